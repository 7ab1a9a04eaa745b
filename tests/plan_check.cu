// Host-side check of the streaming pass's unit planner (plan() in
// verify_params.cuh), compiled with nvcc and run on the CPU: the split's
// invariants over many shapes, the short-pass rule, and the unit sizes that
// the B300 measurements behind the rule chose.
#include <cstdio>

#include "verify_params.cuh"

using namespace sv;

static int g_fail = 0;

static void expect(bool ok, const char *what, int64_t rows, int V, int elem)
{
    if (!ok) {
        ++g_fail;
        std::printf("FAIL %s: rows %lld V %d elem %d\n", what, (long long)rows, V, elem);
    }
}

int main()
{
    const int P = 148 * 3 * 8;  // B300: 148 SMs, 3 CTAs of 8 warps each
    const int Vs[] = {1, 7, 1000, 1024, 4099, 12345, 18992, 32000, 128000, 151936, 262144};
    const int64_t rows_set[] = {1, 7, 36, 112, 244, 290, 510, 576, 1088, 1142, 2278, 8000};
    long long cases = 0;
    for (int elem : {2, 4})
        for (int V : Vs)
            for (int64_t rows : rows_set) {
                const Geometry g = plan(rows, rows, V, elem, P);
                const int gran = 16 / elem, qmax = kPieceBytesMax / elem;
                const int v_up = (V + gran - 1) / gran * gran;
                ++cases;
                expect(g.Q >= gran && g.Q % gran == 0, "Q a multiple of the 16-byte granule",
                       rows, V, elem);
                expect(g.Q <= qmax && g.Q <= v_up, "Q within the largest unit and the row", rows,
                       V, elem);
                expect(g.cpr == (V + g.Q - 1) / g.Q, "units per row", rows, V, elem);
                expect((int64_t)(g.cpr - 1) * g.Q < V, "no empty unit at a row's end", rows, V,
                       elem);
                expect(g.U == rows * g.cpr, "units", rows, V, elem);
                expect(g.P >= 1 && g.P <= P && g.P <= g.U, "warps", rows, V, elem);
                expect(g.nt == rows && g.max_rows == rows && g.slots == 0, "index space", rows,
                       V, elem);
                // the busiest warp at the largest unit; a short pass takes that unit
                const int qs = qmax < v_up ? qmax : v_up;
                const int64_t per_s = (rows * ((V + qs - 1) / qs) + g.P - 1) / g.P;
                const int64_t per = (g.U + g.P - 1) / g.P;
                expect(per >= per_s, "no unit beats the largest on the busiest warp", rows, V,
                       elem);
                if (per_s <= kShortPassUnits)
                    expect(g.Q == qs, "a short pass takes the largest unit", rows, V, elem);
            }
    // draft slots follow the target rows in the index space
    {
        const Geometry g = plan(576, 320, 128000, 2, P);
        expect(g.nt == 320 && g.slots == 256, "draft slots after the target rows", 576, 128000,
               2);
    }
    // the unit sizes behind the measured rule (bf16 rows, B300's 3552 warps)
    struct Pin {
        int64_t rows;
        int V, Q;
    } pins[] = {
        {576, 128000, 2048},   // D-cut verification: 11 units a warp, a short pass
        {244, 151936, 2048},   // B = 16, V = 151936: short
        {2278, 151936, 2000},  // B = 128, V = 151936 at T > 0: bytes, 49 units a warp
        {1142, 151936, 1976},  // B = 64 at T > 0: bytes, 25 units a warp
        {544, 151936, 1952},   // B = 32, K = 16 at T = 0: 12 a warp, bytes (4 KB was slower)
    };
    for (const Pin &q : pins) {
        const Geometry g = plan(q.rows, q.rows, q.V, 2, P);
        if (g.Q != q.Q) {
            ++g_fail;
            std::printf("FAIL pinned unit: rows %lld V %d: Q %d, expected %d\n",
                        (long long)q.rows, q.V, g.Q, q.Q);
        }
    }
    std::printf("cases %lld failures %d\n", cases, g_fail);
    return g_fail != 0;
}
