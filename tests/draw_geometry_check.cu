// Host-side check of the final draw's cluster geometry (draw_geometry() in
// finish_kernel.cuh), compiled with nvcc and run on the CPU: the CTAs per
// draw (16, 8 or 4) by batch size, one wave for batches up to the SM count,
// the merge capacity at the largest depth, the slice table, and a result for
// every vocabulary the calls accept.
#include <cstdio>

#include "finish_kernel.cuh"

using namespace sv;

static int g_fail = 0;

static void expect(bool ok, const char *what, int64_t draws, int V, int e)
{
    if (!ok) {
        ++g_fail;
        std::printf("FAIL %s: draws %lld V %d elem %d\n", what, (long long)draws, V, e);
    }
}

int main()
{
    const int64_t sms = 148;  // B300
    const int Vs[] = {1, 7, 1000, 4099, 18992, 32000, 128000, 151936, 262144, 1 << 20,
                      kMaxVocab};
    const int64_t draws_set[] = {1, 2, 4, 8, 16, 18, 19, 32, 37, 38, 64, 74, 75, 100, 128,
                                 148, 149, 256, 1024, 4096};
    long long cases = 0;
    for (int e : {2, 4})
        for (int V : Vs)
            for (int64_t draws : draws_set) {
                FinishParams fp{};
                const bool ok = draw_geometry(fp, draws, V, e, sms);
                ++cases;
                expect(ok, "a geometry for every vocabulary the calls accept", draws, V, e);
                if (!ok)
                    continue;
                const int gran = 16 / e, ncl = fp.ncl;
                expect(ncl == 4 || ncl == 8 || ncl == 16, "4, 8 or 16 CTAs per draw", draws, V,
                       e);
                // rows 0..2K of a request at K = kMaxDraft: two per warp of the
                // cluster, then one per warp of each CTA
                expect(2 * kSampleWarps * ncl + kSampleWarps >= 2 * kMaxDraft + 1,
                       "merge capacity at the largest depth", draws, V, e);
                expect(fp.R % gran == 0 && (int64_t)fp.R * ncl >= V &&
                           (int64_t)fp.R * (ncl - 1) < V + (int64_t)gran * ncl,
                       "ranges cover the row", draws, V, e);
                const bool dense = draws * ncl > 2 * sms;
                expect(fp.slice >= 1 && fp.slice <= fp.R &&
                           (int64_t)fp.slice * e <= kStageRowBytes,
                       "slice within the range and the stage", draws, V, e);
                expect((fp.R + fp.slice - 1) / fp.slice <= kMaxSlices, "slice table", draws, V,
                       e);
                expect(fp.stage_smem % 128 == 0 && fp.stage_smem >= fp.slice * e,
                       "staging buffer", draws, V, e);
                expect(fp.pv % 2 == 1 && (int64_t)fp.pv * kSampleThreads * 16 >= fp.slice * e,
                       "thread pieces cover a slice (odd count)", draws, V, e);
                if (dense && (fp.R + kStageRowBytes / 2 / e - 1) / (kStageRowBytes / 2 / e) <=
                                 kMaxSlices)
                    expect((int64_t)fp.slice * e <= kStageRowBytes / 2,
                           "a dense grid stages half slices", draws, V, e);
                // the rule, where the vocabulary does not force more CTAs
                if (V <= 262144) {
                    const int want = draws * 16 <= 2 * sms ? 16 : draws * 8 <= 4 * sms ? 8 : 4;
                    expect(ncl == want, "CTAs per draw by batch size", draws, V, e);
                    if (draws <= sms)
                        expect(draws * ncl <= (dense ? 4 : 2) * sms, "one wave", draws, V, e);
                }
            }
    // the geometries behind the measurements (bf16, V = 151936): CTAs per
    // draw and the slice (a whole range when it fits the stage: 48 KB, or
    // 24 KB on a dense grid)
    struct Pin {
        int64_t draws;
        int ncl, slice_kb;
    } pins[] = {{16, 16, 18}, {32, 8, 37}, {64, 8, 24}, {128, 4, 24}};
    for (const Pin &q : pins) {
        FinishParams fp{};
        draw_geometry(fp, q.draws, 151936, 2, sms);
        const int kb = (int)((int64_t)fp.slice * 2 / 1024);
        if (fp.ncl != q.ncl || kb != q.slice_kb) {
            ++g_fail;
            std::printf("FAIL pinned geometry: B %lld: %d CTAs, %d KB slices; expected %d, %d\n",
                        (long long)q.draws, fp.ncl, kb, q.ncl, q.slice_kb);
        }
    }
    std::printf("cases %lld failures %d\n", cases, g_fail);
    return g_fail != 0;
}
