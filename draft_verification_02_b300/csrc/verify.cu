// verify.cu - batched draft verification on sm_103a.
//
// What is computed (per request i with K drafted tokens x_0..x_{K-1}, target
// rows t_0..t_K and, at T > 0, draft rows d_0..d_{K-1}):
//   T = 0: g_j = lowest argmax of t_j; a = first j with x_j != g_j (else K);
//          emit x_0..x_{a-1}, g_a.
//   T > 0: p_j = softmax(t_j / T), q_j = softmax(d_j / T); accept j iff
//          u_j < p_j(x_j) / q_j(x_j); a = first rejection (else K); the final
//          token is the inverse CDF at u_final of w = max(0, p_a - q_a) (or of
//          p_K when every draft is accepted).
// The pages state the procedure (verify the drafted block in one target pass
// by rejection sampling, keep the accepted prefix plus one more token;
// "Tencent Hunyuan Turns Speculative Decoding Into a Full Open-Source Stack",
// "What problem does it solve") and that it is lossless ("Tencent ...
// AngelSpec ...", "Qu'est-ce que le speculative decoding"); the accept and
// residual formulas are the standard ones (Leviathan, Kalman & Matias 2023,
// "Speculative Sampling").
//
// Kernel 1, stream_kernel: the HBM-bound pass.  Every row that must be read
// (all target rows; at T > 0 all draft rows) is cut into units of Q elements;
// the units, in row order, are split into P contiguous, equal ranges, one per
// warp of a persistent grid (a few CTAs per SM).  Each warp keeps a ring of
// kRing units in flight with 1-D TMA bulk copies (cp.async.bulk into shared
// memory, mbarrier completion, bounded waits) and reduces each unit from
// registers: T > 0 takes the maximum with packed bf16x2 max, then sums
// exp2(x*c - m*c) with one FFMA + ex2.approx + FADD per element (the rounding
// of m*c is corrected exactly once per unit); T = 0 keeps the lowest index of
// the maximum.  No fp64 on this path (B300's fp64 rate is a small fraction of
// its fp32 rate).  Every (row, warp) segment leaves one partial.
// Kernel 2, finish_kernel: one CTA per (request, draw chunk), launched as a
// programmatic dependent of kernel 1 so its launch overlaps kernel 1's tail.
// Each CTA merges its request's partials in a fixed order (identical in every
// CTA of the request), runs the accept test and the first-rejection ballot,
// then sums the final-draw weights of its chunk; the request's last CTA
// (atomic ticket) picks the chunk holding u*S and scans inside it.
// Every merge runs in a fixed order, so repeated calls give identical bits.
#include <algorithm>
#include <cfloat>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace sv {

// ---------------------------------------------------------------------------
// parameters
// ---------------------------------------------------------------------------

struct Geometry {  // the unit split of kernel 1, needed by kernel 2 to find partials
    int64_t max_rows;  // target rows (host bound)
    int64_t U;         // units
    int cpr;           // units per row
    int Q;             // elements per unit (the last unit of a row may be shorter)
    int P;             // warp workers
};

struct StreamParams {
    const void *target;
    const void *draft;
    const int32_t *cu;
    int32_t *out_tokens;
    int32_t *out_len;
    int B, V;
    int64_t draft_slots;  // draft rows read (packed index space); 0 at T = 0
    int draft_stride;
    Geometry g;
    int tma;
    int piece_smem;  // bytes per ring slot (multiple of 128)
    float c;         // log2(e) / T
    uint32_t *status;
    uint32_t *cu_flag;
    Partial *part;
};

struct FinishParams {
    const void *target;
    const void *draft;
    const int32_t *tokens;
    const int32_t *cu;
    const float *u_accept;
    const float *u_final;
    int32_t *out_tokens;
    int32_t *out_len;
    float *out_p;
    float *out_q;
    int B, V;
    int64_t draft_rows;  // rows the draft side may index
    int draft_stride;
    Geometry g;
    int NC;          // draw chunks per row
    int nce;         // elements per draw chunk
    int chunk_smem;  // bytes per staged draw chunk (multiple of 128)
    int tma;
    float c;
    uint32_t *status;
    const uint32_t *cu_flag;
    uint32_t *cnt2;
    const Partial *part;
    double *part2;
};

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// 2^x on the SFU (PTX ex2.approx.ftz.f32); results below 2^-126 flush to 0.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Owner warp of unit u when warp w owns units [w*U/P, (w+1)*U/P).
__device__ __forceinline__ int owner_of(int64_t u, const Geometry &g)
{
    return (int)(((u + 1) * (int64_t)g.P - 1) / g.U);
}

// The unit sums use exp2(x*c - fl(m*c)) = exp2((x - m)*c) * 2^-(fl(m*c) - m*c);
// this returns the factor 2^(fl(m*c) - m*c) that undoes the rounding.  The
// rounding error fl(m*c) - m*c is exact as -fma(m, c, -fl(m*c)) and below
// 2^-17 in magnitude, so 1 + delta*ln2 is the factor to fp32 precision.
__device__ __forceinline__ float mc_correction(float m, float mc, float c)
{
    const float delta = -fmaf(m, c, -mc);
    return fmaf(delta, 0.69314718f, 1.0f);
}

// 2^x for x <= 0 given in fp64: split x = n + f exactly (n integer, f in
// [0,1)), take 2^f with CUDA's exp2f (2 ulp) and scale by 2^n.  A handful of
// fp64 operations instead of a full fp64 exp2.
__device__ __forceinline__ float exp2_split(double x)
{
    if (x < -200.0)
        return 0.f;
    const double n = floor(x);
    return ldexpf(exp2f((float)(x - n)), (int)n);
}

__device__ __forceinline__ int64_t draft_index(int draft_stride, const int32_t *cu, int i, int j)
{
    return draft_stride > 0 ? (int64_t)i * draft_stride + j : (int64_t)__ldg(cu + i) + j;
}

__device__ __forceinline__ double qnan_d() { return __longlong_as_double(0x7ff8000000000000ll); }

// ---------------------------------------------------------------------------
// kernel 1: stream the rows
// ---------------------------------------------------------------------------

#ifndef SV_RING
#define SV_RING 3
#endif
#ifndef SV_STREAM_CTAS_PER_SM
#define SV_STREAM_CTAS_PER_SM 2
#endif
constexpr int kRing = SV_RING;
constexpr int kStreamWarps = 8;
constexpr int kStreamThreads = kStreamWarps * 32;

// Per-lane running state of one row segment.  The running sum is fp32 with
// Kahan compensation: one term per unit.
struct LaneAcc {
    float m;     // running max (T > 0) / best value (T = 0)
    float s;     // running sum of exp2((x - m) c)  (T > 0)
    float comp;  // Kahan compensation of s
    int idx;     // best index (T = 0)
    int nan;     // a NaN was seen (T = 0)
};

// Fold a unit's maximum pm into the running (m, s); false when nothing more
// is to be summed (NaN, all masked, or +inf - the merge flags those rows).
__device__ __forceinline__ bool fold_max(LaneAcc &a, float pm, float c)
{
    const float mn = max_nan(a.m, pm);
    if (mn != mn) {
        a.m = mn;
        a.s = __int_as_float(0x7fc00000);
        return false;
    }
    if (mn > a.m) {
        if (a.m != -INFINITY) {
            const float f = exp2f((a.m - mn) * c);
            a.s *= f;
            a.comp *= f;
        }
        a.m = mn;
    }
    return a.m != -INFINITY && a.m != INFINITY && a.s == a.s;
}

// Add one unit's sum (taken relative to fl(m c)) to the running sum.
__device__ __forceinline__ void add_unit(LaneAcc &a, float unit_sum, float mc, float c)
{
    const float y = unit_sum * mc_correction(a.m, mc, c) - a.comp;
    const float t = a.s + y;
    a.comp = (t - a.s) - y;
    a.s = t;
}

// One unit of bf16 data at T > 0 from shared memory (lane-strided 16-byte
// vectors held in registers between the max and the sum); a tail that is not
// a whole vector (plain-load path only) is handled element-wise.
template <int MAXV>
__device__ __forceinline__ void unit_softmax_bf16(const uint16_t *buf, int len, float c,
                                                  LaneAcc &a)
{
    const int lane = threadIdx.x & 31;
    const uint4 *vb = reinterpret_cast<const uint4 *>(buf);
    const int nvec = len >> 3;
    uint4 r[MAXV];
    uint32_t hm = 0xff80ff80u;  // (-inf, -inf)
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const int v = lane + 32 * t;
        if (v < nvec) {
            r[t] = vb[v];
            hm = max_nan_bf16x2(hm, r[t].x);
            hm = max_nan_bf16x2(hm, r[t].y);
            hm = max_nan_bf16x2(hm, r[t].z);
            hm = max_nan_bf16x2(hm, r[t].w);
        }
    }
    float pm = max_nan(bf16_lo(hm), bf16_hi(hm));
    for (int k = nvec * 8 + lane; k < len; k += 32)
        pm = max_nan(pm, bf16_lo((uint32_t)buf[k]));
    if (!fold_max(a, pm, c))
        return;
    const float mc = a.m * c;
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const int v = lane + 32 * t;
        if (v < nvec) {
            const uint32_t w4[4] = {r[t].x, r[t].y, r[t].z, r[t].w};
            float e[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                e[2 * h] = ex2_approx(fmaf(bf16_lo(w4[h]), c, -mc));
                e[2 * h + 1] = ex2_approx(fmaf(bf16_hi(w4[h]), c, -mc));
            }
            acc += ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
        }
    }
    for (int k = nvec * 8 + lane; k < len; k += 32)
        acc += ex2_approx(fmaf(bf16_lo((uint32_t)buf[k]), c, -mc));
    add_unit(a, acc, mc, c);
}

template <int MAXV>
__device__ __forceinline__ void unit_softmax_f32(const float *buf, int len, float c, LaneAcc &a)
{
    const int lane = threadIdx.x & 31;
    const float4 *vb = reinterpret_cast<const float4 *>(buf);
    const int nvec = len >> 2;
    float4 r[MAXV];
    float pm = -INFINITY;
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const int v = lane + 32 * t;
        if (v < nvec) {
            r[t] = vb[v];
            pm = max_nan(pm, max_nan(max_nan(r[t].x, r[t].y), max_nan(r[t].z, r[t].w)));
        }
    }
    for (int k = nvec * 4 + lane; k < len; k += 32)
        pm = max_nan(pm, buf[k]);
    if (!fold_max(a, pm, c))
        return;
    const float mc = a.m * c;
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const int v = lane + 32 * t;
        if (v < nvec) {
            const float e0 = ex2_approx(fmaf(r[t].x, c, -mc));
            const float e1 = ex2_approx(fmaf(r[t].y, c, -mc));
            const float e2 = ex2_approx(fmaf(r[t].z, c, -mc));
            const float e3 = ex2_approx(fmaf(r[t].w, c, -mc));
            acc += (e0 + e1) + (e2 + e3);
        }
    }
    for (int k = nvec * 4 + lane; k < len; k += 32)
        acc += ex2_approx(fmaf(buf[k], c, -mc));
    add_unit(a, acc, mc, c);
}

// T = 0: lowest index of the maximum.  Each lane visits its elements in
// increasing index order, so a strict > keeps the lowest index.
template <int MAXV>
__device__ __forceinline__ void unit_argmax_bf16(const uint16_t *buf, int len, int col0,
                                                 LaneAcc &a)
{
    const int lane = threadIdx.x & 31;
    const uint4 *vb = reinterpret_cast<const uint4 *>(buf);
    const int nvec = len >> 3;
    uint4 r[MAXV];
    uint32_t hm = 0xff80ff80u;
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const int v = lane + 32 * t;
        if (v < nvec) {
            r[t] = vb[v];
            hm = max_nan_bf16x2(hm, r[t].x);
            hm = max_nan_bf16x2(hm, r[t].y);
            hm = max_nan_bf16x2(hm, r[t].z);
            hm = max_nan_bf16x2(hm, r[t].w);
        }
    }
    const float pm = max_nan(bf16_lo(hm), bf16_hi(hm));
    if (pm != pm) {
        a.nan = 1;
    } else if (pm > a.m) {  // locate the first element equal to the new maximum
        int found = INT_MAX;
#pragma unroll
        for (int t = 0; t < MAXV; ++t) {
            const int v = lane + 32 * t;
            if (v < nvec && found == INT_MAX) {
                const uint32_t w4[4] = {r[t].x, r[t].y, r[t].z, r[t].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    if (found == INT_MAX && bf16_lo(w4[h]) == pm)
                        found = v * 8 + 2 * h;
                    if (found == INT_MAX && bf16_hi(w4[h]) == pm)
                        found = v * 8 + 2 * h + 1;
                }
            }
        }
        a.m = pm;
        a.idx = col0 + found;
    }
    for (int k = nvec * 8 + lane; k < len; k += 32) {  // tail (plain path), in order
        const float x = bf16_lo((uint32_t)buf[k]);
        if (x != x)
            a.nan = 1;
        else if (x > a.m) {
            a.m = x;
            a.idx = col0 + k;
        }
    }
}

template <int MAXV>
__device__ __forceinline__ void unit_argmax_f32(const float *buf, int len, int col0, LaneAcc &a)
{
    const int lane = threadIdx.x & 31;
    const float4 *vb = reinterpret_cast<const float4 *>(buf);
    const int nvec = len >> 2;
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const int v = lane + 32 * t;
        if (v < nvec) {
            const float4 q = vb[v];
            const float x4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (x4[h] != x4[h])
                    a.nan = 1;
                else if (x4[h] > a.m) {
                    a.m = x4[h];
                    a.idx = col0 + v * 4 + h;
                }
            }
        }
    }
    for (int k = nvec * 4 + lane; k < len; k += 32) {
        const float x = buf[k];
        if (x != x)
            a.nan = 1;
        else if (x > a.m) {
            a.m = x;
            a.idx = col0 + k;
        }
    }
}

// Reduce the lanes' state of a finished row segment, store its partial and
// reset the state.
template <bool GREEDY>
__device__ __forceinline__ void store_partial(LaneAcc &a, float c, Partial *slot)
{
    const int lane = threadIdx.x & 31;
    Partial out;
    if (GREEDY) {
        float best = a.m;
        int bidx = a.idx;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
            if (ob > best || (ob == best && oi < bidx)) {
                best = ob;
                bidx = oi;
            }
        }
        const int nan = __any_sync(0xffffffffu, a.nan);
        out.m = best;
        out.idx = nan ? -2 : (bidx == INT_MAX ? -1 : bidx);
        out.s = 0.0;
    } else {
        const float m = warp_max_nan(a.m);
        double s = 0.0;
        if (m == m && m != -INFINITY && m != INFINITY) {
            if (a.s != 0.f)
                s = (double)(a.s - a.comp) * (double)exp2f((a.m - m) * c);
        } else if (m != -INFINITY) {
            s = qnan_d();
        }
        s = warp_sum_d(s);
        out.m = m;
        out.idx = 0;
        out.s = s;
    }
    if (lane == 0)
        *slot = out;
    a.m = -INFINITY;
    a.s = 0.f;
    a.comp = 0.f;
    a.idx = INT_MAX;
    a.nan = 0;
}

template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kStreamThreads, SV_STREAM_CTAS_PER_SM)
    stream_kernel(const StreamParams p)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t bars[kStreamWarps][kRing];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int w = blockIdx.x * kStreamWarps + wib;
    const Geometry g = p.g;
    const int B = p.B, V = p.V;
    unsigned char *ring = dsm + (size_t)wib * kRing * p.piece_smem;
    int32_t *cu_s = reinterpret_cast<int32_t *>(dsm + (size_t)kStreamWarps * kRing * p.piece_smem);
    constexpr int MAXV = (kPieceBytesMax / 16 + 31) / 32;  // 16-byte vectors per lane per unit

    pdl_trigger();  // the finish kernel may launch now; it waits for this grid to complete
    if (lane == 0) {
        for (int k = 0; k < kRing; ++k)
            mbar_init(&bars[wib][k], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int64_t u0 = w < g.P ? (int64_t)w * g.U / g.P : 0;
    const int64_t u1 = w < g.P ? (int64_t)(w + 1) * g.U / g.P : 0;
    const T *tbase = reinterpret_cast<const T *>(p.target);
    const T *dbase = reinterpret_cast<const T *>(p.draft);
    const bool padded = !GREEDY && p.draft_stride > 0;

    // Where the unit at (row rg, column chunk q) comes from; false when the
    // row lies past the real rows (nt target, nd draft) and `check` is set.
    auto locate = [&](int64_t rg, int q, const T *&src, int &len, int &col0, int64_t nt,
                      int64_t nd, bool check) -> bool {
        col0 = q * g.Q;
        len = min(g.Q, V - col0);
        if (rg < g.max_rows) {
            if (check && rg >= nt)
                return false;
            src = tbase + rg * (int64_t)V + col0;
            return true;
        }
        const int64_t slot = rg - g.max_rows;
        if (check && slot >= nd)
            return false;
        int64_t row = slot;
        if (padded) {  // packed slot -> (request, position) -> padded row
            int lo = 0, hi = B - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (cu_s[mid] <= slot)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            row = (int64_t)lo * p.draft_stride + (slot - cu_s[lo]);
        }
        src = dbase + row * (int64_t)V + col0;
        return true;
    };

    uint32_t issued = 0, phase = 0;
    auto issue = [&](int64_t rg, int q, int k, int64_t nt, int64_t nd, bool check) {
        const T *src;
        int len, col0;
        if (!locate(rg, q, src, len, col0, nt, nd, check))
            return;
        T *dst = reinterpret_cast<T *>(ring + (size_t)k * p.piece_smem);
        if (p.tma) {
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                const uint32_t bytes = (uint32_t)len * (uint32_t)sizeof(T);
                mbar_arrive_expect_tx(&bars[wib][k], bytes);
                bulk_g2s(dst, src, bytes, &bars[wib][k]);
            }
        } else {
            for (int e = lane; e < len; e += 32)
                dst[e] = src[e];
            __syncwarp();
        }
        issued |= 1u << k;
    };

    // cursors: (row, column chunk) of the next unit to consume and to issue
    int64_t c_rg = u0 / g.cpr;
    int c_q = (int)(u0 - c_rg * g.cpr);
    int64_t i_rg = c_rg;
    int i_q = c_q;
    const int64_t n_units = u1 - u0;
    auto advance = [&](int64_t &rg, int &q) {
        if (++q == g.cpr) {
            q = 0;
            ++rg;
        }
    };

    // Packed rows have known addresses: their first copies start before the
    // offsets arrive (the offsets only tell which rows past the real count
    // to skip).  Padded draft rows need the offsets first.
    int64_t nt = g.max_rows, nd = p.draft_slots;
    int n_issued = 0;
    if (!padded)
        for (; n_issued < kRing && n_issued < n_units; ++n_issued) {
            issue(i_rg, i_q, n_issued, nt, nd, false);
            advance(i_rg, i_q);
        }
    // CTA 0 validates the offsets for both kernels (and every CTA does when
    // it maps padded rows through them).
    if (padded || blockIdx.x == 0) {
        int bad = 0;
        for (int k = threadIdx.x; k <= B; k += kStreamThreads) {
            const int v = __ldg(p.cu + k);
            if (padded)
                cu_s[k] = v;
            if (k < B) {
                const int K = __ldg(p.cu + k + 1) - v;
                if (K < 0 || K > kMaxDraft || (p.draft_stride > 0 && K > p.draft_stride))
                    bad = 1;
            } else if ((int64_t)v + B > g.max_rows) {
                bad = 1;
            }
            if (k == 0 && v != 0)
                bad = 1;
        }
        bad = __syncthreads_or(bad);
        if (blockIdx.x == 0) {
            if (threadIdx.x == 0) {
                *p.cu_flag = bad ? 0u : 1u;
                if (bad)
                    set_status(p.status, ST_INVALID);
            }
            if (bad) {
                for (int64_t k = threadIdx.x; k < g.max_rows; k += kStreamThreads)
                    p.out_tokens[k] = -1;
                for (int k = threadIdx.x; k < B; k += kStreamThreads)
                    p.out_len[k] = -1;
            }
        }
        if (bad) {  // malformed offsets: drain the copies in flight, read nothing more
            if (p.tma)
                for (int k = 0; k < kRing; ++k)
                    if (issued >> k & 1)
                        mbar_wait_bounded(&bars[wib][k], 0);
            return;
        }
    }
    {
        int v = lane == 0 ? __ldg(p.cu + B) : 0;
        v = __shfl_sync(0xffffffffu, v, 0);
        nd = min(nd, (int64_t)v);
        nt = min(g.max_rows, (int64_t)v + B);
    }
    if (padded)
        for (; n_issued < kRing && n_issued < n_units; ++n_issued) {
            issue(i_rg, i_q, n_issued, nt, nd, true);
            advance(i_rg, i_q);
        }

    LaneAcc acc{-INFINITY, 0.f, 0.f, INT_MAX, 0};
    bool seg_active = false;
    int k = 0;  // ring slot of the unit being consumed
    for (int64_t n = 0; n < n_units; ++n) {
        const T *src;
        int len, col0;
        const int64_t rg = c_rg;
        const bool live = locate(c_rg, c_q, src, len, col0, nt, nd, true);
        if (issued >> k & 1) {
            if (p.tma) {
                const bool ok = mbar_wait_bounded(&bars[wib][k], phase >> k & 1);
                if (__any_sync(0xffffffffu, !ok)) {
                    // a copy never completed: flag it, give every copy still in
                    // flight one more bounded wait, and stop (the finish kernel
                    // poisons the outputs when it sees the flag)
                    if (lane == 0)
                        set_status(p.status, ST_TIMEOUT);
                    for (int kk = 0; kk < kRing; ++kk)
                        if (issued >> kk & 1)
                            mbar_wait_bounded(&bars[wib][kk], phase >> kk & 1);
                    return;
                }
                phase ^= 1u << k;
            }
            issued &= ~(1u << k);
            if (live) {
                const T *buf = reinterpret_cast<const T *>(ring + (size_t)k * p.piece_smem);
                if constexpr (GREEDY) {
                    if constexpr (sizeof(T) == 2)
                        unit_argmax_bf16<MAXV>(reinterpret_cast<const uint16_t *>(buf), len, col0,
                                               acc);
                    else
                        unit_argmax_f32<MAXV>(reinterpret_cast<const float *>(buf), len, col0,
                                              acc);
                } else {
                    if constexpr (sizeof(T) == 2)
                        unit_softmax_bf16<MAXV>(reinterpret_cast<const uint16_t *>(buf), len, p.c,
                                                acc);
                    else
                        unit_softmax_f32<MAXV>(reinterpret_cast<const float *>(buf), len, p.c,
                                               acc);
                }
                seg_active = true;
            }
        }
        __syncwarp();  // every lane is done with slot k before it is refilled
        if (n_issued < n_units) {
            issue(i_rg, i_q, k, nt, nd, true);
            advance(i_rg, i_q);
            ++n_issued;
        }
        advance(c_rg, c_q);
        const bool row_ends = (n + 1 == n_units) || (c_rg != rg);
        if (row_ends && seg_active) {
            store_partial<GREEDY>(acc, p.c, p.part + rg + w);
            seg_active = false;
        }
        if (++k == kRing)
            k = 0;
    }
}

// ---------------------------------------------------------------------------
// kernel 2: merge, accept test, final draw
// ---------------------------------------------------------------------------

constexpr int kFinishThreads = 256;
constexpr int kFinishWarps = kFinishThreads / 32;

// Merge the partials of flattened row rg (one warp), T > 0: (m, s) with
// s = sum_v exp2((x_v - m) c).
__device__ __forceinline__ void merge_softmax_row(const FinishParams &p, int64_t rg, float &m_out,
                                                  double &s_out)
{
    const int lane = threadIdx.x & 31;
    const int64_t ua = rg * p.g.cpr, ub = ua + p.g.cpr - 1;
    const int wf = owner_of(ua, p.g), wl = owner_of(ub, p.g);
    float m = -INFINITY;
    for (int w = wf + lane; w <= wl; w += 32)
        m = max_nan(m, __ldcg(&p.part[rg + w].m));
    m = warp_max_nan(m);
    double s = 0.0;
    for (int w = wf + lane; w <= wl; w += 32) {
        const double sw = __ldcg(&p.part[rg + w].s);
        if (sw != 0.0)
            s += sw * (double)exp2f((__ldcg(&p.part[rg + w].m) - m) * p.c);
    }
    s = warp_sum_d(s);
    m_out = m;
    s_out = s;
}

// T = 0: lowest argmax of target row rg; -1 masked row, -2 NaN, -3 +inf.
__device__ __forceinline__ int merge_argmax_row(const FinishParams &p, int64_t rg)
{
    const int lane = threadIdx.x & 31;
    const int64_t ua = rg * p.g.cpr, ub = ua + p.g.cpr - 1;
    const int wf = owner_of(ua, p.g), wl = owner_of(ub, p.g);
    float best = -INFINITY;
    int bidx = INT_MAX, nan = 0;
    for (int w = wf + lane; w <= wl; w += 32) {
        const float m = __ldcg(&p.part[rg + w].m);
        const int ix = __ldcg(&p.part[rg + w].idx);
        if (ix == -2)
            nan = 1;
        else if (ix >= 0 && (m > best || (m == best && ix < bidx))) {
            best = m;
            bidx = ix;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (ob > best || (ob == best && oi < bidx)) {
            best = ob;
            bidx = oi;
        }
    }
    nan = __any_sync(0xffffffffu, nan);
    return nan ? -2 : (bidx == INT_MAX ? -1 : (best == INFINITY ? -3 : bidx));
}

__device__ __forceinline__ bool row_ok(float m, double s)
{
    return isfinite(m) && isfinite(s) && s > 0.0;
}

struct DrawCtx {
    bool resid;
    float c, mct, mcd;  // c and fl(m c) of the two rows
    float sc_t, sc_d;   // 2^(fl(m c) - m c) / s: normalisers including the rounding fix
};

// Final-draw weight of one element (pair).
__device__ __forceinline__ float draw_w(const DrawCtx &d, float t, float x)
{
    const float pt = ex2_approx(fmaf(t, d.c, -d.mct));
    if (!d.resid)
        return pt;  // bonus draw (or all-zero residual): unnormalised p
    const float pd = ex2_approx(fmaf(x, d.c, -d.mcd));
    return fmaxf(pt * d.sc_t - pd * d.sc_d, 0.f);
}

template <typename T>
__device__ __forceinline__ int stage_chunk(const FinishParams &p, const T *trow, const T *drow,
                                           bool resid, int c, T *tb, T *db, uint64_t *bar,
                                           uint32_t &phase)
{
    const int col0 = c * p.nce;
    const int len = min(p.nce, p.V - col0);
    // earlier readers of the buffers are done; once any copy of this call has
    // timed out, nothing more is copied (the request's outputs are poisoned)
    if (__syncthreads_or(threadIdx.x == 0 && (read_status(p.status) & ST_TIMEOUT)))
        return len;
    if (p.tma) {
        if (threadIdx.x == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint32_t bytes = (uint32_t)len * (uint32_t)sizeof(T);
            mbar_arrive_expect_tx(bar, resid ? 2 * bytes : bytes);
            bulk_g2s(tb, trow + col0, bytes, bar);
            if (resid)
                bulk_g2s(db, drow + col0, bytes, bar);
        }
        if (!mbar_wait_bounded(bar, phase)) {
            set_status(p.status, ST_TIMEOUT);
            mbar_wait_bounded(bar, phase);  // the copy in flight, once more
        }
        phase ^= 1u;
    } else {
        for (int k = threadIdx.x; k < len; k += kFinishThreads) {
            tb[k] = trow[col0 + k];
            if (resid)
                db[k] = drow[col0 + k];
        }
        __syncthreads();
    }
    return len;
}

template <typename T>
__device__ __forceinline__ float draw_at(const DrawCtx &d, const T *tb, const T *db, int k)
{
    return draw_w(d, Elem<T>::at(tb, k), d.resid ? Elem<T>::at(db, k) : 0.f);
}

// Sum of the draw weights of a staged chunk (thread-strided fp32, then fp64
// across threads in a fixed order).
template <typename T>
__device__ __forceinline__ double chunk_sum(const DrawCtx &d, const T *tb, const T *db, int len,
                                            double *red)
{
    float acc = 0.f;
    for (int k = threadIdx.x; k < len; k += kFinishThreads)
        acc += draw_at(d, tb, db, k);
    return block_sum_d((double)acc, red);
}

// Smallest k of the staged chunk with base + C(k) > target, C the running sum
// in index order; when rounding leaves none, the last k with weight > 0.
// Warps own contiguous segments; in the segment holding the target, 32
// consecutive elements are scanned per step with a warp prefix sum.
template <typename T>
__device__ int chunk_search(const DrawCtx &d, const T *tb, const T *db, int len, double base,
                            double target, double *wtot, int *s_res)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = (len + kFinishWarps - 1) / kFinishWarps;
    const int k0 = min(len, warp * seg), k1 = min(len, k0 + seg);
    float acc = 0.f;
    for (int k = k0 + lane; k < k1; k += 32)
        acc += draw_at(d, tb, db, k);
    const double tot = warp_sum_d((double)acc);
    __syncthreads();
    if (lane == 0)
        wtot[warp] = tot;
    if (threadIdx.x == 0)
        *s_res = -1;
    __syncthreads();
    double lo = base;
    int wc = -1;
    for (int w2 = 0; w2 < kFinishWarps; ++w2) {
        if (lo + wtot[w2] > target) {
            wc = w2;
            break;
        }
        lo += wtot[w2];
    }
    if (warp == wc) {
        double run = lo;
        for (int kb = k0; kb < k1; kb += 32) {
            const int k = kb + lane;
            const float x = k < k1 ? draw_at(d, tb, db, k) : 0.f;
            float incl = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += n;
            }
            const unsigned hit =
                __ballot_sync(0xffffffffu, k < k1 && run + (double)incl > target);
            if (hit) {
                if (lane == 0)
                    *s_res = kb + __ffs(hit) - 1;
                break;
            }
            run += (double)__shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncthreads();
    int res = *s_res;
    if (res < 0) {
        int best = -1;
        for (int k = threadIdx.x; k < len; k += kFinishThreads)
            if (draw_at(d, tb, db, k) > 0.f)
                best = k;
        if (best >= 0)
            atomicMax(s_res, best);
        __syncthreads();
        res = *s_res;
    }
    return res;
}

template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kFinishThreads) finish_kernel(const FinishParams p)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    T *tb = reinterpret_cast<T *>(dsm);
    T *db = reinterpret_cast<T *>(dsm + p.chunk_smem);
    __shared__ __align__(8) uint64_t bar;
    __shared__ float row_m[2 * kMaxDraft + 1];
    __shared__ double row_s[2 * kMaxDraft + 1];
    __shared__ int row_g[kMaxDraft + 1];
    __shared__ double red[kFinishWarps];
    __shared__ double s_tot[kMaxChunks];
    __shared__ double s_base, s_target;
    __shared__ int s_a, s_bad, s_last, s_res, s_mode, s_cs;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NC = GREEDY ? 1 : p.NC;
    const int i = blockIdx.x / NC, c = blockIdx.x % NC;

    pdl_wait();  // kernel 1 has completed and its writes are visible
    if (__ldcg(p.cu_flag) == 0u)
        return;  // malformed offsets: kernel 1 poisoned every output
    const int cu_i = __ldg(p.cu + i);
    const int K = __ldg(p.cu + i + 1) - cu_i;
    const int64_t t0 = (int64_t)cu_i + i;
    const int64_t gmr = p.g.max_rows;

    if constexpr (GREEDY) {
        for (int rho = warp; rho <= K; rho += kFinishWarps) {
            const int gj = merge_argmax_row(p, t0 + rho);
            if (lane == 0)
                row_g[rho] = gj;
        }
        __syncthreads();
        if (warp != 0)
            return;
        const bool act = lane < K;
        int x = -1;
        bool bad_tok = false;
        if (act) {
            x = __ldg(p.tokens + draft_index(p.draft_stride, p.cu, i, lane));
            bad_tok = x < 0 || x >= p.V;
        }
        bool bad_nf = false;
        for (int jj = lane; jj <= K; jj += 32)
            bad_nf |= row_g[jj] < 0;
        const unsigned nf = __ballot_sync(0xffffffffu, bad_nf);
        const unsigned bt = __ballot_sync(0xffffffffu, bad_tok);
        const unsigned rej = __ballot_sync(0xffffffffu, act && x != row_g[act ? lane : 0]);
        const bool timeout = read_status(p.status) & ST_TIMEOUT;
        if (nf || bt || timeout) {
            if (lane == 0)
                set_status(p.status, (nf ? ST_NONFINITE : 0u) | (bt ? ST_INVALID : 0u));
            for (int jj = lane; jj <= K; jj += 32)
                p.out_tokens[t0 + jj] = -1;
            if (lane == 0)
                p.out_len[i] = -1;
            return;
        }
        const int a = rej ? __ffs(rej) - 1 : K;
        for (int jj = lane; jj <= K; jj += 32)
            p.out_tokens[t0 + jj] = jj < a ? x : (jj == a ? row_g[a] : -1);
        if (lane == 0)
            p.out_len[i] = a;
        return;
    } else {
        // ---- merge (m, s) of the request's 2K+1 rows
        for (int rho = warp; rho < 2 * K + 1; rho += kFinishWarps) {
            const int64_t rg = rho <= K ? t0 + rho : gmr + cu_i + (rho - K - 1);
            float m;
            double s;
            merge_softmax_row(p, rg, m, s);
            if (lane == 0) {
                row_m[rho] = m;
                row_s[rho] = s;
            }
        }
        __syncthreads();
        // ---- accept test and first rejection (warp 0; identical in every CTA)
        if (warp == 0) {
            const bool act = lane < K;
            int x = -1;
            bool bad_tok = false, bad_nf = false, acc = true;
            double pp = 0.0, qq = 0.0;
            int64_t di = 0;
            if (act) {
                di = draft_index(p.draft_stride, p.cu, i, lane);
                x = __ldg(p.tokens + di);
                if (x < 0 || x >= p.V) {
                    bad_tok = true;
                } else {
                    const float mt = row_m[lane], md = row_m[K + 1 + lane];
                    const double st = row_s[lane], sd = row_s[K + 1 + lane];
                    if (!row_ok(mt, st) || !row_ok(md, sd)) {
                        bad_nf = true;
                    } else {
                        const T *trow = reinterpret_cast<const T *>(p.target) + (t0 + lane) * p.V;
                        const T *drw = reinterpret_cast<const T *>(p.draft) + di * p.V;
                        const double gt = Elem<T>::ld_global(trow, x);
                        const double gd = Elem<T>::ld_global(drw, x);
                        pp = (double)exp2_split((gt - (double)mt) * (double)p.c) / st;
                        qq = (double)exp2_split((gd - (double)md) * (double)p.c) / sd;
                        const double ratio = qq > 0.0 ? pp / qq : (pp > 0.0 ? INFINITY : 0.0);
                        acc = (double)__ldg(p.u_accept + di) < ratio;
                    }
                }
            }
            if (lane == 0 && !row_ok(row_m[K], row_s[K]))
                bad_nf = true;
            const unsigned nf = __ballot_sync(0xffffffffu, bad_nf);
            const unsigned bt = __ballot_sync(0xffffffffu, bad_tok);
            const unsigned rej = __ballot_sync(0xffffffffu, act && !acc);
            // bad depends only on the request's data, so every CTA of the
            // request takes the same branch (and the ticket count stays whole);
            // an expired wait only poisons outputs (best effort)
            const bool bad = nf || bt;
            const bool timeout = read_status(p.status) & ST_TIMEOUT;
            const int a = rej ? __ffs(rej) - 1 : K;
            if (c == 0) {  // the request's outputs, written once
                if (bad || timeout) {
                    if (lane == 0)
                        set_status(p.status, (nf ? ST_NONFINITE : 0u) | (bt ? ST_INVALID : 0u));
                    for (int jj = lane; jj <= K; jj += 32)
                        p.out_tokens[t0 + jj] = -1;
                    if (lane == 0)
                        p.out_len[i] = -1;
                } else {
                    if (act && p.out_p)
                        p.out_p[di] = (float)pp;
                    if (act && p.out_q)
                        p.out_q[di] = (float)qq;
                    for (int jj = lane; jj <= K; jj += 32) {
                        if (jj < a)
                            p.out_tokens[t0 + jj] = x;  // jj == lane since a <= 32
                        else if (jj > a)
                            p.out_tokens[t0 + jj] = -1;
                    }
                    if (lane == 0)
                        p.out_len[i] = a;
                }
            }
            if (lane == 0) {
                s_a = a;
                s_bad = bad;
            }
        }
        __syncthreads();
        if (s_bad)
            return;

        // ---- final draw over chunk c of the rows of position a
        const int a = s_a;
        const int64_t trow_i = t0 + a;
        const int64_t drow_i = a < K ? draft_index(p.draft_stride, p.cu, i, a) : -1;
        if (trow_i >= gmr || drow_i >= p.draft_rows) {  // never with valid offsets
            if (tid == 0)
                set_status(p.status, ST_INVALID);
            return;
        }
        DrawCtx d;
        d.resid = drow_i >= 0;
        d.c = p.c;
        {
            const float mt = row_m[a];
            d.mct = mt * p.c;
            d.sc_t = (float)((double)mc_correction(mt, d.mct, p.c) / row_s[a]);
            if (d.resid) {
                const float md = row_m[K + 1 + a];
                d.mcd = md * p.c;
                d.sc_d = (float)((double)mc_correction(md, d.mcd, p.c) / row_s[K + 1 + a]);
            } else {
                d.mcd = 0.f;
                d.sc_d = 0.f;
            }
        }
        const T *trow = reinterpret_cast<const T *>(p.target) + trow_i * p.V;
        const T *drow = d.resid ? reinterpret_cast<const T *>(p.draft) + drow_i * p.V : nullptr;

        if (tid == 0) {
            mbar_init(&bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        uint32_t phase = 0;
        int len = stage_chunk<T>(p, trow, drow, d.resid, c, tb, db, &bar, phase);
        double tot = chunk_sum<T>(d, tb, db, len, red);
        if (tid == 0) {
            p.part2[(int64_t)i * NC + c] = tot;
            __threadfence();
            s_last = atomicAdd(p.cnt2 + i, 1u) == (uint32_t)NC - 1;
        }
        __syncthreads();
        if (!s_last)
            return;
        __threadfence();
        int staged = c;
        if (tid == 0) {
            p.cnt2[i] = 0;  // ready for the next call
            double S = 0.0;
            for (int cc = 0; cc < NC; ++cc) {
                s_tot[cc] = __ldcg(p.part2 + (int64_t)i * NC + cc);
                S += s_tot[cc];
            }
            s_mode = (d.resid && !(S > 0.0)) ? 1 : 0;  // all-zero residual: draw from p_a
        }
        __syncthreads();
        if (s_mode == 1) {
            d.resid = false;
            for (int cc = 0; cc < NC; ++cc) {
                len = stage_chunk<T>(p, trow, drow, false, cc, tb, db, &bar, phase);
                tot = chunk_sum<T>(d, tb, db, len, red);
                if (tid == 0)
                    s_tot[cc] = tot;
                staged = cc;
            }
            __syncthreads();
        }
        if (tid == 0) {
            double S = 0.0;
            for (int cc = 0; cc < NC; ++cc)
                S += s_tot[cc];
            const double target = (double)__ldg(p.u_final + i) * S;
            double cum = 0.0, base = 0.0, tgt = target;
            int cs = -1;
            for (int cc = 0; cc < NC; ++cc) {
                if (cum + s_tot[cc] > target) {
                    cs = cc;
                    base = cum;
                    break;
                }
                cum += s_tot[cc];
            }
            if (cs < 0) {  // u*S at or past the end after rounding: last chunk with mass
                cs = 0;
                double cum2 = 0.0;
                for (int cc = 0; cc < NC; ++cc) {
                    if (s_tot[cc] > 0.0) {
                        cs = cc;
                        base = cum2;
                    }
                    cum2 += s_tot[cc];
                }
                tgt = INFINITY;
            }
            s_cs = cs;
            s_base = base;
            s_target = tgt;
        }
        __syncthreads();
        const int cs = s_cs;
        if (cs != staged)
            len = stage_chunk<T>(p, trow, drow, d.resid, cs, tb, db, &bar, phase);
        else
            len = min(p.nce, p.V - cs * p.nce);
        const int k = chunk_search<T>(d, tb, db, len, s_base, s_target, red, &s_res);
        if (tid == 0) {
            int y = k >= 0 ? cs * p.nce + k : -1;
            if (y < 0)
                set_status(p.status, ST_NONFINITE);
            if (read_status(p.status) & ST_TIMEOUT) {  // staged data may be stale
                y = -1;
                p.out_len[i] = -1;
                for (int jj = 0; jj <= K; ++jj)
                    p.out_tokens[t0 + jj] = -1;
            }
            p.out_tokens[trow_i] = y;
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static int sm_count()
{
    static int n = [] {
        int dev = 0, v = 148;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            return v;
        return 148;
    }();
    return n;
}

// Unit size for a balanced split: U = rows * ceil(V / Q) units over P warps
// puts ceil(U / P) units on the busiest warp.  Pick the Q (a multiple of the
// 16-byte granule, at most kPieceBytesMax) that minimises the busiest warp's
// elements (plus a fixed per-unit cost), preferring larger Q.
static Geometry plan(int64_t rows_total, int64_t max_rows, int V, int elem, int P_max)
{
    Geometry g{};
    g.max_rows = max_rows;
    const int gran = 16 / elem;
    const int qmax = kPieceBytesMax / elem;
    const int64_t total = rows_total * (int64_t)V;
    int64_t P = P_max;
    const int64_t min_work = 2048 / elem;  // at least ~2 KB per warp
    if (total / min_work < P)
        P = std::max<int64_t>(1, total / min_work);
    double best_cost = 1e300;
    int best_q = qmax;
    for (int q = qmax; q >= gran && q >= qmax / 8; q -= gran) {
        const int64_t cpr = (V + q - 1) / q;
        const int64_t U = rows_total * cpr;
        const int64_t per = (U + P - 1) / P;
        const double cost = (double)per * (double)(std::min<int64_t>(q, V) + 64);
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best_q = q;
        }
    }
    g.Q = std::min(best_q, ((V + gran - 1) / gran) * gran);
    g.cpr = (V + g.Q - 1) / g.Q;
    g.U = rows_total * (int64_t)g.cpr;
    g.P = (int)std::min<int64_t>(P, g.U);
    return g;
}

template <typename T, bool GREEDY>
static cudaError_t prepare_stream()
{
    static cudaError_t once = [] {
        const int smem = kStreamWarps * kRing * (int)align_up(kPieceBytesMax, 128) +
                         4 * (kMaxBatch + 1);
        cudaError_t e = cudaFuncSetAttribute(stream_kernel<T, GREEDY>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(stream_kernel<T, GREEDY>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        return e;
    }();
    return once;
}

template <typename T, bool GREEDY>
static cudaError_t prepare_finish()
{
    static cudaError_t once = [] {
        return cudaFuncSetAttribute(finish_kernel<T, GREEDY>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    2 * (kDrawChunkBytes + 128));
    }();
    return once;
}

template <typename T, bool GREEDY>
static cudaError_t launch_typed(const VerifyArgs &a, cudaStream_t s, Tracer &tr)
{
    const int e = (int)sizeof(T);
    const WsLayout L = ws_layout(a.B, a.max_rows, a.V);
    unsigned char *ws = static_cast<unsigned char *>(a.ws);
    const int64_t draft_slots = GREEDY ? 0 : a.max_rows - a.B;
    const int ctas_max = sm_count() * SV_STREAM_CTAS_PER_SM;
    const Geometry g = plan(a.max_rows + draft_slots, a.max_rows, a.V, e,
                            std::min(kMaxWorkers, ctas_max * kStreamWarps));
    const bool row16 = ((int64_t)a.V * e) % 16 == 0;
    const bool tma = row16 && reinterpret_cast<uintptr_t>(a.target) % 16 == 0 &&
                     (GREEDY || reinterpret_cast<uintptr_t>(a.draft) % 16 == 0);
    const double c = GREEDY ? 0.0 : 1.4426950408889634074 / a.temperature;  // log2(e) / T

    StreamParams sp{};
    sp.target = a.target;
    sp.draft = a.draft;
    sp.cu = a.cu;
    sp.out_tokens = a.out_tokens;
    sp.out_len = a.out_len;
    sp.B = a.B;
    sp.V = a.V;
    sp.draft_slots = draft_slots;
    sp.draft_stride = a.draft_stride;
    sp.g = g;
    sp.tma = tma;
    sp.piece_smem = (int)align_up((size_t)g.Q * e, 128);
    sp.c = (float)c;
    sp.status = reinterpret_cast<uint32_t *>(ws + L.status);
    sp.cu_flag = sp.status + 1;
    sp.part = reinterpret_cast<Partial *>(ws + L.part1);

    FinishParams fp{};
    fp.target = a.target;
    fp.draft = a.draft;
    fp.tokens = a.tokens;
    fp.cu = a.cu;
    fp.u_accept = a.u_accept;
    fp.u_final = a.u_final;
    fp.out_tokens = a.out_tokens;
    fp.out_len = a.out_len;
    fp.out_p = a.out_p;
    fp.out_q = a.out_q;
    fp.B = a.B;
    fp.V = a.V;
    fp.draft_rows = a.draft_stride > 0 ? (int64_t)a.B * a.draft_stride : a.max_rows - a.B;
    fp.draft_stride = a.draft_stride;
    fp.g = g;
    const Chunking dc = chunking(a.V, e);
    fp.NC = GREEDY ? 1 : dc.nchunks;
    fp.nce = dc.chunk_elems;
    fp.chunk_smem = (int)align_up((size_t)dc.chunk_elems * e, 128);
    fp.tma = tma;
    fp.c = sp.c;
    fp.status = sp.status;
    fp.cu_flag = sp.cu_flag;
    fp.cnt2 = reinterpret_cast<uint32_t *>(ws + L.cnt2);
    fp.part = sp.part;
    fp.part2 = reinterpret_cast<double *>(ws + L.part2);

    cudaError_t err = prepare_stream<T, GREEDY>();
    if (err == cudaSuccess)
        err = prepare_finish<T, GREEDY>();
    if (err != cudaSuccess)
        return err;
    const int grid1 = (g.P + kStreamWarps - 1) / kStreamWarps;
    const size_t smem1 = (size_t)kStreamWarps * kRing * sp.piece_smem +
                         (a.draft_stride > 0 ? 4 * (size_t)(a.B + 1) : 0);
    tr.begin(s);
    stream_kernel<T, GREEDY><<<grid1, kStreamThreads, smem1, s>>>(sp);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;
    tr.after_kernel(s);

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(a.B * fp.NC));
    cfg.blockDim = dim3(kFinishThreads);
    cfg.dynamicSmemBytes = GREEDY ? 0 : 2 * (size_t)fp.chunk_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((err = cudaLaunchKernelEx(&cfg, finish_kernel<T, GREEDY>, fp)) != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, Tracer &tr)
{
    const bool greedy = a.temperature == 0.0;
    if (a.dtype == 0)
        return greedy ? launch_typed<float, true>(a, s, tr) : launch_typed<float, false>(a, s, tr);
    return greedy ? launch_typed<uint16_t, true>(a, s, tr)
                  : launch_typed<uint16_t, false>(a, s, tr);
}

}  // namespace sv
