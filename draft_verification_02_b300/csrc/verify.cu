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
// Kernel 2, launched as a programmatic dependent of kernel 1: it reads the
// inputs that do not depend on kernel 1 (offsets, drafted tokens, uniforms,
// the logits at the drafted tokens) before waiting for kernel 1 to finish.
//  - T = 0, finish_greedy_kernel: one CTA per request merges the argmax
//    partials and runs the first-mismatch ballot.
//  - T > 0, finish_sample_kernel: one cluster of 8 or 16 CTAs per request.
//    The request's rows are merged one or two per warp of the cluster (their
//    (m, s) and p(x) sent to every CTA through distributed shared memory);
//    every CTA runs the accept test and first-rejection ballot (identical
//    bits everywhere), then weighs its share of the final-draw rows into
//    shared memory and sums the weights.  The range sums are exchanged the
//    same way; the CTA whose range holds u*S finds the token with a block
//    scan of per-thread piece sums and one thread's walk through its piece.
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
    int ncl;    // CTAs per request (cluster size) in the final draw: 8 or 16
    int R;      // vocabulary entries per cluster CTA in the final draw
    int slice;  // entries of one row weighed at a time (multiple of 16 bytes)
    int pv;          // 16-byte vectors per thread piece of a slice (odd)
    int stage_smem;  // bytes per staged row slice (multiple of 128)
    int tma;         // rows 16-byte aligned: TMA bulk copies
    float c;
    uint32_t *status;
    const uint32_t *cu_flag;
    const Partial *part;
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

__device__ __forceinline__ int64_t draft_index(int draft_stride, const int32_t *cu, int i, int j)
{
    return draft_stride > 0 ? (int64_t)i * draft_stride + j : (int64_t)__ldg(cu + i) + j;
}


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

// Units are read from shared memory as lane-strided 16-byte vectors held in
// registers; vectors past the unit's end read as -inf, which neither the
// maximum nor the sum of exp2 sees.  Maxima and sums are trees (short
// dependency chains), not running chains.  A tail that is not a whole vector
// (plain-load path only) is handled element by element.
constexpr uint32_t kNegInfBf16x2 = 0xff80ff80u;

template <int MAXV>
__device__ __forceinline__ void load_unit_bf16(const uint16_t *buf, int nvec, uint4 (&r)[MAXV])
{
    const int lane = threadIdx.x & 31;
    const uint4 *vb = reinterpret_cast<const uint4 *>(buf);
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const int v = lane + 32 * t;
        r[t] = v < nvec ? vb[v] : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2,
                                             kNegInfBf16x2);
    }
}

template <int MAXV>
__device__ __forceinline__ void load_unit_f32(const float *buf, int nvec, float4 (&r)[MAXV])
{
    const int lane = threadIdx.x & 31;
    const float4 *vb = reinterpret_cast<const float4 *>(buf);
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const int v = lane + 32 * t;
        r[t] = v < nvec ? vb[v] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
}

// Tree maximum of a unit held in registers (NaN-propagating).
template <int MAXV>
__device__ __forceinline__ float unit_max_bf16(const uint4 (&r)[MAXV])
{
    uint32_t mx[MAXV];
#pragma unroll
    for (int t = 0; t < MAXV; ++t)
        mx[t] = max_nan_bf16x2(max_nan_bf16x2(r[t].x, r[t].y), max_nan_bf16x2(r[t].z, r[t].w));
#pragma unroll
    for (int w = MAXV / 2; w >= 1; w /= 2)
#pragma unroll
        for (int t = 0; t < w; ++t)
            mx[t] = max_nan_bf16x2(mx[t], mx[t + w]);
    return max_nan(bf16_lo(mx[0]), bf16_hi(mx[0]));
}

template <int MAXV>
__device__ __forceinline__ float unit_max_f32(const float4 (&r)[MAXV])
{
    float mx[MAXV];
#pragma unroll
    for (int t = 0; t < MAXV; ++t)
        mx[t] = max_nan(max_nan(r[t].x, r[t].y), max_nan(r[t].z, r[t].w));
#pragma unroll
    for (int w = MAXV / 2; w >= 1; w /= 2)
#pragma unroll
        for (int t = 0; t < w; ++t)
            mx[t] = max_nan(mx[t], mx[t + w]);
    return mx[0];
}

template <int MAXV>
__device__ __forceinline__ float tree_sum(float (&v)[MAXV])
{
#pragma unroll
    for (int w = MAXV / 2; w >= 1; w /= 2)
#pragma unroll
        for (int t = 0; t < w; ++t)
            v[t] += v[t + w];
    return v[0];
}

// One unit of bf16 data at T > 0.
template <int MAXV>
__device__ __forceinline__ void unit_softmax_bf16(const uint16_t *buf, int len, float c,
                                                  LaneAcc &a)
{
    const int lane = threadIdx.x & 31;
    const int nvec = len >> 3;
    uint4 r[MAXV];
    load_unit_bf16<MAXV>(buf, nvec, r);
    float pm = unit_max_bf16<MAXV>(r);
    for (int k = nvec * 8 + lane; k < len; k += 32)
        pm = max_nan(pm, bf16_lo((uint32_t)buf[k]));
    if (!fold_max(a, pm, c))
        return;
    const float mc = a.m * c;
    float sv[MAXV];
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const uint32_t w4[4] = {r[t].x, r[t].y, r[t].z, r[t].w};
        float e[8];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            e[2 * h] = ex2_approx(fmaf(bf16_lo(w4[h]), c, -mc));
            e[2 * h + 1] = ex2_approx(fmaf(bf16_hi(w4[h]), c, -mc));
        }
        sv[t] = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    }
    float acc = tree_sum<MAXV>(sv);
    for (int k = nvec * 8 + lane; k < len; k += 32)
        acc += ex2_approx(fmaf(bf16_lo((uint32_t)buf[k]), c, -mc));
    add_unit(a, acc, mc, c);
}

template <int MAXV>
__device__ __forceinline__ void unit_softmax_f32(const float *buf, int len, float c, LaneAcc &a)
{
    const int lane = threadIdx.x & 31;
    const int nvec = len >> 2;
    float4 r[MAXV];
    load_unit_f32<MAXV>(buf, nvec, r);
    float pm = unit_max_f32<MAXV>(r);
    for (int k = nvec * 4 + lane; k < len; k += 32)
        pm = max_nan(pm, buf[k]);
    if (!fold_max(a, pm, c))
        return;
    const float mc = a.m * c;
    float sv[MAXV];
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
        const float e0 = ex2_approx(fmaf(r[t].x, c, -mc));
        const float e1 = ex2_approx(fmaf(r[t].y, c, -mc));
        const float e2 = ex2_approx(fmaf(r[t].z, c, -mc));
        const float e3 = ex2_approx(fmaf(r[t].w, c, -mc));
        sv[t] = (e0 + e1) + (e2 + e3);
    }
    float acc = tree_sum<MAXV>(sv);
    for (int k = nvec * 4 + lane; k < len; k += 32)
        acc += ex2_approx(fmaf(buf[k], c, -mc));
    add_unit(a, acc, mc, c);
}

// T = 0: the warp keeps one running (maximum, lowest index) pair, the same in
// every lane.  A unit costs a tree maximum and a warp maximum; only when the
// warp maximum grows does each lane look for its first element equal to it
// (its elements in increasing index order) and the warp take the lowest.
// Earlier units hold lower indices, so a strict > keeps the lowest index.
template <int MAXV>
__device__ __forceinline__ void unit_argmax_bf16(const uint16_t *buf, int len, int col0,
                                                 LaneAcc &a)
{
    const int lane = threadIdx.x & 31;
    const int nvec = len >> 3;
    uint4 r[MAXV];
    load_unit_bf16<MAXV>(buf, nvec, r);
    float pm = unit_max_bf16<MAXV>(r);
    for (int k = nvec * 8 + lane; k < len; k += 32)
        pm = max_nan(pm, bf16_lo((uint32_t)buf[k]));
    const float wm = warp_max_nan(pm);
    if (wm != wm) {
        a.nan = 1;
    } else if (wm > a.m) {
        int found = INT_MAX;
#pragma unroll
        for (int t = 0; t < MAXV; ++t) {
            const uint32_t w4[4] = {r[t].x, r[t].y, r[t].z, r[t].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int k = (lane + 32 * t) * 8 + 2 * h;
                if (found == INT_MAX && bf16_lo(w4[h]) == wm)
                    found = k;
                if (found == INT_MAX && bf16_hi(w4[h]) == wm)
                    found = k + 1;
            }
        }
        for (int k = nvec * 8 + lane; k < len && found == INT_MAX; k += 32)
            if (bf16_lo((uint32_t)buf[k]) == wm)
                found = k;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
        a.m = wm;
        a.idx = col0 + found;
    }
}

template <int MAXV>
__device__ __forceinline__ void unit_argmax_f32(const float *buf, int len, int col0, LaneAcc &a)
{
    const int lane = threadIdx.x & 31;
    const int nvec = len >> 2;
    float4 r[MAXV];
    load_unit_f32<MAXV>(buf, nvec, r);
    float pm = unit_max_f32<MAXV>(r);
    for (int k = nvec * 4 + lane; k < len; k += 32)
        pm = max_nan(pm, buf[k]);
    const float wm = warp_max_nan(pm);
    if (wm != wm) {
        a.nan = 1;
    } else if (wm > a.m) {
        int found = INT_MAX;
#pragma unroll
        for (int t = 0; t < MAXV; ++t) {
            const float x4[4] = {r[t].x, r[t].y, r[t].z, r[t].w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                if (found == INT_MAX && x4[h] == wm)
                    found = (lane + 32 * t) * 4 + h;
        }
        for (int k = nvec * 4 + lane; k < len && found == INT_MAX; k += 32)
            if (buf[k] == wm)
                found = k;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
        a.m = wm;
        a.idx = col0 + found;
    }
}

// Reduce the lanes' state of a finished row segment, store its partial and
// reset the state.
template <bool GREEDY>
__device__ __forceinline__ void store_partial(LaneAcc &a, float c, Partial *slot)
{
    const int lane = threadIdx.x & 31;
    Partial out;
    if (GREEDY) {  // the running (maximum, index) is already the same in every lane
        out.m = a.m;
        out.idx = a.nan ? -2 : (a.idx == INT_MAX ? -1 : a.idx);
        out.s_hi = 0.f;
        out.s_lo = 0.f;
    } else {
        const float m = warp_max_nan(a.m);
        ff s{0.f, 0.f};
        if (m == m && m != -INFINITY && m != INFINITY) {
            if (a.s != 0.f)  // the Kahan pair (s, -comp) rescaled to the warp maximum
                s = ff_mul(fast_two_sum(a.s, -a.comp), exp2f((a.m - m) * c));
        } else if (m != -INFINITY) {
            s.hi = __int_as_float(0x7fc00000);
        }
        s = warp_sum_ff(s);
        out.m = m;
        out.idx = 0;
        out.s_hi = s.hi;
        out.s_lo = s.lo;
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
constexpr int kCluster = 16;               // most CTAs per request in the sampling finish kernel
constexpr int kSampleThreads = 256;        // threads per CTA of the sampling finish kernel
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kStageRowBytes = 48 * 1024;  // largest slice of one row staged at a time
constexpr int kMaxSlices = 64;             // slices per CTA range (bounds V)

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store v at the address `local` has in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ void st_cluster_ff(ff *local, uint32_t rank, ff v)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(v.hi), "f"(v.lo)
                 : "memory");
}

// One partial, read from L2 in a single 16-byte load.
__device__ __forceinline__ Partial load_partial(const Partial *p)
{
    const uint4 r = __ldcg(reinterpret_cast<const uint4 *>(p));
    Partial out;
    out.m = __uint_as_float(r.x);
    out.idx = (int32_t)r.y;
    out.s_hi = __uint_as_float(r.z);
    out.s_lo = __uint_as_float(r.w);
    return out;
}

// Combine two softmax partials (m, s), s = sum exp2((x - m) c) held as a
// float-float pair.  The result does not depend on the order of the two
// arguments, so a butterfly over a warp leaves the same bits in every lane.
__device__ __forceinline__ void lse_combine(float &m, ff &s, float mo, ff so, float c)
{
    if (so.hi == 0.f)
        return;  // empty or fully masked partial
    if (s.hi == 0.f) {
        m = mo;
        s = so;
        return;
    }
    const float mn = max_nan(m, mo);
    if (mn != mn || s.hi != s.hi || so.hi != so.hi) {
        m = __int_as_float(0x7fc00000);
        s = {__int_as_float(0x7fc00000), 0.f};
        return;
    }
    s = ff_add(ff_mul(s, exp2f((m - mn) * c)), ff_mul(so, exp2f((mo - mn) * c)));
    m = mn;
}

// Warps wf..wl left the partials of flattened row rg, in slots rg + wf ..
// rg + wl (warp w's units are contiguous, so its slots never collide).
__device__ __forceinline__ void row_span(const Geometry &g, int64_t rg, int &wf, int &wl)
{
    const int64_t ua = rg * g.cpr;
    wf = owner_of(ua, g);
    wl = owner_of(ua + g.cpr - 1, g);
}

// T = 0: lowest argmax of target row rg; -1 masked row, -2 NaN, -3 +inf.
__device__ __forceinline__ int merge_argmax_row(const Partial *part, const Geometry &g, int64_t rg)
{
    const int lane = threadIdx.x & 31;
    int wf, wl;
    row_span(g, rg, wf, wl);
    float best = -INFINITY;
    int bidx = INT_MAX, nan = 0;
    for (int w = wf + lane; w <= wl; w += 32) {
        const Partial q = load_partial(part + rg + w);
        if (q.idx == -2)
            nan = 1;
        else if (q.idx >= 0 && (q.m > best || (q.m == best && q.idx < bidx))) {
            best = q.m;
            bidx = q.idx;
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

__device__ __forceinline__ bool row_ok(float m, ff s)
{
    return isfinite(m) && isfinite(s.hi) && s.hi > 0.f;
}

// p(x) = 2^((g - m) c) / s for one row given its (m, s): g - m exactly as a
// float-float pair, its product with c to float-float, 2^hi with exp2f and
// the low part to first order, then the division by s.
__device__ __forceinline__ float softmax_at(float g, float m, ff s, float c)
{
    if (g == -INFINITY)
        return 0.f;  // a masked entry
    const ff d = two_sum(g, -m);
    const float xh = __fmul_rn(d.hi, c);
    const float xl = fmaf(d.lo, c, fmaf(d.hi, c, -xh));
    const float num = __fmul_rn(exp2f(xh), fmaf(xl, 0.69314718f, 1.f));
    const float inv = __frcp_rn(s.hi);
    return __fmul_rn(__fmul_rn(num, inv), fmaf(-s.lo, inv, 1.f));
}

// Request i's offsets checked locally, before the streaming kernel's own
// validation is visible: only then are its token / logit addresses formed.
__device__ __forceinline__ bool request_shape_ok(const FinishParams &p, int i, int cu_i, int K)
{
    const int64_t t0 = (int64_t)cu_i + i;
    return cu_i >= 0 && K >= 0 && K <= kMaxDraft && t0 + K < p.g.max_rows &&
           (p.draft_stride > 0 ? K <= p.draft_stride : (int64_t)cu_i + K <= p.draft_rows);
}

template <typename T>
__global__ void __launch_bounds__(kFinishThreads) finish_greedy_kernel(const FinishParams p)
{
    __shared__ int row_g[kMaxDraft + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i = blockIdx.x;

    // inputs that do not depend on kernel 1 are read before waiting for it
    const int cu_i = __ldg(p.cu + i);
    const int K = __ldg(p.cu + i + 1) - cu_i;
    const bool shape = request_shape_ok(p, i, cu_i, K);
    const bool act = shape && warp == 0 && lane < K;
    const int x = act ? __ldg(p.tokens + draft_index(p.draft_stride, p.cu, i, lane)) : -1;

    pdl_wait();  // kernel 1 has completed and its writes are visible
    if (__ldcg(p.cu_flag) == 0u || !shape)
        return;  // malformed offsets: kernel 1 poisoned every output
    const int64_t t0 = (int64_t)cu_i + i;
    for (int rho = warp; rho <= K; rho += kFinishWarps) {
        const int gj = merge_argmax_row(p.part, p.g, t0 + rho);
        if (lane == 0)
            row_g[rho] = gj;
    }
    __syncthreads();
    if (warp != 0)
        return;
    const bool bad_tok = act && (x < 0 || x >= p.V);
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
}

// f / s for a float-float s.
__device__ __forceinline__ float ff_recip_scaled(float f, ff s)
{
    const float inv = __frcp_rn(s.hi);
    return __fmul_rn(__fmul_rn(f, inv), fmaf(-s.lo, inv, 1.f));
}

struct DrawCtx {
    bool resid;
    float c, mct, mcd;  // c and fl(m c) of the two rows
    float sc_t, sc_d;   // 2^(fl(m c) - m c) / s: normalisers including the rounding fix
};

// Final-draw weight of one element: max(0, p - q) after a rejection, the
// unnormalised p for the bonus draw (or an all-zero residual).
__device__ __forceinline__ float draw_w(const DrawCtx &d, float t, float x)
{
    const float pt = ex2_approx(fmaf(t, d.c, -d.mct));
    if (!d.resid)
        return pt;
    const float pd = ex2_approx(fmaf(x, d.c, -d.mcd));
    return fmaxf(fmaf(pt, d.sc_t, -__fmul_rn(pd, d.sc_d)), 0.f);
}

// Sum of the final-draw weights of one thread's contiguous piece (16-byte
// vectors [v0, v1) of a staged slice of len elements), in index order, fp32.
template <typename T>
__device__ __forceinline__ float piece_sum(const DrawCtx d, const T *tb, const T *db, int len,
                                           int v0, int v1)
{
    constexpr int E = Elem<T>::kPerVec;
    const uint4 *tv = reinterpret_cast<const uint4 *>(tb);
    const uint4 *dv = reinterpret_cast<const uint4 *>(db);
    float acc = 0.f;
#pragma unroll 1
    for (int v = v0; v < v1; ++v) {
        float ft[E], fd[E];
        Elem<T>::unpack(tv[v], ft);
        if (d.resid)
            Elem<T>::unpack(dv[v], fd);
#pragma unroll
        for (int h = 0; h < E; ++h) {
            const float w = v * E + h < len ? draw_w(d, ft[h], d.resid ? fd[h] : 0.f) : 0.f;
            acc = __fadd_rn(acc, w);
        }
    }
    return acc;
}

// The same walk, stopping at the first element whose running sum exceeds
// rem: its index in the slice, or (none) the last element with weight > 0
// (-1 if there is none).  The running sums are those of piece_sum, bit for
// bit.
template <typename T>
__device__ __forceinline__ int piece_find(const DrawCtx d, const T *tb, const T *db, int len,
                                          int v0, int v1, float rem)
{
    constexpr int E = Elem<T>::kPerVec;
    const uint4 *tv = reinterpret_cast<const uint4 *>(tb);
    const uint4 *dv = reinterpret_cast<const uint4 *>(db);
    float acc = 0.f;
    int lastp = -1;
#pragma unroll 1
    for (int v = v0; v < v1; ++v) {
        float ft[E], fd[E];
        Elem<T>::unpack(tv[v], ft);
        if (d.resid)
            Elem<T>::unpack(dv[v], fd);
#pragma unroll
        for (int h = 0; h < E; ++h) {
            const int k = v * E + h;
            const float w = k < len ? draw_w(d, ft[h], d.resid ? fd[h] : 0.f) : 0.f;
            acc = __fadd_rn(acc, w);
            if (w > 0.f)
                lastp = k;
            if (acc > rem)
                return k;
        }
    }
    return lastp;
}

// Stage elements [c0, c0 + len) of the draw rows into shared memory (one
// TMA bulk copy per row, or plain loads when the rows are not 16-byte
// aligned), then every thread sums its contiguous piece (kept in piece[]
// for the search) and the pieces are added as float-float pairs in a fixed
// order.  Once any copy of this call has timed out nothing more is copied.
template <typename T>
__device__ __noinline__ ff weigh_slice(const FinishParams &p, const DrawCtx d, const T *trow,
                                       const T *drow, int c0, int len, T *tb, T *db,
                                       uint64_t *bar, uint32_t *phase, float *piece, ff *wred,
                                       int *expired)
{
    constexpr int E = Elem<T>::kPerVec;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // earlier readers of the buffers, piece and wred are done
    const bool stop = __syncthreads_or(tid == 0 && (read_status(p.status) & ST_TIMEOUT));
    if (!stop && len > 0) {
        if (p.tma) {
            if (tid == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                const uint32_t bytes = (uint32_t)len * (uint32_t)sizeof(T);
                mbar_arrive_expect_tx(bar, d.resid ? 2 * bytes : bytes);
                bulk_g2s(tb, trow + c0, bytes, bar);
                if (d.resid)
                    bulk_g2s(db, drow + c0, bytes, bar);
            }
            if (!mbar_wait_bounded(bar, *phase)) {
                set_status(p.status, ST_TIMEOUT);
                *expired = 1;
                mbar_wait_bounded(bar, *phase);  // the copy in flight, once more
            }
            *phase ^= 1u;
        } else {
            for (int k = tid; k < len; k += kSampleThreads) {
                tb[k] = trow[c0 + k];
                if (d.resid)
                    db[k] = drow[c0 + k];
            }
            __syncthreads();
        }
    }
    const int nv = (len + E - 1) / E;
    const int v0 = min(nv, tid * p.pv), v1 = min(nv, v0 + p.pv);
    const float ps = piece_sum<T>(d, tb, db, len, v0, v1);
    piece[tid] = ps;
    const ff ws = warp_sum_ff({ps, 0.f});
    __syncthreads();  // piece[] complete; wred free
    if (lane == 0)
        wred[warp] = ws;
    __syncthreads();
    ff tot = wred[0];
    for (int q = 1; q < kSampleWarps; ++q)
        tot = ff_add(tot, wred[q]);
    return tot;
}

// Store (m, s, p(x)) of row k into the shared memory of cluster CTA `rank`.
__device__ __forceinline__ void st_cluster_row(float *row_m, ff *row_s, float *row_p, int k,
                                               uint32_t rank, float m, ff s, float px)
{
    uint32_t rm, rs, rp;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rm) : "r"(smem_u32(row_m + k)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rs) : "r"(smem_u32(row_s + k)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rp) : "r"(smem_u32(row_p + k)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(rm), "f"(m) : "memory");
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(rs), "f"(s.hi), "f"(s.lo)
                 : "memory");
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(rp), "f"(px) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kSampleThreads, 2) finish_sample_kernel(const FinishParams p)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    T *tb = reinterpret_cast<T *>(dsm);  // staged slice of the target row
    T *db = reinterpret_cast<T *>(dsm + p.stage_smem);  // and of the draft row
    __shared__ __align__(8) uint64_t bar;
    __shared__ float row_m[2 * kMaxDraft + 1];            // written by every CTA of the cluster
    __shared__ __align__(8) ff row_s[2 * kMaxDraft + 1];  // likewise
    __shared__ float row_p[2 * kMaxDraft + 1];            // likewise: p_j(x_j), q_j(x_j)
    __shared__ float piece[kSampleThreads];
    __shared__ ff wred[kSampleWarps];
    __shared__ ff slice_tot[kMaxSlices];
    __shared__ __align__(8) ff cl_sum[2][kCluster];  // written by every CTA of the cluster
    __shared__ ff s_excl[kSampleWarps];
    __shared__ int s_a, s_bad, s_hit, s_last, s_cs, s_past, s_redo, s_expired;
    __shared__ ff s_base, s_target;
    __shared__ DrawCtx s_d;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const int ncl = p.ncl;
    const int i = blockIdx.x / ncl;
    const T *tbase = reinterpret_cast<const T *>(p.target);
    const T *dbase = reinterpret_cast<const T *>(p.draft);

    // ---- inputs that do not depend on kernel 1, read before waiting for it
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        s_expired = 0;
    }
    const int cu_i = __ldg(p.cu + i);
    const int K = __ldg(p.cu + i + 1) - cu_i;
    const bool shape = request_shape_ok(p, i, cu_i, K);
    const int64_t t0 = (int64_t)cu_i + i;
    const int nrows = 2 * K + 1;
    // warp 0, lane j < K: the drafted token and its uniform (accept test)
    const bool act = shape && warp == 0 && lane < K;
    int x = -1;
    float u = 0.f;
    int64_t di = 0;
    if (act) {
        di = draft_index(p.draft_stride, p.cu, i, lane);
        x = __ldg(p.tokens + di);
        u = __ldg(p.u_accept + di);
    }
    // the rows this warp merges (k = rank + ncl * (warp + kSampleWarps * t)):
    // target rows 0..K, then draft rows 0..K-1; the logit at the drafted
    // token of each such row
    int my_k[2];
    float g[2] = {-INFINITY, -INFINITY};
    bool g_ok[2] = {false, false};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        my_k[t] = (int)rank + ncl * (warp + kSampleWarps * t);
        if (!shape || my_k[t] >= nrows)
            my_k[t] = -1;
        else if (my_k[t] != K) {
            const int j = my_k[t] < K ? my_k[t] : my_k[t] - K - 1;
            const int64_t dj = draft_index(p.draft_stride, p.cu, i, j);
            const int xj = __ldg(p.tokens + dj);
            if (xj >= 0 && xj < p.V) {
                g_ok[t] = true;
                g[t] = my_k[t] < K ? Elem<T>::ld_global(tbase + (t0 + j) * p.V, xj)
                                   : Elem<T>::ld_global(dbase + dj * p.V, xj);
            }
        }
    }
    const float uf = __ldg(p.u_final + i);

    pdl_wait();  // kernel 1 has completed and its writes are visible
    if (__ldcg(p.cu_flag) == 0u || !shape)
        return;  // malformed offsets: kernel 1 poisoned every output (same in every CTA)
    cluster_arrive_relaxed();  // (0) this CTA has started
    // an expired wait of kernel 1 only poisons; its flag is read now, off the
    // critical path
    const bool timeout = warp == 0 && (read_status(p.status) & ST_TIMEOUT);

    // ---- (m, s) and p(x) of the request's rows, one or two rows per warp of
    // the cluster, sent to every CTA
    float mm[2] = {-INFINITY, -INFINITY}, px[2] = {0.f, 0.f};
    ff sm[2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (my_k[t] < 0)
            continue;
        const int k = my_k[t];
        const int64_t rg = k <= K ? t0 + k : p.g.max_rows + cu_i + (k - K - 1);
        int wf, wl;
        row_span(p.g, rg, wf, wl);
        for (int w = wf + lane; w <= wl; w += 32) {
            const Partial pt = load_partial(p.part + rg + w);
            lse_combine(mm[t], sm[t], pt.m, {pt.s_hi, pt.s_lo}, p.c);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, mm[t], o);
            const ff so = ff_shfl_xor(sm[t], o);
            lse_combine(mm[t], sm[t], mo, so, p.c);
        }
        px[t] = g_ok[t] && row_ok(mm[t], sm[t]) ? softmax_at(g[t], mm[t], sm[t], p.c) : 0.f;
    }
    cluster_wait_acquire();  // (0) complete: every CTA's shared memory is live
#pragma unroll
    for (int t = 0; t < 2; ++t)
        if (my_k[t] >= 0 && lane < ncl)
            st_cluster_row(row_m, row_s, row_p, my_k[t], (uint32_t)lane, mm[t], sm[t], px[t]);
    cluster_arrive_release();
    cluster_wait_acquire();  // (1) every CTA holds every row's (m, s, p(x))

    // ---- accept test and first rejection (warp 0; identical in every CTA)
    if (warp == 0) {
        bool bad_tok = act && (x < 0 || x >= p.V), bad_nf = false, acc = true;
        float pp = 0.f, qq = 0.f;
        if (act && !bad_tok) {
            if (!row_ok(row_m[lane], row_s[lane]) ||
                !row_ok(row_m[K + 1 + lane], row_s[K + 1 + lane])) {
                bad_nf = true;
            } else {
                pp = row_p[lane];
                qq = row_p[K + 1 + lane];
                const float ratio = qq > 0.f ? __fdiv_rn(pp, qq) : (pp > 0.f ? INFINITY : 0.f);
                acc = u < ratio;
            }
        }
        if (lane == 0 && !row_ok(row_m[K], row_s[K]))
            bad_nf = true;
        const unsigned nf = __ballot_sync(0xffffffffu, bad_nf);
        const unsigned bt = __ballot_sync(0xffffffffu, bad_tok);
        const unsigned rej = __ballot_sync(0xffffffffu, act && !acc);
        // bad depends only on the request's data, so every CTA of the cluster
        // takes the same branch; an expired wait only poisons (best effort)
        const bool bad = nf || bt;
        const int a = rej ? __ffs(rej) - 1 : K;
        if (rank == 0) {  // the request's outputs, written once
            if (bad || timeout) {
                if (lane == 0)
                    set_status(p.status, (nf ? ST_NONFINITE : 0u) | (bt ? ST_INVALID : 0u));
                for (int jj = lane; jj <= K; jj += 32)
                    p.out_tokens[t0 + jj] = -1;
                if (lane == 0)
                    p.out_len[i] = -1;
            } else {
                if (act && p.out_p)
                    p.out_p[di] = pp;
                if (act && p.out_q)
                    p.out_q[di] = qq;
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
            // the final draw's constants, once for the CTA
            DrawCtx d0;
            d0.resid = a < K;
            d0.c = p.c;
            const float mt = row_m[a];
            d0.mct = mt * p.c;
            d0.sc_t = ff_recip_scaled(mc_correction(mt, d0.mct, p.c), row_s[a]);
            d0.mcd = 0.f;
            d0.sc_d = 0.f;
            if (d0.resid) {
                const float md = row_m[K + 1 + a];
                d0.mcd = md * p.c;
                d0.sc_d = ff_recip_scaled(mc_correction(md, d0.mcd, p.c), row_s[K + 1 + a]);
            }
            s_d = d0;
        }
    }
    __syncthreads();
    if (s_bad)
        return;  // same decision in every CTA of the cluster; no more cluster traffic

    // ---- final draw: this CTA weighs its range of the vocabulary
    const int a = s_a;
    const int64_t trow_i = t0 + a;
    const int64_t drow_i = a < K ? draft_index(p.draft_stride, p.cu, i, a) : -1;
    DrawCtx d = s_d;
    const T *trow = tbase + trow_i * p.V;
    const T *drow = d.resid ? dbase + drow_i * p.V : nullptr;
    const int r0 = min(p.V, (int)rank * p.R), r1 = min(p.V, r0 + p.R);
    const int nsl = r1 > r0 ? (r1 - r0 + p.slice - 1) / p.slice : 0;
    int weighed = -1;  // slice staged in shared memory
    uint32_t phase = 0;

    // pass 0 sums max(0, p_a - q_a) (or p_K); an all-zero residual makes a
    // second pass over p_a (the same decision in every CTA)
    int slot = 0;
    for (int pass = 0; pass < 2; ++pass) {
        ff mine{0.f, 0.f};
        for (int sl = 0; sl < nsl; ++sl) {
            const int c0 = r0 + sl * p.slice, len = min(p.slice, r1 - c0);
            const ff ss = weigh_slice<T>(p, d, trow, drow, c0, len, tb, db, &bar, &phase, piece,
                                         wred, &s_expired);
            weighed = sl;
            if (tid == 0)
                slice_tot[sl] = ss;
            mine = ff_add(mine, ss);
        }
        if (tid < ncl)
            st_cluster_ff(&cl_sum[pass][rank], (uint32_t)tid, mine);
        cluster_arrive_release();
        cluster_wait_acquire();  // (2 + pass) every CTA holds every range sum
        slot = pass;
        // S and the range holding u*S, by warp 0 (lane r holds range r): an
        // inclusive float-float scan in range order, the same in every CTA.
        // `past` marks u*S at or beyond the end after rounding: then the
        // last weight > 0 wins.
        if (warp == 0) {
            const ff v = lane < ncl ? cl_sum[pass][lane] : ff{0.f, 0.f};
            ff incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const ff n = ff_shfl_up(incl, o);
                if (lane >= o)
                    incl = ff_add(n, incl);
            }
            const ff S = {__shfl_sync(0xffffffffu, incl.hi, 31),
                          __shfl_sync(0xffffffffu, incl.lo, 31)};
            const ff target = ff_mul(S, uf);
            const unsigned over = __ballot_sync(0xffffffffu, lane < ncl && ff_gt(incl, target));
            const unsigned mass = __ballot_sync(0xffffffffu, lane < ncl && v.hi > 0.f);
            const int cs = over ? __ffs(over) - 1 : (mass ? 31 - __clz(mass) : -1);
            ff excl = ff_shfl_up(incl, 1);
            if (lane == 0)
                excl = {0.f, 0.f};
            const int src = cs < 0 ? 0 : cs;
            const ff base = {__shfl_sync(0xffffffffu, excl.hi, src),
                             __shfl_sync(0xffffffffu, excl.lo, src)};
            if (lane == 0) {
                s_cs = cs;
                s_past = over == 0u;
                s_base = base;
                s_target = target;
                s_redo = !(S.hi > 0.f);
            }
        }
        __syncthreads();
        if (!(d.resid && s_redo))
            break;
        d.resid = false;  // all-zero residual: draw from p_a instead
    }
    // no shared memory of another CTA is touched after this point
    const int cs = s_cs;
    bool past = s_past != 0;
    ff base = s_base;
    const ff target = s_target;
    if ((int)rank != cs) {
        if (cs < 0 && rank == 0 && tid == 0) {  // no mass at all (never with finite rows)
            set_status(p.status, ST_NONFINITE);
            p.out_tokens[trow_i] = -1;
        }
        return;
    }

    // ---- owner CTA: the slice, then the thread piece, then the element
    int sl = -1;
    {
        ff b2 = base;
        for (int s2 = 0; s2 < nsl && !past; ++s2) {
            const ff next = ff_add(b2, slice_tot[s2]);
            if (ff_gt(next, target)) {
                sl = s2;
                break;
            }
            b2 = next;
        }
        if (sl >= 0) {
            base = b2;
        } else {  // the last slice with mass
            past = true;
            ff bl = base;
            b2 = base;
            sl = nsl - 1;
            for (int s2 = 0; s2 < nsl; ++s2) {
                if (slice_tot[s2].hi > 0.f) {
                    sl = s2;
                    bl = b2;
                }
                b2 = ff_add(b2, slice_tot[s2]);
            }
            base = bl;
        }
    }
    const int c0 = r0 + sl * p.slice, len = min(p.slice, r1 - c0);
    if (sl != weighed)
        weigh_slice<T>(p, d, trow, drow, c0, len, tb, db, &bar, &phase, piece, wred, &s_expired);
    // scan of the piece sums (float-float, fixed order).  A piece's lower end
    // is the previous piece's upper end bit for bit, so the pieces tile the
    // slice with no gap and no overlap.
    ff incl{piece[tid], 0.f};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff n = ff_shfl_up(incl, o);
        if (lane >= o)
            incl = ff_add(n, incl);
    }
    ff excl = ff_shfl_up(incl, 1);
    if (lane == 0)
        excl = {0.f, 0.f};
    if (tid == 0) {
        s_hit = INT_MAX;
        s_last = -1;
    }
    if (lane == 31)
        s_excl[warp] = incl;
    __syncthreads();
    ff wbase = base;
    for (int q = 0; q < warp; ++q)
        wbase = ff_add(wbase, s_excl[q]);
    const ff lo = ff_add(wbase, excl), hi = ff_add(wbase, incl);
    if (!past && ff_le(lo, target) && ff_gt(hi, target))
        atomicMin(&s_hit, tid);
    __syncthreads();
    // the piece walk repeats the piece sum's additions, so it meets the same
    // running sums; rem may round up to the piece total: then the piece's
    // last element with weight > 0
    constexpr int E = Elem<T>::kPerVec;
    const int nv = (len + E - 1) / E;
    const int v0 = min(nv, tid * p.pv), v1 = min(nv, v0 + p.pv);
    if (s_hit == tid) {
        const float rem = __fadd_rn(__fsub_rn(target.hi, lo.hi), __fsub_rn(target.lo, lo.lo));
        s_last = piece_find<T>(d, tb, db, len, v0, v1, rem);
    } else if (s_hit == INT_MAX) {  // past the end after rounding: the last element with mass
        const int lp = piece_find<T>(d, tb, db, len, v0, v1, INFINITY);
        if (lp >= 0)
            atomicMax(&s_last, lp);
    }
    __syncthreads();
    if (tid == 0) {
        const int res = s_last;
        int y = res >= 0 ? c0 + res : -1;
        if (y < 0)
            set_status(p.status, ST_NONFINITE);
        if (timeout || s_expired) {  // a copy gave up: the data may be stale
            y = -1;
            p.out_len[i] = -1;
            for (int jj = 0; jj <= K; ++jj)
                p.out_tokens[t0 + jj] = -1;
        }
        p.out_tokens[trow_i] = y;
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

template <typename T>
static cudaError_t prepare_finish_sample()
{
    static cudaError_t once = [] {
        cudaError_t e = cudaFuncSetAttribute(finish_sample_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             2 * kStageRowBytes);
        if (e == cudaSuccess)  // clusters of 16 CTAs
            e = cudaFuncSetAttribute(finish_sample_kernel<T>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return e;
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
    {  // final-draw geometry: ncl ranges of R entries, weighed in slices.  16
        // CTAs per request while the clusters fit the GPU at one CTA per SM
        // (larger clusters are harder to place), else 8.
        const int gran = 16 / e;
        const int ncl = (int64_t)a.B * kCluster <= (int64_t)sm_count() ? kCluster : kCluster / 2;
        fp.ncl = ncl;
        const int R = (int)((((int64_t)a.V + ncl - 1) / ncl + gran - 1) / gran * gran);
        const int slice = std::min(R, kStageRowBytes / e);
        const int nv = (slice * e + 15) / 16;
        fp.R = R;
        fp.slice = slice;
        fp.pv = ((nv + kSampleThreads - 1) / kSampleThreads) | 1;  // odd: no bank conflicts
        fp.stage_smem = (int)align_up((size_t)slice * e, 128);
        if ((R + slice - 1) / slice > kMaxSlices)
            return cudaErrorInvalidValue;  // vocabulary beyond the draw's slice table
    }
    fp.tma = tma;
    fp.c = sp.c;
    fp.status = sp.status;
    fp.cu_flag = sp.cu_flag;
    fp.part = sp.part;

    cudaError_t err = prepare_stream<T, GREEDY>();
    if (err == cudaSuccess && !GREEDY)
        err = prepare_finish_sample<T>();
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
    cfg.blockDim = dim3(kFinishThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    if (GREEDY) {
        cfg.gridDim = dim3((unsigned)a.B);
        cfg.dynamicSmemBytes = 0;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, finish_greedy_kernel<T>, fp);
    } else {
        cfg.gridDim = dim3((unsigned)(a.B * fp.ncl));
        cfg.blockDim = dim3(kSampleThreads);
        cfg.dynamicSmemBytes = 2 * (size_t)fp.stage_smem;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = fp.ncl;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        err = cudaLaunchKernelEx(&cfg, finish_sample_kernel<T>, fp);
    }
    if (err != cudaSuccess)
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
