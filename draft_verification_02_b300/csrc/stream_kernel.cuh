// stream_kernel.cuh - kernel 1 of the verification path: the streaming
// pass over every row that must be read (see verify.cu for the whole path).
#pragma once

#include "verify_params.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// kernel 1: stream the rows
// ---------------------------------------------------------------------------

// Units in flight per warp and CTAs per SM: 2 units of 4 KB with 3 CTAs of 8
// warps per SM (80 registers, 64 KB of ring per CTA).  Measured on B300
// against 3 units with 2 CTAs per SM (the previous setting), streaming
// fraction of the measured HBM peak: B=128, V=151936 at T=0.7 0.936 vs
// 0.894, at T=0 0.874 vs 0.858; B=32, K=16 0.855 vs 0.844, at T=0 0.739 vs
// 0.716; the padded D-cut rows 0.613 vs 0.580.  2 KB units (rings of 4-6, 2
// or 3 CTAs) and one CTA with a ring of 4 were all slower (0.60-0.73).
#ifndef SV_RING
#define SV_RING 2
#endif
#ifndef SV_STREAM_CTAS_PER_SM
#define SV_STREAM_CTAS_PER_SM 3
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
    if (lane == 0 && slot)
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
    Geometry g = p.g;  // the host's split until the offsets arrive (real_split)
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

    int64_t u0 = w < g.P ? (int64_t)w * g.U / g.P : 0;
    int64_t u1 = w < g.P ? (int64_t)(w + 1) * g.U / g.P : 0;
    const T *tbase = reinterpret_cast<const T *>(p.target);
    const T *dbase = reinterpret_cast<const T *>(p.draft);
    const bool padded = !GREEDY && p.draft_stride > 0;

    // Where the unit at (row rg of the split's index space, column chunk q)
    // comes from; false when the row lies past the real rows (nt target, nd
    // draft) and `check` is set.
    int req_hint = 0;  // request of the last slot found (consecutive units share rows)
    auto locate = [&](int64_t rg, int q, const T *&src, int &len, int &col0, int64_t nt,
                      int64_t nd, bool check) -> bool {
        col0 = q * g.Q;
        len = min(g.Q, V - col0);
        if (rg < g.nt) {
            if (check && rg >= nt)
                return false;
            if (!SV_IN_BOUNDS(rg, g.max_rows, p.status))
                return false;
            src = tbase + rg * (int64_t)V + col0;
            return true;
        }
        const int64_t slot = rg - g.nt;
        if (check && slot >= nd)
            return false;
        int64_t row = slot;
        if (padded) {  // packed slot -> (request, position) -> padded row
            int lo = req_hint;
            if (!(cu_s[lo] <= slot && slot < cu_s[lo + 1])) {  // the request holding slot
                lo = 0;
                int hi = B - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (cu_s[mid] <= slot)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                req_hint = lo;
            }
            row = (int64_t)lo * p.draft_stride + (slot - cu_s[lo]);
        }
        if (!SV_IN_BOUNDS(row, p.draft_rows, p.status))
            return false;
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
    int64_t n_units = u1 - u0;
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
    // it maps padded rows through them).  Without offsets (p.cu == nullptr)
    // every row is real.
    if (p.cu != nullptr && (padded || blockIdx.x == 0)) {
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
            if (bad && p.out_tokens) {  // (a shard's row pass has no outputs to poison)
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
    if (p.cu != nullptr) {
        int v = lane == 0 ? __ldg(p.cu + B) : 0;
        v = __shfl_sync(0xffffffffu, v, 0);
        nd = min(nd, (int64_t)v);
        nt = min(g.max_rows, (int64_t)v + B);
        const Geometry gr = real_split(g, B, v);
        if (gr.U != g.U) {
            // a loose host bound: the real rows are split afresh.  The
            // speculative first copies are waited for and dropped.
            bool ok = true;
            if (p.tma)
                for (int k = 0; k < kRing; ++k)
                    if (issued >> k & 1)
                        ok = mbar_wait_bounded(&bars[wib][k], phase >> k & 1) && ok;
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0)
                    set_status(p.status, ST_TIMEOUT);
                for (int k = 0; k < kRing; ++k)  // the copies in flight, once more
                    if (issued >> k & 1)
                        mbar_wait_bounded(&bars[wib][k], phase >> k & 1);
                return;
            }
            if (p.tma)
                for (int k = 0; k < kRing; ++k)
                    if (issued >> k & 1)
                        phase ^= 1u << k;
            issued = 0;
            n_issued = 0;
            __syncwarp();  // every lane is done with the dropped copies' slots
            g = gr;
            u0 = w < g.P ? (int64_t)w * g.U / g.P : 0;
            u1 = w < g.P ? (int64_t)(w + 1) * g.U / g.P : 0;
            n_units = u1 - u0;
            c_rg = u0 / g.cpr;
            c_q = (int)(u0 - c_rg * g.cpr);
            i_rg = c_rg;
            i_q = c_q;
            if (!padded)  // the first copies of the new split
                for (; n_issued < kRing && n_issued < n_units; ++n_issued) {
                    issue(i_rg, i_q, n_issued, nt, nd, true);
                    advance(i_rg, i_q);
                }
        }
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
                bool ok = mbar_wait_bounded(&bars[wib][k], phase >> k & 1);
                if ((uint64_t)(u0 + n) + 1 == p.debug_unit)
                    ok = false;  // test hook: this wait reports expiry (its copy has landed)
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
            store_partial<GREEDY>(acc, p.c,
                                  SV_IN_BOUNDS(rg + w, p.part_cap, p.status) ? p.part + rg + w
                                                                             : nullptr);
            seg_active = false;
        }
        if (++k == kRing)
            k = 0;
    }
}

}  // namespace sv
