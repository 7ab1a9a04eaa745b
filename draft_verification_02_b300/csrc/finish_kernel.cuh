// finish_kernel.cuh - kernel 2 of the verification path: merge, accept test
// and final draw (see verify.cu for the whole path).
#pragma once

#include "verify_params.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// kernel 2: merge, accept test, final draw
// ---------------------------------------------------------------------------

constexpr int kFinishThreads = 256;
constexpr int kFinishWarps = kFinishThreads / 32;
constexpr int kCluster = 16;               // most CTAs per request in the sampling finish kernel
constexpr int kSampleThreads = 256;        // threads per CTA of the sampling finish kernel
constexpr int kSampleWarps = kSampleThreads / 32;
#ifndef SV_STAGE_KB
#define SV_STAGE_KB 48
#endif
constexpr int kStageRowBytes = SV_STAGE_KB * 1024;  // largest slice of one row staged at a time
constexpr int kMaxSlices = 64;             // slices per CTA range (bounds V)

// Slices of at most stage_bytes per row for ncl ranges of a V-entry row;
// false when a range needs more slices than the slice table holds.
inline bool fill_draw_geometry(FinishParams &fp, int ncl, int V, int e, int stage_bytes)
{
    const int gran = 16 / e;
    fp.ncl = ncl;
    const int R = (int)((((int64_t)V + ncl - 1) / ncl + gran - 1) / gran * gran);
    const int slice = std::min(R, stage_bytes / e);
    const int nv = (slice * e + 15) / 16;
    fp.R = R;
    fp.slice = slice;
    fp.pv = ((nv + kSampleThreads - 1) / kSampleThreads) | 1;  // odd: no bank conflicts
    fp.stage_smem = (int)align_up((size_t)slice * e, 128);
    return (R + slice - 1) / slice <= kMaxSlices;
}

// Geometry of a cluster draw over V entries, one cluster per draw: ncl
// ranges of R entries, weighed in slices.  16 CTAs per draw while the
// clusters fit the GPU at two CTAs per SM, else 8 while they fit it at four,
// else 4; a grid of more than two CTAs per SM (a "dense" grid) takes slices
// of half the largest size, so that four CTAs fit an SM, with the
// finish-kernel instance whose registers allow four.  Measured on B300, ms
// per step: B = 16, V = 128000: 16 CTAs 0.0206, 8 CTAs 0.0222, 4 CTAs
// 0.0278; B = 32 at V = 151936: 8 CTAs, 48 KB slices best (0.0690; dense
// from one CTA per SM 0.0705, 16 CTAs 0.0755, 4 CTAs 0.0773); B = 64 at
// V = 151936: 8 CTAs dense 0.0794, 4 CTAs 0.0814, 48 KB slices at three
// CTAs per SM 0.0915; B = 128: 4 CTAs dense (one wave) 0.1403, 8 CTAs dense
// (1.73 waves) 0.1473, 48 KB slices 0.1652.  sms: the GPU's SM count.
// False when the vocabulary exceeds the slice table.
#ifndef SV_DENSE_PER_SM
#define SV_DENSE_PER_SM 2
#endif
inline bool draw_geometry(FinishParams &fp, int64_t draws, int V, int e, int64_t sms)
{
    int ncl = draws * kCluster <= 2 * sms              ? kCluster
              : draws * (kCluster / 2) <= 4 * sms ? kCluster / 2
                                                       : kCluster / 4;
#ifdef SV_NCL
    ncl = SV_NCL;
#endif
    // a vocabulary whose ranges need more slices than the table holds takes
    // more CTAs per draw
    for (; ncl <= kCluster; ncl *= 2) {
        if (draws * ncl > SV_DENSE_PER_SM * sms &&
            fill_draw_geometry(fp, ncl, V, e, kStageRowBytes / 2))
            return true;
        if (fill_draw_geometry(fp, ncl, V, e, kStageRowBytes))
            return true;
    }
    return false;
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

// T = 0: the maximum of flattened row rg and the lowest index holding it
// (INT_MAX when every entry is -inf), merged from the row's partials; nan is
// set when any entry is NaN.  The same result in every lane.
__device__ __forceinline__ void merge_argmax_pair(const Partial *part, const Geometry &g,
                                                  int64_t rg, float &best, int &bidx, bool &nan)
{
    const int lane = threadIdx.x & 31;
    int wf, wl;
    row_span(g, rg, wf, wl);
    best = -INFINITY;
    bidx = INT_MAX;
    int bad = 0;
    for (int w = wf + lane; w <= wl; w += 32) {
        const Partial q = load_partial(part + rg + w);
        if (q.idx == -2)
            bad = 1;
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
    nan = __any_sync(0xffffffffu, bad);
}

// T = 0: lowest argmax of target row rg; -1 masked row, -2 NaN, -3 +inf.
__device__ __forceinline__ int merge_argmax_row(const Partial *part, const Geometry &g, int64_t rg)
{
    float best;
    int bidx;
    bool nan;
    merge_argmax_pair(part, g, rg, best, bidx, nan);
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
    const int cu_tot = __ldg(p.cu + p.B);
    const bool shape = request_shape_ok(p, i, cu_i, K);
    const bool act = shape && warp == 0 && lane < K;
    const int64_t dx = act ? draft_index(p.draft_stride, p.cu, i, lane) : 0;
    const int x = act && SV_IN_BOUNDS(dx, p.draft_rows, p.status) ? __ldg(p.tokens + dx) : -1;

    pdl_wait();  // kernel 1 has completed and its writes are visible
    if (__ldcg(p.cu_flag) == 0u || !shape)
        return;  // malformed offsets: kernel 1 poisoned every output
    const Geometry g = real_split(p.g, p.B, cu_tot);  // kernel 1's split of the real rows
    const int64_t t0 = (int64_t)cu_i + i;
    for (int rho = warp; rho <= K; rho += kFinishWarps) {
        int wf, wl;
        row_span(g, t0 + rho, wf, wl);
        const int gj = SV_IN_BOUNDS(t0 + rho + wl, p.part_cap, p.status)
                           ? merge_argmax_row(p.part, g, t0 + rho)
                           : -2;
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
            if (SV_IN_BOUNDS(t0 + jj, p.g.max_rows, p.status))
                p.out_tokens[t0 + jj] = -1;
        if (lane == 0 && SV_IN_BOUNDS(i, p.B, p.status))
            p.out_len[i] = -1;
        return;
    }
    const int a = rej ? __ffs(rej) - 1 : K;
    for (int jj = lane; jj <= K; jj += 32)
        if (SV_IN_BOUNDS(t0 + jj, p.g.max_rows, p.status))
            p.out_tokens[t0 + jj] = jj < a ? x : (jj == a ? row_g[a] : -1);
    if (lane == 0 && SV_IN_BOUNDS(i, p.B, p.status))
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
// Vectors wholly inside the slice take no per-element bounds test; only the
// slice's last vector can be partial.
template <typename T>
__device__ __forceinline__ float piece_sum(const DrawCtx d, const T *tb, const T *db, int len,
                                           int v0, int v1)
{
    constexpr int E = Elem<T>::kPerVec;
    const uint4 *tv = reinterpret_cast<const uint4 *>(tb);
    const uint4 *dv = reinterpret_cast<const uint4 *>(db);
    const int vfull = min(v1, len / E);
    float acc = 0.f;
    if (d.resid) {
#pragma unroll 1
        for (int v = v0; v < vfull; ++v) {
            float ft[E], fd[E];
            Elem<T>::unpack(tv[v], ft);
            Elem<T>::unpack(dv[v], fd);
#pragma unroll
            for (int h = 0; h < E; ++h)
                acc = __fadd_rn(acc, draw_w(d, ft[h], fd[h]));
        }
    } else {
#pragma unroll 1
        for (int v = v0; v < vfull; ++v) {
            float ft[E];
            Elem<T>::unpack(tv[v], ft);
#pragma unroll
            for (int h = 0; h < E; ++h)
                acc = __fadd_rn(acc, draw_w(d, ft[h], 0.f));
        }
    }
    for (int v = max(v0, vfull); v < v1; ++v) {  // the partial last vector
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
// bit (the same additions in the same order).
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

// piece_find by one warp: the lanes compute the piece's weights (its
// exponentials) into wbuf, then lane 0 adds them in index order with the
// additions of piece_sum, so the running sums are the same bit for bit.
// Every lane of the warp calls it and gets the same index.
template <typename T>
__device__ __forceinline__ int piece_find_warp(const DrawCtx d, const T *tb, const T *db, int len,
                                               int v0, int v1, float rem, float *wbuf)
{
    constexpr int E = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    const int k0 = v0 * E, n = max(0, min(v1 * E, len) - k0);  // the piece's elements
    for (int q = lane; q < n; q += 32) {
        const int k = k0 + q;
        wbuf[q] = draw_w(d, Elem<T>::at(tb, k), d.resid ? Elem<T>::at(db, k) : 0.f);
    }
    __syncwarp();
    int res = -1;
    if (lane == 0) {
        float acc = 0.f;
        for (int q = 0; q < n; ++q) {
            const float w = wbuf[q];
            acc = __fadd_rn(acc, w);
            if (w > 0.f)
                res = k0 + q;
            if (acc > rem) {
                res = k0 + q;
                break;
            }
        }
    }
    return __shfl_sync(0xffffffffu, res, 0);
}

// Stage elements [c0, c0 + len) of the draw rows into shared memory (one
// TMA bulk copy per row, or plain loads when the rows are not 16-byte
// aligned), then every thread sums its contiguous piece (kept in piece[]
// for the search) and the pieces are added as float-float pairs in a fixed
// order.  Once any copy of this call has timed out nothing more is copied.
// With copy == false the slice is already staged.
template <typename T>
__device__ __forceinline__ ff weigh_slice(const FinishParams &p, const DrawCtx d, const T *trow,
                                       const T *drow, int c0, int len, T *tb, T *db,
                                       uint64_t *bar, uint32_t *phase, float *piece, ff *wred,
                                       int *expired, bool copy = true)
{
    constexpr int E = Elem<T>::kPerVec;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // earlier readers of the buffers, piece and wred are done
    const bool stop = __syncthreads_or(tid == 0 && (read_status(p.status) & ST_TIMEOUT));
    if (copy && !stop && len > 0) {
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
    ff ws{ps, 0.f};
#pragma unroll 1
    for (int o = 16; o > 0; o >>= 1)  // warp sum, the same bits in every lane
        ws = ff_add(ws, ff_shfl_xor(ws, o));
    __syncthreads();  // piece[] complete; wred free
    if (lane == 0)
        wred[warp] = ws;
    __syncthreads();
    ff tot = wred[0];
    for (int q = 1; q < kSampleWarps; ++q)
        tot = ff_add(tot, wred[q]);
    return tot;
}

// The same, compiled once out of line.  A kernel that calls it keeps more
// registers per thread (the call's convention), so fewer of its CTAs share
// an SM with the streaming kernel's; measured, that suits small grids.
template <typename T>
__device__ __noinline__ ff weigh_slice_outlined(const FinishParams &p, const DrawCtx d,
                                                const T *trow, const T *drow, int c0, int len,
                                                T *tb, T *db, uint64_t *bar, uint32_t *phase,
                                                float *piece, ff *wred, int *expired, bool copy)
{
    return weigh_slice<T>(p, d, trow, drow, c0, len, tb, db, bar, phase, piece, wred, expired,
                          copy);
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

// Shared-memory state of one CTA's part in a cluster draw.
template <typename T>
struct DrawShared {
    T *tb, *db;  // staged slices of the two rows
    uint64_t *bar;
    float *piece;
    ff *wred, *slice_tot, *s_excl;
    ff (*cl_sum)[kCluster];  // written by every CTA of the cluster
    int *s_hit, *s_last, *s_expired;
};

// The search of the CTA whose range [r0, r1) (nsl slices with totals
// slice_tot, in order) holds the target: base is the running sum before the
// range; past marks a target at or beyond the end of the whole sum after
// rounding (then the last element with weight > 0 wins).  The slice, then the
// thread piece, then the element; `weighed` is the slice already staged (-1
// none).  Returns the drawn index (or -1 if none has weight), in every thread.
template <typename T, bool OUTLINE>
__device__ __forceinline__ int find_in_range(const FinishParams &p, const DrawCtx &d,
                                             const T *trow, const T *drow, int r0, int r1,
                                             int nsl, ff base, ff target, bool past, int weighed,
                                             const ff *slice_tot, const DrawShared<T> &sh,
                                             uint32_t &phase)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    T *tb = sh.tb, *db = sh.db;
    float *piece = sh.piece;
    ff *wred = sh.wred, *s_excl = sh.s_excl;
    int &s_hit = *sh.s_hit, &s_last = *sh.s_last, &s_expired = *sh.s_expired;
    uint64_t &bar = *sh.bar;
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
    if (sl != weighed) {
        if (OUTLINE)
            weigh_slice_outlined<T>(p, d, trow, drow, c0, len, tb, db, &bar, &phase, piece, wred,
                                    &s_expired, true);
        else
            weigh_slice<T>(p, d, trow, drow, c0, len, tb, db, &bar, &phase, piece, wred,
                           &s_expired);
    }
    // scan of the piece sums (float-float, fixed order).  A piece's lower end
    // is the previous piece's upper end bit for bit, so the pieces tile the
    // slice with no gap and no overlap.
    ff incl{piece[tid], 0.f};
#pragma unroll 1
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
    const int hit = s_hit;
    if (hit != INT_MAX) {
        if (warp == hit >> 5) {  // the hit thread's warp walks its piece
            const float rem = __fadd_rn(__fsub_rn(target.hi, lo.hi), __fsub_rn(target.lo, lo.lo));
            const int hl = hit & 31;
            const int k = piece_find_warp<T>(d, tb, db, len, __shfl_sync(0xffffffffu, v0, hl),
                                             __shfl_sync(0xffffffffu, v1, hl),
                                             __shfl_sync(0xffffffffu, rem, hl), piece);
            if (lane == 0)
                s_last = k;
        }
    } else {  // past the end after rounding: the last element with mass
        const int lp = piece_find<T>(d, tb, db, len, v0, v1, INFINITY);
        if (lp >= 0)
            atomicMax(&s_last, lp);
    }
    __syncthreads();
    return s_last >= 0 ? c0 + s_last : -1;
}

// The final draw of one cluster: the CTAs split the vocabulary into ncl
// ranges, weigh theirs (w = max(0, p - q) with d.resid, else the unnormalised
// p), exchange the range sums through distributed shared memory, and the CTA
// whose range holds u*S finds the token.  Returns, in every thread of that
// CTA, the drawn index (or -1 if it found none); -2 in the other CTAs, -1 in
// all CTAs when no range has mass.  Every CTA of the cluster must call it
// (it contains cluster barriers); no shared memory of another CTA is touched
// after it returns.  The CTA's copy barrier starts at phase parity 0.
template <typename T, bool OUTLINE>
__device__ __forceinline__ int draw_token(const FinishParams &p, DrawCtx d, const T *trow,
                                          const T *drow, float uf, uint32_t rank, int ncl,
                                          const DrawShared<T> &sh)
{
    const int tid = threadIdx.x, lane = tid & 31;
    T *tb = sh.tb, *db = sh.db;
    float *piece = sh.piece;
    ff *wred = sh.wred, *slice_tot = sh.slice_tot;
    ff(*cl_sum)[kCluster] = sh.cl_sum;
    int &s_expired = *sh.s_expired;
    uint64_t &bar = *sh.bar;
    const int r0 = min(p.V, (int)rank * p.R), r1 = min(p.V, r0 + p.R);
    const int nsl = r1 > r0 ? (r1 - r0 + p.slice - 1) / p.slice : 0;
    int weighed = -1;  // slice staged in shared memory
    uint32_t phase = 0u;  // parity of the copy barrier's next phase

    // pass 0 sums max(0, p_a - q_a) (or p_K); an all-zero residual makes a
    // second pass over p_a (the same decision in every CTA)
    int cs = -1;
    bool past = true, redo = false;
    ff base{0.f, 0.f}, target{0.f, 0.f};
    for (int pass = 0; pass < 2; ++pass) {
        // the slices last to first: the first (the largest) stays staged for
        // the owner's search, which finds the target there most often
        for (int k = 0; k < nsl; ++k) {
            const int sl = nsl - 1 - k;
            const int c0 = r0 + sl * p.slice, len = min(p.slice, r1 - c0);
            const ff ss =
                OUTLINE ? weigh_slice_outlined<T>(p, d, trow, drow, c0, len, tb, db, &bar, &phase,
                                                  piece, wred, &s_expired, true)
                        : weigh_slice<T>(p, d, trow, drow, c0, len, tb, db, &bar, &phase, piece,
                                         wred, &s_expired);
            weighed = sl;
            if (tid == 0)
                slice_tot[sl] = ss;
        }
        __syncthreads();  // slice_tot complete
        ff mine{0.f, 0.f};  // the range's sum, in slice order
        for (int sl = 0; sl < nsl; ++sl)
            mine = ff_add(mine, slice_tot[sl]);
        if (tid < ncl)
            st_cluster_ff(&cl_sum[pass][rank], (uint32_t)tid, mine);
        cluster_arrive_release();
        cluster_wait_acquire();  // (2 + pass) every CTA holds every range sum
        // S and the range holding u*S, in every warp (lane r holds range r):
        // an inclusive float-float scan in range order, the same bits in every
        // warp of every CTA.  `past` marks u*S at or beyond the end after
        // rounding: then the last weight > 0 wins.
        {
            const ff v = lane < ncl ? cl_sum[pass][lane] : ff{0.f, 0.f};
            ff incl = v;
#pragma unroll 1
            for (int o = 1; o < 32; o <<= 1) {
                const ff n = ff_shfl_up(incl, o);
                if (lane >= o)
                    incl = ff_add(n, incl);
            }
            const ff S = {__shfl_sync(0xffffffffu, incl.hi, 31),
                          __shfl_sync(0xffffffffu, incl.lo, 31)};
            target = ff_mul(S, uf);
            const unsigned over = __ballot_sync(0xffffffffu, lane < ncl && ff_gt(incl, target));
            const unsigned mass = __ballot_sync(0xffffffffu, lane < ncl && v.hi > 0.f);
            cs = over ? __ffs(over) - 1 : (mass ? 31 - __clz(mass) : -1);
            ff excl = ff_shfl_up(incl, 1);
            if (lane == 0)
                excl = {0.f, 0.f};
            const int src = cs < 0 ? 0 : cs;
            base = {__shfl_sync(0xffffffffu, excl.hi, src), __shfl_sync(0xffffffffu, excl.lo, src)};
            past = over == 0u;
            redo = !(S.hi > 0.f);
        }
        if (!(d.resid && redo))
            break;
        d.resid = false;  // all-zero residual: draw from p_a instead
    }
    // no shared memory of another CTA is touched after this point
    if ((int)rank != cs)
        return cs < 0 ? -1 : -2;  // -1: no mass at all (never with finite rows)

    return find_in_range<T, OUTLINE>(p, d, trow, drow, r0, r1, nsl, base, target, past, weighed,
                                     slice_tot, sh, phase);
}

// MINB: CTAs per SM the registers must allow (4 caps them at 64, for grids
// of more than four CTAs per SM; 2 otherwise).
template <typename T, bool OUTLINE, int MINB>
__global__ void __launch_bounds__(kSampleThreads, MINB) finish_sample_kernel(const FinishParams p)
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
    __shared__ int s_hit, s_last, s_expired;

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
    const int cu_tot = __ldg(p.cu + p.B);
    const bool shape = request_shape_ok(p, i, cu_i, K);
    const int64_t t0 = (int64_t)cu_i + i;
    const int nrows = 2 * K + 1;
    // lane j < K of every warp: the drafted token and its uniform (accept test)
    const bool act = shape && lane < K;
    int x = -1;
    float u = 0.f;
    int64_t di = 0;
    if (act) {
        di = draft_index(p.draft_stride, p.cu, i, lane);
        if (SV_IN_BOUNDS(di, p.draft_rows, p.status)) {
            x = __ldg(p.tokens + di);
            u = __ldg(p.u_accept + di);
        }
    }
    // the rows this warp merges: with at most one row per warp of a CTA,
    // every CTA merges all of them (row k = warp), else the rows are spread
    // over the cluster (k = rank + ncl * (warp + kSampleWarps * t)) and sent
    // to every CTA; rows past the cluster's 2 * kSampleWarps * ncl (with
    // clusters of 4 and K = 32 only) are merged by every CTA itself after the
    // exchange.  Target rows 0..K, then draft rows 0..K-1; the logit at the
    // drafted token of each such row.
    const bool local = nrows <= kSampleWarps;
    int my_k[2];
    float g[2] = {-INFINITY, -INFINITY};
    bool g_ok[2] = {false, false};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        my_k[t] = local ? (t == 0 ? warp : nrows) : (int)rank + ncl * (warp + kSampleWarps * t);
        if (!shape || my_k[t] >= nrows)
            my_k[t] = -1;
        else if (my_k[t] != K) {
            const int j = my_k[t] < K ? my_k[t] : my_k[t] - K - 1;
            const int64_t dj = draft_index(p.draft_stride, p.cu, i, j);
            const int xj = SV_IN_BOUNDS(dj, p.draft_rows, p.status) ? __ldg(p.tokens + dj) : -1;
            if (xj >= 0 && xj < p.V &&
                (my_k[t] < K ? SV_IN_BOUNDS(t0 + j, p.g.max_rows, p.status)
                             : SV_IN_BOUNDS(dj, p.draft_rows, p.status))) {
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
    const Geometry gs = real_split(p.g, p.B, cu_tot);  // kernel 1's split of the real rows
    // an expired wait of kernel 1 only poisons; its flag is read now, off the
    // critical path
    const bool timeout = warp == 0 && (read_status(p.status) & ST_TIMEOUT);

    // ---- (m, s) and p(x) of the request's rows, one or two rows per warp of
    // the cluster, sent to every CTA
    // merge of row k's partials into (m, s) across the warp
    auto merge_row = [&](int k, float &m, ff &sr) {
        const int64_t rg = k <= K ? t0 + k : gs.nt + cu_i + (k - K - 1);
        int wf, wl;
        row_span(gs, rg, wf, wl);
        for (int w = wf + lane; w <= wl; w += 32) {
            if (!SV_IN_BOUNDS(rg + w, p.part_cap, p.status))
                continue;
            const Partial pt = load_partial(p.part + rg + w);
            lse_combine(m, sr, pt.m, {pt.s_hi, pt.s_lo}, p.c);
        }
#pragma unroll 1
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m, o);
            const ff so = ff_shfl_xor(sr, o);
            lse_combine(m, sr, mo, so, p.c);
        }
    };
    float mm[2] = {-INFINITY, -INFINITY}, px[2] = {0.f, 0.f};
    ff sm[2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (my_k[t] < 0)
            continue;
        merge_row(my_k[t], mm[t], sm[t]);
        px[t] = g_ok[t] && row_ok(mm[t], sm[t]) ? softmax_at(g[t], mm[t], sm[t], p.c) : 0.f;
    }
    if (local) {  // every CTA merged every row itself
        if (my_k[0] >= 0 && lane == 0) {
            row_m[my_k[0]] = mm[0];
            row_s[my_k[0]] = sm[0];
            row_p[my_k[0]] = px[0];
        }
        __syncthreads();
        cluster_wait_acquire();  // (0) complete (long since)
    } else {
        cluster_wait_acquire();  // (0) complete: every CTA's shared memory is live
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (my_k[t] >= 0 && lane < ncl)
                st_cluster_row(row_m, row_s, row_p, my_k[t], (uint32_t)lane, mm[t], sm[t], px[t]);
        cluster_arrive_release();
        cluster_wait_acquire();  // (1) every CTA holds every row's (m, s, p(x))
        const int spread = 2 * kSampleWarps * ncl;
        if (nrows > spread) {  // the rows past the cluster's share, in every CTA
#pragma unroll 1
            for (int k = spread + warp; k < nrows; k += kSampleWarps) {
                bool ok = false;
                float gj = -INFINITY;
                if (k != K) {  // the logit at the drafted token (the bonus row has none)
                    const int j = k < K ? k : k - K - 1;
                    const int64_t dj = draft_index(p.draft_stride, p.cu, i, j);
                    const int xj =
                        SV_IN_BOUNDS(dj, p.draft_rows, p.status) ? __ldg(p.tokens + dj) : -1;
                    ok = xj >= 0 && xj < p.V &&
                         (k < K ? SV_IN_BOUNDS(t0 + j, p.g.max_rows, p.status)
                                : SV_IN_BOUNDS(dj, p.draft_rows, p.status));
                    if (ok)
                        gj = k < K ? Elem<T>::ld_global(tbase + (t0 + j) * p.V, xj)
                                   : Elem<T>::ld_global(dbase + dj * p.V, xj);
                }
                float m = -INFINITY;
                ff sr{0.f, 0.f};
                merge_row(k, m, sr);
                if (lane == 0) {
                    row_m[k] = m;
                    row_s[k] = sr;
                    row_p[k] = ok && row_ok(m, sr) ? softmax_at(gj, m, sr, p.c) : 0.f;
                }
            }
            __syncthreads();
        }
    }

    // ---- accept test and first rejection: every warp takes the same decision
    // from the same shared rows (no broadcast, no barrier); warp 0 writes
    int a;
    bool bad;
    DrawCtx d;
    {
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
        bad = nf || bt;
        a = rej ? __ffs(rej) - 1 : K;
        if (rank == 0 && warp == 0) {  // the request's outputs, written once
            const bool len_ok = SV_IN_BOUNDS(i, p.B, p.status);
            if (bad || timeout) {
                if (lane == 0)
                    set_status(p.status, (nf ? ST_NONFINITE : 0u) | (bt ? ST_INVALID : 0u));
                for (int jj = lane; jj <= K; jj += 32)
                    if (SV_IN_BOUNDS(t0 + jj, p.g.max_rows, p.status))
                        p.out_tokens[t0 + jj] = -1;
                if (lane == 0 && len_ok)
                    p.out_len[i] = -1;
            } else {
                const bool di_ok = act && SV_IN_BOUNDS(di, p.draft_rows, p.status);
                if (di_ok && p.out_p)
                    p.out_p[di] = pp;
                if (di_ok && p.out_q)
                    p.out_q[di] = qq;
                for (int jj = lane; jj <= K; jj += 32) {
                    if (!SV_IN_BOUNDS(t0 + jj, p.g.max_rows, p.status))
                        continue;
                    if (jj < a)
                        p.out_tokens[t0 + jj] = x;  // jj == lane since a <= 32
                    else if (jj > a)
                        p.out_tokens[t0 + jj] = -1;
                }
                if (lane == 0 && len_ok)
                    p.out_len[i] = a;
            }
        }
        // the final draw's constants
        d.resid = a < K;
        d.c = p.c;
        const float mt = row_m[a];
        d.mct = mt * p.c;
        d.sc_t = ff_recip_scaled(mc_correction(mt, d.mct, p.c), row_s[a]);
        d.mcd = 0.f;
        d.sc_d = 0.f;
        if (d.resid) {
            const float md = row_m[K + 1 + a];
            d.mcd = md * p.c;
            d.sc_d = ff_recip_scaled(mc_correction(md, d.mcd, p.c), row_s[K + 1 + a]);
        }
    }
    if (bad)
        return;  // same decision in every warp and CTA of the cluster; no more cluster traffic

    // ---- final draw: this CTA weighs its range of the vocabulary
    const int64_t trow_i = t0 + a;
    const int64_t drow_i = a < K ? draft_index(p.draft_stride, p.cu, i, a) : -1;
    // (the same verdict in every CTA of the cluster: no cluster barrier is split)
    if (!(SV_IN_BOUNDS(trow_i, p.g.max_rows, p.status) &&
          (drow_i < 0 || SV_IN_BOUNDS(drow_i, p.draft_rows, p.status))))
        return;
    const T *trow = tbase + trow_i * p.V;
    const T *drow = d.resid ? dbase + drow_i * p.V : nullptr;
    const DrawShared<T> sh{tb,     db,      &bar,    piece,      wred,   slice_tot,
                           s_excl, cl_sum,  &s_hit,  &s_last,    &s_expired};
    const int y0 = draw_token<T, OUTLINE>(p, d, trow, drow, uf, rank, ncl, sh);
    if (y0 == -2)
        return;  // another CTA's range holds u*S
    if (tid == 0) {
        int y = y0;
        if (y < 0)
            set_status(p.status, ST_NONFINITE);
        if (timeout || s_expired) {  // a copy gave up: the data may be stale
            y = -1;
            if (SV_IN_BOUNDS(i, p.B, p.status))
                p.out_len[i] = -1;
            for (int jj = 0; jj <= K; ++jj)
                if (SV_IN_BOUNDS(t0 + jj, p.g.max_rows, p.status))
                    p.out_tokens[t0 + jj] = -1;
        }
        p.out_tokens[trow_i] = y;
    }
}

// ---------------------------------------------------------------------------
// prefix confidence of drafted tokens
// ---------------------------------------------------------------------------

struct ConfParams {
    const void *draft;  // [B*Kmax][V], row i*Kmax + j
    const int32_t *tokens;
    const int32_t *kmax;
    int B, Kmax, V;
    Geometry g;  // the streaming pass over the B*Kmax rows
    float c;     // log2(e) / T (T > 0)
    float *out_conf;
    uint32_t *status;
    const Partial *part;
};

// One warp per draft row: conf = q(x) = 2^((g - m) c) / s from the row's
// merged partials (T > 0), or 1 when x is the row's lowest-index maximum
// (T = 0); 0 past kmax[i].  Launched as a programmatic dependent of the
// streaming pass; the token and the logit at it are read before waiting.
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kFinishThreads) confidence_kernel(const ConfParams p)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t r = (int64_t)blockIdx.x * kFinishWarps + warp;
    const int64_t nrow = (int64_t)p.B * p.Kmax;
    bool live = false, bad_k = false, bad_x = false;
    int x = -1;
    float gx = 0.f;
    if (r < nrow) {
        const int i = (int)(r / p.Kmax), j = (int)(r - (int64_t)i * p.Kmax);
        const int km = __ldg(p.kmax + i);
        bad_k = km < 0 || km > p.Kmax;
        live = !bad_k && j < km;
        if (live) {
            x = __ldg(p.tokens + r);
            bad_x = x < 0 || x >= p.V;
            if (!bad_x && !GREEDY)
                gx = Elem<T>::ld_global(reinterpret_cast<const T *>(p.draft) + r * p.V, x);
        }
    }
    pdl_wait();  // the streaming pass has completed and its writes are visible
    if (r >= nrow)
        return;
    float conf = 0.f;
    uint32_t err = 0;
    if (bad_k || bad_x) {
        err = ST_INVALID;
    } else if (live) {
        if constexpr (GREEDY) {
            const int gi = merge_argmax_row(p.part, p.g, r);
            if (gi < 0)
                err = ST_NONFINITE;
            else
                conf = gi == x ? 1.f : 0.f;
        } else {
            int wf, wl;
            row_span(p.g, r, wf, wl);
            float m = -INFINITY;
            ff s{0.f, 0.f};
            for (int w = wf + lane; w <= wl; w += 32) {
                const Partial q = load_partial(p.part + r + w);
                lse_combine(m, s, q.m, {q.s_hi, q.s_lo}, p.c);
            }
#pragma unroll 1
            for (int o = 16; o > 0; o >>= 1) {
                const float mo = __shfl_xor_sync(0xffffffffu, m, o);
                const ff so = ff_shfl_xor(s, o);
                lse_combine(m, s, mo, so, p.c);
            }
            if (row_ok(m, s))
                conf = softmax_at(gx, m, s, p.c);
            else
                err = ST_NONFINITE;
        }
    }
    if (lane == 0) {
        if (err) {
            set_status(p.status, err);
            conf = __int_as_float(0x7fc00000);
        }
        p.out_conf[r] = conf;
    }
}

// ---------------------------------------------------------------------------
// drafted tokens and acceptance statistics
// ---------------------------------------------------------------------------

// T > 0: one CTA per padded draft row r = i*Kmax + j, one read of the row
// from HBM.  The row streams through a ring of two slices (TMA bulk copies).
// Each slice's maximum fixes an integer reference M_k = ceil(max * c), and
// the slice is weighed in it, w = 2^(x c - M_k) <= 1, by thread pieces as in
// the verification draw, into the slice total T_k.  Totals in different
// references meet by exact power-of-two scaling, S = sum_k T_k 2^(M_k - M)
// with M = max_k M_k, so the slice holding u*S is found from the totals;
// that slice is copied once more and walked in its own reference, meeting
// the same running sums as its weighing, bit for bit.  x = the inverse CDF
// of q = softmax(row / T) at u[r]; q(x) = w(x) 2^(M_k - M) / S.  Rows past
// kmax[i] give -1 and 0 and are never read.
constexpr int kMaxRowSlices = 1408;  // 24 KB slices of a row of kMaxVocab f32 logits

// ff scaled by 2^n, exactly unless the low part leaves the normal range
__device__ __forceinline__ ff ff_ldexp(ff v, int n) { return {ldexpf(v.hi, n), ldexpf(v.lo, n)}; }

template <typename T>
__global__ void __launch_bounds__(kSampleThreads, 2) draft_sample_kernel(const FinishParams p)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ float piece[kSampleThreads];
    __shared__ ff wred[kSampleWarps];
    __shared__ float mred[kSampleWarps];
    __shared__ int s_bad, s_hit, s_last, s_sl, s_past, s_expired, s_shift;
    __shared__ ff s_rem, s_S;

    constexpr int E = Elem<T>::kPerVec;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const int i = (int)(r / p.Kmax), j = (int)(r - (int64_t)i * p.Kmax);
    const int km = __ldg(p.kmax + i);
    const bool bad_k = km < 0 || km > p.Kmax;
    if (bad_k || j >= km) {  // the whole CTA: no barrier yet
        if (tid == 0) {
            p.out_tokens[r] = -1;
            p.out_conf[r] = bad_k ? __int_as_float(0x7fc00000) : 0.f;
            if (bad_k)
                set_status(p.status, ST_INVALID);
        }
        return;
    }
    const float uf = __ldg(p.u_final + r);
    const T *row = reinterpret_cast<const T *>(p.target) + r * p.V;
    T *const buf0 = reinterpret_cast<T *>(dsm);
    T *const buf1 = reinterpret_cast<T *>(dsm + p.stage_smem);
    const int nsl = (p.V + p.slice - 1) / p.slice;
    // per slice: its total (float-float) and reference M_k (-inf: no mass)
    ff *const sl_tot = reinterpret_cast<ff *>(dsm + 2 * (size_t)p.stage_smem);
    float *const sl_ref = reinterpret_cast<float *>(sl_tot + nsl);
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        s_expired = 0;
        s_bad = 0;
    }
    __syncthreads();

    auto issue = [&](int sl, T *dst, uint64_t *bar) {  // thread 0: one bulk copy of slice sl
        const int c0 = sl * p.slice, len = min(p.slice, p.V - c0);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint32_t bytes = (uint32_t)len * (uint32_t)sizeof(T);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(dst, row + c0, bytes, bar);
    };
    auto land = [&](int sl, T *dst, uint64_t *bar, uint32_t &ph) {  // slice sl is in dst
        if (p.tma) {
            if (!mbar_wait_bounded(bar, ph)) {
                set_status(p.status, ST_TIMEOUT);
                s_expired = 1;
                mbar_wait_bounded(bar, ph);  // the copy in flight, once more
            }
            ph ^= 1u;
        } else {
            const int c0 = sl * p.slice, len = min(p.slice, p.V - c0);
            for (int k = tid; k < len; k += kSampleThreads)
                dst[k] = row[c0 + k];
            __syncthreads();
        }
    };
    // float-float sum of piece[0 .. kSampleThreads) in a fixed order, by warp 0
    // (every lane gets it)
    auto warp0_sum = [&]() -> ff {
        constexpr int per = kSampleThreads / 32;
        ff w{0.f, 0.f};
#pragma unroll
        for (int q = 0; q < per; ++q)
            w = ff_add(w, ff{piece[lane * per + q], 0.f});
#pragma unroll 1
        for (int o = 16; o > 0; o >>= 1)
            w = ff_add(w, ff_shfl_xor(w, o));
        return w;
    };
    // this thread's piece of a slice of len elements: vectors [v0, v1)
    auto piece_of = [&](int len, int &v0, int &v1) {
        const int nv = (len + E - 1) / E;
        v0 = min(nv, tid * p.pv);
        v1 = min(nv, v0 + p.pv);
    };
    DrawCtx d;
    d.resid = false;
    d.c = p.c;
    d.sc_t = 0.f;
    d.mcd = 0.f;
    d.sc_d = 0.f;

    // ---- one pass over the row: slice maxima, references and totals
    uint32_t ph0 = 0u, ph1 = 0u;
    if (p.tma && tid == 0) {
        issue(0, buf0, &bars[0]);
        if (nsl > 1)
            issue(1, buf1, &bars[1]);
    }
    for (int sl = 0; sl < nsl; ++sl) {
        const bool odd = sl & 1;
        T *const buf = odd ? buf1 : buf0;
        uint64_t *const bar = odd ? &bars[1] : &bars[0];
        if (odd)
            land(sl, buf, bar, ph1);
        else
            land(sl, buf, bar, ph0);
        const int len = min(p.slice, p.V - sl * p.slice);
        // maximum (packed for bf16)
        const uint4 *tv = reinterpret_cast<const uint4 *>(buf);
        const int nfull = len / E;
        float mx = -INFINITY;
        if constexpr (sizeof(T) == 2) {
            uint32_t m2 = 0xff80ff80u;  // -inf, -inf
#pragma unroll 4
            for (int v = tid; v < nfull; v += kSampleThreads) {
                const uint4 x = tv[v];
                m2 = max_nan_bf16x2(m2, max_nan_bf16x2(max_nan_bf16x2(x.x, x.y),
                                                       max_nan_bf16x2(x.z, x.w)));
            }
            mx = max_nan(bf16_lo(m2), bf16_hi(m2));
        } else {
#pragma unroll 4
            for (int v = tid; v < nfull; v += kSampleThreads) {
                const float4 x = reinterpret_cast<const float4 *>(buf)[v];
                mx = max_nan(mx, max_nan(max_nan(x.x, x.y), max_nan(x.z, x.w)));
            }
        }
        for (int k = nfull * E + tid; k < len; k += kSampleThreads)
            mx = max_nan(mx, Elem<T>::at(buf, k));
        mx = warp_max_nan(mx);
        if (lane == 0)
            mred[warp] = mx;
        __syncthreads();
        float sm = mred[0];
        for (int q = 1; q < kSampleWarps; ++q)
            sm = max_nan(sm, mred[q]);
        // the slice's reference: NaN / +inf (or a reference beyond the float
        // range of the weights) make the row an error
        const float ref = sm == -INFINITY ? -INFINITY : ceilf(sm * p.c);
        const bool bad = !(sm == -INFINITY || (ref > -1e30f && ref < 1e30f));
        const bool weigh = !bad && ref > -INFINITY;
        float ps = 0.f;
        if (weigh) {
            d.mct = ref;
            int v0, v1;
            piece_of(len, v0, v1);
            ps = piece_sum<T>(d, buf, nullptr, len, v0, v1);
        }
        piece[tid] = ps;
        __syncthreads();  // every thread is done with the slice and piece[] is complete
        if (warp == 0) {  // the slice total; the other warps go on to the next slice
            const ff tot = weigh ? warp0_sum() : ff{0.f, 0.f};
            if (lane == 0) {
                sl_tot[sl] = tot;
                sl_ref[sl] = bad ? -INFINITY : ref;
                if (bad)
                    s_bad = 1;
                if (p.tma && sl + 2 < nsl)  // the buffer is free: the slice after next
                    issue(sl + 2, buf, bar);
            }
        }
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            set_status(p.status, ST_NONFINITE);
            p.out_tokens[r] = -1;
            p.out_conf[r] = __int_as_float(0x7fc00000);
        }
        return;
    }

    // ---- S and the slice holding u*S (warp 0, slices in chunks of 32)
    if (warp == 0) {
        float M = -INFINITY;
        for (int k = lane; k < nsl; k += 32)
            M = fmaxf(M, sl_ref[k]);
        M = warp_max_nan(M);
        auto scaled = [&](int k) -> ff {  // T_k 2^(M_k - M), exact
            if (k >= nsl || sl_ref[k] == -INFINITY)
                return ff{0.f, 0.f};
            return ff_ldexp(sl_tot[k], max(-300, (int)(sl_ref[k] - M)));
        };
        ff S{0.f, 0.f};
        for (int c0 = 0; c0 < nsl; c0 += 32) {
            ff incl = scaled(c0 + lane);
#pragma unroll 1
            for (int o = 1; o < 32; o <<= 1) {
                const ff n = ff_shfl_up(incl, o);
                if (lane >= o)
                    incl = ff_add(n, incl);
            }
            S = ff_add(S, ff{__shfl_sync(0xffffffffu, incl.hi, 31),
                             __shfl_sync(0xffffffffu, incl.lo, 31)});
        }
        const ff target = ff_mul(S, uf);
        int found = -1, lastm = -1;
        ff run{0.f, 0.f}, base{0.f, 0.f}, lastbase{0.f, 0.f};
        for (int c0 = 0; c0 < nsl && found < 0; c0 += 32) {
            const ff v = scaled(c0 + lane);
            ff incl = v;
#pragma unroll 1
            for (int o = 1; o < 32; o <<= 1) {
                const ff n = ff_shfl_up(incl, o);
                if (lane >= o)
                    incl = ff_add(n, incl);
            }
            ff excl = ff_shfl_up(incl, 1);
            if (lane == 0)
                excl = {0.f, 0.f};
            const ff full = ff_add(run, incl);
            const unsigned over = __ballot_sync(0xffffffffu, c0 + lane < nsl && ff_gt(full, target));
            const unsigned mass = __ballot_sync(0xffffffffu, c0 + lane < nsl && v.hi > 0.f);
            if (mass) {  // the last slice with mass so far, for u*S past the end
                const int src = 31 - __clz(mass);
                lastm = c0 + src;
                lastbase = ff_add(run, ff{__shfl_sync(0xffffffffu, excl.hi, src),
                                          __shfl_sync(0xffffffffu, excl.lo, src)});
            }
            if (over) {
                const int src = __ffs(over) - 1;
                found = c0 + src;
                base = ff_add(run, ff{__shfl_sync(0xffffffffu, excl.hi, src),
                                      __shfl_sync(0xffffffffu, excl.lo, src)});
            }
            run = ff_add(run, ff{__shfl_sync(0xffffffffu, incl.hi, 31),
                                 __shfl_sync(0xffffffffu, incl.lo, 31)});
        }
        if (lane == 0) {
            const bool past = found < 0;
            const int k = past ? lastm : found;
            s_sl = k;
            s_past = past;
            s_S = S;
            if (k >= 0) {
                const int sh = (int)(M - sl_ref[k]);  // >= 0
                s_shift = sh;
                s_rem = ff_ldexp(ff_add(target, ff{-(past ? lastbase : base).hi,
                                                   -(past ? lastbase : base).lo}),
                                 min(sh, 300));
            }
        }
    }
    __syncthreads();
    const int ks = s_sl;
    if (ks < 0) {  // no mass at all (an all-masked row was caught above)
        if (tid == 0) {
            set_status(p.status, ST_NONFINITE);
            p.out_tokens[r] = -1;
            p.out_conf[r] = __int_as_float(0x7fc00000);
        }
        return;
    }

    // ---- the chosen slice once more, its pieces, then one thread's walk
    const int c0 = ks * p.slice, len = min(p.slice, p.V - c0);
    if (p.tma && tid == 0)
        issue(ks, buf0, &bars[0]);
    land(ks, buf0, &bars[0], ph0);
    d.mct = sl_ref[ks];
    int v0, v1;
    piece_of(len, v0, v1);
    const float ps = piece_sum<T>(d, buf0, nullptr, len, v0, v1);
    piece[tid] = ps;
    ff incl{ps, 0.f};
#pragma unroll 1
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
        wred[warp] = incl;
    __syncthreads();
    ff wbase{0.f, 0.f};
    for (int q = 0; q < warp; ++q)
        wbase = ff_add(wbase, wred[q]);
    const ff lo = ff_add(wbase, excl), hi = ff_add(wbase, incl);
    const ff rem = s_rem;
    const bool past = s_past != 0;
    if (!past && ff_le(lo, rem) && ff_gt(hi, rem))
        atomicMin(&s_hit, tid);
    __syncthreads();
    const int hit = s_hit;
    if (hit != INT_MAX) {
        if (warp == hit >> 5) {  // the hit thread's warp walks its piece
            const float rr = __fadd_rn(__fsub_rn(rem.hi, lo.hi), __fsub_rn(rem.lo, lo.lo));
            const int hl = hit & 31;
            const int k = piece_find_warp<T>(d, buf0, nullptr, len,
                                             __shfl_sync(0xffffffffu, v0, hl),
                                             __shfl_sync(0xffffffffu, v1, hl),
                                             __shfl_sync(0xffffffffu, rr, hl), piece);
            if (lane == 0)
                s_last = k;
        }
    } else {  // past the end after rounding: the last element with mass
        const int lp = piece_find<T>(d, buf0, nullptr, len, v0, v1, INFINITY);
        if (lp >= 0)
            atomicMax(&s_last, lp);
    }
    __syncthreads();
    if (tid == 0) {
        int y = s_last >= 0 ? c0 + s_last : -1;
        float conf = __int_as_float(0x7fc00000);
        if (y < 0) {
            set_status(p.status, ST_NONFINITE);
        } else {
            const float w = ex2_approx(fmaf(Elem<T>::ld_global(row, y), d.c, -d.mct));
            conf = __fdiv_rn(ldexpf(w, -min(s_shift, 300)), __fadd_rn(s_S.hi, s_S.lo));
        }
        if (s_expired || (read_status(p.status) & ST_TIMEOUT)) {  // a copy gave up
            y = -1;
            conf = __int_as_float(0x7fc00000);
        }
        p.out_tokens[r] = y;
        p.out_conf[r] = conf;
    }
}

// T = 0: one warp per padded draft row takes the row's lowest-index maximum.
template <typename T>
__global__ void __launch_bounds__(kFinishThreads) draft_greedy_kernel(const FinishParams p)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t r = (int64_t)blockIdx.x * kFinishWarps + warp;
    const int64_t nrow = (int64_t)p.B * p.Kmax;
    int km = 0;
    if (r < nrow)
        km = __ldg(p.kmax + r / p.Kmax);
    pdl_wait();
    if (r >= nrow)
        return;
    const int j = (int)(r % p.Kmax);
    const bool bad_k = km < 0 || km > p.Kmax;
    int y = -1;
    float conf = 0.f;
    uint32_t err = bad_k ? ST_INVALID : 0u;
    if (!bad_k && j < km) {
        const int gi = merge_argmax_row(p.part, p.g, r);
        if (gi < 0)
            err = ST_NONFINITE;
        else {
            y = gi;
            conf = 1.f;
        }
    }
    if (lane == 0) {
        if (err) {
            set_status(p.status, err);
            conf = __int_as_float(0x7fc00000);
        }
        p.out_tokens[r] = y;
        p.out_conf[r] = conf;
    }
}

}  // namespace sv
