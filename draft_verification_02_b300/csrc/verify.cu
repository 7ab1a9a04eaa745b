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
// Kernels
//   rows_kernel  (one CTA per (row, chunk) of every target row and, at T > 0,
//                every draft row): streams one chunk of <= 32 KB into shared
//                memory with a 1-D TMA bulk copy (cp.async.bulk + mbarrier),
//                reduces it (argmax at T = 0; max and sum of exp at T > 0) and
//                writes a partial.  The CTA that completes a request's last
//                chunk (atomic ticket, no spinning) merges the request's
//                partials in a fixed order and runs the accept test and the
//                first-rejection scan (one warp ballot).  At T = 0 it also
//                emits the tokens; that is the whole greedy call.
//   final_kernel (T > 0; one CTA per (request, chunk)): sums the final-draw
//                weights of its chunk; the request's last CTA picks the chunk
//                holding u * S and runs a block scan inside it to find the
//                token.
// Every merge runs in a fixed order, so repeated calls give identical bits.
#include <cfloat>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace sv {

struct VerifyParams {
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
    int64_t max_rows;
    int64_t draft_rows;  // rows the draft side may index (packed or padded)
    int draft_stride;
    int nchunks, chunk_elems;
    int tma;         // rows start on 16-byte boundaries: use TMA bulk copies
    int chunk_smem;  // bytes reserved per staged chunk (multiple of 128)
    float c_hi, c_lo;  // log2(e) / T as an unevaluated pair of floats
    double inv_T;
    uint32_t *status, *cnt1, *cnt2;
    Partial *part1;
    Handoff *hand;
    double *part2;
};

__device__ __forceinline__ int64_t draft_index(const VerifyParams &p, const int32_t *cu, int i,
                                               int j)
{
    return p.draft_stride > 0 ? (int64_t)i * p.draft_stride + j : (int64_t)cu[i] + j;
}

// exp2 argument for (x - m) / T: d * log2(e)/T with the constant split in two
// floats, so the product carries only the final rounding.
__device__ __forceinline__ float exp_arg(float d, float c_hi, float c_lo)
{
    return fmaf(d, c_hi, d * c_lo);
}

__device__ __forceinline__ bool row_ok(float m, double s)
{
    return isfinite(m) && isfinite(s) && s > 0.0;
}

// Thread 0 only: arm `bar` for `len` elements and start the bulk copy.
template <typename T>
__device__ __forceinline__ void tma_issue(T *dst, const T *src, int len, uint64_t *bar)
{
    const uint32_t bytes = (uint32_t)len * (uint32_t)sizeof(T);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(dst, src, bytes, bar);
}

// Every thread: wait for the copy; on expiry flag a timeout and wait once more
// (bounded) so no copy is left writing into shared memory.
__device__ __forceinline__ void tma_wait(uint64_t *bar, uint32_t phase, uint32_t *status)
{
    if (!mbar_wait_bounded(bar, phase)) {
        set_status(status, ST_TIMEOUT);
        mbar_wait_bounded(bar, phase);
    }
}

template <typename T>
__device__ __forceinline__ void plain_copy(T *dst, const T *src, int len)
{
    for (int k = threadIdx.x; k < len; k += kThreads)
        dst[k] = src[k];
}

// CTA 0 only, when the offsets are malformed: poison every output.
__device__ void poison_all(const VerifyParams &p)
{
    if (threadIdx.x == 0)
        set_status(p.status, ST_INVALID);
    for (int64_t k = threadIdx.x; k < p.max_rows; k += kThreads)
        p.out_tokens[k] = -1;
    for (int k = threadIdx.x; k < p.B; k += kThreads) {
        p.out_len[k] = -1;
        p.hand[k].a = -1;
    }
}

// ---------------------------------------------------------------------------
// per-request stages (run by the CTA that completes the request)
// ---------------------------------------------------------------------------

template <typename T>
__device__ void greedy_stage(const VerifyParams &p, const int32_t *cu_s, int i, int *row_g)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = cu_s[i + 1] - cu_s[i];
    const int64_t t0 = (int64_t)cu_s[i] + i;
    for (int rho = warp; rho <= K; rho += kWarps) {
        const Partial *P = p.part1 + (t0 + rho) * p.nchunks;
        float best = -INFINITY;
        int bidx = INT_MAX;
        int nan = 0;
        for (int c = lane; c < p.nchunks; c += 32) {
            const float m = __ldcg(&P[c].m);
            const int ix = __ldcg(&P[c].idx);
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
        if (lane == 0)
            row_g[rho] = nan ? -2 : (bidx == INT_MAX ? -1 : (best == INFINITY ? -3 : bidx));
    }
    __syncthreads();
    if (warp != 0)
        return;
    const int j = lane;
    const bool act = j < K;
    int x = -1;
    bool bad_tok = false;
    if (act) {
        x = __ldg(p.tokens + draft_index(p, cu_s, i, j));
        bad_tok = x < 0 || x >= p.V;
    }
    bool bad_nf = false;
    for (int jj = lane; jj <= K; jj += 32)
        bad_nf |= row_g[jj] < 0;
    const unsigned nf = __ballot_sync(0xffffffffu, bad_nf);
    const unsigned bt = __ballot_sync(0xffffffffu, bad_tok);
    const unsigned rej = __ballot_sync(0xffffffffu, act && x != row_g[j < K ? j : 0]);
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

template <typename T>
__device__ void sample_stage(const VerifyParams &p, const int32_t *cu_s, int i, float *row_m,
                             double *row_s)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = cu_s[i + 1] - cu_s[i];
    const int64_t t0 = (int64_t)cu_s[i] + i;
    const int nrows = 2 * K + 1;
    // merge the chunk partials of every row: m = max, s = sum s_c * exp((m_c - m) / T)
    for (int rho = warp; rho < nrows; rho += kWarps) {
        const int64_t gslot = rho <= K ? t0 + rho : p.max_rows + cu_s[i] + (rho - K - 1);
        const Partial *P = p.part1 + gslot * p.nchunks;
        float m = -INFINITY;
        for (int c = lane; c < p.nchunks; c += 32)
            m = max_nan(m, __ldcg(&P[c].m));
        m = warp_max_nan(m);
        double s = 0.0;
        for (int c = lane; c < p.nchunks; c += 32) {
            const double sc = __ldcg(&P[c].s);
            if (sc != 0.0)
                s += sc * exp(((double)__ldcg(&P[c].m) - (double)m) * p.inv_T);
        }
        s = warp_sum_d(s);
        if (lane == 0) {
            row_m[rho] = m;
            row_s[rho] = s;
        }
    }
    __syncthreads();
    if (warp != 0)
        return;
    const int j = lane;
    const bool act = j < K;
    int x = -1;
    bool bad_tok = false, bad_nf = false, acc = true;
    if (act) {
        const int64_t di = draft_index(p, cu_s, i, j);
        x = __ldg(p.tokens + di);
        if (x < 0 || x >= p.V) {
            bad_tok = true;
        } else {
            const float mt = row_m[j], md = row_m[K + 1 + j];
            const double st = row_s[j], sd = row_s[K + 1 + j];
            if (!row_ok(mt, st) || !row_ok(md, sd)) {
                bad_nf = true;
            } else {
                const T *trow = reinterpret_cast<const T *>(p.target) + (t0 + j) * p.V;
                const T *drow = reinterpret_cast<const T *>(p.draft) + di * p.V;
                const double gt = Elem<T>::ld_global(trow, x);
                const double gd = Elem<T>::ld_global(drow, x);
                const double pp = exp((gt - (double)mt) * p.inv_T) / st;
                const double qq = exp((gd - (double)md) * p.inv_T) / sd;
                const double ratio = qq > 0.0 ? pp / qq : (pp > 0.0 ? INFINITY : 0.0);
                acc = (double)__ldg(p.u_accept + di) < ratio;
                if (p.out_p)
                    p.out_p[di] = (float)pp;
                if (p.out_q)
                    p.out_q[di] = (float)qq;
            }
        }
    }
    if (lane == 0 && !row_ok(row_m[K], row_s[K]))
        bad_nf = true;
    const unsigned nf = __ballot_sync(0xffffffffu, bad_nf);
    const unsigned bt = __ballot_sync(0xffffffffu, bad_tok);
    const unsigned rej = __ballot_sync(0xffffffffu, act && !acc);
    const bool timeout = read_status(p.status) & ST_TIMEOUT;
    if (nf || bt || timeout) {
        if (lane == 0)
            set_status(p.status, (nf ? ST_NONFINITE : 0u) | (bt ? ST_INVALID : 0u));
        for (int jj = lane; jj <= K; jj += 32)
            p.out_tokens[t0 + jj] = -1;
        if (lane == 0) {
            p.out_len[i] = -1;
            p.hand[i].a = -1;
        }
        return;
    }
    const int a = rej ? __ffs(rej) - 1 : K;
    for (int jj = lane; jj <= K; jj += 32) {
        if (jj < a)
            p.out_tokens[t0 + jj] = x;  // jj == lane here, since a <= 32
        else if (jj > a)
            p.out_tokens[t0 + jj] = -1;
    }
    if (lane == 0) {
        p.out_len[i] = a;
        Handoff h;
        h.a = a;
        h.pad = 0;
        h.trow = t0 + a;
        h.drow = a < K ? draft_index(p, cu_s, i, a) : -1;
        h.m_t = row_m[a];
        h.s_t = row_s[a];
        h.m_d = a < K ? row_m[K + 1 + a] : 0.f;
        h.s_d = a < K ? row_s[K + 1 + a] : 0.0;
        p.hand[i] = h;
    }
}

// ---------------------------------------------------------------------------
// kernel 1: row chunks
// ---------------------------------------------------------------------------

template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kThreads) rows_kernel(const VerifyParams p)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    T *buf = reinterpret_cast<T *>(dsm);
    int32_t *cu_s = reinterpret_cast<int32_t *>(dsm + p.chunk_smem);
    __shared__ __align__(8) uint64_t bar;
    __shared__ float red_f[kWarps];
    __shared__ double red_d[kWarps];
    __shared__ int red_i[kWarps];
    __shared__ int s_last;
    __shared__ float row_m[2 * kMaxDraft + 1];
    __shared__ double row_s[2 * kMaxDraft + 1];
    __shared__ int row_g[kMaxDraft + 1];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.B, V = p.V;
    const int64_t tgt_units = p.max_rows * p.nchunks;
    const int64_t u = blockIdx.x;
    const bool is_draft = !GREEDY && u >= tgt_units;
    const int64_t uu = is_draft ? u - tgt_units : u;
    const int64_t slot = uu / p.nchunks;
    const int c = (int)(uu % p.nchunks);
    const int64_t c0 = (int64_t)c * p.chunk_elems;
    const int len = (int)min((int64_t)p.chunk_elems, (int64_t)V - c0);
    const T *base = reinterpret_cast<const T *>(is_draft ? p.draft : p.target);

    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Target rows and packed draft rows have a known address: start the copy
    // before the offsets arrive.
    bool issued = false;
    if (p.tma && (!is_draft || p.draft_stride == 0)) {
        if (tid == 0)
            tma_issue(buf, base + slot * V + c0, len, &bar);
        issued = true;
    }
    for (int k = tid; k <= B; k += kThreads)
        cu_s[k] = __ldg(p.cu + k);
    __syncthreads();
    int bad = 0;
    for (int k = tid; k < B; k += kThreads) {
        const int K = cu_s[k + 1] - cu_s[k];
        if (K < 0 || K > kMaxDraft || (p.draft_stride > 0 && K > p.draft_stride))
            bad = 1;
    }
    if (tid == 0 && (cu_s[0] != 0 || (int64_t)cu_s[B] + B > p.max_rows))
        bad = 1;
    bad = __syncthreads_or(bad);
    if (bad) {
        if (blockIdx.x == 0)
            poison_all(p);
        if (issued)
            tma_wait(&bar, 0, p.status);
        return;
    }
    const int nd = cu_s[B];
    int i, j;
    bool active;
    if (!is_draft) {  // target slot: request i owns rows [cu[i] + i, cu[i+1] + i + 1)
        active = slot < (int64_t)nd + B;
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)cu_s[mid] + mid <= slot)
                lo = mid;
            else
                hi = mid - 1;
        }
        i = lo;
        j = (int)(slot - cu_s[i] - i);
    } else {  // packed draft slot: request i owns [cu[i], cu[i+1])
        active = slot < nd;
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cu_s[mid] <= slot)
                lo = mid;
            else
                hi = mid - 1;
        }
        i = lo;
        j = (int)(slot - cu_s[i]);
    }
    if (!active) {
        if (issued)
            tma_wait(&bar, 0, p.status);
        return;
    }
    const int64_t row = (is_draft && p.draft_stride > 0) ? (int64_t)i * p.draft_stride + j : slot;
    if (p.tma) {
        if (!issued && tid == 0)
            tma_issue(buf, base + row * V + c0, len, &bar);
        tma_wait(&bar, 0, p.status);
    } else {
        plain_copy(buf, base + row * V + c0, len);
        __syncthreads();
    }

    constexpr int VE = Elem<T>::kPerVec;
    const uint4 *vb = reinterpret_cast<const uint4 *>(buf);
    const int nvec = len / VE;
    Partial part;
    if (GREEDY) {
        float best = -INFINITY;
        int bidx = INT_MAX;
        int nan = 0;
        for (int v = tid; v < nvec; v += kThreads) {
            float f[VE];
            Elem<T>::unpack(vb[v], f);
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                nan |= f[e] != f[e];
                if (f[e] > best) {
                    best = f[e];
                    bidx = v * VE + e;
                }
            }
        }
        for (int k = nvec * VE + tid; k < len; k += kThreads) {
            const float x = Elem<T>::at(buf, k);
            nan |= x != x;
            if (x > best) {
                best = x;
                bidx = k;
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
        if (lane == 0) {
            red_f[warp] = best;
            red_i[warp] = bidx;
        }
        nan = __syncthreads_or(nan);
        if (tid == 0) {
            for (int w = 1; w < kWarps; ++w)
                if (red_f[w] > best || (red_f[w] == best && red_i[w] < bidx)) {
                    best = red_f[w];
                    bidx = red_i[w];
                }
            part.m = best;
            part.idx = nan ? -2 : (bidx == INT_MAX ? -1 : (int)(c0 + bidx));
            part.s = 0.0;
        }
    } else {
        float mx = -INFINITY;
        for (int v = tid; v < nvec; v += kThreads) {
            float f[VE];
            Elem<T>::unpack(vb[v], f);
#pragma unroll
            for (int e = 0; e < VE; ++e)
                mx = max_nan(mx, f[e]);
        }
        for (int k = nvec * VE + tid; k < len; k += kThreads)
            mx = max_nan(mx, Elem<T>::at(buf, k));
        const float m = block_max_nan(mx, red_f);
        double s;
        if (m != m) {
            s = __longlong_as_double(0x7ff8000000000000ll);
        } else if (m == -INFINITY) {
            s = 0.0;  // every entry of the chunk is masked
        } else {
            const float ch = p.c_hi, cl = p.c_lo;
            float acc = 0.f;
            for (int v = tid; v < nvec; v += kThreads) {
                float f[VE];
                Elem<T>::unpack(vb[v], f);
                float e[VE];
#pragma unroll
                for (int k = 0; k < VE; ++k)
                    e[k] = exp2f(exp_arg(f[k] - m, ch, cl));
#pragma unroll
                for (int w = 1; w < VE; w <<= 1)
#pragma unroll
                    for (int k = 0; k < VE; k += 2 * w)
                        e[k] += e[k + w];
                acc += e[0];
            }
            for (int k = nvec * VE + tid; k < len; k += kThreads)
                acc += exp2f(exp_arg(Elem<T>::at(buf, k) - m, ch, cl));
            s = block_sum_d((double)acc, red_d);
        }
        part.m = m;
        part.idx = 0;
        part.s = s;
    }
    if (tid == 0) {
        const int64_t gslot = is_draft ? p.max_rows + slot : slot;
        p.part1[gslot * p.nchunks + c] = part;
        __threadfence();
        const int K = cu_s[i + 1] - cu_s[i];
        const uint32_t need = (uint32_t)((GREEDY ? K + 1 : 2 * K + 1) * p.nchunks);
        const uint32_t old = atomicAdd(p.cnt1 + i, 1u);
        s_last = old == need - 1;
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    if (tid == 0)
        p.cnt1[i] = 0;  // ready for the next call
    if (GREEDY)
        greedy_stage<T>(p, cu_s, i, row_g);
    else
        sample_stage<T>(p, cu_s, i, row_m, row_s);
}

// ---------------------------------------------------------------------------
// kernel 2: final draw (T > 0)
// ---------------------------------------------------------------------------

struct DrawCtx {
    const void *trow;
    const void *drow;
    bool resid;
    float m_t, m_d, inv_st, inv_sd;
    float c_hi, c_lo;
};

template <typename T>
__device__ __forceinline__ float draw_weight(const DrawCtx &d, const T *tb, const T *db, int k)
{
    const float pt = exp2f(exp_arg(Elem<T>::at(tb, k) - d.m_t, d.c_hi, d.c_lo));
    if (!d.resid)
        return pt;  // bonus draw (unnormalised p)
    const float pd = exp2f(exp_arg(Elem<T>::at(db, k) - d.m_d, d.c_hi, d.c_lo));
    return fmaxf(pt * d.inv_st - pd * d.inv_sd, 0.f);
}

// Stage chunk c of the draw rows into shared memory (all threads).
template <typename T>
__device__ __forceinline__ int stage_draw_chunk(const VerifyParams &p, const DrawCtx &d, int c,
                                                T *tb, T *db, uint64_t *bar, uint32_t &phase)
{
    const int64_t c0 = (int64_t)c * p.chunk_elems;
    const int len = (int)min((int64_t)p.chunk_elems, (int64_t)p.V - c0);
    const T *ts = reinterpret_cast<const T *>(d.trow) + c0;
    const T *dsrc = d.resid ? reinterpret_cast<const T *>(d.drow) + c0 : nullptr;
    __syncthreads();  // previous users of the buffers are done
    if (p.tma) {
        if (threadIdx.x == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint32_t bytes = (uint32_t)len * (uint32_t)sizeof(T);
            mbar_arrive_expect_tx(bar, d.resid ? 2 * bytes : bytes);
            bulk_g2s(tb, ts, bytes, bar);
            if (d.resid)
                bulk_g2s(db, dsrc, bytes, bar);
        }
        tma_wait(bar, phase, p.status);
        phase ^= 1u;
    } else {
        plain_copy(tb, ts, len);
        if (d.resid)
            plain_copy(db, dsrc, len);
        __syncthreads();
    }
    return len;
}

// Sum of w over this thread's contiguous run of the staged chunk (fp32, in
// index order).  Runs: thread t owns [t*run, min(len, (t+1)*run)).
template <typename T>
__device__ __forceinline__ float run_sum(const DrawCtx &d, const T *tb, const T *db, int len,
                                         int &k0, int &k1)
{
    const int run = (len + kThreads - 1) / kThreads;
    k0 = min(len, (int)threadIdx.x * run);
    k1 = min(len, k0 + run);
    float acc = 0.f;
    for (int k = k0; k < k1; ++k)
        acc += draw_weight<T>(d, tb, db, k);
    return acc;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) final_kernel(const VerifyParams p)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    T *tb = reinterpret_cast<T *>(dsm);
    T *db = reinterpret_cast<T *>(dsm + p.chunk_smem);
    __shared__ __align__(8) uint64_t bar;
    __shared__ double red_d[kWarps];
    __shared__ double s_tot[kMaxChunks];
    __shared__ int s_last, s_chunk, s_claim, s_y, s_mode;
    __shared__ double s_base, s_target;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i = blockIdx.x / p.nchunks, c = blockIdx.x % p.nchunks;
    const Handoff *hp = p.hand + i;
    const int a = __ldcg(&hp->a);
    if (a < 0)
        return;  // poisoned request: nothing to draw
    DrawCtx d;
    const int64_t trow = __ldcg(reinterpret_cast<const long long *>(&hp->trow));
    const int64_t drow = __ldcg(reinterpret_cast<const long long *>(&hp->drow));
    d.resid = drow >= 0;
    if (trow < 0 || trow >= p.max_rows || drow >= p.draft_rows) {  // never from a valid handoff
        if (tid == 0)
            set_status(p.status, ST_INVALID);
        return;
    }
    d.trow = reinterpret_cast<const T *>(p.target) + trow * p.V;
    d.drow = d.resid ? reinterpret_cast<const T *>(p.draft) + drow * p.V : nullptr;
    d.m_t = __ldcg(&hp->m_t);
    d.m_d = __ldcg(&hp->m_d);
    d.inv_st = (float)(1.0 / __ldcg(&hp->s_t));
    d.inv_sd = d.resid ? (float)(1.0 / __ldcg(&hp->s_d)) : 0.f;
    d.c_hi = p.c_hi;
    d.c_lo = p.c_lo;

    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    uint32_t phase = 0;
    int k0, k1;
    int len = stage_draw_chunk<T>(p, d, c, tb, db, &bar, phase);
    float acc = run_sum<T>(d, tb, db, len, k0, k1);
    double tot = block_sum_d((double)acc, red_d);
    if (tid == 0) {
        p.part2[(int64_t)i * p.nchunks + c] = tot;
        __threadfence();
        const uint32_t old = atomicAdd(p.cnt2 + i, 1u);
        s_last = old == (uint32_t)p.nchunks - 1;
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    if (tid == 0) {
        p.cnt2[i] = 0;
        for (int cc = 0; cc < p.nchunks; ++cc)
            s_tot[cc] = __ldcg(p.part2 + (int64_t)i * p.nchunks + cc);
        double S = 0.0;
        for (int cc = 0; cc < p.nchunks; ++cc)
            S += s_tot[cc];
        s_mode = (d.resid && !(S > 0.0)) ? 1 : 0;  // all-zero residual: draw from p_a
    }
    __syncthreads();
    if (s_mode == 1) {
        d.resid = false;
        for (int cc = 0; cc < p.nchunks; ++cc) {
            len = stage_draw_chunk<T>(p, d, cc, tb, db, &bar, phase);
            acc = run_sum<T>(d, tb, db, len, k0, k1);
            tot = block_sum_d((double)acc, red_d);
            if (tid == 0)
                s_tot[cc] = tot;
        }
        __syncthreads();
    }
    if (tid == 0) {
        double S = 0.0;
        for (int cc = 0; cc < p.nchunks; ++cc)
            S += s_tot[cc];
        const double target = (double)__ldg(p.u_final + i) * S;
        double cum = 0.0;
        int cs = -1;
        double base = 0.0;
        for (int cc = 0; cc < p.nchunks; ++cc) {
            if (cum + s_tot[cc] > target) {
                cs = cc;
                base = cum;
                break;
            }
            cum += s_tot[cc];
        }
        int last_pos = 0;
        if (cs < 0) {  // rounding left u*S at or past the end: last chunk with mass
            cs = 0;
            double cum2 = 0.0;
            for (int cc = 0; cc < p.nchunks; ++cc) {
                if (s_tot[cc] > 0.0) {
                    cs = cc;
                    base = cum2;
                }
                cum2 += s_tot[cc];
            }
            last_pos = 1;
        }
        s_chunk = cs;
        s_base = base;
        s_target = last_pos ? INFINITY : target;
        s_claim = INT_MAX;
        s_y = -1;
    }
    __syncthreads();
    const int cs = s_chunk;
    len = stage_draw_chunk<T>(p, d, cs, tb, db, &bar, phase);
    acc = run_sum<T>(d, tb, db, len, k0, k1);
    // exclusive scan of the run sums (fp64, fixed order)
    const double run_d = (double)acc;
    double incl = run_d;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += n;
    }
    const double prev = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 31)
        red_d[warp] = incl;
    __syncthreads();
    double woff = 0.0;
    for (int w = 0; w < warp; ++w)
        woff += red_d[w];
    const double lo = s_base + (woff + (lane ? prev : 0.0));
    const double target = s_target;
    if (k1 > k0 && lo + (double)acc > target)
        atomicMin(&s_claim, tid);
    __syncthreads();
    const int64_t cbase = (int64_t)cs * p.chunk_elems;
    if (s_claim == tid) {
        float run = 0.f;
        int y = -1;
        for (int k = k0; k < k1; ++k) {
            run += draw_weight<T>(d, tb, db, k);
            if (lo + (double)run > target) {
                y = k;
                break;
            }
        }
        s_y = (int)(cbase + y);
    }
    __syncthreads();
    if (s_claim == INT_MAX) {
        // u*S at or past the chunk's end after rounding: last entry with w > 0
        if (tid == 0)
            s_claim = -1;
        __syncthreads();
        int best = -1;
        for (int k = k0; k < k1; ++k)
            if (draw_weight<T>(d, tb, db, k) > 0.f)
                best = k;
        if (best >= 0)
            atomicMax(&s_claim, best);
        __syncthreads();
        if (tid == 0)
            s_y = s_claim >= 0 ? (int)(cbase + s_claim) : -1;
        __syncthreads();
    }
    if (tid == 0) {
        if (s_y < 0)
            set_status(p.status, ST_NONFINITE);
        p.out_tokens[trow] = s_y;
    }
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------

template <typename T, bool GREEDY>
static cudaError_t prepare_rows_kernel()
{
    static cudaError_t once = [] {
        cudaError_t e = cudaFuncSetAttribute(rows_kernel<T, GREEDY>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kChunkBytes + 128 + 4 * (kMaxBatch + 1));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(rows_kernel<T, GREEDY>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        return e;
    }();
    return once;
}

template <typename T>
static cudaError_t prepare_final_kernel()
{
    static cudaError_t once = [] {
        cudaError_t e = cudaFuncSetAttribute(final_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             2 * (kChunkBytes + 128));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(final_kernel<T>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        return e;
    }();
    return once;
}

template <typename T>
static cudaError_t launch_typed(const VerifyArgs &a, cudaStream_t s, Tracer &tr)
{
    const bool greedy = a.temperature == 0.0;
    const Chunking ch = chunking(a.V, (int)sizeof(T));
    const WsLayout L = ws_layout(a.B, a.max_rows, a.V);
    unsigned char *ws = static_cast<unsigned char *>(a.ws);
    VerifyParams p{};
    p.target = a.target;
    p.draft = a.draft;
    p.tokens = a.tokens;
    p.cu = a.cu;
    p.u_accept = a.u_accept;
    p.u_final = a.u_final;
    p.out_tokens = a.out_tokens;
    p.out_len = a.out_len;
    p.out_p = a.out_p;
    p.out_q = a.out_q;
    p.B = a.B;
    p.V = a.V;
    p.max_rows = a.max_rows;
    p.draft_rows = a.draft_stride > 0 ? (int64_t)a.B * a.draft_stride : a.max_rows - a.B;
    p.draft_stride = a.draft_stride;
    p.nchunks = ch.nchunks;
    p.chunk_elems = ch.chunk_elems;
    const bool row16 = ((int64_t)a.V * (int64_t)sizeof(T)) % 16 == 0;
    const bool t16 = reinterpret_cast<uintptr_t>(a.target) % 16 == 0;
    const bool d16 = greedy || reinterpret_cast<uintptr_t>(a.draft) % 16 == 0;
    p.tma = row16 && t16 && d16;
    p.chunk_smem = (int)align_up((size_t)ch.chunk_elems * sizeof(T), 128);
    if (!greedy) {
        const double c = 1.4426950408889634074 / a.temperature;  // log2(e) / T
        p.c_hi = (float)c;
        p.c_lo = (float)(c - (double)p.c_hi);
        p.inv_T = 1.0 / a.temperature;
    }
    p.status = reinterpret_cast<uint32_t *>(ws + L.status);
    p.cnt1 = reinterpret_cast<uint32_t *>(ws + L.cnt1);
    p.cnt2 = reinterpret_cast<uint32_t *>(ws + L.cnt2);
    p.part1 = reinterpret_cast<Partial *>(ws + L.part1);
    p.hand = reinterpret_cast<Handoff *>(ws + L.hand);
    p.part2 = reinterpret_cast<double *>(ws + L.part2);

    cudaError_t e = greedy ? prepare_rows_kernel<T, true>() : prepare_rows_kernel<T, false>();
    if (e != cudaSuccess)
        return e;
    if (!greedy && (e = prepare_final_kernel<T>()) != cudaSuccess)
        return e;
    const int64_t units = (a.max_rows + (greedy ? 0 : a.max_rows - a.B)) * ch.nchunks;
    const size_t smem1 = (size_t)p.chunk_smem + 4 * (size_t)(a.B + 1);
    tr.begin(s);
    if (greedy)
        rows_kernel<T, true><<<(unsigned)units, kThreads, smem1, s>>>(p);
    else
        rows_kernel<T, false><<<(unsigned)units, kThreads, smem1, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    tr.after_kernel(s);
    if (!greedy) {
        final_kernel<T><<<(unsigned)(a.B * ch.nchunks), kThreads, 2 * (size_t)p.chunk_smem, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
        tr.after_kernel(s);
    }
    return cudaSuccess;
}

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, Tracer &tr)
{
    return a.dtype == 0 ? launch_typed<float>(a, s, tr) : launch_typed<uint16_t>(a, s, tr);
}

}  // namespace sv
