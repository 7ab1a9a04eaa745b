// shard.cu - vocabulary-sharded verification: each shard of a tensor-parallel
// target holds the logits of one contiguous vocabulary range, reduces its own
// columns, and only per-row records and per-request masses cross shards.
//
// The split is the target's tensor-parallel output projection ("Tencent
// Hunyuan Turns Speculative Decoding Into a Full Open-Source Stack", "Key
// numbers (Hy3-295B-A21B, TP=8)").  What is computed is the verification of
// verify.cu over the whole vocabulary:
//  - rows: the softmax is shift invariant, so a row's (m, s) over the whole
//    vocabulary is the merge of the shards' (m_r, s_r): m = max m_r and
//    s = sum_r s_r 2^((m_r - m) c).  At T = 0 the lowest index of the row
//    maximum is the shard-order merge of each shard's lowest argmax.
//  - accept: p(x) and q(x) from the merged rows and the logit at x of the
//    shard that holds x; the accept test and first rejection of verify.cu.
//  - final draw: the inverse CDF of the final weights over the whole
//    vocabulary walks the shards' ranges in order, so with S the sum of the
//    shards' masses, the shard whose running-sum range holds u*S draws from
//    its own columns, starting from the running sum before it.
// Kernels (each one CTA per request except the streaming pass):
//  - the streaming pass of verify.cu over the shard's columns, then
//    shard_rows_kernel: a warp per row merges the row's partials into one
//    16-byte record (and reads the logit at the row's drafted token when the
//    shard holds it).
//  - shard_accept_kernel: a warp per row merges the N shards' records (lane
//    r holds shard r's; the merge is commutative bit for bit, so a butterfly
//    leaves the same bits in every lane and on every shard), then warp 0 runs
//    the accept test and the first-rejection ballot and keeps the final
//    draw's constants in the workspace.
//  - shard_mass_kernel: weighs the final rows' columns of this shard in
//    staged slices (1-D TMA bulk copies) and keeps each slice's total.
//  - shard_draw_kernel: the shard-order scan of the gathered masses picks
//    the drawing shard (identical on every shard); that shard finds the
//    slice, the thread piece and the element as the cluster draw of
//    verify.cu does inside its range.
#include <algorithm>
#include <cstdint>

#include "finish_kernel.cuh"

namespace sv {

namespace {

struct __align__(16) ShardRow {  // the layout of spec_shard_row
    float m;
    int32_t x;  // T > 0: the bits of the logit at the drafted token; T = 0: global argmax
    float s_hi, s_lo;
};

struct __align__(16) ShardMass {  // the layout of spec_shard_mass
    ff w, p;
};

enum : int32_t { kSkip = 1, kResid = 2 };

// One request's final draw, written by the accept step, read by the mass and
// draw steps.
struct __align__(16) DrawState {
    int32_t flags;  // kSkip: no draw (a poisoned request); kResid: w = max(0, p - q)
    int32_t a;      // accepted drafts
    int64_t trow;   // target row of the final position (its out_tokens index too)
    int64_t drow;   // draft row of the residual draw, -1 for the bonus draw
    float c, mct, mcd, sc_t, sc_d;  // the DrawCtx constants
    int32_t pad;
};

struct ShardLayout {
    WsLayout base;  // status word, offsets flag, partials of the streaming pass
    size_t state, slices, total;
};

ShardLayout shard_layout(int B, int64_t max_rows)
{
    ShardLayout L{};
    L.base = ws_layout(B, max_rows, 0);
    L.state = L.base.total;
    L.slices = align_up(L.state + (size_t)B * sizeof(DrawState), 256);
    L.total = align_up(L.slices + (size_t)B * kMaxSlices * 2 * sizeof(ff), 256);
    return L;
}

__device__ __forceinline__ bool shard_shape_ok(int64_t max_rows, int64_t draft_rows, int stride,
                                               int i, int cu_i, int K)
{
    const int64_t t0 = (int64_t)cu_i + i;
    return cu_i >= 0 && K >= 0 && K <= kMaxDraft && t0 + K < max_rows &&
           (stride > 0 ? K <= stride : (int64_t)cu_i + K <= draft_rows);
}

__device__ __forceinline__ ShardRow load_row(const ShardRow *r)
{
    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(r));
    return {__uint_as_float(v.x), (int32_t)v.y, __uint_as_float(v.z), __uint_as_float(v.w)};
}

__device__ __forceinline__ ShardMass load_mass(const ShardMass *m)
{
    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(m));
    return {{__uint_as_float(v.x), __uint_as_float(v.y)},
            {__uint_as_float(v.z), __uint_as_float(v.w)}};
}

// ---------------------------------------------------------------------------
// step 1: row records
// ---------------------------------------------------------------------------

struct ShardRowsParams {
    const void *target, *draft;  // the shard's rows, Vs columns each
    const int32_t *tokens, *cu;
    int B, Vs, v_begin;
    int64_t max_rows, draft_rows, n_rec;
    int draft_stride;
    Geometry g;  // the streaming pass's unit split
    float c;
    uint32_t *status;
    const uint32_t *cu_flag;
    const Partial *part;
    int64_t part_cap;
    ShardRow *out;
};

template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kFinishThreads) shard_rows_kernel(const ShardRowsParams p)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i = blockIdx.x;
    const int cu_i = __ldg(p.cu + i);
    const int K = __ldg(p.cu + i + 1) - cu_i;
    const int cu_tot = __ldg(p.cu + p.B);
    const bool shape = shard_shape_ok(p.max_rows, p.draft_rows, p.draft_stride, i, cu_i, K);
    const T *tbase = reinterpret_cast<const T *>(p.target);
    const T *dbase = reinterpret_cast<const T *>(p.draft);

    pdl_wait();  // the streaming pass has completed and its writes are visible
    if (__ldcg(p.cu_flag) == 0u || !shape)
        return;  // malformed offsets: flagged by the streaming pass, poisoned by step 2
    const Geometry g = real_split(p.g, p.B, cu_tot);  // the streaming pass's split
    const int64_t t0 = (int64_t)cu_i + i;
    const int nrows = GREEDY ? K + 1 : 2 * K + 1;  // target rows 0..K, then draft rows
    for (int k = warp; k < nrows; k += kFinishWarps) {
        const bool tgt = k <= K;
        const int j = tgt ? k : k - K - 1;
        const int64_t rg = tgt ? t0 + k : g.nt + cu_i + j;  // row of the streaming pass
        const int64_t dj = k == K ? -1 : draft_index(p.draft_stride, p.cu, i, j);
        const int64_t rec = tgt ? t0 + k : p.max_rows + dj;
        int wf, wl;
        row_span(g, rg, wf, wl);
        ShardRow r{__int_as_float(0x7fc00000), -2, __int_as_float(0x7fc00000), 0.f};
        if (SV_IN_BOUNDS(rg + wl, p.part_cap, p.status)) {
            if (GREEDY) {
                float best;
                int bidx;
                bool nan;
                merge_argmax_pair(p.part, g, rg, best, bidx, nan);
                r = {best, nan ? -2 : (bidx == INT_MAX ? -1 : p.v_begin + bidx), 0.f, 0.f};
            } else {
                float m = -INFINITY;
                ff s{0.f, 0.f};
                for (int w = wf + lane; w <= wl; w += 32) {
                    const Partial pt = load_partial(p.part + rg + w);
                    lse_combine(m, s, pt.m, {pt.s_hi, pt.s_lo}, p.c);
                }
#pragma unroll 1
                for (int o = 16; o > 0; o >>= 1) {
                    const float mo = __shfl_xor_sync(0xffffffffu, m, o);
                    const ff so = ff_shfl_xor(s, o);
                    lse_combine(m, s, mo, so, p.c);
                }
                float gx = 0.f;
                if (dj >= 0 && lane == 0) {
                    const int x = SV_IN_BOUNDS(dj, p.draft_rows, p.status) ? __ldg(p.tokens + dj) : -1;
                    if (x >= p.v_begin && x - p.v_begin < p.Vs)
                        gx = tgt ? Elem<T>::ld_global(tbase + (t0 + j) * (int64_t)p.Vs, x - p.v_begin)
                                 : Elem<T>::ld_global(dbase + dj * (int64_t)p.Vs, x - p.v_begin);
                }
                r = {m, __float_as_int(gx), s.hi, s.lo};
            }
        }
        if (lane == 0 && SV_IN_BOUNDS(rec, p.n_rec, p.status))
            p.out[rec] = r;
    }
}

// ---------------------------------------------------------------------------
// step 2: merge, accept test, first rejection
// ---------------------------------------------------------------------------

struct ShardAcceptParams {
    const ShardRow *rows;  // [n_shards][n_rec]
    int n_shards;
    int32_t begin[kMaxShards + 1];
    const int32_t *tokens, *cu;
    const float *u_accept;
    int B, V;  // V = begin[n_shards]
    int64_t max_rows, draft_rows, n_rec;
    int draft_stride;
    float c;
    int32_t *out_tokens, *out_len;
    float *out_p, *out_q;
    uint32_t *status;
    const uint32_t *cu_flag;
    DrawState *state;
};

template <bool GREEDY>
__global__ void __launch_bounds__(kFinishThreads) shard_accept_kernel(const ShardAcceptParams p)
{
    __shared__ float row_m[2 * kMaxDraft + 1];
    __shared__ __align__(8) ff row_s[2 * kMaxDraft + 1];
    __shared__ float row_p[2 * kMaxDraft + 1];  // p_j(x_j), q_j(x_j)
    __shared__ int row_g[kMaxDraft + 1];        // T = 0: merged argmax (or < 0: error code)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i = blockIdx.x;
    DrawState skip{};
    skip.flags = kSkip;
    skip.drow = -1;
    if (__ldcg(p.cu_flag) == 0u) {
        // this shard's row pass found the offsets malformed (so did every
        // shard's: they all read the same offsets): poison every output
        for (int64_t k = (int64_t)i * kFinishThreads + tid; k < p.max_rows;
             k += (int64_t)gridDim.x * kFinishThreads)
            p.out_tokens[k] = -1;
        if (tid == 0) {
            p.out_len[i] = -1;
            if (!GREEDY)
                p.state[i] = skip;
        }
        return;
    }
    const int cu_i = __ldg(p.cu + i);
    const int K = __ldg(p.cu + i + 1) - cu_i;
    if (!shard_shape_ok(p.max_rows, p.draft_rows, p.draft_stride, i, cu_i, K)) {
        if (tid == 0 && !GREEDY)  // (not reached after a clean validation)
            p.state[i] = skip;
        return;
    }
    const int64_t t0 = (int64_t)cu_i + i;
    const int N = p.n_shards;
    const int nrows = GREEDY ? K + 1 : 2 * K + 1;
    for (int k = warp; k < nrows; k += kFinishWarps) {
        const bool tgt = k <= K;
        const int j = tgt ? k : k - K - 1;
        const int64_t dj = k == K ? -1 : draft_index(p.draft_stride, p.cu, i, j);
        const int64_t rec = tgt ? t0 + k : p.max_rows + dj;
        ShardRow r{-INFINITY, -1, 0.f, 0.f};
        if (lane < N && SV_IN_BOUNDS(rec, p.n_rec, p.status))
            r = load_row(p.rows + (int64_t)lane * p.n_rec + rec);
        if (GREEDY) {
            float best = -INFINITY;
            int bidx = INT_MAX, nan = 0;
            if (lane < N) {
                if (r.x == -2)
                    nan = 1;
                else if (r.x >= 0) {
                    best = r.m;
                    bidx = r.x;
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
                row_g[k] = nan ? -2 : (bidx == INT_MAX ? -1 : (best == INFINITY ? -3 : bidx));
        } else {
            float m = r.m;
            ff s{r.s_hi, r.s_lo};
#pragma unroll 1
            for (int o = 16; o > 0; o >>= 1) {
                const float mo = __shfl_xor_sync(0xffffffffu, m, o);
                const ff so = ff_shfl_xor(s, o);
                lse_combine(m, s, mo, so, p.c);
            }
            const int x = dj >= 0 && SV_IN_BOUNDS(dj, p.draft_rows, p.status) ? __ldg(p.tokens + dj)
                                                                              : -1;
            int owner = -1;
            for (int q = 0; q < N; ++q)
                if (x >= p.begin[q] && x < p.begin[q + 1])
                    owner = q;
            const float gx = __shfl_sync(0xffffffffu, __int_as_float(r.x), owner < 0 ? 0 : owner);
            const float px = owner >= 0 && row_ok(m, s) ? softmax_at(gx, m, s, p.c) : 0.f;
            if (lane == 0) {
                row_m[k] = m;
                row_s[k] = s;
                row_p[k] = px;
            }
        }
    }
    __syncthreads();
    if (warp != 0)
        return;

    const bool act = lane < K;
    int64_t di = 0;
    int x = -1;
    float u = 0.f;
    if (act) {
        di = draft_index(p.draft_stride, p.cu, i, lane);
        if (SV_IN_BOUNDS(di, p.draft_rows, p.status)) {
            x = __ldg(p.tokens + di);
            if (!GREEDY)
                u = __ldg(p.u_accept + di);
        }
    }
    const bool timeout = read_status(p.status) & ST_TIMEOUT;
    const bool bad_tok = act && (x < 0 || x >= p.V);
    bool bad_nf = false, acc = true;
    float pp = 0.f, qq = 0.f;
    if (GREEDY) {
        for (int jj = lane; jj <= K; jj += 32)
            bad_nf |= row_g[jj] < 0;
        acc = !act || x == row_g[act ? lane : 0];
    } else {
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
    }
    const unsigned nf = __ballot_sync(0xffffffffu, bad_nf);
    const unsigned bt = __ballot_sync(0xffffffffu, bad_tok);
    const unsigned rej = __ballot_sync(0xffffffffu, act && !acc);
    const int a = rej ? __ffs(rej) - 1 : K;
    if (nf || bt || timeout) {
        if (lane == 0)
            set_status(p.status, (nf ? ST_NONFINITE : 0u) | (bt ? ST_INVALID : 0u));
        for (int jj = lane; jj <= K; jj += 32)
            if (SV_IN_BOUNDS(t0 + jj, p.max_rows, p.status))
                p.out_tokens[t0 + jj] = -1;
        if (lane == 0) {
            if (SV_IN_BOUNDS(i, p.B, p.status))
                p.out_len[i] = -1;
            if (!GREEDY)
                p.state[i] = skip;
        }
        return;
    }
    if (!GREEDY && act && SV_IN_BOUNDS(di, p.draft_rows, p.status)) {
        if (p.out_p)
            p.out_p[di] = pp;
        if (p.out_q)
            p.out_q[di] = qq;
    }
    for (int jj = lane; jj <= K; jj += 32) {
        if (!SV_IN_BOUNDS(t0 + jj, p.max_rows, p.status))
            continue;
        // jj == lane where jj < a (a <= 32); the final token at T > 0 comes
        // from step 4 (-1 until then)
        p.out_tokens[t0 + jj] = jj < a ? x : (jj == a && GREEDY ? row_g[a] : -1);
    }
    if (lane == 0 && SV_IN_BOUNDS(i, p.B, p.status))
        p.out_len[i] = a;
    if (!GREEDY && lane == 0) {
        DrawState st{};
        st.flags = a < K ? kResid : 0;
        st.a = a;
        st.trow = t0 + a;
        st.drow = a < K ? draft_index(p.draft_stride, p.cu, i, a) : -1;
        st.c = p.c;
        const float mt = row_m[a];
        st.mct = mt * p.c;
        st.sc_t = ff_recip_scaled(mc_correction(mt, st.mct, p.c), row_s[a]);
        if (a < K) {
            const float md = row_m[K + 1 + a];
            st.mcd = md * p.c;
            st.sc_d = ff_recip_scaled(mc_correction(md, st.mcd, p.c), row_s[K + 1 + a]);
        }
        p.state[i] = st;
    }
}

// ---------------------------------------------------------------------------
// steps 3 and 4: the final draw's mass and the draw
// ---------------------------------------------------------------------------

struct ShardDrawParams {
    FinishParams fp;  // target, draft (the shard's rows), V = Vs, slice geometry, tma, status
    const DrawState *state;
    ff *slices;  // [B][kMaxSlices][2]: slice totals of w, then of p
    int v_begin;
    int64_t max_rows, draft_rows;
    ShardMass *out_mass;        // step 3
    const ShardMass *mass_all;  // step 4: [n_shards][B]
    int n_shards, shard;
    const float *u_final;
    int32_t *out_tokens;
};

__device__ __forceinline__ DrawCtx draw_ctx(const DrawState &st)
{
    DrawCtx d;
    d.resid = (st.flags & kResid) != 0;
    d.c = st.c;
    d.mct = st.mct;
    d.mcd = st.mcd;
    d.sc_t = st.sc_t;
    d.sc_d = st.sc_d;
    return d;
}

__device__ __forceinline__ bool state_rows_ok(const ShardDrawParams &q, const DrawState &st)
{
    return !(st.flags & kSkip) && SV_IN_BOUNDS(st.trow, q.max_rows, q.fp.status) &&
           (st.drow < 0 || SV_IN_BOUNDS(st.drow, q.draft_rows, q.fp.status));
}

template <typename T>
__global__ void __launch_bounds__(kSampleThreads) shard_mass_kernel(const ShardDrawParams q)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    const FinishParams &p = q.fp;
    T *tb = reinterpret_cast<T *>(dsm);
    T *db = reinterpret_cast<T *>(dsm + p.stage_smem);
    __shared__ __align__(8) uint64_t bar;
    __shared__ float piece[kSampleThreads];
    __shared__ ff wred[kSampleWarps];
    __shared__ int s_expired;
    const int tid = threadIdx.x, i = blockIdx.x;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        s_expired = 0;
    }
    __syncthreads();
    const DrawState st = q.state[i];
    ShardMass out{{0.f, 0.f}, {0.f, 0.f}};
    if (state_rows_ok(q, st)) {
        const DrawCtx d = draw_ctx(st);
        DrawCtx dp = d;
        dp.resid = false;
        const T *trow = reinterpret_cast<const T *>(p.target) + st.trow * (int64_t)p.V;
        const T *drow = d.resid ? reinterpret_cast<const T *>(p.draft) + st.drow * (int64_t)p.V
                                : nullptr;
        ff *tot = q.slices + (size_t)i * kMaxSlices * 2;
        uint32_t phase = 0;
        const int nsl = (p.V + p.slice - 1) / p.slice;
        for (int sl = 0; sl < nsl; ++sl) {
            const int c0 = sl * p.slice, len = min(p.slice, p.V - c0);
            const ff ws = weigh_slice<T>(p, d, trow, drow, c0, len, tb, db, &bar, &phase, piece,
                                         wred, &s_expired, true);
            out.w = ff_add(out.w, ws);
            // the p weights of the same staged slice (the fallback of an
            // all-zero residual); the w weights already are p for a bonus draw
            const ff ps = d.resid ? weigh_slice<T>(p, dp, trow, nullptr, c0, len, tb, db, &bar,
                                                   &phase, piece, wred, &s_expired, false)
                                  : ws;
            out.p = ff_add(out.p, ps);
            if (tid == 0) {
                tot[2 * sl] = ws;
                tot[2 * sl + 1] = ps;
            }
        }
    }
    if (tid == 0)
        q.out_mass[i] = out;
}

template <typename T>
__global__ void __launch_bounds__(kSampleThreads) shard_draw_kernel(const ShardDrawParams q)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    const FinishParams &p = q.fp;
    T *tb = reinterpret_cast<T *>(dsm);
    T *db = reinterpret_cast<T *>(dsm + p.stage_smem);
    __shared__ __align__(8) uint64_t bar;
    __shared__ float piece[kSampleThreads];
    __shared__ ff wred[kSampleWarps];
    __shared__ ff slice_tot[kMaxSlices];
    __shared__ ff s_excl[kSampleWarps];
    __shared__ int s_hit, s_last, s_expired;
    const int tid = threadIdx.x, lane = tid & 31, i = blockIdx.x;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        s_expired = 0;
    }
    __syncthreads();
    const DrawState st = q.state[i];
    if (!state_rows_ok(q, st))
        return;  // a poisoned request: step 2 wrote its outputs
    const float uf = __ldg(q.u_final + i);
    DrawCtx d = draw_ctx(st);

    // S and the shard holding u*S, in every warp (lane r holds shard r): an
    // inclusive float-float scan in shard order, the same bits on every
    // shard; an all-zero residual scans the p masses instead.  `past` marks
    // u*S at or beyond the end after rounding: then the last weight > 0 wins.
    int use = 0, cs = -1;
    bool past = true;
    ff base{0.f, 0.f}, target{0.f, 0.f};
    const ShardMass mine =
        lane < q.n_shards ? load_mass(q.mass_all + (int64_t)lane * p.B + i)
                          : ShardMass{{0.f, 0.f}, {0.f, 0.f}};
    for (int pass = 0; pass < 2; ++pass) {
        const ff v = pass == 0 ? mine.w : mine.p;
        ff incl = v;
#pragma unroll 1
        for (int o = 1; o < 32; o <<= 1) {
            const ff n = ff_shfl_up(incl, o);
            if (lane >= o)
                incl = ff_add(n, incl);
        }
        const ff S = {__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
        target = ff_mul(S, uf);
        const unsigned over = __ballot_sync(0xffffffffu, lane < q.n_shards && ff_gt(incl, target));
        const unsigned mass = __ballot_sync(0xffffffffu, lane < q.n_shards && v.hi > 0.f);
        cs = over ? __ffs(over) - 1 : (mass ? 31 - __clz(mass) : -1);
        ff excl = ff_shfl_up(incl, 1);
        if (lane == 0)
            excl = {0.f, 0.f};
        const int src = cs < 0 ? 0 : cs;
        base = {__shfl_sync(0xffffffffu, excl.hi, src), __shfl_sync(0xffffffffu, excl.lo, src)};
        past = over == 0u;
        if (!(d.resid && !(S.hi > 0.f)))
            break;
        d.resid = false;  // all-zero residual: draw from p_a instead
        use = 1;
    }
    if (cs != q.shard) {
        if (tid == 0) {
            if (cs < 0)  // no mass on any shard (never with finite rows)
                set_status(p.status, ST_NONFINITE);
            q.out_tokens[st.trow] = -1;  // the drawing shard writes the token
        }
        return;
    }
    const int nsl = (p.V + p.slice - 1) / p.slice;
    if (tid < nsl)
        slice_tot[tid] = q.slices[((size_t)i * kMaxSlices + tid) * 2 + use];
    __syncthreads();
    const T *trow = reinterpret_cast<const T *>(p.target) + st.trow * (int64_t)p.V;
    const T *drow =
        d.resid ? reinterpret_cast<const T *>(p.draft) + st.drow * (int64_t)p.V : nullptr;
    const DrawShared<T> sh{tb,     db,      &bar,   piece,  wred,       slice_tot,
                           s_excl, nullptr, &s_hit, &s_last, &s_expired};
    uint32_t phase = 0;
    const int y = find_in_range<T, false>(p, d, trow, drow, 0, p.V, nsl, base, target, past, -1,
                                          slice_tot, sh, phase);
    if (tid == 0) {
        int tok = y >= 0 ? q.v_begin + y : -1;
        if (y < 0)
            set_status(p.status, ST_NONFINITE);
        if (s_expired || (read_status(p.status) & ST_TIMEOUT))
            tok = -1;  // a copy gave up: the data may be stale
        q.out_tokens[st.trow] = tok;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Slice geometry of the mass and draw steps: the shard's Vs columns in
// slices of at most kStageRowBytes per row.  False when they exceed the
// slice table.
bool shard_draw_geometry(FinishParams &fp, int Vs, int e)
{
    const int gran = 16 / e;
    const int R = (Vs + gran - 1) / gran * gran;
    const int slice = std::min(R, kStageRowBytes / e);
    const int nv = (slice * e + 15) / 16;
    fp.R = R;
    fp.slice = slice;
    fp.pv = ((nv + kSampleThreads - 1) / kSampleThreads) | 1;  // odd: no bank conflicts
    fp.stage_smem = (int)align_up((size_t)slice * e, 128);
    fp.ncl = 1;
    return (Vs + slice - 1) / slice <= kMaxSlices;
}

template <typename T>
cudaError_t prepare_shard_draw()
{
    static cudaError_t once = [] {
        cudaError_t e = cudaFuncSetAttribute(
            shard_mass_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kStageRowBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(shard_draw_kernel<T>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     2 * kStageRowBytes);
        return e;
    }();
    return once;
}

template <typename T, bool GREEDY>
cudaError_t launch_rows_typed(const ShardStatsArgs &a, const StreamParams &sp, cudaStream_t s,
                              Tracer &tr)
{
    const VerifyArgs &v = a.v;
    ShardRowsParams rp{};
    rp.target = v.target;
    rp.draft = v.draft;
    rp.tokens = v.tokens;
    rp.cu = v.cu;
    rp.B = v.B;
    rp.Vs = v.V;
    rp.v_begin = a.v_begin;
    rp.max_rows = v.max_rows;
    rp.draft_rows = v.draft_stride > 0 ? (int64_t)v.B * v.draft_stride : v.max_rows - v.B;
    rp.n_rec = v.max_rows + rp.draft_rows;
    rp.draft_stride = v.draft_stride;
    rp.g = sp.g;
    rp.c = sp.c;
    rp.status = sp.status;
    rp.cu_flag = sp.cu_flag;
    rp.part = sp.part;
    rp.part_cap = sp.part_cap;
    rp.out = static_cast<ShardRow *>(a.out_rows);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)v.B);
    cfg.blockDim = dim3(kFinishThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, shard_rows_kernel<T, GREEDY>, rp);
    if (err != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_draw_typed(const ShardDrawArgs &a, bool draw, cudaStream_t s, Tracer &tr)
{
    const int e = (int)sizeof(T);
    const ShardLayout L = shard_layout(a.B, a.max_rows);
    unsigned char *ws = static_cast<unsigned char *>(a.ws);
    ShardDrawParams q{};
    FinishParams &fp = q.fp;
    fp.target = a.target;
    fp.draft = a.draft;
    fp.B = a.B;
    fp.V = a.V_shard;
    if (!shard_draw_geometry(fp, a.V_shard, e))
        return cudaErrorInvalidValue;
    fp.tma = ((int64_t)a.V_shard * e) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(a.target) % 16 == 0 &&
             (a.draft == nullptr || reinterpret_cast<uintptr_t>(a.draft) % 16 == 0);
    fp.status = reinterpret_cast<uint32_t *>(ws + L.base.status);
    q.state = reinterpret_cast<const DrawState *>(ws + L.state);
    q.slices = reinterpret_cast<ff *>(ws + L.slices);
    q.v_begin = a.v_begin;
    q.max_rows = a.max_rows;
    q.draft_rows = a.draft_stride > 0 ? (int64_t)a.B * a.draft_stride : a.max_rows - a.B;
    q.out_mass = static_cast<ShardMass *>(a.out_mass);
    q.mass_all = static_cast<const ShardMass *>(a.mass_all);
    q.n_shards = a.n_shards;
    q.shard = a.shard;
    q.u_final = a.u_final;
    q.out_tokens = a.out_tokens;
    cudaError_t err = prepare_shard_draw<T>();
    if (err != cudaSuccess)
        return err;
    tr.begin(s);
    if (draw)
        shard_draw_kernel<T><<<a.B, kSampleThreads, 2 * (size_t)fp.stage_smem, s>>>(q);
    else
        shard_mass_kernel<T><<<a.B, kSampleThreads, 2 * (size_t)fp.stage_smem, s>>>(q);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

}  // namespace

size_t shard_ws_bytes(int B, int64_t max_rows) { return shard_layout(B, max_rows).total; }

bool shard_columns_ok(int V_shard, int dtype)
{
    FinishParams fp{};
    return V_shard >= 1 && shard_draw_geometry(fp, V_shard, dtype == 0 ? 4 : 2);
}

cudaError_t launch_shard_stats(const ShardStatsArgs &a, cudaStream_t s, Tracer &tr)
{
    StreamParams sp;
    cudaError_t err = launch_stream_pass(a.v, s, tr, sp);
    if (err != cudaSuccess)
        return err;
    const bool greedy = a.v.temperature == 0.0;
    if (a.v.dtype == 0)
        return greedy ? launch_rows_typed<float, true>(a, sp, s, tr)
                      : launch_rows_typed<float, false>(a, sp, s, tr);
    return greedy ? launch_rows_typed<uint16_t, true>(a, sp, s, tr)
                  : launch_rows_typed<uint16_t, false>(a, sp, s, tr);
}

cudaError_t launch_shard_accept(const ShardAcceptArgs &a, cudaStream_t s, Tracer &tr)
{
    const ShardLayout L = shard_layout(a.B, a.max_rows);
    unsigned char *ws = static_cast<unsigned char *>(a.ws);
    const bool greedy = a.temperature == 0.0;
    ShardAcceptParams p{};
    p.rows = static_cast<const ShardRow *>(a.rows_all);
    p.n_shards = a.n_shards;
    for (int r = 0; r <= a.n_shards; ++r)
        p.begin[r] = a.begin[r];
    p.tokens = a.tokens;
    p.cu = a.cu;
    p.u_accept = a.u_accept;
    p.B = a.B;
    p.V = a.begin[a.n_shards];
    p.max_rows = a.max_rows;
    p.draft_rows = a.draft_stride > 0 ? (int64_t)a.B * a.draft_stride : a.max_rows - a.B;
    p.n_rec = a.max_rows + p.draft_rows;
    p.draft_stride = a.draft_stride;
    p.c = greedy ? 0.f : (float)(1.4426950408889634074 / a.temperature);  // log2(e) / T
    p.out_tokens = a.out_tokens;
    p.out_len = a.out_len;
    p.out_p = a.out_p;
    p.out_q = a.out_q;
    p.status = reinterpret_cast<uint32_t *>(ws + L.base.status);
    p.cu_flag = p.status + 1;
    p.state = reinterpret_cast<DrawState *>(ws + L.state);
    tr.begin(s);
    if (greedy)
        shard_accept_kernel<true><<<a.B, kFinishThreads, 0, s>>>(p);
    else
        shard_accept_kernel<false><<<a.B, kFinishThreads, 0, s>>>(p);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

cudaError_t launch_shard_mass(const ShardDrawArgs &a, cudaStream_t s, Tracer &tr)
{
    return a.dtype == 0 ? launch_draw_typed<float>(a, false, s, tr)
                        : launch_draw_typed<uint16_t>(a, false, s, tr);
}

cudaError_t launch_shard_draw(const ShardDrawArgs &a, cudaStream_t s, Tracer &tr)
{
    return a.dtype == 0 ? launch_draw_typed<float>(a, true, s, tr)
                        : launch_draw_typed<uint16_t>(a, true, s, tr);
}

}  // namespace sv
