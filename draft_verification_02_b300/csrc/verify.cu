// verify.cu - batched draft verification on sm_103a: the launch side of the
// two kernels (stream_kernel.cuh, finish_kernel.cuh).
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
//  - T > 0, finish_sample_kernel: one cluster of 4, 8 or 16 CTAs per
//    request.  The request's rows are merged one or two per warp of the
//    cluster (their (m, s) and p(x) sent to every CTA through distributed
//    shared memory; with 4 CTAs, a 65th row is merged by every CTA itself);
//    every warp of every CTA runs the accept test and first-rejection ballot
//    (identical bits everywhere), then each CTA stages its share of the
//    final-draw rows with TMA and sums the weights.  The range sums are
//    exchanged the same way; the CTA whose range holds u*S finds the token
//    with a block scan of per-thread piece sums, then a warp computes the
//    chosen piece's weights and one lane walks them in order.
// The drafter's kernels (confidence_kernel, draft_sample_kernel,
// draft_greedy_kernel) and the acceptance statistics are launched from here
// too; D-cut from dcut.cu.
// Every merge runs in a fixed order, so repeated calls give identical bits.
#include <algorithm>
#include <cstdint>

#include "finish_kernel.cuh"
#include "stream_kernel.cuh"

namespace sv {

// Acceptance statistics of one verification call, one CTA: per position j
// the requests that tested it (K_i > j, a_i >= j) and accepted it (a_i > j),
// and the mean accepted length over requests with a_i >= 0.  Integer counts,
// so the result does not depend on the order of the atomic adds.
constexpr int kStatsThreads = 1024;

struct StatsParams {
    const int32_t *accept_len;
    const int32_t *cu;
    int B, Kmax;
    int32_t *out_reached;
    int32_t *out_accepted;
    float *out_mean;
    uint32_t *status;
};

__global__ void __launch_bounds__(kStatsThreads) acceptance_stats_kernel(const StatsParams p)
{
    __shared__ int reached[kMaxDraft], accepted[kMaxDraft];
    __shared__ unsigned long long total;
    __shared__ int n, bad;
    const int tid = threadIdx.x;
    if (tid < kMaxDraft)
        reached[tid] = accepted[tid] = 0;
    if (tid == 0) {
        total = 0ull;
        n = 0;
        bad = 0;
    }
    __syncthreads();
    for (int i = tid; i < p.B; i += kStatsThreads) {
        const int a = __ldg(p.accept_len + i);
        const int k = __ldg(p.cu + i + 1) - __ldg(p.cu + i);
        if (a < 0)
            continue;  // a poisoned request
        if (a > k || k > p.Kmax || k < 0) {
            bad = 1;
            continue;
        }
        atomicAdd(&total, (unsigned long long)a);
        atomicAdd(&n, 1);
        for (int j = 0; j < k; ++j) {
            if (a >= j)
                atomicAdd(&reached[j], 1);
            if (a > j)
                atomicAdd(&accepted[j], 1);
        }
    }
    __syncthreads();
    if (tid < p.Kmax) {
        p.out_reached[tid] = bad ? -1 : reached[tid];
        p.out_accepted[tid] = bad ? -1 : accepted[tid];
    }
    if (tid == 0) {
        if (bad)
            set_status(p.status, ST_INVALID);
        *p.out_mean = bad ? __int_as_float(0x7fc00000)
                          : (n > 0 ? (float)((double)total / (double)n) : 0.f);
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

template <typename T, bool OUTLINE, int MINB>
static cudaError_t prepare_finish_sample()
{
    static cudaError_t once = [] {
        cudaError_t e = cudaFuncSetAttribute(finish_sample_kernel<T, OUTLINE, MINB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             2 * kStageRowBytes);
        if (e == cudaSuccess)  // clusters of 16 CTAs
            e = cudaFuncSetAttribute(finish_sample_kernel<T, OUTLINE, MINB>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return e;
    }();
    return once;
}

// Drafting at T > 0: each CTA streams its row through two slices of at most
// this size, which leaves room for four CTAs per SM (measured on drafting
// 512 rows of V = 151936 bf16: 24 KB 42.8 us, 36 KB 52.8 us, 48 KB 54.5 us).
#ifndef SV_DRAFT_STAGE_KB
#define SV_DRAFT_STAGE_KB 24
#endif
constexpr int kDraftStageBytes = SV_DRAFT_STAGE_KB * 1024;

template <typename T>
static cudaError_t prepare_draft_sample()
{
    static cudaError_t once = [] {
        cudaError_t e = cudaFuncSetAttribute(draft_sample_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             2 * kDraftStageBytes + 12 * kMaxRowSlices);
        return e;
    }();
    return once;
}

// Kernel 1's parameters for a verification call (a.out_tokens / a.out_len
// may be null: then malformed offsets are only flagged, not poisoned).
template <typename T, bool GREEDY>
static StreamParams stream_params(const VerifyArgs &a)
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
    sp.part_cap = (int64_t)((L.total - L.part1) / sizeof(Partial));
    sp.draft_rows = a.draft_stride > 0 ? (int64_t)a.B * a.draft_stride : a.max_rows - a.B;
    sp.debug_unit = a.debug_item;
    return sp;
}

template <typename T, bool GREEDY>
static cudaError_t enqueue_stream(const StreamParams &sp, cudaStream_t s, Tracer &tr)
{
    cudaError_t err = prepare_stream<T, GREEDY>();
    if (err != cudaSuccess)
        return err;
    const int grid1 = (sp.g.P + kStreamWarps - 1) / kStreamWarps;
    const size_t smem1 = (size_t)kStreamWarps * kRing * sp.piece_smem +
                         (sp.draft_stride > 0 && !GREEDY ? 4 * (size_t)(sp.B + 1) : 0);
    tr.begin(s);
    stream_kernel<T, GREEDY><<<grid1, kStreamThreads, smem1, s>>>(sp);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

cudaError_t launch_stream_pass(const VerifyArgs &a, cudaStream_t s, Tracer &tr, StreamParams &sp)
{
    const bool greedy = a.temperature == 0.0;
    if (a.dtype == 0) {
        sp = greedy ? stream_params<float, true>(a) : stream_params<float, false>(a);
        return greedy ? enqueue_stream<float, true>(sp, s, tr)
                      : enqueue_stream<float, false>(sp, s, tr);
    }
    sp = greedy ? stream_params<uint16_t, true>(a) : stream_params<uint16_t, false>(a);
    return greedy ? enqueue_stream<uint16_t, true>(sp, s, tr)
                  : enqueue_stream<uint16_t, false>(sp, s, tr);
}

template <typename T, bool GREEDY>
static cudaError_t launch_typed(const VerifyArgs &a, cudaStream_t s, Tracer &tr)
{
    const int e = (int)sizeof(T);
    const StreamParams sp = stream_params<T, GREEDY>(a);
    const Geometry g = sp.g;
    const bool tma = sp.tma != 0;

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
    if (!GREEDY && !draw_geometry(fp, a.B, a.V, e, sm_count()))
        return cudaErrorInvalidValue;  // vocabulary beyond the draw's slice table
    // the finish kernel merges up to two rows per warp of the cluster, then
    // one per warp of each CTA
    if (!GREEDY && 2 * kMaxDraft + 1 > 2 * kSampleWarps * fp.ncl + kSampleWarps)
        return cudaErrorInvalidValue;
    fp.tma = tma;
    fp.c = sp.c;
    fp.status = sp.status;
    fp.cu_flag = sp.cu_flag;
    fp.part = sp.part;
    fp.part_cap = sp.part_cap;

    // The finish kernel with its weighing out of line (more registers, at
    // most two CTAs per SM) when its CTAs can each have an SM and the rows
    // are long, inline otherwise (72 registers, three CTAs per SM).  Measured
    // on B300: B=16, V=128000 (128 CTAs) 22.0 us out of line vs 22.4 inline;
    // B=4, V=1024 10.4 inline vs 10.9; B=32 and B=64 at V >= 128000 0.7-3.3 us
    // faster inline.
    const bool outline = (int64_t)a.B * fp.ncl <= (int64_t)sm_count() && a.V >= 32768;
    // A dense grid (the half-size slices of draw_geometry) takes the
    // instance whose registers allow four CTAs per SM: B=128, V=151936
    // 0.1545 -> 0.1481 ms per step, B=64 0.0915 -> 0.0845; smaller grids
    // keep three (mtp 0.0200 vs 0.0208 with four).
    const bool dense =
        !outline && (int64_t)a.B * fp.ncl > SV_DENSE_PER_SM * (int64_t)sm_count();
    cudaError_t err = cudaSuccess;
    if (!GREEDY)
        err = outline ? prepare_finish_sample<T, true, 2>()
                      : (dense ? prepare_finish_sample<T, false, 4>()
                               : prepare_finish_sample<T, false, 2>());
    if (err != cudaSuccess)
        return err;
    if ((err = enqueue_stream<T, GREEDY>(sp, s, tr)) != cudaSuccess)
        return err;

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
        err = outline ? cudaLaunchKernelEx(&cfg, finish_sample_kernel<T, true, 2>, fp)
              : dense ? cudaLaunchKernelEx(&cfg, finish_sample_kernel<T, false, 4>, fp)
                      : cudaLaunchKernelEx(&cfg, finish_sample_kernel<T, false, 2>, fp);
    }
    if (err != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

// The streaming pass over the B*Kmax padded drafter rows (every row is read):
// the per-row partials the drafting kernels merge.
template <typename T, bool GREEDY>
static cudaError_t launch_draft_pass(const void *draft, int B, int Kmax, int V, double temperature,
                                     void *ws_ptr, cudaStream_t s, Tracer &tr, StreamParams &sp)
{
    const int e = (int)sizeof(T);
    const int64_t rows = (int64_t)B * Kmax;
    const WsLayout L = ws_layout(B, (int64_t)B * (Kmax + 1), V);
    unsigned char *ws = static_cast<unsigned char *>(ws_ptr);
    const int ctas_max = sm_count() * SV_STREAM_CTAS_PER_SM;
    const Geometry g = plan(rows, rows, V, e, std::min(kMaxWorkers, ctas_max * kStreamWarps));
    const double c = GREEDY ? 0.0 : 1.4426950408889634074 / temperature;  // log2(e) / T
    sp = StreamParams{};
    sp.target = draft;  // every draft row is read as a row of the pass
    sp.draft = nullptr;
    sp.cu = nullptr;    // no offsets: every row is real
    sp.B = B;
    sp.V = V;
    sp.draft_slots = 0;
    sp.draft_stride = 0;
    sp.g = g;
    sp.tma = ((int64_t)V * e) % 16 == 0 && reinterpret_cast<uintptr_t>(draft) % 16 == 0;
    sp.piece_smem = (int)align_up((size_t)g.Q * e, 128);
    sp.c = (float)c;
    sp.status = reinterpret_cast<uint32_t *>(ws + L.status);
    sp.cu_flag = sp.status + 1;
    sp.part = reinterpret_cast<Partial *>(ws + L.part1);
    sp.part_cap = (int64_t)((L.total - L.part1) / sizeof(Partial));
    sp.draft_rows = 0;
    cudaError_t err = prepare_stream<T, GREEDY>();
    if (err != cudaSuccess)
        return err;
    const int grid1 = (g.P + kStreamWarps - 1) / kStreamWarps;
    tr.begin(s);
    stream_kernel<T, GREEDY><<<grid1, kStreamThreads, (size_t)kStreamWarps * kRing * sp.piece_smem,
                              s>>>(sp);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

static cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     cudaLaunchAttribute (&attr)[2], int cluster)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cfg;
}

template <typename T, bool GREEDY>
static cudaError_t launch_conf_typed(const ConfArgs &a, cudaStream_t s, Tracer &tr)
{
    const int64_t rows = (int64_t)a.B * a.Kmax;
    StreamParams sp;
    cudaError_t err = launch_draft_pass<T, GREEDY>(a.draft, a.B, a.Kmax, a.V, a.temperature, a.ws,
                                                   s, tr, sp);
    if (err != cudaSuccess)
        return err;
    ConfParams cp{};
    cp.draft = a.draft;
    cp.tokens = a.tokens;
    cp.kmax = a.kmax;
    cp.B = a.B;
    cp.Kmax = a.Kmax;
    cp.V = a.V;
    cp.g = sp.g;
    cp.c = sp.c;
    cp.out_conf = a.out_conf;
    cp.status = sp.status;
    cp.part = sp.part;
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg =
        pdl_config(dim3((unsigned)((rows + kFinishWarps - 1) / kFinishWarps)), dim3(kFinishThreads),
                   0, s, attr, 1);
    if ((err = cudaLaunchKernelEx(&cfg, confidence_kernel<T, GREEDY>, cp)) != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

cudaError_t launch_confidence(const ConfArgs &a, cudaStream_t s, Tracer &tr)
{
    const bool greedy = a.temperature == 0.0;
    if (a.dtype == 0)
        return greedy ? launch_conf_typed<float, true>(a, s, tr)
                      : launch_conf_typed<float, false>(a, s, tr);
    return greedy ? launch_conf_typed<uint16_t, true>(a, s, tr)
                  : launch_conf_typed<uint16_t, false>(a, s, tr);
}

// T > 0: one kernel (draft_sample_kernel reads each row once and draws from
// it); T = 0: the streaming pass over the rows and a warp argmax merge per row.
template <typename T, bool GREEDY>
static cudaError_t launch_draft_typed(const DraftArgs &a, cudaStream_t s, Tracer &tr)
{
    const int e = (int)sizeof(T);
    const int64_t rows = (int64_t)a.B * a.Kmax;
    FinishParams fp{};
    fp.target = a.draft;
    fp.u_final = a.u;
    fp.out_tokens = a.out_tokens;
    fp.out_conf = a.out_conf;
    fp.kmax = a.kmax;
    fp.Kmax = a.Kmax;
    fp.B = a.B;
    fp.V = a.V;
    const WsLayout L = ws_layout(a.B, (int64_t)a.B * (a.Kmax + 1), a.V);
    fp.status = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(a.ws) + L.status);
    fp.cu_flag = fp.status + 1;
    cudaLaunchAttribute attr[2];
    cudaError_t err;
    if (GREEDY) {
        StreamParams sp;
        if ((err = launch_draft_pass<T, true>(a.draft, a.B, a.Kmax, a.V, 0.0, a.ws, s, tr, sp)) !=
            cudaSuccess)
            return err;
        fp.g = sp.g;
        fp.part = sp.part;
        fp.part_cap = sp.part_cap;
        const cudaLaunchConfig_t cfg = pdl_config(
            dim3((unsigned)((rows + kFinishWarps - 1) / kFinishWarps)), dim3(kFinishThreads), 0, s,
            attr, 1);
        err = cudaLaunchKernelEx(&cfg, draft_greedy_kernel<T>, fp);
    } else {
        // one CTA per row; the row streams through two slices of shared memory
        const int gran = 16 / e;
        const int slice = std::min((a.V + gran - 1) / gran * gran, kDraftStageBytes / e);
        if (((int64_t)a.V + slice - 1) / slice > kMaxRowSlices)
            return cudaErrorInvalidValue;
        fp.slice = slice;
        fp.pv = (((slice * e + 15) / 16 + kSampleThreads - 1) / kSampleThreads) | 1;
        fp.stage_smem = (int)align_up((size_t)slice * e, 128);
        if ((err = prepare_draft_sample<T>()) != cudaSuccess)
            return err;
        fp.tma = ((int64_t)a.V * e) % 16 == 0 && reinterpret_cast<uintptr_t>(a.draft) % 16 == 0;
        fp.c = (float)(1.4426950408889634074 / a.temperature);  // log2(e) / T
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)rows);
        cfg.blockDim = dim3(kSampleThreads);
        const int nsl = (int)(((int64_t)a.V + slice - 1) / slice);
        cfg.dynamicSmemBytes = 2 * (size_t)fp.stage_smem + 12 * (size_t)nsl;  // + slice table
        cfg.stream = s;
        tr.begin(s);
        err = cudaLaunchKernelEx(&cfg, draft_sample_kernel<T>, fp);
    }
    if (err != cudaSuccess)
        return err;
    tr.after_kernel(s);
    return cudaSuccess;
}

cudaError_t launch_draft(const DraftArgs &a, cudaStream_t s, Tracer &tr)
{
    const bool greedy = a.temperature == 0.0;
    if (a.dtype == 0)
        return greedy ? launch_draft_typed<float, true>(a, s, tr)
                      : launch_draft_typed<float, false>(a, s, tr);
    return greedy ? launch_draft_typed<uint16_t, true>(a, s, tr)
                  : launch_draft_typed<uint16_t, false>(a, s, tr);
}

cudaError_t launch_acceptance_stats(const StatsArgs &a, cudaStream_t s, Tracer &tr)
{
    StatsParams sp{};
    sp.accept_len = a.accept_len;
    sp.cu = a.cu;
    sp.B = a.B;
    sp.Kmax = a.Kmax;
    sp.out_reached = a.out_reached;
    sp.out_accepted = a.out_accepted;
    sp.out_mean = a.out_mean;
    sp.status = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(a.ws) +
                                             ws_layout(0, 0, 0).status);
    tr.begin(s);
    acceptance_stats_kernel<<<1, kStatsThreads, 0, s>>>(sp);
    if (cudaError_t err = cudaGetLastError(); err != cudaSuccess)
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
