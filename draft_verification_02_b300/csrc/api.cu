// api.cu - the C ABI (include/specverify.h): argument checks, workspace
// sizing, launches on the caller's stream, device status, trace hook.
// Nothing here allocates device memory or synchronises, except
// spec_get_device_status, whose job is to synchronise and read.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "launch.h"
#include "specverify.h"

namespace {

constexpr int kMaxTraceEvents = 16;
thread_local cudaEvent_t g_trace[kMaxTraceEvents];
thread_local int g_trace_n = 0;
thread_local int64_t g_launches = 0;
thread_local uint64_t g_expire_unit = 0;  // test hook: 1 + the unit, 0 = off

sv::Tracer make_tracer()
{
    sv::Tracer t;
    t.events = g_trace_n > 0 ? g_trace : nullptr;
    t.n = g_trace_n;
    return t;
}

int cuda_status(cudaError_t e)
{
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

bool valid_dtype(int dtype) { return dtype == SPEC_F32 || dtype == SPEC_BF16; }

// Checks shared by both verification calls; SPEC_OK when the sizes are usable.
int check_verify_sizes(int32_t B, int32_t V, int64_t max_target_rows, int32_t draft_stride)
{
    if (B < 0 || B > SPEC_MAX_BATCH || V < 1 || draft_stride < 0 || draft_stride > (1 << 20))
        return SPEC_ERR_INVALID_ARG;
    if (max_target_rows < B || max_target_rows > (int64_t)B * (SPEC_MAX_DRAFT + 1))
        return SPEC_ERR_INVALID_ARG;
    if (V > sv::kMaxVocab)
        return SPEC_ERR_INVALID_ARG;
    return SPEC_OK;
}

}  // namespace

namespace sv {

// Inside stream capture a plain record only orders streams; the external
// flag makes it a timestamp node of the graph.
static void record_event(cudaEvent_t e, cudaStream_t s)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else
        cudaEventRecord(e, s);
}

void Tracer::begin(cudaStream_t s)
{
    next = 0;
    if (next < n)
        record_event(events[next++], s);
}

void Tracer::after_kernel(cudaStream_t s)
{
    ++g_launches;
    if (next < n)
        record_event(events[next++], s);
}

}  // namespace sv

extern "C" {

size_t spec_workspace_size(int32_t B, int64_t max_target_rows, int32_t V)
{
    if (B < 0 || max_target_rows < 0 || V < 0)
        return 0;
    if (V > sv::kMaxVocab)
        return 0;
    return sv::ws_layout(B, max_target_rows, V).total;
}

int spec_workspace_init(void *workspace, size_t ws_bytes, spec_stream_t stream)
{
    if (!workspace || ws_bytes == 0)
        return SPEC_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(workspace, 0, ws_bytes, (cudaStream_t)stream));
}

int spec_verify_greedy(const void *target_logits, int dtype, const int32_t *draft_tokens,
                       const int32_t *cu_draft, int32_t B, int32_t V, int64_t max_target_rows,
                       int32_t draft_stride, int32_t *out_tokens, int32_t *out_accept_len,
                       void *workspace, size_t ws_bytes, spec_stream_t stream)
{
    if (!valid_dtype(dtype))
        return SPEC_ERR_INVALID_ARG;
    int st = check_verify_sizes(B, V, max_target_rows, draft_stride);
    if (st != SPEC_OK)
        return st;
    if (B == 0)
        return SPEC_OK;
    if (!target_logits || !cu_draft || !out_tokens || !out_accept_len ||
        (!draft_tokens && max_target_rows > B))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < spec_workspace_size(B, max_target_rows, V))
        return SPEC_ERR_WORKSPACE;
    sv::VerifyArgs a{};
    a.target = target_logits;
    a.draft = nullptr;
    a.dtype = dtype;
    a.tokens = draft_tokens;
    a.cu = cu_draft;
    a.B = B;
    a.V = V;
    a.max_rows = max_target_rows;
    a.draft_stride = draft_stride;
    a.temperature = 0.0;
    a.out_tokens = out_tokens;
    a.out_len = out_accept_len;
    a.ws = workspace;
    a.debug_item = g_expire_unit;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_verify(a, (cudaStream_t)stream, tr));
}

int spec_verify_sample(const void *target_logits, const void *draft_logits, int dtype,
                       const int32_t *draft_tokens, const int32_t *cu_draft, int32_t B,
                       int32_t V, int64_t max_target_rows, int32_t draft_stride,
                       float temperature, const float *u_accept, const float *u_final,
                       int32_t *out_tokens, int32_t *out_accept_len, float *out_p,
                       float *out_q, void *workspace, size_t ws_bytes, spec_stream_t stream)
{
    if (!(temperature >= 0.f) || std::isinf(temperature))
        return SPEC_ERR_INVALID_ARG;
    if (temperature == 0.f)
        return spec_verify_greedy(target_logits, dtype, draft_tokens, cu_draft, B, V,
                                  max_target_rows, draft_stride, out_tokens, out_accept_len,
                                  workspace, ws_bytes, stream);
    if (!valid_dtype(dtype))
        return SPEC_ERR_INVALID_ARG;
    int st = check_verify_sizes(B, V, max_target_rows, draft_stride);
    if (st != SPEC_OK)
        return st;
    if (B == 0)
        return SPEC_OK;
    const bool drafts = max_target_rows > B;
    if (!target_logits || !cu_draft || !out_tokens || !out_accept_len || !u_final ||
        (drafts && (!draft_logits || !draft_tokens || !u_accept)))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < spec_workspace_size(B, max_target_rows, V))
        return SPEC_ERR_WORKSPACE;
    sv::VerifyArgs a{};
    a.target = target_logits;
    a.draft = draft_logits;
    a.dtype = dtype;
    a.tokens = draft_tokens;
    a.cu = cu_draft;
    a.B = B;
    a.V = V;
    a.max_rows = max_target_rows;
    a.draft_stride = draft_stride;
    a.temperature = (double)temperature;
    a.u_accept = u_accept;
    a.u_final = u_final;
    a.out_tokens = out_tokens;
    a.out_len = out_accept_len;
    a.out_p = out_p;
    a.out_q = out_q;
    a.ws = workspace;
    a.debug_item = g_expire_unit;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_verify(a, (cudaStream_t)stream, tr));
}

int dcut_allocate(const float *conf, const int32_t *kmax, int32_t B, int32_t Kmax,
                  int32_t budget, float min_gain, int32_t *out_depth, int32_t *out_cu,
                  float *out_expected_len, void *workspace, size_t ws_bytes,
                  spec_stream_t stream)
{
    if (B < 0 || B > SPEC_MAX_BATCH || Kmax < 0 || Kmax > SPEC_MAX_DRAFT || budget < 0 ||
        std::isnan(min_gain))
        return SPEC_ERR_INVALID_ARG;
    int bp = 1, kp = 1;
    while (bp < B)
        bp <<= 1;
    while (kp < Kmax)
        kp <<= 1;
    if ((int64_t)bp * kp > SPEC_DCUT_MAX_CANDIDATES)
        return SPEC_ERR_INVALID_ARG;
    if (!out_cu || (B > 0 && (!kmax || !out_depth || (Kmax > 0 && !conf))))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < spec_workspace_size(0, 0, 0))
        return SPEC_ERR_WORKSPACE;
    sv::DcutArgs a{};
    a.conf = conf;
    a.kmax = kmax;
    a.B = B;
    a.Kmax = Kmax;
    a.budget = budget;
    a.min_gain = min_gain;
    a.out_depth = out_depth;
    a.out_cu = out_cu;
    a.out_expected = out_expected_len;
    a.ws = workspace;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_dcut(a, (cudaStream_t)stream, tr));
}

int dcut_allocate_cost(const float *conf, const int32_t *kmax, int32_t B, int32_t Kmax,
                       double max_cost, int32_t *out_depth, int32_t *out_cu,
                       double *out_benefit, void *workspace, size_t ws_bytes,
                       spec_stream_t stream)
{
    if (B < 0 || B > SPEC_MAX_BATCH || Kmax < 0 || Kmax > SPEC_MAX_DRAFT || std::isnan(max_cost))
        return SPEC_ERR_INVALID_ARG;
    if (!out_cu || (B > 0 && (!kmax || !out_depth || (Kmax > 0 && !conf))))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < spec_workspace_size(0, 0, 0))
        return SPEC_ERR_WORKSPACE;
    sv::DcutCostArgs a{};
    a.conf = conf;
    a.kmax = kmax;
    a.B = B;
    a.Kmax = Kmax;
    a.max_cost = max_cost;
    a.out_depth = out_depth;
    a.out_cu = out_cu;
    a.out_benefit = out_benefit;
    a.ws = workspace;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_dcut_cost(a, (cudaStream_t)stream, tr));
}

int spec_draft_confidence(const void *draft_logits, int dtype, const int32_t *draft_tokens,
                          const int32_t *kmax, int32_t B, int32_t Kmax, int32_t V,
                          float temperature, float *out_conf, void *workspace, size_t ws_bytes,
                          spec_stream_t stream)
{
    if (!valid_dtype(dtype) || B < 0 || B > SPEC_MAX_BATCH || Kmax < 0 ||
        Kmax > SPEC_MAX_DRAFT || V < 1 || V > sv::kMaxVocab || !(temperature >= 0.f) ||
        std::isinf(temperature))
        return SPEC_ERR_INVALID_ARG;
    if ((int64_t)B * Kmax == 0)
        return SPEC_OK;
    if (!draft_logits || !draft_tokens || !kmax || !out_conf)
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < spec_workspace_size(B, (int64_t)B * (Kmax + 1), V))
        return SPEC_ERR_WORKSPACE;
    sv::ConfArgs a{};
    a.draft = draft_logits;
    a.dtype = dtype;
    a.tokens = draft_tokens;
    a.kmax = kmax;
    a.B = B;
    a.Kmax = Kmax;
    a.V = V;
    a.temperature = (double)temperature;
    a.out_conf = out_conf;
    a.ws = workspace;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_confidence(a, (cudaStream_t)stream, tr));
}

int spec_draft_sample(const void *draft_logits, int dtype, const int32_t *kmax, int32_t B,
                      int32_t Kmax, int32_t V, float temperature, const float *u_draft,
                      int32_t *out_tokens, float *out_conf, void *workspace, size_t ws_bytes,
                      spec_stream_t stream)
{
    if (!valid_dtype(dtype) || B < 0 || B > SPEC_MAX_BATCH || Kmax < 0 ||
        Kmax > SPEC_MAX_DRAFT || V < 1 || V > sv::kMaxVocab || !(temperature >= 0.f) ||
        std::isinf(temperature))
        return SPEC_ERR_INVALID_ARG;
    if ((int64_t)B * Kmax == 0)
        return SPEC_OK;
    if (!draft_logits || !kmax || !out_tokens || !out_conf || (temperature > 0.f && !u_draft))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < spec_workspace_size(B, (int64_t)B * (Kmax + 1), V))
        return SPEC_ERR_WORKSPACE;
    sv::DraftArgs a{};
    a.draft = draft_logits;
    a.dtype = dtype;
    a.kmax = kmax;
    a.B = B;
    a.Kmax = Kmax;
    a.V = V;
    a.temperature = (double)temperature;
    a.u = u_draft;
    a.out_tokens = out_tokens;
    a.out_conf = out_conf;
    a.ws = workspace;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_draft(a, (cudaStream_t)stream, tr));
}

int spec_acceptance_stats(const int32_t *accept_len, const int32_t *cu_draft, int32_t B,
                          int32_t Kmax, int32_t *out_reached, int32_t *out_accepted,
                          float *out_mean, void *workspace, size_t ws_bytes, spec_stream_t stream)
{
    if (B < 0 || B > SPEC_MAX_BATCH || Kmax < 0 || Kmax > SPEC_MAX_DRAFT)
        return SPEC_ERR_INVALID_ARG;
    if ((B > 0 && (!accept_len || !cu_draft)) || (Kmax > 0 && (!out_reached || !out_accepted)) ||
        !out_mean)
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < spec_workspace_size(0, 0, 0))
        return SPEC_ERR_WORKSPACE;
    sv::StatsArgs a{};
    a.accept_len = accept_len;
    a.cu = cu_draft;
    a.B = B;
    a.Kmax = Kmax;
    a.out_reached = out_reached;
    a.out_accepted = out_accepted;
    a.out_mean = out_mean;
    a.ws = workspace;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_acceptance_stats(a, (cudaStream_t)stream, tr));
}

// ---- vocabulary-sharded verification ----

size_t spec_shard_workspace_size(int32_t B, int64_t max_target_rows, int32_t V_shard)
{
    if (check_verify_sizes(B, V_shard, max_target_rows, 0) != SPEC_OK)
        return 0;
    return sv::shard_ws_bytes(B, max_target_rows);
}

int64_t spec_shard_row_count(int32_t B, int64_t max_target_rows, int32_t draft_stride)
{
    if (check_verify_sizes(B, 1, max_target_rows, draft_stride) != SPEC_OK)
        return -1;
    return max_target_rows + (draft_stride > 0 ? (int64_t)B * draft_stride : max_target_rows - B);
}

int spec_shard_row_stats(const void *target_shard, const void *draft_shard, int dtype,
                         const int32_t *draft_tokens, const int32_t *cu_draft, int32_t B,
                         int32_t v_begin, int32_t v_end, int64_t max_target_rows,
                         int32_t draft_stride, float temperature, spec_shard_row *out_rows,
                         void *workspace, size_t ws_bytes, spec_stream_t stream)
{
    if (!valid_dtype(dtype) || !(temperature >= 0.f) || std::isinf(temperature) ||
        v_begin < 0 || v_end <= v_begin)
        return SPEC_ERR_INVALID_ARG;
    const int32_t Vs = v_end - v_begin;
    int st = check_verify_sizes(B, Vs, max_target_rows, draft_stride);
    if (st != SPEC_OK)
        return st;
    if (B == 0)
        return SPEC_OK;
    const bool drafts = max_target_rows > B, greedy = temperature == 0.f;
    if (!target_shard || !cu_draft || !out_rows || (drafts && !draft_tokens) ||
        (drafts && !greedy && !draft_shard))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < sv::shard_ws_bytes(B, max_target_rows))
        return SPEC_ERR_WORKSPACE;
    sv::ShardStatsArgs a{};
    a.v.target = target_shard;
    a.v.draft = greedy ? nullptr : draft_shard;
    a.v.dtype = dtype;
    a.v.tokens = draft_tokens;
    a.v.cu = cu_draft;
    a.v.B = B;
    a.v.V = Vs;
    a.v.max_rows = max_target_rows;
    a.v.draft_stride = draft_stride;
    a.v.temperature = (double)temperature;
    a.v.ws = workspace;
    a.v.debug_item = g_expire_unit;
    a.v_begin = v_begin;
    a.out_rows = out_rows;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_shard_stats(a, (cudaStream_t)stream, tr));
}

int spec_shard_accept(const spec_shard_row *rows_all, int32_t n_shards,
                      const int32_t *shard_begin, const int32_t *draft_tokens,
                      const int32_t *cu_draft, int32_t B, int64_t max_target_rows,
                      int32_t draft_stride, float temperature, const float *u_accept,
                      int32_t *out_tokens, int32_t *out_accept_len, float *out_p, float *out_q,
                      void *workspace, size_t ws_bytes, spec_stream_t stream)
{
    if (n_shards < 1 || n_shards > sv::kMaxShards || !shard_begin || !(temperature >= 0.f) ||
        std::isinf(temperature))
        return SPEC_ERR_INVALID_ARG;
    if (shard_begin[0] != 0)
        return SPEC_ERR_INVALID_ARG;
    for (int r = 0; r < n_shards; ++r)
        if (shard_begin[r + 1] <= shard_begin[r])
            return SPEC_ERR_INVALID_ARG;
    int st = check_verify_sizes(B, shard_begin[n_shards], max_target_rows, draft_stride);
    if (st != SPEC_OK)
        return st;
    if (B == 0)
        return SPEC_OK;
    const bool drafts = max_target_rows > B, greedy = temperature == 0.f;
    if (!rows_all || !cu_draft || !out_tokens || !out_accept_len || (drafts && !draft_tokens) ||
        (drafts && !greedy && !u_accept))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < sv::shard_ws_bytes(B, max_target_rows))
        return SPEC_ERR_WORKSPACE;
    sv::ShardAcceptArgs a{};
    a.rows_all = rows_all;
    a.n_shards = n_shards;
    a.begin = shard_begin;
    a.tokens = draft_tokens;
    a.cu = cu_draft;
    a.B = B;
    a.max_rows = max_target_rows;
    a.draft_stride = draft_stride;
    a.temperature = (double)temperature;
    a.u_accept = u_accept;
    a.out_tokens = out_tokens;
    a.out_len = out_accept_len;
    a.out_p = greedy ? nullptr : out_p;
    a.out_q = greedy ? nullptr : out_q;
    a.ws = workspace;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_shard_accept(a, (cudaStream_t)stream, tr));
}

namespace {

// Checks shared by the two draw steps; fills the common arguments.
int shard_draw_args(const void *target_shard, const void *draft_shard, int dtype, int32_t B,
                    int32_t v_begin, int32_t v_end, int64_t max_target_rows, int32_t draft_stride,
                    void *workspace, size_t ws_bytes, sv::ShardDrawArgs &a)
{
    if (!valid_dtype(dtype) || v_begin < 0 || v_end <= v_begin)
        return SPEC_ERR_INVALID_ARG;
    const int32_t Vs = v_end - v_begin;
    int st = check_verify_sizes(B, Vs, max_target_rows, draft_stride);
    if (st != SPEC_OK)
        return st;
    if (!sv::shard_columns_ok(Vs, dtype))
        return SPEC_ERR_INVALID_ARG;
    if (B > 0 && (!target_shard || (max_target_rows > B && !draft_shard)))
        return SPEC_ERR_INVALID_ARG;
    if (B > 0 && (!workspace || ws_bytes < sv::shard_ws_bytes(B, max_target_rows)))
        return SPEC_ERR_WORKSPACE;
    a.target = target_shard;
    a.draft = draft_shard;
    a.dtype = dtype;
    a.B = B;
    a.v_begin = v_begin;
    a.V_shard = Vs;
    a.max_rows = max_target_rows;
    a.draft_stride = draft_stride;
    a.ws = workspace;
    return SPEC_OK;
}

}  // namespace

int spec_shard_final_mass(const void *target_shard, const void *draft_shard, int dtype,
                          int32_t B, int32_t v_begin, int32_t v_end, int64_t max_target_rows,
                          int32_t draft_stride, spec_shard_mass *out_mass, void *workspace,
                          size_t ws_bytes, spec_stream_t stream)
{
    sv::ShardDrawArgs a{};
    int st = shard_draw_args(target_shard, draft_shard, dtype, B, v_begin, v_end, max_target_rows,
                             draft_stride, workspace, ws_bytes, a);
    if (st != SPEC_OK || B == 0)
        return st;
    if (!out_mass)
        return SPEC_ERR_INVALID_ARG;
    a.out_mass = out_mass;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_shard_mass(a, (cudaStream_t)stream, tr));
}

int spec_shard_final_draw(const void *target_shard, const void *draft_shard, int dtype,
                          const spec_shard_mass *mass_all, int32_t n_shards, int32_t shard,
                          int32_t B, int32_t v_begin, int32_t v_end, int64_t max_target_rows,
                          int32_t draft_stride, const float *u_final, int32_t *out_tokens,
                          void *workspace, size_t ws_bytes, spec_stream_t stream)
{
    if (n_shards < 1 || n_shards > sv::kMaxShards || shard < 0 || shard >= n_shards)
        return SPEC_ERR_INVALID_ARG;
    sv::ShardDrawArgs a{};
    int st = shard_draw_args(target_shard, draft_shard, dtype, B, v_begin, v_end, max_target_rows,
                             draft_stride, workspace, ws_bytes, a);
    if (st != SPEC_OK || B == 0)
        return st;
    if (!mass_all || !u_final || !out_tokens)
        return SPEC_ERR_INVALID_ARG;
    a.mass_all = mass_all;
    a.n_shards = n_shards;
    a.shard = shard;
    a.u_final = u_final;
    a.out_tokens = out_tokens;
    sv::Tracer tr = make_tracer();
    return cuda_status(sv::launch_shard_draw(a, (cudaStream_t)stream, tr));
}

int spec_get_device_status(void *workspace, spec_stream_t stream)
{
    if (!workspace)
        return SPEC_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t word = 0;
    unsigned char *status = static_cast<unsigned char *>(workspace) + sv::ws_layout(0, 0, 0).status;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (cudaMemcpyAsync(&word, status, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof word, s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (word & sv::ST_TIMEOUT)
        return SPEC_ERR_TIMEOUT;
    if (word & sv::ST_INVALID)
        return SPEC_ERR_INVALID_ARG;
    if (word & sv::ST_NONFINITE)
        return SPEC_ERR_NONFINITE;
    return SPEC_OK;
}

const char *spec_status_string(int status)
{
    switch (status) {
    case SPEC_OK:
        return "ok";
    case SPEC_ERR_INVALID_ARG:
        return "invalid argument (or malformed offsets / token id on the device)";
    case SPEC_ERR_WORKSPACE:
        return "workspace missing or too small";
    case SPEC_ERR_CUDA:
        return "CUDA runtime error";
    case SPEC_ERR_NONFINITE:
        return "NaN or +inf logit, or a row with every entry masked";
    case SPEC_ERR_TIMEOUT:
        return "a bounded wait for an asynchronous copy expired";
    default:
        return "unknown status";
    }
}

int spec_set_trace(void *const *events, int n_events)
{
    if (n_events < 0 || n_events > kMaxTraceEvents || (n_events > 0 && !events))
        return SPEC_ERR_INVALID_ARG;
    for (int k = 0; k < n_events; ++k)
        g_trace[k] = static_cast<cudaEvent_t>(events[k]);
    g_trace_n = n_events;
    return SPEC_OK;
}

int64_t spec_kernel_launch_count(void) { return g_launches; }

int spec_test_expire_wait(int64_t unit)
{
    if (unit < -1)
        return SPEC_ERR_INVALID_ARG;
    g_expire_unit = (uint64_t)(unit + 1);
    return SPEC_OK;
}

}  // extern "C"
