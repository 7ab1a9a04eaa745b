// launch.h - host-side interface between the C-ABI layer (api.cu) and the
// kernel launchers (verify.cu, dcut.cu).  Plain structs, no torch types.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// Kernel-boundary hook: records the caller's trace events and counts launches.
struct Tracer {
    cudaEvent_t const *events = nullptr;
    int n = 0;
    int next = 0;
    void begin(cudaStream_t s);
    void after_kernel(cudaStream_t s);
};

struct VerifyArgs {
    const void *target;
    const void *draft;  // nullptr for greedy
    int dtype;          // 0 = f32, 1 = bf16
    const int32_t *tokens;
    const int32_t *cu;
    int B;
    int V;
    int64_t max_rows;
    int draft_stride;
    double temperature;  // 0 = greedy
    const float *u_accept;
    const float *u_final;
    int32_t *out_tokens;
    int32_t *out_len;
    float *out_p;
    float *out_q;
    void *ws;
    uint64_t debug_item;  // test hook: 1 + the streaming unit whose wait reports expiry (0: off)
};

// Enqueue the verification kernels (two launches: the streaming pass and a finish kernel).
cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t stream, Tracer &tr);

struct DcutArgs {
    const float *conf;
    const int32_t *kmax;
    int B;
    int Kmax;
    int budget;
    float min_gain;
    int32_t *out_depth;
    int32_t *out_cu;
    float *out_expected;
    void *ws;
};

cudaError_t launch_dcut(const DcutArgs &a, cudaStream_t stream, Tracer &tr);

struct DcutCostArgs {
    const float *conf;
    const int32_t *kmax;
    int B;
    int Kmax;
    double max_cost;
    int32_t *out_depth;
    int32_t *out_cu;
    double *out_benefit;
    void *ws;
};

cudaError_t launch_dcut_cost(const DcutCostArgs &a, cudaStream_t stream, Tracer &tr);

struct ConfArgs {
    const void *draft;  // [B*Kmax][V]
    int dtype;
    const int32_t *tokens;
    const int32_t *kmax;
    int B;
    int Kmax;
    int V;
    double temperature;  // 0 = greedy
    float *out_conf;
    void *ws;
};

// Enqueue the streaming pass over the B*Kmax draft rows and the per-row
// confidence kernel (2 launches).
cudaError_t launch_confidence(const ConfArgs &a, cudaStream_t stream, Tracer &tr);

struct DraftArgs {
    const void *draft;  // [B*Kmax][V]
    int dtype;
    const int32_t *kmax;
    int B;
    int Kmax;
    int V;
    double temperature;  // 0 = greedy
    const float *u;      // [B*Kmax] (T > 0)
    int32_t *out_tokens;
    float *out_conf;
    void *ws;
};

// Enqueue the streaming pass over the B*Kmax draft rows and the drafting
// kernel (a cluster draw per row, or a warp argmax per row at T = 0).
cudaError_t launch_draft(const DraftArgs &a, cudaStream_t stream, Tracer &tr);

struct StatsArgs {
    const int32_t *accept_len;
    const int32_t *cu;
    int B;
    int Kmax;
    int32_t *out_reached;
    int32_t *out_accepted;
    float *out_mean;
    void *ws;
};

cudaError_t launch_acceptance_stats(const StatsArgs &a, cudaStream_t stream, Tracer &tr);

// Vocabulary-sharded verification (shard.cu): one shard's four steps.
constexpr int kMaxShards = 32;

struct ShardStatsArgs {
    VerifyArgs v;  // the shard's logits (v.V = its column count); no outputs
    int v_begin;   // global token of the shard's column 0
    void *out_rows;
};

struct ShardAcceptArgs {
    const void *rows_all;  // [n_shards][rows]
    int n_shards;
    const int32_t *begin;  // host, n_shards + 1
    const int32_t *tokens;
    const int32_t *cu;
    int B;
    int64_t max_rows;
    int draft_stride;
    double temperature;
    const float *u_accept;
    int32_t *out_tokens;
    int32_t *out_len;
    float *out_p;
    float *out_q;
    void *ws;
};

struct ShardDrawArgs {
    const void *target;
    const void *draft;
    int dtype;
    int B;
    int v_begin;
    int V_shard;
    int64_t max_rows;
    int draft_stride;
    void *out_mass;        // step 3
    const void *mass_all;  // step 4: [n_shards][B]
    int n_shards;
    int shard;
    const float *u_final;
    int32_t *out_tokens;
    void *ws;
};

size_t shard_ws_bytes(int B, int64_t max_rows);
bool shard_columns_ok(int V_shard, int dtype);  // the draw's slice table holds V_shard columns
cudaError_t launch_shard_stats(const ShardStatsArgs &a, cudaStream_t stream, Tracer &tr);
cudaError_t launch_shard_accept(const ShardAcceptArgs &a, cudaStream_t stream, Tracer &tr);
cudaError_t launch_shard_mass(const ShardDrawArgs &a, cudaStream_t stream, Tracer &tr);
cudaError_t launch_shard_draw(const ShardDrawArgs &a, cudaStream_t stream, Tracer &tr);

}  // namespace sv
