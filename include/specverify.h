/*
 * specverify.h - C ABI of the B300 (sm_103a) batched draft-verification
 * library: lossless rejection-sampling verification of drafted tokens, greedy
 * verification at T = 0, and D-cut's batch-level allocation of verification
 * depth.
 *
 * What the calls compute
 * ----------------------
 * Speculative decoding has a cheap drafter propose several tokens; the target
 * model scores the whole drafted block in one forward pass and rejection
 * sampling keeps the accepted prefix plus one extra token ("Tencent Hunyuan
 * Turns Speculative Decoding Into a Full Open-Source Stack", section "What
 * problem does it solve").  The accepted length is the number of drafted
 * tokens approved before the first mismatch ("Tencent rilascia AngelSpec in
 * open source ...", section "Come AngelSpec rende DFly piu selettivo"), and
 * the procedure is lossless: its output law is the target's ("Tencent ...
 * AngelSpec ...", section "Qu'est-ce que le speculative decoding").  The pages
 * do not write the accept/reject formulas; these calls use the standard ones
 * (Leviathan, Kalman & Matias 2023, "Fast Inference from Transformers via
 * Speculative Decoding", section "Speculative Sampling").
 *
 * Layout (all calls)
 * ------------------
 * B requests.  Request i verifies K_i drafted tokens (0 <= K_i <= 32).
 * cu_draft[B+1] (device, int32): cu_draft[0] = 0, cu_draft[i+1] = cu_draft[i] + K_i.
 * Target row j of request i (j = 0..K_i; j = K_i is the bonus row) is row
 *   cu_draft[i] + i + j of target_logits[rows][V] (row-major, stride V).
 * Draft index of (i, j), j < K_i:
 *   draft_stride == 0 (packed): cu_draft[i] + j
 *   draft_stride  > 0 (padded): i * draft_stride + j   (requires K_i <= draft_stride)
 * draft_tokens, draft_logits rows, u_accept, out_p and out_q use the draft index.
 * out_tokens uses the target-row index: out_tokens[cu_draft[i] + i + j] for j = 0..K_i
 * holds the accepted drafts (j < a_i), the final token (j = a_i) and -1 after it.
 *
 * Buffers
 * -------
 * Every pointer is caller-owned DEVICE memory; the library allocates nothing.
 * max_target_rows is a host-known upper bound on cu_draft[B] + B (it sizes
 * the grids, so cu_draft may be produced on the device, e.g. by
 * dcut_allocate, with no host round trip).  target_logits must be readable
 * for max_target_rows rows and out_tokens writable for max_target_rows
 * entries; a packed draft side must be readable for max_target_rows - B rows,
 * a padded one for B * draft_stride rows.  Rows past cu_draft[B] + B may be
 * read (their values are ignored) and are never written.
 * Logits are float32 (SPEC_F32) or bfloat16 (SPEC_BF16); -inf marks a
 * masked vocabulary entry; NaN and +inf are errors.  Pointers should be
 * 16-byte aligned and V * element size a multiple of 16 for the fast TMA
 * path; other shapes run a slower plain-load path with the same results.
 *
 * Streams and errors
 * ------------------
 * Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and returns without synchronising.  Argument errors are returned
 * before anything is enqueued.  Data-dependent errors (NaN/+inf logits, a
 * row with every entry masked, a drafted token outside [0, V), malformed
 * cu_draft, a bounded wait that expired) set a status word inside the
 * workspace and poison the affected outputs (tokens -1, accepted length
 * -1); spec_get_device_status reads and clears that word.  A bounded wait
 * gives up after about two seconds; the kernel then stops copying and
 * returns, and every output of that call is unspecified (some are poisoned).
 * After SPEC_ERR_TIMEOUT, zero the workspace again (spec_workspace_init).
 *
 * Workspace
 * ---------
 * spec_workspace_size(B, max_target_rows, V) bytes of device memory,
 * zero-filled once before first use (spec_workspace_init does this); every
 * call leaves it ready for the next.  One workspace serves one stream at a
 * time: calls on different streams need different workspaces.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *spec_stream_t;

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = -1, /* bad argument, or (device) malformed offsets / token id */
    SPEC_ERR_WORKSPACE = -2,   /* workspace missing or smaller than spec_workspace_size */
    SPEC_ERR_CUDA = -3,        /* a CUDA runtime call or kernel launch failed */
    SPEC_ERR_NONFINITE = -4,   /* (device) NaN or +inf logit, or a fully masked row */
    SPEC_ERR_TIMEOUT = -5      /* (device) a bounded wait for a copy expired */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* Largest K_i, B and B*Kmax the calls accept. */
#define SPEC_MAX_DRAFT 32
#define SPEC_MAX_BATCH 4096
#define SPEC_DCUT_MAX_CANDIDATES 8192

/*
 * Bytes of workspace needed by spec_verify_greedy / spec_verify_sample for up
 * to B requests, max_target_rows target rows and vocabulary V (either dtype),
 * and by dcut_allocate (any B, V = 0).  Returns 0 for invalid sizes.
 */
size_t spec_workspace_size(int32_t B, int64_t max_target_rows, int32_t V);

/* Zero-fill a workspace (enqueued on stream).  Needed once before first use. */
int spec_workspace_init(void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * Greedy verification (T = 0).  g_j = lowest index of the maximum of target
 * row j; draft j is accepted iff draft_tokens[j] == g_j; a_i = first mismatch
 * (K_i if none); the final token is g_{a_i} (the bonus row's argmax when every
 * draft is accepted).  Draft logits are not read.  Two kernel launches.
 * Pages: greedy acceptance rates "at T = 0" ("Tencent ... AngelSpec ...",
 * bullet list); ties to the lowest index is this library's reading.
 *
 *   target_logits  [max_target_rows][V]  f32 or bf16 (dtype)
 *   draft_tokens   draft index -> int32 token id
 *   out_tokens     int32 [max_target_rows]
 *   out_accept_len int32 [B]: a_i
 */
int spec_verify_greedy(const void *target_logits, int dtype, const int32_t *draft_tokens,
                       const int32_t *cu_draft, int32_t B, int32_t V, int64_t max_target_rows,
                       int32_t draft_stride, int32_t *out_tokens, int32_t *out_accept_len,
                       void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * Sampling verification (T > 0).  With p_j = softmax(target row j / T) and
 * q_j = softmax(draft row j / T):
 *   accept draft j iff u_accept[j] < p_j(x_j) / q_j(x_j)  (q_j(x_j) = 0: iff p_j(x_j) > 0)
 *   a_i = first rejected position (K_i if none)
 *   final weights w = max(0, p_a - q_a) after a rejection (w = p_a if that is
 *   all zero), w = p_{K_i} (bonus row) when every draft is accepted;
 *   final token = smallest v with sum_{v' <= v} w(v') > u_final[i] * sum(w).
 * out_p / out_q (draft index, may be NULL) receive p_j(x_j) and q_j(x_j) for
 * every j < K_i.  temperature == 0 runs spec_verify_greedy (out_p/out_q are
 * then left untouched).  Two kernel launches: a streaming pass over every
 * target and draft row, then a per-request pass (accept test, first
 * rejection, final draw) launched as its programmatic dependent.
 *
 *   draft_logits  [draft rows][V], same dtype as target_logits
 *   u_accept      float [draft index] in [0,1)
 *   u_final       float [B] in [0,1)
 */
int spec_verify_sample(const void *target_logits, const void *draft_logits, int dtype,
                       const int32_t *draft_tokens, const int32_t *cu_draft, int32_t B,
                       int32_t V, int64_t max_target_rows, int32_t draft_stride,
                       float temperature, const float *u_accept, const float *u_final,
                       int32_t *out_tokens, int32_t *out_accept_len, float *out_p,
                       float *out_q, void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * D-cut: batch-level allocation of verification depth under a total
 * verify-token budget.  The pages describe D-cut as treating verification
 * capacity as a batch-level shared resource, weighing the expected value of
 * keeping more positions against their cost and sending depth to
 * high-confidence prefixes ("Tencent rilascia AngelSpec in open source ...",
 * "Come AngelSpec rende DFly piu selettivo"; "Tencent Hunyuan Turns
 * Speculative Decoding ...", "What problem does it solve", inference layer).
 *
 * conf[i*Kmax + j] in [0,1] (j < kmax[i]) is request i's confidence in its
 * drafted token j.  P_{i,d} = conf[i][0] * ... * conf[i][d-1] (fp32, left to
 * right).  All (i, d) are ranked by P descending, ties by request then depth
 * ascending; the first min(budget, #{P >= min_gain}) are kept.  out_depth[i]
 * = number kept for request i (always a prefix), out_cu = exclusive prefix
 * sum of out_depth (feeds cu_draft of the verify call; target rows needed =
 * budget + B at most), out_expected_len[i] = sum_{d <= depth_i} P_{i,d}
 * (may be NULL).  The bonus row of every request is always verified and is
 * not counted against the budget.  Invalid confidences set
 * SPEC_ERR_INVALID_ARG on the device and write -1 depths and offsets.
 * One kernel launch (one CTA).  Requires B * Kmax <= SPEC_DCUT_MAX_CANDIDATES.
 */
int dcut_allocate(const float *conf, const int32_t *kmax, int32_t B, int32_t Kmax,
                  int32_t budget, float min_gain, int32_t *out_depth, int32_t *out_cu,
                  float *out_expected_len, void *workspace, size_t ws_bytes,
                  spec_stream_t stream);

/*
 * D-cut in latency-cost units: the scheduling policy that "Tencent AngelSpec
 * Speculative Decoding Framework Deep Dive: MTP + Block Diffusion Dual-Draft
 * Strategy and D-cut High-Concurrency Throughput Optimization" gives in its
 * D-cut section.  cost(d) is the piecewise-linear function through the
 * profiled latency table {1: 1.0, 2: 1.2, 4: 1.5, 8: 2.0, 16: 3.0},
 * constant outside [1, 16].  Request i (kmax[i] >= 1) takes the depth d in 1..kmax[i]
 * maximising benefit(d) = (conf[i][0] * ... * conf[i][d-1]) * d / cost(d)
 * (the first such d); requests are then taken in decreasing benefit (ties by
 * request) and admitted while the running total of their costs stays within
 * max_cost, skipping any that would exceed it.  out_depth[i] = the chosen
 * depth if admitted, else 0 (only its bonus row is verified); out_cu as in
 * dcut_allocate; out_benefit[i] (fp64, may be NULL) = the admitted
 * request's benefit, else 0.  All arithmetic is fp64 (the page computes in
 * Python floats), each operation rounded once, so the depths are those of a
 * plain sequential fp64 evaluation.  Invalid confidences or kmax set
 * SPEC_ERR_INVALID_ARG on the device and write -1 depths and offsets.  One
 * kernel launch (one cluster of 8 CTAs); B <= SPEC_MAX_BATCH.
 */
int dcut_allocate_cost(const float *conf, const int32_t *kmax, int32_t B, int32_t Kmax,
                       double max_cost, int32_t *out_depth, int32_t *out_cu,
                       double *out_benefit, void *workspace, size_t ws_bytes,
                       spec_stream_t stream);

/*
 * Prefix confidence of drafted tokens, the input D-cut ranks: D-cut moves
 * verification depth by per-request prefix confidence ("Tencent Hunyuan
 * Turns Speculative Decoding Into a Full Open-Source Stack", "What problem
 * does it solve", inference layer).  This library's reading: the confidence
 * of drafted token x_{i,j} is the drafter's own probability of it,
 *   out_conf[i*Kmax + j] = softmax(draft row i*Kmax + j / T)(x_{i,j})   j < kmax[i]
 *   out_conf[i*Kmax + j] = 0                                            j >= kmax[i]
 * and at T == 0 (a greedy drafter) 1 when x_{i,j} is the row's lowest-index
 * maximum, else 0.  The output feeds dcut_allocate's conf directly (same
 * [B][Kmax] layout).
 *
 *   draft_logits  [B*Kmax][V] f32 or bf16, padded: row i*Kmax + j (every row
 *                 is read, also those past kmax[i])
 *   draft_tokens  int32 [B*Kmax], kmax int32 [B] (device)
 *   out_conf      float [B*Kmax]
 * A workspace of spec_workspace_size(B, B * (Kmax + 1), V) bytes suffices.
 * A failing row (NaN / +inf / all masked, or a token outside [0, V)) gets
 * NaN and sets the device status; kmax outside [0, Kmax] is
 * SPEC_ERR_INVALID_ARG on the device.  Two kernel launches: the streaming
 * pass over the B*Kmax rows and a per-row kernel, its programmatic dependent.
 */
int spec_draft_confidence(const void *draft_logits, int dtype, const int32_t *draft_tokens,
                          const int32_t *kmax, int32_t B, int32_t Kmax, int32_t V,
                          float temperature, float *out_conf, void *workspace, size_t ws_bytes,
                          spec_stream_t stream);

/*
 * The drafter's own step: draw the drafted tokens from its logits (the step
 * before verification: a lightweight drafter proposes the candidate tokens
 * that the target then checks, "Tencent Hunyuan Turns Speculative Decoding
 * Into a Full Open-Source Stack", "What problem does it solve").  For row
 * r = i*Kmax + j with j < kmax[i], q = softmax(draft row r / T) and
 *   out_tokens[r] = the smallest v with C(v) > u_draft[r] * S   (T > 0)
 *   out_tokens[r] = the row's lowest-index maximum                (T == 0)
 * where C is the running sum of the unnormalised weights 2^((x - m) log2(e)/T)
 * over the vocabulary and S its total (the same inverse-CDF reading as the
 * final draw of spec_verify_sample); out_conf[r] = q(out_tokens[r]) (1 at
 * T == 0), which is the input of dcut_allocate for a drafter that samples.
 * Rows j >= kmax[i] give -1 and 0.
 *
 *   draft_logits  [B*Kmax][V] f32 or bf16, padded (every row is read)
 *   kmax          int32 [B], u_draft float [B*Kmax] in [0, 1) (T > 0; may be
 *                 NULL at T == 0), out_tokens int32 [B*Kmax], out_conf float
 *                 [B*Kmax]; all device pointers
 * A workspace of spec_workspace_size(B, B * (Kmax + 1), V) bytes suffices.
 * A row with NaN / +inf / no finite logit gives -1 and NaN and sets
 * SPEC_ERR_NONFINITE on the device; kmax outside [0, Kmax] sets
 * SPEC_ERR_INVALID_ARG there.  A draw near a CDF boundary may differ from an
 * exact-arithmetic draw by one token (fp32 weights; the float-float running
 * sums keep the error near 1e-7 of S).  T > 0: one kernel launch, one CTA
 * per row that reads the row once, slice by slice (each slice weighed
 * against its own power-of-two reference; the slice holding u*S is weighed
 * again from L2 and walked).  T == 0: two launches, the streaming pass over
 * the B*Kmax rows and a per-row argmax merge, its programmatic dependent.
 */
int spec_draft_sample(const void *draft_logits, int dtype, const int32_t *kmax, int32_t B,
                      int32_t Kmax, int32_t V, float temperature, const float *u_draft,
                      int32_t *out_tokens, float *out_conf, void *workspace, size_t ws_bytes,
                      spec_stream_t stream);

/*
 * The acceptance statistics the pages report per drafter: mean accepted
 * length and acceptance by draft position ("Tencent Hunyuan Turns
 * Speculative Decoding Into a Full Open-Source Stack", "Five angles worth a
 * closer look", item 4: read from the serving engine during training; the
 * French/Russian page's table of acceptance rates by position at T = 0).
 * From one verification call's outputs (accept_len = out_accept_len, cu_draft
 * its offsets), over the requests with accept_len[i] >= 0:
 *   out_reached[j]  = #{ i : K_i > j and a_i >= j }   position j was tested
 *   out_accepted[j] = #{ i : a_i > j }                 and accepted
 *   *out_mean       = sum a_i / #requests (0 with no request), fp32
 * for j < Kmax; the per-position rate is accepted[j] / reached[j].  A request
 * with a_i > K_i or K_i > Kmax sets SPEC_ERR_INVALID_ARG on the device and
 * every output to -1 (mean NaN).  All pointers are device pointers; only the
 * workspace's status word is used (any workspace from spec_workspace_size
 * will do).  One kernel launch (one CTA); B <= SPEC_MAX_BATCH.
 */
int spec_acceptance_stats(const int32_t *accept_len, const int32_t *cu_draft, int32_t B,
                          int32_t Kmax, int32_t *out_reached, int32_t *out_accepted,
                          float *out_mean, void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * Vocabulary-sharded verification
 * -------------------------------
 * A target served tensor-parallel splits its output projection by vocabulary
 * (TP = 8 in "Tencent Hunyuan Turns Speculative Decoding Into a Full
 * Open-Source Stack", section "Key numbers (Hy3-295B-A21B, TP=8)"), so each
 * rank holds the logits of one contiguous vocabulary range, and so may the
 * drafter.  These calls verify such a batch without gathering any logit row:
 * each rank reduces its own columns, and only small per-row and per-request
 * records cross ranks.  The results are those of spec_verify_sample /
 * spec_verify_greedy on the whole vocabulary (same layout, same outputs; the
 * merges round differently, within the same accuracy).
 *
 * N shards, shard r holding global tokens [shard_begin[r], shard_begin[r+1])
 * (shard_begin[0] = 0, strictly increasing, shard_begin[N] = V, N <= 32).
 * Shard r's logits are target_shard[max_target_rows][V_r] (and draft_shard)
 * with V_r = shard_begin[r+1] - shard_begin[r]: column c is token
 * shard_begin[r] + c.  Offsets, drafted tokens and uniforms are the same on
 * every shard.  One verification is, on every shard, in this order:
 *   1. spec_shard_row_stats      -> this shard's row records
 *      (exchange: gather the N shards' records, shard order, on every shard)
 *   2. spec_shard_accept          -> accepted lengths, accepted tokens, p, q
 *      T = 0: the verification is complete here.
 *   3. spec_shard_final_mass      -> this shard's share of the final draw's mass
 *      (exchange: gather the N shards' masses, shard order)
 *   4. spec_shard_final_draw      -> the final token where this shard holds it
 *      (exchange: element-wise max of out_tokens over the shards)
 * Every shard computes step 2 and the choice of the drawing shard in step 4
 * from the same gathered bytes with the same code, so all shards agree
 * bit for bit without further exchange.  The four calls of one
 * verification use one shard workspace (spec_shard_workspace_size), which
 * carries the accepted positions and the draw's constants from step 2 to
 * steps 3 and 4; no other call may use it in between.  Device errors go to
 * that workspace's status word as for spec_verify_sample (read it with
 * spec_get_device_status).  Data errors are poisoned identically on every
 * shard, since they are seen in the gathered records; an expired wait is
 * seen only by the shard it happened on, so after SPEC_ERR_TIMEOUT on any
 * shard every output of that verification is unspecified.
 */

/* One row's record from one shard (16 bytes; exchanged as raw bytes).
 *   T > 0: m = maximum of the shard's logits in the row, s_hi + s_lo = sum
 *          over the shard of 2^((l - m) log2(e) / T) (a float-float pair),
 *          x.gx = the logit at the row's drafted token when this shard holds
 *          that token (0 otherwise).  NaN or +inf in the row make m or s NaN.
 *   T = 0: m = maximum, x.arg = global index of its lowest occurrence (-1
 *          when every entry is -inf, -2 when the row holds a NaN), s = 0. */
typedef struct {
    float m;
    union {
        float gx;
        int32_t arg;
    } x;
    float s_hi, s_lo;
} spec_shard_row;

/* One request's share of the final draw's mass on one shard (16 bytes):
 * w = sum over the shard's columns of the final weights (max(0, p - q) after
 * a rejection, else the unnormalised p of the bonus row); p = the same sum
 * of the unnormalised p (kept for the all-zero residual, where the draw
 * falls back to p).  Float-float pairs. */
typedef struct {
    float w_hi, w_lo, p_hi, p_lo;
} spec_shard_mass;

/* Workspace bytes for one shard of V_shard columns (0 for invalid sizes);
 * zero-fill it once before first use (spec_workspace_init). */
size_t spec_shard_workspace_size(int32_t B, int64_t max_target_rows, int32_t V_shard);

/* Records per shard: max_target_rows target rows, then the draft rows
 * (max_target_rows - B packed, or B * draft_stride padded), by draft index.
 * Records of rows past cu_draft[B] + B (and of padding rows) are not written. */
int64_t spec_shard_row_count(int32_t B, int64_t max_target_rows, int32_t draft_stride);

/*
 * Step 1: this shard's record of every target row and (T > 0) every draft
 * row.  Reads this shard's logits once (the streaming pass of
 * spec_verify_sample over V_r columns) and merges each row.  Two launches.
 *   out_rows  spec_shard_row [spec_shard_row_count(B, max_target_rows, draft_stride)]
 */
int spec_shard_row_stats(const void *target_shard, const void *draft_shard, int dtype,
                         const int32_t *draft_tokens, const int32_t *cu_draft, int32_t B,
                         int32_t v_begin, int32_t v_end, int64_t max_target_rows,
                         int32_t draft_stride, float temperature, spec_shard_row *out_rows,
                         void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * Step 2: merge the N shards' records of each row (in shard order), run the
 * accept test and the first-rejection scan, and write out_accept_len,
 * out_p / out_q (T > 0; may be NULL) and out_tokens except each request's
 * final position (T > 0: -1 there until step 4).  T = 0 writes the final
 * token too (the merged argmax).  One launch.
 *   rows_all     spec_shard_row [N][spec_shard_row_count(...)], shard r's block r
 *   shard_begin  HOST int32 [N + 1]
 */
int spec_shard_accept(const spec_shard_row *rows_all, int32_t n_shards,
                      const int32_t *shard_begin, const int32_t *draft_tokens,
                      const int32_t *cu_draft, int32_t B, int64_t max_target_rows,
                      int32_t draft_stride, float temperature, const float *u_accept,
                      int32_t *out_tokens, int32_t *out_accept_len, float *out_p, float *out_q,
                      void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * Step 3 (T > 0): this shard's share of each request's final-draw mass, from
 * the final rows' columns it holds (the target row a_i and, after a
 * rejection, the draft row a_i).  Requests that step 2 poisoned get zero
 * mass.  One launch.
 *   out_mass  spec_shard_mass [B]
 */
int spec_shard_final_mass(const void *target_shard, const void *draft_shard, int dtype,
                          int32_t B, int32_t v_begin, int32_t v_end, int64_t max_target_rows,
                          int32_t draft_stride, spec_shard_mass *out_mass, void *workspace,
                          size_t ws_bytes, spec_stream_t stream);

/*
 * Step 4 (T > 0): S = the sum of the N shards' w masses in shard order (the
 * p masses when every w is zero after a rejection); the shard whose range
 * holds u_final[i] * S finds the token by the inverse CDF over its columns
 * and writes it (a global token id) at out_tokens[cu_draft[i] + i + a_i];
 * every other shard writes -1 there.  One launch.
 *   mass_all  spec_shard_mass [N][B], shard r's block r
 *   shard     this shard's index r
 */
int spec_shard_final_draw(const void *target_shard, const void *draft_shard, int dtype,
                          const spec_shard_mass *mass_all, int32_t n_shards, int32_t shard,
                          int32_t B, int32_t v_begin, int32_t v_end, int64_t max_target_rows,
                          int32_t draft_stride, const float *u_final, int32_t *out_tokens,
                          void *workspace, size_t ws_bytes, spec_stream_t stream);

/*
 * spec_verify_sample without a workspace, for callers that cannot allocate
 * device memory: an engine whose memory pool already owns all of HBM (for
 * its KV cache), a plugin whose host runtime forbids allocations outside its
 * own allocator, or a loop that must not risk the device-wide
 * synchronisation cudaMalloc can cause.  The pages have no counterpart: this
 * is a deployment convenience of this library.
 *
 * Same arguments, results and kernels as spec_verify_sample (T == 0 runs the
 * greedy verification), minus workspace/ws_bytes.  The scratch is one
 * file-scope device array of SPEC_STATIC_SCRATCH_BYTES bytes inside the
 * library; every GPU that loads the library holds it until the process
 * exits.  The call allocates nothing: it enqueues a memset of the array's
 * status word and request tickets, then the two verification kernels.
 *  - Returns SPEC_ERR_WORKSPACE, with nothing enqueued, when
 *    spec_workspace_size(B, max_target_rows, V) > SPEC_STATIC_SCRATCH_BYTES.
 *  - The first call on each device looks up the array's device address
 *    (with that device current) and keeps it for the life of the process;
 *    make that first call before any stream capture.  A device reset
 *    (cudaDeviceReset) discards the context that address belongs to: after
 *    one, this entry point must not be called again in the same process.
 *  - Every call on a device shares the one array, and it keeps the previous
 *    call's contents: calls that may overlap on the GPU (different streams,
 *    or concurrent host threads) race and must be serialised by the caller.
 *  - The device status word lives in the array and is cleared by the next
 *    call; data errors show as poisoned outputs (accepted length -1).
 */
#define SPEC_STATIC_SCRATCH_BYTES (1 << 20)
int spec_verify_sample_static(const void *target_logits, const void *draft_logits, int dtype,
                              const int32_t *draft_tokens, const int32_t *cu_draft, int32_t B,
                              int32_t V, int64_t max_target_rows, int32_t draft_stride,
                              float temperature, const float *u_accept, const float *u_final,
                              int32_t *out_tokens, int32_t *out_accept_len, float *out_p,
                              float *out_q, spec_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the workspace status word.
 * Returns SPEC_OK or the device-side error (SPEC_ERR_TIMEOUT before
 * SPEC_ERR_INVALID_ARG before SPEC_ERR_NONFINITE when several are set).
 */
int spec_get_device_status(void *workspace, spec_stream_t stream);

/* Static description of a status code. */
const char *spec_status_string(int status);

/*
 * Optional timing hook for benchmarks.  After spec_set_trace(events, n) the
 * calling thread's subsequent calls record events[0] (a cudaEvent_t) on the
 * stream before their first kernel and events[k] after their k-th kernel
 * (k < n).  spec_set_trace(NULL, 0) turns it off.  Thread-local.
 */
int spec_set_trace(void *const *events, int n_events);

/* Number of kernels the calling thread has launched through this library. */
int64_t spec_kernel_launch_count(void);

/*
 * Test hook for the timeout path; never needed in production (unit = -1,
 * the default, turns it off).  The streaming pass of spec_verify_sample /
 * spec_verify_greedy reads the rows in units (pieces of at most 4 KB, each
 * one 1-D bulk copy), numbered from 0 in row order.  After
 * spec_test_expire_wait(unit), the calling thread's later verification calls
 * treat the bounded wait for that unit's copy as expired once the copy has
 * landed: the warp holding it flags SPEC_ERR_TIMEOUT, waits for its other
 * copies in flight and stops, and every output of the call is unspecified
 * (the ones the kernels reach are poisoned).  Thread-local.
 */
int spec_test_expire_wait(int64_t unit);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
