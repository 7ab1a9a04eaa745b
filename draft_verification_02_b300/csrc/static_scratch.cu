// static_scratch.cu - spec_verify_sample_static: sampling (or greedy)
// verification whose scratch memory is a fixed array compiled into this
// library instead of a caller-provided workspace.
//
// Why: some callers cannot allocate device memory at all.  A serving engine
// that has handed the whole HBM to its KV-cache pool, a plugin whose host
// runtime owns every device allocation, or a latency-critical loop where
// cudaMalloc would synchronise the device and stall other streams all need
// a call that touches only the buffers they pass in.  This entry point
// allocates nothing: its scratch is g_scratch below, which every GPU that
// loads the library holds until the process exits.
//
// The verification itself is spec_verify_sample's, unchanged; only where the
// workspace comes from differs.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "common.cuh"
#include "specverify.h"

namespace {

// The scratch every call on a device shares (its size is stated in the
// header as SPEC_STATIC_SCRATCH_BYTES).
static __device__ __align__(256) unsigned char g_scratch[SPEC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  In host code the name
// g_scratch is only a host-side stand-in, never a device address, so the
// address is looked up once per device (with that device current) and kept.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int spec_verify_sample_static(const void *target_logits, const void *draft_logits,
                                         int dtype, const int32_t *draft_tokens,
                                         const int32_t *cu_draft, int32_t B, int32_t V,
                                         int64_t max_target_rows, int32_t draft_stride,
                                         float temperature, const float *u_accept,
                                         const float *u_final, int32_t *out_tokens,
                                         int32_t *out_accept_len, float *out_p, float *out_q,
                                         spec_stream_t stream)
{
    // Argument checks first, with nothing enqueued: without a workspace the
    // regular entry point returns SPEC_ERR_WORKSPACE exactly when every
    // argument is acceptable (and SPEC_OK for an empty batch).
    const int st = spec_verify_sample(target_logits, draft_logits, dtype, draft_tokens, cu_draft,
                                      B, V, max_target_rows, draft_stride, temperature, u_accept,
                                      u_final, out_tokens, out_accept_len, out_p, out_q, nullptr,
                                      0, stream);
    if (st != SPEC_ERR_WORKSPACE)
        return st;
    const size_t need = spec_workspace_size(B, max_target_rows, V);
    if (need == 0)
        return SPEC_ERR_INVALID_ARG;
    if (need > (size_t)SPEC_STATIC_SCRATCH_BYTES)
        return SPEC_ERR_WORKSPACE;  // these sizes need more scratch than the fixed array holds
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return SPEC_ERR_CUDA;
    // The array keeps the previous call's contents.  Its status word must
    // start at zero; the partials are written before they are read.
    const size_t header = sv::ws_layout(B, max_target_rows, V).part1;
    if (cudaMemsetAsync(scratch, 0, header, (cudaStream_t)stream) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return spec_verify_sample(target_logits, draft_logits, dtype, draft_tokens, cu_draft, B, V,
                              max_target_rows, draft_stride, temperature, u_accept, u_final,
                              out_tokens, out_accept_len, out_p, out_q, scratch,
                              SPEC_STATIC_SCRATCH_BYTES, stream);
}
