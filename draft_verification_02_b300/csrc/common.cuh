// common.cuh - device helpers shared by the verification and D-cut kernels:
// inline-PTX wrappers for mbarriers and 1-D TMA bulk copies (sm_90+ forms,
// compiled for sm_103a), a bounded mbarrier wait, NaN-propagating max and
// warp/block reductions, and the workspace layout.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kThreads = 256;  // threads per CTA of the row kernels
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDraft = 32;  // drafted tokens per request (one warp ballot)
constexpr int kMaxBatch = 4096;
constexpr int kDcutMaxCand = 8192;

constexpr int kMaxVocab = 1 << 23;  // largest V the calls accept
#ifndef SV_PIECE_BYTES
#define SV_PIECE_BYTES 4096  // largest unit of the streaming kernel
#endif
constexpr int kPieceBytesMax = SV_PIECE_BYTES;
constexpr int kMaxWorkers = 8192;  // warp workers of the streaming kernel

// Device status bits (the workspace status word).
enum : uint32_t { ST_INVALID = 1u, ST_NONFINITE = 2u, ST_TIMEOUT = 4u };

// Bounded waits give up after this many nanoseconds of %globaltimer.
#ifndef SV_WAIT_NS
#define SV_WAIT_NS 2000000000ull
#endif

// -------------------------------------------------------------------------
// workspace layout
// -------------------------------------------------------------------------

// One (row, segment) partial: softmax (m, s = s_hi + s_lo, a float-float
// sum of exp2((x - m) c)) or argmax (m = value, idx = index).
struct __align__(16) Partial {
    float m;
    int32_t idx;
    float s_hi;
    float s_lo;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: status word and offsets-valid flag (256 bytes; the status word
// must be zero before the first call and every call leaves it so) | stream
// partials, one per (row, warp) segment: at most rows + warps.  The partials
// are written before they are read in every call.
struct WsLayout {
    size_t status, part1, total;
};

inline WsLayout ws_layout(int B, int64_t max_rows, int V)
{
    (void)V;
    WsLayout L{};
    const int64_t rows = max_rows > 0 ? 2 * max_rows - B : 0;
    size_t off = 0;
    L.status = off;
    off += 256;
    L.part1 = off;
    off = align_up(off + (size_t)(max_rows > 0 ? rows + kMaxWorkers : 0) * sizeof(Partial), 256);
    L.total = off;
    return L;
}

// -------------------------------------------------------------------------
// PTX wrappers
// -------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make the initialised barrier visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> shared, completion signalled on `bar` (tx bytes).
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(phase)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `phase` of `bar` to complete, giving up after SV_WAIT_NS
// (the timer is read once every 64 polls, so a wait that completes soon
// costs no timer read).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t phase)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, phase))
            return true;
        if ((it & 63u) == 63u) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0)
                t0 = now;
            else if (now - t0 > SV_WAIT_NS)
                return false;
        }
    }
}

// Thread-block clusters: this CTA's rank, the split cluster barrier, and
// stores into another CTA's shared memory (at the address `local` has there).
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

__device__ __forceinline__ uint32_t cluster_addr(const void *local, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    return remote;
}

__device__ __forceinline__ void st_cluster_u32(const void *local, uint32_t rank, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr(local, rank)), "r"(v)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_u64(const void *local, uint32_t rank, uint64_t v)
{
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(cluster_addr(local, rank)), "l"(v)
                 : "memory");
}

// max that returns NaN when either input is NaN.
__device__ __forceinline__ float max_nan(float a, float b)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ float warp_max_nan(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide NaN-propagating max (kThreads threads, all participate).
__device__ __forceinline__ float block_max_nan(float v, float *scratch /* [kWarps] */)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max_nan(v);
    __syncthreads();
    if (lane == 0)
        scratch[warp] = v;
    __syncthreads();
    float r = scratch[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w)
        r = max_nan(r, scratch[w]);
    return r;
}

// -------------------------------------------------------------------------
// float-float arithmetic (no fp64 on the device: B300's fp64 rate is a
// small fraction of its fp32 rate)
// -------------------------------------------------------------------------

// A value hi + lo with |lo| <= ulp(hi) / 2.
struct ff {
    float hi, lo;
};

// Exact sum: s + e == a + b (Knuth's TwoSum).  The pair is the exact
// rounding of a + b, so it does not depend on the order of a and b.
__device__ __forceinline__ ff two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

// (a + b) renormalised, given |a| >= |b| or a == 0.
__device__ __forceinline__ ff fast_two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// Sum of two float-float values; ff_add(a, b) and ff_add(b, a) give the same
// bits.
__device__ __forceinline__ ff ff_add(ff a, ff b)
{
    const ff s = two_sum(a.hi, b.hi);
    const float lo = __fadd_rn(__fadd_rn(a.lo, b.lo), s.lo);
    return fast_two_sum(s.hi, lo);
}

// Product of a float-float value and a float.
__device__ __forceinline__ ff ff_mul(ff a, float f)
{
    const float p = __fmul_rn(a.hi, f);
    const float e = fmaf(a.hi, f, -p);
    return fast_two_sum(p, fmaf(a.lo, f, e));
}

__device__ __forceinline__ bool ff_gt(ff a, ff b)
{
    return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

__device__ __forceinline__ bool ff_le(ff a, ff b) { return !ff_gt(a, b); }

__device__ __forceinline__ ff ff_shfl_xor(ff v, int o)
{
    return {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}

__device__ __forceinline__ ff ff_shfl_up(ff v, int o)
{
    return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

// Warp sum; every lane gets the same bits (each butterfly step adds the same
// two values in either order).
__device__ __forceinline__ ff warp_sum_ff(ff v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = ff_add(v, ff_shfl_xor(v, o));
    return v;
}

// Element access for the two logit dtypes.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;  // per 16-byte vector
    __device__ __forceinline__ static float at(const float *p, int64_t k) { return p[k]; }
    __device__ __forceinline__ static float ld_global(const float *p, int64_t k)
    {
        return __ldg(p + k);
    }
    __device__ __forceinline__ static void unpack(const uint4 v, float (&f)[4])
    {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
};
template <> struct Elem<uint16_t> {  // bfloat16 bit patterns
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static float at(const uint16_t *p, int64_t k)
    {
        return __uint_as_float((uint32_t)p[k] << 16);
    }
    __device__ __forceinline__ static float ld_global(const uint16_t *p, int64_t k)
    {
        return __uint_as_float((uint32_t)__ldg(p + k) << 16);
    }
    __device__ __forceinline__ static void unpack(const uint4 v, float (&f)[8])
    {
        f[0] = __uint_as_float(v.x << 16);
        f[1] = __uint_as_float(v.x & 0xffff0000u);
        f[2] = __uint_as_float(v.y << 16);
        f[3] = __uint_as_float(v.y & 0xffff0000u);
        f[4] = __uint_as_float(v.z << 16);
        f[5] = __uint_as_float(v.z & 0xffff0000u);
        f[6] = __uint_as_float(v.w << 16);
        f[7] = __uint_as_float(v.w & 0xffff0000u);
    }
};

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits)
{
    atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t read_status(const uint32_t *status)
{
    return *(volatile const uint32_t *)status;
}

// Bounds checks of the debug build (compiled with -DSV_DEBUG): an index
// outside [0, n) of its buffer sets ST_INVALID and the access it guards is
// skipped.  In the normal build every check is the constant true.
#ifdef SV_DEBUG
__device__ __forceinline__ bool in_bounds(int64_t idx, int64_t n, uint32_t *status)
{
    if (idx >= 0 && idx < n)
        return true;
    atomicOr(status, ST_INVALID);
    return false;
}
#define SV_IN_BOUNDS(idx, n, status) ::sv::in_bounds((int64_t)(idx), (int64_t)(n), (status))
#else
#define SV_IN_BOUNDS(idx, n, status) true
#endif

}  // namespace sv
