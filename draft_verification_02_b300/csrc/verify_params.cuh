// verify_params.cuh - what the two verification kernels share: their
// parameter blocks and small device helpers (PDL control, 2^x, bf16
// unpacking, the draft index, the rounding fix of fl(m c)).
#pragma once

#include <algorithm>
#include <cfloat>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace sv {

// ---------------------------------------------------------------------------
// parameters
// ---------------------------------------------------------------------------

// The unit split of kernel 1, needed by kernel 2 to find partials.  Rows
// are numbered in one index space: target rows [0, nt), then draft slots
// (draft slot s is row nt + s); units run through it in order.
struct Geometry {
    int64_t max_rows;  // target rows (host bound)
    int64_t U;         // units
    int cpr;           // units per row
    int Q;             // elements per unit (the last unit of a row may be shorter)
    int P;             // warp workers
    int64_t slots;     // draft slots of the host bound (max_rows - B at T > 0, else 0)
    int64_t nt;        // target rows of the index space (max_rows in the host's split)
};

struct StreamParams {
    const void *target;
    const void *draft;
    const int32_t *cu;
    int32_t *out_tokens;
    int32_t *out_len;
    int B, V;
    int64_t draft_slots;  // draft rows read (packed index space); 0 at T = 0
    int draft_stride;
    Geometry g;
    int tma;
    int piece_smem;  // bytes per ring slot (multiple of 128)
    float c;         // log2(e) / T
    uint32_t *status;
    uint32_t *cu_flag;
    Partial *part;
    int64_t part_cap;     // partials the workspace holds
    int64_t draft_rows;   // draft rows the draft side may index
    uint64_t debug_unit;  // test hook: the wait for unit debug_unit - 1 reports expiry (0: off)
};

struct FinishParams {
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
    int64_t draft_rows;  // rows the draft side may index
    int draft_stride;
    Geometry g;
    int ncl;    // CTAs per request (cluster size) in the final draw: 8 or 16
    int R;      // vocabulary entries per cluster CTA in the final draw
    int slice;  // entries of one row weighed at a time (multiple of 16 bytes)
    int pv;          // 16-byte vectors per thread piece of a slice (odd)
    int stage_smem;  // bytes per staged row slice (multiple of 128)
    int tma;         // rows 16-byte aligned: TMA bulk copies
    const int32_t *kmax;  // drafting only: rows per request that hold a draft
    int Kmax;             // drafting only: rows per request (padded)
    float *out_conf;      // drafting only: q(x) of each drawn token
    float c;
    uint32_t *status;
    const uint32_t *cu_flag;
    const Partial *part;
    int64_t part_cap;  // partials the workspace holds
};

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// 2^x on the SFU (PTX ex2.approx.ftz.f32); results below 2^-126 flush to 0.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The split over the rows that exist.  The host splits its bound (every
// target row up to max_rows, every draft slot); once the real count
// cu_total = cu_draft[B] is known, a looser bound is re-split over the real
// rows only (target rows [0, cu_total + B), then the cu_total draft slots),
// so that no warp is handed rows that do not exist.  Every kernel that reads
// the partials derives the same split from the same offsets.  (Malformed
// offsets are clamped here only to keep the split well formed; such a call
// is poisoned anyway.)
__device__ __forceinline__ Geometry real_split(Geometry g, int B, int cu_total)
{
    const int64_t v = cu_total < 0 ? 0 : cu_total;
    const int64_t nt = min(g.max_rows, v + B);
    const int64_t nd = min(g.slots, v);
    if (nt + nd < g.max_rows + g.slots) {
        g.nt = nt;
        g.U = (nt + nd) * (int64_t)g.cpr;
    }
    return g;
}

// Owner warp of unit u when warp w owns units [w*U/P, (w+1)*U/P).
__device__ __forceinline__ int owner_of(int64_t u, const Geometry &g)
{
    return (int)(((u + 1) * (int64_t)g.P - 1) / g.U);
}

// The unit sums use exp2(x*c - fl(m*c)) = exp2((x - m)*c) * 2^-(fl(m*c) - m*c);
// this returns the factor 2^(fl(m*c) - m*c) that undoes the rounding.  The
// rounding error fl(m*c) - m*c is exact as -fma(m, c, -fl(m*c)) and below
// 2^-17 in magnitude, so 1 + delta*ln2 is the factor to fp32 precision.
__device__ __forceinline__ float mc_correction(float m, float mc, float c)
{
    const float delta = -fmaf(m, c, -mc);
    return fmaf(delta, 0.69314718f, 1.0f);
}

__device__ __forceinline__ int64_t draft_index(int draft_stride, const int32_t *cu, int i, int j)
{
    return draft_stride > 0 ? (int64_t)i * draft_stride + j : (int64_t)__ldg(cu + i) + j;
}

// Enqueue kernel 1 alone for a verification call (verify.cu) and return its
// parameters (where the partials are, the unit geometry).
cudaError_t launch_stream_pass(const VerifyArgs &a, cudaStream_t s, Tracer &tr, StreamParams &sp);

}  // namespace sv
