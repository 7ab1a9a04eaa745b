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

// Unit size for a balanced split: U = rows * ceil(V / Q) units over P warps
// puts ceil(U / P) units on the busiest warp.  Q is a multiple of the
// 16-byte granule, at most kPieceBytesMax.  Every unit costs a warp the same
// instructions whatever its size (the unit loop is unrolled to the largest
// unit), so:
//  - a short pass (at most kShortPassUnits on the busiest warp at the best
//    Q) takes the largest Q with that fewest count: fewest units in all;
//  - a longer pass is bound by bytes and minimises the busiest warp's
//    elements plus a fixed cost per unit (SV_UNIT_COST), preferring larger Q.
// Measured on B300, streaming pass in us (the earlier rule: elements plus
// 64): 576 rows of V = 128000 at T = 1, padded drafts (11 units a warp)
// 36.45 -> 33.80; B = 16 at V = 151936 (7 a warp) 21.27 -> 19.40.  The
// largest Q for longer passes was slower: B = 128 at V = 151936, T = 0.7,
// 113.8 -> 114.1; B = 32, K = 16 at T = 0 (12 a warp) 33.9 -> 34.5.
#ifndef SV_UNIT_COST
#define SV_UNIT_COST 512
#endif
#ifndef SV_SHORT_PASS_UNITS
#define SV_SHORT_PASS_UNITS 11
#endif
constexpr int64_t kShortPassUnits = SV_SHORT_PASS_UNITS;

inline Geometry plan(int64_t rows_total, int64_t max_rows, int V, int elem, int P_max)
{
    Geometry g{};
    g.max_rows = max_rows;
    const int gran = 16 / elem;
    const int qmax = kPieceBytesMax / elem;
    const int64_t total = rows_total * (int64_t)V;
    int64_t P = P_max;
    const int64_t min_work = 2048 / elem;  // at least ~2 KB per warp
    if (total / min_work < P)
        P = std::max<int64_t>(1, total / min_work);
    double best_cost = 1e300;
    int best_q = qmax, fewest_q = qmax;
    int64_t fewest = INT64_MAX;
    for (int q = qmax; q >= gran && q >= qmax / 8; q -= gran) {
        const int64_t cpr = (V + q - 1) / q;
        const int64_t U = rows_total * cpr;
        const int64_t per = (U + P - 1) / P;
        const double cost = (double)per * (double)(std::min<int64_t>(q, V) + SV_UNIT_COST);
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best_q = q;
        }
        if (per < fewest) {
            fewest = per;
            fewest_q = q;
        }
    }
    if (fewest <= kShortPassUnits)
        best_q = fewest_q;
    g.Q = std::min(best_q, ((V + gran - 1) / gran) * gran);
    g.cpr = (V + g.Q - 1) / g.Q;
    g.U = rows_total * (int64_t)g.cpr;
    g.P = (int)std::min<int64_t>(P, g.U);
    g.slots = rows_total - max_rows;
    g.nt = max_rows;
    return g;
}

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
    int ncl;    // CTAs per request (cluster size) in the final draw: 4, 8 or 16
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
