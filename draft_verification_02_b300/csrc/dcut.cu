// dcut.cu - D-cut: batch-level allocation of verification depth, one CTA.
//
// D-cut treats target-verification capacity as a shared batch-level resource
// and moves depth to high-confidence prefixes ("Tencent rilascia AngelSpec in
// open source ...", "Come AngelSpec rende DFly piu selettivo"; "Tencent
// Hunyuan Turns Speculative Decoding Into a Full Open-Source Stack", "What
// problem does it solve", inference layer).  Reading used here: the budget is
// counted in verified draft tokens; the value of verifying request i to depth
// d is the prefix product P_{i,d} = conf_i0 * ... * conf_i(d-1) (the
// probability that the first d drafts are all accepted when conf is the
// conditional acceptance probability), so keeping the `budget` largest
// products over the whole batch maximises the expected number of accepted
// tokens; a product below `min_gain` is never worth its cost.
//
// Kernel: every candidate (i, d) becomes one 64-bit key
//   hi 32 bits: 0x3F800000 - bits(P)   (P in [0,1]: larger P -> smaller key)
//   lo 32 bits: i * Kmax + (d - 1)     (ties: lower request, then lower depth)
// The first keep = min(budget, #{P >= min_gain}) keys in key order are kept.
// No sort is needed: a most-significant-digit radix select (8 bits a pass,
// shared-memory histograms) finds the keep-th smallest key tau, and a request's
// depth is the number of its keys <= tau.  Keys are unique and ascend with d
// in every request (P never grows with d), so the kept keys are a prefix of
// every request and exactly keep in all.
#include <climits>
#include <cstdint>

#include <cstring>

#include "common.cuh"
#include "fp64_exact.cuh"
#include "launch.h"

namespace sv {

// threads of the D-cut CTA: its passes are barrier-bound, so fewer warps
// meet sooner (measured on B=64, Kmax=16: 256 threads 10.4 us traced,
// 512 10.7, 1024 11.0)
#ifndef SV_DCUT_THREADS
#define SV_DCUT_THREADS 256
#endif
constexpr int kDcutThreads = SV_DCUT_THREADS;

struct DcutParams {
    const float *conf;
    const int32_t *kmax;
    int B, Kmax, Kp, Bp;
    int budget;
    float min_gain;
    int32_t *out_depth;
    int32_t *out_cu;
    float *out_expected;
    uint32_t *status;
};

__device__ __forceinline__ int block_excl_scan_int(int v, int *warp_tot /* [32] */, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += n;
    }
    if (lane == 31)
        warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;  // fewer than 32 warps
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o)
                ti += n;
        }
        warp_tot[lane] = ti - t;  // exclusive offset of each warp
        if (lane == 31)
            warp_tot[32] = ti;
    }
    __syncthreads();
    total = warp_tot[32];
    return warp_tot[warp] + incl - v;
}

__global__ void __launch_bounds__(kDcutThreads) dcut_kernel(const DcutParams p)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    const int n = p.B * p.Kmax;         // candidate keys, stored position-major: [d][request]
    const int cs = p.Kmax | 1;          // odd row stride of the staged confidences: no bank conflicts
    uint64_t *keys = reinterpret_cast<uint64_t *>(dsm);
    int *depth_s = reinterpret_cast<int *>(keys + n);
    int *kmax_s = depth_s + p.B;
    float *conf_s = reinterpret_cast<float *>(kmax_s + p.B);  // [B][cs]
    __shared__ int hist[256];
    __shared__ int warp_tot[33];
    __shared__ int s_elig, s_bucket, s_below, s_count;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        s_elig = 0;
    // stage the inputs with coalesced loads (one round trip), then work from
    // shared memory
    for (int r = tid; r < p.B; r += kDcutThreads) {
        depth_s[r] = 0;
        kmax_s[r] = __ldg(p.kmax + r);
    }
    for (int k = tid; k < n; k += kDcutThreads)
        conf_s[(k / p.Kmax) * cs + k % p.Kmax] = __ldg(p.conf + k);
    __syncthreads();

    // 1. prefix products (fp32, left to right) -> keys; validate inputs.  A
    // key orders candidates by (P desc, request asc, depth asc): high word
    // 0x3F800000 - bits(P) (P in [0, 1]), low word request * Kmax + depth - 1;
    // a position past kmax gets a key above every real one.
    int bad = 0, elig = 0;
    for (int r = tid; r < p.B; r += kDcutThreads) {
        int km = kmax_s[r];
        if (km < 0 || km > p.Kmax) {
            bad = 1;
            km = 0;
        }
        float P = 1.f;
        for (int d = 1; d <= p.Kmax; ++d) {
            const uint64_t lo = (uint32_t)(r * p.Kmax + (d - 1));
            uint64_t key;
            if (d <= km) {
                float c = conf_s[r * cs + (d - 1)];
                if (!(c >= 0.f && c <= 1.f)) {
                    bad = 1;
                    c = 0.f;
                }
                P = __fadd_rn(__fmul_rn(P, c), 0.f);  // + 0 turns -0 into +0
                key = ((uint64_t)(0x3F800000u - __float_as_uint(P)) << 32) | lo;
                elig += P >= p.min_gain;
            } else {
                key = (0xFFFFFFFFull << 32) | lo;  // not a candidate
            }
            keys[(d - 1) * p.B + r] = key;
        }
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (tid == 0)
            set_status(p.status, ST_INVALID);
        for (int r = tid; r < p.B; r += kDcutThreads) {
            p.out_depth[r] = -1;
            if (p.out_expected)
                p.out_expected[r] = __int_as_float(0x7fc00000);
        }
        for (int r = tid; r <= p.B; r += kDcutThreads)
            p.out_cu[r] = -1;
        return;
    }
    if (elig)
        atomicAdd(&s_elig, elig);
    __syncthreads();

    // 2. the keep-th smallest key tau (keep = min(budget, eligible)) by a
    // most-significant-digit radix select, 8 bits a pass; it stops once the
    // keys sharing the digits found so far are exactly the ones still needed.
    // Keys are distinct, so exactly `keep` keys are <= tau, and since P never
    // grows with depth they are a prefix of every request.
    const int keep = min(p.budget, s_elig);
    uint64_t tau = 0;
    if (keep > 0) {
        uint64_t prefix = 0, mask = 0;
        int remaining = keep;  // rank of tau among the keys matching prefix
        tau = ~0ull;
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int q = tid; q < 256; q += kDcutThreads)
                hist[q] = 0;
            __syncthreads();
            for (int e = tid; e < n; e += kDcutThreads) {
                const uint64_t k = keys[e];
                if ((k & mask) == prefix)
                    atomicAdd(&hist[(k >> shift) & 255], 1);
            }
            __syncthreads();
            if (warp == 0) {  // the digit holding the remaining-th key: lane l holds digits 8l..8l+7
                int c[8], sum = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    c[q] = hist[lane * 8 + q];
                    sum += c[q];
                }
                int incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o)
                        incl += v;
                }
                const int excl = incl - sum;
                if (excl < remaining && remaining <= incl) {
                    int run = excl;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (run + c[q] >= remaining) {
                            s_bucket = lane * 8 + q;
                            s_below = run;
                            s_count = c[q];
                            break;
                        }
                        run += c[q];
                    }
                }
            }
            __syncthreads();
            remaining -= s_below;
            prefix |= (uint64_t)s_bucket << shift;
            mask |= 0xFFull << shift;
            const bool done = s_count == remaining;  // every key matching prefix is taken
            __syncthreads();  // s_* are read before the next pass writes them
            if (done) {
                tau = prefix | ~mask;
                break;
            }
            tau = prefix;
        }
        // 3. depth of each request: its keys <= tau
        for (int e = tid; e < n; e += kDcutThreads) {
            const uint64_t k = keys[e];
            if (k <= tau)
                atomicAdd(&depth_s[(int)((uint32_t)k / (uint32_t)p.Kmax)], 1);
        }
    }
    __syncthreads();

    // 4. offsets (exclusive scan), depths, expected accepted drafts
    const int per = (p.B + kDcutThreads - 1) / kDcutThreads;
    const int r0 = min(p.B, tid * per), r1 = min(p.B, r0 + per);
    int seg = 0;
    for (int r = r0; r < r1; ++r)
        seg += depth_s[r];
    int total = 0;
    int off = block_excl_scan_int(seg, warp_tot, total);
    for (int r = r0; r < r1; ++r) {
        p.out_cu[r] = off;
        off += depth_s[r];
        p.out_depth[r] = depth_s[r];
        if (p.out_expected) {
            float P = 1.f;
            double e = 0.0;
            for (int d = 1; d <= depth_s[r]; ++d) {
                P = __fadd_rn(__fmul_rn(P, conf_s[r * cs + (d - 1)]), 0.f);
                e += (double)P;
            }
            p.out_expected[r] = (float)e;
        }
    }
    if (tid == 0)
        p.out_cu[p.B] = total;
}

static int next_pow2(int x)
{
    int p = 1;
    while (p < x)
        p <<= 1;
    return p;
}

cudaError_t launch_dcut(const DcutArgs &a, cudaStream_t s, Tracer &tr)
{
    static cudaError_t once = cudaFuncSetAttribute(
        dcut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        8 * kDcutMaxCand + 8 * kMaxBatch + 4 * (kDcutMaxCand + kMaxBatch));
    if (once != cudaSuccess)
        return once;
    DcutParams p{};
    p.conf = a.conf;
    p.kmax = a.kmax;
    p.B = a.B;
    p.Kmax = a.Kmax;
    p.Kp = next_pow2(a.Kmax > 0 ? a.Kmax : 1);
    p.Bp = next_pow2(a.B > 0 ? a.B : 1);
    p.budget = a.budget;
    p.min_gain = a.min_gain;
    p.out_depth = a.out_depth;
    p.out_cu = a.out_cu;
    p.out_expected = a.out_expected;
    const WsLayout L = ws_layout(0, 0, 0);
    p.status = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(a.ws) + L.status);
    const size_t smem = sizeof(uint64_t) * (size_t)a.B * a.Kmax + 8 * (size_t)a.B +
                        4 * (size_t)a.B * (a.Kmax | 1);
    tr.begin(s);
    dcut_kernel<<<1, kDcutThreads, smem, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    tr.after_kernel(s);
    return cudaSuccess;
}

}  // namespace sv

// ---------------------------------------------------------------------------
// D-cut, cost-unit variant
// ---------------------------------------------------------------------------
//
// The deep-dive page ("Tencent AngelSpec Speculative Decoding Framework Deep
// Dive ...", its D-cut scheduler) budgets verification in profiled
// latency-cost units: cost(d) is the piecewise-linear function through the
// table {1: 1.0, 2: 1.2, 4: 1.5, 8: 2.0, 16: 3.0} (constant beyond its
// ends); each request takes the depth maximising benefit(d) = P_d * d /
// cost(d) (the first such d); requests are admitted in decreasing benefit
// (ties by request) while the running cost stays within max_cost, skipping
// those that do not fit.  The page computes in Python floats (binary64);
// every value here is the binary64 value of the same operations in the same
// order, each rounded once, so depths and benefits match a sequential fp64
// evaluation bit for bit.  The roundings are done exactly on the integer
// pipes (fp64_exact.cuh; B300's fp64 pipe is slow), the hardware fp64 path
// only for values outside the normal range.  One cluster of CTAs:
// per-request best depths in parallel across its SMs, ranks by counting,
// then the admission in rank order (sequential by definition), decided
// block-wide from exact sums of the costs, the rounded running total taken
// only where the rounding can matter.

namespace sv {

constexpr int kCostCluster = 8;    // CTAs of the cost kernel's cluster (one per SM)
constexpr int kCostThreads = 512;  // threads per CTA

struct DcutCostParams {
    const float *conf;
    const int32_t *kmax;
    int B, Kmax;
    uint64_t cost_bits[kMaxDraft + 1];   // cost(d) as a double's bits, d = 1..32
    uint64_t cost_recip[kMaxDraft + 1];  // recip116 of cost(d)'s significand
    double max_cost;
    uint64_t max_units;  // floor(max_cost * 2^52) when units_path
    uint64_t half_ulp;   // half a unit in the last place of max_cost + 3, in those units
    int units_path;      // 0 <= max_cost < 1024: the admission adds in units of 2^-52
    int32_t *out_depth;
    int32_t *out_cu;
    double *out_benefit;
    uint32_t *status;
};

// cost(d) of the profiled latency table {1: 1.0, 2: 1.2, 4: 1.5, 8: 2.0,
// 16: 3.0}: piecewise linear through those points, constant outside
// [1, 16].  The table's depths are the powers 2^0 .. 2^4, so depth d in
// (2^k, 2^(k+1)] lies on segment k, whose span is 2^k: the fraction
// (d - 2^k) / 2^k is exact and the cost is one rounded multiply and one
// rounded add in binary64.  Evaluated on the host (each operation a separate
// IEEE binary64 operation: `volatile` keeps them from being fused).
static double latency_cost(int d)
{
    const double at_pow2[5] = {1.0, 1.2, 1.5, 2.0, 3.0};  // cost(2^k), k = 0..4
    if (d <= 1)
        return at_pow2[0];
    if (d >= 16)
        return at_pow2[4];
    int k = 0;
    while ((2 << k) < d)  // 2^k < d <= 2^(k+1)
        ++k;
    const double frac = (double)(d - (1 << k)) / (double)(1 << k);  // exact
    volatile double rise = at_pow2[k + 1] - at_pow2[k];
    volatile double step = rise * frac;
    return at_pow2[k] + step;
}

// Bytes of dynamic shared memory per request: benefit bits, the cost of
// each rank (units of 2^-52, or a double's bits), best depth, rank order,
// depth, the admission decision of each rank.
constexpr int kCostSmemPerReq = 8 + 8 + 4 + 4 + 4 + 1;

// The benefit P_d * d / cost(d) of one (request, depth) pair as a double's
// bits, computed the way the scheduler's fp64 arithmetic does (P_d the
// left-to-right product of the confidences, each operation rounded once):
// on the integer paths (fp64_exact.cuh), or with the fp64 hardware when a
// value leaves the normal range (a subnormal product or confidence).  The
// group of Kp lanes of one request holds its confidences, one per lane
// (cj of lane j); every lane of the group calls this (it shuffles).
__device__ __forceinline__ uint64_t pair_benefit(const uint64_t *cost_bits,
                                                 const uint64_t *cost_recip, float cj, int gbase,
                                                 int Kp, int d)
{
    Dbl P{1ull << 52, -52};  // 1.0
    bool zero = false, slow = false;
    for (int j = 0; j < Kp; ++j) {
        const float c = __shfl_sync(0xffffffffu, cj, gbase + j);
        if (j >= d || zero || slow)
            continue;
        if (c == 0.f) {
            zero = true;
            continue;
        }
        Dbl cd;
        if (!flt_unpack(__float_as_uint(c), cd)) {
            slow = true;
            continue;
        }
        P = mul_round(P, cd);
        slow = P.e + 1075 < 1;
    }
    uint64_t bits = 0;  // +0.0: a zero confidence makes the benefit 0
    if (!zero && !slow && d >= 1 && d <= kMaxDraft) {
        const Dbl x = mul_round(P, int_unpack((uint32_t)d));
        Dbl y;
        dbl_unpack(cost_bits[d], y);
        slow = !dbl_pack(div_round(x, y, cost_recip[d]), bits);
    }
    // the hardware path, from the start (every lane shuffles; only the
    // lanes that need it use the result)
    const bool any_slow = __any_sync(0xffffffffu, slow);
    if (any_slow) {
        double Q = 1.0;
        for (int j = 0; j < Kp; ++j) {
            const float c = __shfl_sync(0xffffffffu, cj, gbase + j);
            if (slow && j < d)
                Q = __dmul_rn(Q, (double)c);
        }
        if (slow)
            bits = (uint64_t)__double_as_longlong(__ddiv_rn(
                __dmul_rn(Q, (double)d), __longlong_as_double((long long)cost_bits[d])));
    }
    return bits;
}

// One cluster of kCostCluster CTAs:
//  1. every (request, depth) pair is one thread somewhere in the cluster
//     (pair_benefit); a group of Kp lanes keeps its request's first maximum
//     (benefits compared as the integer bits of non-negative doubles) and
//     stores (benefit, depth) into the shared memory of every CTA;
//  2. every CTA ranks its share of the requests (larger benefit first, then
//     lower request) by counting, and stores the rank into CTA 0;
//  3. CTA 0 lays out the costs in rank order and admits in rank order: the
//     exact sums of the costs (64-bit integers in units of 2^-52) decide
//     every rank farther than the accumulated rounding margin from
//     max_cost, by a block-wide prefix scan and block-wide searches; a rank
//     inside the margin is decided on the binary64 running total.  The CTA
//     then writes depths, offsets and benefits.
__global__ void __launch_bounds__(kCostThreads) dcut_cost_kernel(const DcutCostParams p)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    uint64_t *rank_cost = reinterpret_cast<uint64_t *>(dsm);  // [B] CTA 0: cost of each rank
    uint64_t *bbits = rank_cost + p.B;                         // [B] benefit bits
    int *best_d = reinterpret_cast<int *>(bbits + p.B);                // [B] 0: no candidate
    int *order = best_d + p.B;                                         // [B] CTA 0: request of each rank
    int *depth = order + p.B;                                          // [B] CTA 0
    __shared__ uint64_t cost_units[kMaxDraft + 1];  // cost(d) in units of 2^-52
    __shared__ uint64_t cost_bits[kMaxDraft + 1];   // cost(d) as a double's bits
    __shared__ uint64_t cost_recip[kMaxDraft + 1];  // recip116 of its significand
    __shared__ int s_bad[kCostCluster];         // written by every CTA of the cluster
    __shared__ int s_ncand;
    __shared__ int warp_tot[33];
    __shared__ uint64_t warp_sum[kCostThreads / 32];  // the admission's scan
    __shared__ uint64_t s_x;
    __shared__ int s_first;
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    if (tid >= 1 && tid <= kMaxDraft) {  // staged: lanes index them by their own depth
        cost_units[tid] = to_units(p.cost_bits[tid]);
        cost_bits[tid] = p.cost_bits[tid];
        cost_recip[tid] = p.cost_recip[tid];
    }
    if (tid < kCostCluster)
        s_bad[tid] = 0;
    if (tid == 0)
        s_ncand = 0;
    __syncthreads();
    cluster_arrive_release();
    cluster_wait_acquire();  // (0) every CTA has started: remote stores may begin

    // 1. the best depth of every request
    int Kp = 1;
    while (Kp < p.Kmax)
        Kp <<= 1;
    const int64_t npairs = (int64_t)p.B * Kp;
    const int64_t stride = (int64_t)kCostCluster * kCostThreads;
    int bad = 0;
    // warp w of CTA q takes the 32 pairs at (w * kCostCluster + q) * 32 first,
    // so that a small batch is spread over every SM of the cluster
    for (int64_t base = ((int64_t)(tid >> 5) * kCostCluster + rank) * 32; base < npairs;
         base += stride) {
        const int64_t t = base + lane;  // groups of Kp lanes never straddle a warp (Kp | 32)
        const int r = (int)(t / Kp), d = (int)(t % Kp) + 1;
        int km = 0;
        float cj = 0.f;  // this lane's confidence: c[r][d - 1]
        if (t < npairs) {
            km = __ldg(p.kmax + r);
            if (km < 0 || km > p.Kmax) {
                bad = 1;
                km = 0;
            }
            if (d <= km) {
                cj = __ldg(p.conf + (int64_t)r * p.Kmax + (d - 1));
                if (!(cj >= 0.f && cj <= 1.f))
                    bad = 1;
            }
        }
        // the group's lanes hold its request's confidences; an invalid one
        // anywhere poisons the whole call, so the values are only used when
        // the whole warp saw valid ones
        const bool warp_bad = __any_sync(0xffffffffu, bad);
        const uint64_t bits =
            pair_benefit(cost_bits, cost_recip, warp_bad ? 0.f : cj, lane & ~(Kp - 1), Kp, d);
        const long long b = t < npairs && d <= km && !warp_bad ? (long long)bits : -1;
        // the group's first maximum: larger benefit, then smaller depth
        long long bb = b;
        int bd = b >= 0 ? d : 0;
        for (int o = Kp >> 1; o > 0; o >>= 1) {
            const long long ob = __shfl_xor_sync(0xffffffffu, bb, o);
            const int od = __shfl_xor_sync(0xffffffffu, bd, o);
            if (ob > bb || (ob == bb && od != 0 && (bd == 0 || od < bd))) {
                bb = ob;
                bd = od;
            }
        }
        if (t < npairs && d == 1) {
            const uint64_t best_bits = km > 0 ? (uint64_t)bb + 1 : 0ull;  // the ranking key
            const int dd = km > 0 ? bd : 0;
            for (uint32_t q = 0; q < kCostCluster; ++q) {
                st_cluster_u64(&bbits[r], q, best_bits);
                st_cluster_u32(&best_d[r], q, (uint32_t)dd);
            }
        }
    }
    if (__syncthreads_or(bad) && tid == 0)
        for (uint32_t q = 0; q < kCostCluster; ++q)
            st_cluster_u32(&s_bad[rank], q, 1u);
    cluster_arrive_release();
    cluster_wait_acquire();  // (1) every CTA holds every request's (benefit, depth)
    int any_bad = 0;
    for (int q = 0; q < kCostCluster; ++q)
        any_bad |= s_bad[q];
    if (any_bad) {  // the same verdict in every CTA: no barrier follows
        if (rank == 0) {
            if (tid == 0)
                set_status(p.status, ST_INVALID);
            for (int r = tid; r < p.B; r += kCostThreads) {
                p.out_depth[r] = -1;
                if (p.out_benefit)
                    p.out_benefit[r] = __longlong_as_double(0x7ff8000000000000ll);
            }
            for (int r = tid; r <= p.B; r += kCostThreads)
                p.out_cu[r] = -1;
        }
        return;
    }

    // 2. rank of every candidate.  Keys: the benefit's bits + 1 for a
    // candidate (benefits >= 0: their bits order as integers), 0 for none,
    // so that no candidate ever counts a non-candidate above it.
    for (int r = rank * kCostThreads + tid; r < p.B; r += kCostCluster * kCostThreads) {
        const uint64_t kb = bbits[r];
        if (kb == 0)
            continue;
        int rk0 = 0, rk1 = 0;
        int q = 0;
        for (; q + 1 < p.B; q += 2) {  // two independent counts
            const uint64_t o0 = bbits[q], o1 = bbits[q + 1];
            rk0 += o0 > kb || (o0 == kb && q < r);
            rk1 += o1 > kb || (o1 == kb && q + 1 < r);
        }
        if (q < p.B)
            rk0 += bbits[q] > kb || (bbits[q] == kb && q < r);
        st_cluster_u32(&order[rk0 + rk1], 0, (uint32_t)r);
    }
    cluster_arrive_release();
    cluster_wait_acquire();  // (2) CTA 0 holds the ranking
    if (rank != 0)
        return;  // no CTA touches another's shared memory after (2)

    // 3. admission in rank order
    int nc = 0;
    for (int r = tid; r < p.B; r += kCostThreads) {
        nc += bbits[r] != 0;
        depth[r] = 0;
    }
    if (nc)
        atomicAdd(&s_ncand, nc);
    __syncthreads();
    const int ncand = s_ncand;
    for (int t = tid; t < ncand; t += kCostThreads) {
        const int dd = best_d[order[t]];
        rank_cost[t] = p.units_path ? cost_units[dd] : cost_bits[dd];
    }
    __syncthreads();
    uint8_t *admitted = reinterpret_cast<uint8_t *>(depth + p.B);  // [B] per rank
    if (p.units_path) {
        // The rounded running total T and the exact sum X of the admitted
        // costs differ by at most k half-ulps after k admissions (every
        // rounded sum is below max_cost + 3), so a step whose exact sum lies
        // farther than (k + 1) half-ulps from max_cost is decided by X alone.
        //  - Until the first rejection every rank is admitted, so X is the
        //    prefix sum of the costs: one block-wide scan finds the first
        //    rank that is not surely admitted.
        //  - After it the remaining budget is below that rank's cost (at
        //    most 3) and every cost is at least 1, so at most two more ranks
        //    fit: each is found by a block-wide search for the next rank
        //    that is not surely rejected.
        // A decision inside the margin (a budget on or next to a reachable
        // sum) is taken on the rounded running total, as the scheduler's
        // binary64 additions would.
        const uint64_t M = p.max_units, hu = p.half_ulp;
        const uint64_t SAT = ~0ull >> 1;  // above every budget
        const int per = (ncand + kCostThreads - 1) / kCostThreads;
        const int t0 = min(ncand, tid * per), t1 = min(ncand, t0 + per);
        uint64_t seg = 0;
        for (int t = t0; t < t1; ++t) {
            admitted[t] = 0;
            seg = min(SAT, seg + rank_cost[t]);
        }
        // exclusive scan of the segment sums (saturating)
        uint64_t incl = seg;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl = min(SAT, incl + n);
        }
        if (lane == 31)
            warp_sum[tid >> 5] = incl;
        if (tid == 0)
            s_first = INT_MAX;
        __syncthreads();
        uint64_t E = incl - seg;  // this thread's exclusive prefix, then each rank's
        for (int w = 0; w < (tid >> 5); ++w)
            E = min(SAT, E + warp_sum[w]);
        int mine = INT_MAX;  // this thread's first rank that is not surely admitted
        for (int t = t0; t < t1; ++t) {
            const uint64_t y = min(SAT, E + rank_cost[t]);
            if (y + (uint64_t)(t + 1) * hu > M) {
                mine = t;
                atomicMin(&s_first, t);
                break;
            }
            E = y;
        }
        __syncthreads();
        const int first = s_first;
        for (int t = t0; t < t1 && t < first; ++t)
            admitted[t] = 1;
        if (first < ncand) {
            if (mine == first)
                s_x = E;  // the exact sum of the ranks before `first`, all admitted
            __syncthreads();
            // From `first` on, each step takes the next rank that is not
            // surely rejected.  A surely admitted one is admitted; one inside
            // the margin is decided on the rounded total T (computed once,
            // when first needed, from the ranks admitted so far), and a
            // rejection at T also rejects every later rank whose cost is no
            // smaller while T stays the same.  The budget left after the first
            // step that is not sure is below one cost, so few steps follow.
            uint64_t X = s_x, T = 0, c_rej = ~0ull;
            bool have_T = false;
            int k = first, cur = first - 1, n_late = 0;
            int late[4];  // ranks admitted from `first` on, in order: at most 3, since
                          // the budget left is below one cost (<= 3) and every cost is >= 1
            for (;;) {
                __syncthreads();  // every thread has read s_first
                if (tid == 0)
                    s_first = INT_MAX;
                __syncthreads();
                const uint64_t lim = M + (uint64_t)(k + 1) * hu;
                for (int t = max(t0, cur + 1); t < t1; ++t)
                    if (rank_cost[t] < c_rej && X + rank_cost[t] <= lim) {
                        atomicMin(&s_first, t);
                        break;
                    }
                __syncthreads();
                const int nx = s_first;
                if (nx >= ncand)
                    break;  // every later rank is rejected
                const uint64_t c = rank_cost[nx];
                bool adm;
                if (X + c + (uint64_t)(k + 1) * hu <= M) {
                    adm = true;  // surely admitted
                    if (have_T)
                        T = add_units_round(T, c);
                } else {  // inside the margin: the rounded total decides
                    if (!have_T) {
                        T = 0;  // the ranks admitted so far, in rank order
                        for (int t = 0; t < first; ++t)
                            T = add_units_round(T, rank_cost[t]);
                        for (int q = 0; q < n_late; ++q)
                            T = add_units_round(T, rank_cost[late[q]]);
                        have_T = true;
                    }
                    const uint64_t nt = add_units_round(T, c);
                    adm = nt <= M;
                    if (adm)
                        T = nt;
                }
                if (adm) {
                    if (tid == 0)
                        admitted[nx] = 1;
                    X += c;
                    ++k;
                    c_rej = ~0ull;
                    if (n_late < 4)
                        late[n_late++] = nx;
                } else {
                    c_rej = c;
                }
                cur = nx;
            }
        }
    } else if (tid == 0) {  // a large budget (or none): the fp64 hardware, one thread
        double total = 0.0;
        for (int t = 0; t < ncand; ++t) {
            const double nt = __dadd_rn(total, __longlong_as_double((long long)rank_cost[t]));
            const bool adm = p.max_cost >= 0.0 && nt <= p.max_cost;
            total = adm ? nt : total;
            admitted[t] = adm;
        }
    }
    __syncthreads();
    for (int t = tid; t < ncand; t += kCostThreads)
        if (admitted[t]) {
            const int r = order[t];
            depth[r] = best_d[r];
        }
    __syncthreads();

    // 4. depths, offsets (exclusive scan), benefits of the admitted requests
    const int per = (p.B + kCostThreads - 1) / kCostThreads;
    const int r0 = min(p.B, tid * per), r1 = min(p.B, r0 + per);
    int seg = 0;
    for (int r = r0; r < r1; ++r)
        seg += depth[r];
    int total = 0;
    int off = block_excl_scan_int(seg, warp_tot, total);
    for (int r = r0; r < r1; ++r) {
        p.out_cu[r] = off;
        off += depth[r];
        p.out_depth[r] = depth[r];
        if (p.out_benefit)
            p.out_benefit[r] =
                depth[r] > 0 ? __longlong_as_double((long long)(bbits[r] - 1)) : 0.0;
    }
    if (tid == 0)
        p.out_cu[p.B] = total;
}

cudaError_t launch_dcut_cost(const DcutCostArgs &a, cudaStream_t s, Tracer &tr)
{
    static cudaError_t once = cudaFuncSetAttribute(
        dcut_cost_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        kCostSmemPerReq * kMaxBatch);
    if (once != cudaSuccess)
        return once;
    DcutCostParams p{};
    p.conf = a.conf;
    p.kmax = a.kmax;
    p.B = a.B;
    p.Kmax = a.Kmax;
    for (int d = 1; d <= kMaxDraft; ++d) {
        const double cost = latency_cost(d);
        std::memcpy(&p.cost_bits[d], &cost, sizeof cost);
        Dbl y;
        dbl_unpack(p.cost_bits[d], y);  // cost(d) in [1, 3]: normal
        p.cost_recip[d] = recip116(y.m);
    }
    // floor(max_cost * 2^52): an admitted total is 0 or a double >= 1, a
    // multiple of 2^-52, so total <= max_cost exactly when its units are <=
    // this.  Totals stay below max_cost + 3 < 2^11 on this path.
    p.max_cost = a.max_cost;
    p.units_path = a.max_cost >= 0.0 && a.max_cost < 1024.0;
    p.max_units = 0;
    p.half_ulp = 0;
    if (p.units_path && a.max_cost > 0.0) {
        uint64_t bits;
        std::memcpy(&bits, &a.max_cost, sizeof bits);
        const int be = (int)((bits >> 52) & 0x7ff);
        const uint64_t m = (bits & ((1ull << 52) - 1)) | (be ? (1ull << 52) : 0ull);
        const int sh = (be ? be : 1) - 1075 + 52;  // max_cost * 2^52 = m * 2^sh
        p.max_units = sh >= 0 ? m << sh : (sh > -64 ? m >> -sh : 0);
    }
    if (p.units_path) {  // the largest sum ever compared is below max_cost + 3
        const uint64_t top = p.max_units + (3ull << 52);
        int L = 64;
        while (L > 0 && !(top >> (L - 1)))
            --L;
        p.half_ulp = L > 53 ? 1ull << (L - 54) : 0;  // no rounding below 2^53 units
    }
    p.out_depth = a.out_depth;
    p.out_cu = a.out_cu;
    p.out_benefit = a.out_benefit;
    const WsLayout L = ws_layout(0, 0, 0);
    p.status = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(a.ws) + L.status);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(kCostCluster);
    cfg.blockDim = dim3(kCostThreads);
    cfg.dynamicSmemBytes = kCostSmemPerReq * (size_t)(a.B > 0 ? a.B : 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCostCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    tr.begin(s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, dcut_cost_kernel, p);
    if (e != cudaSuccess)
        return e;
    tr.after_kernel(s);
    return cudaSuccess;
}

}  // namespace sv
