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

#include "common.cuh"
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
// those that do not fit.  The page computes in Python floats (fp64); every
// decision here is taken in fp64 with each operation explicitly rounded, so
// depths match a sequential fp64 evaluation bit for bit.  One cluster of
// CTAs: per-request best depths in parallel across its SMs, ranks by
// counting, then one thread walks the ranked requests (the admission is
// sequential by definition).

namespace sv {

constexpr int kCostCluster = 8;    // CTAs of the cost kernel's cluster (one per SM)
constexpr int kCostThreads = 512;  // threads per CTA

struct DcutCostParams {
    const float *conf;
    const int32_t *kmax;
    int B, Kmax;
    double max_cost;
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
// rounded add in fp64.
__device__ __forceinline__ double latency_cost(int d)
{
    const double at_pow2[5] = {1.0, 1.2, 1.5, 2.0, 3.0};  // cost(2^k), k = 0..4
    if (d <= 1)
        return at_pow2[0];
    if (d >= 16)
        return at_pow2[4];
    const int k = 31 - __clz(d - 1);  // floor(log2(d - 1)): 2^k < d <= 2^(k+1)
    const double frac = (double)(d - (1 << k)) / (double)(1 << k);  // exact
    return __dadd_rn(at_pow2[k], __dmul_rn(__dsub_rn(at_pow2[k + 1], at_pow2[k]), frac));
}

// Bytes of dynamic shared memory per request.
constexpr int kCostSmemPerReq = 8 + 8 + 4 + 4 + 4;

// One cluster of kCostCluster CTAs (B300's fp64 rate per SM is low, so the
// fp64 benefits are spread over the cluster's SMs):
//  1. every (request, depth) pair is one thread somewhere in the cluster:
//     the prefix product left to right, one multiply by d and one division
//     by cost(d); a group of Kp lanes keeps its request's first maximum and
//     stores (benefit, depth) into the shared memory of every CTA;
//  2. every CTA ranks its share of the requests (larger benefit first, then
//     lower request) by counting, with the benefits compared as the integer
//     bits of non-negative doubles, and stores the rank into CTA 0;
//  3. CTA 0 gathers the costs in rank order, one thread admits in rank order
//     (sequential by definition, each addition rounded in fp64), and the
//     CTA writes depths, offsets and benefits.
__global__ void __launch_bounds__(kCostThreads) dcut_cost_kernel(const DcutCostParams p)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    uint64_t *bbits = reinterpret_cast<uint64_t *>(dsm);             // [B] benefit bits
    double *rank_cost = reinterpret_cast<double *>(bbits + p.B);      // [B] CTA 0
    int *best_d = reinterpret_cast<int *>(rank_cost + p.B);           // [B] 0: no candidate
    int *order = best_d + p.B;                                        // [B] CTA 0: request of each rank
    int *depth = order + p.B;                                         // [B] CTA 0
    __shared__ double cost_tab[kMaxDraft + 1];  // cost(d), d = 1..Kmax
    __shared__ int s_bad[kCostCluster];         // written by every CTA of the cluster
    __shared__ int s_ncand;
    __shared__ int warp_tot[33];
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    if (tid >= 1 && tid <= kMaxDraft)
        cost_tab[tid] = latency_cost(tid);
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
    for (int64_t base = (int64_t)rank * kCostThreads + (tid & ~31); base < npairs; base += stride) {
        const int64_t t = base + lane;  // groups of Kp lanes never straddle a warp (Kp | 32)
        const int r = (int)(t / Kp), d = (int)(t % Kp) + 1;
        int km = 0;
        double b = -1.0;
        if (t < npairs) {
            km = __ldg(p.kmax + r);
            if (km < 0 || km > p.Kmax) {
                bad = 1;
                km = 0;
            }
            if (d <= km) {
                double P = 1.0;
                for (int j = 0; j < d; ++j) {
                    const float c = __ldg(p.conf + (int64_t)r * p.Kmax + j);
                    if (!(c >= 0.f && c <= 1.f))
                        bad = 1;
                    P = __dmul_rn(P, (double)c);
                }
                b = __ddiv_rn(__dmul_rn(P, (double)d), cost_tab[d]);
            }
        }
        // the group's first maximum: larger benefit, then smaller depth
        double bb = b;
        int bd = b >= 0.0 ? d : 0;
        for (int o = Kp >> 1; o > 0; o >>= 1) {
            const double ob = __shfl_xor_sync(0xffffffffu, bb, o);
            const int od = __shfl_xor_sync(0xffffffffu, bd, o);
            if (ob > bb || (ob == bb && od != 0 && (bd == 0 || od < bd))) {
                bb = ob;
                bd = od;
            }
        }
        if (t < npairs && d == 1) {
            const uint64_t bits = km > 0 ? (uint64_t)__double_as_longlong(bb) : 0ull;
            const int dd = km > 0 ? bd : 0;
            for (uint32_t q = 0; q < kCostCluster; ++q) {
                st_cluster_u64(&bbits[r], q, bits);
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

    // 2. rank of every candidate (benefits >= 0: their bits order as integers)
    for (int r = rank * kCostThreads + tid; r < p.B; r += kCostCluster * kCostThreads) {
        if (best_d[r] == 0)
            continue;
        const uint64_t kb = bbits[r];
        int rk = 0;
        for (int q = 0; q < p.B; ++q) {
            const uint64_t o = bbits[q];
            rk += best_d[q] != 0 && (o > kb || (o == kb && q < r));
        }
        st_cluster_u32(&order[rk], 0, (uint32_t)r);
    }
    cluster_arrive_release();
    cluster_wait_acquire();  // (2) CTA 0 holds the ranking
    if (rank != 0)
        return;  // no CTA touches another's shared memory after (2)

    // 3. admission in rank order
    int nc = 0;
    for (int r = tid; r < p.B; r += kCostThreads) {
        nc += best_d[r] != 0;
        depth[r] = 0;
    }
    if (nc)
        atomicAdd(&s_ncand, nc);
    __syncthreads();
    const int ncand = s_ncand;
    for (int t = tid; t < ncand; t += kCostThreads)
        rank_cost[t] = cost_tab[best_d[order[t]]];
    __syncthreads();
    if (tid == 0) {
        double total = 0.0;
        for (int t = 0; t < ncand; ++t) {
            const double nt = __dadd_rn(total, rank_cost[t]);
            if (nt <= p.max_cost) {
                total = nt;
                const int r = order[t];
                depth[r] = best_d[r];
            }
        }
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
                depth[r] > 0 ? __longlong_as_double((long long)bbits[r]) : 0.0;
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
    p.max_cost = a.max_cost;
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
