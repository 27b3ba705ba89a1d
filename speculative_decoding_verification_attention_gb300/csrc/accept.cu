// Batched accept/reject kernels for the verification step.
//
// Greedy: "accept the longest agreeing prefix, then emit one more target
// token" (LLM inference handbook, "How speculative decoding works").
// Stochastic: accept x with probability min(1, p(x)/q(x)); at the first
// rejection resample from max(0, p - q) renormalised (llm-digest,
// "Mechanism" and "Math intuition").
//
// Layout of the work: one thread-block cluster of CS CTAs per sequence;
// CTA `rank` owns a contiguous slice of the vocabulary and each of its 8
// warps a contiguous sub-slice, streamed in 128-element steps (one float4
// per lane, coalesced).  Cluster-wide reductions go through distributed
// shared memory.
//
// Exactness: the accept test u*q < p is evaluated in fp64, where the
// product of two fp32 values is exact.  Residual / bonus mass is summed in
// 64-bit fixed point (2^-61 resolution, truncation of each element), so
// every partial sum is exact and independent of the summation order; the
// draw compares running sums against floor(u * Z) computed exactly from
// the 24-bit mantissa of u.
#include <cooperative_groups.h>
#include <float.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace spec {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStep = 128;   // elements per warp step
constexpr int kUnroll = 8;   // steps whose loads are in flight together

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

struct Slice {
    int64_t begin, end;      // this warp's element range within the row
};

__device__ __forceinline__ Slice warp_slice(int V, int cs, int rank, int warp)
{
    // CTA slice rounded to a multiple of 4 elements, warp sub-slice to kStep
    int64_t cta_len = ((static_cast<int64_t>(V) + cs - 1) / cs + 3) & ~int64_t(3);
    const int64_t v = V;
    int64_t c0 = imin64(v, cta_len * rank), c1 = imin64(v, c0 + cta_len);
    int64_t w_len = ((cta_len + kWarps - 1) / kWarps + kStep - 1) / kStep * kStep;
    int64_t w0 = imin64(c1, c0 + w_len * warp), w1 = imin64(c1, w0 + w_len);
    return {w0, w1};
}

// Load the 4 elements [e, e+4) of row (bounded by `end`); missing ones read
// as `fill`.
__device__ __forceinline__ float4 load4(const float *row, int64_t e, int64_t end, bool vec4,
                                        float fill)
{
    if (vec4 && e + 3 < end) return __ldg(reinterpret_cast<const float4 *>(row + e));
    float4 r;
    r.x = e + 0 < end ? __ldg(row + e + 0) : fill;
    r.y = e + 1 < end ? __ldg(row + e + 1) : fill;
    r.z = e + 2 < end ? __ldg(row + e + 2) : fill;
    r.w = e + 3 < end ? __ldg(row + e + 3) : fill;
    return r;
}

// ------------------------------------------------------------------ greedy
struct ArgMax {
    float v;
    int i;
};

__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b)
{
    // larger value wins; equal values resolve to the lower index
    return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax b{__shfl_xor_sync(0xffffffffu, a.v, o), __shfl_xor_sync(0xffffffffu, a.i, o)};
        a = better(a, b);
    }
    return a;
}

template <int CS>
__global__ void __launch_bounds__(kThreads) accept_greedy_kernel(
    const float *__restrict__ p, const int32_t *__restrict__ draft, int D, int V,
    int32_t *__restrict__ n_accepted, int32_t *__restrict__ token, bool vec4)
{
    __shared__ ArgMax s_warp[kWarps];
    __shared__ ArgMax s_cta[2];  // per row parity, read by the whole cluster
    const int rank = CS > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int b = blockIdx.x / CS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Slice sl = warp_slice(V, CS, rank, warp);

    for (int i = 0; i <= D; ++i) {
        const float *row = p + (static_cast<int64_t>(b) * (D + 1) + i) * V;
        ArgMax best{-FLT_MAX, INT_MAX};
        bool have = false;
        for (int64_t base = sl.begin; base < sl.end; base += kStep * kUnroll) {
            float4 x[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                int64_t e = base + u * kStep + lane * 4;
                x[u] = e < sl.end ? load4(row, e, sl.end, vec4, -FLT_MAX) : make_float4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                int64_t e = base + u * kStep + lane * 4;
                if (e >= sl.end) continue;
                const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (e + k < sl.end && (!have || xs[k] > best.v)) {
                        best = {xs[k], static_cast<int>(e + k)};
                        have = true;
                    }
                }
            }
        }
        best = warp_argmax(best);
        if (lane == 0) s_warp[warp] = best;
        __syncthreads();
        if (threadIdx.x == 0) {
            ArgMax c = s_warp[0];
            for (int w = 1; w < kWarps; ++w) c = better(c, s_warp[w]);
            s_cta[i & 1] = c;
        }
        ArgMax g;
        if constexpr (CS > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            g = *cluster.map_shared_rank(&s_cta[i & 1], 0);
            for (int r = 1; r < CS; ++r) g = better(g, *cluster.map_shared_rank(&s_cta[i & 1], r));
        } else {
            __syncthreads();
            g = s_cta[i & 1];
        }
        const bool stop = (i == D) || (draft[static_cast<int64_t>(b) * D + i] != g.i);
        if (stop) {
            if (rank == 0 && threadIdx.x == 0) {
                n_accepted[b] = i;
                token[b] = g.i;
            }
            break;
        }
    }
    // keep this CTA's shared memory alive until every peer has read it
    if constexpr (CS > 1) cg::this_cluster().sync();
}

// --------------------------------------------------------------- stochastic
// Fixed point with 2^-61 resolution (truncating); probabilities up to 8
// per row sum fit in 64 bits.  Conversion saturates: negatives and NaN -> 0.
__device__ __forceinline__ unsigned long long fix61(float x)
{
    return __float2ull_rz(x * 0x1p61f);
}

__device__ __forceinline__ unsigned long long mass(float pv, float qv, int residual)
{
    unsigned long long a = fix61(pv);
    if (!residual) return a;
    unsigned long long c = fix61(qv);
    return a > c ? a - c : 0ull;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long x, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// floor(u * Z) exactly, for u in [0, 1).
__device__ __forceinline__ unsigned long long scaled_threshold(float u, unsigned long long Z)
{
    const uint32_t bits = __float_as_uint(u);
    const uint32_t e = (bits >> 23) & 0xFFu;
    const unsigned long long mu = e ? ((bits & 0x7FFFFFu) | 0x800000u) : (bits & 0x7FFFFFu);
    const int s = 150 - static_cast<int>(e ? e : 1);   // u = mu * 2^-s, s >= 24
    const unsigned long long lo = mu * Z;
    const unsigned long long hi = __umul64hi(mu, Z);
    if (s >= 128) return 0ull;
    if (s >= 64) return hi >> (s - 64);
    return (hi << (64 - s)) | (lo >> s);
}

template <int CS>
__global__ void __launch_bounds__(kThreads) accept_sample_kernel(
    const float *__restrict__ p, const float *__restrict__ q, const int32_t *__restrict__ draft,
    const float *__restrict__ u_acc, const float *__restrict__ u_res, int D, int V,
    int32_t *__restrict__ n_accepted, int32_t *__restrict__ token, uint32_t *dev_status,
    bool vec4)
{
    __shared__ unsigned long long s_warp[kWarps];
    __shared__ unsigned long long s_cta[2];  // per attempt, read by the whole cluster
    __shared__ int s_j;
    const int rank = CS > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int b = blockIdx.x / CS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Slice sl = warp_slice(V, CS, rank, warp);

    // First rejected draft (every CTA of the cluster computes the same j).
    if (warp == 0) {
        int j = D;
        for (int i0 = 0; i0 < D; i0 += 32) {
            const int i = i0 + lane;
            bool rej = false;
            if (i < D) {
                const int x = draft[static_cast<int64_t>(b) * D + i];
                if (x < 0 || x >= V) {
                    if (rank == 0) report(dev_status, SPEC_DEV_ERR_TOKEN_ID);
                    rej = true;
                } else {
                    const double pv = p[(static_cast<int64_t>(b) * (D + 1) + i) * V + x];
                    const double qv = q[(static_cast<int64_t>(b) * D + i) * V + x];
                    const float uf = u_acc[static_cast<int64_t>(b) * D + i];
                    if (!(uf >= 0.0f && uf < 1.0f) && rank == 0) report(dev_status, SPEC_DEV_ERR_UNIFORM);
                    rej = !(static_cast<double>(uf) * qv < pv);   // exact product
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, rej);
            if (m) {
                j = i0 + __ffs(m) - 1;
                break;
            }
        }
        if (lane == 0) s_j = j;
    }
    __syncthreads();
    const int j = s_j;
    const float *prow = p + (static_cast<int64_t>(b) * (D + 1) + j) * V;
    const float *qrow = j < D ? q + (static_cast<int64_t>(b) * D + j) * V : nullptr;
    float u = u_res[b];
    if (!(u >= 0.0f && u < 1.0f)) {
        if (rank == 0 && threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_UNIFORM);
        u = (u >= 1.0f) ? 0x1.fffffep-1f : 0.0f;
    }
    int residual = j < D;
    int tok = -1;

    for (int attempt = 0; attempt < 2; ++attempt) {
        // Phase 1: exact mass of this warp's sub-slice.
        unsigned long long acc = 0;
        for (int64_t base = sl.begin; base < sl.end; base += kStep * kUnroll) {
            float4 xp[kUnroll], xq[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t e = base + k * kStep + lane * 4;
                xp[k] = e < sl.end ? load4(prow, e, sl.end, vec4, 0.f) : make_float4(0, 0, 0, 0);
                xq[k] = (residual && e < sl.end) ? load4(qrow, e, sl.end, vec4, 0.f)
                                                 : make_float4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                acc += mass(xp[k].x, xq[k].x, residual) + mass(xp[k].y, xq[k].y, residual) +
                       mass(xp[k].z, xq[k].z, residual) + mass(xp[k].w, xq[k].w, residual);
            }
        }
        acc = warp_sum_u64(acc);
        if (lane == 0) s_warp[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long t = 0;
            for (int w = 0; w < kWarps; ++w) t += s_warp[w];
            s_cta[attempt] = t;
        }
        unsigned long long Z = 0, pre = 0, mine = 0;
        if constexpr (CS > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            for (int r = 0; r < CS; ++r) {
                const unsigned long long t = *cluster.map_shared_rank(&s_cta[attempt], r);
                if (r < rank) pre += t;
                if (r == rank) mine = t;
                Z += t;
            }
        } else {
            __syncthreads();
            Z = mine = s_cta[attempt];
        }
        if (Z == 0) {
            if (residual) {   // reading: fall back to the target row itself
                residual = 0;
                if (rank == 0 && threadIdx.x == 0) report(dev_status, SPEC_DEV_INFO_ZERO_RESIDUAL);
                continue;
            }
            if (rank == 0 && threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_ZERO_MASS);
            tok = 0;
            break;
        }
        const unsigned long long T = scaled_threshold(u, Z);
        // Phase 2: the single warp whose range holds the crossing re-reads
        // its sub-slice (now cache-resident) with a running prefix.
        if (pre <= T && T < pre + mine) {
            unsigned long long wpre = pre;
            for (int w = 0; w < warp; ++w) wpre += s_warp[w];
            if (wpre <= T && T < wpre + s_warp[warp]) {
                unsigned long long run = wpre;
                for (int64_t base = sl.begin; base < sl.end; base += kStep) {
                    const int64_t e = base + lane * 4;
                    const float4 xp = e < sl.end ? load4(prow, e, sl.end, vec4, 0.f) : make_float4(0, 0, 0, 0);
                    const float4 xq = (residual && e < sl.end) ? load4(qrow, e, sl.end, vec4, 0.f)
                                                               : make_float4(0, 0, 0, 0);
                    const unsigned long long m[4] = {mass(xp.x, xq.x, residual), mass(xp.y, xq.y, residual),
                                                     mass(xp.z, xq.z, residual), mass(xp.w, xq.w, residual)};
                    const unsigned long long lane_sum = m[0] + m[1] + m[2] + m[3];
                    const unsigned long long incl = warp_incl_scan_u64(lane_sum, lane);
                    const unsigned hit = __ballot_sync(0xffffffffu, run + incl > T);
                    if (hit) {
                        const int L = __ffs(hit) - 1;
                        if (lane == L) {
                            unsigned long long c = run + incl - lane_sum;
                            int v = static_cast<int>(e);
                            for (int k = 0; k < 4; ++k) {
                                c += m[k];
                                if (c > T) { v = static_cast<int>(e) + k; break; }
                            }
                            token[b] = v;
                        }
                        break;
                    }
                    run += __shfl_sync(0xffffffffu, incl, 31);
                }
            }
        }
        break;
    }
    if (rank == 0 && threadIdx.x == 0) {
        n_accepted[b] = j;
        if (tok >= 0) token[b] = tok;
    }
    if constexpr (CS > 1) cg::this_cluster().sync();
}

int pick_cluster(int V)
{
    if (V >= 32768) return 8;
    if (V >= 8192) return 4;
    if (V >= 2048) return 2;
    return 1;
}

template <typename Kernel, typename... Args>
cudaError_t launch_clustered(Kernel k, int B, int cs, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B) * cs);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace

cudaError_t launch_accept_greedy(const float *p, const int32_t *draft, int B, int D, int V,
                                 int32_t *n_acc, int32_t *token, cudaStream_t st)
{
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0);
    switch (pick_cluster(V)) {
    case 8: return launch_clustered(accept_greedy_kernel<8>, B, 8, st, p, draft, D, V, n_acc, token, vec4);
    case 4: return launch_clustered(accept_greedy_kernel<4>, B, 4, st, p, draft, D, V, n_acc, token, vec4);
    case 2: return launch_clustered(accept_greedy_kernel<2>, B, 2, st, p, draft, D, V, n_acc, token, vec4);
    default: return launch_clustered(accept_greedy_kernel<1>, B, 1, st, p, draft, D, V, n_acc, token, vec4);
    }
}

cudaError_t launch_accept_sample(const float *p, const float *q, const int32_t *draft,
                                 const float *u_acc, const float *u_res, int B, int D, int V,
                                 int32_t *n_acc, int32_t *token, uint32_t *dev_status,
                                 cudaStream_t st)
{
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                      (q == nullptr || reinterpret_cast<uintptr_t>(q) % 16 == 0);
    switch (pick_cluster(V)) {
    case 8: return launch_clustered(accept_sample_kernel<8>, B, 8, st, p, q, draft, u_acc, u_res, D, V, n_acc, token, dev_status, vec4);
    case 4: return launch_clustered(accept_sample_kernel<4>, B, 4, st, p, q, draft, u_acc, u_res, D, V, n_acc, token, dev_status, vec4);
    case 2: return launch_clustered(accept_sample_kernel<2>, B, 2, st, p, q, draft, u_acc, u_res, D, V, n_acc, token, dev_status, vec4);
    default: return launch_clustered(accept_sample_kernel<1>, B, 1, st, p, q, draft, u_acc, u_res, D, V, n_acc, token, dev_status, vec4);
    }
}

}  // namespace spec
