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
#include "kernels.h"

namespace cg = cooperative_groups;

namespace spec {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStep = 128;   // elements per warp step
constexpr int kUnroll = 8;   // greedy: steps whose loads are in flight together

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
__global__ void __launch_bounds__(kThreads, 4) accept_greedy_kernel(
    const float *__restrict__ p, const int32_t *__restrict__ draft, int D, int V,
    int32_t *__restrict__ n_accepted, int32_t *__restrict__ token, bool vec4)
{
    __shared__ ArgMax s_warp[kWarps];
    __shared__ ArgMax s_cta[2];  // per row parity, read by the whole cluster
    __shared__ ArgMax s_g[2];    // cluster-wide result, per row parity
    const int rank = CS > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int b = blockIdx.x / CS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Slice sl = warp_slice(V, CS, rank, warp);
    // the drafts are read up front, off the per-row critical path
    __shared__ int32_t s_draft[kMaxDraft];
    for (int i = threadIdx.x; i < D; i += kThreads) s_draft[i] = draft[static_cast<int64_t>(b) * D + i];
    __syncthreads();

    for (int i = 0; i <= D; ++i) {
        const float *row = p + (static_cast<int64_t>(b) * (D + 1) + i) * V;
        // Per lane, elements are visited in increasing index order; only a
        // strictly larger value replaces the best, so ties keep the lowest
        // index.  The index is located only when a float4's max wins.
        ArgMax best{-FLT_MAX, INT_MAX};
        for (int64_t base = sl.begin; base < sl.end; base += kStep * kUnroll) {
            float4 x[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                int64_t e = base + u * kStep + lane * 4;
                x[u] = e < sl.end ? load4(row, e, sl.end, vec4, -INFINITY) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int e = static_cast<int>(base) + u * kStep + lane * 4;
                const float m4 = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
                if (e < sl.end && (m4 > best.v || (best.i == INT_MAX && m4 == m4))) {
                    const int k = x[u].x == m4 ? 0 : x[u].y == m4 ? 1 : x[u].z == m4 ? 2 : 3;
                    if (e + k < sl.end) best = {m4, e + k};
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
            // every peer's result is read at once, one lane per rank
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            if (warp == 0) {
                ArgMax c{-FLT_MAX, INT_MAX};
                if (lane < CS) c = *cluster.map_shared_rank(&s_cta[i & 1], lane);
                c = warp_argmax(c);
                if (lane == 0) s_g[i & 1] = c;
            }
            __syncthreads();
            g = s_g[i & 1];
        } else {
            __syncthreads();
            g = s_cta[i & 1];
        }
        const bool stop = (i == D) || (s_draft[i] != g.i);
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
// Fixed point with 2^-61 resolution: floor(x * 2^61) for 0 <= x < 8 (row
// sums below 8 fit in 64 bits).  x * 2^61 = m * 2^sh with m the 24-bit
// significand and sh = exponent - 89; the result is (m << max(sh, 0)) >>
// max(-sh, 0).  PTX clamps shift counts, so zero, denormals (sh = -89),
// negatives (the sign bit makes sh >= 167), infinities and NaN all give 0
// without special cases.  Integer shifts only: the float-to-64-bit-integer
// conversion instruction runs on the small fp64 pipe of this GPU.
__device__ __forceinline__ unsigned long long fix61(float x)
{
    const uint32_t b = __float_as_uint(x);
    const unsigned long long m = (b & 0x7FFFFFu) | 0x800000u;
    const int sh = static_cast<int>(b >> 23) - 89;
    unsigned long long r;
    asm("{\n\t.reg .u32 l, rr;\n\t"
        "max.s32 l, %1, 0;\n\t"
        "neg.s32 rr, %1;\n\t"
        "max.s32 rr, rr, 0;\n\t"
        "shl.b64 %0, %2, l;\n\t"
        "shr.b64 %0, %0, rr;\n\t}"
        : "=l"(r)
        : "r"(sh), "l"(m));
    return r;
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

// ----------------------------------------------------- stochastic, staged
// Scratch layout in the caller's workspace (see spec_accept_sample):
//   js    int32  [B]                 first rejected draft (or D)
//   cnt   uint32 [B]                 chunks of the sequence finished
//   steps uint64 [B][ceil(V / 128)]  exact residual / bonus mass of every
//                                    128-element step of the needed row
struct SampleScratch {
    int32_t *js;
    uint32_t *cnt;
    unsigned long long *steps;
    int nsteps;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int kChunk = kThreads * 32;      // elements of one streaming CTA
constexpr int kWarpElems = kChunk / kWarps;   // 1024: 8 steps of 128

// Stage 1: first rejected draft of every sequence (one warp per sequence);
// the accept test u * q(x) < p(x) is evaluated in fp64, where it is exact.
__global__ void __launch_bounds__(kThreads) accept_prep_kernel(
    const float *__restrict__ p, const float *__restrict__ q, const int32_t *__restrict__ draft,
    const float *__restrict__ u_acc, int B, int D, int V, SampleScratch sc, uint32_t *dev_status)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarps + warp;
    if (b >= B) return;
    int j = D;
    for (int i0 = 0; i0 < D; i0 += 32) {
        const int i = i0 + lane;
        bool rej = false;
        if (i < D) {
            const int x = draft[static_cast<int64_t>(b) * D + i];
            if (x < 0 || x >= V) {
                report(dev_status, SPEC_DEV_ERR_TOKEN_ID);
                rej = true;
            } else {
                const double pv = p[(static_cast<int64_t>(b) * (D + 1) + i) * V + x];
                const double qv = q[(static_cast<int64_t>(b) * D + i) * V + x];
                const float uf = u_acc[static_cast<int64_t>(b) * D + i];
                if (!(uf >= 0.0f && uf < 1.0f)) report(dev_status, SPEC_DEV_ERR_UNIFORM);
                rej = !(static_cast<double>(uf) * qv < pv);   // exact product
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, rej);
        if (m) {
            j = i0 + __ffs(m) - 1;
            break;
        }
    }
    if (lane == 0) {
        sc.js[b] = j;
        sc.cnt[b] = 0u;
    }
}

// Exact masses of the 8 steps of 128 elements starting at element e0 of a
// row (one warp; lane k of the result holds step k's total, k < 8).
__device__ __forceinline__ unsigned long long warp_step_masses(const float *prow, const float *qrow,
                                                               int residual, int64_t e0, int64_t V,
                                                               bool vec4, int lane)
{
    float4 xp[8], xq[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int64_t e = e0 + k * kStep + lane * 4;
        xp[k] = e < V ? load4(prow, e, V, vec4, 0.f) : make_float4(0, 0, 0, 0);
        xq[k] = (residual && e < V) ? load4(qrow, e, V, vec4, 0.f) : make_float4(0, 0, 0, 0);
    }
    unsigned long long mine = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const unsigned long long m = mass(xp[k].x, xq[k].x, residual) + mass(xp[k].y, xq[k].y, residual) +
                                     mass(xp[k].z, xq[k].z, residual) + mass(xp[k].w, xq[k].w, residual);
        const unsigned long long t = warp_sum_u64(m);
        if (lane == k) mine = t;
    }
    return mine;
}

// Stage 2: every CTA streams one 8192-element chunk of the row its
// sequence needs (the residual row j, or the bonus row D) and writes the
// exact mass of each 128-element step.  The last CTA of a sequence to
// finish finds the crossing of u * Z in the running sum from the step
// masses and re-reads only the 128 elements of that step.
__global__ void __launch_bounds__(kThreads, 2) accept_stream_kernel(
    const float *__restrict__ p, const float *__restrict__ q, const float *__restrict__ u_res,
    int D, int V, int nchunks, SampleScratch sc, int32_t *__restrict__ n_accepted,
    int32_t *__restrict__ token, uint32_t *dev_status, bool vec4)
{
    __shared__ unsigned long long s_wsum[kWarps];
    __shared__ unsigned long long s_run;
    __shared__ int s_step, s_last;
    const int b = blockIdx.y, chunk = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = sc.js[b];
    const float *prow = p + (static_cast<int64_t>(b) * (D + 1) + j) * V;
    const float *qrow = j < D ? q + (static_cast<int64_t>(b) * D + j) * V : nullptr;
    int residual = j < D;
    unsigned long long *steps = sc.steps + static_cast<int64_t>(b) * sc.nsteps;

    {
        const int64_t e0 = static_cast<int64_t>(chunk) * kChunk + warp * kWarpElems;
        const unsigned long long t = warp_step_masses(prow, qrow, residual, e0, V, vec4, lane);
        const int s0 = static_cast<int>(e0 / kStep);
        if (lane < 8 && s0 + lane < sc.nsteps) steps[s0 + lane] = t;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&sc.cnt[b], 1u) == static_cast<unsigned>(nchunks - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    float u = u_res[b];
    if (!(u >= 0.0f && u < 1.0f)) {
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_UNIFORM);
        u = (u >= 1.0f) ? 0x1.fffffep-1f : 0.0f;
    }
    for (int attempt = 0; attempt < 2; ++attempt) {
        // Block-wide exclusive scan of the step masses, 4 consecutive steps per
        // thread per pass.
        const int per_pass = kThreads * 4;
        unsigned long long Z = 0;
        for (int s0 = 0; s0 < sc.nsteps; s0 += per_pass) {
            unsigned long long t = 0;
            for (int k = 0; k < 4; ++k) {
                const int st = s0 + threadIdx.x * 4 + k;
                if (st < sc.nsteps) t += __ldcg(steps + st);
            }
            t = warp_sum_u64(t);
            if (lane == 0) s_wsum[warp] = t;
            __syncthreads();
            for (int w = 0; w < kWarps; ++w) Z += s_wsum[w];
            __syncthreads();
        }
        if (Z == 0) {
            if (residual) {
                // reading: max(0, p - q) has no mass -> draw from the target row
                // itself; this CTA recomputes the step masses of p alone
                residual = 0;
                if (threadIdx.x == 0) report(dev_status, SPEC_DEV_INFO_ZERO_RESIDUAL);
                for (int64_t e0 = warp * kWarpElems; e0 < V; e0 += kChunk) {
                    const unsigned long long t = warp_step_masses(prow, nullptr, 0, e0, V, vec4, lane);
                    const int s0 = static_cast<int>(e0 / kStep);
                    if (lane < 8 && s0 + lane < sc.nsteps) steps[s0 + lane] = t;
                }
                __threadfence_block();
                __syncthreads();
                continue;
            }
            if (threadIdx.x == 0) {
                report(dev_status, SPEC_DEV_ERR_ZERO_MASS);
                n_accepted[b] = j;
                token[b] = 0;
                sc.cnt[b] = 0u;
            }
            return;
        }
        const unsigned long long T = scaled_threshold(u, Z);
        // Locate the step holding the crossing: smallest step s with
        // prefix(s) <= T < prefix(s) + mass(s).
        if (threadIdx.x == 0) s_step = -1;
        unsigned long long base = 0;
        for (int s0 = 0; s0 < sc.nsteps; s0 += per_pass) {
            unsigned long long v[4], t = 0;
            for (int k = 0; k < 4; ++k) {
                const int st = s0 + threadIdx.x * 4 + k;
                v[k] = st < sc.nsteps ? __ldcg(steps + st) : 0ull;
                t += v[k];
            }
            const unsigned long long incl = warp_incl_scan_u64(t, lane);
            if (lane == 31) s_wsum[warp] = incl;
            __syncthreads();
            unsigned long long wpre = base, all = 0;
            for (int w = 0; w < kWarps; ++w) {
                if (w < warp) wpre += s_wsum[w];
                all += s_wsum[w];
            }
            unsigned long long run = wpre + incl - t;
            if (run <= T && T < run + t) {
                for (int k = 0; k < 4; ++k) {
                    if (T < run + v[k]) {
                        s_step = s0 + threadIdx.x * 4 + k;
                        s_run = run;
                        break;
                    }
                    run += v[k];
                }
            }
            base += all;
            __syncthreads();
        }
        if (warp == 0 && s_step >= 0) {
            const int64_t e = static_cast<int64_t>(s_step) * kStep + lane * 4;
            const float4 xp = e < V ? load4(prow, e, V, vec4, 0.f) : make_float4(0, 0, 0, 0);
            const float4 xq = (residual && e < V) ? load4(qrow, e, V, vec4, 0.f) : make_float4(0, 0, 0, 0);
            const unsigned long long m[4] = {mass(xp.x, xq.x, residual), mass(xp.y, xq.y, residual),
                                             mass(xp.z, xq.z, residual), mass(xp.w, xq.w, residual)};
            const unsigned long long lane_sum = m[0] + m[1] + m[2] + m[3];
            const unsigned long long incl = warp_incl_scan_u64(lane_sum, lane);
            const unsigned long long run = s_run;
            const unsigned hit = __ballot_sync(0xffffffffu, run + incl > T);
            const int Lh = hit ? __ffs(hit) - 1 : 31;
            if (lane == Lh) {
                unsigned long long c = run + incl - lane_sum;
                int v = static_cast<int>(e);
                for (int k = 0; k < 4; ++k) {
                    c += m[k];
                    if (c > T) { v = static_cast<int>(e) + k; break; }
                }
                token[b] = v;
            }
        }
        break;
    }
    if (threadIdx.x == 0) {
        n_accepted[b] = j;
        sc.cnt[b] = 0u;     // ready for the next call
    }
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

size_t accept_sample_workspace_bytes(int B, int V)
{
    const size_t nsteps = (static_cast<size_t>(V) + kStep - 1) / kStep;
    return 2 * align256(sizeof(int32_t) * static_cast<size_t>(B)) +
           align256(sizeof(unsigned long long) * nsteps * static_cast<size_t>(B));
}

cudaError_t launch_accept_sample(const float *p, const float *q, const int32_t *draft,
                                 const float *u_acc, const float *u_res, int B, int D, int V,
                                 int32_t *n_acc, int32_t *token, void *workspace,
                                 uint32_t *dev_status, cudaStream_t st)
{
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                      (q == nullptr || reinterpret_cast<uintptr_t>(q) % 16 == 0);
    char *w = static_cast<char *>(workspace);
    SampleScratch sc;
    sc.js = reinterpret_cast<int32_t *>(w);
    sc.cnt = reinterpret_cast<uint32_t *>(w + align256(sizeof(int32_t) * B));
    sc.steps = reinterpret_cast<unsigned long long *>(w + 2 * align256(sizeof(int32_t) * B));
    sc.nsteps = (V + kStep - 1) / kStep;
    accept_prep_kernel<<<(B + kWarps - 1) / kWarps, kThreads, 0, st>>>(p, q, draft, u_acc, B, D, V, sc, dev_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int nchunks = (V + kChunk - 1) / kChunk;
    accept_stream_kernel<<<dim3(nchunks, B), kThreads, 0, st>>>(p, q, u_res, D, V, nchunks, sc, n_acc, token,
                                                               dev_status, vec4);
    return cudaGetLastError();
}

}  // namespace spec
