// Batched accept/reject kernels for the verification step.
//
// Greedy: keep the longest draft prefix the target agrees with and add one
// target token (LLM inference handbook, "How speculative decoding works").
// Stochastic: accept x with probability min(1, p(x)/q(x)); at the first
// rejection resample from max(0, p - q) renormalised (llm-digest,
// "Mechanism" and "Math intuition").
//
// Greedy: one thread-block cluster of CS CTAs per sequence; CTA `rank`
// owns a contiguous slice of the vocabulary and each of its 8 warps a
// contiguous sub-slice, streamed in 128-element steps (one float4 per lane,
// coalesced).  Cluster-wide reductions go through distributed shared
// memory.  Stochastic: three kernels chained by programmatic dependent
// launch (first rejection per sequence; a persistent streaming kernel that
// stages the needed rows by bulk copies and writes exact slice masses; a
// warp per sequence that draws the token).
//
// Exactness: the accept test u*q < p is evaluated in fp64, where the
// product of two fp32 values is exact.  The residual of an element is
// max(0, p - q) with the difference rounded to fp32; residual / bonus masses
// are summed in 64-bit fixed point (2^-61 resolution, truncation of each
// element), so every partial sum is exact and independent of the summation
// order; the draw compares running sums against floor(u * Z) computed
// exactly from the 24-bit mantissa of u.  Against the exact real-number
// residual, each element is off by at most 2^-24 of its value, so a draw
// can differ from the exact one only within 2^-23 Z of a CDF boundary.
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

// Programmatic dependent launch: let the next kernel on the stream be
// scheduled now / wait until the previous one's results are visible.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

__device__ __forceinline__ unsigned long long pack_argmax(ArgMax a)
{
    const uint32_t lo = a.i == INT_MAX ? 0xFFFFFFFFu : static_cast<uint32_t>(a.i);
    return (static_cast<unsigned long long>(__float_as_uint(a.v)) << 32) | lo;
}

__device__ __forceinline__ ArgMax unpack_argmax(unsigned long long w)
{
    const uint32_t lo = static_cast<uint32_t>(w);
    return {__uint_as_float(static_cast<uint32_t>(w >> 32)), lo == 0xFFFFFFFFu ? INT_MAX : static_cast<int>(lo)};
}



constexpr int kGUnroll = 8;    // greedy: 128-element steps whose loads are in flight together

// Greedy acceptance: one thread-block cluster of CS CTAs per sequence, CTA
// `rank` owning a contiguous slice of the vocabulary.  Row by row, each CTA
// reduces its slice to an argmax and sends the result to every CTA of the
// cluster with an asynchronous distributed-shared-memory store that
// completes on the receiver's mbarrier; every CTA then reduces the CS
// results itself and takes the same decision, so no cluster-wide barrier
// sits on the per-row path.  Only rows 0..n_accepted are read.
// BULK (rows 16-byte aligned): each row's slice is staged in shared memory
// in chunks of kGChunk elements, kGSlots of them in flight at once, issued
// by one thread -- no loads held in registers, the arithmetic on a chunk
// starting as soon as it lands; a slice longer than the ring (64 KB at
// V = 131072 against a 48 KB ring, which keeps 4 CTAs on an SM) streams
// through it; thread 0 issues the next row's copies as soon as it has the
// row's decision.  Otherwise every lane loads its elements with register
// loads, kGUnroll 128-element steps in flight.
// The cluster barrier that orders the peers' mbarrier initialisation before
// the first exchange is split: arrived at before row 0 is read, waited for
// only before row 0's result is sent; row 0's copies go out before the
// drafts are read.
// Measured (B = 256, V = 131072): a per-cluster timestamp trace shows a
// cluster living ~7.3 us for a one-row sequence, 2.7 us of it copies, the
// rest start-up, the wait for the cluster's slowest slice plus the exchange
// (~1.7 us) and the final cluster barrier (~1.3 us); one sequence alone
// takes 10.3 us end to end, while each further row costs about its bytes at
// the HBM rate.  Two sequences per cluster (each CTA split into two
// independent halves), 5 or 6 CTAs per SM with smaller rings, and 8 KB
// copies all measured within 3% of this form.
// TREE: the 1 + D rows are the nodes of a draft tree (parent[b][k] < k,
// node tokens tokens[b][k]); from the root the walk moves to the child whose
// token equals the row's argmax (lowest node index among such siblings) and
// stops when none does.  The chain is the tree parent[k] = k - 1 whose node
// k carries draft k - 1.
constexpr int kGChunk = 4096;                                    // elements per bulk copy (16 KB)
constexpr int kGSlots = 3;                                       // copies in flight per CTA
constexpr uint32_t kGSmem = kGSlots * kGChunk * 4 + 128;         // ring + alignment slack
constexpr int kGMinBlocks = 4;                                   // CTAs per SM (4 rings of 48 KB)


template <int CS, bool TREE, bool BULK>
__global__ void __launch_bounds__(kThreads, kGMinBlocks) accept_greedy_kernel(
    const float *__restrict__ p, const int32_t *__restrict__ draft, const int32_t *__restrict__ parent,
    int D, int V, int32_t *__restrict__ n_accepted, int32_t *__restrict__ token, int32_t *__restrict__ path,
    uint32_t *dev_status, bool vec4)
{
    extern __shared__ uint8_t s_graw[];
    float *ring = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(s_graw) + 127) & ~uintptr_t(127));
    __shared__ ArgMax s_warp[kWarps];
    __shared__ __align__(8) unsigned long long s_res[2][CS];   // per row parity, one per CTA
    __shared__ uint64_t s_bar[2];
    __shared__ uint64_t s_full[kGSlots];
    __shared__ int32_t s_draft[kMaxDraft + 1];   // chain: drafts; tree: node tokens
    __shared__ int32_t s_par[TREE ? kMaxDraft + 1 : 1];
    __shared__ int s_abort, s_bad;
    if (cluster_ctas() != static_cast<uint32_t>(CS)) {   // uniform over the grid
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        return;
    }
    const int rank = CS > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int b = blockIdx.x / CS;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Slice sl = warp_slice(V, CS, rank, warp);   // register loads: this warp's elements
    // this CTA's slice [c0, c0 + n) (BULK: a multiple of 4 elements, V % 4 == 0)
    const int64_t cta_len = ((static_cast<int64_t>(V) + CS - 1) / CS + 3) & ~int64_t(3);
    const int64_t c0 = imin64(V, cta_len * rank);
    const int n = static_cast<int>(imin64(V, c0 + cta_len) - c0);
    const int nchunks = (n + kGChunk - 1) / kGChunk;
    volatile int *abort = reinterpret_cast<volatile int *>(&s_abort);
    if (tid == 0) {
        s_bad = 0;
        mbar_init(&s_bar[0], 1);
        mbar_init(&s_bar[1], 1);
        for (int k = 0; k < kGSlots; ++k) mbar_init(&s_full[k], 1);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if constexpr (CS > 1) cluster_arrive_relaxed();   // waited for before the first send
    uint32_t issued[kGSlots] = {};   // thread 0: copies issued per slot (its phase count)
    uint32_t used = 0;               // every thread: chunks consumed so far (slot c % kGSlots)
    // thread 0: arm row i's exchange barrier and copy the first chunks of
    // its slice (row index r of sequence b) into the ring
    auto issue_row = [&](int i, int r) {
        if (CS > 1) mbar_arrive_expect_tx(&s_bar[i & 1], CS * 8);
        if (!BULK) return;
        const float *src = p + (static_cast<int64_t>(b) * (D + 1) + r) * V + c0;
        for (int c = 0; c < nchunks && c < kGSlots; ++c) {
            const uint32_t bytes = static_cast<uint32_t>(imin64(kGChunk, n - c * kGChunk)) * 4u;
            const int slot = static_cast<int>((used + c) % kGSlots);
            mbar_arrive_expect_tx(&s_full[slot], bytes);
            bulk_load(ring + slot * kGChunk, src + c * kGChunk, bytes, &s_full[slot]);
            ++issued[slot];
        }
    };
    // row 0 (the root's row) travels while the drafts are read
    if (tid == 0) issue_row(0, 0);
    if constexpr (TREE) {
        for (int k = tid; k <= D; k += kThreads) {
            s_draft[k] = draft[static_cast<int64_t>(b) * (D + 1) + k];
            const int pa = parent[static_cast<int64_t>(b) * (D + 1) + k];
            s_par[k] = pa;
            if (k == 0 ? pa != -1 : (pa < 0 || pa >= k)) s_bad = 1;
        }
    } else {
        for (int i = tid; i < D; i += kThreads) s_draft[i] = draft[static_cast<int64_t>(b) * D + i];
    }
    __syncthreads();

    // a malformed tree is reported and walked as a lone root
    if (TREE && s_bad && rank == 0 && tid == 0) report(dev_status, SPEC_DEV_ERR_TREE);
    int node = 0;                    // tree: the node whose row this iteration reads
    for (int i = 0; i <= D; ++i) {
        const int par = i & 1;
        const float *row = p + (static_cast<int64_t>(b) * (D + 1) + (TREE ? node : i)) * V + c0;
        // Per lane, elements are visited in increasing index order; only a
        // strictly larger value replaces the best, so ties keep the lowest
        // index.  The index is located only when a float4's max wins.
        ArgMax best{-FLT_MAX, INT_MAX};
        bool ok = true;
        if constexpr (!BULK) {
            const float *grow = p + (static_cast<int64_t>(b) * (D + 1) + (TREE ? node : i)) * V;
            for (int64_t base = sl.begin; base < sl.end; base += kStep * kGUnroll) {
                float4 x[kGUnroll];
#pragma unroll
                for (int u = 0; u < kGUnroll; ++u) {
                    const int64_t e = base + u * kStep + lane * 4;
                    x[u] = e < sl.end ? load4(grow, e, sl.end, vec4, -INFINITY)
                                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
#pragma unroll
                for (int u = 0; u < kGUnroll; ++u) {
                    const int e = static_cast<int>(base) + u * kStep + lane * 4;
                    const float m4 = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
                    if (e < sl.end && (m4 > best.v || (best.i == INT_MAX && m4 == m4))) {
                        const int k = x[u].x == m4 ? 0 : x[u].y == m4 ? 1 : x[u].z == m4 ? 2 : 3;
                        if (e + k < sl.end) best = {m4, e + k};
                    }
                }
            }
        }
        // BULK: every thread runs every chunk iteration (a failed wait only
        // skips the arithmetic), so the refill barriers below always pair up
        for (int c = 0; BULK && c < nchunks; ++c, ++used) {
            const int slot = static_cast<int>(used % kGSlots);
            if (ok) ok = mbar_wait(&s_full[slot], (used / kGSlots) & 1u, abort, dev_status);
            if (ok) {
                const float *src = ring + slot * kGChunk;
                const int len = static_cast<int>(imin64(kGChunk, n - c * kGChunk));
                const int gbase = static_cast<int>(c0) + c * kGChunk;
#pragma unroll 4
                for (int e = tid * 4; e < len; e += kThreads * 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(src + e);
                    const float m4 = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
                    if (m4 > best.v || (best.i == INT_MAX && m4 == m4)) {
                        const int k = x.x == m4 ? 0 : x.y == m4 ? 1 : x.z == m4 ? 2 : 3;
                        best = {m4, gbase + e + k};
                    }
                }
            }
            if (c + kGSlots < nchunks) {   // a slice longer than the ring: refill this slot
                __syncthreads();
                if (tid == 0 && !*abort) {
                    const uint32_t bytes =
                        static_cast<uint32_t>(imin64(kGChunk, n - (c + kGSlots) * kGChunk)) * 4u;
                    mbar_arrive_expect_tx(&s_full[slot], bytes);
                    bulk_load(ring + slot * kGChunk, row + (c + kGSlots) * kGChunk, bytes, &s_full[slot]);
                    ++issued[slot];
                }
            }
        }
        ok = __syncthreads_and(ok);
        best = warp_argmax(best);
        if (lane == 0) s_warp[warp] = best;
        if constexpr (CS > 1) {
            if (i == 0) cluster_wait_acquire();   // every peer's barriers are initialised
        }
        __syncthreads();
        if (warp == 0 && ok) {
            ArgMax c = lane < kWarps ? s_warp[lane] : ArgMax{-FLT_MAX, INT_MAX};
            c = warp_argmax(c);
            // this CTA's result, to every CTA of the cluster (itself included)
            if (lane < CS) {
                const unsigned long long w = pack_argmax(c);
                if constexpr (CS > 1)
                    st_async_peer(peer_smem(&s_res[par][rank], lane), w, peer_smem(&s_bar[par], lane));
                else
                    s_res[par][0] = w;   // a lone CTA: its own result is the row's
            }
        }
        if constexpr (CS > 1) {
            if (ok) ok = mbar_wait_warp(&s_bar[par], (i >> 1) & 1, abort, dev_status);
        } else {
            __syncthreads();
        }
        ArgMax g{-FLT_MAX, INT_MAX};
#pragma unroll
        for (int r = 0; r < CS; ++r) g = better(g, unpack_argmax(s_res[par][r]));
        bool stop;
        int next = -1;
        if constexpr (TREE) {
            // the lowest-index child of `node` carrying the argmax (every
            // thread scans the same small tree, so all agree)
            if (ok && !s_bad)
                for (int k = node + 1; k <= D; ++k)
                    if (s_par[k] == node && s_draft[k] == g.i) { next = k; break; }
            stop = !ok || next < 0;
        } else {
            stop = !ok || i == D || s_draft[i] != g.i;
        }
        if (stop) {
            if (ok && rank == 0 && tid == 0) {
                n_accepted[b] = i;
                token[b] = g.i;
            }
            if (TREE && path && rank == 0)
                for (int x = i + tid; x < D; x += kThreads) path[static_cast<int64_t>(b) * D + x] = -1;
            break;
        }
        if constexpr (TREE) {
            if (path && rank == 0 && tid == 0) path[static_cast<int64_t>(b) * D + i] = next;
            node = next;
        }
        // The next row's copies go out as soon as thread 0 knows the
        // decision: every thread of this CTA finished reading the ring before
        // the barrier that precedes this row's send, and no thread rewrites
        // s_warp or s_res[par] before every CTA has sent its next result.
        if (tid == 0) issue_row(i + 1, TREE ? node : i + 1);
    }
    // unwind after a timed-out wait: let the copies in flight land
    if (tid == 0 && *abort)
        for (int k = 0; k < kGSlots; ++k)
            if (issued[k]) mbar_wait_drain(&s_full[k], (issued[k] - 1u) & 1u, kWaitTimeoutNs);
    // keep this CTA's shared memory alive until every peer is done with it
    if constexpr (CS > 1) cluster_exit_barrier();
}

// --------------------------------------------------------------- stochastic
// Fixed point with 2^-61 resolution: floor(x * 2^61) for 0 <= x < 2 (row
// sums of probabilities fit in 64 bits).  With x = m * 2^(E - 150), m the
// 24-bit significand and E the biased exponent, x * 2^61 = (m << 38) >>
// (127 - E).  m << 38 has a zero low word, so this is one 32-bit shift and
// one 64-bit right shift.  PTX clamps shift counts, so zero and denormals
// (E = 0), negatives (the sign bit makes E >= 256), x >= 2, infinities and
// NaN all give 0 without special cases.  Integer work only: the
// float-to-64-bit-integer conversion runs on the small fp64 pipe.
__device__ __forceinline__ unsigned long long fix61(float x)
{
    const uint32_t bits = __float_as_uint(x);
    const uint32_t m = (bits & 0x7FFFFFu) | 0x800000u;
    const uint32_t sh = 127u - (bits >> 23);
    unsigned long long r;
    asm("{\n\t.reg .b64 t;\n\t"
        "mov.b64 t, {%2, %3};\n\t"
        "shr.b64 %0, t, %1;\n\t}"
        : "=l"(r)
        : "r"(sh), "r"(0u), "r"(m << 6));
    return r;
}

// Mass of one element: p, or the residual max(0, p - q) with the difference
// rounded to fp32 (round to nearest).  Each element's mass is then exact in
// the fixed point, so every sum of masses is exact and order-independent.
__device__ __forceinline__ unsigned long long mass(float pv, float qv, int residual)
{
    return fix61(residual ? fmaxf(__fsub_rn(pv, qv), 0.0f) : pv);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// The same sum; ovf is set when it wraps past 2^64 (a row whose
// probabilities sum to 8 or more overflows the 2^-61 fixed point).
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x, bool &ovf)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long y = x + __shfl_xor_sync(0xffffffffu, x, o);
        ovf |= y < x;
        x = y;
    }
    return x;
}

// Range checks of the probability form, cheap enough for the streaming
// loop.  A value the fixed point represents, 0 <= x < 2 (+0 included, NaN
// not), has bits below 0x40000000: one unsigned max per element covers
// negative values, NaN, infinities and x >= 2 at once.  A group's 512
// masses wrap their 64-bit sums only if they add up to 8 or more; each
// lane keeps the sum of its 4-element masses >> 40 (a 32-bit shadow, at
// most 2 lost per step), and only when some lane's shadow reaches a
// 32nd of the bound is the warp's total formed.
constexpr uint32_t kFixRangeBits = 0x40000000u;        // bits of 2.0f
constexpr uint32_t kShadowBound = (1u << 24) - 128u;   // 2^64 >> 40, less the truncation
__device__ __forceinline__ uint32_t max_bits4(uint32_t acc, float4 r)
{
    return max(max(acc, max(__float_as_uint(r.x), __float_as_uint(r.y))),
               max(__float_as_uint(r.z), __float_as_uint(r.w)));
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

// ------------------------------------------------------- from logits
// The logits form takes p = softmax(zp / T) and q = softmax(zq / T).  Its
// probabilities are the fp32 roundings of the exact softmax -- the fp32
// probability rows the probability form takes -- evaluated two ways:
//  * the accept tests and the row statistics use a fast evaluation: m =
//    max_v z_v, Zf = sum_v 2^((z_v - m) c) with c = fl32(log2 e / T), the
//    hardware base-2 exponential and fp32 sums in a fixed order, and
//    p(x) = 2^((z_x - m) c) / Zf.  Its relative error (about 1e-7, up to
//    1e-6 far below the maximum) can change a decision only when the
//    uniform lies that close to p(x) / q(x);
//  * the one row each sequence draws from (max(0, p_j - q_j), or p_D) is
//    evaluated exactly up to the final rounding: (z - m) / T and exp in
//    double-float arithmetic (unevaluated fp32 pairs hi + lo), the sum Z
//    in double-float, and p_v = e_v / Z rounded to fp32 once.  Each p_v
//    then is the nearest fp32 to the exact softmax unless the exact value
//    lies within about 2^-33 (relative) of a rounding tie.

// Two fp32 values in one 64-bit register (element 0 in the low word) for
// the packed fp32x2 instructions: each rounds both halves exactly like the
// scalar instruction.
using F32x2 = unsigned long long;

__device__ __forceinline__ F32x2 pack2(float lo, float hi)
{
    return (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo_of(F32x2 v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_of(F32x2 v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ F32x2 add2(F32x2 a, F32x2 b)
{
    F32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ F32x2 sub2(F32x2 a, F32x2 b)
{
    F32x2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ F32x2 mul2(F32x2 a, F32x2 b)
{
    F32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ F32x2 fma2(F32x2 a, F32x2 b, F32x2 c)
{
    F32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ F32x2 neg2(F32x2 a) { return a ^ 0x8000000080000000ull; }
__device__ __forceinline__ F32x2 splat2(float x) { return pack2(x, x); }

struct DF {
    float hi, lo;   // the unevaluated sum hi + lo
};

// a + b exactly as hi + lo (Knuth's two-sum; every step rounds to nearest)
__device__ __forceinline__ DF two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, err};
}

// a + b for double-float values, renormalised
__device__ __forceinline__ DF df_add(DF a, DF b)
{
    const DF s = two_sum(a.hi, b.hi);
    const float lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
    const float hi = __fadd_rn(s.hi, lo);
    return {hi, __fsub_rn(lo, __fsub_rn(hi, s.hi))};
}

// 2^(j / 256) for j = 0..255 as (hi, lo) fp32 pairs in the calling CTA's
// shared memory: fp64 products of the constants 2^(2^i / 256), i = 0..7
// (at most eight roundings of 2^-53 each).  Ends with __syncthreads.
__device__ void build_exp2_table(float2 *tab)
{
    const double c[8] = {0x1.00b1afa5abcbfp+0, 0x1.0163da9fb3335p+0, 0x1.02c9a3e778061p+0,
                         0x1.059b0d3158574p+0, 0x1.0b5586cf9890fp+0, 0x1.172b83c7d517bp+0,
                         0x1.306fe0a31b715p+0, 0x1.6a09e667f3bcdp+0};
    for (int j = threadIdx.x; j < 256; j += blockDim.x) {
        double v = 1.0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if ((j >> i) & 1) v = __dmul_rn(v, c[i]);
        const float hi = __double2float_rn(v);
        tab[j] = make_float2(hi, __double2float_rn(__dsub_rn(v, static_cast<double>(hi))));
    }
    __syncthreads();
}

// Parameters of one logits row for the exact evaluation: 1/T = ih + il,
// 1/Z = rh + rl (rh = 0: the row has no softmax, every probability is 0).
struct SoftmaxRow {
    float m, ih, il, rh, rl;
};

// exp(yh + yl) for yh + yl <= 0 as a double-float value, relative error
// about 2^-33; 0 below -83 (e^-83 < 2^-119) and for -inf.
//   k = rint((yh) 256 / ln 2);  r = y - k ln2 / 256, with ln2 / 256 split
//   as C1 + C2 + C3 (C1 has 8 significant bits, so k C1 is exact for
//   |k| < 2^15, and the first fused multiply-add is exact);  |r| <= ~ln2 /
//   512;  e^r - 1 = r + r^2 (1/2 + r/6 + r^2/24) (Taylor, the next term
//   is below 2^-41);  exp(y) = 2^(k >> 8) 2^((k & 255) / 256) e^r.
// Evaluated on a pair of elements at a time with packed fp32x2
// instructions: k is taken with the 1.5 * 2^23 rounding trick (fma(y,
// 256/ln2, 1.5 * 2^23) holds 1.5 * 2^23 + k in its significand, so its bits
// are 0x4B400000 + k), and lanes below -83 are computed on a clamped
// argument and zeroed at the end.  The probability is the double-float
// quotient e / Z = (e_hi + e_lo)(1/Z_hi + 1/Z_lo) rounded once.
struct DF2 {
    F32x2 hi, lo;
};

__device__ __forceinline__ DF2 two_sum2(F32x2 a, F32x2 b)
{
    const F32x2 s = add2(a, b);
    const F32x2 bb = sub2(s, a);
    return {s, add2(sub2(a, sub2(s, bb)), sub2(b, bb))};
}

// A row's exact-evaluation parameters on both lanes.
struct SoftmaxPair {
    F32x2 neg_m, ih, il, rh, rl;
    bool unit_t;   // T = 1: (z - m) / T = z - m
    bool none;     // no softmax: every probability 0
};

__device__ __forceinline__ SoftmaxPair softmax_pair(const SoftmaxRow &r)
{
    return {splat2(-r.m), splat2(r.ih), splat2(r.il), splat2(r.rh), splat2(r.rl),
            r.ih == 1.0f && r.il == 0.0f, r.rh == 0.0f};
}

__device__ __forceinline__ DF2 softmax_exp2(F32x2 z, const SoftmaxPair &r, const float2 *tab)
{
    const DF2 d = two_sum2(z, r.neg_m);   // z - m exactly
    F32x2 yh = d.hi, yl = d.lo;
    if (!r.unit_t) {
        yh = mul2(d.hi, r.ih);
        yl = add2(fma2(d.hi, r.ih, neg2(yh)), fma2(d.hi, r.il, mul2(d.lo, r.ih)));
    }
    const float y0 = lo_of(yh), y1 = hi_of(yh);
    const bool z0 = !(y0 >= -83.0f), z1 = !(y1 >= -83.0f);
    const F32x2 yc = pack2(z0 ? -83.0f : y0, z1 ? -83.0f : y1);
    const F32x2 magic = splat2(0x1.8p+23f);
    const F32x2 rk = fma2(yc, splat2(0x1.715476p+8f), magic);   // 1.5 * 2^23 + k
    const F32x2 nk = sub2(magic, rk);                           // -k
    F32x2 t = fma2(nk, splat2(0x1.62p-9f), yc);
    t = fma2(nk, splat2(0x1.c85fep-18f), t);
    t = fma2(nk, splat2(-0x1.718432p-43f), t);
    const F32x2 rr = add2(t, yl);
    F32x2 sp = fma2(rr, splat2(0x1.555556p-5f), splat2(0x1.555556p-3f));
    sp = fma2(sp, rr, splat2(0.5f));
    sp = mul2(mul2(sp, rr), rr);
    const F32x2 em1 = add2(rr, sp);
    const int k0 = static_cast<int>(static_cast<uint32_t>(rk)) - 0x4B400000;
    const int k1 = static_cast<int>(static_cast<uint32_t>(rk >> 32)) - 0x4B400000;
    const float2 t0 = tab[k0 & 255], t1 = tab[k1 & 255];
    const F32x2 sc = pack2(__int_as_float(((k0 >> 8) + 127) << 23), __int_as_float(((k1 >> 8) + 127) << 23));
    const F32x2 th = pack2(t0.x, t1.x), tl = pack2(t0.y, t1.y);
    F32x2 eh = mul2(th, sc), el = mul2(fma2(th, em1, tl), sc);
    if (z0 | z1) {
        const F32x2 keep = (z0 ? 0ull : 0xFFFFFFFFull) | (z1 ? 0ull : 0xFFFFFFFF00000000ull);
        eh &= keep;
        el &= keep;
    }
    return {eh, el};
}

// softmax_prob of two elements.
__device__ __forceinline__ F32x2 softmax_prob2(F32x2 z, const SoftmaxPair &r, const float2 *tab)
{
    if (r.none) return 0ull;
    const DF2 e = softmax_exp2(z, r, tab);
    const F32x2 qh = mul2(e.hi, r.rh);
    const F32x2 ql = add2(fma2(e.hi, r.rh, neg2(qh)), fma2(e.hi, r.rl, mul2(e.lo, r.rh)));
    return add2(qh, ql);
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The fast probability of the accept tests from the row statistics (m, Zf)
// and c = fl32(log2 e / T); 0 for a row without a softmax (Zf = +inf).
__device__ __forceinline__ float fast_prob(float z, float2 stat, float c)
{
    if (!(stat.y < INFINITY)) return 0.0f;
    return __fdiv_rn(ex2_approx(__fmul_rn(__fsub_rn(z, stat.x), c)), stat.y);
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): word 0 for counter (c0, c1, stream, 0) and key
// = seed; the uniform is its top 24 bits times 2^-24.
__device__ __forceinline__ float philox_u(unsigned long long seed, uint32_t c0, uint32_t c1, uint32_t stream)
{
    uint32_t x0 = c0, x1 = c1, x2 = stream, x3 = 0u;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, x0), lo0 = 0xD2511F53u * x0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, x2), lo1 = 0xCD9E8D57u * x2;
        const uint32_t n0 = hi1 ^ x1 ^ k0, n2 = hi0 ^ x3 ^ k1;
        x0 = n0; x1 = lo1; x2 = n2; x3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return __fmul_rn(__uint2float_rn(x0 >> 8), 0x1p-24f);
}

// Inputs of the stochastic acceptance.  Probability form: p, q and the
// uniforms u_acc, u_res.  Logits form: p, q hold the target / draft logits,
// stats the fast statistics (m, Zf) of every row -- row b (2D + 1) + k is
// target row k for k <= D and draft row k - D - 1 otherwise -- zparts the
// double-float partial sums of exp((z - m) / T) over the nzchunks chunks of
// each sequence's draw rows ([b][0]: the target row, [b][1]: the draft
// row), and the uniforms come from Philox with key `seed`: u_acc[b][i] from
// counter (b, i, 0, 0), u_res[b] from (b, 0, 1, 0).
struct SampleIn {
    const float *p, *q;
    const float *u_acc, *u_res;
    const float2 *stats;
    const float2 *zparts;
    int nzchunks;
    float c_fast;          // fl32(log2 e / T)
    float ih, il;          // 1 / T as a double-float value
    unsigned long long seed;
};

// The exact-evaluation parameters of row k (0..2D) of sequence b, which is
// its draw row `which` (0: target, 1: draft): Z is the sum of the row's
// partial sums in chunk order, 1 / Z refined by one Newton step.  Every
// caller computes the same value from the same inputs.
template <bool LOGITS>
__device__ __forceinline__ SoftmaxRow draw_row(const SampleIn &in, int b, int D, int k, int which)
{
    SoftmaxRow r{0.0f, 1.0f, 0.0f, 1.0f, 0.0f};
    if (LOGITS) {
        const float2 st = __ldcg(in.stats + static_cast<int64_t>(b) * (2 * D + 1) + k);
        r.m = st.x;
        r.ih = in.ih;
        r.il = in.il;
        if (!(st.y < INFINITY)) {
            r.rh = 0.0f;
            return r;
        }
        DF Z{0.0f, 0.0f};
        const float2 *zp = in.zparts + (static_cast<int64_t>(b) * 2 + which) * in.nzchunks;
        for (int c = 0; c < in.nzchunks; ++c) {
            const float2 t = __ldcg(zp + c);
            Z = df_add(Z, DF{t.x, t.y});
        }
        const float rh = __frcp_rn(Z.hi);
        const float err = __fsub_rn(__fmaf_rn(-Z.hi, rh, 1.0f), __fmul_rn(Z.lo, rh));
        r.rh = rh;
        r.rl = __fmul_rn(rh, err);
    }
    return r;
}

template <bool LOGITS>
__device__ __forceinline__ float4 to_prob4(float4 z, const SoftmaxPair &r, const float2 *tab)
{
    if (!LOGITS) return z;
    const F32x2 a = softmax_prob2(pack2(z.x, z.y), r, tab), b = softmax_prob2(pack2(z.z, z.w), r, tab);
    return make_float4(lo_of(a), hi_of(a), lo_of(b), hi_of(b));
}

// Value read for an element past the end of a row: no mass either way.
template <bool LOGITS>
__device__ __forceinline__ float pad_value()
{
    return LOGITS ? -INFINITY : 0.0f;
}

// Scratch in the caller's workspace (see spec_accept_sample):
//   js    int32  [B]            the row j the token is drawn from, which is
//                               also n_accepted; kBonusFlag set when it is a
//                               bonus draw from p[j] (all proposed drafts
//                               accepted), clear for a residual draw from
//                               max(0, p[j] - q[j]) after a rejection
//   gtot  uint64 [B][ngroups]   exact residual / bonus mass of every group
//                               of 4 steps (512 elements)
//   steps uint64 [B][nsteps]    ... and of every 128-element step
struct SampleScratch {
    int32_t *js;
    unsigned long long *gtot;
    unsigned long long *steps;
    int nsteps, ngroups;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int32_t kBonusFlag = 1 << 30;

struct DrawRow {
    int j;          // row of the draw (= n_accepted)
    int residual;   // 1: max(0, p[j] - q[j]); 0: p[j]
};

__device__ __forceinline__ DrawRow decode_draw(int32_t v)
{
    return {v & ~kBonusFlag, (v & kBonusFlag) ? 0 : 1};
}

constexpr int kChunk = 8192;                   // elements of one work item
constexpr int kConsumers = 16;                 // consumer warps of the streaming kernel
constexpr int kGroupSteps = kChunk / kStep / kConsumers;   // 4
constexpr int kGroup = kGroupSteps * kStep;    // 512: one consumer warp's share of an item
constexpr int kRing = 3;                       // items staged at once per CTA
constexpr int kStreamThreads = (kConsumers + 1) * 32;   // + 1 producer warp
constexpr uint32_t kItemBytes = 2 * kChunk * 4;   // p and q slices of one item
constexpr uint32_t kStreamSmem = kRing * kItemBytes + 1024;


// Stage 1: first rejected draft of every sequence (one warp per sequence);
// the accept test u * q(x) < p(x) is evaluated in fp64, where the product
// is exact.
template <bool LOGITS>
__global__ void __launch_bounds__(kThreads) accept_prep_kernel(SampleIn in, const int32_t *__restrict__ draft,
                                                                int B, int D, int V, SampleScratch sc,
                                                                uint32_t *dev_status)
{
    pdl_launch_dependents();
    if (LOGITS) pdl_wait();   // the row softmax parameters come from the previous kernel
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
                float pv = in.p[(static_cast<int64_t>(b) * (D + 1) + i) * V + x];
                float qv = in.q[(static_cast<int64_t>(b) * D + i) * V + x];
                float uf;
                if (LOGITS) {
                    const float2 *st = in.stats + static_cast<int64_t>(b) * (2 * D + 1);
                    pv = fast_prob(pv, __ldcg(st + i), in.c_fast);
                    qv = fast_prob(qv, __ldcg(st + D + 1 + i), in.c_fast);
                    uf = philox_u(in.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i), 0u);
                } else {
                    uf = in.u_acc[static_cast<int64_t>(b) * D + i];
                    if (!(uf >= 0.0f && uf < 1.0f)) report(dev_status, SPEC_DEV_ERR_UNIFORM);
                }
                // the product of two fp32 values is exact in fp64
                rej = !(static_cast<double>(uf) * static_cast<double>(qv) < static_cast<double>(pv));
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, rej);
        if (m) {
            j = i0 + __ffs(m) - 1;
            break;
        }
    }
    if (lane == 0) sc.js[b] = j == D ? (j | kBonusFlag) : j;
}

// Exact masses of the kGroupSteps steps of 128 elements starting at element
// w0 of the n-element slice (sp, sq): staged in shared memory (SMEM,
// n % 4 == 0) or read from global memory.  Lane k of the result holds step
// k's total (k < kGroupSteps).
// Probability form: bad is set when a value turned into mass (max(0, p -
// q), or p for a bonus draw) is negative, NaN or 2 or more, or when the
// group's masses sum to about 8 or more (their 64-bit sums could wrap);
// the fixed point represents neither.
template <bool SMEM, bool LOGITS>
__device__ __forceinline__ unsigned long long warp_step_masses(const float *sp, const float *sq,
                                                               int residual, int w0, int n, bool vec4,
                                                               int lane, const SoftmaxPair &rp,
                                                               const SoftmaxPair &rq, const float2 *tab, bool &bad)
{
    unsigned long long mine = 0;
    uint32_t mb = 0, shadow = 0;
#pragma unroll
    for (int k = 0; k < kGroupSteps; ++k) {
        const int e = w0 + k * kStep + lane * 4;
        unsigned long long m = 0;
        if (e < n) {
            float4 xp, xq = make_float4(0, 0, 0, 0);
            if (SMEM) {
                xp = *reinterpret_cast<const float4 *>(sp + e);
                if (residual) xq = *reinterpret_cast<const float4 *>(sq + e);
            } else {
                xp = load4(sp, e, n, vec4, pad_value<LOGITS>());
                if (residual) xq = load4(sq, e, n, vec4, pad_value<LOGITS>());
            }
            xp = to_prob4<LOGITS>(xp, rp, tab);
            if (residual) xq = to_prob4<LOGITS>(xq, rq, tab);
            float4 r;
            if (residual) {
                r = make_float4(fmaxf(__fsub_rn(xp.x, xq.x), 0.0f), fmaxf(__fsub_rn(xp.y, xq.y), 0.0f),
                                fmaxf(__fsub_rn(xp.z, xq.z), 0.0f), fmaxf(__fsub_rn(xp.w, xq.w), 0.0f));
            } else if (!LOGITS) {
                // x + 0 turns -0 into +0, the one sign-bit value the range check must pass
                r = make_float4(__fadd_rn(xp.x, 0.0f), __fadd_rn(xp.y, 0.0f), __fadd_rn(xp.z, 0.0f),
                                __fadd_rn(xp.w, 0.0f));
            } else {
                r = xp;
            }
            m = fix61(r.x) + fix61(r.y) + fix61(r.z) + fix61(r.w);
            if (!LOGITS) {
                mb = max_bits4(mb, r);
                shadow += static_cast<uint32_t>(m >> 40);
            }
        }
        const unsigned long long t = warp_sum_u64(m);
        if (lane == k) mine = t;
    }
    if (!LOGITS) {
        bad |= mb >= kFixRangeBits;
        if (__any_sync(0xffffffffu, shadow >= kShadowBound / 32u)) {
            uint32_t tot = shadow;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
            bad |= tot >= kShadowBound;
        }
    }
    return mine;
}

// Stage 2, persistent: each CTA takes work items (sequence b, 8192-element
// chunk of the one row b needs -- the residual row j, or the bonus row D)
// round robin.  The producer warp stages up to kRing items ahead in shared
// memory with bulk copies; each of the 16 consumer warps turns 512 elements
// of an item into 4 exact step masses and their group total.
// LOGITS: the staged slices are logits, turned into probabilities with the
// softmax parameters of their rows as they are consumed.
template <bool LOGITS>
__global__ void __launch_bounds__(kStreamThreads, 1) accept_stream_kernel(
    SampleIn in, int D, int V, int nchunks, int items, SampleScratch sc, uint32_t *dev_status, bool bulk)
{
    const float *__restrict__ p = in.p;
    const float *__restrict__ q = in.q;
    extern __shared__ uint8_t s_raw[];
    float *ring = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(s_raw) + 127) & ~uintptr_t(127));
    __shared__ uint64_t full[kRing], empty[kRing];
    __shared__ int s_j[kRing];
    __shared__ SoftmaxRow s_rp[kRing], s_rq[kRing];   // LOGITS: the draw rows' parameters
    __shared__ float2 s_tab[LOGITS ? 256 : 1];
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort = reinterpret_cast<volatile int *>(&s_abort);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kConsumers); }
        s_abort = 0;
        fence_mbar_init();
    }
    if (LOGITS) build_exp2_table(s_tab);
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait();   // js (and, for logits, the draw rows' sums) come from the previous kernels

    if (warp == kConsumers) {
        if (lane == 0) {
            for (int k = 0;; ++k) {
                const int item = blockIdx.x + k * gridDim.x;
                if (item >= items) break;
                const int slot = k % kRing;
                if (k >= kRing && !mbar_wait(&empty[slot], ((k / kRing) - 1) & 1, abort, dev_status)) break;
                const int b = item / nchunks, chunk = item % nchunks;
                const int32_t code = __ldcg(sc.js + b);
                s_j[slot] = code;
                const DrawRow dr = decode_draw(code);
                const int j = dr.j;
                if (LOGITS) {
                    s_rp[slot] = draw_row<true>(in, b, D, j, 0);
                    s_rq[slot] = dr.residual ? draw_row<true>(in, b, D, D + 1 + j, 1) : s_rp[slot];
                }
                if (bulk) {
                    const int64_t e0 = static_cast<int64_t>(chunk) * kChunk;
                    const uint32_t bytes = static_cast<uint32_t>(imin64(kChunk, V - e0)) * 4;  // % 16 == 0
                    float *dst = ring + slot * (2 * kChunk);
                    mbar_arrive_expect_tx(&full[slot], dr.residual ? 2 * bytes : bytes);
                    bulk_load(dst, p + (static_cast<int64_t>(b) * (D + 1) + j) * V + e0, bytes, &full[slot]);
                    if (dr.residual)
                        bulk_load(dst + kChunk, q + (static_cast<int64_t>(b) * D + j) * V + e0, bytes,
                                  &full[slot]);
                } else {
                    mbar_arrive(&full[slot]);   // consumers read global memory directly
                }
            }
        }
        return;
    }

    for (int k = 0;; ++k) {
        const int item = blockIdx.x + k * gridDim.x;
        if (item >= items) break;
        const int slot = k % kRing;
        if (!mbar_wait_warp(&full[slot], (k / kRing) & 1, abort, dev_status)) break;
        const int b = item / nchunks, chunk = item % nchunks;
        const DrawRow dr = decode_draw(s_j[slot]);
        const int j = dr.j;
        const int residual = dr.residual;
        SoftmaxRow rp{0.0f, 1.0f, 0.0f, 1.0f, 0.0f}, rq = rp;
        if (LOGITS) {
            rp = s_rp[slot];
            rq = s_rq[slot];
        }
        const int64_t e0 = static_cast<int64_t>(chunk) * kChunk;
        const int n = static_cast<int>(imin64(kChunk, V - e0));
        const float *sp, *sq;
        if (bulk) {
            sp = ring + slot * (2 * kChunk);
            sq = sp + kChunk;
        } else {
            sp = p + (static_cast<int64_t>(b) * (D + 1) + j) * V + e0;
            sq = residual ? q + (static_cast<int64_t>(b) * D + j) * V + e0 : nullptr;
        }
        bool bad = false;
        const unsigned long long t =
            bulk ? warp_step_masses<true, LOGITS>(sp, sq, residual, warp * kGroup, n, true, lane, softmax_pair(rp),
                                                   softmax_pair(rq), s_tab, bad)
                 : warp_step_masses<false, LOGITS>(sp, sq, residual, warp * kGroup, n, false, lane, softmax_pair(rp),
                                                   softmax_pair(rq), s_tab, bad);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);   // this warp is done with the slot
        const int s0 = chunk * (kChunk / kStep) + warp * kGroupSteps;
        if (lane < kGroupSteps && s0 + lane < sc.nsteps)
            sc.steps[static_cast<int64_t>(b) * sc.nsteps + s0 + lane] = t;
        const unsigned long long gt = warp_sum_u64(lane < kGroupSteps ? t : 0ull);
        if (!LOGITS && __any_sync(0xffffffffu, bad) && lane == 0) report(dev_status, SPEC_DEV_ERR_PROB);
        const int gi = chunk * kConsumers + warp;
        if (lane == 0 && gi < sc.ngroups) sc.gtot[static_cast<int64_t>(b) * sc.ngroups + gi] = gt;
    }
}

// Logits form, between stages 1 and 2: the exact row sums Z = sum_v
// exp((z_v - m) / T) of each sequence's draw rows (the target row j and,
// for a residual draw, the draft row j), in double-float.  One CTA per
// (sequence, 8192-element chunk): each thread evaluates 32 elements of
// each row (all its loads in flight first), the CTA adds the threads' sums
// in a fixed order and writes the chunk's partial sum to zparts.
constexpr int kZChunk = 8192;
constexpr int kZPerThread = kZChunk / kThreads;   // 32

__device__ __forceinline__ DF warp_sum_df(DF a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const DF x{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
        a = df_add(a, x);
    }
    return a;
}

__global__ void __launch_bounds__(kThreads) logits_draw_sums_kernel(SampleIn in, int D, int V, SampleScratch sc,
                                                                     bool vec4, float2 *__restrict__ zparts)
{
    __shared__ float2 s_tab[256];
    __shared__ DF s_w[kWarps];
    build_exp2_table(s_tab);
    pdl_launch_dependents();
    pdl_wait();   // the draw row comes from the previous kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x / in.nzchunks, chunk = blockIdx.x % in.nzchunks;
    const DrawRow dr = decode_draw(__ldcg(sc.js + b));
    const int j = dr.j;
    const int64_t e0 = static_cast<int64_t>(chunk) * kZChunk;
    const int n = static_cast<int>(imin64(kZChunk, V - e0));
    for (int which = 0; which < (dr.residual ? 2 : 1); ++which) {
        const int k = which ? D + 1 + j : j;
        const float2 st = __ldcg(in.stats + static_cast<int64_t>(b) * (2 * D + 1) + k);
        const float *row = (which ? in.q + (static_cast<int64_t>(b) * D + j) * V
                                  : in.p + (static_cast<int64_t>(b) * (D + 1) + j) * V) + e0;
        DF acc{0.0f, 0.0f};
        if (st.y < INFINITY) {
            const SoftmaxPair r = softmax_pair(SoftmaxRow{st.x, in.ih, in.il, 1.0f, 0.0f});
            float4 z[kZPerThread / 4];
#pragma unroll
            for (int u = 0; u < kZPerThread / 4; ++u) {
                const int e = (u * kThreads + threadIdx.x) * 4;
                z[u] = e < n ? load4(row, e, n, vec4, -INFINITY) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            DF2 a2{0ull, 0ull};   // two running sums (even and odd elements), hi + lo each
#pragma unroll
            for (int u = 0; u < kZPerThread / 4; ++u) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const DF2 e = softmax_exp2(h ? pack2(z[u].z, z[u].w) : pack2(z[u].x, z[u].y), r, s_tab);
                    const DF2 t = two_sum2(a2.hi, e.hi);
                    a2.hi = t.hi;
                    a2.lo = add2(a2.lo, add2(t.lo, e.lo));
                }
            }
            acc = df_add(DF{lo_of(a2.hi), lo_of(a2.lo)}, DF{hi_of(a2.hi), hi_of(a2.lo)});
        }
        acc = warp_sum_df(acc);
        if (lane == 0) s_w[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            DF t = s_w[0];
            for (int w = 1; w < kWarps; ++w) t = df_add(t, s_w[w]);
            zparts[(static_cast<int64_t>(b) * 2 + which) * in.nzchunks + chunk] = make_float2(t.hi, t.lo);
        }
        __syncthreads();
    }
}

// Stage 3: one warp per sequence draws the token: Z = sum of the group
// masses, then the group, the step and finally the element whose running
// sum first exceeds floor(u * Z) (re-reading only the 128 elements of one
// step).
template <bool LOGITS>
__global__ void __launch_bounds__(kThreads) accept_finalize_kernel(
    SampleIn in, int B, int D, int V, SampleScratch sc, int32_t *__restrict__ n_accepted,
    int32_t *__restrict__ token, uint32_t *dev_status, bool vec4)
{
    const float *__restrict__ p = in.p;
    const float *__restrict__ q = in.q;
    __shared__ float2 s_tab[LOGITS ? 256 : 1];
    if (LOGITS) build_exp2_table(s_tab);
    pdl_wait();   // step and group masses come from the previous kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarps + warp;
    if (b >= B) return;
    const DrawRow dr = decode_draw(sc.js[b]);
    const int j = dr.j;
    int residual = dr.residual;
    const float *prow = p + (static_cast<int64_t>(b) * (D + 1) + j) * V;
    const float *qrow = residual ? q + (static_cast<int64_t>(b) * D + j) * V : nullptr;
    unsigned long long *steps = sc.steps + static_cast<int64_t>(b) * sc.nsteps;
    unsigned long long *gtot = sc.gtot + static_cast<int64_t>(b) * sc.ngroups;
    const SoftmaxPair rp = softmax_pair(draw_row<LOGITS>(in, b, D, j, 0));
    const SoftmaxPair rq = residual ? softmax_pair(draw_row<LOGITS>(in, b, D, D + 1 + j, 1)) : rp;

    float u = LOGITS ? philox_u(in.seed, static_cast<uint32_t>(b), 0u, 1u) : in.u_res[b];
    if (!(u >= 0.0f && u < 1.0f)) {
        if (lane == 0) report(dev_status, SPEC_DEV_ERR_UNIFORM);
        u = (u >= 1.0f) ? 0x1.fffffep-1f : 0.0f;
    }
    unsigned long long Z = 0;
    bool ovf = false;
    for (int attempt = 0; attempt < 2; ++attempt) {
        unsigned long long z = 0;
        for (int g = lane; g < sc.ngroups; g += 32) {
            const unsigned long long y = z + gtot[g];
            ovf |= y < z;
            z = y;
        }
        Z = warp_sum_u64(z, ovf);
        if (Z != 0 || !residual) break;
        // reading: max(0, p - q) has no mass -> draw from the target row
        // itself; this warp recomputes the step and group masses of p
        residual = 0;
        if (lane == 0) report(dev_status, SPEC_DEV_INFO_ZERO_RESIDUAL);
        for (int g = 0; g < sc.ngroups; ++g) {
            const int64_t g0 = static_cast<int64_t>(g) * kGroup;
            const int n = static_cast<int>(imin64(kGroup, V - g0));
            const unsigned long long t =
                warp_step_masses<false, LOGITS>(prow + g0, nullptr, 0, 0, n, false, lane, rp, rq, s_tab, ovf);
            if (lane < kGroupSteps && g * kGroupSteps + lane < sc.nsteps) steps[g * kGroupSteps + lane] = t;
            const unsigned long long gt = warp_sum_u64(lane < kGroupSteps ? t : 0ull);
            if (lane == 0) gtot[g] = gt;
        }
        __syncwarp();
    }
    if (__any_sync(0xffffffffu, ovf) && lane == 0) report(dev_status, SPEC_DEV_ERR_PROB);
    if (Z == 0) {
        if (lane == 0) {
            report(dev_status, SPEC_DEV_ERR_ZERO_MASS);
            n_accepted[b] = j;
            token[b] = 0;
        }
        return;
    }
    const unsigned long long T = scaled_threshold(u, Z);
    // the group holding the crossing: smallest g with prefix(g) <= T < prefix(g) + mass(g)
    int found = -1;
    unsigned long long run_g = 0, base = 0;
    for (int g0 = 0; g0 < sc.ngroups && found < 0; g0 += 32) {
        const int g = g0 + lane;
        const unsigned long long v = g < sc.ngroups ? gtot[g] : 0ull;
        const unsigned long long incl = warp_incl_scan_u64(v, lane);
        const unsigned long long run = base + incl - v;
        const unsigned hit = __ballot_sync(0xffffffffu, g < sc.ngroups && run <= T && T < run + v);
        if (hit) {
            const int l = __ffs(hit) - 1;
            found = g0 + l;
            run_g = __shfl_sync(0xffffffffu, run, l);
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    int tok = 0;
    if (found >= 0) {
        // the step within the group
        const int st = found * kGroupSteps + (lane % kGroupSteps);
        const unsigned long long v = (lane < kGroupSteps && st < sc.nsteps) ? steps[st] : 0ull;
        const unsigned long long incl = warp_incl_scan_u64(v, lane);
        const unsigned long long run = run_g + incl - v;
        const unsigned hit = __ballot_sync(0xffffffffu, lane < kGroupSteps && run <= T && T < run + v);
        const int l = hit ? __ffs(hit) - 1 : 0;
        const int step = found * kGroupSteps + l;
        const unsigned long long run_s = __shfl_sync(0xffffffffu, run, l);
        // the element within the step
        const int64_t e = static_cast<int64_t>(step) * kStep + lane * 4;
        const float pad = pad_value<LOGITS>();
        const float4 xp =
            to_prob4<LOGITS>(e < V ? load4(prow, e, V, vec4, pad) : make_float4(pad, pad, pad, pad), rp, s_tab);
        const float4 xq = (residual && e < V) ? to_prob4<LOGITS>(load4(qrow, e, V, vec4, pad), rq, s_tab)
                                              : make_float4(0, 0, 0, 0);
        const unsigned long long m[4] = {mass(xp.x, xq.x, residual), mass(xp.y, xq.y, residual),
                                         mass(xp.z, xq.z, residual), mass(xp.w, xq.w, residual)};
        const unsigned long long lane_sum = m[0] + m[1] + m[2] + m[3];
        const unsigned long long lincl = warp_incl_scan_u64(lane_sum, lane);
        const unsigned ehit = __ballot_sync(0xffffffffu, run_s + lincl > T);
        const int Lh = ehit ? __ffs(ehit) - 1 : 31;
        unsigned long long c = run_s + lincl - lane_sum;
        int v_tok = static_cast<int>(e);
        for (int k = 0; k < 4; ++k) {
            c += m[k];
            if (c > T) { v_tok = static_cast<int>(e) + k; break; }
        }
        tok = __shfl_sync(0xffffffffu, v_tok, Lh);
    }
    if (lane == 0) {
        n_accepted[b] = j;
        token[b] = tok;
    }
}

// ------------------------------------------------------------------ AdaSD
// AdaSD relaxed acceptance ("Adaptive speculative decoding", section AdaSD):
// the entropy of the draft distribution decides where the drafter stops and
// the Jensen-Shannon distance between draft and target distributions lets a
// draft token be accepted where min(1, p/q) would reject it.
//   H(q_i)   = -sum_v q ln q                       (natural log, 0 ln 0 = 0)
//   JSD_i    = (sum_v p ln p + q ln q - s ln s) / 2 + ln 2 * sum_v s / 2,
//              s = p + q  (= (KL(p||m) + KL(q||m)) / 2 with m = s / 2)
//   JS_i     = sqrt(max(0, JSD_i))
//   d_eff    = first i with H(q_i) > tau_H, else D
//   draft i < d_eff accepted iff u_acc q(x) < p(x) (exact) or JS_i <= tau_JS;
//   the token is drawn as in the stochastic acceptance from row j (residual
//   after a rejection at j, else the bonus row d_eff).
// Stage A streams the D (p_i, q_i) row pairs of every sequence once, one
// 8192-element chunk per CTA, and writes each chunk's two partial sums;
// stage B (a warp per sequence) adds the partials in a fixed order, takes
// the decisions and hands the draw row to the streaming and finalising
// kernels of the stochastic acceptance.  The sums are fp32 (the logarithms
// from the hardware approximation), so H and JS are close to, not equal
// to, the exact values; decisions can differ from exact ones only for a
// statistic within that error of its threshold.
constexpr int kAdaChunk = 8192;
constexpr int kAdaVec = kAdaChunk / (4 * kThreads);   // float4 loads per thread and row: 8

__device__ __forceinline__ float xlogx(float x) { return x > 0.0f ? x * __logf(x) : 0.0f; }

__global__ void __launch_bounds__(kThreads) adasd_stats_kernel(const float *__restrict__ p,
                                                                const float *__restrict__ q, int D, int V,
                                                                int nchunks, bool vec4, float2 *__restrict__ parts)
{
    __shared__ float2 s_w[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int item = blockIdx.x;
    const int r = item / nchunks, c = item % nchunks;
    const int b = r / D, i = r % D;
    const int64_t e0 = static_cast<int64_t>(c) * kAdaChunk;
    const int n = static_cast<int>(imin64(kAdaChunk, V - e0));
    const float *pr = p + (static_cast<int64_t>(b) * (D + 1) + i) * V + e0;
    const float *qr = q + (static_cast<int64_t>(b) * D + i) * V + e0;
    float4 xp[kAdaVec], xq[kAdaVec];
#pragma unroll
    for (int u = 0; u < kAdaVec; ++u) {   // every load of the thread in flight at once
        const int e = (u * kThreads + threadIdx.x) * 4;
        xp[u] = e < n ? load4(pr, e, n, vec4, 0.0f) : make_float4(0.f, 0.f, 0.f, 0.f);
        xq[u] = e < n ? load4(qr, e, n, vec4, 0.0f) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_launch_dependents();
    float h = 0.0f, js = 0.0f, sum = 0.0f;
#pragma unroll
    for (int u = 0; u < kAdaVec; ++u) {
        const float pv[4] = {xp[u].x, xp[u].y, xp[u].z, xp[u].w};
        const float qv[4] = {xq[u].x, xq[u].y, xq[u].z, xq[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float qlq = xlogx(qv[k]);
            const float s = pv[k] + qv[k];
            h += qlq;
            js += xlogx(pv[k]) + qlq - xlogx(s);
            sum += s;
        }
    }
    js += 0.69314718f * sum;   // + ln 2 * sum of s
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        h += __shfl_xor_sync(0xffffffffu, h, o);
        js += __shfl_xor_sync(0xffffffffu, js, o);
    }
    if (lane == 0) s_w[warp] = make_float2(h, js);
    __syncthreads();
    if (threadIdx.x == 0) {
        float2 t = s_w[0];
        for (int w = 1; w < kWarps; ++w) {
            t.x += s_w[w].x;
            t.y += s_w[w].y;
        }
        parts[static_cast<int64_t>(r) * nchunks + c] = t;
    }
}

// Stage B: one warp per sequence.
__global__ void __launch_bounds__(kThreads) adasd_prep_kernel(
    const float *__restrict__ p, const float *__restrict__ q, const int32_t *__restrict__ draft,
    const float *__restrict__ u_acc, const float2 *__restrict__ parts, int nchunks, float tau_h, float tau_js,
    int B, int D, int V, float *__restrict__ entropy, float *__restrict__ js_dist, int32_t *__restrict__ d_eff,
    SampleScratch sc, uint32_t *dev_status)
{
    pdl_launch_dependents();
    pdl_wait();   // the partial sums come from the previous kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarps + warp;
    if (b >= B) return;
    int de = D;          // first position whose draft entropy exceeds tau_H
    int j = -1;          // first position that fails both tests
    for (int i = 0; i < D; ++i) {
        const int64_t r = static_cast<int64_t>(b) * D + i;
        float h = 0.0f, s = 0.0f;
        for (int c = lane; c < nchunks; c += 32) {
            const float2 v = __ldcg(parts + r * nchunks + c);
            h += v.x;
            s += v.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {   // the same order on every lane
            h += __shfl_xor_sync(0xffffffffu, h, o);
            s += __shfl_xor_sync(0xffffffffu, s, o);
        }
        const float H = -h, JS = sqrtf(fmaxf(0.5f * s, 0.0f));
        if (lane == 0) {
            if (entropy) entropy[r] = H;
            if (js_dist) js_dist[r] = JS;
        }
        if (de < D) continue;   // past the stop: statistics only
        if (H > tau_h) {
            de = i;
            continue;
        }
        if (j >= 0) continue;   // already decided
        const int x = draft[r];
        bool ok;
        if (x < 0 || x >= V) {
            if (lane == 0) report(dev_status, SPEC_DEV_ERR_TOKEN_ID);
            ok = false;
        } else {
            const double pv = p[(static_cast<int64_t>(b) * (D + 1) + i) * V + x];
            const double qv = q[r * V + x];
            const float uf = u_acc[r];
            if (!(uf >= 0.0f && uf < 1.0f) && lane == 0) report(dev_status, SPEC_DEV_ERR_UNIFORM);
            // the product of two fp32 values is exact in fp64
            ok = static_cast<double>(uf) * qv < pv || JS <= tau_js;
        }
        if (!ok) j = i;
    }
    if (lane == 0) {
        sc.js[b] = j >= 0 ? j : (de | kBonusFlag);
        if (d_eff) d_eff[b] = de;
    }
}

// Logits row statistics: for every row of the target and draft logits,
// m = max_v z_v and Zf = sum_v 2^((z_v - m) c), c = fl32(log2 e / T) (the
// fast evaluation of the accept tests: hardware exponential, fp32 sums in
// a fixed order).
//
// One thread-block cluster of CS CTAs works on one row at a time, CTA
// `rank` owning the elements [rank * slice, (rank + 1) * slice); clusters
// walk the rows round robin, several clusters' CTAs sharing an SM so that
// one CTA's copy or exchange overlaps another's arithmetic.  BULK: the
// slice is staged in shared memory by one bulk copy, so every logit is read
// from HBM once; otherwise both passes read global memory (the second from
// L2).  Pass 1 takes the slice maximum; the CTAs exchange their maxima
// through distributed shared memory (asynchronous stores that complete on
// the receiver's mbarrier; no cluster-wide barrier per row).  Pass 2 sums
// the exponentials; the partial sums go to the row's owner (rank = row
// iteration mod CS), which adds them in rank order and writes (m, Zf).
// Rows whose maximum is not finite, or that hold NaN or +inf, get Zf = +inf
// (every probability 0) and set SPEC_DEV_ERR_LOGITS.
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr int kStatsThreads = 256;
constexpr int kStatsWarps = kStatsThreads / 32;
constexpr int kStatsMinBlocks = 3;                 // CTAs per SM (shared memory allows 3 slices of 64 KB)

template <int CS, bool BULK>
__global__ void __launch_bounds__(kStatsThreads, kStatsMinBlocks) logits_rowstats_kernel(
    const float *__restrict__ zp, const float *__restrict__ zq, int B, int D, int V, float c_fast, int slice,
    bool vec4, float2 *__restrict__ stats, uint32_t *dev_status)
{
    extern __shared__ uint8_t s_raw[];
    float *buf = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(s_raw) + 127) & ~uintptr_t(127));
    __shared__ uint64_t full, bar_max[2], bar_sum[2];
    __shared__ unsigned long long s_xmax[2][CS];   // (bad << 32) | bits of CTA c's max, by row parity
    __shared__ unsigned long long s_xsum[2][CS];   // CTA c's partial sum (bits), owned rows
    __shared__ float s_wmax[kStatsWarps];
    __shared__ int s_wbad[kStatsWarps];
    __shared__ float s_wsum[kStatsWarps];
    __shared__ int s_abort;
    volatile int *abort = reinterpret_cast<volatile int *>(&s_abort);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (cluster_ctas() != static_cast<uint32_t>(CS)) {   // uniform over the grid
        if (tid == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        return;
    }
    uint32_t rank = 0;
    if (CS > 1) asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int cluster = blockIdx.x / CS, nclusters = gridDim.x / CS;
    const int rows_per_b = 2 * D + 1;
    const int R = B * rows_per_b;
    const int64_t e0 = static_cast<int64_t>(rank) * slice;
    const int len = static_cast<int>(imin64(slice, imin64(V, e0 + slice) - imin64(V, e0)));
    auto row_src = [&](int r) -> const float * {
        const int b = r / rows_per_b, k = r % rows_per_b;
        const float *base = k <= D ? zp + (static_cast<int64_t>(b) * (D + 1) + k) * V
                                   : zq + (static_cast<int64_t>(b) * D + (k - D - 1)) * V;
        return base + e0;
    };
    if (tid == 0) {
        mbar_init(&full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_max[i], 1);
            mbar_init(&bar_sum[i], 1);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (CS > 1) cluster_sync_all();   // every peer's barriers exist before the first send
    else __syncthreads();
    pdl_launch_dependents();

    // the owner of row iteration k (k % CS == rank) collects the partial sums
    auto finish_row = [&](int k, int r, float m, int rbad) {
        const int slot = (k / CS) & 1;
        if (CS > 1 && !mbar_wait(&bar_sum[slot], ((k / CS) >> 1) & 1, abort, dev_status)) return;
        float z = 0.0f;
        for (int c = 0; c < CS; ++c) z = __fadd_rn(z, __uint_as_float(static_cast<uint32_t>(s_xsum[slot][c])));
        float2 st;
        if (rbad || !(z > 0.0f)) {
            report(dev_status, SPEC_DEV_ERR_LOGITS);
            st = make_float2(0.0f, INFINITY);
        } else {
            st = make_float2(m, z);
        }
        stats[r] = st;
    };
    int pend_k = -1, pend_r = 0, pend_bad = 0;   // thread 0: an owned row whose sums are still due
    float pend_m = 0.0f;
    uint32_t loads = 0;   // thread 0: copies issued

    int k = 0;
    for (int r = cluster; r < R; r += nclusters, ++k) {
        const int owner = k % CS;
        if (tid == 0) {
            if (BULK && len > 0 && !*abort) {
                mbar_arrive_expect_tx(&full, static_cast<uint32_t>(len) * 4u);
                bulk_load(buf, row_src(r), static_cast<uint32_t>(len) * 4u, &full);
                ++loads;
                // the next row's slice travels to L2 while this one is worked on
                if (r + nclusters < R) prefetch_l2(row_src(r + nclusters), static_cast<uint32_t>(len) * 4u);
            }
            if (CS > 1) {
                mbar_arrive_expect_tx(&bar_max[k & 1], CS * 8u);
                if (owner == static_cast<int>(rank)) mbar_arrive_expect_tx(&bar_sum[(k / CS) & 1], CS * 8u);
            }
            // while this row's slice lands: the sums of the previous owned row
            if (pend_k >= 0) {
                finish_row(pend_k, pend_r, pend_m, pend_bad);
                pend_k = -1;
            }
        }
        const float *src = row_src(r);
        if (BULK) {
            // row iteration k's copy completes phase k of `full`
            if (len > 0) mbar_wait(&full, static_cast<uint32_t>(k) & 1u, abort, dev_status);
            src = buf;
        }
        // pass 1: the maximum; a NaN anywhere makes the running sum NaN
        float mx = -INFINITY;
        unsigned long long acc2 = 0ull;
        for (int i = tid * 4; i < len; i += kStatsThreads * 4) {
            const float4 v = BULK ? *reinterpret_cast<const float4 *>(src + i) : load4(src, i, len, vec4, -INFINITY);
            mx = max3(mx, max3(v.x, v.y, v.z), v.w);
            acc2 = add2(acc2, add2(pack2(v.x, v.y), pack2(v.z, v.w)));
        }
        const bool bad = lo_of(acc2) != lo_of(acc2) || hi_of(acc2) != hi_of(acc2);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const int wbad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            s_wmax[warp] = mx;
            s_wbad[warp] = wbad;
        }
        __syncthreads();
        if (tid < CS) {
            float cm = s_wmax[0];
            int cb = s_wbad[0];
            for (int w = 1; w < kStatsWarps; ++w) {
                cm = fmaxf(cm, s_wmax[w]);
                cb |= s_wbad[w];
            }
            const unsigned long long word = (static_cast<unsigned long long>(cb ? 1u : 0u) << 32) | __float_as_uint(cm);
            if (CS > 1)
                st_async_peer(peer_smem(&s_xmax[k & 1][rank], static_cast<uint32_t>(tid)), word,
                              peer_smem(&bar_max[k & 1], static_cast<uint32_t>(tid)));
            else
                s_xmax[k & 1][0] = word;
        }
        if (CS > 1) mbar_wait(&bar_max[k & 1], (k >> 1) & 1, abort, dev_status);
        else __syncthreads();
        float m = -INFINITY;
        int rbad = 0;
#pragma unroll
        for (int c = 0; c < CS; ++c) {
            const unsigned long long w = s_xmax[k & 1][c];
            m = fmaxf(m, __uint_as_float(static_cast<uint32_t>(w)));
            rbad |= static_cast<int>(w >> 32);
        }
        rbad |= !(m > -INFINITY) | !(m < INFINITY);
        // pass 2: the sum of the exponentials, in a fixed order
        float acc = 0.0f;
        if (!rbad) {
            for (int i = tid * 4; i < len; i += kStatsThreads * 4) {
                const float4 v = BULK ? *reinterpret_cast<const float4 *>(src + i) : load4(src, i, len, vec4, -INFINITY);
                const float e0 = ex2_approx(__fmul_rn(__fsub_rn(v.x, m), c_fast));
                const float e1 = ex2_approx(__fmul_rn(__fsub_rn(v.y, m), c_fast));
                const float e2 = ex2_approx(__fmul_rn(__fsub_rn(v.z, m), c_fast));
                const float e3 = ex2_approx(__fmul_rn(__fsub_rn(v.w, m), c_fast));
                acc = __fadd_rn(acc, __fadd_rn(__fadd_rn(e0, e1), __fadd_rn(e2, e3)));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
        if (lane == 0) s_wsum[warp] = acc;
        __syncthreads();   // also: every thread is done with this slice
        if (tid == 0) {
            float t = s_wsum[0];
            for (int w = 1; w < kStatsWarps; ++w) t = __fadd_rn(t, s_wsum[w]);
            const int slot = (k / CS) & 1;
            if (CS > 1)
                st_async_peer(peer_smem(&s_xsum[slot][rank], static_cast<uint32_t>(owner)), __float_as_uint(t),
                              peer_smem(&bar_sum[slot], static_cast<uint32_t>(owner)));
            else
                s_xsum[slot][0] = __float_as_uint(t);
            if (owner == static_cast<int>(rank)) {
                pend_k = k;
                pend_r = r;
                pend_m = m;
                pend_bad = rbad;
            }
        }
    }
    if (tid == 0) {
        if (pend_k >= 0) finish_row(pend_k, pend_r, pend_m, pend_bad);
        // unwind after a timed-out wait: let a copy still in flight land
        if (BULK && *abort && loads) mbar_wait_drain(&full, (loads - 1u) & 1u, kWaitTimeoutNs);
    }
    // keep this CTA's shared memory alive until every peer is done with it
    if (CS > 1) cluster_sync_all();
}

// ------------------------------------------------------- stochastic tree
// Stochastic acceptance over a draft tree: the children of node k (nodes
// whose parent is k, in increasing index) carry tokens drafted from
// q[b][k].  At the current node the working row starts as p; a child with
// token x is accepted iff u * q(x) < r(x), and after a rejection the row
// becomes max(0, r - q) renormalised, before the next sibling is tried;
// when no child is accepted the token is drawn from the row.  A chain is
// the stochastic acceptance above (and the rule is lossless for siblings
// drafted independently from q).
// One cluster per sequence.  The row is kept unnormalised: R_0 = p and
// R_j = max(0, R_{j-1} - S_{j-1} q) with S_0 = 1 and S_j = sum_v R_j(v), so
// r_j = R_j / S_j.  Unrolled, R_j = max(0, p - c_j q) with c_j = S_0 + ... +
// S_{j-1} (a clipped element stays clipped as c grows), which is how each
// R_j(v) is evaluated: one fp32 fused multiply-add from p(v), q(v) and c_j,
// whatever the depth, by the same function for one element and for a whole
// pass.  c_j accumulates in fp64 from the exact S's and is rounded to fp32
// once.  Each S_j is the exact sum of the elements' 2^-61 fixed-point
// masses, and a test after j rejections is u q(x) S_j < R_j(x) in fp64.  An
// empty residual (S = 0) leaves the row as it was and is reported.
constexpr int kTSThreads = 256;
constexpr int kTSWarps = kTSThreads / 32;
constexpr int kTSGroup = 4 * kStep;   // 512 elements: 4 steps of 128

// R_j(v) for j >= 1 (RES) or R_0(v) = p(v)
template <bool RES>
__device__ __forceinline__ float tree_row_value(float pv, float qv, float c)
{
    return RES ? fmaxf(__fmaf_rn(-c, qv, pv), 0.0f) : pv;
}

template <bool RES>
__device__ __forceinline__ unsigned long long tree_masses4(const float4 &xp, const float4 &xq, float c)
{
    return (fix61(tree_row_value<RES>(xp.x, xq.x, c)) + fix61(tree_row_value<RES>(xp.y, xq.y, c))) +
           (fix61(tree_row_value<RES>(xp.z, xq.z, c)) + fix61(tree_row_value<RES>(xp.w, xq.w, c)));
}

// Exact masses of R per 512-element group of a slice of n elements (warp w
// takes groups w, w + kTSWarps, ...), into gtot; returns the sum of the
// warp's groups (in every lane).  With 16-byte aligned rows (vec4) every
// group inside the slice takes four unconditional float4 loads per operand
// (q only for a residual); the ragged last group is checked.
template <bool RES>
__device__ __forceinline__ unsigned long long tree_group_totals(const float *prow, const float *qrow, float c, int n,
                                                                bool vec4, unsigned long long *gtot, int ngroups)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nfull = vec4 ? n / kTSGroup : 0;
    const float4 *p4 = reinterpret_cast<const float4 *>(prow) + lane;
    const float4 *q4 = reinterpret_cast<const float4 *>(qrow) + lane;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    unsigned long long part = 0;
    for (int g = warp; g < nfull; g += kTSWarps) {
        float4 xp[4], xq[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            xp[k] = __ldg(p4 + g * (kTSGroup / 4) + k * 32);
            xq[k] = RES ? __ldg(q4 + g * (kTSGroup / 4) + k * 32) : zero;
        }
        const unsigned long long m0 = tree_masses4<RES>(xp[0], xq[0], c) + tree_masses4<RES>(xp[1], xq[1], c);
        const unsigned long long m1 = tree_masses4<RES>(xp[2], xq[2], c) + tree_masses4<RES>(xp[3], xq[3], c);
        const unsigned long long m = warp_sum_u64(m0 + m1);
        if (lane == 0) gtot[g] = m;
        part += m;
    }
    for (int g = nfull + warp; g < ngroups; g += kTSWarps) {
        unsigned long long m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t e = static_cast<int64_t>(g) * kTSGroup + k * kStep + lane * 4;
            const float4 xp = e < n ? load4(prow, e, n, vec4, 0.0f) : zero;
            const float4 xq = (RES && e < n) ? load4(qrow, e, n, vec4, 0.0f) : zero;
            m += tree_masses4<RES>(xp, xq, c);
        }
        m = warp_sum_u64(m);
        if (lane == 0) gtot[g] = m;
        part += m;
    }
    return part;
}

// CS CTAs (a cluster) per sequence, CTA `rank` owning the vocabulary slice
// [c0, c0 + n).  Every CTA takes the same decisions: the tests read the two
// gathered values from global memory, and each row sum is the CTAs' exact
// slice sums, sent to every CTA of the cluster by asynchronous shared-memory
// stores that complete on the receiver's mbarrier and added in rank order.
// The final draw exchanges the slice totals the same way; the CTA whose
// prefix holds the threshold finds the token in its slice.
template <int CS>
__global__ void __launch_bounds__(kTSThreads) accept_tree_sample_kernel(
    const float *__restrict__ p, const float *__restrict__ q, const int32_t *__restrict__ tokens,
    const int32_t *__restrict__ parent, const float *__restrict__ u_acc, const float *__restrict__ u_res, int D,
    int V, int32_t *__restrict__ n_accepted, int32_t *__restrict__ token, int32_t *__restrict__ path,
    uint32_t *dev_status, bool vec4)
{
    extern __shared__ unsigned long long s_gtot[];   // one total per 512-element group of the slice
    __shared__ int32_t s_par[kMaxDraft + 1], s_tok[kMaxDraft + 1];
    __shared__ unsigned long long s_wpart[kTSWarps];
    __shared__ __align__(8) unsigned long long s_x[2][CS];   // exchanged partials, per parity
    __shared__ uint64_t s_xbar[2];
    __shared__ int s_bad, s_abort;
    if (cluster_ctas() != static_cast<uint32_t>(CS)) {   // uniform over the grid
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        return;
    }
    const int rank = CS > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int b = blockIdx.x / CS, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = 1 + D;
    const int64_t cta_len = ((static_cast<int64_t>(V) + CS - 1) / CS + 3) & ~int64_t(3);
    const int64_t c0 = imin64(V, cta_len * rank);
    const int n = static_cast<int>(imin64(V, c0 + cta_len) - c0);
    volatile int *abort = reinterpret_cast<volatile int *>(&s_abort);
    if (tid == 0) {
        s_bad = 0;
        s_abort = 0;
        mbar_init(&s_xbar[0], 1);
        mbar_init(&s_xbar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if constexpr (CS > 1) cluster_arrive_relaxed();   // waited for before the first send
    for (int k = tid; k < T; k += kTSThreads) {
        const int pa = parent[static_cast<int64_t>(b) * T + k];
        const int tk = tokens[static_cast<int64_t>(b) * T + k];
        s_par[k] = pa;
        s_tok[k] = tk;
        if (k == 0 ? pa != -1 : (pa < 0 || pa >= k)) atomicOr(&s_bad, 1);
        if (k > 0 && (tk < 0 || tk >= V)) atomicOr(&s_bad, 2);
    }
    __syncthreads();
    const int bad = s_bad;
    // a malformed tree (or a token out of range) is walked as a lone root
    if (bad && rank == 0 && tid == 0) report(dev_status, (bad & 1) ? SPEC_DEV_ERR_TREE : SPEC_DEV_ERR_TOKEN_ID);
    if (path && rank == 0 && tid < D) path[static_cast<int64_t>(b) * D + tid] = -1;

    // sum over the cluster of each CTA's value (identical in every CTA)
    uint32_t nx = 0;    // exchanges so far
    bool ok = true;
    auto exchange = [&](unsigned long long mine) -> unsigned long long {
        const int slot = static_cast<int>(nx & 1u);
        if constexpr (CS > 1) {
            if (tid == 0) mbar_arrive_expect_tx(&s_xbar[slot], CS * 8);
            if (nx == 0) cluster_wait_acquire();   // every peer's barriers are initialised
            if (tid < CS) st_async_peer(peer_smem(&s_x[slot][rank], tid), mine, peer_smem(&s_xbar[slot], tid));
            // one warp spins (spinning warps would take issue slots from the
            // passes of the SM's other CTAs); the others block in the barrier
            // and then take the completed phase, without waiting, to acquire
            // the peers' stores themselves
            if (ok && warp == 0) ok = mbar_wait(&s_xbar[slot], (nx >> 1) & 1u, abort, dev_status);
            ok = __syncthreads_and(ok);
            if (ok && warp != 0) (void)mbar_try_wait(smem_u32(&s_xbar[slot]), (nx >> 1) & 1u);
        } else {
            if (tid == 0) s_x[slot][0] = mine;
            __syncthreads();
        }
        unsigned long long t = 0;
#pragma unroll
        for (int r = 0; r < CS; ++r) t += s_x[slot][r];
        ++nx;
        return t;
    };

    // the current row R_j: j rejections so far, c_j (fp64 and rounded to
    // fp32) and S_j (exact, and in fp64); c_0 = 0 and S_0 = 1
    int cur = 0, depth = 0, j = 0;
    double Cj = 0.0, Sj = 1.0;
    float cf = 0.0f;
    const float *prow = p, *qrow = q;
    const int ngroups = (n + kTSGroup - 1) / kTSGroup;
    int gtot_j = -1;            // s_gtot holds the group totals of R_gtot_j of the current node
    unsigned long long gtot_sum = 0;   // ... and their sum
    // group totals of R (p, or the residual with coefficient c) over this
    // CTA's slice into s_gtot; returns their sum.  The warps' partials are
    // read before the exchange that follows every call, whose barrier keeps
    // the next call from rewriting them early.
    auto slice_totals = [&](bool res, float c) -> unsigned long long {
        const unsigned long long part =   // res is uniform over the cluster
            res ? tree_group_totals<true>(prow + c0, qrow + c0, c, n, vec4, s_gtot, ngroups)
                : tree_group_totals<false>(prow + c0, qrow + c0, c, n, vec4, s_gtot, ngroups);
        if (lane == 0) s_wpart[warp] = part;
        __syncthreads();
        unsigned long long t = 0;
#pragma unroll
        for (int w = 0; w < kTSWarps; ++w) t += s_wpart[w];
        return t;
    };
    for (;;) {
        prow = p + (static_cast<int64_t>(b) * T + cur) * V;
        qrow = q + (static_cast<int64_t>(b) * T + cur) * V;
        j = 0;
        Cj = 0.0;
        Sj = 1.0;
        cf = 0.0f;
        gtot_j = -1;
        int next = -1;
        for (int c = cur + 1; c < T && !bad && ok; ++c) {
            if (s_par[c] != cur) continue;
            const int x = s_tok[c];
            float u = u_acc[static_cast<int64_t>(b) * T + c];
            if (!(u >= 0.0f && u < 1.0f)) {
                if (rank == 0 && tid == 0) report(dev_status, SPEC_DEV_ERR_UNIFORM);
                u = (u >= 1.0f) ? 0x1.fffffep-1f : 0.0f;
            }
            const float px = prow[x], qx = qrow[x];
            bool acc;
            if (j == 0) {
                acc = static_cast<double>(u) * static_cast<double>(qx) < static_cast<double>(px);
            } else {
                const float rx = tree_row_value<true>(px, qx, cf);
                acc = static_cast<double>(u) * static_cast<double>(qx) * Sj < static_cast<double>(rx);
            }
            if (acc) {
                next = c;
                break;
            }
            // R_{j+1} = max(0, p - c_{j+1} q) with c_{j+1} = c_j + S_j; its
            // group totals are kept: if no later sibling is accepted, the
            // draw uses them as they are
            if (j == 0 && vec4 && tid == 0 && n >= 4) {   // the node's first pass
                prefetch_l2(prow + c0, static_cast<uint32_t>(n & ~3) * 4u);
                prefetch_l2(qrow + c0, static_cast<uint32_t>(n & ~3) * 4u);
            }
            const double Cn = Cj + Sj;
            const float cn = static_cast<float>(Cn);
            const unsigned long long mine = slice_totals(true, cn);
            const unsigned long long Sn = exchange(mine);
            if (Sn == 0) {
                gtot_j = -1;   // the totals are of an empty row, not of R_j
                if (rank == 0 && tid == 0) report(dev_status, SPEC_DEV_INFO_ZERO_RESIDUAL);
            } else {
                ++j;
                Cj = Cn;
                cf = cn;
                Sj = static_cast<double>(Sn) * 0x1p-61;
                gtot_j = j;
                gtot_sum = mine;
            }
        }
        if (next < 0 || !ok) break;
        if (path && rank == 0 && tid == 0) path[static_cast<int64_t>(b) * D + depth] = next;
        ++depth;
        cur = next;
    }

    // the token: inverse CDF of R_j over the row with u_res; this CTA's
    // slice holds the cumulative masses base .. base + total
    float u = u_res[b];
    if (!(u >= 0.0f && u < 1.0f)) {
        if (rank == 0 && tid == 0) report(dev_status, SPEC_DEV_ERR_UNIFORM);
        u = (u >= 1.0f) ? 0x1.fffffep-1f : 0.0f;
    }
    // the last rejection's pass already left R_j's group totals
    unsigned long long mine;
    if (gtot_j == j) {
        mine = gtot_sum;
    } else {
        if (vec4 && tid == 0 && n >= 4) {
            prefetch_l2(prow + c0, static_cast<uint32_t>(n & ~3) * 4u);
            if (j > 0) prefetch_l2(qrow + c0, static_cast<uint32_t>(n & ~3) * 4u);
        }
        mine = slice_totals(j > 0, cf);
    }
    const unsigned long long Z = ok ? exchange(mine) : 0ull;
    unsigned long long base = 0;
    for (int r = 0; r < rank; ++r) base += s_x[(nx - 1) & 1u][r];
    const unsigned long long Tt = Z ? scaled_threshold(u, Z) : 0ull;
    const bool owner = Z != 0 && base <= Tt && Tt < base + mine;
    if (ok && Z == 0 && rank == 0 && tid == 0) {
        report(dev_status, SPEC_DEV_ERR_ZERO_MASS);
        n_accepted[b] = depth;
        token[b] = 0;
    }
    if (ok && owner && warp == 0) {
        int tok = 0;
        // the group: smallest g with prefix(g) <= Tt < prefix(g) + mass(g)
        int found = -1;
        unsigned long long run_g = 0, gbase = base;
        for (int g0 = 0; g0 < ngroups && found < 0; g0 += 32) {
            const int g = g0 + lane;
            const unsigned long long v = g < ngroups ? s_gtot[g] : 0ull;
            const unsigned long long incl = warp_incl_scan_u64(v, lane);
            const unsigned long long run = gbase + incl - v;
            const unsigned hit = __ballot_sync(0xffffffffu, g < ngroups && v > 0 && run <= Tt && Tt < run + v);
            if (hit) {
                const int l = __ffs(hit) - 1;
                found = g0 + l;
                run_g = __shfl_sync(0xffffffffu, run, l);
            }
            gbase += __shfl_sync(0xffffffffu, incl, 31);
        }
        // the element: walk the group's 512 elements, 128 at a time
        auto rv = [&](float pv, float qv) { return j > 0 ? tree_row_value<true>(pv, qv, cf) : pv; };
        unsigned long long run = run_g;
        for (int k = 0; k < 4 && found >= 0; ++k) {
            const int64_t e = static_cast<int64_t>(found) * kTSGroup + k * kStep + lane * 4;
            float4 xp = make_float4(0.f, 0.f, 0.f, 0.f), xq = xp;
            if (e < n) {
                xp = load4(prow + c0, e, n, vec4, 0.0f);
                if (j > 0) xq = load4(qrow + c0, e, n, vec4, 0.0f);
            }
            const unsigned long long m0 = e < n ? fix61(rv(xp.x, xq.x)) : 0ull;
            const unsigned long long m1 = e < n ? fix61(rv(xp.y, xq.y)) : 0ull;
            const unsigned long long m2 = e < n ? fix61(rv(xp.z, xq.z)) : 0ull;
            const unsigned long long m3 = e < n ? fix61(rv(xp.w, xq.w)) : 0ull;
            const unsigned long long ls = m0 + m1 + m2 + m3;
            const unsigned long long incl = warp_incl_scan_u64(ls, lane);
            const unsigned hit = __ballot_sync(0xffffffffu, run + incl > Tt);
            if (hit) {
                const int l = __ffs(hit) - 1;
                if (lane == l) {
                    unsigned long long cc = run + incl - ls;
                    const unsigned long long mm[4] = {m0, m1, m2, m3};
                    int k4 = 3;
                    for (int i = 0; i < 4; ++i) {
                        cc += mm[i];
                        if (cc > Tt) { k4 = i; break; }
                    }
                    tok = static_cast<int>(c0 + e) + k4;
                }
                tok = __shfl_sync(0xffffffffu, tok, l);
                found = -1;   // done
            } else {
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (lane == 0) {
            n_accepted[b] = depth;
            token[b] = tok;
        }
    }
    // keep this CTA's shared memory alive until every peer is done with it
    if constexpr (CS > 1) cluster_exit_barrier();
}

}  // namespace

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel k, dim3 grid, dim3 block, uint32_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

int pick_cluster(int V)
{
    if (V >= 32768) return 8;
    if (V >= 8192) return 4;
    if (V >= 2048) return 2;
    return 1;
}

template <int CS, bool TREE, bool BULK>
cudaError_t launch_greedy_cs(const float *p, const int32_t *draft, const int32_t *parent, int B, int D,
                             int V, int32_t *n_acc, int32_t *token, int32_t *path, uint32_t *dev_status,
                             bool vec4, cudaStream_t st)
{
    const uint32_t smem = BULK ? kGSmem : 0u;
    if (BULK) {
        const cudaError_t e = cudaFuncSetAttribute(accept_greedy_kernel<CS, TREE, BULK>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B) * CS);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_greedy_kernel<CS, TREE, BULK>, p, draft, parent, D, V, n_acc, token,
                              path, dev_status, vec4);
}

template <bool TREE, bool BULK>
cudaError_t launch_greedy_bulk(const float *p, const int32_t *draft, const int32_t *parent, int B, int D,
                               int V, int32_t *n_acc, int32_t *token, int32_t *path, uint32_t *dev_status,
                               bool vec4, cudaStream_t st)
{
    switch (pick_cluster(V)) {
    case 8: return launch_greedy_cs<8, TREE, BULK>(p, draft, parent, B, D, V, n_acc, token, path, dev_status, vec4, st);
    case 4: return launch_greedy_cs<4, TREE, BULK>(p, draft, parent, B, D, V, n_acc, token, path, dev_status, vec4, st);
    case 2: return launch_greedy_cs<2, TREE, BULK>(p, draft, parent, B, D, V, n_acc, token, path, dev_status, vec4, st);
    default: return launch_greedy_cs<1, TREE, BULK>(p, draft, parent, B, D, V, n_acc, token, path, dev_status, vec4, st);
    }
}

template <bool TREE>
cudaError_t launch_greedy(const float *p, const int32_t *draft, const int32_t *parent, int B, int D,
                          int V, int32_t *n_acc, int32_t *token, int32_t *path, uint32_t *dev_status,
                          cudaStream_t st)
{
    // rows staged by bulk copies need 16-byte aligned rows
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0);
    if (vec4) return launch_greedy_bulk<TREE, true>(p, draft, parent, B, D, V, n_acc, token, path, dev_status, vec4, st);
    return launch_greedy_bulk<TREE, false>(p, draft, parent, B, D, V, n_acc, token, path, dev_status, vec4, st);
}

cudaError_t launch_accept_greedy(const float *p, const int32_t *draft, int B, int D, int V,
                                 int32_t *n_acc, int32_t *token, uint32_t *dev_status, cudaStream_t st)
{
    return launch_greedy<false>(p, draft, nullptr, B, D, V, n_acc, token, nullptr, dev_status, st);
}

cudaError_t launch_accept_tree_greedy(const float *p, const int32_t *tokens, const int32_t *parent, int B,
                                      int D, int V, int32_t *n_acc, int32_t *token, int32_t *path,
                                      uint32_t *dev_status, cudaStream_t st)
{
    return launch_greedy<true>(p, tokens, parent, B, D, V, n_acc, token, path, dev_status, st);
}

template <int CS>
cudaError_t launch_tree_sample_cs(const float *p, const float *q, const int32_t *tokens, const int32_t *parent,
                                  const float *u_acc, const float *u_res, int B, int D, int V, int32_t *n_acc,
                                  int32_t *token, int32_t *path, uint32_t *dev_status, bool vec4, cudaStream_t st)
{
    const int64_t cta_len = ((static_cast<int64_t>(V) + CS - 1) / CS + 3) & ~int64_t(3);
    const uint32_t smem = static_cast<uint32_t>((cta_len + kTSGroup - 1) / kTSGroup) * 8u;
    if (smem > 48u * 1024u) {
        const cudaError_t e = cudaFuncSetAttribute(accept_tree_sample_kernel<CS>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B) * CS);
    cfg.blockDim = dim3(kTSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_tree_sample_kernel<CS>, p, q, tokens, parent, u_acc, u_res, D, V, n_acc,
                              token, path, dev_status, vec4);
}

cudaError_t launch_accept_tree_sample(const float *p, const float *q, const int32_t *tokens, const int32_t *parent,
                                      const float *u_acc, const float *u_res, int B, int D, int V,
                                      int32_t *n_acc, int32_t *token, int32_t *path, uint32_t *dev_status,
                                      cudaStream_t st)
{
    // slices start on 16-byte boundaries when rows do (V % 4 == 0)
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(q) % 16 == 0);
    switch (pick_cluster(V)) {
    case 8: return launch_tree_sample_cs<8>(p, q, tokens, parent, u_acc, u_res, B, D, V, n_acc, token, path,
                                            dev_status, vec4, st);
    case 4: return launch_tree_sample_cs<4>(p, q, tokens, parent, u_acc, u_res, B, D, V, n_acc, token, path,
                                            dev_status, vec4, st);
    case 2: return launch_tree_sample_cs<2>(p, q, tokens, parent, u_acc, u_res, B, D, V, n_acc, token, path,
                                            dev_status, vec4, st);
    default: return launch_tree_sample_cs<1>(p, q, tokens, parent, u_acc, u_res, B, D, V, n_acc, token, path,
                                             dev_status, vec4, st);
    }
}

namespace {

// The AdaSD decision stage's inputs and outputs.
struct AdaArgs {
    const float2 *parts;
    int nchunks;
    float tau_h, tau_js;
    float *entropy, *js_dist;
    int32_t *d_eff;
};

// Stages 1-3 of the stochastic acceptance (prep, stream, finalize) on the
// scratch that starts at `workspace`.  LOGITS: the first stage waits for the
// row statistics of the kernel before it (programmatic dependent launch).
// ada: the AdaSD decision stage replaces the first stage.
template <bool LOGITS>
cudaError_t launch_sample_stages(const SampleIn &in, const int32_t *draft, int B, int D, int V, int32_t *n_acc,
                                 int32_t *token, void *workspace, uint32_t *dev_status, cudaStream_t st,
                                 const AdaArgs *ada = nullptr)
{
    // bulk copies need 16-byte aligned rows: V % 4 == 0 and aligned bases
    const bool bulk = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(in.p) % 16 == 0) &&
                      (in.q == nullptr || reinterpret_cast<uintptr_t>(in.q) % 16 == 0);
    char *w = static_cast<char *>(workspace);
    SampleScratch sc;
    sc.nsteps = (V + kStep - 1) / kStep;
    sc.ngroups = (V + kGroup - 1) / kGroup;
    sc.js = reinterpret_cast<int32_t *>(w);
    w += align256(sizeof(int32_t) * B);
    sc.gtot = reinterpret_cast<unsigned long long *>(w);
    w += align256(sizeof(unsigned long long) * static_cast<size_t>(sc.ngroups) * B);
    sc.steps = reinterpret_cast<unsigned long long *>(w);

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(accept_stream_kernel<LOGITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kStreamSmem));
    if (e != cudaSuccess) return e;

    const unsigned sgrid = static_cast<unsigned>((B + kWarps - 1) / kWarps);
    if (ada) {
        // AdaSD: the decisions come from the row statistics of the kernel before
        e = launch_pdl(adasd_prep_kernel, dim3(sgrid), dim3(kThreads), 0u, st, in.p, in.q, draft, in.u_acc,
                       ada->parts, ada->nchunks, ada->tau_h, ada->tau_js, B, D, V, ada->entropy, ada->js_dist,
                       ada->d_eff, sc, dev_status);
    } else if (LOGITS) {
        e = launch_pdl(accept_prep_kernel<LOGITS>, dim3(sgrid), dim3(kThreads), 0u, st, in, draft, B, D, V, sc,
                       dev_status);
        // the exact sums of each sequence's draw rows
        if (e == cudaSuccess)
            e = launch_pdl(logits_draw_sums_kernel, dim3(static_cast<unsigned>(B) * in.nzchunks), dim3(kThreads), 0u,
                           st, in, D, V, sc, bulk, const_cast<float2 *>(in.zparts));
    } else {
        accept_prep_kernel<LOGITS><<<sgrid, kThreads, 0, st>>>(in, draft, B, D, V, sc, dev_status);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const int nchunks = (V + kChunk - 1) / kChunk;
    const long long items = static_cast<long long>(B) * nchunks;
    const int grid = static_cast<int>(items < sms ? items : sms);
    e = launch_pdl(accept_stream_kernel<LOGITS>, dim3(grid), dim3(kStreamThreads), kStreamSmem, st, in, D, V,
                   nchunks, static_cast<int>(items), sc, dev_status, bulk);
    if (e != cudaSuccess) return e;
    return launch_pdl(accept_finalize_kernel<LOGITS>, dim3(sgrid), dim3(kThreads), 0u, st, in, B, D, V, sc,
                      n_acc, token, dev_status, bulk);
}

constexpr uint32_t kStatsStaticSmem = 1024;   // bound on the row-statistics kernel's static shared memory

template <int CS, bool BULK>
cudaError_t launch_rowstats_cs(const float *zp, const float *zq, int B, int D, int V, float c_fast, int slice,
                               bool vec4, float2 *stats, uint32_t *dev_status, cudaStream_t st)
{
    auto kernel = logits_rowstats_kernel<CS, BULK>;
    const uint32_t smem = BULK ? static_cast<uint32_t>(slice) * 4u + 128u : 0u;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kStatsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many clusters as fit on the device at once, at most one per row
    const long long rows = static_cast<long long>(B) * (2 * D + 1);
    int clusters = 0;
    cfg.gridDim = dim3(CS);
    e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    if (clusters > rows) clusters = static_cast<int>(rows);
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * CS));
    return cudaLaunchKernelEx(&cfg, kernel, zp, zq, B, D, V, c_fast, slice, vec4, stats, dev_status);
}

template <int CS>
cudaError_t launch_rowstats(const float *zp, const float *zq, int B, int D, int V, float c_fast, float2 *stats,
                            uint32_t *dev_status, cudaStream_t st)
{
    const int slice = ((V + CS - 1) / CS + 3) & ~3;
    const bool aligned = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(zp) % 16 == 0) &&
                         (zq == nullptr || reinterpret_cast<uintptr_t>(zq) % 16 == 0);
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    const bool fits = static_cast<long long>(slice) * 4 + 128 + kStatsStaticSmem <= optin;
    if (aligned && fits)
        return launch_rowstats_cs<CS, true>(zp, zq, B, D, V, c_fast, slice, true, stats, dev_status, st);
    return launch_rowstats_cs<CS, false>(zp, zq, B, D, V, c_fast, slice, aligned, stats, dev_status, st);
}

}  // namespace

size_t accept_sample_workspace_bytes(int B, int V)
{
    const size_t nsteps = (static_cast<size_t>(V) + kStep - 1) / kStep;
    const size_t ngroups = (static_cast<size_t>(V) + kGroup - 1) / kGroup;
    return align256(sizeof(int32_t) * static_cast<size_t>(B)) +
           align256(sizeof(unsigned long long) * ngroups * static_cast<size_t>(B)) +
           align256(sizeof(unsigned long long) * nsteps * static_cast<size_t>(B));
}

cudaError_t launch_accept_sample(const float *p, const float *q, const int32_t *draft,
                                 const float *u_acc, const float *u_res, int B, int D, int V,
                                 int32_t *n_acc, int32_t *token, void *workspace,
                                 uint32_t *dev_status, cudaStream_t st)
{
    const SampleIn in{p, q, u_acc, u_res, nullptr, nullptr, 0, 0.0f, 1.0f, 0.0f, 0ull};
    return launch_sample_stages<false>(in, draft, B, D, V, n_acc, token, workspace, dev_status, st);
}

namespace {

size_t adasd_parts_bytes(int B, int D, int V)
{
    const size_t nchunks = (static_cast<size_t>(V) + kAdaChunk - 1) / kAdaChunk;
    return align256(sizeof(float2) * static_cast<size_t>(B) * D * nchunks);
}

size_t adasd_stats_bytes(int B, int D) { return align256(sizeof(float) * static_cast<size_t>(B) * D); }

}  // namespace

size_t accept_adasd_workspace_bytes(int B, int D, int V)
{
    return adasd_parts_bytes(B, D, V) + 2 * adasd_stats_bytes(B, D) + accept_sample_workspace_bytes(B, V);
}

cudaError_t launch_accept_adasd(const float *p, const float *q, const int32_t *draft, const float *u_acc,
                                const float *u_res, float tau_h, float tau_js, int B, int D, int V, int32_t *n_acc,
                                int32_t *token, int32_t *d_eff, float *entropy, float *js_dist, void *workspace,
                                uint32_t *dev_status, cudaStream_t st)
{
    char *w = static_cast<char *>(workspace);
    AdaArgs ada;
    ada.parts = reinterpret_cast<const float2 *>(w);
    ada.nchunks = (V + kAdaChunk - 1) / kAdaChunk;
    w += adasd_parts_bytes(B, D, V);
    ada.entropy = entropy ? entropy : reinterpret_cast<float *>(w);
    w += adasd_stats_bytes(B, D);
    ada.js_dist = js_dist ? js_dist : reinterpret_cast<float *>(w);
    w += adasd_stats_bytes(B, D);
    ada.tau_h = tau_h;
    ada.tau_js = tau_js;
    ada.d_eff = d_eff;
    if (D > 0) {
        const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                          (reinterpret_cast<uintptr_t>(q) % 16 == 0);
        const long long items = static_cast<long long>(B) * D * ada.nchunks;
        adasd_stats_kernel<<<static_cast<unsigned>(items), kThreads, 0, st>>>(
            p, q, D, V, ada.nchunks, vec4, const_cast<float2 *>(ada.parts));
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const SampleIn in{p, q, u_acc, u_res, nullptr, nullptr, 0, 0.0f, 1.0f, 0.0f, 0ull};
    return launch_sample_stages<false>(in, draft, B, D, V, n_acc, token, w, dev_status, st, &ada);
}

namespace {

size_t logits_stats_bytes(int B, int D)
{
    return align256(sizeof(float2) * static_cast<size_t>(B) * (2 * static_cast<size_t>(D) + 1));
}

int logits_zchunks(int V) { return (V + kZChunk - 1) / kZChunk; }

size_t logits_zparts_bytes(int B, int V)
{
    return align256(sizeof(float2) * static_cast<size_t>(B) * 2 * logits_zchunks(V));
}

}  // namespace

size_t accept_sample_logits_workspace_bytes(int B, int D, int V)
{
    return logits_stats_bytes(B, D) + logits_zparts_bytes(B, V) + accept_sample_workspace_bytes(B, V);
}

cudaError_t launch_accept_sample_logits(const float *zp, const float *zq, const int32_t *draft, float temperature,
                                        unsigned long long seed, int B, int D, int V, int32_t *n_acc,
                                        int32_t *token, void *workspace, uint32_t *dev_status, cudaStream_t st)
{
    char *w = static_cast<char *>(workspace);
    float2 *stats = reinterpret_cast<float2 *>(w);
    w += logits_stats_bytes(B, D);
    float2 *zparts = reinterpret_cast<float2 *>(w);
    w += logits_zparts_bytes(B, V);
    // fast evaluation: c = fl32(log2 e / T); exact one: 1 / T as hi + lo
    const double inv = 1.0 / static_cast<double>(temperature);
    const float c_fast = static_cast<float>(1.4426950408889634 * inv);
    const float ih = static_cast<float>(inv);
    const float il = static_cast<float>(inv - static_cast<double>(ih));
    cudaError_t e;
    switch (pick_cluster(V)) {
    case 8: e = launch_rowstats<8>(zp, zq, B, D, V, c_fast, stats, dev_status, st); break;
    case 4: e = launch_rowstats<4>(zp, zq, B, D, V, c_fast, stats, dev_status, st); break;
    case 2: e = launch_rowstats<2>(zp, zq, B, D, V, c_fast, stats, dev_status, st); break;
    default: e = launch_rowstats<1>(zp, zq, B, D, V, c_fast, stats, dev_status, st); break;
    }
    if (e != cudaSuccess) return e;
    const SampleIn in{zp, zq, nullptr, nullptr, stats, zparts, logits_zchunks(V), c_fast, ih, il, seed};
    return launch_sample_stages<true>(in, draft, B, D, V, n_acc, token, w, dev_status, st);
}

}  // namespace spec
