// Verify GEMM y[M][N] = x[M][K] . w[N][K]^T, bf16 in, fp32 accumulate in
// tensor memory, bf16 out.
//
// "Draft length and performance of linear layers" (co-design blog): with
// speculation every target linear layer runs at GEMM-M = M(1+D); the
// representative expert GEMM is N = K = 6144.  Small M streams the weights
// (HBM-bound); large M is a dense contraction on the tensor cores.
//
// Two warp-specialised kernels (warp 0: TMA producer, warp 1: MMA issuer,
// warps 2-5: epilogue), operands staged by TMA with the 128-byte swizzle,
// tcgen05.mma kind::f16 accumulating in TMEM:
//  * gemm_pair_kernel (M > 256): CTA pairs (clusters of 2) run one
//    tcgen05.mma of M = 256 together.  Each CTA loads its own 128 rows of x
//    and one half of the tile's w rows; the pair's tensor cores read both
//    halves, so each w byte crosses from L2 into one SM only.  Tiles are
//    whole (no split K) with ragged widths (multiples of 32 columns, chosen
//    so the tiles spread evenly over the pairs).
//  * gemm_split_kernel (M <= 256, when every tile's cluster fits at once):
//    A = w rows (128 per tile), B = the M rows of x padded to BN, so the
//    MMA is not mostly padding; the output is written transposed.  Each
//    tile's k-blocks are split over the S CTAs of a thread-block cluster,
//    whose fp32 pieces meet in their shared memory and are added in k
//    order (see the kernel).
//  * gemm_split_pair_kernel (64 < M <= 256, N a multiple of 256, when its
//    clusters fit and are not fewer CTAs): the same split with each MMA
//    shared by a CTA pair, each CTA staging half of the x rows.
//  * gemm_swap_kernel (M <= 256, otherwise): the same orientation; the
//    k-block iterations of all tiles are split evenly over the CTAs
//    (stream-K, see gemm_schedule.h): every piece of a tile cut between
//    CTAs leaves its fp32 partial in the workspace and counts itself in;
//    the last piece to arrive adds them all in k order (so results are
//    deterministic) and writes the tile.  No CTA waits for another.
// Output blocks of 32 x 32 are staged in shared memory by each epilogue warp and written by TMA tensor stores (coalesced, asynchronous;
// rows past M are clipped).
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "gemm.h"
#include "gemm_schedule.h"
#include "tmap.h"

namespace spec {
namespace {

constexpr int kBM = 128;       // MMA M
constexpr int kBK = 64;        // K per stage: one 128-byte swizzle row
constexpr int kThreads = 192;  // 6 warps
constexpr uint32_t kTileA = kBM * kBK * 2;

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// After an abort: wait (bounded) for the last copies this producer issued,
// so no TMA write lands in shared memory after the CTA has exited.
__device__ __forceinline__ void drain_copies(uint64_t *full, uint32_t issued, int stages)
{
    const uint32_t first = issued > static_cast<uint32_t>(stages) ? issued - stages : 0;
    for (uint32_t i = first; i < issued; ++i)
        mbar_wait_drain(&full[i % stages], (i / stages) & 1, 100000000ull);
}

// After an abort: wait (bounded) until every MMA this thread issued has
// finished, before tensor memory is released.
__device__ __forceinline__ void drain_mmas(uint64_t *drain)
{
    umma_commit(drain);
    mbar_wait_drain(drain, 0, 100000000ull);
}

// Issue the 4 MMAs (K = 16 each) of one 64-wide K block.
template <int N>
__device__ __forceinline__ void mma_kblock(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem,
                                           bool accumulate_first)
{
    constexpr uint32_t idesc = idesc_f16(kBM, N, /*bf16*/ 1, 0, 0);
#pragma unroll
    for (int k = 0; k < kBK / 16; ++k) {
        const uint64_t a = sdesc(a_smem + k * 32, 16, 1024);
        const uint64_t b = sdesc(b_smem + k * 32, 16, 1024);
        umma_f16_ss(d_tmem, a, b, idesc, (accumulate_first || k > 0) ? 1u : 0u);
    }
}

__device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Partial tiles (128 rows x BN fp32) are laid out in 32-column units of
// 16 KB, each [8 column quads][128 rows][4]: a warp's float4 accesses to one
// quad are contiguous, and a unit is one bulk copy.
__device__ __forceinline__ uint32_t unit_index(int quad, int row)
{
    return static_cast<uint32_t>((quad * kBM + row) * 4);
}
__device__ __forceinline__ uint32_t partial_index(int cc, int quad, int row)
{
    return static_cast<uint32_t>(cc * 32 * kBM) + unit_index(quad, row);
}

// Partial slot of the piece that unit v's CTA `rank` holds: two per CTA,
// for the first and the last segment of its stream-K range.
__device__ __forceinline__ int piece_slot(int v, int rank, bool first_segment, int unit_ctas)
{
    return (v * unit_ctas + rank) * 2 + (first_segment ? 0 : 1);
}

// Whether unit f's stream-K range starts exactly at tile t's first k-block
// (then f's piece of t is its first segment).
__device__ __forceinline__ bool other_first(const SkGrid &g, int f, int t)
{
    return g.begin(f) == static_cast<long long>(t - g.dp_tiles) * g.kblocks;
}

// Output staging: each epilogue warp owns two 32 x 32 bf16 blocks (2 KB).
constexpr uint32_t kOutBlock = 32 * 32 * 2;
constexpr uint32_t kOutStaging = 4 * 2 * kOutBlock;

__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one bulk group of this thread still reading its shared source
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every bulk group of this thread has finished reading its shared source
// (the writes themselves complete by the end of the grid)
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Column quads of 32-column chunk cc that a cut tile's pieces publish and
// add: a swap tile has a column per row of x, so only the quads that hold
// rows m < M.
__device__ __forceinline__ int live_quads(int M, int cc)
{
    const int q = (M - cc * 32 + 3) / 4;
    return q < 8 ? q : 8;
}

// Take the warp's next 2 KB staging buffer (the store issued from it two
// blocks ago has finished reading it).
__device__ __forceinline__ uint8_t *next_out_buffer(uint8_t *obuf, uint32_t nst, int lane)
{
    if (lane == 0) bulk_wait_read_1();
    __syncwarp();
    return obuf + (nst & 1u) * kOutBlock;
}

// Make the staged block visible to the TMA unit and store it with lane 0.
__device__ __forceinline__ void issue_out_store(const CUtensorMap *tm, const uint8_t *buf, int lane, int x, int y,
                                                uint32_t &nst)
{
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tm, buf, x, y);
        bulk_commit();
    }
    ++nst;
}

// Swap orientation: tile row = w row n = y column, tile column = x row m, so
// the warp's 32 tile rows x 32 columns (chunk cc) are transposed while
// staged and stored at (x = 128 t + 32 quad, y = 32 cc).
__device__ __forceinline__ void store_out_swap(const CUtensorMap *tm_y, uint8_t *obuf, uint32_t &nst, int lane,
                                               int t, int quad, int cc, const float (&a)[32])
{
    uint8_t *buf = next_out_buffer(obuf, nst, lane);
    __nv_bfloat16 *b = reinterpret_cast<__nv_bfloat16 *>(buf);
#pragma unroll
    for (int j = 0; j < 32; ++j) b[j * 32 + lane] = __float2bfloat16_rn(a[j]);
    issue_out_store(tm_y, buf, lane, t * kBM + quad * 32, cc * 32, nst);
}

// Pair tiles: 32 columns of the warp's 32 rows, row-major, at (x = column,
// y = row) of y.
__device__ __forceinline__ void store_out_rows(const CUtensorMap *tm_y, uint8_t *obuf, uint32_t &nst, int lane,
                                               int x, int y, const uint32_t (&r)[32])
{
    uint8_t *buf = next_out_buffer(obuf, nst, lane);
    uint4 *b = reinterpret_cast<uint4 *>(buf + lane * 64);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        uint4 o;
        o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
        o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
        o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
        o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
        b[v] = o;
    }
    issue_out_store(tm_y, buf, lane, x, y, nst);
}

template <int BN, int STAGES>
struct TiledSmem {
    static constexpr uint32_t kTileB = BN * kBK * 2;
    static constexpr uint32_t kStage = kTileA + kTileB;
    static constexpr uint32_t kBytes = STAGES * kStage + kOutStaging + 1024 /*align*/ + 256 /*barriers*/;
    static_assert(STAGES * kStage >= kBM * BN * 4, "a partial tile must fit in the stage ring");
};

constexpr int stages_for(int bn) { return bn >= 256 ? 4 : bn >= 128 ? 6 : 8; }

// Weight streaming: 128-row w tiles, A = w, B = x padded to BN rows, single
// CTAs, stream-K split.
template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_y, int M, int N, SkGrid grid, float *__restrict__ part,
                uint32_t *__restrict__ flags, uint32_t *dev_status)
{
    using L = TiledSmem<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *out_stage = smem + STAGES * L::kStage;   // 4 warps x 2 output blocks
    uint64_t *full = reinterpret_cast<uint64_t *>(out_stage + kOutStaging);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint64_t *pub_bar = drain + 1;      // 4 epilogue warps stored a partial
    uint64_t *dec_bar = pub_bar + 1;    // whether this piece arrived last is known
    uint64_t *red_full = dec_bar + 1;   // other pieces' partials landed in the ring
    uint64_t *red_empty = red_full + 1; // 4 epilogue warps finished reading them
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(red_empty + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *s_last = abort + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = 0;
    const int c = static_cast<int>(blockIdx.x);
    constexpr int kUnit = 1;   // CTAs per unit of the split
    if (cluster_ctas() != 1u) {   // uniform over the grid
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], 4); }
        mbar_init(drain, 1);
        mbar_init(pub_bar, 4);
        mbar_init(dec_bar, 1);
        mbar_init(red_full, 1);
        mbar_init(red_empty, 4);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(tmem_slot, 2 * BN); tmem_relinquish(); }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_y);
        SegWalker wk(grid, c);
        Seg s;
        uint32_t it = 0;
        while (!*abort && wk.next(s)) {
            for (int kb = s.kb0; kb < s.kb1; ++kb, ++it) {
                const int st = it % STAGES;
                if (it >= STAGES && !mbar_wait(&empty[st], ((it / STAGES) & 1) ^ 1, abort, dev_status)) break;
                uint8_t *sa = smem + st * L::kStage;
                mbar_arrive_expect_tx(&full[st], L::kStage);
                tma_load_2d(sa, &tm_w, &full[st], kb * kBK, s.t * kBM);
                tma_load_2d(sa + kTileA, &tm_x, &full[st], kb * kBK, 0);
            }
        }
        if (*abort) drain_copies(full, it, STAGES);
    } else if (warp == 1 && lane == 0) {
        SegWalker wk(grid, c);
        Seg s;
        uint32_t it = 0, lt = 0;
        while (!*abort && wk.next(s)) {
            const uint32_t ab = lt & 1;
            if (lt >= 2 && !mbar_wait(&acc_empty[ab], ((lt >> 1) & 1) ^ 1, abort, dev_status)) break;
            tc_fence_after();
            const uint32_t d = tmem + ab * BN;
            bool ok = true;
            for (int kb = s.kb0; kb < s.kb1; ++kb, ++it) {
                const int st = it % STAGES;
                if (!mbar_wait(&full[st], (it / STAGES) & 1, abort, dev_status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + st * L::kStage);
                mma_kblock<BN>(d, sa, sa + kTileA, kb > s.kb0);
                umma_commit(&empty[st]);
            }
            if (!ok) break;
            umma_commit(&acc_full[ab]);
            ++lt;
        }
    } else if (warp >= 2) {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        // only the 32-column chunks that hold rows of x are needed
        const int nchunks = (M + 31) / 32 < BN / 32 ? (M + 31) / 32 : BN / 32;
        SegWalker wk(grid, c);
        Seg s;
        uint32_t lt = 0, npub = 0, nred = 0, ndec = 0;
        uint8_t *obuf = out_stage + (warp - 2) * 2 * kOutBlock;
        uint32_t nst = 0;   // output blocks this warp has stored
        while (!*abort && wk.next(s)) {
            const uint32_t ab = lt & 1;
            if (!mbar_wait_warp(&acc_full[ab], (lt >> 1) & 1, abort, dev_status)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((quad * 32) << 16) + ab * BN;
            bool ok = true;
            if (s.kb0 == 0 && s.kb1 == grid.kblocks) {
                // a whole tile
#pragma unroll 1
                for (int cc = 0; cc < nchunks; ++cc) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + cc * 32, r);
                    tmem_ld_wait();
                    float a[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) a[j] = __uint_as_float(r[j]);
                    store_out_swap(&tm_y, obuf, nst, lane, s.t, quad, cc, a);
                }
            } else {
                // A piece of a cut tile: publish the fp32 partial, then count
                // the tile's published pieces; the last piece to arrive adds
                // all of them in k order and writes the tile.  No CTA ever
                // waits for another, so residency is never assumed.
                int f, l;
                sk_tile_units(grid, s.t, f, l);
                const int me = c;
                const int my_slot = piece_slot(me, rank, sk_first_segment(grid, me, s), kUnit);
                float *slot = part + static_cast<size_t>(my_slot) * kBM * BN;
                uint32_t *cnt = flags + (s.t - grid.dp_tiles) * kUnit + rank;
                // A piece that ends its unit's range usually finishes with or
                // after the others: if all of them have arrived already it is
                // the last for sure and need not publish its own partial.
                bool sure_last = false;
                if (!wk.has_more()) {
                    uint32_t seen = 0;
                    if (lane == 0) seen = ld_acquire(cnt);
                    sure_last = __shfl_sync(0xffffffffu, seen, 0) == static_cast<uint32_t>(l - f);
                }
#pragma unroll 1
                for (int cc = 0; cc < nchunks && !sure_last; ++cc) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + cc * 32, r);
                    tmem_ld_wait();
                    const int nq = live_quads(M, cc);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        if (q4 < nq)
                            __stcg(reinterpret_cast<float4 *>(slot + partial_index(cc, q4, row)),
                                   make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                                               __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3])));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(pub_bar);
                if (threadIdx.x == 64) {
                    bool last = false;
                    if (mbar_wait(pub_bar, npub & 1, abort, dev_status)) {
                        if (sure_last) {
                            last = true;
                        } else {
                            __threadfence();
                            last = atomicAdd(cnt, 1u) == static_cast<uint32_t>(l - f);
                        }
                        if (last) {
                            __threadfence();
                            *cnt = 0u;   // zero again for the next call
                        }
                    }
                    *s_last = last ? 1 : 0;
                    mbar_arrive(dec_bar);
                }
                __syncwarp();
                ++npub;
                ok = mbar_wait_warp(dec_bar, ndec & 1, abort, dev_status);
                ++ndec;
                if (ok && *s_last) {
                    // other pieces' partials: through the stage ring with bulk
                    // copies when this is the unit's last segment (the ring is
                    // idle then) and they are large, else straight from L2 (a
                    // swap tile with one 32-column chunk holds a few KB per
                    // piece: plain loads save the copies' barrier round trip)
                    const bool ring_ok = !wk.has_more() && nchunks != 1;
                    const float *ring = reinterpret_cast<const float *>(smem);
                    const int others = l - f;
                    const int per_pass_chunks =
                        ring_ok ? imin((STAGES * static_cast<int>(L::kStage)) / (others * 32 * kBM * 4), nchunks)
                                : 1;
                    for (int c0 = 0; c0 < nchunks && ok; c0 += per_pass_chunks) {
                        const int c1 = imin(nchunks, c0 + per_pass_chunks);
                        if (ring_ok) {
                            if (threadIdx.x == 64) {
                                bool go = nred == 0 || mbar_wait(red_empty, (nred - 1) & 1, abort, dev_status);
                                if (go) {
                                    fence_proxy_async_all();
                                    uint32_t bytes = 0;
                                    for (int cc = c0; cc < c1; ++cc) bytes += live_quads(M, cc) * kBM * 16;
                                    mbar_arrive_expect_tx(red_full, bytes * others);
                                    int k = 0;
                                    for (int v = f; v <= l; ++v) {
                                        if (v == me) continue;
                                        const float *src = part + static_cast<size_t>(
                                            piece_slot(v, rank, v != f || other_first(grid, f, s.t), kUnit)) * kBM * BN;
                                        // a unit's quads are its outer index: the live ones are its first bytes
                                        for (int cc = c0; cc < c1; ++cc)
                                            bulk_load(smem + ((cc - c0) * others + k) * 32 * kBM * 4,
                                                      src + cc * 32 * kBM, live_quads(M, cc) * kBM * 16, red_full);
                                        ++k;
                                    }
                                }
                            }
                            __syncwarp();
                            ok = mbar_wait_warp(red_full, nred & 1, abort, dev_status);
                            if (!ok) break;
                        }
#pragma unroll 1
                        for (int cc = c0; cc < c1; ++cc) {
                            uint32_t r[32];
                            tmem_ld_32x32b_x32(tbase + cc * 32, r);
                            tmem_ld_wait();
                            float a[32];
                            int k = 0;
                            for (int v = f; v <= l; ++v) {
                                float4 pv[8];
                                if (v == me) {
#pragma unroll
                                    for (int q4 = 0; q4 < 8; ++q4)
                                        pv[q4] = make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                                                             __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]));
                                } else {
                                    // columns past the live quads are rows m >= M, never stored
                                    const int nq = live_quads(M, cc);
                                    if (ring_ok) {
                                        const float *u = ring + ((cc - c0) * others + k) * 32 * kBM;
#pragma unroll
                                        for (int q4 = 0; q4 < 8; ++q4)
                                            pv[q4] = q4 < nq ? *reinterpret_cast<const float4 *>(u + unit_index(q4, row))
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                                    } else {
                                        const float *src = part + static_cast<size_t>(piece_slot(
                                            v, rank, v != f || other_first(grid, f, s.t), kUnit)) * kBM * BN;
#pragma unroll
                                        for (int q4 = 0; q4 < 8; ++q4)
                                            pv[q4] = q4 < nq ? __ldcg(reinterpret_cast<const float4 *>(src + partial_index(cc, q4, row)))
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                                    }
                                    ++k;
                                }
                                // k order, the same whichever piece arrived last
#pragma unroll
                                for (int q4 = 0; q4 < 8; ++q4) {
                                    if (v == f) {
                                        a[4 * q4] = pv[q4].x; a[4 * q4 + 1] = pv[q4].y;
                                        a[4 * q4 + 2] = pv[q4].z; a[4 * q4 + 3] = pv[q4].w;
                                    } else {
                                        a[4 * q4] += pv[q4].x; a[4 * q4 + 1] += pv[q4].y;
                                        a[4 * q4 + 2] += pv[q4].z; a[4 * q4 + 3] += pv[q4].w;
                                    }
                                }
                            }
                            store_out_swap(&tm_y, obuf, nst, lane, s.t, quad, cc, a);
                        }
                        if (ring_ok) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(red_empty);
                            ++nred;
                        }
                    }
                }
            }
            if (!ok) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
            ++lt;
        }
        if (lane == 0) bulk_wait_read_all();   // staged output read before the CTA's shared memory goes
    }
    __syncwarp();
    __syncthreads();
    if (*abort && threadIdx.x == 32) drain_mmas(drain);
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 2 * BN); }
}

// ------------------------------------------------- weight streaming, split K
// M <= 256 with few 128-row w tiles (N = 6144: 48): tile t's k-blocks are
// cut into S equal ranges, one per CTA of a cluster of S (rank r takes
// k-blocks [r K/S, (r + 1) K/S) of K/64), all of a tile's CTAs resident
// together.  Each CTA streams its range (KPS k-blocks per stage) into its
// own tensor-memory accumulator.  Once every CTA of the cluster has
// finished its MMAs (a cluster barrier), their stage rings are idle and
// receive the partial sums: 32-column chunk cc of the tile belongs to CTA
// cc % S, and every other CTA sends its fp32 piece of the chunk into slot
// (cc / S, rank) of the owner's ring by asynchronous shared-memory stores
// that complete on the owner's mbarrier.  The owner adds the S pieces in
// rank (= k) order, its own read from its tensor memory, and stores the
// chunk as bf16.  Against stream-K this
// removes the fp32 partials' round trip through L2 and the tile fix-up
// that one CTA did alone after all others had finished.
template <int BN>
struct SplitCfg {
    static constexpr int kKps = 2;                                      // k-blocks per stage
    static constexpr int kStages = BN >= 256 ? 2 : BN >= 128 ? 3 : 4;
    static constexpr uint32_t kTileB = BN * kBK * 2;
    static constexpr uint32_t kStage = kKps * (kTileA + kTileB);
    static constexpr uint32_t kRing = kStages * kStage;
    static constexpr uint32_t kBytes = kRing + kOutStaging + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr uint32_t kChunkBytes = 32 * kBM * 4;            // one fp32 piece of a chunk
};

// Whether a cluster of S CTAs can hold the pieces its CTAs receive (each
// owns ceil(chunks / S) chunks of S pieces) in one CTA's stage ring.
template <int BN>
__host__ __device__ constexpr bool split_fits(int S)
{
    return S >= 2 && S <= 8 &&
           static_cast<uint32_t>(S * ((BN / 32 + S - 1) / S)) * SplitCfg<BN>::kChunkBytes <= SplitCfg<BN>::kRing;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_split_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_y, int M, int kblocks, uint32_t *dev_status)
{
    using C = SplitCfg<BN>;
    constexpr int STAGES = C::kStages, KPS = C::kKps;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *out_stage = smem + C::kRing;   // 4 warps x 2 output blocks
    uint64_t *full = reinterpret_cast<uint64_t *>(out_stage + kOutStaging);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *recv = acc_full + 1;    // the pieces of this CTA's chunks landed
    uint64_t *drain = recv + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = static_cast<int>(cluster_ctas());
    if (!split_fits<BN>(S) || kblocks < S) {   // uniform over the grid
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        return;
    }
    const int rank = static_cast<int>(cluster_rank());
    const int t = static_cast<int>(blockIdx.x) / S;
    const int kb0 = rank * kblocks / S, kb1 = (rank + 1) * kblocks / S;
    const int nchunks = (M + 31) / 32 < BN / 32 ? (M + 31) / 32 : BN / 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(acc_full, 1);
        mbar_init(recv, 1);
        mbar_init(drain, 1);
        *abort = 0;
        // the bytes this CTA will receive: S - 1 pieces of each chunk it owns
        uint32_t bytes = 0;
        for (int cc = rank; cc < nchunks; cc += S)
            bytes += static_cast<uint32_t>((S - 1) * live_quads(M, cc)) * kBM * 16;
        mbar_arrive_expect_tx(recv, bytes);
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(tmem_slot, BN); tmem_relinquish(); }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_y);
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1 && !*abort; kb += KPS, ++it) {
            const int nk = kb1 - kb < KPS ? kb1 - kb : KPS;
            const int st = static_cast<int>(it % STAGES);
            if (it >= static_cast<uint32_t>(STAGES) &&
                !mbar_wait(&empty[st], ((it / STAGES) & 1) ^ 1, abort, dev_status)) break;
            uint8_t *sa = smem + st * C::kStage;
            mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(nk) * (kTileA + C::kTileB));
            for (int q = 0; q < nk; ++q) {
                tma_load_2d(sa + q * kTileA, &tm_w, &full[st], (kb + q) * kBK, t * kBM);
                tma_load_2d(sa + KPS * kTileA + q * C::kTileB, &tm_x, &full[st], (kb + q) * kBK, 0);
            }
        }
        if (*abort) drain_copies(full, it, STAGES);
    } else if (warp == 1 && lane == 0) {
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; kb += KPS, ++it) {
            const int nk = kb1 - kb < KPS ? kb1 - kb : KPS;
            const int st = static_cast<int>(it % STAGES);
            if (!mbar_wait(&full[st], (it / STAGES) & 1, abort, dev_status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + st * C::kStage);
            for (int q = 0; q < nk; ++q)
                mma_kblock<BN>(tmem, sa + q * kTileA, sa + KPS * kTileA + q * C::kTileB, it > 0 || q > 0);
            umma_commit(&empty[st]);
        }
        if (ok) umma_commit(acc_full);
    } else if (warp >= 2) {
        ok = mbar_wait_warp(acc_full, 0, abort, dev_status);
        tc_fence_after();
    }
    // every CTA of the cluster is done with its stage ring (its MMAs have
    // completed: the epilogue warps arrive after the accumulator is final)
    __syncwarp();
    cluster_arrive_release();
    cluster_wait_acquire();
    tc_fence_after();

    if (warp >= 2) {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t tbase = tmem + ((quad * 32) << 16);
        // send: this CTA's piece of every chunk it does not own to the owner
#pragma unroll 1
        for (int cc = 0; cc < nchunks && ok && !*abort; ++cc) {
            if (cc % S == rank) continue;
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + cc * 32, r);
            tmem_ld_wait();
            const uint32_t owner = static_cast<uint32_t>(cc % S);
            const float *slot =
                reinterpret_cast<const float *>(smem) + static_cast<size_t>((cc / S) * S + rank) * (32 * kBM);
            const uint32_t dst = peer_smem(slot, owner);
            const uint32_t bar = peer_smem(recv, owner);
            const int nq = live_quads(M, cc);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                if (q4 < nq)
                    st_async_peer_v4(dst + unit_index(q4, row) * 4, r[4 * q4], r[4 * q4 + 1], r[4 * q4 + 2],
                                     r[4 * q4 + 3], bar);
        }
        // receive: the S pieces of each owned chunk, added in k order
        if (ok) ok = mbar_wait_warp(recv, 0, abort, dev_status);
        uint8_t *obuf = out_stage + (warp - 2) * 2 * kOutBlock;
        uint32_t nst = 0;
#pragma unroll 1
        for (int cc = rank; cc < nchunks && ok; cc += S) {
            const int nq = live_quads(M, cc);
            const float *base = reinterpret_cast<const float *>(smem) + static_cast<size_t>((cc / S) * S) * (32 * kBM);
            uint32_t own[32];
            tmem_ld_32x32b_x32(tbase + cc * 32, own);
            tmem_ld_wait();
            float a[32];
            for (int src = 0; src < S; ++src) {
                const float *u = base + static_cast<size_t>(src) * (32 * kBM);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    float4 v = make_float4(__uint_as_float(own[4 * q4]), __uint_as_float(own[4 * q4 + 1]),
                                           __uint_as_float(own[4 * q4 + 2]), __uint_as_float(own[4 * q4 + 3]));
                    if (src != rank)
                        v = q4 < nq ? *reinterpret_cast<const float4 *>(u + unit_index(q4, row))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                    if (src == 0) {
                        a[4 * q4] = v.x; a[4 * q4 + 1] = v.y; a[4 * q4 + 2] = v.z; a[4 * q4 + 3] = v.w;
                    } else {
                        a[4 * q4] += v.x; a[4 * q4 + 1] += v.y; a[4 * q4 + 2] += v.z; a[4 * q4 + 3] += v.w;
                    }
                }
            }
            store_out_swap(&tm_y, obuf, nst, lane, t, quad, cc, a);
        }
        if (lane == 0) bulk_wait_read_all();   // staged output read before the CTA's shared memory goes
        tc_fence_before();                     // the tensor-memory reads, before the deallocation
    }
    // no CTA leaves while a peer may still send into it
    __syncwarp();
    cluster_exit_barrier();
    __syncthreads();
    if (*abort && threadIdx.x == 32) drain_mmas(drain);
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, BN); }
}

// ------------------------------------------------------------- CTA pairs
// M > 256: one tcgen05.mma of M = 256 per 16-deep K step, shared by the two
// CTAs of a cluster.  Per 64-wide k-block each CTA stages its own 128 rows
// of x (16 KB) and its half of the tile's w rows (W / 2 rows, at most 16 KB;
// W a multiple of 32, so each half is whole 16-row groups) in its shared
// memory.  Both CTAs' copies of a stage complete on the even CTA's barrier
// (the .cta_group::2 form of the TMA load may signal the barrier of the
// pair's other CTA), the even CTA issues the MMAs once the stage has landed
// in both, and the commit signals the stage free in both CTAs.  The
// accumulator (128 rows x W fp32 per CTA) lives in each CTA's tensor memory
// and each CTA's epilogue writes its own 128 output rows.
// A stage carries kPairKps k-blocks: [x kb][x kb + 1][w kb][w kb + 1].
// A ring of tensor copies completes about one stage per ~0.45 us per SM
// whatever the stage's bytes (16 to 64 KB) and the ring depth (a copy
// micro-benchmark on GB300), so a stage must carry enough work: with one
// k-block per stage a stage completed every ~0.37 us whatever the tile
// width, the bytes staged and the stage count (6 to 8), and the MMAs, which
// need 0.21 us per k-block at 256 x 160 tiles, waited.  Measured and no
// faster: a second producer warp filling alternate stages, each pair
// starting at its own k-block, three k-blocks per stage in two stages
// (slower: a stage's refill waits for its MMAs), x shared by two pairs
// through cluster multicast (clusters of 4), TMA prefetches into L2 ahead
// of the loads, direct global stores from eight epilogue warps.
constexpr int kPairKps = 2;
constexpr int kPairStages = 3;
constexpr uint32_t kPairTileB = 128 * kBK * 2;            // up to 128 w rows per CTA
constexpr uint32_t kPairStage = kPairKps * (kTileA + kPairTileB);   // 64 KB
constexpr uint32_t kPairSmem = kPairStages * kPairStage + kOutStaging + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t kPairTmemCols = 256;                   // one accumulator, W <= 256
constexpr uint16_t kPairMask = 0x3;

// Tiled 2-D TMA load into this CTA's shared memory whose completion is
// counted on `bar_cluster`, a barrier of this CTA or of its pair peer
// (cluster-window address).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const void *tmap, uint32_t bar_cluster, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w_narrow,
                     const __grid_constant__ CUtensorMap tm_w_wide, const __grid_constant__ CUtensorMap tm_y,
                     int M, PairGrid g, uint32_t *dev_status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *out_stage = smem + kPairStages * kPairStage;   // 4 warps x 2 output blocks
    uint64_t *full = reinterpret_cast<uint64_t *>(out_stage + kOutStaging);   // (even CTA) stage landed in both
    uint64_t *empty = full + kPairStages;        // the pair's MMAs are done with the stage
    uint64_t *acc_full = empty + kPairStages;
    uint64_t *acc_empty = acc_full + 1;          // (even CTA) both CTAs' epilogues read the accumulator
    uint64_t *drain = acc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (cluster_ctas() != 2u) {   // uniform over the grid
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        return;
    }
    const uint32_t rank = cluster_rank();
    const int c = static_cast<int>(blockIdx.x >> 1);
    const int pairs = static_cast<int>(gridDim.x >> 1);
    const int tiles = g.tiles();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kPairTmemCols);
        tmem_relinquish_pair();
        tc_fence_before();
    }
    cluster_sync_all();   // both CTAs' barriers and allocations exist before anything targets them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the pair's accumulators must sit at the same tensor-memory address
    if (ld_cluster_u32(cluster_smem(tmem_slot, rank ^ 1u)) != tmem) {
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        *abort = 1;
    }
    __syncthreads();

    if (warp == 0 && lane == 0) {
        // producer: this CTA's x rows and half of the tile's w rows, counted
        // on the even CTA's full barrier (which expects both CTAs' bytes)
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w_narrow);
        tma_prefetch_desc(&tm_w_wide);
        tma_prefetch_desc(&tm_y);
        const uint32_t full0 = cluster_smem(full, 0);
        uint32_t it = 0;
        for (int t = c; t < tiles && !*abort; t += pairs) {
            const int mt = t % g.tiles_m, nt = t / g.tiles_m;
            const int half = g.width(nt) / 2;
            const CUtensorMap *tw = half == 16 * g.q ? &tm_w_narrow : &tm_w_wide;
            const uint32_t bytes = kTileA + static_cast<uint32_t>(half) * kBK * 2;
            const int row_x = (2 * mt + static_cast<int>(rank)) * kBM;
            const int row_w = g.col0(nt) + static_cast<int>(rank) * half;
            bool ok = true;
            for (int kb0 = 0; kb0 < g.kblocks; kb0 += kPairKps, ++it) {
                const int nk = g.kblocks - kb0 < kPairKps ? g.kblocks - kb0 : kPairKps;
                const int st = it % kPairStages;
                if (it >= kPairStages &&
                    !mbar_wait(&empty[st], ((it / kPairStages) & 1) ^ 1, abort, dev_status)) { ok = false; break; }
                uint8_t *sa = smem + st * kPairStage;
                if (rank == 0) mbar_arrive_expect_tx(&full[st], 2 * bytes * nk);
                for (int q = 0; q < nk; ++q) {
                    tma_load_2d_pair(sa + q * kTileA, &tm_x, full0 + st * 8, (kb0 + q) * kBK, row_x);
                    tma_load_2d_pair(sa + kPairKps * kTileA + q * kPairTileB, tw, full0 + st * 8, (kb0 + q) * kBK,
                                     row_w);
                }
            }
            if (!ok) break;
        }
        if (!*abort) {
            // the last commits signal this CTA's empty barriers (and mean its
            // copies were consumed): wait for them before this CTA may exit
            const uint32_t first = it > static_cast<uint32_t>(kPairStages) ? it - kPairStages : 0;
            for (uint32_t i = first; i < it; ++i)
                if (!mbar_wait(&empty[i % kPairStages], (i / kPairStages) & 1, abort, dev_status)) break;
        }
        if (*abort) {
            // copies in flight complete on the even CTA's full barriers: drain
            // those (bounded), then give any straggler 0.2 ms to land
            if (rank == 0) drain_copies(full, it, kPairStages);
            const unsigned long long t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 200000ull) {
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // MMA issuer (even CTA)
        uint32_t it = 0, lt = 0;
        for (int t = c; t < tiles && !*abort; t += pairs, ++lt) {
            const int nt = t / g.tiles_m;
            const uint32_t idesc = idesc_f16(2 * kBM, g.width(nt), /*bf16*/ 1, 0, 0);
            if (lt >= 1 && !mbar_wait(acc_empty, (lt - 1) & 1, abort, dev_status)) break;
            tc_fence_after();
            bool ok = true;
            for (int kb0 = 0; kb0 < g.kblocks; kb0 += kPairKps, ++it) {
                const int nk = g.kblocks - kb0 < kPairKps ? g.kblocks - kb0 : kPairKps;
                const int st = it % kPairStages;
                if (!mbar_wait(&full[st], (it / kPairStages) & 1, abort, dev_status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + st * kPairStage);
                for (int q = 0; q < nk; ++q) {
                    const uint32_t a = sa + q * kTileA, b = sa + kPairKps * kTileA + q * kPairTileB;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        umma_f16_ss_pair(tmem, sdesc(a + k * 32, 16, 1024), sdesc(b + k * 32, 16, 1024), idesc,
                                         (kb0 > 0 || q > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit_pair(&empty[st], kPairMask);
            }
            if (!ok) break;
            umma_commit_pair(acc_full, kPairMask);
        }
    } else if (warp >= 2) {
        // epilogue: this CTA's 128 rows of each tile, 32 rows per warp
        const int quad = warp & 3;
        uint8_t *obuf = out_stage + (warp - 2) * 2 * kOutBlock;
        const uint32_t acc_empty0 = cluster_smem(acc_empty, 0);
        uint32_t nst = 0, lt = 0;
        for (int t = c; t < tiles && !*abort; t += pairs, ++lt) {
            const int mt = t % g.tiles_m, nt = t / g.tiles_m;
            const int W = g.width(nt), n0 = g.col0(nt);
            if (!mbar_wait_warp(acc_full, lt & 1, abort, dev_status)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((quad * 32) << 16);
            const int y0 = (2 * mt + static_cast<int>(rank)) * kBM + quad * 32;
#pragma unroll 1
            for (int cc = y0 < M ? 0 : W; cc < W; cc += 32) {   // rows past M: nothing to store
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + cc, r);
                tmem_ld_wait();
                store_out_rows(&tm_y, obuf, nst, lane, n0 + cc, y0, r);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty0);
        }
        if (lane == 0) bulk_wait_read_all();   // staged output read before the CTA's shared memory goes
    }
    __syncwarp();
    __syncthreads();
    if (*abort && rank == 0 && threadIdx.x == 32) {
        // let every pair MMA issued so far finish before tensor memory goes
        umma_commit_pair(drain, 0x1);
        mbar_wait_drain(drain, 0, 100000000ull);
    }
    cluster_sync_all();   // neither CTA exits while the other may still signal or read it
    if (warp == 1) { tc_fence_after(); tmem_dealloc_pair(tmem, kPairTmemCols); }
}

// ------------------------------------- weight streaming, split K, CTA pairs
// 64 < M <= 256 with N a multiple of 256: the split above with each MMA
// shared by a CTA pair (tcgen05 cta_group::2).  A pair tile is 256 w rows
// (128 per CTA, the MMA's M side) and the pair's MMAs read half of the
// padded x rows from each CTA (the N side), so an SM takes in half of x per
// k-block instead of all of it: at M = 256 the x rows of a k-block are
// twice its w rows, and the single-CTA split streams at the SMs' L2 read
// rate, not HBM's.  A cluster holds S pairs (2S CTAs); pair p takes
// k-blocks [p K/S, (p + 1) K/S) of the pair tile and CTA 2p + h holds w
// rows h * 128 .. + 127 of it.  Both CTAs' copies of a stage complete on
// the pair's even CTA's barrier, whose MMA thread issues the pair's MMAs
// and commits to both.  After the cluster barrier the pieces of each
// 32-column chunk are exchanged among the S CTAs that hold the same w rows
// (the same h) exactly as in the single-CTA split, and added in k order.
template <int BN>
struct SplitPairCfg {
    static constexpr int kKps = 2;                                      // k-blocks per stage
    static constexpr int kStages = BN >= 256 ? 3 : 4;
    static constexpr uint32_t kTileB = (BN / 2) * kBK * 2;             // this CTA's half of the x rows
    static constexpr uint32_t kStage = kKps * (kTileA + kTileB);
    static constexpr uint32_t kRing = kStages * kStage;
    static constexpr uint32_t kBytes = kRing + kOutStaging + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr uint32_t kChunkBytes = 32 * kBM * 4;
};

// S pairs per cluster (2S CTAs, at most 8): each CTA receives the pieces of
// ceil(chunks / S) chunks from S sources in its stage ring.
template <int BN>
__host__ __device__ constexpr bool split_pair_fits(int S)
{
    return (BN == 128 || BN == 256) && S >= 2 && 2 * S <= 8 &&
           static_cast<uint32_t>(S * ((BN / 32 + S - 1) / S)) * SplitPairCfg<BN>::kChunkBytes <=
               SplitPairCfg<BN>::kRing;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_split_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_y, int M, int kblocks, uint32_t *dev_status)
{
    using C = SplitPairCfg<BN>;
    constexpr int STAGES = C::kStages, KPS = C::kKps;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *out_stage = smem + C::kRing;   // 4 warps x 2 output blocks
    uint64_t *full = reinterpret_cast<uint64_t *>(out_stage + kOutStaging);   // (even CTA) stage landed in both
    uint64_t *empty = full + STAGES;        // the pair's MMAs are done with the stage
    uint64_t *acc_full = empty + STAGES;
    uint64_t *recv = acc_full + 1;          // the pieces of this CTA's chunks landed
    uint64_t *drain = recv + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int CS = static_cast<int>(cluster_ctas());
    const int S = CS / 2;
    if ((CS & 1) || !split_pair_fits<BN>(S) || kblocks < S) {   // uniform over the grid
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        return;
    }
    const uint32_t rank = cluster_rank();
    const int p = static_cast<int>(rank >> 1), h = static_cast<int>(rank & 1u);
    const int T = static_cast<int>(blockIdx.x) / CS;
    const int kb0 = p * kblocks / S, kb1 = (p + 1) * kblocks / S;
    const int nchunks = (M + 31) / 32 < BN / 32 ? (M + 31) / 32 : BN / 32;
    const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (2 * p));

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(acc_full, 1);
        mbar_init(recv, 1);
        mbar_init(drain, 1);
        *abort = 0;
        // the bytes this CTA will receive: S - 1 pieces of each chunk it owns
        uint32_t bytes = 0;
        for (int cc = p; cc < nchunks; cc += S) bytes += static_cast<uint32_t>((S - 1) * live_quads(M, cc)) * kBM * 16;
        mbar_arrive_expect_tx(recv, bytes);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, BN);
        tmem_relinquish_pair();
        tc_fence_before();
    }
    cluster_sync_all();   // every CTA's barriers and allocation exist before anything targets them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the pair's accumulators must sit at the same tensor-memory address
    if (ld_cluster_u32(cluster_smem(tmem_slot, rank ^ 1u)) != tmem) {
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        *abort = 1;
    }
    __syncthreads();

    bool ok = true;
    if (warp == 0 && lane == 0) {
        // producer: this CTA's 128 w rows and half of the x rows, counted on
        // the pair's even CTA's full barrier (which expects both CTAs' bytes)
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_y);
        const uint32_t full_even = cluster_smem(full, rank & ~1u);
        const uint32_t bytes = kTileA + C::kTileB;
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1 && !*abort; kb += KPS, ++it) {
            const int nk = kb1 - kb < KPS ? kb1 - kb : KPS;
            const int st = static_cast<int>(it % STAGES);
            if (it >= static_cast<uint32_t>(STAGES) &&
                !mbar_wait(&empty[st], ((it / STAGES) & 1) ^ 1, abort, dev_status)) break;
            uint8_t *sa = smem + st * C::kStage;
            if (h == 0) mbar_arrive_expect_tx(&full[st], 2 * bytes * static_cast<uint32_t>(nk));
            for (int q = 0; q < nk; ++q) {
                tma_load_2d_pair(sa + q * kTileA, &tm_w, full_even + st * 8, (kb + q) * kBK, (2 * T + h) * kBM);
                tma_load_2d_pair(sa + KPS * kTileA + q * C::kTileB, &tm_x, full_even + st * 8, (kb + q) * kBK,
                                 h * (BN / 2));
            }
        }
        if (*abort) {
            // copies in flight complete on the even CTA's full barriers: drain
            // those (bounded), then give any straggler 0.2 ms to land
            if (h == 0) drain_copies(full, it, STAGES);
            const unsigned long long t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 200000ull) {
            }
        }
    } else if (warp == 1 && lane == 0 && h == 0) {
        // MMA issuer (the pair's even CTA)
        constexpr uint32_t idesc = idesc_f16(2 * kBM, BN, /*bf16*/ 1, 0, 0);
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; kb += KPS, ++it) {
            const int nk = kb1 - kb < KPS ? kb1 - kb : KPS;
            const int st = static_cast<int>(it % STAGES);
            if (!mbar_wait(&full[st], (it / STAGES) & 1, abort, dev_status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + st * C::kStage);
            for (int q = 0; q < nk; ++q) {
                const uint32_t a = sa + q * kTileA, b = sa + KPS * kTileA + q * C::kTileB;
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                    umma_f16_ss_pair(tmem, sdesc(a + k * 32, 16, 1024), sdesc(b + k * 32, 16, 1024), idesc,
                                     (it > 0 || q > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit_pair(&empty[st], pair_mask);
        }
        if (ok) umma_commit_pair(acc_full, pair_mask);
    } else if (warp >= 2) {
        ok = mbar_wait_warp(acc_full, 0, abort, dev_status);
        tc_fence_after();
    }
    // every pair of the cluster is done with its stage rings (its MMAs have
    // completed: the epilogue warps arrive after the accumulator is final)
    __syncwarp();
    cluster_arrive_release();
    cluster_wait_acquire();
    tc_fence_after();

    if (warp >= 2) {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t tbase = tmem + ((quad * 32) << 16);
        // send: this CTA's piece of every chunk it does not own to the CTA of
        // the owning pair that holds the same w rows
#pragma unroll 1
        for (int cc = 0; cc < nchunks && ok && !*abort; ++cc) {
            if (cc % S == p) continue;
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + cc * 32, r);
            tmem_ld_wait();
            const uint32_t owner = static_cast<uint32_t>(2 * (cc % S) + h);
            const float *slot =
                reinterpret_cast<const float *>(smem) + static_cast<size_t>((cc / S) * S + p) * (32 * kBM);
            const uint32_t dst = peer_smem(slot, owner);
            const uint32_t bar = peer_smem(recv, owner);
            const int nq = live_quads(M, cc);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                if (q4 < nq)
                    st_async_peer_v4(dst + unit_index(q4, row) * 4, r[4 * q4], r[4 * q4 + 1], r[4 * q4 + 2],
                                     r[4 * q4 + 3], bar);
        }
        // receive: the S pieces of each owned chunk, added in k order
        if (ok) ok = mbar_wait_warp(recv, 0, abort, dev_status);
        uint8_t *obuf = out_stage + (warp - 2) * 2 * kOutBlock;
        uint32_t nst = 0;
#pragma unroll 1
        for (int cc = p; cc < nchunks && ok; cc += S) {
            const int nq = live_quads(M, cc);
            const float *base = reinterpret_cast<const float *>(smem) + static_cast<size_t>((cc / S) * S) * (32 * kBM);
            uint32_t own[32];
            tmem_ld_32x32b_x32(tbase + cc * 32, own);
            tmem_ld_wait();
            float a[32];
            for (int src = 0; src < S; ++src) {
                const float *u = base + static_cast<size_t>(src) * (32 * kBM);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    float4 v = make_float4(__uint_as_float(own[4 * q4]), __uint_as_float(own[4 * q4 + 1]),
                                           __uint_as_float(own[4 * q4 + 2]), __uint_as_float(own[4 * q4 + 3]));
                    if (src != p)
                        v = q4 < nq ? *reinterpret_cast<const float4 *>(u + unit_index(q4, row))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                    if (src == 0) {
                        a[4 * q4] = v.x; a[4 * q4 + 1] = v.y; a[4 * q4 + 2] = v.z; a[4 * q4 + 3] = v.w;
                    } else {
                        a[4 * q4] += v.x; a[4 * q4 + 1] += v.y; a[4 * q4 + 2] += v.z; a[4 * q4 + 3] += v.w;
                    }
                }
            }
            store_out_swap(&tm_y, obuf, nst, lane, 2 * T + h, quad, cc, a);
        }
        if (lane == 0) bulk_wait_read_all();   // staged output read before the CTA's shared memory goes
        tc_fence_before();                     // the tensor-memory reads, before the deallocation
    }
    __syncwarp();
    __syncthreads();
    if (*abort && h == 0 && threadIdx.x == 32) {
        // let every pair MMA issued so far finish before tensor memory goes
        umma_commit_pair(drain, static_cast<uint16_t>(1u << rank));
        mbar_wait_drain(drain, 0, 100000000ull);
    }
    cluster_sync_all();   // no CTA exits while another may still send into it, signal or read it
    if (warp == 1) { tc_fence_after(); tmem_dealloc_pair(tmem, BN); }
}

template <typename Kern>
cudaError_t set_smem(Kern k, uint32_t bytes)
{
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <int BN>
cudaError_t run_swap(const GemmPlan &p, const CUtensorMap &tx, const CUtensorMap &tw, const CUtensorMap &ty,
                     int M, int N, void *workspace, uint32_t *dev_status, cudaStream_t st)
{
    constexpr int STAGES = stages_for(BN);
    auto k = gemm_swap_kernel<BN, STAGES>;
    cudaError_t e = set_smem(k, TiledSmem<BN, STAGES>::kBytes);
    if (e != cudaSuccess) return e;
    uint32_t *flags = static_cast<uint32_t *>(workspace);
    float *part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kFlagBytes);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = TiledSmem<BN, STAGES>::kBytes;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, k, tx, tw, ty, M, N, p.sk, part, flags, dev_status);
}

cudaLaunchConfig_t pair_config(int grid, cudaStream_t st, cudaLaunchAttribute (&attr)[1])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kPairSmem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;   // the two CTAs of a pair MMA
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Units (CTA pairs, or single CTAs for the swap orientation) that can be
// resident at once, from the occupancy calculator; 0 if the query fails.
template <int BN>
int max_swap_units()
{
    constexpr int STAGES = stages_for(BN);
    auto k = gemm_swap_kernel<BN, STAGES>;
    if (set_smem(k, TiledSmem<BN, STAGES>::kBytes) != cudaSuccess) return 0;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, TiledSmem<BN, STAGES>::kBytes) !=
            cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return per_sm > 0 ? sms : 0;   // one CTA per SM
}

template <typename Kern>
cudaError_t set_smem(Kern k, uint32_t bytes);

template <int BN>
cudaLaunchConfig_t split_config(int grid, int S, cudaStream_t st, cudaLaunchAttribute (&attr)[1])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SplitCfg<BN>::kBytes;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;   // the CTAs sharing a tile's k-blocks
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int BN>
cudaError_t run_split(const GemmPlan &p, const CUtensorMap &tx, const CUtensorMap &tw, const CUtensorMap &ty,
                      int M, int K, uint32_t *dev_status, cudaStream_t st)
{
    cudaError_t e = set_smem(gemm_split_kernel<BN>, SplitCfg<BN>::kBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = split_config<BN>(p.grid, p.split, st, attr);
    return cudaLaunchKernelEx(&cfg, gemm_split_kernel<BN>, tx, tw, ty, M, K / kBK, dev_status);
}

// Clusters of S split CTAs that can be resident at once (0 if the query
// fails or the ring cannot hold the exchanged pieces).
template <int BN>
int max_split_clusters(int S)
{
    if (!split_fits<BN>(S)) return 0;
    if (set_smem(gemm_split_kernel<BN>, SplitCfg<BN>::kBytes) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = split_config<BN>(S, S, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_split_kernel<BN>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int BN>
cudaLaunchConfig_t split_pair_config(int grid, int S, cudaStream_t st, cudaLaunchAttribute (&attr)[1])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SplitPairCfg<BN>::kBytes;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;   // S CTA pairs sharing a pair tile's k-blocks
    attr[0].val.clusterDim.x = 2 * S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int BN>
cudaError_t run_split_pair(const GemmPlan &p, const CUtensorMap &tx, const CUtensorMap &tw, const CUtensorMap &ty,
                           int M, int K, uint32_t *dev_status, cudaStream_t st)
{
    cudaError_t e = set_smem(gemm_split_pair_kernel<BN>, SplitPairCfg<BN>::kBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = split_pair_config<BN>(p.grid, p.split, st, attr);
    return cudaLaunchKernelEx(&cfg, gemm_split_pair_kernel<BN>, tx, tw, ty, M, K / kBK, dev_status);
}

// Clusters of S CTA pairs that can be resident at once (0 if the query
// fails or S cannot be used).
template <int BN>
int max_split_pair_clusters(int S)
{
    if (!split_pair_fits<BN>(S)) return 0;
    if (set_smem(gemm_split_pair_kernel<BN>, SplitPairCfg<BN>::kBytes) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = split_pair_config<BN>(2 * S, S, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_split_pair_kernel<BN>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

bool split_pair_fits_bn(int bn, int S)
{
    return bn == 128 ? split_pair_fits<128>(S) : bn == 256 ? split_pair_fits<256>(S) : false;
}

bool split_fits_bn(int bn, int S)
{
    switch (bn) {
    case 32: return split_fits<32>(S);
    case 64: return split_fits<64>(S);
    case 128: return split_fits<128>(S);
    default: return split_fits<256>(S);
    }
}

int max_pair_units()
{
    if (set_smem(gemm_pair_kernel, kPairSmem) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(2, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

int query_max_units(int bn, bool swap)
{
    if (!swap) return max_pair_units();
    switch (bn) {
    case 32: return max_swap_units<32>();
    case 64: return max_swap_units<64>();
    case 128: return max_swap_units<128>();
    default: return max_swap_units<256>();
    }
}

}  // namespace

SplitCaps split_caps_estimate(int sms)
{
    SplitCaps c{};
    for (int S = 2; S <= 8; ++S) c.max_clusters[S] = sms / S;
    for (int S = 2; S <= 4; ++S) c.pair_clusters[S] = sms / (2 * S);
    return c;
}

SplitCaps split_caps_device(int bn)
{
    // per device and width; the answers never change for a process
    static std::atomic<int> cache[64][4][9];
    static std::atomic<int> pair_cache[64][4][5];
    SplitCaps c{};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return c;
    const int b = bn == 32 ? 0 : bn == 64 ? 1 : bn == 128 ? 2 : 3;
    for (int S = 2; S <= 8; ++S) {
        std::atomic<int> &slot = cache[dev][b][S];
        int v = slot.load(std::memory_order_relaxed);
        if (v == 0) {
            switch (bn) {
            case 32: v = max_split_clusters<32>(S); break;
            case 64: v = max_split_clusters<64>(S); break;
            case 128: v = max_split_clusters<128>(S); break;
            default: v = max_split_clusters<256>(S); break;
            }
            slot.store(v > 0 ? v : -1, std::memory_order_relaxed);
        }
        c.max_clusters[S] = v > 0 ? v : 0;
    }
    for (int S = 2; S <= 4; ++S) {
        std::atomic<int> &slot = pair_cache[dev][b][S];
        int v = slot.load(std::memory_order_relaxed);
        if (v == 0) {
            v = bn == 128 ? max_split_pair_clusters<128>(S) : bn == 256 ? max_split_pair_clusters<256>(S) : -1;
            slot.store(v > 0 ? v : -1, std::memory_order_relaxed);
        }
        c.pair_clusters[S] = v > 0 ? v : 0;
    }
    return c;
}

int gemm_max_units(int bn, bool swap)
{
    // per device and kernel variant; the answer never changes for a process
    static std::atomic<int> cache[64][5];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int v_idx = swap ? (bn == 32 ? 0 : bn == 64 ? 1 : bn == 128 ? 2 : 3) : 4;
    std::atomic<int> &slot = cache[dev][v_idx];
    int v = slot.load(std::memory_order_relaxed);
    if (v <= 0) {
        v = query_max_units(bn, swap);
        slot.store(v, std::memory_order_relaxed);
    }
    return v;
}

// Pair tiles: choose the number of column tiles.  Widths are multiples of
// 32 columns (each CTA's half of the pair MMA's N then covers whole 16-row
// groups of w) within [32, 256]; the cost of a candidate is the number of
// waves of tiles over the resident pairs times the widest tile plus a fixed
// per-tile overhead of kPairOverheadCols columns (the x rows every k-block
// stages whatever the width, the pipeline fill, the epilogue).  N = K =
// 6144, 76 pairs: M = 512 takes 38 column tiles of 160 or 192 columns, one
// tile per pair, where 256-column tiles would leave 28 pairs idle.
constexpr int kPairOverheadCols = 32;

PairGrid plan_pairs(int M, int N, int K, int max_pairs)
{
    PairGrid g{};
    g.tiles_m = (M + 2 * kBM - 1) / (2 * kBM);
    g.kblocks = K / kBK;
    const int n32 = N / 32;
    const int lo = (n32 + 7) / 8;   // widths <= 256
    long long best = -1;
    for (int tn = lo; tn <= n32; ++tn) {
        const long long tiles = static_cast<long long>(g.tiles_m) * tn;
        const long long waves = (tiles + max_pairs - 1) / max_pairs;
        const long long cost = waves * (32LL * ((n32 + tn - 1) / tn) + kPairOverheadCols);
        // on a tie, more (narrower) tiles: the same makespan with less work
        // on most pairs
        if (best < 0 || cost <= best) {
            best = cost;
            g.tiles_n = tn;
        }
    }
    g.q = n32 / g.tiles_n;
    g.r = n32 % g.tiles_n;
    g.pairs = g.tiles() < max_pairs ? g.tiles() : max_pairs;
    return g;
}

GemmPlan plan_gemm(int M, int N, int K, int max_units_swap, int max_units_pair, const SplitCaps &caps)
{
    GemmPlan p{};
    const int kblocks = K / kBK;
    if (M > 256) {
        p.swap = false;
        const int cap = max_units_pair < 1 ? 1 : max_units_pair > kMaxCtas / 2 ? kMaxCtas / 2 : max_units_pair;
        p.pg = plan_pairs(M, N, K, cap);
        p.bn = p.pg.width(0);
        p.grid = 2 * p.pg.pairs;
        p.workspace_bytes = 0;   // whole tiles: nothing to add across CTAs
        return p;
    }
    // Weight streaming: 128-row w tiles cut so that every SM streams, each
    // into about three pieces (min_iters = ceil(kblocks / 3); at K = 6144,
    // 48 tiles become 144 equal thirds).  Measured against a limit of five
    // pieces for narrow tiles and three for wide ones: M = 8 26.2 -> 25.2
    // us, M = 64 28.6 -> 26.6 us, M = 256 37.0 -> 36.1 us.
    p.swap = true;
    p.bn = M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    const int tiles = N / kBM;
    // Split K over clusters when every tile's cluster can be resident at
    // once: the largest S (at most K / 64) whose clusters all fit and whose
    // exchanged pieces fit a stage ring; S single CTAs per 128-row tile, or
    // (M > 64, N a multiple of 256) S CTA pairs per 256-row tile, which
    // halve the x rows each SM takes in -- preferred unless they would use
    // fewer CTAs.
    int S1 = 0, S2 = 0;
    for (int S = 8; S >= 2 && !S1; --S)
        if (S <= kblocks && split_fits_bn(p.bn, S) && caps.max_clusters[S] >= tiles) S1 = S;
    if (M > 64 && N % 256 == 0)
        for (int S = 4; S >= 2 && !S2; --S)
            if (S <= kblocks && split_pair_fits_bn(p.bn, S) && caps.pair_clusters[S] >= N / 256) S2 = S;
    if (S2 && (N / 256) * 2 * S2 >= tiles * S1) {
        p.split = S2;
        p.split_pairs = true;
        p.grid = (N / 256) * 2 * S2;
        p.workspace_bytes = 0;   // the pieces meet in shared memory
        return p;
    }
    if (S1) {
        p.split = S1;
        p.grid = tiles * S1;
        p.workspace_bytes = 0;
        return p;
    }
    p.sk.tiles_m = 1;
    const int div = 3;
    const int min_iters = (kblocks + div - 1) / div > 8 ? (kblocks + div - 1) / div : 8;
    int cap = max_units_swap;
    // Stream-K: whole-tile waves while more than two waves remain, the rest
    // cut into equal k-block ranges, one per unit.
    const long long iters = static_cast<long long>(tiles) * kblocks;
    cap = cap < kMaxCtas ? cap : kMaxCtas;
    cap = cap < 1 ? 1 : cap;
    long long u = iters / min_iters;
    u = u < 1 ? 1 : u > cap ? cap : u;
    const int units = static_cast<int>(u);
    const int waves = tiles / units;
    p.grid = units;
    p.sk.tiles = tiles;
    p.sk.kblocks = kblocks;
    p.sk.G = units;
    p.sk.dp_tiles = waves >= 2 ? (waves - 1) * units : 0;
    p.sk.sk_iters = static_cast<long long>(tiles - p.sk.dp_tiles) * kblocks;
    p.workspace_bytes = kFlagBytes + 2 * static_cast<size_t>(p.grid) * kBM * p.bn * 4;
    return p;
}

cudaError_t launch_gemm(const GemmPlan &p, const void *x, const void *w, void *y, int M, int N, int K,
                        void *workspace, uint32_t *dev_status, cudaStream_t st)
{
    const uint64_t dx[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t dw[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
    const uint64_t sk[1] = {static_cast<uint64_t>(K) * 2};
    const uint64_t dy[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t sy[1] = {static_cast<uint64_t>(N) * 2};
    CUtensorMap tx, tw, ty;
    if (p.swap) {
        // x padded to bn rows, 128-row w tiles; y written in 32 x 32 blocks
        const uint32_t bx[2] = {64, static_cast<uint32_t>(p.bn)};
        const uint32_t bw[2] = {64, static_cast<uint32_t>(kBM)};
        const uint32_t by[2] = {32, 32};
        if (!encode_bf16_tmap(&tx, x, 2, dx, sk, bx) || !encode_bf16_tmap(&tw, w, 2, dw, sk, bw) ||
            !encode_bf16_tmap_plain(&ty, y, 2, dy, sy, by))
            return cudaErrorInvalidValue;
        if (p.split >= 2 && p.split_pairs) {
            // the pair's B operand: half of the padded x rows per CTA
            const uint32_t bxh[2] = {64, static_cast<uint32_t>(p.bn / 2)};
            CUtensorMap txh;
            if (!encode_bf16_tmap(&txh, x, 2, dx, sk, bxh)) return cudaErrorInvalidValue;
            return p.bn == 128 ? run_split_pair<128>(p, txh, tw, ty, M, K, dev_status, st)
                               : run_split_pair<256>(p, txh, tw, ty, M, K, dev_status, st);
        }
        if (p.split >= 2) {
            switch (p.bn) {
            case 32: return run_split<32>(p, tx, tw, ty, M, K, dev_status, st);
            case 64: return run_split<64>(p, tx, tw, ty, M, K, dev_status, st);
            case 128: return run_split<128>(p, tx, tw, ty, M, K, dev_status, st);
            default: return run_split<256>(p, tx, tw, ty, M, K, dev_status, st);
            }
        }
        switch (p.bn) {
        case 32: return run_swap<32>(p, tx, tw, ty, M, N, workspace, dev_status, st);
        case 64: return run_swap<64>(p, tx, tw, ty, M, N, workspace, dev_status, st);
        case 128: return run_swap<128>(p, tx, tw, ty, M, N, workspace, dev_status, st);
        default: return run_swap<256>(p, tx, tw, ty, M, N, workspace, dev_status, st);
        }
    }
    // pairs: 128 x rows per CTA; half of a tile's w rows per CTA (16q rows
    // for the narrow tiles, 16(q + 1) for the wide ones); y in 32 x 32 blocks
    CUtensorMap tw2;
    const uint32_t bx[2] = {64, static_cast<uint32_t>(kBM)};
    const uint32_t bw_n[2] = {64, static_cast<uint32_t>(16 * p.pg.q)};
    const uint32_t bw_w[2] = {64, static_cast<uint32_t>(16 * (p.pg.q + 1))};
    const uint32_t by[2] = {32, 32};
    if (!encode_bf16_tmap(&tx, x, 2, dx, sk, bx) || !encode_bf16_tmap(&tw, w, 2, dw, sk, bw_n) ||
        !encode_bf16_tmap(&tw2, w, 2, dw, sk, bw_w) || !encode_bf16_tmap_plain(&ty, y, 2, dy, sy, by))
        return cudaErrorInvalidValue;
    cudaError_t e = set_smem(gemm_pair_kernel, kPairSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config(p.grid, st, attr);
    (void)workspace;
    return cudaLaunchKernelEx(&cfg, gemm_pair_kernel, tx, tw, tw2, ty, M, p.pg, dev_status);
}

}  // namespace spec
