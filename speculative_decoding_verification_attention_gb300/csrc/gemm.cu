// Verify GEMM y[M][N] = x[M][K] . w[N][K]^T, bf16 in, fp32 accumulate in
// tensor memory, bf16 out.
//
// "Draft length and performance of linear layers" (co-design blog): with
// speculation every target linear layer runs at GEMM-M = M(1+D); the
// representative expert GEMM is N = K = 6144.  Small M streams the weights
// (HBM-bound); large M is a dense contraction on the tensor cores.
//
// One warp-specialised kernel (warp 0: TMA producer, warp 1: MMA issuer,
// warps 2-5: epilogue), operands staged by TMA with the 128-byte swizzle,
// tcgen05.mma kind::f16 (M = 128) accumulating in TMEM, two accumulators so
// one piece's epilogue overlaps the next piece's main loop.  Two operand
// orientations:
//  * tiled (M > 256): A = x rows, B = w rows.  CTAs run in pairs (clusters
//    of 2) on 256 x BN tiles, 128 rows each; each CTA loads half of the w
//    tile and multicasts it to both, halving the L2 -> SM traffic of w.
//  * swap (M <= 256): A = w rows (128 per tile), B = the M rows of x padded
//    to MPAD, so the MMA is not mostly padding; the output is written
//    transposed.
// Both split the k-block iterations of all tiles evenly over the CTAs
// (stream-K, see gemm_schedule.h).  Every piece of a tile cut between CTAs
// leaves its fp32 partial in the workspace and counts itself in; the last
// piece to arrive adds them all in k order (so results are deterministic)
// and writes the tile.  No CTA waits for another.  Output blocks of 32 x 32
// are staged in shared memory by each epilogue warp and written by TMA
// tensor stores (coalesced, asynchronous; rows past M are clipped).
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "gemm.h"
#include "gemm_schedule.h"

namespace cg = cooperative_groups;

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
// add: swap tiles have a column per row of x, so only the quads that hold
// rows m < M; tiled ones all 8.
template <bool SWAP>
__device__ __forceinline__ int live_quads(int M, int cc)
{
    if (!SWAP) return 8;
    const int q = (M - cc * 32 + 3) / 4;
    return q < 8 ? q : 8;
}

// Write 32 columns (chunk cc) of this warp's 32 tile rows as one bf16 block:
// staged in the warp's next buffer, then one TMA store by lane 0.  Tiled:
// tile row = y row, block at (x = nt BN + 32 cc, y = 128 mt + 32 quad).
// Swap: tile row = w row n = y column, tile column = x row m, so the block
// is transposed while staged, at (x = 128 t + 32 quad, y = 32 cc).
template <bool SWAP>
__device__ __forceinline__ void store_out(const CUtensorMap *tm_y, uint8_t *obuf, uint32_t &nst, int lane,
                                          int t, int mt, int nt, int BN, int quad, int cc, const float (&a)[32])
{
    uint8_t *buf = obuf + (nst & 1u) * kOutBlock;
    if (lane == 0) bulk_wait_read_1();   // the store issued from this buffer two blocks ago has read it
    __syncwarp();
    if (SWAP) {
        __nv_bfloat16 *b = reinterpret_cast<__nv_bfloat16 *>(buf);
#pragma unroll
        for (int j = 0; j < 32; ++j) b[j * 32 + lane] = __float2bfloat16_rn(a[j]);
    } else {
        uint4 *b = reinterpret_cast<uint4 *>(buf + lane * 64);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint4 o;
            o.x = pack_bf16x2(a[8 * v + 0], a[8 * v + 1]);
            o.y = pack_bf16x2(a[8 * v + 2], a[8 * v + 3]);
            o.z = pack_bf16x2(a[8 * v + 4], a[8 * v + 5]);
            o.w = pack_bf16x2(a[8 * v + 6], a[8 * v + 7]);
            b[v] = o;
        }
    }
    fence_proxy_async_smem();   // the staged block is visible to the TMA unit
    __syncwarp();
    if (lane == 0) {
        if (SWAP) tma_store_2d(tm_y, buf, t * kBM + quad * 32, cc * 32);
        else tma_store_2d(tm_y, buf, nt * BN + cc * 32, mt * kBM + quad * 32);
        bulk_commit();
    }
    ++nst;
}

template <int BN, int STAGES>
struct TiledSmem {
    static constexpr uint32_t kTileB = BN * kBK * 2;
    static constexpr uint32_t kStage = kTileA + kTileB;
    static constexpr uint32_t kBytes = STAGES * kStage + kOutStaging + 1024 /*align*/ + 256 /*barriers*/;
    static_assert(STAGES * kStage >= kBM * BN * 4, "a partial tile must fit in the stage ring");
};

constexpr int stages_for(int bn) { return bn >= 256 ? 4 : bn >= 128 ? 6 : 8; }

// SWAP = false: 256 x BN tiles on CTA pairs, A = x, B = w (shared half by
// half through multicast).  SWAP = true: 128-row w tiles, A = w, B = x
// padded to BN rows, single CTAs.
template <int BN, int STAGES, bool SWAP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
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
    // tiled: CTA within its pair, and the pair index (the unit of the split)
    const int rank = SWAP ? 0 : static_cast<int>(blockIdx.x & 1);
    const int c = SWAP ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x >> 1);
    constexpr int kUnit = SWAP ? 1 : 2;   // CTAs per unit of the split
    constexpr uint16_t kPair = 0x3;
    if (cluster_ctas() != static_cast<uint32_t>(kUnit)) {   // uniform over the grid
        if (threadIdx.x == 0) report(dev_status, SPEC_DEV_ERR_LAUNCH);
        return;
    }

    if (threadIdx.x == 0) {
        // tiled: a stage is free once the MMAs of both CTAs of the pair read it
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kUnit); }
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
    if constexpr (SWAP) __syncthreads();
    else cg::this_cluster().sync();   // the peer's barriers exist before anything targets them
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
            const int mt = 2 * (s.t % grid.tiles_m) + rank, nt = s.t / grid.tiles_m;
            for (int kb = s.kb0; kb < s.kb1; ++kb, ++it) {
                const int st = it % STAGES;
                if (it >= STAGES && !mbar_wait(&empty[st], ((it / STAGES) & 1) ^ 1, abort, dev_status)) break;
                uint8_t *sa = smem + st * L::kStage;
                mbar_arrive_expect_tx(&full[st], L::kStage);
                if constexpr (SWAP) {
                    tma_load_2d(sa, &tm_w, &full[st], kb * kBK, s.t * kBM);
                    tma_load_2d(sa + kTileA, &tm_x, &full[st], kb * kBK, 0);
                } else {
                    // this CTA's rows of x, plus its half of the shared w
                    // tile, which lands in both CTAs of the pair
                    tma_load_2d(sa, &tm_x, &full[st], kb * kBK, mt * kBM);
                    tma_load_2d_multicast(sa + kTileA + rank * (L::kTileB / 2), &tm_w, &full[st],
                                          kb * kBK, nt * BN + rank * (BN / 2), kPair);
                }
            }
        }
        if (*abort) {
            drain_copies(full, it, STAGES);
        } else if (!SWAP) {
            // the peer's MMAs signal this CTA's empty barriers: wait for their
            // last arrivals before this CTA may exit
            for (uint32_t i = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0; i < it; ++i)
                if (!mbar_wait(&empty[i % STAGES], (i / STAGES) & 1, abort, dev_status)) break;
        }
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
                if constexpr (SWAP) umma_commit(&empty[st]);
                else umma_commit_multicast(&empty[st], kPair);
            }
            if (!ok) break;
            umma_commit(&acc_full[ab]);
            ++lt;
        }
    } else if (warp >= 2) {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        // swap: only the 32-column chunks that hold rows of x are needed
        const int nchunks = SWAP ? (M + 31) / 32 < BN / 32 ? (M + 31) / 32 : BN / 32 : BN / 32;
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
            const int mt = 2 * (s.t % grid.tiles_m) + rank, nt = s.t / grid.tiles_m;
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
                    store_out<SWAP>(&tm_y, obuf, nst, lane, s.t, mt, nt, BN, quad, cc, a);
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
                    const int nq = live_quads<SWAP>(M, cc);
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
                    const bool ring_ok = !wk.has_more() && !(SWAP && nchunks == 1);
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
                                    for (int cc = c0; cc < c1; ++cc) bytes += live_quads<SWAP>(M, cc) * kBM * 16;
                                    mbar_arrive_expect_tx(red_full, bytes * others);
                                    int k = 0;
                                    for (int v = f; v <= l; ++v) {
                                        if (v == me) continue;
                                        const float *src = part + static_cast<size_t>(
                                            piece_slot(v, rank, v != f || other_first(grid, f, s.t), kUnit)) * kBM * BN;
                                        // a unit's quads are its outer index: the live ones are its first bytes
                                        for (int cc = c0; cc < c1; ++cc)
                                            bulk_load(smem + ((cc - c0) * others + k) * 32 * kBM * 4,
                                                      src + cc * 32 * kBM, live_quads<SWAP>(M, cc) * kBM * 16, red_full);
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
                                    const int nq = live_quads<SWAP>(M, cc);
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
                            store_out<SWAP>(&tm_y, obuf, nst, lane, s.t, mt, nt, BN, quad, cc, a);
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
    if constexpr (SWAP) __syncthreads();
    else cg::this_cluster().sync();   // neither CTA of a pair exits while the other may signal it
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 2 * BN); }
}

template <typename Kern>
cudaError_t set_smem(Kern k, uint32_t bytes)
{
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <int BN, bool SWAP>
cudaLaunchConfig_t kernel_config(int grid, cudaStream_t st, cudaLaunchAttribute (&attr)[2])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = TiledSmem<BN, stages_for(BN)>::kBytes;
    cfg.stream = st;
    int n = 0;
    if (!SWAP) {
        attr[n].id = cudaLaunchAttributeClusterDimension;   // CTA pairs share the w tile
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cfg;
}

template <int BN, bool SWAP>
cudaError_t run(const GemmPlan &p, const CUtensorMap &tx, const CUtensorMap &tw, const CUtensorMap &ty,
                int M, int N, void *workspace, uint32_t *dev_status, cudaStream_t st)
{
    constexpr int STAGES = stages_for(BN);
    auto k = gemm_kernel<BN, STAGES, SWAP>;
    cudaError_t e = set_smem(k, TiledSmem<BN, STAGES>::kBytes);
    if (e != cudaSuccess) return e;
    uint32_t *flags = static_cast<uint32_t *>(workspace);
    float *part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kFlagBytes);
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = kernel_config<BN, SWAP>(p.grid, st, attr);
    return cudaLaunchKernelEx(&cfg, k, tx, tw, ty, M, N, p.sk, part, flags, dev_status);
}

// Units (CTA pairs, or single CTAs for the swap orientation) that can be
// resident at once, from the occupancy calculator; 0 if the query fails.
template <int BN, bool SWAP>
int max_units_for()
{
    constexpr int STAGES = stages_for(BN);
    auto k = gemm_kernel<BN, STAGES, SWAP>;
    if (set_smem(k, TiledSmem<BN, STAGES>::kBytes) != cudaSuccess) return 0;
    int n = 0;
    if (SWAP) {
        int dev = 0, sms = 0, per_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads,
                                                          TiledSmem<BN, STAGES>::kBytes) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        n = per_sm > 0 ? sms : 0;   // one CTA per SM
    } else {
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = kernel_config<BN, SWAP>(2, nullptr, attr);
        cfg.numAttrs = 1;   // the occupancy query takes the cluster shape only
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
    }
    return n;
}

int query_max_units(int bn, bool swap)
{
    if (swap) {
        switch (bn) {
        case 32: return max_units_for<32, true>();
        case 64: return max_units_for<64, true>();
        case 128: return max_units_for<128, true>();
        default: return max_units_for<256, true>();
        }
    }
    return bn == 256 ? max_units_for<256, false>() : max_units_for<128, false>();
}

}  // namespace

int gemm_max_units(int bn, bool swap)
{
    // per device and kernel variant; the answer never changes for a process
    static std::atomic<int> cache[64][6];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int v_idx = swap ? (bn == 32 ? 0 : bn == 64 ? 1 : bn == 128 ? 2 : 3) : (bn == 256 ? 5 : 4);
    std::atomic<int> &slot = cache[dev][v_idx];
    int v = slot.load(std::memory_order_relaxed);
    if (v <= 0) {
        v = query_max_units(bn, swap);
        slot.store(v, std::memory_order_relaxed);
    }
    return v;
}

GemmPlan plan_gemm(int M, int N, int K, int max_units_swap, int max_units_tiled)
{
    GemmPlan p{};
    const int kblocks = K / kBK;
    int tiles, min_iters, cap;
    if (M <= 256) {
        // Weight streaming: 128-row w tiles cut so that every SM streams,
        // each into about three pieces (min_iters = ceil(kblocks / 3); at
        // K = 6144, 48 tiles become 144 equal thirds).  Measured against a
        // limit of five pieces for narrow tiles and three for wide ones:
        // M = 8 26.2 -> 25.2 us, M = 64 28.6 -> 26.6 us, M = 256 37.0 ->
        // 36.1 us.
        p.swap = true;
        p.bn = M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
        tiles = N / kBM;
        p.sk.tiles_m = 1;
        const int div = 3;
        min_iters = (kblocks + div - 1) / div > 8 ? (kblocks + div - 1) / div : 8;
        cap = max_units_swap;
    } else {
        // 256 x BN tiles on CTA pairs; a tile is cut into at most three
        // pieces (min_iters = ceil(kblocks / 2)), or not at all (below).
        p.swap = false;
        p.bn = N % 256 == 0 ? 256 : 128;
        p.sk.tiles_m = ((M + kBM - 1) / kBM + 1) / 2;
        tiles = p.sk.tiles_m * (N / p.bn);
        min_iters = (kblocks + 1) / 2 > 16 ? (kblocks + 1) / 2 : 16;
        cap = max_units_tiled;
    }
    // Stream-K: whole-tile waves while more than two waves remain, the rest
    // cut into equal k-block ranges, one per unit.
    const long long iters = static_cast<long long>(tiles) * kblocks;
    const int unit_ctas = p.swap ? 1 : 2;
    cap = cap < kMaxCtas / unit_ctas ? cap : kMaxCtas / unit_ctas;
    cap = cap < 1 ? 1 : cap;
    long long u = iters / min_iters;
    u = u < 1 ? 1 : u > cap ? cap : u;
    // Tiled orientation with at least half a wave of tiles but no more than
    // one: one whole tile per CTA pair.  Cut tiles would keep every pair
    // busy, but adding their pieces (fp32 partials through L2, at the same
    // per-SM L2 rate that feeds the MMAs) costs more than the idle pairs:
    // N = K = 6144, M = 512: 50.8 -> 45.1 us, M = 768: 55.1 -> 45.1 us.
    if (!p.swap && tiles <= cap && 2 * tiles >= cap) u = tiles;
    const int units = static_cast<int>(u);
    const int waves = tiles / units;
    p.grid = unit_ctas * units;
    p.sk.tiles = tiles;
    p.sk.kblocks = kblocks;
    p.sk.G = units;
    p.sk.dp_tiles = waves >= 2 ? (waves - 1) * units : 0;
    p.sk.sk_iters = static_cast<long long>(tiles - p.sk.dp_tiles) * kblocks;
    p.workspace_bytes = kFlagBytes + 2 * static_cast<size_t>(p.grid) * kBM * p.bn * 4;
    return p;
}

cudaError_t launch_gemm(const GemmPlan &p, const CUtensorMap &t_x, const CUtensorMap &t_w,
                        const CUtensorMap &t_y, void *y, int M, int N, void *workspace,
                        uint32_t *dev_status, cudaStream_t st)
{
    (void)y;   // written through t_y
    if (p.swap) {
        switch (p.bn) {
        case 32: return run<32, true>(p, t_x, t_w, t_y, M, N, workspace, dev_status, st);
        case 64: return run<64, true>(p, t_x, t_w, t_y, M, N, workspace, dev_status, st);
        case 128: return run<128, true>(p, t_x, t_w, t_y, M, N, workspace, dev_status, st);
        default: return run<256, true>(p, t_x, t_w, t_y, M, N, workspace, dev_status, st);
        }
    }
    if (p.bn == 256) return run<256, false>(p, t_x, t_w, t_y, M, N, workspace, dev_status, st);
    return run<128, false>(p, t_x, t_w, t_y, M, N, workspace, dev_status, st);
}

}  // namespace spec
