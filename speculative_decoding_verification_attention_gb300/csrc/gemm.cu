// Verify GEMM y[M][N] = x[M][K] . w[N][K]^T, bf16 in, fp32 accumulate in
// tensor memory, bf16 out.
//
// "Draft length and performance of linear layers" (co-design blog): with
// speculation every target linear layer runs at GEMM-M = M(1+D); the
// representative expert GEMM is N = K = 6144.  Small M streams the weights
// (HBM-bound); large M is a dense contraction on the tensor cores.
//
// Two kernels, both warp-specialised (warp 0: TMA producer, warp 1: MMA
// issuer, warps 2-5: epilogue), operands staged by TMA with the 128-byte
// swizzle, tcgen05.mma kind::f16 (M = 128) accumulating in TMEM:
//  * gemm_tiled: persistent over 128 x BN output tiles, two TMEM
//    accumulators so one tile's epilogue overlaps the next tile's
//    main loop.  A = x, B = w.
//  * gemm_swap: for small M the weight rows take the MMA M side (A = w,
//    128 rows per tile) and the M rows of x the N side (B = x, padded to
//    MPAD).  K is split across a thread-block cluster; the partial sums are
//    reduced in fixed order through distributed shared memory.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "gemm.h"

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

// ------------------------------------------------------------------ tiled
template <int BN, int STAGES>
struct TiledSmem {
    static constexpr uint32_t kTileB = BN * kBK * 2;
    static constexpr uint32_t kStage = kTileA + kTileB;
    static constexpr uint32_t kBytes = STAGES * kStage + 1024 /*align*/ + 256 /*barriers*/;
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tiled(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
               __nv_bfloat16 *__restrict__ y, int M, int N, int K, uint32_t *dev_status)
{
    using L = TiledSmem<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * L::kStage);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_m = (M + kBM - 1) / kBM, tiles_n = N / BN;
    const int tiles = tiles_m * tiles_n;
    const int kblocks = K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], 4); }
        mbar_init(drain, 1);
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
        uint32_t it = 0;
        for (int t = blockIdx.x; t < tiles && !*abort; t += gridDim.x) {
            const int mt = t % tiles_m, nt = t / tiles_m;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                if (it >= STAGES && !mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, abort, dev_status)) break;
                uint8_t *sa = smem + s * L::kStage;
                mbar_arrive_expect_tx(&full[s], L::kStage);
                tma_load_2d(sa, &tm_x, &full[s], kb * kBK, mt * kBM);
                tma_load_2d(sa + kTileA, &tm_w, &full[s], kb * kBK, nt * BN);
            }
        }
        if (*abort) drain_copies(full, it, STAGES);
    } else if (warp == 1 && lane == 0) {
        uint32_t it = 0, lt = 0;
        for (int t = blockIdx.x; t < tiles && !*abort; t += gridDim.x, ++lt) {
            const uint32_t ab = lt & 1;
            if (lt >= 2 && !mbar_wait(&acc_empty[ab], ((lt >> 1) & 1) ^ 1, abort, dev_status)) break;
            tc_fence_after();
            const uint32_t d = tmem + ab * BN;
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                if (!mbar_wait(&full[s], (it / STAGES) & 1, abort, dev_status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * L::kStage);
                mma_kblock<BN>(d, sa, sa + kTileA, kb > 0);
                umma_commit(&empty[s]);
            }
            if (!ok) break;
            umma_commit(&acc_full[ab]);
        }
    } else if (warp >= 2) {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        uint32_t lt = 0;
        for (int t = blockIdx.x; t < tiles && !*abort; t += gridDim.x, ++lt) {
            const uint32_t ab = lt & 1;
            if (!mbar_wait_warp(&acc_full[ab], (lt >> 1) & 1, abort, dev_status)) break;
            tc_fence_after();
            const int mt = t % tiles_m, nt = t / tiles_m;
            const int m = mt * kBM + row;
            __nv_bfloat16 *yrow = y + static_cast<int64_t>(m) * N + nt * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + ((quad * 32) << 16) + ab * BN + c * 32, r);
                tmem_ld_wait();
                if (m < M) {
                    uint4 *dst = reinterpret_cast<uint4 *>(yrow + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                        o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                        o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                        o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                        dst[v] = o;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
        }
    }
    __syncwarp();
    __syncthreads();
    if (*abort && threadIdx.x == 32) drain_mmas(drain);
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 2 * BN); }
}

// ------------------------------------------------------------------- swap
template <int MPAD, int STAGES>
struct SwapSmem {
    static constexpr uint32_t kTileB = MPAD * kBK * 2;
    static constexpr uint32_t kStage = kTileA + kTileB;
    static constexpr uint32_t kPipe = STAGES * kStage;
    static constexpr uint32_t kRed = kBM * MPAD * 4;    // fp32 partial of one CTA
    static constexpr uint32_t kMain = kPipe > kRed ? kPipe : kRed;
    static constexpr uint32_t kBytes = kMain + 1024 + 256;
};

template <int MPAD, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_swap(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
              __nv_bfloat16 *__restrict__ y, int M, int N, int K, int splits, uint32_t *dev_status)
{
    using L = SwapSmem<MPAD, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kMain);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *drain = acc_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *red = reinterpret_cast<float *>(smem);   // reused after the main loop

    static_assert(MPAD >= 32 && MPAD % 32 == 0, "epilogue reads 32 columns at a time");
    constexpr int kTmemCols = MPAD;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = blockIdx.x % splits;
    const int nt = blockIdx.x / splits;
    const int kblocks = K / kBK;
    const int per = (kblocks + splits - 1) / splits;
    const int kb0 = min(kblocks, rank * per), kb1 = min(kblocks, kb0 + per);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(&acc_full[0], 1);
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_x);
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = it % STAGES;
            if (it >= STAGES && !mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, abort, dev_status)) break;
            uint8_t *sa = smem + s * L::kStage;
            mbar_arrive_expect_tx(&full[s], L::kStage);
            tma_load_2d(sa, &tm_w, &full[s], kb * kBK, nt * kBM);
            tma_load_2d(sa + kTileA, &tm_x, &full[s], kb * kBK, 0);
        }
        if (*abort) drain_copies(full, it, STAGES);
    } else if (warp == 1 && lane == 0) {
        bool ok = true;
        for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
            const int s = it % STAGES;
            if (!mbar_wait(&full[s], (it / STAGES) & 1, abort, dev_status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * L::kStage);
            mma_kblock<MPAD>(tmem, sa, sa + kTileA, it > 0);
            umma_commit(&empty[s]);
        }
        // completes once every MMA above has finished (also with none issued)
        if (ok) umma_commit(&acc_full[0]);
    }

    __syncwarp();   // reconverge the producer / MMA warps before cluster barriers

    // Epilogue warps: fetch this CTA's partial (rows = weight rows n, columns
    // = x rows m); split 0 reduces the others' partials in rank order.
    const bool has_k = kb1 > kb0;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;                 // weight row within the tile
    const bool epi = warp >= 2;
    bool ok = true;
    if (epi) {
        ok = mbar_wait_warp(&acc_full[0], 0, abort, dev_status);
        tc_fence_after();
    }
    if (splits > 1) {
        if (epi && rank != 0 && ok) {
            for (int c = 0; c < MPAD / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + ((quad * 32) << 16) + c * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    red[(c * 32 + j) * kBM + row] = has_k ? __uint_as_float(r[j]) : 0.0f;
            }
        }
        cg::this_cluster().sync();
    }
    if (epi && rank == 0 && ok) {
        const int n = nt * kBM + row;
        for (int c = 0; c < MPAD / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tmem + ((quad * 32) << 16) + c * 32, r);
            tmem_ld_wait();
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = has_k ? __uint_as_float(r[j]) : 0.0f;
            if (splits > 1) {
                cg::cluster_group cluster = cg::this_cluster();
                for (int s = 1; s < splits; ++s) {
                    const float *rr = cluster.map_shared_rank(red, s);
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[j] += rr[(c * 32 + j) * kBM + row];
                }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int m = c * 32 + j;
                if (m < M) y[static_cast<int64_t>(m) * N + n] = __float2bfloat16_rn(acc[j]);
            }
        }
    }
    if (splits > 1) cg::this_cluster().sync();
    __syncthreads();
    if (*abort && threadIdx.x == 32) drain_mmas(drain);
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, kTmemCols); }
}

template <typename Kern>
cudaError_t set_smem(Kern k, uint32_t bytes)
{
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <int MPAD>
cudaError_t run_swap(const CUtensorMap &tw, const CUtensorMap &tx, __nv_bfloat16 *y, int M, int N,
                     int K, int splits, uint32_t *dev_status, cudaStream_t st)
{
    constexpr int STAGES = MPAD >= 256 ? 4 : 6;
    using L = SwapSmem<MPAD, STAGES>;
    auto k = gemm_swap<MPAD, STAGES>;
    cudaError_t e = set_smem(k, L::kBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N / kBM) * splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, tw, tx, y, M, N, K, splits, dev_status);
}

template <int BN>
cudaError_t run_tiled(const CUtensorMap &tx, const CUtensorMap &tw, __nv_bfloat16 *y, int M, int N,
                      int K, int num_sms, uint32_t *dev_status, cudaStream_t st)
{
    constexpr int STAGES = BN >= 256 ? 4 : 6;
    using L = TiledSmem<BN, STAGES>;
    auto k = gemm_tiled<BN, STAGES>;
    cudaError_t e = set_smem(k, L::kBytes);
    if (e != cudaSuccess) return e;
    const int tiles = ((M + kBM - 1) / kBM) * (N / BN);
    const int grid = tiles < num_sms ? tiles : num_sms;
    k<<<grid, kThreads, L::kBytes, st>>>(tx, tw, y, M, N, K, dev_status);
    return cudaGetLastError();
}

}  // namespace

GemmPlan plan_gemm(int M, int N, int K, int num_sms)
{
    GemmPlan p{};
    (void)K;
    if (M <= 256) {
        p.swap = true;
        p.mpad = M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
        const int tiles = N / kBM;
        int s = num_sms / (tiles > 0 ? tiles : 1);
        s = s < 1 ? 1 : s > 4 ? 4 : s;
        const int kblocks = K / kBK;
        while (s > 1 && kblocks < s * 2) --s;
        p.splits = s;
        p.bn = 0;
    } else {
        p.swap = false;
        p.splits = 1;
        // pick the tile width that wastes the least of the last wave
        const int tiles_m = (M + kBM - 1) / kBM;
        double best = 1e30;
        for (int bn : {256, 128}) {
            if (N % bn) continue;
            const int tiles = tiles_m * (N / bn);
            const int waves = (tiles + num_sms - 1) / num_sms;
            const double cost = static_cast<double>(waves) * bn * (bn == 256 ? 0.92 : 1.0);
            if (cost < best) { best = cost; p.bn = bn; }
        }
    }
    return p;
}

cudaError_t launch_gemm(const GemmPlan &p, const CUtensorMap &t_x, const CUtensorMap &t_w,
                        void *y, int M, int N, int K, int num_sms, uint32_t *dev_status,
                        cudaStream_t st)
{
    __nv_bfloat16 *yy = static_cast<__nv_bfloat16 *>(y);
    if (p.swap) {
        switch (p.mpad) {
        case 32: return run_swap<32>(t_w, t_x, yy, M, N, K, p.splits, dev_status, st);
        case 64: return run_swap<64>(t_w, t_x, yy, M, N, K, p.splits, dev_status, st);
        case 128: return run_swap<128>(t_w, t_x, yy, M, N, K, p.splits, dev_status, st);
        default: return run_swap<256>(t_w, t_x, yy, M, N, K, p.splits, dev_status, st);
        }
    }
    if (p.bn == 256) return run_tiled<256>(t_x, t_w, yy, M, N, K, num_sms, dev_status, st);
    return run_tiled<128>(t_x, t_w, yy, M, N, K, num_sms, dev_status, st);
}

}  // namespace spec
