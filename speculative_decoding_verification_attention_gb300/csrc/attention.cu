// Verify attention over a paged bf16 KV cache.
//
// "Draft length and attention performance" (co-design blog): the D draft
// tokens reuse the KV cache of the sequence, so the G query heads of a KV
// head and the 1+D positions form one GEMM with M = G(1+D) against a single
// K/V stream; decode intensity ~2G becomes ~2G(1+D).  Row r = i*G + g of KV
// head h is query head h*G + g at position i and sees keys
// j < kv_len - D + i.
//
// Kernel structure (one CTA per SM, 8 warps):
//   warp 0      TMA producer: K and V tiles of 128 keys, page by page, into a
//               ring of shared-memory stages (128-byte swizzle).
//   warp 1      tcgen05 issuer of S = Q K^T (bf16, M = 128 rows x N = 128
//               keys, fp32 in TMEM).
//   warp 2      loads the 128 query rows of each segment into shared memory
//               and zeroes the V rows of keys past the end of a sequence.
//   warp 3      tcgen05 issuer of O += P V (P read from TMEM, fp32
//               accumulator in TMEM), as soon as a stream's P is ready.
//   warps 4-11  softmax, as two streams that take alternate key tiles (each
//               with its own S buffers and O accumulator in TMEM): one thread
//               per query row reads its S row from TMEM, masks, keeps an
//               online max / sum with lazy rescaling of O (only when the max
//               grows by more than 2^8), and writes P back into its S buffer
//               as a bf16 pair hi + lo; at the end of a segment the two
//               streams are merged and the normalised output or a partial
//               result is written.
// The KV stream of all (b, h) units is split evenly across CTA groups (see
// attn_schedule.h); units cut by a group boundary are merged by
// attention_combine.  G(1+D) > 128 uses several 128-row m-tiles, each its
// own CTA of the same group, so the same K/V tiles are read concurrently
// and served from L2.
//
// P is split as P = hi + lo with hi = P truncated to bf16 and
// lo = bf16(P - hi) (about 16 significant bits), and O += hi V + lo V takes two bf16 MMAs that read
// the A operand straight from tensor memory.  Rounding P to a single bf16
// would cost about 2e-3 relative error in O; the pair keeps it near 1e-5
// and leaves V in bf16 as stored.
#include <cuda_bf16.h>

#include "attention.h"
#include "attn_schedule.h"
#include "common.cuh"

namespace spec {
namespace {

constexpr int kBM = 128;
constexpr int kBN = kKeyTile;
constexpr int kThreads = 384;                 // 12 warps
constexpr int kCombineThreads = 512;          // 4 threads per row, a quarter of its columns each
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int HD>
struct AttnSmem {
    static constexpr int kSub = HD / 64;                   // 64-column chunks
    static constexpr uint32_t kQ = kBM * HD * 2;
    static constexpr uint32_t kSubBytes = kBN * 128;       // one 64-column chunk of a K/V tile
    static constexpr uint32_t kKV = kSub * kSubBytes;      // one K or V tile
    static constexpr int kStages = HD == 128 ? 3 : 6;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kQ;
    static constexpr uint32_t kOffV = kOffK + kStages * kKV;
    static constexpr uint32_t kOffML = kOffV + kStages * kKV;   // float2 per row: stream merge
    static constexpr uint32_t kOffBar = kOffML + kBM * 8;
    static constexpr uint32_t kBytes = kOffBar + 512 + 1024;
};

struct PlanShared {
    int64_t total, gbegin, gend, ub0;
    int b0, h0, groups_eff, found;
    int64_t warp_tot[(kThreads > kCombineThreads ? kThreads : kCombineThreads) / 32];
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int64_t warp_incl_scan64(int64_t x, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Block-wide inclusive scan of one int64 per thread (all threads call).
__device__ int64_t block_incl_scan64(int64_t x, PlanShared *ps, int64_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t incl = warp_incl_scan64(x, lane);
    if (lane == 31) ps->warp_tot[warp] = incl;
    __syncthreads();
    int64_t before = 0, all = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
        if (w < warp) before += ps->warp_tot[w];
        all += ps->warp_tot[w];
    }
    __syncthreads();
    *total = all;
    return incl + before;
}

// Total tile count, this group's range and the unit holding its first tile.
__device__ void plan_group(const AttnArgs &a, int g, PlanShared *ps)
{
    int64_t local = 0;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        const int nk = seq_tiles(a.kv_len[b], a.D, a.max_len);
        if (nk == 0 && blockIdx.x == 0) report(a.dev_status, SPEC_DEV_ERR_KV_LEN);
        local += static_cast<int64_t>(a.Hkv) * nk;
    }
    int64_t total;
    block_incl_scan64(local, ps, &total);
    const int ge = effective_groups(total, a.groups);
    const int64_t gb = g < ge ? group_begin(total, ge, g) : total;
    const int64_t gn = g < ge ? group_begin(total, ge, g + 1) : total;
    if (threadIdx.x == 0) {
        ps->total = total; ps->groups_eff = ge; ps->gbegin = gb; ps->gend = gn;
        ps->found = 0; ps->b0 = a.B; ps->h0 = 0; ps->ub0 = total;
    }
    __syncthreads();
    if (gb >= gn) return;
    int64_t base = 0;
    for (int c0 = 0; c0 < a.B; c0 += blockDim.x) {
        const int b = c0 + threadIdx.x;
        const int nk = b < a.B ? seq_tiles(a.kv_len[b], a.D, a.max_len) : 0;
        const int64_t span = static_cast<int64_t>(a.Hkv) * nk;
        int64_t chunk_total;
        const int64_t incl = block_incl_scan64(span, ps, &chunk_total);
        const int64_t lo = base + incl - span;
        if (span > 0 && lo <= gb && gb < base + incl) {
            const int h = static_cast<int>((gb - lo) / nk);
            ps->b0 = b; ps->h0 = h; ps->ub0 = lo + static_cast<int64_t>(h) * nk; ps->found = 1;
        }
        __syncthreads();
        if (ps->found) break;
        base += chunk_total;
    }
}

// TREE: rows see the prefix plus their root-to-node path (a.tree_mask);
// otherwise the chain mask, compiled without the tree's per-key bit tests.
template <int HD, bool TREE>
__global__ void __launch_bounds__(kThreads, 1)
    verify_attention_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const AttnArgs a)
{
    using L = AttnSmem<HD>;
    constexpr int S = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    __shared__ PlanShared ps;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + L::kOffQ;
    uint8_t *sK = smem + L::kOffK;
    uint8_t *sV = smem + L::kOffV;
    float2 *sML = reinterpret_cast<float2 *>(smem + L::kOffML);
    uint64_t *kv_full = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *kv_empty = kv_full + S;
    uint64_t *v_ready = kv_empty + S;
    uint64_t *s_full = v_ready + S;       // [stream]: S of the stream's current tile is in TMEM
    uint64_t *s_empty = s_full + 2;       // [stream]: its P.V has run, the S/P columns are free
    uint64_t *p_full = s_empty + 2;       // [stream]: P written
    uint64_t *p_empty = p_full + 2;       // [stream]: P.V done (O updated)
    uint64_t *q_full = p_empty + 2;
    uint64_t *q_empty = q_full + 1;
    uint64_t *ml_ready = q_empty + 1;     // stream 1 published (m, l) and its O is final
    uint64_t *o_taken = ml_ready + 1;     // stream 0 has read stream 1's O
    uint64_t *drain = o_taken + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x / a.nt, mt = blockIdx.x % a.nt;
    // TMEM: O of stream s at column s*HD; the S/P buffer of stream s at
    // 2*HD + s*128.  After the softmax has read S it writes P over it: for
    // keys [16c, 16c + 16), hi in columns 16c..16c+7 and lo in 16c+8..16c+15
    // (two bf16 per column), i.e. exactly over those keys' own S columns.
    constexpr uint32_t kCols = 512;
    constexpr uint32_t kColS = 2 * HD;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&v_ready[i], 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&p_empty[i], 1);
        }
        mbar_init(q_full, 32);
        mbar_init(q_empty, 1);
        mbar_init(ml_ready, 4);
        mbar_init(o_taken, 4);
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(tmem_slot, kCols); tmem_relinquish(); }
    plan_group(a, g, &ps);
    __syncthreads();
    // the merge kernel may be scheduled as CTAs of this grid leave; it waits
    // for this grid's completion before it reads a partial result
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    SegmentWalker walk;
    walk.init(a.kv_len, a.B, a.D, a.Hkv, a.max_len, g, ps.gbegin, ps.gend, ps.b0, ps.h0, ps.ub0);
    const int Hq = a.Hkv * a.G;
    Segment seg;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            uint32_t kg = 0;
            bool ok = true;
            while (ok && walk.next(seg)) {
                const int Lb = a.kv_len[seg.b];
                const int32_t *bt = a.block_table + static_cast<int64_t>(seg.b) * a.max_pages;
                for (int t = seg.tile_begin; t < seg.tile_end; ++t, ++kg) {
                    const int st = kg % S;
                    // page ids are looked up before waiting for the stage, so the
                    // block-table loads overlap the wait
                    const int key0 = t * kBN;
                    const int nvalid = min(kBN, Lb - key0);
                    int rows[kBN / 16];
                    int nbox = 0;
                    uint32_t bytes = 0;
                    for (int r0 = 0; r0 < kBN; r0 += a.box_rows, ++nbox) {
                        rows[nbox] = -1;
                        if (r0 >= nvalid) continue;
                        const int key = key0 + r0;
                        const int page = bt[key / a.page_size];
                        if (page < 0 || page >= a.num_pages) { report(a.dev_status, SPEC_DEV_ERR_PAGE_ID); continue; }
                        rows[nbox] = page * a.page_size + key % a.page_size;
                        bytes += 2u * L::kSub * a.box_rows * 128u;
                    }
                    if (kg >= S && !mbar_wait(&kv_empty[st], ((kg / S) & 1) ^ 1, abort, a.dev_status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&kv_full[st], bytes);
                    uint8_t *dk = sK + st * L::kKV;
                    uint8_t *dv = sV + st * L::kKV;
                    for (int i = 0; i < nbox; ++i) {
                        if (rows[i] < 0) continue;
                        const int r0 = i * a.box_rows;
#pragma unroll
                        for (int sub = 0; sub < L::kSub; ++sub) {
                            tma_load_3d(dk + sub * L::kSubBytes + r0 * 128, &tm_k, &kv_full[st], sub * 64, seg.h, rows[i]);
                            tma_load_3d(dv + sub * L::kSubBytes + r0 * 128, &tm_v, &kv_full[st], sub * 64, seg.h, rows[i]);
                        }
                    }
                }
            }
            if (*abort) {
                const uint32_t first = kg > static_cast<uint32_t>(S) ? kg - S : 0;
                for (uint32_t i = first; i < kg; ++i) mbar_wait_drain(&kv_full[i % S], (i / S) & 1, 100000000ull);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // -------------------------------------------- tcgen05 issuers
        // Tile k of a segment belongs to stream k & 1.  Warp 1 issues
        // S = QK^T for all tiles in order; warp 3 issues O += PV with one
        // cursor per stream, whichever stream's P is ready first.  Two
        // issuing threads keep a ready P.V from queueing behind a QK issue.
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_f16(kBM, kBN, 1, 0, 0);
            constexpr uint32_t idesc_pv = idesc_f16(kBM, HD, 1, 0, 1);
            // descriptors of the tile bases; a K step or a stage only moves
            // the start-address field
            const uint64_t dq0 = sdesc(smem_u32(sQ), 16, 1024);
            const uint64_t dk0 = sdesc(smem_u32(sK), 16, 1024);
            const uint64_t dv0 = sdesc(smem_u32(sV), L::kSubBytes, 1024);
            struct Cursor {
                SegmentWalker w;
                Segment seg;
                bool valid;
                int k, step;
                uint32_t j, base, si;   // global tile, segment's first global tile, segment index
                __device__ void start(const SegmentWalker &w0, int k0, int st)
                {
                    w = w0; k = k0; step = st; j = 0; base = 0; si = 0;
                    valid = w.next(seg);
                    settle(k0);
                }
                // move on while the current segment has no tile for this cursor
                __device__ void settle(int k_restart)
                {
                    while (valid && k >= seg.tile_end - seg.tile_begin) {
                        base += seg.tile_end - seg.tile_begin;
                        ++si;
                        k = k_restart;
                        valid = w.next(seg);
                    }
                    j = base + k;
                }
                __device__ void advance(int k_restart)
                {
                    k += step;
                    settle(k_restart);
                }
            };
            const bool qk_role = warp == 1;
            Cursor cq, cp[2];
            if (qk_role) {
                cq.start(walk, 0, 1);
                cp[0].valid = cp[1].valid = false;
            } else {
                cq.valid = false;
                cp[0].start(walk, 0, 2);
                cp[1].start(walk, 1, 2);
            }
            uint32_t nqk[2] = {0, 0}, npv[2] = {0, 0};
            unsigned long long t_idle = 0;
            uint32_t spins = 0;
            while (cq.valid || cp[0].valid || cp[1].valid) {
                bool progress = false;
                if (cq.valid) {
                    const int n = cq.seg.tile_end - cq.seg.tile_begin;
                    const uint32_t j = cq.j, st = j % S, sm = cq.k & 1, jq = nqk[sm];
                    if ((cq.k != 0 || mbar_test(q_full, cq.si & 1)) && mbar_test(&kv_full[st], (j / S) & 1) &&
                        (jq == 0 || mbar_test(&s_empty[sm], (jq - 1) & 1))) {
                        tc_fence_after();
                        const uint32_t d = tmem + kColS + sm * kBN;
#pragma unroll
                        for (int kk = 0; kk < HD / 16; ++kk) {
                            const uint64_t ad = dq0 + ((static_cast<uint32_t>(kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
                            const uint64_t bd = dk0 + ((st * L::kKV + static_cast<uint32_t>(kk >> 2) * L::kSubBytes + (kk & 3) * 32) >> 4);
                            umma_f16_ss(d, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        umma_commit(&s_full[sm]);
                        if (cq.k == n - 1) umma_commit(q_empty);
                        ++nqk[sm];
                        cq.advance(0);
                        progress = true;
                    }
                }
#pragma unroll
                for (int sm = 0; sm < 2; ++sm) {
                    Cursor &c = cp[sm];
                    if (!c.valid) continue;
                    const uint32_t j = c.j, st = j % S, jp = npv[sm];
                    if (mbar_test(&p_full[sm], jp & 1) && mbar_test(&v_ready[st], (j / S) & 1)) {
                        tc_fence_after();
                        const bool first = c.k < 2;     // first tile of this stream in the segment
                        const uint32_t p_tm = tmem + kColS + sm * kBN;
                        const uint32_t d = tmem + sm * HD;
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {
                            const uint64_t bd = dv0 + ((st * L::kKV + kk * 2048) >> 4);
                            umma_f16_ts(d, p_tm + kk * 16, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
                            umma_f16_ts(d, p_tm + kk * 16 + 8, bd, idesc_pv, 1u);
                        }
                        umma_commit(&p_empty[sm]);
                        umma_commit(&kv_empty[st]);
                        umma_commit(&s_empty[sm]);   // S/P columns reusable
                        ++npv[sm];
                        c.advance(sm);
                        progress = true;
                    }
                }
                if (progress) {
                    spins = 0;
                } else if ((++spins & 255u) == 0) {
                    if (*abort) break;
                    const unsigned long long now = globaltimer_ns();
                    if (spins == 256) t_idle = now;
                    else if (now - t_idle > kWaitTimeoutNs) {
                        *abort = 1;
                        report(a.dev_status, SPEC_DEV_ERR_TIMEOUT);
                        break;
                    }
                }
            }
        }
    } else if (warp == 2) {
        // ------------------------------- Q loader + V tail clearing (warp 2)
        const int ct = lane;
        uint32_t kg = 0, si = 0;
        bool ok = true;
        while (ok && walk.next(seg)) {
            if (si >= 1 && !mbar_wait(q_empty, (si - 1) & 1, abort, a.dev_status)) break;
            for (int rr = 0; rr < 4; ++rr) {
                const int rl = ct + rr * 32;
                const int r = mt * kBM + rl;
                if (r < a.R) {
                    const int i = r / a.G, gg = r % a.G;
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        a.q + ((static_cast<int64_t>(seg.b) * (a.D + 1) + i) * Hq + seg.h * a.G + gg) * HD);
#pragma unroll 4
                    for (int c = 0; c < HD / 8; ++c) {
                        const uint4 v = __ldg(src + c);
                        *reinterpret_cast<uint4 *>(sQ + (c >> 3) * (kBM * 128) + sw128_offset(rl, c & 7)) = v;
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < HD / 8; ++c)
                        *reinterpret_cast<uint4 *>(sQ + (c >> 3) * (kBM * 128) + sw128_offset(rl, c & 7)) = make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(q_full);
            const int Lb = a.kv_len[seg.b];
            for (int t = seg.tile_begin; t < seg.tile_end; ++t, ++kg) {
                const int st = kg % S;
                if (!mbar_wait(&kv_full[st], (kg / S) & 1, abort, a.dev_status)) { ok = false; break; }
                // Keys past the end of the sequence get P = 0, but 0 * NaN would
                // still poison O: clear those V rows (they hold whatever the
                // page or the stage held before).
                const int nvalid = min(kBN, Lb - t * kBN);
                if (nvalid < kBN) {
                    uint8_t *vt = sV + st * L::kKV;
                    for (int idx = ct; idx < L::kSub * kBN * 8; idx += 32) {
                        const int row = (idx & (kBN * 8 - 1)) >> 3;
                        if (row >= nvalid) *reinterpret_cast<uint4 *>(vt + idx * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&v_ready[st]);
            }
            ++si;
        }
    } else {
        // --------------------------------- softmax / epilogue, two streams
        // Warps 4-7 are stream 0, warps 8-11 stream 1; both streams own the
        // same 128 query rows (TMEM lanes) and take alternate key tiles.
        const int sm = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int rl = quad * 32 + lane;
        const int r = mt * kBM + rl;
        const bool row_ok = r < a.R;
        // a warp whose 32 rows are all padding (G(1+D) not a multiple of
        // 128) only has to write P = 0
        const bool pad_warp = mt * kBM + quad * 32 >= a.R;
        const int i_row = row_ok ? r / a.G : 0;
        const int g_row = row_ok ? r % a.G : 0;
        const uint32_t t_lane = tmem + ((quad * 32) << 16);
        const uint32_t t_o = t_lane + sm * HD;
        const uint32_t t_s = t_lane + kColS + sm * kBN;
        const float sc = a.scale_log2;
        uint32_t ns = 0, si = 0;     // tiles of this stream so far; segments
        bool ok = true;
        while (ok && walk.next(seg)) {
            const int n = seg.tile_end - seg.tile_begin;
            const int Lb = a.kv_len[seg.b];
            // Visible keys of this row: j < vis_end, plus key vis_end + x
            // for every bit x of vis_bits.  Chain: the prefix and drafts
            // 0..i (vis_bits = 0).  Tree: the prefix before the 1+D tree
            // keys, plus the tree keys on the root-to-node path.
            int vis_end;
            unsigned long long vis_bits;
            if (TREE) {
                vis_end = row_ok ? Lb - a.D - 1 : 0;
                vis_bits = row_ok ? a.tree_mask[static_cast<int64_t>(seg.b) * (a.D + 1) + i_row] : 0ull;
            } else {
                vis_end = row_ok ? Lb - a.D + i_row : 0;
                vis_bits = 0ull;
            }
            const int limit = vis_end;   // keys j < limit are visible for sure
            float m_ref = -INFINITY, l = 0.f;
            int ks = 0;
            for (int k = sm; k < n; k += 2, ++ks, ++ns) {
                if (!mbar_wait_warp(&s_full[sm], ns & 1, abort, a.dev_status)) { ok = false; break; }
                tc_fence_after();
                // S(ns) exists only after the stream's previous P.V finished
                // (the issuer waits for that before S = QK^T), so this confirms
                // that phase at once and keeps the p_empty waits in step.
                if (ns >= 1 && !mbar_wait_warp(&p_empty[sm], (ns - 1) & 1, abort, a.dev_status)) { ok = false; break; }
                if (pad_warp) {
                    uint32_t z[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) z[c] = 0u;
#pragma unroll
                    for (int q = 0; q < kBN / 32; ++q) tmem_st_32x32b_x32(t_s + 32 * q, z);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[sm]);
                    continue;
                }
                const int key0 = (seg.tile_begin + k) * kBN;
                const int nvis = limit - key0;            // keys [0, nvis) of the tile are visible
                // whether key c of the tile is visible (the slow path only)
                auto visible = [&](int c) {
                    if (!TREE) return c < nvis;
                    const unsigned x = static_cast<unsigned>(c - nvis);
                    return c < nvis || (x < 64u && ((vis_bits >> x) & 1ull));
                };
                // pass 1: row max of the raw scores
                float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll 1
                for (int q = 0; q < kBN / 32; q += 2) {
                    uint32_t x0[32], x1[32];
                    tmem_ld_32x32b_x32(t_s + 32 * q, x0);
                    tmem_ld_32x32b_x32(t_s + 32 * q + 32, x1);
                    tmem_ld_wait();
                    if (key0 + kBN <= limit) {
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            m0 = fmaxf(m0, fmaxf(__uint_as_float(x0[c]), __uint_as_float(x0[c + 1])));
                            m1 = fmaxf(m1, fmaxf(__uint_as_float(x1[c]), __uint_as_float(x1[c + 1])));
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            if (visible(32 * q + c)) m0 = fmaxf(m0, __uint_as_float(x0[c]));
                            if (visible(32 * q + 32 + c)) m1 = fmaxf(m1, __uint_as_float(x1[c]));
                        }
                    }
                }
                // max commutes with the positive scale: scale once
                const float mx = fmaxf(m0, m1) * sc;
                // Lazy rescaling: a row moves its reference max only when the
                // tile max exceeds it by more than 2^8.  The decision is per
                // row, but the TMEM access below is warp-collective, so the
                // whole warp takes the branch when any row needs it (rows that
                // do not keep alpha = 1).  The previous P.V of this stream is
                // already complete (confirmed above).
                const bool mine = mx > m_ref + kRescaleLog2;
                if (__any_sync(0xffffffffu, mine)) {
                    const float alpha = mine ? ex2(m_ref - mx) : 1.0f;   // 0 when m_ref = -inf
                    if (ks > 0) {
#pragma unroll 1
                        for (int c = 0; c < HD / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld_32x32b_x32(t_o + c * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st_32x32b_x32(t_o + c * 32, o);
                        }
                        tmem_st_wait();
                    }
                    if (mine) {
                        l *= alpha;
                        m_ref = mx;
                    }
                }
                // pass 2: p = 2^(s * scale_log2 - m_ref) (one FFMA and one MUFU
                // per key; masked keys give 0; a row with no visible key yet,
                // m_ref = -inf, writes zeros), split into hi + lo bf16 and
                // written over the same keys' S columns.
                const float neg_m = -m_ref;
                const bool live = m_ref != -INFINITY;
                const bool full = live && nvis >= kBN;   // no key of this tile is masked
                float l0 = 0.f, l1 = 0.f;
#pragma unroll 1
                for (int q = 0; q < kBN / 32; ++q) {
                    uint32_t x[32], pw[32];
                    tmem_ld_32x32b_x32(t_s + 32 * q, x);
                    tmem_ld_wait();
                    if (!full) {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (!live || !visible(32 * q + c)) x[c] = __float_as_uint(-INFINITY);
                    }
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        // masked keys: fma(-inf, sc, -m) = -inf and 2^-inf = 0;
                        // rows with m_ref = -inf have every key masked
                        const float p0 = ex2(fmaf(__uint_as_float(x[c]), sc, live ? neg_m : 0.f));
                        const float p1 = ex2(fmaf(__uint_as_float(x[c + 1]), sc, live ? neg_m : 0.f));
                        l0 += p0;
                        l1 += p1;
                        // hi = p truncated to bf16 (exact: the top half of p),
                        // lo = bf16(p - hi): hi + lo carries ~16 bits of p
                        const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
                        const uint32_t hw = __byte_perm(b0, b1, 0x7632);
                        const __nv_bfloat162 lb = __floats2bfloat162_rn(p0 - __uint_as_float(b0 & 0xFFFF0000u),
                                                                        p1 - __uint_as_float(b1 & 0xFFFF0000u));
                        // 16-key group gi = c / 16 of this chunk: hi words first, then lo
                        const int gi = c >> 4, wi = (c & 15) >> 1;
                        pw[gi * 16 + wi] = hw;
                        pw[gi * 16 + 8 + wi] = *reinterpret_cast<const uint32_t *>(&lb);
                    }
                    tmem_st_32x32b_x32(t_s + 32 * q, pw);
                }
                l += l0 + l1;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[sm]);
            }
            if (!ok) break;
            // Segment end: each stream's O is final once its last P.V is done.
            if (ks > 0 && !mbar_wait_warp(&p_empty[sm], (ns - 1) & 1, abort, a.dev_status)) break;
            tc_fence_before();
            if (sm == 1) {
                sML[rl] = make_float2(m_ref, l);
                __syncwarp();
                if (lane == 0) mbar_arrive(ml_ready);
                // stream 0 reads this stream's O before it may be overwritten
                if (!mbar_wait_warp(o_taken, si & 1, abort, a.dev_status)) break;
                tc_fence_after();
            } else {
                if (!mbar_wait_warp(ml_ready, si & 1, abort, a.dev_status)) break;
                tc_fence_after();
                const bool has1 = n >= 2;
                const float2 ml1 = sML[rl];
                const float m1v = has1 ? ml1.x : -INFINITY;
                const float M = fmaxf(m_ref, m1v);
                const float w0 = m_ref == -INFINITY ? 0.f : ex2(m_ref - M);
                const float w1 = m1v == -INFINITY ? 0.f : ex2(m1v - M);
                const float lsum = w0 * l + (has1 ? w1 * ml1.y : 0.f);
                float *dst;
                if (seg.slot < 0) {
                    dst = a.out + ((static_cast<int64_t>(seg.b) * (a.D + 1) + i_row) * Hq + seg.h * a.G + g_row) * HD;
                } else {
                    dst = a.part_o + ((static_cast<int64_t>(seg.slot) * a.nt + mt) * kBM + rl) * HD;
                }
                const float inv = (seg.slot < 0 && lsum > 0.f) ? 1.0f / lsum : 1.0f;
                const float c0w = w0 * inv, c1w = w1 * inv;
#pragma unroll 1
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o0[32], o1[32];
                    tmem_ld_32x32b_x32(t_lane + c * 32, o0);
                    if (has1) tmem_ld_32x32b_x32(t_lane + HD + c * 32, o1);
                    tmem_ld_wait();
                    if (row_ok) {
                        float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float4 v;
                            v.x = __uint_as_float(o0[4 * e]) * c0w;
                            v.y = __uint_as_float(o0[4 * e + 1]) * c0w;
                            v.z = __uint_as_float(o0[4 * e + 2]) * c0w;
                            v.w = __uint_as_float(o0[4 * e + 3]) * c0w;
                            if (has1) {
                                v.x += __uint_as_float(o1[4 * e]) * c1w;
                                v.y += __uint_as_float(o1[4 * e + 1]) * c1w;
                                v.z += __uint_as_float(o1[4 * e + 2]) * c1w;
                                v.w += __uint_as_float(o1[4 * e + 3]) * c1w;
                            }
                            d4[e] = v;
                        }
                    }
                }
                if (row_ok) {
                    if (seg.slot < 0) {
                        if (a.lse)
                            a.lse[(static_cast<int64_t>(seg.b) * (a.D + 1) + i_row) * Hq + seg.h * a.G + g_row] =
                                (M + __log2f(lsum)) * kLn2;
                    } else {
                        a.part_ml[(static_cast<int64_t>(seg.slot) * a.nt + mt) * kBM + rl] = make_float2(M, lsum);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_taken);
            }
            ++si;
        }
    }

    __syncwarp();
    __syncthreads();
    if (*abort && threadIdx.x == 32) {
        umma_commit(drain);
        mbar_wait_drain(drain, 0, 100000000ull);
    }
    __syncthreads();
    if (*abort && threadIdx.x == 96) {
        umma_commit(drain);
        mbar_wait_drain(drain, 1, 100000000ull);
    }
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, kCols); }
}

// Merge the partial results of units split across groups.  Block (g, mt):
// if group g's range begins inside a unit that started in an earlier group
// and ends within g, g is that unit's last group and merges it.
template <int HD>
__global__ void __launch_bounds__(kCombineThreads) attention_combine_kernel(const AttnArgs a)
{
    __shared__ PlanShared ps;
    const int g = blockIdx.x, mt = blockIdx.y;
    plan_group(a, g, &ps);
    if (ps.gbegin >= ps.gend || !ps.found) return;
    const int b = ps.b0, h = ps.h0;
    const int64_t ub = ps.ub0;
    const int nk = seq_tiles(a.kv_len[b], a.D, a.max_len);
    if (ub >= ps.gbegin || ub + nk > ps.gend) return;
    const int ge = ps.groups_eff;
    const int64_t total = ps.total;
    const int g_first = group_of(ub, total, ge);
    const int Hq = a.Hkv * a.G;
    // launched as a programmatic dependent of the attention grid: its
    // partial results are complete and visible only after this wait
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // four threads per row, each a quarter of its columns: short load chains
    // and 512 contiguous bytes per row across the four
    constexpr int kQ = kCombineThreads / kBM;   // threads per row
    constexpr int kCols = HD / kQ;              // columns per thread
    const int rl = threadIdx.x / kQ, c0 = (threadIdx.x % kQ) * kCols;
    {
        const int r = mt * kBM + rl;
        if (r >= a.R) return;
        const int i = r / a.G, gg = r % a.G;
        float M = -INFINITY;
        for (int q = g_first; q <= g; ++q) {
            const int64_t qb = group_begin(total, ge, q), qe = group_begin(total, ge, q + 1);
            if (qb >= qe) continue;
            const int slot = (ub <= qb) ? 2 * q : 2 * q + 1;
            M = fmaxf(M, a.part_ml[(static_cast<int64_t>(slot) * a.nt + mt) * kBM + rl].x);
        }
        float lsum = 0.f;
        float acc[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
        for (int q = g_first; q <= g; ++q) {
            const int64_t qb = group_begin(total, ge, q), qe = group_begin(total, ge, q + 1);
            if (qb >= qe) continue;
            const int slot = (ub <= qb) ? 2 * q : 2 * q + 1;
            const int64_t row = (static_cast<int64_t>(slot) * a.nt + mt) * kBM + rl;
            const float2 ml = a.part_ml[row];
            const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
            lsum += w * ml.y;
            const float4 *src = reinterpret_cast<const float4 *>(a.part_o + row * HD + c0);
#pragma unroll
            for (int c = 0; c < kCols / 4; ++c) {
                const float4 v = src[c];
                acc[4 * c] += w * v.x; acc[4 * c + 1] += w * v.y;
                acc[4 * c + 2] += w * v.z; acc[4 * c + 3] += w * v.w;
            }
        }
        const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
        const int64_t orow = (static_cast<int64_t>(b) * (a.D + 1) + i) * Hq + h * a.G + gg;
        float4 *dst = reinterpret_cast<float4 *>(a.out + orow * HD + c0);
#pragma unroll
        for (int c = 0; c < kCols / 4; ++c)
            dst[c] = make_float4(acc[4 * c] * inv, acc[4 * c + 1] * inv, acc[4 * c + 2] * inv, acc[4 * c + 3] * inv);
        if (a.lse && c0 == 0) a.lse[orow] = (M + __log2f(lsum)) * kLn2;
    }
}

template <int HD>
cudaError_t run(const CUtensorMap &tk, const CUtensorMap &tv, const AttnArgs &a, cudaStream_t st)
{
    using L = AttnSmem<HD>;
    auto k = a.tree_mask ? verify_attention_kernel<HD, true> : verify_attention_kernel<HD, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kBytes));
    if (e != cudaSuccess) return e;
    k<<<a.groups * a.nt, kThreads, L::kBytes, st>>>(tk, tv, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.groups, a.nt);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attention_combine_kernel<HD>, a);
}

}  // namespace

int attention_groups(int nt, int num_sms)
{
    const int g = num_sms / nt;
    return g < 1 ? 1 : g;
}

size_t attention_workspace_bytes(int nt, int head_dim, int num_sms)
{
    const size_t slots = 2 * static_cast<size_t>(attention_groups(nt, num_sms));
    const size_t rows = slots * nt * kBM;
    const size_t o = rows * head_dim * sizeof(float);
    return ((o + 255) & ~size_t(255)) + rows * sizeof(float2);
}

cudaError_t launch_verify_attention(const CUtensorMap &tk, const CUtensorMap &tv, const AttnArgs &a,
                                    int head_dim, cudaStream_t st)
{
    return head_dim == 128 ? run<128>(tk, tv, a, st) : run<64>(tk, tv, a, st);
}

namespace {

// One thread per (sequence, node): walk up to the root, collecting the
// path's bits.  Nodes are in topological order (parent < node), so a walk
// ends within T steps; anything else is reported and the node keeps its own
// bit only.
__global__ void tree_mask_kernel(const int32_t *__restrict__ parent, int B, int T,
                                 unsigned long long *__restrict__ mask, uint32_t *dev_status)
{
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<int64_t>(B) * T) return;
    const int k = static_cast<int>(idx % T);
    const int32_t *par = parent + (idx - k);
    bool ok = k == 0 ? par[0] == -1 : true;
    unsigned long long m = 1ull << k;
    int a = k;
    for (int steps = 0; ok && a > 0 && steps < T; ++steps) {
        const int pa = par[a];
        if (pa < 0 || pa >= a) {
            ok = false;
            break;
        }
        m |= 1ull << pa;
        a = pa;
    }
    if (ok && par[0] != -1) ok = false;
    if (!ok) {
        report(dev_status, SPEC_DEV_ERR_TREE);
        m = 1ull << k;
    }
    mask[idx] = m;
}

}  // namespace

cudaError_t launch_tree_masks(const int32_t *parent, int B, int T, unsigned long long *mask,
                              uint32_t *dev_status, cudaStream_t st)
{
    const int64_t n = static_cast<int64_t>(B) * T;
    if (n == 0) return cudaSuccess;
    tree_mask_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(parent, B, T, mask, dev_status);
    return cudaGetLastError();
}

}  // namespace spec
