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
//   warp 0      TMA producer: K and V tiles of 64 keys, page by page, into a
//               ring of shared-memory stages (128-byte swizzle).
//   warp 1      tcgen05 issuer: S = Q K^T (bf16, fp32 in TMEM, two S
//               buffers) and O += P V (fp16, fp32 accumulator in TMEM).
//   warps 2-3   load the 128 query rows of each segment into shared memory;
//               convert each V tile bf16 -> fp16 in place (zeroing keys past
//               the end of the sequence).
//   warps 4-7   softmax: one thread per query row reads its S row from TMEM,
//               masks, keeps an online max / sum with lazy rescaling of O
//               (only when the max grows by more than 2^8), writes P as fp16
//               to shared memory; at the end of a segment reads O from TMEM
//               and writes the normalised output or a partial result.
// The KV stream of all (b, h) units is split evenly across CTA groups (see
// attn_schedule.h); units cut by a group boundary are merged by
// attention_combine.  G(1+D) > 128 uses several 128-row m-tiles, each its
// own CTA of the same group, so the same K/V tiles are read concurrently
// and served from L2.
//
// P is kept in fp16 rather than bf16: rounding P to bf16 alone gives about
// 2e-3 relative error in O; fp16 (11-bit significand) keeps it near 3e-4.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attention.h"
#include "attn_schedule.h"
#include "common.cuh"

namespace spec {
namespace {

constexpr int kBM = 128;
constexpr int kBN = kKeyTile;
constexpr int kThreads = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int HD>
struct AttnSmem {
    static constexpr int kSub = HD / 64;                   // 64-column chunks
    static constexpr uint32_t kQ = kBM * HD * 2;
    static constexpr uint32_t kKV = kBN * HD * 2;          // one K or V tile
    static constexpr int kStages = HD == 128 ? 4 : 6;
    static constexpr uint32_t kP = kBM * kBN * 2;          // one fp16 P buffer
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kQ;
    static constexpr uint32_t kOffV = kOffK + kStages * kKV;
    static constexpr uint32_t kOffP = kOffV + kStages * kKV;
    static constexpr uint32_t kOffBar = kOffP + 2 * kP;
    static constexpr uint32_t kBytes = kOffBar + 256 + 1024;
};

struct PlanShared {
    int64_t total, gbegin, gend, ub0;
    int b0, h0, groups_eff, found;
    int64_t warp_tot[kThreads / 32];
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
    for (int w = 0; w < kThreads / 32; ++w) {
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
    for (int b = threadIdx.x; b < a.B; b += kThreads) {
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
    for (int c0 = 0; c0 < a.B; c0 += kThreads) {
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

template <int HD>
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
    uint8_t *sP = smem + L::kOffP;
    uint64_t *kv_full = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *kv_empty = kv_full + S;
    uint64_t *v_ready = kv_empty + S;
    uint64_t *s_full = v_ready + S;
    uint64_t *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2;
    uint64_t *p_empty = p_full + 2;
    uint64_t *q_full = p_empty + 2;
    uint64_t *q_empty = q_full + 1;
    uint64_t *drain = q_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x / a.nt, mt = blockIdx.x % a.nt;
    constexpr uint32_t kCols = 256;        // O: HD columns, S: 2 x 64 columns
    constexpr uint32_t kColS = HD;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
            mbar_init(&v_ready[s], 64);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], 4);
            mbar_init(&p_full[s], 4);
            mbar_init(&p_empty[s], 1);
        }
        mbar_init(q_full, 64);
        mbar_init(q_empty, 1);
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(tmem_slot, kCols); tmem_relinquish(); }
    plan_group(a, g, &ps);
    __syncthreads();
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
                    if (kg >= S && !mbar_wait(&kv_empty[st], ((kg / S) & 1) ^ 1, abort, a.dev_status)) { ok = false; break; }
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
                    mbar_arrive_expect_tx(&kv_full[st], bytes);
                    uint8_t *dk = sK + st * L::kKV;
                    uint8_t *dv = sV + st * L::kKV;
                    for (int i = 0; i < nbox; ++i) {
                        if (rows[i] < 0) continue;
                        const int r0 = i * a.box_rows;
#pragma unroll
                        for (int sub = 0; sub < L::kSub; ++sub) {
                            tma_load_3d(dk + sub * (kBN * 128) + r0 * 128, &tm_k, &kv_full[st], sub * 64, seg.h, rows[i]);
                            tma_load_3d(dv + sub * (kBN * 128) + r0 * 128, &tm_v, &kv_full[st], sub * 64, seg.h, rows[i]);
                        }
                    }
                }
            }
            if (*abort) {
                const uint32_t first = kg > static_cast<uint32_t>(S) ? kg - S : 0;
                for (uint32_t i = first; i < kg; ++i) mbar_wait_drain(&kv_full[i % S], (i / S) & 1, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------- tcgen05 issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_f16(kBM, kBN, 1, 0, 0);
            constexpr uint32_t idesc_pv = idesc_f16(kBM, HD, 0, 0, 1);
            const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV),
                           p_base = smem_u32(sP);
            uint32_t kg = 0, si = 0;
            bool ok = true;
            auto issue_pv = [&](uint32_t j, bool first) -> bool {
                const uint32_t pb = j & 1, st = j % S;
                if (!mbar_wait(&p_full[pb], (j >> 1) & 1, abort, a.dev_status)) return false;
                if (!mbar_wait(&v_ready[st], (j / S) & 1, abort, a.dev_status)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t ad = sdesc(p_base + pb * L::kP + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc(v_base + st * L::kKV + kk * 2048, kBN * 128, 1024);
                    umma_f16_ss(tmem, ad, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
                }
                umma_commit(&p_empty[pb]);
                umma_commit(&kv_empty[st]);
                return true;
            };
            while (ok && walk.next(seg)) {
                const int n = seg.tile_end - seg.tile_begin;
                if (!mbar_wait(q_full, si & 1, abort, a.dev_status)) break;
                for (int k = 0; k < n && ok; ++k) {
                    const uint32_t j = kg + k, st = j % S, sb = j & 1;
                    if (!mbar_wait(&kv_full[st], (j / S) & 1, abort, a.dev_status)) { ok = false; break; }
                    if (j >= 2 && !mbar_wait(&s_empty[sb], ((j >> 1) & 1) ^ 1, abort, a.dev_status)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint64_t ad = sdesc(q_base + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = sdesc(k_base + st * L::kKV + (kk >> 2) * (kBN * 128) + (kk & 3) * 32, 16, 1024);
                        umma_f16_ss(tmem + kColS + sb * kBN, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&s_full[sb]);
                    if (k == n - 1) umma_commit(q_empty);
                    if (k >= 1 && !issue_pv(j - 1, k - 1 == 0)) { ok = false; break; }
                }
                if (!ok) break;
                if (!issue_pv(kg + n - 1, n == 1)) break;
                kg += n;
                ++si;
            }
        }
    } else if (warp < 4) {
        // ------------------------------- Q loader + V bf16 -> fp16 converter
        const int ct = threadIdx.x - 64;       // 0..63
        uint32_t kg = 0, si = 0;
        bool ok = true;
        while (ok && walk.next(seg)) {
            if (si >= 1 && !mbar_wait(q_empty, (si - 1) & 1, abort, a.dev_status)) break;
            for (int rr = 0; rr < 2; ++rr) {
                const int rl = ct + rr * 64;
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
                const int nvalid = min(kBN, Lb - t * kBN);
                uint8_t *vt = sV + st * L::kKV;
#pragma unroll 4
                for (int idx = ct; idx < L::kSub * kBN * 8; idx += 64) {
                    const int row = (idx & (kBN * 8 - 1)) >> 3;
                    uint4 *pch = reinterpret_cast<uint4 *>(vt + idx * 16);
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (row < nvalid) {
                        const uint4 in = *pch;
                        const uint32_t iw[4] = {in.x, in.y, in.z, in.w};
                        uint32_t ow[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float lo = __uint_as_float(iw[e] << 16);
                            const float hi = __uint_as_float(iw[e] & 0xFFFF0000u);
                            const __half2 h2 = __floats2half2_rn(lo, hi);
                            ow[e] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        w = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                    *pch = w;
                }
                fence_proxy_async_smem();
                mbar_arrive(&v_ready[st]);
            }
            ++si;
        }
    } else {
        // --------------------------------------------- softmax / epilogue
        const int quad = warp & 3;
        const int rl = quad * 32 + lane;
        const int r = mt * kBM + rl;
        const bool row_ok = r < a.R;
        const int i_row = row_ok ? r / a.G : 0;
        const int g_row = row_ok ? r % a.G : 0;
        const uint32_t t_lane = tmem + ((quad * 32) << 16);
        uint32_t kg = 0;
        bool ok = true;
        while (ok && walk.next(seg)) {
            const int n = seg.tile_end - seg.tile_begin;
            const int Lb = a.kv_len[seg.b];
            const int limit = row_ok ? Lb - a.D + i_row : 0;    // keys j < limit are visible
            float m_ref = -INFINITY, l = 0.f;
            for (int k = 0; k < n; ++k) {
                const uint32_t j = kg + k, sb = j & 1, pb = j & 1;
                if (!mbar_wait_warp(&s_full[sb], (j >> 1) & 1, abort, a.dev_status)) { ok = false; break; }
                tc_fence_after();
                uint32_t s0[32], s1[32];
                tmem_ld_32x32b_x32(t_lane + kColS + sb * kBN, s0);
                tmem_ld_32x32b_x32(t_lane + kColS + sb * kBN + 32, s1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                // Raw scores; keys at or past this row's limit become -inf.  Only
                // the tail tiles of a sequence need the mask.
                const int key0 = (seg.tile_begin + k) * kBN;
                float x[kBN];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    x[c] = __uint_as_float(s0[c]);
                    x[c + 32] = __uint_as_float(s1[c]);
                }
                if (key0 + kBN > limit) {
                    const int nvis = limit - key0;       // may be <= 0
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c >= nvis) x[c] = -INFINITY;
                }
                float m0 = fmaxf(x[0], x[1]), m1 = fmaxf(x[2], x[3]);
#pragma unroll
                for (int c = 4; c < kBN; c += 4) {
                    m0 = fmaxf(m0, fmaxf(x[c], x[c + 1]));
                    m1 = fmaxf(m1, fmaxf(x[c + 2], x[c + 3]));
                }
                // max commutes with the positive scale: scale once
                const float mx = fmaxf(m0, m1) * a.scale_log2;
                // Lazy rescaling: a row moves its reference max only when the
                // tile max exceeds it by more than 2^8.  The decision is per
                // row, but the TMEM access below is warp-collective, so the
                // whole warp takes the branch when any row needs it (rows that
                // do not keep alpha = 1).
                const bool mine = mx > m_ref + kRescaleLog2;
                if (__any_sync(0xffffffffu, mine)) {
                    const float alpha = mine ? ex2(m_ref - mx) : 1.0f;   // 0 when m_ref = -inf
                    if (k > 0) {
                        // O holds the P.V sums of this segment so far: wait for the
                        // last of them, then scale the rows in tensor memory.
                        const uint32_t jp = j - 1;
                        if (!mbar_wait_warp(&p_empty[jp & 1], (jp >> 1) & 1, abort, a.dev_status)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < HD / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld_32x32b_x32(t_lane + c * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st_32x32b_x32(t_lane + c * 32, o);
                        }
                        tmem_st_wait();
                    }
                    if (mine) {
                        l *= alpha;
                        m_ref = mx;
                    }
                }
                if (j >= 2 && !mbar_wait_warp(&p_empty[pb], ((j >> 1) & 1) ^ 1, abort, a.dev_status)) { ok = false; break; }
                // p = 2^(s * scale_log2 - m_ref): one FFMA and one MUFU per key;
                // masked keys (-inf) give 0.  A row with no visible key yet
                // (m_ref = -inf) writes zeros.
                uint32_t ph[kBN / 2];
                const float neg_m = -m_ref;
                const float sc = a.scale_log2;
                float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
                if (m_ref != -INFINITY) {
#pragma unroll
                    for (int c = 0; c < kBN; c += 4) {
                        const float p0 = ex2(fmaf(x[c], sc, neg_m));
                        const float p1 = ex2(fmaf(x[c + 1], sc, neg_m));
                        const float p2 = ex2(fmaf(x[c + 2], sc, neg_m));
                        const float p3 = ex2(fmaf(x[c + 3], sc, neg_m));
                        l0 += p0; l1 += p1; l2 += p2; l3 += p3;
                        const __half2 h01 = __floats2half2_rn(p0, p1);
                        const __half2 h23 = __floats2half2_rn(p2, p3);
                        ph[c / 2] = *reinterpret_cast<const uint32_t *>(&h01);
                        ph[c / 2 + 1] = *reinterpret_cast<const uint32_t *>(&h23);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kBN / 2; ++c) ph[c] = 0u;
                }
                l += (l0 + l1) + (l2 + l3);
                uint8_t *prow = sP + pb * L::kP;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(prow + sw128_offset(rl, c)) =
                        make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[pb]);
            }
            if (!ok) break;
            // segment end: O is complete once the last P.V has finished
            const uint32_t jl = kg + n - 1;
            if (!mbar_wait_warp(&p_empty[jl & 1], (jl >> 1) & 1, abort, a.dev_status)) break;
            tc_fence_after();
            float *dst;
            if (seg.slot < 0) {
                dst = a.out + ((static_cast<int64_t>(seg.b) * (a.D + 1) + i_row) * Hq + seg.h * a.G + g_row) * HD;
            } else {
                dst = a.part_o + ((static_cast<int64_t>(seg.slot) * a.nt + mt) * kBM + rl) * HD;
            }
            const float inv = (seg.slot < 0 && l > 0.f) ? 1.0f / l : 1.0f;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(t_lane + c * 32, o);
                tmem_ld_wait();
                if (row_ok) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        d4[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                            __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                }
            }
            if (row_ok) {
                if (seg.slot < 0) {
                    if (a.lse)
                        a.lse[(static_cast<int64_t>(seg.b) * (a.D + 1) + i_row) * Hq + seg.h * a.G + g_row] =
                            (m_ref + __log2f(l)) * kLn2;
                } else {
                    a.part_ml[(static_cast<int64_t>(seg.slot) * a.nt + mt) * kBM + rl] = make_float2(m_ref, l);
                }
            }
            tc_fence_before();
            kg += n;
        }
    }

    __syncwarp();
    __syncthreads();
    if (*abort && threadIdx.x == 32) {
        umma_commit(drain);
        mbar_wait_drain(drain, 0, 100000000ull);
    }
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, kCols); }
}

// Merge the partial results of units split across groups.  Block (g, mt):
// if group g's range begins inside a unit that started in an earlier group
// and ends within g, g is that unit's last group and merges it.
template <int HD>
__global__ void __launch_bounds__(kThreads) attention_combine_kernel(const AttnArgs a)
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
    for (int rl = threadIdx.x; rl < kBM; rl += kThreads) {
        const int r = mt * kBM + rl;
        if (r >= a.R) continue;
        const int i = r / a.G, gg = r % a.G;
        float M = -INFINITY;
        for (int q = g_first; q <= g; ++q) {
            const int64_t qb = group_begin(total, ge, q), qe = group_begin(total, ge, q + 1);
            if (qb >= qe) continue;
            const int slot = (ub <= qb) ? 2 * q : 2 * q + 1;
            M = fmaxf(M, a.part_ml[(static_cast<int64_t>(slot) * a.nt + mt) * kBM + rl].x);
        }
        float lsum = 0.f;
        float acc[HD];
#pragma unroll
        for (int c = 0; c < HD; ++c) acc[c] = 0.f;
        for (int q = g_first; q <= g; ++q) {
            const int64_t qb = group_begin(total, ge, q), qe = group_begin(total, ge, q + 1);
            if (qb >= qe) continue;
            const int slot = (ub <= qb) ? 2 * q : 2 * q + 1;
            const int64_t row = (static_cast<int64_t>(slot) * a.nt + mt) * kBM + rl;
            const float2 ml = a.part_ml[row];
            const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
            lsum += w * ml.y;
            const float4 *src = reinterpret_cast<const float4 *>(a.part_o + row * HD);
#pragma unroll
            for (int c = 0; c < HD / 4; ++c) {
                const float4 v = src[c];
                acc[4 * c] += w * v.x; acc[4 * c + 1] += w * v.y;
                acc[4 * c + 2] += w * v.z; acc[4 * c + 3] += w * v.w;
            }
        }
        const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
        float4 *dst = reinterpret_cast<float4 *>(a.out + ((static_cast<int64_t>(b) * (a.D + 1) + i) * Hq + h * a.G + gg) * HD);
#pragma unroll
        for (int c = 0; c < HD / 4; ++c)
            dst[c] = make_float4(acc[4 * c] * inv, acc[4 * c + 1] * inv, acc[4 * c + 2] * inv, acc[4 * c + 3] * inv);
        if (a.lse)
            a.lse[(static_cast<int64_t>(b) * (a.D + 1) + i) * Hq + h * a.G + gg] = (M + __log2f(lsum)) * kLn2;
    }
}

template <int HD>
cudaError_t run(const CUtensorMap &tk, const CUtensorMap &tv, const AttnArgs &a, cudaStream_t st)
{
    using L = AttnSmem<HD>;
    auto k = verify_attention_kernel<HD>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kBytes));
    if (e != cudaSuccess) return e;
    k<<<a.groups * a.nt, kThreads, L::kBytes, st>>>(tk, tv, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    attention_combine_kernel<HD><<<dim3(a.groups, a.nt), kThreads, 0, st>>>(a);
    return cudaGetLastError();
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

}  // namespace spec
