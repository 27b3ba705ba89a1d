// C-ABI entry points: host-side validation, then launches on the caller's
// stream.  Nothing here allocates device memory.
#include <cmath>
#include <cstdio>

#include "attention.h"
#include "attn_schedule.h"
#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "tmap.h"

using namespace spec;

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t tree_mask_bytes(int B, int D)
{
    return (static_cast<size_t>(B) * (D + 1) * 8 + 255) & ~size_t(255);
}

spec_status_t from_cuda(cudaError_t e)
{
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *spec_status_string(int status)
{
    switch (status) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT";
    default: return "SPEC_ERR_UNKNOWN";
    }
}

int spec_version(void) { return 100; }

spec_status_t spec_accept_greedy(const float *p, const int32_t *draft, int B, int D, int V,
                                 int32_t *n_accepted, int32_t *token, uint32_t *dev_status,
                                 void *stream)
{
    if (B < 0 || D < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (D > kMaxDraft || V > (1 << 26)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!p || !n_accepted || !token || (D > 0 && !draft)) return SPEC_ERR_INVALID_ARG;
    if (!aligned(p, 4) || !aligned(n_accepted, 4) || !aligned(token, 4)) return SPEC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * 8 > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
    return from_cuda(launch_accept_greedy(p, draft, B, D, V, n_accepted, token, dev_status,
                                          static_cast<cudaStream_t>(stream)));
}

spec_status_t spec_accept_tree_greedy(const float *p, const int32_t *tokens, const int32_t *parent,
                                      int B, int D, int V, int32_t *n_accepted, int32_t *token,
                                      int32_t *path, uint32_t *dev_status, void *stream)
{
    if (B < 0 || D < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (D > kMaxDraft || V > (1 << 26)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!p || !tokens || !parent || !n_accepted || !token) return SPEC_ERR_INVALID_ARG;
    if (!aligned(p, 4) || !aligned(tokens, 4) || !aligned(parent, 4) || !aligned(n_accepted, 4) ||
        !aligned(token, 4) || (path && !aligned(path, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * 8 > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
    return from_cuda(launch_accept_tree_greedy(p, tokens, parent, B, D, V, n_accepted, token, path,
                                               dev_status, static_cast<cudaStream_t>(stream)));
}

spec_status_t spec_accept_tree_sample(const float *p, const float *q, const int32_t *tokens,
                                      const int32_t *parent, const float *u_acc, const float *u_res, int B,
                                      int D, int V, int32_t *n_accepted, int32_t *token, int32_t *path,
                                      uint32_t *dev_status, void *stream)
{
    if (B < 0 || D < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (D > kMaxDraft || V > (1 << 22)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!p || !q || !tokens || !parent || !u_acc || !u_res || !n_accepted || !token)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(p, 4) || !aligned(q, 4) || !aligned(tokens, 4) || !aligned(parent, 4) || !aligned(u_acc, 4) ||
        !aligned(u_res, 4) || !aligned(n_accepted, 4) || !aligned(token, 4) || (path && !aligned(path, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (B > 0x7fffffff / 2) return SPEC_ERR_UNSUPPORTED;
    return from_cuda(launch_accept_tree_sample(p, q, tokens, parent, u_acc, u_res, B, D, V, n_accepted, token, path,
                                               dev_status, static_cast<cudaStream_t>(stream)));
}

size_t spec_accept_sample_workspace_size(int B, int V)
{
    if (B < 0 || V < 1 || V > (1 << 26)) return 0;
    return accept_sample_workspace_bytes(B, V);
}

spec_status_t spec_accept_sample(const float *p, const float *q, const int32_t *draft,
                                 const float *u_acc, const float *u_res, int B, int D, int V,
                                 int32_t *n_accepted, int32_t *token, void *workspace,
                                 size_t workspace_bytes, uint32_t *dev_status, void *stream)
{
    if (B < 0 || D < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (D > kMaxDraft || V > (1 << 26)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!p || !u_res || !n_accepted || !token) return SPEC_ERR_INVALID_ARG;
    if (D > 0 && (!q || !draft || !u_acc)) return SPEC_ERR_INVALID_ARG;
    if (!aligned(p, 4) || (q && !aligned(q, 4)) || !aligned(n_accepted, 4) || !aligned(token, 4))
        return SPEC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * 8 > 0x7fffffffLL || B > 65535) return SPEC_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < accept_sample_workspace_bytes(B, V) || !aligned(workspace, 256))
        return SPEC_ERR_WORKSPACE;
    return from_cuda(launch_accept_sample(p, q, draft, u_acc, u_res, B, D, V, n_accepted, token,
                                          workspace, dev_status, static_cast<cudaStream_t>(stream)));
}

size_t spec_accept_adasd_workspace_size(int B, int D, int V)
{
    if (B < 0 || D < 0 || D > kMaxDraft || V < 1 || V > (1 << 26)) return 0;
    return accept_adasd_workspace_bytes(B, D, V);
}

spec_status_t spec_accept_adasd(const float *p, const float *q, const int32_t *draft, const float *u_acc,
                                const float *u_res, float tau_entropy, float tau_js, int B, int D, int V,
                                int32_t *n_accepted, int32_t *token, int32_t *draft_len, float *entropy,
                                float *js_distance, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                                void *stream)
{
    if (B < 0 || D < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (tau_entropy != tau_entropy || tau_js != tau_js) return SPEC_ERR_INVALID_ARG;   // NaN thresholds
    if (D > kMaxDraft || V > (1 << 26)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!p || !u_res || !n_accepted || !token) return SPEC_ERR_INVALID_ARG;
    if (D > 0 && (!q || !draft || !u_acc)) return SPEC_ERR_INVALID_ARG;
    if (!aligned(p, 4) || (q && !aligned(q, 4)) || !aligned(n_accepted, 4) || !aligned(token, 4) ||
        (draft_len && !aligned(draft_len, 4)) || (entropy && !aligned(entropy, 4)) ||
        (js_distance && !aligned(js_distance, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (B > 65535) return SPEC_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < accept_adasd_workspace_bytes(B, D, V) || !aligned(workspace, 256))
        return SPEC_ERR_WORKSPACE;
    return from_cuda(launch_accept_adasd(p, D > 0 ? q : nullptr, draft, u_acc, u_res, tau_entropy, tau_js, B, D, V,
                                         n_accepted, token, draft_len, entropy, js_distance, workspace, dev_status,
                                         static_cast<cudaStream_t>(stream)));
}

size_t spec_accept_sample_logits_workspace_size(int B, int D, int V)
{
    if (B < 0 || D < 0 || D > kMaxDraft || V < 1 || V > (1 << 26)) return 0;
    return accept_sample_logits_workspace_bytes(B, D, V);
}

spec_status_t spec_accept_sample_logits(const float *target_logits, const float *draft_logits,
                                        const int32_t *draft, float temperature, uint64_t seed, int B, int D,
                                        int V, int32_t *n_accepted, int32_t *token, void *workspace,
                                        size_t workspace_bytes, uint32_t *dev_status, void *stream)
{
    if (B < 0 || D < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (!(temperature > 0.0f) || !(temperature < INFINITY)) return SPEC_ERR_INVALID_ARG;
    if (D > kMaxDraft || V > (1 << 26)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !n_accepted || !token) return SPEC_ERR_INVALID_ARG;
    if (D > 0 && (!draft_logits || !draft)) return SPEC_ERR_INVALID_ARG;
    if (!aligned(target_logits, 4) || (draft_logits && !aligned(draft_logits, 4)) || !aligned(n_accepted, 4) ||
        !aligned(token, 4) || (draft && !aligned(draft, 4)))
        return SPEC_ERR_INVALID_ARG;
    if (B > 65535) return SPEC_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < accept_sample_logits_workspace_bytes(B, D, V) || !aligned(workspace, 256))
        return SPEC_ERR_WORKSPACE;
    return from_cuda(launch_accept_sample_logits(target_logits, D > 0 ? draft_logits : nullptr, draft, temperature,
                                                 seed, B, D, V, n_accepted, token, workspace, dev_status,
                                                 static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

constexpr int kMaxRows = 1024;      // G * (1 + D)
constexpr int kSmFallback = 256;    // upper bound when no device is current

bool attention_shape_supported(int D, int Hkv, int G, int head_dim)
{
    return D >= 0 && D <= kMaxDraft && Hkv >= 1 && G >= 1 &&
           static_cast<long long>(G) * (1 + D) <= kMaxRows && (head_dim == 64 || head_dim == 128);
}

}  // namespace

extern "C" {

size_t spec_verify_attention_workspace_size(int B, int D, int Hkv, int G, int head_dim,
                                            int max_kv_len)
{
    if (B < 0 || max_kv_len < 0 || !attention_shape_supported(D, Hkv, G, head_dim)) return 0;
    int sms = device_sm_count();
    if (sms <= 0) sms = kSmFallback;
    const int nt = (G * (1 + D) + 127) / 128;
    return attention_workspace_bytes(nt, head_dim, sms);
}

}  // extern "C"

namespace {

// Chain (tree_parent == NULL) or tree verify attention.  The tree's node
// masks go after the chain workspace.
spec_status_t verify_attention_impl(const void *q_bf16, const void *k_pages_bf16,
                                    const void *v_pages_bf16, int num_pages,
                                    const int32_t *block_table, int max_pages_per_seq,
                                    const int32_t *kv_len, const int32_t *tree_parent, int B, int D,
                                    int Hkv, int G, int head_dim, int page_size,
                                    float softmax_scale, float *out_f32, float *lse_f32,
                                    void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                                    void *stream)
{
    if (B < 0 || D < 0 || Hkv < 1 || G < 1 || head_dim < 1 || page_size < 1 || num_pages < 1 ||
        max_pages_per_seq < 1)
        return SPEC_ERR_INVALID_ARG;
    if (!attention_shape_supported(D, Hkv, G, head_dim) || page_size % 16 != 0)
        return SPEC_ERR_UNSUPPORTED;
    if (static_cast<long long>(num_pages) * page_size > 0x7fffffffLL ||
        static_cast<long long>(max_pages_per_seq) * page_size > 0x7fffffffLL)
        return SPEC_ERR_UNSUPPORTED;
    if (!(softmax_scale > 0.0f) || softmax_scale > 1e30f) return SPEC_ERR_INVALID_ARG;
    if (B == 0) return SPEC_OK;
    if (!q_bf16 || !k_pages_bf16 || !v_pages_bf16 || !block_table || !kv_len || !out_f32)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(q_bf16, 16) || !aligned(k_pages_bf16, 16) || !aligned(v_pages_bf16, 16) ||
        !aligned(out_f32, 16) || !aligned(block_table, 4) || !aligned(kv_len, 4) ||
        (lse_f32 && !aligned(lse_f32, 4)) || (tree_parent && !aligned(tree_parent, 4)))
        return SPEC_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return SPEC_ERR_CUDA;
    const int nt = (G * (1 + D) + 127) / 128;
    const size_t chain_need = attention_workspace_bytes(nt, head_dim, sms);
    const size_t need = chain_need + (tree_parent ? tree_mask_bytes(B, D) : 0);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SPEC_ERR_WORKSPACE;

    CUtensorMap tk, tv;
    const int box_rows = page_size % 64 == 0 ? 64 : page_size % 32 == 0 ? 32 : 16;
    const uint64_t dims[3] = {static_cast<uint64_t>(head_dim), static_cast<uint64_t>(Hkv),
                              static_cast<uint64_t>(num_pages) * page_size};
    const uint64_t strides[2] = {static_cast<uint64_t>(head_dim) * 2,
                                 static_cast<uint64_t>(Hkv) * head_dim * 2};
    const uint32_t box[3] = {64, 1, static_cast<uint32_t>(box_rows)};
    if (!encode_bf16_tmap(&tk, k_pages_bf16, 3, dims, strides, box) ||
        !encode_bf16_tmap(&tv, v_pages_bf16, 3, dims, strides, box))
        return SPEC_ERR_CUDA;

    AttnArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(q_bf16);
    a.block_table = block_table;
    a.kv_len = kv_len;
    a.out = out_f32;
    a.lse = lse_f32;
    a.part_o = static_cast<float *>(workspace);
    a.nt = nt;
    a.groups = attention_groups(nt, sms);
    const size_t o_bytes = static_cast<size_t>(2) * a.groups * nt * 128 * head_dim * sizeof(float);
    a.part_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + ((o_bytes + 255) & ~size_t(255)));
    a.dev_status = dev_status;
    a.B = B; a.D = D; a.Hkv = Hkv; a.G = G; a.R = G * (1 + D);
    a.page_size = page_size; a.box_rows = box_rows; a.max_pages = max_pages_per_seq;
    a.num_pages = num_pages;
    a.max_len = static_cast<int64_t>(max_pages_per_seq) * page_size;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.tree_mask = nullptr;
    if (tree_parent) {
        unsigned long long *masks =
            reinterpret_cast<unsigned long long *>(static_cast<char *>(workspace) + chain_need);
        const cudaError_t e = launch_tree_masks(tree_parent, B, D + 1, masks, dev_status,
                                                static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return from_cuda(e);
        a.tree_mask = masks;
    }
    return from_cuda(launch_verify_attention(tk, tv, a, head_dim, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

spec_status_t spec_verify_attention(const void *q_bf16, const void *k_pages_bf16,
                                    const void *v_pages_bf16, int num_pages,
                                    const int32_t *block_table, int max_pages_per_seq,
                                    const int32_t *kv_len, int B, int D, int Hkv, int G,
                                    int head_dim, int page_size, float softmax_scale,
                                    float *out_f32, float *lse_f32, void *workspace,
                                    size_t workspace_bytes, uint32_t *dev_status, void *stream)
{
    return verify_attention_impl(q_bf16, k_pages_bf16, v_pages_bf16, num_pages, block_table,
                                 max_pages_per_seq, kv_len, nullptr, B, D, Hkv, G, head_dim, page_size,
                                 softmax_scale, out_f32, lse_f32, workspace, workspace_bytes,
                                 dev_status, stream);
}

size_t spec_verify_tree_attention_workspace_size(int B, int D, int Hkv, int G, int head_dim,
                                                 int max_kv_len)
{
    const size_t chain = spec_verify_attention_workspace_size(B, D, Hkv, G, head_dim, max_kv_len);
    return B > 0 && D >= 0 ? chain + tree_mask_bytes(B, D) : chain;
}

spec_status_t spec_verify_tree_attention(const void *q_bf16, const void *k_pages_bf16,
                                         const void *v_pages_bf16, int num_pages,
                                         const int32_t *block_table, int max_pages_per_seq,
                                         const int32_t *kv_len, const int32_t *tree_parent, int B,
                                         int D, int Hkv, int G, int head_dim, int page_size,
                                         float softmax_scale, float *out_f32, float *lse_f32,
                                         void *workspace, size_t workspace_bytes,
                                         uint32_t *dev_status, void *stream)
{
    if (B > 0 && !tree_parent) return SPEC_ERR_INVALID_ARG;
    return verify_attention_impl(q_bf16, k_pages_bf16, v_pages_bf16, num_pages, block_table,
                                 max_pages_per_seq, kv_len, tree_parent, B, D, Hkv, G, head_dim,
                                 page_size, softmax_scale, out_f32, lse_f32, workspace,
                                 workspace_bytes, dev_status, stream);
}


int spec_verify_attention_plan(int B, const int32_t *kv_len_host, int D, int Hkv, int num_groups,
                               int32_t *segments, int max_segments)
{
    if (B < 0 || D < 0 || Hkv < 1 || num_groups < 1 || (B > 0 && !kv_len_host) ||
        max_segments < 0 || (max_segments > 0 && !segments))
        return -1;
    const int64_t max_len = INT64_MAX;
    const int64_t total = total_tiles_serial(kv_len_host, B, D, Hkv, max_len);
    const int ge = effective_groups(total, num_groups);
    int n = 0;
    for (int g = 0; g < ge; ++g) {
        const int64_t gb = group_begin(total, ge, g), gn = group_begin(total, ge, g + 1);
        if (gb >= gn) continue;
        int b0, h0;
        int64_t ub0;
        locate_serial(kv_len_host, B, D, Hkv, max_len, gb, b0, h0, ub0);
        SegmentWalker w;
        w.init(kv_len_host, B, D, Hkv, max_len, g, gb, gn, b0, h0, ub0);
        Segment s;
        while (w.next(s)) {
            if (n < max_segments) {
                int32_t *o = segments + 6 * static_cast<int64_t>(n);
                o[0] = g; o[1] = s.b; o[2] = s.h; o[3] = s.tile_begin; o[4] = s.tile_end; o[5] = s.slot;
            }
            ++n;
        }
    }
    return n;
}

}  // extern "C"

extern "C" {

size_t spec_verify_gemm_workspace_size(int M, int N, int K)
{
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    int sms = device_sm_count();
    if (sms <= 0) sms = kSmFallback;
    // an upper bound: the stream-K plan (split K needs no workspace, and the
    // device decides between the two)
    return plan_gemm(M, N, K, sms, sms / 2, SplitCaps{}).workspace_bytes;
}

int spec_verify_gemm_plan(int M, int N, int K, int num_sms, int32_t *segments, int max_segments)
{
    if (M <= 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 64 != 0 || num_sms <= 0 ||
        max_segments < 0 || (max_segments > 0 && !segments))
        return -1;
    const GemmPlan plan = plan_gemm(M, N, K, num_sms, num_sms / 2, split_caps_estimate(num_sms));
    int n = 0;
    if (!plan.swap) {
        // pairs: whole tiles, pair c taking tiles c, c + pairs, ...
        const PairGrid &g = plan.pg;
        for (int c = 0; c < g.pairs; ++c)
            for (int t = c; t < g.tiles(); t += g.pairs) {
                if (n < max_segments) {
                    int32_t *r = segments + 6 * static_cast<size_t>(n);
                    r[0] = c;
                    r[1] = t;
                    r[2] = 0;
                    r[3] = g.kblocks;
                    r[4] = c;
                    r[5] = g.width(t / g.tiles_m);
                }
                ++n;
            }
        return n;
    }
    if (plan.split >= 2 && plan.split_pairs) {
        // split K over S CTA pairs: CTA c = T 2S + 2p + h takes k-blocks
        // [p K/S, (p + 1) K/S) of 128-row tile 2T + h; pair 0's rows name
        // the last CTA holding the same tile (pair S - 1)
        const int S = plan.split, CS = 2 * S, kblocks = K / 64;
        for (int c = 0; c < plan.grid; ++c) {
            if (n < max_segments) {
                const int T = c / CS, pp = (c % CS) >> 1, h = c & 1;
                int32_t *row = segments + 6 * static_cast<size_t>(n);
                row[0] = c;
                row[1] = 2 * T + h;
                row[2] = pp * kblocks / S;
                row[3] = (pp + 1) * kblocks / S;
                row[4] = pp == 0 ? c + 2 * (S - 1) : -1;
                row[5] = plan.bn;
            }
            ++n;
        }
        return n;
    }
    if (plan.split >= 2) {
        // split K: CTA c = t S + r takes k-blocks [r K/S, (r + 1) K/S) of
        // tile t; rank 0's row names the last CTA of the tile's cluster
        const int S = plan.split, kblocks = K / 64;
        for (int c = 0; c < plan.grid; ++c) {
            if (n < max_segments) {
                const int t = c / S, r = c % S;
                int32_t *row = segments + 6 * static_cast<size_t>(n);
                row[0] = c;
                row[1] = t;
                row[2] = r * kblocks / S;
                row[3] = (r + 1) * kblocks / S;
                row[4] = r == 0 ? c + S - 1 : -1;
                row[5] = plan.bn;
            }
            ++n;
        }
        return n;
    }
    for (int c = 0; c < plan.sk.G; ++c) {
        SegWalker wk(plan.sk, c);
        Seg s;
        while (wk.next(s)) {
            if (n < max_segments) {
                int32_t *r = segments + 6 * static_cast<size_t>(n);
                r[0] = c;
                r[1] = s.t;
                r[2] = s.kb0;
                r[3] = s.kb1;
                r[4] = s.kb0 == 0 ? sk_last_contributor(plan.sk, c, s) : -1;
                r[5] = plan.bn;
            }
            ++n;
        }
    }
    return n;
}

int spec_verify_gemm_plan_cluster(int M, int N, int K, int num_sms)
{
    if (M <= 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 64 != 0 || num_sms <= 0) return -1;
    const GemmPlan plan = plan_gemm(M, N, K, num_sms, num_sms / 2, split_caps_estimate(num_sms));
    if (!plan.swap) return 2;
    if (plan.split < 2) return 1;
    return plan.split_pairs ? 2 * plan.split : plan.split;
}

spec_status_t spec_verify_gemm(const void *x_bf16, const void *w_bf16, void *y_bf16, int M, int N,
                               int K, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                               void *stream)
{
    if (M < 0 || N < 0 || K < 0) return SPEC_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SPEC_OK;
    if (M > 65536 || N % 128 != 0 || K % 64 != 0 || K == 0 || N > (1 << 20) || K > (1 << 20))
        return SPEC_ERR_UNSUPPORTED;
    if (!x_bf16 || !w_bf16 || !y_bf16) return SPEC_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(w_bf16, 16) || !aligned(y_bf16, 16))
        return SPEC_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return SPEC_ERR_CUDA;
    // only the variant this call runs is asked for its residency
    const GemmPlan probe = plan_gemm(M, N, K, sms, sms / 2, SplitCaps{});
    const int units = gemm_max_units(probe.bn, probe.swap);
    if (units <= 0) return SPEC_ERR_CUDA;
    const GemmPlan plan = plan_gemm(M, N, K, probe.swap ? units : sms, probe.swap ? sms / 2 : units,
                                    probe.swap ? split_caps_device(probe.bn) : SplitCaps{});
    if (plan.workspace_bytes > 0 &&
        (!workspace || workspace_bytes < plan.workspace_bytes || !aligned(workspace, 256)))
        return SPEC_ERR_WORKSPACE;
    return from_cuda(launch_gemm(plan, x_bf16, w_bf16, y_bf16, M, N, K, workspace, dev_status,
                                 static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
