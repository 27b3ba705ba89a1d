// Verify-attention launch interface (host side).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace spec {

struct AttnArgs {
    const __nv_bfloat16 *q;
    const int32_t *block_table;
    const int32_t *kv_len;
    float *out;
    float *lse;                // may be null
    float *part_o;             // workspace: [2*groups][nt][128][head_dim]
    float2 *part_ml;           // workspace: [2*groups][nt][128] (max, sum)
    uint32_t *dev_status;      // may be null
    const unsigned long long *tree_mask;   // null: chain; else [B][1+D] root-to-node bits
    int B, D, Hkv, G, R, nt;
    int page_size, box_rows, max_pages, num_pages, groups;
    int64_t max_len;
    float scale_log2;          // softmax_scale * log2(e)
};

int attention_groups(int nt, int num_sms);
size_t attention_workspace_bytes(int nt, int head_dim, int num_sms);
cudaError_t launch_verify_attention(const CUtensorMap &tk, const CUtensorMap &tv,
                                    const AttnArgs &a, int head_dim, cudaStream_t st);

// Root-to-node bit masks of draft trees: mask[b][k] has bit a set for every
// node a on the path from the root to node k.  parent [B][T] (T <= 64);
// a malformed tree sets SPEC_DEV_ERR_TREE and gives its nodes their own bit
// only.
cudaError_t launch_tree_masks(const int32_t *parent, int B, int T, unsigned long long *mask,
                              uint32_t *dev_status, cudaStream_t st);

}  // namespace spec
