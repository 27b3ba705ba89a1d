// Launch functions implemented by the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace spec {

constexpr int kMaxDraft = 63;

cudaError_t launch_accept_greedy(const float *p, const int32_t *draft, int B, int D, int V,
                                 int32_t *n_acc, int32_t *token, uint32_t *dev_status, cudaStream_t st);

cudaError_t launch_accept_tree_greedy(const float *p, const int32_t *tokens, const int32_t *parent, int B,
                                      int D, int V, int32_t *n_acc, int32_t *token, int32_t *path,
                                      uint32_t *dev_status, cudaStream_t st);

cudaError_t launch_accept_tree_sample(const float *p, const float *q, const int32_t *tokens, const int32_t *parent,
                                      const float *u_acc, const float *u_res, int B, int D, int V,
                                      int32_t *n_acc, int32_t *token, int32_t *path, uint32_t *dev_status,
                                      cudaStream_t st);

size_t accept_sample_workspace_bytes(int B, int V);

cudaError_t launch_accept_sample(const float *p, const float *q, const int32_t *draft,
                                 const float *u_acc, const float *u_res, int B, int D, int V,
                                 int32_t *n_acc, int32_t *token, void *workspace,
                                 uint32_t *dev_status, cudaStream_t st);

size_t accept_sample_logits_workspace_bytes(int B, int D, int V);

cudaError_t launch_accept_sample_logits(const float *zp, const float *zq, const int32_t *draft, float temperature,
                                        unsigned long long seed, int B, int D, int V, int32_t *n_acc,
                                        int32_t *token, void *workspace, uint32_t *dev_status, cudaStream_t st);

size_t accept_adasd_workspace_bytes(int B, int D, int V);

cudaError_t launch_accept_adasd(const float *p, const float *q, const int32_t *draft, const float *u_acc,
                                const float *u_res, float tau_h, float tau_js, int B, int D, int V, int32_t *n_acc,
                                int32_t *token, int32_t *d_eff, float *entropy, float *js_dist, void *workspace,
                                uint32_t *dev_status, cudaStream_t st);

}  // namespace spec
