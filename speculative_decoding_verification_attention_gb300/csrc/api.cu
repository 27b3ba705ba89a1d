// C-ABI entry points: host-side validation, then launches on the caller's
// stream.  Nothing here allocates device memory.
#include <cstdio>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "tmap.h"

using namespace spec;

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

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
    (void)dev_status;
    if (B < 0 || D < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (D > kMaxDraft || V > (1 << 26)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!p || !n_accepted || !token || (D > 0 && !draft)) return SPEC_ERR_INVALID_ARG;
    if (!aligned(p, 4) || !aligned(n_accepted, 4) || !aligned(token, 4)) return SPEC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * 8 > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
    return from_cuda(launch_accept_greedy(p, draft, B, D, V, n_accepted, token,
                                          static_cast<cudaStream_t>(stream)));
}

spec_status_t spec_accept_sample(const float *p, const float *q, const int32_t *draft,
                                 const float *u_acc, const float *u_res, int B, int D, int V,
                                 int32_t *n_accepted, int32_t *token, uint32_t *dev_status,
                                 void *stream)
{
    if (B < 0 || D < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
    if (D > kMaxDraft || V > (1 << 26)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!p || !u_res || !n_accepted || !token) return SPEC_ERR_INVALID_ARG;
    if (D > 0 && (!q || !draft || !u_acc)) return SPEC_ERR_INVALID_ARG;
    if (!aligned(p, 4) || (q && !aligned(q, 4)) || !aligned(n_accepted, 4) || !aligned(token, 4))
        return SPEC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * 8 > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
    return from_cuda(launch_accept_sample(p, q, draft, u_acc, u_res, B, D, V, n_accepted, token,
                                          dev_status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// Entry points whose kernels are not built yet.
extern "C" {

size_t spec_verify_attention_workspace_size(int, int, int, int, int, int) { return 0; }

spec_status_t spec_verify_attention(const void *, const void *, const void *, int,
                                    const int32_t *, int, const int32_t *, int, int, int, int,
                                    int, int, float, float *, float *, void *, size_t,
                                    uint32_t *, void *)
{
    return SPEC_ERR_UNSUPPORTED;
}

int spec_verify_attention_plan(int, const int32_t *, int, int, int, int32_t *, int) { return -1; }


}  // extern "C"

extern "C" {

size_t spec_verify_gemm_workspace_size(int, int, int) { return 0; }

spec_status_t spec_verify_gemm(const void *x_bf16, const void *w_bf16, void *y_bf16, int M, int N,
                               int K, void *workspace, size_t workspace_bytes, void *stream)
{
    (void)workspace;
    (void)workspace_bytes;
    if (M < 0 || N < 0 || K < 0) return SPEC_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SPEC_OK;
    if (M > 65536 || N % 128 != 0 || K % 64 != 0 || K == 0 || N > (1 << 20) || K > (1 << 20))
        return SPEC_ERR_UNSUPPORTED;
    if (!x_bf16 || !w_bf16 || !y_bf16) return SPEC_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(w_bf16, 16) || !aligned(y_bf16, 16))
        return SPEC_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return SPEC_ERR_CUDA;
    const GemmPlan plan = plan_gemm(M, N, K, sms);
    CUtensorMap tx, tw;
    const uint64_t dx[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t dw[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
    const uint64_t st[1] = {static_cast<uint64_t>(K) * 2};
    const uint32_t bx[2] = {64, static_cast<uint32_t>(plan.swap ? plan.mpad : 128)};
    const uint32_t bw[2] = {64, static_cast<uint32_t>(plan.swap ? 128 : plan.bn)};
    if (!encode_bf16_tmap(&tx, x_bf16, 2, dx, st, bx) || !encode_bf16_tmap(&tw, w_bf16, 2, dw, st, bw))
        return SPEC_ERR_CUDA;
    return from_cuda(launch_gemm(plan, tx, tw, y_bf16, M, N, K, sms, nullptr,
                                 static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
