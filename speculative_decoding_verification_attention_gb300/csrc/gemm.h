// Verify GEMM launch plan (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spec {

struct GemmPlan {
    bool swap;     // weights on the MMA M side (small M)
    int mpad;      // swap: x rows padded to the MMA N size
    int splits;    // swap: K split across a cluster of this many CTAs
    int bn;        // tiled: output tile width
};

GemmPlan plan_gemm(int M, int N, int K, int num_sms);

cudaError_t launch_gemm(const GemmPlan &p, const CUtensorMap &t_x, const CUtensorMap &t_w,
                        void *y, int M, int N, int K, int num_sms, uint32_t *dev_status,
                        cudaStream_t st);

}  // namespace spec
