// Verify GEMM launch plan (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gemm_schedule.h"

namespace spec {

// Workspace of the GEMM: an arrival counter per stream-K tile and CTA rank
// (fewer than 2 * kMaxCtas of them) in the first kFlagBytes, then two fp32
// 128 x BN partial tiles per CTA (its first and last stream-K segment).
constexpr int kMaxCtas = 256;
constexpr size_t kFlagBytes = 4096;

struct GemmPlan {
    bool swap;     // w rows on the MMA M side (M <= 256), x rows padded to bn
    int bn;        // MMA N: output tile width, or (swap) padded rows of x
    int grid;      // CTAs (tiled: in pairs), all co-resident
    SkGrid sk;     // stream-K decomposition; units are CTA pairs (tiled) or CTAs (swap)
    size_t workspace_bytes;  // ready flags + fp32 partial slots
};

// max_units_*: units (single CTAs for the swap orientation, CTA pairs for
// the tiled one) that can be resident at once.
GemmPlan plan_gemm(int M, int N, int K, int max_units_swap, int max_units_tiled);

// Resident units of the kernel variant on the current device (0 if the
// query fails).
int gemm_max_units(int bn, bool swap);

// t_y: y as bf16 [M][N] with 32 x 32 boxes and no swizzle (output stores).
cudaError_t launch_gemm(const GemmPlan &p, const CUtensorMap &t_x, const CUtensorMap &t_w,
                        const CUtensorMap &t_y, void *y, int M, int N, void *workspace,
                        uint32_t *dev_status, cudaStream_t st);

}  // namespace spec
