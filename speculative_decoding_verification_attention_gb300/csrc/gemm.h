// Verify GEMM launch plan (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gemm_schedule.h"

namespace spec {

// Workspace of the weight-streaming GEMM (M <= 256): an arrival counter per
// stream-K tile (fewer than kMaxCtas of them) in the first kFlagBytes, then
// two fp32 128 x BN partial tiles per CTA (its first and last stream-K
// segment).  The CTA-pair GEMM (M > 256) needs none.
constexpr int kMaxCtas = 256;
constexpr size_t kFlagBytes = 4096;

struct GemmPlan {
    bool swap;     // w rows on the MMA M side (M <= 256), x rows padded to bn
    int bn;        // swap: padded rows of x (MMA N); pairs: width of the first tile
    int grid;      // CTAs (pairs: in clusters of 2), all co-resident
    int split;     // swap: S >= 2 when each tile's k-blocks are split S ways in a cluster, else 0
    bool split_pairs;  // split: S CTA pairs per cluster over 256-row tiles (else S single CTAs)
    SkGrid sk;     // swap, split 0: stream-K decomposition over single CTAs
    PairGrid pg;   // pairs: ragged whole tiles
    size_t workspace_bytes;  // stream-K: ready flags + fp32 partial slots; split, pairs: 0
};

// Resident clusters of the split-K weight-streaming kernels: of S single
// CTAs (index S = 2..8) and of S CTA pairs (2S CTAs, index S = 2..4); 0
// where S cannot be used.
struct SplitCaps {
    int max_clusters[9];
    int pair_clusters[5];
};

// The resident clusters on the current device for x padded to bn rows, and
// an estimate from the SM count alone (host planning without a device).
SplitCaps split_caps_device(int bn);
SplitCaps split_caps_estimate(int sms);

// max_units_*: units (single CTAs for the swap orientation, CTA pairs for
// M > 256) that can be resident at once; caps: where split K is possible
// (all zero: stream-K only).
GemmPlan plan_gemm(int M, int N, int K, int max_units_swap, int max_units_pair, const SplitCaps &caps);

// Resident units of the kernel variant on the current device (0 if the
// query fails).
int gemm_max_units(int bn, bool swap);

// Encodes the tensor maps of x [M][K], w [N][K] and y [M][N] (bf16,
// row-major) and launches the plan's kernel on st.
cudaError_t launch_gemm(const GemmPlan &p, const void *x, const void *w, void *y, int M, int N, int K,
                        void *workspace, uint32_t *dev_status, cudaStream_t st);

}  // namespace spec
