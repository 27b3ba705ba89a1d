// Host helpers: TMA tensor-map encoding through the driver entry point, and
// the device's SM count.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spec {

// Tiled bf16 tensor map with the 128-byte swizzle.  dims/strides_bytes are
// innermost first (strides exclude dim 0); box innermost extent must be
// 64 elements (128 bytes).  Returns false on failure.
bool encode_bf16_tmap(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                      const uint64_t *strides_bytes, const uint32_t *box);

// Tiled bf16 tensor map without swizzle (row-major boxes in shared memory),
// e.g. for TMA stores of output blocks.  Same argument convention.
bool encode_bf16_tmap_plain(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                            const uint64_t *strides_bytes, const uint32_t *box);

// SM count of the current device (cached per device), or -1.
int device_sm_count();

}  // namespace spec
