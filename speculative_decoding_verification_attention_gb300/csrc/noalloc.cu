// Verify attention for callers that cannot allocate device memory.
//
// spec_verify_attention needs a caller-provided scratch buffer for the
// partial results of KV ranges split across CTAs.  Some callers have no way
// to provide one: a plugin inside an inference engine that owns all device
// memory through its own pool and forbids third-party allocations, or a
// latency-critical serving loop where cudaMalloc / cudaFree would
// synchronise the device.  This entry point takes its scratch from a fixed
// array compiled into the library instead, and allocates nothing.
#include <mutex>

#include "../../include/spec_verify.h"

namespace {

// The scratch array.  Every GPU that loads the library holds it until the
// process exits.  Host code must not pass this name to a kernel: on the
// host it is only a stand-in, so the device address is looked up below.
__device__ __align__(256) unsigned char g_attention_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
spec_status_t scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attention_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SPEC_OK;
}

}  // namespace

extern "C" spec_status_t spec_verify_attention_noalloc(
    const void *q_bf16, const void *k_pages_bf16, const void *v_pages_bf16, int num_pages,
    const int32_t *block_table, int max_pages_per_seq, const int32_t *kv_len, int B, int D,
    int Hkv, int G, int head_dim, int page_size, float softmax_scale, float *out_f32,
    float *lse_f32, uint32_t *dev_status, void *stream)
{
    if (max_pages_per_seq < 1 || page_size < 1) return SPEC_ERR_INVALID_ARG;
    const long long max_len = static_cast<long long>(max_pages_per_seq) * page_size;
    const size_t need = spec_verify_attention_workspace_size(
        B, D, Hkv, G, head_dim, max_len > 0x7fffffffLL ? 0x7fffffff : static_cast<int>(max_len));
    if (need > SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_WORKSPACE;
    void *scratch = nullptr;
    const spec_status_t st = scratch_for_current_device(&scratch);
    if (st != SPEC_OK) return st;
    // The partial results are always written before they are read, so the
    // scratch needs no clearing between calls.
    return spec_verify_attention(q_bf16, k_pages_bf16, v_pages_bf16, num_pages, block_table,
                                 max_pages_per_seq, kv_len, B, D, Hkv, G, head_dim, page_size,
                                 softmax_scale, out_f32, lse_f32, scratch,
                                 SPEC_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
