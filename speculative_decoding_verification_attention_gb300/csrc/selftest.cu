// Self-test of the bounded device wait that every kernel of the library
// uses on its mbarriers (no counterpart on the pages).  A wait that runs out
// must record SPEC_DEV_ERR_TIMEOUT, raise the kernel's abort flag and
// return, leaving the CUDA context usable; this entry point lets a test make
// a wait run out on purpose, on a barrier that nothing arrives on, with no
// copy or MMA in flight.
#include "common.cuh"

namespace spec {
namespace {

// One CTA of two warps.  Warp 0 waits on `bar` (phase 0) with the library's
// bounded wait limited to limit_ns.  Lane 0 of warp 1 arrives on it after
// arrive_after_ns, or never when arrive_after_ns is ~0.  Both paths end:
// the wait by its limit, the delayed arrival by its own deadline.
__global__ void __launch_bounds__(64, 1)
    bounded_wait_selftest_kernel(unsigned long long limit_ns, unsigned long long arrive_after_ns,
                                 unsigned long long *__restrict__ result, uint32_t *dev_status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        const unsigned long long t0 = globaltimer_ns();
        const bool ok = mbar_wait_warp(&bar, 0, &abort_flag, dev_status, limit_ns);
        const unsigned long long t1 = globaltimer_ns();
        if (lane == 0) {
            result[0] = ok ? 1ull : 0ull;
            result[1] = static_cast<unsigned long long>(*static_cast<volatile int *>(&abort_flag));
            result[2] = t1 - t0;
        }
    } else if (lane == 0 && arrive_after_ns != ~0ull) {
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < arrive_after_ns) __nanosleep(1000);
        mbar_arrive(&bar);
    }
    __syncthreads();
}

}  // namespace
}  // namespace spec

extern "C" spec_status_t spec_selftest_bounded_wait(uint64_t wait_limit_ns, uint64_t arrive_after_ns,
                                                    uint64_t *result, uint32_t *dev_status, void *stream)
{
    constexpr uint64_t kMaxNs = 10000000000ull;   // 10 s
    if (!result || wait_limit_ns == 0 || wait_limit_ns > kMaxNs) return SPEC_ERR_INVALID_ARG;
    if (arrive_after_ns != ~0ull && arrive_after_ns > kMaxNs) return SPEC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(result) % 8 != 0) return SPEC_ERR_INVALID_ARG;
    spec::bounded_wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
        wait_limit_ns, arrive_after_ns, reinterpret_cast<unsigned long long *>(result), dev_status);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
