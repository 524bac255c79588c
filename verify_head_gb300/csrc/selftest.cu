// Self-test of the bounded-wait path used by the tensor-core kernels: a wait
// on an mbarrier that no thread or copy ever completes must give up after the
// time limit, raise the error word and let the kernel return normally.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/verifyhead.h"
#include "vh_kernels.h"
#include "vh_ptx.cuh"

namespace {

__global__ void k_selftest_wait(unsigned int* flag, unsigned long long timeout_ns) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x == 0) {
        vh::ptx::mbar_init(&bar, 1);  // one arrival expected; none will come
        vh::ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned long long t0 = vh::ptx::globaltimer();
        bool done = false;
        while (!done) {
            if (vh::ptx::mbar_try_wait(&bar, 0u)) break;
            if (vh::ptx::globaltimer() - t0 > timeout_ns) {
                atomicOr(flag, 1u);
                done = true;
            }
        }
        // balance the barrier so that no phase is left pending at exit
        vh::ptx::mbar_arrive(&bar);
    }
}

inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" {

size_t vh_workspace_error_offset(void) { return vh::kWsErrorOffset; }

vh_status vh_selftest_bounded_wait(unsigned int* flag, unsigned int timeout_us, void* stream) {
    if (!flag) return VH_ERR_NULL;
    if (!aligned4(flag)) return VH_ERR_ALIGN;
    if (timeout_us < 1 || timeout_us > 1000000) return VH_ERR_SHAPE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return VH_ERR_DEVICE;
    }
    k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(flag, (unsigned long long)timeout_us * 1000ull);
    if (cudaGetLastError() != cudaSuccess) return VH_ERR_LAUNCH;
    return VH_OK;
}

}  // extern "C"
