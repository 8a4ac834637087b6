// Test-only kernels for the bounded waits every kernel of the library uses
// (gdn_tma.cuh): a wait on an mbarrier phase that nothing completes must give up
// after its time limit, a wait that watches an abort flag must return as soon as
// another warp sets it, and a completed phase must return at once.  Each kernel
// records what the wait returned and how long it took (globaltimer, ns).
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_tma.cuh"

namespace {

// mode 0: nothing arrives (the phase never completes)
// mode 1: warp 1 sets the abort flag after ~20 us; warp 0 waits with mbar_wait_or_abort
// mode 2: the phase is completed by an arrive before the wait
__global__ void wait_kernel(int mode, long long* out) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        gdn::mbar_init(&bar, 1);
        gdn::fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    if (mode == 2 && threadIdx.x == 0) gdn::mbar_arrive(&bar);
    __syncthreads();
    if (warp == 1 && lane == 0 && mode == 1) {
        const unsigned long long t0 = gdn::global_ns();
        while (gdn::global_ns() - t0 < 20000ull) {
        }
        abort_flag = 1;
    }
    if (warp == 0 && lane == 0) {
        const unsigned long long t0 = gdn::global_ns();
        bool ok;
        if (mode == 1)
            ok = gdn::mbar_wait_or_abort(&bar, 0, reinterpret_cast<const volatile int*>(&abort_flag));
        else
            ok = gdn::mbar_wait_bounded(&bar, 0);
        out[0] = ok ? 1 : 0;
        out[1] = (long long)(gdn::global_ns() - t0);
    }
}

}  // namespace

// Runs one wait_kernel launch of the given mode on the default stream; out_host[0] = the
// wait's result (1 completed, 0 gave up), out_host[1] = its duration in ns.  Returns the
// CUDA error code (0 on success).
extern "C" int gdn_test_wait(int mode, long long* out_host) {
    long long* d = nullptr;
    cudaError_t e = cudaMalloc(&d, 2 * sizeof(long long));
    if (e != cudaSuccess) return (int)e;
    wait_kernel<<<1, 64>>>(mode, d);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(out_host, d, 2 * sizeof(long long), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return (int)e;
}
