// selftest.cu -- makes the kernels' bounded-wait failure path run, on purpose,
// without a fault: a test aid behind conv_check_wait_timeout (include/conv.h).
//
// Every mbarrier wait in the convolution kernels gives up after a time limit
// (mbar_wait: 2 s; mbar_wait_limit is the same loop with the limit as argument),
// latches a bit in the device status word, raises the CTA's abort flag so the
// other roles leave their loops, frees tensor memory and returns.  A working
// pipeline never takes that path, so this kernel builds the situation with the
// same helpers: one role waits (with the caller's short limit) on a barrier
// that nothing completes; a second role waits on another such barrier with the
// kernels' own 2 s limit and must leave early through the abort flag.  No wait
// is unbounded, nothing traps, and the context stays usable afterwards.
#include "conv.h"
#include "conv_internal.h"
#include "ptx.cuh"

namespace convgb {

namespace {

__global__ void __launch_bounds__(128, 1)
    wait_timeout_kernel(unsigned long long limit_ns, unsigned* status, unsigned long long* elapsed_ns) {
    __shared__ uint64_t never[2];   // barriers no thread arrives on
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&never[0], 1);
        mbar_init(&never[1], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {  // the role that owns tensor memory, as in the GEMM kernels
        tmem_alloc(&tmem_slot, 32);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1 && lane == 0) {
        // a consumer whose data never lands: the short limit runs out
        if (!mbar_wait_limit(&never[0], 0, abort, limit_ns)) record_status(status, kStatusTimeoutMma, abort);
    } else if (warp == 2 && lane == 0) {
        // another role blocked on its own barrier with the kernels' 2 s limit: it sees
        // the abort flag and leaves long before that; it times its own wait
        const uint64_t t0 = globaltimer_ns();
        if (!mbar_wait(&never[1], 0, abort)) record_status(status, kStatusTimeoutEpilogue, abort);
        const uint64_t t1 = globaltimer_ns();
        if (elapsed_ns != nullptr) *elapsed_ns = t1 - t0;
    }
    __syncwarp();      // the waiting lanes rejoin their warps before the CTA barrier
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_slot, 32);
    }
}

}  // namespace

}  // namespace convgb

extern "C" conv_status conv_check_wait_timeout(unsigned long long limit_ns, unsigned long long* elapsed_ns,
                                               void* stream) {
    using namespace convgb;
    if (limit_ns == 0 || limit_ns > kWaitTimeoutNs) return CONV_ERR_INVALID_ARG;
    if (elapsed_ns != nullptr && reinterpret_cast<uintptr_t>(elapsed_ns) % 8u != 0) return CONV_ERR_MISALIGNED;
    unsigned* status = nullptr;
    if (device_status_word(&status) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    wait_timeout_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, status, elapsed_ns);
    if (cudaGetLastError() != cudaSuccess) return CONV_ERR_CUDA;
    return CONV_OK;
}
