// mma_rate.cu -- the dense BF16 tensor rate of this GPU's SMs, measured.
//
// One CTA per SM issues `iters` back-to-back tcgen05.mma of M = 128, N = 256,
// K = 16 (BF16 operands from shared memory, FP32 accumulation in TMEM: the
// largest single-SM shape) and counts its SM's cycles from the first issue to
// the completion of the last.  2 * 128 * 256 * 16 * iters / cycles is the dense
// BF16 FLOP per clock per SM; times the SM count and the clock under load it is
// the chip's clock-derived peak, a second denominator beside a measured library
// GEMM.  The operands are zeros: the tensor pipe's rate does not depend on them.
#include "conv.h"
#include "conv_internal.h"
#include "tc_common.cuh"

namespace convgb {

namespace {

constexpr int kRateThreads = 128;
constexpr uint32_t kRateA = 128 * 128;  // 128 pixel rows x 128 bytes (K = 64 BF16), 128-byte swizzle
constexpr uint32_t kRateB = 256 * 128;  // 256 weight rows x 128 bytes
// more than half of an SM's shared memory, so no two CTAs share an SM
constexpr int kRateSmem = 120 * 1024;
constexpr int kRateMaxIters = 1 << 20;

__global__ void __launch_bounds__(kRateThreads, 1)
    mma_rate_kernel(int iters, unsigned long long* cycles, unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_slot;
    uint8_t* a = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* b = a + kRateA;
    for (uint32_t i = threadIdx.x * 16u; i < kRateA + kRateB; i += kRateThreads * 16u)
        *reinterpret_cast<uint4*>(a + i) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&done, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(&tmem_slot, 256);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (threadIdx.x == 0) {
        const uint32_t idesc = idesc_bf16_f32(128, 256);
        const uint64_t ad = sdesc_sw128(smem_addr(a)), bd = sdesc_sw128(smem_addr(b));
        const long long t0 = clock64();
        for (int i = 0; i < iters; ++i)  // the four K = 16 slices of the 128-byte rows in turn
            mma_bf16(tmem, ad + 2 * (i & 3), bd + 2 * (i & 3), idesc, i > 0 ? 1u : 0u);
        mma_commit(&done);
        const bool ok = mbar_wait(&done, 0, nullptr);
        const long long t1 = clock64();
        cycles[blockIdx.x] = ok ? static_cast<unsigned long long>(t1 - t0) : 0ull;
        if (!ok) record_status(status, kStatusTimeoutMma, nullptr);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

}  // namespace convgb

extern "C" conv_status conv_measure_mma_rate(int iters, unsigned long long* cycles, int grid, void* stream) {
    using namespace convgb;
    if (iters <= 0 || iters > kRateMaxIters || cycles == nullptr || grid <= 0) return CONV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(cycles) % 8u != 0) return CONV_ERR_MISALIGNED;
    unsigned* status = nullptr;
    static SmemLimitCache limits;
    if (device_status_word(&status) != cudaSuccess ||
        ensure_smem_limit(reinterpret_cast<const void*>(mma_rate_kernel), kRateSmem, limits) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    mma_rate_kernel<<<grid, kRateThreads, kRateSmem, static_cast<cudaStream_t>(stream)>>>(iters, cycles, status);
    if (cudaGetLastError() != cudaSuccess) return CONV_ERR_CUDA;
    return CONV_OK;
}
