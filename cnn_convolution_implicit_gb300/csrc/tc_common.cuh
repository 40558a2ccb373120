// tc_common.cuh -- pieces shared by the tcgen05 kernels: the fused
// bias + ReLU + BF16 epilogue of one 32-column TMEM chunk.
//
// Epilogue fusion follows "GPU lesson 9: how a GPU executes neural-network
// convolution" (lincklin.cn), section 31: the accumulator gets the bias, then
// the activation, in registers, and is written once.
#pragma once

#include "ptx.cuh"

namespace convgb {

// v: 32 FP32 accumulators of one output pixel (columns co .. co+31, raw bits).
// bias: bias + co, or nullptr.  dst: y + pixel*C_out + co (16-byte aligned).
__device__ __forceinline__ void epilogue_store32(const uint32_t (&v)[32], const float* bias, int relu,
                                                 __nv_bfloat16* dst, bool valid) {
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
    if (bias != nullptr) {
        const float4* b4 = reinterpret_cast<const float4*>(bias);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 b = __ldg(b4 + i);
            f[4 * i + 0] += b.x;
            f[4 * i + 1] += b.y;
            f[4 * i + 2] += b.z;
            f[4 * i + 3] += b.w;
        }
    }
    if (relu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = fmaxf(f[i], 0.0f);
    }
    if (!valid) return;
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 q;
        q.x = pack_bf16x2(f[8 * i + 0], f[8 * i + 1]);
        q.y = pack_bf16x2(f[8 * i + 2], f[8 * i + 3]);
        q.z = pack_bf16x2(f[8 * i + 4], f[8 * i + 5]);
        q.w = pack_bf16x2(f[8 * i + 6], f[8 * i + 7]);
        d4[i] = q;
    }
}

}  // namespace convgb
