// tc_common.cuh -- pieces shared by the tcgen05 kernels: the fused
// bias + ReLU + BF16 epilogue of one 32-column TMEM chunk.
//
// Epilogue fusion follows "GPU lesson 9: how a GPU executes neural-network
// convolution" (lincklin.cn), section 31: the accumulator gets the bias, then
// the activation, in registers, and is written once.
#pragma once

#include "ptx.cuh"

namespace convgb {

// Staging of one 32-column chunk for a TMA store: thread `r` (0..31) writes the
// bias + ReLU + BF16 result of its row (64 bytes) into a 32 x 64-byte tile laid
// out in the 64-byte swizzle pattern (16-byte chunk j of row r at chunk
// j ^ ((r >> 1) & 3)), which the Y tensor map (box 32 x 32, SWIZZLE_64B) reads.
// Eight consecutive rows hit eight distinct bank groups, so the warp's stores
// are conflict-free.  SMEM_BIAS: `bias` and `scale` point to shared memory
// (else global, read through the read-only path).  `scale` (optional) multiplies
// the accumulator before the bias is added.
template <bool SMEM_BIAS = false>
__device__ __forceinline__ void stage_row32(const uint32_t (&v)[32], const float* bias, int relu, uint8_t* stg,
                                            int r, const float* scale = nullptr) {
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
    if (scale != nullptr) {  // per-channel scale first (a folded batch norm), then the shift
        const float4* s4 = reinterpret_cast<const float4*>(scale);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 s = SMEM_BIAS ? s4[i] : __ldg(s4 + i);
            f[4 * i + 0] *= s.x;
            f[4 * i + 1] *= s.y;
            f[4 * i + 2] *= s.z;
            f[4 * i + 3] *= s.w;
        }
    }
    if (bias != nullptr) {
        const float4* b4 = reinterpret_cast<const float4*>(bias);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 b = SMEM_BIAS ? b4[i] : __ldg(b4 + i);
            f[4 * i + 0] += b.x;
            f[4 * i + 1] += b.y;
            f[4 * i + 2] += b.z;
            f[4 * i + 3] += b.w;
        }
    }
    uint8_t* row = stg + r * 64;
    const int sw = (r >> 1) & 3;
    if (relu) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 q;
            q.x = pack_bf16x2_relu(f[8 * j + 0], f[8 * j + 1]);
            q.y = pack_bf16x2_relu(f[8 * j + 2], f[8 * j + 3]);
            q.z = pack_bf16x2_relu(f[8 * j + 4], f[8 * j + 5]);
            q.w = pack_bf16x2_relu(f[8 * j + 6], f[8 * j + 7]);
            *reinterpret_cast<uint4*>(row + ((j ^ sw) << 4)) = q;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 q;
            q.x = pack_bf16x2(f[8 * j + 0], f[8 * j + 1]);
            q.y = pack_bf16x2(f[8 * j + 2], f[8 * j + 3]);
            q.z = pack_bf16x2(f[8 * j + 4], f[8 * j + 5]);
            q.w = pack_bf16x2(f[8 * j + 6], f[8 * j + 7]);
            *reinterpret_cast<uint4*>(row + ((j ^ sw) << 4)) = q;
        }
    }
}

}  // namespace convgb
