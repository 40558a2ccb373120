// fp32x2.cuh -- packed FP32 fused multiply-add (fma.rn.f32x2) for the CUDA-core
// kernels.  Each of the two lanes rounds exactly as fmaf does, so a kernel that
// pairs its independent sums this way produces the same bits with half the FMA
// instructions.
#pragma once

namespace convgb {

// {a, b} as one 64-bit operand (a in the low lane).
__device__ __forceinline__ unsigned long long f32x2_pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

// {v, v}
__device__ __forceinline__ unsigned long long f32x2_dup(float v) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ void f32x2_unpack(unsigned long long v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

// d = a * b + d in both lanes.
__device__ __forceinline__ void f32x2_fma(unsigned long long& d, unsigned long long a, unsigned long long b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

}  // namespace convgb
