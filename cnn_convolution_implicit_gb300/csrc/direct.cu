// direct.cu -- general direct convolution on CUDA cores, any shape.
//
// One thread per output element with the sum held in a register: the simplest
// mapping of "GPU lesson 9: how a GPU executes neural-network convolution"
// (lincklin.cn), section 5, with the index map of section 2 (plus dilation and
// groups) and zero padding as an address test (section 26).  It runs the tiny
// FP32 layer and every shape the tensor-core and depthwise kernels do not take
// (odd channel counts, groups not aligned to the MMA tile, BF16 with
// C_out % 16 != 0, ...).  Threads are ordered with the output channel fastest
// so a warp writes a contiguous NHWC run and reads the same input pixels.
//
// Transposed convolution ("Convolution variants and their matrix operations",
// lpnh.cn/news/2674933, sections 2.3 and 4.2: the adjoint of the convolution,
// each input pixel (i, j) contributing to output (i*S + kh*D - P,
// j*S + kw*D - P)) runs here in gather form: output (ho, wo) takes input row
// i = (ho + P - kh*D) / S for every kernel row kh where the division is exact
// and i is inside the input, likewise for columns.
#include "conv_internal.h"
#include "ptx.cuh"

namespace convgb {

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) {
    return v;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) direct_kernel(const DirectParams p) {
    const ConvGeom& g = p.g;
    const long long total = g.pixels * g.C_out;
    const Tin* x = static_cast<const Tin*>(p.x);
    const Tin* w = static_cast<const Tin*>(p.w);
    Tout* y = static_cast<Tout*>(p.y);
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int co = static_cast<int>(i % g.C_out);
        const long long pix = i / g.C_out;
        const int wo = static_cast<int>(pix % g.W_out);
        const long long t = pix / g.W_out;
        const int ho = static_cast<int>(t % g.H_out);
        const int n = static_cast<int>(t / g.H_out);
        const int grp = co / g.cout_g;
        const Tin* wco = w + static_cast<long long>(co) * g.Kh * g.Kw * g.cin_g;
        float acc = 0.f;
        if (p.transposed) {
            for (int kh = 0; kh < g.Kh; ++kh) {
                const int nh = ho + g.P - kh * g.D;
                if (nh < 0 || nh % g.S != 0 || nh / g.S >= g.H) continue;
                const int hi = nh / g.S;
                for (int kw = 0; kw < g.Kw; ++kw) {
                    const int nw = wo + g.P - kw * g.D;
                    if (nw < 0 || nw % g.S != 0 || nw / g.S >= g.W) continue;
                    const int wi = nw / g.S;
                    const Tin* xp = x + ((static_cast<long long>(n) * g.H + hi) * g.W + wi) * g.C_in + grp * g.cin_g;
                    const Tin* wp = wco + (kh * g.Kw + kw) * g.cin_g;
                    for (int ci = 0; ci < g.cin_g; ++ci) acc = fmaf(to_f32(xp[ci]), to_f32(wp[ci]), acc);
                }
            }
        }
        for (int kh = 0; kh < g.Kh && !p.transposed; ++kh) {
            const int hi = ho * g.S + kh * g.D - g.P;
            if (hi < 0 || hi >= g.H) continue;
            for (int kw = 0; kw < g.Kw; ++kw) {
                const int wi = wo * g.S + kw * g.D - g.P;
                if (wi < 0 || wi >= g.W) continue;
                const Tin* xp = x + ((static_cast<long long>(n) * g.H + hi) * g.W + wi) * g.C_in + grp * g.cin_g;
                const Tin* wp = wco + (kh * g.Kw + kw) * g.cin_g;
                for (int ci = 0; ci < g.cin_g; ++ci) acc = fmaf(to_f32(xp[ci]), to_f32(wp[ci]), acc);
            }
        }
        if (p.scale) acc *= p.scale[co];
        if (p.bias) acc += p.bias[co];
        if (p.relu) acc = fmaxf(acc, 0.f);
        if constexpr (sizeof(Tout) == 2) {
            y[i] = __float2bfloat16_rn(acc);
        } else {
            y[i] = acc;
        }
    }
}

cudaError_t launch_direct(const DirectParams& p, cudaStream_t stream) {
    const long long total = p.g.pixels * p.g.C_out;
    const long long blocks_needed = (total + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(blocks_needed < (1ll << 20) ? blocks_needed : (1ll << 20));
    if (p.in_bf16) {
        direct_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks, 256, 0, stream>>>(p);
    } else if (p.out_bf16) {
        direct_kernel<float, __nv_bfloat16><<<blocks, 256, 0, stream>>>(p);
    } else {
        direct_kernel<float, float><<<blocks, 256, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace convgb
