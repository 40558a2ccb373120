// depthwise.cu -- FP32 depthwise convolution (G = C_in = C_out) as a direct
// kernel on CUDA cores.
//
// Depthwise convolution does no cross-channel sum ("GPU lesson 9: how a GPU
// executes neural-network convolution", lincklin.cn, section 23) and so has
// too little arithmetic per byte for tensor cores: it is bound by memory
// traffic (section 24).  It is computed directly with the shared-memory halo
// tile of sections 12-13: a CTA owns T x T output pixels of 32 channels and
// loads the (T-1)*S + (Kh-1)*D + 1 rows by as many columns of input they read
// (an 18 x 18 tile for 16 x 16 outputs of a 3x3 kernel) with one 4-D TMA tile
// copy from the NHWC tensor.  The copy's out-of-bounds zero fill is the zero
// padding (section 26).  Dilated kernels read only the Kh*Kw live taps.
//
// Each thread owns 4 channels (one float4, 128-bit shared loads and global
// stores) of one output column and walks T/RG output rows, holding its
// channels' weights in registers (lesson 9, sections 14 and 17-18).
#include "conv_internal.h"
#include "ptx.cuh"

namespace convgb {

namespace {

constexpr int kDwChannels = 32;  // channels per CTA: one 128-byte TMA row
constexpr int kDwRowGroups = 2;  // output-row groups per CTA

__device__ __forceinline__ void fma4(float4& acc, const float4& a, const float4& w) {
    acc.x = fmaf(a.x, w.x, acc.x);
    acc.y = fmaf(a.y, w.y, acc.y);
    acc.z = fmaf(a.z, w.z, acc.z);
    acc.w = fmaf(a.w, w.w, acc.w);
}

}  // namespace

// K > 0: square K x K kernel known at compile time; K == 0: any Kh x Kw.
template <int K, int T>
__global__ void __launch_bounds__(8 * T * kDwRowGroups)
    depthwise_kernel(const __grid_constant__ CUtensorMap x_map, const DepthwiseParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    float* tile = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int Kh = K > 0 ? K : p.g.Kh;
    const int Kw = K > 0 ? K : p.g.Kw;
    const int S = p.g.S, D = p.g.D;

    int b = blockIdx.x;
    const int cb = b % p.cblocks;
    b /= p.cblocks;
    const int tw = b % p.tiles_w;
    b /= p.tiles_w;
    const int th = b % p.tiles_h;
    const int n = b / p.tiles_h;
    const int ho0 = th * T, wo0 = tw * T, c0 = cb * kDwChannels;

    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t bytes = static_cast<uint32_t>(kDwChannels * 4 * p.in_w * p.in_h);
        mbar_arrive_expect_tx(&bar, bytes);
        tma_load_4d(tile, &x_map, &bar, c0, wo0 * S - p.g.P, ho0 * S - p.g.P, n);
    }

    const int c4 = threadIdx.x & 7;
    const int col = (threadIdx.x >> 3) % T;
    const int rg = (threadIdx.x >> 3) / T;
    const int c = c0 + 4 * c4;
    constexpr int kRows = T / kDwRowGroups;

    // Weights of this thread's 4 channels, tap-major, while the tile is in flight.
    constexpr int kTaps = K > 0 ? K * K : 1;
    float4 wreg[kTaps];
    if (K > 0) {
#pragma unroll
        for (int t = 0; t < kTaps; ++t) {
            wreg[t] = make_float4(__ldg(p.w + (c + 0) * kTaps + t), __ldg(p.w + (c + 1) * kTaps + t),
                                  __ldg(p.w + (c + 2) * kTaps + t), __ldg(p.w + (c + 3) * kTaps + t));
        }
    }
    float4 bias = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.bias) bias = *reinterpret_cast<const float4*>(p.bias + c);

    if (!mbar_wait(&bar, 0, &abort_flag)) {
        record_status(p.status, kStatusTimeoutDepthwise, &abort_flag);
        return;
    }

    const int wo = wo0 + col;
    const float4* t4 = reinterpret_cast<const float4*>(tile);
#pragma unroll 1
    for (int r = 0; r < kRows; ++r) {
        const int lr = rg * kRows + r;
        const int ho = ho0 + lr;
        float4 acc = bias;
        if (K > 0) {
#pragma unroll
            for (int kh = 0; kh < (K > 0 ? K : 1); ++kh)
#pragma unroll
                for (int kw = 0; kw < (K > 0 ? K : 1); ++kw) {
                    const int ih = lr * S + kh * D, iw = col * S + kw * D;
                    fma4(acc, t4[(ih * p.in_w + iw) * (kDwChannels / 4) + c4], wreg[kh * K + kw]);
                }
        } else {
            for (int kh = 0; kh < Kh; ++kh)
                for (int kw = 0; kw < Kw; ++kw) {
                    const int ih = lr * S + kh * D, iw = col * S + kw * D;
                    const int t = kh * Kw + kw;
                    const float4 wv = make_float4(__ldg(p.w + (c + 0) * Kh * Kw + t), __ldg(p.w + (c + 1) * Kh * Kw + t),
                                                  __ldg(p.w + (c + 2) * Kh * Kw + t), __ldg(p.w + (c + 3) * Kh * Kw + t));
                    fma4(acc, t4[(ih * p.in_w + iw) * (kDwChannels / 4) + c4], wv);
                }
        }
        if (p.relu) {
            acc.x = fmaxf(acc.x, 0.f);
            acc.y = fmaxf(acc.y, 0.f);
            acc.z = fmaxf(acc.z, 0.f);
            acc.w = fmaxf(acc.w, 0.f);
        }
        if (ho < p.g.H_out && wo < p.g.W_out) {
            const long long o = ((static_cast<long long>(n) * p.g.H_out + ho) * p.g.W_out + wo) * p.g.C_out + c;
            if (p.out_bf16) {
                uint2 q;
                q.x = pack_bf16x2(acc.x, acc.y);
                q.y = pack_bf16x2(acc.z, acc.w);
                *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.y) + o) = q;
            } else {
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + o) = acc;
            }
        }
    }
}

int depthwise_tile_for(const ConvGeom& g) {
    // 14 or 16 output pixels per side, whichever wastes fewer lanes on the ragged edge.
    auto waste = [&](int t) {
        const long long th = (g.H_out + t - 1) / t, tw = (g.W_out + t - 1) / t;
        return static_cast<double>(th * tw * t * t) / (static_cast<double>(g.H_out) * g.W_out);
    };
    const int t = waste(14) < waste(16) ? 14 : 16;
    const int in_h = (t - 1) * g.S + (g.Kh - 1) * g.D + 1;
    const int in_w = (t - 1) * g.S + (g.Kw - 1) * g.D + 1;
    if (in_h > 256 || in_w > 256) return 0;                      // TMA box limit
    if (static_cast<long long>(in_h) * in_w * kDwChannels * 4 > 200 * 1024) return 0;
    return t;
}

template <int K, int T>
static cudaError_t launch_dw(const CUtensorMap& x_map, const DepthwiseParams& p, cudaStream_t stream) {
    const int smem = p.in_h * p.in_w * kDwChannels * 4 + 128;
    cudaError_t e = cudaFuncSetAttribute(depthwise_kernel<K, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long blocks = static_cast<long long>(p.g.N) * p.tiles_h * p.tiles_w * p.cblocks;
    depthwise_kernel<K, T><<<static_cast<unsigned>(blocks), 8 * T * kDwRowGroups, smem, stream>>>(x_map, p);
    return cudaGetLastError();
}

cudaError_t launch_depthwise(const CUtensorMap& x_map, const DepthwiseParams& p, cudaStream_t stream) {
    const bool k3 = p.g.Kh == 3 && p.g.Kw == 3;
    if (p.tile == 14) return k3 ? launch_dw<3, 14>(x_map, p, stream) : launch_dw<0, 14>(x_map, p, stream);
    return k3 ? launch_dw<3, 16>(x_map, p, stream) : launch_dw<0, 16>(x_map, p, stream);
}

}  // namespace convgb
