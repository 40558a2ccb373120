// depthwise.cu -- FP32 depthwise convolution (G = C_in = C_out) as a direct
// kernel on CUDA cores.
//
// Depthwise convolution does no cross-channel sum ("GPU lesson 9: how a GPU
// executes neural-network convolution", lincklin.cn, section 23) and so has
// too little arithmetic per byte for tensor cores: it is bound by memory
// traffic (section 24).  It is computed directly with the shared-memory halo
// tile of sections 12-13: a tile of TH x TW output pixels and 32 channels
// reads the ((TH-1)*S + (Kh-1)*D + 1) x ((TW-1)*S + (Kw-1)*D + 1) input pixels
// under it (e.g. 30 x 10 for 28 x 8 outputs of a 3x3 kernel), fetched with one
// 4-D TMA tile copy from the NHWC tensor; the copy's out-of-bounds zero fill is
// the zero padding (section 26), and a dilated kernel reads only its Kh*Kw
// live taps.
//
// The kernel is persistent (one CTA per SM) and keeps a ring of `stages` halo
// tiles in flight, so HBM reads of the next tiles overlap the arithmetic and
// stores of the current one.  Each of the 256 threads owns 4 channels (one
// float4: 128-bit shared loads and global stores) of one output column and
// walks a run of output rows.  For stride 1 / dilation 1 it keeps the last Kh-1 input rows of its
// Kh x Kw window in registers and reads one new row per output row (lesson 9,
// sections 6 and 17-18: input reuse held in registers, several outputs per
// thread); weights live in registers.
#include "conv_internal.h"
#include "ptx.cuh"

namespace convgb {

namespace {

constexpr int kDwChannels = 32;  // channels per tile: one 128-byte TMA row
constexpr int kDwThreads = 256;  // 8 channel quads x TW columns x (32 / TW) row groups

__device__ __forceinline__ void fma4(float4& acc, const float4& a, const float4& w) {
    acc.x = fmaf(a.x, w.x, acc.x);
    acc.y = fmaf(a.y, w.y, acc.y);
    acc.z = fmaf(a.z, w.z, acc.z);
    acc.w = fmaf(a.w, w.w, acc.w);
}

struct DwTile {
    int n, ho0, wo0, c0;
};

__device__ __forceinline__ DwTile dw_decode(const DepthwiseParams& p, int t) {
    DwTile d;
    const int cb = t % p.cblocks;
    t /= p.cblocks;
    const int tw = t % p.tiles_w;
    t /= p.tiles_w;
    const int th = t % p.tiles_h;
    d.n = t / p.tiles_h;
    d.ho0 = th * p.tile_h;
    d.wo0 = tw * p.tile_w;
    d.c0 = cb * kDwChannels;
    return d;
}

__device__ __forceinline__ void dw_store(const DepthwiseParams& p, int n, int ho, int wo, int c, float4 acc) {
    if (p.relu) {
        acc.x = fmaxf(acc.x, 0.f);
        acc.y = fmaxf(acc.y, 0.f);
        acc.z = fmaxf(acc.z, 0.f);
        acc.w = fmaxf(acc.w, 0.f);
    }
    if (ho >= p.g.H_out || wo >= p.g.W_out) return;
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

}  // namespace

// K > 0: square K x K kernel known at compile time; K == 0: any Kh x Kw.
template <int K, int TW>
__global__ void __launch_bounds__(kDwThreads, 1)
    depthwise_kernel(const __grid_constant__ CUtensorMap x_map, const DepthwiseParams p) {
    constexpr int kRowGroups = kDwThreads / (8 * TW);
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t full[8];
    __shared__ int abort_flag;
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int Kh = K > 0 ? K : p.g.Kh;
    const int Kw = K > 0 ? K : p.g.Kw;
    const int S = p.g.S, D = p.g.D;
    const int stage_bytes = p.in_h * p.in_w * kDwChannels * 4;
    const uint32_t box_bytes = static_cast<uint32_t>(stage_bytes);
    const int num_tiles = p.num_tiles;
    const int my_count = blockIdx.x < num_tiles ? (num_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    int issued = 0;            // tiles whose TMA thread 0 has issued
    auto issue = [&](int i) {  // TMA of this CTA's i-th tile into slot i % stages
        const int slot = i % p.stages;
        issued = i + 1;
        const DwTile t = dw_decode(p, blockIdx.x + i * gridDim.x);
        mbar_arrive_expect_tx(&full[slot], box_bytes);
        tma_load_4d(ring + slot * stage_bytes, &x_map, &full[slot], t.c0, t.wo0 * S - p.g.P, t.ho0 * S - p.g.P, t.n);
    };
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&x_map);
        for (int i = 0; i < p.stages && i < my_count; ++i) issue(i);
    }

    const int c4 = threadIdx.x & 7;
    const int col = (threadIdx.x >> 3) % TW;
    const int rg = (threadIdx.x >> 3) / TW;
    const int rows = p.tile_h / kRowGroups;
    const bool rolling = K == 3 && S == 1 && D == 1;
    constexpr int kTaps = K > 0 ? K * K : 1;
    const int in_row4 = p.in_w * (kDwChannels / 4);  // float4 per input row

    for (int i = 0; i < my_count; ++i) {
        const DwTile t = dw_decode(p, blockIdx.x + i * gridDim.x);
        const int c = t.c0 + 4 * c4;
        // weights and bias of this thread's 4 channels (L1-resident), before the wait
        float4 wreg[kTaps];
        if (K > 0) {
#pragma unroll
            for (int k = 0; k < kTaps; ++k)
                wreg[k] = make_float4(__ldg(p.w + (c + 0) * kTaps + k), __ldg(p.w + (c + 1) * kTaps + k),
                                      __ldg(p.w + (c + 2) * kTaps + k), __ldg(p.w + (c + 3) * kTaps + k));
        }
        float4 bias = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.bias) bias = __ldg(reinterpret_cast<const float4*>(p.bias + c));

        const int slot = i % p.stages;
        const bool ok = mbar_wait(&full[slot], static_cast<uint32_t>((i / p.stages) & 1), &abort_flag);
        if (__syncthreads_or(!ok)) {  // block-uniform exit
            if (!ok) record_status(p.status, kStatusTimeoutDepthwise, &abort_flag);
            break;
        }
        const float4* t4 = reinterpret_cast<const float4*>(ring + slot * stage_bytes);
        const int wo = t.wo0 + col;
        const int lr0 = rg * rows;

        if (rolling) {
            // window rows r, r+1 held in registers; one new input row per output row
            const float4* base = t4 + (lr0 * p.in_w + col) * (kDwChannels / 4) + c4;
            float4 a0 = base[0], a1 = base[8], a2 = base[16];
            float4 b0 = base[in_row4], b1 = base[in_row4 + 8], b2 = base[in_row4 + 16];
            const int ho_first = t.ho0 + lr0;
            const int nrows = min(rows, p.g.H_out - ho_first);  // rows of this thread inside the image
            const long long row_stride = static_cast<long long>(p.g.W_out) * p.g.C_out;
            const long long o0 = ((static_cast<long long>(t.n) * p.g.H_out + ho_first) * p.g.W_out + wo) * p.g.C_out + c;
            const bool col_ok = wo < p.g.W_out;
            float* yf = reinterpret_cast<float*>(p.y) + o0;
            __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(p.y) + o0;
            const float4* cr = base + 2 * in_row4;
#pragma unroll 2
            for (int r = 0; r < nrows; ++r) {
                const float4 d0 = cr[0], d1 = cr[8], d2 = cr[16];
                cr += in_row4;
                float4 acc = bias;
                fma4(acc, a0, wreg[0]);
                fma4(acc, a1, wreg[1 % kTaps]);
                fma4(acc, a2, wreg[2 % kTaps]);
                fma4(acc, b0, wreg[3 % kTaps]);
                fma4(acc, b1, wreg[4 % kTaps]);
                fma4(acc, b2, wreg[5 % kTaps]);
                fma4(acc, d0, wreg[6 % kTaps]);
                fma4(acc, d1, wreg[7 % kTaps]);
                fma4(acc, d2, wreg[8 % kTaps]);
                if (p.relu) {
                    acc.x = fmaxf(acc.x, 0.f);
                    acc.y = fmaxf(acc.y, 0.f);
                    acc.z = fmaxf(acc.z, 0.f);
                    acc.w = fmaxf(acc.w, 0.f);
                }
                if (col_ok) {
                    if (p.out_bf16) {
                        uint2 q;
                        q.x = pack_bf16x2(acc.x, acc.y);
                        q.y = pack_bf16x2(acc.z, acc.w);
                        *reinterpret_cast<uint2*>(yb) = q;
                    } else {
                        *reinterpret_cast<float4*>(yf) = acc;
                    }
                }
                yf += row_stride;
                yb += row_stride;
                a0 = b0; a1 = b1; a2 = b2;
                b0 = d0; b1 = d1; b2 = d2;
            }
        } else {
            for (int r = 0; r < rows; ++r) {
                const int lr = lr0 + r;
                float4 acc = bias;
                for (int kh = 0; kh < Kh; ++kh)
                    for (int kw = 0; kw < Kw; ++kw) {
                        const int ih = lr * S + kh * D, iw = col * S + kw * D;
                        float4 wv;
                        if (K > 0) {
                            wv = wreg[(kh * Kw + kw) % kTaps];
                        } else {
                            const int k = kh * Kw + kw, taps = Kh * Kw;
                            wv = make_float4(__ldg(p.w + (c + 0) * taps + k), __ldg(p.w + (c + 1) * taps + k),
                                             __ldg(p.w + (c + 2) * taps + k), __ldg(p.w + (c + 3) * taps + k));
                        }
                        fma4(acc, t4[(ih * p.in_w + iw) * (kDwChannels / 4) + c4], wv);
                    }
                dw_store(p, t.n, t.ho0 + lr, wo, c, acc);
            }
        }
        __syncthreads();  // every thread is done with this slot
        if (threadIdx.x == 0 && i + p.stages < my_count && !abort_flag) issue(i + p.stages);
    }
    // Leave no copy in flight: wait (bounded) for every issued fill of each slot.
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages && s < issued; ++s) {
            const int fills = (issued - 1 - s) / p.stages + 1;  // fills issued into slot s
            if (!mbar_wait(&full[s], static_cast<uint32_t>((fills - 1) & 1), nullptr))
                record_status(p.status, kStatusTimeoutDrain, nullptr);
        }
    }
}

int depthwise_config(const ConvGeom& g, int smem_optin, DepthwiseParams& d) {
    // Tile width 8 or 16 columns (a warp never straddles two row groups),
    // height from {32, 28, 24, 16} with the least ragged-edge waste, then as
    // many ring stages (<= 8) as fit in shared memory; shrink the height if
    // fewer than two stages fit (large strides or dilations).
    auto padded = [](int extent, int t) { return ((extent + t - 1) / t) * t; };
    const int tw = padded(g.W_out, 8) < padded(g.W_out, 16) ? 8 : 16;
    const int rg = kDwThreads / (8 * tw);
    const int cand[4] = {32, 28, 24, 16};
    int th = 0;
    for (int i = 0; i < 4; ++i)
        if (cand[i] % rg == 0 && (th == 0 || padded(g.H_out, cand[i]) < padded(g.H_out, th))) th = cand[i];
    for (;;) {
        const int in_h = (th - 1) * g.S + (g.Kh - 1) * g.D + 1;
        const int in_w = (tw - 1) * g.S + (g.Kw - 1) * g.D + 1;
        const long long stage = static_cast<long long>(in_h) * in_w * kDwChannels * 4;
        long long stages = (smem_optin - 1024 - 128) / stage;
        if (stages > 8) stages = 8;
        if (in_h <= 256 && in_w <= 256 && (stages >= 2 || (th <= rg && stages >= 1))) {
            d.tile_w = tw;
            d.tile_h = th;
            d.in_h = in_h;
            d.in_w = in_w;
            d.stages = static_cast<int>(stages);
            d.smem_bytes = static_cast<int>(stages * stage + 128);
            break;
        }
        if (th <= rg) return 0;
        th = th / 2 >= rg ? (th / 2) / rg * rg : rg;
    }
    d.tiles_h = (g.H_out + d.tile_h - 1) / d.tile_h;
    d.tiles_w = (g.W_out + d.tile_w - 1) / d.tile_w;
    d.cblocks = g.C_in / kDwChannels;
    const long long tiles = static_cast<long long>(g.N) * d.tiles_h * d.tiles_w * d.cblocks;
    if (tiles > 0x7fffffffLL) return 0;
    d.num_tiles = static_cast<int>(tiles);
    return 1;
}

template <int K, int TW>
static cudaError_t launch_dw(const CUtensorMap& x_map, const DepthwiseParams& p, int grid, cudaStream_t stream) {
    cudaError_t e =
        cudaFuncSetAttribute(depthwise_kernel<K, TW>, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess) return e;
    depthwise_kernel<K, TW><<<grid, kDwThreads, p.smem_bytes, stream>>>(x_map, p);
    return cudaGetLastError();
}

cudaError_t launch_depthwise(const CUtensorMap& x_map, const DepthwiseParams& p, int grid, cudaStream_t stream) {
    const bool k3 = p.g.Kh == 3 && p.g.Kw == 3;
    if (p.tile_w == 8) return k3 ? launch_dw<3, 8>(x_map, p, grid, stream) : launch_dw<0, 8>(x_map, p, grid, stream);
    return k3 ? launch_dw<3, 16>(x_map, p, grid, stream) : launch_dw<0, 16>(x_map, p, grid, stream);
}

}  // namespace convgb
