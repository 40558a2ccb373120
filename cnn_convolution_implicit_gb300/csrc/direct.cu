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
// Layers with at least 32 output channels per group take a register-tiled
// form of the same sums (lesson 9, section 11: output-stationary tiling with
// the operands staged in shared memory): a CTA owns 64 or 128 output pixels x
// 64 output channels of one group, each thread 8 pixels x 4 channels in
// registers; the reduction runs tap by tap in chunks of 16 input channels,
// double-buffered in shared memory, so every staged input value feeds 64 FMAs
// of its CTA and every staged weight 64 or 128.
//
// Transposed convolution ("Convolution variants and their matrix operations",
// lpnh.cn/news/2674933, sections 2.3 and 4.2: the adjoint of the convolution,
// each input pixel (i, j) contributing to output (i*S + kh*D - P,
// j*S + kw*D - P)) runs here in gather form: output (ho, wo) takes input row
// i = (ho + P - kh*D) / S for every kernel row kh where the division is exact
// and i is inside the input, likewise for columns.
#include "conv_internal.h"
#include "fp32x2.cuh"
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

// Input element (n, hi, wi) of the tap (kh, kw) for output (ho, wo), forward
// or transposed (gather form); false where it falls in the padding or, for the
// transposed form, where the division by the stride is not exact.
__device__ __forceinline__ bool source_pixel(const ConvGeom& g, bool transposed, int ho, int wo, int kh, int kw,
                                             int& hi, int& wi) {
    if (!transposed) {
        hi = ho * g.S + kh * g.D - g.P;
        wi = wo * g.S + kw * g.D - g.P;
        return hi >= 0 && hi < g.H && wi >= 0 && wi < g.W;
    }
    const int nh = ho + g.P - kh * g.D, nw = wo + g.P - kw * g.D;
    if (nh < 0 || nw < 0 || nh % g.S != 0 || nw % g.S != 0) return false;
    hi = nh / g.S;
    wi = nw / g.S;
    return hi < g.H && wi < g.W;
}

// Four consecutive channels [c, c + 4) of one input pixel (zero past `limit`).
template <typename Tin>
__device__ __forceinline__ void load4(const Tin* src, int c, int limit, bool vec, float (&r)[4]) {
    if (src != nullptr && vec && c + 4 <= limit) {
        if constexpr (sizeof(Tin) == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src + c);
            r[0] = v.x;
            r[1] = v.y;
            r[2] = v.z;
            r[3] = v.w;
        } else {
            const uint2 v = *reinterpret_cast<const uint2*>(src + c);
            r[0] = __uint_as_float(v.x << 16);
            r[1] = __uint_as_float(v.x & 0xffff0000u);
            r[2] = __uint_as_float(v.y << 16);
            r[3] = __uint_as_float(v.y & 0xffff0000u);
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = (src != nullptr && c + i < limit) ? to_f32(src[c + i]) : 0.f;
}

template <typename Tin, typename Tout, int BM>
__global__ void __launch_bounds__(2 * BM) direct_tiled_kernel(const DirectParams p, const int vec_x, const int vec_y) {
    constexpr int kThreads = 2 * BM;
    constexpr int kPitchA = BM + 4;        // row pitch (floats): the two loader halves land 16 banks apart
    constexpr int kPitchB = kDtTileN + 4;  // the 8 rows of one warp's weight stores land 4 banks apart
    constexpr int kBLoads = kDtTileN * kDtChunk / kThreads;
    constexpr int kALoads = kDtChunk / 2;  // channels of the chunk each loader thread fetches
    __shared__ __align__(16) float As[2][kDtChunk][kPitchA];
    __shared__ __align__(16) float Bs[2][kDtChunk][kPitchB];
    const ConvGeom& g = p.g;
    const Tin* x = static_cast<const Tin*>(p.x);
    const Tin* w = static_cast<const Tin*>(p.w);
    Tout* y = static_cast<Tout*>(p.y);
    const int tid = threadIdx.x;
    const long long pix0 = static_cast<long long>(blockIdx.x) * BM;
    const int co_blocks = (g.cout_g + kDtTileN - 1) / kDtTileN;
    const int grp = blockIdx.y / co_blocks;
    const int cb0 = (blockIdx.y - grp * co_blocks) * kDtTileN;  // first output channel (within the group)

    // loader role: one pixel of the tile, half of the chunk's channels
    const int lp = tid >> 1;
    const int lc = (tid & 1) * kALoads;
    const long long lpix = pix0 + lp;
    const bool lpix_ok = lpix < g.pixels;
    int ln = 0, lho = 0, lwo = 0;
    if (lpix_ok) {
        lwo = static_cast<int>(lpix % g.W_out);
        const long long t = lpix / g.W_out;
        lho = static_cast<int>(t % g.H_out);
        ln = static_cast<int>(t / g.H_out);
    }
    const Tin* xg = x + static_cast<long long>(grp) * g.cin_g;
    const long long w_per_co = static_cast<long long>(g.Kh) * g.Kw * g.cin_g;
    const Tin* wg = w + static_cast<long long>(grp) * g.cout_g * w_per_co;

    float ra[kALoads], rb[kBLoads];
    auto fetch = [&](int kh, int kw, int ci0) {
        const Tin* src = nullptr;
        int hi, wi;
        if (lpix_ok && source_pixel(g, p.transposed != 0, lho, lwo, kh, kw, hi, wi))
            src = xg + ((static_cast<long long>(ln) * g.H + hi) * g.W + wi) * g.C_in;
#pragma unroll
        for (int i = 0; i < kALoads; i += 4)
            load4(src, ci0 + lc + i, g.cin_g, vec_x != 0, *reinterpret_cast<float(*)[4]>(ra + i));
        const int tap = kh * g.Kw + kw;
#pragma unroll
        for (int i = 0; i < kBLoads; ++i) {
            const int e = tid + i * kThreads;
            const int co = cb0 + e / kDtChunk, ci = ci0 + e % kDtChunk;
            rb[i] = (co < g.cout_g && ci < g.cin_g) ? to_f32(wg[co * w_per_co + tap * g.cin_g + ci]) : 0.f;
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int i = 0; i < kALoads; ++i) As[buf][lc + i][lp] = ra[i];
#pragma unroll
        for (int i = 0; i < kBLoads; ++i) {
            const int e = tid + i * kThreads;
            Bs[buf][e % kDtChunk][e / kDtChunk] = rb[i];
        }
    };

    // compute role: pixels [ty*8, ty*8 + 8) x channels [tx*4, tx*4 + 4) of the tile
    const int tx = tid & 15, ty = tid >> 4;
    unsigned long long acc2[8][2];  // channel pairs {4tx, 4tx+1}, {4tx+2, 4tx+3} of each pixel
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[i][0] = acc2[i][1] = 0ull;

    const int chunks_per_tap = (g.cin_g + kDtChunk - 1) / kDtChunk;
    const int nchunks = g.Kh * g.Kw * chunks_per_tap;
    int kh = 0, kw = 0, ci0 = 0;  // running position of the next chunk to fetch
    auto advance = [&]() {
        ci0 += kDtChunk;
        if (ci0 >= g.cin_g) {
            ci0 = 0;
            if (++kw == g.Kw) {
                kw = 0;
                ++kh;
            }
        }
    };
    fetch(kh, kw, ci0);
    advance();
    stash(0);
    __syncthreads();
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c & 1;
        const bool more = c + 1 < nchunks;
        if (more) {  // next chunk's global loads in flight during this chunk's FMAs
            fetch(kh, kw, ci0);
            advance();
        }
#pragma unroll
        for (int k = 0; k < kDtChunk; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 8]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 8 + 4]);
            const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const unsigned long long b01 = f32x2_pack(b.x, b.y), b23 = f32x2_pack(b.z, b.w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const unsigned long long ai = f32x2_dup(av[i]);
                f32x2_fma(acc2[i][0], ai, b01);
                f32x2_fma(acc2[i][1], ai, b23);
            }
        }
        if (more) stash(buf ^ 1);
        __syncthreads();
    }

    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f32x2_unpack(acc2[i][0], acc[i][0], acc[i][1]);
        f32x2_unpack(acc2[i][1], acc[i][2], acc[i][3]);
    }
    // epilogue: scale, bias, ReLU, NHWC store of 4 consecutive channels per pixel
    const int co = cb0 + tx * 4;
    if (co >= g.cout_g) return;
    const int cabs = grp * g.cout_g + co;
    float sc[4], bi[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const bool ok = co + j < g.cout_g;
        sc[j] = (p.scale && ok) ? p.scale[cabs + j] : 1.f;
        bi[j] = (p.bias && ok) ? p.bias[cabs + j] : 0.f;
    }
    const bool full4 = vec_y != 0 && co + 4 <= g.cout_g;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const long long pix = pix0 + ty * 8 + i;
        if (pix >= g.pixels) break;
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[j] = p.scale ? acc[i][j] * sc[j] : acc[i][j];
            v[j] += bi[j];
            if (p.relu) v[j] = fmaxf(v[j], 0.f);
        }
        Tout* yp = y + pix * g.C_out + cabs;
        if (full4) {
            if constexpr (sizeof(Tout) == 4) {
                *reinterpret_cast<float4*>(yp) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
                uint2 u;
                u.x = *reinterpret_cast<const uint32_t*>(&lo);
                u.y = *reinterpret_cast<const uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(yp) = u;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (co + j >= g.cout_g) break;
                if constexpr (sizeof(Tout) == 4)
                    yp[j] = v[j];
                else
                    yp[j] = __float2bfloat16_rn(v[j]);
            }
        }
    }
}

void direct_shape(const ConvGeom& g, int num_sms, int& tile_m, unsigned& gx, unsigned& gy, int& block) {
    const long long co_blocks = (g.cout_g + kDtTileN - 1) / kDtTileN;
    const long long ny = static_cast<long long>(g.G) * co_blocks;
    if (g.cout_g >= 32 && ny <= 65535 && g.pixels > 0) {
        // 128 pixels per CTA unless that leaves fewer than two CTAs per SM
        const long long ctas128 = (g.pixels + 127) / 128 * ny;
        tile_m = ctas128 >= 2LL * num_sms ? 128 : 64;
        const long long nx = (g.pixels + tile_m - 1) / tile_m;
        if (nx <= 0x7fffffffLL) {
            gx = static_cast<unsigned>(nx);
            gy = static_cast<unsigned>(ny);
            block = 2 * tile_m;
            return;
        }
    }
    tile_m = 0;
    const long long total = g.pixels * g.C_out;
    const long long blocks = (total + 255) / 256;
    gx = static_cast<unsigned>(blocks < (1ll << 20) ? blocks : (1ll << 20));
    gy = 1;
    block = 256;
}

template <typename Tin, typename Tout>
static void launch_direct_typed(const DirectParams& p, unsigned gx, unsigned gy, int vec_x, int vec_y,
                                cudaStream_t stream) {
    if (p.tile_m == 128)
        direct_tiled_kernel<Tin, Tout, 128><<<dim3(gx, gy), 256, 0, stream>>>(p, vec_x, vec_y);
    else if (p.tile_m == 64)
        direct_tiled_kernel<Tin, Tout, 64><<<dim3(gx, gy), 128, 0, stream>>>(p, vec_x, vec_y);
    else
        direct_kernel<Tin, Tout><<<gx, 256, 0, stream>>>(p);
}

cudaError_t launch_direct(const DirectParams& p, int num_sms, cudaStream_t stream) {
    if (p.g.pixels == 0 || p.g.C_out == 0) return cudaSuccess;
    int tile_m = 0, block = 0;
    unsigned gx = 0, gy = 0;
    direct_shape(p.g, num_sms, tile_m, gx, gy, block);
    DirectParams q = p;
    q.tile_m = tile_m;
    // vector accesses: 4 channels per load / store where every such run is aligned
    const unsigned in_align = p.in_bf16 ? 8u : 16u, out_align = p.out_bf16 ? 8u : 16u;
    const int vec_x = (p.g.C_in % 4 == 0 && p.g.cin_g % 4 == 0 &&
                       reinterpret_cast<uintptr_t>(p.x) % in_align == 0) ? 1 : 0;
    const int vec_y = (p.g.C_out % 4 == 0 && p.g.cout_g % 4 == 0 &&
                       reinterpret_cast<uintptr_t>(p.y) % out_align == 0) ? 1 : 0;
    if (p.in_bf16)
        launch_direct_typed<__nv_bfloat16, __nv_bfloat16>(q, gx, gy, vec_x, vec_y, stream);
    else if (p.out_bf16)
        launch_direct_typed<float, __nv_bfloat16>(q, gx, gy, vec_x, vec_y, stream);
    else
        launch_direct_typed<float, float>(q, gx, gy, vec_x, vec_y, stream);
    return cudaGetLastError();
}

}  // namespace convgb
