// winograd.cu -- FP32 3x3 stride-1 convolution by Winograd's minimal filtering
// F(2x2, 3x3) on CUDA cores.
//
// "Convolution vs inner product" (lnrq.cn/news/4475), section 2.2, and
// "Convolution variants and their matrix operations" (lpnh.cn/news/2674933),
// section 3.3: a 4x4 input tile d and a 3x3 kernel g are mapped to a 4x4
// transformed space, V = B^T d B and U = G g G^T; 16 element-wise products
// (summed over input channels) M = sum_c U * V give a 2x2 output tile
// Y = A^T M A.  That is 4 multiplies per output instead of 9.  The transform
// matrices are those of polynomial interpolation at 0, 1, -1 and infinity (the
// published F(2x2, 3x3) of Lavin and Gray):
//   B^T = [1 0 -1 0; 0 1 1 0; 0 -1 1 0; 0 1 0 -1]
//   G   = [1 0 0; 1/2 1/2 1/2; 1/2 -1/2 1/2; 0 0 1]
//   A^T = [1 1 1 0; 0 1 -1 -1]
// The pages warn that it costs precision; the library runs it only on request
// (CONV_FLAG_WINOGRAD).  On this part the multiplies are what an FP32 direct
// convolution spends its time on, so that is where it applies; BF16 layers
// run on the tensor cores, where a transformed-space GEMM would move 4x the
// data for fewer, narrower MMAs.
//
// CTA: 4 x 8 Winograd tiles (8 x 16 outputs) of one image x 32 output
// channels, 256 threads, input channels in chunks of 16:
//   1. the 10 x 18 input patch of the chunk into shared memory (zero outside
//      the image: the padding) by asynchronous copies issued during the
//      previous chunk's products, into the other of two patch buffers;
//   2. thread (tile, channel) computes V = B^T d B; thread (filter, channel)
//      computes U = G g G^T;
//   3. thread (component xi of 16, 8 tiles, 8 filters) accumulates its 8 x 8
//      block of M[xi] over the chunk: 64 FMAs (32 packed pairs) per 16 shared loads;
// then the 16 components of each (tile, filter) meet in shared memory and
// thread (tile, filter) computes Y = A^T M A, scale, bias, ReLU and stores.
#include "conv_internal.h"
#include "fp32x2.cuh"
#include "ptx.cuh"

namespace convgb {

namespace {

constexpr int kWgTilesH = 4, kWgTilesW = 8;                    // Winograd tiles per CTA
constexpr int kWgTiles = kWgTilesH * kWgTilesW;                // 32
constexpr int kWgCo = 32;                                      // output channels per CTA
constexpr int kWgCi = 16;                                      // input channels per chunk
constexpr int kWgPatchH = 2 * kWgTilesH + 2, kWgPatchW = 2 * kWgTilesW + 2;  // 10 x 18 inputs
constexpr int kWgRow = 36;                                     // floats per (component, channel) row (32 + skew)
constexpr int kWgMStride = 33;                                 // floats per tile row of M (32 + skew)
constexpr int kWgPatchFloats = kWgCi * kWgPatchH * kWgPatchW;  // 1440
constexpr int kWgVFloats = 16 * kWgCi * kWgRow;                // 4608
constexpr int kWgMFloats = 16 * kWgTiles * kWgMStride;         // 16896
constexpr int kWgSmemFloats =
    kWgMFloats > 2 * kWgPatchFloats + 2 * kWgVFloats ? kWgMFloats : 2 * kWgPatchFloats + 2 * kWgVFloats;

// 4-byte asynchronous global -> shared copy; an invalid source reads nothing and fills zero.
__device__ __forceinline__ void cp_async_f32(float* dst, const float* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <typename Tout>
__global__ void __launch_bounds__(kWgThreads, 2) winograd_kernel(const WinogradParams p) {
    extern __shared__ __align__(16) float smem[];  // kWgSmemFloats
    float* patch = smem;                   // two buffers of [ci][10][18]
    float* Vs = smem + 2 * kWgPatchFloats; // [16][ci][kWgRow]: tiles
    float* Us = Vs + kWgVFloats;           // [16][ci][kWgRow]: filters
    float* Ms = smem;                      // after the channel loop: [16][tile][kWgMStride]

    const ConvGeom& g = p.g;
    const int tid = threadIdx.x;
    const int tiles_w = (g.W_out + 1) / 2, tiles_h = (g.H_out + 1) / 2;
    const int blocks_w = (tiles_w + kWgTilesW - 1) / kWgTilesW;
    const int blocks_h = (tiles_h + kWgTilesH - 1) / kWgTilesH;
    int b = blockIdx.x;
    const int bw = b % blocks_w;
    b /= blocks_w;
    const int bh = b % blocks_h;
    const int n = b / blocks_h;
    const int co0 = blockIdx.y * kWgCo;
    const int in_h0 = 2 * kWgTilesH * bh - g.P, in_w0 = 2 * kWgTilesW * bw - g.P;

    // product-phase roles: component xi, 8 tiles (tg), 8 filters (cg)
    const int xi = tid >> 4, tg = (tid >> 2) & 3, cg = tid & 3;
    const int skew = (xi & 1) * 4;  // the two components of a warp read different banks
    unsigned long long acc2[8][4];  // filter pairs {2c, 2c+1} of each tile
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc2[a][c] = 0ull;

    const float* x = static_cast<const float*>(p.x);
    const float* w = static_cast<const float*>(p.w);
    // patch element e = tid + i * kWgThreads: channel e % kWgCi of patch pixel e / kWgCi
    constexpr int kPatchCopies = (kWgPatchFloats + kWgThreads - 1) / kWgThreads;
    auto issue_patch = [&](int c0, float* dst) {
#pragma unroll 1
        for (int i = 0; i < kPatchCopies; ++i) {
            const int e = tid + i * kWgThreads;
            if (e >= kWgPatchFloats) break;
            const int ci = e % kWgCi, pix = e / kWgCi;
            const int r = pix / kWgPatchW, q = pix - r * kWgPatchW;
            const int h = in_h0 + r, ww = in_w0 + q, c = c0 + ci;
            const bool ok = h >= 0 && h < g.H && ww >= 0 && ww < g.W && c < g.C_in;
            const float* src = ok ? x + ((static_cast<long long>(n) * g.H + h) * g.W + ww) * g.C_in + c : x;
            cp_async_f32(dst + ci * (kWgPatchH * kWgPatchW) + pix, src, ok);
        }
    };
    issue_patch(0, patch);
    cp_async_commit_wait_all();
    __syncthreads();
    for (int c0 = 0, pb = 0; c0 < g.C_in; c0 += kWgCi, pb ^= 1) {
        const float* cur = patch + pb * kWgPatchFloats;
        // 2b. U = G g G^T for (filter, channel) pairs; weights [C_out][3][3][C_in],
        // channel fastest across threads so a warp reads 32-byte runs
#pragma unroll 1
        for (int half = 0; half < kWgCi / 8; ++half) {
            const int f = tid >> 3, ci = (tid & 7) + 8 * half;
            const int co = co0 + f, c = c0 + ci;
            float gg[3][3], t[4][3];
#pragma unroll
            for (int i = 0; i < 3; ++i)
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    gg[i][j] = (co < g.C_out && c < g.C_in) ? __ldg(w + (static_cast<long long>(co) * 9 + i * 3 + j) *
                                                                          g.C_in + c)
                                                            : 0.f;
#pragma unroll
            for (int j = 0; j < 3; ++j) {  // rows: G g
                t[0][j] = gg[0][j];
                t[1][j] = 0.5f * (gg[0][j] + gg[1][j] + gg[2][j]);
                t[2][j] = 0.5f * (gg[0][j] - gg[1][j] + gg[2][j]);
                t[3][j] = gg[2][j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // columns: (G g) G^T
                const float u0 = t[i][0], u1 = 0.5f * (t[i][0] + t[i][1] + t[i][2]);
                const float u2 = 0.5f * (t[i][0] - t[i][1] + t[i][2]), u3 = t[i][2];
                const int k = 4 * i;
                Us[((k + 0) * kWgCi + ci) * kWgRow + ((k + 0) & 1) * 4 + f] = u0;
                Us[((k + 1) * kWgCi + ci) * kWgRow + ((k + 1) & 1) * 4 + f] = u1;
                Us[((k + 2) * kWgCi + ci) * kWgRow + ((k + 2) & 1) * 4 + f] = u2;
                Us[((k + 3) * kWgCi + ci) * kWgRow + ((k + 3) & 1) * 4 + f] = u3;
            }
        }
        __syncthreads();
        // 2a. V = B^T d B for (tile, channel) pairs
#pragma unroll 1
        for (int half = 0; half < kWgCi / 8; ++half) {
            const int t = tid & 31, ci = (tid >> 5) + 8 * half;
            const int lh = t / kWgTilesW, lw = t - lh * kWgTilesW;
            const float* d0 = cur + ci * (kWgPatchH * kWgPatchW) + (2 * lh) * kWgPatchW + 2 * lw;
            float d[4][4], u[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) d[i][j] = d0[i * kWgPatchW + j];
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // rows: B^T d
                u[0][j] = d[0][j] - d[2][j];
                u[1][j] = d[1][j] + d[2][j];
                u[2][j] = d[2][j] - d[1][j];
                u[3][j] = d[1][j] - d[3][j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // columns: (B^T d) B
                const float v0 = u[i][0] - u[i][2], v1 = u[i][1] + u[i][2];
                const float v2 = u[i][2] - u[i][1], v3 = u[i][1] - u[i][3];
                const int k = 4 * i;
                Vs[((k + 0) * kWgCi + ci) * kWgRow + ((k + 0) & 1) * 4 + t] = v0;
                Vs[((k + 1) * kWgCi + ci) * kWgRow + ((k + 1) & 1) * 4 + t] = v1;
                Vs[((k + 2) * kWgCi + ci) * kWgRow + ((k + 2) & 1) * 4 + t] = v2;
                Vs[((k + 3) * kWgCi + ci) * kWgRow + ((k + 3) & 1) * 4 + t] = v3;
            }
        }
        __syncthreads();
        // the next chunk's patch copies are in flight during the products
        if (c0 + kWgCi < g.C_in) {
            issue_patch(c0 + kWgCi, patch + (pb ^ 1) * kWgPatchFloats);
            cp_async_commit();
        }
        // 3. M[xi] += V[xi] (8 tiles) x U[xi] (8 filters) over the chunk's channels
#pragma unroll
        for (int ci = 0; ci < kWgCi; ++ci) {
            const float4* vp = reinterpret_cast<const float4*>(Vs + (xi * kWgCi + ci) * kWgRow + skew + 8 * tg);
            const float4* up = reinterpret_cast<const float4*>(Us + (xi * kWgCi + ci) * kWgRow + skew + 8 * cg);
            const float4 va = vp[0], vb = vp[1], ua = up[0], ub = up[1];
            const float v[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
            const unsigned long long u2[4] = {f32x2_pack(ua.x, ua.y), f32x2_pack(ua.z, ua.w), f32x2_pack(ub.x, ub.y),
                                              f32x2_pack(ub.z, ub.w)};
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const unsigned long long va2 = f32x2_dup(v[a]);
#pragma unroll
                for (int c = 0; c < 4; ++c) f32x2_fma(acc2[a][c], va2, u2[c]);
            }
        }
        cp_async_commit_wait_all();
        __syncthreads();  // the next patch has landed; the next chunk overwrites V and U
    }

    // the 16 components of every (tile, filter) into shared memory
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float* m = Ms + (xi * kWgTiles + 8 * tg + a) * kWgMStride + 8 * cg + 2 * c;
            f32x2_unpack(acc2[a][c], m[0], m[1]);
        }
    __syncthreads();

    // Y = A^T M A, then scale, bias, ReLU; thread = (tile, filter), filters fastest
    Tout* y = static_cast<Tout*>(p.y);
    for (int pr = tid; pr < kWgTiles * kWgCo; pr += kWgThreads) {
        const int f = pr % kWgCo, t = pr / kWgCo;
        const int co = co0 + f;
        const int lh = t / kWgTilesW, lw = t - lh * kWgTilesW;
        const int ho = 2 * (kWgTilesH * bh + lh), wo = 2 * (kWgTilesW * bw + lw);
        if (co >= g.C_out || ho >= g.H_out || wo >= g.W_out) continue;
        float m[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) m[i][j] = Ms[((4 * i + j) * kWgTiles + t) * kWgMStride + f];
        float r[2][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // rows: A^T M
            r[0][j] = m[0][j] + m[1][j] + m[2][j];
            r[1][j] = m[1][j] - m[2][j] - m[3][j];
        }
        const float sc = p.scale ? __ldg(p.scale + co) : 1.f;
        const float bi = p.bias ? __ldg(p.bias + co) : 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int h = ho + i, ww = wo + j;
                if (h >= g.H_out || ww >= g.W_out) continue;
                float v = j == 0 ? r[i][0] + r[i][1] + r[i][2] : r[i][1] - r[i][2] - r[i][3];  // (A^T M) A
                if (p.scale) v *= sc;
                if (p.bias) v += bi;
                if (p.relu) v = fmaxf(v, 0.f);
                const long long o = ((static_cast<long long>(n) * g.H_out + h) * g.W_out + ww) * g.C_out + co;
                if constexpr (sizeof(Tout) == 2)
                    y[o] = __float2bfloat16_rn(v);
                else
                    y[o] = v;
            }
        }
    }
}

}  // namespace

bool winograd_supported(const ConvGeom& g) {
    return g.Kh == 3 && g.Kw == 3 && g.S == 1 && g.D == 1 && g.G == 1 && g.H_out >= 1 && g.W_out >= 1;
}

void winograd_grid(const ConvGeom& g, unsigned& gx, unsigned& gy) {
    const long long tiles_w = (g.W_out + 1) / 2, tiles_h = (g.H_out + 1) / 2;
    const long long blocks = static_cast<long long>(g.N) * ((tiles_h + kWgTilesH - 1) / kWgTilesH) *
                             ((tiles_w + kWgTilesW - 1) / kWgTilesW);
    gx = static_cast<unsigned>(blocks);
    gy = static_cast<unsigned>((g.C_out + kWgCo - 1) / kWgCo);
}

int winograd_smem_bytes() { return kWgSmemFloats * 4; }

cudaError_t launch_winograd(const WinogradParams& p, cudaStream_t stream) {
    unsigned gx, gy;
    winograd_grid(p.g, gx, gy);
    const int smem = winograd_smem_bytes();
    static SmemLimitCache limits_f32, limits_bf16;
    cudaError_t e;
    if (p.out_bf16) {
        e = ensure_smem_limit(reinterpret_cast<const void*>(winograd_kernel<__nv_bfloat16>), smem, limits_bf16);
        if (e != cudaSuccess) return e;
        winograd_kernel<__nv_bfloat16><<<dim3(gx, gy), kWgThreads, smem, stream>>>(p);
    } else {
        e = ensure_smem_limit(reinterpret_cast<const void*>(winograd_kernel<float>), smem, limits_f32);
        if (e != cudaSuccess) return e;
        winograd_kernel<float><<<dim3(gx, gy), kWgThreads, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace convgb
