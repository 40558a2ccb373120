// conv_internal.h -- parameter blocks and launchers shared between the plan
// code (conv_api.cu) and the kernel translation units.  Not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace convgb {

// Geometry of one convolution (NHWC activations, [C_out][Kh][Kw][C_in/G] weights).
struct ConvGeom {
    int N, C_in, H, W, C_out, Kh, Kw, S, P, D, G;
    int H_out, W_out;
    int cin_g, cout_g;
    long long pixels;  // N * H_out * W_out
};

// ---------------------------------------------------------------- direct (CUDA cores)
struct DirectParams {
    ConvGeom g;
    const void* x;
    const void* w;
    const float* bias;  // nullptr when no bias
    void* y;
    int relu;
    int in_bf16;   // x, w are BF16 (else FP32)
    int out_bf16;  // y is BF16 (else FP32)
};
cudaError_t launch_direct(const DirectParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- depthwise (FP32, TMA halo tile)
struct DepthwiseParams {
    ConvGeom g;
    const float* w;     // [C][Kh][Kw]
    const float* bias;  // nullptr when no bias
    void* y;
    int relu;
    int out_bf16;
    int tile;           // output tile edge (tile x tile pixels) per CTA
    int tiles_h, tiles_w, cblocks;
    int in_h, in_w;     // halo box extent
    unsigned* status;
};
// Box {32 channels, in_w, in_h, 1} of the 4-D NHWC map; 0 if the shape is not supported.
int depthwise_tile_for(const ConvGeom& g);
cudaError_t launch_depthwise(const CUtensorMap& x_map, const DepthwiseParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- tcgen05 GEMM (1x1 and implicit)
constexpr int kTcBlockM = 128;    // pixels per tile (TMEM lanes)
constexpr int kTcBlockK = 64;     // BF16 elements per K-step (one 128-byte swizzle row)
constexpr int kTcThreads = 192;   // producer warp, MMA warp, 4 epilogue warps

enum TcMode { kTcMode1x1 = 0, kTcModeIm2col = 1 };

struct TcGemmParams {
    ConvGeom g;
    int mode;          // TcMode
    int n_tile;        // accumulator columns per tile (<= 256)
    int mma_n;         // N of each MMA (<= 256, multiple of 16)
    int gpc;           // sub-GEMMs (groups, or a slice of one group) per tile
    int kblk;          // (C_in/G) / 64
    int ksteps;        // Kh * Kw * kblk K-steps per sub-GEMM
    int num_m_tiles, num_n_tiles, num_tiles;
    int stages;
    int tmem_cols;     // power of two >= 2 * n_tile
    int smem_bytes;
    int relu;
    const float* bias;
    __nv_bfloat16* y;
    unsigned* status;
};
cudaError_t launch_tc_gemm(const CUtensorMap& a_map, const CUtensorMap& b_map, const TcGemmParams& p, int grid,
                           cudaStream_t stream);

// ---------------------------------------------------------------- tcgen05 small-K (stem)
constexpr int kSkThreads = 320;   // producer, MMA, 4 epilogue, 4 transform warps

struct SmallKParams {
    ConvGeom g;
    const __nv_bfloat16* x;
    const __nv_bfloat16* w;   // [C_out][Ktot]
    const float* bias;
    __nv_bfloat16* y;
    int relu;
    int ktot;          // C_in * Kh * Kw  (<= 64)
    int kmma;          // number of K=16 MMAs (ceil(ktot / 16))
    int segs;          // 128-pixel segments per output row
    int num_tiles;
    int row_bytes;     // W * C_in * 2
    int raw_bytes;     // Kh * row_bytes rounded up to 1024
    int stages;
    int tmem_cols;
    int smem_bytes;
    unsigned* status;
};
cudaError_t launch_tc_smallk(const SmallKParams& p, int grid, cudaStream_t stream);

}  // namespace convgb
