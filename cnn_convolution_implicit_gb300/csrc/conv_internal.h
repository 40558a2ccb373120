// conv_internal.h -- parameter blocks and launchers shared between the plan
// code (conv_api.cu) and the kernel translation units.  Not part of the ABI.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace convgb {

// Per-device dynamic shared-memory limit already set on one kernel (zero-initialised
// when declared static; atomic, so plans driven from different host threads may
// launch the same kernel concurrently).
using SmemLimitCache = std::atomic<int>[64];

// Raise a kernel's dynamic shared-memory limit only when a launch needs more
// than what was set before on this device (`limits` is the caller's per-kernel
// cache).  The limit is a per-function attribute, so a plan's later launches
// cost no extra runtime call.  Concurrent first calls may both set it: harmless,
// and the cache only ever grows.
inline cudaError_t ensure_smem_limit(const void* func, int bytes, SmemLimitCache& limits) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    }
    if (limits[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) {
        int cur = limits[dev].load(std::memory_order_relaxed);
        while (cur < bytes && !limits[dev].compare_exchange_weak(cur, bytes, std::memory_order_relaxed)) {
        }
    }
    return e;
}

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
    const float* bias;   // nullptr when no bias
    const float* scale;  // nullptr when no per-channel scale
    void* y;
    int relu;
    int in_bf16;     // x, w are BF16 (else FP32)
    int out_bf16;    // y is BF16 (else FP32)
    int transposed;  // transposed convolution (gather form): x is the H x W input, y the H_out x W_out output
    int tile_m;      // 0: one thread per output; 64 or 128: register-tiled kernel with that many pixels per CTA
};
// Register-tiled direct kernel: a CTA computes kDtTileN output channels of one
// group for tile_m output pixels, the reduction in chunks of kDtChunk channels of one tap.
constexpr int kDtTileN = 64;
constexpr int kDtChunk = 16;
// Launch shape of the direct path: tile_m as above, the grid and block size.
void direct_shape(const ConvGeom& g, int num_sms, int& tile_m, unsigned& gx, unsigned& gy, int& block);
cudaError_t launch_direct(const DirectParams& p, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- Winograd F(2x2, 3x3) (FP32)
constexpr int kWgThreads = 256;
struct WinogradParams {
    ConvGeom g;           // 3x3, S = 1, D = 1, G = 1
    const void* x;        // FP32 NHWC
    const void* w;        // FP32 [C_out][3][3][C_in]
    const float* bias;    // nullptr when no bias
    const float* scale;   // nullptr when no per-channel scale
    void* y;
    int relu;
    int out_bf16;
};
bool winograd_supported(const ConvGeom& g);
void winograd_grid(const ConvGeom& g, unsigned& gx, unsigned& gy);
int winograd_smem_bytes();
cudaError_t launch_winograd(const WinogradParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- depthwise (FP32, TMA halo tile)
struct DepthwiseParams {
    ConvGeom g;
    const float* w;      // [C][Kh][Kw]
    const float* bias;   // nullptr when no bias
    const float* scale;  // nullptr when no per-channel scale
    void* y;
    int relu;
    int out_bf16;
    int tile_h, tile_w;  // output pixels per tile (32 channels each)
    int tiles_h, tiles_w, cblocks, num_tiles;
    int in_h, in_w;      // halo box extent (TMA box {32, in_w, in_h, 1})
    int stages;          // halo tiles in flight per CTA (<= 8)
    int smem_bytes;
    int fixed_cb;        // each CTA keeps one channel block (grid a multiple of cblocks)
    int grid;
    unsigned* status;
};
// Fills the tiling fields of d; returns 0 if the shape does not fit the kernel.
int depthwise_config(const ConvGeom& g, int smem_per_sm, int num_sms, DepthwiseParams& d);
cudaError_t launch_depthwise(const CUtensorMap& x_map, const DepthwiseParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- tcgen05 GEMM (1x1 and implicit)
constexpr int kTcBlockM = 128;    // pixels per tile (TMEM lanes)
constexpr int kTcBlockK = 64;     // BF16 elements per K-step (one 128-byte swizzle row)
constexpr int kTcThreads = 576;   // producer warp, MMA warp, 4 x 4 epilogue warps
constexpr int kTcHaloThreads = 608;  // halo mode: + a weight producer warp (the halo producer is warp 0)
constexpr int kTcBWarp = 18;      // halo mode: the weight (B operand) producer warp
// Two pixel tiles per CTA: a second MMA-issuing warp (tile 1's MMAs; warp 1 issues tile 0's)
// after the other warps: warp 18, or 19 in halo mode.
__host__ __device__ constexpr int tc_mma2_warp(bool halo) { return halo ? 19 : 18; }
__host__ __device__ constexpr int tc_threads(bool halo, bool dual) {
    return (halo ? kTcHaloThreads : kTcThreads) + (dual ? 32 : 0);
}
constexpr int kTcMaxGroupsPerTile = 8;  // groups packed side by side in one accumulator (<= ring stages)

enum TcMode { kTcMode1x1 = 0, kTcModeIm2col = 1, kTcModeRect = 2, kTcModePhase = 3, kTcModeHalo = 4 };

// kTcModeHalo (stride 1): pixel tiles are 8 wide x 16 high, so each 8-row core-matrix
// group of the MMA's A operand is one output row segment.  One TMA box per 64-channel
// block brings the tile's input halo (kTcHaloTileW + (Kw-1)*D) x (16 + (Kh-1)*D) pixels
// (x2 wide for two tiles per CTA) into shared memory, and every tap (kh, kw) reads it
// through a descriptor whose start is shifted by kh*D*halo_w + kw*D pixel rows and
// whose 8-row stride is halo_w rows.
constexpr int kTcHaloTileW = 8;
constexpr int kTcHaloTileH = 16;
constexpr int kTcMaxHaloStages = 4;

// Transposed convolution (kTcModePhase, any stride S): output pixels split into
// S x S phases by (h mod S, w mod S); phase residue r of one axis uses the kernel
// taps k with (r + P - k*D) divisible by S, reading input row (q + off) for phase
// row q, off = (r + P - k*D) / S.
constexpr int kTcMaxPhaseStride = 4;
constexpr int kTcMaxPhaseTaps = 8;
struct TcPhaseAxis {
    int8_t cnt[kTcMaxPhaseStride];                    // taps per residue
    int8_t k[kTcMaxPhaseStride][kTcMaxPhaseTaps];     // kernel index of each tap
    int8_t off[kTcMaxPhaseStride][kTcMaxPhaseTaps];   // input offset of each tap
};

struct TcGemmParams {
    ConvGeom g;
    int mode;          // TcMode
    int n_tile;        // accumulator columns per tile (<= 256)
    int mma_n;         // N of each MMA (<= 256, multiple of 16)
    int gpc;           // sub-GEMMs (groups, or a slice of one group) per tile
    int kblk;          // (C_in/G) / 64
    int ksteps;        // Kh * Kw * kblk K-steps per sub-GEMM
    int num_m_tiles, num_n_tiles, num_tiles;
    int rect_w, rect_h;              // kTcModeRect: pixel tile = rect_h x rect_w output pixels
    int rect_tiles_w, rect_tiles_h;  // rectangles per image row / column
    int ychunk;                      // output channels per TMA store (32: 64-byte rows)
    int stages;
    int tmem_cols;     // power of two >= 2 * n_tile
    int smem_bytes;
    int pair;          // 1: CTA-pair kernel (B rows split across the two CTAs)
    int dual;          // 1: two pixel tiles per CTA (M = 256, two accumulators; n_tile <= 128)
    int halo;          // 1: kTcModeHalo (one input halo per 64-channel block feeds every tap)
    int halo_w, halo_h;  // kTcModeHalo: halo box extent in pixels (TMA box {64, halo_w, halo_h, 1})
    int halo_bytes;      // kTcModeHalo: one halo stage (box bytes rounded up to 1024)
    int halo_stages;     // kTcModeHalo: halos in flight (stages is then the weight ring)
    int btaps;           // kTcModeHalo: taps per weight stage (one barrier wait feeds btaps x 4 MMAs)
    int bres;            // 1x1 mode: the tile's weights stay in shared memory (loaded once per CTA; the ring carries A only)
    int swap;            // two tiles per CTA of 128 channels (per-tap modes): weights are the MMA's M operand
    int ps;            // kTcModePhase: the transposed convolution's stride S (phases = S*S)
    int hq, wq;        // kTcModePhase: output rows / columns per phase (H_out / S, W_out / S)
    TcPhaseAxis ph, pw;
    int relu;
    const float* bias;
    const float* scale;  // nullptr when no per-channel scale
    __nv_bfloat16* y;
    unsigned* status;
};
// a_map: rect and phase modes 4-D tiled {C_in, W, H, N} box {64, rect_w, rect_h, 1}; im2col
// mode 4-D im2col; 1x1 mode 2-D {C_in, pixels} box {64, 128}; all 128-byte swizzle.
// y_map: rect mode 4-D {C_out, W_out, H_out, N} box {32, rect_w, 32/rect_w, 1},
// phase mode 5-D {C_out, S, W_out/S, S, N*H_out/S} box {32, 1, rect_w, 1, 32/rect_w}
// (one phase's pixels of 32/rect_w rows), else 2-D {C_out, pixels} box {32, 32};
// 64-byte swizzle.  p.pair selects the
// CTA-pair kernel (grid even, clusters of 2).
cudaError_t launch_tc_gemm(const CUtensorMap& a_map, const CUtensorMap& b_map, const CUtensorMap& y_map,
                           const TcGemmParams& p, int grid, cudaStream_t stream);

// Co-resident 2-CTA clusters of the pair kernel at p.smem_bytes (0 if unknown).
int tc_gemm_pair_max_clusters(const TcGemmParams& p);

// ---------------------------------------------------------------- tcgen05 small-K (stem)
constexpr int kSkTransformThreads = 192;  // 6 transform warps
constexpr int kSkMaxStages = 8;
constexpr int kSkMaxRows = 8;             // row segments per stage at most
constexpr int kSkThreads = 320 + kSkTransformThreads;  // producer, MMA, 2 x 4 epilogue, transform warps

struct SmallKParams {
    ConvGeom g;
    const __nv_bfloat16* x;
    const __nv_bfloat16* w;   // [C_out][Ktot]
    const float* bias;
    const float* scale;       // nullptr when no per-channel scale
    __nv_bfloat16* y;
    int relu;
    int ktot;          // C_in * Kh * Kw  (<= 64)
    int kmma;          // number of K=16 MMAs (ceil(ktot / 16))
    int a_row_bytes;   // 64 (K <= 32, 64-byte swizzle) or 128 (128-byte swizzle)
    int segs;          // 128-pixel segments per output row
    int rows_per_tile; // row segments (MMAs of M = 128) per pipeline stage
    int num_segments;  // N * H_out * segs
    int num_tiles;     // ceil(num_segments / rows_per_tile)
    int row_bytes;     // W * C_in * 2
    int raw_bytes;     // rows_per_tile * Kh * row_bytes rounded up to 1024
    int row_runs;      // 1: a stage's input rows come in as one bulk copy per run of overlapping rows
    int stages;
    int tmem_cols;
    int smem_bytes;
    unsigned* status;
};
cudaError_t launch_tc_smallk(const SmallKParams& p, int grid, cudaStream_t stream);

// ---------------------------------------------------------------- fused depthwise 3x3 + pointwise 1x1 block
constexpr int kBkTileH = 16;          // output tile: 16 rows x 8 columns = 128 pixels (TMEM lanes)
constexpr int kBkTileW = 8;
constexpr int kBkChunk = 32;          // depthwise channels per halo copy (one 128-byte FP32 row)
constexpr int kBkHaloBytes = (kBkTileH + 2) * (kBkTileW + 2) * kBkChunk * 4;  // 23,040
constexpr int kBkThreads = 480;       // halo producer, MMA, 2 x 4 epilogue, 4 depthwise, weight producer
constexpr int kBkMaxKblk = 4;         // C <= 256: the whole BF16 A tile (128 x C) stays in shared memory

struct BlockParams {
    int N, C, H, W, C_out, P;
    int H_out, W_out;
    int tiles_w, tiles_h, num_tiles;  // 16 x 8 output tiles
    int kblk;                         // C / 64 (A k-blocks)
    int chunks;                       // C / 32 (halo copies per tile)
    int slices, slice_n;              // pointwise GEMM N slices (slice_n <= 256, multiple of 32)
    int halo_stages, b_stages;
    int tmem_cols;
    int smem_bytes;
    int dw_relu, pw_relu;
    const float* w_dw;      // [C][3][3]
    const float* dw_scale;  // nullptr: 1
    const float* dw_bias;   // nullptr: 0
    const float* pw_scale;  // nullptr: none
    const float* pw_bias;   // nullptr: none
    unsigned* status;
};
// x_map: FP32 4-D {C, W, H, N}, box {32, 10, 18, 1}, no swizzle.  w_map: BF16
// 2-D {C, C_out}, box {64, slice_n}, 128-byte swizzle.  y_map: BF16 4-D
// {C_out, W_out, H_out, N}, box {32, 8, 4, 1}, 64-byte swizzle.
cudaError_t launch_dwpw_block(const CUtensorMap& x_map, const CUtensorMap& w_map, const CUtensorMap& y_map,
                              const BlockParams& p, int grid, cudaStream_t stream);
// Shared memory the block kernel needs for a configuration.
int dwpw_block_smem_bytes(int C, int C_out, int slice_n, int halo_stages, int b_stages);

// Helpers of the plan code, shared with the block plan (conv_api.cu).
bool tensor_map_encoder_ready();
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* base, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle);
cudaError_t device_status_word(unsigned** word);

}  // namespace convgb
