// block_api.cu -- C ABI of the fused depthwise-separable block
// (conv_block_plan_*, conv_block_forward in include/conv.h): shape checks,
// launch configuration, TMA descriptors and launch of dwpw_block_kernel.
//
// The block is the depthwise 3x3 + pointwise 1x1 pair of "GPU lesson 9: how a
// GPU executes neural-network convolution" (lincklin.cn), section 25, with the
// depthwise output kept on chip (the fusion that section describes).
#include <new>

#include "../../include/conv.h"
#include "conv_internal.h"
#include "status_slots.h"

using namespace convgb;

struct conv_block_plan {
    BlockParams bp;
    int device;
    int status_slot;  // index of the plan's own status word, -1: the library-wide word
    int num_sms;
    int grid;
    const void* cache_x;
    const void* cache_w;
    const void* cache_y;
    bool cache_valid;
    CUtensorMap map_x;
    CUtensorMap map_w;
    CUtensorMap map_y;
};

namespace {

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int pow2_at_least(int v) {
    int r = 32;
    while (r < v) r <<= 1;
    return r;
}

conv_status encode_block_maps(conv_block_plan* pl, const void* x, const void* w_pw, void* y) {
    if (pl->cache_valid && pl->cache_x == x && pl->cache_w == w_pw && pl->cache_y == y) return CONV_OK;
    pl->cache_valid = false;
    if (!tensor_map_encoder_ready()) return CONV_ERR_CUDA;
    const BlockParams& b = pl->bp;
    const cuuint64_t C = b.C, Co = b.C_out;
    {
        const cuuint64_t dims[4] = {C, static_cast<cuuint64_t>(b.W), static_cast<cuuint64_t>(b.H),
                                    static_cast<cuuint64_t>(b.N)};
        const cuuint64_t strides[3] = {C * 4, C * 4 * b.W, C * 4 * b.W * b.H};
        const cuuint32_t box[4] = {kBkChunk, kBkTileW + 2, kBkTileH + 2, 1};
        if (encode_tiled(&pl->map_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(x), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
            return CONV_ERR_CUDA;
    }
    {
        const cuuint64_t dims[2] = {C, Co};
        const cuuint64_t strides[1] = {C * 2};
        const cuuint32_t box[2] = {kTcBlockK, static_cast<cuuint32_t>(b.slice_n)};
        if (encode_tiled(&pl->map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w_pw), dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return CONV_ERR_CUDA;
    }
    {
        const cuuint64_t dims[4] = {Co, static_cast<cuuint64_t>(b.W_out), static_cast<cuuint64_t>(b.H_out),
                                    static_cast<cuuint64_t>(b.N)};
        const cuuint64_t strides[3] = {Co * 2, Co * 2 * b.W_out, Co * 2 * b.W_out * b.H_out};
        const cuuint32_t box[4] = {32, kBkTileW, 32 / kBkTileW, 1};
        if (encode_tiled(&pl->map_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, y, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
            return CONV_ERR_CUDA;
    }
    pl->cache_x = x;
    pl->cache_w = w_pw;
    pl->cache_y = y;
    pl->cache_valid = true;
    return CONV_OK;
}

}  // namespace

extern "C" {

conv_status conv_block_plan_create(conv_block_plan** out, int N, int C, int H, int W, int C_out, int K, int P,
                                   unsigned flags) {
    if (out == nullptr) return CONV_ERR_INVALID_ARG;
    *out = nullptr;
    if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || C_out <= 0 || K <= 0 || P < 0) return CONV_ERR_INVALID_ARG;
    if (flags & ~(CONV_BLOCK_DW_RELU | CONV_BLOCK_PW_RELU)) return CONV_ERR_INVALID_ARG;
    const long long Ho = static_cast<long long>(H) + 2LL * P - (K - 1);
    const long long Wo = static_cast<long long>(W) + 2LL * P - (K - 1);
    if (Ho < 1 || Wo < 1) return CONV_ERR_INVALID_ARG;
    if (K != 3 || P > 2 || C % 64 != 0 || C > kBkMaxKblk * 64 || C_out % 32 != 0) return CONV_ERR_UNSUPPORTED;
    // output-channel slices: the fewest equal slices of <= 256 channels, each a multiple of 32
    int slices = (C_out + 255) / 256;
    while (C_out % slices != 0 || (C_out / slices) % 32 != 0) ++slices;
    const long long tiles_w = (Wo + kBkTileW - 1) / kBkTileW, tiles_h = (Ho + kBkTileH - 1) / kBkTileH;
    const long long tiles = static_cast<long long>(N) * tiles_w * tiles_h;
    if (tiles > 0x7fffffffLL || static_cast<long long>(N) * H * W * C > (1LL << 40)) return CONV_ERR_UNSUPPORTED;

    conv_block_plan* pl = new (std::nothrow) conv_block_plan();
    if (pl == nullptr) return CONV_ERR_NO_MEMORY;
    BlockParams& b = pl->bp;
    b.N = N; b.C = C; b.H = H; b.W = W; b.C_out = C_out; b.P = P;
    b.H_out = static_cast<int>(Ho); b.W_out = static_cast<int>(Wo);
    b.tiles_w = static_cast<int>(tiles_w);
    b.tiles_h = static_cast<int>(tiles_h);
    b.num_tiles = static_cast<int>(tiles);
    b.kblk = C / 64;
    b.chunks = C / kBkChunk;
    b.slices = slices;
    b.slice_n = C_out / slices;
    b.tmem_cols = pow2_at_least(2 * b.slice_n);
    b.dw_relu = (flags & CONV_BLOCK_DW_RELU) ? 1 : 0;
    b.pw_relu = (flags & CONV_BLOCK_PW_RELU) ? 1 : 0;
    pl->cache_valid = false;

    int smem_optin = 232448;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        cudaGetLastError();
        pl->device = -1;
        pl->num_sms = 152;
        b.status = nullptr;
        pl->status_slot = -1;
    } else if ((pl->status_slot = -1, cudaGetDevice(&pl->device)) != cudaSuccess ||
               cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->device) != cudaSuccess ||
               cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, pl->device) !=
                   cudaSuccess ||
               acquire_status_word(pl->device, &b.status, &pl->status_slot) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return CONV_ERR_CUDA;
    }
    // deepest halo ring first (it hides the HBM latency of the input), then the weight ring
    b.halo_stages = b.b_stages = 0;
    for (int hs = 4; hs >= 2 && b.halo_stages == 0; --hs)
        for (int bs = 4; bs >= 2; --bs)
            if (dwpw_block_smem_bytes(C, C_out, b.slice_n, hs, bs) <= smem_optin) {
                b.halo_stages = hs;
                b.b_stages = bs;
                break;
            }
    if (b.halo_stages == 0) {
        release_status_word(pl->device, pl->status_slot);
        delete pl;
        return CONV_ERR_UNSUPPORTED;
    }
    b.smem_bytes = dwpw_block_smem_bytes(C, C_out, b.slice_n, b.halo_stages, b.b_stages);
    pl->grid = b.num_tiles < pl->num_sms ? b.num_tiles : pl->num_sms;
    *out = pl;
    return CONV_OK;
}

conv_status conv_block_plan_output_shape(const conv_block_plan* p, int* H_out, int* W_out) {
    if (p == nullptr || H_out == nullptr || W_out == nullptr) return CONV_ERR_INVALID_ARG;
    *H_out = p->bp.H_out;
    *W_out = p->bp.W_out;
    return CONV_OK;
}

conv_status conv_block_plan_launch_info(const conv_block_plan* p, int* grid, int* block, int* smem_bytes,
                                        int* halo_stages, int* weight_stages) {
    if (p == nullptr) return CONV_ERR_INVALID_ARG;
    if (grid) *grid = p->grid;
    if (block) *block = kBkThreads;
    if (smem_bytes) *smem_bytes = p->bp.smem_bytes;
    if (halo_stages) *halo_stages = p->bp.halo_stages;
    if (weight_stages) *weight_stages = p->bp.b_stages;
    return CONV_OK;
}

conv_status conv_block_forward(conv_block_plan* p, const void* x, const void* w_dw, const void* dw_scale,
                               const void* dw_bias, const void* w_pw, const void* pw_scale, const void* pw_bias,
                               void* y, void* stream) {
    if (p == nullptr || x == nullptr || w_dw == nullptr || w_pw == nullptr || y == nullptr)
        return CONV_ERR_INVALID_ARG;
    for (const void* ptr : {x, w_dw, dw_scale, dw_bias, w_pw, pw_scale, pw_bias, static_cast<const void*>(y)})
        if (ptr != nullptr && !aligned16(ptr)) return CONV_ERR_MISALIGNED;
    if (p->device < 0) return CONV_ERR_CUDA;  // host-only plan
    int cur = -1;  // the plan belongs to the device current at its creation
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    if (cur != p->device) return CONV_ERR_INVALID_ARG;
    const conv_status s = encode_block_maps(p, x, w_pw, y);
    if (s != CONV_OK) return s;
    BlockParams b = p->bp;
    b.w_dw = static_cast<const float*>(w_dw);
    b.dw_scale = static_cast<const float*>(dw_scale);
    b.dw_bias = static_cast<const float*>(dw_bias);
    b.pw_scale = static_cast<const float*>(pw_scale);
    b.pw_bias = static_cast<const float*>(pw_bias);
    if (launch_dwpw_block(p->map_x, p->map_w, p->map_y, b, p->grid, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    return CONV_OK;
}

conv_status conv_block_plan_device_status(const conv_block_plan* p, void* stream, int* code) {
    if (p == nullptr || code == nullptr) return CONV_ERR_INVALID_ARG;
    *code = 0;
    if (p->device < 0) return CONV_ERR_CUDA;  // host-only plan
    return read_status_word(p->device, p->bp.status, stream, code);
}

conv_status conv_block_plan_destroy(conv_block_plan* p) {
    if (p != nullptr) release_status_word(p->device, p->status_slot);
    delete p;
    return CONV_OK;
}

}  // extern "C"
