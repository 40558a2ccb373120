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
// The kernel is persistent (two CTAs per SM) and each CTA keeps a ring of
// `stages` halo tiles in flight, so HBM reads of the next tiles overlap the
// arithmetic and stores of the current one.  When the channel blocks fit in the grid, every
// CTA stays on one 32-channel block, so its weights are read once.  Each of
// the 256 threads owns 4 channels (one float4: 128-bit shared loads and global
// stores) of one output column and walks a run of output rows.  For stride 1
// and dilation 1 with a 3x3 kernel it keeps the last two input rows of its
// window in registers and reads one new row per output row (lesson 9, sections
// 6 and 17-18: input reuse held in registers, several outputs per thread).
#include "conv_internal.h"
#include "ptx.cuh"

namespace convgb {

namespace {

constexpr int kDwChannels = 32;  // channels per tile: one 128-byte TMA row
constexpr int kDwThreads = 256;  // 8 channel quads x TW columns x (32 / TW) row groups
constexpr int kDwMaxStages = 8;
constexpr int kDwCtasPerSm = 2;  // two resident CTAs: one computes and stores while the other's loads land
constexpr int kDwStagesCap = 2;

__device__ __forceinline__ void fma4(float4& acc, const float4& a, const float4& w) {
    acc.x = fmaf(a.x, w.x, acc.x);
    acc.y = fmaf(a.y, w.y, acc.y);
    acc.z = fmaf(a.z, w.z, acc.z);
    acc.w = fmaf(a.w, w.w, acc.w);
}

struct DwTile {
    int n, ho0, wo0, cb;
};

// Tile `i` of this CTA.  With fixed_cb the CTA's channel block is
// blockIdx.x % cblocks and it walks the spatial tiles; otherwise it walks the
// flat tile list (channel block fastest).
__device__ __forceinline__ DwTile dw_tile(const DepthwiseParams& p, int i) {
    int t, cb;
    if (p.fixed_cb) {
        const int per = gridDim.x / p.cblocks;
        cb = blockIdx.x % p.cblocks;
        t = blockIdx.x / p.cblocks + i * per;
    } else {
        const int flat = blockIdx.x + i * gridDim.x;
        cb = flat % p.cblocks;
        t = flat / p.cblocks;
    }
    DwTile d;
    d.cb = cb;
    const int tw = t % p.tiles_w;
    t /= p.tiles_w;
    const int th = t % p.tiles_h;
    d.n = t / p.tiles_h;
    d.ho0 = th * p.tile_h;
    d.wo0 = tw * p.tile_w;
    return d;
}

__device__ __forceinline__ int dw_count(const DepthwiseParams& p) {
    if (p.fixed_cb) {
        const int per = gridDim.x / p.cblocks;
        const int first = blockIdx.x / p.cblocks;
        const int spatial = p.num_tiles / p.cblocks;
        return first < spatial ? (spatial - 1 - first) / per + 1 : 0;
    }
    return blockIdx.x < p.num_tiles ? (p.num_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
}

struct DwOut {
    float* yf;
    __nv_bfloat16* yb;
    long long stride;  // elements between consecutive output rows
    int relu, out_bf16;
    int affine;         // per-channel scale: acc * scale + shift (the sum then started at 0)
    float4 scale, shift;
};

__device__ __forceinline__ void dw_emit(DwOut& o, float4 acc, bool ok) {
    if (o.affine) {
        acc.x = fmaf(acc.x, o.scale.x, o.shift.x);
        acc.y = fmaf(acc.y, o.scale.y, o.shift.y);
        acc.z = fmaf(acc.z, o.scale.z, o.shift.z);
        acc.w = fmaf(acc.w, o.scale.w, o.shift.w);
    }
    if (o.relu) {
        acc.x = fmaxf(acc.x, 0.f);
        acc.y = fmaxf(acc.y, 0.f);
        acc.z = fmaxf(acc.z, 0.f);
        acc.w = fmaxf(acc.w, 0.f);
    }
    if (ok) {
        if (o.out_bf16) {
            uint2 q;
            q.x = pack_bf16x2(acc.x, acc.y);
            q.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2*>(o.yb) = q;
        } else {
            *reinterpret_cast<float4*>(o.yf) = acc;
        }
    }
    o.yf += o.stride;
    o.yb += o.stride;
}

// One output row of the 3x3 stride-1 window: rows (r0, r1) from registers,
// the new row r2 read from shared memory into `n`.
__device__ __forceinline__ float4 dw_row3(const float4 (&w)[9], const float4& bias, const float4 (&r0)[3],
                                          const float4 (&r1)[3], float4 (&n)[3], const float4* src) {
    n[0] = src[0];
    n[1] = src[8];
    n[2] = src[16];
    float4 acc = bias;
    fma4(acc, r0[0], w[0]);
    fma4(acc, r0[1], w[1]);
    fma4(acc, r0[2], w[2]);
    fma4(acc, r1[0], w[3]);
    fma4(acc, r1[1], w[4]);
    fma4(acc, r1[2], w[5]);
    fma4(acc, n[0], w[6]);
    fma4(acc, n[1], w[7]);
    fma4(acc, n[2], w[8]);
    return acc;
}

}  // namespace

// K > 0: square K x K kernel known at compile time; K == 0: any Kh x Kw.
template <int K, int TW>
__global__ void __launch_bounds__(kDwThreads, kDwCtasPerSm)
    depthwise_kernel(const __grid_constant__ CUtensorMap x_map, const DepthwiseParams p) {
    constexpr int kRowGroups = kDwThreads / (8 * TW);
    constexpr int kTaps = K > 0 ? K * K : 1;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t full[kDwMaxStages];
    __shared__ int abort_flag;
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int Kh = K > 0 ? K : p.g.Kh;
    const int Kw = K > 0 ? K : p.g.Kw;
    const int S = p.g.S, D = p.g.D;
    const int stage_bytes = p.in_h * p.in_w * kDwChannels * 4;
    const int my_count = dw_count(p);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    int issued = 0;  // tiles whose TMA thread 0 has issued
    auto issue = [&](int i) {
        const int slot = i % p.stages;
        issued = i + 1;
        const DwTile t = dw_tile(p, i);
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(stage_bytes));
        tma_load_4d(ring + slot * stage_bytes, &x_map, &full[slot], t.cb * kDwChannels, t.wo0 * S - p.g.P,
                    t.ho0 * S - p.g.P, t.n);
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
    const int in_row4 = p.in_w * (kDwChannels / 4);  // float4 per input row

    float4 wreg[kTaps];
    float4 bias = make_float4(0.f, 0.f, 0.f, 0.f);   // the sum's starting value
    float4 scale = make_float4(1.f, 1.f, 1.f, 1.f), shift = bias;
    int cur_cb = -1;

    for (int i = 0; i < my_count; ++i) {
        const DwTile t = dw_tile(p, i);
        const int c = t.cb * kDwChannels + 4 * c4;
        if (t.cb != cur_cb) {  // weights and bias of this thread's 4 channels
            cur_cb = t.cb;
            if (K > 0) {
#pragma unroll
                for (int k = 0; k < kTaps; ++k)
                    wreg[k] = make_float4(__ldg(p.w + (c + 0) * kTaps + k), __ldg(p.w + (c + 1) * kTaps + k),
                                          __ldg(p.w + (c + 2) * kTaps + k), __ldg(p.w + (c + 3) * kTaps + k));
            }
            if (p.bias) bias = __ldg(reinterpret_cast<const float4*>(p.bias + c));
            if (p.scale) {  // scaled sum + shift: start the sum at zero
                scale = __ldg(reinterpret_cast<const float4*>(p.scale + c));
                shift = bias;
                bias = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }

        const int slot = i % p.stages;
        const bool ok = mbar_wait(&full[slot], static_cast<uint32_t>((i / p.stages) & 1), &abort_flag);
        if (__syncthreads_or(!ok)) {  // block-uniform exit
            if (!ok) record_status(p.status, kStatusTimeoutDepthwise, &abort_flag);
            break;
        }
        const float4* t4 = reinterpret_cast<const float4*>(ring + slot * stage_bytes);
        const int wo = t.wo0 + col;
        const int lr0 = rg * rows;
        const int ho_first = t.ho0 + lr0;
        const int nrows = min(rows, p.g.H_out - ho_first);  // rows of this thread inside the image
        const bool col_ok = wo < p.g.W_out;
        DwOut o;
        const long long o0 =
            ((static_cast<long long>(t.n) * p.g.H_out + ho_first) * p.g.W_out + wo) * p.g.C_out + c;
        o.yf = reinterpret_cast<float*>(p.y) + o0;
        o.yb = reinterpret_cast<__nv_bfloat16*>(p.y) + o0;
        o.stride = static_cast<long long>(p.g.W_out) * p.g.C_out;
        o.relu = p.relu;
        o.out_bf16 = p.out_bf16;
        o.affine = p.scale != nullptr;
        o.scale = scale;
        o.shift = shift;

        bool done = false;
        if constexpr (K == 3) {
            if (rolling) {
                // three register rows cycle through the roles (top, middle, new): no copies
                const float4* src = t4 + (lr0 * p.in_w + col) * (kDwChannels / 4) + c4;
                float4 ra[3] = {src[0], src[8], src[16]};
                src += in_row4;
                float4 rb[3] = {src[0], src[8], src[16]};
                src += in_row4;
                float4 rc[3];
                int r = 0;
                for (; r + 3 <= nrows; r += 3) {
                    dw_emit(o, dw_row3(wreg, bias, ra, rb, rc, src), col_ok);
                    src += in_row4;
                    dw_emit(o, dw_row3(wreg, bias, rb, rc, ra, src), col_ok);
                    src += in_row4;
                    dw_emit(o, dw_row3(wreg, bias, rc, ra, rb, src), col_ok);
                    src += in_row4;
                }
                if (r < nrows) {
                    dw_emit(o, dw_row3(wreg, bias, ra, rb, rc, src), col_ok);
                    src += in_row4;
                    if (r + 1 < nrows) dw_emit(o, dw_row3(wreg, bias, rb, rc, ra, src), col_ok);
                }
                done = true;
            }
        }
        if (!done) {
            for (int r = 0; r < nrows; ++r) {
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
                dw_emit(o, acc, col_ok);
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

int depthwise_config(const ConvGeom& g, int smem_per_sm, int num_sms, DepthwiseParams& d) {
    // Tile width 8 or 16 columns (a warp never straddles two row groups),
    // height from {32, 28, 24, 16} with the least ragged-edge waste, then as
    // many ring stages (<= 8) as fit in a CTA's share of shared memory (two
    // CTAs per SM); shrink the height if fewer than two stages fit (large
    // strides or dilations).
    const int smem_per_cta = smem_per_sm / kDwCtasPerSm - 1024;  // 1 KB per CTA is reserved
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
        long long stages = (smem_per_cta - 128 - 256) / stage;  // alignment slack, static barriers
        // two stages per CTA (four tiles in flight per SM) measured faster than three
        if (stages > kDwStagesCap) stages = kDwStagesCap;
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
    // grid: two CTAs per SM; a multiple of the channel blocks when they fit, so
    // each CTA keeps one channel block (and its weights) for its whole run
    const int slots = kDwCtasPerSm * num_sms;
    d.fixed_cb = d.cblocks <= slots ? 1 : 0;
    int grid = d.fixed_cb ? (slots / d.cblocks) * d.cblocks : slots;
    if (grid > d.num_tiles) grid = d.num_tiles;  // still a multiple of cblocks
    d.grid = grid;
    return 1;
}

template <int K, int TW>
static cudaError_t launch_dw(const CUtensorMap& x_map, const DepthwiseParams& p, cudaStream_t stream) {
    static SmemLimitCache limits;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(depthwise_kernel<K, TW>), p.smem_bytes, limits);
    if (e != cudaSuccess) return e;
    depthwise_kernel<K, TW><<<p.grid, kDwThreads, p.smem_bytes, stream>>>(x_map, p);
    return cudaGetLastError();
}

cudaError_t launch_depthwise(const CUtensorMap& x_map, const DepthwiseParams& p, cudaStream_t stream) {
    const bool k3 = p.g.Kh == 3 && p.g.Kw == 3;
    if (p.tile_w == 8) return k3 ? launch_dw<3, 8>(x_map, p, stream) : launch_dw<0, 8>(x_map, p, stream);
    return k3 ? launch_dw<3, 16>(x_map, p, stream) : launch_dw<0, 16>(x_map, p, stream);
}

}  // namespace convgb
