// dwpw_block.cu -- a depthwise-separable block (depthwise 3x3, FP32, then
// pointwise 1x1, BF16 tensor cores) in one kernel.
//
// The two stages of a depthwise-separable convolution ("GPU lesson 9: how a
// GPU executes neural-network convolution", lincklin.cn, section 25) normally
// write the depthwise feature map to memory and read it back for the
// pointwise GEMM; the same section names kernel fusion as the way to drop that
// round trip, at the price of registers, shared memory and scheduling.  Here
// the depthwise output never leaves the SM: it is rounded to BF16 and written
// straight into shared memory in the tensor core's operand layout, where
// tcgen05.mma consumes it as the A operand of the 1x1 GEMM (lesson 9, section
// 21).  Memory traffic is the FP32 input and the BF16 output only.
//
// One CTA per SM, persistent over 16 x 8-pixel output tiles of one image.
// Per tile:
//   * the halo producer (warp 0) copies the 18 x 10 input pixels under the
//     tile, 32 channels at a time, with 4-D TMA (zero fill = padding, lesson 9
//     section 26) into a ring of halo buffers;
//   * four depthwise warps (10..13) share every halo copy, one warp per four
//     output rows; they compute the 3x3 sums in FP32 (each input row is read
//     once per thread and feeds the output rows it belongs to; a thread owns
//     four channels of two adjacent columns), apply the optional per-channel
//     scale, shift and ReLU, round to BF16 and store the 128 x C A tile in
//     the 128-byte swizzled K-major layout, one 32-channel half k-block per
//     halo copy;
//   * the weight producer (warp 14) streams [slice_n x 64] blocks of the
//     pointwise weights through a ring;
//   * the MMA warp (1) runs, per N slice of the output channels, the K = C
//     reduction into one of two TMEM accumulators; a k-block of A is released
//     to the depthwise warps of the next tile once the last slice has read it.
//     With exactly two slices (both accumulators) it goes k-block major, both
//     slices per k-block, so each k-block returns as soon as it is consumed;
//   * eight epilogue warps (2..9, one group per accumulator) apply the
//     pointwise scale, bias and ReLU, round to BF16 and TMA-store NHWC rows
//     through one staging tile each (the shared memory this leaves for a third
//     halo stage measured faster than a second staging tile).
#include "conv_internal.h"
#include "fp32x2.cuh"
#include "tc_common.cuh"

namespace convgb {

namespace {

constexpr uint32_t kBkKblkBytes = kTcBlockM * kTcBlockK * 2;  // 16 KB: 128 pixels x 64 channels BF16
constexpr uint32_t kBkStoreTile = 32 * 64;                     // 32 pixels x 32 channels BF16
constexpr int kBkHaloW = kBkTileW + 2;
constexpr int kBkHaloH = kBkTileH + 2;
static_assert(kBkHaloBytes == kBkHaloH * kBkHaloW * kBkChunk * 4, "one halo copy: 18 x 10 pixels x 32 FP32 channels");
constexpr int kBkDwWarp0 = 10;
constexpr int kBkDwWarps = 4;
constexpr int kBkWeightWarp = 14;

struct BkSmem {
    uint8_t* a;
    uint8_t* b;
    uint8_t* out;
    uint8_t* halo;
    float* wdw;  // [chunk][tap][32]
    float* dsc;  // [C]
    float* dbi;  // [C]
    uint64_t* hfull;
    uint64_t* hempty;
    uint64_t* bfull;
    uint64_t* bempty;
    uint64_t* afull;
    uint64_t* aempty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint32_t* tmem_slot;
    int* abort;
};

__device__ __forceinline__ BkSmem bk_carve(uint8_t* raw, const BlockParams& p) {
    BkSmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = s.a + p.kblk * kBkKblkBytes;
    s.out = s.b + p.b_stages * p.slice_n * 128;
    s.halo = s.out + 8 * kBkStoreTile;
    s.wdw = reinterpret_cast<float*>(s.halo + p.halo_stages * kBkHaloBytes);
    s.dsc = s.wdw + p.C * 9;
    s.dbi = s.dsc + p.C;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.dbi + p.C);
    s.hfull = bars;
    s.hempty = s.hfull + p.halo_stages;
    s.bfull = s.hempty + p.halo_stages;
    s.bempty = s.bfull + p.b_stages;
    s.afull = s.bempty + p.b_stages;
    s.aempty = s.afull + kBkMaxKblk;
    s.tfull = s.aempty + kBkMaxKblk;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
    return s;
}

struct BkTile {
    int n, ho0, wo0;
};

__device__ __forceinline__ BkTile bk_tile(const BlockParams& p, int m) {
    BkTile t;
    const int per_img = p.tiles_h * p.tiles_w;
    t.n = m / per_img;
    const int r = m - t.n * per_img;
    const int th = r / p.tiles_w;
    t.ho0 = th * kBkTileH;
    t.wo0 = (r - th * p.tiles_w) * kBkTileW;
    return t;
}

// acc += a * w on four channels as two packed FP32 FMAs (each lane rounds as
// fmaf, so the sums match the standalone depthwise kernel bit for bit): half
// the FMA instructions of the depthwise warps, which share their issue slots
// with the epilogue warps.
__device__ __forceinline__ void fma4(float4& acc, const float4& a, const float4& w) {
    unsigned long long lo = f32x2_pack(acc.x, acc.y), hi = f32x2_pack(acc.z, acc.w);
    f32x2_fma(lo, f32x2_pack(a.x, a.y), f32x2_pack(w.x, w.y));
    f32x2_fma(hi, f32x2_pack(a.z, a.w), f32x2_pack(w.z, w.w));
    f32x2_unpack(lo, acc.x, acc.y);
    f32x2_unpack(hi, acc.z, acc.w);
}

// Wait until every fill issued into a ring of `stages` barriers has landed.
__device__ __forceinline__ void drain_ring(uint64_t* full, int stages, long long issued, unsigned* status,
                                          volatile int* abort) {
    for (int s = 0; s < stages; ++s) {
        const long long fills = issued / stages + (s < issued % stages ? 1 : 0);
        if (fills == 0) continue;
        if (!mbar_wait(&full[s], static_cast<uint32_t>((fills - 1) & 1), nullptr))
            record_status(status, kStatusTimeoutDrain, abort);
    }
}

// Depthwise output of one pixel's four channels -> optional scale/shift, ReLU
// -> BF16 -> the A tile (128-byte swizzle: 16-byte chunk c of row p sits at
// chunk c ^ (p & 7)).
__device__ __forceinline__ void bk_emit(float4 v, const float4& sc, const float4& bi, bool affine, bool relu,
                                        uint8_t* a_kb, int pix, int c16, int half) {
    if (affine) {
        v.x = fmaf(v.x, sc.x, bi.x);
        v.y = fmaf(v.y, sc.y, bi.y);
        v.z = fmaf(v.z, sc.z, bi.z);
        v.w = fmaf(v.w, sc.w, bi.w);
    }
    uint2 q;
    if (relu) {
        q.x = pack_bf16x2_relu(v.x, v.y);
        q.y = pack_bf16x2_relu(v.z, v.w);
    } else {
        q.x = pack_bf16x2(v.x, v.y);
        q.y = pack_bf16x2(v.z, v.w);
    }
    *reinterpret_cast<uint2*>(a_kb + pix * 128 + ((c16 ^ (pix & 7)) << 4) + half * 8) = q;
}

}  // namespace

__global__ void __launch_bounds__(kBkThreads, 1)
    dwpw_block_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                      const __grid_constant__ CUtensorMap y_map, const BlockParams p) {
    extern __shared__ uint8_t smem_raw[];
    const BkSmem sm = bk_carve(smem_raw, p);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = sm.abort;
    const uint32_t b_bytes = static_cast<uint32_t>(p.slice_n) * 128u;

    // depthwise weights, scale and shift into shared memory, regrouped so a
    // channel quad's weights for one tap are one 16-byte load
    for (int i = threadIdx.x; i < p.C * 9; i += blockDim.x) {
        const int c = i / 9, tap = i - 9 * (i / 9);
        sm.wdw[((c >> 5) * 9 + tap) * 32 + (c & 31)] = __ldg(p.w_dw + i);
    }
    for (int c = threadIdx.x; c < p.C; c += blockDim.x) {
        sm.dsc[c] = p.dw_scale ? __ldg(p.dw_scale + c) : 1.f;
        sm.dbi[c] = p.dw_bias ? __ldg(p.dw_bias + c) : 0.f;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.halo_stages; ++s) {
            mbar_init(&sm.hfull[s], 1);
            mbar_init(&sm.hempty[s], kBkDwWarps);  // every depthwise warp reads every halo copy
        }
        for (int s = 0; s < p.b_stages; ++s) {
            mbar_init(&sm.bfull[s], 1);
            mbar_init(&sm.bempty[s], 1);
        }
        for (int k = 0; k < kBkMaxKblk; ++k) {
            mbar_init(&sm.afull[k], 2 * kBkDwWarps);  // two 32-channel halves, each written by all DW warps
            mbar_init(&sm.aempty[k], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.tfull[b], 1);
            mbar_init(&sm.tempty[b], 4);
        }
        mbar_init(sm.drain, 1);
        *sm.abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&x_map);
        tma_prefetch_desc(&w_map);
        tma_prefetch_desc(&y_map);
    }
    if (warp == 1) {
        tmem_alloc(sm.tmem_slot, p.tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ halo producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int m = blockIdx.x; m < p.num_tiles && ok; m += gridDim.x) {
                const BkTile t = bk_tile(p, m);
                for (int j = 0; j < p.chunks; ++j) {
                    if (!mbar_wait(&sm.hempty[stage], phase ^ 1u, abort)) {
                        record_status(p.status, kStatusTimeoutProducer, abort);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.hfull[stage], kBkHaloBytes);
                    tma_load_4d(sm.halo + stage * kBkHaloBytes, &x_map, &sm.hfull[stage], j * kBkChunk, t.wo0 - p.P,
                                t.ho0 - p.P, t.n);
                    ++issued;
                    if (++stage == p.halo_stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            drain_ring(sm.hfull, p.halo_stages, issued, p.status, abort);
        }
    } else if (warp == kBkWeightWarp) {
        // ------------------------------------------------------------ pointwise weight producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            // the MMA issuer's order: k-block major with two slices, else slice major
            const bool kb_major = p.slices == 2;
            for (int m = blockIdx.x; m < p.num_tiles && ok; m += gridDim.x) {
                for (int i = 0; i < p.slices * p.kblk; ++i) {
                    const int sl = kb_major ? (i & 1) : i / p.kblk;
                    const int kb = kb_major ? (i >> 1) : i - sl * p.kblk;
                    if (!mbar_wait(&sm.bempty[stage], phase ^ 1u, abort)) {
                        record_status(p.status, kStatusTimeoutProducer, abort);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.bfull[stage], b_bytes);
                    tma_load_2d(sm.b + stage * b_bytes, &w_map, &sm.bfull[stage], kb * kTcBlockK, sl * p.slice_n);
                    ++issued;
                    if (++stage == p.b_stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            drain_ring(sm.bfull, p.b_stages, issued, p.status, abort);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kTcBlockM, p.slice_n);
            int stage = 0;
            uint32_t phase = 0;
            int local_tile = 0, unit = 0;
            bool ok = true;
            for (int m = blockIdx.x; m < p.num_tiles && ok; m += gridDim.x, ++local_tile) {
                const uint32_t tile_par = static_cast<uint32_t>(local_tile) & 1u;
                if (p.slices == 2) {
                    // Two slices fill both TMEM accumulators: k-block major, each k-block of A
                    // feeds both slices and returns to the depthwise warps at once, so the
                    // next tile's depthwise work never waits for the second slice's MMAs.
                    const uint32_t use = tile_par;
                    if (!mbar_wait(&sm.tempty[0], use ^ 1u, abort) || !mbar_wait(&sm.tempty[1], use ^ 1u, abort)) {
                        record_status(p.status, kStatusTimeoutMma, abort);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int kb = 0; kb < p.kblk && ok; ++kb) {
                        if (!mbar_wait(&sm.afull[kb], tile_par, abort)) {
                            record_status(p.status, kStatusTimeoutMma, abort);
                            ok = false;
                            break;
                        }
                        for (int sl = 0; sl < 2; ++sl) {
                            if (!mbar_wait(&sm.bfull[stage], phase, abort)) {
                                record_status(p.status, kStatusTimeoutMma, abort);
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t d = tmem_base + static_cast<uint32_t>(sl * p.slice_n);
                            const uint64_t adesc = sdesc_sw128(smem_addr(sm.a + kb * kBkKblkBytes));
                            const uint64_t bdesc = sdesc_sw128(smem_addr(sm.b + stage * b_bytes));
#pragma unroll
                            for (int k = 0; k < kTcBlockK / 16; ++k)
                                mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                            mma_commit(&sm.bempty[stage]);
                            if (++stage == p.b_stages) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                        if (ok) mma_commit(&sm.aempty[kb]);  // the next tile may overwrite it
                    }
                    if (ok) {
                        mma_commit(&sm.tfull[0]);
                        mma_commit(&sm.tfull[1]);
                    }
                    unit += 2;
                    continue;
                }
                for (int sl = 0; sl < p.slices && ok; ++sl, ++unit) {
                    const int buf = unit & 1;
                    const uint32_t use = static_cast<uint32_t>(unit >> 1) & 1u;
                    if (!mbar_wait(&sm.tempty[buf], use ^ 1u, abort)) {
                        record_status(p.status, kStatusTimeoutMma, abort);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + static_cast<uint32_t>(buf * p.slice_n);
                    for (int kb = 0; kb < p.kblk; ++kb) {
                        if ((sl == 0 && !mbar_wait(&sm.afull[kb], tile_par, abort)) ||
                            !mbar_wait(&sm.bfull[stage], phase, abort)) {
                            record_status(p.status, kStatusTimeoutMma, abort);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = sdesc_sw128(smem_addr(sm.a + kb * kBkKblkBytes));
                        const uint64_t bdesc = sdesc_sw128(smem_addr(sm.b + stage * b_bytes));
#pragma unroll
                        for (int k = 0; k < kTcBlockK / 16; ++k)
                            mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                        mma_commit(&sm.bempty[stage]);
                        if (sl == p.slices - 1) mma_commit(&sm.aempty[kb]);  // the next tile may overwrite it
                        if (++stage == p.b_stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) mma_commit(&sm.tfull[buf]);
                }
            }
            mma_commit(sm.drain);
            if (!mbar_wait(sm.drain, 0, nullptr)) record_status(p.status, kStatusTimeoutDrain, abort);
        }
    } else if (warp >= kBkDwWarp0) {
        // ------------------------------------------------------------ depthwise 3x3
        // All four warps take every halo copy in order (so each waits on every
        // ring phase in turn); warp d computes output rows 4d..4d+3.  Thread:
        // channel quad q (channels 4q..4q+3 of the chunk) of output columns
        // 2cp and 2cp+1.  Input row r of the warp's six halo rows feeds its
        // output rows r (kernel row 0), r-1 (row 1) and r-2 (row 2); three
        // accumulator rows rotate, so each halo value is read once per thread.
        constexpr int kRows = kBkTileH / kBkDwWarps;  // 4 output rows per warp
        const int dw = warp - kBkDwWarp0;
        const int q = lane & 7, cp = lane >> 3;
        const bool relu = p.dw_relu != 0;
        const bool affine = p.dw_scale != nullptr || p.dw_bias != nullptr;
        int local_tile = 0;
        long long idx = 0;  // halo copies consumed so far
        bool ok = true;
        for (int m = blockIdx.x; m < p.num_tiles && ok; m += gridDim.x, ++local_tile) {
            const uint32_t tile_par = static_cast<uint32_t>(local_tile) & 1u;
            for (int j = 0; j < p.chunks; ++j, ++idx) {
                const int kb = j >> 1;
                const int stage = static_cast<int>(idx % p.halo_stages);
                const uint32_t hpar = static_cast<uint32_t>((idx / p.halo_stages) & 1);
                const bool got = mbar_wait(&sm.aempty[kb], tile_par ^ 1u, abort) &&
                                 mbar_wait(&sm.hfull[stage], hpar, abort);
                if (!__all_sync(0xffffffffu, got)) {
                    record_status(p.status, kStatusTimeoutDepthwise, abort);
                    ok = false;
                    break;
                }
                float4 w[9];
                const float4* w4 = reinterpret_cast<const float4*>(sm.wdw) + j * 9 * 8 + q;
#pragma unroll
                for (int t = 0; t < 9; ++t) w[t] = w4[t * 8];
                const float4 sc = reinterpret_cast<const float4*>(sm.dsc)[j * 8 + q];
                const float4 bi = reinterpret_cast<const float4*>(sm.dbi)[j * 8 + q];
                const float4* h4 = reinterpret_cast<const float4*>(sm.halo + stage * kBkHaloBytes) +
                                   (dw * kRows * kBkHaloW + 2 * cp) * 8 + q;
                uint8_t* a_kb = sm.a + kb * kBkKblkBytes;
                const int c16 = (j & 1) * 4 + (q >> 1);
                const int half = q & 1;
                const int pix0 = dw * kRows * kBkTileW + 2 * cp;
                float4 acc[3][2];
#pragma unroll
                for (int r = 0; r < kRows + 2; ++r) {
                    float4 in[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) in[k] = h4[(r * kBkHaloW + k) * 8];
#pragma unroll
                    for (int col = 0; col < 2; ++col) {
                        if (r < kRows) {  // output row r: kernel row 0 starts its sum
                            float4& a0 = acc[r % 3][col];
                            a0 = make_float4(0.f, 0.f, 0.f, 0.f);
                            fma4(a0, in[col], w[0]);
                            fma4(a0, in[col + 1], w[1]);
                            fma4(a0, in[col + 2], w[2]);
                        }
                        if (r >= 1 && r - 1 < kRows) {  // output row r-1: kernel row 1
                            float4& a1 = acc[(r + 2) % 3][col];
                            fma4(a1, in[col], w[3]);
                            fma4(a1, in[col + 1], w[4]);
                            fma4(a1, in[col + 2], w[5]);
                        }
                        if (r >= 2) {  // output row r-2: kernel row 2 completes it
                            float4& a2 = acc[(r + 1) % 3][col];
                            fma4(a2, in[col], w[6]);
                            fma4(a2, in[col + 1], w[7]);
                            fma4(a2, in[col + 2], w[8]);
                            bk_emit(a2, sc, bi, affine, relu, a_kb, pix0 + (r - 2) * kBkTileW + col, c16, half);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.hempty[stage]);  // this warp's halo reads are done
                fence_proxy_async_smem();                         // A writes -> visible to the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.afull[kb]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Group e drains the accumulator units that land in buffer e.  Warp
        // quarter q owns TMEM lanes 32q..32q+31 = tile rows 4q..4q+3.
        const int quarter = warp & 3;
        const int group = (warp - 2) >> 2;
        uint8_t* stg = sm.out + (warp - 2) * kBkStoreTile;
        int unit = 0;
        for (int m = blockIdx.x; m < p.num_tiles; m += gridDim.x) {
            const BkTile t = bk_tile(p, m);
            const int h = t.ho0 + 4 * quarter;
            const bool rows_exist = h < p.H_out;
            bool stop = false;
            for (int sl = 0; sl < p.slices; ++sl, ++unit) {
                const int buf = unit & 1;
                if (buf != group) continue;
                const uint32_t use = static_cast<uint32_t>(unit >> 1) & 1u;
                const bool ready = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[buf], use, abort));
                if (!ready) {
                    record_status(p.status, kStatusTimeoutEpilogue, abort);
                    stop = true;
                    break;
                }
                tc_fence_after();
                const int co0 = sl * p.slice_n;
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(buf * p.slice_n);
                // one 32-column chunk at a time: the TMEM load latency is short next to
                // the staging and store work, and a second register buffer would spill
                for (int cc = 0; cc < p.slice_n; cc += 32) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_ld32(t_row + static_cast<uint32_t>(cc), v);
                    tmem_ld_wait(v);
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    uint8_t* dst = stg;
                    stage_row32<false>(v, p.pw_bias ? p.pw_bias + co0 + cc : nullptr, p.pw_relu, dst, lane,
                                       p.pw_scale ? p.pw_scale + co0 + cc : nullptr);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && rows_exist) {
                        tma_store_4d(&y_map, dst, co0 + cc, t.wo0, h, t.n);
                        bulk_commit();
                    }
                }
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.tempty[buf]);
            }
            if (stop) break;
        }
        if (lane == 0) bulk_wait_all();
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

int dwpw_block_smem_bytes(int C, int C_out, int slice_n, int halo_stages, int b_stages) {
    const int bars = (2 * halo_stages + 2 * b_stages + 2 * kBkMaxKblk + 5) * 8 + 16;
    (void)C_out;
    return 1024 + (C / 64) * static_cast<int>(kBkKblkBytes) + b_stages * slice_n * 128 +
           8 * static_cast<int>(kBkStoreTile) + halo_stages * kBkHaloBytes + C * 11 * 4 + bars;
}

cudaError_t launch_dwpw_block(const CUtensorMap& x_map, const CUtensorMap& w_map, const CUtensorMap& y_map,
                              const BlockParams& p, int grid, cudaStream_t stream) {
    static SmemLimitCache limits;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(dwpw_block_kernel), p.smem_bytes, limits);
    if (e != cudaSuccess) return e;
    dwpw_block_kernel<<<grid, kBkThreads, p.smem_bytes, stream>>>(x_map, w_map, y_map, p);
    return cudaGetLastError();
}

}  // namespace convgb
