// tc_gemm.cu -- BF16 convolution as an implicit GEMM on tcgen05 tensor cores.
//
// The convolution-as-GEMM mapping of "GPU lesson 9: how a GPU executes
// neural-network convolution" (lincklin.cn), section 19 (M = C_out,
// N = N*H_out*W_out, K = C_in*Kh*Kw), computed as an implicit GEMM (section
// 11; "Convolution variants and their matrix operations", lpnh.cn/news/2674933,
// section 3.3): the im2col matrix is never stored.  Each K-step is one kernel
// tap (kh, kw) and one 64-channel block; the TMA engine gathers the 128 input
// pixels of that tap straight from the NHWC tensor in im2col mode, with its
// out-of-bounds zero fill standing in for the padding (lesson 9, section 26)
// and the tap offset (kh*D, kw*D) gathering only the Kh*Kw live taps of a
// dilated kernel (variants page, section 4.2).  A 1x1 / stride-1 / pad-0
// convolution is a plain GEMM (lesson 9, section 21) and uses a 2-D tiled map.
//
// Operand roles on the tensor core: the MMA's M side is the pixel tile (128
// TMEM lanes), its N side the output channels; D = Y^T of the logical GEMM, so
// each TMEM lane holds one output pixel's contiguous NHWC channel vector.
// Groups are independent GEMMs (variants page, sections 2.2 and 4.3): a tile
// packs `gpc` groups side by side in TMEM columns, each with its own K loop.
//
// Warp roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer (one lane): A (pixels x 64 ch) and B (C_out x 64) per K-step
//   warp 1      TMEM allocator; one lane issues tcgen05.mma and commits
//   warps 2..5  epilogue: tcgen05.ld -> +bias -> ReLU -> BF16 -> smem -> TMA store (NHWC)
// Shared memory holds a ring of `stages` (A, B) buffers; TMEM holds two
// accumulators so the epilogue of tile i overlaps the MMAs of tile i+1.
#include "conv_internal.h"
#include "tc_common.cuh"

namespace convgb {

namespace {

constexpr uint32_t kABytes = kTcBlockM * kTcBlockK * 2;  // 16 KB

constexpr uint32_t kStageOutBytes = 32 * 64;  // one 32-row x 32-column BF16 store tile

struct TcSmem {
    uint8_t* a;
    uint8_t* b;
    uint8_t* out;  // per epilogue warp: two store tiles
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint32_t* tmem_slot;
    int* abort;
};

__device__ __forceinline__ TcSmem carve(uint8_t* raw, const TcGemmParams& p) {
    TcSmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const uint32_t b_bytes = static_cast<uint32_t>(p.mma_n) * 128u;
    s.a = base;
    s.b = base + p.stages * kABytes;
    s.out = s.b + p.stages * b_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.out + 4 * 2 * kStageOutBytes);
    s.full = bars;
    s.empty = bars + p.stages;
    s.tfull = bars + 2 * p.stages;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
    return s;
}

// Sub-GEMM j of n-tile nt: its group, first weight row, and TMEM column offset.
__device__ __forceinline__ void sub_gemm(const TcGemmParams& p, int nt, int j, int& grp, int& brow) {
    if (p.g.cout_g >= p.n_tile) {  // one group spans one or more n-tiles
        brow = nt * p.n_tile;
        grp = brow / p.g.cout_g;
    } else {                       // several groups packed in one n-tile
        grp = nt * p.gpc + j;
        brow = grp * p.g.cout_g;
    }
}

}  // namespace

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_conv_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap b_map,
                   const __grid_constant__ CUtensorMap y_map, const TcGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const TcSmem sm = carve(smem_raw, p);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = sm.abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.tfull[b], 1);
            mbar_init(&sm.tempty[b], 4 * 32);
        }
        mbar_init(sm.drain, 1);
        *sm.abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&a_map);
        tma_prefetch_desc(&b_map);
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

    const int HWo = p.g.H_out * p.g.W_out;
    const uint32_t b_bytes = static_cast<uint32_t>(p.mma_n) * 128u;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
                const int m = tile / p.num_n_tiles;
                const int nt = tile - m * p.num_n_tiles;
                const long long pix0 = static_cast<long long>(m) * kTcBlockM;
                const int n0 = static_cast<int>(pix0 / HWo);
                const int rem = static_cast<int>(pix0 - static_cast<long long>(n0) * HWo);
                const int ho0 = rem / p.g.W_out;
                const int wo0 = rem - ho0 * p.g.W_out;
                for (int j = 0; j < p.gpc && ok; ++j) {
                    int grp, brow;
                    sub_gemm(p, nt, j, grp, brow);
                    for (int ks = 0; ks < p.ksteps; ++ks) {
                        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
                            record_status(p.status, kStatusTimeoutProducer, abort);
                            ok = false;
                            break;
                        }
                        const int tap = ks / p.kblk;
                        const int kb = ks - tap * p.kblk;
                        const int kh = tap / p.g.Kw;
                        const int kw = tap - kh * p.g.Kw;
                        const int c = grp * p.g.cin_g + kb * kTcBlockK;
                        uint8_t* a_dst = sm.a + stage * kABytes;
                        uint8_t* b_dst = sm.b + stage * b_bytes;
                        mbar_arrive_expect_tx(&sm.full[stage], kABytes + b_bytes);
                        if (p.mode == kTcMode1x1) {
                            tma_load_2d(a_dst, &a_map, &sm.full[stage], c, static_cast<int>(pix0));
                        } else {
                            tma_load_im2col_4d(a_dst, &a_map, &sm.full[stage], c, wo0 * p.g.S - p.g.P,
                                               ho0 * p.g.S - p.g.P, n0, static_cast<uint16_t>(kw * p.g.D),
                                               static_cast<uint16_t>(kh * p.g.D));
                        }
                        tma_load_2d(b_dst, &b_map, &sm.full[stage], tap * p.g.cin_g + kb * kTcBlockK, brow);
                        ++issued;
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // Drain: every issued fill must have landed before the CTA may exit.
            for (int s = 0; s < p.stages; ++s) {
                const long long fills = issued / p.stages + (s < issued % p.stages ? 1 : 0);
                if (fills > 0 && !mbar_wait(&sm.full[s], static_cast<uint32_t>((fills - 1) & 1), nullptr))
                    record_status(p.status, kStatusTimeoutDrain, abort);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kTcBlockM, p.mma_n);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++local) {
                const int buf = local & 1;
                const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
                if (!mbar_wait(&sm.tempty[buf], use ^ 1u, abort)) {
                    record_status(p.status, kStatusTimeoutMma, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t d_base = tmem_base + static_cast<uint32_t>(buf * p.n_tile);
                for (int j = 0; j < p.gpc && ok; ++j) {
                    const uint32_t d = d_base + static_cast<uint32_t>(j * p.mma_n);
                    for (int ks = 0; ks < p.ksteps; ++ks) {
                        if (!mbar_wait(&sm.full[stage], phase, abort)) {
                            record_status(p.status, kStatusTimeoutMma, abort);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = sdesc_sw128(smem_addr(sm.a + stage * kABytes));
                        const uint64_t bdesc = sdesc_sw128(smem_addr(sm.b + stage * b_bytes));
#pragma unroll
                        for (int k = 0; k < kTcBlockK / 16; ++k) {
                            // +32 bytes along K inside the swizzle row = +2 in the >>4 address field
                            mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, (ks | k) != 0 ? 1u : 0u);
                        }
                        mma_commit(&sm.empty[stage]);
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (ok) mma_commit(&sm.tfull[buf]);
            }
            // Drain: all MMAs this thread issued complete before TMEM is freed.
            mma_commit(sm.drain);
            if (!mbar_wait(sm.drain, 0, nullptr)) record_status(p.status, kStatusTimeoutDrain, abort);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // TMEM -> registers (+bias, ReLU, BF16) -> swizzled smem tile -> TMA store,
        // 32 pixels x 32 channels at a time, two store tiles in flight per warp.
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        uint8_t* stg = sm.out + (warp - 2) * 2 * kStageOutBytes;
        int sbuf = 0;
        int local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const int buf = local & 1;
            const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
            // warp-uniform outcome, so the .sync.aligned TMEM loads below stay converged
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[buf], use, abort));
            if (!ready) {
                record_status(p.status, kStatusTimeoutEpilogue, abort);
                break;
            }
            tc_fence_after();
            const int m = tile / p.num_n_tiles;
            const int nt = tile - m * p.num_n_tiles;
            const long long row0 = static_cast<long long>(m) * kTcBlockM + quarter * 32;
            const bool rows_exist = row0 < p.g.pixels;
            const int co0 = nt * p.n_tile;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(buf * p.n_tile);
            for (int c = 0; c < p.n_tile; c += 32) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld32(t_row + static_cast<uint32_t>(c), v);
                tmem_ld_wait();
                if (lane == 0) bulk_wait_read_le1();  // the tile written two chunks ago is free
                __syncwarp();
                uint8_t* dst = stg + sbuf * kStageOutBytes;
                stage_row32(v, p.bias ? p.bias + co0 + c : nullptr, p.relu, dst, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && rows_exist) {
                    tma_store_2d(&y_map, dst, co0 + c, static_cast<int>(row0));
                    bulk_commit();
                }
                sbuf ^= 1;
            }
            tc_fence_before();
            mbar_arrive(&sm.tempty[buf]);
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

// ---------------------------------------------------------------------------
// CTA-pair variant (cluster of 2 on two SMs): one tcgen05.mma.cta_group::2 per
// K slice computes 256 pixels x N.  Each CTA loads its own 128-pixel A tile and
// half of the weight rows (N/2), so the weight traffic from L2 per pixel halves
// and a ring stage is 32 KB instead of 48 KB at N = 256 (six stages instead of
// four).  The leader CTA (cluster rank 0) issues the MMAs; both CTAs' TMA loads
// complete on the leader's `full` barrier, the MMA commits arrive on both CTAs'
// `empty` / `tfull` barriers, and both CTAs' epilogue warps arrive on the
// leader's `tempty` barrier.  Each CTA's TMEM holds the accumulator rows of its
// own pixels, so the epilogue is unchanged.
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_conv_pair_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap b_map,
                        const __grid_constant__ CUtensorMap y_map, const TcGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const int half_n = p.mma_n / 2;
    TcGemmParams q = p;
    q.mma_n = half_n;  // this CTA's share of the weight rows sizes its B buffers
    const TcSmem sm = carve(smem_raw, q);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = sm.abort;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int num_pair_tiles = ((p.num_m_tiles + 1) / 2) * p.num_n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.tfull[b], 1);
            mbar_init(&sm.tempty[b], 2 * 4);  // one arrival per epilogue warp of both CTAs
        }
        mbar_init(sm.drain, 1);
        *sm.abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&a_map);
        tma_prefetch_desc(&b_map);
        tma_prefetch_desc(&y_map);
    }
    if (warp == 1) {
        tmem_alloc_pair(sm.tmem_slot, p.tmem_cols);
        tmem_relinquish_pair();
        tc_fence_before();
    }
    __syncthreads();
    cluster_sync_all();  // the peer's barriers exist before anything signals them
    tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;

    const int HWo = p.g.H_out * p.g.W_out;
    const uint32_t b_bytes = static_cast<uint32_t>(half_n) * 128u;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int pt = pair; pt < num_pair_tiles && ok; pt += num_pairs) {
                const int mp = pt / p.num_n_tiles;
                const int nt = pt - mp * p.num_n_tiles;
                const int m = 2 * mp + static_cast<int>(rank);  // past the last tile: zero-filled, not stored
                const long long pix0 = static_cast<long long>(m) * kTcBlockM;
                const int n0 = static_cast<int>(pix0 / HWo);
                const int rem = static_cast<int>(pix0 - static_cast<long long>(n0) * HWo);
                const int ho0 = rem / p.g.W_out;
                const int wo0 = rem - ho0 * p.g.W_out;
                for (int j = 0; j < p.gpc && ok; ++j) {
                    int grp, brow;
                    sub_gemm(p, nt, j, grp, brow);
                    for (int ks = 0; ks < p.ksteps; ++ks) {
                        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
                            record_status(p.status, kStatusTimeoutProducer, abort);
                            ok = false;
                            break;
                        }
                        const int tap = ks / p.kblk;
                        const int kb = ks - tap * p.kblk;
                        const int kh = tap / p.g.Kw;
                        const int kw = tap - kh * p.g.Kw;
                        const int c = grp * p.g.cin_g + kb * kTcBlockK;
                        uint8_t* a_dst = sm.a + stage * kABytes;
                        uint8_t* b_dst = sm.b + stage * b_bytes;
                        const uint32_t full_leader = mapa_shared(smem_addr(&sm.full[stage]), 0);
                        if (leader) mbar_arrive_expect_tx(&sm.full[stage], 2 * (kABytes + b_bytes));
                        if (p.mode == kTcMode1x1) {
                            tma_load_2d_pair(a_dst, &a_map, full_leader, c, static_cast<int>(pix0));
                        } else {
                            tma_load_im2col_4d_pair(a_dst, &a_map, full_leader, c, wo0 * p.g.S - p.g.P,
                                                    ho0 * p.g.S - p.g.P, n0, static_cast<uint16_t>(kw * p.g.D),
                                                    static_cast<uint16_t>(kh * p.g.D));
                        }
                        tma_load_2d_pair(b_dst, &b_map, full_leader, tap * p.g.cin_g + kb * kTcBlockK,
                                         brow + static_cast<int>(rank) * half_n);
                        ++issued;
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // Drain: every fill this CTA issued has landed.  The leader sees its
            // full barriers complete; the peer sees the MMA release each slot
            // after consuming it (which needs the fill to have landed).
            for (int s = 0; s < p.stages; ++s) {
                const long long fills = issued / p.stages + (s < issued % p.stages ? 1 : 0);
                if (fills == 0) continue;
                const uint32_t par = static_cast<uint32_t>((fills - 1) & 1);
                const bool done = leader ? mbar_wait(&sm.full[s], par, nullptr) : mbar_wait(&sm.empty[s], par, nullptr);
                if (!done) record_status(p.status, kStatusTimeoutDrain, abort);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader only)
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_bf16_f32(2 * kTcBlockM, p.mma_n);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int pt = pair; pt < num_pair_tiles && ok; pt += num_pairs, ++local) {
                const int buf = local & 1;
                const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
                if (!mbar_wait_cluster(&sm.tempty[buf], use ^ 1u, abort)) {
                    record_status(p.status, kStatusTimeoutMma, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t d_base = tmem_base + static_cast<uint32_t>(buf * p.n_tile);
                for (int j = 0; j < p.gpc && ok; ++j) {
                    const uint32_t d = d_base + static_cast<uint32_t>(j * p.mma_n);
                    for (int ks = 0; ks < p.ksteps; ++ks) {
                        if (!mbar_wait(&sm.full[stage], phase, abort)) {
                            record_status(p.status, kStatusTimeoutMma, abort);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = sdesc_sw128(smem_addr(sm.a + stage * kABytes));
                        const uint64_t bdesc = sdesc_sw128(smem_addr(sm.b + stage * b_bytes));
#pragma unroll
                        for (int k = 0; k < kTcBlockK / 16; ++k)
                            mma_bf16_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, (ks | k) != 0 ? 1u : 0u);
                        mma_commit_pair(&sm.empty[stage], 0x3);
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (ok) mma_commit_pair(&sm.tfull[buf], 0x3);
            }
            mma_commit_pair(sm.drain, 0x1);
            if (!mbar_wait(sm.drain, 0, nullptr)) record_status(p.status, kStatusTimeoutDrain, abort);
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int quarter = warp & 3;
        uint8_t* stg = sm.out + (warp - 2) * 2 * kStageOutBytes;
        int sbuf = 0;
        int local = 0;
        for (int pt = pair; pt < num_pair_tiles; pt += num_pairs, ++local) {
            const int buf = local & 1;
            const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[buf], use, abort));
            if (!ready) {
                record_status(p.status, kStatusTimeoutEpilogue, abort);
                break;
            }
            tc_fence_after();
            const int mp = pt / p.num_n_tiles;
            const int nt = pt - mp * p.num_n_tiles;
            const int m = 2 * mp + static_cast<int>(rank);
            const long long row0 = static_cast<long long>(m) * kTcBlockM + quarter * 32;
            const bool rows_exist = row0 < p.g.pixels;
            const int co0 = nt * p.n_tile;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(buf * p.n_tile);
            for (int c = 0; c < p.n_tile; c += 32) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld32(t_row + static_cast<uint32_t>(c), v);
                tmem_ld_wait();
                if (lane == 0) bulk_wait_read_le1();
                __syncwarp();
                uint8_t* dst = stg + sbuf * kStageOutBytes;
                stage_row32(v, p.bias ? p.bias + co0 + c : nullptr, p.relu, dst, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && rows_exist) {
                    tma_store_2d(&y_map, dst, co0 + c, static_cast<int>(row0));
                    bulk_commit();
                }
                sbuf ^= 1;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa_shared(smem_addr(&sm.tempty[buf]), 0));
        }
        if (lane == 0) bulk_wait_all();
    }

    __syncthreads();
    cluster_sync_all();  // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, p.tmem_cols);
    }
}

cudaError_t launch_tc_gemm_pair(const CUtensorMap& a_map, const CUtensorMap& b_map, const CUtensorMap& y_map,
                                const TcGemmParams& p, int grid, cudaStream_t stream) {
    cudaError_t e =
        cudaFuncSetAttribute(tc_conv_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, tc_conv_pair_kernel, a_map, b_map, y_map, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int tc_gemm_pair_max_clusters(const TcGemmParams& p) {
    if (cudaFuncSetAttribute(tc_conv_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_conv_pair_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_tc_gemm(const CUtensorMap& a_map, const CUtensorMap& b_map, const CUtensorMap& y_map,
                           const TcGemmParams& p, int grid, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(tc_conv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess) return e;
    tc_conv_kernel<<<grid, kTcThreads, p.smem_bytes, stream>>>(a_map, b_map, y_map, p);
    return cudaGetLastError();
}

}  // namespace convgb
