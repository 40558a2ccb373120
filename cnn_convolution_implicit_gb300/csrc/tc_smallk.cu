// tc_smallk.cu -- BF16 convolution with a short reduction (C_in*Kh*Kw <= 64),
// e.g. a 3-channel stem layer, as an implicit GEMM on tcgen05.
//
// Same mapping as the main implicit GEMM ("GPU lesson 9: how a GPU executes
// neural-network convolution", lincklin.cn, sections 11 and 19), but a pixel
// carries only C_in = 3 channels (6 bytes), below the TMA's 16-byte granule, so
// the im2col gather happens in shared memory instead.  Lesson 9 section 20
// names exactly this case (C_in = 3 under-fills the tensor core); the reduction
// is padded with zeros up to the next multiple of 16 and the layer stays bound
// by memory traffic, not by the MMA.
//
// One tile = up to 128 output pixels of one output row (n, ho).  The Kh input
// rows it reads (h_i = ho*S + kh*D - P) are whole, contiguous NHWC rows and
// come in by bulk copy; transform warps then build the 128 x K operand with
// the index map of lesson 9 section 2 and zero padding as an address test
// (section 26), writing the 128-byte-swizzled layout the MMA descriptor reads.
// The whole weight matrix (C_out x K, K <= 64) stays in shared memory.
//
// Warp roles (320 threads, persistent):
//   warp 0      bulk-copy producer (one lane)
//   warp 1      TMEM allocator; one lane issues tcgen05.mma
//   warps 2..5  epilogue (tcgen05.ld -> +bias -> ReLU -> BF16 -> NHWC store)
//   warps 6..9  transform: raw rows -> swizzled A tile
#include "conv_internal.h"
#include "tc_common.cuh"

namespace convgb {

namespace {

constexpr uint32_t kSkABytes = 128 * 128;  // 128 pixels x 64 BF16

struct SkSmem {
    uint8_t* b;
    uint8_t* a;
    uint8_t* raw;
    uint64_t* raw_full;
    uint64_t* a_full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint32_t* tmem_slot;
    int* abort;
};

__device__ __forceinline__ SkSmem carve(uint8_t* raw, const SmallKParams& p) {
    SkSmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.b = base;
    s.a = s.b + p.g.C_out * 128;
    s.raw = s.a + p.stages * kSkABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.raw + p.stages * p.raw_bytes);
    s.raw_full = bars;
    s.a_full = bars + p.stages;
    s.empty = bars + 2 * p.stages;
    s.tfull = bars + 3 * p.stages;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
    return s;
}

struct SkTile {
    int n, ho, wo0, npix;
};

__device__ __forceinline__ SkTile decode(const SmallKParams& p, int tile) {
    SkTile t;
    const int per_img = p.g.H_out * p.segs;
    t.n = tile / per_img;
    const int r = tile - t.n * per_img;
    t.ho = r / p.segs;
    const int seg = r - t.ho * p.segs;
    t.wo0 = seg * 128;
    t.npix = min(128, p.g.W_out - t.wo0);
    return t;
}

// Byte offset of element k of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
    return static_cast<uint32_t>(r * 128 + ((((k >> 3) ^ (r & 7)) & 7) << 4) + ((k & 7) << 1));
}

}  // namespace

__global__ void __launch_bounds__(kSkThreads, 1) tc_smallk_kernel(const SmallKParams p) {
    extern __shared__ uint8_t smem_raw[];
    const SkSmem sm = carve(smem_raw, p);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = sm.abort;

    // Resident weights: row co = w[co][0..ktot), zero beyond ktot, swizzled.
    {
        const uint16_t* w16 = reinterpret_cast<const uint16_t*>(p.w);
        for (int idx = threadIdx.x; idx < p.g.C_out * 64; idx += blockDim.x) {
            const int co = idx >> 6;
            const int k = idx & 63;
            const uint16_t v = k < p.ktot ? w16[static_cast<long long>(co) * p.ktot + k] : uint16_t(0);
            *reinterpret_cast<uint16_t*>(sm.b + sw128_offset(co, k)) = v;
        }
        fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sm.raw_full[s], 1);
            mbar_init(&sm.a_full[s], 128);
            mbar_init(&sm.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.tfull[b], 1);
            mbar_init(&sm.tempty[b], 128);
        }
        mbar_init(sm.drain, 1);
        *sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sm.tmem_slot, p.tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;
    const int n_tile = p.g.C_out;

    if (warp == 0) {
        // ------------------------------------------------------------ bulk-copy producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            const char* xb = reinterpret_cast<const char*>(p.x);
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
                    record_status(p.status, kStatusTimeoutProducer, abort);
                    break;
                }
                const SkTile t = decode(p, tile);
                uint32_t bytes = 0;
                for (int kh = 0; kh < p.g.Kh; ++kh) {
                    const int hi = t.ho * p.g.S - p.g.P + kh * p.g.D;
                    if (hi >= 0 && hi < p.g.H) bytes += static_cast<uint32_t>(p.row_bytes);
                }
                mbar_arrive_expect_tx(&sm.raw_full[stage], bytes);
                uint8_t* dst = sm.raw + stage * p.raw_bytes;
                for (int kh = 0; kh < p.g.Kh; ++kh) {
                    const int hi = t.ho * p.g.S - p.g.P + kh * p.g.D;
                    if (hi < 0 || hi >= p.g.H) continue;
                    const char* src = xb + (static_cast<long long>(t.n) * p.g.H + hi) * p.row_bytes;
                    bulk_load(dst + kh * p.row_bytes, src, static_cast<uint32_t>(p.row_bytes), &sm.raw_full[stage]);
                }
                ++issued;
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            for (int s = 0; s < p.stages; ++s) {
                const long long fills = issued / p.stages + (s < issued % p.stages ? 1 : 0);
                if (fills > 0 && !mbar_wait(&sm.raw_full[s], static_cast<uint32_t>((fills - 1) & 1), nullptr))
                    record_status(p.status, kStatusTimeoutDrain, abort);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, n_tile);
            const uint64_t bdesc = sdesc_sw128(smem_addr(sm.b));
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
                const int buf = local & 1;
                const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
                if (!mbar_wait(&sm.tempty[buf], use ^ 1u, abort) || !mbar_wait(&sm.a_full[stage], phase, abort)) {
                    record_status(p.status, kStatusTimeoutMma, abort);
                    break;
                }
                tc_fence_after();
                const uint64_t adesc = sdesc_sw128(smem_addr(sm.a + stage * kSkABytes));
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * n_tile);
                for (int k = 0; k < p.kmma; ++k) mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, k != 0 ? 1u : 0u);
                mma_commit(&sm.empty[stage]);
                mma_commit(&sm.tfull[buf]);
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            mma_commit(sm.drain);
            if (!mbar_wait(sm.drain, 0, nullptr)) record_status(p.status, kStatusTimeoutDrain, abort);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        int local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const int buf = local & 1;
            const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[buf], use, abort));
            if (!ready) {
                record_status(p.status, kStatusTimeoutEpilogue, abort);
                break;
            }
            tc_fence_after();
            const SkTile t = decode(p, tile);
            const bool valid = row < t.npix;
            const long long pix =
                (static_cast<long long>(t.n) * p.g.H_out + t.ho) * p.g.W_out + t.wo0 + (valid ? row : 0);
            __nv_bfloat16* yrow = p.y + pix * p.g.C_out;
            const uint32_t t_row =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * n_tile);
            for (int c = 0; c < n_tile; c += 32) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld32(t_row + static_cast<uint32_t>(c), v);
                tmem_ld_wait();
                epilogue_store32(v, p.bias ? p.bias + c : nullptr, p.relu, yrow + c, valid);
            }
            tc_fence_before();
            mbar_arrive(&sm.tempty[buf]);
        }
    } else {
        // ------------------------------------------------------------ transform (im2col in smem)
        const int r = threadIdx.x - 192;  // A row = pixel within the tile
        const uint16_t* raw16 = reinterpret_cast<const uint16_t*>(sm.raw);
        const int row_elems = p.row_bytes >> 1;
        const int raw_elems = p.raw_bytes >> 1;
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
            if (!mbar_wait(&sm.raw_full[stage], phase, abort)) {
                record_status(p.status, kStatusTimeoutTransform, abort);
                break;
            }
            const SkTile t = decode(p, tile);
            const uint16_t* src = raw16 + stage * raw_elems;
            uint8_t* arow = sm.a + stage * kSkABytes;
            const int wo = t.wo0 + r;
            const bool pix_ok = r < t.npix;
            for (int j = 0; j < 2 * p.kmma; ++j) {  // 16-byte chunks of 8 K-elements
                uint32_t q[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    uint32_t pair = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int k = j * 8 + e + h;
                        uint32_t v = 0;
                        if (pix_ok && k < p.ktot) {
                            const int ci = k % p.g.C_in;
                            const int tap = k / p.g.C_in;
                            const int kh = tap / p.g.Kw;
                            const int kw = tap - kh * p.g.Kw;
                            const int hi = t.ho * p.g.S - p.g.P + kh * p.g.D;
                            const int wi = wo * p.g.S - p.g.P + kw * p.g.D;
                            if (hi >= 0 && hi < p.g.H && wi >= 0 && wi < p.g.W)
                                v = src[kh * row_elems + wi * p.g.C_in + ci];
                        }
                        pair |= v << (16 * h);
                    }
                    q[e >> 1] = pair;
                }
                *reinterpret_cast<uint4*>(arow + sw128_offset(r, j * 8)) = make_uint4(q[0], q[1], q[2], q[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.a_full[stage]);
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

cudaError_t launch_tc_smallk(const SmallKParams& p, int grid, cudaStream_t stream) {
    cudaError_t e =
        cudaFuncSetAttribute(tc_smallk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess) return e;
    tc_smallk_kernel<<<grid, kSkThreads, p.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace convgb
