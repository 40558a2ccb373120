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
// A row segment is up to 128 output pixels of one output row (n, ho).  The Kh
// input rows it reads (h_i = ho*S + kh*D - P) are whole, contiguous NHWC rows
// and come in by bulk copy; transform warps then build its 128 x K operand with
// the index map of lesson 9 section 2 and zero padding as an address test
// (section 26), writing the swizzled K-major layout the MMA descriptor reads
// (64-byte rows with the 64-byte swizzle when K <= 32, else 128-byte rows).
// One pipeline stage carries `rows_per_tile` segments (one M = 128 MMA each,
// side by side in TMEM), so the per-stage barrier and epilogue costs are
// shared by several rows.  The whole weight matrix (C_out x K) stays in shared
// memory.
//
// Warp roles (512 threads, persistent):
//   warp 0       bulk-copy producer (one lane)
//   warp 1       TMEM allocator; one lane issues tcgen05.mma
//   warps 2..9   epilogue, two groups of four (one per TMEM accumulator buffer):
//                tcgen05.ld -> +bias -> ReLU -> BF16 -> smem -> TMA store
//   warps 10..15 transform: raw rows -> swizzled A tiles
// The 3-channel 3x3 case is compiled with its K decomposition as constants;
// other shapes read it from a per-CTA table.
#include "conv_internal.h"
#include "tc_common.cuh"

namespace convgb {

namespace {

constexpr uint32_t kSkOutBytes = 32 * 64;  // one 32-row x 32-column BF16 store tile

struct SkSmem {
    uint8_t* b;
    uint8_t* a;
    uint8_t* raw;
    uint8_t* out;  // per epilogue warp: two store tiles
    uint64_t* raw_full;
    uint64_t* a_full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint32_t* tmem_slot;
    int* abort;
    int* tab_off;    // per K index: kh*row_elems + kw*D*C_in + ci
    int* tab_kwd;    // per K index: kw*D
    int* tab_kh;     // per K index: kh, or -1 beyond the reduction (zero padding of K)
    int* seg_base;   // per stage and row segment: raw-buffer row of the segment's kernel row 0
    float* bias;     // [C_out] copy of the bias
    float* scale;    // [C_out] copy of the per-channel scale (when given)
};

__device__ __forceinline__ uint32_t a_tile_bytes(const SmallKParams& p) { return 128u * p.a_row_bytes; }

__device__ __forceinline__ SkSmem carve(uint8_t* raw, const SmallKParams& p) {
    SkSmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.b = base;
    const uint32_t b_bytes = (static_cast<uint32_t>(p.g.C_out * p.a_row_bytes) + 1023u) & ~1023u;
    s.a = s.b + b_bytes;
    s.raw = s.a + p.stages * p.rows_per_tile * a_tile_bytes(p);
    s.out = s.raw + p.stages * p.raw_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.out + 8 * 2 * kSkOutBytes);
    s.raw_full = bars;
    s.a_full = bars + p.stages;
    s.empty = bars + 2 * p.stages;
    s.tfull = bars + 3 * p.stages;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
    s.tab_off = s.abort + 1;
    s.tab_kwd = s.tab_off + 64;
    s.tab_kh = s.tab_kwd + 64;
    // 16-byte aligned: the epilogue reads it as float4 (the barrier count above varies with `stages`)
    s.seg_base = s.tab_kh + 64;
    s.bias = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(s.seg_base + kSkMaxStages * kSkMaxRows) + 15) & ~uintptr_t(15));
    s.scale = s.bias + ((p.g.C_out + 3) & ~3);
    return s;
}

struct SkSeg {
    int n, ho, wo0, npix;
};

// Row segment u: output row (n, ho), pixels [wo0, wo0 + npix).
__device__ __forceinline__ SkSeg segment(const SmallKParams& p, int u) {
    SkSeg t;
    const int per_img = p.g.H_out * p.segs;
    t.n = u / per_img;
    const int r = u - t.n * per_img;
    t.ho = r / p.segs;
    const int seg = r - t.ho * p.segs;
    t.wo0 = seg * 128;
    t.npix = min(128, p.g.W_out - t.wo0);
    return t;
}

// The input rows of the row segments of one stage.  With row runs, segments in
// a row of one image whose input rows overlap or touch form one run, copied as
// one contiguous block of whole NHWC rows (a 3x3 stride-2 stem reads 9 rows for
// 4 output rows, not 12); rows outside the image are never copied (they read
// as zero padding).  Otherwise every segment gets its Kh rows, one copy each.
// emit(n, first_row, rows, raw_row) is called per copy; base[j] receives the
// raw-buffer row that holds segment j's kernel row 0 (it may lie before the
// copied rows when that row is padding).
template <typename F>
__device__ __forceinline__ void stage_rows(const SmallKParams& p, int tile, int* base, F&& emit) {
    const int R = p.rows_per_tile;
    if (!p.row_runs) {
        for (int j = 0; j < R; ++j) {
            const int u = tile * R + j;
            if (u >= p.num_segments) break;
            const SkSeg t = segment(p, u);
            if (base) base[j] = j * p.g.Kh;
            for (int kh = 0; kh < p.g.Kh; ++kh) {
                const int hi = t.ho * p.g.S - p.g.P + kh * p.g.D;
                if (hi >= 0 && hi < p.g.H) emit(t.n, hi, 1, j * p.g.Kh + kh);
            }
        }
        return;
    }
    int run_n = -1, run_lo = 0, run_hi = -1, raw0 = 0, next_raw = 0;
    for (int j = 0; j < R; ++j) {
        const int u = tile * R + j;
        if (u >= p.num_segments) break;
        const SkSeg t = segment(p, u);
        const int top = t.ho * p.g.S - p.g.P;  // input row of kernel row 0
        const int lo = top > 0 ? top : 0;
        const int last = top + p.g.Kh - 1;
        const int hi = last < p.g.H - 1 ? last : p.g.H - 1;
        if (lo > hi) {  // every kernel row is padding
            if (base) base[j] = 0;
            continue;
        }
        if (t.n != run_n || lo > run_hi + 1) {  // a new run
            if (run_n >= 0) emit(run_n, run_lo, run_hi - run_lo + 1, raw0);
            raw0 = next_raw;
            run_n = t.n;
            run_lo = lo;
            run_hi = hi;
        } else if (hi > run_hi) {
            run_hi = hi;
        }
        next_raw = raw0 + (run_hi - run_lo + 1);
        if (base) base[j] = raw0 + (top - run_lo);
    }
    if (run_n >= 0) emit(run_n, run_lo, run_hi - run_lo + 1, raw0);
}

// Byte offset of element k of row r in a swizzled K-major tile with 64- or
// 128-byte rows (16-byte chunk j of row r sits at chunk j ^ f(r)).
__device__ __forceinline__ uint32_t sw_offset(int r, int k, int row_bytes) {
    if (row_bytes == 128) return static_cast<uint32_t>(r * 128 + ((((k >> 3) ^ (r & 7)) & 7) << 4) + ((k & 7) << 1));
    return static_cast<uint32_t>(r * 64 + ((((k >> 3) ^ (r >> 1)) & 3) << 4) + ((k & 7) << 1));
}

// Shared-memory descriptor for a K-major tile of 64-byte rows, 64-byte swizzle:
// stride byte offset 8 rows x 64 B = 512 (>> 4 = 32), swizzle mode 4.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(512 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(4) << 61);
}

__device__ __forceinline__ uint64_t a_desc(const SmallKParams& p, uint32_t saddr) {
    return p.a_row_bytes == 128 ? sdesc_sw128(saddr) : sdesc_sw64(saddr);
}

// Gather the 8 K-elements of chunk j for one pixel row.  CIN/KH/KW > 0: the
// decomposition k -> (kh, kw, ci) is constant-folded; 0: read from the tables.
template <int CIN, int KH, int KW>
__device__ __forceinline__ uint4 gather_chunk(const SkSmem& sm, const SmallKParams& p, const uint16_t* src, int j,
                                              int wbase, unsigned long long rowmask) {
    uint32_t q[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        uint32_t pair = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = j * 8 + e + h;
            uint32_t v = 0;
            if constexpr (CIN > 0) {
                if (k < CIN * KH * KW) {
                    const int ci = k % CIN, tap = k / CIN, kh = tap / KW, kw = tap % KW;
                    const int wi = wbase + kw * p.g.D;
                    if (((rowmask >> kh) & 1ull) && wi >= 0 && wi < p.g.W)
                        v = src[kh * (p.row_bytes >> 1) + wi * CIN + ci];
                }
            } else {
                const int kh = sm.tab_kh[k];
                const int wi = wbase + sm.tab_kwd[k];
                if (kh >= 0 && ((rowmask >> kh) & 1ull) && wi >= 0 && wi < p.g.W)
                    v = src[wbase * p.g.C_in + sm.tab_off[k]];
            }
            pair |= v << (16 * h);
        }
        q[e >> 1] = pair;
    }
    return make_uint4(q[0], q[1], q[2], q[3]);
}

}  // namespace

template <int CIN, int KH, int KW>
__global__ void __launch_bounds__(kSkThreads, 1)
    tc_smallk_kernel(const __grid_constant__ CUtensorMap y_map, const SmallKParams p) {
    extern __shared__ uint8_t smem_raw[];
    const SkSmem sm = carve(smem_raw, p);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = sm.abort;
    const int R = p.rows_per_tile;
    const int n_tile = p.g.C_out;

    // Resident weights: row co = w[co][0..ktot), zero beyond ktot, swizzled.
    {
        const uint16_t* w16 = reinterpret_cast<const uint16_t*>(p.w);
        const int kw = p.a_row_bytes / 2;
        for (int idx = threadIdx.x; idx < p.g.C_out * kw; idx += blockDim.x) {
            const int co = idx / kw;
            const int k = idx - co * kw;
            const uint16_t v = k < p.ktot ? w16[static_cast<long long>(co) * p.ktot + k] : uint16_t(0);
            *reinterpret_cast<uint16_t*>(sm.b + sw_offset(co, k, p.a_row_bytes)) = v;
        }
        fence_proxy_async_smem();
        // K index -> (kh, kw, ci) decomposition, once per CTA (no divisions in the gather loop)
        for (int k = threadIdx.x; k < 64; k += blockDim.x) {
            if (k < p.ktot) {
                const int ci = k % p.g.C_in, tap = k / p.g.C_in;
                const int kh = tap / p.g.Kw, kwi = tap - kh * p.g.Kw;
                sm.tab_off[k] = kh * (p.row_bytes >> 1) + kwi * p.g.D * p.g.C_in + ci;
                sm.tab_kwd[k] = kwi * p.g.D;
                sm.tab_kh[k] = kh;
            } else {
                sm.tab_off[k] = 0;
                sm.tab_kwd[k] = 0;
                sm.tab_kh[k] = -1;
            }
        }
        for (int c = threadIdx.x; c < p.g.C_out; c += blockDim.x) {
            sm.bias[c] = p.bias ? p.bias[c] : 0.f;
            sm.scale[c] = p.scale ? p.scale[c] : 1.f;
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sm.raw_full[s], 1);
            mbar_init(&sm.a_full[s], kSkTransformThreads);
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
                int* base = sm.seg_base + stage * kSkMaxRows;
                uint32_t bytes = 0;  // segment bases (read by the transform warps) and the stage's byte count
                stage_rows(p, tile, base, [&](int, int, int rows, int) {
                    bytes += static_cast<uint32_t>(rows * p.row_bytes);
                });
                mbar_arrive_expect_tx(&sm.raw_full[stage], bytes);
                uint8_t* dst = sm.raw + stage * p.raw_bytes;
                stage_rows(p, tile, nullptr, [&](int n, int row, int rows, int raw_row) {
                    const char* src = xb + (static_cast<long long>(n) * p.g.H + row) * p.row_bytes;
                    bulk_load(dst + raw_row * p.row_bytes, src, static_cast<uint32_t>(rows * p.row_bytes),
                              &sm.raw_full[stage]);
                });
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
            const uint64_t bdesc = a_desc(p, smem_addr(sm.b));
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
                const int rows = min(R, p.num_segments - tile * R);
                // K slices outer, segments inner: consecutive MMAs go to independent accumulators
                for (int k = 0; k < p.kmma; ++k)
                    for (int j = 0; j < rows; ++j) {
                        const uint64_t adesc = a_desc(p, smem_addr(sm.a + (stage * R + j) * a_tile_bytes(p)));
                        const uint32_t d = tmem_base + static_cast<uint32_t>((buf * R + j) * n_tile);
                        mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, k != 0 ? 1u : 0u);
                    }
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
    } else if (warp < 10) {
        // ------------------------------------------------------------ epilogue
        // Two groups of four warps, one per TMEM accumulator buffer (so two
        // stages drain at once); the next chunk's TMEM load is in flight while
        // the current one is converted and staged.
        const int quarter = warp & 3;
        const int group = (warp - 2) >> 2;
        uint8_t* stg = sm.out + (warp - 2) * 2 * kSkOutBytes;
        const int chunks = n_tile / 32;
        int sbuf = 0;
        int local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const int buf = local & 1;
            if (buf != group) continue;
            const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[buf], use, abort));
            if (!ready) {
                record_status(p.status, kStatusTimeoutEpilogue, abort);
                break;
            }
            tc_fence_after();
            const int rows = min(R, p.num_segments - tile * R);
            const int items = rows * chunks;  // (segment, 32-column chunk) pairs
            const uint32_t t_q = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(buf * R * n_tile);
            auto t_addr = [&](int it) {
                const int j = it / chunks;
                return t_q + static_cast<uint32_t>(j * n_tile + (it - j * chunks) * 32);
            };
            auto process = [&](const uint32_t(&v)[32], int it) {
                const int j = it / chunks;
                const int c = (it - j * chunks) * 32;
                const SkSeg t = segment(p, tile * R + j);
                const int wo_row0 = t.wo0 + quarter * 32;  // first output column of this warp's rows
                const bool rows_exist = quarter * 32 < t.npix;
                if (lane == 0) bulk_wait_read_le1();
                __syncwarp();
                uint8_t* dst = stg + sbuf * kSkOutBytes;
                stage_row32<true>(v, p.bias ? sm.bias + c : nullptr, p.relu, dst, lane,
                                  p.scale ? sm.scale + c : nullptr);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && rows_exist) {  // columns past W_out fall outside the map: not written
                    tma_store_3d(&y_map, dst, c, wo_row0, t.n * p.g.H_out + t.ho);
                    bulk_commit();
                }
                sbuf ^= 1;
            };
            uint32_t va[32], vb[32];
            __syncwarp();
            tmem_ld32(t_addr(0), va);
            for (int it = 0; it < items; it += 2) {
                tmem_ld_wait(va);
                if (it + 1 < items) {
                    __syncwarp();
                    tmem_ld32(t_addr(it + 1), vb);
                }
                process(va, it);
                if (it + 1 < items) {
                    tmem_ld_wait(vb);
                    if (it + 2 < items) {
                        __syncwarp();
                        tmem_ld32(t_addr(it + 2), va);
                    }
                    process(vb, it + 1);
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.tempty[buf]);
        }
        if (lane == 0) bulk_wait_all();
    } else {
        // ------------------------------------------------------------ transform (im2col in smem)
        const int tid = threadIdx.x - 320;  // 0..kSkTransformThreads-1
        const uint16_t* raw16 = reinterpret_cast<const uint16_t*>(sm.raw);
        const int raw_elems = p.raw_bytes >> 1;
        const int row_elems = p.row_bytes >> 1;
        const int nchunks = 2 * p.kmma;
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
            if (!mbar_wait(&sm.raw_full[stage], phase, abort)) {
                record_status(p.status, kStatusTimeoutTransform, abort);
                break;
            }
            for (int idx = tid; idx < R * 128; idx += kSkTransformThreads) {
                const int j = idx >> 7;   // row segment within the stage
                const int r = idx & 127;  // A row = pixel within the segment
                const int u = tile * R + j;
                uint8_t* arow = sm.a + (stage * R + j) * a_tile_bytes(p);
                unsigned long long rowmask = 0;  // input rows that exist (the rest read as zero)
                int wbase = 0;
                if (u < p.num_segments) {
                    const SkSeg t = segment(p, u);
                    for (int kh = 0; kh < p.g.Kh; ++kh) {
                        const int hi = t.ho * p.g.S - p.g.P + kh * p.g.D;
                        if (hi >= 0 && hi < p.g.H) rowmask |= 1ull << kh;
                    }
                    wbase = (t.wo0 + r) * p.g.S - p.g.P;  // input column of tap kw = 0
                    if (r >= t.npix) rowmask = 0;         // rows past the segment: zeros
                }
                const uint16_t* src = raw16 + stage * raw_elems + sm.seg_base[stage * kSkMaxRows + j] * row_elems;
                if constexpr (CIN > 0) {
                    constexpr int kChunks = ((CIN * KH * KW + 15) / 16) * 2;
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        *reinterpret_cast<uint4*>(arow + sw_offset(r, c * 8, p.a_row_bytes)) =
                            gather_chunk<CIN, KH, KW>(sm, p, src, c, wbase, rowmask);
                } else {
                    for (int c = 0; c < nchunks; ++c)
                        *reinterpret_cast<uint4*>(arow + sw_offset(r, c * 8, p.a_row_bytes)) =
                            gather_chunk<0, 0, 0>(sm, p, src, c, wbase, rowmask);
                }
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

template <int CIN, int KH, int KW>
static cudaError_t launch_sk(const CUtensorMap& y_map, const SmallKParams& p, int grid, cudaStream_t stream) {
    static int limits[64] = {};
    cudaError_t e =
        ensure_smem_limit(reinterpret_cast<const void*>(tc_smallk_kernel<CIN, KH, KW>), p.smem_bytes, limits);
    if (e != cudaSuccess) return e;
    tc_smallk_kernel<CIN, KH, KW><<<grid, kSkThreads, p.smem_bytes, stream>>>(y_map, p);
    return cudaGetLastError();
}

cudaError_t launch_tc_smallk(const CUtensorMap& y_map, const SmallKParams& p, int grid, cudaStream_t stream) {
    if (p.g.C_in == 3 && p.g.Kh == 3 && p.g.Kw == 3) return launch_sk<3, 3, 3>(y_map, p, grid, stream);
    return launch_sk<0, 0, 0>(y_map, p, grid, stream);
}

}  // namespace convgb
