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
//                tcgen05.ld -> +bias -> ReLU -> BF16 -> 16-byte global stores (a lane
//                owns one output pixel: its 32-channel run is 64 contiguous bytes)
//   warps 10..15 transform: raw rows -> swizzled A tiles
// The 3-channel 3x3 case is compiled with its K decomposition as constants;
// other shapes read it from a per-CTA table.
#include "conv_internal.h"
#include "tc_common.cuh"

namespace convgb {

namespace {

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
    uint64_t* ready;  // the resident weights, tables and bias are in place
    uint32_t* tmem_slot;
    int* abort;
    int* tab_off;    // per K index: kh*row_elems + kw*D*C_in + ci
    int* tab_kwd;    // per K index: kw*D
    int* tab_kh;     // per K index: kh, or -1 beyond the reduction (zero padding of K)
    int4* seg_info;  // per stage and row segment: {raw row of kernel row 0, live kernel rows, w0, pixels}
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
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.raw + p.stages * p.raw_bytes);
    s.raw_full = bars;
    s.a_full = bars + p.stages;
    s.empty = bars + 2 * p.stages;
    s.tfull = bars + 3 * p.stages;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.ready = s.drain + 1;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.ready + 1);
    s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
    s.tab_off = s.abort + 1;
    s.tab_kwd = s.tab_off + 64;
    s.tab_kh = s.tab_kwd + 64;
    // 16-byte aligned: the epilogue reads it as float4 (the barrier count above varies with `stages`)
    s.seg_info = reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(s.tab_kh + 64) + 15) & ~uintptr_t(15));
    s.bias = reinterpret_cast<float*>(s.seg_info + kSkMaxStages * kSkMaxRows);
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

// The segment after t (no division: segments run along the row, then rows, then images).
__device__ __forceinline__ void next_segment(const SmallKParams& p, SkSeg& t) {
    t.wo0 += 128;
    if (t.wo0 >= p.g.W_out) {
        t.wo0 = 0;
        if (++t.ho == p.g.H_out) {
            t.ho = 0;
            ++t.n;
        }
    }
    t.npix = min(128, p.g.W_out - t.wo0);
}

// The first segments of a CTA's stages: segment blockIdx.x * R, then gridDim.x * R
// segments further each time, stepped as a mixed-radix number (segment, row,
// image) with one carry per digit instead of divisions.
struct SkStageWalk {
    SkSeg t;
    int seg, d_seg, d_ho, d_n;
    __device__ __forceinline__ SkStageWalk(const SmallKParams& p) {
        t = segment(p, blockIdx.x * p.rows_per_tile);
        seg = t.wo0 / 128;
        const SkSeg d = segment(p, gridDim.x * p.rows_per_tile);
        d_seg = d.wo0 / 128;
        d_ho = d.ho;
        d_n = d.n;
    }
    __device__ __forceinline__ void next(const SmallKParams& p) {
        seg += d_seg;
        int c = 0;
        if (seg >= p.segs) {
            seg -= p.segs;
            c = 1;
        }
        t.ho += d_ho + c;
        c = 0;
        if (t.ho >= p.g.H_out) {
            t.ho -= p.g.H_out;
            c = 1;
        }
        t.n += d_n + c;
        t.wo0 = seg * 128;
        t.npix = min(128, p.g.W_out - t.wo0);
    }
};

// The input rows of the row segments of one stage.  With row runs, segments in
// a row of one image whose input rows overlap or touch form one run, copied as
// one contiguous block of whole NHWC rows (a 3x3 stride-2 stem reads 9 rows for
// 4 output rows, not 12); rows outside the image are never copied (they read
// as zero padding).  Otherwise every segment gets its Kh rows, one copy each.
// emit(n, first_row, rows, raw_row) is called per copy.  info[j] (when given)
// receives what the transform warps need of segment j: the raw-buffer row that
// holds its kernel row 0 (it may lie before the copied rows when that row is
// padding), its live kernel rows kh_lo | kh_hi << 8 (kh_lo > kh_hi: none), the
// input column of its first pixel's tap kw = 0, and its pixel count (0 past
// the last segment).
// `t` is the stage's first segment, tile * rows_per_tile.
template <typename F>
__device__ __forceinline__ void stage_rows(const SmallKParams& p, int tile, SkSeg t, int4* info, F&& emit) {
    const int R = p.rows_per_tile;
    int run_n = -1, run_lo = 0, run_hi = -1, raw0 = 0, next_raw = 0;
    for (int j = 0; j < R; ++j, next_segment(p, t)) {
        if (tile * R + j >= p.num_segments) {
            if (info) info[j] = make_int4(0, 1, 0, 0);
            continue;
        }
        const int top = t.ho * p.g.S - p.g.P;  // input row of kernel row 0
        // live kernel rows: top + kh*D inside [0, H)
        int kh_lo, kh_last;
        if (p.g.D == 1) {
            kh_lo = top >= 0 ? 0 : -top;
            kh_last = p.g.H - 1 - top;
        } else {
            kh_lo = top >= 0 ? 0 : (-top + p.g.D - 1) / p.g.D;
            kh_last = (p.g.H - 1 - top) >= 0 ? (p.g.H - 1 - top) / p.g.D : -1;
        }
        const int kh_hi = kh_last < p.g.Kh - 1 ? kh_last : p.g.Kh - 1;
        int base;
        if (!p.row_runs) {
            base = j * p.g.Kh;
            for (int kh = kh_lo; kh <= kh_hi; ++kh) emit(t.n, top + kh * p.g.D, 1, j * p.g.Kh + kh);
        } else if (kh_lo > kh_hi) {  // every kernel row is padding
            base = 0;
        } else {
            const int lo = top + kh_lo, hi = top + kh_hi;  // D = 1 in run mode
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
            base = raw0 + (top - run_lo);
        }
        if (info) info[j] = make_int4(base, kh_lo | (kh_hi << 8), t.wo0 * p.g.S - p.g.P, t.npix);
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
    tc_smallk_kernel(const SmallKParams p) {
    extern __shared__ uint8_t smem_raw[];
    const SkSmem sm = carve(smem_raw, p);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = sm.abort;
    const int R = p.rows_per_tile;
    const int n_tile = p.g.C_out;

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
        mbar_init(sm.ready, kSkThreads - 32);
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

    if (warp != 0) {
        // Resident operands, loaded by every warp but the producer's while its first
        // input copies are in flight.  Weights: row co = w[co][0..ktot), zero beyond
        // ktot, swizzled.
        const int t0 = threadIdx.x - 32, nt = kSkThreads - 32;
        // every global load of a round is issued before its stores (one memory latency per round)
        const bool has_c = t0 < p.g.C_out;  // C_out <= 256 < nt: one channel per thread
        float bias_v = 0.f, scale_v = 1.f;
        if (has_c) {
            if (p.bias) bias_v = p.bias[t0];
            if (p.scale) scale_v = p.scale[t0];
        }
        const uint16_t* w16 = reinterpret_cast<const uint16_t*>(p.w);
        const int kw = p.a_row_bytes / 2;
        const int wtotal = p.g.C_out * kw;
        for (int base = t0; base < wtotal; base += 4 * nt) {
            uint16_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int idx = base + u * nt;
                const int co = idx / kw;
                const int k = idx - co * kw;
                v[u] = (idx < wtotal && k < p.ktot) ? w16[static_cast<long long>(co) * p.ktot + k] : uint16_t(0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int idx = base + u * nt;
                if (idx < wtotal) {
                    const int co = idx / kw;
                    *reinterpret_cast<uint16_t*>(sm.b + sw_offset(co, idx - co * kw, p.a_row_bytes)) = v[u];
                }
            }
        }
        fence_proxy_async_smem();
        // K index -> (kh, kw, ci) decomposition, once per CTA (no divisions in the gather loop)
        for (int k = t0; k < 64; k += nt) {
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
        if (has_c) {
            sm.bias[t0] = bias_v;
            sm.scale[t0] = scale_v;
        }
        mbar_arrive(sm.ready);
        if (!mbar_wait(sm.ready, 0, abort)) record_status(p.status, kStatusTimeoutTransform, abort);
    }

    if (warp == 0) {
        // ------------------------------------------------------------ bulk-copy producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            const char* xb = reinterpret_cast<const char*>(p.x);
            SkStageWalk walk(p);
            // One segment per output row and whole images per stage: a stage is R consecutive
            // rows of one image, and its input rows are one run in closed form.
            const bool whole_rows = p.segs == 1 && p.row_runs && p.g.H_out % R == 0;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
                    record_status(p.status, kStatusTimeoutProducer, abort);
                    break;
                }
                // segment info for the transform warps, then one copy per run of rows; the
                // stage's arrival comes last, after every copy's bytes are expected
                uint8_t* dst = sm.raw + stage * p.raw_bytes;
                auto emit = [&](int n, int row, int rows, int raw_row) {
                    const uint32_t bytes = static_cast<uint32_t>(rows * p.row_bytes);
                    mbar_expect_tx(&sm.raw_full[stage], bytes);
                    bulk_load(dst + raw_row * p.row_bytes, xb + (static_cast<long long>(n) * p.g.H + row) * p.row_bytes,
                              bytes, &sm.raw_full[stage]);
                };
                if (whole_rows) {
                    const int top0 = walk.t.ho * p.g.S - p.g.P;  // input row of kernel row 0, first row
                    const int lo = max(top0, 0);
                    const int hi = min(top0 + (R - 1) * p.g.S + p.g.Kh - 1, p.g.H - 1);
                    int4* info = sm.seg_info + stage * kSkMaxRows;
                    for (int j = 0; j < R; ++j) {
                        const int top = top0 + j * p.g.S;
                        const int kh_lo = max(0, -top), kh_hi = min(p.g.Kh - 1, p.g.H - 1 - top);
                        info[j] = make_int4(kh_lo <= kh_hi ? top - lo : 0, kh_lo | (kh_hi << 8), -p.g.P, p.g.W_out);
                    }
                    if (hi >= lo) emit(walk.t.n, lo, hi - lo + 1, 0);
                } else {
                    stage_rows(p, tile, walk.t, sm.seg_info + stage * kSkMaxRows, emit);
                }
                mbar_arrive(&sm.raw_full[stage]);
                walk.next(p);
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
            // descriptor of A tile 0; tile i starts a_tile_bytes * i further (address field in 16-byte units)
            const uint64_t adesc0 = a_desc(p, smem_addr(sm.a));
            const uint32_t tile16 = a_tile_bytes(p) >> 4;
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
                const uint64_t adesc_s = adesc0 + static_cast<uint64_t>(stage * R) * tile16;
                const uint32_t d_s = tmem_base + static_cast<uint32_t>(buf * R * n_tile);
                for (int k = 0; k < p.kmma; ++k)
                    for (int j = 0; j < rows; ++j)
                        mma_bf16(d_s + static_cast<uint32_t>(j * n_tile), adesc_s + static_cast<uint64_t>(j) * tile16 + 2 * k,
                                 bdesc + 2 * k, idesc, k != 0 ? 1u : 0u);
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
        // stages drain at once).  One 32-column TMEM load at a time keeps the
        // epilogue within its registers (a second buffer spilled and measured slower;
        // 16-column halves, each load in flight during the other's stores, slower too).
        const int quarter = warp & 3;
        const int group = (warp - 2) >> 2;
        const int chunks = n_tile / 32;
        int local = 0;
        SkStageWalk walk(p);
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local, walk.next(p)) {
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
                SkSeg t = walk.t;  // segment tile * R + j
                for (int q = 0; q < j; ++q) next_segment(p, t);
                if (quarter * 32 + lane < t.npix) {
                    const int wo = t.wo0 + quarter * 32 + lane;
                    float f[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
                    if (p.scale) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) f[i] *= sm.scale[c + i];
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] += sm.bias[c + i];
                    uint4* dst = reinterpret_cast<uint4*>(
                        p.y + ((static_cast<long long>(t.n) * p.g.H_out + t.ho) * p.g.W_out + wo) * p.g.C_out + c);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w4;
                        if (p.relu) {
                            w4.x = pack_bf16x2_relu(f[8 * q4 + 0], f[8 * q4 + 1]);
                            w4.y = pack_bf16x2_relu(f[8 * q4 + 2], f[8 * q4 + 3]);
                            w4.z = pack_bf16x2_relu(f[8 * q4 + 4], f[8 * q4 + 5]);
                            w4.w = pack_bf16x2_relu(f[8 * q4 + 6], f[8 * q4 + 7]);
                        } else {
                            w4.x = pack_bf16x2(f[8 * q4 + 0], f[8 * q4 + 1]);
                            w4.y = pack_bf16x2(f[8 * q4 + 2], f[8 * q4 + 3]);
                            w4.z = pack_bf16x2(f[8 * q4 + 4], f[8 * q4 + 5]);
                            w4.w = pack_bf16x2(f[8 * q4 + 6], f[8 * q4 + 7]);
                        }
                        dst[q4] = w4;
                    }
                }
            };
            for (int it = 0; it < items; ++it) {
                uint32_t va[32];
                __syncwarp();
                tmem_ld32(t_addr(it), va);
                tmem_ld_wait(va);
                process(va, it);
            }
            tc_fence_before();
            mbar_arrive(&sm.tempty[buf]);
        }
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
            uint32_t done_mask = 0;  // bit q: this thread's q-th row was packed by the fast path
            if constexpr (CIN == 3 && KH == 3 && KW == 3) {
                // Adjacent taps (D = 1): each kernel row's 9 values (3 taps x 3 channels) are
                // one contiguous run of the input row; read it as 5 words, realign by the
                // run's 16-bit parity, zero the taps outside the row (a run that starts or
                // ends up to two pixels outside reads a few bytes of the neighbouring shared
                // memory, then masks them) and pack the three runs back to back.  A thread's
                // (at most 3) rows issue all their loads before any packing, so their
                // shared-memory latencies overlap.
                if (p.g.D == 1) {
                    uint32_t wv[3][3][5];
                    uint32_t hm[3], shq[3];
                    uint8_t* arow_q[3];
                    int rq[3];
#pragma unroll
                    for (int q = 0; q < 3; ++q) {
                        const int idx = tid + q * kSkTransformThreads;
                        hm[q] = 0;
                        shq[q] = 0;
                        rq[q] = 0;
                        arow_q[q] = sm.a;
                        if (idx >= R * 128) continue;
                        const int j = idx >> 7, r = idx & 127;
                        const int4 info = sm.seg_info[stage * kSkMaxRows + j];
                        if (r >= info.w) {  // past the segment: its products are never stored
                            done_mask |= 1u << q;
                            continue;
                        }
                        const int kh_lo = info.y & 0xff, kh_hi = info.y >> 8;
                        const int wbase = info.z + r * p.g.S;  // input column of tap kw = 0
                        if (kh_lo > kh_hi || wbase < -2 || wbase >= p.g.W) continue;  // generic path
                        const int o = wbase * 3;
                        shq[q] = static_cast<uint32_t>(o & 1) * 16u;
#pragma unroll
                        for (int kw = 0; kw < 3; ++kw)
                            if (wbase + kw >= 0 && wbase + kw < p.g.W) hm[q] |= 7u << (3 * kw);
                        const uint16_t* src = raw16 + stage * raw_elems + info.x * row_elems;
#pragma unroll
                        for (int kh = 0; kh < 3; ++kh) {
                            const uint32_t* w32 = reinterpret_cast<const uint32_t*>(src + kh * row_elems) + (o >> 1);
                            const bool live = kh >= kh_lo && kh <= kh_hi;
#pragma unroll
                            for (int i = 0; i < 5; ++i) wv[q][kh][i] = live ? w32[i] : 0u;
                        }
                        arow_q[q] = sm.a + (stage * R + j) * a_tile_bytes(p);
                        rq[q] = r;
                        done_mask |= 1u << q;
                    }
#pragma unroll
                    for (int q = 0; q < 3; ++q) {
                        if (hm[q] == 0) continue;  // not packed here (or skipped)
                        uint32_t wm[5];
#pragma unroll
                        for (int i = 0; i < 5; ++i)
                            wm[i] = (((hm[q] >> (2 * i)) & 1u) ? 0x0000ffffu : 0u) |
                                    (((hm[q] >> (2 * i + 1)) & 1u) ? 0xffff0000u : 0u);
                        uint32_t a[3][5];
#pragma unroll
                        for (int kh = 0; kh < 3; ++kh) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                a[kh][i] = __funnelshift_r(wv[q][kh][i], wv[q][kh][i + 1], shq[q]) & wm[i];
                            a[kh][4] = (wv[q][kh][4] >> shq[q]) & wm[4];
                        }
                        const uint4 q0 = make_uint4(a[0][0], a[0][1], a[0][2], a[0][3]);
                        const uint4 q1 = make_uint4(a[0][4] | (a[1][0] << 16), __funnelshift_r(a[1][0], a[1][1], 16),
                                                    __funnelshift_r(a[1][1], a[1][2], 16),
                                                    __funnelshift_r(a[1][2], a[1][3], 16));
                        const uint4 q2 = make_uint4(__funnelshift_r(a[1][3], a[1][4], 16), a[2][0], a[2][1], a[2][2]);
                        const uint4 q3 = make_uint4(a[2][3], a[2][4], 0u, 0u);
                        uint8_t* arow = arow_q[q];
                        const int r = rq[q];
                        *reinterpret_cast<uint4*>(arow + sw_offset(r, 0, p.a_row_bytes)) = q0;
                        *reinterpret_cast<uint4*>(arow + sw_offset(r, 8, p.a_row_bytes)) = q1;
                        *reinterpret_cast<uint4*>(arow + sw_offset(r, 16, p.a_row_bytes)) = q2;
                        *reinterpret_cast<uint4*>(arow + sw_offset(r, 24, p.a_row_bytes)) = q3;
                    }
                }
            }
            for (int idx = tid, q = 0; idx < R * 128; idx += kSkTransformThreads, ++q) {
                if (q < 3 && ((done_mask >> q) & 1u)) continue;  // packed by the fast path
                const int j = idx >> 7;   // row segment within the stage
                const int r = idx & 127;  // A row = pixel within the segment
                uint8_t* arow = sm.a + (stage * R + j) * a_tile_bytes(p);
                const int4 info = sm.seg_info[stage * kSkMaxRows + j];
                if (r >= info.w) continue;  // past the segment: its products are never stored
                const int kh_lo = info.y & 0xff, kh_hi = info.y >> 8;
                // input rows that exist (the rest read as zero)
                const unsigned long long rowmask =
                    kh_lo <= kh_hi ? ((2ull << kh_hi) - 1) & ~((1ull << kh_lo) - 1) : 0ull;
                const int wbase = info.z + r * p.g.S;  // input column of tap kw = 0
                const uint16_t* src = raw16 + stage * raw_elems + info.x * row_elems;
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
static cudaError_t launch_sk(const SmallKParams& p, int grid, cudaStream_t stream) {
    static SmemLimitCache limits;
    cudaError_t e =
        ensure_smem_limit(reinterpret_cast<const void*>(tc_smallk_kernel<CIN, KH, KW>), p.smem_bytes, limits);
    if (e != cudaSuccess) return e;
    tc_smallk_kernel<CIN, KH, KW><<<grid, kSkThreads, p.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_tc_smallk(const SmallKParams& p, int grid, cudaStream_t stream) {
    if (p.g.C_in == 3 && p.g.Kh == 3 && p.g.Kw == 3) return launch_sk<3, 3, 3>(p, grid, stream);
    return launch_sk<0, 0, 0>(p, grid, stream);
}

}  // namespace convgb
