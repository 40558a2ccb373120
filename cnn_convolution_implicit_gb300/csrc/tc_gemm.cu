// tc_gemm.cu -- BF16 convolution as an implicit GEMM on tcgen05 tensor cores.
//
// The convolution-as-GEMM mapping of "GPU lesson 9: how a GPU executes
// neural-network convolution" (lincklin.cn), section 19 (M = C_out,
// N = N*H_out*W_out, K = C_in*Kh*Kw), computed as an implicit GEMM (section
// 11; "Convolution variants and their matrix operations", lpnh.cn/news/2674933,
// section 3.3): the im2col matrix is never stored.  Each K-step is one kernel
// tap (kh, kw) and one 64-channel block, and the TMA engine gathers the 128
// input pixels of that tap straight from the NHWC tensor:
//   * stride 1 (kTcModeRect): the output tile is a rectangle of TH x TW pixels,
//     and the tap's input pixels are the same rectangle shifted by
//     (kh*D - P, kw*D - P) -- one 4-D tiled box;
//   * other strides (kTcModeIm2col): 128 consecutive output pixels, loaded in
//     the TMA's im2col mode with per-tap offsets (kw*D, kh*D);
//   * 1x1 / stride 1 / pad 0 (kTcMode1x1): a plain GEMM (lesson 9, section
//     21) over the [pixels][C_in] matrix.
// Out-of-bounds input reads zero-fill, which is the zero padding (lesson 9,
// section 26); the tap offsets read only the Kh*Kw live taps of a dilated
// kernel (variants page, section 4.2).
//
// Operand roles on the tensor core: the MMA's M side is the pixel tile (128
// TMEM lanes), its N side the output channels; D = Y^T of the logical GEMM, so
// each TMEM lane holds one output pixel's contiguous NHWC channel vector.
// Groups are independent GEMMs (variants page, sections 2.2 and 4.3): a tile
// packs `gpc` groups side by side in TMEM columns, each with its own K loop.
//
// Warp roles (576 threads, 608 in halo mode; one CTA per SM, persistent over tiles):
//   warp 0      TMA producer (one lane): A (pixels x 64 ch) and B (C_out x 64) per
//               K-step; in halo mode the halos only
//   warp 18     halo mode: TMA producer (one lane) of the weight stages
//   warp 1      TMEM allocator; one lane issues tcgen05.mma and commits
//   warps 2..17 epilogue, four groups of four, two per TMEM accumulator (each
//               group drains half of its columns): tcgen05.ld -> +bias -> ReLU ->
//               BF16 -> swizzled smem -> TMA store, 32 columns per step
// Shared memory holds a ring of `stages` (A, B) buffers; TMEM holds two
// accumulators so the epilogue of tile i overlaps the MMAs of tile i+1.
//
// PAIR = true runs the same pipeline on a cluster of two CTAs (two SMs): one
// tcgen05.mma.cta_group::2 per K slice computes 256 pixels x N, each CTA
// loading its own 128-pixel A tile and half of the weight rows (N/2).  The
// leader CTA (cluster rank 0) issues the MMAs; both CTAs' TMA loads complete
// on the leader's `full` barrier; the MMA commits arrive on both CTAs' `empty`
// and `tfull` barriers; both CTAs' epilogue warps arrive on the leader's
// `tempty` barrier.
#include "conv_internal.h"
#include "tc_common.cuh"

namespace convgb {

namespace {

constexpr uint32_t kABytes = kTcBlockM * kTcBlockK * 2;  // 16 KB
constexpr uint32_t kOutTileBytes = 32 * 64;               // one store tile: 32 pixels x 32 channels

struct TcSmem {
    uint8_t* a;    // A ring (per-tap modes) or halo ring (halo mode)
    uint8_t* b;
    uint8_t* out;  // per epilogue warp: two store tiles
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint64_t* hfull;   // halo mode: halo landed
    uint64_t* hempty;  // halo mode: every tap of the halo consumed
    uint64_t* bfull;   // resident weights landed
    uint32_t* tmem_slot;
    int* abort;
};

// a_bytes: one A stage (per-tap modes) or one halo stage (halo mode, p.halo_stages of them);
// b_total: the weight ring, or the resident weights.
__device__ __forceinline__ TcSmem carve(uint8_t* raw, const TcGemmParams& p, uint32_t a_bytes, uint32_t b_total) {
    TcSmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int a_stages = p.halo ? p.halo_stages : p.stages;
    s.a = base;
    s.b = s.a + a_stages * a_bytes;
    s.out = s.b + b_total;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.out + 8 * 2 * kOutTileBytes);
    s.full = bars;
    s.empty = bars + p.stages;
    s.tfull = bars + 2 * p.stages;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.hfull = s.drain + 1;
    s.hempty = s.hfull + kTcMaxHaloStages;
    s.bfull = s.hempty + kTcMaxHaloStages;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.bfull + 1);
    s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
    return s;
}

// Sub-GEMM j of n-tile nt: its group and first weight row.
__device__ __forceinline__ void sub_gemm(const TcGemmParams& p, int nt, int j, int& grp, int& brow) {
    if (p.g.cout_g >= p.n_tile) {  // one group spans one or more n-tiles
        brow = nt * p.n_tile;
        grp = brow / p.g.cout_g;
    } else {                       // several groups packed in one n-tile
        grp = nt * p.gpc + j;
        brow = grp * p.g.cout_g;
    }
}

// Where pixel tile m sits.  Linear modes: pixels [m*128, m*128 + 128) in
// (n, ho, wo) order.  Rect and halo modes: image n, rows [ho0, ho0 + TH), cols
// [wo0, wo0 + TW).
struct PixTile {
    long long pix0;
    int n, ho0, wo0;
    int rh, rw;   // phase mode: the tile's output phase (h mod S, w mod S); ho0, wo0 are phase-grid coordinates
    bool exists;  // m is a real tile (the pair kernel may run one past the end)
};

template <bool PHASE, bool PAIR = false>
__device__ __forceinline__ PixTile pix_tile(const TcGemmParams& p, int m) {
    PixTile t;
    t.exists = m < p.num_m_tiles;
    t.rh = t.rw = 0;
    if constexpr (PHASE) {  // phases fastest: neighbouring tiles read the same input rectangle
        const int nph = p.ps * p.ps;
        const int per_img = p.rect_tiles_h * p.rect_tiles_w;
        int ph, q;
        if constexpr (PAIR) {  // a pair is two neighbouring tiles of one phase (one tap list for both)
            const int pr = m >> 1;
            ph = pr % nph;
            q = (pr / nph) * 2 + (m & 1);
            t.exists = t.exists && q < p.g.N * per_img;  // an odd tile count leaves one tile unpaired
        } else {
            ph = m % nph;
            q = m / nph;
        }
        t.rh = ph / p.ps;
        t.rw = ph - t.rh * p.ps;
        t.n = q / per_img;
        const int r = q - t.n * per_img;
        const int th = r / p.rect_tiles_w;
        t.ho0 = th * p.rect_h;
        t.wo0 = (r - th * p.rect_tiles_w) * p.rect_w;
        t.pix0 = 0;
    } else if (p.mode == kTcModeRect || p.mode == kTcModeHalo) {
        const int per_img = p.rect_tiles_h * p.rect_tiles_w;
        t.n = m / per_img;
        const int r = m - t.n * per_img;
        const int th = r / p.rect_tiles_w;
        t.ho0 = th * p.rect_h;
        t.wo0 = (r - th * p.rect_tiles_w) * p.rect_w;
        t.pix0 = 0;
    } else {
        const int HWo = p.g.H_out * p.g.W_out;
        t.pix0 = static_cast<long long>(m) * kTcBlockM;
        t.n = static_cast<int>(t.pix0 / HWo);
        const int rem = static_cast<int>(t.pix0 - static_cast<long long>(t.n) * HWo);
        t.ho0 = rem / p.g.W_out;
        t.wo0 = rem - t.ho0 * p.g.W_out;
    }
    return t;
}

// K-steps of one sub-GEMM of a tile: taps x 64-channel blocks (phase mode: the
// taps of the tile's phase only).
template <bool PHASE>
__device__ __forceinline__ int tile_ksteps(const TcGemmParams& p, int rh, int rw) {
    if constexpr (PHASE) return p.ph.cnt[rh] * p.pw.cnt[rw] * p.kblk;
    return p.ksteps;
}

// One tap of a tile's K loop: kernel indices, input offsets (rect / phase
// modes) and the weight tap it multiplies.
struct Tap {
    int kh, kw, dh, dw, wtap;
};

// A operand of one K-step: 128 pixels x 64 channels of tap (kh, kw).
template <bool PAIR, bool PHASE>
__device__ __forceinline__ void load_a(const TcGemmParams& p, const CUtensorMap* map, uint8_t* dst, uint64_t* bar,
                                       uint32_t bar_cluster, const PixTile& t, int c, const Tap& tp) {
    const int kh = tp.kh, kw = tp.kw;
    if (!PHASE && p.mode == kTcMode1x1) {
        if constexpr (PAIR)
            tma_load_2d_pair(dst, map, bar_cluster, c, static_cast<int>(t.pix0));
        else
            tma_load_2d(dst, map, bar, c, static_cast<int>(t.pix0));
    } else if (PHASE || p.mode == kTcModeRect) {
        const int w = t.wo0 + tp.dw, h = t.ho0 + tp.dh;
        if constexpr (PAIR)
            tma_load_4d_pair(dst, map, bar_cluster, c, w, h, t.n);
        else
            tma_load_4d(dst, map, bar, c, w, h, t.n);
    } else {
        const int w = t.wo0 * p.g.S - p.g.P, h = t.ho0 * p.g.S - p.g.P;
        const uint16_t ow = static_cast<uint16_t>(kw * p.g.D), oh = static_cast<uint16_t>(kh * p.g.D);
        if constexpr (PAIR)
            tma_load_im2col_4d_pair(dst, map, bar_cluster, c, w, h, t.n, ow, oh);
        else
            tma_load_im2col_4d(dst, map, bar, c, w, h, t.n, ow, oh);
    }
}

// ---------------------------------------------------------------- halo mode
// The halo mode's K loop runs channel blocks outer, taps inner: a "block" is
// one (unit, sub-GEMM, 64-channel block) and owns one halo; its Kh*Kw taps each
// take one weight stage.  A CTA walks its blocks with running counters (the
// producer keeps two walkers, one for the halos it issues ahead and one for the
// weights): only a new unit costs divisions, to place its pixel tile.
struct HaloWalk {
    int u, nt, j, kb;  // unit, its n-tile, sub-GEMM, channel block
    int c, brow;       // first input channel and first weight row of the block
    int w0, h0, n;     // the halo box origin of the unit's tile
};

template <bool PAIR, bool DUAL>
__device__ __forceinline__ void halo_walk_block(const TcGemmParams& p, HaloWalk& w) {
    int grp, brow;
    sub_gemm(p, w.nt, w.j, grp, brow);
    w.c = grp * p.g.cin_g + w.kb * kTcBlockK;
    w.brow = brow;
}

template <bool PAIR, bool DUAL>
__device__ __forceinline__ void halo_walk_unit(const TcGemmParams& p, HaloWalk& w, uint32_t rank) {
    const int mu = w.u / p.num_n_tiles;
    w.nt = w.u - mu * p.num_n_tiles;
    const int m = PAIR ? 2 * mu + static_cast<int>(rank) : (DUAL ? 2 * mu : mu);
    PixTile t = pix_tile<false, PAIR || DUAL>(p, m);
    if (!t.exists) t = pix_tile<false, PAIR || DUAL>(p, p.num_m_tiles - 1);  // loaded, never stored
    w.w0 = t.wo0 - p.g.P;
    w.h0 = t.ho0 - p.g.P;
    w.n = t.n;
    halo_walk_block<PAIR, DUAL>(p, w);
}

template <bool PAIR, bool DUAL>
__device__ __forceinline__ void halo_walk_start(const TcGemmParams& p, HaloWalk& w, int unit0, uint32_t rank) {
    w.u = unit0;
    w.j = w.kb = 0;
    halo_walk_unit<PAIR, DUAL>(p, w, rank);
}

template <bool PAIR, bool DUAL>
__device__ __forceinline__ void halo_walk_next(const TcGemmParams& p, HaloWalk& w, int unit_step, int num_units,
                                               uint32_t rank) {
    if (++w.kb < p.kblk) {
        halo_walk_block<PAIR, DUAL>(p, w);
        return;
    }
    w.kb = 0;
    if (++w.j < p.gpc) {
        halo_walk_block<PAIR, DUAL>(p, w);
        return;
    }
    w.j = 0;
    w.u += unit_step;
    if (w.u < num_units) halo_walk_unit<PAIR, DUAL>(p, w, rank);
}

// Every fill of a ring this thread issued has landed (the leader sees its full
// barriers complete; a pair's peer sees the MMA release each slot, which needs
// the fill landed), so the CTA may exit with no copy in flight.
__device__ __forceinline__ void drain_ring(uint64_t* full, uint64_t* empty, int stages, long long issued, bool leader,
                                           unsigned* status, volatile int* abort) {
    for (int s = 0; s < stages; ++s) {
        const long long fills = issued / stages + (s < issued % stages ? 1 : 0);
        if (fills == 0) continue;
        const uint32_t par = static_cast<uint32_t>((fills - 1) & 1);
        const bool done = leader ? mbar_wait(&full[s], par, nullptr) : mbar_wait(&empty[s], par, nullptr);
        if (!done) record_status(status, kStatusTimeoutDrain, abort);
    }
}

// Producers (one thread per role).  ROLE 0 issues the blocks' halos in order,
// up to halo_stages ahead of the MMAs; ROLE 1 issues the weight stages.  A weight
// stage holds `btaps` consecutive taps of one block (the last stage of a block
// may hold fewer), so every barrier wait of the MMA issuer is followed by enough
// MMAs to cover its latency.  Each role drains its own ring before returning.
// RESB (resident weights, one SM per unit): ROLE 1 loads the n-tile's rows for every
// channel block and tap once, and the MMAs read them in place.
template <bool PAIR, bool DUAL, int ROLE, bool RESB = false>
__device__ __forceinline__ void halo_producer(const TcGemmParams& p, const CUtensorMap* a_map,
                                              const CUtensorMap* b_map, const TcSmem& sm, int unit0, int unit_step,
                                              int num_units, uint32_t rank, bool leader, volatile int* abort) {
    const int T = p.g.Kh * p.g.Kw;
    const int my_units = unit0 < num_units ? (num_units - 1 - unit0) / unit_step + 1 : 0;
    const int nblocks = my_units * p.gpc * p.kblk;
    if (nblocks == 0) return;
    HaloWalk w;
    halo_walk_start<PAIR, DUAL>(p, w, unit0, rank);
    long long issued = 0;
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    if constexpr (ROLE == 0) {
        const int HS = p.halo_stages;
        const uint32_t h_tx = (PAIR ? 2u : 1u) * static_cast<uint32_t>(p.halo_w * p.halo_h) * 128u;
        for (int blk = 0; blk < nblocks; ++blk) {
            if (!mbar_wait(&sm.hempty[st], ph ^ 1u, abort)) {
                record_status(p.status, kStatusTimeoutProducer, abort);
                break;
            }
            if (leader) mbar_arrive_expect_tx(&sm.hfull[st], h_tx);
            uint8_t* dst = sm.a + st * p.halo_bytes;
            if constexpr (PAIR)
                tma_load_4d_pair(dst, a_map, mapa_shared(smem_addr(&sm.hfull[st]), 0), w.c, w.w0, w.h0, w.n);
            else
                tma_load_4d(dst, a_map, &sm.hfull[st], w.c, w.w0, w.h0, w.n);
            ++issued;
            if (++st == HS) {
                st = 0;
                ph ^= 1u;
            }
            if (blk + 1 < nblocks) halo_walk_next<PAIR, DUAL>(p, w, unit_step, num_units, rank);
        }
        drain_ring(sm.hfull, sm.hempty, HS, issued, leader, p.status, abort);
    } else if constexpr (RESB) {
        static_assert(!PAIR, "resident weights run one SM per unit");
        const uint32_t b_tap = static_cast<uint32_t>(p.mma_n) * 128u;
        mbar_arrive_expect_tx(sm.bfull, b_tap * static_cast<uint32_t>(T * p.kblk));
        for (int kb = 0; kb < p.kblk; ++kb)
            for (int tap = 0; tap < T; ++tap)
                tma_load_2d(sm.b + (kb * T + tap) * b_tap, b_map, sm.bfull, tap * p.g.cin_g + kb * kTcBlockK, w.brow);
        if (!mbar_wait(sm.bfull, 0, nullptr)) record_status(p.status, kStatusTimeoutDrain, abort);
    } else {
        const int BT = p.btaps, BS = p.stages;
        const int b_rows = PAIR ? p.mma_n / 2 : p.mma_n;
        const uint32_t b_tap = static_cast<uint32_t>(b_rows) * 128u;  // one tap's weight rows in this CTA
        const uint32_t b_tx = (PAIR ? 2u : 1u) * b_tap;
        for (int blk = 0; blk < nblocks && ok; ++blk) {
            for (int tap0 = 0; tap0 < T; tap0 += BT) {
                if (!mbar_wait(&sm.empty[st], ph ^ 1u, abort)) {
                    record_status(p.status, kStatusTimeoutProducer, abort);
                    ok = false;
                    break;
                }
                const int nt = T - tap0 < BT ? T - tap0 : BT;
                if (leader) mbar_arrive_expect_tx(&sm.full[st], b_tx * static_cast<uint32_t>(nt));
                uint8_t* b_dst = sm.b + st * b_tap * static_cast<uint32_t>(BT);
                const uint32_t full_leader = PAIR ? mapa_shared(smem_addr(&sm.full[st]), 0) : 0u;
                for (int i = 0; i < nt; ++i) {
                    const int kcol = (tap0 + i) * p.g.cin_g + w.kb * kTcBlockK;
                    if constexpr (PAIR)
                        tma_load_2d_pair(b_dst + i * b_tap, b_map, full_leader, kcol,
                                         w.brow + static_cast<int>(rank) * b_rows);
                    else
                        tma_load_2d(b_dst + i * b_tap, b_map, &sm.full[st], kcol, w.brow);
                }
                ++issued;
                if (++st == BS) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (blk + 1 < nblocks) halo_walk_next<PAIR, DUAL>(p, w, unit_step, num_units, rank);
        }
        drain_ring(sm.full, sm.empty, BS, issued, leader, p.status, abort);
    }
}

// MMA issuer (one thread of the leader).  Per block: wait for its halo; per
// weight stage: wait once, then for each of its taps issue the K = 64 slice as
// four K = 16 MMAs whose A descriptor starts at the tap's shifted halo row.
// part: 0 or 1 = only that pixel tile's MMAs (two tiles per CTA, one issuing thread per
// tile), 2 = every MMA.
template <bool PAIR, bool DUAL, bool RESB = false>
__device__ __forceinline__ void halo_mma(const TcGemmParams& p, const TcSmem& sm, uint32_t tmem_base, int unit0,
                                         int unit_step, int num_units, volatile int* abort, int part) {
    const uint32_t idesc = idesc_bf16_f32((PAIR ? 2 : 1) * kTcBlockM, p.mma_n);
    const int T = p.g.Kh * p.g.Kw;
    const int BT = RESB ? T : p.btaps;  // resident weights: every tap of a block after one halo wait
    const int b_rows = PAIR ? p.mma_n / 2 : p.mma_n;
    const uint32_t b_tap = static_cast<uint32_t>(b_rows) * 128u;
    const uint32_t b_stage = b_tap * static_cast<uint32_t>(BT);
    const uint32_t sbo = static_cast<uint32_t>(p.halo_w) * 128u;   // 8 output rows apart: one halo row
    const uint32_t row_kh = static_cast<uint32_t>(p.g.D * p.halo_w) * 128u;
    const uint32_t row_kw = static_cast<uint32_t>(p.g.D) * 128u;
    int hs = 0, bs = 0;
    uint32_t hph = 0, bph = 0;
    int local = 0;
    bool ok = true;
    if (RESB && unit0 < num_units && !mbar_wait(sm.bfull, 0, abort)) {
        record_status(p.status, kStatusTimeoutMma, abort);
        ok = false;
    }
    for (int u = unit0; u < num_units && ok; u += unit_step, ++local) {
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
        const bool free_acc = PAIR ? mbar_wait_cluster(&sm.tempty[buf], use ^ 1u, abort)
                                   : mbar_wait(&sm.tempty[buf], use ^ 1u, abort);
        if (!free_acc) {
            record_status(p.status, kStatusTimeoutMma, abort);
            break;
        }
        tc_fence_after();
        const uint32_t d_base = tmem_base + static_cast<uint32_t>(buf * (DUAL ? 2 : 1) * p.n_tile);
        for (int j = 0; j < p.gpc && ok; ++j) {
            const uint32_t d = d_base + static_cast<uint32_t>(j * p.mma_n);
            for (int kb = 0; kb < p.kblk && ok; ++kb) {
                if (!mbar_wait(&sm.hfull[hs], hph, abort)) {
                    record_status(p.status, kStatusTimeoutMma, abort);
                    ok = false;
                    break;
                }
                const uint32_t hbase = smem_addr(sm.a + hs * p.halo_bytes);
                int kh = 0, kw = 0;
                for (int tap0 = 0; tap0 < T; tap0 += BT) {
                    if (!RESB && !mbar_wait(&sm.full[bs], bph, abort)) {
                        record_status(p.status, kStatusTimeoutMma, abort);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nt = T - tap0 < BT ? T - tap0 : BT;
                    const uint32_t bbase = RESB ? smem_addr(sm.b) + static_cast<uint32_t>(kb * T) * b_tap
                                                : smem_addr(sm.b + bs * b_stage);
                    for (int i = 0; i < nt; ++i) {
                        const uint32_t a_addr =
                            hbase + static_cast<uint32_t>(kh) * row_kh + static_cast<uint32_t>(kw) * row_kw;
                        const uint64_t adesc = sdesc_sw128_rows(a_addr, sbo);
                        const uint64_t bdesc = sdesc_sw128(bbase + static_cast<uint32_t>(i) * b_tap);
                        const uint32_t first = (kb | tap0 | i) != 0 ? 1u : 0u;
                        if (!DUAL || part != 1) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                if constexpr (PAIR)
                                    mma_bf16_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, (first | k) != 0 ? 1u : 0u);
                                else
                                    mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, (first | k) != 0 ? 1u : 0u);
                            }
                        }
                        if (DUAL && part != 0) {
                            const uint64_t adesc1 = sdesc_sw128_rows(a_addr + 8u * 128u, sbo);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_bf16(d + static_cast<uint32_t>(p.n_tile), adesc1 + 2 * k, bdesc + 2 * k, idesc,
                                         (first | k) != 0 ? 1u : 0u);
                        }
                        if (++kw == p.g.Kw) {
                            kw = 0;
                            ++kh;
                        }
                    }
                    if constexpr (!RESB) {
                        if constexpr (PAIR)
                            mma_commit_pair(&sm.empty[bs], 0x3);
                        else
                            mma_commit(&sm.empty[bs]);
                        if (++bs == p.stages) {
                            bs = 0;
                            bph ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    mma_commit_pair(&sm.hempty[hs], 0x3);
                else
                    mma_commit(&sm.hempty[hs]);
                if (++hs == p.halo_stages) {
                    hs = 0;
                    hph ^= 1u;
                }
            }
        }
        if (ok) {
            if constexpr (PAIR)
                mma_commit_pair(&sm.tfull[buf], 0x3);
            else
                mma_commit(&sm.tfull[buf]);
        }
    }
    if constexpr (PAIR)
        mma_commit_pair(sm.drain, 0x1);
    else
        mma_commit(sm.drain);
    if (!mbar_wait(sm.drain, 0, nullptr)) record_status(p.status, kStatusTimeoutDrain, abort);
}

}  // namespace

// PHASE: the transposed-convolution phase mode (kTcModePhase), compiled
// separately so the convolution modes keep their own loops.
// DUAL: two pixel tiles per CTA (M = 256 on one SM) for tiles of at most 128
// output channels: each K-step loads both tiles' A operands and one weight
// block and issues the MMAs of both into two accumulators, so the producer's
// per-K-step work feeds twice the tensor work.
// HALO: the halo mode (kTcModeHalo, stride 1): one input halo per 64-channel
// block feeds every tap through shifted descriptors.
// RESB: resident weights (1x1 and halo modes): every CTA keeps one n-tile (the grid
// is a multiple of the n-tile count), whose weight rows for the whole reduction load
// once into shared memory; the ring carries pixels only and the MMA issuer waits on
// A (halo) stages alone.
// SWAP: two tiles per CTA of 128 output channels (per-tap modes): the weights are the
// MMA's M = 128 operand and both tiles' 256 pixels its N, so one M128 N256 MMA per K = 16
// reads 12 KB of operands where two M128 N128 MMAs read 16 KB (the tensor core reads
// its shared-memory operands at 128 bytes per clock, which N = 128 MMAs already fill).
// TMEM then holds D with output channels on the lanes; the epilogue transposes it.
template <bool PAIR, bool PHASE, bool DUAL, bool HALO = false, bool RESB = false, bool SWAP = false>
__global__ void __launch_bounds__(tc_threads(HALO, DUAL), 1)
    tc_conv_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap b_map,
                   const __grid_constant__ CUtensorMap y_map, const TcGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    constexpr bool TWO = PAIR || DUAL;                   // work units of two pixel tiles
    // 1x1 with resident weights: every epilogue warp drains every tile (a quarter of its
    // columns each), so a tile drains in half the time; the MMAs of the next tile meanwhile
    // fill the other accumulator.  (Pointwise layer 64.4 -> 61.5 us; the per-tap and halo
    // kernels measured slower this way and keep two groups per accumulator.)
    constexpr bool ALLW = RESB && !HALO && !PAIR && !DUAL;
    constexpr uint32_t a_stage = DUAL ? 2 * kABytes : kABytes;
    const int b_rows = PAIR ? p.mma_n / 2 : p.mma_n;  // weight rows this CTA loads per K-step
    const uint32_t b_bytes = static_cast<uint32_t>(b_rows) * 128u;
    const TcSmem sm = carve(smem_raw, p, HALO ? static_cast<uint32_t>(p.halo_bytes) : a_stage,
                            RESB ? b_bytes * static_cast<uint32_t>(p.ksteps)
                                 : (HALO ? b_bytes * static_cast<uint32_t>(p.btaps) : b_bytes) *
                                       static_cast<uint32_t>(p.stages));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort = sm.abort;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // work units: a tile (single) or a pair of adjacent pixel tiles (PAIR)
    const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int unit_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int num_units = TWO ? ((p.num_m_tiles + 1) / 2) * p.num_n_tiles : p.num_tiles;

    if (threadIdx.x == 0) {
        // two tiles per CTA: both MMA-issuing threads commit to the barriers that release
        // a stage, a halo, an accumulator or the final drain
        constexpr uint32_t mma_threads = (DUAL && !SWAP) ? 2 : 1;
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], mma_threads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.tfull[b], mma_threads);
            mbar_init(&sm.tempty[b], ALLW ? 16 : (PAIR ? 2 * 8 : 8));  // one arrival per warp that drains it (both CTAs)
        }
        mbar_init(sm.drain, mma_threads);
        mbar_init(sm.bfull, 1);
        if constexpr (HALO) {
            for (int h = 0; h < p.halo_stages; ++h) {
                mbar_init(&sm.hfull[h], 1);
                mbar_init(&sm.hempty[h], mma_threads);
            }
        }
        *sm.abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&a_map);
        tma_prefetch_desc(&b_map);
        tma_prefetch_desc(&y_map);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(sm.tmem_slot, p.tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(sm.tmem_slot, p.tmem_cols);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // the peer's barriers exist before anything signals them
    tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;

    if (HALO && (warp == 0 || warp == kTcBWarp)) {
        if (lane == 0) {
            if (warp == 0)
                halo_producer<PAIR, DUAL, 0>(p, &a_map, &b_map, sm, unit0, unit_step, num_units, rank, leader, abort);
            else
                halo_producer<PAIR, DUAL, 1, RESB && HALO>(p, &a_map, &b_map, sm, unit0, unit_step, num_units, rank, leader,
                                                   abort);
        }
    } else if (HALO && (warp == 1 || (DUAL && warp == tc_mma2_warp(true)))) {
        if (lane == 0 && leader)
            halo_mma<PAIR, DUAL, RESB && HALO>(p, sm, tmem_base, unit0, unit_step, num_units, abort,
                                       DUAL ? (warp == 1 ? 0 : 1) : 2);
    } else if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            const uint32_t a_b_bytes = RESB ? (PAIR ? 2u * kABytes : a_stage)
                                            : (PAIR ? 2u * (kABytes + b_bytes) : a_stage + b_bytes);
            if (RESB && unit0 < num_units) {
                // resident weights: every CTA's units share one n-tile (the grid is a multiple of the
                // n-tile count), so its weight rows for every K-step load once
                int grp, brow;
                sub_gemm(p, unit0 % p.num_n_tiles, 0, grp, brow);
                const uint32_t bfull_leader = PAIR ? mapa_shared(smem_addr(sm.bfull), 0) : 0u;
                if (leader) mbar_arrive_expect_tx(sm.bfull, (PAIR ? 2u : 1u) * b_bytes * static_cast<uint32_t>(p.ksteps));
                for (int ks = 0; ks < p.ksteps; ++ks) {
                    if constexpr (PAIR)
                        tma_load_2d_pair(sm.b + ks * b_bytes, &b_map, bfull_leader, ks * kTcBlockK,
                                         brow + static_cast<int>(rank) * b_rows);
                    else
                        tma_load_2d(sm.b + ks * b_bytes, &b_map, sm.bfull, ks * kTcBlockK, brow);
                }
            }
            for (int u = unit0; u < num_units && ok; u += unit_step) {
                const int mu = u / p.num_n_tiles;
                const int nt = u - mu * p.num_n_tiles;
                const int m = PAIR ? 2 * mu + static_cast<int>(rank) : (DUAL ? 2 * mu : mu);
                PixTile t = pix_tile<PHASE, TWO>(p, m);
                // a missing tile loads a valid one whose result is never stored (phase mode: its own
                // coordinates, past the last image, which read as zeros: its phase stays its pair's)
                if (!t.exists && !PHASE) t = pix_tile<PHASE, TWO>(p, p.num_m_tiles - 1);
                PixTile t1 = t;  // DUAL: the second tile of the unit
                if constexpr (DUAL) {
                    t1 = pix_tile<PHASE, true>(p, m + 1);
                    if (!t1.exists && !PHASE) t1 = t;
                }
                const int ksteps = tile_ksteps<PHASE>(p, t.rh, t.rw);
                for (int j = 0; j < p.gpc && ok; ++j) {
                    int grp, brow;
                    sub_gemm(p, nt, j, grp, brow);
                    int c_kb = 0, c_kh = 0, c_kw = 0, c_tap = 0;
                    for (int ks = 0; ks < ksteps; ++ks) {
                        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
                            record_status(p.status, kStatusTimeoutProducer, abort);
                            ok = false;
                            break;
                        }
                        Tap tp;
                        int kb;
                        if constexpr (PHASE) {  // running counters over the phase's row and column taps
                            kb = c_kb;
                            tp.kh = p.ph.k[t.rh][c_kh];
                            tp.kw = p.pw.k[t.rw][c_kw];
                            tp.dh = p.ph.off[t.rh][c_kh];
                            tp.dw = p.pw.off[t.rw][c_kw];
                            tp.wtap = tp.kh * p.g.Kw + tp.kw;
                            if (++c_kb == p.kblk) {
                                c_kb = 0;
                                if (++c_kw == p.pw.cnt[t.rw]) {
                                    c_kw = 0;
                                    ++c_kh;
                                }
                            }
                        } else {  // running counters: no division per K-step
                            kb = c_kb;
                            tp.kh = c_kh;
                            tp.kw = c_kw;
                            tp.dh = c_kh * p.g.D - p.g.P;
                            tp.dw = c_kw * p.g.D - p.g.P;
                            tp.wtap = c_tap;
                            if (++c_kb == p.kblk) {
                                c_kb = 0;
                                ++c_tap;
                                if (++c_kw == p.g.Kw) {
                                    c_kw = 0;
                                    ++c_kh;
                                }
                            }
                        }
                        const int c = grp * p.g.cin_g + kb * kTcBlockK;
                        uint8_t* a_dst = sm.a + stage * a_stage;
                        uint8_t* b_dst = sm.b + stage * b_bytes;
                        const uint32_t full_leader = PAIR ? mapa_shared(smem_addr(&sm.full[stage]), 0) : 0u;
                        if (leader) mbar_arrive_expect_tx(&sm.full[stage], a_b_bytes);
                        load_a<PAIR, PHASE>(p, &a_map, a_dst, &sm.full[stage], full_leader, t, c, tp);
                        if constexpr (DUAL) load_a<PAIR, PHASE>(p, &a_map, a_dst + kABytes, &sm.full[stage], 0u, t1, c, tp);
                        const int kcol = tp.wtap * p.g.cin_g + kb * kTcBlockK;
                        if constexpr (!RESB) {
                            if constexpr (PAIR)
                                tma_load_2d_pair(b_dst, &b_map, full_leader, kcol, brow + static_cast<int>(rank) * b_rows);
                            else
                                tma_load_2d(b_dst, &b_map, &sm.full[stage], kcol, brow);
                        }
                        ++issued;
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // Drain: every fill this CTA issued has landed before it may exit.  The
            // leader sees its full barriers complete; a pair's peer sees the MMA
            // release each slot after consuming it (which needs the fill landed).
            for (int s = 0; s < p.stages; ++s) {
                const long long fills = issued / p.stages + (s < issued % p.stages ? 1 : 0);
                if (fills == 0) continue;
                const uint32_t par = static_cast<uint32_t>((fills - 1) & 1);
                const bool done = leader ? mbar_wait(&sm.full[s], par, nullptr) : mbar_wait(&sm.empty[s], par, nullptr);
                if (!done) record_status(p.status, kStatusTimeoutDrain, abort);
            }
            // the resident weights (a peer's land on the leader's barrier, which its MMA
            // waited for before releasing the stages waited on above)
            if (RESB && leader && unit0 < num_units && !mbar_wait(sm.bfull, 0, nullptr))
                record_status(p.status, kStatusTimeoutDrain, abort);
        }
    } else if (warp == 1 || (DUAL && !SWAP && warp == tc_mma2_warp(false))) {
        // ------------------------------------------------------------ MMA issuer (leader only)
        // Two tiles per CTA: warp 1 issues tile 0's MMAs and a second warp tile 1's, each
        // waiting for the same stages (one thread issues at most one MMA per ~55 clocks)
        const int part = DUAL ? (warp == 1 ? 0 : 1) : 2;
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_bf16_f32((PAIR ? 2 : 1) * kTcBlockM, p.mma_n);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            if (RESB && unit0 < num_units) {
                ok = mbar_wait(sm.bfull, 0, abort);
                if (!ok) record_status(p.status, kStatusTimeoutMma, abort);
            }
            for (int u = unit0; u < num_units && ok; u += unit_step, ++local) {
                const int buf = local & 1;
                const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
                const bool free_acc = PAIR ? mbar_wait_cluster(&sm.tempty[buf], use ^ 1u, abort)
                                           : mbar_wait(&sm.tempty[buf], use ^ 1u, abort);
                if (!free_acc) {
                    record_status(p.status, kStatusTimeoutMma, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t d_base = tmem_base + static_cast<uint32_t>(buf * (DUAL ? 2 : 1) * p.n_tile);
                int ksteps = p.ksteps;
                if constexpr (PHASE) {  // the phase of tile m (no pairs in this mode)
                    const int ph = (u / p.num_n_tiles) % (p.ps * p.ps);
                    ksteps = tile_ksteps<PHASE>(p, ph / p.ps, ph % p.ps);
                }
                for (int j = 0; j < p.gpc && ok; ++j) {
                    const uint32_t d = d_base + static_cast<uint32_t>(j * p.mma_n);
                    for (int ks = 0; ks < ksteps; ++ks) {
                        if (!mbar_wait(&sm.full[stage], phase, abort)) {
                            record_status(p.status, kStatusTimeoutMma, abort);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = sdesc_sw128(smem_addr(sm.a + stage * a_stage));
                        const uint64_t bdesc = sdesc_sw128(smem_addr(sm.b + (RESB ? ks : stage) * b_bytes));
                        if constexpr (SWAP) {
                            // weights (128 rows) x both tiles' pixels (256 rows of the stage's A block)
                            constexpr uint32_t idesc_sw = idesc_bf16_f32(kTcBlockM, 2 * kTcBlockM);
#pragma unroll
                            for (int k = 0; k < kTcBlockK / 16; ++k)
                                mma_bf16(d, bdesc + 2 * k, adesc + 2 * k, idesc_sw, (ks | k) != 0 ? 1u : 0u);
                        } else if (!DUAL || part != 1) {
#pragma unroll
                            for (int k = 0; k < kTcBlockK / 16; ++k) {
                                // +32 bytes along K inside the swizzle row = +2 in the >>4 address field
                                if constexpr (PAIR)
                                    mma_bf16_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, (ks | k) != 0 ? 1u : 0u);
                                else
                                    mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, (ks | k) != 0 ? 1u : 0u);
                            }
                        }
                        if (DUAL && part != 0) {  // the unit's second tile: A at +16 KB, its own accumulator
                            const uint64_t adesc1 = sdesc_sw128(smem_addr(sm.a + stage * a_stage + kABytes));
#pragma unroll
                            for (int k = 0; k < kTcBlockK / 16; ++k)
                                mma_bf16(d + static_cast<uint32_t>(p.n_tile), adesc1 + 2 * k, bdesc + 2 * k, idesc,
                                         (ks | k) != 0 ? 1u : 0u);
                        }
                        if constexpr (PAIR)
                            mma_commit_pair(&sm.empty[stage], 0x3);
                        else
                            mma_commit(&sm.empty[stage]);
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (ok) {
                    if constexpr (PAIR)
                        mma_commit_pair(&sm.tfull[buf], 0x3);
                    else
                        mma_commit(&sm.tfull[buf]);
                }
            }
            // Drain: all MMAs this thread issued complete before TMEM is freed.
            if constexpr (PAIR)
                mma_commit_pair(sm.drain, 0x1);
            else
                mma_commit(sm.drain);
            if (!mbar_wait(sm.drain, 0, nullptr)) record_status(p.status, kStatusTimeoutDrain, abort);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Four groups of four warps, two per TMEM accumulator: the groups of
        // buffer e take the tiles that land in it, each draining half of the
        // columns, so two tiles drain at once with twice the warps on each.  Per
        // 32 columns: tcgen05.ld -> scale, +bias, ReLU, BF16 -> swizzled smem
        // tile (one per warp) -> TMA store.
        const int quarter = warp & 3;             // TMEM lane quarter this warp may access
        const int egroup = (warp - 2) >> 2;       // 0..3
        const int group = egroup >> 1;            // = the accumulator buffer it drains
        const int chalf = egroup & 1;             // which half of the columns
        uint8_t* stg = sm.out + (warp - 2) * kOutTileBytes;
        int local = 0;
        for (int u = unit0; u < num_units; u += unit_step, ++local) {
            const int buf = local & 1;
            if (!ALLW && buf != group) continue;
            const uint32_t use = static_cast<uint32_t>(local >> 1) & 1u;
            // warp-uniform outcome, so the .sync.aligned TMEM loads below stay converged
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[buf], use, abort));
            if (!ready) {
                record_status(p.status, kStatusTimeoutEpilogue, abort);
                break;
            }
            tc_fence_after();
            const int mu = u / p.num_n_tiles;
            const int nt = u - mu * p.num_n_tiles;
            // DUAL: group half h drains tile h of the unit (all its columns)
            const int m = PAIR ? 2 * mu + static_cast<int>(rank) : (DUAL ? 2 * mu + chalf : mu);
            const PixTile t = pix_tile<PHASE, TWO>(p, m);
            if constexpr (SWAP) {
                // D holds output channels on TMEM lanes and the unit's 256 pixels on columns
                // (tile h: columns 128h ..): this warp drains channels 32*quarter .. of its tile,
                // 32 pixels per step; lane pairs swap halves so that each lane writes whole
                // 32-bit words (two channels of one pixel) into the pixel-major staging tile
                const int co = nt * p.n_tile + 32 * quarter;  // this warp's first output channel
                const float bl = p.bias ? __ldg(p.bias + co + lane) : 0.f;
                const float sl = p.scale ? __ldg(p.scale + co + lane) : 1.f;
                const uint32_t t_col = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(buf * 2 * p.n_tile + chalf * p.n_tile);
                const int odd = lane & 1;
                for (int cc = 0; cc < kTcBlockM / 32; ++cc) {
                    bool rows_exist;
                    int yc1, yc2, yc3;
                    if (PHASE) {
                        const int h = t.ho0 + cc * 32 / p.rect_w;
                        rows_exist = t.exists && h < p.hq && t.wo0 < p.wq;
                        yc1 = t.wo0;
                        yc2 = h;
                        yc3 = t.n;
                    } else if (p.mode == kTcModeRect || p.mode == kTcModeHalo) {
                        const int h = t.ho0 + cc * 32 / p.rect_w;
                        rows_exist = t.exists && h < p.g.H_out && t.wo0 < p.g.W_out;
                        yc1 = t.wo0;
                        yc2 = h;
                        yc3 = t.n;
                    } else {
                        const long long row0 = t.pix0 + cc * 32;
                        rows_exist = t.exists && row0 < p.g.pixels;
                        yc1 = static_cast<int>(row0);
                        yc2 = yc3 = 0;
                    }
                    uint32_t v[32];
                    __syncwarp();
                    tmem_ld32(t_col + static_cast<uint32_t>(cc * 32), v);
                    tmem_ld_wait(v);
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    float f[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        f[i] = p.scale ? fmaf(__uint_as_float(v[i]), sl, bl) : __uint_as_float(v[i]) + bl;
                    // even lane 2k writes pixels 0..15 of channels 2k, 2k+1; odd lane 2k+1 pixels 16..31
                    const int c2 = (lane & ~1) * 2;  // byte offset of the channel pair in a 64-byte row
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float mine = odd ? f[i + 16] : f[i];
                        const float send = odd ? f[i] : f[i + 16];
                        const float other = __shfl_xor_sync(0xffffffffu, send, 1);
                        const float lo = odd ? other : mine, hi = odd ? mine : other;
                        const uint32_t w = p.relu ? pack_bf16x2_relu(lo, hi) : pack_bf16x2(lo, hi);
                        const int r = i + 16 * odd;  // pixel row of the staging tile
                        const int byte = r * 64 + ((((c2 >> 4) ^ ((r >> 1) & 3)) << 4) | (c2 & 15));
                        *reinterpret_cast<uint32_t*>(stg + byte) = w;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && rows_exist) {
                        if (PHASE)
                            tma_store_5d(&y_map, stg, co, t.rw, yc1, t.rh, yc3 * p.hq + yc2);
                        else if (p.mode == kTcModeRect || p.mode == kTcModeHalo)
                            tma_store_4d(&y_map, stg, co, yc1, yc2, yc3);
                        else
                            tma_store_2d(&y_map, stg, co, yc1);
                        bulk_commit();
                    }
                }
            } else {
                // this warp's 32 pixels: rect mode = 32/TW rows of the rectangle, else 32 linear pixels
                bool rows_exist;
                int yc1, yc2, yc3;
                if (PHASE) {
                    const int h = t.ho0 + quarter * 32 / p.rect_w;  // phase-grid row
                    rows_exist = t.exists && h < p.hq && t.wo0 < p.wq;
                    yc1 = t.wo0;
                    yc2 = h;
                    yc3 = t.n;
                } else if (p.mode == kTcModeRect || p.mode == kTcModeHalo) {
                    const int h = t.ho0 + quarter * 32 / p.rect_w;
                    rows_exist = t.exists && h < p.g.H_out && t.wo0 < p.g.W_out;
                    yc1 = t.wo0;
                    yc2 = h;
                    yc3 = t.n;
                } else {
                    const long long row0 = t.pix0 + quarter * 32;
                    rows_exist = t.exists && row0 < p.g.pixels;
                    yc1 = static_cast<int>(row0);
                    yc2 = yc3 = 0;
                }
                const int co0 = nt * p.n_tile;
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(buf * (DUAL ? 2 : 1) * p.n_tile + (DUAL ? chalf * p.n_tile : 0));
                // this group's half of the columns, 32 per step, one staging tile per warp
                const int chunks = p.n_tile / 32;
                const int c_lo = ALLW ? 32 * ((chunks * egroup) / 4)
                                      : DUAL ? 0 : (chalf == 0 ? 0 : ((chunks + 1) / 2) * 32);
                const int c_hi = ALLW ? 32 * ((chunks * (egroup + 1)) / 4)
                                      : DUAL ? p.n_tile : (chalf == 0 ? ((chunks + 1) / 2) * 32 : p.n_tile);
                for (int c = c_lo; c < c_hi; c += 32) {
                    uint32_t v[32];
                    if constexpr (ALLW) {
                        __syncwarp();
                        tmem_ld32(t_row + static_cast<uint32_t>(c), v);
                        if (lane == 0) bulk_wait_read_all();
                        tmem_ld_wait(v);
                        __syncwarp();
                        stage_row32(v, p.bias ? p.bias + co0 + c : nullptr, p.relu, stg, lane,
                                    p.scale ? p.scale + co0 + c : nullptr);
                    } else {
                        // lane l loads the scale and shift of channel co0 + c + l before the TMEM
                        // load, and shuffles hand them round: no global load waits behind the
                        // accumulator (body with a folded batch norm 145.4 -> 136.8 us, body 136.3 ->
                        // 134.2, dilated 27.5 -> 26.7; the 1x1 kernel above measured slower this way)
                        const float sl = p.scale ? __ldg(p.scale + co0 + c + lane) : 1.f;
                        const float bl = p.bias ? __ldg(p.bias + co0 + c + lane) : 0.f;
                        __syncwarp();
                        tmem_ld32(t_row + static_cast<uint32_t>(c), v);
                        tmem_ld_wait(v);
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
                        if (p.scale) {
    #pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const float si = __shfl_sync(0xffffffffu, sl, i), bi = __shfl_sync(0xffffffffu, bl, i);
                                v[i] = __float_as_uint(fmaf(__uint_as_float(v[i]), si, bi));
                            }
                        } else if (p.bias) {
    #pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[i] = __float_as_uint(__uint_as_float(v[i]) + __shfl_sync(0xffffffffu, bl, i));
                        }
                        stage_row32(v, nullptr, p.relu, stg, lane, nullptr);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && rows_exist) {
                        if (PHASE)
                            tma_store_5d(&y_map, stg, co0 + c, t.rw, yc1, t.rh, yc3 * p.hq + yc2);
                        else if (p.mode == kTcModeRect || p.mode == kTcModeHalo)
                            tma_store_4d(&y_map, stg, co0 + c, yc1, yc2, yc3);
                        else
                            tma_store_2d(&y_map, stg, co0 + c, yc1);
                        bulk_commit();
                    }
                }
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_remote(mapa_shared(smem_addr(&sm.tempty[buf]), 0));
                else
                    mbar_arrive(&sm.tempty[buf]);
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, p.tmem_cols);
        else
            tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// per-device dynamic shared-memory limit already set on the pair kernel
static SmemLimitCache g_pair_smem_limits;

namespace {

// Launch one instantiation: clusters of two CTAs for SM pairs, else plain.
template <bool PAIR, bool PHASE, bool DUAL, bool HALO, bool RESB = false, bool SWAP = false>
cudaError_t launch_one(const CUtensorMap& a_map, const CUtensorMap& b_map, const CUtensorMap& y_map,
                       const TcGemmParams& p, int grid, cudaStream_t stream) {
    static SmemLimitCache limits;
    auto* fn = tc_conv_kernel<PAIR, PHASE, DUAL, HALO, RESB, SWAP>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(fn), p.smem_bytes, limits);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(tc_threads(HALO, DUAL), 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = PAIR ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, fn, a_map, b_map, y_map, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_gemm(const CUtensorMap& a_map, const CUtensorMap& b_map, const CUtensorMap& y_map,
                           const TcGemmParams& p, int grid, cudaStream_t stream) {
    if (p.halo) {
        if (p.bres) {
            if (p.dual) return launch_one<false, false, true, true, true>(a_map, b_map, y_map, p, grid, stream);
            return launch_one<false, false, false, true, true>(a_map, b_map, y_map, p, grid, stream);
        }
        if (p.pair) return launch_one<true, false, false, true>(a_map, b_map, y_map, p, grid, stream);
        if (p.dual) return launch_one<false, false, true, true>(a_map, b_map, y_map, p, grid, stream);
        return launch_one<false, false, false, true>(a_map, b_map, y_map, p, grid, stream);
    }
    if (p.bres) {
        if (p.pair) return launch_one<true, false, false, false, true>(a_map, b_map, y_map, p, grid, stream);
        return launch_one<false, false, false, false, true>(a_map, b_map, y_map, p, grid, stream);
    }
    if (p.pair) {
        static SmemLimitCache pair_phase_limits;
        cudaError_t e = p.mode == kTcModePhase
                            ? ensure_smem_limit(reinterpret_cast<const void*>(tc_conv_kernel<true, true, false>), p.smem_bytes,
                                                pair_phase_limits)
                            : ensure_smem_limit(reinterpret_cast<const void*>(tc_conv_kernel<true, false, false>),
                                                p.smem_bytes, g_pair_smem_limits);
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
        e = p.mode == kTcModePhase ? cudaLaunchKernelEx(&cfg, tc_conv_kernel<true, true, false>, a_map, b_map, y_map, p)
                                   : cudaLaunchKernelEx(&cfg, tc_conv_kernel<true, false, false>, a_map, b_map, y_map, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (p.dual && p.swap) {  // two pixel tiles per CTA, weights as the M operand
        if (p.mode == kTcModePhase) return launch_one<false, true, true, false, false, true>(a_map, b_map, y_map, p, grid, stream);
        return launch_one<false, false, true, false, false, true>(a_map, b_map, y_map, p, grid, stream);
    }
    if (p.dual) {  // two pixel tiles per CTA
        static SmemLimitCache dual_limits, dual_phase_limits;
        const bool ph = p.mode == kTcModePhase;
        const void* fn = ph ? reinterpret_cast<const void*>(tc_conv_kernel<false, true, true>)
                            : reinterpret_cast<const void*>(tc_conv_kernel<false, false, true>);
        cudaError_t e = ensure_smem_limit(fn, p.smem_bytes, ph ? dual_phase_limits : dual_limits);
        if (e != cudaSuccess) return e;
        if (ph)
            tc_conv_kernel<false, true, true><<<grid, tc_threads(false, true), p.smem_bytes, stream>>>(a_map, b_map, y_map, p);
        else
            tc_conv_kernel<false, false, true><<<grid, tc_threads(false, true), p.smem_bytes, stream>>>(a_map, b_map, y_map, p);
        return cudaGetLastError();
    }
    if (p.mode == kTcModePhase) {
        static SmemLimitCache phase_limits;
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(tc_conv_kernel<false, true, false>), p.smem_bytes,
                                          phase_limits);
        if (e != cudaSuccess) return e;
        tc_conv_kernel<false, true, false><<<grid, kTcThreads, p.smem_bytes, stream>>>(a_map, b_map, y_map, p);
        return cudaGetLastError();
    }
    static SmemLimitCache limits;
    cudaError_t e =
        ensure_smem_limit(reinterpret_cast<const void*>(tc_conv_kernel<false, false, false>), p.smem_bytes, limits);
    if (e != cudaSuccess) return e;
    tc_conv_kernel<false, false, false><<<grid, kTcThreads, p.smem_bytes, stream>>>(a_map, b_map, y_map, p);
    return cudaGetLastError();
}

int tc_gemm_pair_max_clusters(const TcGemmParams& p) {
    static SmemLimitCache halo_pair_limits;
    const void* fn = p.halo ? reinterpret_cast<const void*>(tc_conv_kernel<true, false, false, true>)
                            : reinterpret_cast<const void*>(tc_conv_kernel<true, false, false>);
    if (ensure_smem_limit(fn, p.smem_bytes, p.halo ? halo_pair_limits : g_pair_smem_limits) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(p.halo ? kTcHaloThreads : kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = p.halo ? cudaOccupancyMaxActiveClusters(&n, tc_conv_kernel<true, false, false, true>, &cfg)
                                 : cudaOccupancyMaxActiveClusters(&n, tc_conv_kernel<true, false, false>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace convgb
