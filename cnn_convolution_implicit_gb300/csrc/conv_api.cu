// conv_api.cu -- the C ABI (include/conv.h): plan creation, shape checks,
// kernel choice, TMA descriptor encoding and launch.
//
// Shape math: H_out = floor((H + 2P - D(Kh-1) - 1)/S) + 1 ("Convolution
// variants and their matrix operations", lpnh.cn/news/2674933, section 6.2;
// the printed formula is garbled, this is its reading), with the effective
// dilated kernel K + (K-1)(D-1) (same page, section 2.3).  GEMM extents
// M = C_out, N = N*H_out*W_out, K = (C_in/G)*Kh*Kw ("GPU lesson 9: how a GPU
// executes neural-network convolution", lincklin.cn, section 19).
//
// Kernel choice by shape (the channel-alignment concerns of lesson 9 sections
// 20 and 33 decide it):
//   FP32, G = C_in = C_out, C % 32 == 0   -> depthwise halo-tile kernel
//   BF16, 1x1, S=1, P=0, G=1, aligned      -> tcgen05 GEMM with tiled TMA
//   BF16, (C_in/G) % 64 == 0, aligned      -> tcgen05 implicit GEMM, TMA im2col
//   BF16, G=1, C_in*Kh*Kw <= 64            -> tcgen05 small-K kernel (stem)
//   BF16 transposed, aligned, S | H_out    -> tcgen05 implicit GEMM, phase mode
//   FP32 3x3 s1 d1 G=1 with WINOGRAD flag  -> Winograd F(2x2, 3x3) kernel
//   anything else                          -> direct CUDA-core kernel
#include <mutex>
#include <new>

#include <cudaTypedefs.h>

#include "../../include/conv.h"
#include "conv_internal.h"
#include "status_slots.h"

using namespace convgb;

// Device status word: bits latched by kernels whose bounded waits gave up.
__device__ unsigned int g_conv_status_word;

// Per-plan status words (status_slots.h): a fixed array per device, taken and given
// back on the host under a lock.
constexpr int kStatusSlots = 1024;
constexpr int kMaxStatusDevices = 64;
__device__ unsigned int g_conv_status_slots[kStatusSlots];

namespace convgb {
namespace {
std::mutex g_slot_mutex;
bool g_slot_used[kMaxStatusDevices][kStatusSlots];
}  // namespace

cudaError_t acquire_status_word(int device, unsigned** word, int* slot) {
    *slot = -1;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_conv_status_word);
    if (e != cudaSuccess || device < 0 || device >= kMaxStatusDevices) return e;
    int idx = -1;
    {
        std::lock_guard<std::mutex> lock(g_slot_mutex);
        for (int i = 0; i < kStatusSlots && idx < 0; ++i)
            if (!g_slot_used[device][i]) {
                g_slot_used[device][i] = true;
                idx = i;
            }
    }
    if (idx < 0) return cudaSuccess;  // every word is taken: share the library-wide one
    unsigned* base = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&base), g_conv_status_slots);
    if (e == cudaSuccess) e = cudaMemset(base + idx, 0, sizeof(unsigned));  // a previous owner's bits
    if (e != cudaSuccess) {
        release_status_word(device, idx);
        return e;
    }
    *word = base + idx;
    *slot = idx;
    return cudaSuccess;
}

void release_status_word(int device, int slot) {
    if (slot < 0 || device < 0 || device >= kMaxStatusDevices) return;
    std::lock_guard<std::mutex> lock(g_slot_mutex);
    g_slot_used[device][slot] = false;
}
}  // namespace convgb

struct conv_plan {
    ConvGeom g;
    conv_dtype dtype;
    unsigned flags;
    int path;
    int device;
    int num_sms;
    int smem_optin;
    int smem_per_sm;
    int pair_clusters;  // co-resident 2-CTA clusters of the pair kernel (0: unknown)
    unsigned* status;
    int status_slot;    // index of the plan's own status word, -1: the library-wide word
    // per-path configuration
    TcGemmParams tc;
    SmallKParams sk;
    DepthwiseParams dw;
    // descriptor cache, keyed by the pointers it was encoded for
    const void* cache_x;
    const void* cache_w;
    const void* cache_y;
    bool cache_valid;
    CUtensorMap map_a;  // the type carries its own 64-byte alignment
    CUtensorMap map_b;
    CUtensorMap map_y;
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
PFN_cuTensorMapEncodeIm2col_v12000 g_encode_im2col = nullptr;
std::once_flag g_entry_once;
bool g_entry_ok = false;

bool load_entry_points() {
    std::call_once(g_entry_once, [] {
        cudaDriverEntryPointQueryResult q1, q2;
        void* f1 = nullptr;
        void* f2 = nullptr;
        const cudaError_t e1 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000,
                                                                cudaEnableDefault, &q1);
        const cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f2, 12000,
                                                                cudaEnableDefault, &q2);
        if (e1 == cudaSuccess && e2 == cudaSuccess && q1 == cudaDriverEntryPointSuccess &&
            q2 == cudaDriverEntryPointSuccess && f1 && f2) {
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f1);
            g_encode_im2col = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(f2);
            g_entry_ok = true;
        }
    });
    return g_entry_ok;
}

int out_extent(int in, int k, int s, int p, int d) {
    const long long num = static_cast<long long>(in) + 2LL * p - static_cast<long long>(d) * (k - 1) - 1;
    if (num < 0) return 0;
    return static_cast<int>(num / s + 1);
}

// Transposed convolution: (in - 1)*s - 2p + d(k - 1) + 1, or 0 when not positive.
int out_extent_transposed(int in, int k, int s, int p, int d) {
    const long long v = static_cast<long long>(in - 1) * s - 2LL * p + static_cast<long long>(d) * (k - 1) + 1;
    return v > 0 && v <= 0x7fffffffLL ? static_cast<int>(v) : 0;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int pow2_at_least(int v) {
    int r = 32;
    while (r < v) r <<= 1;
    return r;
}

// Taps of one axis of a transposed convolution, per output phase residue r:
// kernel index k with (r + P - k*D) divisible by S, input offset (r + P - k*D)/S.
// False if a residue has no tap or an offset does not fit the table.
bool phase_axis(int K, int S, int P, int D, TcPhaseAxis& a) {
    for (int r = 0; r < S; ++r) {
        int n = 0;
        for (int k = 0; k < K; ++k) {
            const int num = r + P - k * D;
            if (((num % S) + S) % S != 0) continue;
            const int off = num / S;
            if (off < -128 || off > 127 || n >= kTcMaxPhaseTaps) return false;
            a.k[r][n] = static_cast<int8_t>(k);
            a.off[r][n] = static_cast<int8_t>(off);
            ++n;
        }
        if (n == 0) return false;
        a.cnt[r] = static_cast<int8_t>(n);
    }
    return true;
}

// tcgen05 GEMM configuration; false when the shape does not fit it.
// Narrowest per-tile N the plan runs on SM pairs by default.
constexpr int kPairMinN = 256;
// Widest per-tile N that runs two pixel tiles per CTA.
constexpr int kDualMaxN = 128;

bool configure_tc(conv_plan* pl, bool one_by_one, bool transposed = false) {
    const ConvGeom& g = pl->g;
    TcGemmParams& t = pl->tc;
    if (g.cin_g % kTcBlockK != 0) return false;
    if (g.cout_g % 16 != 0) return false;
    const long long ktot = static_cast<long long>(g.cin_g) * g.Kh * g.Kw;
    if ((ktot * 2) % 16 != 0) return false;
    int n_tile, mma_n, gpc;
    if (g.cout_g >= 256) {
        if (g.cout_g % 256 != 0) return false;
        n_tile = mma_n = 256;
        gpc = 1;
    } else {
        // groups packed per tile: the MMA issuer holds one ring stage per group at
        // once, so gpc is also bounded by the stages that fit
        mma_n = g.cout_g;
        const int stage_bytes = kTcBlockM * kTcBlockK * 2 + mma_n * 128;
        const int max_gpc_stages = (pl->smem_optin - (1024 + 256 + 8 * 2 * 32 * 64)) / stage_bytes;
        gpc = 0;
        for (int c = g.G; c >= 1; --c)
            if (g.G % c == 0 && c * g.cout_g <= 256 && (c * g.cout_g) % 32 == 0 && c <= kTcMaxGroupsPerTile &&
                c <= max_gpc_stages) {
                gpc = c;
                break;
            }
        if (gpc == 0) return false;
        n_tile = gpc * g.cout_g;
    }
    if (transposed) {
        // phase mode: S x S output phases, each a stride-1 gather over the input
        if (g.S > kTcMaxPhaseStride || g.Kh > kTcMaxPhaseTaps || g.Kw > kTcMaxPhaseTaps) return false;
        if (g.H_out % g.S != 0 || g.W_out % g.S != 0) return false;
        if (!phase_axis(g.Kh, g.S, g.P, g.D, t.ph) || !phase_axis(g.Kw, g.S, g.P, g.D, t.pw)) return false;
        t.ps = g.S;
        t.hq = g.H_out / g.S;
        t.wq = g.W_out / g.S;
    } else if (!one_by_one) {
        // im2col bounding box corners must fit the 4-D map's signed 8-bit range
        const int lo = -g.P;
        const int up_w = g.P - (g.Kw - 1) * g.D, up_h = g.P - (g.Kh - 1) * g.D;
        if (lo < -128 || up_w < -128 || up_h < -128 || g.P > 127) return false;
        if (g.S > 8) return false;
        if ((g.Kw - 1) * g.D > 65535 || (g.Kh - 1) * g.D > 65535) return false;
    }
    if (g.pixels > 0x7fffffffLL) return false;
    t.g = g;
    t.mode = transposed ? kTcModePhase : one_by_one ? kTcMode1x1 : (g.S == 1 ? kTcModeRect : kTcModeIm2col);
    t.n_tile = n_tile;
    t.mma_n = mma_n;
    t.gpc = gpc;
    t.kblk = g.cin_g / kTcBlockK;
    t.ksteps = g.Kh * g.Kw * t.kblk;
    if (t.mode == kTcModeRect || t.mode == kTcModePhase) {
        // 128-pixel rectangle (of the output, or of one phase's output grid), 8 /
        // 16 / 32 wide: the one that pads least (ties go to 16 x 8).  A warp's 32
        // TMEM lanes are 32/TW whole rows of it; in phase mode a warp's rows must
        // not cross the end of the phase grid (its store view runs on into the
        // next image), so the grid height must be a multiple of 32/TW.
        const bool phase = t.mode == kTcModePhase;
        const int eh = phase ? t.hq : g.H_out, ew = phase ? t.wq : g.W_out;
        auto padded = [](int extent, int t) { return static_cast<long long>((extent + t - 1) / t) * t; };
        int best = 0;
        long long best_area = 0;
        for (int tw : {16, 8, 32}) {
            if (phase && eh % (32 / tw) != 0) continue;
            const long long area = padded(ew, tw) * padded(eh, kTcBlockM / tw);
            if (best == 0 || area < best_area) {
                best = tw;
                best_area = area;
            }
        }
        // halo mode (stride 1, not forced per tap): 8 x 16 tiles, one halo per channel block
        if (t.mode == kTcModeRect && !(pl->flags & CONV_FLAG_PER_TAP)) {
            t.mode = kTcModeHalo;
            best = kTcHaloTileW;
        }
        t.rect_w = best;
        t.rect_h = kTcBlockM / best;
        t.rect_tiles_w = (ew + t.rect_w - 1) / t.rect_w;
        t.rect_tiles_h = (eh + t.rect_h - 1) / t.rect_h;
        const long long m_tiles =
            static_cast<long long>(g.N) * t.rect_tiles_w * t.rect_tiles_h * (phase ? t.ps * t.ps : 1);
        if (m_tiles > 0x3fffffffLL) return false;
        t.num_m_tiles = static_cast<int>(m_tiles);
    } else {
        t.rect_w = t.rect_h = t.rect_tiles_w = t.rect_tiles_h = 0;
        t.num_m_tiles = static_cast<int>((g.pixels + kTcBlockM - 1) / kTcBlockM);
    }
    t.num_n_tiles = g.C_out / n_tile;
    t.num_tiles = t.num_m_tiles * t.num_n_tiles;
    t.ychunk = 32;
    // SM pairs (one MMA over 2 x 128 pixels, weight rows split between the two
    // CTAs) on request, when there are at least two pixel tiles to pair up.
    // SM pairs (one MMA over 2 x 128 pixels, weight rows split between the two CTAs):
    // on request, else by default where each tile is a long reduction over a wide tile
    // (a pair doubles the MMA work per K-step its producers issue, which pays when
    // the MMAs dominate; for short reductions and narrow groups it measured slower)
    int min_ksteps = t.ksteps;
    if (transposed) {  // the shortest phase's reduction
        int ch = 64, cw = 64;
        for (int r = 0; r < t.ps; ++r) {
            ch = t.ph.cnt[r] < ch ? t.ph.cnt[r] : ch;
            cw = t.pw.cnt[r] < cw ? t.pw.cnt[r] : cw;
        }
        min_ksteps = ch * cw * t.kblk;
    }
    // One group per tile where two pixel tiles per CTA can pair up instead: packing
    // groups side by side adds no operand reuse (each group reads its own channels
    // and weights), but it makes units coarse (36 K-steps for four packed 3x3
    // groups, 3.4 units per SM on the dilated layer) and rules out the two-tile mode
    // (dilated grouped layer 56.0 -> 41.6 us).
    if (gpc > 1 && !(pl->flags & CONV_FLAG_SM_PAIRS) && g.cout_g <= kDualMaxN && g.cout_g % 32 == 0 &&
        t.num_m_tiles >= 2 && min_ksteps >= 4) {  // (the epilogue drains 32-column chunks)
        gpc = 1;
        n_tile = g.cout_g;
        t.gpc = 1;
        t.n_tile = n_tile;
        t.num_n_tiles = g.C_out / n_tile;
        t.num_tiles = t.num_m_tiles * t.num_n_tiles;
    }
    const bool auto_pairs = !one_by_one && gpc == 1 && mma_n >= kPairMinN && min_ksteps >= 9;
    const bool want_pairs = (pl->flags & CONV_FLAG_SM_PAIRS) || (auto_pairs && !(pl->flags & CONV_FLAG_ONE_SM));
    t.pair = (t.num_m_tiles >= 2 && want_pairs) ? 1 : 0;
    // Two pixel tiles per CTA (M = 256 on one SM) for narrow tiles with a real
    // reduction: each K-step then feeds twice the tensor work for one weight block and
    // one more A copy (a 2-K-step 1x1 layer measured slower: its epilogue dominates).
    t.dual = (!t.pair && gpc == 1 && n_tile <= kDualMaxN && t.num_m_tiles >= 2 && min_ksteps >= 4) ? 1 : 0;
    // Two tiles of 128 channels: one M128 N256 MMA (weights x both tiles' pixels) per K = 16 reads
    // 12 KB of shared-memory operands instead of two M128 N128 MMAs' 16 KB (the per-tap modes;
    // the halo mode's operands are the shifted halo windows).
    t.swap = (t.dual && n_tile == kDualMaxN && mma_n == kDualMaxN) ? 1 : 0;
    if ((t.pair || t.dual) && transposed) {  // both tiles of a unit in one phase: round each phase's count up
        const long long spatial = static_cast<long long>(g.N) * t.rect_tiles_w * t.rect_tiles_h;
        t.num_m_tiles = static_cast<int>(((spatial + 1) / 2) * 2 * t.ps * t.ps);
        t.num_tiles = t.num_m_tiles * t.num_n_tiles;
    }
    const int b_rows = t.pair ? mma_n / 2 : mma_n;
    const int fixed = 1024 + 256 + 8 * 2 * 32 * 64;  // alignment, barriers, epilogue store tiles
    t.halo = 0;
    t.halo_w = t.halo_h = t.halo_bytes = t.halo_stages = 0;
    t.btaps = 1;
    t.bres = 0;
    if (t.mode == kTcModeHalo) {
        // one box {64 ch, halo_w, halo_h} per 64-channel block: the tile (two side by side
        // for two tiles per CTA) plus the (K-1)*D border its taps reach
        long long hw = (t.dual ? 2 : 1) * kTcHaloTileW + static_cast<long long>(g.Kw - 1) * g.D;
        const long long hh = kTcHaloTileH + static_cast<long long>(g.Kh - 1) * g.D;
        const int taps = g.Kh * g.Kw;
        // Taps per weight stage: each barrier wait of the MMA issuer costs a few hundred
        // clocks under load, so a stage should carry >= 1,536 clocks of tensor work (a
        // K = 16 MMA of M = 128 rows and N columns takes N/2 clocks per SM at the full
        // rate; measured on the body layer: 1, 2, 3 taps per stage took 191, 154, 136 us).
        // The largest such count that still leaves two halos and two weight stages in
        // shared memory, with three halos when that keeps as many weight stages.
        const int tap_clk = (t.dual ? 2 : 1) * (kTcBlockK / 16) * (mma_n / 2);
        int bt_max = (1536 + tap_clk - 1) / tap_clk;
        if (bt_max > taps) bt_max = taps;
        int hs = 0, bs = 0, hbytes = 0, bt = 0;
        long long wbytes = 0;
        if (hw <= 256 && hh <= 256) {
            hbytes = static_cast<int>((hw * hh * 128 + 1023) / 1024 * 1024);
            // Resident weights (one SM per unit): where every CTA keeps one n-tile and its
            // rows for all taps and channel blocks fit beside two halos, they load once and
            // the MMA issuer waits only for halos.
            wbytes = static_cast<long long>(t.ksteps) * mma_n * 128;
            if (!t.pair && gpc == 1 && t.num_n_tiles <= 8 &&
                fixed + 2LL * hbytes + wbytes <= static_cast<long long>(pl->smem_optin)) {
                t.bres = 1;
                hs = fixed + 3LL * hbytes + wbytes <= static_cast<long long>(pl->smem_optin) ? 3 : 2;
                bt = taps;
                bs = 1;
            }
        }
        if (hbytes > 0 && !t.bres) {
            for (int cbt = bt_max; cbt >= 1 && hs == 0; --cbt) {
                const long long stage = static_cast<long long>(cbt) * b_rows * 128;
                auto fit = [&](int h) {
                    const long long left = static_cast<long long>(pl->smem_optin) - fixed - static_cast<long long>(h) * hbytes;
                    return left > 0 ? left / stage : 0;
                };
                const long long n2 = fit(2), n3 = fit(3);
                if (n2 < 2) continue;
                bt = cbt;
                hs = (n3 >= 2 && n3 >= (n2 < 8 ? n2 : 8)) ? 3 : 2;
                const long long nb = hs == 3 ? n3 : n2;
                bs = static_cast<int>(nb > 8 ? 8 : nb);
            }
        }
        if (hs > 0) {
            t.halo = 1;
            t.swap = 0;  // the halo mode's A operands are shifted halo windows
            t.halo_w = static_cast<int>(hw);
            t.halo_h = static_cast<int>(hh);
            t.halo_bytes = hbytes;
            t.halo_stages = hs;
            if (t.dual) {  // a unit is a 16 x 16 region: both of its 8 x 16 tiles sit in one tile row
                t.rect_tiles_w = 2 * ((g.W_out + 2 * kTcHaloTileW - 1) / (2 * kTcHaloTileW));
                t.num_m_tiles = g.N * t.rect_tiles_w * t.rect_tiles_h;
                t.num_tiles = t.num_m_tiles * t.num_n_tiles;
            }
            t.btaps = bt;
            t.stages = bs;
            t.smem_bytes = fixed + hs * hbytes + (t.bres ? static_cast<int>(wbytes) : bs * bt * b_rows * 128);
        } else {  // the halo does not fit: per-tap rectangle tiles
            t.mode = kTcModeRect;
            int best = 0;
            long long best_area = 0;
            auto padded = [](int extent, int tl) { return static_cast<long long>((extent + tl - 1) / tl) * tl; };
            for (int tw : {16, 8, 32}) {
                const long long area = padded(g.W_out, tw) * padded(g.H_out, kTcBlockM / tw);
                if (best == 0 || area < best_area) {
                    best = tw;
                    best_area = area;
                }
            }
            t.rect_w = best;
            t.rect_h = kTcBlockM / best;
            t.rect_tiles_w = (g.W_out + t.rect_w - 1) / t.rect_w;
            t.rect_tiles_h = (g.H_out + t.rect_h - 1) / t.rect_h;
            t.num_m_tiles = g.N * t.rect_tiles_w * t.rect_tiles_h;
            t.num_tiles = t.num_m_tiles * t.num_n_tiles;
        }
    }
    if (!t.halo) {
        const int stage_bytes = (t.dual ? 2 : 1) * kTcBlockM * kTcBlockK * 2 + b_rows * 128;
        int stages = (pl->smem_optin - fixed) / stage_bytes;
        if (stages > 8) stages = 8;
        if (stages < 2 || stages < gpc) return false;
        t.stages = stages;
        t.smem_bytes = fixed + stages * stage_bytes;
    }
    // 1x1 layers: where one n-tile's weight rows for the whole reduction fit beside an A
    // ring of at least four stages, they stay in shared memory (loaded once per CTA) and
    // the ring carries the pixels only.  The weights were the larger part of each stage
    // (a 256-row block against 128 pixel rows) and came from L2 again for every tile.
    // Every CTA's units share one n-tile (the grid is a multiple of the n-tile count).
    if (t.mode == kTcMode1x1 && gpc == 1 && !t.dual && t.num_n_tiles <= 8) {
        const bool pairs = t.pair != 0;
        const long long wbytes = static_cast<long long>(t.ksteps) * (pairs ? mma_n / 2 : mma_n) * 128;
        const long long left = static_cast<long long>(pl->smem_optin) - fixed - wbytes;
        long long st = left > 0 ? left / (kTcBlockM * kTcBlockK * 2) : 0;
        if (st > 8) st = 8;
        if (st >= 4) {
            t.bres = 1;
            t.pair = pairs ? 1 : 0;
            t.stages = static_cast<int>(st);
            t.smem_bytes = fixed + static_cast<int>(wbytes) + t.stages * kTcBlockM * kTcBlockK * 2;
        }
    }
    t.tmem_cols = pow2_at_least((t.dual ? 4 : 2) * n_tile);
    t.relu = (pl->flags & CONV_FLAG_RELU) ? 1 : 0;
    t.status = pl->status;
    return true;
}

// The Winograd launch grid (spatial blocks x 32-channel blocks) within CUDA's limits.
bool winograd_grid_fits(const ConvGeom& g) {
    const long long tiles_w = (g.W_out + 1) / 2, tiles_h = (g.H_out + 1) / 2;
    const long long blocks = static_cast<long long>(g.N) * ((tiles_h + 3) / 4) * ((tiles_w + 7) / 8);
    return blocks <= 0x7fffffffLL && (g.C_out + 31) / 32 <= 65535;
}

bool configure_smallk(conv_plan* pl) {
    const ConvGeom& g = pl->g;
    SmallKParams& s = pl->sk;
    if (g.G != 1) return false;
    const int ktot = g.C_in * g.Kh * g.Kw;
    if (ktot > 64) return false;
    if (g.C_out % 32 != 0 || g.C_out > 256) return false;
    const long long row_bytes = static_cast<long long>(g.W) * g.C_in * 2;
    if (row_bytes % 16 != 0) return false;
    const long long segs = (g.W_out + 127) / 128;
    const long long segments = static_cast<long long>(g.N) * g.H_out * segs;
    if (segments > 0x7fffffffLL) return false;
    s.g = g;
    s.ktot = ktot;
    s.kmma = (ktot + 15) / 16;
    s.a_row_bytes = s.kmma * 16 <= 32 ? 64 : 128;
    s.segs = static_cast<int>(segs);
    s.num_segments = static_cast<int>(segments);
    s.row_bytes = static_cast<int>(row_bytes);
    const int b_bytes = (g.C_out * s.a_row_bytes + 1023) / 1024 * 1024;
    const int fixed = 1024 + b_bytes + 1024 + 3 * 64 * 4 + 16 + kSkMaxStages * kSkMaxRows * 16 +
                      2 * (g.C_out + 4) * 4;
    // row segments per stage (2 * rows * C_out TMEM columns): as many as allow a two-stage ring
    int rows = 256 / g.C_out < 4 ? 256 / g.C_out : 4;
    int stages = 0;
    for (; rows >= 1; --rows) {
        const long long raw = (static_cast<long long>(rows) * g.Kh * row_bytes + 1023) / 1024 * 1024;
        if (raw > 48 * 1024) continue;
        const long long stage_bytes = static_cast<long long>(rows) * 128 * s.a_row_bytes + raw;
        stages = static_cast<int>((pl->smem_optin - fixed) / stage_bytes);
        if (stages >= 2) {
            s.raw_bytes = static_cast<int>(raw);
            break;
        }
    }
    if (rows < 1 || stages < 2) return false;
    if (stages > kSkMaxStages) stages = kSkMaxStages;
    s.rows_per_tile = rows;
    // consecutive output rows of one image read overlapping, contiguous input rows
    // when the kernel rows are adjacent and the stride skips none of them: one copy
    // of their union fits in the stage's Kh rows per segment
    s.row_runs = (g.D == 1 && g.S <= g.Kh) ? 1 : 0;
    s.num_tiles = static_cast<int>((segments + rows - 1) / rows);
    s.stages = stages;
    s.smem_bytes = fixed + stages * (rows * 128 * s.a_row_bytes + s.raw_bytes);
    s.tmem_cols = pow2_at_least(2 * rows * g.C_out);
    s.relu = (pl->flags & CONV_FLAG_RELU) ? 1 : 0;
    s.status = pl->status;
    return true;
}

bool configure_depthwise(conv_plan* pl) {
    const ConvGeom& g = pl->g;
    DepthwiseParams& d = pl->dw;
    if (!(g.G == g.C_in && g.C_out == g.C_in)) return false;
    if (g.C_in % 32 != 0) return false;
    if (!depthwise_config(g, pl->smem_per_sm, pl->num_sms, d)) return false;
    d.g = g;
    d.relu = (pl->flags & CONV_FLAG_RELU) ? 1 : 0;
    d.out_bf16 = (pl->flags & CONV_FLAG_OUT_BF16) ? 1 : 0;
    d.status = pl->status;
    return true;
}

// Y store map of the tcgen05 paths: BF16, boxes of `ychunk` channels x 32
// pixels, 128-byte swizzle (64 channels) or 64-byte swizzle (32 channels).
CUresult encode_y_map(conv_plan* pl, void* y) {
    const ConvGeom& g = pl->g;
    const TcGemmParams& t = pl->tc;
    const CUtensorMapSwizzle sw = t.ychunk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (t.mode == kTcModePhase) {
        // y viewed as {C_out, S (column phase), W_out/S, S (row phase), N*H_out/S}: one
        // box is 32 channels x TW pixels of one phase x 32/TW phase rows
        const cuuint64_t S = static_cast<cuuint64_t>(t.ps), Co = static_cast<cuuint64_t>(g.C_out);
        const cuuint32_t box[5] = {static_cast<cuuint32_t>(t.ychunk), 1, static_cast<cuuint32_t>(t.rect_w), 1,
                                   static_cast<cuuint32_t>(32 / t.rect_w)};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        const cuuint64_t dims[5] = {Co, S, static_cast<cuuint64_t>(t.wq), S,
                                    static_cast<cuuint64_t>(g.N) * static_cast<cuuint64_t>(t.hq)};
        const cuuint64_t strides[4] = {Co * 2, S * Co * 2, static_cast<cuuint64_t>(g.W_out) * Co * 2,
                                       S * static_cast<cuuint64_t>(g.W_out) * Co * 2};
        return g_encode_tiled(&pl->map_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, y, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (t.mode == kTcModeRect || t.mode == kTcModeHalo) {  // {C_out, W_out, H_out, N}: 32/TW rows of TW pixels per store
        const cuuint32_t box[4] = {static_cast<cuuint32_t>(t.ychunk), static_cast<cuuint32_t>(t.rect_w),
                                   static_cast<cuuint32_t>(32 / t.rect_w), 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.C_out), static_cast<cuuint64_t>(g.W_out),
                                    static_cast<cuuint64_t>(g.H_out), static_cast<cuuint64_t>(g.N)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.C_out) * 2,
                                       static_cast<cuuint64_t>(g.W_out) * g.C_out * 2,
                                       static_cast<cuuint64_t>(g.H_out) * g.W_out * g.C_out * 2};
        return g_encode_tiled(&pl->map_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, y, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(t.ychunk), 32};
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(g.C_out), static_cast<cuuint64_t>(g.pixels)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(g.C_out) * 2};
    return g_encode_tiled(&pl->map_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

conv_status encode_maps(conv_plan* pl, const void* x, const void* w, void* y) {
    if (pl->cache_valid && pl->cache_x == x && pl->cache_w == w && pl->cache_y == y) return CONV_OK;
    pl->cache_valid = false;
    if (!load_entry_points()) return CONV_ERR_CUDA;
    const ConvGeom& g = pl->g;
    CUresult r = CUDA_SUCCESS;
    if (pl->path == CONV_PATH_GEMM_1X1 || pl->path == CONV_PATH_IMPLICIT_GEMM) {
        if (pl->path == CONV_PATH_GEMM_1X1) {
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(g.C_in), static_cast<cuuint64_t>(g.pixels)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(g.C_in) * 2};
            const cuuint32_t box[2] = {kTcBlockK, kTcBlockM};
            const cuuint32_t estr[2] = {1, 1};
            r = g_encode_tiled(&pl->map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides,
                               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else if (pl->tc.mode == kTcModeHalo) {  // one box per 64-channel block: the tile's halo
            const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.C_in), static_cast<cuuint64_t>(g.W),
                                        static_cast<cuuint64_t>(g.H), static_cast<cuuint64_t>(g.N)};
            const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.C_in) * 2,
                                           static_cast<cuuint64_t>(g.W) * g.C_in * 2,
                                           static_cast<cuuint64_t>(g.H) * g.W * g.C_in * 2};
            const cuuint32_t box[4] = {kTcBlockK, static_cast<cuuint32_t>(pl->tc.halo_w),
                                       static_cast<cuuint32_t>(pl->tc.halo_h), 1};
            const cuuint32_t estr[4] = {1, 1, 1, 1};
            r = g_encode_tiled(&pl->map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else if (pl->tc.mode == kTcModeRect || pl->tc.mode == kTcModePhase) {
            const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.C_in), static_cast<cuuint64_t>(g.W),
                                        static_cast<cuuint64_t>(g.H), static_cast<cuuint64_t>(g.N)};
            const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.C_in) * 2,
                                           static_cast<cuuint64_t>(g.W) * g.C_in * 2,
                                           static_cast<cuuint64_t>(g.H) * g.W * g.C_in * 2};
            const cuuint32_t box[4] = {kTcBlockK, static_cast<cuuint32_t>(pl->tc.rect_w),
                                       static_cast<cuuint32_t>(pl->tc.rect_h), 1};
            const cuuint32_t estr[4] = {1, 1, 1, 1};
            r = g_encode_tiled(&pl->map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.C_in), static_cast<cuuint64_t>(g.W),
                                        static_cast<cuuint64_t>(g.H), static_cast<cuuint64_t>(g.N)};
            const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.C_in) * 2,
                                           static_cast<cuuint64_t>(g.W) * g.C_in * 2,
                                           static_cast<cuuint64_t>(g.H) * g.W * g.C_in * 2};
            const int lower[2] = {-g.P, -g.P};
            const int upper[2] = {g.P - (g.Kw - 1) * g.D, g.P - (g.Kh - 1) * g.D};
            const cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(g.S), static_cast<cuuint32_t>(g.S), 1};
            r = g_encode_im2col(&pl->map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                                lower, upper, kTcBlockK, kTcBlockM, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) return CONV_ERR_CUDA;
        const long long ktot = static_cast<long long>(g.cin_g) * g.Kh * g.Kw;
        const cuuint64_t bdims[2] = {static_cast<cuuint64_t>(ktot), static_cast<cuuint64_t>(g.C_out)};
        const cuuint64_t bstrides[1] = {static_cast<cuuint64_t>(ktot) * 2};
        const cuuint32_t bbox[2] = {kTcBlockK,
                                    static_cast<cuuint32_t>(pl->tc.pair ? pl->tc.mma_n / 2 : pl->tc.mma_n)};
        const cuuint32_t bestr[2] = {1, 1};
        r = g_encode_tiled(&pl->map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), bdims, bstrides,
                           bbox, bestr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return CONV_ERR_CUDA;
        if (encode_y_map(pl, y) != CUDA_SUCCESS) return CONV_ERR_CUDA;
    } else if (pl->path == CONV_PATH_DEPTHWISE) {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.C_in), static_cast<cuuint64_t>(g.W),
                                    static_cast<cuuint64_t>(g.H), static_cast<cuuint64_t>(g.N)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.C_in) * 4, static_cast<cuuint64_t>(g.W) * g.C_in * 4,
                                       static_cast<cuuint64_t>(g.H) * g.W * g.C_in * 4};
        const cuuint32_t box[4] = {32, static_cast<cuuint32_t>(pl->dw.in_w), static_cast<cuuint32_t>(pl->dw.in_h), 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        r = g_encode_tiled(&pl->map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(x), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return CONV_ERR_CUDA;
    }
    pl->cache_x = x;
    pl->cache_w = w;
    pl->cache_y = y;
    pl->cache_valid = true;
    return CONV_OK;
}

}  // namespace

namespace convgb {

bool tensor_map_encoder_ready() { return load_entry_points(); }

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* base, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
    if (!load_entry_points()) return CUDA_ERROR_NOT_INITIALIZED;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return g_encode_tiled(map, type, rank, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

cudaError_t device_status_word(unsigned** word) {
    return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_conv_status_word);
}

conv_status read_status_word(int device, unsigned* word, void* stream, int* code) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    if (cur != device) return CONV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned v = 0;
    // after everything queued on the stream before this call
    if (cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    if (v != 0 && (cudaMemsetAsync(word, 0, sizeof(unsigned), st) != cudaSuccess ||
                   cudaStreamSynchronize(st) != cudaSuccess)) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    *code = static_cast<int>(v);
    return v ? CONV_ERR_TIMEOUT : CONV_OK;
}

}  // namespace convgb

extern "C" {

conv_status conv_plan_create(conv_plan** out, int N, int C_in, int H, int W, int C_out, int Kh, int Kw, int S,
                             int P, int D, int G, conv_dtype dtype, unsigned flags) {
    if (out == nullptr) return CONV_ERR_INVALID_ARG;
    *out = nullptr;
    if (N <= 0 || C_in <= 0 || H <= 0 || W <= 0 || C_out <= 0 || Kh <= 0 || Kw <= 0 || S <= 0 || P < 0 || D <= 0 ||
        G <= 0)
        return CONV_ERR_INVALID_ARG;
    if (C_in % G != 0 || C_out % G != 0) return CONV_ERR_INVALID_ARG;
    if (dtype != CONV_F32 && dtype != CONV_BF16) return CONV_ERR_INVALID_ARG;
    if (flags & ~(CONV_FLAG_BIAS | CONV_FLAG_RELU | CONV_FLAG_OUT_BF16 | CONV_FLAG_SM_PAIRS | CONV_FLAG_TRANSPOSED |
                  CONV_FLAG_WINOGRAD | CONV_FLAG_ONE_SM | CONV_FLAG_PER_TAP))
        return CONV_ERR_INVALID_ARG;
    if ((flags & CONV_FLAG_SM_PAIRS) && (flags & CONV_FLAG_ONE_SM)) return CONV_ERR_INVALID_ARG;
    if ((flags & CONV_FLAG_OUT_BF16) && dtype != CONV_F32) return CONV_ERR_INVALID_ARG;
    const bool transposed = (flags & CONV_FLAG_TRANSPOSED) != 0;
    const int Ho = transposed ? out_extent_transposed(H, Kh, S, P, D) : out_extent(H, Kh, S, P, D);
    const int Wo = transposed ? out_extent_transposed(W, Kw, S, P, D) : out_extent(W, Kw, S, P, D);
    if (Ho < 1 || Wo < 1) return CONV_ERR_INVALID_ARG;

    conv_plan* pl = new (std::nothrow) conv_plan();
    if (pl == nullptr) return CONV_ERR_NO_MEMORY;
    ConvGeom& g = pl->g;
    g.N = N; g.C_in = C_in; g.H = H; g.W = W; g.C_out = C_out;
    g.Kh = Kh; g.Kw = Kw; g.S = S; g.P = P; g.D = D; g.G = G;
    g.H_out = Ho; g.W_out = Wo;
    g.cin_g = C_in / G; g.cout_g = C_out / G;
    g.pixels = static_cast<long long>(N) * Ho * Wo;
    pl->dtype = dtype;
    pl->flags = flags;
    pl->cache_valid = false;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        // No device: a host-only plan (shape checks and kernel choice against
        // a 152-SM, 227 KB-per-block part).  conv_forward on it fails with
        // CONV_ERR_CUDA; nothing falls back to the host.
        cudaGetLastError();
        pl->device = -1;
        pl->num_sms = 152;
        pl->smem_optin = 232448;
        pl->smem_per_sm = 233472;
        pl->status = nullptr;
        pl->status_slot = -1;
    } else if ((pl->status_slot = -1, cudaGetDevice(&pl->device)) != cudaSuccess ||
               cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->device) != cudaSuccess ||
               cudaDeviceGetAttribute(&pl->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, pl->device) !=
                   cudaSuccess ||
               cudaDeviceGetAttribute(&pl->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, pl->device) !=
                   cudaSuccess ||
               acquire_status_word(pl->device, &pl->status, &pl->status_slot) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return CONV_ERR_CUDA;
    }

    pl->path = CONV_PATH_DIRECT;
    pl->pair_clusters = 0;
    if (transposed) {
        if (dtype == CONV_BF16 && configure_tc(pl, false, true)) pl->path = CONV_PATH_IMPLICIT_GEMM;
    } else if (dtype == CONV_F32) {
        if ((flags & CONV_FLAG_WINOGRAD) && winograd_supported(g) && winograd_grid_fits(g))
            pl->path = CONV_PATH_WINOGRAD;
        else if (configure_depthwise(pl))
            pl->path = CONV_PATH_DEPTHWISE;
    } else {
        const bool pointwise = Kh == 1 && Kw == 1 && S == 1 && P == 0 && G == 1;
        if (pointwise && configure_tc(pl, true))
            pl->path = CONV_PATH_GEMM_1X1;
        else if (configure_tc(pl, false))
            pl->path = CONV_PATH_IMPLICIT_GEMM;
        else if (configure_smallk(pl))
            pl->path = CONV_PATH_SMALL_K_GEMM;
        if ((pl->path == CONV_PATH_GEMM_1X1 || pl->path == CONV_PATH_IMPLICIT_GEMM) && pl->tc.pair &&
            pl->device >= 0)
            pl->pair_clusters = tc_gemm_pair_max_clusters(pl->tc);
    }
    *out = pl;
    return CONV_OK;
}

conv_status conv_plan_output_shape(const conv_plan* p, int* H_out, int* W_out) {
    if (p == nullptr || H_out == nullptr || W_out == nullptr) return CONV_ERR_INVALID_ARG;
    *H_out = p->g.H_out;
    *W_out = p->g.W_out;
    return CONV_OK;
}

conv_status conv_plan_info(const conv_plan* p, int* path, long long* gemm_m, long long* gemm_n, long long* gemm_k) {
    if (p == nullptr) return CONV_ERR_INVALID_ARG;
    if (path) *path = p->path;
    if (p->flags & CONV_FLAG_TRANSPOSED) {  // Y_col = W^T X
        if (gemm_m) *gemm_m = static_cast<long long>(p->g.C_out) * p->g.Kh * p->g.Kw;
        if (gemm_n) *gemm_n = static_cast<long long>(p->g.N) * p->g.H * p->g.W;
        if (gemm_k) *gemm_k = p->g.cin_g;
        return CONV_OK;
    }
    if (gemm_m) *gemm_m = p->g.C_out;
    if (gemm_n) *gemm_n = p->g.pixels;
    if (gemm_k) *gemm_k = static_cast<long long>(p->g.cin_g) * p->g.Kh * p->g.Kw;
    return CONV_OK;
}

int conv_plan_num_sms(const conv_plan* p) { return p ? p->num_sms : 0; }

conv_status conv_plan_gemm_config(const conv_plan* p, int* mode, int* n_tile, int* pair, int* dual,
                                  int* resident_weights, int* swapped) {
    if (p == nullptr || (p->path != CONV_PATH_GEMM_1X1 && p->path != CONV_PATH_IMPLICIT_GEMM))
        return CONV_ERR_INVALID_ARG;
    const TcGemmParams& t = p->tc;
    if (mode) *mode = t.mode;
    if (n_tile) *n_tile = t.n_tile;
    if (pair) *pair = t.pair;
    if (dual) *dual = t.dual;
    if (resident_weights) *resident_weights = t.bres;
    if (swapped) *swapped = t.swap;
    return CONV_OK;
}

conv_status conv_plan_launch_info(const conv_plan* p, int* grid, int* block, int* smem_bytes, int* stages,
                                  int* cluster) {
    if (p == nullptr) return CONV_ERR_INVALID_ARG;
    int gr = 0, bl = 0, sm = 0, st = 0, cl = 1;
    switch (p->path) {
        case CONV_PATH_GEMM_1X1:
        case CONV_PATH_IMPLICIT_GEMM: {
            const TcGemmParams& t = p->tc;
            bl = tc_threads(t.halo != 0, t.dual != 0);
            sm = t.smem_bytes;
            st = t.stages;
            if (t.pair) {
                const int pair_tiles = ((t.num_m_tiles + 1) / 2) * t.num_n_tiles;
                int clusters = p->pair_clusters > 0 ? p->pair_clusters : p->num_sms / 2;
                if (clusters > pair_tiles) clusters = pair_tiles;
                if (t.bres) {  // whole n-tile sets, so every cluster keeps one n-tile
                    clusters -= clusters % t.num_n_tiles;
                    if (clusters == 0) clusters = t.num_n_tiles;
                }
                gr = 2 * clusters;
                cl = 2;
            } else {
                const int units = t.dual ? ((t.num_m_tiles + 1) / 2) * t.num_n_tiles : t.num_tiles;
                gr = units < p->num_sms ? units : p->num_sms;
                if (t.bres) {  // whole n-tile sets, so every CTA keeps one n-tile
                    gr -= gr % t.num_n_tiles;
                    if (gr == 0) gr = t.num_n_tiles;
                }
            }
            break;
        }
        case CONV_PATH_SMALL_K_GEMM:
            bl = kSkThreads;
            sm = p->sk.smem_bytes;
            st = p->sk.stages;
            gr = p->sk.num_tiles < p->num_sms ? p->sk.num_tiles : p->num_sms;
            break;
        case CONV_PATH_WINOGRAD: {
            unsigned gx = 0, gy = 0;
            winograd_grid(p->g, gx, gy);
            gr = static_cast<int>(gx * gy);
            bl = kWgThreads;
            sm = winograd_smem_bytes();
            break;
        }
        case CONV_PATH_DEPTHWISE:
            bl = 256;
            sm = p->dw.smem_bytes;
            st = p->dw.stages;
            gr = p->dw.grid;
            break;
        default: {
            int tile_m = 0;
            unsigned gx = 0, gy = 0;
            direct_shape(p->g, p->num_sms, tile_m, gx, gy, bl);
            const long long blocks = static_cast<long long>(gx) * gy;
            gr = static_cast<int>(blocks < 0x7fffffffLL ? blocks : 0x7fffffffLL);
            sm = tile_m == 0 ? 0 : 2 * kDtChunk * (tile_m + 4 + kDtTileN + 4) * 4;  // static shared memory
            break;
        }
    }
    if (grid) *grid = gr;
    if (block) *block = bl;
    if (smem_bytes) *smem_bytes = sm;
    if (stages) *stages = st;
    if (cluster) *cluster = cl;
    return CONV_OK;
}

namespace {
conv_status forward_impl(conv_plan* p, const void* x, const void* w, const float* scale, const void* bias, void* y,
                         void* stream);
}  // namespace

conv_status conv_forward(conv_plan* p, const void* x, const void* w, const void* bias, void* y, void* stream) {
    return forward_impl(p, x, w, nullptr, bias, y, stream);
}

conv_status conv_forward_affine(conv_plan* p, const void* x, const void* w, const void* scale, const void* bias,
                                void* y, void* stream) {
    if (scale == nullptr) return CONV_ERR_INVALID_ARG;
    if (!aligned16(scale)) return CONV_ERR_MISALIGNED;
    return forward_impl(p, x, w, static_cast<const float*>(scale), bias, y, stream);
}

}  // extern "C"

namespace {
conv_status forward_impl(conv_plan* p, const void* x, const void* w, const float* scale, const void* bias, void* y,
                         void* stream) {
    if (p == nullptr || x == nullptr || w == nullptr || y == nullptr) return CONV_ERR_INVALID_ARG;
    if (p->device < 0) return CONV_ERR_CUDA;  // host-only plan: no device to run on
    // the plan's SM count, cluster occupancy, shared-memory limits and status word belong
    // to the device current at creation: another current device is a caller error
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    if (cur != p->device) return CONV_ERR_INVALID_ARG;
    const bool has_bias = (p->flags & CONV_FLAG_BIAS) != 0;
    if (has_bias && bias == nullptr) return CONV_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (has_bias && !aligned16(bias)))
        return CONV_ERR_MISALIGNED;
    const float* b = has_bias ? static_cast<const float*>(bias) : nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (p->path) {
        case CONV_PATH_GEMM_1X1:
        case CONV_PATH_IMPLICIT_GEMM: {
            conv_status s = encode_maps(p, x, w, y);
            if (s != CONV_OK) return s;
            TcGemmParams t = p->tc;
            t.bias = b;
            t.scale = scale;
            t.y = static_cast<__nv_bfloat16*>(y);
            int grid = 0;
            conv_plan_launch_info(p, &grid, nullptr, nullptr, nullptr, nullptr);
            e = launch_tc_gemm(p->map_a, p->map_b, p->map_y, t, grid, st);
            break;
        }
        case CONV_PATH_SMALL_K_GEMM: {  // plain and bulk copies only: no tensor maps
            SmallKParams s = p->sk;
            s.x = static_cast<const __nv_bfloat16*>(x);
            s.w = static_cast<const __nv_bfloat16*>(w);
            s.bias = b;
            s.scale = scale;
            s.y = static_cast<__nv_bfloat16*>(y);
            const int grid = s.num_tiles < p->num_sms ? s.num_tiles : p->num_sms;
            e = launch_tc_smallk(s, grid, st);
            break;
        }
        case CONV_PATH_WINOGRAD: {
            WinogradParams wp;
            wp.g = p->g;
            wp.x = x;
            wp.w = w;
            wp.bias = b;
            wp.scale = scale;
            wp.y = y;
            wp.relu = (p->flags & CONV_FLAG_RELU) ? 1 : 0;
            wp.out_bf16 = (p->flags & CONV_FLAG_OUT_BF16) ? 1 : 0;
            e = launch_winograd(wp, st);
            break;
        }
        case CONV_PATH_DEPTHWISE: {
            conv_status s = encode_maps(p, x, w, y);
            if (s != CONV_OK) return s;
            DepthwiseParams d = p->dw;
            d.w = static_cast<const float*>(w);
            d.bias = b;
            d.scale = scale;
            d.y = y;
            e = launch_depthwise(p->map_a, d, st);
            break;
        }
        default: {
            DirectParams d;
            d.g = p->g;
            d.x = x;
            d.w = w;
            d.bias = b;
            d.scale = scale;
            d.y = y;
            d.relu = (p->flags & CONV_FLAG_RELU) ? 1 : 0;
            d.in_bf16 = p->dtype == CONV_BF16 ? 1 : 0;
            d.out_bf16 = (p->dtype == CONV_BF16 || (p->flags & CONV_FLAG_OUT_BF16)) ? 1 : 0;
            d.transposed = (p->flags & CONV_FLAG_TRANSPOSED) ? 1 : 0;
            d.tile_m = 0;  // chosen by the launcher
            e = launch_direct(d, p->num_sms, st);
            break;
        }
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    return CONV_OK;
}

}  // namespace

extern "C" {

conv_status conv_plan_destroy(conv_plan* p) {
    if (p != nullptr) release_status_word(p->device, p->status_slot);
    delete p;
    return CONV_OK;
}

conv_status conv_plan_device_status(const conv_plan* p, void* stream, int* code) {
    if (p == nullptr || code == nullptr) return CONV_ERR_INVALID_ARG;
    *code = 0;
    if (p->device < 0) return CONV_ERR_CUDA;  // host-only plan
    return read_status_word(p->device, p->status, stream, code);
}

const char* conv_status_string(conv_status s) {
    switch (s) {
        case CONV_OK: return "ok";
        case CONV_ERR_INVALID_ARG: return "invalid argument";
        case CONV_ERR_UNSUPPORTED: return "unsupported convolution";
        case CONV_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case CONV_ERR_CUDA: return "CUDA call failed";
        case CONV_ERR_NO_MEMORY: return "host allocation failed";
        case CONV_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

conv_status conv_device_status(int* code) {
    if (code == nullptr) return CONV_ERR_INVALID_ARG;
    *code = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return CONV_ERR_CUDA;
    // the library-wide word and every plan's own word
    static unsigned words[kStatusSlots];  // guarded: conv_device_status may run on several threads
    static std::mutex words_mutex;
    std::lock_guard<std::mutex> lock(words_mutex);
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_conv_status_word, sizeof(v)) != cudaSuccess ||
        cudaMemcpyFromSymbol(words, g_conv_status_slots, sizeof(words)) != cudaSuccess)
        return CONV_ERR_CUDA;
    unsigned any = v;
    for (int i = 0; i < kStatusSlots; ++i) any |= words[i];
    if (any != 0) {
        const unsigned zero = 0;
        for (int i = 0; i < kStatusSlots; ++i) words[i] = 0;
        if (cudaMemcpyToSymbol(g_conv_status_word, &zero, sizeof(zero)) != cudaSuccess ||
            cudaMemcpyToSymbol(g_conv_status_slots, words, sizeof(words)) != cudaSuccess)
            return CONV_ERR_CUDA;
    }
    *code = static_cast<int>(any);
    return any ? CONV_ERR_TIMEOUT : CONV_OK;
}

}  // extern "C"
