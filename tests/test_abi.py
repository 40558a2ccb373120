"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/conv.h declares, validates shapes, and picks kernels."""
import ctypes
import os
import re

import pytest
import torch

import cnn_convolution_implicit_gb300 as cg
from cnn_convolution_implicit_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "conv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(conv_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    L = cg.lib()
    declared = header_functions()
    assert set(declared) == set(binding.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings():
    L = cg.lib()
    for code in range(7):
        assert L.conv_status_string(code)
    assert L.conv_status_string(99) == b"unknown status"


def _create(*args):
    L = cg.lib()
    h = ctypes.c_void_p(1234)
    st = L.conv_plan_create(ctypes.byref(h), *args)
    return st, h


@pytest.mark.parametrize("args", [
    (0, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 0, 0),        # N = 0
    (1, 3, 8, 8, 4, 3, 3, 0, 1, 1, 1, 0, 0),        # S = 0
    (1, 3, 8, 8, 4, 3, 3, 1, -1, 1, 1, 0, 0),       # P < 0
    (1, 3, 8, 8, 4, 3, 3, 1, 1, 0, 1, 0, 0),        # D = 0
    (1, 6, 8, 8, 4, 3, 3, 1, 1, 1, 4, 0, 0),        # C_in % G
    (1, 8, 8, 8, 6, 3, 3, 1, 1, 1, 4, 0, 0),        # C_out % G
    (1, 3, 2, 2, 4, 5, 5, 1, 0, 1, 1, 0, 0),        # empty output
    (1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 1, 4),        # OUT_BF16 with BF16 input
    (1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 2, 0),        # bad dtype
    (1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 0, 256),      # unknown flag
    (1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 0, 512),      # unknown flag
    (1, 3, 2, 2, 4, 3, 3, 1, 3, 1, 1, 0, 16),       # transposed with an empty output: (2-1) - 6 + 2 + 1 < 1
])
def test_create_rejects_bad_shapes(args):
    st, h = _create(*args)
    assert st == 1 and h.value is None


def test_create_null_out_and_null_plan_calls():
    L = cg.lib()
    assert L.conv_plan_create(None, 1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 0, 0) == 1
    assert L.conv_plan_destroy(None) == 0
    a, b = ctypes.c_int(), ctypes.c_int()
    assert L.conv_plan_output_shape(None, ctypes.byref(a), ctypes.byref(b)) == 1
    assert L.conv_forward(None, 16, 16, None, 16, None) == 1
    assert L.conv_forward_affine(None, 16, 16, 16, None, 16, None) == 1
    assert L.conv_device_status(None) == 1
    p = cg.ConvPlan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, 1, "f32")
    assert L.conv_forward_affine(p._plan, 256, 256, None, None, 256, None) == 1   # scale required
    assert L.conv_forward_affine(p._plan, 256, 256, 260, None, 256, None) == 3    # misaligned scale


@pytest.mark.parametrize("shape,path", [
    ((32, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1, "bf16"), "implicit_gemm"),
    ((32, 3, 224, 224, 32, 3, 3, 2, 1, 1, 1, "bf16"), "small_k_gemm"),
    ((64, 256, 56, 56, 256, 3, 3, 1, 1, 1, 256, "f32"), "depthwise"),
    ((64, 256, 56, 56, 512, 1, 1, 1, 0, 1, 1, "bf16"), "gemm_1x1"),
    ((16, 256, 64, 64, 256, 3, 3, 1, 2, 2, 4, "bf16"), "implicit_gemm"),
    ((1, 3, 32, 32, 8, 3, 3, 1, 1, 1, 1, "f32"), "direct"),
    ((2, 64, 9, 9, 24, 3, 3, 1, 1, 1, 1, "bf16"), "direct"),          # C_out % 16 != 0
    ((2, 96, 9, 9, 64, 3, 3, 1, 1, 1, 1, "bf16"), "direct"),          # C_in not a multiple of 64, K > 64
    ((2, 128, 9, 9, 64, 1, 1, 2, 0, 1, 1, "bf16"), "implicit_gemm"),  # strided 1x1 -> im2col
    ((2, 128, 9, 9, 64, 3, 3, 1, 1, 1, 2, "bf16"), "implicit_gemm"),  # 2 groups packed per tile
    ((2, 48, 9, 9, 48, 3, 3, 1, 1, 1, 48, "f32"), "direct"),          # depthwise, C % 32 != 0
    ((2, 64, 9, 9, 64, 3, 3, 1, 1, 1, 64, "bf16"), "direct"),         # BF16 depthwise
    ((2, 4, 30, 300, 64, 3, 3, 1, 1, 1, 1, "bf16"), "small_k_gemm"),  # 3 segments per row
])
def test_kernel_choice(shape, path):
    *dims, dtype = shape
    p = cg.ConvPlan(*dims, dtype=dtype, bias=True, relu=True)
    assert p.path == path


def test_gemm_extents_body_layer():
    """Per image, the 112x112x128 -> 256 3x3 layer is a 256 x 12544 x 1152 GEMM
    ("Convolution variants and their matrix operations", section 3.3)."""
    p = cg.ConvPlan(1, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1, "bf16")
    assert p.gemm_mnk == (256, 12544, 1152)
    assert (p.H_out, p.W_out) == (112, 112)


def test_output_shape_matches_formula():
    for (H, K, S, P, D) in [(224, 3, 2, 1, 1), (64, 3, 1, 2, 2), (7, 5, 3, 0, 1), (9, 2, 2, 3, 3)]:
        p = cg.ConvPlan(1, 8, H, H, 8, K, K, S, P, D, 1, "f32")
        exp = (H + 2 * P - D * (K - 1) - 1) // S + 1
        assert (p.H_out, p.W_out) == (exp, exp)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device behaviour")
def test_forward_without_device_fails_loudly():
    p = cg.ConvPlan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, 1, "f32")
    L = cg.lib()
    assert L.conv_forward(p._plan, 256, 256, 256, 256, None) == 4  # CONV_ERR_CUDA, nothing launched


# ----------------------------------------------------------------- fused depthwise-separable block
def _block_create(*args):
    L = cg.lib()
    h = ctypes.c_void_p(1234)
    st = L.conv_block_plan_create(ctypes.byref(h), *args)
    return st, h


@pytest.mark.parametrize("args,status", [
    ((0, 64, 8, 8, 32, 3, 1, 0), 1),       # N = 0
    ((1, 64, 8, 8, 32, 3, -1, 0), 1),      # P < 0
    ((1, 64, 1, 1, 32, 3, 0, 0), 1),       # empty output
    ((1, 64, 8, 8, 32, 3, 1, 4), 1),       # unknown flag
    ((1, 64, 8, 8, 32, 5, 2, 0), 2),       # 5x5 depthwise: not fused
    ((1, 64, 8, 8, 32, 3, 3, 0), 2),       # P > 2
    ((1, 96, 8, 8, 32, 3, 1, 0), 2),       # C % 64 != 0
    ((1, 320, 8, 8, 32, 3, 1, 0), 2),      # C > 256
    ((1, 64, 8, 8, 48, 3, 1, 0), 2),       # C_out % 32 != 0
])
def test_block_create_rejects(args, status):
    st, h = _block_create(*args)
    assert st == status and h.value is None


@pytest.mark.parametrize("C_out,slices", [(32, 1), (256, 1), (320, 2), (384, 2), (512, 2), (352, 11), (768, 3)])
def test_block_output_slices_and_stages(C_out, slices):
    p = cg.BlockPlan(2, 128, 12, 12, C_out, 3, 1)
    assert (p.H_out, p.W_out) == (12, 12)
    assert p.launch["block"] == 480
    assert p.launch["halo_stages"] >= 2 and p.launch["weight_stages"] >= 2
    assert p.launch["smem_bytes"] <= 232448


def test_block_full_size_launch():
    p = cg.BlockPlan(64, 256, 56, 56, 512, 3, 1)
    assert (p.H_out, p.W_out) == (56, 56)
    tiles = 64 * 4 * 7  # 16 x 8 output tiles: 56 / 16 -> 4 rows of tiles, 56 / 8 -> 7 columns
    assert 1 <= p.launch["grid"] <= tiles
    if not torch.cuda.is_available():
        assert p.launch["grid"] == 152  # host-only plan: one persistent CTA per SM of a 152-SM part


def test_block_null_and_misaligned_calls():
    L = cg.lib()
    assert L.conv_block_plan_create(None, 1, 64, 8, 8, 32, 3, 1, 0) == 1
    assert L.conv_block_plan_destroy(None) == 0
    a, b = ctypes.c_int(), ctypes.c_int()
    assert L.conv_block_plan_output_shape(None, ctypes.byref(a), ctypes.byref(b)) == 1
    assert L.conv_block_plan_launch_info(None, None, None, None, None, None) == 1
    assert L.conv_block_forward(None, 16, 16, None, None, 16, None, None, 16, None) == 1
    p = cg.BlockPlan(1, 64, 8, 8, 32, 3, 1)
    assert L.conv_block_forward(p._plan, None, 256, None, None, 256, None, None, 256, None) == 1
    assert L.conv_block_forward(p._plan, 256, 256, 260, None, 256, None, None, 256, None) == 3
    assert L.conv_block_forward(p._plan, 256, 256, None, None, 256, None, 264, 256, None) == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device behaviour")
def test_block_forward_without_device_fails_loudly():
    p = cg.BlockPlan(1, 64, 8, 8, 32, 3, 1)
    L = cg.lib()
    assert L.conv_block_forward(p._plan, 256, 256, None, None, 256, None, None, 256, None) == 4


@pytest.mark.parametrize("shape,path", [
    ((16, 256, 56, 56, 128, 4, 4, 2, 1, 1, 1, "bf16"), "implicit_gemm"),   # the upsampling layer
    ((2, 64, 9, 7, 64, 3, 3, 1, 1, 1, 1, "bf16"), "implicit_gemm"),        # stride 1
    ((2, 64, 6, 6, 32, 3, 3, 2, 1, 1, 1, "bf16"), "direct"),               # H_out = 11, not a multiple of S
    ((2, 64, 6, 6, 32, 1, 1, 2, 0, 1, 1, "bf16"), "direct"),               # odd phases have no tap
    ((2, 64, 6, 6, 32, 9, 9, 2, 4, 1, 1, "bf16"), "direct"),               # K > 8
    ((2, 64, 6, 6, 32, 5, 5, 5, 0, 1, 1, "bf16"), "direct"),               # S > 4
    ((2, 64, 8, 8, 64, 3, 3, 1, 1, 1, 64, "f32"), "direct"),               # FP32 depthwise-shaped: direct
])
def test_transposed_kernel_choice(shape, path):
    *dims, dtype = shape
    p = cg.ConvPlan(*dims, dtype=dtype, bias=True, relu=True, transposed=True)
    assert p.path == path
    N, C_in, H, W, C_out, Kh, Kw, S, P, D, G = dims
    assert p.H_out == (H - 1) * S - 2 * P + D * (Kh - 1) + 1
    assert p.W_out == (W - 1) * S - 2 * P + D * (Kw - 1) + 1
    # matrix form Y_col = W^T X (variants page, section 4.2)
    assert p.gemm_mnk == (C_out * Kh * Kw, N * H * W, C_in // G)


@pytest.mark.parametrize("shape,winograd,path", [
    ((8, 64, 56, 56, 64, 3, 3, 1, 1, 1, 1, "f32"), True, "winograd"),
    ((8, 64, 56, 56, 64, 3, 3, 1, 1, 1, 1, "f32"), False, "direct"),     # opt-in only
    ((1, 3, 32, 32, 8, 3, 3, 1, 1, 1, 1, "f32"), True, "winograd"),      # ragged channels
    ((2, 8, 9, 9, 8, 3, 3, 2, 1, 1, 1, "f32"), True, "direct"),          # stride 2
    ((2, 8, 9, 9, 8, 3, 3, 1, 2, 2, 1, "f32"), True, "direct"),          # dilation 2
    ((2, 8, 9, 9, 8, 5, 5, 1, 2, 1, 1, "f32"), True, "direct"),          # 5x5
    ((2, 8, 9, 9, 8, 3, 3, 1, 1, 1, 2, "f32"), True, "direct"),          # groups
    ((2, 64, 9, 9, 64, 3, 3, 1, 1, 1, 64, "f32"), True, "depthwise"),    # depthwise keeps its kernel
    ((2, 128, 9, 9, 128, 3, 3, 1, 1, 1, 1, "bf16"), True, "implicit_gemm"),  # BF16: tensor cores
    ((2 ** 27, 4, 64, 64, 8, 3, 3, 1, 1, 1, 1, "f32"), True, "direct"),  # its grid would pass 2**31 blocks
])
def test_winograd_kernel_choice(shape, winograd, path):
    *dims, dtype = shape
    p = cg.ConvPlan(*dims, dtype=dtype, bias=True, relu=True, winograd=winograd)
    assert p.path == path


@pytest.mark.parametrize("shape,sm_pairs,cluster", [
    ((32, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1), None, 2),    # body: long full-width reduction -> pairs
    ((32, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1), False, 1),   # forced one SM
    ((64, 256, 56, 56, 512, 1, 1, 1, 0, 1, 1), None, 1),      # pointwise: 4 K-steps -> one SM (resident weights)
    ((64, 256, 56, 56, 512, 1, 1, 1, 0, 1, 1), True, 2),      # forced pairs
    ((16, 256, 64, 64, 256, 3, 3, 1, 2, 2, 4), None, 1),      # grouped: N = 64 per group -> one SM
    ((4, 128, 31, 29, 256, 3, 3, 2, 1, 1, 1), None, 2),       # strided (im2col mode), 18 K-steps, 8 tiles
])
def test_sm_pair_choice(shape, sm_pairs, cluster):
    p = cg.ConvPlan(*shape, dtype="bf16", bias=True, relu=True, sm_pairs=sm_pairs)
    assert p.launch["cluster"] == cluster


def test_sm_pair_flags_are_exclusive():
    st, h = _create(1, 128, 8, 8, 256, 3, 3, 1, 1, 1, 1, 1, 8 | 64)
    assert st == 1 and h.value is None


# ----------------------------------------------------------------- tensor-rate measurement helper
def test_mma_rate_rejects_bad_arguments_without_launching():
    """Invalid counts, a null or misaligned cycles array, or an empty grid return before
    any CUDA call (the pointers are only checked, never dereferenced)."""
    L = cg.lib()
    buf = (ctypes.c_ulonglong * 4)()
    base = ctypes.addressof(buf)
    assert L.conv_measure_mma_rate(0, ctypes.c_void_p(base), 1, None) == 1  # CONV_ERR_INVALID_ARG
    assert L.conv_measure_mma_rate((1 << 20) + 1, ctypes.c_void_p(base), 1, None) == 1
    assert L.conv_measure_mma_rate(16, None, 1, None) == 1
    assert L.conv_measure_mma_rate(16, ctypes.c_void_p(base), 0, None) == 1
    assert L.conv_measure_mma_rate(16, ctypes.c_void_p(base + 4), 1, None) == 3  # CONV_ERR_MISALIGNED
    assert list(buf) == [0, 0, 0, 0]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device behaviour")
def test_mma_rate_without_device_fails_loudly():
    L = cg.lib()
    buf = (ctypes.c_ulonglong * 1)()
    assert L.conv_measure_mma_rate(16, ctypes.c_void_p(ctypes.addressof(buf)), 1, None) == 4  # CONV_ERR_CUDA


# Stride-1 BF16 implicit-GEMM plans take the halo mode (one input halo per 64-channel
# block, 8 x 16 output tiles, a second producer warp: 608 threads); CONV_FLAG_PER_TAP,
# other strides, 1x1 layers and halos wider than a TMA box (256) keep one box per tap.
@pytest.mark.parametrize("shape,halo", [
    ((32, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1), True),     # body layer (SM pairs)
    ((16, 256, 64, 64, 256, 3, 3, 1, 2, 2, 4), True),       # dilated grouped (two tiles per CTA)
    ((2, 64, 12, 12, 64, 5, 5, 1, 2, 1, 1), True),          # 5x5
    ((2, 64, 10, 14, 64, 1, 3, 1, 1, 1, 1), True),          # 1x3
    ((2, 512, 8, 8, 128, 3, 3, 1, 2, 2, 8), True),          # groups packed side by side
    ((1, 128, 9, 11, 256, 3, 3, 2, 1, 1, 1), False),        # stride 2: TMA im2col mode
    ((2, 256, 9, 13, 512, 1, 1, 1, 0, 1, 1), False),        # 1x1 GEMM
    ((1, 64, 4, 300, 64, 1, 3, 1, 125, 125, 1), False),     # halo 8 + 2*125 = 258 columns > 256
])
def test_halo_mode_choice(shape, halo):
    """The halo mode adds a weight-producer warp to the per-tap kernel's 576 threads (18
    warps); two pixel tiles per CTA add a second MMA-issuing warp in either mode."""
    p = cg.ConvPlan(*shape, dtype="bf16", bias=True, relu=True)
    assert p.path in ("implicit_gemm", "gemm_1x1")
    assert p.launch["smem_bytes"] <= 232448
    assert p.launch["stages"] >= (1 if p.gemm["resident_weights"] else 2)
    assert (p.gemm["mode"] == 4) == halo
    q = cg.ConvPlan(*shape, dtype="bf16", bias=True, relu=True, per_tap=True)
    assert q.path == p.path and q.launch["block"] in (576, 608) and q.gemm["mode"] != 4
    assert p.launch["block"] == q.launch["block"] + (32 if halo else 0)


# Resident weights: where one n-tile's weight rows for the whole reduction fit in shared
# memory beside the operand ring (two halos in the halo mode, four A stages in the 1x1
# mode), on one SM per unit; every CTA keeps one n-tile, so the grid is a multiple of the
# n-tile count.  (shape, resident, n-tiles)
@pytest.mark.parametrize("shape,resident,sm_pairs", [
    ((16, 256, 64, 64, 256, 3, 3, 1, 2, 2, 4), 1, None),   # dilated grouped: 9 taps x 64 rows (72 KB)
    ((64, 256, 56, 56, 512, 1, 1, 1, 0, 1, 1), 1, None),   # pointwise: 4 blocks x 256 rows (128 KB)
    ((3, 256, 9, 13, 768, 1, 1, 1, 0, 1, 1), 1, None),     # three n-tiles
    ((2, 256, 21, 19, 64, 3, 3, 1, 1, 1, 2), 1, None),     # two channel blocks per tap, two groups
    ((2, 64, 10, 14, 256, 1, 3, 1, 1, 1, 1), 1, None),     # halo mode, one tile per CTA
    ((64, 256, 56, 56, 512, 1, 1, 1, 0, 1, 1), 1, True),   # 1x1 on SM pairs: half the rows per SM
    ((32, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1), 0, None),  # body: 18 K-steps x 128 rows do not fit
    ((2, 64, 12, 12, 64, 5, 5, 1, 2, 1, 1), 0, None),      # 25 taps x 64 rows beside two halos do not fit
    ((4, 128, 31, 29, 256, 3, 3, 2, 1, 1, 1), 0, None),    # strided (im2col mode): weights stream
])
def test_resident_weights_choice(shape, resident, sm_pairs):
    p = cg.ConvPlan(*shape, dtype="bf16", bias=True, relu=True, sm_pairs=sm_pairs)
    assert p.gemm["resident_weights"] == resident
    assert p.launch["smem_bytes"] <= 232448
    if resident:
        n_tiles = shape[4] // p.gemm["n_tile"]
        per_cta = p.launch["grid"] // p.launch["cluster"]
        assert per_cta % n_tiles == 0


def test_gemm_config_other_paths():
    """conv_plan_gemm_config answers for the tensor-core GEMM paths only."""
    p = cg.ConvPlan(2, 64, 9, 9, 64, 3, 3, 1, 1, 1, 64, dtype="f32", bias=True, relu=True)
    assert p.path == "depthwise" and p.gemm is None
    assert cg.lib().conv_plan_gemm_config(None, None, None, None, None, None, None) == 1


# Swapped operands (weights on the MMA's M side, both tiles' pixels on N) for two-tile units of
# exactly 128 output channels in the per-tap modes; never in the halo mode or at other widths.
@pytest.mark.parametrize("shape,flags,swapped", [
    ((16, 256, 56, 56, 128, 4, 4, 2, 1, 1, 1), {"transposed": True}, 1),  # transposed upsampling (phase mode)
    ((4, 128, 29, 23, 128, 3, 3, 2, 1, 1, 1), {}, 1),                      # strided (im2col mode)
    ((2, 256, 9, 13, 128, 1, 1, 1, 0, 1, 1), {}, 1),                       # 1x1, two tiles per CTA
    ((2, 64, 13, 11, 128, 3, 3, 1, 1, 1, 1), {"per_tap": True}, 1),        # one box per tap
    ((2, 64, 13, 11, 128, 3, 3, 1, 1, 1, 1), {}, 0),                       # halo mode
    ((16, 256, 64, 64, 256, 3, 3, 1, 2, 2, 4), {}, 0),                     # 64-channel groups
    ((2, 128, 13, 11, 64, 3, 3, 2, 1, 1, 1), {}, 0),                       # 64 channels
])
def test_swapped_operand_choice(shape, flags, swapped):
    p = cg.ConvPlan(*shape, dtype="bf16", bias=True, relu=True, **flags)
    assert p.gemm["swapped"] == swapped
    if swapped:
        assert p.gemm["dual"] == 1 and p.gemm["n_tile"] == 128


def test_wait_timeout_check_rejects_bad_arguments_without_launching():
    """conv_check_wait_timeout validates its limit and pointer before any CUDA call; with
    no device a valid call fails loudly (CONV_ERR_CUDA), it never runs on the host."""
    L = cg.lib()
    assert L.conv_check_wait_timeout(0, None, None) == 1                 # limit 0
    assert L.conv_check_wait_timeout(2_000_000_001, None, None) == 1     # above the kernels' own 2 s
    assert L.conv_check_wait_timeout(1_000_000, ctypes.c_void_p(12), None) == 3  # misaligned
    import torch
    if not torch.cuda.is_available():
        assert L.conv_check_wait_timeout(1_000_000, None, None) == 4


def test_plan_status_words_validate_arguments():
    """conv_plan_device_status / conv_block_plan_device_status reject NULL arguments; a
    host-only plan (no device at creation) has no word of its own and fails loudly."""
    L = cg.lib()
    code = ctypes.c_int(7)
    assert L.conv_plan_device_status(None, None, ctypes.byref(code)) == 1
    assert L.conv_block_plan_device_status(None, None, ctypes.byref(code)) == 1
    p = cg.ConvPlan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, 1, "f32")
    b = cg.BlockPlan(1, 64, 8, 8, 32, 3, 1)
    assert L.conv_plan_device_status(p._plan, None, None) == 1
    assert L.conv_block_plan_device_status(b._plan, None, None) == 1
    if not torch.cuda.is_available():
        assert L.conv_plan_device_status(p._plan, None, ctypes.byref(code)) == 4
        assert code.value == 0
        code.value = 7
        assert L.conv_block_plan_device_status(b._plan, None, ctypes.byref(code)) == 4
        assert code.value == 0
