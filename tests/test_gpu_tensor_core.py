"""GPU parity: the tcgen05 paths (implicit GEMM with TMA im2col, 1x1 GEMM,
small-K stem kernel) against the FP64 oracle.  BF16 inputs, FP32 accumulate,
BF16 output; tolerance |y - y_ref| <= 2e-2 * (1 + |y_ref|)."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_full, check_points, oracle_full, run, sample_points
from workloads import ConvShape, draw, inputs

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------- small shapes, every output
@pytest.mark.parametrize("shape,path", [
    # implicit GEMM, several K-steps per tap, ragged last pixel tile
    (ConvShape(2, 64, 13, 11, 32, 3, 3, 1, 1, 1, 1, "bf16", True, True), "implicit_gemm"),
    (ConvShape(1, 128, 9, 11, 256, 3, 3, 2, 1, 1, 1, "bf16", True, False), "implicit_gemm"),  # stride 2
    (ConvShape(2, 64, 12, 12, 64, 5, 5, 1, 2, 1, 1, "bf16", False, True), "implicit_gemm"),   # 5x5
    (ConvShape(2, 64, 15, 13, 64, 3, 3, 1, 3, 3, 1, "bf16", True, True), "implicit_gemm"),    # dilation 3
    (ConvShape(2, 64, 10, 14, 64, 1, 3, 1, 1, 1, 1, "bf16", True, False), "implicit_gemm"),   # 1x3, Kh != Kw
    (ConvShape(2, 64, 14, 10, 64, 3, 1, 1, 1, 1, 1, "bf16", True, False), "implicit_gemm"),   # 3x1
    (ConvShape(2, 64, 11, 9, 32, 3, 3, 2, 0, 1, 1, "bf16", True, True), "implicit_gemm"),     # no padding
    (ConvShape(1, 64, 7, 9, 32, 3, 3, 1, 1, 1, 1, "bf16", True, True), "implicit_gemm"),      # < 1 tile
    (ConvShape(2, 128, 9, 9, 64, 1, 1, 2, 0, 1, 1, "bf16", True, True), "implicit_gemm"),     # strided 1x1
    # groups: packed per tile, and one group spanning a tile
    (ConvShape(2, 128, 9, 9, 64, 3, 3, 1, 1, 1, 2, "bf16", True, True), "implicit_gemm"),
    (ConvShape(2, 512, 8, 8, 128, 3, 3, 1, 2, 2, 8, "bf16", True, True), "implicit_gemm"),
    (ConvShape(1, 256, 8, 8, 256, 3, 3, 1, 2, 2, 4, "bf16", True, True), "implicit_gemm"),
    # 1x1 GEMM path, including two N-tiles and a ragged pixel tail
    (ConvShape(2, 64, 7, 9, 32, 1, 1, 1, 0, 1, 1, "bf16", True, True), "gemm_1x1"),
    (ConvShape(3, 256, 9, 13, 512, 1, 1, 1, 0, 1, 1, "bf16", True, True), "gemm_1x1"),
    (ConvShape(1, 128, 5, 5, 96, 1, 1, 1, 0, 1, 1, "bf16", False, False), "gemm_1x1"),
    # small-K kernel
    (ConvShape(2, 3, 40, 40, 32, 3, 3, 2, 1, 1, 1, "bf16", True, True), "small_k_gemm"),
    (ConvShape(2, 3, 17, 24, 64, 3, 3, 1, 1, 1, 1, "bf16", True, False), "small_k_gemm"),
    (ConvShape(1, 4, 6, 300, 32, 3, 3, 1, 1, 1, 1, "bf16", True, True), "small_k_gemm"),      # 3 segments
    (ConvShape(2, 1, 20, 32, 32, 7, 7, 2, 3, 1, 1, "bf16", True, True), "small_k_gemm"),      # 49 taps
    (ConvShape(1, 8, 12, 16, 256, 2, 2, 1, 0, 2, 1, "bf16", False, True), "small_k_gemm"),    # dilation
    (ConvShape(3, 3, 30, 24, 32, 3, 3, 2, 1, 1, 1, "bf16", True, True), "small_k_gemm"),      # H_out 15: stages cross images
    (ConvShape(1, 3, 2, 16, 32, 3, 3, 1, 3, 1, 1, "bf16", True, False), "small_k_gemm"),      # rows that are all padding
    (ConvShape(2, 3, 16, 24, 32, 3, 3, 1, 2, 1, 1, "bf16", True, True), "small_k_gemm"),      # P = 2: two taps off each side
    (ConvShape(2, 3, 21, 16, 32, 1, 1, 2, 0, 1, 1, "bf16", True, True), "small_k_gemm"),      # S > K: row per copy
    # whole-row stages (one segment per row, H_out a multiple of the rows per stage: copies in closed form)
    (ConvShape(1, 3, 4, 16, 32, 3, 3, 1, 3, 1, 1, "bf16", True, False), "small_k_gemm"),      # all-padding rows
    (ConvShape(2, 3, 14, 24, 32, 3, 3, 1, 2, 1, 1, "bf16", True, True), "small_k_gemm"),      # P = 2
    (ConvShape(2, 3, 16, 24, 64, 3, 3, 2, 1, 1, 1, "bf16", True, True), "small_k_gemm"),      # C_out = 64
])
@pytest.mark.parametrize("sm_pairs", [False, True], ids=["single_sm", "sm_pairs"])
def test_tensor_core_small_shapes_full(shape, path, sm_pairs):
    """Every output, on both tcgen05 GEMM kernels: CTA pairs (cta_group::2, M = 256)
    and one CTA per tile (cta_group::1, M = 128)."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    x, w, b = draw(shape, (31, 32, 33))
    plan, y = run(shape, x, w, b, plan=ConvPlan.for_shape(shape, sm_pairs=sm_pairs))
    assert plan.path == path
    check_full(shape, y, oracle_full(shape, x, w, b))


def test_small_k_random_sweep():
    """Random BF16 shapes that plan to the small-K kernel (C_in * Kh * Kw <= 64): strides,
    paddings, dilations and widths that split rows into several segments; every output."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    rng = np.random.default_rng(23)
    done = 0
    while done < 12:
        C_in = int(rng.integers(1, 8))
        K = int(rng.choice([1, 2, 3, 5, 7]))
        if C_in * K * K > 64:
            continue
        W = int(rng.choice([8, 16, 24, 40, 136, 264]))
        if (W * C_in * 2) % 16 != 0:
            continue
        s = ConvShape(int(rng.integers(1, 4)), C_in, int(rng.integers(2, 24)), W, int(rng.choice([32, 64, 96, 128])),
                      K, K, int(rng.choice([1, 2, 3])), int(rng.integers(0, 4)), int(rng.choice([1, 2])), 1, "bf16",
                      bool(rng.integers(0, 2)), bool(rng.integers(0, 2)))
        if s.H_out < 1 or s.W_out < 1 or ConvPlan.for_shape(s).path != "small_k_gemm":
            continue
        x, w, b = draw(s, (800 + done, 810 + done, 820 + done))
        plan, y = run(s, x, w, b)
        check_full(s, y, oracle_full(s, x, w, b))
        done += 1


def test_measured_mma_rate():
    """conv_measure_mma_rate: every SM's chain of M128 N256 K16 MMAs completes and gives a
    FLOP-per-clock rate in a plausible band (dense BF16 on one SM is a few thousand FLOP
    per clock), the same on every SM within 10 %."""
    from cnn_convolution_implicit_gb300 import measure_mma_rate
    fpc, per_sm, sms = measure_mma_rate(1 << 14)
    assert sms == torch.cuda.get_device_properties(0).multi_processor_count
    assert np.all(np.isfinite(per_sm)) and len(per_sm) == sms
    assert 2048 <= fpc <= 16384, fpc
    assert np.all(np.abs(per_sm / fpc - 1) < 0.1), (per_sm.min(), per_sm.max())


def test_two_calls_same_plan_are_identical():
    s = ConvShape(2, 128, 13, 13, 256, 3, 3, 1, 1, 1, 1, "bf16", True, True)
    x, w, b = draw(s, (41, 42, 43))
    plan, y1 = run(s, x, w, b)
    plan, y2 = run(s, x, w, b, plan=plan)
    assert torch.equal(y1, y2)


# ----------------------------------------------------------------- full-size layers
def test_stem_full_size_all_outputs():
    """N=32, 3->32, 224 -> 112, 3x3 s2 p1, bias+ReLU: every output against the oracle."""
    s, x, w, b = inputs("stem")
    plan, y = run(s, x, w, b)
    assert plan.path == "small_k_gemm"
    check_full(s, y, oracle_full(s, x, w, b))


def test_body_full_size_one_sm_kernel():
    """The one-SM-per-tile kernel on the full body layer (the plan's own choice there is SM
    pairs): seeded points."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    s, x, w, b = inputs("body")
    plan, y = run(s, x, w, b, plan=ConvPlan.for_shape(s, sm_pairs=False))
    assert plan.launch["cluster"] == 1
    check_points(s, y, x, w, b, sample_points(s, 4096, 13))


def test_body_full_size():
    """N=32, 128->256, 112x112, 3x3 s1 p1, bias+ReLU (halo mode on SM pairs): every output
    of the batch against the FP64 oracle, in chunks of images to bound host memory."""
    s, x, w, b = inputs("body")
    plan, y = run(s, x, w, b)
    assert plan.path == "implicit_gemm" and plan.launch["block"] == 608 and plan.launch["cluster"] == 2  # halo, pairs
    for n0 in range(0, s.N, 8):
        ref = oracle.conv2d(x[n0:n0 + 8], w, b, 1, 1, 1, 1, True)
        check_full(s, y[n0:n0 + 8], ref)


def test_pointwise_full_size():
    """N64, 256 -> 512, 56x56 1x1 + bias + ReLU: every output of the batch against the
    FP64 oracle ("Convolution variants", section 6.4: compare every element)."""
    s, x, w, b = inputs("pw")
    plan, y = run(s, x, w, b)
    assert plan.path == "gemm_1x1"
    check_full(s, y, oracle_full(s, x, w, b))


def test_dilated_grouped_full_size():
    """N16, 256 -> 256, 64x64, 3x3 d2 p2 g4 + bias + ReLU (halo mode, two tiles per CTA):
    every output of the batch against the FP64 oracle."""
    s, x, w, b = inputs("dilated")
    plan, y = run(s, x, w, b)
    assert plan.path == "implicit_gemm" and plan.launch["block"] == 640  # halo mode, two MMA warps
    check_full(s, y, oracle_full(s, x, w, b))


# stride-1 implicit-GEMM shapes of the small-shape list, run with one TMA box per tap
# (CONV_FLAG_PER_TAP) instead of the default halo tiles
PER_TAP_SHAPES = [
    ConvShape(2, 64, 13, 11, 32, 3, 3, 1, 1, 1, 1, "bf16", True, True),
    ConvShape(2, 64, 12, 12, 64, 5, 5, 1, 2, 1, 1, "bf16", False, True),
    ConvShape(2, 64, 15, 13, 64, 3, 3, 1, 3, 3, 1, "bf16", True, True),
    ConvShape(2, 64, 10, 14, 64, 1, 3, 1, 1, 1, 1, "bf16", True, False),
    ConvShape(2, 128, 9, 9, 64, 3, 3, 1, 1, 1, 2, "bf16", True, True),
    ConvShape(1, 256, 8, 8, 256, 3, 3, 1, 2, 2, 4, "bf16", True, True),
    ConvShape(2, 128, 20, 27, 256, 3, 3, 1, 1, 1, 1, "bf16", True, True),
]


@pytest.mark.parametrize("shape", PER_TAP_SHAPES, ids=lambda s: "K%dx%dD%dG%d_%dx%d" % (s.Kh, s.Kw, s.D, s.G, s.H, s.W))
@pytest.mark.parametrize("sm_pairs", [False, True], ids=["single_sm", "sm_pairs"])
def test_per_tap_mode_full(shape, sm_pairs):
    """Every output with one input box per tap (the per-tap mode): same results as the
    halo mode up to the order of the FP32 sum, both against the oracle."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    x, w, b = draw(shape, (61, 62, 63))
    ref = oracle_full(shape, x, w, b)
    plan, y = run(shape, x, w, b, plan=ConvPlan.for_shape(shape, sm_pairs=sm_pairs, per_tap=True))
    assert plan.path == "implicit_gemm" and plan.launch["block"] in (576, 608)
    check_full(shape, y, ref)
    plan_h, y_h = run(shape, x, w, b, plan=ConvPlan.for_shape(shape, sm_pairs=sm_pairs))
    assert plan_h.launch["block"] == plan.launch["block"] + 32  # the halo mode's weight-producer warp
    check_full(shape, y_h, ref)


# Resident weights: each CTA keeps one n-tile's weight rows for the whole reduction in
# shared memory (halo mode with one and two tiles per CTA, 1x1 mode on one SM and on SM
# pairs), including two channel blocks per tap, several n-tiles and ragged tiles.
RESIDENT_SHAPES = [
    (ConvShape(2, 256, 21, 19, 64, 3, 3, 1, 1, 1, 2, "bf16", True, True), None),
    (ConvShape(2, 64, 10, 14, 256, 1, 3, 1, 1, 1, 1, "bf16", True, False), None),
    (ConvShape(1, 128, 11, 35, 64, 3, 3, 1, 2, 2, 2, "bf16", False, True), None),
    (ConvShape(3, 256, 9, 13, 768, 1, 1, 1, 0, 1, 1, "bf16", True, True), None),
    (ConvShape(3, 256, 9, 13, 768, 1, 1, 1, 0, 1, 1, "bf16", True, True), True),
    (ConvShape(2, 128, 7, 9, 96, 1, 1, 1, 0, 1, 1, "bf16", False, False), None),
]


@pytest.mark.parametrize("shape,sm_pairs", RESIDENT_SHAPES,
                         ids=lambda v: ("K%dx%dG%d_%dto%d" % (v.Kh, v.Kw, v.G, v.C_in, v.C_out))
                         if isinstance(v, ConvShape) else str(v))
def test_resident_weights_full(shape, sm_pairs):
    """Every output of plans whose weights stay in shared memory across tiles."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    x, w, b = draw(shape, (71, 72, 73))
    plan, y = run(shape, x, w, b, plan=ConvPlan.for_shape(shape, sm_pairs=sm_pairs))
    assert plan.gemm["resident_weights"] == 1
    check_full(shape, y, oracle_full(shape, x, w, b))


# Swapped operands: two tiles per CTA of 128 output channels, the weights on the MMA's M side and
# both tiles' 256 pixels on N; the epilogue transposes D (channels on TMEM lanes) back to NHWC.
SWAPPED_SHAPES = [
    (ConvShape(4, 128, 29, 23, 128, 3, 3, 2, 1, 1, 1, "bf16", True, True), {}),             # im2col mode
    (ConvShape(3, 256, 9, 13, 128, 1, 1, 1, 0, 1, 1, "bf16", True, False), {}),             # 1x1 mode
    (ConvShape(2, 64, 13, 11, 128, 3, 3, 1, 1, 1, 1, "bf16", False, True), {"per_tap": True}),  # one box per tap
    (ConvShape(2, 256, 19, 17, 256, 3, 3, 2, 1, 1, 2, "bf16", True, True), {}),             # two groups of 128
]


@pytest.mark.parametrize("shape,kw", SWAPPED_SHAPES, ids=["im2col", "1x1", "per_tap", "groups"])
def test_swapped_operands_full(shape, kw):
    """Every output of plans whose weights are the MMA's M operand."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    x, w, b = draw(shape, (81, 82, 83))
    plan, y = run(shape, x, w, b, plan=ConvPlan.for_shape(shape, **kw))
    assert plan.gemm["swapped"] == 1
    check_full(shape, y, oracle_full(shape, x, w, b))


def test_halo_mode_random_sweep():
    """Random stride-1 BF16 shapes in the halo mode (kernel sizes 1-5 per axis, dilation
    1-3, padding, groups, ragged 8 x 16 tiles, widths that leave a lone right-hand tile of
    a two-tile unit): every output against the oracle."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    rng = np.random.default_rng(29)
    done = 0
    while done < 16:
        G = int(rng.choice([1, 1, 2, 4]))
        cin_g = 64 * int(rng.integers(1, 3))
        cout_g = int(rng.choice([32, 64, 96, 128, 256]))
        Kh, Kw = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        D = int(rng.integers(1, 4))
        s = ConvShape(int(rng.integers(1, 3)), cin_g * G, int(rng.integers(3, 30)), int(rng.integers(3, 40)),
                      cout_g * G, Kh, Kw, 1, int(rng.integers(0, 4)), D, G, "bf16",
                      bool(rng.integers(0, 2)), bool(rng.integers(0, 2)))
        if s.H_out < 1 or s.W_out < 1 or Kh * Kw == 1:
            continue
        plan = ConvPlan.for_shape(s)
        if plan.path != "implicit_gemm" or plan.launch["block"] not in (608, 640):  # halo mode
            continue
        x, w, b = draw(s, (900 + done, 910 + done, 920 + done))
        _, y = run(s, x, w, b, plan=plan)
        check_full(s, y, oracle_full(s, x, w, b))
        done += 1


def test_depthwise_separable_block():
    """DW 3x3 (FP32, BF16 out) then PW 1x1 256->512 + bias + ReLU on the full-size block.
    The PW output is checked against the oracle fed the BF16 intermediate, and the
    block end to end against the FP64 oracle of both layers."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    from workloads import WORKLOADS, b_device, w_device, x_device
    sd, x, wd, _ = inputs("dw")
    sp, _, wp, bp = inputs("pw")
    dw_plan = ConvPlan(sd.N, sd.C_in, sd.H, sd.W, sd.C_out, 3, 3, 1, 1, 1, sd.G, "f32", False, False,
                       out_bf16=True)
    pw_plan = ConvPlan.for_shape(sp)
    mid = dw_plan.forward(x_device(x, "f32"), w_device(wd, "f32"))
    y = pw_plan.forward(mid, w_device(wp, "bf16"), b_device(bp))
    torch.cuda.synchronize()
    mid_nchw = mid.float().cpu().permute(0, 3, 1, 2).contiguous().double().numpy()
    pts = sample_points(sp, 4096, 6)
    check_points(sp, y, mid_nchw, wp, bp, pts)
    # end to end: FP64 depthwise, FP64 pointwise
    ref_mid = oracle.conv2d(x, wd, None, 1, 1, 1, sd.G, False)
    check_points(sp, y, ref_mid, wp, bp, pts)
