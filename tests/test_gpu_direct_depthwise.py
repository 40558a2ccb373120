"""GPU parity: direct CUDA-core kernel and FP32 depthwise halo-tile kernel
against the FP64 oracle (elementwise, tolerance in tests/parity.py)."""
import numpy as np
import pytest
import torch

from parity import F32_TOL, check_full, check_points, oracle_full, run, sample_points
from workloads import ConvShape, draw, inputs, random_shape

pytestmark = pytest.mark.gpu


def test_tiny_fp32_layer_full():
    """N=1, 3->8, 32x32, 3x3 s1 p1, FP32 with bias: every output."""
    s, x, w, b = inputs("tiny_f32")
    plan, y = run(s, x, w, b)
    assert plan.path == "direct"
    check_full(s, y, oracle_full(s, x, w, b))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_direct_random_sweep(dtype):
    """Random small shapes over K in {1,2,3,5}, S, P, D, G (all taken by the direct kernel)."""
    rng = np.random.default_rng(11 if dtype == "f32" else 12)
    for i in range(40):
        s = random_shape(rng, dtype)
        x, w, b = draw(s, (100 + i, 200 + i, 300 + i), "uniform", "uniform", "uniform")
        plan, y = run(s, x, w, b)
        check_full(s, y, oracle_full(s, x, w, b))


@pytest.mark.parametrize("shape,tile_m", [
    # register-tiled direct kernel: >= 32 output channels per group
    (ConvShape(2, 16, 13, 11, 32, 3, 3, 1, 1, 1, 1, "f32", True, True), 64),      # half a channel block
    (ConvShape(3, 13, 17, 19, 96, 3, 3, 2, 1, 1, 1, "f32", True, False), 64),     # ragged chunk, scalar loads
    (ConvShape(2, 64, 20, 20, 64, 3, 3, 1, 2, 2, 2, "f32", True, True), 64),      # 2 groups, dilation 2
    (ConvShape(1, 24, 9, 9, 40, 5, 5, 1, 2, 1, 1, "bf16", True, True), 64),       # BF16, C_out % 16 != 0
    (ConvShape(2, 6, 10, 10, 36, 1, 1, 1, 0, 1, 1, "f32", False, False), 64),     # 1x1, 36 channels
    (ConvShape(2, 8, 9, 7, 48, 3, 3, 1, 1, 1, 1, "f32", True, True, out_bf16=True), 64),  # FP32 in, BF16 out
    (ConvShape(4, 8, 100, 100, 32, 3, 3, 1, 1, 1, 1, "f32", True, True), 128),    # 128-pixel tiles
    (ConvShape(2, 12, 130, 121, 70, 3, 3, 1, 1, 1, 1, "f32", True, False), 128),  # 128 pixels, odd channels
])
def test_direct_tiled_kernel(shape, tile_m):
    """Every output of the register-tiled direct kernel: both pixel-tile sizes, ragged
    pixel tails, partial channel blocks and reduction chunks, groups, BF16 in and out."""
    x, w, b = draw(shape, (400, 401, 402), "normal", "kaiming", "uniform")
    plan, y = run(shape, x, w, b)
    assert plan.path == "direct"
    assert plan.launch["block"] == 2 * tile_m, plan.launch
    check_full(shape, y, oracle_full(shape, x, w, b))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_direct_tiled_random_sweep(dtype):
    """Random shapes with >= 32 output channels per group that plan to the direct path
    (so the register-tiled kernel runs): K in {1,2,3,5}, S, P, D, groups, ragged
    channel counts, both pixel-tile sizes' code paths; every output against the oracle."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    rng = np.random.default_rng(21 if dtype == "f32" else 22)
    done = 0
    while done < 12:
        G = int(rng.choice([1, 1, 2]))
        cin_g = int(rng.integers(1, 41))
        if dtype == "bf16" and cin_g % 64 == 0:
            continue
        cout_g = int(rng.choice([32, 40, 48, 64, 72, 96]))
        K = int(rng.choice([1, 2, 3, 5]))
        s = ConvShape(int(rng.integers(1, 3)), G * cin_g, int(rng.integers(3, 21)), int(rng.integers(3, 21)),
                      G * cout_g, K, K, int(rng.choice([1, 2, 3])), int(rng.integers(0, 4)), int(rng.choice([1, 2])),
                      G, dtype, bool(rng.integers(0, 2)), bool(rng.integers(0, 2)))
        if s.H_out < 1 or s.W_out < 1 or ConvPlan.for_shape(s).path != "direct":
            continue
        x, w, b = draw(s, (700 + done, 710 + done, 720 + done), "uniform", "uniform", "uniform")
        plan, y = run(s, x, w, b)
        assert plan.launch["block"] in (128, 256), plan.launch
        check_full(s, y, oracle_full(s, x, w, b))
        done += 1


def test_depthwise_full_size_layer():
    """N=64, C=256, 56x56, depthwise 3x3 s1 p1 FP32: every output (0.46 G MACs in FP64)."""
    s, x, w, b = inputs("dw")
    plan, y = run(s, x, w, b)
    assert plan.path == "depthwise"
    check_full(s, y, oracle_full(s, x, w, b))


@pytest.mark.parametrize("C,H,W,K,S,P,D,bias,relu", [
    (32, 14, 14, 3, 1, 1, 1, False, False),      # one tile exactly
    (64, 17, 23, 3, 1, 1, 1, True, True),        # ragged tiles on both axes
    (32, 16, 16, 5, 1, 2, 1, True, False),       # 5x5, generic-K kernel
    (32, 31, 29, 3, 2, 1, 1, False, True),       # stride 2
    (96, 20, 20, 3, 1, 2, 2, True, True),        # dilation 2: 9 live taps of a 5x5 window
    (32, 9, 40, 3, 1, 0, 1, False, False),       # no padding
    (32, 1, 1, 3, 1, 1, 1, True, False),         # 1x1 image: only the centre tap is live
    (32, 12, 12, 1, 1, 0, 1, True, True),        # 1x1 depthwise = per-channel scale
])
def test_depthwise_shapes(C, H, W, K, S, P, D, bias, relu):
    s = ConvShape(2, C, H, W, C, K, K, S, P, D, C, "f32", bias, relu)
    x, w, b = draw(s, (7, 8, 9), "normal", "kaiming", "uniform")
    plan, y = run(s, x, w, b)
    assert plan.path == "depthwise"
    check_full(s, y, oracle_full(s, x, w, b))


def test_depthwise_bf16_output_block_mode():
    """FP32 depthwise writing BF16 (the intermediate of the depthwise-separable block)."""
    s = ConvShape(3, 64, 21, 19, 64, 3, 3, 1, 1, 1, 64, "f32", True, True, out_bf16=True)
    x, w, b = draw(s, (21, 22, 23))
    plan, y = run(s, x, w, b)
    assert plan.path == "depthwise" and y.dtype == torch.bfloat16
    check_full(s, y, oracle_full(s, x, w, b))


def test_depthwise_full_size_sampled_in_bench_launch_config():
    """The same plan object twice (descriptor cache hit) and sampled points."""
    s, x, w, b = inputs("dw")
    plan, y1 = run(s, x, w, b)
    plan, y2 = run(s, x, w, b, plan=plan)
    assert torch.equal(y1, y2)
    check_points(s, y2, x, w, b, sample_points(s, 4096, 5))
