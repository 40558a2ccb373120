"""GPU parity of the transposed convolution (CONV_FLAG_TRANSPOSED) against the FP64
oracle (variants page, sections 2.3 and 4.2: the adjoint of the convolution)."""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_TOL, F32_TOL
from workloads import ConvShape, b_device, draw, inputs, w_device_transposed, x_device

pytestmark = pytest.mark.gpu

CASES = [
    # N, C_in, H, W, C_out, K, S, P, D, G, dtype, bias, relu, expected path
    (2, 64, 7, 9, 32, 4, 2, 1, 1, 1, "bf16", True, True, "implicit_gemm"),     # 4x4 s2 p1: 4 taps per phase
    (2, 128, 6, 5, 64, 2, 2, 0, 1, 1, "bf16", True, False, "implicit_gemm"),   # K = S: one tap per phase
    (1, 128, 5, 6, 64, 4, 2, 1, 1, 2, "bf16", True, True, "implicit_gemm"),    # two groups (packed per tile with SM pairs)
    (2, 64, 9, 7, 64, 3, 1, 1, 1, 1, "bf16", False, True, "implicit_gemm"),    # stride 1: one phase, 9 taps
    (2, 64, 9, 7, 48, 3, 1, 1, 1, 1, "bf16", False, True, "direct"),           # C_out % 32 != 0
    (1, 64, 6, 6, 32, 3, 3, 0, 1, 1, "bf16", True, False, "implicit_gemm"),    # S = 3
    (1, 64, 5, 7, 32, 3, 1, 2, 2, 1, "bf16", True, True, "implicit_gemm"),     # dilation 2, negative offsets
    (2, 64, 4, 5, 32, 4, 4, 0, 1, 1, "bf16", True, False, "implicit_gemm"),    # S = 4
    (3, 64, 11, 13, 64, 4, 2, 1, 1, 1, "bf16", True, True, "implicit_gemm"),   # several tiles, ragged grids
    (2, 64, 6, 6, 32, 3, 2, 1, 1, 1, "bf16", True, True, "direct"),            # H_out = 11: S does not divide
    (1, 64, 6, 6, 32, 1, 2, 0, 1, 1, "bf16", True, False, "direct"),           # odd phases have no tap
    (2, 96, 5, 5, 32, 4, 2, 1, 1, 1, "bf16", True, True, "direct"),            # C_in % 64 != 0
    (1, 3, 8, 8, 8, 4, 2, 1, 1, 1, "f32", True, False, "direct"),              # FP32
    (2, 8, 5, 6, 12, 3, 2, 0, 2, 4, "f32", True, True, "direct"),              # FP32 groups + dilation
    (2, 16, 7, 7, 40, 4, 2, 1, 1, 1, "f32", True, True, "direct"),             # FP32, register-tiled kernel
    (1, 24, 6, 5, 64, 3, 3, 1, 2, 2, "f32", True, False, "direct"),            # FP32 tiled, 2 groups, S = 3
]


def _run_case(case, seed, scale=False, sm_pairs=None):
    from cnn_convolution_implicit_gb300 import ConvPlan, device_status
    N, C_in, H, W, C_out, K, S, P, D, G, dtype, bias, relu, path = case
    s = ConvShape(N, C_in, H, W, C_out, K, K, S, P, D, G, dtype, bias, relu, transposed=True)
    x, w, b = draw(s, (seed, seed + 1, seed + 2))
    plan = ConvPlan.for_shape(s, sm_pairs=sm_pairs)
    if sm_pairs and path == "implicit_gemm":
        assert plan.launch["cluster"] == 2
    assert plan.path == path, (plan.path, path)
    assert (plan.H_out, plan.W_out) == (s.H_out, s.W_out)
    sc = np.random.default_rng(seed + 3).uniform(-2, 2, C_out).astype(np.float32) if scale else None
    y = plan.forward(x_device(x, dtype), w_device_transposed(w, dtype, G), b_device(b) if bias else None,
                     scale=None if sc is None else b_device(sc))
    torch.cuda.synchronize()
    assert device_status() == 0
    ref = oracle.conv_transpose2d(x, w, b if bias else None, S, P, D, G, relu, scale=sc)
    got = y.float().cpu().double().numpy().transpose(0, 3, 1, 2)
    assert got.shape == ref.shape
    tol = BF16_TOL if dtype == "bf16" else F32_TOL
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert np.all(np.isfinite(got))
    assert float(err.max()) <= tol, "max scaled error %.3e at %s" % (
        float(err.max()), np.unravel_index(int(err.argmax()), err.shape))
    if dtype == "f32":
        assert np.linalg.norm(got - ref) <= F32_TOL * np.linalg.norm(ref)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s_K%dS%dP%dD%dG%d_%dx%d_%s" % (
    c[10], c[5], c[6], c[7], c[8], c[9], c[2], c[3], c[13]))
def test_transposed_matches_oracle(case):
    _run_case(case, 8100 + case[2] * 7 + case[5])


@pytest.mark.parametrize("case", [c for c in CASES if c[13] == "implicit_gemm" and c[9] == 1],
                         ids=lambda c: "pairs_K%dS%dP%dD%d_%dx%d" % (c[5], c[6], c[7], c[8], c[2], c[3]))
def test_transposed_sm_pairs(case):
    """The phase mode on SM pairs (forced): both tiles of a pair are neighbours in one phase,
    an odd tile count leaves one tile paired with an empty one."""
    _run_case(case, 8300 + case[2] * 5 + case[6], sm_pairs=True)


def test_transposed_affine_epilogue():
    """conv_forward_affine on the phase-mode path: per-channel scale before the bias."""
    _run_case((2, 64, 7, 9, 32, 4, 2, 1, 1, 1, "bf16", True, True, "implicit_gemm"), 8200, scale=True)


def test_upsample_full_size():
    """The full-size 56x56 -> 112x112 4x4 s2 p1 layer (N16, 256 -> 128): every output
    against the oracle's transposed convolution."""
    from cnn_convolution_implicit_gb300 import ConvPlan, device_status
    from parity import check_full
    s, x, w, b = inputs("upsample")
    plan = ConvPlan.for_shape(s)
    assert plan.path == "implicit_gemm"
    y = plan.forward(x_device(x, "bf16"), w_device_transposed(w, "bf16", s.G), b_device(b))
    torch.cuda.synchronize()
    assert device_status() == 0
    ref = oracle.conv_transpose2d(x, w, b, s.S, s.P, s.D, s.G, s.relu)
    check_full(s, y, ref)


@pytest.mark.parametrize("case,scale", [
    ((2, 128, 7, 9, 128, 4, 2, 1, 1, 1, "bf16", True, True, "implicit_gemm"), False),
    ((3, 64, 11, 13, 128, 4, 2, 1, 1, 1, "bf16", True, False, "implicit_gemm"), True),
    ((2, 256, 6, 6, 128, 3, 3, 0, 1, 1, "bf16", False, True, "implicit_gemm"), False),
], ids=["K4S2", "K4S2_affine_ragged", "K3S3"])
def test_transposed_swapped_operands(case, scale):
    """Two phase tiles of 128 output channels per CTA with the weights as the MMA's M operand
    and both tiles' pixels as N (D transposed in TMEM, transposed again by the epilogue)."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    N, C_in, H, W, C_out, K, S, P, D, G, dtype, bias, relu, path = case
    s = ConvShape(N, C_in, H, W, C_out, K, K, S, P, D, G, dtype, bias, relu, transposed=True)
    assert ConvPlan.for_shape(s).gemm["swapped"] == 1
    _run_case(case, 8400 + H, scale=scale)
