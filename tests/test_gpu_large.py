"""GPU parity at sizes past 2**31 elements: every kernel path on a tensor whose element
offsets do not fit in 32 bits (the input for the 1x1 GEMM, depthwise, Winograd and fused
block paths, the output for the implicit-GEMM, transposed, small-K and register-tiled
direct paths).  Inputs are drawn on the
device from a seeded generator; sampled outputs in the first, a middle and the last image
(whose addresses lie past 2**31 elements) are checked against the FP64 oracle, which reads
only those images."""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_TOL, F32_TOL
from workloads import ConvShape, b_device, w_device

pytestmark = pytest.mark.gpu

BIG = 2 ** 31


def _x_device(s: ConvShape, seed: int) -> torch.Tensor:
    """NHWC input ~ N(0, 1) drawn on the device (rounded once to BF16 for BF16 shapes)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((s.N, s.H, s.W, s.C_in), generator=g, device="cuda", dtype=torch.float32)
    return x.to(torch.bfloat16) if s.dtype == "bf16" else x


def _weights(s: ConvShape, seed: int):
    rng = np.random.default_rng(seed)
    cin_g = s.C_in // s.G
    w = rng.normal(0.0, np.sqrt(2.0 / (cin_g * s.Kh * s.Kw)), (s.C_out, cin_g, s.Kh, s.Kw)).astype(np.float32)
    b = rng.normal(0.0, 0.01, s.C_out).astype(np.float32)
    if s.dtype == "bf16":  # the oracle reads the values the GPU receives
        w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    return w, b


def _check_sampled(s: ConvShape, x, w, b, y, count=192, seed=0):
    """Outputs at seeded points of images 0, N//2 and N-1 (plus the last image's corners)
    against the oracle run on just those three images."""
    imgs = [0, s.N // 2, s.N - 1]
    rng = np.random.default_rng(seed)
    pts = np.stack([rng.integers(0, 3, count), rng.integers(0, s.C_out, count),
                    rng.integers(0, s.H_out, count), rng.integers(0, s.W_out, count)], 1)
    corners = [(2, co, ho, wo) for co in (0, s.C_out - 1) for ho in (0, s.H_out - 1) for wo in (0, s.W_out - 1)]
    pts = np.concatenate([pts, np.array(corners)], 0).astype(np.int64)
    x_sub = x[imgs].float().cpu().numpy().astype(np.float64)  # NHWC, three images
    ref = oracle.conv2d_points(x_sub, w, b, pts, s.S, s.P, s.D, s.G, s.relu, x_layout="NHWC")
    n_idx = torch.tensor(imgs, device=y.device)[torch.from_numpy(pts[:, 0]).to(y.device)]
    idx = torch.from_numpy(pts).to(y.device)
    got = y[n_idx, idx[:, 2], idx[:, 3], idx[:, 1]].double().cpu().numpy()
    tol = BF16_TOL if (s.dtype == "bf16" or s.out_bf16) else F32_TOL
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert np.all(np.isfinite(got))
    assert float(err.max()) <= tol, "max scaled error %.3e at point %s" % (float(err.max()), pts[int(err.argmax())])


@pytest.mark.parametrize("shape,path,big", [
    # 1x1 GEMM: input 2049 x 64 x 64 x 256 = 2.148e9 elements
    (ConvShape(2049, 256, 64, 64, 128, 1, 1, 1, 0, 1, 1, "bf16", True, True), "gemm_1x1", "x"),
    # depthwise: input (and output) 130 x 128 x 128 x 1024 = 2.18e9 elements
    (ConvShape(130, 1024, 128, 128, 1024, 3, 3, 1, 1, 1, 1024, "f32", True, False), "depthwise", "x"),
    # implicit GEMM (SM pairs): output 670 x 112 x 112 x 256 = 2.15e9 elements
    (ConvShape(670, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1, "bf16", True, True), "implicit_gemm", "y"),
    # small-K stem: output 5400 x 112 x 112 x 32 = 2.17e9 elements
    (ConvShape(5400, 3, 224, 224, 32, 3, 3, 2, 1, 1, 1, "bf16", True, True), "small_k_gemm", "y"),
    # register-tiled direct FP32: output 34 x 1000 x 1000 x 64 = 2.18e9 elements
    (ConvShape(34, 4, 1000, 1000, 64, 1, 1, 1, 0, 1, 1, "f32", True, False), "direct", "y"),
], ids=["gemm_1x1", "depthwise", "implicit_gemm", "small_k", "direct"])
def test_past_2_31_elements(shape, path, big):
    from cnn_convolution_implicit_gb300 import ConvPlan, device_status
    s = shape
    n_big = s.N * (s.H * s.W * s.C_in if big == "x" else s.H_out * s.W_out * s.C_out)
    assert n_big > BIG
    plan = ConvPlan.for_shape(s)
    assert plan.path == path
    x = _x_device(s, 4242)
    w, b = _weights(s, 4243)
    y = plan.forward(x, w_device(w, s.dtype), b_device(b))
    torch.cuda.synchronize()
    assert device_status() == 0
    _check_sampled(s, x, w, b, y)
    del x, y
    torch.cuda.empty_cache()


def _points(s: ConvShape, count=192, seed=0):
    rng = np.random.default_rng(seed)
    pts = np.stack([rng.integers(0, 3, count), rng.integers(0, s.C_out, count),
                    rng.integers(0, s.H_out, count), rng.integers(0, s.W_out, count)], 1)
    corners = [(2, co, ho, wo) for co in (0, s.C_out - 1) for ho in (0, s.H_out - 1) for wo in (0, s.W_out - 1)]
    return np.concatenate([pts, np.array(corners)], 0).astype(np.int64)


def _gather(y, imgs, pts):
    n_idx = torch.tensor(imgs, device=y.device)[torch.from_numpy(pts[:, 0]).to(y.device)]
    idx = torch.from_numpy(pts).to(y.device)
    return y[n_idx, idx[:, 2], idx[:, 3], idx[:, 1]].double().cpu().numpy()


def _assert_close(got, ref, tol, pts):
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert np.all(np.isfinite(got))
    assert float(err.max()) <= tol, "max scaled error %.3e at point %s" % (float(err.max()), pts[int(err.argmax())])


def test_winograd_past_2_31_elements():
    """Winograd F(2x2, 3x3) on an FP32 input of 130 x 128 x 128 x 1024 = 2.18e9 elements."""
    from cnn_convolution_implicit_gb300 import ConvPlan, device_status
    s = ConvShape(130, 1024, 128, 128, 64, 3, 3, 1, 1, 1, 1, "f32", True, True)
    assert s.N * s.H * s.W * s.C_in > BIG
    plan = ConvPlan.for_shape(s, winograd=True)
    assert plan.path == "winograd"
    x = _x_device(s, 5151)
    w, b = _weights(s, 5152)
    y = plan.forward(x, w_device(w, "f32"), b_device(b))
    torch.cuda.synchronize()
    assert device_status() == 0
    _check_sampled(s, x, w, b, y)
    del x, y
    torch.cuda.empty_cache()


def test_transposed_past_2_31_elements():
    """Transposed 4x4 s2 p1 (phase mode) with an output of 172 x 224 x 224 x 256 = 2.2e9 elements."""
    from cnn_convolution_implicit_gb300 import ConvPlan, device_status
    from workloads import w_device_transposed
    s = ConvShape(172, 256, 112, 112, 256, 4, 4, 2, 1, 1, 1, "bf16", True, True, transposed=True)
    assert s.N * s.H_out * s.W_out * s.C_out > BIG
    plan = ConvPlan.for_shape(s)
    assert plan.path == "implicit_gemm"
    x = _x_device(s, 6161)
    rng = np.random.default_rng(6162)
    w = rng.normal(0.0, np.sqrt(2.0 / (s.C_in * 4)), (s.C_in, s.C_out, 4, 4)).astype(np.float32)  # IOHW
    w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    b = rng.normal(0.0, 0.01, s.C_out).astype(np.float32)
    y = plan.forward(x, w_device_transposed(w, "bf16", 1), b_device(b))
    torch.cuda.synchronize()
    assert device_status() == 0
    imgs = [0, s.N // 2, s.N - 1]
    pts = _points(s)
    x_sub = x[imgs].float().cpu().numpy().astype(np.float64)
    ref = oracle.conv_transpose2d_points(x_sub, w, b, pts, s.S, s.P, s.D, s.G, s.relu, x_layout="NHWC")
    _assert_close(_gather(y, imgs, pts), ref, BF16_TOL, pts)
    del x, y
    torch.cuda.empty_cache()


def test_block_past_2_31_elements():
    """The fused depthwise-separable block on an FP32 input of 520 x 128 x 128 x 256 = 2.18e9
    elements (output 4.4e9): sampled outputs against the oracle's two stages on three images,
    the intermediate rounded to BF16 as the kernel holds it."""
    from cnn_convolution_implicit_gb300 import BlockPlan, device_status
    N, C, H, W, C_out = 520, 256, 128, 128, 512
    assert N * H * W * C > BIG
    g = torch.Generator(device="cuda").manual_seed(7171)
    x = torch.randn((N, H, W, C), generator=g, device="cuda", dtype=torch.float32)
    rng = np.random.default_rng(7172)
    w_dw = rng.normal(0.0, np.sqrt(2.0 / 9), (C, 1, 3, 3)).astype(np.float32)
    w_pw = rng.normal(0.0, np.sqrt(2.0 / C), (C_out, C, 1, 1)).astype(np.float32)
    w_pw = torch.from_numpy(w_pw).to(torch.bfloat16).float().numpy()
    b_pw = rng.normal(0.0, 0.01, C_out).astype(np.float32)
    plan = BlockPlan(N, C, H, W, C_out, 3, 1, dw_relu=False, pw_relu=True)
    y = plan.forward(x, torch.from_numpy(np.ascontiguousarray(w_dw[:, 0])).cuda(),
                     torch.from_numpy(w_pw[:, :, 0, 0]).to(torch.bfloat16).cuda(), pw_bias=b_device(b_pw))
    torch.cuda.synchronize()
    assert device_status() == 0
    imgs = [0, N // 2, N - 1]
    x_sub = x[imgs].permute(0, 3, 1, 2).contiguous().cpu().numpy().astype(np.float64)
    mid = oracle.round_bf16(oracle.conv2d(x_sub, w_dw, None, 1, 1, 1, C, False))
    s = ConvShape(3, C, H, W, C_out, 1, 1, 1, 0, 1, 1, "bf16", True, True)
    pts = _points(s)
    ref = oracle.conv2d_points(mid, w_pw, b_pw, pts, 1, 0, 1, 1, True)
    _assert_close(_gather(y, imgs, pts), ref, BF16_TOL, pts)
    del x, y
    torch.cuda.empty_cache()
