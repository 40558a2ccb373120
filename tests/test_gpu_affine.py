"""GPU parity of the folded-batch-norm epilogue (conv_forward_affine):
y = act(scale[co] * sum + bias[co]) on every kernel path, against the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from cnn_convolution_implicit_gb300 import ConvPlan, device_status
from parity import check_full, check_points, sample_points
from workloads import ConvShape, b_device, draw, inputs, w_device, x_device

pytestmark = pytest.mark.gpu


def run_affine(s, x, w, b, sc, plan=None):
    plan = plan or ConvPlan.for_shape(s)
    y = plan.forward(x_device(x, s.dtype), w_device(w, s.dtype), b_device(b) if s.bias else None,
                     scale=torch.from_numpy(sc.astype(np.float32)).cuda())
    torch.cuda.synchronize()
    assert device_status() == 0
    return plan, y


@pytest.mark.parametrize("shape,path", [
    (ConvShape(2, 5, 9, 11, 6, 3, 3, 1, 1, 1, 1, "f32", True, True), "direct"),
    (ConvShape(2, 8, 9, 7, 8, 3, 3, 2, 1, 2, 2, "bf16", True, False), "direct"),
    (ConvShape(2, 8, 9, 7, 48, 3, 3, 1, 1, 1, 1, "f32", True, True), "direct"),   # register-tiled kernel
    (ConvShape(2, 64, 17, 19, 64, 3, 3, 1, 1, 1, 64, "f32", True, True), "depthwise"),
    (ConvShape(2, 64, 17, 19, 64, 3, 3, 1, 1, 1, 64, "f32", False, False), "depthwise"),
    (ConvShape(2, 128, 13, 11, 256, 3, 3, 1, 1, 1, 1, "bf16", True, True), "implicit_gemm"),
    (ConvShape(2, 64, 13, 11, 64, 3, 3, 2, 1, 1, 1, "bf16", True, True), "implicit_gemm"),
    (ConvShape(1, 256, 8, 8, 256, 3, 3, 1, 2, 2, 4, "bf16", True, True), "implicit_gemm"),
    (ConvShape(2, 256, 7, 9, 512, 1, 1, 1, 0, 1, 1, "bf16", True, True), "gemm_1x1"),
    (ConvShape(2, 3, 40, 40, 32, 3, 3, 2, 1, 1, 1, "bf16", True, True), "small_k_gemm"),
])
def test_affine_epilogue_every_path(shape, path):
    x, w, b = draw(shape, (51, 52, 53))
    sc = np.random.default_rng(54).uniform(-2.0, 2.0, shape.C_out)
    plan, y = run_affine(shape, x, w, b, sc)
    assert plan.path == path
    ref = oracle.conv2d(x, w, b if shape.bias else None, shape.S, shape.P, shape.D, shape.G, shape.relu,
                        scale=sc.astype(np.float32).astype(np.float64))
    check_full(shape, y, ref)


def test_affine_body_layer_points():
    """The body layer with a folded batch norm (gamma/sqrt(var+eps) scale, beta - mean*scale shift)."""
    s, x, w, b = inputs("body")
    rng = np.random.default_rng(55)
    gamma, var, mean = rng.uniform(0.5, 1.5, 256), rng.uniform(0.5, 2.0, 256), rng.standard_normal(256) * 0.1
    sc = (gamma / np.sqrt(var + 1e-5)).astype(np.float32)
    shift = (b - mean * sc).astype(np.float32)
    plan, y = run_affine(s, x, w, shift, sc)
    ref = oracle.conv2d_points(x, w, shift.astype(np.float64), sample_points(s, 4096, 56), 1, 1, 1, 1, True,
                               scale=sc.astype(np.float64))
    pts = sample_points(s, 4096, 56)
    idx = torch.from_numpy(pts).to(y.device)
    got = y[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]].double().cpu().numpy()
    assert np.max(np.abs(got - ref) / (1 + np.abs(ref))) <= 2e-2
