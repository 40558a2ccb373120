"""GPU parity of the FP32 Winograd F(2x2, 3x3) path (CONV_FLAG_WINOGRAD) against the FP64
direct-convolution oracle: in exact arithmetic the method computes the convolution itself
("Convolution vs inner product", lnrq.cn, section 2.2), so the convolution's definition is
the reference, at the FP32 tolerance of the library's FP32 paths."""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_TOL, F32_TOL, check_full, run
from workloads import ConvShape, b_device, draw, inputs, w_device, x_device

pytestmark = pytest.mark.gpu

CASES = [
    # N, C_in, H, W, C_out, P, bias, relu, out_bf16
    (1, 3, 32, 32, 8, 1, True, False, False),       # the tiny FP32 layer's shape
    (2, 5, 7, 6, 4, 1, True, True, False),          # channels not multiples of 8 / 32
    (1, 16, 13, 11, 40, 0, False, False, False),    # P = 0, odd sizes: ragged last tiles
    (2, 64, 17, 9, 33, 2, True, True, False),       # P = 2, two output-channel blocks
    (1, 24, 30, 70, 64, 1, True, False, False),     # several tile blocks per image
    (2, 8, 12, 12, 32, 1, True, True, True),        # BF16 output
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N%dC%d_%dx%d_Co%d_P%d%s" % (c[:6] + ("_bf16" if c[8] else "",)))
def test_winograd_matches_oracle(case):
    from cnn_convolution_implicit_gb300 import ConvPlan, device_status
    N, C_in, H, W, C_out, P, bias, relu, out_bf16 = case
    s = ConvShape(N, C_in, H, W, C_out, 3, 3, 1, P, 1, 1, "f32", bias, relu, out_bf16)
    x, w, b = draw(s, (9100 + C_in, 9101 + C_out, 9102))
    plan = ConvPlan.for_shape(s, winograd=True)
    assert plan.path == "winograd"
    _, y = run(s, x, w, b, plan)
    ref = oracle.conv2d(x, w, b if bias else None, 1, P, 1, 1, relu)
    check_full(s, y, ref, BF16_TOL if out_bf16 else F32_TOL)


def test_winograd_affine_epilogue():
    from cnn_convolution_implicit_gb300 import ConvPlan, device_status
    s = ConvShape(2, 32, 15, 14, 48, 3, 3, 1, 1, 1, 1, "f32", True, True)
    x, w, b = draw(s, (9200, 9201, 9202))
    sc = np.random.default_rng(9203).uniform(-2, 2, 48).astype(np.float32)
    plan = ConvPlan.for_shape(s, winograd=True)
    y = plan.forward(x_device(x, "f32"), w_device(w, "f32"), b_device(b), scale=b_device(sc))
    torch.cuda.synchronize()
    assert device_status() == 0
    check_full(s, y, oracle.conv2d(x, w, b, 1, 1, 1, 1, True, scale=sc), F32_TOL)


def test_winograd_full_layer_and_direct_path():
    """The N8 64 -> 64 56x56 FP32 layer: the whole output against the oracle, and the
    Winograd and direct GPU paths within the FP32 tolerance of each other."""
    from cnn_convolution_implicit_gb300 import ConvPlan
    s, x, w, b = inputs("f32_3x3")
    _, yw = run(s, x, w, b, ConvPlan.for_shape(s, winograd=True))
    _, yd = run(s, x, w, b, ConvPlan.for_shape(s))
    ref = oracle.conv2d(x, w, b, 1, 1, 1, 1, True)
    ew = check_full(s, yw, ref, F32_TOL)
    ed = check_full(s, yd, ref, F32_TOL)
    diff = (yw - yd).abs().max().item()
    assert diff <= 1e-4, diff
    print("max scaled error: winograd %.2e, direct %.2e" % (ew, ed))
