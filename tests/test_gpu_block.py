"""GPU parity of the fused depthwise-separable block (conv_block_forward): depthwise
3x3 FP32 -> BF16 -> pointwise 1x1 on tensor cores in one kernel, against the FP64
oracle of the two stages (lesson 9, section 25) with the BF16 intermediate."""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_TOL
from workloads import ConvShape, b_device, draw, inputs, x_device

pytestmark = pytest.mark.gpu


def _block_inputs(N, C, H, W, C_out, P, seed, dw_affine=False, pw_scale=False, pw_bias=True):
    dws = ConvShape(N, C, H, W, C, 3, 3, 1, P, 1, C, "f32", dw_affine, False)
    x, wdw, dwb = draw(dws, (seed, seed + 1, seed + 2))
    Ho, Wo = H + 2 * P - 2, W + 2 * P - 2
    pws = ConvShape(N, C, Ho, Wo, C_out, 1, 1, 1, 0, 1, 1, "bf16", pw_bias, False)
    _, wpw, pwb = draw(pws, (seed + 3, seed + 4, seed + 5))
    rng = np.random.default_rng(seed + 6)
    dwsc = rng.uniform(0.5, 1.5, C).astype(np.float32) if dw_affine else None
    pwsc = rng.uniform(-2.0, 2.0, C_out).astype(np.float32) if pw_scale else None
    return x, wdw, dwsc, dwb, wpw, pwsc, pwb


def _run(plan, x, wdw, dwsc, dwb, wpw, pwsc, pwb):
    from cnn_convolution_implicit_gb300 import device_status
    dev = lambda a: None if a is None else b_device(a)  # noqa: E731
    y = plan.forward(x_device(x, "f32"), torch.from_numpy(np.ascontiguousarray(wdw[:, 0], np.float32)).cuda(),
                     torch.from_numpy(np.ascontiguousarray(wpw[:, :, 0, 0], np.float32)).to(torch.bfloat16).cuda(),
                     dev(dwsc), dev(dwb), dev(pwsc), dev(pwb))
    torch.cuda.synchronize()
    assert device_status() == 0
    return y


def _check(y, ref, tol=BF16_TOL):
    got = y.float().cpu().double().numpy().transpose(0, 3, 1, 2)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    worst = float(err.max())
    assert worst <= tol, "max scaled error %.3e at %s" % (worst, np.unravel_index(int(err.argmax()), err.shape))
    return worst


CASES = [
    # N, C, H, W, C_out, P, dw_relu, pw_relu, dw_affine, pw_scale, pw_bias
    (2, 64, 13, 13, 32, 1, False, True, False, False, True),      # one 32-channel slice, ragged tiles
    (2, 128, 20, 17, 96, 0, True, False, False, False, False),    # P = 0, depthwise ReLU, no pointwise bias
    (1, 192, 9, 30, 384, 2, False, True, False, True, True),      # P = 2, three k-blocks, two 192 slices
    (2, 256, 20, 20, 320, 1, True, True, True, True, True),       # both stages affine (folded batch norms)
    (3, 256, 16, 8, 512, 1, False, True, False, False, True),     # exact 16 x 8 tiles, two 256 slices
    (1, 64, 40, 40, 768, 1, False, False, True, False, True),     # three slices: buffers alternate across tiles
    (2, 128, 33, 9, 352, 1, False, True, False, True, False),     # eleven 32-channel slices
    (8, 64, 64, 64, 64, 1, False, True, False, False, True),      # 256 tiles: CTAs loop, ring phases wrap
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N%d_C%d_%dx%d_Co%d_P%d" % c[:6])
def test_block_matches_oracle(case):
    from cnn_convolution_implicit_gb300 import BlockPlan
    N, C, H, W, C_out, P, dw_relu, pw_relu, dw_aff, pw_sc, pw_b = case
    ins = _block_inputs(N, C, H, W, C_out, P, 7000 + C_out + H, dw_aff, pw_sc, pw_b)
    x, wdw, dwsc, dwb, wpw, pwsc, pwb = ins
    plan = BlockPlan(N, C, H, W, C_out, 3, P, dw_relu=dw_relu, pw_relu=pw_relu)
    y = _run(plan, *ins)
    ref = oracle.dwpw_block(x, wdw, wpw, P, dwsc, dwb, dw_relu, pwsc, pwb, pw_relu, round_mid=True)
    worst = _check(y, ref)
    # the block end to end against the unrounded FP64 chain, at the same tolerance
    ref64 = oracle.dwpw_block(x, wdw, wpw, P, dwsc, dwb, dw_relu, pwsc, pwb, pw_relu, round_mid=False)
    _check(y, ref64)
    # a second call on the same plan (cached descriptors) gives the same bits
    y2 = _run(plan, *ins)
    assert torch.equal(y, y2), worst


def test_block_full_size_and_matches_two_kernel_path():
    """The full-size block (N64, 256 -> 512, 56x56): every output against the oracle (with
    the BF16 intermediate, and end to end in FP64), and bit-identical to the two-launch
    path (depthwise kernel writing BF16, then the 1x1 GEMM kernel), which computes the
    same sums in the same order."""
    from cnn_convolution_implicit_gb300 import BlockPlan, ConvPlan, device_status
    from parity import check_full
    from workloads import w_device
    sd, x, wd, _ = inputs("dw")
    sp, _, wp, bp = inputs("pw")
    plan = BlockPlan(sd.N, sd.C_in, sd.H, sd.W, sp.C_out, 3, 1, dw_relu=False, pw_relu=True)
    xd = x_device(x, "f32")
    wdd = torch.from_numpy(np.ascontiguousarray(wd[:, 0], np.float32)).cuda()
    wpd = w_device(wp, "bf16").reshape(sp.C_out, sp.C_in)
    bd = b_device(bp)
    y = plan.forward(xd, wdd, wpd, pw_bias=bd)
    torch.cuda.synchronize()
    assert device_status() == 0
    # two-kernel reference path on the GPU
    dw_plan = ConvPlan(sd.N, sd.C_in, sd.H, sd.W, sd.C_out, 3, 3, 1, 1, 1, sd.G, "f32", False, False, out_bf16=True)
    mid = dw_plan.forward(xd, w_device(wd, "f32"))
    y2 = ConvPlan.for_shape(sp).forward(mid, w_device(wp, "bf16"), bd)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    # every output against the FP64 oracle: the BF16-rounded intermediate, and end to end
    ref = oracle.dwpw_block(x, wd, wp, 1, pw_bias=bp, pw_relu=True, round_mid=True)
    check_full(sp, y, ref)
    ref64 = oracle.dwpw_block(x, wd, wp, 1, pw_bias=bp, pw_relu=True, round_mid=False)
    check_full(sp, y, ref64)


def test_block_rejects_bad_tensors():
    from cnn_convolution_implicit_gb300 import BlockPlan
    plan = BlockPlan(1, 64, 8, 8, 32, 3, 1)
    x = torch.zeros(1, 8, 8, 64, device="cuda")
    wdw = torch.zeros(64, 3, 3, device="cuda")
    wpw = torch.zeros(32, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        plan.forward(x.double(), wdw, wpw)
    with pytest.raises(ValueError):
        plan.forward(x, wdw, wpw.float())
    with pytest.raises(ValueError):
        plan.forward(x, wdw, wpw, pw_bias=torch.zeros(31, device="cuda"))
    y = plan.forward(x, wdw, wpw)
    torch.cuda.synchronize()
    assert float(y.float().abs().max()) == 0.0
