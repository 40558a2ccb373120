"""Pins for the FP64 oracle (CPU only).

Each test ties the oracle to something other than itself: numbers the pages
print (tests/golden/), closed forms, identities the pages state (1x1 conv is a
GEMM, grouped conv is G independent convs, dilation is a zero-inserted dense
kernel), and two independent restatements on small random shapes (torch's
float64 CPU conv2d and a numpy explicit-im2col GEMM).
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import ConvShape, random_shape

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def conv(x, w, b=None, s=1, p=0, d=1, g=1, relu=False):
    return oracle.conv2d(x, w, b, stride=s, padding=p, dilation=d, groups=g, relu=relu)


# ----------------------------------------------------------------- im2col restatement
def im2col_gemm(x, w, b, s, p, d, g, relu):
    """Explicit im2col + matmul per group (lesson 9 sections 7-8; variants page 3.1),
    written independently of the oracle: pad with zeros, gather each window
    column by slicing, multiply by the flattened kernel."""
    N, C, H, W = x.shape
    Co, Cg, Kh, Kw = w.shape
    Ho = (H + 2 * p - d * (Kh - 1) - 1) // s + 1
    Wo = (W + 2 * p - d * (Kw - 1) - 1) // s + 1
    xp = np.zeros((N, C, H + 2 * p, W + 2 * p))
    xp[:, :, p:p + H, p:p + W] = x
    out = np.zeros((N, Co, Ho, Wo))
    cog = Co // g
    for n in range(N):
        for gi in range(g):
            cols = np.zeros((Cg * Kh * Kw, Ho * Wo))
            r = 0
            for c in range(Cg):
                for kh in range(Kh):
                    for kw in range(Kw):
                        patch = xp[n, gi * Cg + c,
                                   kh * d: kh * d + s * (Ho - 1) + 1: s,
                                   kw * d: kw * d + s * (Wo - 1) + 1: s]
                        cols[r] = patch.reshape(-1)
                        r += 1
            wm = w[gi * cog:(gi + 1) * cog].reshape(cog, -1)
            out[n, gi * cog:(gi + 1) * cog] = (wm @ cols).reshape(cog, Ho, Wo)
    if b is not None:
        out += b[None, :, None, None]
    if relu:
        out = np.maximum(out, 0.0)
    return out


# ----------------------------------------------------------------- 1. lesson 9 worked example
def test_lesson9_im2col_worked_example():
    """3x3 input a..i, 2x2 kernel, stride 1 (lesson 9, section 8).  With a one-hot
    kernel at tap t the oracle's four outputs are column t of the printed X_col."""
    lines = [l.split() for l in open(os.path.join(GOLDEN, "lesson9_im2col_2x2.txt"))
             if l.strip() and not l.startswith("#")]
    letters = lines[0][1:]
    val = {ch: float(i + 1) for i, ch in enumerate(letters)}
    xcol = np.array([[val[ch] for ch in l[2:]] for l in lines[1:]])
    assert xcol.shape == (4, 4)
    assert np.array_equal(xcol, xcol.T)  # the printed matrix is symmetric
    x = np.array([val[ch] for ch in letters]).reshape(1, 1, 3, 3)
    for t in range(4):
        w = np.zeros((1, 1, 2, 2))
        w[0, 0, t // 2, t % 2] = 1.0
        y = conv(x, w)
        assert y.shape == (1, 1, 2, 2)
        assert np.array_equal(y.reshape(-1), xcol[:, t])
    # the full X_col also comes out of the independent restatement
    w = np.arange(1, 5, dtype=float).reshape(1, 1, 2, 2)
    assert np.array_equal(conv(x, w).reshape(-1), xcol @ w.reshape(-1))


# ----------------------------------------------------------------- 2. variants page 4x4 example
def test_variants_4x4_example(facts):
    """1x4x4 input, 3x3 kernel, S1 P0 -> 2x2 output; X_col is 9x4 (variants page 3.1)."""
    rng = np.random.default_rng(1)
    n_in, n_out = facts["small_in"], facts["small_out"]
    x = rng.standard_normal((1, 1, n_in, n_in))
    assert oracle.out_size(n_in, 3, 1, 0, 1) == n_out
    xcol = np.zeros((facts["small_xcol_rows"], facts["small_xcol_cols"]))
    for t in range(9):
        w = np.zeros((1, 1, 3, 3))
        w[0, 0, t // 3, t % 3] = 1.0
        xcol[t] = conv(x, w).reshape(-1)
    # each column is one window, flattened row-major
    for j in range(4):
        ho, wo = divmod(j, 2)
        assert np.array_equal(xcol[:, j], x[0, 0, ho:ho + 3, wo:wo + 3].reshape(-1))


# ----------------------------------------------------------------- 3. MAC counts
@pytest.mark.parametrize("cin,key", [(3, "macs_3x3_cin3"), (64, "macs_3x3_cin64"),
                                     (256, "macs_3x3_cin256")])
def test_mac_counts_interior(cin, key, facts):
    x = np.ones((1, cin, 6, 6))
    w = np.ones((2, cin, 3, 3))
    assert oracle.macs_at(x, w, 0, 1, 2, 3, padding=1) == facts[key]


def test_mac_counts_groups_depthwise_borders():
    x = np.ones((1, 8, 7, 7))
    # grouped: (C_in/G) * K^2 per output
    w = np.ones((4, 2, 3, 3))
    assert oracle.macs_at(x, w, 0, 3, 3, 3, padding=1, groups=4) == 2 * 9
    # depthwise: one channel per output, 9 taps
    w = np.ones((8, 1, 3, 3))
    assert oracle.macs_at(x, w, 0, 5, 3, 3, padding=1, groups=8) == 9
    # zero padding skips taps: corner 4, edge 6
    w = np.ones((1, 8, 3, 3))
    assert oracle.macs_at(x, w, 0, 0, 0, 0, padding=1) == 4 * 8
    assert oracle.macs_at(x, w, 0, 0, 0, 3, padding=1) == 6 * 8
    # dilation: still 9 live taps, never the 25 of the 5x5 window
    assert oracle.macs_at(x, w, 0, 0, 3, 3, padding=2, dilation=2) == 9 * 8


# ----------------------------------------------------------------- 4. shapes
def test_stem_shape(facts):
    n = facts["stem_in"]
    assert oracle.out_size(n, 3, 2, 1, 1) == facts["stem_out"]
    x = np.zeros((1, 3, n, n))
    w = np.zeros((facts["stem_cout"], 3, 3, 3))
    assert conv(x, w, s=2, p=1).shape == (1, facts["stem_cout"], facts["stem_out"], facts["stem_out"])


def test_output_size_sweep_against_torch():
    for H in range(1, 12):
        for K in (1, 2, 3, 5):
            for S in (1, 2, 3):
                for P in range(0, 4):
                    for D in (1, 2, 3):
                        ho = oracle.out_size(H, K, S, P, D)
                        keff = K + (K - 1) * (D - 1)
                        # dilation only widens the window: same size as the dense K_eff kernel
                        assert ho == oracle.out_size(H, keff, S, P, 1)
                        if H + 2 * P < keff:
                            assert ho == 0
                            continue
                        t = F.conv2d(torch.zeros(1, 1, H, H), torch.zeros(1, 1, K, K),
                                     stride=S, padding=P, dilation=D)
                        assert ho == t.shape[-1]


def test_dilated_effective_kernel(facts):
    k, d = facts["dilated_k"], facts["dilated_d"]
    assert k + (k - 1) * (d - 1) == facts["dilated_k_eff"]
    assert oracle.out_size(64, k, 1, 2, d) == 64
    x = np.ones((1, 1, 9, 9))
    w = np.ones((1, 1, k, k))
    assert oracle.macs_at(x, w, 0, 0, 4, 4, padding=2, dilation=d) == facts["dilated_live_taps"]


# ----------------------------------------------------------------- 5. 1x1 == GEMM
def test_1x1_is_gemm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 16, 5, 7))
    w = rng.standard_normal((12, 16, 1, 1))
    y = conv(x, w)
    ref = np.einsum("oc,nchw->nohw", w[:, :, 0, 0], x)
    gemm = (w[:, :, 0, 0] @ x.transpose(1, 0, 2, 3).reshape(16, -1)).reshape(12, 2, 5, 7).transpose(1, 0, 2, 3)
    assert np.allclose(y, gemm, rtol=1e-12, atol=1e-12)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- 6. dilation == zero-inserted dense kernel
def test_dilation_bit_equals_dense_kernel_with_zero_taps():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 3, 11, 10))
    w = rng.standard_normal((4, 3, 3, 3))
    b = rng.standard_normal(4)
    dense = np.zeros((4, 3, 5, 5))
    dense[:, :, ::2, ::2] = w
    y_d = conv(x, w, b, p=2, d=2)
    y_dense = conv(x, dense, b, p=2, d=1)
    assert y_d.shape == y_dense.shape == (2, 4, 11, 10)
    assert np.array_equal(y_d, y_dense)


# ----------------------------------------------------------------- 7. groups == independent convs
@pytest.mark.parametrize("g", [2, 4, 8])
def test_groups_bit_equal_independent_convs(g):
    rng = np.random.default_rng(4 + g)
    cin, cout = 8, 16
    x = rng.standard_normal((2, cin, 7, 6))
    w = rng.standard_normal((cout, cin // g, 3, 3))
    b = rng.standard_normal(cout)
    y = conv(x, w, b, s=2, p=1, g=g)
    cg, og = cin // g, cout // g
    for gi in range(g):
        part = conv(x[:, gi * cg:(gi + 1) * cg], w[gi * og:(gi + 1) * og], b[gi * og:(gi + 1) * og], s=2, p=1)
        assert np.array_equal(y[:, gi * og:(gi + 1) * og], part)


def test_depthwise_is_per_channel():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 6, 8, 8))
    w = rng.standard_normal((6, 1, 3, 3))
    y = conv(x, w, p=1, g=6)
    for c in range(6):
        assert np.array_equal(y[:, c:c + 1], conv(x[:, c:c + 1], w[c:c + 1], p=1))


# ----------------------------------------------------------------- 8. closed forms
def test_all_ones_input_closed_form():
    """All-ones input with fixed weights (variants page 6.4): interior = sum(w) + b,
    border = sum of the in-bounds taps + b."""
    w = np.arange(1, 10, dtype=float).reshape(1, 1, 3, 3)
    b = np.array([0.5])
    y = conv(np.ones((1, 1, 5, 5)), w, b, p=1)[0, 0]
    assert y[2, 2] == w.sum() + 0.5
    assert y[0, 0] == w[0, 0, 1:, 1:].sum() + 0.5
    assert y[0, 2] == w[0, 0, 1:, :].sum() + 0.5
    assert y[4, 4] == w[0, 0, :2, :2].sum() + 0.5


def test_zero_input_gives_relu_of_bias():
    b = np.array([-1.5, 0.0, 2.25])
    w = np.ones((3, 2, 3, 3))
    y = conv(np.zeros((1, 2, 4, 4)), w, b, p=1)
    assert np.all(y == b[None, :, None, None])
    yr = conv(np.zeros((1, 2, 4, 4)), w, b, p=1, relu=True)
    assert np.all(yr == np.maximum(b, 0)[None, :, None, None])


def test_bias_before_relu():
    # acc = -1, bias = +2: bias-then-ReLU gives 1; ReLU-then-bias would also give 1,
    # so use acc = -3, bias = +2: bias-then-ReLU gives 0, ReLU-then-bias gives 2.
    x = np.full((1, 1, 1, 1), -3.0)
    w = np.ones((1, 1, 1, 1))
    assert conv(x, w, np.array([2.0]), relu=True)[0, 0, 0, 0] == 0.0


def test_translation_equivariance_interior():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((1, 2, 12, 12))
    w = rng.standard_normal((3, 2, 3, 3))
    y = conv(x, w)
    xs = np.roll(x, shift=(2, 1), axis=(2, 3))
    ys = conv(xs, w)
    assert np.allclose(ys[:, :, 2:, 1:], y[:, :, :-2, :-1], rtol=0, atol=0)


# ----------------------------------------------------------------- 9. brute force vs two restatements
def test_random_sweep_against_torch_and_im2col():
    rng = np.random.default_rng(7)
    for _ in range(150):
        s = random_shape(rng, "f32")
        x = rng.standard_normal((s.N, s.C_in, s.H, s.W))
        w = rng.standard_normal((s.C_out, s.C_in // s.G, s.Kh, s.Kw))
        b = rng.standard_normal(s.C_out) if s.bias else None
        y = conv(x, w, b, s.S, s.P, s.D, s.G, s.relu)
        t = F.conv2d(torch.from_numpy(x), torch.from_numpy(w),
                     None if b is None else torch.from_numpy(b),
                     stride=s.S, padding=s.P, dilation=s.D, groups=s.G)
        if s.relu:
            t = torch.relu(t)
        r = im2col_gemm(x, w, b, s.S, s.P, s.D, s.G, s.relu)
        assert y.shape == tuple(t.shape) == r.shape, s
        scale = 1.0 + np.abs(y)
        assert np.max(np.abs(y - t.numpy()) / scale) < 1e-12, s
        assert np.max(np.abs(y - r) / scale) < 1e-12, s


# ----------------------------------------------------------------- 10. im2col size arithmetic
def test_body_layer_im2col_arithmetic(facts):
    """112x112x128 -> 256 at 3x3 (variants page 3.3): X_col is (C_in*K*K) x (H_out*W_out)."""
    s = ConvShape(1, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1)
    rows = s.C_in * s.Kh * s.Kw
    cols = oracle.out_size(112, 3, 1, 1, 1) ** 2
    assert rows == facts["body_xcol_rows"] and cols == facts["body_xcol_cols"]
    # the page's "about 1447 x 10^4" is loose: 1152*12544 = 14,450,688
    assert rows * cols / 1e4 == pytest.approx(facts["body_xcol_entries_wan"], rel=5e-3)
    assert round(rows * cols * 4 / 2**20) == facts["body_xcol_mb"]
    assert round(112 * 112 * 128 * 4 / 2**20, 1) == pytest.approx(facts["body_input_mb"], abs=0.3)
    assert rows * cols // (112 * 112 * 128) == facts["body_inflation"]


# ----------------------------------------------------------------- layout / points plumbing
def test_nhwc_and_ohwi_layouts_bit_equal():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 6, 7, 5))
    w = rng.standard_normal((4, 3, 3, 2))
    b = rng.standard_normal(4)
    y = oracle.conv2d(x, w, b, 2, 1, 2, 2, True)
    y2 = oracle.conv2d(x.transpose(0, 2, 3, 1), w.transpose(0, 2, 3, 1), b, 2, 1, 2, 2, True,
                       x_layout="NHWC", w_layout="OHWI", y_layout="NHWC")
    assert np.array_equal(y, y2.transpose(0, 3, 1, 2))


def test_points_bit_equal_full():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 4, 9, 9))
    w = rng.standard_normal((6, 2, 3, 3))
    b = rng.standard_normal(6)
    y = oracle.conv2d(x, w, b, 1, 1, 1, 2, True)
    pts = np.stack([rng.integers(0, 2, 50), rng.integers(0, 6, 50),
                    rng.integers(0, 9, 50), rng.integers(0, 9, 50)], 1)
    v = oracle.conv2d_points(x, w, b, pts, 1, 1, 1, 2, True)
    assert np.array_equal(v, y[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]])
    with pytest.raises(ValueError):
        oracle.conv2d_points(x, w, b, np.array([[0, 6, 0, 0]]), 1, 1, 1, 2, True)


def test_rejects_bad_descriptors():
    with pytest.raises(ValueError):
        oracle.conv2d(np.zeros((1, 3, 4, 4)), np.zeros((2, 2, 3, 3)), groups=1)
    with pytest.raises(ValueError):
        oracle.conv2d(np.zeros((1, 2, 2, 2)), np.zeros((2, 2, 5, 5)))  # empty output


# ----------------------------------------------------------------- folded batch norm (scale + shift)
def test_scale_one_is_bit_identical():
    rng = np.random.default_rng(20)
    x = rng.standard_normal((2, 4, 7, 6))
    w = rng.standard_normal((6, 2, 3, 3))
    b = rng.standard_normal(6)
    y = oracle.conv2d(x, w, b, 1, 1, 1, 2, True)
    assert np.array_equal(y, oracle.conv2d(x, w, b, 1, 1, 1, 2, True, scale=np.ones(6)))


def test_scale_folds_into_weights():
    """scale[co] * (w * x) == (scale[co] * w) * x: folding the scale into the weights."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((2, 6, 9, 8))
    w = rng.standard_normal((9, 2, 3, 3))
    b = rng.standard_normal(9)
    sc = rng.standard_normal(9)
    y = oracle.conv2d(x, w, b, 2, 1, 2, 3, False, scale=sc)
    y2 = oracle.conv2d(x, w * sc[:, None, None, None], b, 2, 1, 2, 3, False)
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-12)


def test_folded_batch_norm_matches_batch_norm():
    """Inference batch norm after the conv (torch's float64 batch_norm) equals the
    conv with scale = gamma / sqrt(var + eps), shift = beta - mean * scale."""
    rng = np.random.default_rng(22)
    x = rng.standard_normal((2, 3, 8, 8))
    w = rng.standard_normal((5, 3, 3, 3))
    mean, var = rng.standard_normal(5), rng.uniform(0.5, 2.0, 5)
    gamma, beta, eps = rng.standard_normal(5), rng.standard_normal(5), 1e-5
    conv = F.conv2d(torch.from_numpy(x), torch.from_numpy(w), padding=1)
    ref = torch.relu(F.batch_norm(conv, torch.from_numpy(mean), torch.from_numpy(var),
                                  torch.from_numpy(gamma), torch.from_numpy(beta), False, 0.0, eps)).numpy()
    sc = gamma / np.sqrt(var + eps)
    y = oracle.conv2d(x, w, beta - mean * sc, 1, 1, 1, 1, True, scale=sc)
    assert np.allclose(y, ref, rtol=1e-11, atol=1e-11)


def test_scale_all_ones_closed_form_and_points():
    w = np.arange(1, 10, dtype=float).reshape(1, 1, 3, 3)
    y = oracle.conv2d(np.ones((1, 1, 5, 5)), w, np.array([0.5]), padding=1, scale=np.array([-2.0]))[0, 0]
    assert y[2, 2] == -2.0 * w.sum() + 0.5
    pts = np.array([[0, 0, 2, 2], [0, 0, 0, 0]])
    v = oracle.conv2d_points(np.ones((1, 1, 5, 5)), w, np.array([0.5]), pts, 1, 1, scale=np.array([-2.0]))
    assert v[0] == y[2, 2] and v[1] == y[0, 0]


# ----------------------------------------------------------------- BF16 rounding and the block
def test_round_bf16_matches_torch_on_float32_values():
    """Nearest-even rounding to BF16 agrees with torch's float32 -> bfloat16 conversion
    on random values, exact ties, signed zeros, subnormals and the largest finite values."""
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    ties = (rng.integers(0, 2**16, 4000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)  # exact halves
    ties = ties[np.isfinite(ties)]
    special = np.array([0.0, -0.0, 1.0, -1.0, 1.00390625, 1.01171875, 1e-40, -3e-39, 3.3e38, -3.38e38,
                        np.float32(2**-126), np.float32(2**-133) * 3], dtype=np.float32)
    for v in (vals, ties, special, rng.standard_normal(100000).astype(np.float32)):
        ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
        got = oracle.round_bf16(v.astype(np.float64))
        assert np.array_equal(got, ref), v[np.argmax(got != ref)]


def test_round_bf16_ties_go_to_even():
    # 1 + 2**-8 lies halfway between 1 and 1 + 2**-7: even mantissa is 1.0
    assert oracle.round_bf16(1 + 2.0**-8) == 1.0
    assert oracle.round_bf16(1 + 3 * 2.0**-8) == 1 + 2 * 2.0**-7
    assert oracle.round_bf16(-(1 + 2.0**-8)) == -1.0


def test_block_identity_depthwise_is_pointwise_of_rounded_input():
    """With a centre-tap depthwise kernel (no scale, shift, ReLU) the block is the 1x1
    conv of bf16(x): a numpy GEMM over channels."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, 64, 5, 6))
    wdw = np.zeros((64, 1, 3, 3))
    wdw[:, 0, 1, 1] = 1.0
    wpw = rng.standard_normal((32, 64, 1, 1))
    b = rng.standard_normal(32)
    y = oracle.dwpw_block(x, wdw, wpw, 1, pw_bias=b)
    xr = oracle.round_bf16(x)
    ref = np.einsum("oc,nchw->nohw", wpw[:, :, 0, 0], xr) + b[None, :, None, None]
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-12)


def test_block_stages_apply_in_order():
    """The depthwise stage's scale, shift and ReLU act before the rounding and the
    pointwise sum: a negative depthwise shift under dw ReLU zeroes the pointwise input."""
    x = np.ones((1, 64, 4, 4))
    wdw = np.ones((64, 1, 3, 3))
    wpw = np.ones((32, 64, 1, 1))
    y = oracle.dwpw_block(x, wdw, wpw, 1, dw_scale=np.full(64, 0.5), dw_bias=np.full(64, -10.0),
                          dw_relu=True, pw_bias=np.full(32, 0.25))
    assert np.all(y == 0.25)
    # without the ReLU: interior depthwise sum 9 * 0.5 - 10 = -5.5, pointwise 64 * -5.5 + 0.25
    y = oracle.dwpw_block(x, wdw, wpw, 1, dw_scale=np.full(64, 0.5), dw_bias=np.full(64, -10.0),
                          pw_bias=np.full(32, 0.25))
    assert y[0, 0, 1, 1] == 64 * -5.5 + 0.25
    # a corner sees 4 taps: 4 * 0.5 - 10 = -8
    assert y[0, 3, 0, 0] == 64 * -8.0 + 0.25


# ----------------------------------------------------------------- transposed convolution
def _adjoint_shapes():
    rng = np.random.default_rng(21)
    out = []
    while len(out) < 40:
        G = int(rng.choice([1, 1, 2]))
        A, B = G * int(rng.integers(1, 4)), G * int(rng.integers(1, 4))
        K, S, D = int(rng.choice([1, 2, 3, 4])), int(rng.choice([1, 2, 3])), int(rng.choice([1, 2]))
        P = int(rng.integers(0, D * (K - 1) + 1))
        Hy, Wy = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        H = (Hy - 1) * S - 2 * P + D * (K - 1) + 1
        W = (Wy - 1) * S - 2 * P + D * (K - 1) + 1
        if H >= 1 and W >= 1:
            out.append((int(rng.integers(1, 3)), A, B, H, W, Hy, Wy, K, S, P, D, G))
    return out


@pytest.mark.parametrize("shape", _adjoint_shapes())
def test_transposed_is_the_adjoint_of_the_convolution(shape):
    """<conv(x), y> == <x, conv_transpose(y)> with the same weight array: the transposed
    convolution is the convolution's matrix transpose (variants page, section 4.2)."""
    N, A, B, H, W, Hy, Wy, K, S, P, D, G = shape
    rng = np.random.default_rng(abs(hash(shape)) % 2**32)
    w = rng.standard_normal((A, B // G, K, K))      # conv: [C_out=A][C_in/G]; transposed: [C_in=A][C_out/G]
    x = rng.standard_normal((N, B, H, W))
    y = rng.standard_normal((N, A, Hy, Wy))
    cx = oracle.conv2d(x, w, None, S, P, D, G)
    assert cx.shape == y.shape
    ty = oracle.conv_transpose2d(y, w, None, S, P, D, G)
    assert ty.shape == x.shape
    lhs, rhs = float(np.sum(cx * y)), float(np.sum(x * ty))
    assert abs(lhs - rhs) <= 1e-11 * (1 + abs(lhs)), (lhs, rhs)


@pytest.mark.parametrize("K,S,P,D,G", [(3, 2, 1, 1, 1), (4, 2, 1, 1, 1), (2, 2, 0, 1, 2), (3, 3, 2, 1, 1),
                                       (3, 2, 0, 2, 1), (5, 1, 2, 1, 1), (1, 2, 0, 1, 1)])
def test_transposed_equals_zero_insertion_then_stride1_conv(K, S, P, D, G):
    """The construction of the variants page, section 4.2: insert S-1 zeros between
    neighbouring input pixels, pad by D(K-1)-P, run a stride-1 convolution with the
    kernel flipped and its in/out channel roles swapped."""
    rng = np.random.default_rng(22 + K + S)
    C_in, C_out, H, W = 2 * G, 3 * G, 4, 5
    x = rng.standard_normal((2, C_in, H, W))
    w = rng.standard_normal((C_in, C_out // G, K, K))
    b = rng.standard_normal(C_out)
    y = oracle.conv_transpose2d(x, w, b, S, P, D, G)
    z = np.zeros((2, C_in, (H - 1) * S + 1, (W - 1) * S + 1))
    z[:, :, ::S, ::S] = x
    cin_g, cout_g = C_in // G, C_out // G
    wf = np.zeros((C_out, cin_g, K, K))
    for g in range(G):
        for co in range(cout_g):
            for ci in range(cin_g):
                wf[g * cout_g + co, ci] = w[g * cin_g + ci, co, ::-1, ::-1]
    ref = oracle.conv2d(z, wf, b, 1, D * (K - 1) - P, D, G)
    assert y.shape == ref.shape
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_transposed_stride_equals_kernel_stamps_blocks():
    """K = S = 2, P = 0: every input pixel stamps a copy of the kernel scaled by its value
    into its own 2x2 output block (no overlap)."""
    x = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    w = np.array([[[[1.0, 10.0], [100.0, 1000.0]]]])
    y = oracle.conv_transpose2d(x, w, None, 2, 0)[0, 0]
    ref = np.block([[1 * w[0, 0], 2 * w[0, 0]], [3 * w[0, 0], 4 * w[0, 0]]])
    assert np.array_equal(y, ref)
    # K = 3, S = 2: neighbouring stamps overlap on one shared row / column and add
    w3 = np.ones((1, 1, 3, 3))
    y3 = oracle.conv_transpose2d(np.ones((1, 1, 2, 2)), w3, None, 2, 0)[0, 0]
    assert y3.shape == (5, 5)
    assert y3[2, 2] == 4.0 and y3[0, 2] == 2.0 and y3[2, 0] == 2.0 and y3[0, 0] == 1.0


def test_transposed_points_match_full_output():
    rng = np.random.default_rng(23)
    x = rng.standard_normal((2, 4, 6, 5))
    w = rng.standard_normal((4, 3, 4, 4))
    b = rng.standard_normal(6)
    full = oracle.conv_transpose2d(x, w, b, 2, 1, 1, 2, True)
    pts = np.stack([rng.integers(0, 2, 300), rng.integers(0, 6, 300), rng.integers(0, full.shape[2], 300),
                    rng.integers(0, full.shape[3], 300)], 1)
    got = oracle.conv_transpose2d_points(x, w, b, pts, 2, 1, 1, 2, True)
    ref = full[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_transposed_matches_torch_and_size_formula():
    rng = np.random.default_rng(24)
    for _ in range(60):
        G = int(rng.choice([1, 2]))
        C_in, C_out = G * int(rng.integers(1, 4)), G * int(rng.integers(1, 4))
        K, S, D = int(rng.choice([1, 2, 3, 4])), int(rng.choice([1, 2, 3])), int(rng.choice([1, 2]))
        P = int(rng.integers(0, 3))
        H, W = int(rng.integers(1, 7)), int(rng.integers(1, 7))
        Ho = (H - 1) * S - 2 * P + D * (K - 1) + 1
        Wo = (W - 1) * S - 2 * P + D * (K - 1) + 1
        assert oracle.out_size_transposed(H, K, S, P, D) == max(Ho, 0)
        if Ho < 1 or Wo < 1:
            continue
        x = rng.standard_normal((2, C_in, H, W))
        w = rng.standard_normal((C_in, C_out // G, K, K))
        b = rng.standard_normal(C_out)
        y = oracle.conv_transpose2d(x, w, b, S, P, D, G)
        t = torch.nn.functional.conv_transpose2d(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b),
                                                 S, P, 0, G, D).numpy()
        assert y.shape == t.shape and np.allclose(y, t, rtol=1e-12, atol=1e-12)
    # the upsampling layer the pages describe: 56 -> 112 with K = 4, S = 2, P = 1
    assert oracle.out_size_transposed(56, 4, 2, 1, 1) == 112


# ----------------------------------------------------------------- Winograd F(2x2, 3x3)
def test_winograd_1d_minimal_filtering_is_exact():
    """F(2, 3): y = A^T[(G g) * (B^T d)] equals the 2-output correlation exactly (integer
    data, binary-exact halves): the transforms are right, not just close."""
    BT, G, AT = oracle.WINO_BT, oracle.WINO_G, oracle.WINO_AT
    d, g = np.array([1.0, 2.0, 3.0, 4.0]), np.array([1.0, 1.0, 1.0])
    assert np.array_equal(AT @ ((G @ g) * (BT @ d)), [6.0, 9.0])
    rng = np.random.default_rng(31)
    for _ in range(200):
        d = rng.integers(-50, 50, 4).astype(np.float64)
        g = rng.integers(-50, 50, 3).astype(np.float64)
        ref = np.array([d[0] * g[0] + d[1] * g[1] + d[2] * g[2], d[1] * g[0] + d[2] * g[1] + d[3] * g[2]])
        assert np.array_equal(AT @ ((G @ g) * (BT @ d)), ref)


@pytest.mark.parametrize("N,C,H,W,Co,P", [(2, 5, 7, 6, 4, 1), (1, 3, 8, 8, 8, 0), (2, 4, 5, 9, 3, 2),
                                          (1, 16, 13, 11, 6, 1), (1, 2, 3, 3, 2, 0), (1, 1, 1, 1, 1, 1)])
def test_winograd_equals_direct_convolution_in_fp64(N, C, H, W, Co, P):
    """In exact arithmetic the method computes the convolution itself: in FP64 it matches the
    direct oracle to rounding, for odd and even sizes (ragged last tiles) and P = 0, 1, 2."""
    rng = np.random.default_rng(32 + H)
    x = rng.standard_normal((N, C, H, W))
    w = rng.standard_normal((Co, C, 3, 3))
    b = rng.standard_normal(Co)
    sc = rng.uniform(0.5, 2.0, Co)
    y = oracle.winograd_conv2d(x, w, b, P, True, scale=sc)
    r = oracle.conv2d(x, w, b, 1, P, 1, 1, True, scale=sc)
    assert y.shape == r.shape
    assert np.max(np.abs(y - r)) <= 1e-12 * (1 + np.max(np.abs(r)))


def _direct_fp32_in_order(x, w):
    """3x3 stride-1 pad-1 convolution summed in FP32 in one fixed order (channel, kernel
    row, kernel column), each product added to the running output: a plain loop's rounding."""
    N, C, H, W = x.shape
    xp = np.pad(x.astype(np.float32), ((0, 0), (0, 0), (1, 1), (1, 1)))
    w32 = w.astype(np.float32)
    y = np.zeros((N, w.shape[0], H, W), np.float32)
    for c in range(C):
        for i in range(3):
            for j in range(3):
                y += xp[:, c:c + 1, i:i + H, j:j + W] * w32[None, :, c, i, j, None, None]
    return y.astype(np.float64)


def test_winograd_multiply_count_and_fp32_tolerance():
    """4 multiplies per output instead of 9 (16 per 2x2 tile): the pages' 2.25x.  On
    Kaiming-scale multi-channel data its FP32 result stays within the FP32 tolerance the
    library's FP32 paths are held to."""
    assert oracle.WINO_BT.shape[0] * oracle.WINO_BT.shape[0] / (oracle.WINO_AT.shape[0] ** 2) == 4.0
    assert 9 / (16 / 4) == 2.25
    rng = np.random.default_rng(33)
    x = rng.standard_normal((2, 64, 16, 16))
    w = rng.standard_normal((32, 64, 3, 3)) * np.sqrt(2.0 / 576)
    ref = oracle.conv2d(x, w, None, 1, 1)
    wino32 = oracle.winograd_conv2d(x.astype(np.float32), w.astype(np.float32), None, 1, dtype=np.float32)
    e_w = np.linalg.norm(wino32 - ref) / np.linalg.norm(ref)
    assert np.max(np.abs(wino32 - ref) / (1 + np.abs(ref))) <= 1e-5 and e_w <= 1e-5


@pytest.mark.parametrize("seed", range(6))
def test_winograd_precision_caveat_single_channel(seed):
    """The pages' precision caveat of Winograd ("Convolution vs inner product", lnrq.cn,
    section 2.2; "Convolution variants and their matrix operations", section 3.3), where it
    shows: with one input channel no channel sum's ordering hides it, and the transforms'
    own rounding (the input transform adds up to four values, the output transform four
    products' sums) leaves F(2x2, 3x3) in FP32 with a larger normwise error than the nine
    products summed in order: measured 1.6-1.8x over seeds; pinned at > 1.3x."""
    rng = np.random.default_rng(100 + seed)
    x = rng.standard_normal((4, 1, 32, 32))
    w = rng.standard_normal((16, 1, 3, 3))
    ref = oracle.conv2d(x, w, None, 1, 1)
    wino32 = oracle.winograd_conv2d(x.astype(np.float32), w.astype(np.float32), None, 1, dtype=np.float32)
    direct32 = _direct_fp32_in_order(x, w)
    e_w = np.linalg.norm(wino32 - ref) / np.linalg.norm(ref)
    e_d = np.linalg.norm(direct32 - ref) / np.linalg.norm(ref)
    assert e_w > 1.3 * e_d, (e_w, e_d)
    assert e_w <= 1e-5
