"""Seeded input generators: reproducible, BF16 values exact, shapes as stated."""
import numpy as np
import torch

import oracle
from workloads import WORKLOADS, ConvShape, draw, inputs, round_bf16


def test_shapes_and_output_sizes_match_oracle():
    for name, wl in WORKLOADS.items():
        s = wl.shape
        size = oracle.out_size_transposed if s.transposed else oracle.out_size
        assert s.H_out == size(s.H, s.Kh, s.S, s.P, s.D), name
        assert s.W_out == size(s.W, s.Kw, s.S, s.P, s.D), name
    assert WORKLOADS["upsample"].shape.H_out == 112
    assert WORKLOADS["stem"].shape.H_out == 112
    assert WORKLOADS["dilated"].shape.H_out == 64
    assert WORKLOADS["body"].shape.flops == 2 * 32 * 112 * 112 * 256 * 1152


def test_draws_are_reproducible_and_bf16_exact():
    s = ConvShape(2, 16, 9, 9, 32, 3, 3, 1, 1, 1, 1, "bf16", True, True)
    a = draw(s, (11, 12, 13))
    b = draw(s, (11, 12, 13))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    x, w, _ = a
    assert np.array_equal(round_bf16(x), x) and np.array_equal(round_bf16(w), w)
    t = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(t, x)


def test_distributions():
    s = ConvShape(4, 64, 32, 32, 128, 3, 3, 1, 1, 1, 1, "f32", True, False)
    x, w, b = draw(s, (1, 2, 3))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs(w.std() - np.sqrt(2.0 / (64 * 9))) < 0.002
    assert abs(b.std() - 0.01) < 0.003


def test_tiny_workload_is_uniform():
    s, x, w, b = inputs("tiny_f32")
    assert x.min() >= -1 and x.max() <= 1 and w.min() >= -1 and b.max() <= 1
    assert x.shape == (1, 3, 32, 32) and w.shape == (8, 3, 3, 3)


def test_transposed_flop_count_matches_oracle_tap_counts():
    """The transposed workload's FLOPs count each (output pixel, tap) pair whose input
    pixel exists: checked against the oracle's own per-point multiply count on a small case."""
    s = ConvShape(1, 1, 5, 4, 1, 4, 4, 2, 1, 1, 1, "f32", False, False, transposed=True)
    x = np.ones((1, 1, 5, 4))
    w = np.ones((1, 1, 4, 4))
    y = oracle.conv_transpose2d(x, w, None, 2, 1)  # all-ones: each output counts its live taps
    assert s.flops == 2 * int(round(y.sum()))


def test_transposed_weight_marshalling():
    """[C_in][C_out/G][Kh][Kw] -> [C_out][Kh][Kw][C_in/G]: a permutation per group."""
    from workloads import w_device_transposed
    rng = np.random.default_rng(3)
    G, cin_g, cout_g = 2, 3, 4
    w = rng.standard_normal((G * cin_g, cout_g, 2, 3)).astype(np.float32)
    d = w_device_transposed(w, "f32", G, device="cpu").numpy()
    for g in range(G):
        for co in range(cout_g):
            for ci in range(cin_g):
                assert np.array_equal(d[g * cout_g + co, :, :, ci], w[g * cin_g + ci, co])
