"""Seeded input generators: reproducible, BF16 values exact, shapes as stated."""
import numpy as np
import torch

import oracle
from workloads import WORKLOADS, ConvShape, draw, inputs, round_bf16


def test_shapes_and_output_sizes_match_oracle():
    for name, wl in WORKLOADS.items():
        s = wl.shape
        assert s.H_out == oracle.out_size(s.H, s.Kh, s.S, s.P, s.D), name
        assert s.W_out == oracle.out_size(s.W, s.Kw, s.S, s.P, s.D), name
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
