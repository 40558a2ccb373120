"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare against the FP64 oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
from cnn_convolution_implicit_gb300 import ConvPlan, device_status
from workloads import b_device, w_device, x_device

# Tolerances (elementwise, against the FP64 oracle):
#   BF16 tensor paths: |y - y_ref| <= 2e-2 * (1 + |y_ref|)
#   FP32 paths:        |y - y_ref| <= 1e-5 * (1 + |y_ref|), and the normwise
#                      relative error ||y - y_ref|| / ||y_ref|| <= 1e-5.
BF16_TOL = 2e-2
F32_TOL = 1e-5


def tolerance(shape):
    return BF16_TOL if (shape.dtype == "bf16" or shape.out_bf16) else F32_TOL


def run(shape, x, w, b, plan=None):
    """Run the CUDA path on NCHW/OIHW host arrays; returns (plan, y NHWC device tensor)."""
    plan = plan or ConvPlan.for_shape(shape)
    xd = x_device(x, shape.dtype)
    wd = w_device(w, shape.dtype)
    bd = b_device(b) if shape.bias else None
    y = plan.forward(xd, wd, bd)
    torch.cuda.synchronize()
    assert device_status() == 0
    return plan, y


def oracle_full(shape, x, w, b):
    return oracle.conv2d(x, w, b if shape.bias else None, shape.S, shape.P, shape.D, shape.G, shape.relu)


def check_full(shape, y_nhwc, ref_nchw, tol=None):
    """Elementwise check of a whole output; returns the max scaled error."""
    tol = tol if tol is not None else tolerance(shape)
    y = y_nhwc.float().cpu().double().numpy().transpose(0, 3, 1, 2)
    assert y.shape == ref_nchw.shape
    err = np.abs(y - ref_nchw) / (1.0 + np.abs(ref_nchw))
    worst = float(err.max()) if err.size else 0.0
    assert np.all(np.isfinite(y))
    assert worst <= tol, "max scaled error %.3e > %.1e at %s" % (
        worst, tol, np.unravel_index(int(err.argmax()), err.shape))
    if tol == F32_TOL:
        den = np.linalg.norm(ref_nchw)
        if den > 0:
            assert np.linalg.norm(y - ref_nchw) / den <= F32_TOL
    return worst


def sample_points(shape, count, seed):
    """Seeded output points (n, co, ho, wo) plus every corner and the last pixel."""
    rng = np.random.default_rng(seed)
    Ho, Wo = shape.H_out, shape.W_out
    pts = np.stack([rng.integers(0, shape.N, count), rng.integers(0, shape.C_out, count),
                    rng.integers(0, Ho, count), rng.integers(0, Wo, count)], 1)
    extra = []
    for n in (0, shape.N - 1):
        for ho in (0, Ho - 1):
            for wo in (0, Wo - 1):
                for co in (0, shape.C_out - 1):
                    extra.append((n, co, ho, wo))
    return np.concatenate([pts, np.array(extra)], 0).astype(np.int64)


def check_points(shape, y_nhwc, x, w, b, pts, tol=None):
    tol = tol if tol is not None else tolerance(shape)
    ref = oracle.conv2d_points(x, w, b if shape.bias else None, pts, shape.S, shape.P, shape.D,
                               shape.G, shape.relu)
    idx = torch.from_numpy(pts).to(y_nhwc.device)
    got = y_nhwc[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]].double().cpu().numpy()
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    worst = float(err.max())
    assert np.all(np.isfinite(got))
    assert worst <= tol, "max scaled error %.3e > %.1e at point %s" % (worst, tol, pts[int(err.argmax())])
    return worst
