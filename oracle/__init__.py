"""FP64 CPU oracle for the forward 2D convolution -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it.

The arithmetic lives in ``conv_oracle.c`` (plain seven-loop FP64 nest, OpenMP
over (n, co)); this module compiles it with gcc on first use and marshals
numpy arrays into it through ctypes.  What it computes, with the passages it
follows, is stated at the top of ``conv_oracle.c``:

* dot-product definition and index map: "GPU lesson 9: how a GPU executes
  neural-network convolution" (lincklin.cn), section 2;
* zero padding by address predicate: lesson 9, section 26;
* dilation, effective kernel, output size, groups: "Convolution variants and
  their matrix operations" (lpnh.cn/news/2674933), sections 2.2, 2.3, 4.2,
  4.3, 6.2;
* bias after the sum, then ReLU: lesson 9, section 31 (with its per-channel
  scale and shift, a folded batch norm: y = act(scale * sum + shift));
* transposed convolution, the adjoint of the convolution (variants page,
  sections 2.3 and 4.2: zero insertion between input pixels, then a stride-1
  convolution; in matrix form the weight enters transposed), output extent
  (H - 1)*S - 2P + D*(K - 1) + 1;
* the depthwise-separable block, depthwise 3x3 then pointwise 1x1 (lesson 9,
  section 25), with its intermediate rounded to BF16 (``round_bf16``, the
  pointwise GEMM's operand type).

Every function here is pinned by ``tests/test_oracle.py`` against values the
pages print, closed forms, and two independent restatements.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("N", "C_in", "H", "W", "C_out", "Kh", "Kw", "S", "P", "D", "G", "relu")] + \
               [(n, ctypes.c_int64) for n in
                ("xs_n", "xs_c", "xs_h", "xs_w", "ws_o", "ws_i", "ws_h", "ws_w",
                 "ys_n", "ys_c", "ys_h", "ys_w")]


def build(force: bool = False) -> str:
    """Compile ``conv_oracle.c`` into ``liboracle.so`` beside it (gcc, -O2, OpenMP)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.POINTER
        lib.oracle_out_size.argtypes = [ctypes.c_int] * 5
        lib.oracle_out_size.restype = ctypes.c_int
        lib.oracle_conv2d_f64.argtypes = [P(_Desc), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_conv2d_f64.restype = ctypes.c_int
        lib.oracle_conv2d_points_f64.argtypes = [P(_Desc), ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_conv2d_points_f64.restype = ctypes.c_int
        lib.oracle_conv2d_macs_at.argtypes = [P(_Desc), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_conv2d_macs_at.restype = ctypes.c_long
        lib.oracle_out_size_transposed.argtypes = [ctypes.c_int] * 5
        lib.oracle_out_size_transposed.restype = ctypes.c_int
        lib.oracle_conv_transpose2d_f64.argtypes = lib.oracle_conv2d_f64.argtypes
        lib.oracle_conv_transpose2d_f64.restype = ctypes.c_int
        lib.oracle_conv_transpose2d_points_f64.argtypes = lib.oracle_conv2d_points_f64.argtypes
        lib.oracle_conv_transpose2d_points_f64.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def out_size(size: int, k: int, s: int, p: int, d: int) -> int:
    """Output extent floor((size + 2p - d(k-1) - 1)/s) + 1, or 0 if the window never fits."""
    return int(_load().oracle_out_size(size, k, s, p, d))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


# Logical axis order: x/y (n, c, h, w); w (o, i, h, w).
_ACT_LAYOUTS = {"NCHW": "nchw", "NHWC": "nhwc"}
_W_LAYOUTS = {"OIHW": "oihw", "OHWI": "ohwi"}


def _strides(arr: np.ndarray, layout: str, logical: str):
    """Element strides of ``arr`` (C-contiguous in ``layout`` order) per logical axis."""
    st = [s // arr.itemsize for s in arr.strides]
    return [st[layout.index(a)] for a in logical]


def _logical_shape(arr: np.ndarray, layout: str, logical: str):
    return [arr.shape[layout.index(a)] for a in logical]


def _desc(x, w, x_layout, w_layout, y_layout, stride, padding, dilation, groups, relu, y=None):
    xl, wl = _ACT_LAYOUTS[x_layout], _W_LAYOUTS[w_layout]
    N, C_in, H, W = _logical_shape(x, xl, "nchw")
    C_out, Cin_g, Kh, Kw = _logical_shape(w, wl, "oihw")
    if Cin_g * groups != C_in:
        raise ValueError("weight input-channel extent %d x groups %d != C_in %d" % (Cin_g, groups, C_in))
    d = _Desc()
    d.N, d.C_in, d.H, d.W, d.C_out = N, C_in, H, W, C_out
    d.Kh, d.Kw, d.S, d.P, d.D, d.G = Kh, Kw, stride, padding, dilation, groups
    d.relu = 1 if relu else 0
    d.xs_n, d.xs_c, d.xs_h, d.xs_w = _strides(x, xl, "nchw")
    d.ws_o, d.ws_i, d.ws_h, d.ws_w = _strides(w, wl, "oihw")
    if y is not None:
        d.ys_n, d.ys_c, d.ys_h, d.ys_w = _strides(y, _ACT_LAYOUTS[y_layout], "nchw")
    return d


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def conv2d(x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, relu=False,
           x_layout="NCHW", w_layout="OIHW", y_layout="NCHW", nthreads=0, scale=None):
    """Full FP64 output of the convolution (see module docstring).

    ``scale`` ([C_out] or None) multiplies each channel's sum before the bias
    is added: y = act(scale[co] * sum + bias[co]) (a folded batch norm).

    ``x`` is given in ``x_layout`` ("NCHW" or "NHWC"), ``w`` in ``w_layout``
    ("OIHW" = [C_out][C_in/G][Kh][Kw], or "OHWI" = [C_out][Kh][Kw][C_in/G]),
    ``bias`` is [C_out] or None.  The result is returned in ``y_layout``.
    """
    lib = _load()
    x, w = _f64(x), _f64(w)
    b = None if bias is None else _f64(bias)
    sc = None if scale is None else _f64(scale)
    xl = _ACT_LAYOUTS[x_layout]
    N, C_in, H, W = _logical_shape(x, xl, "nchw")
    C_out, _, Kh, Kw = _logical_shape(w, _W_LAYOUTS[w_layout], "oihw")
    Ho = out_size(H, Kh, stride, padding, dilation)
    Wo = out_size(W, Kw, stride, padding, dilation)
    if Ho <= 0 or Wo <= 0:
        raise ValueError("empty output (H_out=%d, W_out=%d)" % (Ho, Wo))
    shape = {"NCHW": (N, C_out, Ho, Wo), "NHWC": (N, Ho, Wo, C_out)}[y_layout]
    y = np.empty(shape, dtype=np.float64)
    d = _desc(x, w, x_layout, w_layout, y_layout, stride, padding, dilation, groups, relu, y)
    rc = lib.oracle_conv2d_f64(ctypes.byref(d), x.ctypes.data, w.ctypes.data,
                               None if sc is None else sc.ctypes.data,
                               None if b is None else b.ctypes.data, y.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the convolution descriptor")
    return y


def conv2d_points(x, w, bias, pts, stride=1, padding=0, dilation=1, groups=1, relu=False,
                  x_layout="NCHW", w_layout="OIHW", nthreads=0, scale=None):
    """FP64 values at selected outputs; ``pts`` is an int array [npts, 4] of (n, co, ho, wo)."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    b = None if bias is None else _f64(bias)
    sc = None if scale is None else _f64(scale)
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
    out = np.empty(pts.shape[0], dtype=np.float64)
    d = _desc(x, w, x_layout, w_layout, "NCHW", stride, padding, dilation, groups, relu)
    rc = lib.oracle_conv2d_points_f64(ctypes.byref(d), x.ctypes.data, w.ctypes.data,
                                      None if sc is None else sc.ctypes.data,
                                      None if b is None else b.ctypes.data, pts.ctypes.data,
                                      pts.shape[0], out.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the descriptor or a point")
    return out


def macs_at(x, w, n, co, ho, wo, stride=1, padding=0, dilation=1, groups=1,
            x_layout="NCHW", w_layout="OIHW"):
    """Number of multiply terms the oracle takes for output (n, co, ho, wo)."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    d = _desc(x, w, x_layout, w_layout, "NCHW", stride, padding, dilation, groups, False)
    return int(lib.oracle_conv2d_macs_at(ctypes.byref(d), x.ctypes.data, w.ctypes.data,
                                         n, co, ho, wo))


def round_bf16(a):
    """Round to the nearest BF16 value (8 significant bits, ties to even), returned as float64.

    BF16 keeps FP32's exponent range with a 7-bit stored mantissa; below the normal
    range its spacing stays 2**-133.  Written from that definition: scale each value
    by its own ulp, round half-to-even, scale back."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)                        # a = m * 2**e, 0.5 <= |m| < 1
    ulp = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.rint(a / ulp) * ulp                # np.rint rounds halves to even
    big = np.abs(r) > np.ldexp(255.0, 120)    # beyond the largest finite BF16 (0x7f7f)
    return np.where(big, np.copysign(np.inf, a), r)


def dwpw_block(x, w_dw, w_pw, padding=1, dw_scale=None, dw_bias=None, dw_relu=False,
               pw_scale=None, pw_bias=None, pw_relu=False, round_mid=True, nthreads=0):
    """Depthwise-separable block (lesson 9, section 25): depthwise KxK, stride 1, then 1x1.

    x NCHW [N][C][H][W]; w_dw [C][1][K][K] (groups = C); w_pw [C_out][C][1][1].
    Intermediate t = act_dw(dw_scale * dw(x) + dw_bias), rounded to BF16 when
    ``round_mid`` (the pointwise GEMM's operand type), then
    y = act_pw(pw_scale * pw(t) + pw_bias).  Returns y (NCHW, float64)."""
    C = np.asarray(x).shape[1]
    mid = conv2d(x, w_dw, dw_bias, 1, padding, 1, C, dw_relu, nthreads=nthreads, scale=dw_scale)
    if round_mid:
        mid = round_bf16(mid)
    return conv2d(mid, w_pw, pw_bias, 1, 0, 1, 1, pw_relu, nthreads=nthreads, scale=pw_scale)


def out_size_transposed(size: int, k: int, s: int, p: int, d: int) -> int:
    """Transposed-convolution output extent (size - 1)*s - 2p + d(k - 1) + 1, or 0 if not positive."""
    return int(_load().oracle_out_size_transposed(size, k, s, p, d))


def _tdesc(x, w, x_layout, w_layout, y_layout, stride, padding, dilation, groups, relu, y=None):
    """Descriptor of a transposed convolution; w is logical [C_in][C_out/G][Kh][Kw]
    ("IOHW", torch's ConvTranspose2d layout) or "IHWO" = [C_in][Kh][Kw][C_out/G]."""
    xl = _ACT_LAYOUTS[x_layout]
    N, C_in, H, W = _logical_shape(x, xl, "nchw")
    wl = {"IOHW": "iohw", "IHWO": "ihwo"}[w_layout]
    Cin_w, Cout_g, Kh, Kw = _logical_shape(w, wl, "iohw")
    if Cin_w != C_in:
        raise ValueError("weight input-channel extent %d != C_in %d" % (Cin_w, C_in))
    d = _Desc()
    d.N, d.C_in, d.H, d.W, d.C_out = N, C_in, H, W, Cout_g * groups
    d.Kh, d.Kw, d.S, d.P, d.D, d.G = Kh, Kw, stride, padding, dilation, groups
    d.relu = 1 if relu else 0
    d.xs_n, d.xs_c, d.xs_h, d.xs_w = _strides(x, xl, "nchw")
    d.ws_o, d.ws_i, d.ws_h, d.ws_w = _strides(w, wl, "iohw")
    if y is not None:
        d.ys_n, d.ys_c, d.ys_h, d.ys_w = _strides(y, _ACT_LAYOUTS[y_layout], "nchw")
    return d


def conv_transpose2d(x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, relu=False,
                     x_layout="NCHW", w_layout="IOHW", y_layout="NCHW", nthreads=0, scale=None):
    """Full FP64 transposed convolution (scatter order).  x [N][C_in][H][W] (NCHW) or
    NHWC; w [C_in][C_out/G][Kh][Kw] ("IOHW") or [C_in][Kh][Kw][C_out/G] ("IHWO");
    optional per-channel scale, then bias, then ReLU."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    b = None if bias is None else _f64(bias)
    sc = None if scale is None else _f64(scale)
    d0 = _tdesc(x, w, x_layout, w_layout, y_layout, stride, padding, dilation, groups, relu)
    Ho = out_size_transposed(d0.H, d0.Kh, stride, padding, dilation)
    Wo = out_size_transposed(d0.W, d0.Kw, stride, padding, dilation)
    if Ho <= 0 or Wo <= 0:
        raise ValueError("empty output (H_out=%d, W_out=%d)" % (Ho, Wo))
    shape = {"NCHW": (d0.N, d0.C_out, Ho, Wo), "NHWC": (d0.N, Ho, Wo, d0.C_out)}[y_layout]
    y = np.empty(shape, dtype=np.float64)
    d = _tdesc(x, w, x_layout, w_layout, y_layout, stride, padding, dilation, groups, relu, y)
    rc = lib.oracle_conv_transpose2d_f64(ctypes.byref(d), x.ctypes.data, w.ctypes.data,
                                         None if sc is None else sc.ctypes.data,
                                         None if b is None else b.ctypes.data, y.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the transposed-convolution descriptor")
    return y


def conv_transpose2d_points(x, w, bias, pts, stride=1, padding=0, dilation=1, groups=1, relu=False,
                            x_layout="NCHW", w_layout="IOHW", nthreads=0, scale=None):
    """FP64 transposed-convolution values at (n, co, h, w) points, gather order."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    b = None if bias is None else _f64(bias)
    sc = None if scale is None else _f64(scale)
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
    out = np.empty(pts.shape[0], dtype=np.float64)
    d = _tdesc(x, w, x_layout, w_layout, "NCHW", stride, padding, dilation, groups, relu)
    rc = lib.oracle_conv_transpose2d_points_f64(ctypes.byref(d), x.ctypes.data, w.ctypes.data,
                                                None if sc is None else sc.ctypes.data,
                                                None if b is None else b.ctypes.data, pts.ctypes.data,
                                                pts.shape[0], out.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the descriptor or a point")
    return out


# ----------------------------------------------------------------- Winograd F(2x2, 3x3)
# "Convolution vs inner product" (lnrq.cn/news/4475), section 2.2, and "Convolution
# variants and their matrix operations" (lpnh.cn/news/2674933), section 3.3: for a 3x3
# kernel, Winograd's minimal filtering F(2x2, 3x3) maps a 4x4 input tile and the kernel
# into a transformed space where 16 element-wise products give a 2x2 output tile: 4
# multiplies per output instead of 9 (2.25x fewer), at some cost in precision.
#
# The transforms come from the polynomial-interpolation construction with the points
# 0, 1, -1 and infinity (Toom-Cook; the published form of Lavin and Gray, 2015):
#   1-D F(2, 3):  y = A^T [ (G g) * (B^T d) ],  d = 4 inputs, g = 3 taps, y = 2 outputs,
#   y_i = sum_k d_{i+k} g_k (the cross-correlation of the definition).
#   2-D nests it:  Y = A^T [ (G g G^T) * (B^T d B) ] A.
WINO_BT = np.array([[1, 0, -1, 0],
                    [0, 1, 1, 0],
                    [0, -1, 1, 0],
                    [0, 1, 0, -1]], dtype=np.float64)
WINO_G = np.array([[1, 0, 0],
                   [0.5, 0.5, 0.5],
                   [0.5, -0.5, 0.5],
                   [0, 0, 1]], dtype=np.float64)
WINO_AT = np.array([[1, 1, 1, 0],
                    [0, 1, -1, -1]], dtype=np.float64)


def winograd_conv2d(x, w, bias=None, padding=1, relu=False, scale=None, dtype=np.float64):
    """3x3, stride 1, dilation 1, groups 1 convolution by Winograd F(2x2, 3x3), computed in
    ``dtype`` (float64 by default; float32 shows the method's precision cost).

    x NCHW [N][C_in][H][W], w OIHW [C_out][C_in][3][3].  Steps, in the method's order:
    pad and cut the input into 4x4 tiles at stride 2; V = B^T d B per tile and channel;
    U = G g G^T per filter; M = sum over input channels of U * V (16 products per tile and
    channel pair); Y = A^T M A; crop to the output size; scale, bias, ReLU."""
    x = np.asarray(x, dtype=dtype)
    w = np.asarray(w, dtype=dtype)
    N, C, H, W = x.shape
    Co, Ci, Kh, Kw = w.shape
    if (Kh, Kw) != (3, 3) or Ci != C:
        raise ValueError("Winograd F(2x2, 3x3) needs 3x3 kernels over all input channels")
    Ho, Wo = H + 2 * padding - 2, W + 2 * padding - 2
    if Ho < 1 or Wo < 1:
        raise ValueError("empty output")
    th, tw = (Ho + 1) // 2, (Wo + 1) // 2
    # zero-padded input covering every tile (2 outputs per tile need 4 inputs)
    xp = np.zeros((N, C, 2 * th + 2, 2 * tw + 2), dtype=dtype)
    hs, ws = min(H, 2 * th + 2 - padding), min(W, 2 * tw + 2 - padding)
    xp[:, :, padding:padding + hs, padding:padding + ws] = x[:, :, :hs, :ws]
    d = np.lib.stride_tricks.sliding_window_view(xp, (4, 4), axis=(2, 3))[:, :, ::2, ::2]  # N C th tw 4 4
    BT, G, AT = WINO_BT.astype(dtype), WINO_G.astype(dtype), WINO_AT.astype(dtype)
    V = np.einsum("ij,nctwjk,lk->nctwil", BT, d, BT)          # B^T d B
    U = np.einsum("ij,ocjk,lk->ocil", G, w, G)                 # G g G^T
    M = np.einsum("ocil,nctwil->notwil", U, V)                 # 16 products per (tile, c), summed over c
    Y = np.einsum("ij,notwjk,lk->notwil", AT, M, AT)           # A^T M A: 2x2 per tile
    y = Y.transpose(0, 1, 2, 4, 3, 5).reshape(N, Co, 2 * th, 2 * tw)[:, :, :Ho, :Wo]
    y = y.astype(np.float64)
    if scale is not None:
        y = y * np.asarray(scale, dtype=np.float64)[None, :, None, None]
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :, None, None]
    if relu:
        y = np.maximum(y, 0.0)
    return y
