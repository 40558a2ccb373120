"""Thin ctypes binding over libconv.so (include/conv.h).

Argument marshalling only: shapes, dtypes, device pointers and the CUDA
stream are checked and passed through; every step of the convolution runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.  There
is no CPU path: if the library is missing or no GPU is present, calls fail.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libconv.so")

CONV_F32, CONV_BF16 = 0, 1
CONV_FLAG_BIAS, CONV_FLAG_RELU, CONV_FLAG_OUT_BF16, CONV_FLAG_SM_PAIRS, CONV_FLAG_TRANSPOSED = 1, 2, 4, 8, 16
CONV_FLAG_WINOGRAD, CONV_FLAG_ONE_SM, CONV_FLAG_PER_TAP = 32, 64, 128
STATUS = {0: "CONV_OK", 1: "CONV_ERR_INVALID_ARG", 2: "CONV_ERR_UNSUPPORTED", 3: "CONV_ERR_MISALIGNED",
          4: "CONV_ERR_CUDA", 5: "CONV_ERR_NO_MEMORY", 6: "CONV_ERR_TIMEOUT"}
PATHS = {0: "direct", 1: "depthwise", 2: "gemm_1x1", 3: "implicit_gemm", 4: "small_k_gemm", 5: "winograd"}

# Every symbol include/conv.h declares.
EXPORTS = ("conv_plan_create", "conv_plan_output_shape", "conv_plan_info", "conv_forward",
           "conv_plan_destroy", "conv_status_string", "conv_device_status", "conv_plan_num_sms",
           "conv_plan_launch_info", "conv_forward_affine", "conv_block_plan_create",
           "conv_block_plan_output_shape", "conv_block_forward", "conv_block_plan_launch_info",
           "conv_block_plan_destroy", "conv_measure_mma_rate", "conv_check_wait_timeout",
           "conv_plan_gemm_config", "conv_plan_device_status", "conv_block_plan_device_status")
CONV_BLOCK_DW_RELU, CONV_BLOCK_PW_RELU = 1, 2

_lock = threading.Lock()
_lib = None


class ConvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (what, STATUS.get(status, str(status)), _status_text(status)))


def _status_text(status: int) -> str:
    try:
        return lib().conv_status_string(status).decode()
    except Exception:  # pragma: no cover - only while the library itself is broken
        return "?"


def lib():
    """Load libconv.so (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            from . import build as _build
            if not _build.up_to_date():
                _build.build()
            L = ctypes.CDLL(LIB_PATH)
            c_int, c_ll, vp = ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p
            L.conv_plan_create.argtypes = [ctypes.POINTER(vp)] + [c_int] * 11 + [c_int, ctypes.c_uint]
            L.conv_plan_create.restype = c_int
            L.conv_plan_output_shape.argtypes = [vp, ctypes.POINTER(c_int), ctypes.POINTER(c_int)]
            L.conv_plan_output_shape.restype = c_int
            L.conv_plan_info.argtypes = [vp, ctypes.POINTER(c_int), ctypes.POINTER(c_ll),
                                         ctypes.POINTER(c_ll), ctypes.POINTER(c_ll)]
            L.conv_plan_info.restype = c_int
            L.conv_forward.argtypes = [vp, vp, vp, vp, vp, vp]
            L.conv_forward.restype = c_int
            L.conv_forward_affine.argtypes = [vp, vp, vp, vp, vp, vp, vp]
            L.conv_forward_affine.restype = c_int
            L.conv_plan_destroy.argtypes = [vp]
            L.conv_plan_destroy.restype = c_int
            L.conv_status_string.argtypes = [c_int]
            L.conv_status_string.restype = ctypes.c_char_p
            L.conv_device_status.argtypes = [ctypes.POINTER(c_int)]
            L.conv_device_status.restype = c_int
            L.conv_plan_num_sms.argtypes = [vp]
            L.conv_plan_num_sms.restype = c_int
            L.conv_plan_launch_info.argtypes = [vp] + [ctypes.POINTER(c_int)] * 5
            L.conv_plan_launch_info.restype = c_int
            L.conv_plan_gemm_config.argtypes = [vp] + [ctypes.POINTER(c_int)] * 6
            L.conv_plan_gemm_config.restype = c_int
            L.conv_plan_device_status.argtypes = [vp, vp, ctypes.POINTER(c_int)]
            L.conv_plan_device_status.restype = c_int
            L.conv_block_plan_device_status.argtypes = [vp, vp, ctypes.POINTER(c_int)]
            L.conv_block_plan_device_status.restype = c_int
            L.conv_block_plan_create.argtypes = [ctypes.POINTER(vp)] + [c_int] * 7 + [ctypes.c_uint]
            L.conv_block_plan_create.restype = c_int
            L.conv_block_plan_output_shape.argtypes = [vp, ctypes.POINTER(c_int), ctypes.POINTER(c_int)]
            L.conv_block_plan_output_shape.restype = c_int
            L.conv_block_forward.argtypes = [vp] * 10
            L.conv_block_forward.restype = c_int
            L.conv_block_plan_launch_info.argtypes = [vp] + [ctypes.POINTER(c_int)] * 5
            L.conv_block_plan_launch_info.restype = c_int
            L.conv_block_plan_destroy.argtypes = [vp]
            L.conv_block_plan_destroy.restype = c_int
            L.conv_measure_mma_rate.argtypes = [c_int, vp, c_int, vp]
            L.conv_measure_mma_rate.restype = c_int
            L.conv_check_wait_timeout.argtypes = [ctypes.c_ulonglong, vp, vp]
            L.conv_check_wait_timeout.restype = c_int
            _lib = L
        return _lib


def device_status() -> int:
    """Synchronise the device and read/clear the library's timeout word (0 = clean)."""
    code = ctypes.c_int(0)
    st = lib().conv_device_status(ctypes.byref(code))
    if st not in (0, 6):
        raise ConvError(st, "conv_device_status")
    return code.value


def _plan_status(fn, plan, stream, name) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    code = ctypes.c_int(0)
    st = fn(plan, ctypes.c_void_p(stream.cuda_stream), ctypes.byref(code))
    if st not in (0, 6):
        raise ConvError(st, name)
    return code.value


class ConvPlan:
    """A planned convolution: shapes fixed, pointers supplied per call.

    Tensors are NHWC activations [N][H][W][C], weights [C_out][Kh][Kw][C_in/G]
    and an FP32 bias [C_out].  dtype "bf16": BF16 x, w, y.  dtype "f32": FP32
    x, w and FP32 y (BF16 y with out_bf16=True).  transposed=True plans the
    transposed convolution (the adjoint of the convolution with the same S, P,
    D, G; output (H - 1)*S - 2P + D(Kh - 1) + 1 rows), same weight layout.
    winograd=True asks FP32 3x3 stride-1 ungrouped plans to run Winograd F(2x2, 3x3).
    sm_pairs: None lets the plan choose SM pairs or one SM per tile for the tensor-core
    GEMM paths; True / False force one or the other.
    """

    def __init__(self, N, C_in, H, W, C_out, Kh, Kw, S=1, P=0, D=1, G=1, dtype="bf16",
                 bias=True, relu=False, out_bf16=False, sm_pairs=None, transposed=False, winograd=False,
                 per_tap=False):
        L = lib()
        self._plan = None
        flags = (CONV_FLAG_BIAS if bias else 0) | (CONV_FLAG_RELU if relu else 0) | \
                (CONV_FLAG_OUT_BF16 if out_bf16 else 0) | (CONV_FLAG_SM_PAIRS if sm_pairs is True else 0) | \
                (CONV_FLAG_ONE_SM if sm_pairs is False else 0) | \
                (CONV_FLAG_TRANSPOSED if transposed else 0) | (CONV_FLAG_WINOGRAD if winograd else 0) | \
                (CONV_FLAG_PER_TAP if per_tap else 0)
        dt = {"bf16": CONV_BF16, "f32": CONV_F32}[dtype]
        h = ctypes.c_void_p()
        st = L.conv_plan_create(ctypes.byref(h), N, C_in, H, W, C_out, Kh, Kw, S, P, D, G, dt, flags)
        if st != 0:
            raise ConvError(st, "conv_plan_create")
        self._plan = h
        self.shape = (N, C_in, H, W, C_out, Kh, Kw, S, P, D, G)
        self.dtype, self.bias, self.relu, self.out_bf16 = dtype, bias, relu, out_bf16
        self.transposed = transposed
        ho, wo = ctypes.c_int(), ctypes.c_int()
        L.conv_plan_output_shape(h, ctypes.byref(ho), ctypes.byref(wo))
        self.H_out, self.W_out = ho.value, wo.value
        path, m, n, k = ctypes.c_int(), ctypes.c_longlong(), ctypes.c_longlong(), ctypes.c_longlong()
        L.conv_plan_info(h, ctypes.byref(path), ctypes.byref(m), ctypes.byref(n), ctypes.byref(k))
        self.path = PATHS[path.value]
        self.gemm_mnk = (m.value, n.value, k.value)
        self.num_sms = L.conv_plan_num_sms(h)
        li = [ctypes.c_int() for _ in range(5)]
        L.conv_plan_launch_info(h, *[ctypes.byref(v) for v in li])
        self.launch = dict(zip(("grid", "block", "smem_bytes", "stages", "cluster"), [v.value for v in li]))
        gc = [ctypes.c_int(0) for _ in range(6)]
        if L.conv_plan_gemm_config(h, *[ctypes.byref(v) for v in gc]) == 0:
            self.gemm = dict(zip(("mode", "n_tile", "pair", "dual", "resident_weights", "swapped"), [v.value for v in gc]))
        else:
            self.gemm = None  # not a tensor-core GEMM plan

    @classmethod
    def for_shape(cls, s, sm_pairs=None, winograd=False, per_tap=False):
        """Plan from a workloads.ConvShape-like object."""
        return cls(s.N, s.C_in, s.H, s.W, s.C_out, s.Kh, s.Kw, s.S, s.P, s.D, s.G, s.dtype,
                   s.bias, s.relu, s.out_bf16, sm_pairs, getattr(s, "transposed", False), winograd, per_tap)

    def close(self):
        if self._plan is not None and _lib is not None:
            _lib.conv_plan_destroy(self._plan)
        self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ torch side
    def out_dtype(self):
        import torch
        return torch.bfloat16 if (self.dtype == "bf16" or self.out_bf16) else torch.float32

    def empty_output(self, device="cuda"):
        import torch
        N, _, _, _, C_out = self.shape[:5]
        return torch.empty((N, self.H_out, self.W_out, C_out), dtype=self.out_dtype(), device=device)

    def forward(self, x, w, bias=None, y=None, stream=None, scale=None):
        """Launch on ``stream`` (default: torch's current stream); returns y.

        ``scale`` (CUDA float32 [C_out], optional) multiplies each channel's sum
        before the bias: y = act(scale * sum + bias), a folded batch norm."""
        import torch
        N, C_in, H, W, C_out, Kh, Kw, S, P, D, G = self.shape
        dt = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        if not (x.is_cuda and w.is_cuda):
            raise ValueError("x and w must be CUDA tensors")
        if x.dtype != dt or w.dtype != dt:
            raise ValueError("x and w must be %s" % dt)
        if tuple(x.shape) != (N, H, W, C_in) or not x.is_contiguous():
            raise ValueError("x must be a contiguous NHWC tensor of shape %s" % ((N, H, W, C_in),))
        if tuple(w.shape) != (C_out, Kh, Kw, C_in // G) or not w.is_contiguous():
            raise ValueError("w must be a contiguous tensor of shape %s" % ((C_out, Kh, Kw, C_in // G),))
        if self.bias:
            if bias is None or bias.dtype != torch.float32 or tuple(bias.shape) != (C_out,) or \
                    not bias.is_contiguous() or not bias.is_cuda:
                raise ValueError("bias must be a contiguous CUDA float32 tensor of shape (%d,)" % C_out)
        if y is None:
            y = self.empty_output(x.device)
        elif tuple(y.shape) != (N, self.H_out, self.W_out, C_out) or y.dtype != self.out_dtype() or \
                not y.is_contiguous():
            raise ValueError("y has the wrong shape, dtype or layout")
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        bptr = bias.data_ptr() if (self.bias and bias is not None) else None
        if scale is None:
            st = lib().conv_forward(self._plan, x.data_ptr(), w.data_ptr(), bptr, y.data_ptr(), stream.cuda_stream)
            if st != 0:
                raise ConvError(st, "conv_forward")
        else:
            if scale.dtype != torch.float32 or tuple(scale.shape) != (C_out,) or not scale.is_contiguous() or \
                    not scale.is_cuda:
                raise ValueError("scale must be a contiguous CUDA float32 tensor of shape (%d,)" % C_out)
            st = lib().conv_forward_affine(self._plan, x.data_ptr(), w.data_ptr(), scale.data_ptr(), bptr,
                                           y.data_ptr(), stream.cuda_stream)
            if st != 0:
                raise ConvError(st, "conv_forward_affine")
        return y

    __call__ = forward

    def device_status(self, stream=None) -> int:
        """Read and clear the plan's own status word after the work queued on ``stream``
        (default: torch's current stream); waits for that stream only.  0 = clean."""
        return _plan_status(lib().conv_plan_device_status, self._plan, stream, "conv_plan_device_status")


class BlockPlan:
    """Fused depthwise-separable block: depthwise 3x3 (FP32) -> BF16 -> pointwise 1x1
    (BF16 tensor cores), one kernel (include/conv.h, conv_block_forward).

    x NHWC FP32 [N][H][W][C]; w_dw FP32 [C][3][3]; w_pw BF16 [C_out][C]; optional
    FP32 per-channel scale / shift for each stage; y NHWC BF16 [N][H_out][W_out][C_out].
    """

    def __init__(self, N, C, H, W, C_out, K=3, P=1, dw_relu=False, pw_relu=True):
        L = lib()
        self._plan = None
        flags = (CONV_BLOCK_DW_RELU if dw_relu else 0) | (CONV_BLOCK_PW_RELU if pw_relu else 0)
        h = ctypes.c_void_p()
        st = L.conv_block_plan_create(ctypes.byref(h), N, C, H, W, C_out, K, P, flags)
        if st != 0:
            raise ConvError(st, "conv_block_plan_create")
        self._plan = h
        self.shape = (N, C, H, W, C_out, K, P)
        self.dw_relu, self.pw_relu = dw_relu, pw_relu
        ho, wo = ctypes.c_int(), ctypes.c_int()
        L.conv_block_plan_output_shape(h, ctypes.byref(ho), ctypes.byref(wo))
        self.H_out, self.W_out = ho.value, wo.value
        li = [ctypes.c_int() for _ in range(5)]
        L.conv_block_plan_launch_info(h, *[ctypes.byref(v) for v in li])
        self.launch = dict(zip(("grid", "block", "smem_bytes", "halo_stages", "weight_stages"),
                               [v.value for v in li]))

    def close(self):
        if self._plan is not None and _lib is not None:
            _lib.conv_block_plan_destroy(self._plan)
        self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def empty_output(self, device="cuda"):
        import torch
        N, C_out = self.shape[0], self.shape[4]
        return torch.empty((N, self.H_out, self.W_out, C_out), dtype=torch.bfloat16, device=device)

    def forward(self, x, w_dw, w_pw, dw_scale=None, dw_bias=None, pw_scale=None, pw_bias=None, y=None,
                stream=None):
        """Launch on ``stream`` (default: torch's current stream); returns y."""
        import torch
        N, C, H, W, C_out, K, P = self.shape

        def need(t, name, shape, dtype):
            if t is None or not t.is_cuda or t.dtype != dtype or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError("%s must be a contiguous CUDA %s tensor of shape %s" % (name, dtype, shape))

        need(x, "x", (N, H, W, C), torch.float32)
        need(w_dw, "w_dw", (C, K, K), torch.float32)
        need(w_pw, "w_pw", (C_out, C), torch.bfloat16)
        for t, name, n in ((dw_scale, "dw_scale", C), (dw_bias, "dw_bias", C), (pw_scale, "pw_scale", C_out),
                           (pw_bias, "pw_bias", C_out)):
            if t is not None:
                need(t, name, (n,), torch.float32)
        if y is None:
            y = self.empty_output(x.device)
        else:
            need(y, "y", (N, self.H_out, self.W_out, C_out), torch.bfloat16)
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        st = lib().conv_block_forward(self._plan, x.data_ptr(), w_dw.data_ptr(), ptr(dw_scale), ptr(dw_bias),
                                      w_pw.data_ptr(), ptr(pw_scale), ptr(pw_bias), y.data_ptr(),
                                      stream.cuda_stream)
        if st != 0:
            raise ConvError(st, "conv_block_forward")
        return y

    __call__ = forward

    def device_status(self, stream=None) -> int:
        """The block plan's own status word, as ConvPlan.device_status."""
        return _plan_status(lib().conv_block_plan_device_status, self._plan, stream,
                            "conv_block_plan_device_status")


_plan_cache = {}


def measure_mma_rate(iters: int = 1 << 16, device=None):
    """Dense BF16 tcgen05 rate of every SM (conv_measure_mma_rate): returns
    (FLOP per clock per SM, one value per SM, median first) and the SM count."""
    import numpy as np
    import torch
    L = lib()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    st = L.conv_measure_mma_rate(int(iters), ctypes.c_void_p(cycles.data_ptr()), sms,
                                 ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise ConvError(st, "conv_measure_mma_rate")
    torch.cuda.synchronize(dev)
    if device_status() != 0:
        raise ConvError(6, "conv_measure_mma_rate")
    c = cycles.cpu().numpy().astype(np.float64)
    per_sm = 2.0 * 128 * 256 * 16 * iters / c
    return float(np.median(per_sm)), per_sm, sms


def check_wait_timeout(limit_ns: int, device=None):
    """Run conv_check_wait_timeout: one role's bounded wait on a barrier nothing completes
    gives up after ``limit_ns``, a second role leaves through the abort flag.  Returns
    (the status word conv_device_status read and cleared, the second role's wait in ns)."""
    import torch
    L = lib()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    elapsed = torch.zeros(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    st = L.conv_check_wait_timeout(int(limit_ns), ctypes.c_void_p(elapsed.data_ptr()),
                                   ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise ConvError(st, "conv_check_wait_timeout")
    torch.cuda.synchronize(dev)
    code = device_status()
    return code, int(elapsed.item())


def conv2d(x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, relu=False, out_bf16=False,
           y=None, stream=None):
    """Functional form: x NHWC [N][H][W][C_in], w [C_out][Kh][Kw][C_in/G], bias FP32 or None."""
    import torch
    N, H, W, C_in = x.shape
    C_out, Kh, Kw, _ = w.shape
    dtype = "bf16" if x.dtype == torch.bfloat16 else "f32"
    key = (x.device.index, N, C_in, H, W, C_out, Kh, Kw, stride, padding, dilation, groups, dtype,
           bias is not None, relu, out_bf16)
    plan = _plan_cache.get(key)
    if plan is None:
        plan = ConvPlan(N, C_in, H, W, C_out, Kh, Kw, stride, padding, dilation, groups, dtype,
                        bias is not None, relu, out_bf16)
        _plan_cache[key] = plan
    return plan.forward(x, w, bias, y=y, stream=stream)
