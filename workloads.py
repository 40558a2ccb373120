"""Seeded synthetic inputs for the convolution workloads.

Shared by the CUDA path's tests/benchmark and by the oracle checks.  It holds
no convolution arithmetic: only shapes, seeded draws, the one-time BF16
rounding of the drawn inputs, and layout marshalling (NCHW <-> NHWC).

Shapes are the layer shapes the source pages discuss:

* ``tiny_f32``   -- N=1, 3 -> 8 channels, 32x32, 3x3 s1 p1, FP32, bias; X, W, b ~ U[-1, 1].
* ``stem``       -- N=32, 3 -> 32, 224x224 -> 112x112, 3x3 s2 p1, BF16, bias+ReLU
  (the 224x224x3 / 32 filters / stride 2 / pad 1 layer of "Convolution
  variants and their matrix operations", section 2.1).
* ``body``       -- N=32, 128 -> 256, 112x112, 3x3 s1 p1, BF16, bias+ReLU (the
  112x112x128 -> 256 layer of the same page, sections 3.2-3.3).
* ``dw``         -- N=64, C=256, 56x56, depthwise 3x3 s1 p1, FP32, no bias
  (first half of the depthwise-separable block, lesson 9 section 25).
* ``pw``         -- the block's pointwise 1x1, 256 -> 512, BF16, bias+ReLU.
* ``dilated``    -- N=16, 256 -> 256, 64x64, 3x3 d2 p2 s1, groups 4, BF16,
  bias+ReLU (variants page, sections 2.2-2.3 and 4.2).
* ``f32_3x3``    -- N=8, 64 -> 64, 56x56, 3x3 s1 p1, FP32, bias+ReLU (a first-stage
  residual-network convolution kept in FP32: the Winograd F(2x2, 3x3) comparison).
* ``upsample``   -- N=16, 256 -> 128, 56x56 -> 112x112 transposed convolution,
  4x4 s2 p1, BF16, bias+ReLU (the upsampling layer of the variants page,
  sections 2.3 and 4.2, with the kernel size divisible by the stride as the
  page advises against checkerboard overlap).

Transposed shapes draw their weight as [C_in][C_out/G][Kh][Kw] (the matrix the
operation transposes) with Kaiming fan-in = taps reaching one output,
(C_in/G)*ceil(Kh/S)*ceil(Kw/S).

Value recipe: X ~ N(0, 1) unless stated; W ~ N(0, 2/fan_in) with
fan_in = (C_in/G)*Kh*Kw (Kaiming normal); bias ~ N(0, 0.01^2).  Config i
draws X, W, bias from torch CPU generators seeded 1000*i + {0, 1, 2}; the
block's pointwise weights use 1000*i + 3 and its bias 1000*i + 4.  Draws are
FP32; BF16 workloads round them once (round-to-nearest-even) and every
consumer reads exactly those rounded values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class ConvShape:
    N: int
    C_in: int
    H: int
    W: int
    C_out: int
    Kh: int
    Kw: int
    S: int = 1
    P: int = 0
    D: int = 1
    G: int = 1
    dtype: str = "bf16"          # "f32" or "bf16" (input / weight storage type)
    bias: bool = True
    relu: bool = False
    out_bf16: bool = False       # FP32 depthwise writing a BF16 result (block mode)
    transposed: bool = False     # transposed convolution (the adjoint of the convolution)

    @property
    def H_out(self) -> int:
        if self.transposed:
            return (self.H - 1) * self.S - 2 * self.P + self.D * (self.Kh - 1) + 1
        return (self.H + 2 * self.P - self.D * (self.Kh - 1) - 1) // self.S + 1

    @property
    def W_out(self) -> int:
        if self.transposed:
            return (self.W - 1) * self.S - 2 * self.P + self.D * (self.Kw - 1) + 1
        return (self.W + 2 * self.P - self.D * (self.Kw - 1) - 1) // self.S + 1

    @property
    def pixels(self) -> int:
        return self.N * self.H_out * self.W_out

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs: 2 per multiply-add over live taps only.  Transposed:
        2 per multiply-add of an (output pixel, tap) pair whose input pixel exists."""
        if self.transposed:
            def pairs(n_in, n_out, k):
                ho = np.arange(n_out)[:, None] + self.P - self.D * np.arange(k)[None, :]
                return int(np.sum((ho >= 0) & (ho % self.S == 0) & (ho // self.S < n_in)))
            taps = pairs(self.H, self.H_out, self.Kh) * pairs(self.W, self.W_out, self.Kw)
            return 2 * self.N * taps * self.C_out * (self.C_in // self.G)
        return 2 * self.pixels * self.C_out * (self.C_in // self.G) * self.Kh * self.Kw

    @property
    def algorithmic_bytes(self) -> int:
        """Read X, W and bias once, write Y once."""
        e = 2 if self.dtype == "bf16" else 4
        eo = 2 if (self.dtype == "bf16" or self.out_bf16) else 4
        x = self.N * self.H * self.W * self.C_in * e
        w = self.C_out * (self.C_in // self.G) * self.Kh * self.Kw * e
        b = self.C_out * 4 if self.bias else 0
        y = self.pixels * self.C_out * eo
        return x + w + b + y


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    shape: ConvShape
    x_dist: str = "normal"        # "normal" or "uniform"
    w_dist: str = "kaiming"       # "kaiming" or "uniform"
    b_dist: str = "normal001"     # "normal001" or "uniform"
    description: str = ""


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1,
                         ConvShape(1, 3, 32, 32, 8, 3, 3, 1, 1, 1, 1, "f32", True, False),
                         "uniform", "uniform", "uniform",
                         "Conv2d fp32, N=1, 3->8, 32x32, 3x3 s1 p1, bias"),
    "stem": Workload("stem", 2,
                     ConvShape(32, 3, 224, 224, 32, 3, 3, 2, 1, 1, 1, "bf16", True, True),
                     description="stem conv bf16, N=32, 3->32, 224->112, 3x3 s2 p1, bias+ReLU"),
    "body": Workload("body", 3,
                     ConvShape(32, 128, 112, 112, 256, 3, 3, 1, 1, 1, 1, "bf16", True, True),
                     description="body conv bf16, N=32, 128->256, 112x112, 3x3 s1 p1, bias+ReLU"),
    "dw": Workload("dw", 4,
                   ConvShape(64, 256, 56, 56, 256, 3, 3, 1, 1, 1, 256, "f32", False, False),
                   description="depthwise 3x3 fp32, N=64, C=256, 56x56, s1 p1, groups=256"),
    "pw": Workload("pw", 4,
                   ConvShape(64, 256, 56, 56, 512, 1, 1, 1, 0, 1, 1, "bf16", True, True),
                   description="pointwise 1x1 bf16, N=64, 256->512, 56x56, bias+ReLU"),
    "dilated": Workload("dilated", 5,
                        ConvShape(16, 256, 64, 64, 256, 3, 3, 1, 2, 2, 4, "bf16", True, True),
                        description="dilated grouped conv bf16, N=16, 256->256, 64x64, 3x3 d2 p2 g4, bias+ReLU"),
    "f32_3x3": Workload("f32_3x3", 7,
                        ConvShape(8, 64, 56, 56, 64, 3, 3, 1, 1, 1, 1, "f32", True, True),
                        description="conv fp32, N=8, 64->64, 56x56, 3x3 s1 p1, bias+ReLU"),
    "upsample": Workload("upsample", 6,
                         ConvShape(16, 256, 56, 56, 128, 4, 4, 2, 1, 1, 1, "bf16", True, True, transposed=True),
                         description="transposed conv bf16, N=16, 256->128, 56x56 -> 112x112, 4x4 s2 p1, bias+ReLU"),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round FP32 values once to BF16 (RNE) and return them as FP32."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def draw(shape: ConvShape, seeds, x_dist="normal", w_dist="kaiming", b_dist="normal001"):
    """Draw (x NCHW, w OIHW, bias) as FP32 numpy arrays; BF16 shapes are pre-rounded.

    ``seeds`` = (seed_x, seed_w, seed_b).
    """
    s = shape
    cin_g = s.C_in // s.G
    if x_dist == "uniform":
        x = torch.rand(s.N, s.C_in, s.H, s.W, generator=_gen(seeds[0])) * 2 - 1
    else:
        x = torch.randn(s.N, s.C_in, s.H, s.W, generator=_gen(seeds[0]))
    # conv: w [C_out][C_in/G][Kh][Kw]; transposed: w [C_in][C_out/G][Kh][Kw]
    wshape = (s.C_in, s.C_out // s.G, s.Kh, s.Kw) if s.transposed else (s.C_out, cin_g, s.Kh, s.Kw)
    if w_dist == "uniform":
        w = torch.rand(*wshape, generator=_gen(seeds[1])) * 2 - 1
    else:
        fan_in = cin_g * s.Kh * s.Kw
        if s.transposed:
            fan_in = cin_g * (-(-s.Kh // s.S)) * (-(-s.Kw // s.S))
        std = math.sqrt(2.0 / fan_in)
        w = torch.randn(*wshape, generator=_gen(seeds[1])) * std
    b = None
    if s.bias:
        if b_dist == "uniform":
            b = torch.rand(s.C_out, generator=_gen(seeds[2])) * 2 - 1
        else:
            b = torch.randn(s.C_out, generator=_gen(seeds[2])) * 0.01
        b = b.numpy()
    x, w = x.numpy(), w.numpy()
    if s.dtype == "bf16":
        x, w = round_bf16(x), round_bf16(w)
    return x, w, b


def inputs(name: str):
    """(shape, x NCHW, w OIHW, bias) for a named workload."""
    wl = WORKLOADS[name]
    i = wl.index
    if name == "pw":
        seeds = (1000 * i + 5, 1000 * i + 3, 1000 * i + 4)
    else:
        seeds = (1000 * i, 1000 * i + 1, 1000 * i + 2)
    x, w, b = draw(wl.shape, seeds, wl.x_dist, wl.w_dist, wl.b_dist)
    return wl.shape, x, w, b


def random_shape(rng: np.random.Generator, dtype="bf16", max_c=8, max_hw=9) -> ConvShape:
    """A small random convolution (N<=2, C<=max_c, H,W<=max_hw, K in {1,2,3,5},
    S in {1,2,3}, P in [0,3], D in {1,2,3}, G dividing both channel counts)
    whose output is non-empty."""
    while True:
        N = int(rng.integers(1, 3))
        G = int(rng.choice([1, 1, 2, 4]))
        C_in = G * int(rng.integers(1, max(2, max_c // G + 1)))
        C_out = G * int(rng.integers(1, max(2, max_c // G + 1)))
        H, W = int(rng.integers(1, max_hw + 1)), int(rng.integers(1, max_hw + 1))
        Kh, Kw = int(rng.choice([1, 2, 3, 5])), int(rng.choice([1, 2, 3, 5]))
        S, P, D = int(rng.choice([1, 2, 3])), int(rng.integers(0, 4)), int(rng.choice([1, 2, 3]))
        s = ConvShape(N, C_in, H, W, C_out, Kh, Kw, S, P, D, G, dtype,
                      bool(rng.integers(0, 2)), bool(rng.integers(0, 2)))
        if s.H_out >= 1 and s.W_out >= 1:
            return s


# ---------------------------------------------------------------- layout marshalling
def x_device(x_nchw: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """NCHW values -> contiguous NHWC tensor [N][H][W][C] of the storage dtype."""
    t = torch.from_numpy(np.ascontiguousarray(x_nchw, dtype=np.float32)).permute(0, 2, 3, 1).contiguous()
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    return t.to(device)


def w_device_transposed(w_iohw: np.ndarray, dtype: str, groups: int = 1, device="cuda") -> torch.Tensor:
    """Transposed-convolution weights [C_in][C_out/G][Kh][Kw] -> the library's
    [C_out][Kh][Kw][C_in/G] (a permutation per group, no flip)."""
    C_in, cout_g, Kh, Kw = w_iohw.shape
    cin_g = C_in // groups
    w = np.asarray(w_iohw, dtype=np.float32).reshape(groups, cin_g, cout_g, Kh, Kw)
    w = w.transpose(0, 2, 3, 4, 1).reshape(groups * cout_g, Kh, Kw, cin_g)
    t = torch.from_numpy(np.ascontiguousarray(w))
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float32).to(device)


def w_device(w_oihw: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """OIHW weights -> contiguous [C_out][Kh][Kw][C_in/G] tensor of the storage dtype."""
    t = torch.from_numpy(np.ascontiguousarray(w_oihw, dtype=np.float32)).permute(0, 2, 3, 1).contiguous()
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    return t.to(device)


def b_device(b, device="cuda"):
    if b is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(b, dtype=np.float32)).to(device)


def y_to_nchw(y_nhwc: torch.Tensor) -> np.ndarray:
    """Device NHWC result -> float64 NCHW numpy array."""
    return y_nhwc.float().cpu().permute(0, 3, 1, 2).contiguous().double().numpy()
