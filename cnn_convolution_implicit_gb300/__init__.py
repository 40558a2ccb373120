"""GB300 (sm_103a) forward 2D convolution: implicit GEMM on tcgen05 tensor cores,
a 1x1 GEMM path, a small-K (stem) path, a TMA halo-tile depthwise kernel and a
direct fallback kernel, behind the C ABI of include/conv.h.

    from cnn_convolution_implicit_gb300 import ConvPlan, conv2d
"""
from .binding import (CONV_BF16, CONV_F32, EXPORTS, PATHS, BlockPlan, ConvError, ConvPlan,
                      check_wait_timeout, conv2d, device_status, lib, measure_mma_rate)

__all__ = ["ConvPlan", "BlockPlan", "conv2d", "ConvError", "device_status", "lib", "measure_mma_rate",
           "check_wait_timeout", "PATHS", "EXPORTS", "CONV_BF16", "CONV_F32"]
