"""GPU: the bounded-wait failure path of the pipelined kernels, made to run on purpose
without a fault (a barrier that nothing completes), and the context afterwards."""
import numpy as np
import pytest
import torch

from parity import check_full, oracle_full, run
from workloads import ConvShape, b_device, draw, w_device, x_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [1_000_000, 20_000_000])
def test_wait_gives_up_reports_and_context_survives(limit_ns):
    """One role's wait on a never-completed mbarrier gives up after the given limit (bit 2);
    a second role waiting with the kernels' own 2 s limit leaves through the CTA's abort flag
    (bit 4) well before that; conv_device_status reports CONV_ERR_TIMEOUT with both bits and
    clears them; a following convolution on the same context is parity-green."""
    from cnn_convolution_implicit_gb300 import ConvPlan, check_wait_timeout, device_status
    assert device_status() == 0
    code, elapsed = check_wait_timeout(limit_ns)
    assert code == 2 | 4, code
    assert limit_ns <= elapsed < limit_ns + 200_000_000, elapsed  # not the 2 s limit of the second role
    assert device_status() == 0                                    # the word was cleared
    s = ConvShape(2, 128, 13, 11, 256, 3, 3, 1, 1, 1, 1, "bf16", True, True)
    x, w, b = draw(s, (71, 72, 73))
    _, y = run(s, x, w, b, plan=ConvPlan.for_shape(s))
    check_full(s, y, oracle_full(s, x, w, b))


def test_plan_status_words_attribute_timeouts():
    """Each plan reads only its own status word, in the order of one stream.  A plan made
    after all 1,024 words are taken shares the library-wide word, which is where the
    wait-timeout check latches its bits: that plan reports them (and clears them), a plan
    with its own word stays clean, and conv_device_status then finds nothing left."""
    import ctypes
    import gc
    from cnn_convolution_implicit_gb300 import ConvPlan, binding, device_status, lib
    binding._plan_cache.clear()  # plans other tests left alive hold words of the pool
    gc.collect()
    assert device_status() == 0
    s = ConvShape(2, 128, 13, 11, 256, 3, 3, 1, 1, 1, 1, "bf16", True, True)
    x, w, b = draw(s, (81, 82, 83))
    own = ConvPlan.for_shape(s)
    xd, wd, bd = x_device(x, s.dtype), w_device(w, s.dtype), b_device(b)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        y = own.forward(xd, wd, bd)
    assert own.device_status(side) == 0           # after the forward, in the side stream's order
    check_full(s, y, oracle_full(s, x, w, b))
    plans = [ConvPlan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, 1, "bf16") for _ in range(1025)]
    shared = plans[-1]                            # at least 1,025 plans alive: no word left
    L = lib()
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream()
    assert L.conv_check_wait_timeout(1_000_000, ctypes.c_void_p(elapsed.data_ptr()),
                                     ctypes.c_void_p(stream.cuda_stream)) == 0
    assert own.device_status() == 0
    assert shared.device_status() == 2 | 4        # read after the check in stream order
    assert shared.device_status() == 0            # and cleared
    assert device_status() == 0
    del plans, shared


def test_block_plan_status_word_in_stream_order():
    """A fused-block forward on a side stream leaves the block plan's own status word clean,
    read after that stream's work; the forward's output matches the same plan on the
    default stream bit for bit."""
    from cnn_convolution_implicit_gb300 import BlockPlan, device_status
    assert device_status() == 0
    g = torch.Generator().manual_seed(91)
    N, C, H, W, Co = 2, 128, 17, 20, 96
    plan = BlockPlan(N, C, H, W, Co, 3, 1)
    x = torch.randn(N, H, W, C, generator=g).cuda()
    wdw = (torch.randn(C, 3, 3, generator=g) * 0.3).cuda()
    wpw = (torch.randn(Co, C, generator=g) * 0.1).to(torch.bfloat16).cuda()
    bias = torch.randn(Co, generator=g).cuda()
    ref = plan.forward(x, wdw, wpw, pw_bias=bias)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        y = plan.forward(x, wdw, wpw, pw_bias=bias)
    assert plan.device_status(side) == 0
    assert torch.equal(y.view(torch.int16).cpu(), ref.view(torch.int16).cpu())
    assert device_status() == 0
