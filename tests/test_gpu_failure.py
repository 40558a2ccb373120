"""GPU: the bounded-wait failure path of the pipelined kernels, made to run on purpose
without a fault (a barrier that nothing completes), and the context afterwards."""
import numpy as np
import pytest
import torch

from parity import check_full, oracle_full, run
from workloads import ConvShape, draw

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
