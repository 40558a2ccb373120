"""The forward calls are CUDA-graph capturable: a graph of conv_forward (and of the fused
block) replays to the same bits as the eager call, and a replay after the input changed in
place computes the new result (the graph holds the buffers, not the values)."""
import numpy as np
import pytest
import torch

from workloads import b_device, inputs, w_device, x_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_f32", "stem", "body", "dw", "dilated", "upsample", "f32_3x3"])
def test_conv_forward_replays_in_a_cuda_graph(name):
    from cnn_convolution_implicit_gb300 import ConvPlan, device_status
    from workloads import w_device_transposed
    s, x, w, b = inputs(name)
    plan = ConvPlan.for_shape(s)
    xd = x_device(x, s.dtype)
    wd = w_device_transposed(w, s.dtype, s.G) if s.transposed else w_device(w, s.dtype)
    bd = b_device(b) if s.bias else None
    y = plan.empty_output()
    plan.forward(xd, wd, bd, y)  # first call: tensor maps encoded and cached for these pointers
    torch.cuda.synchronize()
    y_eager = y.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plan.forward(xd, wd, bd, y)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert device_status() == 0
    assert torch.equal(y, y_eager)
    xd.mul_(-0.5)  # new values in the same buffer
    graph.replay()
    torch.cuda.synchronize()
    y_new = plan.forward(xd, wd, bd)
    torch.cuda.synchronize()
    assert device_status() == 0
    assert torch.equal(y, y_new) and not torch.equal(y_new, y_eager)


def test_block_forward_replays_in_a_cuda_graph():
    from cnn_convolution_implicit_gb300 import BlockPlan, device_status
    sd, x, wd, _ = inputs("dw")
    sp, _, wp, bp = inputs("pw")
    plan = BlockPlan(sd.N, sd.C_in, sd.H, sd.W, sp.C_out, 3, 1, dw_relu=False, pw_relu=True)
    xd = x_device(x, "f32")
    wdd = torch.from_numpy(np.ascontiguousarray(wd[:, 0], np.float32)).cuda()
    wpd = w_device(wp, "bf16").reshape(sp.C_out, sp.C_in)
    bd = b_device(bp)
    y = plan.empty_output()
    plan.forward(xd, wdd, wpd, pw_bias=bd, y=y)
    torch.cuda.synchronize()
    y_eager = y.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plan.forward(xd, wdd, wpd, pw_bias=bd, y=y)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert device_status() == 0
    assert torch.equal(y, y_eager)
