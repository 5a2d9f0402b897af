"""The pipelined host path (lmoe_forward_host through lmoe.HostPipeline): batches in pinned
host memory, copies on their own streams overlapped with the neighbouring batches' compute.
Every batch's output must equal the plain device call's, bit for bit, whatever the overlap
and whatever the batch sizes."""
import pytest
import torch

import gpu_helpers as H
from latent_compressed_expert_gb300 import lmoe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from latent_compressed_expert_gb300 import build
    build.build()
    lmoe.load()
    return torch.device("cuda:0")


@pytest.mark.parametrize("depth", [1, 2, 3, 4])
def test_pipelined_batches_equal_plain_calls(dev, depth):
    sh = H.mid_shape()
    w = {k: v.to(dev) for k, v in synth.make_weights(sh, seed=61).items()}
    layer = lmoe.Layer(sh, w)
    xs = [synth.make_x(sh, seed=61 + i, T=(357 if i == 3 else sh.T)) for i in range(6)]
    ref = []
    for x in xs:
        xd = x.to(dev)
        ref.append(layer.forward(xd, residual=xd).cpu())
    torch.cuda.synchronize()
    pipe = lmoe.HostPipeline(layer, depth=depth)
    x_host = [x.pin_memory() for x in xs]
    y_host = [torch.empty_like(x).pin_memory() for x in xs]
    for xh, yh in zip(x_host, y_host):
        pipe.submit(xh, yh)
    pipe.synchronize()
    assert layer.device_error() == 0
    for yh, r in zip(y_host, ref):
        assert torch.equal(yh.view(torch.int16), r.view(torch.int16))
