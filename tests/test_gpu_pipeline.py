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


@pytest.mark.parametrize("T", [64, 1000])
def test_forward_replays_from_a_cuda_graph(dev, T):
    """lmoe_forward enqueues only kernels, memsets and event-free copies on its stream, so a
    whole layer call (split-K dense GEMMs at T = 64, the routed GEMMs' pairs at T = 1000) can be
    captured into a CUDA graph and replayed; each replay gives the eager call's bits."""
    sh = H.mid_shape(T)
    w = {k: v.to(dev) for k, v in synth.make_weights(sh, seed=63).items()}
    layer = lmoe.Layer(sh, w)
    x = synth.make_x(sh, seed=64).to(dev)
    ref = layer.forward(x, residual=x).clone()
    torch.cuda.synchronize()
    y = torch.empty_like(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm up the kernels' attributes outside the capture
        layer.forward(x, residual=x, y=y)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x, residual=x, y=y)
    for _ in range(2):
        y.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        assert layer.device_error() == 0
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_cluster_kernels_replay_from_a_cuda_graph(dev):
    """The same at a size where the dense GEMMs and the down GEMM run over SM pairs (clusters of
    two CTAs, launched with a cluster dimension): 8192 tokens, d = 2048, 1024 tokens per expert
    in 256-token chunks.  Each replay gives the eager call's bits."""
    sh = synth.LayerShape("pairgraph", T=8192, d=2048, L=2048, E=16, K=2, I=256, S=1, Is=256)
    w = synth.make_weights(sh, seed=65, device=dev)
    layer = lmoe.Layer(sh, w)
    x = synth.make_x(sh, seed=66, device=dev)
    ref = layer.forward(x, residual=x).clone()
    torch.cuda.synchronize()
    y = torch.empty_like(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(x, residual=x, y=y)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x, residual=x, y=y)
    for _ in range(2):
        y.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        assert layer.device_error() == 0
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
