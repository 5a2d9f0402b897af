"""Failure detection without a GPU fault: a device-side wait is made to run out (the first
GEMM waits on an mbarrier that nothing arrives on), every role of that kernel gives up
within the wait limit, frees its tensor memory and returns; the host reads the time-out
from the workspace flag, and the next call on the same context is correct again."""
import numpy as np
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


def test_stalled_wait_reports_timeout_and_context_recovers(dev, oracle_mod, monkeypatch):
    sh = synth.TINY
    w = synth.make_weights(sh, seed=9)
    layer = lmoe.Layer(sh, {k: v.to(dev) for k, v in w.items()})
    x = synth.make_x(sh, seed=9)
    xd = x.to(dev)
    logits = synth.make_logits(sh.T, sh.E, seed=9)
    monkeypatch.setenv("LMOE_WAIT_LIMIT_MS", "200")
    monkeypatch.setenv("LMOE_FAULT_INJECT", "stall")
    layer.forward(xd, residual=xd, logits_in=logits.to(dev))
    torch.cuda.synchronize()
    assert layer.device_error() == lmoe.LMOE_ERR_DEVICE_TIMEOUT
    assert layer.device_error() == lmoe.LMOE_OK  # reading clears the flag
    monkeypatch.delenv("LMOE_FAULT_INJECT")
    y, dbg = layer.forward(xd, residual=xd, logits_in=logits.to(dev), debug=True)
    torch.cuda.synchronize()
    assert layer.device_error() == lmoe.LMOE_OK
    ref = oracle_mod.forward(w, x, sh.K, residual=x, tau="batch", logits_in=logits.numpy())
    H.assert_layer_close(y, dbg["y_f32"], ref.y, "after-timeout")


def test_stalled_wait_over_sm_pairs(dev, monkeypatch):
    """The same at a size where the first GEMM runs over SM pairs (8192 tokens, d = 2048: 320
    cluster tiles of 256 x 256, K = 2048).  Rank 0's MMA issuer stalls; rank 0's other roles see
    its abort flag, rank 1's run into their own wait limits, both CTAs of each cluster meet at
    the teardown barrier and free their tensor memory.  The call reports the time-out, and the
    next call on the context gives an earlier call's bits.  Routing runs on given logits, so
    the stalled GEMM's unwritten output reaches no index."""
    sh = synth.LayerShape("pairstall", T=8192, d=2048, L=2048, E=16, K=2, I=256, S=1, Is=256)
    w = synth.make_weights(sh, seed=19, device=dev)
    layer = lmoe.Layer(sh, w)
    x = synth.make_x(sh, seed=19, device=dev)
    logits = synth.make_logits(sh.T, sh.E, seed=19).to(dev)
    y0 = layer.forward(x, residual=x, logits_in=logits).clone()
    torch.cuda.synchronize()
    assert layer.device_error() == lmoe.LMOE_OK
    monkeypatch.setenv("LMOE_WAIT_LIMIT_MS", "200")
    monkeypatch.setenv("LMOE_FAULT_INJECT", "stall")
    layer.forward(x, residual=x, logits_in=logits)
    torch.cuda.synchronize()
    assert layer.device_error() == lmoe.LMOE_ERR_DEVICE_TIMEOUT
    assert layer.device_error() == lmoe.LMOE_OK  # reading clears the flag
    monkeypatch.delenv("LMOE_FAULT_INJECT")
    y2 = layer.forward(x, residual=x, logits_in=logits)
    torch.cuda.synchronize()
    assert layer.device_error() == lmoe.LMOE_OK
    assert torch.equal(y2.view(torch.int16), y0.view(torch.int16))
