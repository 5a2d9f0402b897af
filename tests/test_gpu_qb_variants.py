"""Quantile-Balancing variants on the GPU: streaming (EMA) thresholds, load statistics over
steps, and the 448-expert / top-8 pool the pages set against 896 / top-16
("The 2.8-Trillion-Parameter Problem", LatentMoE bullet of the summary).  Routing decisions
and counters are bit-exact against the oracle on identical logits."""
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


@pytest.mark.parametrize("beta", [0.0, 0.3, 0.9, 1.0])
def test_tau_ema_bit_exact(dev, oracle_mod, beta):
    rng = np.random.default_rng(int(beta * 10) + 1)
    E = 896
    prev = rng.uniform(0.2, 0.95, E).astype(np.float32)
    step = rng.uniform(0.2, 0.95, E).astype(np.float32)
    for first in (False, True):
        t = torch.from_numpy(prev.copy()).to(dev)
        lmoe.tau_ema(torch.from_numpy(step).to(dev), t, beta, first)
        ref = oracle_mod.tau_ema(prev, step, beta, first)
        assert np.array_equal(t.cpu().numpy().view(np.int32), ref.view(np.int32))


def test_load_stats_bit_exact(dev, oracle_mod):
    rng = np.random.default_rng(3)
    E = 1500  # more experts than threads of the kernel's block
    stats = lmoe.LoadStats(E, dev)
    ref = None
    for step in range(6):
        c = rng.integers(0, 300, E).astype(np.int32)
        c[rng.choice(E, 20, replace=False)] = 0
        stats.update(torch.from_numpy(c).to(dev))
        ref = oracle_mod.load_stats_update(ref, c)
    assert np.array_equal(stats.acc.cpu().numpy().astype(np.uint64), ref)


def test_streaming_thresholds_in_the_forward(dev, oracle_mod):
    """Three batches: the first initialises the streaming thresholds, the next two fold
    theirs in with beta = 0.8; every batch is routed against the updated thresholds, and
    the layer's load counters accumulate each step's counts."""
    sh = H.mid_shape()
    w = synth.make_weights(sh, seed=41)
    wd = {k: v.to(dev) for k, v in w.items()}
    layer = lmoe.Layer(sh, wd)
    k = oracle_mod.fair_share_rank(sh.T, sh.K, sh.E)
    tau = torch.zeros(sh.E, dtype=torch.float32, device=dev)
    stats = lmoe.LoadStats(sh.E, dev)
    ref_tau, ref_acc = None, None
    for step in range(3):
        x = synth.make_x(sh, seed=41 + step).to(dev)
        logits = synth.make_logits(sh.T, sh.E, seed=141 + step)
        _, dbg = layer.forward(x, residual=x, logits_in=logits.to(dev), debug=True, tau_ema=tau,
                               ema_beta=0.8, ema_first=step == 0, load_stats=stats)
        torch.cuda.synchronize()
        assert layer.device_error() == 0
        lg = logits.numpy()
        ref_tau = oracle_mod.tau_ema(ref_tau, oracle_mod.thresholds(lg, k), 0.8, first=step == 0)
        assert np.array_equal(tau.cpu().numpy().view(np.int32), ref_tau.view(np.int32)), step
        assert np.array_equal(dbg["tau"].cpu().numpy().view(np.int32), ref_tau.view(np.int32))
        idx, gate, _ = oracle_mod.route(lg, ref_tau, sh.K)
        assert np.array_equal(dbg["idx"].cpu().numpy(), idx)
        assert np.array_equal(dbg["gate"].cpu().numpy().view(np.int32), gate.view(np.int32))
        ref_acc = oracle_mod.load_stats_update(ref_acc, np.bincount(idx.ravel(), minlength=sh.E))
    assert np.array_equal(stats.acc.cpu().numpy().astype(np.uint64), ref_acc)
    s = stats.summary()
    assert s["steps"] == 3 and s["fair_share"] == pytest.approx(sh.T * sh.K / sh.E)


def test_pool_448_top8_layer(dev, oracle_mod):
    """The alternative pool: 448 experts, 8 per token (the same 1/56 activation ratio), at
    a reduced width; every token against the oracle, routing on identical logits."""
    sh = synth.LayerShape("p448", T=1024, d=1024, L=512, E=448, K=8, I=256, S=2, Is=512)
    w = synth.make_weights(sh, seed=51)
    wd = {k: v.to(dev) for k, v in w.items()}
    layer = lmoe.Layer(sh, wd)
    x = synth.make_x(sh, seed=51)
    xd = x.to(dev)
    logits = synth.make_logits(sh.T, sh.E, seed=52)
    y, dbg = layer.forward(xd, residual=xd, logits_in=logits.to(dev), debug=True)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ref = oracle_mod.forward(w, x, sh.K, residual=x, tau="batch", logits_in=logits.numpy())
    assert np.array_equal(dbg["tau"].cpu().numpy().view(np.int32), ref.tau.view(np.int32))
    assert np.array_equal(dbg["idx"].cpu().numpy(), ref.idx)
    H.assert_layer_close(y, dbg["y_f32"], ref.y, "pool448")
    counts = dbg["counts"].cpu().numpy()
    assert counts.sum() == sh.T * sh.K and counts.max() <= 3 * sh.T * sh.K / sh.E
