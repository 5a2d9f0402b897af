"""GPU parity of the routed branch's backward pass (lmoe_routed_backward) against the oracle's
(PyTorch fp64 autodiff of the branch, pinned to finite differences).  Routing is shared
through lmoe_io.logits_in, so both sides differentiate the same selection.

Tolerance (derived): the device path rounds five intermediates to bf16 (the latent, the
expert outputs, do, dh and the gate/value gradients, each relative 2^-9) and accumulates in
fp32.  A gradient element is a sum of n products of two such operands (n: an expert's tokens
for the weights, L or 2I features for the latent), so its error is at most ~2^-8 sum|terms|,
which under sign cancellation is ~sqrt(n) times the element's typical size: per tensor the
mean relative error is at most 1.5e-2, the RMS error at most 2.5e-2 of the tensor's RMS, and
the largest element error at most 0.15 of it (the tail at n ~ 30-150)."""
import numpy as np
import pytest
import torch

from latent_compressed_expert_gb300 import lmoe, synth

pytestmark = pytest.mark.gpu

MEAN_REL = 1.5e-2
RMS_REL = 2.5e-2
MAX_REL_RMS = 0.15


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from latent_compressed_expert_gb300 import build
    build.build()
    lmoe.load()
    return torch.device("cuda:0")


def _stats(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return {"finite": bool(np.all(np.isfinite(got))), "max_over_rms": float(err.max() / rms),
            "rms_rel": float(np.sqrt(np.mean(err * err)) / rms),
            "mean_rel": float(err.sum() / np.abs(ref).sum())}


def _ok(s):
    return (s["finite"] and s["mean_rel"] <= MEAN_REL and s["rms_rel"] <= RMS_REL
            and s["max_over_rms"] <= MAX_REL_RMS)


@pytest.mark.parametrize("shape", [
    synth.LayerShape("b1", T=256, d=512, L=256, E=32, K=4, I=128, S=2, Is=128),
    synth.LayerShape("b2", T=300, d=512, L=384, E=16, K=6, I=192, S=0, Is=0),  # ragged tiles
])
def test_routed_backward_matches_oracle(dev, oracle_mod, shape):
    import oracle.backward as B
    sh = shape
    w = synth.make_weights(sh, seed=81)
    wd = {k: v.to(dev) for k, v in w.items()}
    layer = lmoe.Layer(sh, wd)
    layer.enable_backward(wd)
    x = synth.make_x(sh, seed=82)
    logits = synth.make_logits(sh.T, sh.E, seed=83)
    xd = x.to(dev)
    _, dbg = layer.forward(xd, residual=xd, logits_in=logits.to(dev), debug=True)
    dz = torch.randn(sh.T, sh.L, generator=torch.Generator().manual_seed(84))
    g = layer.backward(dz.to(dev))
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    lat = oracle_mod.latent(x, w["w_down"])
    idx, gate, _ = oracle_mod.route(logits.numpy(), oracle_mod.thresholds(
        logits.numpy(), oracle_mod.fair_share_rank(sh.T, sh.K, sh.E)), sh.K)
    assert np.array_equal(dbg["idx"].cpu().numpy(), idx)
    ref = B.routed_backward(lat, idx, gate, w["w_gate"], w["w_value"], w["w_edown"],
                            w["gamma"].numpy(), dz.numpy())
    stats = {key: _stats(g[key].cpu().numpy(), ref[key])
             for key in ("dlat", "dgate", "dgamma", "dw_gate", "dw_value", "dw_edown")}
    assert all(_ok(v) for v in stats.values()), (sh.name, stats)
    # experts no token chose have zero weight gradients
    unused = np.setdiff1d(np.arange(sh.E), np.unique(idx))
    if len(unused):
        assert float(g["dw_edown"][torch.as_tensor(unused)].abs().max()) == 0.0


LAYER_KEYS = ("dx", "dgamma", "dw_down", "dw_router", "dw_gate", "dw_value", "dw_edown", "dw_up",
              "dw_sgate", "dw_svalue", "dw_sdown")


@pytest.mark.parametrize("shape", [
    synth.LayerShape("b1", T=256, d=512, L=256, E=32, K=4, I=128, S=2, Is=128),
    synth.LayerShape("b2", T=300, d=512, L=384, E=16, K=6, I=192, S=0, Is=0),  # ragged tiles
])
def test_layer_backward_matches_oracle(dev, oracle_mod, shape):
    """lmoe_backward against the oracle's whole-layer backward.  The GPU routes on the
    oracle's own fp32 logits (logits_in), so the selection is shared and the gates are those
    of lat W_r^T on both sides."""
    import oracle.backward as B
    sh = shape
    w = synth.make_weights(sh, seed=91)
    w["gamma"] = torch.linspace(0.6, 1.4, sh.L)
    wd = {k: v.to(dev) for k, v in w.items()}
    layer = lmoe.Layer(sh, wd)
    layer.enable_backward(wd)
    x = synth.make_x(sh, seed=92)
    r = oracle_mod.forward(w, x, sh.K, residual=None)
    logits = torch.as_tensor(r.logits).to(dev)
    xd = x.to(dev)
    _, dbg = layer.forward(xd, residual=xd, logits_in=logits, debug=True)
    assert np.array_equal(dbg["idx"].cpu().numpy(), r.idx)
    dy = torch.randn(sh.T, sh.d, generator=torch.Generator().manual_seed(93)).to(torch.bfloat16)
    g = layer.backward_layer(xd, dy.to(dev), logits=logits)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ref = B.layer_backward(x, r.idx, w, dy.double().numpy())
    keys = [k for k in LAYER_KEYS if ref[k].size > 0]
    stats = {k: _stats(g[k].cpu().numpy(), ref[k]) for k in keys}
    assert all(_ok(v) for v in stats.values()), (sh.name, stats)


def test_saved_pre_activations_match_recompute(dev):
    """A training forward keeps the routed pre-activations (lmoe_io.save_pre); the backward
    that uses them equals, bit for bit, the one that recomputes them (same GEMM, same
    accumulation order)."""
    sh = synth.LayerShape("b1", T=256, d=512, L=256, E=32, K=4, I=128, S=2, Is=128)
    w = synth.make_weights(sh, seed=95)
    wd = {k: v.to(dev) for k, v in w.items()}
    layer = lmoe.Layer(sh, wd)
    layer.enable_backward(wd)
    x = synth.make_x(sh, seed=96).to(dev)
    dy = torch.randn(sh.T, sh.d, generator=torch.Generator().manual_seed(97)).to(torch.bfloat16)
    dy = dy.to(dev)
    layer.forward(x, residual=x)
    g0 = {k: v.clone() for k, v in layer.backward_layer(x, dy).items()}
    layer.forward(x, residual=x, train=True)
    g1 = layer.backward_layer(x, dy)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    for k in g0:
        assert torch.equal(g0[k], g1[k]), k
