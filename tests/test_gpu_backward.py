"""GPU parity of the routed branch's backward pass (lmoe_routed_backward) against the oracle's
(PyTorch fp64 autodiff of the branch, pinned to finite differences).  Routing is shared
through lmoe_io.logits_in, so both sides differentiate the same selection.

Tolerance (derived): the device path rounds five intermediates to bf16 (the latent, the
expert outputs, do, dh and the gate/value gradients, each relative 2^-9) and accumulates in
fp32.  A gradient element is a sum of n products of two such operands (n: an expert's tokens
for the weights, L or 2I features for the latent), so its error is at most ~2^-8 sum|terms|,
which under sign cancellation is ~sqrt(n) times the element's typical size: per tensor the
mean relative error is at most 1.5e-2, the RMS error at most 2.5e-2 of the tensor's RMS, and
the largest element error at most 0.15 of it (the tail at n ~ 30-150).  With one or two
tokens per expert an element is a single product, with no sum to average its error, and
the gradient is a heavy-tailed outer product (largest element 15-40 times the RMS): there
the largest error is bounded by a single product's, 2^-7 of itself, with a factor 2 of
margin: max(0.15 RMS, 2^-6 of the largest magnitude)."""
import numpy as np
import pytest
import torch

from latent_compressed_expert_gb300 import lmoe, synth

pytestmark = pytest.mark.gpu

MEAN_REL = 1.5e-2
RMS_REL = 2.5e-2
MAX_REL_RMS = 0.15
MAX_REL_PEAK = 2.0 ** -6


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
            "max_over_peak": float(err.max() / np.abs(ref).max()),
            "rms_rel": float(np.sqrt(np.mean(err * err)) / rms),
            "mean_rel": float(err.sum() / np.abs(ref).sum())}


def _ok(s):
    return (s["finite"] and s["mean_rel"] <= MEAN_REL and s["rms_rel"] <= RMS_REL
            and (s["max_over_rms"] <= MAX_REL_RMS or s["max_over_peak"] <= MAX_REL_PEAK))


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


LAYER_KEYS = ("dx", "dgamma", "dw_down", "dw_gate", "dw_value", "dw_edown", "dw_up",
              "dw_sgate", "dw_svalue", "dw_sdown")
EXPERT_KEYS = ("dw_gate", "dw_value", "dw_edown")


def _router_sigma(ref, idx, E):
    """Standard deviation of the rounding error of each router weight-gradient element,
    dW_r = sum_t dlogit[t]^T lat[t] with dlogit_j = (dg_j - sum_i g_i dg_i) / S * s_j (1 - s_j)
    and dg_j = <du, o_j>.  The device computes dg_j from bf16 expert outputs o (and a du
    that inherits their rounding): independent errors of at most 2^-9 relative per term,
    whose variances add, so sd(dg_j) <= 2^-8 sqrt(sum_l (du_l o_jl)^2) with margin.  They
    propagate through the normalisation (where the difference may cancel, which is why a
    tensor-wide ratio does not bound this gradient at a few tokens) and, with the bf16
    stores of dlogit and of the latent (2^-8 each, with margin), through the token sum."""
    du, o, s, g, lat = ref["du"], ref["o"], ref["s"], ref["gate"], ref["lat"]
    sd_dg = 2.0 ** -8 * np.sqrt(np.einsum("tl,tjl->tj", du * du, o * o))
    dg = np.einsum("tl,tjl->tj", du, o)
    S = s.sum(1, keepdims=True)
    dl = (dg - (g * dg).sum(1, keepdims=True)) / S * s * (1.0 - s)
    sd_dl = np.sqrt((s * (1.0 - s) / S) ** 2 * (sd_dg ** 2 + (g * g * sd_dg ** 2).sum(1, keepdims=True))
                    + (2.0 ** -8 * dl) ** 2)
    T = idx.shape[0]
    sd_mat = np.zeros((T, E))
    dl_mat = np.zeros((T, E))
    rows = np.repeat(np.arange(T), idx.shape[1])
    sd_mat[rows, idx.ravel()] = sd_dl.ravel()
    dl_mat[rows, idx.ravel()] = dl.ravel()
    return np.sqrt((sd_mat ** 2).T @ lat ** 2 + 2.0 ** -16 * (dl_mat ** 2).T @ lat ** 2)


@pytest.mark.parametrize("shape", [
    synth.LayerShape("b1", T=256, d=512, L=256, E=32, K=4, I=128, S=2, Is=128),
    synth.LayerShape("b2", T=300, d=512, L=384, E=16, K=6, I=192, S=0, Is=0),  # ragged tiles
    # one token, and seven: most experts get no rows, every segment and the dense weight
    # gradients' single K-block are partial
    synth.LayerShape("b_t1", T=1, d=512, L=256, E=32, K=4, I=128, S=2, Is=128),
    synth.LayerShape("b_t7", T=7, d=512, L=256, E=32, K=4, I=128, S=2, Is=128),
    # one expert per token: the gate is s/s = 1 whatever s, so the router gets no gradient
    synth.LayerShape("b_k1", T=130, d=512, L=256, E=16, K=1, I=128, S=2, Is=128),
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
    ref = B.layer_backward(x, r.idx, w, dy.double().numpy(), intermediates=True)
    # experts no token chose have exactly zero gradients; the statistics cover the others
    # (at a few tokens most experts are idle, and their zeros would dilute the RMS)
    used = np.unique(r.idx)
    idle = np.setdiff1d(np.arange(sh.E), used)
    got = {k: g[k].cpu().numpy() for k in LAYER_KEYS + ("dw_router",) if ref[k].size > 0}
    for k in EXPERT_KEYS + ("dw_router",):
        assert np.all(got[k][idle] == 0.0), k
    stats = {k: _stats(got[k][used] if k in EXPERT_KEYS else got[k],
                       ref[k][used] if k in EXPERT_KEYS else ref[k])
             for k in LAYER_KEYS if ref[k].size > 0}
    bad = {k: v for k, v in stats.items() if not _ok(v)}
    assert not bad, (sh.name, bad)
    if sh.K == 1:
        assert np.all(got["dw_router"] == 0.0)
    # the router's gradient: every element within 6 standard deviations of its rounding
    excess = np.abs(got["dw_router"] - ref["dw_router"]) - 6.0 * _router_sigma(ref, r.idx, sh.E)
    assert excess.max() <= 1e-6 * np.abs(ref["dw_router"]).max(), (sh.name, excess.max())


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


def test_prefill_backward_sampled_tokens_and_linearity(dev, oracle_mod):
    """The benchmark's backward at the full K3 prefill shape (T=8192, E=896, top-16, x with
    0.1 % outliers).  The oracle computes every token's latent and logits, the in-batch
    thresholds and the routing (bit-exact against the device on the same logits), then dx of
    sampled tokens, one at a time.  Every weight gradient sums over thousands of tokens, so
    at this size they are held to a property: each backward step is linear in dy and
    doubling is exact in binary floating point, so backward(2 dy) is 2 backward(dy), bit for
    bit, in every output."""
    import gpu_helpers as H
    import oracle.backward as B
    sh = synth.PREFILL
    gain = synth.outlier_router_gain(sh, 0.001, 1000.0)
    w = synth.make_weights(sh, seed=4, device=dev, router_gain=gain)
    x = synth.make_x(sh, seed=4, device=dev, outlier_frac=0.001)
    wh = H.weights_to_host(w)
    xh = x.cpu()
    lat = oracle_mod.latent(xh, wh["w_down"])
    lg32 = oracle_mod.router_logits(lat, wh["w_router"]).astype(np.float32)
    tau = oracle_mod.thresholds(lg32, oracle_mod.fair_share_rank(sh.T, sh.K, sh.E))
    idx, _, _ = oracle_mod.route(lg32, tau, sh.K)
    layer = lmoe.Layer(sh, w)
    layer.enable_backward(w)
    logits = torch.as_tensor(lg32).to(dev)
    _, dbg = layer.forward(x, residual=x, logits_in=logits, train=True, debug=True)
    assert np.array_equal(dbg["idx"].cpu().numpy(), idx)
    dy = torch.randn(sh.T, sh.d, generator=torch.Generator(device=dev).manual_seed(5),
                     device=dev).to(torch.bfloat16)
    g = {k: v.clone() for k, v in layer.backward_layer(x, dy, logits=logits).items()}
    g2 = layer.backward_layer(x, dy * 2, logits=logits)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    for k in ("dx", "dgamma", "dw_in", "dw_router", "dw_gu", "dw_edown", "dw_out"):
        assert torch.equal(g2[k], 2 * g[k]), k
    rows = np.array([0, 1, 4095, 8191] + list(np.random.default_rng(6).choice(sh.T, 2, replace=False)))
    ref = B.layer_dx_rows(xh[rows], idx[rows], wh, dy[rows].double().cpu().numpy())
    s = _stats(g["dx"][rows].cpu().numpy(), ref)
    assert _ok(s), s
