"""Pins of the backward oracle (oracle/backward.py): its re-statement of the routed branch
equals the pinned C oracle's forward, and its gradients equal central finite differences of
that forward on tiny inputs (every input: latent, gates, gamma and the three weights)."""
import numpy as np
import pytest
import torch

from latent_compressed_expert_gb300 import synth


def _case(seed=0, n=5, L=16, E=6, K=3, I=8, c=100.0):
    rng = np.random.default_rng(seed)
    lat = rng.standard_normal((n, L))
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(n)]).astype(np.int32)
    gate = rng.uniform(0.1, 0.6, (n, K)).astype(np.float32)
    wg = torch.randn(E, I, L, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    wv = torch.randn(E, I, L, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
    wd = (torch.randn(E, L, I, generator=torch.Generator().manual_seed(seed + 2)) * 0.3).to(torch.bfloat16)
    gamma = rng.uniform(0.5, 1.5, L).astype(np.float32)
    dz = rng.standard_normal((n, L))
    return lat, idx, gate, wg, wv, wd, gamma, dz


@pytest.mark.parametrize("c", [100.0, 2.0])
def test_restated_forward_equals_c_oracle(oracle_mod, c):
    import oracle.backward as B
    lat, idx, gate, wg, wv, wd, gamma, dz = _case(1, c=c)
    z_c = oracle_mod.routed(lat, idx, gate, wg, wv, wd, gamma, c, 1e-6)
    g = B.routed_backward(lat, idx, gate, wg, wv, wd, gamma, dz, c, 1e-6)
    assert np.allclose(g["z"], z_c, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("c", [100.0, 2.0])   # c = 2 puts many pre-activations on the cap
def test_gradients_equal_finite_differences(oracle_mod, c):
    """Central differences of the C oracle's forward (a different implementation from the
    differentiated one), on a few entries of every input."""
    import oracle.backward as B
    lat, idx, gate, wg, wv, wd, gamma, dz = _case(2, c=c)
    g = B.routed_backward(lat, idx, gate, wg, wv, wd, gamma, dz, c, 1e-6)
    wgf, wvf, wdf = (w.double().numpy() for w in (wg, wv, wd))

    def loss(lat_, gate_, gamma_, wg_, wv_, wd_):
        # the C oracle takes bf16 weights: evaluate through the torch re-statement for
        # weight perturbations, and through the C oracle for the others
        return float(np.sum(dz * B.routed_forward_t(
            torch.as_tensor(lat_), idx, torch.as_tensor(gate_.astype(np.float64)),
            torch.as_tensor(wg_), torch.as_tensor(wv_), torch.as_tensor(wd_),
            torch.as_tensor(gamma_.astype(np.float64)), c, 1e-6).numpy()))

    def loss_c(lat_, gate_, gamma_):
        return float(np.sum(dz * oracle_mod.routed(lat_, idx, gate_, wg, wv, wd, gamma_, c, 1e-6)))

    rng = np.random.default_rng(3)
    h = 1e-5
    for _ in range(6):
        t, l = rng.integers(lat.shape[0]), rng.integers(lat.shape[1])
        a, b = lat.copy(), lat.copy()
        a[t, l] += h
        b[t, l] -= h
        fd = (loss_c(a, gate, gamma) - loss_c(b, gate, gamma)) / (2 * h)
        assert fd == pytest.approx(g["dlat"][t, l], rel=1e-5, abs=1e-7)
    for _ in range(4):
        t, j = rng.integers(gate.shape[0]), rng.integers(gate.shape[1])
        a, b = gate.astype(np.float64).copy(), gate.astype(np.float64).copy()
        a[t, j] += h
        b[t, j] -= h
        fd = (loss(lat, a, gamma, wgf, wvf, wdf) - loss(lat, b, gamma, wgf, wvf, wdf)) / (2 * h)
        assert fd == pytest.approx(g["dgate"][t, j], rel=1e-5, abs=1e-7)
    for name, arr, key in (("wg", wgf, "dw_gate"), ("wv", wvf, "dw_value"), ("wd", wdf, "dw_edown")):
        for _ in range(4):
            ix = tuple(rng.integers(s) for s in arr.shape)
            a, b = arr.copy(), arr.copy()
            a[ix] += h
            b[ix] -= h
            args_a = {"wg": wgf, "wv": wvf, "wd": wdf}
            args_b = dict(args_a)
            args_a[name], args_b[name] = a, b
            fd = (loss(lat, gate, gamma, args_a["wg"], args_a["wv"], args_a["wd"]) -
                  loss(lat, gate, gamma, args_b["wg"], args_b["wv"], args_b["wd"])) / (2 * h)
            assert fd == pytest.approx(g[key][ix], rel=1e-5, abs=1e-7), name
    l = rng.integers(len(gamma))
    a, b = gamma.astype(np.float64).copy(), gamma.astype(np.float64).copy()
    a[l] += h
    b[l] -= h
    # (gamma enters the C oracle as fp32, which would round the perturbation away)
    fd = (loss(lat, gate, a, wgf, wvf, wdf) - loss(lat, gate, b, wgf, wvf, wdf)) / (2 * h)
    assert fd == pytest.approx(g["dgamma"][l], rel=1e-5, abs=1e-7)


# --- the whole layer (layer_backward) ---------------------------------------------------

def _layer_case(S, seed=5, T=7):
    sh = synth.LayerShape("tiny_bwd", T=T, d=48, L=32, E=8, K=3, I=16, S=S, Is=16 if S else 0)
    w = synth.make_weights(sh, seed=seed)
    w["gamma"] = torch.linspace(0.6, 1.4, sh.L)
    x = synth.make_x(sh, seed=seed + 1)
    return sh, w, x


@pytest.mark.parametrize("S", [2, 0])
def test_layer_restatement_equals_c_oracle(oracle_mod, S):
    """With the C oracle's routing and fp32 gates the restated layer reproduces its output,
    latent and logits; the restatement's own fp64 gates match route's fp32 gates to within
    the fp32 sigmoid's error."""
    import oracle.backward as B
    sh, w, x = _layer_case(S)
    r = oracle_mod.forward(w, x, sh.K, residual=None, tau="batch")
    w64 = {k: B._f64(v) for k, v in w.items()}
    x64 = B._f64(x)
    y, parts = B.layer_forward_t(x64, r.idx, w64, gate=torch.as_tensor(r.gate.astype(np.float64)))
    rms = float(np.sqrt(np.mean(r.y ** 2)))
    assert np.allclose(y.numpy(), r.y, rtol=1e-10, atol=1e-10 * rms)
    assert np.allclose(parts["lat"].numpy(), r.lat, rtol=1e-12, atol=1e-12)
    lg = parts["logits"].numpy()
    assert np.all(np.abs(lg - r.logits) <= 2.0 ** -24 * np.abs(lg) + 1e-30)
    _, own = B.layer_forward_t(x64, r.idx, w64)
    assert np.allclose(own["gate"].numpy(), r.gate, rtol=2e-6, atol=0)


@pytest.mark.parametrize("S,c", [(2, 100.0), (2, 2.0), (0, 100.0)])
def test_layer_gradients_equal_finite_differences(S, c):
    """Central differences of the restated layer (routing held fixed) on a few entries of x,
    gamma and every weight."""
    import oracle.backward as B
    sh, w, x = _layer_case(S, seed=11)
    rng = np.random.default_rng(12)
    idx = np.stack([rng.choice(sh.E, sh.K, replace=False) for _ in range(sh.T)]).astype(np.int32)
    dy = rng.standard_normal((sh.T, sh.d))
    g = B.layer_backward(x, idx, w, dy, c=c)
    base = {k: B._f64(v) for k, v in w.items()}
    base["x"] = B._f64(x)
    key = {"x": "dx", "gamma": "dgamma"}

    def loss(vals):
        wd = {k: v for k, v in vals.items() if k != "x"}
        y, _ = B.layer_forward_t(vals["x"], idx, wd, c=c)
        return float(torch.sum(torch.as_tensor(dy) * y))

    h = 1e-6
    names = ["x", "gamma"] + [n for n in B.LAYER_WEIGHTS if base[n].numel() > 0]
    for name in names:
        for _ in range(3):
            ix = tuple(int(rng.integers(s)) for s in base[name].shape)
            a, b = dict(base), dict(base)
            a[name] = base[name].clone()
            b[name] = base[name].clone()
            a[name][ix] += h
            b[name][ix] -= h
            fd = (loss(a) - loss(b)) / (2 * h)
            assert fd == pytest.approx(g[key.get(name, "d" + name)][ix], rel=1e-5, abs=1e-7), name


def test_layer_dx_rows_equals_whole_batch():
    """Token by token, with each token's experts' weights only, the restatement gives the
    whole batch's dx (a token's gradient depends on that token alone given the routing)."""
    import oracle.backward as B
    sh, w, x = _layer_case(2, seed=21, T=6)
    rng = np.random.default_rng(22)
    idx = np.stack([rng.choice(sh.E, sh.K, replace=False) for _ in range(sh.T)]).astype(np.int32)
    dy = rng.standard_normal((sh.T, sh.d))
    whole = B.layer_backward(x, idx, w, dy)["dx"]
    rows = np.array([0, 3, 5])
    part = B.layer_dx_rows(x[rows], idx[rows], w, dy[rows])
    assert np.allclose(part, whole[rows], rtol=1e-11, atol=1e-13)
