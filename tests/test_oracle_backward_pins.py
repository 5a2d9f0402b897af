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
