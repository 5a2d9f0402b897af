"""Pins of the CPU oracle to facts fixed outside itself: closed forms, library routines on
special cases, brute force on tiny inputs, and invariants of the layer's definition.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a wrong sign,
index or transposed operand) fails at least one of them.  CPU only.
"""
import math

import numpy as np
import pytest
import torch

from latent_compressed_expert_gb300 import synth


# ----------------------------------------------------------------------------------------
# Router score (fp32 sigmoid, specified bit for bit)
# ----------------------------------------------------------------------------------------

def _sig64(z):
    z = np.clip(np.asarray(z, dtype=np.float64), -88.0, 88.0)
    return 1.0 / (1.0 + np.exp(-z))


def test_sigmoid_accuracy_against_libm(oracle_mod):
    """Within 3 fp32 ulps of the logistic function computed with libm in double, over a
    dense sample of [-90, 90] (the method rounds three times: exp to about 1 ulp, then
    1 + e, then the division); a wrong polynomial coefficient, range-reduction constant or
    scaling step breaks this by orders of magnitude."""
    rng = np.random.default_rng(0)
    z = np.concatenate([np.linspace(-90, 90, 400_001), rng.uniform(-90, 90, 200_000),
                        rng.normal(0, 3, 200_000)]).astype(np.float32)
    s = oracle_mod.scores(z)
    ref = _sig64(z.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(s.astype(np.float64) - ref) / ulp
    assert err.max() <= 3.0, (err.max(), z[np.argmax(err)])


def test_sigmoid_special_values(oracle_mod):
    sig = oracle_mod.sigmoid32
    assert sig(0.0) == 0.5
    assert sig(88.0) == 1.0 and sig(1e30) == 1.0 and sig(float("inf")) == 1.0
    assert sig(20.0) == 1.0  # exp(-20) < 2^-24: rounds to exactly 1
    lo = sig(-88.0)
    assert lo == sig(-1e30) == sig(float("-inf"))
    assert 0.0 < lo < 1.2e-38  # subnormal, about e^-88
    assert abs(lo - math.exp(-88.0)) <= 2 * 2.0 ** -149


def test_sigmoid_symmetry_and_monotone(oracle_mod):
    """s(z) + s(-z) = 1 up to rounding, and s is non-decreasing over dense runs of
    consecutive fp32 values (including the points where the range reduction switches n)."""
    z = np.linspace(-30, 30, 100_001).astype(np.float32)
    s1 = oracle_mod.scores(z).astype(np.float64)
    s2 = oracle_mod.scores(-z).astype(np.float64)
    assert np.abs(s1 + s2 - 1.0).max() <= 2 * 2.0 ** -24
    for centre in (0.0, 0.3465736, 1.0397208, -1.0397208, 5.5451775, -60.65, 17.0):
        base = np.float32(centre).view(np.int32)
        bits = np.arange(-200_000, 200_000, dtype=np.int64) + int(base)
        zz = bits.astype(np.int32).view(np.float32)
        zz = np.sort(zz[np.isfinite(zz)])
        ss = oracle_mod.scores(zz)
        assert np.all(np.diff(ss.astype(np.float64)) >= 0.0), centre


def test_sigmoid_is_monotone_up_to_one_ulp_over_all_fp32(oracle_mod):
    """Every fp32 input in [-88, 88], in increasing order (2.24e9 values; outside the clamp
    the score is constant).  The score never steps down by more than one ulp, and it does
    step down by one ulp in a few hundred places (the roundings of the polynomial and the
    division): a selection by score is not a selection by logit, which is why thresholds,
    candidates and top-K all compare the scores themselves."""
    one, more = oracle_mod.sigmoid_decreases()
    assert more == 0
    assert 0 < one < 10_000, one


# ----------------------------------------------------------------------------------------
# Quantile-Balancing thresholds
# ----------------------------------------------------------------------------------------

def test_fair_share_rank(oracle_mod):
    r = oracle_mod.fair_share_rank
    assert r(8192, 16, 896) == 146      # 8192*16/896 = 146.29
    assert r(32768, 16, 896) == 585     # 585.14
    assert r(4096, 4, 64) == 256
    assert r(64, 4, 16) == 16
    assert r(64, 16, 896) == 1          # floor would be 1
    assert r(10, 1, 896) == 1           # clamped up to 1
    assert r(3, 16, 16) == 3            # clamped down to T
    assert r(0, 16, 896) == 0


@pytest.mark.parametrize("T,E,k", [(64, 16, 16), (257, 33, 5), (100, 7, 100), (50, 9, 1)])
def test_thresholds_brute_force(oracle_mod, T, E, k):
    """tau[e] is the k-th largest score of column e: compare with Python's sorted() on each
    column, and check the counting property that defines a k-th largest value."""
    lg = synth.make_uniform_logits(T, E, seed=T + E, quantum=0.25).numpy()
    tau = oracle_mod.thresholds(lg, k)
    s = oracle_mod.scores(lg)
    for e in range(E):
        col = sorted((float(v) for v in s[:, e]), reverse=True)
        assert tau[e] == np.float32(col[k - 1])
        assert (s[:, e] >= tau[e]).sum() >= k
        assert (s[:, e] > tau[e]).sum() < k


# ----------------------------------------------------------------------------------------
# Top-K routing
# ----------------------------------------------------------------------------------------

def _route_brute(s, tau, K):
    T, E = s.shape
    idx = np.empty((T, K), np.int32)
    gate = np.empty((T, K), np.float32)
    for t in range(T):
        a = [(float(np.float32(s[t, e] - (tau[e] if tau is not None else 0.0))), e)
             for e in range(E)]
        order = sorted(a, key=lambda p: (-p[0], p[1]))[:K]
        tot = np.float32(0.0)
        for _, e in order:
            tot = np.float32(tot + s[t, e])
        for j, (_, e) in enumerate(order):
            idx[t, j] = e
            gate[t, j] = np.float32(s[t, e] / tot)
    return idx, gate


@pytest.mark.parametrize("T,E,K,quantum", [(64, 16, 4, None), (97, 33, 7, 0.5),
                                           (40, 16, 16, None), (30, 64, 1, 0.125)])
def test_route_brute_force(oracle_mod, T, E, K, quantum):
    """Selection and gates equal a full Python sort by (a descending, expert ascending),
    bit for bit, with balancing thresholds from the same batch and without."""
    lg = synth.make_uniform_logits(T, E, seed=7 * T + E, quantum=quantum).numpy()
    s = oracle_mod.scores(lg)
    tau = oracle_mod.thresholds(lg, oracle_mod.fair_share_rank(T, K, E))
    for t_ in (tau, None):
        idx, gate, sc = oracle_mod.route(lg, t_, K)
        assert np.array_equal(sc, s)
        bi, bg = _route_brute(s, t_, K)
        assert np.array_equal(idx, bi)
        assert np.array_equal(gate.view(np.int32), bg.view(np.int32))


def test_route_plain_topk_is_stable_argsort(oracle_mod):
    """Without thresholds the selection is numpy's stable argsort of -s (ties to the lower
    expert id), truncated to K."""
    lg = synth.make_uniform_logits(200, 50, seed=3, quantum=0.5).numpy()
    s = oracle_mod.scores(lg)
    idx, _, _ = oracle_mod.route(lg, None, 6)
    ref = np.argsort(-s, axis=1, kind="stable")[:, :6]
    assert np.array_equal(idx, ref)


def test_route_selection_count_and_ratio(oracle_mod):
    """Each token gets exactly K distinct experts (16 of 896: about 1.8 % of the pool), and
    the gates of a token sum to 1 and keep the ratios of the scores."""
    T, E, K = 256, 896, 16
    lg = synth.make_logits(T, E, seed=1).numpy()
    tau = oracle_mod.thresholds(lg, oracle_mod.fair_share_rank(T, K, E))
    idx, gate, s = oracle_mod.route(lg, tau, K)
    assert all(len(set(r)) == K for r in idx.tolist())
    assert idx.min() >= 0 and idx.max() < E
    assert round(100.0 * K / E, 1) == 1.8
    assert idx.size == T * K
    assert np.allclose(gate.sum(1), 1.0, atol=4e-7 * K)
    ratio = gate[:, :1] / gate
    sref = np.take_along_axis(s, idx, 1)
    assert np.allclose(ratio, sref[:, :1] / sref, rtol=1e-6)


def test_route_saturated_ties(oracle_mod):
    """Scores that saturate to exactly 1.0 tie; the lower expert ids win."""
    lg = np.full((3, 10), 30.0, np.float32)
    lg[1, 5:] = 40.0
    lg[2, :] = -5.0
    lg[2, 7] = 25.0
    idx, gate, s = oracle_mod.route(lg, None, 3)
    assert np.all(s[:2] == 1.0)
    assert idx[0].tolist() == [0, 1, 2]
    assert idx[1].tolist() == [0, 1, 2]
    assert idx[2].tolist() == [7, 0, 1]
    assert np.all(gate[0] == np.float32(1.0 / 3.0))


def test_quantile_balancing_caps_loads(oracle_mod):
    """With thresholds from the batch, a skewed router's per-expert load falls toward the
    fair share T*K/E; without them a Zipf-biased router overloads its favourites."""
    T, E, K = 2048, 128, 8
    lg = synth.make_logits(T, E, seed=4, zipf_s=1.1).numpy()
    k = oracle_mod.fair_share_rank(T, K, E)
    tau = oracle_mod.thresholds(lg, k)
    plain, _, _ = oracle_mod.route(lg, None, K)
    bal, _, _ = oracle_mod.route(lg, tau, K)
    lp = np.bincount(plain.ravel(), minlength=E)
    lb = np.bincount(bal.ravel(), minlength=E)
    fair = T * K / E
    assert lp.max() / fair > 4.0
    assert lb.max() / fair < 1.6
    assert (lb == 0).sum() == 0


# ----------------------------------------------------------------------------------------
# SiTU-GLU
# ----------------------------------------------------------------------------------------

def _silu(x):
    return torch.nn.functional.silu(torch.as_tensor(x, dtype=torch.float64)).numpy()


def test_situ_reduces_to_swiglu_without_cap(oracle_mod):
    """As the cap c grows without bound SiTU-GLU is SwiGLU: silu(g) * v (torch's silu)."""
    rng = np.random.default_rng(1)
    g, v = rng.normal(0, 5, 10_000), rng.normal(0, 5, 10_000)
    got = oracle_mod.situ(g, v, c=1e9)
    ref = _silu(g) * v
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_situ_taylor_bound_near_zero(oracle_mod):
    """c tanh(x/c) differs from x by at most |x|^3/(3c^2); hence SiTU-GLU differs from
    SwiGLU by at most (|silu g| |v|^3 + 1.1 |v| |g|^3) / (3 c^2), which is below 1e-6 for
    |g|, |v| <= 0.3 and c = 100."""
    c = 100.0
    x = np.linspace(-3.0, 3.0, 241)
    g, v = [a.ravel() for a in np.meshgrid(x, x)]
    got = oracle_mod.situ(g, v, c)
    sw = _silu(g) * v
    bound = (np.abs(_silu(g)) * np.abs(v) ** 3 + 1.1 * np.abs(v) * np.abs(g) ** 3) / (3 * c * c)
    assert np.all(np.abs(got - sw) <= bound + 1e-15)
    small = (np.abs(g) <= 0.3) & (np.abs(v) <= 0.3)
    assert np.abs(got - sw)[small].max() < 1e-6
    # and the difference is not zero: the cap is active, with the sign of a tanh shrink
    assert np.abs(got - sw)[~small].max() > 1e-5


def test_situ_caps_both_branches(oracle_mod):
    """Both branches saturate near +-c: |out| <= c^2 (equality only once exp(-c) is lost
    to rounding), silu of the capped gate stays in
    (-0.2785, c), the output is odd in v, and huge inputs give about +-c^2."""
    c = 100.0
    rng = np.random.default_rng(2)
    g = rng.normal(0, 1e4, 20_000)
    v = rng.normal(0, 1e4, 20_000)
    out = oracle_mod.situ(g, v, c)
    assert np.all(np.abs(out) <= c * c)
    vc = c * np.tanh(np.clip(v, -1e3, 1e3) / c)
    with np.errstate(divide="ignore", invalid="ignore"):
        sg = np.where(np.abs(vc) > 1e-3, out / vc, np.nan)
    sg = sg[np.isfinite(sg)]
    assert sg.min() > -0.2785 and sg.max() <= c * (1 + 1e-8)
    assert np.allclose(oracle_mod.situ(g, -v, c), -out)
    big = oracle_mod.situ(np.array([1e6, -1e6, 1e6]), np.array([1e6, 1e6, -1e6]), c)
    silu_c = c / (1 + math.exp(-c))
    assert np.allclose(big, [silu_c * c, -c * math.exp(-c) * c / (1 + math.exp(-c)), -silu_c * c],
                       rtol=1e-12, atol=1e-30)


# ----------------------------------------------------------------------------------------
# Dense steps against a library matmul
# ----------------------------------------------------------------------------------------

def _f64(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def test_latent_router_output_against_numpy(oracle_mod):
    sh = synth.TINY
    w = synth.make_weights(sh, seed=11)
    x = synth.make_x(sh, seed=11, T=9)
    lat = oracle_mod.latent(x, w["w_down"])
    ref = _f64(x) @ _f64(w["w_down"]).T
    assert np.allclose(lat, ref, rtol=1e-12, atol=1e-12)
    lg = oracle_mod.router_logits(lat, w["w_router"])
    assert np.allclose(lg, ref @ _f64(w["w_router"]).T, rtol=1e-12, atol=1e-12)
    rng = np.random.default_rng(0)
    z = rng.normal(size=(9, sh.L))
    ys = rng.normal(size=(9, sh.d))
    y = oracle_mod.output(z, ys, w["w_up"], residual=x)
    assert np.allclose(y, _f64(x) + z @ _f64(w["w_up"]).T + ys, rtol=1e-12, atol=1e-12)
    y0 = oracle_mod.output(z, ys, w["w_up"], residual=None)
    assert np.allclose(y0, z @ _f64(w["w_up"]).T + ys, rtol=1e-12, atol=1e-12)


def test_shared_experts_are_swiglu_ffns_without_cap(oracle_mod):
    """With the cap lifted, the shared path is the sum over the two shared experts of a
    SwiGLU FFN (torch matmul + silu), each at the full hidden width."""
    sh = synth.TINY
    w = synth.make_weights(sh, seed=12)
    x = synth.make_x(sh, seed=12, T=7)
    got = oracle_mod.shared(x, w["w_sgate"], w["w_svalue"], w["w_sdown"], c=1e9)
    xt = x.double()
    ref = torch.zeros(7, sh.d, dtype=torch.float64)
    for s in range(sh.S):
        hg = xt @ w["w_sgate"][s].double().T
        hv = xt @ w["w_svalue"][s].double().T
        ref += (torch.nn.functional.silu(hg) * hv) @ w["w_sdown"][s].double().T
    assert np.allclose(got, ref.numpy(), rtol=1e-10, atol=1e-10)


# ----------------------------------------------------------------------------------------
# Routed path: brute force with masked gates, and invariants
# ----------------------------------------------------------------------------------------

def _dense_masked(oracle_mod, lat, idx, gate, w, c=100.0, eps=1e-6):
    """Evaluate every expert on every token densely (library matmuls) and mix them with a
    gate matrix that is zero outside the selected experts."""
    n, L = lat.shape
    E = w["w_gate"].shape[0]
    G = np.zeros((n, E))
    for t in range(n):
        for j in range(idx.shape[1]):
            G[t, idx[t, j]] += float(gate[t, j])
    u = np.zeros((n, L))
    for e in range(E):
        hg = lat @ _f64(w["w_gate"][e]).T
        hv = lat @ _f64(w["w_value"][e]).T
        h = oracle_mod.situ(hg, hv, c)
        u += G[:, e:e + 1] * (h @ _f64(w["w_edown"][e]).T)
    ms = (u * u).mean(1, keepdims=True)
    return _f64(w["gamma"])[None, :] * u / np.sqrt(ms + eps)


def test_routed_equals_dense_masked_mixture(oracle_mod):
    """I1: the gathered routed path equals a dense evaluation of all experts with the gates
    masked to the selected ones (tiny shape, hot rows that hit the cap, random gamma)."""
    sh = synth.TINY
    w = synth.make_weights(sh, seed=13, hot_row_frac=0.01)
    w["gamma"] = torch.rand(sh.L, generator=torch.Generator().manual_seed(5)) + 0.5
    x = synth.make_x(sh, seed=13)
    r = oracle_mod.forward(w, x, sh.K, residual=x)
    ref = _dense_masked(oracle_mod, r.lat, r.idx, r.gate, w)
    assert np.allclose(r.z, ref, rtol=1e-10, atol=1e-10)
    # the hot rows really do push pre-activations past the cap
    hg = np.concatenate([r.lat @ _f64(w["w_gate"][e]).T for e in range(sh.E)], 1)
    assert np.abs(hg).max() > 300.0


def test_rmsnorm_unit_rms_and_gate_scale_invariance(oracle_mod):
    """RMSNorm output has RMS sqrt(ms/(ms+eps)) before gamma; scaling every gate by alpha
    changes the output only through eps (I3)."""
    sh = synth.TINY
    w = synth.make_weights(sh, seed=14)
    x = synth.make_x(sh, seed=14, T=16)
    r = oracle_mod.forward(w, x, sh.K)
    rms = np.sqrt((r.z ** 2).mean(1))
    assert np.all(np.abs(rms - 1.0) < 1e-4)
    z2 = oracle_mod.routed(r.lat, r.idx, r.gate * np.float32(3.0), w["w_gate"], w["w_value"],
                           w["w_edown"], w["gamma"].numpy())
    assert np.allclose(z2, r.z, rtol=1e-5, atol=1e-5)
    z3 = oracle_mod.routed(r.lat, r.idx, r.gate, w["w_gate"], w["w_value"], w["w_edown"],
                           w["gamma"].numpy(), eps=0.0)
    assert np.allclose(np.sqrt((z3 ** 2).mean(1)), 1.0, rtol=1e-12)


def test_zero_routed_output_leaves_residual_plus_shared(oracle_mod):
    """I2: with every routed down-projection zero the aggregated latent is zero, RMSNorm
    maps it to zero (eps > 0), and the layer is residual + shared experts."""
    sh = synth.TINY
    w = synth.make_weights(sh, seed=15)
    w["w_edown"] = torch.zeros_like(w["w_edown"])
    x = synth.make_x(sh, seed=15, T=12)
    r = oracle_mod.forward(w, x, sh.K, residual=x)
    assert np.all(r.z == 0.0)
    assert np.allclose(r.y, _f64(x) + r.ys, rtol=0, atol=1e-12)


def test_expert_permutation_invariance(oracle_mod):
    """I4: relabelling the experts (weights and router rows together) leaves the layer's
    output unchanged wherever the selection has no exact tie at the K-th place.  Under
    in-batch balancing such ties are structural: each expert's k-th ranked token sits at
    a = 0 exactly, so a token can tie for several experts; there the lower id wins and a
    relabelling may change the pick.  Both cases are checked."""
    sh = synth.TINY
    w = synth.make_weights(sh, seed=16)
    x = synth.make_x(sh, seed=16)
    perm = torch.randperm(sh.E, generator=torch.Generator().manual_seed(3))
    w2 = dict(w)
    for k in ("w_router", "w_gate", "w_value", "w_edown"):
        w2[k] = w[k][perm].contiguous()
    for tau in (None, "batch"):
        r = oracle_mod.forward(w, x, sh.K, residual=x, tau=tau)
        r2 = oracle_mod.forward(w2, x, sh.K, residual=x, tau=tau)
        s = oracle_mod.scores(r.logits)
        a = s - (r.tau if r.tau is not None else 0.0)
        srt = -np.sort(-a, axis=1)
        clean = srt[:, sh.K - 1] != srt[:, sh.K]
        assert clean.sum() >= sh.T // 2
        assert np.array_equal(perm.numpy()[r2.idx][clean], r.idx[clean])
        assert np.allclose(r2.y[clean], r.y[clean], rtol=1e-12, atol=1e-12)
        if tau is None:
            assert clean.all()


def test_token_permutation_equivariance(oracle_mod):
    """I5: permuting the tokens permutes the output rows; in-batch thresholds do not
    change."""
    sh = synth.TINY
    w = synth.make_weights(sh, seed=17)
    x = synth.make_x(sh, seed=17)
    r = oracle_mod.forward(w, x, sh.K, residual=x)
    perm = torch.randperm(sh.T, generator=torch.Generator().manual_seed(4))
    xp = x[perm].contiguous()
    r2 = oracle_mod.forward(w, xp, sh.K, residual=xp)
    assert np.array_equal(r2.tau, r.tau)
    assert np.allclose(r2.y, r.y[perm.numpy()], rtol=1e-12, atol=1e-12)


def test_all_experts_without_balancing_is_dense_moe(oracle_mod):
    """I6: K = E without thresholds is the dense mixture of all experts with gates
    s / sum(s)."""
    sh = synth.TINY
    w = synth.make_weights(sh, seed=18)
    x = synth.make_x(sh, seed=18, T=10)
    r = oracle_mod.forward(w, x, sh.E, residual=None, tau=None)
    s = oracle_mod.scores(r.logits).astype(np.float64)
    G = s / s.sum(1, keepdims=True)
    idx_all = np.tile(np.arange(sh.E, dtype=np.int32), (10, 1))
    ref = _dense_masked(oracle_mod, r.lat, idx_all, G.astype(np.float32), w)
    assert np.allclose(r.z, ref, rtol=1e-6, atol=1e-6)
    assert sorted(r.idx[0].tolist()) == list(range(sh.E))


# ----------------------------------------------------------------------------------------
# streaming thresholds and load statistics
# ----------------------------------------------------------------------------------------
def test_tau_ema_limits_and_convergence(oracle_mod):
    rng = np.random.default_rng(7)
    a = rng.uniform(0.3, 0.9, 50).astype(np.float32)
    b = rng.uniform(0.3, 0.9, 50).astype(np.float32)
    assert np.array_equal(oracle_mod.tau_ema(a, b, 0.0), b)             # beta 0: this step
    assert np.array_equal(oracle_mod.tau_ema(a, b, 1.0), a)             # beta 1: frozen
    assert np.array_equal(oracle_mod.tau_ema(a, b, 0.9, first=True), b)  # initialisation
    # a constant step threshold is approached geometrically: |t_n - b| <= beta^n |t_0 - b|
    t = a.copy()
    for n in range(1, 40):
        t = oracle_mod.tau_ema(t, b, 0.75)
        bound = 0.75 ** n * np.abs(a.astype(np.float64) - b) + n * 2.0 ** -24
        assert np.all(np.abs(t.astype(np.float64) - b) <= bound)
    # between the two: a convex combination
    m = oracle_mod.tau_ema(a, b, 0.3).astype(np.float64)
    assert np.all(m >= np.minimum(a, b) - 1e-7) and np.all(m <= np.maximum(a, b) + 1e-7)


def test_load_stats_accumulate_counts(oracle_mod):
    rng = np.random.default_rng(8)
    E = 16
    steps = [rng.integers(0, 20, E) for _ in range(5)]
    steps[2][3] = 0
    acc = None
    for c in steps:
        acc = oracle_mod.load_stats_update(acc, c)
    S = np.array(steps, dtype=np.int64)
    assert acc[0] == 5 and acc[1] == S.sum() and acc[2] == S.max(1).sum() and acc[3] == S.max()
    assert np.array_equal(acc[4:4 + E], S.sum(0))
    assert np.array_equal(acc[4 + E:4 + 2 * E], (S * S).sum(0))
    assert np.array_equal(acc[4 + 2 * E:4 + 3 * E], (S == 0).sum(0))
    assert np.array_equal(acc[4 + 3 * E:], S.max(0))
    # invariants: pairs are conserved, the per-step maximum bounds the mean, and the largest
    # count of any expert is the largest per-expert maximum
    assert acc[4:4 + E].sum() == acc[1]
    assert acc[3] * acc[0] >= acc[2] and acc[3] == acc[4 + 3 * E:].max()
    assert np.all(acc[4 + E:4 + 2 * E] * acc[0] >= acc[4:4 + E] ** 2)  # Cauchy-Schwarz


# ----------------------------------------------------------------------------------------
# expert-parallel dispatch and combine
# ----------------------------------------------------------------------------------------
def _ep_case(seed, T=40, K=6, E=48):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    return rng, idx


@pytest.mark.parametrize("R", [1, 4, 8, 48])
def test_ep_dispatch_pairs(oracle_mod, R):
    rng, idx = _ep_case(11)
    T, K = idx.shape
    E = 48
    rows = torch.randn(T, 16).to(torch.bfloat16)
    d = oracle_mod.ep_dispatch(idx, E, R, rows)
    per = E // R
    ranks = idx // per
    # one pair per (token, distinct rank), in (rank, token) order
    assert d["P"] == sum(len(set(ranks[t])) for t in range(T))
    keys = [(int(r), int(t)) for r in range(R) for t in range(T) if r in set(ranks[t])]
    got = [(r, int(t)) for r in range(R) for t in d["send_tok"][d["send_off"][r]:d["send_off"][r + 1]]]
    assert got == keys
    # every slot of every token goes to exactly one pair, the one of its expert's rank
    seen = np.zeros((T, K), dtype=int)
    for r in range(R):
        for p in range(d["send_off"][r], d["send_off"][r + 1]):
            t, sl = d["send_tok"][p], int(d["send_slots"][p])
            for j in range(K):
                if sl >> j & 1:
                    assert ranks[t, j] == r
                    seen[t, j] += 1
    assert np.all(seen == 1)
    # rows are copies of the token's row
    assert np.array_equal(d["send_rows"], rows.view(torch.int16).numpy().view(np.uint16)[d["send_tok"]])
    if R == 1:
        assert d["P"] == T
    if R == E:
        assert d["P"] == T * K


def test_ep_combine_sums_to_the_gated_mixture(oracle_mod):
    """Summed over ranks, the returned rows give sum_j gate_j o_j: exactly so with one rank
    (one fma chain over all slots, then one bf16 rounding), and within the bf16 rounding of
    each rank's partial otherwise."""
    rng, idx = _ep_case(12)
    T, K = idx.shape
    E, W = 48, 24
    gate = rng.uniform(0.05, 0.3, (T, K)).astype(np.float32)
    inv = rng.permutation(T * K).reshape(T, K).astype(np.int32)
    o = torch.randn(T * K, W).to(torch.bfloat16)
    of = o.float().numpy().astype(np.float64)
    exact = np.einsum("tk,tkw->tw", gate.astype(np.float64), of[inv])
    for R in (1, 4, 48):
        d = oracle_mod.ep_dispatch(idx, E, R)
        part, u = oracle_mod.ep_combine(d, inv, gate, o, T)
        pf = (part.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        bound = np.zeros((T, W))
        for p in range(d["P"]):
            bound[d["send_tok"][p]] += np.abs(pf[p]) * 2.0 ** -8 + 1e-6
        assert np.all(np.abs(u - exact) <= bound + 1e-5 * np.abs(exact)), R
        if R == 1:
            assert np.array_equal(u, pf.astype(np.float32))
