"""Thresholds over a batch spread across ranks, on one GPU.

Quantile Balancing reads each expert's threshold off the scores of the whole step's batch
("Part 1 of Inside Kimi K3", Quantile Balancing passage).  When the batch is split over
ranks, each part contributes its k largest scores per expert (lmoe_threshold_candidates),
the parts' candidates are stacked (the all-gather), and lmoe_thresholds on the stack gives
the threshold of the whole batch.  Checked here:
  - the candidates against a brute-force selection on the oracle's scores (bit-exact),
    including ties, saturated scores, parts smaller than k and an empty part;
  - thresholds from stacked candidates against the oracle's thresholds of the whole batch
    (bit-exact) for several splits;
  - the layer's two phases (router, then experts) against the one-call layer, and the
    parts of a split batch against the whole batch, token for token, bit for bit.
"""
import numpy as np
import pytest
import torch

import gpu_helpers as H
from latent_compressed_expert_gb300 import lmoe, synth

pytestmark = pytest.mark.gpu

FLT_MAX_BITS = np.float32(-np.finfo(np.float32).max).view(np.int32)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from latent_compressed_expert_gb300 import build
    build.build()
    lmoe.load()
    return torch.device("cuda:0")


def _logits(T, E, kind, seed):
    if kind == "normal":
        return synth.make_logits(T, E, seed)
    if kind == "ties":
        return synth.make_uniform_logits(T, E, seed, quantum=0.25)
    if kind == "saturated":
        return synth.make_logits(T, E, seed, scale=30.0)
    raise ValueError(kind)


def _expected_candidates(oracle_mod, lg: np.ndarray, k: int) -> np.ndarray:
    """Per column: the logits of the min(k, T) largest scores (scores above the min(k,T)-th
    largest first, then tokens equal to it, each in token order), then -FLT_MAX."""
    T, E = lg.shape
    out = np.full((k, E), -np.finfo(np.float32).max, dtype=np.float32)
    if T == 0:
        return out
    s = oracle_mod.scores(lg)
    kk = min(k, T)
    for e in range(E):
        col = s[:, e]
        order = sorted(range(T), key=lambda t: (-float(col[t]), t))
        v = col[order[kk - 1]]
        gt = [t for t in range(T) if col[t] > v]
        eq = [t for t in range(T) if col[t] == v][: kk - len(gt)]
        out[:kk, e] = lg[gt + eq, e]
    return out


@pytest.mark.parametrize("T,E,k,kind", [
    (3000, 64, 146, "normal"), (1000, 64, 146, "ties"), (500, 96, 146, "saturated"),
    (50, 32, 146, "normal"),            # fewer tokens than k: padding rows
    (146, 16, 146, "ties"),             # exactly k tokens
    (1, 16, 4, "normal"), (0, 16, 8, "normal"),
    (40000, 16, 300, "ties"),           # column too long to stage in shared memory
])
def test_candidates_bit_exact(dev, oracle_mod, T, E, k, kind):
    lg = _logits(T, E, kind, seed=T + 7 * E + k)
    cand = lmoe.threshold_candidates(lg.to(dev), k)
    ref = _expected_candidates(oracle_mod, lg.numpy(), k)
    got = cand.cpu().numpy()
    assert np.array_equal(got.view(np.int32), ref.view(np.int32))
    if T < k:
        assert np.all(got[T:].view(np.int32) == FLT_MAX_BITS)


SPLITS = [[8192], [3000, 5192], [50, 4000, 4142], [2048, 2048, 2048, 2048], [0, 8192]]


@pytest.mark.parametrize("kind", ["normal", "ties", "saturated"])
def test_thresholds_from_stacked_candidates(dev, oracle_mod, kind):
    T, E, K = 8192, 896, 16
    lg = _logits(T, E, kind, seed=11)
    k = oracle_mod.fair_share_rank(T, K, E)
    ref = oracle_mod.thresholds(lg.numpy(), k)
    lgd = lg.to(dev)
    for split in SPLITS:
        parts, t0 = [], 0
        for n in split:
            parts.append(lmoe.threshold_candidates(lgd[t0:t0 + n].contiguous(), k))
            t0 += n
        tau = lmoe.thresholds(torch.cat(parts, 0), K, k_rank=k)
        assert np.array_equal(tau.cpu().numpy().view(np.int32), ref.view(np.int32)), split


def _mid_layer(dev, max_tokens=None):
    sh = H.mid_shape()
    w = synth.make_weights(sh, seed=21, device="cpu")
    wd = {k: v.to(dev) for k, v in w.items()}
    return sh, wd


def test_two_phases_equal_one_call(dev):
    sh, wd = _mid_layer(dev)
    layer = lmoe.Layer(sh, wd)
    x = synth.make_x(sh, seed=22).to(dev)
    y_all, d_all = layer.forward(x, residual=x, debug=True)
    y_all = y_all.clone()
    assert layer.last_kernel_launches == 12
    # router phase, then experts phase solving the in-batch thresholds itself
    assert layer.forward(x, phase=lmoe.PHASE_ROUTER) is None
    assert layer.last_kernel_launches == 2
    y2, d2 = layer.forward(x, residual=x, phase=lmoe.PHASE_EXPERTS, debug=True)
    assert layer.last_kernel_launches == 10     # + the router scores (both layouts)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    for key in ("logits", "tau", "idx", "gate", "counts"):
        assert torch.equal(d_all[key], d2[key]), key
    assert torch.equal(y_all.view(torch.int16), y2.view(torch.int16))
    # one rank: the global path reduces to the in-batch thresholds
    y3 = layer.forward_global(x, residual=x)
    torch.cuda.synchronize()
    assert torch.equal(y_all.view(torch.int16), y3.view(torch.int16))


@pytest.mark.parametrize("split", [[400, 600], [1, 333, 666]])
def test_split_batch_matches_whole_batch(dev, split):
    """Each part runs on its own workspace, as a rank would; the stacked candidates give
    the whole batch's thresholds, and every token's routing and output equal the one-call
    layer on the whole batch."""
    sh, wd = _mid_layer(dev)
    T = sum(split)
    whole = lmoe.Layer(sh, wd, max_tokens=T)
    x = synth.make_x(sh, seed=23, T=T).to(dev)
    y_all, d_all = whole.forward(x, residual=x, debug=True)
    k = lmoe.fair_share_rank(T, sh.K, sh.E)
    ranks, cands, t0 = [], [], 0
    for n in split:
        r = lmoe.Layer(sh, wd, max_tokens=n)
        xs = x[t0:t0 + n].contiguous()
        cands.append(r.forward(xs, phase=lmoe.PHASE_ROUTER, cand_k=k))
        assert r.last_kernel_launches == 3
        ranks.append((r, xs, t0))
        t0 += n
    tau = lmoe.thresholds(torch.cat(cands, 0), sh.K, k_rank=k)
    assert torch.equal(tau.view(torch.int32), d_all["tau"].view(torch.int32))
    for r, xs, t0 in ranks:
        n = xs.shape[0]
        y, d = r.forward(xs, residual=xs, tau=tau, phase=lmoe.PHASE_EXPERTS, debug=True)
        assert r.last_kernel_launches == 8
        torch.cuda.synchronize()
        assert r.device_error() == 0
        assert torch.equal(d["idx"], d_all["idx"][t0:t0 + n])
        assert torch.equal(d["gate"].view(torch.int32), d_all["gate"][t0:t0 + n].view(torch.int32))
        assert torch.equal(y.view(torch.int16), y_all[t0:t0 + n].view(torch.int16))
