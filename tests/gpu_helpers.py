"""Shared pieces of the GPU parity tests: running the oracle on a subset of tokens, the
output tolerance, and the near-tie rule for routing decisions taken on two different
(but each correct within its precision) sets of router logits."""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import torch

from latent_compressed_expert_gb300 import synth

# Output tolerance for bf16 operands with fp32 accumulation (stated for the layer):
#   max |y - y_ref| <= 2e-2 * RMS(y_ref)  and  sum |y - y_ref| / sum |y_ref| <= 5e-3.
# It is held, exactly as written, to the value the output GEMM computes in fp32 before its
# bf16 store (lmoe_io.y_f32_out); the returned bf16 y must then be that value rounded to
# nearest even, bit for bit, and meet the mean bound too.  (The store alone moves an element
# by up to half a bf16 ulp of itself, which exceeds 2e-2 * RMS wherever |y| > ~5 RMS: the
# heavy-tailed outputs once pre-activations hit the SiTU-GLU cap.)
MAX_ERR_REL_RMS = 2e-2
MEAN_REL_ERR = 5e-3


def half_ulp_bf16(ref):
    """Half the bf16 spacing at each value (fp32 spacing times 2^16, halved)."""
    return np.spacing(np.abs(np.asarray(ref, dtype=np.float32))).astype(np.float64) * 32768.0


def error_stats(y, ref):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(y - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    excess = np.maximum(err - half_ulp_bf16(ref), 0.0)
    return {"max_err": float(err.max()), "rms_ref": rms,
            "max_err_over_rms": float(err.max() / rms) if rms > 0 else float("inf"),
            "max_excess_over_rms": float(excess.max() / rms) if rms > 0 else float("inf"),
            "mean_rel_err": float(err.sum() / max(np.abs(ref).sum(), 1e-300))}


def _np(t):
    return t.detach().float().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def assert_layer_close(y, y_f32, ref, tag=""):
    """The layer's output against the oracle's.  y: the bf16 output rows (torch); y_f32: the
    same rows before the bf16 store (lmoe_io.y_f32_out); ref: the oracle's fp64 rows.
    Checks the stated bound literally on y_f32, that y is y_f32 rounded to nearest even, and
    the mean bound on y.  Returns the statistics of both."""
    assert y.dtype == torch.bfloat16 and y_f32.dtype == torch.float32, tag
    rounded = y_f32.to(torch.bfloat16)
    assert torch.equal(rounded.view(torch.int16), y.view(torch.int16)), \
        (tag, "bf16 output is not the fp32 value rounded to nearest")
    v = _np(y_f32).astype(np.float64)
    assert np.all(np.isfinite(v)), tag
    s32 = error_stats(v, ref)
    s16 = error_stats(_np(y), ref)
    assert s32["max_err_over_rms"] <= MAX_ERR_REL_RMS, (tag, "before the store", s32)
    assert s32["mean_rel_err"] <= MEAN_REL_ERR, (tag, "before the store", s32)
    assert s16["mean_rel_err"] <= MEAN_REL_ERR, (tag, "bf16", s16)
    return {"f32": s32, "bf16": s16}


def assert_close(y, ref, tag=""):
    """Two bf16 outputs of the device path, each rounded from its own fp32 value (split or
    unsplit reductions, the no-allocation entry point): the stated bound plus half a bf16 ulp
    of the reference for the rounding of y."""
    s = error_stats(y, ref)
    assert np.all(np.isfinite(np.asarray(y, dtype=np.float64))), tag
    assert s["max_excess_over_rms"] <= MAX_ERR_REL_RMS, (tag, s)
    assert s["mean_rel_err"] <= MEAN_REL_ERR, (tag, s)
    return s


def weights_to_host(w: dict) -> dict:
    return {k: v.detach().cpu() for k, v in w.items()}


def oracle_rows(oracle, w_host: dict, x_rows, idx_rows, gate_rows, residual_rows=None,
                c=100.0, eps=1e-6):
    """Layer output of the given tokens with the given routing (fp64 oracle).  Only the
    experts these tokens use are handed to the oracle (indices remapped accordingly)."""
    idx_rows = np.asarray(idx_rows, dtype=np.int64)
    used, remap = np.unique(idx_rows, return_inverse=True)
    remap = remap.reshape(idx_rows.shape).astype(np.int32)
    sel = torch.as_tensor(used)
    lat = oracle.latent(x_rows, w_host["w_down"])
    z = oracle.routed(lat, remap, gate_rows, w_host["w_gate"][sel].contiguous(),
                      w_host["w_value"][sel].contiguous(), w_host["w_edown"][sel].contiguous(),
                      w_host["gamma"].numpy(), c, eps)
    ys = oracle.shared(x_rows, w_host["w_sgate"], w_host["w_svalue"], w_host["w_sdown"], c)
    return oracle.output(z, ys, w_host["w_up"], residual_rows)


def routing_agrees_up_to_ties(oracle, logits_ref, tau_ref, idx_gpu, K, delta):
    """Per token: True where the GPU's expert set equals the oracle's.  Where they differ,
    assert that every expert in the symmetric difference has an oracle key a = s - tau
    within `delta` of the oracle's K-th largest key (a near-tie that the logits' rounding
    decides).  Returns the boolean mask of tokens with identical sets."""
    idx_ref, _, s_ref = oracle.route(logits_ref, tau_ref, K)
    a = s_ref.astype(np.float64) - (tau_ref.astype(np.float64)[None, :] if tau_ref is not None else 0.0)
    same = np.zeros(len(idx_gpu), dtype=bool)
    for t in range(len(idx_gpu)):
        g, r = set(idx_gpu[t].tolist()), set(idx_ref[t].tolist())
        if g == r:
            same[t] = True
            continue
        kth = np.sort(a[t])[::-1][K - 1]
        for e in g ^ r:
            assert abs(a[t, e] - kth) <= delta, (t, e, a[t, e], kth, delta)
    return same, idx_ref


def mid_shape(T=1000):
    """Several tiles in every GEMM dimension, ragged tails, expert segments of ~125 rows."""
    return synth.LayerShape("mid", T=T, d=1024, L=512, E=64, K=8, I=256, S=2, Is=512)


def with_T(sh, T):
    return replace(sh, T=T)
