"""Backward pass of the routed-expert branch -- TEST INFRASTRUCTURE ONLY (the product path
never imports this module).

Two functions: ``routed_backward`` for the routed branch alone (from dz at the RMSNorm output),
and ``layer_backward`` for the whole layer (from dy at the layer output).

The branch, as the forward oracle (``lmoe_oracle.c``, ``oracle_routed``) defines it, for a
token t with selected experts e_j and gates g_j (routing is a discrete choice and is held
fixed; the gates carry gradient):
    G_j = lat_t . W_g[e_j]^T,  V_j = lat_t . W_v[e_j]^T             [I]
    h_j = silu(c tanh(G_j / c)) * c tanh(V_j / c)                   SiTU-GLU
    o_j = h_j . W_ed[e_j]^T                                         [L]
    u_t = sum_j g_j o_j,   z_t = gamma * u_t / sqrt(mean(u_t^2) + eps)
Given dz = dLoss/dz this module returns dLoss/d(lat, gate, gamma, W_g, W_v, W_ed), in
float64, by PyTorch's reverse-mode autodiff of a plain re-statement of those lines (the
library routine serves as the differentiation step; the re-statement is pinned to the C
oracle's forward, and the gradients to finite differences, in the CPU tests).

Sources: "The 2.8-Trillion-Parameter Problem" (Towards AI article, "Part 1 of Inside Kimi
K3", stabilizers passage: SiTU-GLU and the RMSNorm were introduced to keep training of the
routed branch stable); the same page and "苏神复盘 Kimi K3" (Stable LatentMoE bullet) for the
branch itself.
"""
from __future__ import annotations

import numpy as np
import torch


def _bf16_values(w) -> torch.Tensor:
    if isinstance(w, torch.Tensor):
        return w.detach().to(torch.float64).cpu()
    u = np.ascontiguousarray(w)
    if u.dtype == np.int16:
        u = u.view(np.uint16)
    return torch.from_numpy((u.astype(np.uint32) << 16).view(np.float32).astype(np.float64))


def routed_forward_t(lat, idx, gate, wg, wv, wed, gamma, c=100.0, eps=1e-6, keep=None):
    """The branch in float64 torch ops (differentiable in lat, gate, gamma and weights).
    keep: a dict that receives the expert outputs "o" [n, K, L] and their gated sum "u"."""
    n, K = idx.shape
    E, I, L = wg.shape
    idx_t = torch.as_tensor(np.asarray(idx), dtype=torch.long)
    G = torch.einsum("tl,tkil->tki", lat, wg[idx_t])
    V = torch.einsum("tl,tkil->tki", lat, wv[idx_t])
    gc = c * torch.tanh(G / c)
    vc = c * torch.tanh(V / c)
    h = gc * torch.sigmoid(gc) * vc
    o = torch.einsum("tki,tkli->tkl", h, wed[idx_t])
    u = (gate.unsqueeze(-1) * o).sum(1)
    if keep is not None:
        keep["o"], keep["u"] = o, u
    r = torch.rsqrt((u * u).mean(-1, keepdim=True) + eps)
    return gamma * u * r


def routed_backward(lat, idx, gate, w_gate, w_value, w_edown, gamma, dz, c=100.0, eps=1e-6):
    """Gradients of sum(dz * z) with respect to lat [n, L], gate [n, K], gamma [L],
    W_g, W_v [E, I, L] and W_ed [E, L, I].  Weights may be bf16 tensors or bit arrays."""
    lat_t = torch.as_tensor(np.asarray(lat, dtype=np.float64)).requires_grad_(True)
    gate_t = torch.as_tensor(np.asarray(gate, dtype=np.float64)).requires_grad_(True)
    gam_t = torch.as_tensor(np.asarray(gamma, dtype=np.float64)).requires_grad_(True)
    wg = _bf16_values(w_gate).requires_grad_(True)
    wv = _bf16_values(w_value).requires_grad_(True)
    wed = _bf16_values(w_edown).requires_grad_(True)
    z = routed_forward_t(lat_t, idx, gate_t, wg, wv, wed, gam_t, c, eps)
    z.backward(torch.as_tensor(np.asarray(dz, dtype=np.float64)))
    return {"z": z.detach().numpy(), "dlat": lat_t.grad.numpy(), "dgate": gate_t.grad.numpy(),
            "dgamma": gam_t.grad.numpy(), "dw_gate": wg.grad.numpy(),
            "dw_value": wv.grad.numpy(), "dw_edown": wed.grad.numpy()}


def _f64(a) -> torch.Tensor:
    """A float64 copy of a tensor, a bf16 bit array (int16/uint16) or a float array."""
    if isinstance(a, torch.Tensor):
        return a.detach().to(torch.float64).cpu().clone()
    a = np.asarray(a)
    if a.dtype in (np.int16, np.uint16):
        return _bf16_values(a)
    return torch.as_tensor(a.astype(np.float64))


def _situ(g, v, c):
    gc = c * torch.tanh(g / c)
    return gc * torch.sigmoid(gc) * (c * torch.tanh(v / c))


def layer_forward_t(x, idx, w: dict, c=100.0, eps=1e-6, gate=None, keep=None, local_idx=None):
    """The whole layer without its residual term, in float64 torch ops, with routing held at
    ``idx`` (the forward oracle's ``latent``, ``router_logits``, ``route``, ``routed``,
    ``shared`` and ``output``):
        lat = x W_down^T,  logits = lat W_r^T,  s = sigmoid(logits),
        g_j = s[e_j] / sum_i s[e_i]   (the selected experts),
        z = routed branch (see the module docstring),
        hs_s = SiTU-GLU(x W_sg[s]^T, x W_sv[s]^T),  y = z W_up^T + sum_s hs_s W_sd[s]^T.
    ``gate`` replaces the computed gates when given (to pin the rest of the restatement to
    the C oracle, which takes fp32 gates).  keep: as for ``routed_forward_t``, plus the
    selected experts' scores "s".  local_idx: when the routed weights given are only the
    selected experts' (w_gate etc. indexed by these instead of idx).  Returns
    (y, {"lat", "logits", "gate", "z"})."""
    idx_t = torch.as_tensor(np.asarray(idx), dtype=torch.long)
    lat = x @ w["w_down"].T
    logits = lat @ w["w_router"].T
    s = torch.sigmoid(torch.gather(logits, 1, idx_t))
    if gate is None:
        gate = s / s.sum(1, keepdim=True)
    if keep is not None:
        keep["s"] = s
    z = routed_forward_t(lat, idx if local_idx is None else local_idx, gate, w["w_gate"],
                         w["w_value"], w["w_edown"], w["gamma"], c, eps, keep)
    y = z @ w["w_up"].T
    if w["w_sgate"].shape[0] > 0:
        G = torch.einsum("td,sid->tsi", x, w["w_sgate"])
        V = torch.einsum("td,sid->tsi", x, w["w_svalue"])
        y = y + torch.einsum("tsi,sdi->td", _situ(G, V, c), w["w_sdown"])
    return y, {"lat": lat, "logits": logits, "gate": gate, "z": z}


LAYER_WEIGHTS = ("w_down", "w_router", "w_gate", "w_value", "w_edown", "w_up", "w_sgate",
                 "w_svalue", "w_sdown")


def layer_backward(x, idx, w: dict, dy, c=100.0, eps=1e-6, intermediates=False) -> dict:
    """Gradients of sum(dy * y) for the layer (``layer_forward_t``) with respect to x (through
    the latent and the shared experts; the residual adds dy itself), gamma and every weight,
    in float64: keys dx, dgamma and "d" + weight name (dw_down [L, d], dw_router [E, L],
    dw_gate, dw_value, dw_edown, dw_up [d, L], dw_sgate, dw_svalue, dw_sdown); "y" is the
    forward value.  x, dy: [n, d]; weights bf16 tensors or bit arrays, gamma fp32.
    intermediates: also return du (dLoss/du, u the gated sum of the expert outputs), o, the
    selected scores s, the gates and the latent, for error bounds."""
    xt = _f64(x).requires_grad_(True)
    wt = {k: _f64(w[k]).requires_grad_(True) for k in LAYER_WEIGHTS + ("gamma",)}
    keep = {} if intermediates else None
    y, parts = layer_forward_t(xt, idx, wt, c, eps, keep=keep)
    if intermediates:
        keep["u"].retain_grad()
    y.backward(torch.as_tensor(np.asarray(dy, dtype=np.float64)))
    out = {"y": y.detach().numpy(), "dx": xt.grad.numpy(), "dgamma": wt["gamma"].grad.numpy()}
    if intermediates:
        # for error bounds: du = dLoss/du, the expert outputs o, scores s, gates, latent
        out.update({"du": keep["u"].grad.numpy(), "o": keep["o"].detach().numpy(),
                    "s": keep["s"].detach().numpy(),
                    "gate": parts["gate"].detach().numpy(),
                    "lat": parts["lat"].detach().numpy()})
    for k in LAYER_WEIGHTS:
        g = wt[k].grad  # None for weights the forward does not reach (no shared experts)
        out["d" + k] = g.numpy() if g is not None else np.zeros(tuple(wt[k].shape))
    return out


def _rows_of(a, sel: np.ndarray) -> torch.Tensor:
    """float64 copy of the rows `sel` of a weight stack (tensor or bf16 bit array)."""
    if isinstance(a, torch.Tensor):
        return _f64(a.index_select(0, torch.as_tensor(sel, dtype=torch.long)))
    return _f64(np.asarray(a)[sel])


def layer_dx_rows(x, idx, w: dict, dy, c=100.0, eps=1e-6) -> np.ndarray:
    """dx (as ``layer_backward``) for individual tokens, one at a time.  Given the routing, a
    token's output and its gradient depend on that token alone.  Only its K experts'
    weights enter, so a full-size layer fits in memory.  x, dy: [n, d]; idx: [n, K]."""
    dense = {k: _f64(w[k]) for k in ("w_down", "w_router", "gamma", "w_up", "w_sgate",
                                     "w_svalue", "w_sdown")}
    xs = _f64(x)
    dys = torch.as_tensor(np.asarray(dy, dtype=np.float64))
    idx = np.asarray(idx)
    K = idx.shape[1]
    local = np.arange(K)[None, :]
    dx = np.empty(tuple(xs.shape))
    for t in range(xs.shape[0]):
        wt = dict(dense)
        for k in ("w_gate", "w_value", "w_edown"):
            wt[k] = _rows_of(w[k], idx[t])
        xt = xs[t:t + 1].clone().requires_grad_(True)
        y, _ = layer_forward_t(xt, idx[t:t + 1], wt, c, eps, local_idx=local)
        y.backward(dys[t:t + 1])
        dx[t] = xt.grad[0].numpy()
    return dx
