"""Backward pass of the routed-expert branch -- TEST INFRASTRUCTURE ONLY (the product path
never imports this module).

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


def routed_forward_t(lat, idx, gate, wg, wv, wed, gamma, c=100.0, eps=1e-6):
    """The branch in float64 torch ops (differentiable in lat, gate, gamma and weights)."""
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
