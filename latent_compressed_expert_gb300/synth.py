"""Seeded synthetic inputs for the Stable Latent MoE layer.

This module draws random numbers and nothing else: it holds none of the layer's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.  Every tensor is
generated from a ``torch.Generator`` seeded from (seed, tensor name), in fixed-size chunks,
so the same call gives the same bits on every run of the same device type.

Workloads (sizes of the K3 layer as the pages state them: hidden 7168, latent 3584 =
half of it, 896 routed experts with 16 active per token, 2 shared experts; the expert
intermediate sizes 512 / 2048 are this build's choice, the pages give none):
    tiny     T=64    d=256  L=128  E=16  K=4  I=64  S=2 Is=128   (CPU-sized)
    e64      T=4096  d=7168 L=3584 E=64  K=4  I=512 S=2 Is=2048
    prefill  T=8192  d=7168 L=3584 E=896 K=16 I=512 S=2 Is=2048
    decode   T=64    same widths as prefill
    skew     T=32768 same widths, router logits with a Zipf(1.1) per-expert bias
Distributions: x ~ N(0,1) (optionally a fraction of elements times 1000); every weight
~ N(0, 1/fan_in); gamma = 1; optionally a fraction of the gate/value rows times 500 so
that pre-activations reach the SiTU-GLU cap.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class LayerShape:
    name: str
    T: int      # tokens
    d: int      # hidden width
    L: int      # latent width
    E: int      # routed experts
    K: int      # experts per token
    I: int      # routed expert intermediate size
    S: int      # shared experts
    Is: int     # shared expert intermediate size
    c: float = 100.0    # SiTU-GLU cap
    eps: float = 1e-6   # RMSNorm epsilon

    def with_tokens(self, T: int) -> "LayerShape":
        return replace(self, T=T)


TINY = LayerShape("tiny", T=64, d=256, L=128, E=16, K=4, I=64, S=2, Is=128)
E64 = LayerShape("e64", T=4096, d=7168, L=3584, E=64, K=4, I=512, S=2, Is=2048)
PREFILL = LayerShape("prefill", T=8192, d=7168, L=3584, E=896, K=16, I=512, S=2, Is=2048)
DECODE = LayerShape("decode", T=64, d=7168, L=3584, E=896, K=16, I=512, S=2, Is=2048)
SKEW = LayerShape("skew", T=32768, d=7168, L=3584, E=896, K=16, I=512, S=2, Is=2048)

SHAPES = {s.name: s for s in (TINY, E64, PREFILL, DECODE, SKEW)}

_CHUNK = 1 << 24  # elements drawn per generator call


def _gen(seed: int, name: str, device) -> torch.Generator:
    h = hashlib.sha256(f"{seed}/{name}".encode()).digest()
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def _normal(shape, std: float, g: torch.Generator, device, dtype) -> torch.Tensor:
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        tmp = torch.randn(m, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[s:s + m].copy_(tmp)
    return out


def _pick(count: int, frac: float, g: torch.Generator, device) -> torch.Tensor:
    m = max(1, int(round(count * frac)))
    return torch.randperm(count, generator=g, device=device)[:m]


def outlier_router_gain(sh: LayerShape, outlier_frac: float, outlier_scale: float) -> float:
    """Router weight gain that keeps the router logits ~N(0, 1) when x carries outliers:
    the latent's expected mean square grows from 1 to 1 + frac * (scale^2 - 1), so the
    router's N(0, 1/fan_in) weights are scaled by the inverse square root of that."""
    return (1.0 + outlier_frac * (outlier_scale ** 2 - 1.0)) ** -0.5


def make_weights(sh: LayerShape, seed: int, device="cpu", hot_row_frac: float = 0.0,
                 hot_scale: float = 500.0, router_gain: float = 1.0) -> dict:
    """All weights of one layer, bf16 [out, in] (gamma fp32).  ``hot_row_frac`` > 0 scales
    that fraction (at least one) of the routed and shared gate and value rows by
    ``hot_scale``; ``router_gain`` scales the router's standard deviation."""
    bf = torch.bfloat16
    w = {}
    w["w_down"] = _normal((sh.L, sh.d), sh.d ** -0.5, _gen(seed, "w_down", device), device, bf)
    w["w_router"] = _normal((sh.E, sh.L), router_gain * sh.L ** -0.5,
                            _gen(seed, "w_router", device), device, bf)
    w["w_gate"] = _normal((sh.E, sh.I, sh.L), sh.L ** -0.5, _gen(seed, "w_gate", device), device, bf)
    w["w_value"] = _normal((sh.E, sh.I, sh.L), sh.L ** -0.5, _gen(seed, "w_value", device), device, bf)
    w["w_edown"] = _normal((sh.E, sh.L, sh.I), sh.I ** -0.5, _gen(seed, "w_edown", device), device, bf)
    w["gamma"] = torch.ones(sh.L, dtype=torch.float32, device=device)
    w["w_up"] = _normal((sh.d, sh.L), sh.L ** -0.5, _gen(seed, "w_up", device), device, bf)
    w["w_sgate"] = _normal((sh.S, sh.Is, sh.d), sh.d ** -0.5, _gen(seed, "w_sgate", device), device, bf)
    w["w_svalue"] = _normal((sh.S, sh.Is, sh.d), sh.d ** -0.5, _gen(seed, "w_svalue", device), device, bf)
    w["w_sdown"] = _normal((sh.S, sh.d, sh.Is), max(sh.Is, 1) ** -0.5, _gen(seed, "w_sdown", device),
                           device, bf)
    if hot_row_frac > 0.0:
        for name in ("w_gate", "w_value", "w_sgate", "w_svalue"):
            t = w[name]
            rows = t.view(-1, t.shape[-1])
            sel = _pick(rows.shape[0], hot_row_frac, _gen(seed, name + "/hot", device), device)
            rows[sel] = (rows[sel].float() * hot_scale).to(bf)
    return w


def make_x(sh: LayerShape, seed: int, device="cpu", outlier_frac: float = 0.0,
           outlier_scale: float = 1000.0, T: int | None = None) -> torch.Tensor:
    """Hidden states [T, d] bf16 ~ N(0,1); ``outlier_frac`` of the elements times
    ``outlier_scale``."""
    T = sh.T if T is None else T
    x = _normal((T, sh.d), 1.0, _gen(seed, f"x/{T}", device), device, torch.float32)
    if outlier_frac > 0.0 and x.numel() > 0:
        sel = _pick(x.numel(), outlier_frac, _gen(seed, f"x/{T}/outliers", device), device)
        x.view(-1)[sel] *= outlier_scale
    return x.to(torch.bfloat16)


def make_logits(T: int, E: int, seed: int, device="cpu", zipf_s: float | None = None,
                scale: float = 1.0) -> torch.Tensor:
    """Router logits [T, E] fp32 ~ N(0, scale^2).  With ``zipf_s``, expert e gets the added
    bias -zipf_s * ln(rank_e), rank a seeded permutation of 1..E, so that a few experts
    dominate the raw scores."""
    z = _normal((T, E), scale, _gen(seed, f"logits/{T}x{E}", device), device, torch.float32)
    if zipf_s is not None:
        z += zipf_bias(E, seed, zipf_s, device).unsqueeze(0)
    return z


def zipf_bias(E: int, seed: int, s: float = 1.1, device="cpu") -> torch.Tensor:
    """Per-expert router bias [E] fp32 of the skewed-router workload: -s * ln(rank_e), with
    rank a seeded permutation of 1..E."""
    rank = torch.randperm(E, generator=_gen(seed, f"zipf/{E}", device), device=device) + 1
    return (-s * torch.log(rank.to(torch.float32))).contiguous()


def make_uniform_logits(T: int, E: int, seed: int, device="cpu", lo=-4.0, hi=4.0,
                        quantum: float | None = None) -> torch.Tensor:
    """Logits uniform in [lo, hi); with ``quantum``, rounded to multiples of it, which makes
    exact ties frequent."""
    g = _gen(seed, f"ulogits/{T}x{E}", device)
    z = torch.rand((T, E), generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo
    if quantum is not None:
        z = torch.round(z / quantum) * quantum
    return z


def shape_dict(sh: LayerShape) -> dict:
    return {"T": sh.T, "d": sh.d, "L": sh.L, "E": sh.E, "K": sh.K, "I": sh.I, "S": sh.S,
            "Is": sh.Is}
