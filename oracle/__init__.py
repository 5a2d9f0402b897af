"""CPU oracle of the Stable Latent MoE feed-forward layer -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
import this package.  The product path (the CUDA library and its Python binding) never
imports, links or calls it, and it shares no code with them.

The arithmetic lives in ``lmoe_oracle.c`` (fp64, fp32 routing, OpenMP over tokens); this
module compiles it with gcc on first use and wraps each function with ctypes.  Every step
cites the passage it follows in the C source.  ``forward`` chains the steps in the order
the layer defines them:

    lat    = x . W_down^T                              latent down-projection
    z      = lat . W_r^T   (rounded to fp32)           router logits
    tau    = k-th largest sigmoid score per expert     Quantile Balancing (in-batch)
    idx, g = top-K of fl32(s - tau), gates s / sum s   routing
    z_n    = RMSNorm(sum_j g_j SiTU-FFN_{idx_j}(lat))  routed experts in the latent
    ys     = sum_s SiTU-FFN_s(x)                       shared experts at full width
    y      = residual + z_n . W_up^T + ys

``backward.py`` differentiates the routed branch (PyTorch fp64 autodiff of a plain
re-statement, pinned to this forward and to finite differences).

The routed experts also have an e4m3 variant (``routed_fp8``, ``forward(expert_fp8=True)``):
per-row quantisation of both GEMM operands, defined in the C source.

Parity status: every function is pinned by the CPU tests in ``tests/test_oracle_*.py``
(closed forms, library special cases, brute force on tiny inputs, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lmoe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dbl_p = ctypes.POINTER(ctypes.c_double)
_flt_p = ctypes.POINTER(ctypes.c_float)
_u16_p = ctypes.POINTER(ctypes.c_uint16)
_i32_p = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math) and return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_sigmoid32.restype = ctypes.c_float
        lib.oracle_sigmoid32.argtypes = [ctypes.c_float]
        lib.oracle_situ.restype = ctypes.c_double
        lib.oracle_situ.argtypes = [ctypes.c_double] * 3
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_sigmoid_decreases.restype = None
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_bf16_round.restype = ctypes.c_float
        lib.oracle_bf16_round.argtypes = [ctypes.c_double]
        lib.oracle_bf16_tie_distance.restype = ctypes.c_double
        lib.oracle_bf16_tie_distance.argtypes = [ctypes.c_double]
        lib.oracle_ep_dispatch.restype = ctypes.c_longlong
        for name in ("oracle_quantize_rows", "oracle_routed_fp8", "oracle_tau_ema",
                     "oracle_load_stats_update", "oracle_ep_combine"):
            getattr(lib, name).restype = None
        for name in ("oracle_latent", "oracle_router_logits", "oracle_scores",
                     "oracle_thresholds", "oracle_route", "oracle_situ_vec",
                     "oracle_routed", "oracle_shared", "oracle_output"):
            getattr(lib, name).restype = None
        _lib = lib
        return lib


def _p(a: np.ndarray, ptype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ptype)


def _u16(a) -> np.ndarray:
    """bf16 bit patterns as a C-contiguous uint16 array (accepts numpy uint16/int16 or a
    torch bf16 tensor)."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.detach().contiguous().view(torch.int16).cpu().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def sigmoid32(z: float) -> float:
    return float(_load().oracle_sigmoid32(ctypes.c_float(z)))


def sigmoid_decreases() -> tuple[int, int]:
    """(steps down by one ulp, larger steps down) of the routing score between consecutive
    fp32 inputs, over all of [-88, 88]."""
    a, b = ctypes.c_longlong(), ctypes.c_longlong()
    _load().oracle_sigmoid_decreases(ctypes.byref(a), ctypes.byref(b))
    return int(a.value), int(b.value)


def scores(logits: np.ndarray) -> np.ndarray:
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    out = np.empty_like(lg)
    _load().oracle_scores(ctypes.c_longlong(lg.size), _p(lg, _flt_p), _p(out, _flt_p))
    return out


def situ(g, v, c: float = 100.0) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    assert g.shape == v.shape
    out = np.empty_like(g)
    _load().oracle_situ_vec(ctypes.c_longlong(g.size), _p(g, _dbl_p), _p(v, _dbl_p),
                            ctypes.c_double(c), _p(out, _dbl_p))
    return out


def fair_share_rank(T: int, K: int, E: int) -> int:
    """k = max(1, floor(T*K/E)), at most T: the rank of the Quantile-Balancing threshold."""
    if T <= 0:
        return 0
    return min(T, max(1, (T * K) // E))


def thresholds(logits: np.ndarray, k: int) -> np.ndarray:
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    tau = np.empty(E, dtype=np.float32)
    _load().oracle_thresholds(T, E, int(k), _p(lg, _flt_p), _p(tau, _flt_p))
    return tau


def tau_ema(tau_ema_prev, tau_step, beta: float, first: bool = False) -> np.ndarray:
    """One step of the streaming thresholds: fma(beta, prev - step, step) in fp32."""
    step = np.ascontiguousarray(tau_step, dtype=np.float32)
    out = (np.array(step) if tau_ema_prev is None
           else np.ascontiguousarray(tau_ema_prev, dtype=np.float32).copy())
    _load().oracle_tau_ema(len(step), ctypes.c_float(beta), 1 if first else 0,
                           _p(step, _flt_p), _p(out, _flt_p))
    return out


def load_stats_update(acc, counts) -> np.ndarray:
    """Accumulate one step's per-expert counts into the 64-bit counters (4 + 4E)."""
    c = np.ascontiguousarray(counts, dtype=np.int32)
    E = len(c)
    a = (np.zeros(4 + 4 * E, dtype=np.uint64) if acc is None
         else np.ascontiguousarray(acc, dtype=np.uint64).copy())
    _load().oracle_load_stats_update(E, _p(c, _i32_p),
                                     a.ctypes.data_as(ctypes.POINTER(ctypes.c_ulonglong)))
    return a


_u32_p = ctypes.POINTER(ctypes.c_uint32)


def ep_dispatch(idx, E: int, R: int, rows=None) -> dict:
    """Expert-parallel dispatch over R ranks: the (token, rank) pairs in (rank, token) order,
    their slot masks, and (with rows, bf16 [T, W]) the rows each pair carries."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, K = idx.shape
    assert E % R == 0
    rr = None if rows is None else _u16(rows)
    W = 0 if rr is None else rr.shape[1]
    pmax = T * min(K, R)
    off = np.zeros(R + 1, dtype=np.int32)
    tok = np.zeros(pmax, dtype=np.int32)
    slots = np.zeros(pmax, dtype=np.uint32)
    srows = np.zeros((pmax, max(W, 1)), dtype=np.uint16)
    P = _load().oracle_ep_dispatch(T, K, E, R, _p(idx, _i32_p), W,
                                   None if rr is None else _p(rr, _u16_p), _p(off, _i32_p),
                                   _p(tok, _i32_p), _p(slots, _u32_p),
                                   None if rr is None else _p(srows, _u16_p))
    out = {"P": int(P), "send_off": off, "send_tok": tok[:P], "send_slots": slots[:P]}
    if rr is not None:
        out["send_rows"] = srows[:P, :W]
    return out


def ep_combine(disp: dict, inv, gate, o, T: int):
    """Expert-parallel combine: per pair the bf16 gate-weighted sum of its slots' output rows
    (o: bf16 [T*K, W], rows addressed through inv [T, K]), then per token the fp32 sum of its
    pairs' rows in rank order.  Returns (part uint16 [P, W], u fp32 [T, W])."""
    inv = np.ascontiguousarray(inv, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    ou = _u16(o)
    K = inv.shape[1]
    W = ou.shape[1]
    P = disp["P"]
    tok = np.ascontiguousarray(disp["send_tok"], dtype=np.int32)
    slots = np.ascontiguousarray(disp["send_slots"], dtype=np.uint32)
    part = np.zeros((P, W), dtype=np.uint16)
    u = np.zeros((T, W), dtype=np.float32)
    _load().oracle_ep_combine(T, K, ctypes.c_longlong(P), _p(tok, _i32_p), _p(slots, _u32_p),
                              _p(inv, _i32_p), _p(gate, _flt_p), W, _p(ou, _u16_p),
                              _p(part, _u16_p), _p(u, _flt_p))
    return part, u


def route(logits: np.ndarray, tau, K: int):
    """Returns (idx int32 [T,K], gate fp32 [T,K], scores fp32 [T,E])."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    idx = np.empty((T, K), dtype=np.int32)
    gate = np.empty((T, K), dtype=np.float32)
    sc = np.empty((T, E), dtype=np.float32)
    tp = None
    if tau is not None:
        tau = np.ascontiguousarray(tau, dtype=np.float32)
        assert tau.shape == (E,)
        tp = _p(tau, _flt_p)
    _load().oracle_route(T, E, K, _p(lg, _flt_p), tp, _p(idx, _i32_p), _p(gate, _flt_p),
                         _p(sc, _flt_p))
    return idx, gate, sc


def latent(x, w_down) -> np.ndarray:
    x, w_down = _u16(x), _u16(w_down)
    n, d = x.shape
    L = w_down.shape[0]
    assert w_down.shape == (L, d)
    lat = np.empty((n, L), dtype=np.float64)
    _load().oracle_latent(n, d, L, _p(x, _u16_p), _p(w_down, _u16_p), _p(lat, _dbl_p))
    return lat


def router_logits(lat: np.ndarray, w_router) -> np.ndarray:
    lat = np.ascontiguousarray(lat, dtype=np.float64)
    w_router = _u16(w_router)
    n, L = lat.shape
    E = w_router.shape[0]
    assert w_router.shape == (E, L)
    out = np.empty((n, E), dtype=np.float64)
    _load().oracle_router_logits(n, L, E, _p(lat, _dbl_p), _p(w_router, _u16_p),
                                 _p(out, _dbl_p))
    return out


def routed(lat, idx, gate, w_gate, w_value, w_edown, gamma, c=100.0, eps=1e-6):
    lat = np.ascontiguousarray(lat, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    w_gate, w_value, w_edown = _u16(w_gate), _u16(w_value), _u16(w_edown)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    n, L = lat.shape
    E, I, L2 = w_gate.shape
    K = idx.shape[1]
    assert L2 == L and w_value.shape == w_gate.shape and w_edown.shape == (E, L, I)
    assert gate.shape == idx.shape == (n, K) and gamma.shape == (L,)
    assert n == 0 or (idx.min() >= 0 and idx.max() < E)
    z = np.empty((n, L), dtype=np.float64)
    _load().oracle_routed(n, L, E, K, I, _p(lat, _dbl_p), _p(idx, _i32_p), _p(gate, _flt_p),
                          _p(w_gate, _u16_p), _p(w_value, _u16_p), _p(w_edown, _u16_p),
                          _p(gamma, _flt_p), ctypes.c_double(c), ctypes.c_double(eps),
                          _p(z, _dbl_p))
    return z


_u8_p = ctypes.POINTER(ctypes.c_uint8)


def e4m3_decode(codes) -> np.ndarray:
    """Values of e4m3 codes (uint8 array) as float64."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3 codes (ties to even, saturating at 448) of fp32 values."""
    lib = _load()
    xf = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in xf.ravel()],
                    dtype=np.uint8).reshape(xf.shape)


def bf16_round(x) -> np.ndarray:
    """fp64 values rounded to the nearest bf16 (ties to even), as float32."""
    lib = _load()
    xd = np.asarray(x, dtype=np.float64)
    return np.array([lib.oracle_bf16_round(float(v)) for v in xd.ravel()],
                    dtype=np.float32).reshape(xd.shape)


def quantize_rows(x):
    """Per-row e4m3 quantisation of fp32 rows [rows, cols]: (codes uint8, scales fp32),
    with x ~ decode(codes) * scale."""
    xf = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = xf.shape
    codes = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty(rows, dtype=np.float32)
    if rows:
        _load().oracle_quantize_rows(ctypes.c_longlong(rows), cols, _p(xf, _flt_p),
                                     _p(codes, _u8_p), _p(scales, _flt_p))
    return codes, scales


def _bf16_values(w) -> np.ndarray:
    """bf16 weights (torch tensor or uint16 bits) as float32 values."""
    u = _u16(w)
    return (u.astype(np.uint32) << 16).view(np.float32)


def quantize_expert_weights(w_gate, w_value, w_edown) -> dict:
    """The routed experts' weights quantised row by row (one row = one output feature of
    one expert): qg, qv [E, I, L] + sg, sv [E, I]; qd [E, L, I] + sd [E, L]."""
    out = {}
    for name, w in (("g", w_gate), ("v", w_value), ("d", w_edown)):
        v = _bf16_values(w)
        E, R, C = v.shape
        q, s = quantize_rows(v.reshape(E * R, C))
        out["q" + name] = q.reshape(E, R, C)
        out["s" + name] = s.reshape(E, R)
    return out


def bf16_tie_distance(x) -> np.ndarray:
    """Relative distance of each value from the nearest bf16 rounding tie."""
    lib = _load()
    xd = np.asarray(x, dtype=np.float64)
    return np.array([lib.oracle_bf16_tie_distance(float(v)) for v in xd.ravel()]).reshape(xd.shape)


def routed_fp8(lat, idx, gate, wq: dict, gamma, c=100.0, eps=1e-6, tie_margin=2.0 ** -16,
               return_ties=False):
    """Routed experts with e4m3 operands (weights from quantize_expert_weights).
    return_ties: also return, per token, how many of its quantised rows (its latent and its
    K SiTU outputs) have a scale that hinges on a bf16 rounding near-tie (relative distance
    below tie_margin): there an evaluation that differs in the last fp32 bits may quantise
    the whole row differently."""
    lat = np.ascontiguousarray(lat, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    qg, qv, qd = (np.ascontiguousarray(wq[k]) for k in ("qg", "qv", "qd"))
    sg, sv, sd = (np.ascontiguousarray(wq[k], dtype=np.float32) for k in ("sg", "sv", "sd"))
    n, L = lat.shape
    E, I, L2 = qg.shape
    K = idx.shape[1]
    assert L2 == L and qv.shape == qg.shape and qd.shape == (E, L, I)
    assert sg.shape == sv.shape == (E, I) and sd.shape == (E, L)
    assert n == 0 or (idx.min() >= 0 and idx.max() < E)
    z = np.empty((n, L), dtype=np.float64)
    ties = np.zeros(n, dtype=np.int32)
    _load().oracle_routed_fp8(n, L, E, K, I, _p(lat, _dbl_p), _p(idx, _i32_p),
                              _p(gate, _flt_p), _p(qg, _u8_p), _p(sg, _flt_p), _p(qv, _u8_p),
                              _p(sv, _flt_p), _p(qd, _u8_p), _p(sd, _flt_p), _p(gamma, _flt_p),
                              ctypes.c_double(c), ctypes.c_double(eps), _p(z, _dbl_p),
                              _p(ties, _i32_p), ctypes.c_double(tie_margin))
    return (z, ties) if return_ties else z


def shared(x, w_sgate, w_svalue, w_sdown, c=100.0):
    x = _u16(x)
    w_sgate, w_svalue, w_sdown = _u16(w_sgate), _u16(w_svalue), _u16(w_sdown)
    n, d = x.shape
    S, Is, d2 = w_sgate.shape
    assert d2 == d and w_svalue.shape == w_sgate.shape and w_sdown.shape == (S, d, Is)
    ys = np.empty((n, d), dtype=np.float64)
    _load().oracle_shared(n, d, S, Is, _p(x, _u16_p), _p(w_sgate, _u16_p),
                          _p(w_svalue, _u16_p), _p(w_sdown, _u16_p), ctypes.c_double(c),
                          _p(ys, _dbl_p))
    return ys


def output(z, ys, w_up, residual=None):
    z = np.ascontiguousarray(z, dtype=np.float64)
    ys = np.ascontiguousarray(ys, dtype=np.float64)
    w_up = _u16(w_up)
    n, L = z.shape
    d = w_up.shape[0]
    assert w_up.shape == (d, L) and ys.shape == (n, d)
    rp = None
    if residual is not None:
        residual = _u16(residual)
        assert residual.shape == (n, d)
        rp = _p(residual, _u16_p)
    y = np.empty((n, d), dtype=np.float64)
    _load().oracle_output(n, d, L, _p(z, _dbl_p), _p(ys, _dbl_p), _p(w_up, _u16_p), rp,
                          _p(y, _dbl_p))
    return y


@dataclass
class OracleResult:
    y: np.ndarray            # [n, d] fp64 layer output
    lat: np.ndarray          # [n, L] fp64 latent
    logits: np.ndarray       # [n, E] fp32 router logits used for routing
    tau: np.ndarray | None   # [E] fp32 thresholds used (None: no balancing)
    idx: np.ndarray          # [n, K] int32
    gate: np.ndarray         # [n, K] fp32
    z: np.ndarray            # [n, L] fp64 normalised aggregated latent
    ys: np.ndarray           # [n, d] fp64 shared-expert output
    scale_ties: np.ndarray | None = None  # expert_fp8: per token, rows quantised at a near-tie


def forward(w: dict, x, K: int, residual=None, tau="batch", logits_in=None, c=100.0,
            eps=1e-6, expert_fp8: bool = False, tie_margin: float = 2.0 ** -16) -> OracleResult:
    """The whole layer on the rows of ``x``.

    w: dict of weights (bf16 tensors or uint16 bit arrays, fp32 gamma) with keys w_down,
       w_router, w_gate, w_value, w_edown, gamma, w_up, w_sgate, w_svalue, w_sdown.
    tau: "batch" -> thresholds solved over the rows of x (k = fair_share_rank);
         None -> plain top-K without balancing; an array -> those thresholds.
    logits_in: fp32 [n, E] router logits to route on instead of the computed ones.
    expert_fp8: routed experts with e4m3 operands (``routed_fp8``); tie_margin is its
    near-tie margin for ``scale_ties``.
    """
    xs = _u16(x)
    n = xs.shape[0]
    lat = latent(xs, w["w_down"])
    if logits_in is None:
        lg = router_logits(lat, w["w_router"]).astype(np.float32)
    else:
        lg = np.ascontiguousarray(logits_in, dtype=np.float32)
    E = lg.shape[1]
    if isinstance(tau, str):
        assert tau == "batch"
        tau_v = thresholds(lg, fair_share_rank(n, K, E))
    elif tau is None:
        tau_v = None
    else:
        tau_v = np.ascontiguousarray(tau, dtype=np.float32)
    idx, gate, _ = route(lg, tau_v, K)
    gamma = w["gamma"]
    if hasattr(gamma, "detach"):
        gamma = gamma.detach().float().cpu().numpy()
    ties = None
    if expert_fp8:
        wq = quantize_expert_weights(w["w_gate"], w["w_value"], w["w_edown"])
        z, ties = routed_fp8(lat, idx, gate, wq, gamma, c, eps, tie_margin=tie_margin,
                             return_ties=True)
    else:
        z = routed(lat, idx, gate, w["w_gate"], w["w_value"], w["w_edown"], gamma, c, eps)
    ys = shared(xs, w["w_sgate"], w["w_svalue"], w["w_sdown"], c)
    y = output(z, ys, w["w_up"], residual)
    return OracleResult(y=y, lat=lat, logits=lg, tau=tau_v, idx=idx, gate=gate, z=z, ys=ys,
                        scale_ties=ties)
