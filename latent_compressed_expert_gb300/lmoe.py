"""ctypes binding of liblmoe.so (include/lmoe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; PyTorch provides device
memory and the current stream.  There is no CPU fallback: if the library is missing or
its CUDA calls fail, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "liblmoe.so")

LMOE_OK = 0
LMOE_ERR_INVALID_ARG = 1
LMOE_ERR_UNSUPPORTED = 2
LMOE_ERR_CUDA = 3
LMOE_ERR_DEVICE_TIMEOUT = 4
LMOE_ERR_WORKSPACE_TOO_SMALL = 5

# Every symbol the header declares, with its ctypes signature.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class Dims(ctypes.Structure):
    _fields_ = [("T", _i), ("d", _i), ("L", _i), ("E", _i), ("K", _i), ("I", _i), ("S", _i),
                ("Is", _i), ("c", _f), ("eps", _f), ("expert_fp8", _i)]


class Weights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("w_down", "w_router", "w_gate", "w_value", "w_edown", "gamma",
                                   "w_up", "w_sgate", "w_svalue", "w_sdown")]


class IO(ctypes.Structure):
    _fields_ = [("tau_in", _vp), ("balance", _i), ("logits_in", _vp), ("logits_out", _vp),
                ("tau_out", _vp), ("idx_out", _vp), ("gate_out", _vp), ("counts_out", _vp),
                ("stage_events", ctypes.POINTER(_vp)), ("kernel_launches", _i),
                ("aux_stream", _vp), ("aux_events", _vp * 2), ("shared_sms", _i),
                ("phase", _i), ("cand_out", _vp), ("cand_k", _i),
                ("tau_ema", _vp), ("ema_beta", _f), ("ema_first", _i), ("load_stats", _vp),
                ("save_pre", _vp), ("save_pre_shared", _vp), ("y_f32_out", _vp),
                ("logit_bias", _vp)]


OVERLAP_MIN_T = 512  # LMOE_OVERLAP_MIN_T
HOST_PIPE_MAX_DEPTH = 4  # LMOE_HOST_PIPE_MAX_DEPTH


class HostPipe(ctypes.Structure):
    _fields_ = [("depth", _i), ("max_tokens", _i), ("x_dev", _vp * HOST_PIPE_MAX_DEPTH),
                ("y_dev", _vp * HOST_PIPE_MAX_DEPTH), ("upload", _vp), ("compute", _vp),
                ("download", _vp), ("uploaded", _vp * HOST_PIPE_MAX_DEPTH),
                ("computed", _vp * HOST_PIPE_MAX_DEPTH),
                ("downloaded", _vp * HOST_PIPE_MAX_DEPTH), ("calls", ctypes.c_ulonglong)]

# enum lmoe_phase
PHASE_ALL, PHASE_ROUTER, PHASE_EXPERTS = 0, 1, 2


# enum lmoe_stage
STAGES = ["latent_shared", "router", "thresholds", "route", "dispatch", "expert_gate_up",
          "expert_down", "combine", "output"]
NUM_STAGES = len(STAGES)


SIGNATURES = {
    "lmoe_packed_bytes": (_sz, [ctypes.POINTER(Dims)]),
    "lmoe_pack_weights": (_i, [ctypes.POINTER(Dims), ctypes.POINTER(Weights), _vp, _sz, _vp]),
    "lmoe_workspace_bytes": (_sz, [ctypes.POINTER(Dims)]),
    "lmoe_thresholds": (_i, [_vp, _i, _i, _i, _i, _vp, _vp]),
    "lmoe_threshold_candidates": (_i, [_vp, _i, _i, _i, _vp, _vp]),
    "lmoe_fair_share_rank": (_i, [ctypes.c_longlong, _i, _i]),
    "lmoe_quantize_e4m3": (_i, [_vp, ctypes.c_longlong, _i, _vp, _vp, _vp]),
    "lmoe_tau_ema": (_i, [_vp, _vp, _i, _f, _i, _vp]),
    "lmoe_packed_backward_bytes": (_sz, [ctypes.POINTER(Dims)]),
    "lmoe_pack_backward_weights": (_i, [ctypes.POINTER(Dims), ctypes.POINTER(Weights), _vp, _vp,
                                        _sz, _vp]),
    "lmoe_backward_workspace_bytes": (_sz, [ctypes.POINTER(Dims)]),
    "lmoe_backward": (_i, [ctypes.POINTER(Dims), _vp, _vp, _vp, _sz, _vp, _vp, _vp, _vp, _vp,
                           _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lmoe_routed_backward_workspace_bytes": (_sz, [ctypes.POINTER(Dims)]),
    "lmoe_routed_backward": (_i, [ctypes.POINTER(Dims), _vp, _vp, _vp, _sz, _vp, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _vp, _sz, _vp]),
    "lmoe_ep_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "lmoe_ep_dispatch": (_i, [_vp, _i, _i, _i, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lmoe_ep_combine": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp,
                             _vp, _vp]),
    "lmoe_load_stats_update": (_i, [_vp, _i, _vp, _vp]),
    "lmoe_route": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "lmoe_forward": (_i, [ctypes.POINTER(Dims), _vp, _vp, _vp, _vp, _vp, _sz, ctypes.POINTER(IO),
                          _vp]),
    "lmoe_gemm_bf16": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp]),
    "lmoe_gemm_wgrad_bf16": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp]),
    "lmoe_forward_noalloc": (_i, [ctypes.POINTER(Dims), _vp, _vp, _vp, _vp, ctypes.POINTER(IO),
                                  _vp]),
    "lmoe_forward_host": (_i, [ctypes.POINTER(Dims), _vp, _vp, _i, _vp, _vp, _sz,
                               ctypes.POINTER(IO), ctypes.POINTER(HostPipe)]),
    "lmoe_noalloc_last_device_error": (_i, []),
    "lmoe_last_device_error": (_i, [_vp]),
    "lmoe_error_string": (ctypes.c_char_p, [_i]),
    "lmoe_version": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


def load():
    """Load liblmoe.so (built by ``python -m latent_compressed_expert_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run "
                               "`python -m latent_compressed_expert_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class LmoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = load().lmoe_error_string(code).decode()
        super().__init__(f"{what}: {msg} (status {code})")
        self.code = code


def _check(code: int, what: str):
    if code != LMOE_OK:
        raise LmoeError(code, what)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("lmoe: tensors must be CUDA device tensors")
    if not t.is_contiguous():
        raise ValueError("lmoe: tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _expect(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"lmoe: {name} must be {dtype} {tuple(shape)}, got {t.dtype} "
                         f"{tuple(t.shape)}")


def make_dims(T, d, L, E, K, I, S, Is, c=100.0, eps=1e-6, expert_fp8=False) -> Dims:
    return Dims(T, d, L, E, K, I, S, Is, c, eps, 1 if expert_fp8 else 0)


def dims_of(shape, T=None, expert_fp8=False) -> Dims:
    """Dims from an object with T, d, L, E, K, I, S, Is (and optionally c, eps)."""
    return make_dims(shape.T if T is None else T, shape.d, shape.L, shape.E, shape.K, shape.I,
                     shape.S, shape.Is, getattr(shape, "c", 100.0), getattr(shape, "eps", 1e-6),
                     expert_fp8)


def packed_bytes(dims: Dims) -> int:
    return int(load().lmoe_packed_bytes(ctypes.byref(dims)))


SPLITK_BYTES = 12 << 20  # the optional split-K region of lmoe_workspace_bytes (T <= 128)
NOALLOC_SCRATCH_BYTES = 24 << 20  # LMOE_NOALLOC_SCRATCH_BYTES: lmoe_forward_noalloc's array


def workspace_base_bytes(dims: Dims) -> int:
    """The smallest workspace lmoe_forward accepts: lmoe_workspace_bytes less the optional
    split-K region of small batches."""
    full = workspace_bytes(dims)
    return full - SPLITK_BYTES if full and 0 < dims.T <= 128 else full


def workspace_bytes(dims: Dims) -> int:
    return int(load().lmoe_workspace_bytes(ctypes.byref(dims)))


def pack_weights(dims: Dims, w: dict, stream=None) -> torch.Tensor:
    """Repack a dict of unpacked weights (bf16 [out, in], gamma fp32) into one device
    buffer in the layout lmoe_forward reads."""
    D = dims
    bf = torch.bfloat16
    _expect(w["w_down"], bf, (D.L, D.d), "w_down")
    _expect(w["w_router"], bf, (D.E, D.L), "w_router")
    _expect(w["w_gate"], bf, (D.E, D.I, D.L), "w_gate")
    _expect(w["w_value"], bf, (D.E, D.I, D.L), "w_value")
    _expect(w["w_edown"], bf, (D.E, D.L, D.I), "w_edown")
    _expect(w["gamma"], torch.float32, (D.L,), "gamma")
    _expect(w["w_up"], bf, (D.d, D.L), "w_up")
    if D.S > 0:
        _expect(w["w_sgate"], bf, (D.S, D.Is, D.d), "w_sgate")
        _expect(w["w_svalue"], bf, (D.S, D.Is, D.d), "w_svalue")
        _expect(w["w_sdown"], bf, (D.S, D.d, D.Is), "w_sdown")
    nbytes = packed_bytes(D)
    if nbytes == 0:
        raise LmoeError(LMOE_ERR_UNSUPPORTED, "lmoe_packed_bytes")
    dev = w["w_down"].device
    packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    W = Weights(*[_ptr(w.get(n)) for n, _ in Weights._fields_])
    _check(load().lmoe_pack_weights(ctypes.byref(D), ctypes.byref(W), _ptr(packed), nbytes,
                                    _stream(stream)), "lmoe_pack_weights")
    return packed


def thresholds(logits: torch.Tensor, K: int, k_rank: int = 0, stream=None) -> torch.Tensor:
    T, E = logits.shape
    _expect(logits, torch.float32, (T, E), "logits")
    tau = torch.empty(E, dtype=torch.float32, device=logits.device)
    _check(load().lmoe_thresholds(_ptr(logits), T, E, K, k_rank, _ptr(tau), _stream(stream)),
           "lmoe_thresholds")
    return tau


def quantize_e4m3(x: torch.Tensor, stream=None):
    """Per-row e4m3 codes (uint8) and fp32 scales of bf16 rows (lmoe_quantize_e4m3)."""
    rows, cols = x.shape
    _expect(x, torch.bfloat16, (rows, cols), "x")
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    scales = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check(load().lmoe_quantize_e4m3(_ptr(x), rows, cols, _ptr(codes), _ptr(scales),
                                     _stream(stream)), "lmoe_quantize_e4m3")
    return codes, scales


def tau_ema(tau_step: torch.Tensor, tau_ema_: torch.Tensor, beta: float, first: bool = False,
            stream=None) -> torch.Tensor:
    """Fold one step's thresholds into the streaming thresholds, in place (lmoe_tau_ema)."""
    E = tau_step.shape[0]
    _expect(tau_step, torch.float32, (E,), "tau_step")
    _expect(tau_ema_, torch.float32, (E,), "tau_ema")
    _check(load().lmoe_tau_ema(_ptr(tau_step), _ptr(tau_ema_), E, beta, 1 if first else 0,
                               _stream(stream)), "lmoe_tau_ema")
    return tau_ema_


class LoadStats:
    """64-bit per-expert load counters on the device (layout at lmoe_load_stats_update),
    updated by ``Layer.forward(load_stats=...)`` or ``update(counts)``."""

    def __init__(self, E: int, device):
        self.E = E
        self.acc = torch.zeros(4 + 4 * E, dtype=torch.int64, device=device)

    def update(self, counts: torch.Tensor, stream=None):
        _expect(counts, torch.int32, (self.E,), "counts")
        _check(load().lmoe_load_stats_update(_ptr(counts), self.E, _ptr(self.acc),
                                             _stream(stream)), "lmoe_load_stats_update")

    def summary(self) -> dict:
        a = self.acc.cpu().numpy().astype(float)
        E, steps = self.E, max(a[0], 1.0)
        mean = a[1] / steps / E                     # tokens per expert per step
        per = a[4:4 + E] / steps
        return {"steps": int(a[0]), "fair_share": mean,
                "mean_max_over_mean": a[2] / steps / mean if mean else None,
                "worst_max_over_mean": a[3] / mean if mean else None,
                "expert_cv": float(per.std() / per.mean()) if per.mean() else None,
                "idle_expert_steps": int(a[4 + 2 * E:4 + 3 * E].sum())}


def ep_dispatch(idx: torch.Tensor, E: int, R: int, rows: torch.Tensor | None = None,
                stream=None) -> dict:
    """Expert-parallel dispatch over R ranks (lmoe_ep_dispatch): pair offsets per rank, the
    token and slot mask of each pair, and (with rows, bf16 [T, W]) each pair's row."""
    T, K = idx.shape
    _expect(idx, torch.int32, (T, K), "idx")
    dev = idx.device
    pmax = T * min(K, R)
    W = 0
    if rows is not None:
        W = rows.shape[1]
        _expect(rows, torch.bfloat16, (T, W), "rows")
    ws_bytes = int(load().lmoe_ep_workspace_bytes(T, K, E, R))
    if ws_bytes == 0:
        raise LmoeError(LMOE_ERR_UNSUPPORTED, "lmoe_ep_workspace_bytes")
    d = {"ws": torch.empty(ws_bytes, dtype=torch.uint8, device=dev),
         "send_off": torch.empty(R + 1, dtype=torch.int32, device=dev),
         "send_tok": torch.empty(pmax, dtype=torch.int32, device=dev),
         "send_slots": torch.empty(pmax, dtype=torch.int32, device=dev),
         "send_rows": torch.empty((pmax, W), dtype=torch.bfloat16, device=dev) if W else None,
         "E": E, "R": R}
    _check(load().lmoe_ep_dispatch(_ptr(idx), T, K, E, R, _ptr(rows), W, _ptr(d["send_rows"]),
                                   _ptr(d["send_off"]), _ptr(d["send_tok"]), _ptr(d["send_slots"]),
                                   _ptr(d["ws"]), ws_bytes, _stream(stream)), "lmoe_ep_dispatch")
    return d


def ep_combine(idx: torch.Tensor, disp: dict, inv: torch.Tensor, gate: torch.Tensor,
               o: torch.Tensor, stream=None):
    """Expert-parallel combine (lmoe_ep_combine): (part bf16 [pairs, W], u fp32 [T, W])."""
    T, K = idx.shape
    W = o.shape[1]
    _expect(o, torch.bfloat16, (o.shape[0], W), "o")
    _expect(inv, torch.int32, (T, K), "inv")
    _expect(gate, torch.float32, (T, K), "gate")
    part = torch.empty((T * min(K, disp["R"]), W), dtype=torch.bfloat16, device=o.device)
    u = torch.empty((T, W), dtype=torch.float32, device=o.device)
    _check(load().lmoe_ep_combine(_ptr(idx), T, K, disp["E"], disp["R"], _ptr(disp["send_off"]),
                                  _ptr(disp["send_tok"]), _ptr(disp["send_slots"]), _ptr(inv),
                                  _ptr(gate), _ptr(o), W, _ptr(part), _ptr(u), _ptr(disp["ws"]),
                                  _stream(stream)), "lmoe_ep_combine")
    return part, u


def fair_share_rank(T: int, K: int, E: int) -> int:
    """The threshold's rank among a column's T scores (lmoe_fair_share_rank)."""
    k = int(load().lmoe_fair_share_rank(T, K, E))
    if k < 0:
        raise LmoeError(LMOE_ERR_INVALID_ARG, "lmoe_fair_share_rank")
    return k


def threshold_candidates(logits: torch.Tensor, k: int, stream=None) -> torch.Tensor:
    """[k, E] candidates this batch contributes to thresholds solved over several batches
    (lmoe_threshold_candidates)."""
    T, E = logits.shape
    _expect(logits, torch.float32, (T, E), "logits")
    cand = torch.empty((k, E), dtype=torch.float32, device=logits.device)
    _check(load().lmoe_threshold_candidates(_ptr(logits), T, E, k, _ptr(cand), _stream(stream)),
           "lmoe_threshold_candidates")
    return cand


def gather_candidates(cand: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather every rank's [k, E] candidates into [world * k, E], rank order: the one
    exchange of a batch spread over ranks.  torch.distributed moves the bytes."""
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size(group) == 1:
        return cand
    world = dist.get_world_size(group)
    parts = [torch.empty_like(cand) for _ in range(world)]
    dist.all_gather(parts, cand.contiguous(), group=group)
    return torch.cat(parts, dim=0)


def global_token_count(T: int, device, group=None) -> int:
    """Sum of the ranks' batch sizes."""
    import torch.distributed as dist
    if not dist.is_initialized():
        return T
    dev = device if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([T], dtype=torch.int64, device=dev)
    dist.all_reduce(t, group=group)
    return int(t.item())


def route(logits: torch.Tensor, tau, K: int, want_scores: bool = False, stream=None):
    """Returns (idx int32 [T,K], gate fp32 [T,K]) and, with want_scores, scores [T,E]."""
    T, E = logits.shape
    _expect(logits, torch.float32, (T, E), "logits")
    if tau is not None:
        _expect(tau, torch.float32, (E,), "tau")
    dev = logits.device
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    gate = torch.empty((T, K), dtype=torch.float32, device=dev)
    sc = torch.empty((T, E), dtype=torch.float32, device=dev) if want_scores else None
    _check(load().lmoe_route(_ptr(logits), _ptr(tau), T, E, K, _ptr(idx), _ptr(gate), _ptr(sc),
                             _stream(stream)), "lmoe_route")
    return (idx, gate, sc) if want_scores else (idx, gate)


def gemm_bf16(A: torch.Tensor, B: torch.Tensor, stream=None) -> torch.Tensor:
    """C = A . B^T (fp32) on the tcgen05 GEMM of the library."""
    M, Kd = A.shape
    N = B.shape[0]
    _expect(A, torch.bfloat16, (M, Kd), "A")
    _expect(B, torch.bfloat16, (N, Kd), "B")
    C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    flag = torch.zeros(4, dtype=torch.int32, device=A.device)
    _check(load().lmoe_gemm_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, Kd, _ptr(flag),
                                 _stream(stream)), "lmoe_gemm_bf16")
    return C, flag


def gemm_wgrad_bf16(A: torch.Tensor, B: torch.Tensor, stream=None) -> torch.Tensor:
    """C = A^T . B (fp32) over all rows of token-major A [T, M] and B [T, N], as the backward's
    weight gradients compute it."""
    T, M = A.shape
    N = B.shape[1]
    _expect(A, torch.bfloat16, (T, M), "A")
    _expect(B, torch.bfloat16, (T, N), "B")
    C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    words = torch.zeros(4, dtype=torch.int32, device=A.device)
    _check(load().lmoe_gemm_wgrad_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, T, _ptr(words),
                                       _stream(stream)), "lmoe_gemm_wgrad_bf16")
    return C, words


def last_device_error(workspace: torch.Tensor) -> int:
    return int(load().lmoe_last_device_error(_ptr(workspace)))


class Layer:
    """One Stable Latent MoE layer on the device: packed weights + a workspace sized for up
    to ``max_tokens`` tokens.  ``forward`` is one lmoe_forward call."""

    def __init__(self, shape, weights: dict, max_tokens: int | None = None, stream=None,
                 overlap: bool = False, shared_sms: int = 0, expert_fp8: bool = False):
        """overlap: run the shared experts on an auxiliary stream beside the routed path for
        batches of at least OVERLAP_MIN_T tokens (shared_sms SMs for them; 0 = a third).
        Off by default: the routed expert GEMMs are limited per SM, so the SMs lent to the
        shared experts slow them down more than the concurrency gains.
        expert_fp8: routed experts with e4m3 operands (weights quantised when packed)."""
        self.shape = shape
        self.expert_fp8 = expert_fp8
        self.max_tokens = shape.T if max_tokens is None else max_tokens
        self.dims = dims_of(shape, T=self.max_tokens, expert_fp8=expert_fp8)
        self.device = weights["w_down"].device
        self.packed = pack_weights(self.dims, weights, stream)
        self.ws_bytes = workspace_bytes(self.dims)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.overlap = overlap
        self.shared_sms = shared_sms
        self.aux_stream = torch.cuda.Stream(device=self.device) if overlap else None
        self.aux_events = []
        if overlap:
            for _ in range(2):
                ev = torch.cuda.Event()
                ev.record(torch.cuda.current_stream(self.device))  # create the event now
                self.aux_events.append(ev)

    def forward(self, x: torch.Tensor, residual: torch.Tensor | None = None, y=None,
                tau: torch.Tensor | None = None, balance: bool = True,
                logits_in: torch.Tensor | None = None, debug: bool = False, stream=None,
                stage_events=None, phase: int = PHASE_ALL, cand_k: int = 0,
                tau_ema: torch.Tensor | None = None, ema_beta: float = 0.9,
                ema_first: bool = False, load_stats: "LoadStats | None" = None,
                train: bool = False, logit_bias: torch.Tensor | None = None):
        """One lmoe_forward call.  stage_events: optional list of NUM_STAGES + 1
        torch.cuda.Event(enable_timing=True) recorded at the stage boundaries.  After the
        call, ``self.last_kernel_launches`` holds the number of kernels it launched.
        phase: PHASE_ALL, or one half of the layer: PHASE_ROUTER (returns the [cand_k, E]
        threshold candidates when cand_k > 0, else None) then PHASE_EXPERTS (x gives the
        batch size only).  tau_ema: [E] streaming thresholds, updated in place with this
        batch's (ema_beta, ema_first) and routed against.  load_stats: a LoadStats that this
        step's per-expert counts are added to.  train: also keep the routed experts'
        pre-activations (lmoe_io.save_pre) for the next ``backward`` / ``backward_layer``
        (needs ``enable_backward``).  logit_bias: [E] fp32 added to the router logits the
        layer computes (lmoe_io.logit_bias)."""
        sh = self.shape
        T = x.shape[0]
        if T > self.max_tokens:
            raise ValueError(f"lmoe: {T} tokens exceed the workspace's {self.max_tokens}")
        _expect(x, torch.bfloat16, (T, sh.d), "x")
        if residual is not None:
            _expect(residual, torch.bfloat16, (T, sh.d), "residual")
        if y is None:
            y = torch.empty((T, sh.d), dtype=torch.bfloat16, device=x.device)
        dims = dims_of(sh, T=T, expert_fp8=self.expert_fp8)
        io = IO()
        io.balance = 1 if balance else 0
        io.phase = phase
        cand = None
        if phase == PHASE_ROUTER and cand_k > 0:
            cand = torch.empty((cand_k, sh.E), dtype=torch.float32, device=x.device)
            io.cand_out = _ptr(cand)
            io.cand_k = cand_k
        if self.overlap and T >= OVERLAP_MIN_T and T <= self.max_tokens:
            io.aux_stream = ctypes.c_void_p(self.aux_stream.cuda_stream)
            io.aux_events[0] = self.aux_events[0].cuda_event
            io.aux_events[1] = self.aux_events[1].cuda_event
            io.shared_sms = self.shared_sms
        dbg = {}
        if tau is not None:
            _expect(tau, torch.float32, (sh.E,), "tau")
            io.tau_in = _ptr(tau)
        if logits_in is not None:
            _expect(logits_in, torch.float32, (T, sh.E), "logits_in")
            io.logits_in = _ptr(logits_in)
        if logit_bias is not None:
            _expect(logit_bias, torch.float32, (sh.E,), "logit_bias")
            io.logit_bias = _ptr(logit_bias)
        if tau_ema is not None:
            _expect(tau_ema, torch.float32, (sh.E,), "tau_ema")
            io.tau_ema = _ptr(tau_ema)
            io.ema_beta = ema_beta
            io.ema_first = 1 if ema_first else 0
        if load_stats is not None:
            io.load_stats = _ptr(load_stats.acc)
        self._pre_rows = None
        if train:
            if getattr(self, "pre_buf", None) is None:
                raise RuntimeError("lmoe: forward(train=True) needs enable_backward() first")
            io.save_pre = _ptr(self.pre_buf)
            if self.pre_shared_buf is not None:
                io.save_pre_shared = _ptr(self.pre_shared_buf)
            self._pre_rows = T
        if debug:
            dev = x.device
            dbg["logits"] = torch.empty((T, sh.E), dtype=torch.float32, device=dev)
            dbg["tau"] = torch.empty(sh.E, dtype=torch.float32, device=dev)
            dbg["idx"] = torch.empty((T, sh.K), dtype=torch.int32, device=dev)
            dbg["gate"] = torch.empty((T, sh.K), dtype=torch.float32, device=dev)
            dbg["counts"] = torch.empty(sh.E, dtype=torch.int32, device=dev)
            if phase != PHASE_ROUTER:
                # the output before its bf16 store (y is this, rounded to nearest even)
                dbg["y_f32"] = torch.empty((T, sh.d), dtype=torch.float32, device=dev)
                io.y_f32_out = _ptr(dbg["y_f32"])
            io.logits_out = _ptr(dbg["logits"])
            io.tau_out = _ptr(dbg["tau"])
            io.idx_out = _ptr(dbg["idx"])
            io.gate_out = _ptr(dbg["gate"])
            io.counts_out = _ptr(dbg["counts"])
        if stage_events is not None:
            if len(stage_events) != NUM_STAGES + 1:
                raise ValueError(f"lmoe: need {NUM_STAGES + 1} stage events")
            handles = []
            for ev in stage_events:
                if not ev.cuda_event:      # torch creates its events lazily
                    ev.record(torch.cuda.current_stream() if stream is None else stream)
                handles.append(ev.cuda_event)
            arr = (_vp * len(handles))(*handles)
            io.stage_events = ctypes.cast(arr, ctypes.POINTER(_vp))
        _check(load().lmoe_forward(ctypes.byref(dims), _ptr(self.packed), _ptr(x), _ptr(residual),
                                   _ptr(y), _ptr(self.workspace), self.ws_bytes,
                                   ctypes.byref(io), _stream(stream)), "lmoe_forward")
        self.last_kernel_launches = io.kernel_launches
        if phase == PHASE_ROUTER:
            return (cand, dbg) if debug else cand
        return (y, dbg) if debug else y

    def forward_global(self, x: torch.Tensor, residual: torch.Tensor | None = None, y=None,
                       group=None, global_tokens: int | None = None, debug: bool = False,
                       stage_events=None):
        """The layer on this rank's part of a batch spread over the ranks of ``group``, with
        one set of Quantile-Balancing thresholds solved over the whole batch: router phase
        with candidates, all-gather of the candidates, lmoe_thresholds on them, experts
        phase.  Runs on the current stream (the collectives order against it)."""
        sh = self.shape
        T = x.shape[0]
        Tg = global_token_count(T, x.device, group) if global_tokens is None else global_tokens
        if Tg == 0:  # every rank's part is empty
            return self.forward(x, residual, y, debug=debug)
        k = fair_share_rank(Tg, sh.K, sh.E)
        r = self.forward(x, phase=PHASE_ROUTER, cand_k=k, debug=debug, stage_events=stage_events)
        launches = self.last_kernel_launches
        cand, dbg0 = r if debug else (r, None)
        tau = thresholds(gather_candidates(cand, group), sh.K, k_rank=k)
        out = self.forward(x, residual, y, tau=tau, phase=PHASE_EXPERTS, debug=debug,
                           stage_events=stage_events)
        self.last_kernel_launches += launches + 1
        if debug:
            out[1]["logits"] = dbg0["logits"]
            out[1]["candidates"] = cand
        return out

    def forward_host(self, x_host: torch.Tensor, y_host: torch.Tensor, x_dev: torch.Tensor,
                     y_dev: torch.Tensor, residual_from_x: bool = True, stream=None,
                     qb: str = "local", **kw):
        """End-to-end call from host memory: copy x (pinned host) to the device, run the
        layer, copy y back to pinned host memory; all on one stream, asynchronous.  Extra
        keyword arguments go to ``forward`` (tau, balance, logits_in), or, with
        qb="global", to ``forward_global`` (group, global_tokens)."""
        x_dev.copy_(x_host, non_blocking=True)
        resid = x_dev if residual_from_x else None
        if qb == "global":
            self.forward_global(x_dev, resid, y=y_dev, **kw)
        else:
            self.forward(x_dev, residual=resid, y=y_dev, stream=stream, **kw)
        y_host.copy_(y_dev, non_blocking=True)
        return y_host

    def device_error(self) -> int:
        return last_device_error(self.workspace)

    def enable_backward(self, weights: dict, stream=None):
        """Pack the transposed weights and allocate the scratch of ``backward`` and
        ``backward_layer``."""
        D = self.dims
        nb = int(load().lmoe_packed_backward_bytes(ctypes.byref(D)))
        if nb == 0:
            raise LmoeError(LMOE_ERR_UNSUPPORTED, "lmoe_packed_backward_bytes")
        self.packed_bwd = torch.empty(nb, dtype=torch.uint8, device=self.device)
        W = Weights(*[_ptr(weights.get(n)) for n, _ in Weights._fields_])
        _check(load().lmoe_pack_backward_weights(ctypes.byref(D), ctypes.byref(W),
                                                 _ptr(self.packed), _ptr(self.packed_bwd), nb,
                                                 _stream(stream)),
               "lmoe_pack_backward_weights")
        self.bwd_bytes = int(load().lmoe_backward_workspace_bytes(ctypes.byref(D)))
        # the routed pre-activations a training forward keeps (lmoe_io.save_pre)
        sh = self.shape
        self.pre_buf = torch.empty((self.max_tokens * sh.K, 2 * sh.I), dtype=torch.bfloat16,
                                   device=self.device)
        self.pre_shared_buf = None if sh.S == 0 else torch.empty(
            (self.max_tokens, 2 * sh.S * sh.Is), dtype=torch.bfloat16, device=self.device)
        self.bwd_ws = torch.empty(self.bwd_bytes, dtype=torch.uint8, device=self.device)

    def backward_launches(self, T: int) -> int:
        """Kernels one lmoe_routed_backward call for T tokens launches: combine backward, two
        dgamma passes, two grouped dgrad GEMMs (and the pre-activation GEMM when the last
        forward was not a training step), SiTU backward, slot sum, latent row gather, row
        map and two grouped weight-gradient GEMMs."""
        return 11 + (0 if getattr(self, "_pre_rows", None) == T else 1)

    def _saved_pre(self, T: int, shared: bool = False):
        """The routed (or shared) experts' pre-activations kept by the last forward, if it
        was a training step of T tokens; else None (the backward recomputes them)."""
        if getattr(self, "_pre_rows", None) != T:
            return None
        return _ptr(self.pre_shared_buf if shared else self.pre_buf)

    def backward(self, dz: torch.Tensor, stream=None) -> dict:
        """Gradients of the routed branch for the batch of the last ``forward`` call
        (lmoe_routed_backward): dz [T, L] fp32 -> dlat, dgate, dgamma, dw_gate, dw_value,
        dw_edown (fp32)."""
        sh = self.shape
        T = dz.shape[0]
        _expect(dz, torch.float32, (T, sh.L), "dz")
        dims = dims_of(sh, T=T, expert_fp8=self.expert_fp8)
        dev = dz.device
        f = torch.float32
        out = {"dlat": torch.empty((T, sh.L), dtype=f, device=dev),
               "dgate": torch.empty((T, sh.K), dtype=f, device=dev),
               "dgamma": torch.empty(sh.L, dtype=f, device=dev),
               "dw_gu": torch.empty((sh.E, 2 * sh.I, sh.L), dtype=f, device=dev),
               "dw_edown": torch.empty((sh.E, sh.L, sh.I), dtype=f, device=dev)}
        bwd_bytes = int(load().lmoe_routed_backward_workspace_bytes(ctypes.byref(dims)))
        _check(load().lmoe_routed_backward(
            ctypes.byref(dims), _ptr(self.packed), _ptr(self.packed_bwd), _ptr(self.workspace),
            self.ws_bytes, _ptr(dz), self._saved_pre(T), _ptr(out["dlat"]), _ptr(out["dgate"]), _ptr(out["dgamma"]),
            _ptr(out["dw_gu"]), _ptr(out["dw_edown"]), _ptr(self.bwd_ws), bwd_bytes,
            _stream(stream)), "lmoe_routed_backward")
        out["dw_gate"] = out["dw_gu"][:, :sh.I]
        out["dw_value"] = out["dw_gu"][:, sh.I:]
        return out

    def layer_backward_launches(self, T: int) -> int:
        """Kernels one lmoe_backward call launches: the routed branch's, plus the row map of
        dw_in, the dz GEMM, router backward and its GEMM, the dx GEMM and three
        weight-gradient GEMMs; with shared experts also the dhs GEMM and their SiTU backward,
        and their pre-activation GEMM unless the last forward was a training step."""
        shared = 0
        if self.shape.S > 0:
            shared = 2 + (0 if getattr(self, "_pre_rows", None) == T else 1)
        return self.backward_launches(T) + 8 + shared

    def backward_layer(self, x: torch.Tensor, dy: torch.Tensor, logits=None,
                       stream=None) -> dict:
        """Gradients of the whole layer for the batch of the last ``forward`` call
        (lmoe_backward): x [T, d] bf16 (that call's input), dy [T, d] bf16 ->
        dx (through the latent and the shared experts; the residual adds dy), dgamma and
        every weight's gradient, fp32, in the weights' own shapes (dw_up, dw_sdown and the
        shared gate/value gradients are views into the packed gradient buffers).  logits:
        the fp32 [T, E] logits the forward routed on, when it was given ``logits_in``."""
        sh = self.shape
        T = x.shape[0]
        _expect(x, torch.bfloat16, (T, sh.d), "x")
        _expect(dy, torch.bfloat16, (T, sh.d), "dy")
        if logits is not None:
            _expect(logits, torch.float32, (T, sh.E), "logits")
        dims = dims_of(sh, T=T, expert_fp8=self.expert_fp8)
        dev = x.device
        f = torch.float32
        S, Is, L, d = sh.S, sh.Is, sh.L, sh.d
        sw = S * Is
        out = {"dx": torch.empty((T, d), dtype=f, device=dev),
               "dgamma": torch.empty(L, dtype=f, device=dev),
               "dw_in": torch.empty((L + 2 * sw, d), dtype=f, device=dev),
               "dw_router": torch.empty((sh.E, L), dtype=f, device=dev),
               "dw_gu": torch.empty((sh.E, 2 * sh.I, L), dtype=f, device=dev),
               "dw_edown": torch.empty((sh.E, L, sh.I), dtype=f, device=dev),
               "dw_out": torch.empty((d, L + sw), dtype=f, device=dev)}
        bwd_bytes = int(load().lmoe_backward_workspace_bytes(ctypes.byref(dims)))
        _check(load().lmoe_backward(
            ctypes.byref(dims), _ptr(self.packed), _ptr(self.packed_bwd), _ptr(self.workspace),
            self.ws_bytes, _ptr(x), _ptr(logits), _ptr(dy), self._saved_pre(T),
            self._saved_pre(T, shared=True), _ptr(out["dx"]),
            _ptr(out["dgamma"]), _ptr(out["dw_in"]), _ptr(out["dw_router"]), _ptr(out["dw_gu"]),
            _ptr(out["dw_edown"]), _ptr(out["dw_out"]), _ptr(self.bwd_ws), bwd_bytes,
            _stream(stream)), "lmoe_backward")
        out["dw_down"] = out["dw_in"][:L]
        out["dw_sgate"] = out["dw_in"][L:L + sw].view(S, Is, d)
        out["dw_svalue"] = out["dw_in"][L + sw:].view(S, Is, d)
        out["dw_gate"] = out["dw_gu"][:, :sh.I]
        out["dw_value"] = out["dw_gu"][:, sh.I:]
        out["dw_up"] = out["dw_out"][:, :L]
        out["dw_sdown"] = out["dw_out"][:, L:].unflatten(1, (S, Is)).permute(1, 0, 2)
        return out


class HostPipeline:
    """The layer on batches that live in pinned host memory, overlapped across batches: each
    ``submit`` is one lmoe_forward_host call (the upload of x, the layer and the download of
    y on three streams, through one of ``depth`` device staging slots), so batch i + 1's
    upload and batch i - 1's download run while batch i computes.  The library orders every
    reuse of a slot with the pipe's events; this class owns the slots, streams and events.
    ``synchronize`` waits for every submitted batch."""

    def __init__(self, layer: "Layer", depth: int = 2):
        if not 1 <= depth <= HOST_PIPE_MAX_DEPTH:
            raise ValueError(f"lmoe: pipeline depth must be 1..{HOST_PIPE_MAX_DEPTH}")
        self.layer = layer
        self.depth = depth
        T, d = layer.max_tokens, layer.shape.d
        dev = layer.device
        self.x = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        self.y = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        self.up = torch.cuda.Stream(device=dev)
        self.compute = torch.cuda.Stream(device=dev)
        self.down = torch.cuda.Stream(device=dev)
        self.events = [[torch.cuda.Event() for _ in range(3)] for _ in range(depth)]
        for evs in self.events:  # torch creates its events lazily: record each once
            for ev in evs:
                ev.record(self.compute)
        self.compute.synchronize()
        p = HostPipe()
        p.depth, p.max_tokens = depth, T
        for k in range(depth):
            p.x_dev[k] = self.x[k].data_ptr()
            p.y_dev[k] = self.y[k].data_ptr()
            p.uploaded[k] = self.events[k][0].cuda_event
            p.computed[k] = self.events[k][1].cuda_event
            p.downloaded[k] = self.events[k][2].cuda_event
        p.upload = self.up.cuda_stream
        p.compute = self.compute.cuda_stream
        p.download = self.down.cuda_stream
        p.calls = 0
        self.pipe = p

    def submit(self, x_host: torch.Tensor, y_host: torch.Tensor, residual_from_x: bool = True,
               tau: torch.Tensor | None = None, balance: bool = True,
               logit_bias: torch.Tensor | None = None):
        """Enqueue one batch: x_host [T, d] bf16 pinned in, y_host pinned out."""
        layer, sh = self.layer, self.layer.shape
        T = x_host.shape[0]
        if T > layer.max_tokens:
            raise ValueError(f"lmoe: {T} tokens exceed the pipeline's {layer.max_tokens}")
        _expect(x_host, torch.bfloat16, (T, sh.d), "x_host")
        _expect(y_host, torch.bfloat16, (T, sh.d), "y_host")
        if x_host.is_cuda or y_host.is_cuda or not x_host.is_contiguous() or \
                not y_host.is_contiguous():
            raise ValueError("lmoe: x_host and y_host must be contiguous host tensors")
        io = IO()
        io.balance = 1 if balance else 0
        if tau is not None:
            _expect(tau, torch.float32, (sh.E,), "tau")
            io.tau_in = _ptr(tau)
        if logit_bias is not None:
            _expect(logit_bias, torch.float32, (sh.E,), "logit_bias")
            io.logit_bias = _ptr(logit_bias)
        dims = dims_of(sh, T=T, expert_fp8=layer.expert_fp8)
        _check(load().lmoe_forward_host(ctypes.byref(dims), _ptr(layer.packed),
                                        ctypes.c_void_p(x_host.data_ptr()),
                                        1 if residual_from_x else 0,
                                        ctypes.c_void_p(y_host.data_ptr()),
                                        _ptr(layer.workspace), layer.ws_bytes, ctypes.byref(io),
                                        ctypes.byref(self.pipe)), "lmoe_forward_host")
        layer.last_kernel_launches = io.kernel_launches

    def synchronize(self):
        for s in (self.up, self.compute, self.down):
            s.synchronize()
