"""Benchmark of the Stable Latent MoE layer on GB300.

Workload (one "step" = one lmoe_forward over one batch): the K3 prefill layer, T=8192
tokens, d=7168, latent 3584, E=896 routed experts, top-16, 2 shared experts (I_s=2048),
routed I=512, bf16 with fp32 accumulation; x ~ N(0,1) with 0.1 % of its elements x1000;
weights ~ N(0, 1/fan_in) (router weights scaled to keep the logits ~N(0,1) under those
outliers); in-batch Quantile-Balancing thresholds; residual = x.  Synthetic data, seed 2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch on its own GPU
(weak scaling); the time is the max over ranks.  By default each rank solves its own
thresholds (no collective on the data path); ``--qb global`` solves one set over all
ranks' batches (router phase, all-gather of threshold candidates, experts phase).
``--impl reference`` times the CPU oracle (the only reference there is) on host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import glob
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from latent_compressed_expert_gb300 import lmoe, synth  # noqa: E402

METRIC = "latent-MoE layer tokens/s at 896E/top-16; TFLOP/s & % bf16 / HBM roofline"
UNIT = "tokens/s"
SEED = 2
OUTLIER_FRAC, OUTLIER_SCALE = 0.001, 1000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------------------
# algorithmic work of each stage (what the method must read/write/compute at minimum)
# ----------------------------------------------------------------------------------------
def stage_work(sh, touched: int, residual: bool = True, fp8: bool = False) -> dict:
    T, d, L, E, K, I, S, Is = sh.T, sh.d, sh.L, sh.E, sh.K, sh.I, sh.S, sh.Is
    sw = S * Is
    bf, f4 = 2, 4
    TK = T * K
    w = {
        "latent_shared": (2.0 * T * d * (L + 2 * sw),
                          (T * d + (L + 2 * sw) * d + T * L + T * sw) * bf),
        "router": (2.0 * T * L * E, (T * L + E * L) * bf + T * E * f4),
        "thresholds": (0.0, T * E * f4 + E * f4),
        "route": (0.0, T * E * f4 + E * f4 + T * K * 8),
        # indices only: idx read, per-block masks/bases, inv and source-token written
        "dispatch": (0.0, T * K * 4 * 3 + 2 * ((T + 31) // 32) * E * 4),
        # the latent rows are gathered inside the GEMM: read once (L2 serves the repeats)
        "expert_gate_up": (2.0 * T * K * L * 2 * I,
                           touched * 2 * I * L * bf + T * L * bf + T * K * I * bf),
        "expert_down": (2.0 * T * K * I * L, touched * L * I * bf + T * K * (I + L) * bf),
        "combine": (0.0, T * K * L * bf + T * K * 8 + T * L * bf + L * f4),
        "output": (2.0 * T * (L + sw) * d,
                   (T * (L + sw) + d * (L + sw) + T * d * (2 if residual else 1)) * bf),
    }
    if fp8:
        # e4m3 operands: one byte per weight plus a scale per row; the stage also quantises
        # its activation rows (bf16 read, codes + scale written) before the GEMM reads them
        w["expert_gate_up"] = (2.0 * TK * L * 2 * I,
                               touched * 2 * I * (L + f4) + T * L * bf + T * (L + f4)
                               + T * L + TK * I * bf)
        w["expert_down"] = (2.0 * TK * I * L,
                            TK * I * bf + TK * (I + f4) + touched * L * (I + f4) + TK * I
                            + TK * L * bf)
    return {k: {"flop": v[0], "bytes": float(v[1])} for k, v in w.items()}


def layer_work(sh, touched: int, fp8: bool = False) -> tuple[float, float]:
    """FLOP of the layer (461.5 MFLOP per token at the K3 shape) and its algorithmic bytes:
    every touched weight once, x and the residual read, y written."""
    T, d, L, E, K, I, S, Is = sh.T, sh.d, sh.L, sh.E, sh.K, sh.I, sh.S, sh.Is
    flop_tok = 2.0 * (d * L + L * E + K * (L * 2 * I + I * L) + 3 * S * Is * d + L * d)
    routed = touched * 3 * I * L * (1 if fp8 else 2) + (touched * (2 * I + L) * 4 if fp8 else 0)
    wbytes = (L * d + E * L + L * d + 3 * S * Is * d) * 2 + routed + L * 4
    return flop_tok * T, float(wbytes + 3 * T * d * 2)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"]))}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# The source files that define each stage's kernel and its launch configuration (the
# launcher sits in the kernel's own .cu), plus the headers every kernel includes.
_COMMON_SRC = ("common.cuh", "kernels.cuh", "ptx.cuh", "lmoe.h")
STAGE_SOURCES = {
    "latent_shared": ("gemm.cu",), "router": ("gemm.cu",), "output": ("gemm.cu",),
    "thresholds": ("routing.cu",), "route": ("routing.cu",), "dispatch": ("dispatch.cu",),
    "expert_gate_up": ("gemm_grouped.cu",), "expert_down": ("gemm_grouped.cu",),
    "combine": ("dispatch.cu",),
}


_COMMENT = re.compile(rb"/\*.*?\*/|//[^\n]*", re.S)


def kernel_source_hash(stage: str) -> str:
    """Hash of the sources of one stage's kernel, comments and blank space left out: a
    stored ncu figure is valid while it matches."""
    h = hashlib.sha256()
    for name in sorted(STAGE_SOURCES[stage] + _COMMON_SRC):
        path = os.path.join(ROOT, "include" if name.endswith(".h") else
                            os.path.join("latent_compressed_expert_gb300", "csrc"), name)
        with open(path, "rb") as f:
            code = b" ".join(_COMMENT.sub(b" ", f.read()).split())
        h.update(name.encode())
        h.update(code)
    return h.hexdigest()[:16]


def ncu_traffic(stage: str, table: str = "stages"):
    """DRAM bytes per launch of a stage's kernel from a committed ncu summary, if it was
    captured from the current sources of that kernel; else None.  table: "stages" (bf16
    routed experts) or "stages_fp8"."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        t = json.load(f)
    s = t.get(table, {}).get(stage)
    if s is None or s.get("kernel_source_hash") != kernel_source_hash(stage):
        return None
    return float(s["dram_bytes_per_launch"])


# ----------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------
# the CPU oracle on a bounded sample (reported baseline, and the reference arm)
# ----------------------------------------------------------------------------------------
def batch_thresholds(oracle, wh, xh, K):
    """The batch-wide part of the layer on the host: the latent and router logits of every
    token, and the Quantile-Balancing thresholds over the whole batch.  Returns
    (lat, logits, tau, seconds)."""
    t0 = time.perf_counter()
    lat = oracle.latent(xh, wh["w_down"])
    lg = oracle.router_logits(lat, wh["w_router"]).astype(np.float32)
    tau = oracle.thresholds(lg, oracle.fair_share_rank(lg.shape[0], K, lg.shape[1]))
    return lat, lg, tau, time.perf_counter() - t0


def oracle_rest(oracle, wh, x_rows, lat_rows, lg_rows, tau, K, c=100.0, eps=1e-6):
    """The per-token rest of the layer for some tokens, given their latent and logits and the
    batch's thresholds: routing, routed experts, combine and RMSNorm, shared experts,
    up-projection and residual."""
    idx, gate, _ = oracle.route(lg_rows, tau, K)
    z = oracle.routed(lat_rows, idx, gate, wh["w_gate"], wh["w_value"], wh["w_edown"],
                      wh["gamma"].numpy(), c, eps)
    ys = oracle.shared(x_rows, wh["w_sgate"], wh["w_svalue"], wh["w_sdown"], c)
    return oracle.output(z, ys, wh["w_up"], x_rows)


def oracle_tokens(oracle, wh, x_rows, tau, K):
    """The whole layer's per-token work for some tokens (latent, logits, then the rest),
    routed against thresholds solved over their whole batch."""
    lat = oracle.latent(x_rows, wh["w_down"])
    lg = oracle.router_logits(lat, wh["w_router"]).astype(np.float32)
    return oracle_rest(oracle, wh, x_rows, lat, lg, tau, K)


def host_weights(w):
    return {k: v.detach().cpu() for k, v in w.items()}


SUBSET_TOKENS = 512


def cpu_baseline(sh, wh, xh, args):
    """The fp64 oracle on the host cores: the batch-wide stage (latent and logits of all T
    tokens, thresholds over the batch) timed in full, and the per-token rest of the layer on
    a fixed subset of 512 tokens; the layer's host time for the batch is the first plus the
    second scaled by T / 512 (its cost is linear in tokens)."""
    import oracle
    oracle.build()
    lat, lg, tau, t_batch = batch_thresholds(oracle, wh, xh, sh.K)
    n = min(sh.T, args.cpu_tokens if args.cpu_tokens > 0 else SUBSET_TOKENS)
    rows = np.linspace(0, sh.T - 1, n).astype(np.int64)  # fixed, spread over the batch
    t0 = time.perf_counter()
    oracle_rest(oracle, wh, xh[rows].contiguous(), lat[rows], lg[rows], tau, sh.K)
    t_rest = time.perf_counter() - t0
    t_layer = t_batch + t_rest * sh.T / n
    return {"value": sh.T / t_layer, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"latent, router logits and thresholds of all {sh.T} tokens ({t_batch:.1f} s) "
                      f"+ the rest of the layer for a fixed subset of {n} tokens "
                      f"({t_rest:.1f} s), scaled to the batch: {t_layer:.1f} s per {sh.T}-token step",
            "batch_stage_s": t_batch, "subset_tokens": n, "subset_rest_s": t_rest}


# ----------------------------------------------------------------------------------------
def dist_setup(n_gpus, backend=None):
    """Rank, world size and local rank from the torchrun environment; one GPU per rank."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    on_gpu = dist.get_backend() == "nccl"
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


SMALL = synth.LayerShape("small", T=1024, d=7168, L=3584, E=128, K=16, I=512, S=2, Is=2048)
# the K3 routing shape (T=8192, E=896, top-16) with narrow widths: the threshold, top-K and
# dispatch kernels run at full size on a device footprint of well under 1 GB
ROUTING = synth.LayerShape("routing", T=8192, d=512, L=256, E=896, K=16, I=64, S=2, Is=128)
# the alternative pool the pages weigh against 896 / top-16: 448 experts, 8 per token
POOL448 = synth.LayerShape("pool448", T=8192, d=7168, L=3584, E=448, K=8, I=512, S=2, Is=2048)
WGRAD = synth.LayerShape("wgrad", T=584, d=7168, L=3584, E=64, K=16, I=512, S=2, Is=2048)
# the skewed workload's expert load (~585 tokens per expert, tensor-bound routed GEMMs) on
# 128 experts: a profiling case of a few GB
SKEW_SMALL = synth.LayerShape("skew_small", T=4688, d=7168, L=3584, E=128, K=16, I=512, S=2,
                              Is=2048)
SHAPES = {"prefill": synth.PREFILL, "decode": synth.DECODE, "e64": synth.E64,
          "skew": synth.SKEW, "small": SMALL, "routing": ROUTING, "pool448": POOL448,
          "wgrad": WGRAD, "skew_small": SKEW_SMALL}
DESCRIPTIONS = {
    "prefill": "K3 Stable Latent MoE layer, prefill: in-batch Quantile-Balancing thresholds; "
               "x~N(0,1) with 0.1% of elements x1000; residual = x",
    "decode": "K3 layer, decode: thresholds from a 8192-token prefill batch of the same "
              "layer passed in; x~N(0,1); residual = x",
    "e64": "K3 widths with a reduced pool (E=64, top-4): in-batch thresholds; x~N(0,1); "
           "residual = x",
    "skew": "K3 layer, skewed router: a per-expert Zipf(1.1) bias -1.1 ln(rank) added to "
            "the router logits in the router GEMM's epilogue, in-batch thresholds; x~N(0,1); "
            "residual = x",
    "small": "K3 widths, 128 experts, T=1024 (profiling case: ~128 tokens per expert as "
             "in prefill, a few GB on the device); x as in prefill",
    "pool448": "K3 widths with the alternative pool of 448 routed experts, top-8 (the same "
               "1/56 activation ratio, half the routed FLOPs); x as in prefill; in-batch "
               "thresholds",
    "routing": "K3 routing shape with narrow widths (profiling case for the threshold, "
               "top-K and dispatch kernels at T=8192, E=896, top-16); x~N(0,1); in-batch "
               "thresholds",
    "skew_small": "K3 widths, 128 experts, T=4688 (profiling case: ~585 tokens per expert as "
                  "in the skewed workload after balancing, a few GB on the device); x~N(0,1); "
                  "in-batch thresholds",
    "wgrad": "K3 widths, 64 experts, T=584 (profiling case for the backward's weight-gradient "
             "GEMMs: 146 tokens per expert as in prefill, a few GB on the device); x as in "
             "prefill",
}


class Workload:
    """Inputs and routing arguments of one bench configuration."""

    def __init__(self, name, dev, rank, overlap=False, shared_sms=0, qb="local", world=1,
                 expert_fp8=False):
        self.name = name
        self.qb = qb
        self.fp8 = expert_fp8
        self.sh = sh = SHAPES[name]
        outliers = name in ("prefill", "small", "pool448", "wgrad")
        gain = synth.outlier_router_gain(sh, OUTLIER_FRAC, OUTLIER_SCALE) if outliers else 1.0
        self.w = synth.make_weights(sh, SEED, device=dev, router_gain=gain)
        self.x = synth.make_x(sh, SEED + 1000 * rank, device=dev,
                              outlier_frac=OUTLIER_FRAC if outliers else 0.0,
                              outlier_scale=OUTLIER_SCALE)
        self.layer = lmoe.Layer(sh, self.w, max_tokens=max(sh.T, 8192 if name == "decode" else 0),
                                overlap=overlap, shared_sms=shared_sms, expert_fp8=expert_fp8)
        self.kwargs = {}
        self.extra = {}
        if qb == "global":
            if name not in ("prefill", "e64", "small", "routing", "pool448", "wgrad"):
                raise ValueError("--qb global applies to the in-batch-threshold workloads")
            # thresholds over all ranks' batches together (all-gather of candidates)
            self.kwargs["global_tokens"] = sh.T * world
        if name == "decode":
            # thresholds of a prefill batch through the same layer
            xp = synth.make_x(sh, SEED + 7, device=dev, T=8192)
            _, dbg = self.layer.forward(xp, debug=True)
            self.kwargs["tau"] = dbg["tau"].clone()
            del xp, dbg
        if name == "skew":
            # the Zipf bias enters in the router GEMM's epilogue, so the step routes on
            # biased logits it computes itself
            self.kwargs["logit_bias"] = synth.zipf_bias(sh.E, SEED, 1.1, device=dev)
            _, plain = self.layer.forward(self.x, debug=True, balance=False,
                                          logit_bias=self.kwargs["logit_bias"])
            fair = sh.T * sh.K / sh.E
            c0 = plain["counts"].float()
            self.extra["load_before"] = {"max_over_mean": float(c0.max() / fair),
                                         "min_over_mean": float(c0.min() / fair),
                                         "idle_experts": int((c0 == 0).sum())}
            del plain

    def forward(self, **kw):
        if self.qb == "global":
            return self.layer.forward_global(self.x, residual=self.x, **self.kwargs, **kw)
        return self.layer.forward(self.x, residual=self.x, **self.kwargs, **kw)

    def config(self, world):
        sh = self.sh
        return {"workload": f"{DESCRIPTIONS[self.name]}. T={sh.T} tokens, d={sh.d}, "
                            f"latent {sh.L}, E={sh.E} routed top-{sh.K}, {sh.S} shared experts "
                            f"(I_s={sh.Is}), routed I={sh.I}",
                "shape": self.name, "tokens_per_gpu": sh.T, "global_tokens": sh.T * world,
                "l2": "inputs larger than L2: the expert weights streamed per step exceed it",
                "parallelism": f"replicas x{world}, independent batches" if self.qb == "local"
                               else f"data parallel x{world}, Quantile-Balancing thresholds over "
                                    f"the {sh.T * world}-token global batch (all-gather of "
                                    f"per-rank candidates)",
                "shared_experts": "in line" if not self.layer.overlap else
                                  f"second stream, {self.layer.shared_sms or 'default'} SMs",
                "routed_experts": "e4m3 operands, one fp32 scale per row" if self.fp8
                                  else "bf16"}


def make_inputs(sh, dev, rank, outliers=True):
    """The same weights and x that Workload draws (for the CPU-only reference arm)."""
    gain = synth.outlier_router_gain(sh, OUTLIER_FRAC, OUTLIER_SCALE) if outliers else 1.0
    w = synth.make_weights(sh, SEED, device=dev, router_gain=gain)
    x = synth.make_x(sh, SEED + 1000 * rank, device=dev,
                     outlier_frac=OUTLIER_FRAC if outliers else 0.0, outlier_scale=OUTLIER_SCALE)
    return w, x


def run_reference(args):
    """The oracle (the only reference there is) on the host cores.  Set-up: the batch-wide
    stage (latent and logits of all T tokens, thresholds over the batch), timed and
    reported.  Each step: the whole layer's per-token work (latent, logits, routing against
    those thresholds, experts, shared experts, output) for a sub-batch of n tokens, sized so
    that warm-up and steps take about 2-3 minutes; value = tokens per second of those steps."""
    world, rank, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    sh = SHAPES[args.shape]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w, x = make_inputs(sh, dev, 0, outliers=args.shape in ("prefill", "small"))
    wh = host_weights(w)
    xh = x.cpu()
    del w, x
    import oracle
    oracle.build()
    _, _, tau, t_batch = batch_thresholds(oracle, wh, xh, sh.K)
    t0 = time.perf_counter()
    oracle_tokens(oracle, wh, xh[:4].contiguous(), tau, sh.K)
    rate = 4 / (time.perf_counter() - t0)
    n = int(max(1, min(64, rate * 150.0 / max(1, args.steps + args.warmup))))
    for i in range(args.warmup):
        oracle_tokens(oracle, wh, xh[i * n:(i + 1) * n].contiguous(), tau, sh.K)
    t0 = time.perf_counter()
    for i in range(args.steps):
        s = (i * n) % (sh.T - n)
        oracle_tokens(oracle, wh, xh[s:s + n].contiguous(), tau, sh.K)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    cores = oracle.num_threads()
    sample = (f"{n} tokens of the {sh.T}-token batch per step through the whole layer's "
              f"per-token work, routed against thresholds solved over the whole batch "
              f"(that batch-wide stage took {t_batch:.1f} s once, before the steps)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{DESCRIPTIONS[args.shape]}. T={sh.T} tokens, d={sh.d}, "
                                   f"latent {sh.L}, E={sh.E} routed top-{sh.K}, {sh.S} shared "
                                   f"experts (I_s={sh.Is}), routed I={sh.I}",
                       "shape": args.shape, "tokens_per_gpu": sh.T, "global_tokens": sh.T},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, "batch_stage_s": t_batch},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# Timed regions shorter than this are compared with the burst bf16 peak, longer ones with the
# sustained one (a kernel timed alone vs. inside a long run under the power cap).
BURST_REGION_S = 1.0


def pick_peak(peaks, region_s):
    if region_s < BURST_REGION_S:
        return peaks["bf16_tflops"], "bf16 burst"
    return peaks["bf16_tflops_sustained"], "bf16 sustained"


def time_workload(wl, steps, warmup, world, local, stream):
    """`warmup` untimed steps, then `steps` timed ones between a barrier and device
    synchronisations, with CUDA events at every stage boundary on the launching stream and
    nvidia-smi clock samples.  Returns the step time (max over ranks) and per-stage means."""
    layer, x = wl.layer, wl.x
    y = torch.empty_like(x)
    for _ in range(warmup):  # also learns how many experts a step touches
        _, dbg = wl.forward(y=y, debug=True)
    torch.cuda.synchronize()
    if layer.device_error() != 0:
        raise RuntimeError(f"device-side error during warm-up ({wl.name})")
    counts = dbg["counts"].cpu().numpy()
    launches = layer.last_kernel_launches
    del dbg
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(lmoe.NUM_STAGES + 1)]
           for _ in range(steps)]
    for e in evs:  # create the events outside the timed region
        for ev in e:
            ev.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(steps):
            wl.forward(y=y, stage_events=evs[i])
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(end)
    if layer.device_error() != 0:
        raise RuntimeError(f"device-side error in the timed region ({wl.name})")
    stage_ms = {name: float(np.mean([evs[i][s].elapsed_time(evs[i][s + 1])
                                     for i in range(steps)]))
                for s, name in enumerate(lmoe.STAGES)}
    return {"ms": max_over_ranks(ms, world), "stage_ms": stage_ms, "counts": counts,
            "touched": int((counts > 0).sum()), "launches": launches, "clocks": clk.summary(),
            "y": y}


def dominant_roofline(wl, r, peaks, peak_src, region_s):
    """Roofline of the stage that takes the most time: algorithmic FLOP or bytes of one
    launch over its mean CUDA-event duration, against the measured peak of its bound."""
    sh = wl.sh
    work = stage_work(sh, r["touched"], fp8=wl.fp8)
    stage_ms = r["stage_ms"]
    dom = max(stage_ms, key=stage_ms.get)
    dw = work[dom]
    t_s = stage_ms[dom] / 1e3
    tflops, kind = pick_peak(peaks, region_s)
    t_flop = dw["flop"] / (tflops * 1e12)
    t_byte = dw["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if t_flop >= t_byte:
        roof = {"bound": "tensor", "achieved": dw["flop"] / t_s / 1e12, "peak": tflops,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": dw["bytes"] / t_s / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
        kind = "HBM copy"
    roof["frac"] = roof["achieved"] / roof["peak"]
    # the stored figures are captures of the prefill workload (in-batch thresholds)
    roof["traffic"] = (ncu_traffic(dom, "stages_fp8" if wl.fp8 and dom.startswith("expert")
                                   else "stages")
                       if wl.name == "prefill" and wl.qb == "local" else None)
    roof["kernel"] = dom
    roof["peak_source"] = f"{peak_src} ({kind})"
    roof["algorithmic"] = {"flop": dw["flop"], "bytes": dw["bytes"]}
    stages = {}
    for name in lmoe.STAGES:
        sw_ = work[name]
        t = stage_ms[name] / 1e3
        stages[name] = {"ms": round(stage_ms[name], 4),
                        "tflops": round(sw_["flop"] / t / 1e12, 1) if t > 0 and sw_["flop"] else None,
                        "gbs": round(sw_["bytes"] / t / 1e9, 1) if t > 0 else None}
    return roof, stages


def load_summary(sh, counts):
    fair = sh.T * sh.K / sh.E
    return {"max_over_mean": float(counts.max() / fair),
            "min_over_mean": float(counts.min() / fair),
            "idle_experts": int((counts == 0).sum())}


# The other workloads of the layer reported inside the headline line: steps per timed
# region (each region stays well under a second).
CONFIG_STEPS = {"decode": 60, "skew": 10, "e64": 40}


def run_configs(args, dev, rank, world, local, stream, peaks, peak_src):
    """Decode, skewed-router and reduced-pool (E=64) workloads, each timed as the headline
    is (device-resident inputs, CUDA events, max over ranks)."""
    out = {}
    for name in ("decode", "skew", "e64"):
        wl = Workload(name, dev, rank, world=world, expert_fp8=args.experts == "fp8")
        steps = min(args.steps, CONFIG_STEPS[name])
        r = time_workload(wl, steps, 3, world, local, stream)
        sh = wl.sh
        step_s = r["ms"] / 1e3 / steps
        region_s = r["ms"] / 1e3
        flop, nbytes = layer_work(sh, r["touched"], fp8=wl.fp8)
        tflops, kind = pick_peak(peaks, region_s)
        roof, stages = dominant_roofline(wl, r, peaks, peak_src, region_s)
        c = {"workload": wl.config(world)["workload"], "steps": steps, "warmup": 3,
             "ms_per_step": r["ms"] / steps, "value": world * sh.T / step_s, "unit": UNIT,
             "tflops": flop / step_s / 1e12, "frac_bf16_peak": flop / step_s / 1e12 / tflops,
             "bf16_peak": f"{tflops} TFLOP/s ({peak_src}, {kind})",
             "experts_touched": r["touched"], "roofline": roof, "stages": stages,
             "clocks": r["clocks"], "gpu_launches": r["launches"] * steps}
        if name == "decode":
            c["decode_weight_gbs"] = nbytes / step_s / 1e9
            c["decode_frac_hbm"] = c["decode_weight_gbs"] / peaks["hbm_gbs"]
            c["decode_target_frac_hbm"] = 0.70
            c["decode_bytes"] = ("weights of the experts the step touches, the dense weights, "
                                 "x, residual and y, each once")
        if name == "skew":
            c["load"] = {"before_balancing": wl.extra["load_before"],
                         "after_balancing": load_summary(sh, r["counts"])}
        else:
            c["load"] = load_summary(sh, r["counts"])
        out[name] = c
        del wl, r
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    world, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (the layer has no CPU path)")
    dev = torch.device("cuda", local)
    wl = Workload(args.shape, dev, rank, overlap=args.overlap, shared_sms=args.shared_sms,
                  qb=args.qb, world=world, expert_fp8=args.experts == "fp8")
    sh, layer, x, w = wl.sh, wl.layer, wl.x, wl.w
    stream = torch.cuda.current_stream()

    # ---- timed region: device-resident inputs
    r = time_workload(wl, args.steps, args.warmup, world, local, stream)
    ms_max, stage_ms, counts, touched = r["ms"], r["stage_ms"], r["counts"], r["touched"]
    launches_per_step = r["launches"]
    y = r["y"]

    # ---- end to end through the C ABI with host buffers: every step uploads its x from
    # pinned host memory and downloads its y; lmoe_forward_host (lmoe.HostPipeline) overlaps
    # one step's copies with the neighbouring steps' compute (global thresholds need the
    # collective between phases, so that mode uses the serial host path)
    x_host = x.cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    if wl.qb == "global":
        x_dev = torch.empty_like(x)
        run_e2e = lambda: layer.forward_host(x_host, y_host, x_dev, y, qb=wl.qb, **wl.kwargs)
        finish = torch.cuda.synchronize
        first_stream = last_stream = stream
    else:
        pipe = lmoe.HostPipeline(layer, depth=2)
        run_e2e = lambda: pipe.submit(x_host, y_host, **wl.kwargs)
        finish = pipe.synchronize
        first_stream, last_stream = pipe.up, pipe.down
    for _ in range(max(1, args.warmup)):
        run_e2e()
    finish()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    e0.record(first_stream)
    for _ in range(args.steps):
        run_e2e()
    e1.record(last_stream)
    finish()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    if wl.qb != "global":
        del pipe

    T = sh.T
    value = world * T * args.steps / (ms_max / 1e3)
    e2e_value = world * T * args.steps / (e2e_ms / 1e3)
    peaks, peak_src = load_peaks()
    flop, nbytes = layer_work(sh, touched, fp8=wl.fp8)
    step_s = ms_max / 1e3 / args.steps
    region_s = ms_max / 1e3
    tflops, kind = pick_peak(peaks, region_s)
    roof, stages = dominant_roofline(wl, r, peaks, peak_src, region_s)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16, routed experts e4m3" if wl.fp8 else "bf16",
            "data": "synthetic (seeded; random-init weights of the K3 layer shape)",
            "config": wl.config(world),
            "tflops": flop / step_s / 1e12,
            "frac_bf16_peak": flop / step_s / 1e12 / tflops,
            "bf16_peak": f"{tflops} TFLOP/s ({peak_src}, {kind}: timed region {region_s:.3f} s)",
            "layer_roofline_ms": 1e3 * max(flop / (tflops * 1e12),
                                           nbytes / (peaks["hbm_gbs"] * 1e9)),
            "experts_touched": touched,
            "roofline": roof, "stages": stages,
            "clocks": r["clocks"],
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": x.numel() * 2,
                    "d2h_bytes_per_step": y.numel() * 2,
                    "path": "lmoe_forward_host (C ABI, pinned host x and y; copies on their "
                            "own streams through 2 device staging slots, overlapped with the "
                            "neighbouring steps' compute)"
                            if wl.qb != "global" else "Layer.forward_host (serial)"},
            "gpu_launches": launches_per_step * args.steps}

    line["load"] = load_summary(sh, counts)
    if wl.name == "skew":
        line["load"] = {"before_balancing": wl.extra["load_before"],
                        "after_balancing": load_summary(sh, counts)}
    if wl.name == "decode":
        line["decode_weight_gbs"] = layer_work(sh, touched, fp8=wl.fp8)[1] / step_s / 1e9
    # the CPU baseline runs on host copies; the device copies of this workload are freed
    # before the other workloads are built
    wh = host_weights(w) if rank == 0 and world == 1 and not args.no_cpu_baseline else None
    xh = x.cpu() if wh is not None else None
    if args.shape == "prefill" and not args.no_configs:
        del wl, layer, x, w, y, r
        torch.cuda.empty_cache()
        line["configs"] = run_configs(args, dev, rank, world, local, stream, peaks, peak_src)
    if wh is not None:
        line["cpu_baseline"] = cpu_baseline(sh, wh, xh, args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_backward(args):
    """The backward pass after each forward step, at the K3 prefill workload: the whole layer
    (lmoe_backward, from dy) or the routed branch alone (lmoe_routed_backward, from dz).  The
    forward is timed as in the headline, the backward alone with CUDA events around it."""
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    wl = Workload(args.shape, dev, rank)
    sh, layer, x = wl.sh, wl.layer, wl.x
    layer.enable_backward(wl.w)
    whole = args.backward == "layer"
    y = torch.empty_like(x)
    gen = torch.Generator(device=dev).manual_seed(SEED)
    if whole:
        grad = torch.randn(sh.T, sh.d, generator=gen, device=dev).to(torch.bfloat16)
        step_bwd = lambda: layer.backward_layer(x, grad)  # noqa: E731
    else:
        grad = torch.randn(sh.T, sh.L, generator=gen, device=dev)
        step_bwd = lambda: layer.backward(grad)  # noqa: E731
    for _ in range(args.warmup):
        wl.forward(y=y, train=True)
        step_bwd()
    torch.cuda.synchronize()
    if layer.device_error() != 0:
        raise RuntimeError("device-side error during warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            ev[i][0].record()
            wl.forward(y=y, train=True)  # a training step keeps the routed pre-activations
            ev[i][1].record()
            step_bwd()
            ev[i][2].record()
        torch.cuda.synchronize()
    barrier(world)
    fwd_launches = layer.last_kernel_launches
    bwd_launches = (layer.layer_backward_launches(sh.T) if whole
                    else layer.backward_launches(sh.T))
    fwd = max_over_ranks(float(np.mean([e[0].elapsed_time(e[1]) for e in ev])), world)
    bwd = max_over_ranks(float(np.mean([e[1].elapsed_time(e[2]) for e in ev])), world)
    T, TK, L, I, E, d = sh.T, sh.T * sh.K, sh.L, sh.I, sh.E, sh.d
    sw = sh.S * sh.Is
    # routed: dgrad x2, wgrad x2 (2 flop per multiply-add each; the forward keeps the
    # gate/value pre-activations, so none are recomputed)
    flop = 12.0 * TK * L * I
    grad_bytes = 4.0 * E * 3 * I * L
    if whole:
        # dz/dhs and dW_out, dx and dW_in, router dgrad and dW_router (the training forward
        # keeps the shared experts' pre-activations too)
        flop += 2.0 * T * d * (L + sw) * 2 + 2.0 * T * (L + 2 * sw) * d * 2 \
            + 2.0 * T * E * L * 2
        grad_bytes += 4.0 * (d * (L + sw) + (L + 2 * sw) * d + E * L)
    peaks, _ = load_peaks()
    what = "layer" if whole else "routed-branch"
    where = "K3 prefill" if args.shape == "prefill" else f"{args.shape} workload"
    line = {"metric": f"{what} backward tokens/s ({where})",
            "value": world * sh.T / (bwd / 1e3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": bwd,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; random-init weights of the K3 layer shape; "
                    + ("dy" if whole else "dz") + " ~ N(0,1))",
            "config": {"workload": wl.config(world)["workload"],
                       "backward": "whole layer: dx and every weight's gradient (fp32)" if whole
                       else "routed branch: dlat, dgate, dgamma, dW_g, dW_v, dW_ed (fp32)",
                       "forward": "training step (keeps the routed pre-activations)"},
            "forward_ms": fwd, "backward_ms": bwd,
            "backward_tflops": flop / (bwd / 1e3) / 1e12,
            "weight_gradient_bytes": grad_bytes,
            "weight_gradient_write_ms_at_hbm_peak": grad_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3,
            "clocks": clk.summary(),
            "gpu_launches": (fwd_launches + bwd_launches) * args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_ep(args):
    """Expert-parallel dispatch and combine, packed and unpacked on one GPU, at the K3 prefill
    routing shape over R ranks: the bytes that would cross the interconnect per token with
    latent rows (L = 3584) against hidden rows (d = 7168), and the pack/unpack kernels' time.
    The transfer itself is not run (one GPU)."""
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    sh, R = synth.PREFILL, args.ep_ranks
    T, K, E = sh.T, sh.K, sh.E
    logits = synth.make_logits(T, E, SEED + rank, device=dev)
    tau = lmoe.thresholds(logits, K)
    idx, gate = lmoe.route(logits, tau, K)
    # expert outputs in expert-segment order, as the routed GEMMs leave them
    order = np.argsort(idx.cpu().numpy().ravel(), kind="stable")
    inv = torch.from_numpy(np.argsort(order).astype(np.int32).reshape(T, K)).to(dev)
    res = {}
    for name, W in (("latent", sh.L), ("hidden", sh.d)):
        rows = synth.make_x(synth.LayerShape("ep", T=T, d=W, L=W, E=E, K=K, I=64, S=0, Is=0),
                            SEED + rank, device=dev)
        o = synth.make_x(synth.LayerShape("ep", T=T * K, d=W, L=W, E=E, K=K, I=64, S=0, Is=0),
                         SEED + 1 + rank, device=dev)
        for _ in range(args.warmup):
            d = lmoe.ep_dispatch(idx, E, R, rows)
            lmoe.ep_combine(idx, d, inv, gate, o)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        torch.cuda.synchronize()
        barrier(world)
        t_disp = t_comb = 0.0
        for _ in range(args.steps):
            ev[0].record()
            d = lmoe.ep_dispatch(idx, E, R, rows)
            ev[1].record()
            lmoe.ep_combine(idx, d, inv, gate, o)
            ev[2].record()
            torch.cuda.synchronize()
            t_disp += ev[0].elapsed_time(ev[1])
            t_comb += ev[1].elapsed_time(ev[2])
        barrier(world)
        P = int(d["send_off"][R].item())
        res[name] = {"width": W, "pairs_per_token": P / T,
                     "interconnect_bytes_per_token": {"dispatch": P * W * 2 / T,
                                                       "combine": P * W * 2 / T},
                     "dispatch_ms": max_over_ranks(t_disp / args.steps, world),
                     "combine_ms": max_over_ranks(t_comb / args.steps, world)}
    lat = res["latent"]
    ms = lat["dispatch_ms"] + lat["combine_ms"]
    line = {"metric": "EP dispatch+combine pack/unpack tokens/s (latent rows)",
            "value": world * T / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded logits and rows)",
            "config": {"workload": f"K3 prefill routing (T={T}, E={E}, top-{K}, in-batch "
                                   f"thresholds) over {R} ranks of {E // R} experts; rows of the "
                                   f"latent ({sh.L}) and of the hidden state ({sh.d})",
                       "ranks": R, "transfer": "not run (one GPU): buffers are what would cross "
                                               "the interconnect"},
            "latent": lat, "hidden": res["hidden"],
            "byte_ratio_hidden_over_latent": (res["hidden"]["interconnect_bytes_per_token"]
                                              ["dispatch"] /
                                              lat["interconnect_bytes_per_token"]["dispatch"]),
            "gpu_launches": 5 * args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--shape", choices=sorted(SHAPES) + ["ep"], default="prefill",
                    help="workload (prefill is the headline; the others are extra lines)")
    ap.add_argument("--cpu-tokens", type=int, default=0,
                    help="tokens of the fixed subset the CPU baseline runs the per-token rest "
                         "of the layer on (0: 512)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="prefill: leave out the decode, skew and e64 workloads of the line")
    ap.add_argument("--overlap", action="store_true",
                    help="run the shared experts on a second stream beside the routed path")
    ap.add_argument("--shared-sms", type=int, default=0,
                    help="SMs for the shared experts when they overlap (0: library default)")
    ap.add_argument("--backward", nargs="?", const="layer", choices=("layer", "routed"),
                    help="time the backward pass after each forward step: the whole layer "
                         "(lmoe_backward, the default) or the routed branch alone")
    ap.add_argument("--ep-ranks", type=int, default=8,
                    help="--shape ep: ranks the experts are spread over")
    ap.add_argument("--experts", choices=["bf16", "fp8"], default="bf16",
                    help="routed-expert GEMM operands: bf16, or e4m3 with per-row scales")
    ap.add_argument("--qb", choices=["local", "global"], default="local",
                    help="thresholds per rank's batch (local) or over all ranks' batches "
                         "(global: router phase, all-gather of candidates, experts phase)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        if args.shape == "ep":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the layer; "
                              "--shape ep measures pack/unpack kernels only"}), flush=True)
            return 0
        return run_reference(args)
    if args.backward:
        return run_backward(args)
    return run_ep(args) if args.shape == "ep" else run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
