"""The C-ABI library builds, loads and exports every function include/lmoe.h declares; the
host-side argument checks and size queries behave as documented.  No call here launches
a kernel, so these run without a GPU."""
import ctypes
import os
import re

import pytest

from latent_compressed_expert_gb300 import build, lmoe, synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "lmoe.h")


# Calls below pass fake device addresses that the host-side checks must reject before any
# CUDA call; they are host-logic tests and stay off machines with a GPU, where a check that
# let one through would touch a bogus address.
no_gpu = pytest.mark.skipif(__import__("torch").cuda.is_available(),
                            reason="fake-pointer host checks run on CPU-only machines")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return lmoe.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lmoe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"lmoe_forward", "lmoe_route", "lmoe_thresholds"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    # and the binding knows a signature for each of them
    assert set(names) == set(lmoe.SIGNATURES)


def test_version_and_error_strings(lib):
    assert lib.lmoe_version().decode().startswith("lmoe")
    for code in range(6):
        assert lib.lmoe_error_string(code)
    assert lib.lmoe_error_string(99) == b"unknown status"


def test_size_queries(lib):
    d = lmoe.dims_of(synth.PREFILL)
    pb = lmoe.packed_bytes(d)
    # every weight once (bf16) plus gamma (fp32), up to 1 KB alignment per piece
    sh = synth.PREFILL
    weights = (sh.L * sh.d + sh.E * sh.L + 3 * sh.E * sh.I * sh.L + sh.d * sh.L
               + 3 * sh.S * sh.Is * sh.d) * 2 + sh.L * 4
    assert weights <= pb <= weights + 6 * 1024
    # the expert outputs o [T*K, L] dominate; the permuted latent is never materialised
    o_bytes = sh.T * sh.K * sh.L * 2
    assert o_bytes < lmoe.workspace_bytes(d) < 2 * o_bytes
    # T = 0 is valid and small
    assert 0 < lmoe.workspace_bytes(lmoe.dims_of(synth.PREFILL, T=0)) < 1 << 20


def test_fp8_size_queries(lib):
    sh = synth.PREFILL
    d16 = lmoe.dims_of(sh)
    d8 = lmoe.dims_of(sh, expert_fp8=True)
    routed = sh.E * 3 * sh.I * sh.L
    # the routed experts take one byte per weight plus a fp32 scale per row
    scales = sh.E * (2 * sh.I + sh.L) * 4
    assert lmoe.packed_bytes(d16) - lmoe.packed_bytes(d8) == pytest.approx(routed - scales,
                                                                         abs=8 * 1024)
    # the workspace adds the quantised latent and SiTU output with their scales
    extra = sh.T * (sh.L + 4) + sh.T * sh.K * (sh.I + 4)
    assert lmoe.workspace_bytes(d8) - lmoe.workspace_bytes(d16) == pytest.approx(extra,
                                                                                abs=2048)
    # FP8 needs L and I in multiples of 128 (one 128-byte K-block of codes)
    assert lmoe.packed_bytes(lmoe.dims_of(synth.TINY, expert_fp8=True)) == 0


@no_gpu
@pytest.mark.parametrize("field,value,code", [
    ("d", 100, lmoe.LMOE_ERR_UNSUPPORTED),    # not a multiple of 64
    ("L", 96, lmoe.LMOE_ERR_UNSUPPORTED),
    ("I", 32, lmoe.LMOE_ERR_UNSUPPORTED),
    ("K", 33, lmoe.LMOE_ERR_UNSUPPORTED),     # K > 32
    ("E", 8, lmoe.LMOE_ERR_UNSUPPORTED),      # K = 16 > E
    ("E", 900, lmoe.LMOE_ERR_UNSUPPORTED),    # not a multiple of 16
    ("T", -1, lmoe.LMOE_ERR_INVALID_ARG),
    ("c", 0.0, lmoe.LMOE_ERR_INVALID_ARG),
])
def test_unsupported_dims_are_rejected(lib, field, value, code):
    d = lmoe.dims_of(synth.PREFILL)
    setattr(d, field, value)
    assert lmoe.packed_bytes(d) == 0 and lmoe.workspace_bytes(d) == 0
    rc = lib.lmoe_forward(ctypes.byref(d), None, None, None, None, None, 0, None, None)
    assert rc == code


@no_gpu
def test_forward_argument_checks(lib):
    d = lmoe.dims_of(synth.TINY)
    # missing buffers
    assert lib.lmoe_forward(ctypes.byref(d), None, None, None, None, None, 0, None, None) \
        == lmoe.LMOE_ERR_INVALID_ARG
    # T == 0 is a no-op that touches nothing
    d0 = lmoe.dims_of(synth.TINY, T=0)
    assert lib.lmoe_forward(ctypes.byref(d0), None, None, None, None, None, 0, None, None) \
        == lmoe.LMOE_OK
    # misaligned pointers are rejected before any launch
    fake = ctypes.c_void_p(0x1000)
    bad = ctypes.c_void_p(0x1001)
    ws = lmoe.workspace_bytes(d)
    assert lib.lmoe_forward(ctypes.byref(d), fake, bad, None, fake, fake, ws, None, None) \
        == lmoe.LMOE_ERR_INVALID_ARG
    # y aliasing x is rejected
    assert lib.lmoe_forward(ctypes.byref(d), fake, fake, None, fake, ctypes.c_void_p(0x2000),
                            ws, None, None) == lmoe.LMOE_ERR_INVALID_ARG
    # a workspace one byte short of the base size is rejected (the split-K region of a small
    # batch is optional)
    base = lmoe.workspace_base_bytes(d)
    assert base == ws - 12 * 2 ** 20
    assert lib.lmoe_forward(ctypes.byref(d), fake, fake, None, ctypes.c_void_p(0x3000),
                            ctypes.c_void_p(0x4000), base - 1, None, None) \
        == lmoe.LMOE_ERR_WORKSPACE_TOO_SMALL


@no_gpu
def test_route_and_threshold_argument_checks(lib):
    fake = ctypes.c_void_p(0x1000)
    assert lib.lmoe_route(fake, None, 4, 8, 9, fake, fake, None, None) == lmoe.LMOE_ERR_UNSUPPORTED
    assert lib.lmoe_route(fake, None, 4, 64, 33, fake, fake, None, None) == lmoe.LMOE_ERR_UNSUPPORTED
    assert lib.lmoe_route(fake, None, 4, 8192, 4, fake, fake, None, None) == lmoe.LMOE_ERR_UNSUPPORTED
    assert lib.lmoe_route(fake, None, -1, 8, 4, fake, fake, None, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_route(None, None, 4, 8, 4, None, None, None, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_route(None, None, 0, 8, 4, None, None, None, None) == lmoe.LMOE_OK
    assert lib.lmoe_thresholds(fake, 10, 8, 4, 11, fake, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_thresholds(None, 10, 8, 4, 0, None, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_thresholds(None, 0, 8, 4, 0, None, None) == lmoe.LMOE_OK
    assert lib.lmoe_gemm_bf16(fake, fake, fake, 4, 24, 64, fake, None) == lmoe.LMOE_ERR_UNSUPPORTED
    assert lib.lmoe_gemm_bf16(fake, fake, fake, 4, 32, 96, fake, None) == lmoe.LMOE_ERR_UNSUPPORTED
    assert lib.lmoe_gemm_bf16(fake, fake, fake, 4, 32, 64, None, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_gemm_wgrad_bf16(fake, fake, fake, 12, 32, 64, fake, None) == lmoe.LMOE_ERR_UNSUPPORTED
    assert lib.lmoe_gemm_wgrad_bf16(fake, fake, fake, 16, 24, 64, fake, None) == lmoe.LMOE_ERR_UNSUPPORTED
    assert lib.lmoe_gemm_wgrad_bf16(fake, fake, fake, 16, 32, -1, fake, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_gemm_wgrad_bf16(fake, fake, fake, 16, 32, 64, None, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_gemm_wgrad_bf16(fake, fake, fake, 0, 32, 64, fake, None) == lmoe.LMOE_OK


def test_binding_refuses_cpu_tensors(lib):
    import torch
    logits = torch.zeros(4, 16)
    with pytest.raises(ValueError):
        lmoe.route(logits, None, 4)


@no_gpu
def test_phase_and_candidate_argument_checks(lib):
    d = lmoe.dims_of(synth.TINY)
    fake = ctypes.c_void_p(0x1000)
    ws = lmoe.workspace_bytes(d)

    def fwd(x, y, **fields):
        io = lmoe.IO()
        io.balance = 1
        for k, v in fields.items():
            setattr(io, k, v)
        return lib.lmoe_forward(ctypes.byref(d), fake, x, None, y, ctypes.c_void_p(0x4000), ws,
                                ctypes.byref(io), None)

    assert fwd(fake, ctypes.c_void_p(0x2000), phase=3) == lmoe.LMOE_ERR_INVALID_ARG
    assert fwd(fake, ctypes.c_void_p(0x2000), phase=-1) == lmoe.LMOE_ERR_INVALID_ARG
    # candidates only come out of the router phase, and need their rank
    assert fwd(fake, ctypes.c_void_p(0x2000), cand_out=0x5000, cand_k=4) \
        == lmoe.LMOE_ERR_INVALID_ARG
    assert fwd(fake, None, phase=lmoe.PHASE_ROUTER, cand_out=0x5000, cand_k=0) \
        == lmoe.LMOE_ERR_INVALID_ARG
    assert fwd(fake, None, phase=lmoe.PHASE_EXPERTS, cand_out=0x5000, cand_k=4) \
        == lmoe.LMOE_ERR_INVALID_ARG
    # the router phase needs x, the experts phase needs y
    assert fwd(None, None, phase=lmoe.PHASE_ROUTER) == lmoe.LMOE_ERR_INVALID_ARG
    assert fwd(None, None, phase=lmoe.PHASE_EXPERTS) == lmoe.LMOE_ERR_INVALID_ARG
    # lmoe_threshold_candidates
    c = lib.lmoe_threshold_candidates
    assert c(None, 10, 8, 4, fake, None) == lmoe.LMOE_ERR_INVALID_ARG   # logits missing
    assert c(fake, 10, 8, 4, None, None) == lmoe.LMOE_ERR_INVALID_ARG   # cand missing
    assert c(fake, 10, 8, 0, fake, None) == lmoe.LMOE_ERR_INVALID_ARG   # k < 1
    assert c(fake, 10, 0, 4, fake, None) == lmoe.LMOE_ERR_INVALID_ARG   # E < 1
    assert c(fake, -1, 8, 4, fake, None) == lmoe.LMOE_ERR_INVALID_ARG   # T < 0
    # lmoe_quantize_e4m3
    q = lib.lmoe_quantize_e4m3
    assert q(None, 4, 16, fake, fake, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert q(fake, -1, 16, fake, fake, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert q(fake, 4, 24, fake, fake, None) == lmoe.LMOE_ERR_UNSUPPORTED  # cols % 16
    assert q(None, 0, 16, None, None, None) == lmoe.LMOE_OK
    # streaming thresholds and load statistics
    assert lib.lmoe_tau_ema(fake, fake, 8, 1.5, 0, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_tau_ema(None, fake, 8, 0.5, 0, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_tau_ema(None, None, 0, 0.5, 0, None) == lmoe.LMOE_OK
    assert lib.lmoe_load_stats_update(fake, 0, fake, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert lib.lmoe_load_stats_update(None, 8, fake, None) == lmoe.LMOE_ERR_INVALID_ARG
    assert fwd(fake, ctypes.c_void_p(0x2000), tau_ema=0x6000, ema_beta=2.0) \
        == lmoe.LMOE_ERR_INVALID_ARG


def test_backward_size_queries(lib):
    sh = synth.PREFILL
    d = lmoe.dims_of(sh)
    routed = lib.lmoe_routed_backward_workspace_bytes(ctypes.byref(d))
    layer = lib.lmoe_backward_workspace_bytes(ctypes.byref(d))
    # the layer's scratch extends the routed branch's by its dense buffers: dz, dlat_r and
    # dlat (fp32), dhs, the shared pre-activations, [dlat | dgv_s] and dlogit (bf16)
    sw = sh.S * sh.Is
    extra = sh.T * (12 * sh.L + 2 * sw + 4 * sw + 2 * (sh.L + 2 * sw) + 2 * sh.E + 4 * sh.K)
    assert layer - routed == pytest.approx(extra, abs=64 * 1024)
    # the routed branch's: do, the slot-order latent and its gradient ([TK, L] bf16 each),
    # dh [TK, I], pre-activations and their gradients [TK, 2I], plus u (fp32 [T, L])
    TK = sh.T * sh.K
    acts = TK * (3 * 2 * sh.L + 2 * sh.I + 2 * 2 * 2 * sh.I)
    assert acts < routed < acts + sh.T * sh.L * 4 + 4 * 1024 * 1024
    # the transposed pack holds every routed and dense weight once (bf16)
    pb = lib.lmoe_packed_backward_bytes(ctypes.byref(d))
    weights = 2 * (3 * sh.E * sh.I * sh.L + (sh.L + sw) * sh.d + sh.L * sh.E
                   + sh.d * (sh.L + 2 * sw))
    assert weights <= pb <= weights + 8 * 1024 * 1024
    d8 = lmoe.dims_of(sh, expert_fp8=True)
    assert lib.lmoe_backward_workspace_bytes(ctypes.byref(d8)) == 0


@no_gpu
def test_backward_argument_checks(lib):
    d = lmoe.dims_of(synth.TINY)
    fake = ctypes.c_void_p(0x1000)
    ws = lmoe.workspace_bytes(d)
    bw = lib.lmoe_backward_workspace_bytes(ctypes.byref(d))
    f = lib.lmoe_backward

    def call(dims=d, x=fake, dy=fake, ws_bytes=ws, bw_bytes=bw, dx=fake):
        return f(ctypes.byref(dims), fake, fake, fake, ws_bytes, x, None, dy, None, None, dx,
                 fake, fake, fake, fake, fake, fake, fake, bw_bytes, None)

    assert call(x=None) == lmoe.LMOE_ERR_INVALID_ARG
    assert call(dy=None) == lmoe.LMOE_ERR_INVALID_ARG
    assert call(dx=ctypes.c_void_p(0x1004)) == lmoe.LMOE_ERR_INVALID_ARG   # misaligned
    assert f(ctypes.byref(d), fake, fake, fake, ws, fake, None, fake, ctypes.c_void_p(0x1002),
             None, fake, fake, fake, fake, fake, fake, fake, fake, bw, None) \
        == lmoe.LMOE_ERR_INVALID_ARG                                          # pre misaligned
    assert call(bw_bytes=bw - 1) == lmoe.LMOE_ERR_WORKSPACE_TOO_SMALL
    assert call(ws_bytes=lmoe.workspace_base_bytes(d) - 1) == lmoe.LMOE_ERR_WORKSPACE_TOO_SMALL
    assert call(dims=lmoe.dims_of(synth.TINY, T=0), ws_bytes=1 << 30, bw_bytes=1 << 30) \
        == lmoe.LMOE_OK
    d8 = lmoe.dims_of(synth.PREFILL, expert_fp8=True)
    assert call(dims=d8) == lmoe.LMOE_ERR_UNSUPPORTED
    # the transposed pack needs the forward's packed buffer
    W = lmoe.Weights()
    assert lib.lmoe_pack_backward_weights(ctypes.byref(d), ctypes.byref(W), None, fake, 1 << 30,
                                          None) == lmoe.LMOE_ERR_INVALID_ARG


def _c_layout(struct, fields, tmp_path):
    """sizeof and offsetof of a struct of include/lmoe.h, from a C program gcc compiles."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    body = "".join(f'  printf("%zu\\n", offsetof({struct}, {f}));\n' for f in fields)
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "lmoe.h"\n'
                   f'int main(void) {{\n  printf("%zu\\n", sizeof({struct}));\n{body}'
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I" + os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    return int(out[0]), [int(v) for v in out[1:]]


@pytest.mark.parametrize("struct,cls", [("lmoe_dims", lmoe.Dims), ("lmoe_weights", lmoe.Weights),
                                        ("lmoe_io", lmoe.IO), ("lmoe_host_pipe", lmoe.HostPipe)])
def test_binding_structs_match_the_header(struct, cls, tmp_path):
    """The ctypes mirrors of the header's structs have the same size and field offsets, so
    every option reaches the library in its own field."""
    names = [f for f, _ in cls._fields_]
    size, offs = _c_layout(struct, names, tmp_path)
    assert ctypes.sizeof(cls) == size
    assert [getattr(cls, f).offset for f in names] == offs


def test_noalloc_constants_match_the_header():
    src = open(HEADER).read()
    m = re.search(r"#define\s+LMOE_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "LMOE_NOALLOC_SCRATCH_BYTES not found"
    assert lmoe.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
    m = re.search(r"#define\s+LMOE_OVERLAP_MIN_T\s+(\d+)", src)
    assert m and lmoe.OVERLAP_MIN_T == int(m.group(1))


def test_noalloc_limit_is_the_documented_batch(lib):
    """The array holds the base workspace of a K3 decode batch of up to 152 tokens, as the
    header states; 153 tokens exceed it."""
    fits = [T for T in range(1, 400)
            if lmoe.workspace_base_bytes(lmoe.dims_of(synth.DECODE, T=T))
            <= lmoe.NOALLOC_SCRATCH_BYTES]
    assert max(fits) == 152 and fits == list(range(1, 153))
    assert "up to 152 tokens" in open(HEADER).read()


def test_fair_share_rank_matches_the_oracle(lib, oracle_mod):
    """The library's rank (used by the thresholds and by a batch spread over ranks) is the
    oracle's, pinned to the pages' fair share; invalid arguments give -1."""
    for T in (0, 1, 7, 55, 56, 57, 64, 1000, 8192, 32768, 40000, 1 << 24):
        for K, E in ((16, 896), (8, 448), (4, 64), (16, 16), (1, 4096), (32, 33)):
            assert lmoe.fair_share_rank(T, K, E) == oracle_mod.fair_share_rank(T, K, E)
    assert lib.lmoe_fair_share_rank(-1, 16, 896) == -1
    assert lib.lmoe_fair_share_rank(100, 0, 896) == -1
    assert lib.lmoe_fair_share_rank(100, 16, 0) == -1


@no_gpu
def test_forward_host_argument_checks(lib):
    """lmoe_forward_host rejects a bad pipe or batch before it enqueues anything."""
    d = lmoe.dims_of(synth.TINY)
    fake = ctypes.c_void_p(1 << 20)
    ws = lmoe.workspace_bytes(d)

    def pipe(depth=2, max_tokens=synth.TINY.T):
        p = lmoe.HostPipe()
        p.depth, p.max_tokens = depth, max_tokens
        for k in range(lmoe.HOST_PIPE_MAX_DEPTH):
            p.x_dev[k] = (1 << 20) + (k << 16)
            p.y_dev[k] = (1 << 24) + (k << 16)
            p.uploaded[k] = p.computed[k] = p.downloaded[k] = 4096 + k
        p.upload, p.compute, p.download = 8, 16, 24
        return p

    def call(p, x=fake, y=fake, dims=d):
        return lib.lmoe_forward_host(ctypes.byref(dims), fake, x, 1, y, fake, ws, None,
                                     ctypes.byref(p))

    assert call(pipe(depth=0)) == lmoe.LMOE_ERR_INVALID_ARG
    assert call(pipe(depth=lmoe.HOST_PIPE_MAX_DEPTH + 1)) == lmoe.LMOE_ERR_INVALID_ARG
    assert call(pipe(max_tokens=synth.TINY.T - 1)) == lmoe.LMOE_ERR_INVALID_ARG
    assert call(pipe(), x=None) == lmoe.LMOE_ERR_INVALID_ARG
    assert call(pipe(), y=None) == lmoe.LMOE_ERR_INVALID_ARG
    bad = lmoe.dims_of(synth.TINY)
    bad.d = 100
    assert call(pipe(), dims=bad) == lmoe.LMOE_ERR_UNSUPPORTED
    p = pipe()
    p.calls = 5
    assert lib.lmoe_forward_host(ctypes.byref(d), fake, fake, 1, fake, fake, 16, None,
                                 ctypes.byref(p)) == lmoe.LMOE_ERR_WORKSPACE_TOO_SMALL
    assert p.calls == 5  # nothing was enqueued
