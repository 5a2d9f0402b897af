"""lmoe_forward_noalloc: the layer for callers that cannot allocate device memory (a
plug-in whose host framework owns every device allocation, a serving loop where an
allocation would synchronise the device).  Its scratch is a fixed 24 MiB array inside the
library, so it must give the output of lmoe_forward with a caller-allocated workspace on
every call, however many calls share that array, must refuse batches whose scratch would
not fit, and must let the caller read a device-side error recorded in the array.  This
file is collected last, so a failure here stops a -x run only after every other test has
run."""
import ctypes

import numpy as np
import pytest
import torch

import gpu_helpers as H
from latent_compressed_expert_gb300 import lmoe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from latent_compressed_expert_gb300 import build
    build.build()
    return lmoe.load()


def _noalloc(lib, layer, x, residual, y):
    dims = lmoe.dims_of(layer.shape, T=x.shape[0])
    io = lmoe.IO()
    io.balance = 1
    return lib.lmoe_forward_noalloc(ctypes.byref(dims), lmoe._ptr(layer.packed), lmoe._ptr(x),
                                    lmoe._ptr(residual), lmoe._ptr(y), ctypes.byref(io),
                                    lmoe._stream())


@pytest.fixture(scope="module")
def decode_layer(lib):
    sh = synth.DECODE
    w = synth.make_weights(sh, seed=3, device="cuda")
    return lmoe.Layer(sh, w)


SMALL = synth.LayerShape("small", T=300, d=1024, L=512, E=64, K=8, I=256, S=2, Is=512)


@pytest.mark.parametrize("which", ["decode", "small"])
def test_noalloc_matches_forward_with_workspace(lib, decode_layer, which):
    if which == "decode":
        layer = decode_layer
    else:
        layer = lmoe.Layer(SMALL, synth.make_weights(SMALL, seed=7, device="cuda"))
    sh = layer.shape
    for call in range(2):
        x = synth.make_x(sh, seed=10 + call, device="cuda")
        ref = layer.forward(x, residual=x)
        y = torch.full_like(x, float("nan"))
        assert _noalloc(lib, layer, x, x, y) == lmoe.LMOE_OK
        torch.cuda.synchronize()
        H.assert_close(y.float().cpu().numpy(), ref.float().cpu().numpy(), f"{which}/call{call}")


def _largest_batch_that_fits(sh):
    """Largest batch whose base workspace fits the array (its size from the header's
    constant, mirrored by the binding), searched from the sizes the library reports."""
    T = 1
    while lmoe.workspace_base_bytes(lmoe.dims_of(sh, T=T + 1)) <= lmoe.NOALLOC_SCRATCH_BYTES:
        T += 1
    return T


def test_noalloc_at_its_largest_batch_and_refusal_beyond(lib, decode_layer):
    """The largest K3 decode batch the array holds gives lmoe_forward's output; one token
    more is refused with nothing enqueued."""
    sh = synth.DECODE
    T = _largest_batch_that_fits(sh)
    assert T >= 64
    x = synth.make_x(sh, seed=5, device="cuda", T=T)
    dims = lmoe.dims_of(sh, T=T)
    ws_bytes = lmoe.workspace_bytes(dims)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(x)
    io = lmoe.IO()
    io.balance = 1
    assert lib.lmoe_forward(ctypes.byref(dims), lmoe._ptr(decode_layer.packed), lmoe._ptr(x),
                            lmoe._ptr(x), lmoe._ptr(ref), lmoe._ptr(ws), ws_bytes,
                            ctypes.byref(io), lmoe._stream()) == lmoe.LMOE_OK
    y = torch.full_like(x, float("nan"))
    assert _noalloc(lib, decode_layer, x, x, y) == lmoe.LMOE_OK
    torch.cuda.synchronize()
    assert lib.lmoe_noalloc_last_device_error() == lmoe.LMOE_OK
    H.assert_close(y.float().cpu().numpy(), ref.float().cpu().numpy(), f"T{T}")
    # one token more: refused before anything is enqueued
    x1 = synth.make_x(sh, seed=6, device="cuda", T=T + 1)
    assert lmoe.workspace_base_bytes(lmoe.dims_of(sh, T=T + 1)) > lmoe.NOALLOC_SCRATCH_BYTES
    y1 = torch.full_like(x1, 7.0)
    assert _noalloc(lib, decode_layer, x1, x1, y1) == lmoe.LMOE_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((y1 == 7.0).all())  # nothing was enqueued


def test_noalloc_device_error_is_readable(lib, monkeypatch):
    """A bounded device wait that runs out inside lmoe_forward_noalloc is reported by
    lmoe_noalloc_last_device_error, which clears it; the next call is correct.  The wait is
    made to run out on purpose (LMOE_FAULT_INJECT=stall: the first GEMM's MMA role waits on
    a barrier nothing arrives on, for LMOE_WAIT_LIMIT_MS), which faults nothing."""
    sh = synth.TINY
    w = {k: v.to("cuda") for k, v in synth.make_weights(sh, seed=9).items()}
    layer = lmoe.Layer(sh, w)
    x = synth.make_x(sh, seed=9).to("cuda")
    logits = synth.make_logits(sh.T, sh.E, seed=9).to("cuda")

    def call(y):
        dims = lmoe.dims_of(sh, T=sh.T)
        io = lmoe.IO()
        io.balance = 1
        io.logits_in = lmoe._ptr(logits)
        return lib.lmoe_forward_noalloc(ctypes.byref(dims), lmoe._ptr(layer.packed),
                                        lmoe._ptr(x), lmoe._ptr(x), lmoe._ptr(y),
                                        ctypes.byref(io), lmoe._stream())

    monkeypatch.setenv("LMOE_WAIT_LIMIT_MS", "200")
    monkeypatch.setenv("LMOE_FAULT_INJECT", "stall")
    y = torch.empty_like(x)
    assert call(y) == lmoe.LMOE_OK
    torch.cuda.synchronize()
    assert lib.lmoe_noalloc_last_device_error() == lmoe.LMOE_ERR_DEVICE_TIMEOUT
    assert lib.lmoe_noalloc_last_device_error() == lmoe.LMOE_OK  # reading clears it
    monkeypatch.delenv("LMOE_FAULT_INJECT")
    assert call(y) == lmoe.LMOE_OK
    torch.cuda.synchronize()
    assert lib.lmoe_noalloc_last_device_error() == lmoe.LMOE_OK
    ref = layer.forward(x, residual=x, logits_in=logits)
    torch.cuda.synchronize()
    H.assert_close(y.float().cpu().numpy(), ref.float().cpu().numpy(), "after-timeout")
