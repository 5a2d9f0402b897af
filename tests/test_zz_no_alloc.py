"""lmoe_forward_noalloc: the layer for callers that cannot allocate device memory (a
plug-in whose host framework owns every device allocation, a serving loop where an
allocation would synchronise the device).  Its scratch is a fixed 24 MiB array inside the
library, so it must give the output of lmoe_forward with a caller-allocated workspace on
every call, however many calls share that array, and must refuse batches whose scratch
would not fit.  This file is collected last, so a failure here stops a -x run only after
every other test has run."""
import ctypes

import numpy as np
import pytest
import torch

import gpu_helpers as H
from latent_compressed_expert_gb300 import lmoe, synth

pytestmark = pytest.mark.gpu


def lmoe_scratch_bytes():
    """LMOE_NOALLOC_SCRATCH_BYTES of include/lmoe.h."""
    return 24 << 20


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


def test_noalloc_refuses_batches_beyond_its_array(lib, decode_layer):
    T = 256  # needs ~39 MiB of scratch at the K3 widths
    assert lmoe.workspace_bytes(lmoe.dims_of(synth.DECODE, T=T)) > lmoe_scratch_bytes()
    x = synth.make_x(synth.DECODE, seed=5, device="cuda", T=T)
    y = torch.full_like(x, 7.0)
    assert _noalloc(lib, decode_layer, x, x, y) == lmoe.LMOE_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())  # nothing was enqueued
