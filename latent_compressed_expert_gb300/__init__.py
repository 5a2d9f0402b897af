"""GB300-native Stable Latent MoE feed-forward layer (Kimi K3): hand-written sm_103a CUDA
kernels behind the C ABI of include/lmoe.h, with a thin ctypes binding.

    from latent_compressed_expert_gb300 import lmoe, synth
    layer = lmoe.Layer(synth.PREFILL, weights)   # packs weights, allocates the workspace
    y = layer.forward(x, residual=x)

The seeded input generators live in ``synth``; the binding in ``lmoe`` loads the library
lazily and raises if it has not been built.
"""
__all__ = ["lmoe", "synth"]
