"""Block-diffusion attention on GB300 (sm_103a).

Exact softmax attention over a [noisy | clean] sequence of length 2n under the
block-diffusion mask, forward and backward, in hand-written tcgen05/TMA CUDA
kernels behind the C ABI of ``libdfa.so`` (``include/dfa.h``).  PyTorch only
provides device memory, streams and autograd plumbing.

    from block_diffusion_masked_gb300 import diffusion_attn_func
    out = diffusion_attn_func(q, k, v, block_size=4)  # (batch, 2n, heads, headdim) bf16

The binding is imported lazily so that ``inputs`` can be used without CUDA.
"""

from __future__ import annotations

__all__ = ["diffusion_attn_func", "diffusion_attn_varlen_func", "causal_attn_func", "binding"]


def __getattr__(name):
    import importlib

    if name in ("diffusion_attn_func", "diffusion_attn_varlen_func", "causal_attn_func",
                "DiffusionAttnFunc", "DiffusionAttnVarlenFunc", "CausalAttnFunc"):
        return getattr(importlib.import_module(__name__ + ".autograd"), name)
    if name in ("binding", "autograd", "inputs", "build"):
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
