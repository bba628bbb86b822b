"""CPU float64 oracle for block-diffusion attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes anything under this package; only the tests, the smoke check of
``__graft_entry__`` and the CPU baseline leg of ``bench.py`` use it.  It
shares no code with the CUDA path: it materialises the full masked score
matrix and takes the plain definition of attention and of its gradients.
"""

from .attention import (  # noqa: F401
    HALF_NOISY,
    HALF_CLEAN,
    visible,
    diffusion_mask,
    causal_mask,
    visible_pairs,
    masked_attention_forward,
    masked_attention_backward,
    diffusion_forward,
    diffusion_backward,
    diffusion_varlen_forward,
    diffusion_varlen_backward,
    causal_forward,
    causal_backward,
    online_softmax_row,
)
