"""dfa_backward_noalloc: the backward pass for callers that cannot let a
library allocate device memory (a framework whose own allocator must account
for every byte, or a latency-critical step where an allocation could block
or fail).  Its scratch lives in a fixed array inside the library.

Checked through the C ABI against dfa_backward on two calls in a row (the
second on different data, so stale scratch from the first would show), and
the second call also against the float64 oracle.  Kept in its own file,
collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_masked_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_GRAD = 2e-2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_masked_gb300 import binding, build

    build.build()
    handle = binding.lib()
    fn = handle.dfa_backward_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    return handle


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _normwise(got, ref):
    g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
    return float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-30))


@pytest.mark.parametrize("B,n,H,d,bs,seed", [(1, 200, 2, 128, 16, 1), (2, 130, 1, 64, 3, 2)])
def test_noalloc_backward_matches_backward(lib, B, n, H, d, bs, seed):
    from block_diffusion_masked_gb300 import binding

    dev = torch.device("cuda", 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for call in range(2):
        q, k, v, do = (t.to(dev) for t in inputs.make_inputs(B, n, H, d, seed=seed + 10 * call))
        out, lse = binding.dfa_forward(q, k, v, bs)
        ref = binding.dfa_backward(q, k, v, out, do, lse, bs)
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = lib.dfa_backward_noalloc(_p(q), _p(k), _p(v), _p(out), _p(do), _p(lse), _p(got[0]),
                                      _p(got[1]), _p(got[2]), B, n, H, d, bs, stream)
        assert rc == 0, rc
        torch.cuda.synchronize()
        assert binding.dfa_status() == 0
        for g, r in zip(got, ref):
            assert torch.isfinite(g).all()
            assert _normwise(g, r) <= TOL_GRAD
    # the second call's gradients against the oracle
    f64 = lambda t: t.float().cpu().double().numpy()  # noqa: E731
    refs = oracle.diffusion_backward(f64(q), f64(k), f64(v), f64(do), bs)
    floor = 1e-3 * max(np.abs(r).max() for r in refs)
    for g, r in zip(got, refs):
        assert np.abs(f64(g) - r).max() / max(np.abs(r).max(), floor) <= TOL_GRAD


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    p = ctypes.c_void_p(0x1000)
    # 8 x 2*8192 x 16 x 128 floats is far more than the fixed 32 MiB scratch
    rc = lib.dfa_backward_noalloc(p, p, p, p, p, p, p, p, p, 8, 8192, 16, 128, 16,
                                  ctypes.c_void_p(0))
    assert rc == -1  # DFA_EINVAL, before any work is enqueued
