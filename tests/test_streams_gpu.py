"""Launches on different streams that run at the same time.

The persistent kernels take work items from a counter the library keeps per
stream.  Two problems started back to back on two streams must each produce
the results of a run on its own: an item taken by the wrong launch would
leave tiles unwritten or written twice.  out, lse, dk and dv come from one
CTA each and are compared exactly; dq is a sum of float32 atomics whose
order varies, compared to a tight tolerance.
"""

import pytest
import torch

from block_diffusion_masked_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_masked_gb300 import binding, build

    build.build()
    binding.lib()
    return binding


def _problem(seed, d):
    dev = torch.device("cuda", 0)
    return [t.to(dev) for t in inputs.make_inputs(4, 512, 8, d, seed=seed)]


def _run(b, q, k, v, do, bs):
    out, lse = b.dfa_forward(q, k, v, bs)
    dq, dk, dv = b.dfa_backward(q, k, v, out, do, lse, bs)
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
def test_concurrent_streams_match_serial_runs(b, d):
    p1, p2 = _problem(11, d), _problem(12, d)
    ref1 = _run(b, *p1, 16)
    ref2 = _run(b, *p2, 32)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s1):
            got1 = _run(b, *p1, 16)
        with torch.cuda.stream(s2):
            got2 = _run(b, *p2, 32)
        torch.cuda.synchronize()
        assert b.dfa_status() == b.DFA_OK
        for got, ref in ((got1, ref1), (got2, ref2)):
            out, lse, dq, dk, dv = got
            assert torch.equal(out, ref[0])
            assert torch.equal(lse, ref[1])
            assert torch.equal(dk, ref[3])
            assert torch.equal(dv, ref[4])
            err = (dq.float() - ref[2].float()).abs().max() / ref[2].float().abs().max()
            assert float(err) < 1e-2
