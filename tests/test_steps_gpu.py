"""The step-wise entry points against the one-call forward and backward.

dfa_fwd_main with a dq accumulator zeroes it inside the forward launch, and
dfa_bwd_preprocess with dq_acc NULL then computes D only.  The accumulator
is filled with a large value first, so that any 16-byte group the forward
misses shows.  out, lse, dk and dv come from the same kernels as the one-call
path and must be identical; dq is a sum of float32 atomics whose order
varies, compared to a tight tolerance, and also against the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
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


def _steps(b, q, k, v, do, bs, mode):
    B, L, H, d = q.shape
    dev = q.device
    out = torch.empty_like(q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    dq_acc = torch.full(q.shape, 1.0e30, dtype=torch.float32, device=dev)
    delta = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    b.dfa_fwd_main(q, k, v, out, lse, dq_acc, bs, mode=mode)
    torch.cuda.synchronize()
    zeroed = bool((dq_acc == 0).all())
    dk, dv, dq = torch.empty_like(k), torch.empty_like(v), torch.empty_like(q)
    b.dfa_bwd_preprocess(out, do, delta, None)
    b.dfa_bwd_main(q, k, v, do, lse, delta, dq_acc, dk, dv, bs, mode=mode)
    b.dfa_bwd_dq_convert(dq_acc, dq)
    torch.cuda.synchronize()
    assert b.dfa_status() == b.DFA_OK
    return zeroed, out, lse, dq, dk, dv


def _one_call(b, q, k, v, do, bs, mode):
    B, L, H, d = q.shape
    if mode == b.MODE_CAUSAL:
        n = L // 2
        qc, kc, vc, doc = (t.view(2 * B, n, H, d) for t in (q, k, v, do))
        out, lse = b.dfa_causal_forward(qc, kc, vc)
        dq, dk, dv = b.dfa_causal_backward(qc, kc, vc, out, doc, lse)
        res = (out, lse, dq, dk, dv)
        return tuple(t.view(B, L, H, d) if t.dim() == 4 else t for t in res)
    out, lse = b.dfa_forward(q, k, v, bs)
    dq, dk, dv = b.dfa_backward(q, k, v, out, do, lse, bs)
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("mode_name", ["diffusion", "causal"])
@pytest.mark.parametrize("B,n,H,d,bs", [(2, 300, 3, 64, 16), (2, 256, 4, 128, 32),
                                        (2, 200, 2, 256, 8)])
def test_steps_match_one_call(b, mode_name, B, n, H, d, bs):
    mode = b.MODE_DIFFUSION if mode_name == "diffusion" else b.MODE_CAUSAL
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in inputs.make_inputs(B, n, H, d, seed=21))
    zeroed, *got = _steps(b, q, k, v, do, bs, mode)
    assert zeroed, "the forward left part of the dq accumulator unzeroed"
    ref = _one_call(b, q, k, v, do, bs, mode)
    torch.cuda.synchronize()
    out, lse, dq, dk, dv = got
    lse_ref = ref[1].reshape(lse.shape)
    assert torch.equal(out, ref[0])
    assert torch.equal(lse, lse_ref)
    assert torch.equal(dk, ref[3])
    assert torch.equal(dv, ref[4])
    err = (dq.float() - ref[2].float()).abs().max() / ref[2].float().abs().max()
    assert float(err) < 1e-2


def test_steps_dq_against_oracle(b):
    B, n, H, d, bs = 1, 256, 2, 128, 16
    qh, kh, vh, doh = inputs.make_inputs(B, n, H, d, seed=22)
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in (qh, kh, vh, doh))
    zeroed, out, lse, dq, dk, dv = _steps(b, q, k, v, do, bs, b.MODE_DIFFUSION)
    assert zeroed
    as64 = lambda t: t.float().cpu().double().numpy()  # noqa: E731
    rq, _, _ = oracle.diffusion_backward(as64(qh), as64(kh), as64(vh), as64(doh), bs)
    got = as64(dq)
    assert np.abs(got - rq).max() / np.abs(rq).max() < 2e-2
