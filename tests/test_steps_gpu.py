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
    """The step API on q (B, 2n, H, d) (diffusion) or (Bc, n, H, d) (causal)."""
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
    b.dfa_bwd_preprocess(out, do, delta, None, mode=mode)
    b.dfa_bwd_main(q, k, v, do, lse, delta, dq_acc, dk, dv, bs, mode=mode)
    b.dfa_bwd_dq_convert(dq_acc, dq, mode=mode)
    torch.cuda.synchronize()
    assert b.dfa_status() == b.DFA_OK
    return zeroed, out, lse, dq, dk, dv


def _one_call(b, q, k, v, do, bs, mode):
    if mode == b.MODE_CAUSAL:
        out, lse = b.dfa_causal_forward(q, k, v)
        dq, dk, dv = b.dfa_causal_backward(q, k, v, out, do, lse)
        return out, lse, dq, dk, dv
    out, lse = b.dfa_forward(q, k, v, bs)
    dq, dk, dv = b.dfa_backward(q, k, v, out, do, lse, bs)
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("mode_name", ["diffusion", "causal"])
@pytest.mark.parametrize("B,n,H,d,bs", [(2, 300, 3, 64, 16), (2, 256, 4, 128, 32),
                                        (2, 200, 2, 256, 8), (1, 129, 2, 128, 4)])
def test_steps_match_one_call(b, mode_name, B, n, H, d, bs):
    """Diffusion on (B, 2n); causal on the 2B sequences of length n and, for
    an odd count, on the first 2B - 1 of them."""
    mode = b.MODE_DIFFUSION if mode_name == "diffusion" else b.MODE_CAUSAL
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in inputs.make_inputs(B, n, H, d, seed=21))
    if mode == b.MODE_CAUSAL:
        Bc = 2 * B - 1 if B > 1 else 2 * B
        q, k, v, do = (t.view(2 * B, n, H, d)[:Bc].contiguous() for t in (q, k, v, do))
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


@pytest.mark.parametrize("Bc,n,H,Hk,d", [(3, 200, 4, 2, 128), (2, 129, 6, 2, 64),
                                         (1, 150, 2, 1, 256)])
def test_causal_grouped_heads_step_api(b, Bc, n, H, Hk, d):
    """The step API in the causal mode with grouped key/value heads (query
    head h reads key/value head h // (H / Hk)) against the oracle's causal
    attention with the same head map."""
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(31 + Bc)
    mk = lambda h: torch.randn(Bc, n, h, d, generator=g).to(torch.bfloat16)  # noqa: E731
    qh, kh, vh, doh = mk(H), mk(Hk), mk(Hk), mk(H)
    q, k, v, do = (t.to(dev) for t in (qh, kh, vh, doh))
    out = torch.empty_like(q)
    lse = torch.empty((Bc, H, n), dtype=torch.float32, device=dev)
    dq_acc = torch.empty(q.shape, dtype=torch.float32, device=dev)
    delta = torch.empty((Bc, H, n), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    b.dfa_fwd_main_gqa(q, k, v, out, lse, dq_acc, 1, mode=b.MODE_CAUSAL)
    b.dfa_bwd_preprocess(out, do, delta, None, mode=b.MODE_CAUSAL)
    b.dfa_bwd_main_gqa(q, k, v, do, lse, delta, dq_acc, dk, dv, 1, mode=b.MODE_CAUSAL)
    b.dfa_bwd_dq_convert(dq_acc, dq, mode=b.MODE_CAUSAL)
    torch.cuda.synchronize()
    assert b.dfa_status() == b.DFA_OK
    as64 = lambda t: t.float().cpu().double().numpy()  # noqa: E731
    ro, rl = oracle.causal_forward(as64(qh), as64(kh), as64(vh))
    rq, rk, rv = oracle.causal_backward(as64(qh), as64(kh), as64(vh), as64(doh))
    nw = lambda a, r: np.abs(a - r).max() / np.abs(r).max()  # noqa: E731
    assert nw(as64(out), ro) <= 1e-2
    assert np.abs(as64(lse) - rl).max() <= 1e-3
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert nw(as64(got), ref) <= 2e-2


@pytest.mark.parametrize("B,L,H,d", [(2, 600, 3, 64), (1, 2050, 32, 128), (3, 70, 8, 256),
                                     (1, 10, 2100, 64), (2, 9, 1, 128), (1, 1, 5, 256)])
@pytest.mark.parametrize("zero", [False, True])
def test_preprocess_delta_and_zeroing(b, B, L, H, d, zero):
    """D = rowsum(dout * out) ("FlashAttention: Exact Attention Without
    Materialization", section 4.5), laid out (batch, head, position), for
    few and very many heads (the latter stored without shared-memory
    staging), ragged position counts, every head dimension; and the dq
    accumulator zeroed when passed.  Compared with the float64 sum of the
    same bf16 products."""
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(31 + L + H + d)
    out = torch.randn(B, L, H, d, generator=g).to(torch.bfloat16)
    dout = torch.randn(B, L, H, d, generator=g).to(torch.bfloat16)
    ref = (out.double() * dout.double()).sum(-1).permute(0, 2, 1).contiguous()  # (B, H, L)
    delta = torch.full((B, H, L), float("nan"), dtype=torch.float32, device=dev)
    acc = torch.full((B, L, H, d), 7.0, dtype=torch.float32, device=dev) if zero else None
    mode = b.MODE_CAUSAL  # rows of L positions per batch entry, L odd allowed
    b.dfa_bwd_preprocess(out.to(dev), dout.to(dev), delta, acc, mode=mode)
    torch.cuda.synchronize()
    assert b.dfa_status() == b.DFA_OK
    got = delta.cpu().double()
    assert bool(torch.isfinite(got).all())
    bar = 1e-5 * (out.double().abs() * dout.double().abs()).sum(-1).permute(0, 2, 1) + 1e-6
    assert bool(((got - ref).abs() <= bar).all()), float((got - ref).abs().max())
    if zero:
        assert bool((acc == 0).all())
