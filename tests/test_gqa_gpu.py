"""GPU parity of grouped key/value heads (MQA / GQA) through the C ABI.

"Fast Diffusion Attention" lists MQA / GQA among the supported shapes and a
"GQA-grouped backward" in which one thread block sums dK / dV over the query
heads of a key/value head.  Here k and v carry H_kv heads (query head h
reads head h // (H / H_kv)), and the kernels' out, lse, dq, dk, dv are
compared with the float64 oracle on the same seeded inputs, at sizes that
span several tiles with ragged tails, for every head dimension.  Bars as in
the plain parity tests: normwise 1e-2 for out, 2e-2 for the gradients,
1e-3 absolute for lse.
"""

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_masked_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2
TOL_GRAD = 2e-2
TOL_LSE = 1e-3


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_masked_gb300 import binding, build

    build.build()
    binding.lib()
    return binding


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _grouped_inputs(B, n, H, Hk, d, seed):
    q, _, _, do = inputs.make_inputs(B, n, H, d, seed=seed)
    _, k, v = inputs.make_inputs(B, n, Hk, d, seed=seed + 1, with_dout=False)
    return q, k, v, do


def _errors(got, ref):
    # A gradient can be exactly zero (every row seeing a single key makes
    # dS = 0): then measure it against 1e-3 of the largest gradient.
    floor = 1e-3 * max(np.abs(r).max() for r in ref.values())
    return {name: float(np.abs(got[name] - r).max() / max(np.abs(r).max(), floor))
            for name, r in ref.items()}


CASES = [
    # (B, n, H, H_kv, d, bs)
    (1, 1, 2, 1, 64, 1),
    (1, 67, 4, 2, 64, 3),
    (2, 129, 4, 1, 64, 16),
    (1, 200, 4, 2, 128, 7),
    (1, 130, 6, 3, 128, 1),
    (1, 256, 4, 1, 128, 64),
    (1, 67, 4, 2, 256, 3),
    (1, 130, 2, 1, 256, 16),
]


@pytest.mark.parametrize("B,n,H,Hk,d,bs", CASES)
def test_grouped_matches_oracle(b, B, n, H, Hk, d, bs):
    q, k, v, do = _grouped_inputs(B, n, H, Hk, d, seed=300 + n + H + Hk + d)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    out, lse = b.dfa_forward_gqa(qd, kd, vd, bs)
    dq, dk, dv = b.dfa_backward_gqa(qd, kd, vd, out, dod, lse, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    ro, rl = oracle.diffusion_forward(qn, kn, vn, bs)
    rq, rk, rv = oracle.diffusion_backward(qn, kn, vn, don, bs)
    e_out = float(np.abs(_np(out) - ro).max() / np.abs(ro).max())
    e_lse = float(np.abs(lse.cpu().double().numpy() - rl).max())
    errs = _errors({"dq": _np(dq), "dk": _np(dk), "dv": _np(dv)}, {"dq": rq, "dk": rk, "dv": rv})
    assert e_out <= TOL_OUT, (e_out, errs)
    assert e_lse <= TOL_LSE, (e_lse, errs)
    for name, e in errs.items():
        assert e <= TOL_GRAD, errs


@pytest.mark.parametrize("d", [64, 128, 256])
def test_one_group_per_head_is_the_plain_path(b, d):
    # H_kv == H runs the very same kernels as dfa_forward / dfa_backward:
    # bitwise equal results.
    q, k, v, do = inputs.make_inputs(1, 131, 2, d, seed=41 + d)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o1, l1 = b.dfa_forward(qd, kd, vd, 5)
    o2, l2 = b.dfa_forward_gqa(qd, kd, vd, 5)
    g1 = b.dfa_backward(qd, kd, vd, o1, dod, l1, 5)
    g2 = b.dfa_backward_gqa(qd, kd, vd, o1, dod, l1, 5)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # dq sums float32 atomics in arrival order; dk and dv are plain stores
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    dq_gap = (g1[0].float() - g2[0].float()).abs().max().item()
    assert dq_gap <= 1e-2 * g1[0].float().abs().max().item()


def test_grouped_agrees_with_repeated_heads(b):
    # The forward of a grouped call equals the plain forward on k, v with
    # each key/value head repeated for its query heads (same tiles, same
    # order of operations: bitwise); the grouped dk, dv equal the group sums
    # of the plain gradients within the gradient bar.
    B, n, H, Hk, d, bs = 1, 150, 4, 2, 128, 4
    q, k, v, do = _grouped_inputs(B, n, H, Hk, d, seed=77)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    kr = kd.repeat_interleave(H // Hk, dim=2).contiguous()
    vr = vd.repeat_interleave(H // Hk, dim=2).contiguous()
    og, lg = b.dfa_forward_gqa(qd, kd, vd, bs)
    orr, lr = b.dfa_forward(qd, kr, vr, bs)
    _, dkg, dvg = b.dfa_backward_gqa(qd, kd, vd, og, dod, lg, bs)
    _, dkr, dvr = b.dfa_backward(qd, kr, vr, orr, dod, lr, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert torch.equal(og, orr) and torch.equal(lg, lr)
    for got, rep in ((dkg, dkr), (dvg, dvr)):
        s = rep.float().view(B, 2 * n, Hk, H // Hk, d).sum(3)
        assert (got.float() - s).abs().max().item() <= TOL_GRAD * s.abs().max().item()


def test_heads_must_divide(b):
    q, _, _ = inputs.make_inputs(1, 8, 3, 64, seed=1, with_dout=False)
    _, k, v = inputs.make_inputs(1, 8, 2, 64, seed=2, with_dout=False)
    dev = torch.device("cuda", 0)
    with pytest.raises(ValueError):
        b.dfa_forward_gqa(q.to(dev), k.to(dev), v.to(dev), 2)


def test_autograd_function_grouped(b):
    from block_diffusion_masked_gb300 import diffusion_attn_func

    B, n, H, Hk, d, bs = 1, 96, 4, 1, 64, 8
    q, k, v, do = _grouped_inputs(B, n, H, Hk, d, seed=5)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    out = diffusion_attn_func(qd, kd, vd, bs)
    out.backward(do.to(dev))
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    ro, _ = oracle.diffusion_forward(qn, kn, vn, bs)
    rq, rk, rv = oracle.diffusion_backward(qn, kn, vn, don, bs)
    assert float(np.abs(_np(out) - ro).max() / np.abs(ro).max()) <= TOL_OUT
    errs = _errors({"dq": _np(qd.grad), "dk": _np(kd.grad), "dv": _np(vd.grad)},
                   {"dq": rq, "dk": rk, "dv": rv})
    assert max(errs.values()) <= TOL_GRAD, errs


@pytest.mark.parametrize("d,Hk", [(64, 1), (128, 2), (256, 1)])
def test_grouped_step_api_matches_one_call(b, d, Hk):
    # dfa_fwd_main_gqa (zeroing the dq accumulator) + preprocess +
    # dfa_bwd_main_gqa + convert: the same kernels as the one-call API.
    B, n, H, bs = 2, 150, 4, 8
    q, k, v, do = _grouped_inputs(B, n, H, Hk, d, seed=88 + d)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, 2 * n), dtype=torch.float32, device=dev)
    dq_acc = torch.full(qd.shape, 1.0e30, dtype=torch.float32, device=dev)
    delta = torch.empty((B, H, 2 * n), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    b.dfa_fwd_main_gqa(qd, kd, vd, out, lse, dq_acc, bs)
    b.dfa_bwd_preprocess(out, dod, delta, None)
    b.dfa_bwd_main_gqa(qd, kd, vd, dod, lse, delta, dq_acc, dk, dv, bs)
    b.dfa_bwd_dq_convert(dq_acc, dq)
    ro, rl = b.dfa_forward_gqa(qd, kd, vd, bs)
    rq, rk, rv = b.dfa_backward_gqa(qd, kd, vd, ro, dod, rl, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert torch.equal(out, ro) and torch.equal(lse, rl)
    assert torch.equal(dk, rk) and torch.equal(dv, rv)
    gap = (dq.float() - rq.float()).abs().max().item()
    assert gap <= 1e-2 * rq.float().abs().max().item()
