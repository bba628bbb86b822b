"""GPU parity of packed (varlen) batches through the C ABI.

"Fast Diffusion Attention" schedules packed samples of different lengths in
one launch, longest first.  Each sample of the packed (rows, heads, headdim)
tensors is [noisy | clean] with its own half length; the kernels' out, lse,
dq, dk, dv are compared with the float64 oracle on the same seeded inputs:
ragged halves, zero-length samples, grouped key/value heads and every head
dimension.  Bars as in the batched parity tests.
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


def _packed(halves, H, Hk, d, seed):
    """q, k, v, dout packed along the rows, sample b of 2 * halves[b] rows."""
    rows = 2 * sum(halves)
    q, _, _, do = inputs.make_inputs(1, rows // 2, H, d, seed=seed)
    _, k, v = inputs.make_inputs(1, rows // 2, Hk, d, seed=seed + 1, with_dout=False)
    cu = np.concatenate([[0], np.cumsum([2 * n for n in halves])]).astype(int).tolist()
    return q[0], k[0], v[0], do[0], cu


def _errors(got, ref):
    floor = 1e-3 * max(np.abs(r).max() for r in ref.values())
    return {name: float(np.abs(got[name] - r).max() / max(np.abs(r).max(), floor))
            for name, r in ref.items()}


CASES = [
    # (halves per sample, H, H_kv, d, bs)
    ([67, 0, 130, 5], 2, 2, 64, 3),
    ([1, 200, 64], 4, 2, 64, 16),
    ([129, 300, 0, 17], 2, 2, 128, 7),
    ([256, 128, 1], 4, 1, 128, 64),
    ([100, 3, 250], 2, 1, 128, 1),
    ([67, 130], 2, 2, 256, 3),
    ([200, 0, 31], 2, 1, 256, 16),
]


@pytest.mark.parametrize("halves,H,Hk,d,bs", CASES)
def test_varlen_matches_oracle(b, halves, H, Hk, d, bs):
    q, k, v, do, cu = _packed(halves, H, Hk, d, seed=500 + sum(halves) + d + H)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    out, lse = b.dfa_forward_varlen(qd, kd, vd, cu, bs)
    dq, dk, dv = b.dfa_backward_varlen(qd, kd, vd, out, dod, lse, cu, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    ro, rl = oracle.diffusion_varlen_forward(qn, kn, vn, cu, bs)
    rq, rk, rv = oracle.diffusion_varlen_backward(qn, kn, vn, don, cu, bs)
    e_out = float(np.abs(_np(out) - ro).max() / np.abs(ro).max())
    e_lse = float(np.abs(lse.cpu().double().numpy() - rl).max())
    errs = _errors({"dq": _np(dq), "dk": _np(dk), "dv": _np(dv)}, {"dq": rq, "dk": rk, "dv": rv})
    assert e_out <= TOL_OUT, (e_out, e_lse, errs)
    assert e_lse <= TOL_LSE, (e_out, e_lse, errs)
    assert max(errs.values()) <= TOL_GRAD, errs


@pytest.mark.parametrize("d", [64, 128, 256])
def test_equal_lengths_match_the_batched_path(b, d):
    # Samples of one length run the same tiles as the batched call: out, lse,
    # dk and dv are bitwise those of the batched kernels (dq sums float32
    # atomics in arrival order).
    B, n, H, bs = 3, 131, 2, 5
    q, k, v, do = inputs.make_inputs(B, n, H, d, seed=61 + d)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    ob, lb = b.dfa_forward(qd, kd, vd, bs)
    gb = b.dfa_backward(qd, kd, vd, ob, dod, lb, bs)
    pk = lambda t: t.reshape(B * 2 * n, H, d)  # noqa: E731
    cu = [0, 2 * n, 4 * n, 6 * n]
    ov, lv = b.dfa_forward_varlen(pk(qd), pk(kd), pk(vd), cu, bs)
    gv = b.dfa_backward_varlen(pk(qd), pk(kd), pk(vd), ov, pk(dod), lv, cu, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert torch.equal(ov, pk(ob))
    assert torch.equal(lv, lb.permute(1, 0, 2).reshape(H, B * 2 * n))
    assert torch.equal(gv[1], pk(gb[1])) and torch.equal(gv[2], pk(gb[2]))
    gap = (gv[0].float() - pk(gb[0]).float()).abs().max().item()
    assert gap <= 1e-2 * gb[0].float().abs().max().item()


def test_all_samples_empty_is_a_no_op(b):
    q, k, v, do, _ = _packed([2], 2, 2, 64, seed=3)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (t.to(dev)[:0] for t in (q, k, v))
    out, lse = b.dfa_forward_varlen(qd, kd, vd, [0, 0, 0], 4)
    torch.cuda.synchronize()
    assert out.shape == (0, 2, 64) and lse.shape == (2, 0)


def test_odd_sample_length_is_refused(b):
    from block_diffusion_masked_gb300.binding import DfaError

    q, k, v, _, _ = _packed([3, 4], 2, 2, 64, seed=4)
    dev = torch.device("cuda", 0)
    with pytest.raises(DfaError):
        b.dfa_forward_varlen(q.to(dev), k.to(dev), v.to(dev), [0, 5, 14], 2)


def test_autograd_varlen_function(b):
    from block_diffusion_masked_gb300 import diffusion_attn_varlen_func

    q, k, v, do, cu = _packed([40, 0, 97], 4, 2, 64, seed=8)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    out = diffusion_attn_varlen_func(qd, kd, vd, cu, 8)
    out.backward(do.to(dev))
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    ro, _ = oracle.diffusion_varlen_forward(qn, kn, vn, cu, 8)
    rq, rk, rv = oracle.diffusion_varlen_backward(qn, kn, vn, don, cu, 8)
    assert float(np.abs(_np(out) - ro).max() / np.abs(ro).max()) <= TOL_OUT
    errs = _errors({"dq": _np(qd.grad), "dk": _np(kd.grad), "dv": _np(vd.grad)},
                   {"dq": rq, "dk": rk, "dv": rv})
    assert max(errs.values()) <= TOL_GRAD, errs


@pytest.mark.parametrize("d,det", [(64, False), (128, False), (256, False), (128, True)])
def test_neighbour_samples_do_not_leak(b, d, det):
    """Non-finite values in one sample must not reach another sample's
    results: every sample is read through its own tensor maps, so rows past
    the end of a half read zero instead of the next sample's rows.  Sample 1
    (and the empty sample 2) sit between samples 0 and 3; inf and NaN are
    planted in all of sample 1's q, k, v, dout.  Samples 0 and 3 (ragged
    halves, so their last tiles run into the neighbours) must match the
    oracle on their own rows, finite everywhere."""
    halves = [67, 45, 0, 130]
    H, Hk, bs = 2, 1, 5
    q, k, v, do, cu = _packed(halves, H, Hk, d, seed=640 + d)
    a1, e1 = cu[1], cu[2]  # sample 1's rows
    for t, val in ((q, float("inf")), (k, float("nan")), (v, float("-inf")), (do, float("nan"))):
        t[a1:e1] = val
        t[a1 + 1] = float("inf")
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    out, lse = b.dfa_forward_varlen(qd, kd, vd, cu, bs)
    if det:
        dq, dk, dv = b.dfa_backward_ex(qd, kd, vd, out, dod, lse, bs, cu_seqlens=cu,
                                       deterministic=True)
    else:
        dq, dk, dv = b.dfa_backward_varlen(qd, kd, vd, out, dod, lse, cu, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    for s in (0, 3):
        a, e = cu[s], cu[s + 1]
        sub = [0, e - a]
        ro, rl = oracle.diffusion_varlen_forward(qn[a:e], kn[a:e], vn[a:e], sub, bs)
        rq, rk, rv = oracle.diffusion_varlen_backward(qn[a:e], kn[a:e], vn[a:e], don[a:e], sub,
                                                      bs)
        got = {"out": _np(out[a:e]), "dq": _np(dq[a:e]), "dk": _np(dk[a:e]),
               "dv": _np(dv[a:e])}
        for name, t in got.items():
            assert np.isfinite(t).all(), (s, name)
        g_lse = lse[:, a:e].cpu().double().numpy()
        assert np.isfinite(g_lse).all()
        assert np.abs(g_lse - rl).max() <= TOL_LSE
        errs = _errors(got, {"out": ro, "dq": rq, "dk": rk, "dv": rv})
        assert errs["out"] <= TOL_OUT, (s, errs)
        for name in ("dq", "dk", "dv"):
            assert errs[name] <= TOL_GRAD, (s, errs)
