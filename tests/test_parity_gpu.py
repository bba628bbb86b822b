"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Same seeded bf16 inputs on both sides.  Error measure (normwise, per tensor):
max |gpu - oracle| / max |oracle|.  Bars: 1e-2 for out, 2e-2 for dq, dk and
dv (bf16 inputs, fp32 accumulation); |lse - oracle| <= 1e-3 absolute.
Small shapes are compared in full here; the full-size workloads are run at
full size and compared on sampled (batch, head) pairs in test_accuracy_gpu.py.
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


def normwise(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def _run_gpu(b, q, k, v, do, bs, backward=True):
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    out, lse = b.dfa_forward(qd, kd, vd, bs)
    grads = b.dfa_backward(qd, kd, vd, out, dod, lse, bs) if backward else None
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    res = {"out": _np(out), "lse": lse.cpu().double().numpy()}
    if backward:
        res.update(dq=_np(grads[0]), dk=_np(grads[1]), dv=_np(grads[2]))
    return res


def _check(res, q, k, v, do, bs, heads=None, backward=True):
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    if heads is None:
        B, _, H, _ = q.shape
        heads = [(bb, hh) for bb in range(B) for hh in range(H)]
    out, lse = oracle.diffusion_forward(qn, kn, vn, bs, heads=heads)
    sel = tuple(np.array(x) for x in zip(*heads))

    def pick(a, layout):  # layout "bshd" or "bhs"
        return a[sel[0], :, sel[1]] if layout == "bshd" else a[sel[0], sel[1]]

    errs = {"out": normwise(pick(res["out"], "bshd"), pick(out, "bshd")),
            "lse": float(np.abs(pick(res["lse"], "bhs") - pick(lse, "bhs")).max())}
    if backward:
        dq, dk, dv = oracle.diffusion_backward(qn, kn, vn, don, bs, heads=heads)
        refs = {"dq": pick(dq, "bshd"), "dk": pick(dk, "bshd"), "dv": pick(dv, "bshd")}
        # A gradient can be exactly zero (every row seeing a single key makes
        # dS = 0): then measure it against 1e-3 of the largest gradient.
        floor = 1e-3 * max(np.abs(r).max() for r in refs.values())
        for name, ref in refs.items():
            got = pick(res[name], "bshd")
            errs[name] = float(np.abs(got - ref).max() / max(np.abs(ref).max(), floor))
    assert np.isfinite(list(errs.values())).all(), errs
    assert errs["out"] <= TOL_OUT, errs
    assert errs["lse"] <= TOL_LSE, errs
    for name in ("dq", "dk", "dv"):
        if name in errs:
            assert errs[name] <= TOL_GRAD, errs
    return errs


def test_tiny_workload(b):
    w = inputs.WORKLOADS["tiny"]
    q, k, v, do = inputs.make_workload_inputs(w)
    res = _run_gpu(b, q, k, v, do, w.block_size)
    _check(res, q, k, v, do, w.block_size)


EDGE = [
    # (B, n, H, d, bs): ragged halves, block sizes that cut tiles, bs > n
    (1, 1, 1, 64, 1),
    (1, 67, 2, 64, 1),
    (1, 67, 2, 128, 3),
    (2, 129, 1, 128, 5),
    (1, 129, 2, 64, 64),
    (1, 200, 1, 128, 300),
    (1, 256, 2, 128, 16),
    (2, 300, 1, 64, 7),
    (1, 384, 1, 128, 128),
    (1, 130, 1, 128, 1),
]


@pytest.mark.parametrize("B,n,H,d,bs", EDGE)
def test_edge_cases(b, B, n, H, d, bs):
    q, k, v, do = inputs.make_inputs(B, n, H, d, seed=100 + n + bs)
    res = _run_gpu(b, q, k, v, do, bs)
    _check(res, q, k, v, do, bs)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("step", [0.5, 2.0])
def test_rising_scores_move_the_reference(b, d, step):
    """Scores that rise from one 64-key half-tile to the next by about 2^8
    or more in the softmax's base-2 units ("FlashAttention: Exact Attention
    Without Materialization", section 4.2: the online softmax rescales its
    running sum and output whenever the maximum grows): the kernels' reference
    maximum then moves on almost every tile, with the two halves of a tile
    disagreeing, and O and the row sum are rescaled.  out and lse must stay
    within the bars against the oracle.  (The backward, which reads the
    stored LSE and has no running maximum, is not compared here: on these
    inputs dQ sums large cancelling terms against K entries up to 32, so its
    normwise error measures bf16 rounding of dS rather than the kernel.)"""
    B, n, H, bs = 1, 300, 2, 16
    q, k, v, do = inputs.make_inputs(B, n, H, d, seed=900 + d)
    pos = torch.arange(2 * n) % n
    ramp = (pos // 64).float() * 16.0 * step
    q[..., 0] = 8.0
    k[..., 0] = ramp.view(1, -1, 1).to(k.dtype)
    res = _run_gpu(b, q, k, v, do, bs, backward=False)
    _check(res, q, k, v, do, bs, backward=False)


@pytest.mark.parametrize("n,bs", [(67, 3), (256, 64), (300, 1)])
def test_headdim_256(b, n, bs):
    q, k, v, do = inputs.make_inputs(1, n, 2, 256, seed=7 + n)
    res = _run_gpu(b, q, k, v, do, bs)
    _check(res, q, k, v, do, bs)


@pytest.mark.parametrize("Bc,n,H,d", [(4, 200, 2, 128), (1, 200, 2, 128), (3, 131, 2, 128),
                                      (3, 77, 2, 64), (1, 300, 2, 256), (5, 129, 1, 64)])
def test_causal_yardstick(b, Bc, n, H, d):
    """Causal attention on Bc sequences of length n ("The right yardstick"),
    any Bc (odd counts and a single sequence included), ragged lengths."""
    q, k, v, do = (t.view(-1, n, H, d)[:Bc].contiguous()
                   for t in inputs.make_inputs((Bc + 1) // 2, n, H, d, seed=11 + Bc))
    dev = torch.device("cuda", 0)
    qc, kc, vc, doc = (t.to(dev) for t in (q, k, v, do))
    out, lse = b.dfa_causal_forward(qc, kc, vc)
    dq, dk, dv = b.dfa_causal_backward(qc, kc, vc, out, doc, lse)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    ro, rl = oracle.causal_forward(qn, kn, vn)
    rq, rk, rv = oracle.causal_backward(qn, kn, vn, don)
    assert normwise(_np(out), ro) <= TOL_OUT
    assert np.abs(lse.cpu().double().numpy() - rl).max() <= TOL_LSE
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert normwise(_np(got), ref) <= TOL_GRAD


def test_autograd_function(b):
    from block_diffusion_masked_gb300 import diffusion_attn_func

    q, k, v, do = inputs.make_inputs(1, 96, 2, 64, seed=5)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    out = diffusion_attn_func(qd, kd, vd, 8)
    out.backward(do.to(dev))
    res = {"out": _np(out), "lse": np.zeros((1, 2, 192)), "dq": _np(qd.grad), "dk": _np(kd.grad),
           "dv": _np(vd.grad)}
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    ro, _ = oracle.diffusion_forward(qn, kn, vn, 8)
    rq, rk, rv = oracle.diffusion_backward(qn, kn, vn, don, 8)
    assert normwise(res["out"], ro) <= TOL_OUT
    for name, ref in (("dq", rq), ("dk", rk), ("dv", rv)):
        assert normwise(res[name], ref) <= TOL_GRAD

# The full-size configurations are compared on sampled heads, against both
# the tolerance bars and the pages' "twice a straightforward PyTorch bf16
# implementation" criterion, in test_accuracy_gpu.py.
