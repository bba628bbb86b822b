"""Grouped, packed and FP8 paths at the benchmark's full size, sampled.

The bench's variant lines (`--variant gqa|varlen|fp8`) run the small
workload's shapes (8 x 2048 rows, 16 heads, headdim 128, block size 16).
Here the same calls run at that size on the GPU and the oracle recomputes a
few outputs one head (or one sample) at a time: for grouped heads every
query head of one key/value head, so that its dk and dv are complete; for
the packed batch one sample, cut out and given to the batched oracle (which
the varlen pins tie to the varlen oracle).  Bars as in the smaller parity
tests.
"""

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_masked_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

W = inputs.WORKLOADS["small"]


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


def _rel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def test_gqa_full_size_sampled(b):
    H, Hk, d, bs = W.heads, W.heads // 4, W.headdim, W.block_size
    q, _, _, do = inputs.make_workload_inputs(W)
    _, k, v = inputs.make_inputs(W.batch, W.n, Hk, d, seed=W.seed + 1, with_dout=False)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    out, lse = b.dfa_forward_gqa(qd, kd, vd, bs)
    dq, dk, dv = b.dfa_backward_gqa(qd, kd, vd, out, dod, lse, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    bb, hk = 5, 2  # one key/value head of one sample, with its 4 query heads
    hs = [hk * (H // Hk) + i for i in range(H // Hk)]
    sel = lambda t: _np(t[bb:bb + 1])  # noqa: E731
    qn, kn, vn, don = (sel(t) for t in (q, k, v, do))
    heads = [(0, h) for h in hs]
    ro, rl = oracle.diffusion_forward(qn, kn, vn, bs, heads=heads)
    rq, rk, rv = oracle.diffusion_backward(qn, kn, vn, don, bs, heads=heads)
    assert _rel(_np(out[bb][:, hs]), ro[0][:, hs]) <= 1e-2
    assert np.abs(lse[bb, hs].cpu().double().numpy() - rl[0, hs]).max() <= 1e-3
    assert _rel(_np(dq[bb][:, hs]), rq[0][:, hs]) <= 2e-2
    assert _rel(_np(dk[bb][:, hk]), rk[0][:, hk]) <= 2e-2
    assert _rel(_np(dv[bb][:, hk]), rv[0][:, hk]) <= 2e-2


def test_varlen_full_size_sampled(b):
    H, d, bs = W.heads, W.headdim, W.block_size
    halves = [1536, 1280, 1152, 1024, 1024, 896, 768, 512]  # the bench's mix
    rows = 2 * sum(halves)
    q, k, v, do = (t[0] for t in inputs.make_inputs(1, rows // 2, H, d, seed=W.seed))
    cu = np.concatenate([[0], np.cumsum([2 * h for h in halves])]).astype(int).tolist()
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    out, lse = b.dfa_forward_varlen(qd, kd, vd, cu, bs)
    dq, dk, dv = b.dfa_backward_varlen(qd, kd, vd, out, dod, lse, cu, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    for s, h in ((0, 3), (7, 11)):  # the longest sample and the shortest
        a, e = cu[s], cu[s + 1]
        qn, kn, vn, don = (_np(t[a:e])[None] for t in (q, k, v, do))
        ro, rl = oracle.diffusion_forward(qn, kn, vn, bs, heads=[(0, h)])
        rq, rk, rv = oracle.diffusion_backward(qn, kn, vn, don, bs, heads=[(0, h)])
        assert _rel(_np(out[a:e, h]), ro[0, :, h]) <= 1e-2
        assert np.abs(lse[h, a:e].cpu().double().numpy() - rl[0, h]).max() <= 1e-3
        for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
            assert _rel(_np(got[a:e, h]), ref[0, :, h]) <= 2e-2


def test_fp8_full_size_sampled(b):
    H, d, bs = W.heads, W.headdim, W.block_size
    q, k, v = inputs.make_workload_inputs(W, with_dout=False)
    scales = [float(t.float().abs().max()) / 448.0 for t in (q, k, v)]
    q8, k8, v8 = ((t.float() / s).to(torch.float8_e4m3fn) for t, s in zip((q, k, v), scales))
    dev = torch.device("cuda", 0)
    out, lse = b.dfa_forward_fp8(q8.to(dev), k8.to(dev), v8.to(dev), *scales, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    bb = 6
    qn, kn, vn = (t[bb:bb + 1].float().double().numpy() * s
                  for t, s in zip((q8, k8, v8), scales))
    heads = [(0, 0), (0, H - 1)]
    ro, rl = oracle.diffusion_forward(qn, kn, vn, bs, heads=heads)
    for _, h in heads:
        err = np.abs(_np(out[bb][:, h]) - ro[0][:, h]).max() / np.abs(vn[0][:, h]).max()
        assert err <= 2.0 ** -4 + 2.0 ** -8
        assert np.abs(lse[bb, h].cpu().double().numpy() - rl[0, h]).max() <= 1e-3
