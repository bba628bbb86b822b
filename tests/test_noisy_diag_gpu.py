"""GPU parity of the noisy-diagonal backward option (DFA_NOISY_DIAG_PASS).

"Fast Diffusion Attention", "Hopper: the FlashAttention-3 generation": the
block-diagonal noisy-noisy part of the backward runs on its own, writing the
noisy queries' first dQ and the complete dK / dV of the noisy keys, and the
main backward then visits the clean key tiles only.  Here that is two
launches of the same kernel (noisy key tiles, then clean key tiles), taken
when no block crosses a 128-key tile.  Checked, for every head dimension,
grouped heads and ragged halves:

* against the float64 oracle with the bars of the plain parity tests
  (normwise 1e-2 for out, 2e-2 for the gradients);
* dK and dV bitwise equal to the single launch (each key tile's sums are
  the same work in the same order);
* dQ equal to the single launch's up to the order of float32 additions;
* through the step API, that the noisy rows of the dQ accumulator are
  overwritten: junk left there beforehand does not reach dQ.

Block sizes that do not divide the tile fall back to the single launch
(bitwise equal results).
"""

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_masked_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_GRAD = 2e-2


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


def _inputs(B, n, H, Hk, d, seed):
    q, _, _, do = inputs.make_inputs(B, n, H, d, seed=seed)
    _, k, v = inputs.make_inputs(B, n, Hk, d, seed=seed + 1, with_dout=False)
    dev = torch.device("cuda", 0)
    return tuple(t.to(dev) for t in (q, k, v, do))


def _applies(n, bs):
    return 128 % min(bs, n) == 0 or n <= 128


def _same_to_rounding(x, y):
    """bf16 of float32 sums taken in another order: a unit in the last place
    of the value, or a float32 reassociation error where terms cancel."""
    x, y = x.float(), y.float()
    bar = x.abs() * 2.0 ** -7 + 1e-5 * float(x.abs().max())
    assert bool(((x - y).abs() <= bar).all()), float(((x - y).abs() / bar).max())


CASES = [
    # (B, n, H, Hk, d, bs)
    (2, 300, 2, 2, 128, 16),
    (1, 512, 2, 2, 128, 1),
    (1, 256, 4, 2, 128, 64),
    (2, 200, 2, 2, 128, 128),
    (1, 100, 2, 2, 128, 512),   # one tile per half: applies with any block size
    (1, 300, 2, 2, 128, 48),    # block crosses a tile: single launch
    (2, 300, 2, 2, 64, 4),
    (1, 257, 4, 1, 64, 32),
    (1, 300, 2, 2, 64, 24),     # single launch
    (1, 300, 2, 2, 256, 8),
    (2, 129, 4, 2, 256, 128),
    (1, 200, 2, 2, 256, 3),     # single launch
]


@pytest.mark.parametrize("B,n,H,Hk,d,bs", CASES)
def test_against_oracle_and_single_launch(b, B, n, H, Hk, d, bs):
    q, k, v, do = _inputs(B, n, H, Hk, d, seed=7100 + n + d + bs)
    out, lse = b.dfa_forward_gqa(q, k, v, bs)
    one = b.dfa_backward_ex(q, k, v, out, do, lse, bs)
    two = b.dfa_backward_ex(q, k, v, out, do, lse, bs, noisy_diag_pass=True)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert torch.equal(one[1], two[1]) and torch.equal(one[2], two[2])
    if not _applies(n, bs):
        assert torch.equal(one[0], two[0])
    else:
        # bf16 of float32 sums in another order: at most a unit in the last place
        _same_to_rounding(one[0], two[0])
    qn, kn, vn, don = (_np(t) for t in (q, k, v, do))
    ref = oracle.diffusion_backward(qn, kn, vn, don, bs)
    floor = 1e-3 * max(np.abs(r).max() for r in ref)
    for name, got, r in zip(("dq", "dk", "dv"), two, ref):
        err = float(np.abs(_np(got) - r).max() / max(np.abs(r).max(), floor))
        assert err <= TOL_GRAD, (name, err)


@pytest.mark.parametrize("d,bs", [(64, 16), (128, 4), (256, 64)])
def test_step_api_overwrites_noisy_rows(b, d, bs):
    B, n, H = 2, 300, 2
    q, k, v, do = _inputs(B, n, H, H, d, seed=7300 + d)
    dev = q.device
    out, lse = b.dfa_forward(q, k, v, bs)
    delta = torch.empty(B, H, 2 * n, dtype=torch.float32, device=dev)
    dq_acc = torch.empty(B, 2 * n, H, d, dtype=torch.float32, device=dev)
    b.dfa_bwd_preprocess(out, do, delta, dq_acc)
    ref_acc = dq_acc.clone()
    dk0, dv0 = torch.empty_like(k), torch.empty_like(v)
    b.dfa_bwd_main_gqa(q, k, v, do, lse, delta, ref_acc, dk0, dv0, bs)
    # junk in the noisy rows: the noisy-diagonal launch stores over it
    g = torch.Generator(device=dev).manual_seed(11)
    dq_acc[:, :n] = torch.randn(B, n, H, d, generator=g, device=dev) * 1e3
    dk1, dv1 = torch.empty_like(k), torch.empty_like(v)
    b.dfa_bwd_main_ex(q, k, v, do, lse, delta, dq_acc, dk1, dv1, bs, noisy_diag_pass=True)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    scale = float(ref_acc.abs().max())
    assert float((dq_acc - ref_acc).abs().max()) <= 1e-5 * scale


def test_full_size_mid_workload(b):
    """The mid configuration at full size: dK / dV bitwise, dQ to rounding."""
    w = inputs.WORKLOADS["mid"]
    q, k, v, do = (t.to(torch.device("cuda", 0)) for t in inputs.make_workload_inputs(w))
    out, lse = b.dfa_forward(q, k, v, w.block_size)
    one = b.dfa_backward_ex(q, k, v, out, do, lse, w.block_size)
    two = b.dfa_backward_ex(q, k, v, out, do, lse, w.block_size, noisy_diag_pass=True)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert torch.equal(one[1], two[1]) and torch.equal(one[2], two[2])
    _same_to_rounding(one[0], two[0])
