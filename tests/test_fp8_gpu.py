"""GPU parity of the FP8 (e4m3) forward through the C ABI.

"Fast Diffusion Attention" lists an FP8 forward.  Here q, k, v are e4m3
with per-tensor descales; the reference is the float64 oracle applied to
the dequantized inputs (e4m3 -> float64 is exact).  The bar follows the
pages' accuracy methodology ("Accuracy": at most twice the error of a
straightforward PyTorch implementation in the same precision): the
comparator, inside this test only, is a float32 PyTorch forward on the
dequantized inputs on the GPU that rounds the unnormalised probabilities
exp(s - rowmax) to e4m3 before P V, divides by the float32 row sums of the
unrounded probabilities and rounds out to bf16 -- the precision the FP8
kernel computes in.  lse: |lse - oracle| <= 1e-3.
"""

import math

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


def _quantize(x):
    """Per-tensor e4m3 quantisation: (x8, descale) with x ~= x8 * descale."""
    scale = float(x.float().abs().max()) / 448.0
    return (x.float() / scale).to(torch.float8_e4m3fn), scale


@pytest.mark.parametrize("B,n,H,Hk,bs", [
    (1, 67, 2, 2, 3),
    (2, 300, 4, 2, 16),
    (1, 1000, 2, 1, 1),
    (1, 256, 2, 2, 64),
    (1, 1, 2, 1, 1),
])
def test_fp8_forward_matches_oracle(b, B, n, H, Hk, bs):
    d = 128
    q, _, _, _ = inputs.make_inputs(B, n, H, d, seed=700 + n, with_dout=True)
    _, k, v = inputs.make_inputs(B, n, Hk, d, seed=701 + n, with_dout=False)
    (q8, qs), (k8, ks), (v8, vs) = (_quantize(t) for t in (q, k, v))
    dev = torch.device("cuda", 0)
    out, lse = b.dfa_forward_fp8(q8.to(dev), k8.to(dev), v8.to(dev), qs, ks, vs, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    qn, kn, vn = (t.float().double().numpy() * s for t, s in ((q8, qs), (k8, ks), (v8, vs)))
    ro, rl = oracle.diffusion_forward(qn, kn, vn, bs)
    got = out.float().cpu().double().numpy()
    pt = _pytorch_fp8_forward(q8, k8, v8, qs, ks, vs, bs, dev)
    err, err_pt = np.abs(got - ro).max(), np.abs(pt - ro).max()
    assert err <= 2.0 * err_pt, (err, err_pt)
    assert np.abs(lse.cpu().double().numpy() - rl).max() <= 1e-3


def _pytorch_fp8_forward(q8, k8, v8, qs, ks, vs, bs, dev):
    """Straightforward float32 PyTorch forward with P rounded to e4m3."""
    B, L, H, d = q8.shape
    G = H // k8.shape[2]
    mask = torch.from_numpy(oracle.diffusion_mask(L // 2, bs)).to(dev)
    out = np.zeros((B, L, H, d))
    for bb in range(B):
        for h in range(H):
            q = q8[bb, :, h].to(dev).float() * qs
            k = k8[bb, :, h // G].to(dev).float() * ks
            v = v8[bb, :, h // G].to(dev).float() * vs
            s = (q @ k.t()) / math.sqrt(d)
            s = s.masked_fill(~mask, float("-inf"))
            p = torch.exp(s - s.max(dim=-1, keepdim=True).values)
            o = (p.to(torch.float8_e4m3fn).float() @ v) / p.sum(dim=-1, keepdim=True)
            out[bb, :, h] = o.to(torch.bfloat16).double().cpu().numpy()
    return out


def test_fp8_rejects_other_head_dims(b):
    from block_diffusion_masked_gb300.binding import DfaError

    q = torch.zeros((1, 8, 2, 64), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(DfaError):
        b.dfa_forward_fp8(q, q, q, 1.0, 1.0, 1.0, 2)


@pytest.mark.parametrize("n,Hk", [(300, 2), (67, 1)])
def test_fp8_two_step_equals_one_call(b, n, Hk):
    # dfa_fp8_transpose_v + dfa_forward_fp8_vt: bitwise the one-call forward
    B, H, d, bs = 2, 4, 128, 16
    q, _, _, _ = inputs.make_inputs(B, n, H, d, seed=710 + n)
    _, k, v = inputs.make_inputs(B, n, Hk, d, seed=711 + n, with_dout=False)
    (q8, qs), (k8, ks), (v8, vs) = (_quantize(t) for t in (q, k, v))
    dev = torch.device("cuda", 0)
    q8, k8, v8 = q8.to(dev), k8.to(dev), v8.to(dev)
    o1, l1 = b.dfa_forward_fp8(q8, k8, v8, qs, ks, vs, bs)
    vt = b.dfa_fp8_transpose_v(v8)
    o2, l2 = b.dfa_forward_fp8_vt(q8, k8, vt, Hk, qs, ks, vs, bs)
    torch.cuda.synchronize()
    assert b.dfa_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
