"""GPU parity of the FP8 (e4m3) forward through the C ABI.

"Fast Diffusion Attention" lists an FP8 forward.  Here q, k, v are e4m3
with per-tensor descales; the oracle is the float64 definition applied to
the dequantized inputs (e4m3 -> float64 is exact).  The kernels accumulate
Q K^T and P V in float32 from exact e4m3 products and round only P to e4m3
(relative error <= 2^-4 for e4m3's normal range), with row sums taken
before that rounding.  So |out - oracle| <= 2^-4 * max|v| per element, plus
the bf16 rounding of out (2^-9 relative) and the underflow of
probabilities below e4m3's smallest subnormal, negligible for these
inputs: the bar is (2^-4 + 2^-8) * max|v|.  lse comes from float32 sums of
exact products: |lse - oracle| <= 1e-3.
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
    err = np.abs(got - ro).max() / np.abs(vn).max()
    assert err <= 2.0 ** -4 + 2.0 ** -8, err
    assert np.abs(lse.cpu().double().numpy() - rl).max() <= 1e-3


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
