"""Pins of the oracle's packed (varlen) batches.

"Fast Diffusion Attention" describes varlen batches: samples of different
lengths packed along the rows, each attended to on its own.  The oracle's
varlen functions are pinned here against things other than themselves: the
batched oracle (itself pinned) when all lengths agree, PyTorch float64
autograd on each sample cut out by hand, central finite differences,
independence of the samples, and zero-length samples.
"""

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_equal_lengths_match_the_batched_oracle():
    B, n, H, Hk, d, bs = 3, 5, 4, 2, 3, 2
    q, do = _rand((B, 2 * n, H, d), 1), _rand((B, 2 * n, H, d), 2)
    k, v = _rand((B, 2 * n, Hk, d), 3), _rand((B, 2 * n, Hk, d), 4)
    cu = [0, 2 * n, 4 * n, 6 * n]
    pk = lambda x: x.reshape(B * 2 * n, *x.shape[2:])  # noqa: E731
    out, lse = oracle.diffusion_varlen_forward(pk(q), pk(k), pk(v), cu, bs)
    ro, rl = oracle.diffusion_forward(q, k, v, bs)
    assert np.allclose(out, pk(ro), rtol=0, atol=1e-13)
    assert np.allclose(lse, rl.transpose(1, 0, 2).reshape(H, B * 2 * n), rtol=0, atol=1e-13)
    dq, dk, dv = oracle.diffusion_varlen_backward(pk(q), pk(k), pk(v), pk(do), cu, bs)
    rq, rk, rv = oracle.diffusion_backward(q, k, v, do, bs)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.allclose(got, pk(ref), rtol=0, atol=1e-12)


def _torch_sample(q, k, v, dout, n, bs):
    """float64 autograd on one sample, mask built from the mask rules' text."""
    L = 2 * n
    pos = torch.arange(L)
    clean = pos >= n
    blk = (pos % n) // bs
    qc, kc = clean[:, None], clean[None, :]
    bi, bj = blk[:, None], blk[None, :]
    mask = ((~qc) & (~kc) & (bi == bj)) | ((~qc) & kc & (bj < bi)) | (qc & kc & (bj <= bi))
    H, Hk = q.shape[1], k.shape[1]
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kr = tk.repeat_interleave(H // Hk, dim=1)
    vr = tv.repeat_interleave(H // Hk, dim=1)
    s = torch.einsum("lhd,mhd->hlm", tq, kr) / np.sqrt(q.shape[2])
    s = s.masked_fill(~mask, float("-inf"))
    p = torch.softmax(s, dim=-1)
    out = torch.einsum("hlm,mhd->lhd", p, vr)
    (out * torch.tensor(dout)).sum().backward()
    return out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("lengths,bs", [([6, 0, 10, 4], 2), ([14, 2], 3), ([8, 8, 12], 16)])
def test_ragged_batch_matches_per_sample_autograd(lengths, bs):
    H, Hk, d = 4, 2, 3
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(int)
    rows = int(cu[-1])
    q, do = _rand((rows, H, d), 5), _rand((rows, H, d), 6)
    k, v = _rand((rows, Hk, d), 7), _rand((rows, Hk, d), 8)
    out, _ = oracle.diffusion_varlen_forward(q, k, v, cu, bs)
    dq, dk, dv = oracle.diffusion_varlen_backward(q, k, v, do, cu, bs)
    for b in range(len(lengths)):
        a, e = cu[b], cu[b + 1]
        if e == a:
            continue
        ro, rq, rk, rv = _torch_sample(q[a:e], k[a:e], v[a:e], do[a:e], (e - a) // 2, bs)
        for got, ref in ((out[a:e], ro), (dq[a:e], rq), (dk[a:e], rk), (dv[a:e], rv)):
            assert np.abs(got - ref).max() < 1e-12


def test_varlen_gradients_match_finite_differences():
    H, Hk, d, bs = 2, 1, 2, 2
    cu = [0, 4, 10]
    rows = cu[-1]
    q, do = _rand((rows, H, d), 9), _rand((rows, H, d), 10)
    k, v = _rand((rows, Hk, d), 11), _rand((rows, Hk, d), 12)

    def loss(qq, kk, vv):
        return float((oracle.diffusion_varlen_forward(qq, kk, vv, cu, bs)[0] * do).sum())

    grads = oracle.diffusion_varlen_backward(q, k, v, do, cu, bs)
    h = 1e-6
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.abs(num - g).max() / np.abs(num).max() < 1e-6


def test_samples_are_independent():
    H, d, bs = 2, 3, 2
    cu = [0, 6, 14]
    q, k, v = (_rand((14, H, d), s) for s in (13, 14, 15))
    out, lse = oracle.diffusion_varlen_forward(q, k, v, cu, bs)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for x in (q2, k2, v2):
        x[6:] = _rand((8, H, d), 99)  # change the second sample only
    out2, lse2 = oracle.diffusion_varlen_forward(q2, k2, v2, cu, bs)
    assert np.array_equal(out[:6], out2[:6]) and np.array_equal(lse[:, :6], lse2[:, :6])


def test_bad_lengths_raise():
    q = np.zeros((6, 1, 2))
    with pytest.raises(ValueError):
        oracle.diffusion_varlen_forward(q, q, q, [0, 3, 6], 1)  # odd lengths
    with pytest.raises(ValueError):
        oracle.diffusion_varlen_forward(q, q, q, [0, 4], 1)  # does not cover the rows


def test_planted_cross_sample_mask_is_caught(monkeypatch):
    # A mask over the whole packed sequence (samples not separated) must
    # break the per-sample pin.
    from oracle import attention as oa

    def merged(cu_seqlens, rows):
        return [(0, rows)]

    monkeypatch.setattr(oa, "_varlen_samples", merged)
    H, d, bs = 1, 3, 2
    cu = [0, 4, 12]
    q, k, v, do = (_rand((12, H, d), s) for s in (16, 17, 18, 19))
    out, _ = oa.diffusion_varlen_forward(q, k, v, cu, bs)
    ro, *_ = _torch_sample(q[:4], k[:4], v[:4], do[:4], 2, bs)
    assert np.abs(out[:4] - ro).max() > 1e-3
