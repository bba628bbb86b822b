"""Pins of the oracle's grouped key/value heads (MQA / GQA).

"Fast Diffusion Attention" lists multi-query and grouped-query attention
among the supported shapes ("GQA-grouped backward"): k and v carry H_kv
heads, each read by H / H_kv consecutive query heads, and the gradient of a
key/value head sums over those query heads.  The oracle's grouped code is
pinned here against things other than itself: finite differences of the
loss, PyTorch autograd through an explicitly repeated key/value tensor, and
PyTorch's causal attention.
"""

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _torch_reference(q, k, v, dout, mask):
    """float64 PyTorch attention with repeated key/value heads and autograd.

    q, dout: (B, L, H, d); k, v: (B, L, H_kv, d); mask: (L, L) bool.  The
    repeat's backward sums each group's gradients, independently of the
    oracle's own accumulation.
    """
    H, Hk = q.shape[2], k.shape[2]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    kr = tk.repeat_interleave(H // Hk, dim=2)
    vr = tv.repeat_interleave(H // Hk, dim=2)
    s = torch.einsum("blhd,bmhd->bhlm", tq, kr) / np.sqrt(q.shape[3])
    s = s.masked_fill(~torch.tensor(mask), float("-inf"))
    p = torch.softmax(s, dim=-1)
    out = torch.einsum("bhlm,bmhd->blhd", p, vr)
    (out * torch.tensor(dout)).sum().backward()
    return out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("B,n,H,Hk,d,bs", [(2, 6, 4, 2, 5, 2), (1, 7, 3, 1, 4, 3),
                                           (1, 5, 6, 3, 3, 1)])
def test_grouped_oracle_matches_torch_autograd(B, n, H, Hk, d, bs):
    L = 2 * n
    q, do = _rand((B, L, H, d), 1), _rand((B, L, H, d), 2)
    k, v = _rand((B, L, Hk, d), 3), _rand((B, L, Hk, d), 4)
    out, _ = oracle.diffusion_forward(q, k, v, bs)
    dq, dk, dv = oracle.diffusion_backward(q, k, v, do, bs)
    ro, rq, rk, rv = _torch_reference(q, k, v, do, oracle.diffusion_mask(n, bs))
    for got, ref in ((out, ro), (dq, rq), (dk, rk), (dv, rv)):
        assert got.shape == ref.shape
        assert np.abs(got - ref).max() < 1e-12 * max(1.0, np.abs(ref).max())


def test_grouped_gradients_match_finite_differences():
    B, n, H, Hk, d, bs = 1, 4, 4, 2, 3, 2
    L = 2 * n
    q, do = _rand((B, L, H, d), 5), _rand((B, L, H, d), 6)
    k, v = _rand((B, L, Hk, d), 7), _rand((B, L, Hk, d), 8)

    def loss(qq, kk, vv):
        return float((oracle.diffusion_forward(qq, kk, vv, bs)[0] * do).sum())

    grads = oracle.diffusion_backward(q, k, v, do, bs)
    h = 1e-6
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g).max() / np.abs(num).max()
        assert err < 1e-6, (which, err)


def test_one_group_per_head_is_plain_multi_head():
    # H_kv == H: every query head reads its own key/value head.
    B, n, H, d, bs = 1, 6, 3, 4, 2
    q, k, v, do = (_rand((B, 2 * n, H, d), s) for s in (9, 10, 11, 12))
    out, lse = oracle.diffusion_forward(q, k, v, bs)
    for h in range(H):
        o, s = oracle.masked_attention_forward(q[0, :, h], k[0, :, h], v[0, :, h],
                                               oracle.diffusion_mask(n, bs))
        assert np.array_equal(out[0, :, h], o) and np.array_equal(lse[0, h], s)


def test_grouped_causal_oracle_matches_sdpa():
    B, L, H, Hk, d = 2, 9, 4, 2, 5
    q, do = _rand((B, L, H, d), 13), _rand((B, L, H, d), 14)
    k, v = _rand((B, L, Hk, d), 15), _rand((B, L, Hk, d), 16)
    out, _ = oracle.causal_forward(q, k, v)
    tq = torch.tensor(q).transpose(1, 2)
    tk = torch.tensor(k).repeat_interleave(H // Hk, dim=2).transpose(1, 2)
    tv = torch.tensor(v).repeat_interleave(H // Hk, dim=2).transpose(1, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    assert np.abs(out - ref.transpose(1, 2).numpy()).max() < 1e-12


def test_heads_must_divide():
    q = np.zeros((1, 4, 3, 2))
    k = np.zeros((1, 4, 2, 2))
    with pytest.raises(ValueError):
        oracle.diffusion_forward(q, k, k, 1)


def test_planted_head_mapping_mistake_is_caught(monkeypatch):
    # Interleaving the groups (h % H_kv instead of h // (H / H_kv)) must break
    # the autograd pin.
    from oracle import attention as oa

    def wrong(q, k):
        hk = k.shape[2]
        return lambda h: h % hk

    monkeypatch.setattr(oa, "_kv_head", wrong)
    B, n, H, Hk, d, bs = 1, 5, 4, 2, 3, 2
    q, do = _rand((B, 2 * n, H, d), 17), _rand((B, 2 * n, H, d), 18)
    k, v = _rand((B, 2 * n, Hk, d), 19), _rand((B, 2 * n, Hk, d), 20)
    out, _ = oa.diffusion_forward(q, k, v, bs)
    ro, *_ = _torch_reference(q, k, v, do, oa.diffusion_mask(n, bs))
    assert np.abs(out - ro).max() > 1e-3
