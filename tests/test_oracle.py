"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test checks the oracle against the pages (hand-drawn masks, the printed
pair count, the worked online-softmax example), against library routines for
the special cases where block-diffusion attention reduces to textbook
attention (PyTorch's causal and unmasked attention in float64), against
per-row gathers written independently of the full-matrix code, and against
finite differences for the gradients.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _read_mask(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c == "1" for c in line.replace(" ", "")])
    return np.array(rows, dtype=bool)


# ---------------------------------------------------------------- the mask

@pytest.mark.parametrize("name,n,bs", [("mask_n6_bs2.txt", 6, 2), ("mask_n5_bs2.txt", 5, 2)])
def test_mask_matches_hand_drawn(name, n, bs):
    want = _read_mask(name)
    assert want.shape == (2 * n, 2 * n)
    np.testing.assert_array_equal(oracle.diffusion_mask(n, bs), want)
    for i in range(2 * n):
        for j in range(2 * n):
            assert oracle.visible(i, j, n, bs) == want[i, j]


@pytest.mark.parametrize("n,bs", [(64, 4), (6, 2), (12, 3), (32, 32), (16, 1), (40, 8)])
def test_pair_count_printed_formula(n, bs):
    # "The right yardstick": n^2 + n*block_size visible pairs per sample.
    assert n % bs == 0
    assert int(oracle.diffusion_mask(n, bs).sum()) == n * n + n * bs
    assert oracle.visible_pairs(n, bs) == n * n + n * bs


def test_pair_count_tiny_workload():
    assert int(oracle.diffusion_mask(64, 4).sum()) == 4352


@pytest.mark.parametrize("n", range(1, 14))
def test_pair_count_any_block_size(n):
    for bs in range(1, n + 3):
        assert oracle.visible_pairs(n, bs) == int(oracle.diffusion_mask(n, bs).sum())


def test_every_row_has_a_visible_key():
    for n in range(1, 12):
        for bs in range(1, n + 2):
            assert oracle.diffusion_mask(n, bs).any(axis=1).all()


# ------------------------------------------- special cases and gathers

def _gather_row_attention(q, k, v, keys, scale):
    """Attention of one query row over an explicit list of keys."""
    s = np.array([scale * float(np.dot(q, k[j])) for j in keys])
    w = np.exp(s - s.max())
    w = w / w.sum()
    return sum(w[t] * v[j] for t, j in enumerate(keys)), math.log(np.exp(s - s.max()).sum()) + s.max()


@pytest.mark.parametrize("n,bs,d", [(7, 2, 5), (9, 3, 4), (8, 8, 3), (6, 10, 4)])
def test_rows_equal_per_row_gather(n, bs, d):
    # Clean rows: block-causal attention on the clean half alone.  Noisy rows:
    # attention over (clean keys of earlier blocks) + (noisy keys of own block),
    # i.e. the KV-cache reading of "Block diffusion in one picture".
    L = 2 * n
    q, k, v = (_rand((L, d), s) for s in (1, 2, 3))
    scale = 1 / math.sqrt(d)
    out, lse = oracle.masked_attention_forward(q, k, v, oracle.diffusion_mask(n, bs))
    for i in range(L):
        r, b = i % n, (i % n) // bs
        if i >= n:
            keys = [n + t for t in range(n) if t // bs <= b]
        else:
            keys = [n + t for t in range(n) if t // bs < b] + [t for t in range(n) if t // bs == b]
        o_i, lse_i = _gather_row_attention(q[i], k, v, keys, scale)
        np.testing.assert_allclose(out[i], o_i, rtol=1e-12, atol=1e-12)
        assert abs(lse[i] - lse_i) < 1e-12


def test_clean_half_ignores_noisy_half():
    n, bs, d = 10, 3, 6
    q, k, v = (_rand((2 * n, d), s) for s in (4, 5, 6))
    mask = oracle.diffusion_mask(n, bs)
    out1, _ = oracle.masked_attention_forward(q, k, v, mask)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:n] += 3.0
    k2[:n] -= 2.0
    v2[:n] *= 5.0
    out2, _ = oracle.masked_attention_forward(q2, k2, v2, mask)
    np.testing.assert_array_equal(out1[n:], out2[n:])


def _sdpa(q, k, v, causal):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64)[None, None] for x in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)[0, 0].numpy()


def _sdpa_grads(q, k, v, dout, causal):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                                         is_causal=causal)[0, 0]
    (o * torch.tensor(dout, dtype=torch.float64)).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("n,d", [(9, 4), (16, 8)])
def test_block_size_one_clean_half_is_causal(n, d):
    # "Accuracy": with block_size = 1 the clean half is causal attention.
    q, k, v, do = (_rand((2 * n, d), s) for s in (7, 8, 9, 10))
    do[:n] = 0.0   # no gradient flows in from the noisy rows
    mask = oracle.diffusion_mask(n, 1)
    out, _ = oracle.masked_attention_forward(q, k, v, mask)
    np.testing.assert_allclose(out[n:], _sdpa(q[n:], k[n:], v[n:], True), rtol=1e-12, atol=1e-13)
    dq, dk, dv = oracle.masked_attention_backward(q, k, v, do, mask)
    gq, gk, gv = _sdpa_grads(q[n:], k[n:], v[n:], do[n:], True)
    np.testing.assert_allclose(dq[n:], gq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk[n:], gk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv[n:], gv, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("n,bs,d", [(8, 8, 4), (7, 20, 5)])
def test_block_size_at_least_n_is_full_attention_per_half(n, bs, d):
    q, k, v, do = (_rand((2 * n, d), s) for s in (11, 12, 13, 14))
    mask = oracle.diffusion_mask(n, bs)
    out, _ = oracle.masked_attention_forward(q, k, v, mask)
    dq, dk, dv = oracle.masked_attention_backward(q, k, v, do, mask)
    for sl in (slice(0, n), slice(n, 2 * n)):
        np.testing.assert_allclose(out[sl], _sdpa(q[sl], k[sl], v[sl], False), rtol=1e-12, atol=1e-13)
        gq, gk, gv = _sdpa_grads(q[sl], k[sl], v[sl], do[sl], False)
        np.testing.assert_allclose(dq[sl], gq, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dk[sl], gk, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dv[sl], gv, rtol=1e-10, atol=1e-12)


def test_causal_yardstick_oracle_matches_sdpa():
    B, L, H, d = 2, 13, 2, 8
    q, k, v, do = (_rand((B, L, H, d), s) for s in (15, 16, 17, 18))
    out, lse = oracle.causal_forward(q, k, v)
    dq, dk, dv = oracle.causal_backward(q, k, v, do)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(out[b, :, h], _sdpa(q[b, :, h], k[b, :, h], v[b, :, h], True),
                                       rtol=1e-12, atol=1e-13)
            g = _sdpa_grads(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], True)
            for mine, ref in zip((dq, dk, dv), g):
                np.testing.assert_allclose(mine[b, :, h], ref, rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------- invariants

def test_probabilities_and_lse_invariants():
    n, bs, d = 11, 3, 4
    L = 2 * n
    q, k = _rand((L, d), 20), _rand((L, d), 21)
    mask = oracle.diffusion_mask(n, bs)
    ones = np.ones((L, 1))
    out, lse = oracle.masked_attention_forward(q, k, ones, mask)
    np.testing.assert_allclose(out[:, 0], 1.0, rtol=0, atol=1e-14)     # rows of P sum to 1
    s = (q @ k.T) / math.sqrt(d)
    for i in range(L):
        vis = s[i][mask[i]]
        ref = vis.max() + math.log(np.exp(vis - vis.max()).sum())
        assert abs(lse[i] - ref) < 1e-12


def test_masked_pairs_have_exactly_zero_gradient():
    # dout only on clean rows: clean queries see no noisy keys, so every
    # gradient at a noisy position is exactly zero.
    n, bs, d = 12, 4, 5
    q, k, v, do = (_rand((2 * n, d), s) for s in (22, 23, 24, 25))
    do[:n] = 0.0
    dq, dk, dv = oracle.masked_attention_backward(q, k, v, do, oracle.diffusion_mask(n, bs))
    assert np.all(dq[:n] == 0.0) and np.all(dk[:n] == 0.0) and np.all(dv[:n] == 0.0)
    assert np.abs(dq[n:]).max() > 0 and np.abs(dk[n:]).max() > 0


# ------------------------------------------------ finite differences

@pytest.mark.parametrize("n,bs,d", [(5, 2, 4), (8, 3, 4), (4, 1, 3)])
def test_gradients_match_finite_differences(n, bs, d):
    L = 2 * n
    q, k, v, do = (_rand((L, d), s) for s in (30, 31, 32, 33))
    mask = oracle.diffusion_mask(n, bs)

    def loss(qq, kk, vv):
        return float((oracle.masked_attention_forward(qq, kk, vv, mask)[0] * do).sum())

    grads = oracle.masked_attention_backward(q, k, v, do, mask)
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


# --------------------------------------------- the online-softmax example

def _read_example():
    blocks, rec = [], {}
    with open(os.path.join(GOLDEN, "online_softmax_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "block":
                blocks.append([float(x) for x in vals])
            else:
                rec[key] = [float(x) for x in vals]
    return blocks, rec


def test_online_softmax_worked_example():
    blocks, rec = _read_example()
    m1, _, _, hist1 = oracle.online_softmax_row(blocks[:1])
    assert m1 == rec["after_block1_max"][0]
    np.testing.assert_allclose(hist1[-1], np.exp(rec["after_block1_weights_exp"]), rtol=1e-15)
    m2, ell, _, hist = oracle.online_softmax_row(blocks)
    assert m2 == rec["after_block2_max"][0]
    np.testing.assert_allclose(hist[-1], np.exp(rec["after_block2_weights_exp"]), rtol=1e-15)
    allscores = np.concatenate([np.array(b) for b in blocks])
    ref = np.exp(allscores - allscores.max())
    ref = ref / ref.sum()
    np.testing.assert_allclose(hist[-1] / ell, ref, rtol=1e-15)


def test_online_softmax_equals_plain_softmax_with_values():
    rng = np.random.default_rng(40)
    s = rng.standard_normal(23) * 3
    vals = rng.standard_normal((23, 4))
    cuts = [0, 5, 6, 15, 23]
    blocks = [s[a:b] for a, b in zip(cuts[:-1], cuts[1:])]
    vblocks = [vals[a:b] for a, b in zip(cuts[:-1], cuts[1:])]
    _, ell, z, _ = oracle.online_softmax_row(blocks, vblocks)
    w = np.exp(s - s.max())
    np.testing.assert_allclose(z / ell, (w / w.sum()) @ vals, rtol=1e-13)


# ------------------------------------- planted mistakes are caught

def _mutant_masks(n, bs):
    pos = np.arange(2 * n)
    clean = pos >= n
    blk = (pos % n) // bs
    qc, kc, bi, bj = clean[:, None], clean[None, :], blk[:, None], blk[None, :]
    good_nn = (~qc) & (~kc) & (bi == bj)
    good_nc = (~qc) & kc & (bj < bi)
    good_cc = qc & kc & (bj <= bi)
    yield "nc_inclusive", good_nn | ((~qc) & kc & (bj <= bi)) | good_cc
    yield "cc_strict", good_nn | good_nc | (qc & kc & (bj < bi) | (qc & kc & (pos[:, None] == pos[None, :])))
    yield "nn_causal", ((~qc) & (~kc) & (bi == bj) & (pos[None, :] <= pos[:, None])) | good_nc | good_cc
    yield "cn_open", good_nn | good_nc | good_cc | (qc & (~kc) & (bj < bi))


@pytest.mark.parametrize("n,bs", [(6, 2), (8, 4)])
def test_pins_catch_planted_mask_mistakes(n, bs):
    # Each mutant differs from the page's rule in one place; the hand-drawn
    # mask or the pair count must reject it.
    want = _read_mask("mask_n6_bs2.txt") if (n, bs) == (6, 2) else None
    for name, m in _mutant_masks(n, bs):
        caught = (int(m.sum()) != n * n + n * bs) or (want is not None and not np.array_equal(m, want))
        if not caught:
            # fall back to the per-row gather pin
            q, k, v = (_rand((2 * n, 3), s) for s in (50, 51, 52))
            out, _ = oracle.masked_attention_forward(q, k, v, m)
            ref, _ = oracle.masked_attention_forward(q, k, v, oracle.diffusion_mask(n, bs))
            caught = not np.allclose(out, ref)
        assert caught, name


def test_planted_gradient_mistake_is_caught():
    # Dropping the "- D" term of dS must break the finite-difference pin.
    n, bs, d = 4, 2, 3
    q, k, v, do = (_rand((2 * n, d), s) for s in (60, 61, 62, 63))
    mask = oracle.diffusion_mask(n, bs)
    scale = 1 / math.sqrt(d)
    p, _ = oa._probabilities(q, k, mask, scale)
    wrong_dq = scale * ((p * (do @ v.T)) @ k)
    def loss(qq):
        return float((oracle.masked_attention_forward(qq, k, v, mask)[0] * do).sum())
    num = np.zeros_like(q)
    for idx in np.ndindex(*q.shape):
        a, b = q.copy(), q.copy()
        a[idx] += 1e-6
        b[idx] -= 1e-6
        num[idx] = (loss(a) - loss(b)) / 2e-6
    assert np.abs(num - wrong_dq).max() / np.abs(num).max() > 1e-3
    good_dq = oracle.masked_attention_backward(q, k, v, do, mask)[0]
    assert np.abs(num - good_dq).max() / np.abs(num).max() < 1e-6
