"""The library's tile enumeration against a brute-force walk over the mask.

For every query tile the forward enumeration must visit every key tile that
holds a visible pair and no other; for every key tile the backward
enumeration must visit every query tile that holds a visible pair and no
other; the "fully visible" flag must be exact.  The mask comes from the
oracle ("Fast Diffusion Attention", "Block diffusion in one picture"; causal
inside each half for the yardstick).
"""

import numpy as np
import pytest

import oracle
from block_diffusion_masked_gb300 import build as build_mod

RULES = {(0, 0): 0, (0, 1): 1, (1, 1): 2}  # (query half, key half) -> NN, NC, CC


@pytest.fixture(scope="module")
def b():
    build_mod.build()
    from block_diffusion_masked_gb300 import binding

    binding.lib()
    return binding


def _mask(mode, n, bs):
    if mode == 0:
        return oracle.diffusion_mask(n, bs)
    m = np.zeros((2 * n, 2 * n), dtype=bool)
    c = oracle.causal_mask(n)
    m[:n, :n] = c
    m[n:, n:] = c
    return m


def _tile(mask, n, qh, qt, bm, kh, kt, bn):
    """Visibility of a bm x bn tile, rows/keys past the half counted hidden."""
    t = np.zeros((bm, bn), dtype=bool)
    for a in range(bm):
        r = qt * bm + a
        if r >= n:
            continue
        for c in range(bn):
            k = kt * bn + c
            if k < n:
                t[a, c] = mask[qh * n + r, kh * n + k]
    return t


CASES = [(n, bs) for n in (1, 2, 5, 8, 13, 17, 24, 31) for bs in (1, 2, 3, 4, 5, 8, 9, 40)]
TILES = [(4, 4), (8, 4), (4, 8), (3, 5), (16, 16)]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("n,bs", CASES)
def test_forward_enumeration_is_exact(b, mode, n, bs):
    mask = _mask(mode, n, bs)
    for bm, bn in TILES:
        visits = 0
        for qh in (0, 1):
            for qt in range(-(-n // bm)):
                segs = b.dfa_fwd_segments(mode, n, bs, bm, bn, qh, qt)
                got = set()
                for kh, rule, t0, t1 in segs:
                    expect_rule = 3 if mode == 1 else RULES[(qh, kh)]
                    assert rule == expect_rule
                    for kt in range(t0, t1):
                        got.add((kh, kt))
                        t = _tile(mask, n, qh, qt, bm, kh, kt, bn)
                        full = bool(t.all())
                        assert b.dfa_tile_full(rule, n, bs, qt * bm, bm, kt * bn, bn) == int(full)
                visits += len(got)
                want = set()
                for kh in (0, 1):
                    for kt in range(-(-n // bn)):
                        if _tile(mask, n, qh, qt, bm, kh, kt, bn).any():
                            want.add((kh, kt))
                assert got == want, (qh, qt, bm, bn)
        assert b.dfa_tile_visits(mode, n, bs, bm, bn, 0) == visits


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("n,bs", CASES)
def test_backward_enumeration_is_exact(b, mode, n, bs):
    mask = _mask(mode, n, bs)
    for bm, bn in TILES:
        visits = 0
        for kh in (0, 1):
            for kt in range(-(-n // bn)):
                segs = b.dfa_bwd_segments(mode, n, bs, bm, bn, kh, kt)
                got = set()
                for qh, rule, t0, t1 in segs:
                    expect_rule = 3 if mode == 1 else RULES[(qh, kh)]
                    assert rule == expect_rule
                    for qt in range(t0, t1):
                        got.add((qh, qt))
                        t = _tile(mask, n, qh, qt, bm, kh, kt, bn)
                        assert b.dfa_tile_full(rule, n, bs, qt * bm, bm, kt * bn, bn) == int(t.all())
                visits += len(got)
                want = set()
                for qh in (0, 1):
                    for qt in range(-(-n // bm)):
                        if _tile(mask, n, qh, qt, bm, kh, kt, bn).any():
                            want.add((qh, qt))
                assert got == want, (kh, kt, bm, bn)
        assert b.dfa_tile_visits(mode, n, bs, bm, bn, 1) == visits


def test_noisy_diagonal_overhead_matches_page():
    # "Fast Diffusion Attention", "Visit only the visible tiles": the only
    # work beyond causal attention on the halves is the noisy diagonal, about
    # 5% more tiles at 2K tokens per half and 1% at 16K (128-wide tiles, a
    # block size smaller than the tile: one extra key tile per noisy query tile).
    build_mod.build()
    from block_diffusion_masked_gb300 import binding as bb

    for n, lo, hi in ((2048, 0.04, 0.08), (16384, 0.005, 0.015)):
        diff = bb.dfa_tile_visits(0, n, 16, 128, 128, 0)
        causal = bb.dfa_tile_visits(1, n, 1, 128, 128, 0)
        assert lo < diff / causal - 1 < hi, (n, diff, causal)


def _visits(b, pass_, mode, n, bs, half, tile, bm, bn):
    fn = b.dfa_fwd_segments if pass_ == 0 else b.dfa_bwd_segments
    return sum(e - s for (_, _, s, e) in fn(mode, n, bs, bm, bn, half, tile))


@pytest.mark.parametrize("pass_", [0, 1])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("batch,heads,n,bs,group", [
    (1, 1, 300, 16, 1), (2, 3, 700, 1, 2), (3, 5, 1024, 64, 4), (2, 4, 512, 512, 3),
    (1, 7, 129, 7, 7), (4, 2, 2048, 16, 3), (3, 2, 640, 1, 2),
])
def test_work_order_is_longest_first_with_short_tail(b, pass_, mode, batch, heads, n, bs, group):
    """The persistent kernels take items in this order from a counter: it must
    cover every (batch, head, half, tile) once, go longest first for each
    (batch, head) inside the grouped part, and end on the shortest items.
    In the causal mode `batch` counts sequences (any number, odd included):
    sequence s is reported as half s % 2 of sample s // 2, and the
    (sequence, head) pairs take the place of the (batch, head) pairs."""
    bm, bn = (128, 128) if pass_ == 0 else (64, 128)
    tiles = -(-n // (bm if pass_ == 0 else bn))
    BH = batch * heads
    per_pair = tiles if mode == 1 else 2 * tiles
    total = BH * per_pair
    order = [b.dfa_work_item(pass_, mode, w, batch, heads, tiles, group) for w in range(total)]
    if mode == 1:
        expect = [(s // 2, y, s % 2, t) for s in range(batch) for y in range(heads)
                  for t in range(tiles)]
    else:
        expect = [(x, y, h, t) for x in range(batch) for y in range(heads) for h in range(2)
                  for t in range(tiles)]
    assert sorted(order) == sorted(expect)
    pair = (lambda x, y, h: (2 * x + h, y)) if mode == 1 else (lambda x, y, h: (x, y))
    bs_eff = min(bs, n)
    vis = [_visits(b, pass_, mode, n, bs_eff, h, t, bm, bn) for (_, _, h, t) in order]
    if mode == 1:
        tail = min(tiles, 2)
    else:
        tail = min(2 * tiles, 4) if pass_ == 0 else tiles
    head = total - BH * tail
    if head > 0:
        if n % 128 == 0:  # a ragged last tile can be shorter than a tail item
            assert max(vis[head:]) <= min(vis[:head])
        seen = {}
        for (x, y, h, _), c in zip(order[:head], vis[:head]):
            key = pair(x, y, h)
            assert c <= seen.get(key, c)
            seen[key] = c
    # tail: rank by rank over all pairs, each rank covering every pair once
    pairs = sorted({pair(x, y, h) for (x, y, h, _) in expect})
    for r in range(tail):
        chunk = order[head + r * BH: head + (r + 1) * BH]
        assert sorted(pair(x, y, h) for (x, y, h, _) in chunk) == pairs
    with pytest.raises(b.DfaError):
        b.dfa_work_item(pass_, mode, total, batch, heads, tiles, group)


@pytest.mark.parametrize("batch,heads,n,bs,group", [
    (1, 1, 300, 16, 1), (2, 3, 700, 4, 2), (3, 5, 1024, 64, 4), (1, 7, 129, 128, 7),
    (4, 2, 2048, 16, 3), (2, 2, 100, 512, 1),
])
def test_noisy_diag_passes_split_the_backward(b, batch, heads, n, bs, group):
    """The two launches of the noisy-diagonal option ("Fast Diffusion
    Attention", "Hopper": a dedicated pass over the noisy diagonal, the main
    pass over the clean key tiles): together they cover exactly the items of
    the single backward pass; the clean pass goes longest first per pair and
    ends on its two shortest ranks; every noisy item visits only the query
    rows of its own key tile when the block size divides the tile."""
    bm, bn = 64, 128
    tiles = -(-n // bn)
    BH = batch * heads
    total = BH * tiles
    clean = [b.dfa_work_item(2, 0, w, batch, heads, tiles, group) for w in range(total)]
    noisy = [b.dfa_work_item(3, 0, w, batch, heads, tiles, group) for w in range(total)]
    single = [b.dfa_work_item(1, 0, w, batch, heads, tiles, group) for w in range(2 * total)]
    assert all(h == 1 for (_, _, h, _) in clean)
    assert all(h == 0 for (_, _, h, _) in noisy)
    assert sorted(clean + noisy) == sorted(single)
    assert len(set(clean)) == total and len(set(noisy)) == total
    bs_eff = min(bs, n)
    vis = [_visits(b, 1, 0, n, bs_eff, h, t, bm, bn) for (_, _, h, t) in clean]
    tail = min(tiles, 2)
    head = total - BH * tail
    seen = {}
    for (x, y, _, _), c in zip(clean[:head], vis[:head]):
        assert c <= seen.get((x, y), c)
        seen[(x, y)] = c
    pairs = sorted({(x, y) for (x, y, _, _) in clean})
    for r in range(tail):
        chunk = clean[head + r * BH: head + (r + 1) * BH]
        assert sorted((x, y) for (x, y, _, _) in chunk) == pairs
    if bn % bs_eff == 0 or n <= bn:
        # each noisy query row is visited by exactly one noisy key tile
        rows = []
        for t in range(tiles):
            for (qh, _, s, e) in b.dfa_bwd_segments(0, n, bs_eff, bm, bn, 0, t):
                assert qh == 0
                lo, hi = s * bm, min(e * bm, n)
                assert t * bn <= lo and hi <= (t + 1) * bn
                rows += range(lo, hi)
        assert sorted(rows) == list(range(n))
    for pass_ in (2, 3):
        with pytest.raises(b.DfaError):
            b.dfa_work_item(pass_, 0, total, batch, heads, tiles, group)
        with pytest.raises(b.DfaError):
            b.dfa_work_item(pass_, 1, 0, batch, heads, tiles, group)
