"""Plain float64 definition of attention under the block-diffusion mask.

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
baseline leg of the benchmark; never by the product path.  Every result
here is the textbook definition written out on the full score matrix, with
NumPy matmuls as the only library steps.  No tiling, no online softmax, no
reordering of sums beyond what a matmul does internally.

Sources (the web pages this build follows):

* "Fast Diffusion Attention", section "Block diffusion in one picture":
  the sequence is the concatenation [noisy | clean] of two halves of n
  tokens, cut into blocks of ``block_size`` tokens.  A noisy block sees
  itself (both directions) and the clean blocks strictly before it; a clean
  block sees itself and the clean blocks before it; nothing else is visible.
* Same page, section "The right yardstick": the visible pairs of one sample
  number n^2 + n*block_size (when block_size divides n); the yardstick is
  causal attention on the 2B halves of length n; FLOPs count visible pairs
  only, 4*pairs*headdim*heads forward and 2.5x that backward.
* "FlashAttention: Exact Attention Without Materialization", sections 2.3
  (stable softmax), 4.2 (online softmax), 4.3 (worked example) and 4.5
  (backward pass: store the output and one log-sum-exp per row, recompute
  the probabilities).

Readings where the pages are silent (each is listed in the design notes):

* blocks start at position 0 of each half; when block_size does not divide
  n the last block of a half is short; block_size > n makes one block per
  half;
* "previous clean blocks" means strictly earlier blocks;
* the softmax scale is 1/sqrt(headdim);
* the log-sum-exp is the natural log of the sum of exp(scaled scores), laid
  out (batch, heads, 2n).

Every function here is pinned by a CPU test against something other than
itself (finite differences, per-row gathers, PyTorch's own causal and
unmasked attention, closed-form pair counts, the printed worked example).
"""

from __future__ import annotations

import math

import numpy as np

HALF_NOISY = 0
HALF_CLEAN = 1


# --------------------------------------------------------------------------
# The mask ("Fast Diffusion Attention", "Block diffusion in one picture")
# --------------------------------------------------------------------------

def visible(i: int, j: int, n: int, block_size: int) -> bool:
    """Whether query position i may attend to key position j, 0 <= i, j < 2n.

    Positions < n are the noisy half, positions >= n the clean half; the
    block of a position is its offset inside its half divided by block_size.
    """
    qi_clean, kj_clean = i >= n, j >= n
    bi, bj = (i % n) // block_size, (j % n) // block_size
    if not qi_clean and not kj_clean:      # noisy query, noisy key: own block
        return bi == bj
    if not qi_clean and kj_clean:          # noisy query, clean key: earlier blocks
        return bj < bi
    if qi_clean and kj_clean:              # clean query, clean key: block-causal
        return bj <= bi
    return False                           # clean query never sees noisy keys


def diffusion_mask(n: int, block_size: int) -> np.ndarray:
    """Boolean (2n, 2n) matrix M with M[i, j] = visible(i, j)."""
    pos = np.arange(2 * n)
    clean = pos >= n
    blk = (pos % n) // block_size
    qc, kc = clean[:, None], clean[None, :]
    bi, bj = blk[:, None], blk[None, :]
    nn = (~qc) & (~kc) & (bi == bj)
    nc = (~qc) & kc & (bj < bi)
    cc = qc & kc & (bj <= bi)
    return nn | nc | cc


def causal_mask(length: int) -> np.ndarray:
    """Lower-triangular (length, length) mask of causal attention."""
    return np.tril(np.ones((length, length), dtype=bool))


def visible_pairs(n: int, block_size: int) -> int:
    """Visible (query, key) pairs of one sample, counted row by row.

    Row r of a half (block b = r // block_size, block end e = min(n, (b+1)*bs)):
    a clean row sees e clean keys; a noisy row sees the b*bs clean keys of the
    earlier blocks plus the e - b*bs noisy keys of its own block, i.e. also e.
    So each half holds sum_r e(r) pairs.  When block_size divides n this is
    (n^2 + n*block_size)/2 per half, n^2 + n*block_size per sample, the count
    printed in "The right yardstick".
    """
    total = 0
    for r in range(n):
        b = r // block_size
        total += min(n, (b + 1) * block_size)
    return 2 * total


# --------------------------------------------------------------------------
# Attention on one head under an arbitrary mask (plain definition)
# --------------------------------------------------------------------------

def _probabilities(q, k, mask, scale):
    """P = softmax(scale * q k^T) over the visible keys of each row, plus LSE.

    Stable softmax as in section 2.3 of the FlashAttention page: subtract the
    row maximum before exponentiating.  Masked scores are -inf, so their
    probability is exactly 0.  Every row must keep one visible key.
    """
    s = scale * (q @ k.T)
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    if not np.all(np.isfinite(m)):
        raise ValueError("a query row has no visible key")
    e = np.exp(s - m)
    ell = e.sum(axis=1, keepdims=True)
    p = e / ell
    lse = (m + np.log(ell))[:, 0]
    return p, lse


def masked_attention_forward(q, k, v, mask, scale=None):
    """out = softmax(scale q k^T + mask) v and the natural-log LSE per row.

    q, k, v: float64 (L, d); mask: bool (L, L).  Returns out (L, d), lse (L,).
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[1])
    p, lse = _probabilities(q, k, mask, scale)
    return p @ v, lse


def masked_attention_backward(q, k, v, dout, mask, scale=None):
    """Gradients of L = sum(dout * out) with respect to q, k and v.

    Analytic backward of softmax attention, recomputing P from q and k as the
    FlashAttention page (section 4.5) prescribes:
        dV = P^T dO,   dP = dO V^T,   D_i = sum_j P_ij dP_ij,
        dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q.
    dS is exactly zero wherever the mask hides a pair, because P is.
    Returns dq, dk, dv, each (L, d) float64.
    """
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[1])
    p, _ = _probabilities(q, k, mask, scale)
    dv = p.T @ dout
    dp = dout @ v.T
    delta = (p * dp).sum(axis=1, keepdims=True)
    ds = p * (dp - delta)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


# --------------------------------------------------------------------------
# Batched wrappers in the layout of the pages' API:
# q, k, v, out: (batch, 2n, heads, headdim); lse: (batch, heads, 2n).
# --------------------------------------------------------------------------

def _check_layout(q):
    if q.ndim != 4 or q.shape[1] % 2:
        raise ValueError("expected (batch, 2n, heads, headdim) with an even 2n")


def _kv_head(q, k):
    """Map query head h to its key/value head.

    Multi-query and grouped-query attention ("Fast Diffusion Attention",
    "GQA-grouped backward"): k and v carry H_kv heads, H_kv dividing the H
    query heads; query head h reads key/value head h // (H / H_kv), so each
    key/value head serves a run of H / H_kv consecutive query heads (the
    pages do not spell out the grouping; this is the usual one).
    """
    H, Hk = q.shape[2], k.shape[2]
    if Hk < 1 or H % Hk:
        raise ValueError("key/value heads must divide query heads")
    g = H // Hk
    return lambda h: h // g


def diffusion_forward(q, k, v, block_size, heads=None):
    """Block-diffusion attention forward for every (batch, head) or a subset.

    ``heads`` optionally lists (b, h) pairs to compute; the others are left
    as NaN.  Returns out (B, 2n, H, d) and lse (B, H, 2n), float64.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    _check_layout(q)
    B, L, H, d = q.shape
    kvh = _kv_head(q, k)
    mask = diffusion_mask(L // 2, block_size)
    out = np.full((B, L, H, d), np.nan)
    lse = np.full((B, H, L), np.nan)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        o, s = masked_attention_forward(q[b, :, h], k[b, :, kvh(h)], v[b, :, kvh(h)], mask)
        out[b, :, h] = o
        lse[b, h] = s
    return out, lse


def diffusion_backward(q, k, v, dout, block_size, heads=None):
    """Gradients dq (B, 2n, H, d) and dk, dv (B, 2n, H_kv, d), float64.

    With fewer key/value heads than query heads, the gradient of a key/value
    head is the sum over the query heads that read it.  ``heads`` lists
    (b, h) pairs of query heads to compute; dk, dv are then summed over the
    listed heads only (a full key/value head needs all of its query heads).
    """
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    _check_layout(q)
    B, L, H, d = q.shape
    kvh = _kv_head(q, k)
    mask = diffusion_mask(L // 2, block_size)
    dq = np.full((B, L, H, d), np.nan)
    dk, dv = (np.full(k.shape, np.nan) for _ in range(2))
    touched = set()
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        hk = kvh(h)
        g = masked_attention_backward(q[b, :, h], k[b, :, hk], v[b, :, hk], dout[b, :, h], mask)
        dq[b, :, h] = g[0]
        if (b, hk) not in touched:  # first query head of this key/value head
            touched.add((b, hk))
            dk[b, :, hk] = 0.0
            dv[b, :, hk] = 0.0
        dk[b, :, hk] += g[1]
        dv[b, :, hk] += g[2]
    return dq, dk, dv


# --------------------------------------------------------------------------
# Packed batches of different lengths ("Fast Diffusion Attention": varlen
# batches; the API is modeled on FlashAttention's varlen call).
# q, out: (rows, heads, headdim); k, v: (rows, kv_heads, headdim); lse:
# (heads, rows).  Sample b is rows [cu[b], cu[b+1]), [noisy | clean].
# --------------------------------------------------------------------------

def _varlen_samples(cu_seqlens, rows):
    cu = [int(x) for x in cu_seqlens]
    if not cu or cu[0] != 0 or cu[-1] != rows:
        raise ValueError("cu_seqlens must start at 0 and end at the packed rows")
    out = []
    for b in range(len(cu) - 1):
        a, e = cu[b], cu[b + 1]
        if e < a or (e - a) % 2:
            raise ValueError("every sample length must be even and non-negative")
        out.append((a, e))
    return out


def diffusion_varlen_forward(q, k, v, cu_seqlens, block_size):
    """Forward on a packed batch: each sample is attended to on its own.

    Returns out (rows, H, d) and lse (H, rows), float64.  Every sample uses
    the mask of its own half length, with the same block size.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    rows, H, d = q.shape
    kvh = _kv_head(q[None], k[None])
    out = np.zeros((rows, H, d))
    lse = np.zeros((H, rows))
    for a, e in _varlen_samples(cu_seqlens, rows):
        if e == a:
            continue
        mask = diffusion_mask((e - a) // 2, block_size)
        for h in range(H):
            o, s = masked_attention_forward(q[a:e, h], k[a:e, kvh(h)], v[a:e, kvh(h)], mask)
            out[a:e, h] = o
            lse[h, a:e] = s
    return out, lse


def diffusion_varlen_backward(q, k, v, dout, cu_seqlens, block_size):
    """Gradients of a packed batch: dq (rows, H, d), dk, dv (rows, H_kv, d)."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    rows, H, d = q.shape
    kvh = _kv_head(q[None], k[None])
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for a, e in _varlen_samples(cu_seqlens, rows):
        if e == a:
            continue
        mask = diffusion_mask((e - a) // 2, block_size)
        for h in range(H):
            hk = kvh(h)
            g = masked_attention_backward(q[a:e, h], k[a:e, hk], v[a:e, hk], dout[a:e, h], mask)
            dq[a:e, h] = g[0]
            dk[a:e, hk] += g[1]
            dv[a:e, hk] += g[2]
    return dq, dk, dv


def causal_forward(q, k, v, heads=None):
    """Causal attention on (Bc, L, H, d): the yardstick of "The right yardstick"."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, L, H, d = q.shape
    kvh = _kv_head(q, k)
    mask = causal_mask(L)
    out = np.full((B, L, H, d), np.nan)
    lse = np.full((B, H, L), np.nan)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        o, s = masked_attention_forward(q[b, :, h], k[b, :, kvh(h)], v[b, :, kvh(h)], mask)
        out[b, :, h] = o
        lse[b, h] = s
    return out, lse


def causal_backward(q, k, v, dout, heads=None):
    """Gradients of causal attention on (Bc, L, H, d), float64."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    B, L, H, d = q.shape
    kvh = _kv_head(q, k)
    mask = causal_mask(L)
    dq = np.full((B, L, H, d), np.nan)
    dk, dv = (np.full(k.shape, np.nan) for _ in range(2))
    touched = set()
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        hk = kvh(h)
        g = masked_attention_backward(q[b, :, h], k[b, :, hk], v[b, :, hk], dout[b, :, h], mask)
        dq[b, :, h] = g[0]
        if (b, hk) not in touched:  # first query head of this key/value head
            touched.add((b, hk))
            dk[b, :, hk] = 0.0
            dv[b, :, hk] = 0.0
        dk[b, :, hk] += g[1]
        dv[b, :, hk] += g[2]
    return dq, dk, dv


# --------------------------------------------------------------------------
# The online-softmax recurrence ("FlashAttention: Exact Attention Without
# Materialization", section 4.2), on one score row split into blocks.
# Not used by the functions above; it exists so that the printed worked
# example of section 4.3 can be checked step by step.
# --------------------------------------------------------------------------

def online_softmax_row(blocks, values=None):
    """Run the running-max / running-sum recurrence over score blocks.

    blocks: list of 1-D score arrays of one row.  values: optional list of
    (len(block), dv) arrays.  Returns (m, ell, z, history) where history
    records, after each block, the rescaled weights of every score seen so
    far (relative to the current maximum).  The final probabilities are
    history[-1] / ell and, with values, the output is z / ell.
    """
    m = -np.inf
    ell = 0.0
    z = None
    weights = np.zeros(0)
    history = []
    for t, s in enumerate(blocks):
        s = np.asarray(s, dtype=np.float64)
        m_new = max(m, float(s.max()))
        old_scale = math.exp(m - m_new) if np.isfinite(m) else 0.0
        p = np.exp(s - m_new)
        ell = old_scale * ell + p.sum()
        if values is not None:
            contrib = p @ np.asarray(values[t], dtype=np.float64)
            z = contrib if z is None else old_scale * z + contrib
        weights = np.concatenate([weights * old_scale, p])
        m = m_new
        history.append(weights.copy())
    return m, ell, z, history
