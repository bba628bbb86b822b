// Tile geometry of block-diffusion attention, shared by the host scheduler
// and the kernels.
//
// Source: "Fast Diffusion Attention", sections "Block diffusion in one
// picture" (the mask) and "Visit only the visible tiles" (the two halves are
// tiled separately; a query tile visits exactly the key tiles that intersect
// the mask, and in the backward pass a key tile visits exactly the query
// tiles that see it; only tiles cut by a block boundary are masked element by
// element).
//
// Every rule below makes the visible set of one query row a single interval
// of key positions inside one half, and the set of query rows that see one
// key a single interval of query positions; both interval ends are
// non-decreasing in the row (resp. key) index.  Unions over a tile and the
// "fully visible" test therefore only look at the first and last row.
#pragma once

#if defined(__CUDACC__)
#define DFA_HD __host__ __device__ __forceinline__
#else
#define DFA_HD inline
#endif

namespace dfa {

enum Half : int { HALF_NOISY = 0, HALF_CLEAN = 1 };
enum Mode : int { MODE_DIFFUSION = 0, MODE_CAUSAL = 1 };
// Which (query half, key half) pair a tile belongs to.
enum Rule : int { RULE_NONE = -1, RULE_NN = 0, RULE_NC = 1, RULE_CC = 2, RULE_CAUSAL = 3 };

struct Interval {
  int lo, hi;  // [lo, hi), empty when lo >= hi
};

struct Segment {
  int half;     // the other side's half (key half forward, query half backward)
  int rule;
  int t_begin;  // first tile index inside that half
  int t_end;    // one past the last tile
};

DFA_HD int imin(int a, int b) { return a < b ? a : b; }
DFA_HD int cdiv(int a, int b) { return (a + b - 1) / b; }

DFA_HD int rule_for(int mode, int q_half, int k_half) {
  if (mode == MODE_CAUSAL) return q_half == k_half ? RULE_CAUSAL : RULE_NONE;
  if (q_half == HALF_NOISY) return k_half == HALF_NOISY ? RULE_NN : RULE_NC;
  return k_half == HALF_CLEAN ? RULE_CC : RULE_NONE;
}

// Keys (positions inside their half) visible to query row r of its half.
// block_size must already be clamped to [1, n].
DFA_HD Interval key_interval(int rule, int r, int n, int bs) {
  if (r < 0 || r >= n) return {0, 0};
  const int b0 = (r / bs) * bs;
  const int b1 = imin(n, b0 + bs);
  switch (rule) {
    case RULE_NN: return {b0, b1};        // own noisy block, both directions
    case RULE_NC: return {0, b0};         // clean blocks strictly before
    case RULE_CC: return {0, b1};         // clean blocks up to its own
    case RULE_CAUSAL: return {0, r + 1};
    default: return {0, 0};
  }
}

// Query rows (inside their half) that see key j of its half.
DFA_HD Interval query_interval(int rule, int j, int n, int bs) {
  if (j < 0 || j >= n) return {0, 0};
  const int b0 = (j / bs) * bs;
  const int b1 = imin(n, b0 + bs);
  switch (rule) {
    case RULE_NN: return {b0, b1};
    case RULE_NC: return {b1, n};         // noisy rows of strictly later blocks
    case RULE_CC: return {b0, n};
    case RULE_CAUSAL: return {j, n};
    default: return {0, 0};
  }
}

// Every pair of the tile [qs, qs+bm) x [ks, ks+bn) is visible (no padding rows
// or keys, no block boundary cutting it).
DFA_HD bool tile_full(int rule, int n, int bs, int qs, int bm, int ks, int bn) {
  if (rule == RULE_NONE || qs + bm > n || ks + bn > n || qs < 0 || ks < 0) return false;
  const Interval first = key_interval(rule, qs, n, bs);
  const Interval last = key_interval(rule, qs + bm - 1, n, bs);
  return last.lo <= ks && ks + bn <= first.hi;
}

// Forward: key-tile segments of query tile qt of half q_half.  Clean keys
// first, then the noisy diagonal.  Returns the number of segments (0..2).
DFA_HD int fwd_segments(int mode, int n, int bs, int bm, int bn, int q_half, int qt,
                        Segment* seg) {
  const int qs = qt * bm;
  const int qe = imin(n, qs + bm);
  int cnt = 0;
  if (qs >= qe) return 0;
  for (int kh = HALF_CLEAN; kh >= HALF_NOISY; --kh) {
    const int rule = rule_for(mode, q_half, kh);
    if (rule == RULE_NONE) continue;
    const int lo = key_interval(rule, qs, n, bs).lo;
    const int hi = key_interval(rule, qe - 1, n, bs).hi;
    if (lo >= hi) continue;
    seg[cnt].half = kh;
    seg[cnt].rule = rule;
    seg[cnt].t_begin = lo / bn;
    seg[cnt].t_end = cdiv(hi, bn);
    ++cnt;
  }
  return cnt;
}

// Backward: query-tile segments that see key tile kt of half k_half.  Clean
// queries first, then noisy queries.
DFA_HD int bwd_segments(int mode, int n, int bs, int bm, int bn, int k_half, int kt,
                        Segment* seg) {
  const int ks = kt * bn;
  const int ke = imin(n, ks + bn);
  int cnt = 0;
  if (ks >= ke) return 0;
  for (int qh = HALF_CLEAN; qh >= HALF_NOISY; --qh) {
    const int rule = rule_for(mode, qh, k_half);
    if (rule == RULE_NONE) continue;
    const int lo = query_interval(rule, ks, n, bs).lo;
    const int hi = query_interval(rule, ke - 1, n, bs).hi;
    if (lo >= hi) continue;
    seg[cnt].half = qh;
    seg[cnt].rule = rule;
    seg[cnt].t_begin = lo / bm;
    seg[cnt].t_end = cdiv(hi, bm);
    ++cnt;
  }
  return cnt;
}

// Deterministic dQ: the key tiles that reach query tile qt of half q_half
// add into its dQ one after another, in the order the backward's work
// order takes them (clean key tiles before noisy ones, increasing index;
// the same order fwd_segments lists them).  Position of key tile kt of half
// k_half in that order (bm: query rows per tile, bn: keys per tile).
DFA_HD int dq_ordinal(int mode, int n, int bs, int bm, int bn, int q_half, int qt, int k_half,
                      int kt) {
  Segment s[2] = {{0, RULE_NONE, 0, 0}, {0, RULE_NONE, 0, 0}};
  const int cnt = fwd_segments(mode, n, bs, bm, bn, q_half, qt, s);
  if (cnt > 0 && s[0].half == k_half) return kt - s[0].t_begin;
  return (s[0].t_end - s[0].t_begin) + kt - s[1].t_begin;
}

// Offset of the log-sum-exp (and of D = rowsum(dO * O), laid out alike) of
// row r of half `half` of sample b, head h.  Diffusion mode: lse is
// (B, H, 2n).  Causal mode: sequence s of length n is half s % 2 of
// "sample" s / 2 (so that its rows start at (2b + half) * n as a half's
// do), and lse is (sequences, H, n).
DFA_HD long long lse_offset(int mode, int b, int h, int half, int r, int H, int n) {
  if (mode == MODE_CAUSAL)
    return ((2LL * b + half) * H + h) * static_cast<long long>(n) + r;
  return (static_cast<long long>(b) * H + h) * (2LL * n) + static_cast<long long>(half) * n + r;
}

// Halves of a batched launch: every sample has two (noisy, clean); in the
// causal mode B counts sequences, each one "half".
DFA_HD long long launch_halves(int mode, int B) {
  return mode == MODE_CAUSAL ? static_cast<long long>(B) : 2LL * B;
}

// Work items of a batched pass over `tiles` tiles per half.
DFA_HD long long pass_items(int mode, int B, int H, int tiles) {
  return launch_halves(mode, B) * H * tiles;
}

// Work decoding.  An item's "rank" orders the items of one (batch, head)
// longest first ("Fast Diffusion Attention", "Hopper": the scheduler hands
// out tiles longest first).  The (batch, head) pairs are cut into groups of
// `group` heads whose items are handed out together, so the group's tensors
// stay in L2 while its tiles run ("Ampere and Ada": L2-aware block order).
// The shortest ranks of every (batch, head) are held back and handed out
// last, rank by rank over all pairs: they reuse little from L2, and ending on
// short items lets the persistent kernels, which take items from a shared
// counter, finish together.
// Forward: one item per (batch, head, half, query tile): query tiles in
// decreasing index, both halves side by side; the last two tiles of each
// half form the tail.  Backward: key tiles; in the diffusion mode the clean
// key tiles (seen by clean and noisy queries) in increasing index, then the
// noisy key tiles (seen only by their own noisy blocks), which form the
// tail; in the causal mode key tiles in increasing index.  In the causal
// mode B counts sequences and the (sequence, head) pairs take the place of
// the (batch, head) pairs, one half each; the last two tiles of each
// sequence form the tail.
struct WorkItem {
  int b, h, half, tile;
};

// Split w into (rank inside its (batch, head), batch-head index) for groups
// of `group` heads with `per_bh` items each.
DFA_HD void group_split(int w, int BH, int group, int per_bh, int* rank, int* bh) {
  const int g = w / (group * per_bh);
  const int first = g * group;
  const int gsize = imin(group, BH - first);
  const int idx = w - first * per_bh;
  *rank = idx / gsize;
  *bh = first + idx % gsize;
}

// Ranks [0, ranks - tail) group by group, then the last `tail` ranks of all
// (batch, head) pairs.
DFA_HD void work_split(int w, int BH, int group, int ranks, int tail, int* rank, int* bh) {
  const int head = ranks - tail;
  const long long grouped = static_cast<long long>(BH) * head;
  if (w < grouped) {
    group_split(w, BH, group, head, rank, bh);
    return;
  }
  const long long t = w - grouped;
  *rank = head + static_cast<int>(t / BH);
  *bh = static_cast<int>(t % BH);
}

// Ranks per (batch, head) pair, or per (sequence, head) pair in the causal
// mode, and how many of them form the tail.
DFA_HD int pass_ranks(int mode, int tiles) { return mode == MODE_CAUSAL ? tiles : 2 * tiles; }

DFA_HD int fwd_tail_ranks(int mode, int tiles) {
  return mode == MODE_CAUSAL ? imin(tiles, 2) : imin(2 * tiles, 4);
}

DFA_HD int bwd_tail_ranks(int mode, int tiles) {
  return mode == MODE_CAUSAL ? imin(tiles, 2) : tiles;
}

// Causal mode: pair index bh = s * H + h of sequence s -> sample s / 2,
// half s % 2.
DFA_HD void causal_split(int bh, int H, WorkItem* it) {
  const int s = bh / H;
  it->b = s >> 1;
  it->half = s & 1;
  it->h = bh % H;
}

DFA_HD WorkItem fwd_work(int w, int mode, int B, int H, int tiles, int group) {
  int rank, bh;
  work_split(w, B * H, group, pass_ranks(mode, tiles), fwd_tail_ranks(mode, tiles), &rank, &bh);
  WorkItem it;
  if (mode == MODE_CAUSAL) {
    it.tile = tiles - 1 - rank;
    causal_split(bh, H, &it);
    return it;
  }
  it.tile = tiles - 1 - (rank >> 1);
  it.half = rank & 1;
  it.b = bh / H;
  it.h = bh % H;
  return it;
}

DFA_HD WorkItem bwd_work(int w, int mode, int B, int H, int tiles, int group) {
  int rank, bh;
  work_split(w, B * H, group, pass_ranks(mode, tiles), bwd_tail_ranks(mode, tiles), &rank, &bh);
  WorkItem it;
  if (mode == MODE_CAUSAL) {
    it.tile = rank;
    causal_split(bh, H, &it);
    return it;
  }
  if (rank < tiles) {
    it.half = HALF_CLEAN;
    it.tile = rank;
  } else {
    it.half = HALF_NOISY;
    it.tile = rank - tiles;
  }
  it.b = bh / H;
  it.h = bh % H;
  return it;
}

// Backward items of one key half only (the two passes of the noisy-diagonal
// specialisation, "Fast Diffusion Attention", "Hopper": a dedicated pass
// over the noisy diagonal, then the main pass over the clean key tiles).
// Clean key tiles longest first (increasing index) with the last two ranks
// of every pair as the tail; noisy key tiles, all equally short, rank by
// rank over all pairs.  `pass`: 1 clean key tiles, 2 noisy key tiles.
DFA_HD WorkItem bwd_work_pass(int w, int pass, int B, int H, int tiles, int group) {
  int rank, bh;
  const int tail = pass == 1 ? imin(tiles, 2) : tiles;
  work_split(w, B * H, group, tiles, tail, &rank, &bh);
  WorkItem it;
  it.half = pass == 1 ? HALF_CLEAN : HALF_NOISY;
  it.tile = rank;
  it.b = bh / H;
  it.h = bh % H;
  return it;
}

// The noisy-diagonal pass may store the noisy queries' dQ instead of adding
// it when every noisy query row is seen by the noisy keys of one key tile
// only: no block crosses a tile boundary (block size divides the tile) or
// the half is a single tile.
DFA_HD bool diag_pass_applies(int n, int bs, int tile) {
  return tile % bs == 0 || n <= tile;
}

// Heads per group: the group's working set (bytes_per_bh each) kept within
// about half of L2, and the heads spread evenly over the fewest groups that
// allows.  Even groups matter: a group's longest items start when the group
// does, so a small last group would leave its long items running alone at
// the end of the launch.
inline int l2_group(long long bytes_per_bh, long long l2_bytes, int BH) {
  long long g = (l2_bytes / 2) / (bytes_per_bh > 0 ? bytes_per_bh : 1);
  if (g < 1) g = 1;
  if (g > BH) g = BH;
  const long long groups = (BH + g - 1) / g;
  return static_cast<int>((BH + groups - 1) / groups);
}

}  // namespace dfa
