// Backward kernel of block-diffusion attention, headdim 64, on sm_103a.
//
// Recompute-based backward of "FlashAttention: Exact Attention Without
// Materialization", section 4.5: from q, k, v, dout, the forward's
// log-sum-exp and D = rowsum(dout * out), recompute the probabilities on
// chip and accumulate the gradients.  Key-tile major: a work item is one
// 128-key tile of one half of one (batch, head); its CTA keeps K and V in
// shared memory and the dK and dV accumulators in TMEM, and walks exactly
// the 128-query tiles that see it ("Fast Diffusion Attention", "Visit only
// the visible tiles"): a clean key tile is seen by the clean queries of its
// block onward and by the noisy queries of the later blocks; a noisy key
// tile only by the noisy queries of its own blocks.
//
// Per query tile g (counted over the CTA's whole run), b = g % 2:
//   S^T  = K Q^T                    -> TMEM S[b]
//   dP^T = V dO^T                   -> TMEM dP (one buffer)
//   P^T  = exp(scale S^T - LSE)  (0 on hidden pairs),
//   dS^T = scale * P^T (dP^T - D)   (the softmax scale of dQ and dK)
//        written back as bf16 into the columns of dP, dS^T also to shared
//   dV  += P^T dO,  dK += dS^T Q    (A operand read from TMEM)
//   dQ   = dS K                     -> TMEM S[b] (S is consumed by then),
//        then added to a float32 accumulator in device memory: each warp
//        stages its 32 query rows x 32 head dims in shared memory and adds
//        them with one bulk tensor reduce (deterministic mode: one query row
//        per thread with 16-byte atomics, in order).
// Persistent: one CTA per SM takes items from a work counter until none are
// left (the same order and counter as the other kernels); the barrier phases
// run on across items, the next item's first query tiles load while the
// current item ends, and K / V reload once the current item's products are
// done.  At the end of an item warpgroup 0 writes dV and warpgroup 1 dK; the
// next item's first dV / dK products wait until both have been read out.
// Warp roles (384 threads): two compute warpgroups that both work on every
// query tile, warpgroup b on its query columns [64 b, 64 b + 64) (thread t
// of a warpgroup owns key row t of the tile, TMEM lane t): with one dP
// buffer, dP^T of a tile waits for the dV / dK products of the tile before
// it, so tiles follow one another and the softmax-gradient work of a tile
// is split between the warpgroups rather than alternated; the dQ of a tile
// is added during the next tile's turn, each warpgroup adding 32 of its head
// dims.  Warp 8 loads (TMA for Q/dO, plain loads
// for LSE/D); warp 9 issues S^T, warp 10 dP^T, dV and dK, warp 11 dQ (on
// three schedulers, so that the busy compute warps sharing a scheduler with
// one of them do not starve the tensor pipe).  The load/MMA
// warpgroup drops to 72 registers and the compute warpgroups rise to 216
// (setmaxnreg; launched with 168: 256 * 48 == 128 * 96), so a 64-query
// slice of S^T and dP^T is read from TMEM in one batch.
#include <cuda_bf16.h>

#include <type_traits>

#include "geometry.cuh"
#include "params.cuh"
#include "sm100.cuh"

namespace dfa {

template <int D, int BMQ>
struct BwdCfg {
  static constexpr int BN = 128;  // keys per tile (MMA M)
  static constexpr int STAGES = 3;
  static constexpr int kChunks = D / 64;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kQBytes = BMQ * D * 2;
  static constexpr int kDSBytes = BN * BMQ * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVBytes;
  static constexpr int kOffQ = kOffV + kKVBytes;
  static constexpr int kOffDO = kOffQ + STAGES * kQBytes;
  static constexpr int kOffDS = kOffDO + STAGES * kQBytes;    // 2 buffers
  static constexpr int kOffLSE = kOffDS + 2 * kDSBytes;       // STAGES x BMQ floats
  static constexpr int kOffDEL = kOffLSE + STAGES * BMQ * 4;  // STAGES x BMQ floats
  static constexpr int kOffBar = kOffDEL + STAGES * BMQ * 4;
  enum {
    BAR_KV = 0,
    BAR_QFULL = 1,
    BAR_QEMPTY = BAR_QFULL + STAGES,
    BAR_SFULL = BAR_QEMPTY + STAGES,  // [2] per tile parity
    BAR_DPFULL = BAR_SFULL + 2,       // [2]
    BAR_PDS = BAR_DPFULL + 2,         // [2]
    BAR_MMA2 = BAR_PDS + 2,           // [2]
    BAR_DQFREE = BAR_MMA2 + 2,        // [2]
    BAR_ITEMDONE = BAR_DQFREE + 2,    // every product of an item done
    BAR_ACCFREE = BAR_ITEMDONE + 1,   // dK / dV of an item read out of TMEM
    BAR_ITEMFULL = BAR_ACCFREE + 1,   // [4] item index published
    BAR_ALL = BAR_ITEMFULL + 4,       // every MMA done (TMEM release)
    NUM_BARS = BAR_ALL + 1
  };
  static constexpr int kOffItem = kOffBar + NUM_BARS * 8;  // 4 decoded items (BwdItem)
  static constexpr int kOffTmemSlot = kOffItem + 4 * 128;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;
  static constexpr int kTmemS = 0;          // S[b] at b * BMQ; dQ of the tile after S is read
  static constexpr int kTmemDP = 2 * BMQ;   // dP, then P^T / dS^T
  static constexpr int kTmemDK = kTmemDP + BMQ;
  static constexpr int kTmemDV = kTmemDK + D;
  static constexpr int kTmemCols = 512;
  static constexpr int kThreads = 384;
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;    // S^T; owns TMEM
  static constexpr int kMma2Warp = 10;  // dP^T, dV, dK
  static constexpr int kMma3Warp = 11;  // dQ
  static_assert(kTmemDV + D <= kTmemCols, "TMEM budget");
  static_assert(D <= BMQ, "dQ must fit in an S buffer");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(BMQ == 128 && D == 64, "layout of this kernel: 128-query tiles, headdim 64");
};

// One work item: key tile of one key/value head and the query tiles that
// see it (at most two segments per query head, kept in scalars so that
// nothing is indexed dynamically).  With grouped key/value heads
// ("Fast Diffusion Attention": GQA-grouped backward) the item walks the same
// query tiles of each of the kv_group query heads h0, h0 + 1, ... that read
// its key/value head, so that dK and dV sum over the group in TMEM.  The
// producer decodes each item once and publishes the decoded form to the
// other roles through a ring in shared memory; v < 0 means no work is left.
struct BwdItem {
  int v;
  WorkItem wi;  // wi.h: the key/value head
  int n0, nth, ntiles;  // tiles of segment 0, per query head, in all
  int h0;               // first query head of the group
  int half0, rule0, tb0, half1, rule1, tb1;
  int n, bs, row0;  // half length, block size (clamped) and, varlen, first row
  int slot;         // varlen: the sample's slot (its tensor maps)
  // Tile t is local tile l of query head h0 + hh.  Without grouping
  // (GQA false: one query head per key/value head) l = t and hh = 0.
  template <bool GQA>
  __device__ __forceinline__ void split(int t, int& hh, int& l) const {
    hh = 0;
    l = t;
    if constexpr (GQA) {
      if (l >= nth) {
        hh = l / nth;
        l -= hh * nth;
      }
    }
  }
  __device__ __forceinline__ int ltile(int l) const { return l < n0 ? tb0 + l : tb1 + (l - n0); }
  __device__ __forceinline__ int lhalf(int l) const { return l < n0 ? half0 : half1; }
};

static_assert(sizeof(BwdItem) <= 128, "item ring slot");

template <int BMQ, int BN, bool GQA, bool VARLEN>
__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int v) {
  BwdItem it;
  it.v = v;
  if (v < 0) return it;
  if constexpr (VARLEN) {
    it.slot = varlen_slot(p.vl, p.vl_slots, v);
    const VarlenSlot sl = p.vl[it.slot];
    it.wi = bwd_work(v - sl.off, MODE_DIFFUSION, 1, p.Hk, cdiv(sl.n, BN), sl.group);
    it.wi.b = sl.b;
    it.n = sl.n;
    it.bs = imin(p.bs, sl.n);
    it.row0 = sl.row0;
  } else {
    it.wi = p.pass ? bwd_work_pass(v, p.pass, p.B, p.Hk, p.k_tiles, p.group)
                   : bwd_work(v, p.mode, p.B, p.Hk, p.k_tiles, p.group);
    it.n = p.n;
    it.bs = p.bs;
    it.row0 = 0;  // unused: batched rows come from wi.b
    it.slot = 0;
  }
  it.h0 = GQA ? it.wi.h * p.kv_group : it.wi.h;
  Segment seg[2] = {{0, RULE_NONE, 0, 0}, {0, RULE_NONE, 0, 0}};
  const int nseg = bwd_segments(p.mode, it.n, it.bs, BMQ, BN, it.wi.half, it.wi.tile, seg);
  it.n0 = nseg > 0 ? seg[0].t_end - seg[0].t_begin : 0;
  it.nth = it.n0 + (nseg > 1 ? seg[1].t_end - seg[1].t_begin : 0);
  it.ntiles = GQA ? it.nth * p.kv_group : it.nth;
  it.half0 = seg[0].half;
  it.rule0 = seg[0].rule;
  it.tb0 = seg[0].t_begin;
  it.half1 = seg[1].half;
  it.rule1 = seg[1].rule;
  it.tb1 = seg[1].t_begin;
  return it;
}

template <int D, int BMQ, bool GQA, bool VARLEN, bool DET>
__global__ void __launch_bounds__(384, 1) dfa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D, BMQ>;
  constexpr int BN = C::BN;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  // Slot s of the item ring; written by the producer before it arrives on
  // ITEMFULL[s] (release), read by the other roles after their wait (acquire).
  auto ring = [&](int s) { return reinterpret_cast<BwdItem*>(smem + C::kOffItem + 128 * s); };
  const AbortFlag ab{abort_flag, p.status};
  const size_t L = 2 * static_cast<size_t>(p.n);  // rows of one sample (two halves)
#define BAR(i) (sbase + C::kOffBar + 8 * (i))

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::BAR_KV), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(BAR(C::BAR_QFULL + s), 1);
      mbar_init(BAR(C::BAR_QEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(C::BAR_SFULL + b), 1);
      mbar_init(BAR(C::BAR_DPFULL + b), 1);
      mbar_init(BAR(C::BAR_PDS + b), 8);    // every compute warp
      mbar_init(BAR(C::BAR_MMA2 + b), 1);
      mbar_init(BAR(C::BAR_DQFREE + b), 8);
    }
    mbar_init(BAR(C::BAR_ITEMDONE), 2);  // warps 10 and 11
    mbar_init(BAR(C::BAR_ACCFREE), 8);
    for (int s = 0; s < 4; ++s) mbar_init(BAR(C::BAR_ITEMFULL + s), 1);
    mbar_init(BAR(C::BAR_ALL), 3);  // the three MMA-issuing warps
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(sbase + C::kOffTmemSlot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::kOffTmemSlot);
  // The prologue above touches only shared memory and TMEM.  Global memory
  // (inputs, outputs, the work counter) waits for the stream's previous
  // kernel; the next kernel may be launched now (its CTAs take each SM as
  // this kernel's CTA there exits).
  grid_dependency_wait();
  grid_launch_dependents();

  // Items are numbered k = 0, 1, ... in the order this CTA takes them, query
  // tiles g = 0, 1, ... over all of the CTA's items; every barrier phase
  // below is counted in one of the two.  Slot k % 4 of the item ring holds
  // item k; the loader writes it only after item k - 2 is done, which needs
  // both compute warpgroups to have read the dK / dV of item k - 3, so every
  // reader of the slot's previous item has taken its index.
  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
   if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ loads
    if (lane == 0 && !VARLEN) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    constexpr int kPerLane = BMQ / 32;
    bool ok = true;
    int g = 0, k = 0, q_issued = 0, kv_issued = 0;
    // Q, dO and the negated -LSE * log2(e), -D of the item's t-th query tile
    // into the stage of global tile gg.  Rows past the half: probability 0.
    auto load_q = [&](const BwdItem& it, int t, int gg) -> bool {
      int hh, l;
      it.template split<GQA>(t, hh, l);
      const int qt = it.ltile(l);
      const int half = it.lhalf(l);
      const int h = it.h0 + hh;  // query head
      // lse and delta: laid out alike, (batch, heads, 2n) (causal:
      // (sequences, heads, n)) or, varlen, (heads, rows)
      float lse_r[kPerLane], del_r[kPerLane];
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) {
        const int q = qt * BMQ + lane + 32 * e;
        const bool valid = q < it.n;
        const long long off =
            VARLEN ? static_cast<long long>(h) * p.rows + it.row0 + static_cast<long long>(half) * it.n + q
                   : lse_offset(p.mode, it.wi.b, h, half, q, p.H, p.n);
        lse_r[e] = valid ? p.lse[off] * -1.4426950408889634f : -INFINITY;
        // -D * scale: the softmax scale is folded into dS (see the compute)
        del_r[e] = valid ? -p.delta[off] * p.scale : 0.f;
      }
      const int st = gg % STAGES;
      const int round = gg / STAGES;
      if (round > 0) {
        int w = 0;
        if (lane == 0) w = mbar_wait(BAR(C::BAR_QEMPTY + st), (round - 1) & 1, ab) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, w, 0) == 0) return false;
      }
      float* lse_s = reinterpret_cast<float*>(smem + C::kOffLSE) + st * BMQ;
      float* del_s = reinterpret_cast<float*>(smem + C::kOffDEL) + st * BMQ;
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) {
        lse_s[lane + 32 * e] = lse_r[e];
        del_s[lane + 32 * e] = del_r[e];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(BAR(C::BAR_QFULL + st), 2 * C::kQBytes);
        // Varlen: the sample's own maps (rows past its halves read zero).
        const CUtensorMap* mq = VARLEN ? &p.vl_maps[it.slot].q : &p.tm_q;
        const CUtensorMap* mdo = VARLEN ? &p.vl_maps[it.slot].dout : &p.tm_do;
        const HalfRows qr = in_rows<VARLEN>(it.wi.b, half);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_5d(sbase + C::kOffQ + st * C::kQBytes + c * BMQ * 128, mq,
                      BAR(C::BAR_QFULL + st), 64 * c, h, qr.base + qt * BMQ, qr.c3, qr.c4);
          tma_load_5d(sbase + C::kOffDO + st * C::kQBytes + c * BMQ * 128, mdo,
                      BAR(C::BAR_QFULL + st), 64 * c, h, qr.base + qt * BMQ, qr.c3, qr.c4);
        }
      }
      __syncwarp();
      q_issued = gg + 1;
      return true;
    };
    while (ok) {
      int v = -1;
      if (lane == 0) v = sched_next(p.sched, p.items);
      v = __shfl_sync(0xffffffffu, v, 0);
      const BwdItem it = bwd_item<BMQ, BN, GQA, VARLEN>(p, v);
      if (lane == 0) {
        *ring(k & 3) = it;
        mbar_arrive(BAR(C::BAR_ITEMFULL + (k & 3)));
      }
      if (v < 0) break;
      if (VARLEN && lane == 0) {
        // this launch's maps of the item's sample, as memory holds them
        tensormap_acquire(&p.vl_maps[it.slot].q);
        tensormap_acquire(&p.vl_maps[it.slot].dout);
        tensormap_acquire(&p.vl_maps[it.slot].k);
        tensormap_acquire(&p.vl_maps[it.slot].v);
      }
      // The first query tiles only need stages the current item frees before
      // its last products, so they go ahead of the K / V load, which waits
      // for the whole item.
      const int pre = imin(it.ntiles, STAGES - 1);
      for (int t = 0; t < pre && ok; ++t) ok = load_q(it, t, g + t);
      if (!ok) break;
      if (k > 0) {
        int w = 0;
        if (lane == 0) w = mbar_wait(BAR(C::BAR_ITEMDONE), (k - 1) & 1, ab) ? 1 : 0;
        if (!(ok = __shfl_sync(0xffffffffu, w, 0) != 0)) break;
      }
      if (lane == 0) {
        const CUtensorMap* mk = VARLEN ? &p.vl_maps[it.slot].k : &p.tm_k;
        const CUtensorMap* mv = VARLEN ? &p.vl_maps[it.slot].v : &p.tm_v;
        const HalfRows kr = in_rows<VARLEN>(it.wi.b, it.wi.half);
        const int krow = kr.base + it.wi.tile * BN;
        mbar_arrive_expect_tx(BAR(C::BAR_KV), 2 * C::kKVBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_5d(sbase + C::kOffK + c * BN * 128, mk, BAR(C::BAR_KV), 64 * c, it.wi.h,
                      krow, kr.c3, kr.c4);
          tma_load_5d(sbase + C::kOffV + c * BN * 128, mv, BAR(C::BAR_KV), 64 * c, it.wi.h,
                      krow, kr.c3, kr.c4);
        }
      }
      __syncwarp();
      kv_issued = k + 1;
      for (int t = pre; t < it.ntiles && ok; ++t) ok = load_q(it, t, g + t);
      g += it.ntiles;
      ++k;
    }
    // Unwinding after a failed wait: let the copies in flight land.
    if (!ok && lane == 0) {
      if (kv_issued > 0) mbar_wait_limited(BAR(C::BAR_KV), (kv_issued - 1) & 1, 100000000ull);
      for (int t = (q_issued > STAGES ? q_issued - STAGES : 0); t < q_issued; ++t)
        mbar_wait_limited(BAR(C::BAR_QFULL + t % STAGES), (t / STAGES) & 1, 100000000ull);
    }
    __syncwarp();
   } else if (warp == C::kMmaWarp || warp == C::kMma2Warp || warp == C::kMma3Warp) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 9: S^T of every tile (it overwrites S[b], which held dQ of tile
    // g - 2: DQFREE).  Warp 10, in its own order: dV / dK of tile g - 1, then
    // dP^T of tile g, which overwrites the dP columns those products read
    // P^T / dS^T from.  Warp 11: dQ of every tile (MMA2: dQ in S[b]).
    if (lane == 0) {
      const bool s_warp = warp == C::kMmaWarp;
      const bool dq_warp = warp == C::kMma3Warp;
      constexpr uint32_t kIdS = idesc_bf16(BN, BMQ, false, false);  // K Q^T, V dO^T
      constexpr uint32_t kIdKV = idesc_bf16(BN, D, false, true);    // P^T dO, dS^T Q
      constexpr uint32_t kIdDQ = idesc_bf16(BMQ, D, true, true);    // dS K
      // Descriptors of the stage-0 / buffer-0 tiles; the others are reached by
      // adding byte offsets >> 4 to the start-address field.
      const uint64_t dK_kmaj = sdesc_sw128(sbase + C::kOffK, 16, 1024);
      const uint64_t dV_kmaj = sdesc_sw128(sbase + C::kOffV, 16, 1024);
      const uint64_t dK_mn = sdesc_sw128(sbase + C::kOffK, BN * 128, 1024);
      const uint64_t dQ_kmaj = sdesc_sw128(sbase + C::kOffQ, 16, 1024);
      const uint64_t dO_kmaj = sdesc_sw128(sbase + C::kOffDO, 16, 1024);
      const uint64_t dQ_mn = sdesc_sw128(sbase + C::kOffQ, BMQ * 128, 1024);
      const uint64_t dO_mn = sdesc_sw128(sbase + C::kOffDO, BMQ * 128, 1024);
      const uint64_t dDS_mn = sdesc_sw128(sbase + C::kOffDS, BN * 128, 1024);
      auto adv = [](uint64_t d, uint32_t bytes) { return d + static_cast<uint64_t>(bytes >> 4); };
      bool ok = true;
      int g = 0, k = 0;

      auto issue_dp = [&](int gg) {
        const uint32_t st_off = (gg % STAGES) * C::kQBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
          mma_ss(tmem + C::kTmemDP, adv(dV_kmaj, koff), adv(dO_kmaj, st_off + qoff), kIdS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(C::BAR_DPFULL + (gg & 1)));
      };
      // dV and dK of global tile gg, once its P^T / dS^T are in place;
      // `first`: the item's first tile, which starts the dK / dV sums.
      auto issue_second = [&](int gg, bool first) -> bool {
        const int b = gg & 1;
        const uint32_t st_off = (gg % STAGES) * C::kQBytes;
        if (!mbar_wait(BAR(C::BAR_PDS + b), (gg >> 1) & 1, ab)) return false;
        // dK / dV of the previous item must be read out before they restart.
        if (first && k >= 1 && !mbar_wait(BAR(C::BAR_ACCFREE), (k - 1) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t pds = tmem + C::kTmemDP;
#pragma unroll
        for (int kk = 0; kk < BMQ / 16; ++kk) {
          // P^T / dS^T of queries [16kk, 16kk+16): columns of 32-query chunk
          // kk/2, P^T in its first 16 columns, dS^T in its last 16.
          const uint32_t col = 32 * (kk >> 1) + 8 * (kk & 1);
          const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
          mma_ts(tmem + C::kTmemDV, pds + col, adv(dO_mn, st_off + kk * 16 * 128), kIdKV, acc);
          mma_ts(tmem + C::kTmemDK, pds + col + 16, adv(dQ_mn, st_off + kk * 16 * 128), kIdKV,
                 acc);
        }
        // dQ^T reads no Q / dO: the stage is free once dV / dK are done.
        mma_commit(BAR(C::BAR_QEMPTY + (gg % STAGES)));
        return true;
      };
      // dQ of global tile gg (warp 11): dS K into S[b], whose S^T the
      // warpgroup has read once P^T / dS^T are in place.
      auto issue_dq = [&](int gg) -> bool {
        const int b = gg & 1;
        if (!mbar_wait(BAR(C::BAR_PDS + b), (gg >> 1) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t ds_off = b * C::kDSBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ss(tmem + C::kTmemS + b * BMQ, adv(dDS_mn, ds_off + kk * 16 * 128),
                 adv(dK_mn, kk * 16 * 128), kIdDQ, kk > 0 ? 1u : 0u);
        mma_commit(BAR(C::BAR_MMA2 + b));
        return true;
      };

      while (ok) {
        if (!(ok = mbar_wait(BAR(C::BAR_ITEMFULL + (k & 3)), (k >> 2) & 1, ab))) break;
        const BwdItem it = *ring(k & 3);
        if (it.v < 0) break;
        // Every role waits for the item's K / V: ITEMDONE(k) then counts
        // commits made after ITEMDONE(k - 1) completed.
        if (!(ok = mbar_wait(BAR(C::BAR_KV), k & 1, ab))) break;
        if (dq_warp) {
          for (int i = 0; i < it.ntiles && ok; ++i) ok = issue_dq(g + i);
          if (!ok) break;
          // ITEMDONE counts one commit from each of warps 10 and 11.
          mma_commit(BAR(C::BAR_ITEMDONE));
          g += it.ntiles;
          ++k;
          continue;
        }
        for (int i = 0; i < it.ntiles && ok; ++i) {
          const int gg = g + i;
          const int b = gg & 1;
          const int st = gg % STAGES;
          if (!(ok = mbar_wait(BAR(C::BAR_QFULL + st), (gg / STAGES) & 1, ab))) break;
          if (s_warp) {
            // S[b] held dQ of tile gg-2: wait until it has been read out.
            if (gg >= 2 && !(ok = mbar_wait(BAR(C::BAR_DQFREE + b), ((gg - 2) >> 1) & 1, ab)))
              break;
            tc_fence_after();
            const uint32_t st_off = st * C::kQBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
              const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
              mma_ss(tmem + C::kTmemS + b * BMQ, adv(dK_kmaj, koff),
                     adv(dQ_kmaj, st_off + qoff), kIdS, kk > 0 ? 1u : 0u);
            }
            mma_commit(BAR(C::BAR_SFULL + b));
          } else {
            // One dP buffer: it still holds P^T / dS^T of tile gg-1 until the
            // dV / dK products of tile gg-1 have been issued (the previous
            // item's last tile was issued at that item's end).
            if (i >= 1 && !(ok = issue_second(gg - 1, i == 1))) break;
            tc_fence_after();
            issue_dp(gg);
          }
        }
        if (!ok) break;
        if (!s_warp) {
          if (it.ntiles > 0) {
            if (!(ok = issue_second(g + it.ntiles - 1, it.ntiles == 1))) break;
          } else if (k >= 1 && !(ok = mbar_wait(BAR(C::BAR_ACCFREE), (k - 1) & 1, ab))) {
            break;
          }
          // Every S^T of the item precedes its P^T / dS^T, so the last
          // products of warps 10 and 11 complete the item.
          mma_commit(BAR(C::BAR_ITEMDONE));
        }
        g += it.ntiles;
        ++k;
      }
      // Every MMA is complete when BAR_ALL fires (TMEM release).
      mma_commit(BAR(C::BAR_ALL));
    }
    __syncwarp();
   }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;");
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2;                // this warpgroup handles tiles g % 2 == wg
    const int row = (warp & 3) * 32 + lane;  // key row of the tile / TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    const uint64_t dscale2 = f2_pack(p.scale, p.scale);

    // dQ of global tile gg (TMEM S[gg % 2], lane = query `row` of the tile,
    // columns = head dims); warpgroup wg adds head dims [32 wg, 32 wg + 32)
    // of every query row.  The warp stages its 32 rows x 32 dims (float32,
    // 128-byte swizzled) in its own quarter of the tile's dS^T buffer --
    // the part it writes itself, free once the tile's dQ product, its only
    // reader, has completed -- and one lane adds the box into the
    // accumulator with a bulk tensor reduce; before the warp writes that
    // buffer again (two tiles later) it waits until the copy has read it.
    // Deterministic mode: 16-byte atomics in the counters' order.
    auto drain_dq = [&](const BwdItem& it, int gg, int t) -> bool {
      constexpr int DW = D / 2;  // head dims per warpgroup
      constexpr int kStageBytes = 32 * DW * 4;  // a warp's 32 rows x DW dims, float32
      static_assert(8 * kStageBytes <= C::kDSBytes, "staging inside one dS^T buffer");
      const int b = gg & 1;
      if (!mbar_wait_warp(BAR(C::BAR_MMA2 + b), (gg >> 1) & 1, ab)) return false;
      tc_fence_after();
      uint32_t dq[DW];
      tmem_ld32(t_lane + C::kTmemS + b * BMQ + DW * wg, dq);
      tmem_wait_ld();
      tmem_pin<DW>(dq);
      tc_fence_before();
      mbar_arrive_warp(BAR(C::BAR_DQFREE + b));
      int hh, l;
      it.template split<GQA>(t, hh, l);
      const int qs = it.ltile(l) * BMQ;
      const int q = qs + row;
      const int n = VARLEN ? it.n : p.n;
      const size_t first = VARLEN ? static_cast<size_t>(it.row0) : it.wi.b * L;
      unsigned* sem = nullptr;
      if constexpr (DET) {
        // The 4 warps of this warpgroup add the tile's dQ after the key
        // tiles the work order takes earlier: wait for them.
        const int ord = dq_ordinal(p.mode, n, VARLEN ? it.bs : p.bs, BMQ, BN, it.lhalf(l),
                                   it.ltile(l), it.wi.half, it.wi.tile);
        sem = p.dq_sem + static_cast<size_t>(it.h0 + hh) * p.sem_rows + first +
              static_cast<size_t>(it.lhalf(l)) * n + qs;
        // the 8 compute warps of every earlier contribution have signalled
        if (!sem_wait_warp(sem, static_cast<unsigned>(8 * ord), ab)) return false;
      }
      if constexpr (!DET) {
        const uint32_t stg = sbase + C::kOffDS + b * C::kDSBytes + warp * kStageBytes;
#pragma unroll
        for (int c = 0; c < DW / 4; ++c)
          st_shared_v4(stg + lane * 128 + ((c ^ (lane & 7)) << 4), dq[4 * c], dq[4 * c + 1],
                       dq[4 * c + 2], dq[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && qs + (warp & 3) * 32 < n) {
          // Varlen: through the sample's own map, so that rows of the box
          // past the half are skipped rather than added to the next sample.
          const CUtensorMap* mdq = VARLEN ? &p.vl_maps[it.slot].dq : &p.tm_dq;
          const HalfRows dr = in_rows<VARLEN>(it.wi.b, it.lhalf(l));
          if (p.pass == 2)  // noisy-diagonal pass: the rows' first contribution
            tma_store_5d(mdq, stg, DW * wg, it.h0 + hh, dr.base + qs + (warp & 3) * 32, dr.c3,
                         dr.c4);
          else
            tma_reduce_add_5d(mdq, stg, DW * wg, it.h0 + hh, dr.base + qs + (warp & 3) * 32,
                              dr.c3, dr.c4);
          bulk_commit_group();
        }
        return true;
      }
      if (q < n) {
        const size_t pos = static_cast<size_t>(it.lhalf(l)) * n + q;
        float* dst = p.dq_acc + ((first + pos) * p.H + it.h0 + hh) * D + DW * wg;
        if (p.pass == 2) {
          // noisy-diagonal pass: this item's contribution is the row's first
#pragma unroll
          for (int c = 0; c < DW; c += 4) st_global_v4(dst + c, dq[c], dq[c + 1], dq[c + 2], dq[c + 3]);
        } else {
#pragma unroll
          for (int c = 0; c < DW; c += 4)
            red_add_v4_f32(dst + c, __uint_as_float(dq[c]), __uint_as_float(dq[c + 1]),
                           __uint_as_float(dq[c + 2]), __uint_as_float(dq[c + 3]));
        }
      }
      if constexpr (DET) sem_signal_warp(sem);
      return true;
    };

    // P^T and dS^T of one 64-query slice h: S^T and dP^T in (one batch of
    // TMEM loads), bf16 P^T / dS^T back into the dP columns of each 32-query
    // chunk (P^T in its first 16 columns, dS^T in its last 16), dS^T also into
    // the swizzled shared tile.  Pairs of columns go through packed f32x2
    // arithmetic: x = s * sl2 - lse2, p = 2^x, ds = p * (dp - D) * scale; -LSE
    // and -D of four columns come in one shared load.  `masked`: a hidden
    // pair's p is cleared by AND with its column's mask bit (keep_lo /
    // keep_hi: columns 0-31 / 32-63 of the slice); a slice the mask does not
    // cut skips that.
    auto slice = [&](int h, uint32_t s_col, uint32_t ds_s, uint32_t nlse_s, uint32_t ndel_s,
                     uint32_t keep_lo, uint32_t keep_hi, auto masked) {
      uint32_t sr[64], dpr[64];
      tmem_ld32(s_col + 64 * h, sr);
      tmem_ld32(s_col + 64 * h + 32, sr + 32);
      tmem_ld32(t_lane + C::kTmemDP + 64 * h, dpr);
      tmem_ld32(t_lane + C::kTmemDP + 64 * h + 32, dpr + 32);
      tmem_wait_ld();
      tmem_pin<64>(sr);
      tmem_pin<64>(dpr);
      const uint64_t scale2 = f2_pack(sl2, sl2);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int cbase = 64 * h + 32 * cc;  // first query column of the chunk
        const uint32_t keep = cc ? keep_hi : keep_lo;
        uint32_t wp[16], wd[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          uint32_t la, lb, lc, ld, da, db, dc, dd4;
          ld_shared_v4(nlse_s + 4 * (cbase + 4 * e4), la, lb, lc, ld);
          ld_shared_v4(ndel_s + 4 * (cbase + 4 * e4), da, db, dc, dd4);
          const uint32_t nl[4] = {la, lb, lc, ld};
          const uint32_t nd[4] = {da, db, dc, dd4};
#pragma unroll
          for (int hp = 0; hp < 2; ++hp) {
            const int e = 2 * e4 + hp;       // pair inside the chunk
            const int cl = 32 * cc + 2 * e;  // column inside the slice
            const uint64_t x =
                f2_fma(f2_pack(__uint_as_float(sr[cl]), __uint_as_float(sr[cl + 1])), scale2,
                       f2_pack(__uint_as_float(nl[2 * hp]), __uint_as_float(nl[2 * hp + 1])));
            float x0, x1;
            f2_unpack(x, x0, x1);
            float p0 = ex2_approx(x0);
            float p1 = ex2_approx(x1);
            if constexpr (decltype(masked)::value) {
              p0 = __uint_as_float(__float_as_uint(p0) & bit_spread(keep, 2 * e));
              p1 = __uint_as_float(__float_as_uint(p1) & bit_spread(keep, 2 * e + 1));
            }
            const uint64_t pp = f2_pack(p0, p1);
            // (dP - D) * scale: dS carries the softmax scale, so dQ and dK
            // need no scaling afterwards
            const uint64_t dd =
                f2_fma(f2_pack(__uint_as_float(dpr[cl]), __uint_as_float(dpr[cl + 1])), dscale2,
                       f2_pack(__uint_as_float(nd[2 * hp]), __uint_as_float(nd[2 * hp + 1])));
            float d0, d1;
            f2_unpack(f2_mul(pp, dd), d0, d1);
            wp[e] = pack_bf16x2(p0, p1);
            wd[e] = pack_bf16x2(d0, d1);
          }
        }
        const int chunk = 2 * h + cc;
        tmem_st16(t_lane + C::kTmemDP + 32 * chunk, wp);
        tmem_st16(t_lane + C::kTmemDP + 32 * chunk + 16, wd);
        const int a = chunk >> 1;  // 64-column swizzle atom
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const int u = (chunk & 1) * 4 + u4;  // 16-byte unit inside the row
          const uint32_t off = a * (BN * 128) + row * 128 + ((u ^ (row & 7)) << 4);
          st_shared_v4(ds_s + off, wd[4 * u4], wd[4 * u4 + 1], wd[4 * u4 + 2], wd[4 * u4 + 3]);
        }
      }
    };

    bool ok = true;
    int g = 0, k = 0;
    while (ok) {
      if (!(ok = mbar_wait_warp(BAR(C::BAR_ITEMFULL + (k & 3)), (k >> 2) & 1, ab))) break;
      const BwdItem it = *ring(k & 3);
      if (it.v < 0) break;
      if constexpr (VARLEN && !DET) {
        // this launch's dq map of the item's sample, as memory holds it
        if (lane == 0) tensormap_acquire(&p.vl_maps[it.slot].dq);
      }
      const int ks = it.wi.tile * BN;
      const int j = ks + row;  // key inside its half
      // Query rows that see key j, per segment of the item: computed once,
      // so a tile needs no division and no per-tile visibility test.
      const int n = VARLEN ? it.n : p.n;
      const int bs = VARLEN ? it.bs : p.bs;
      const Interval iv0 = query_interval(it.rule0, j, n, bs);
      const Interval iv1 = query_interval(it.rule1, j, n, bs);
      // Both warpgroups work on every tile, warpgroup wg on query columns
      // [64 wg, 64 wg + 64); a tile's dQ is added during the next tile's
      // turn, so its product has completed by then.
      for (int i = 0; i < it.ntiles && ok; ++i) {
        const int gg = g + i;
        const int st = gg % STAGES;
        const int b = gg & 1;
        if (!(ok = mbar_wait_warp(BAR(C::BAR_SFULL + b), (gg >> 1) & 1, ab))) break;
        if (!(ok = mbar_wait_warp(BAR(C::BAR_DPFULL + b), (gg >> 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t nlse_s = sbase + C::kOffLSE + 4 * st * BMQ;
        const uint32_t ndel_s = sbase + C::kOffDEL + 4 * st * BMQ;
        int hh, l;
        it.template split<GQA>(i, hh, l);
        const int qs = it.ltile(l) * BMQ;
        // Columns (queries) that see key j, as a 128-bit mask in 4 words.
        const Interval iv = l < it.n0 ? iv0 : iv1;
        uint32_t keep[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int lo0 = iv.lo - qs - 32 * w, hi0 = iv.hi - qs - 32 * w;
          const int lo = lo0 < 0 ? 0 : (lo0 > 32 ? 32 : lo0);
          const int hi = hi0 < lo ? lo : (hi0 > 32 ? 32 : hi0);
          const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
          const uint32_t below_lo = lo >= 32 ? 0xffffffffu : ((1u << lo) - 1u);
          keep[w] = below_hi & ~below_lo;
        }
        const uint32_t s_col = t_lane + C::kTmemS + b * BMQ;
        const uint32_t ds_s = sbase + C::kOffDS + b * C::kDSBytes;
        if constexpr (!DET) {
          // this warp's quarter of buffer b staged the dQ of tile gg - 2
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
        const uint32_t klo = keep[2 * wg], khi = keep[2 * wg + 1];
        if (__all_sync(0xffffffffu, (klo & khi) == 0xffffffffu))
          slice(wg, s_col, ds_s, nlse_s, ndel_s, klo, khi, std::false_type{});
        else
          slice(wg, s_col, ds_s, nlse_s, ndel_s, klo, khi, std::true_type{});
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive_warp(BAR(C::BAR_PDS + b));
        if (i >= 1 && !(ok = drain_dq(it, gg - 1, i - 1))) break;
      }
      if (!ok) break;
      if (it.ntiles > 0 && !(ok = drain_dq(it, g + it.ntiles - 1, it.ntiles - 1))) break;

      // -------------------------------------------------------- item epilogue
      // Warpgroup 0 writes dV, warpgroup 1 writes dK, once the item's MMAs
      // are done; TMEM is released as soon as both have read their part.
      if (!(ok = mbar_wait_warp(BAR(C::BAR_ITEMDONE), k & 1, ab))) break;
      tc_fence_after();
      const uint32_t col = wg == 0 ? C::kTmemDV : C::kTmemDK;
      uint32_t o[D];
      if (it.ntiles > 0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(t_lane + col + 32 * c, o + 32 * c);
        tmem_wait_ld();
        tmem_pin<D>(o);
      } else {
#pragma unroll
        for (int e = 0; e < D; ++e) o[e] = 0u;
      }
      tc_fence_before();
      mbar_arrive_warp(BAR(C::BAR_ACCFREE));
      if (j < n) {
        const size_t pos = static_cast<size_t>(it.wi.half) * n + j;
        const size_t first = VARLEN ? static_cast<size_t>(it.row0) : it.wi.b * L;
        const size_t off = ((first + pos) * p.Hk + it.wi.h) * D;
        __nv_bfloat16* dst = (wg == 0 ? p.dv : p.dk) + off;
        const float mul = 1.f;  // dK: the scale is already in dS
#pragma unroll
        for (int g8 = 0; g8 < D / 8; ++g8) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w4[e] = pack_bf16x2(__uint_as_float(o[g8 * 8 + 2 * e]) * mul,
                                __uint_as_float(o[g8 * 8 + 2 * e + 1]) * mul);
          st_global_v4(dst + 8 * g8, w4[0], w4[1], w4[2], w4[3]);
        }
      }
      g += it.ntiles;
      ++k;
    }
    // The last bulk reduce-adds must be complete before the CTA exits.
    if constexpr (!DET) {
      if (lane == 0) bulk_wait_all();
    }
  }
#undef BAR

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    // Every MMA must be complete before the TMEM is released.
    if (lane == 0) mbar_wait_limited(sbase + C::kOffBar + 8 * C::BAR_ALL, 0, 1000000000ull);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0) sched_finish(p.sched);
}

template <int D, int BMQ, bool GQA, bool VARLEN, bool DET = false>
static cudaError_t launch_bwd_impl(const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D, BMQ>;
  auto kern = dfa_bwd_kernel<D, BMQ, GQA, VARLEN, DET>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // the noisy-diagonal passes take the key tiles of one half only
  const long long items = VARLEN ? p.units
                          : p.pass ? static_cast<long long>(p.B) * p.Hk * p.k_tiles
                                   : pass_items(p.mode, p.B, p.Hk, p.k_tiles);
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  BwdParams q = p;
  q.items = static_cast<int>(items);
  const long long grid = items < sms ? items : sms;
  return launch_chained(kern, dim3(static_cast<unsigned>(grid)), dim3(C::kThreads), C::kSmemBytes,
                        stream, q);
}

cudaError_t launch_backward(const BwdParams& p, int headdim, cudaStream_t stream) {
  switch (headdim) {
    // grouped key/value heads have their own instantiation
    case 64:
      if (p.dq_sem)  // deterministic mode
        return p.vl ? launch_bwd_impl<64, 128, true, true, true>(p, stream)
                    : launch_bwd_impl<64, 128, true, false, true>(p, stream);
      if (p.vl) return launch_bwd_impl<64, 128, true, true>(p, stream);
      return p.kv_group > 1 ? launch_bwd_impl<64, 128, true, false>(p, stream)
                            : launch_bwd_impl<64, 128, false, false>(p, stream);
    case 128: return launch_backward_d128(p, stream);
    case 256: return launch_backward_d256(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfa
