// Backward kernel of block-diffusion attention, headdim 64, 128 and 256, on
// sm_103a.
//
// Recompute-based backward of "FlashAttention: Exact Attention Without
// Materialization", section 4.5.  Key-tile major: a work item is one 128-key
// tile of one half of one (batch, head); its CTA keeps K and V in shared
// memory and the dK and dV accumulators in TMEM, and walks exactly the
// 64-query tiles that see it ("Fast Diffusion Attention", "Visit only the
// visible tiles").
//
// Per query tile (tensor cores, accumulators in TMEM):
//   S^T  = K Q^T     -> TMEM S        dP^T = V dO^T   -> TMEM dP
//   P^T  = exp(scale S^T - LSE) (0 on hidden pairs),
//   dS^T = scale * P^T (dP^T - D)  (the softmax scale of dQ and dK, taken
//        here once per element instead of on every dQ and dK element)
//        bf16 P^T -> TMEM (two buffers), dS^T -> a shared-memory tile
//        (two; headdim 256: one, and dS^T also -> TMEM beside P^T)
//   dV  += P^T dO  (A operand read from TMEM),
//   dK  += dS^T Q  (A operand read from the shared dS^T tile; headdim 64
//        and 256: from TMEM)
//   dQ^T = K^T dS^T  -> TMEM DQ, then added to a float32 accumulator in
//        device memory (each warp covers 32 consecutive head dims of a
//        query; headdim 64: 16)
// TMEM (512 columns): S 64 | dP 64 | P 2 x 32 (headdim 256: P / dS 64) |
// DQ 64 | dK 128 | dV 128; headdim 64: S 64 | dP 64 | P / dS 2 x 64 |
// DQ (an M = 64 product: lanes 0-15 of each lane quarter) 64 | dK 64 |
// dV 64.  With two P^T buffers and two dS^T tiles a tile's P^T / dS^T are
// written while the tile before is still in its products: the compute
// warpgroups wait only for the products of the tile before that.
// With headdim 256 the dK and dV accumulators of all head dims would need
// every TMEM column, so an item covers one 128-wide half of the head
// dimension of its key tile: it recomputes S^T and dP^T in full (their
// contraction runs over all 256 dims) and accumulates dK, dV and dQ for its
// half only; the two halves of a key tile are neighbouring items.  K and V
// (128 KB) then leave room for a single Q / dO stage.
//
// Persistent: one CTA per SM takes items from a work counter until none are
// left, so the load of the next item's K and V and of its first query tiles
// overlaps the end of the current item, and short items fill the SMs that
// finish early.  The compute warpgroups all work on every query tile, each
// on its own query columns; a tile's dQ is read out of TMEM during the next
// tile's turn, once that tile's P^T / dS^T are handed over, so no warpgroup
// waits for the products of the tile it has just finished.  S and dP are
// released as soon as they are in registers, so the scores of the next tile
// are computed while the warpgroups work.  At the end of an item the first
// half of the warpgroups writes dV and the second half dK; the next item's
// first dV / dK products wait until all have been read out of TMEM.
// With headdim 64 and 128 each warp adds its part of dQ into the float32
// accumulator with a bulk tensor reduce from a shared staging tile; with 256
// (no shared memory left) each thread adds its own with atomics.
// Warps: 4 per compute warpgroup, then one TMA producer and three MMA
// issuers (S^T; dV / dK then dQ^T; dP^T), on three schedulers: a single
// issuing warp is slowed by the busy compute warps sharing its scheduler,
// and S^T and dP^T, which every tile waits for, are issued in parallel.  The control warps drop registers to the compute
// warpgroups (setmaxnreg) within the pool the launch provides.
#include <cuda_bf16.h>

#include <type_traits>

#include "geometry.cuh"
#include "params.cuh"
#include "sm100.cuh"

namespace dfa {

template <int D_, int STAGES_, int NWG_, int KVBUF_>
struct Bwd2Cfg {
  static constexpr int D = D_;
  // K / V buffers: with two, the next item's K and V load while the current
  // item runs, and its first products need not wait for the current item's
  // last ones.
  static constexpr int KVBUF = KVBUF_;
  static constexpr int NWG = NWG_;             // compute warpgroups
  static constexpr int kComputeWarps = 4 * NWG;
  static constexpr int kWarpLoad = kComputeWarps;      // TMA producer
  static constexpr int kWarpS = kComputeWarps + 1;     // S^T issuer, owns TMEM
  static constexpr int kWarpKV = kComputeWarps + 2;    // dV / dK and dQ^T issuer
  static constexpr int kWarpDP = kComputeWarps + 3;    // dP^T issuer
  static constexpr int kThreads = 32 * (kComputeWarps + 4);
  // setmaxnreg split: the launch gives every thread kRegLaunch registers;
  // the 4 control warps drop to kRegCtl, the compute warps rise to
  // kRegCompute, within the launch's pool.
  static constexpr int kRegLaunch = NWG == 2 ? 168 : 96;
  static constexpr int kRegCtl = NWG == 2 ? 136 : 64;
  static constexpr int kRegCompute = NWG == 2 ? 184 : 104;
  static_assert(kRegCtl * 128 + kRegCompute * 128 * NWG <= kRegLaunch * kThreads,
                "register split exceeds the launch pool");
  static constexpr int DH = D < 128 ? D : 128;  // head dims accumulated per item
  static constexpr int NDH = D / DH;   // items per key tile
  static constexpr int BN = 128;  // keys per tile (MMA M)
  static constexpr int BMQ = 64;  // queries per tile
  static constexpr int HC = BMQ / NWG;  // query columns per compute warpgroup
  static constexpr int STAGES = STAGES_;
  static constexpr int kChunks = D / 64;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kQBytes = BMQ * D * 2;
  static constexpr int kDSBytes = BN * BMQ * 2;
  // Headdim 256: Q and dO go through two rings of 64-dim chunks instead of
  // whole-tile stages.  An item needs the chunks of the other head-dim half
  // only for S^T and dP^T, those of its own half also for dV and dK; so the
  // other half's chunks (OH ring, 2 slots) are released as soon as S^T and
  // dP^T complete and the own half's (DH ring, 3 slots) after dV and dK,
  // and the next tile's chunks load while the current tile is still at work
  // -- K and V (128 KB) leave room for five chunk slots, not two stages.
  static constexpr bool kChunkRing = D == 256;
  static constexpr int kOhSlots = 2;
  static constexpr int kDhSlots = 3;
  static constexpr int kSlotBytes = 2 * BMQ * 128;  // a Q chunk, then a dO chunk
  static constexpr int kQBars = kChunkRing ? kOhSlots + kDhSlots : STAGES;
  static constexpr int kLseBufs = kChunkRing ? 2 : STAGES;  // -LSE, -D buffers
  static constexpr int kOffK = 0;                          // [KVBUF]
  static constexpr int kOffV = kOffK + KVBUF * kKVBytes;   // [KVBUF]
  static constexpr int kOffQ = kOffV + KVBUF * kKVBytes;   // ring: the chunk slots
  static constexpr int kOffDO = kOffQ + STAGES * kQBytes;  // (no ring)
  // dS^T tiles in shared memory (the A operand of dK += dS^T Q and the B
  // operand of dQ^T = K^T dS^T): two with headdim 128, so that a tile's dS^T
  // is written while the tile before is still in its products; one with
  // 256 (no room for a second).
  static constexpr int kDSBufs = kChunkRing ? 1 : 2;
  static constexpr int kOffDS =
      kChunkRing ? kOffQ + (kOhSlots + kDhSlots) * kSlotBytes : kOffDO + STAGES * kQBytes;
  // dQ staging, one tile per compute warp: float32 [HC queries][32 head
  // dims] (headdim 64: 16), the source of that warp's bulk reduce-add into
  // the accumulator (with 256 the shared memory is full and dQ goes out
  // with per-thread atomics).
  // Headdim 64: dQ^T (M = 64 head dims) lies in lanes [32 q, 32 q + 16) of
  // each lane quarter q, so each warp stages its 16 head dims x HC queries.
  static constexpr bool kD64 = D == 64;
  static constexpr bool kTmaDQ = (D == 128 && KVBUF == 1) || kD64;
  static constexpr int kDQSBytes = HC * (kD64 ? 16 : 32) * 4;
  static constexpr int kOffDQS = kOffDS + kDSBufs * kDSBytes;
  static constexpr int kOffLSE = kOffDQS + (kTmaDQ ? kComputeWarps * kDQSBytes : 0);  // kLseBufs x BMQ floats
  static constexpr int kOffDEL = kOffLSE + kLseBufs * BMQ * 4;  // kLseBufs x BMQ floats
  static constexpr int kOffBar = kOffDEL + kLseBufs * BMQ * 4;
  enum {
    BAR_KVFULL = 0,  // [KVBUF] K and V of an item loaded
    BAR_QFULL = KVBUF,  // [kQBars] per stage, or per ring slot (OH slots first)
    BAR_QEMPTY = BAR_QFULL + kQBars,
    BAR_SDPFULL = BAR_QEMPTY + kQBars,  // S^T and dP^T of a tile computed
    BAR_SDPFREE = BAR_SDPFULL + 1,      // S^T / dP^T read into registers
    BAR_PDSFULL = BAR_SDPFREE + 1,      // [2] per tile parity: P^T / dS^T of a tile in place
    BAR_MMA2 = BAR_PDSFULL + 2,         // [kDSBufs] per dS^T tile: dV, dK, dQ of a tile done
    BAR_DQFREE = BAR_MMA2 + 2,          // dQ of a tile read out of TMEM
    BAR_ITEMDONE = BAR_DQFREE + 1,      // [KVBUF] every MMA of an item done
    BAR_ACCFREE = BAR_ITEMDONE + KVBUF, // dK / dV of an item read out of TMEM
    BAR_ITEMFULL = BAR_ACCFREE + 1,     // [4] item index published
    BAR_ALL = BAR_ITEMFULL + 4,         // every MMA of the CTA done
    NUM_BARS = BAR_ALL + 1
  };
  static constexpr int kOffItem = kOffBar + NUM_BARS * 8;  // 4 decoded items (Bwd2Item)
  static constexpr int kOffTmemSlot = kOffItem + 4 * 128;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  // The dynamic shared memory starts 1024-byte aligned (the kernel checks
  // this, for the 128-byte swizzle of the TMA boxes and MMA operands).
  static constexpr int kSmemBytes = kOffAbort + 4;
  static constexpr int kTmemS = 0;
  static constexpr int kTmemDP = 64;
  // Headdim 128: P^T of tile g at kTmemP + 32 (g % 2) (64 queries, bf16
  // pairs).  Headdim 256: one buffer of P^T and dS^T together, 32-column
  // chunk c holding P^T of queries [32 c, 32 c + 32) in its first 16 columns
  // and dS^T in the last 16 (both A operands read from TMEM: with a single
  // dS^T tile, reading it from shared memory buys no overlap and costs the
  // ring's shared-memory bandwidth).  Headdim 64: two such buffers, tile g
  // in kTmemP + 64 (g % 2) (dK += dS^T Q with N = 64 head dims would need
  // more shared-memory bandwidth than there is with both operands there);
  // dQ^T (M = 64) then dK and dV of 64 columns each.
  static constexpr int kTmemP = 128;
  static constexpr int kTmemDQ = kD64 ? 256 : 192;
  static constexpr int kTmemDK = kD64 ? 320 : 256;
  static constexpr int kTmemDV = 384;
  // Headdim 64: K and V of the item as the A operands of S^T and dP^T (32
  // columns each): an N = 64 product with both operands in shared memory
  // reads them faster than the port delivers.
  static constexpr int kTmemKA = 448;
  static constexpr int kTmemVA = 480;
  static constexpr int kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// One work item: key tile of one key/value head, head-dim half and the
// query tiles that see it (at most two segments per query head, kept in
// scalars so that nothing is indexed dynamically).  With grouped key/value
// heads ("Fast Diffusion Attention": GQA-grouped backward) the item walks
// the same query tiles of each of the kv_group query heads that read its
// key/value head, h0, h0 + 1, ..., so that dK and dV sum over the group in
// TMEM.  The producer decodes each item once and publishes the decoded form
// to the other roles through a ring in shared memory; v < 0 means no work is
// left.
struct Bwd2Item {
  int v;
  WorkItem wi;  // wi.h: the key/value head
  int dh;
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

static_assert(sizeof(Bwd2Item) <= 128, "item ring slot");

template <int NDH, int BMQ, int BN, bool GQA, bool VARLEN>
__device__ __forceinline__ Bwd2Item bwd2_item(const BwdParams& p, int v) {
  Bwd2Item it;
  it.v = v;
  if (v < 0) return it;
  it.dh = v % NDH;
  if constexpr (VARLEN) {
    const int u = v / NDH;
    it.slot = varlen_slot(p.vl, p.vl_slots, u);
    const VarlenSlot sl = p.vl[it.slot];
    it.wi = bwd_work(u - sl.off, MODE_DIFFUSION, 1, p.Hk, cdiv(sl.n, BN), sl.group);
    it.wi.b = sl.b;
    it.n = sl.n;
    it.bs = imin(p.bs, sl.n);
    it.row0 = sl.row0;
  } else {
    it.wi = p.pass ? bwd_work_pass(v / NDH, p.pass, p.B, p.Hk, p.k_tiles, p.group)
                   : bwd_work(v / NDH, p.mode, p.B, p.Hk, p.k_tiles, p.group);
    it.n = p.n;
    it.bs = p.bs;
    it.row0 = 0;  // unused: batched rows come from wi.b
    it.slot = 0;
  }
  it.h0 = GQA ? it.wi.h * p.kv_group : it.wi.h;
  Segment seg[2] = {};
  const int nseg = bwd_segments(p.mode, it.n, it.bs, BMQ, BN, it.wi.half, it.wi.tile, seg);
  it.n0 = nseg > 0 ? seg[0].t_end - seg[0].t_begin : 0;
  it.nth = it.n0 + (nseg > 1 ? seg[1].t_end - seg[1].t_begin : 0);
  it.ntiles = GQA ? it.nth * p.kv_group : it.nth;
  it.half0 = seg[0].half;
  it.rule0 = seg[0].rule;
  it.tb0 = seg[0].t_begin;
  it.half1 = nseg > 1 ? seg[1].half : 0;
  it.rule1 = nseg > 1 ? seg[1].rule : 0;
  it.tb1 = nseg > 1 ? seg[1].t_begin : 0;
  return it;
}

// One 128-row x 256-bit block of a 128-byte-swizzled shared tile (the A
// operand of one K = 16 step) into TMEM: lane r receives row r's eight
// 32-bit words, the layout of an A operand read from TMEM.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <int D_, int STAGES_, int NWG_, int KVBUF_, bool GQA, bool VARLEN, bool DET>
__global__ void __launch_bounds__(Bwd2Cfg<D_, STAGES_, NWG_, KVBUF_>::kThreads, 1)
    dfa_bwd2_kernel(const __grid_constant__ BwdParams p) {
  using C = Bwd2Cfg<D_, STAGES_, NWG_, KVBUF_>;
  constexpr int DH = C::DH;
  constexpr int D = C::D;
  constexpr int BN = C::BN;
  constexpr int BMQ = C::BMQ;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem_raw) & 1023u) {
    // not the layout this kernel was built for: report, take no work
    if (threadIdx.x == 0) {
      atomicOr(p.status, kStatusIndex);
      sched_finish(p.sched);
    }
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  // Slot s of the item ring; written by the producer before it arrives on
  // ITEMFULL[s] (release), read by the other roles after their wait (acquire).
  auto ring = [&](int s) { return reinterpret_cast<Bwd2Item*>(smem + C::kOffItem + 128 * s); };
  const AbortFlag ab{abort_flag, p.status};
#define BAR(i) (sbase + C::kOffBar + 8 * (i))

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::KVBUF; ++s) {
      mbar_init(BAR(C::BAR_KVFULL + s), 1);
      mbar_init(BAR(C::BAR_ITEMDONE + s), 1);  // the warp issuing dV / dK and dQ
    }
    for (int s = 0; s < C::kQBars; ++s) {
      mbar_init(BAR(C::BAR_QFULL + s), 1);
      // ring: an OH slot is released by the S^T and the dP^T warps, a DH
      // slot (like a stage) by the warp issuing dV / dK
      mbar_init(BAR(C::BAR_QEMPTY + s), C::kChunkRing && s < C::kOhSlots ? 2 : 1);
    }
    mbar_init(BAR(C::BAR_SDPFULL), 2);  // the S^T and the dP^T warps
    mbar_init(BAR(C::BAR_SDPFREE), C::kComputeWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(C::BAR_PDSFULL + b), C::kComputeWarps);
      mbar_init(BAR(C::BAR_MMA2 + b), 1);  // (the second unused with one dS^T tile)
    }
    mbar_init(BAR(C::BAR_DQFREE), C::kComputeWarps);
    mbar_init(BAR(C::BAR_ACCFREE), C::kComputeWarps);
    for (int s = 0; s < 4; ++s) mbar_init(BAR(C::BAR_ITEMFULL + s), 1);
    mbar_init(BAR(C::BAR_ALL), 3);  // one commit per issuing warp
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kWarpS) {
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
  // below is counted in one of the two.  The item ring holds the index of
  // item k in slot k % 4: the loader writes slot k only after item
  // k - 1 - KVBUF is done, and an item is done only after every compute
  // warpgroup has read the dK / dV of the item before it, so a slot is never
  // overwritten before every reader has taken its index.
  if (warp >= C::kComputeWarps) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegCtl));
   if (warp == C::kWarpLoad) {
    // ------------------------------------------------------------ loads
    if (lane == 0 && !VARLEN) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    bool ok = true;
    int g = 0, k = 0, q_issued = 0, kv_issued = 0;
    // -LSE * log2(e) and -D of the item's t-th query tile, read into
    // registers (stage_rows) and stored into buffer `buf` (store_rows).
    float lse_r[2], del_r[2];
    auto stage_rows = [&](const Bwd2Item& it, int t) {
      int hh, l;
      it.template split<GQA>(t, hh, l);
      const int qt = it.ltile(l);
      const int half = it.lhalf(l);
      const int h = it.h0 + hh;  // query head
      // lse and delta: laid out alike, (batch, heads, 2n) (causal:
      // (sequences, heads, n)) or, varlen, (heads, rows)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int q = qt * BMQ + lane + 32 * e;
        const bool valid = q < it.n;
        const long long off =
            VARLEN ? static_cast<long long>(h) * p.rows + it.row0 + static_cast<long long>(half) * it.n + q
                   : lse_offset(p.mode, it.wi.b, h, half, q, p.H, p.n);
        lse_r[e] = valid ? p.lse[off] * -1.4426950408889634f : -INFINITY;
        // -D * scale: the softmax scale is folded into dS (see the compute)
        del_r[e] = valid ? -p.delta[off] * p.scale : 0.f;
      }
    };
    auto store_rows = [&](int buf) {
      float* lse_s = reinterpret_cast<float*>(smem + C::kOffLSE) + buf * BMQ;
      float* del_s = reinterpret_cast<float*>(smem + C::kOffDEL) + buf * BMQ;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        lse_s[lane + 32 * e] = lse_r[e];
        del_s[lane + 32 * e] = del_r[e];
      }
      __syncwarp();
    };
    // Lane 0 waits on `bar` for `parity`; false when the wait gave up.
    auto warp_wait = [&](uint32_t bar, int parity) -> bool {
      int w = 0;
      if (lane == 0) w = mbar_wait(bar, parity, ab) ? 1 : 0;
      return __shfl_sync(0xffffffffu, w, 0) != 0;
    };
    // Q, dO, -LSE * log2(e) and -D of the item's t-th query tile into the
    // stage of global tile gg.
    auto load_q = [&](const Bwd2Item& it, int t, int gg) -> bool {
      int hh, l;
      it.template split<GQA>(t, hh, l);
      const int qt = it.ltile(l);
      const int half = it.lhalf(l);
      const int h = it.h0 + hh;  // query head
      stage_rows(it, t);
      const int st = gg % STAGES;
      const int round = gg / STAGES;
      if (round > 0 && !warp_wait(BAR(C::BAR_QEMPTY + st), (round - 1) & 1)) return false;
      store_rows(st);
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
    // Ring (headdim 256): the Q and dO chunks c of the item's t-th query
    // tile into ring slot `slot` (lane 0).
    int oh_last = -1, dh_last = -1;  // last tile with OH chunks, last DH chunk issued
    auto ring_chunk = [&](const Bwd2Item& it, int t, int c, int slot) {
      int hh, l;
      it.template split<GQA>(t, hh, l);
      const int qt = it.ltile(l);
      const int h = it.h0 + hh;
      const CUtensorMap* mq = VARLEN ? &p.vl_maps[it.slot].q : &p.tm_q;
      const CUtensorMap* mdo = VARLEN ? &p.vl_maps[it.slot].dout : &p.tm_do;
      const HalfRows qr = in_rows<VARLEN>(it.wi.b, it.lhalf(l));
      const uint32_t dst = sbase + C::kOffQ + slot * C::kSlotBytes;
      mbar_arrive_expect_tx(BAR(C::BAR_QFULL + slot), C::kSlotBytes);
      tma_load_5d(dst, mq, BAR(C::BAR_QFULL + slot), 64 * c, h, qr.base + qt * BMQ, qr.c3, qr.c4);
      tma_load_5d(dst + BMQ * 128, mdo, BAR(C::BAR_QFULL + slot), 64 * c, h, qr.base + qt * BMQ,
                  qr.c3, qr.c4);
    };
    // Tile gg's first own-half chunk (with its -LSE, -D rows) and its two
    // other-half chunks.  DH chunk s = 2 gg + j goes to slot kOhSlots + s % 3;
    // that slot last held chunk s - 3, of tile gg - 2 (j = 0), whose dV / dK
    // are then complete -- and with them the compute that read the rows
    // buffer gg & 1.  The OH slots last held tile gg - 1's chunks, free once
    // its S^T and dP^T are complete.
    auto ring_first = [&](const Bwd2Item& it, int t, int gg) -> bool {
      const int s0 = 2 * gg;
      const int slot0 = C::kOhSlots + s0 % C::kDhSlots;
      stage_rows(it, t);
      if (s0 >= C::kDhSlots &&
          !warp_wait(BAR(C::BAR_QEMPTY + slot0), (s0 / C::kDhSlots - 1) & 1))
        return false;
      store_rows(gg & 1);
      if (lane == 0) ring_chunk(it, t, 2 * it.dh, slot0);
      dh_last = s0;
      for (int i = 0; i < C::kOhSlots; ++i) {
        if (gg >= 1 && !warp_wait(BAR(C::BAR_QEMPTY + i), (gg - 1) & 1)) return false;
        if (lane == 0) ring_chunk(it, t, 2 * (1 - it.dh) + i, i);
      }
      oh_last = gg;
      __syncwarp();
      return true;
    };
    // Tile gg's second own-half chunk: its slot last held chunk 2 gg - 2, of
    // tile gg - 1.
    auto ring_last = [&](const Bwd2Item& it, int t, int gg) -> bool {
      const int s1 = 2 * gg + 1;
      const int slot1 = C::kOhSlots + s1 % C::kDhSlots;
      if (s1 >= C::kDhSlots &&
          !warp_wait(BAR(C::BAR_QEMPTY + slot1), (s1 / C::kDhSlots - 1) & 1))
        return false;
      if (lane == 0) ring_chunk(it, t, 2 * it.dh + 1, slot1);
      dh_last = s1;
      __syncwarp();
      return true;
    };
    while (ok) {
      int v = -1;
      if (lane == 0) v = sched_next(p.sched, p.items);
      v = __shfl_sync(0xffffffffu, v, 0);
      const Bwd2Item it = bwd2_item<C::NDH, BMQ, BN, GQA, VARLEN>(p, v);
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
      // K / V buffer `kvs` was last used by item k - KVBUF.  With one buffer
      // the first query tiles only need stages that the current item frees
      // before its last product, so they go ahead of the K / V load, which
      // waits for the whole item; with two the K / V load goes first.
      const int kvs = k % C::KVBUF;
      const int pre = C::KVBUF == 1 ? imin(it.ntiles, STAGES - 1) : 0;
      if constexpr (C::kChunkRing) {
        // the first tile's chunks that the current item frees before its
        // last products go ahead of the K / V load
        if (it.ntiles > 0) ok = ring_first(it, 0, g);
      } else {
        for (int t = 0; t < pre && ok; ++t) ok = load_q(it, t, g + t);
      }
      if (!ok) break;
      if (k >= C::KVBUF) {
        int w = 0;
        if (lane == 0)
          w = mbar_wait(BAR(C::BAR_ITEMDONE + kvs), (k / C::KVBUF - 1) & 1, ab) ? 1 : 0;
        if (!(ok = __shfl_sync(0xffffffffu, w, 0) != 0)) break;
      }
      if (lane == 0) {
        const CUtensorMap* mk = VARLEN ? &p.vl_maps[it.slot].k : &p.tm_k;
        const CUtensorMap* mv = VARLEN ? &p.vl_maps[it.slot].v : &p.tm_v;
        const HalfRows kr = in_rows<VARLEN>(it.wi.b, it.wi.half);
        const int krow = kr.base + it.wi.tile * BN;
        const uint32_t full = BAR(C::BAR_KVFULL + kvs);
        mbar_arrive_expect_tx(full, 2 * C::kKVBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_5d(sbase + C::kOffK + kvs * C::kKVBytes + c * BN * 128, mk, full, 64 * c,
                      it.wi.h, krow, kr.c3, kr.c4);
          tma_load_5d(sbase + C::kOffV + kvs * C::kKVBytes + c * BN * 128, mv, full, 64 * c,
                      it.wi.h, krow, kr.c3, kr.c4);
        }
      }
      __syncwarp();
      kv_issued = k + 1;
      if constexpr (C::kChunkRing) {
        for (int t = 0; t < it.ntiles && ok; ++t) {
          if (t > 0) ok = ring_first(it, t, g + t);
          if (ok) ok = ring_last(it, t, g + t);
        }
      } else {
        for (int t = pre; t < it.ntiles && ok; ++t) ok = load_q(it, t, g + t);
      }
      g += it.ntiles;
      ++k;
    }
    // Unwinding after a failed wait: let the copies in flight land.
    if (!ok && lane == 0) {
      if (kv_issued > 0)
        mbar_wait_limited(BAR(C::BAR_KVFULL + (kv_issued - 1) % C::KVBUF),
                          ((kv_issued - 1) / C::KVBUF) & 1, 100000000ull);
      if constexpr (C::kChunkRing) {
        if (oh_last >= 0)
          for (int i = 0; i < C::kOhSlots; ++i)
            mbar_wait_limited(BAR(C::BAR_QFULL + i), oh_last & 1, 100000000ull);
        for (int s = (dh_last >= C::kDhSlots ? dh_last - C::kDhSlots + 1 : 0); s <= dh_last; ++s)
          mbar_wait_limited(BAR(C::BAR_QFULL + C::kOhSlots + s % C::kDhSlots),
                            (s / C::kDhSlots) & 1, 100000000ull);
      } else {
        for (int t = (q_issued > STAGES ? q_issued - STAGES : 0); t < q_issued; ++t)
          mbar_wait_limited(BAR(C::BAR_QFULL + t % STAGES), (t / STAGES) & 1, 100000000ull);
      }
    }
    __syncwarp();
   } else {
    // ------------------------------------------------------------ MMA issuers
    // Three independent streams of products, each issued by its own warp so
    // that their issue overlaps: warp 9 issues S^T of every tile, warp 11
    // dP^T, warp 10 dV, dK and then dQ^T.  Everything one stream needs from
    // another is ordered through the compute warpgroups' barriers (S^T / dP^T
    // complete -> P^T / dS^T written -> second products); SDPFULL counts one
    // commit from each of warps 9 and 11 (each waits for SDPFREE of the
    // previous tile first, so neither runs a phase ahead).
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(BN, BMQ, false, false);  // K Q^T, V dO^T
      constexpr uint32_t kIdKV = idesc_bf16(BN, DH, false, true);   // P^T dO, dS^T Q
      constexpr uint32_t kIdDQ = idesc_bf16(DH, BMQ, true, true);   // K^T dS^T
      auto adv = [](uint64_t d, uint32_t bytes) { return d + static_cast<uint64_t>(bytes >> 4); };
      bool ok = true;
      int g = 0, k = 0;
      if (warp == C::kWarpS || warp == C::kWarpDP) {
        const bool dp = warp == C::kWarpDP;
        const uint64_t dK_kmaj0 = sdesc_sw128(sbase + C::kOffK, 16, 1024);
        const uint64_t dV_kmaj0 = sdesc_sw128(sbase + C::kOffV, 16, 1024);
        const uint64_t dQ_kmaj = sdesc_sw128(sbase + C::kOffQ, 16, 1024);
        const uint64_t dO_kmaj = sdesc_sw128(sbase + C::kOffDO, 16, 1024);
        while (ok) {
          if (!(ok = mbar_wait(BAR(C::BAR_ITEMFULL + (k & 3)), (k >> 2) & 1, ab))) break;
          const Bwd2Item it = *ring(k & 3);
          if (it.v < 0) break;
          const int kvs = k % C::KVBUF;
          const uint64_t dK_kmaj = adv(dK_kmaj0, kvs * C::kKVBytes);
          const uint64_t dV_kmaj = adv(dV_kmaj0, kvs * C::kKVBytes);
          if (!(ok = mbar_wait(BAR(C::BAR_KVFULL + kvs), (k / C::KVBUF) & 1, ab))) break;
          if constexpr (C::kChunkRing) {
            // S^T = K Q^T or dP^T = V dO^T chunk by chunk, in the order the
            // chunks arrive: own-half chunk 0, the other half's two (whose
            // slots are then released), own-half chunk 1.
            const uint32_t acc = dp ? C::kTmemDP : C::kTmemS;
            const uint64_t a0 = dp ? dV_kmaj : dK_kmaj;
            auto chunk = [&](int c, int slot, bool first) {
              const uint64_t b = sdesc_sw128(
                  sbase + C::kOffQ + slot * C::kSlotBytes + (dp ? BMQ * 128 : 0), 16, 1024);
#pragma unroll
              for (int sub = 0; sub < 4; ++sub)
                mma_ss(tmem + acc, adv(a0, c * (BN * 128) + sub * 32), adv(b, sub * 32), kIdS,
                       (first && sub == 0) ? 0u : 1u);
            };
            for (int i = 0; i < it.ntiles && ok; ++i) {
              const int gg = g + i;
              const int s0 = 2 * gg, s1 = s0 + 1;
              const int slot0 = C::kOhSlots + s0 % C::kDhSlots;
              const int slot1 = C::kOhSlots + s1 % C::kDhSlots;
              if (gg >= 1 && !(ok = mbar_wait(BAR(C::BAR_SDPFREE), (gg - 1) & 1, ab))) break;
              if (!(ok = mbar_wait(BAR(C::BAR_QFULL + slot0), (s0 / C::kDhSlots) & 1, ab))) break;
              tc_fence_after();
              chunk(2 * it.dh, slot0, true);
              for (int j = 0; j < C::kOhSlots && ok; ++j) {
                if (!(ok = mbar_wait(BAR(C::BAR_QFULL + j), gg & 1, ab))) break;
                tc_fence_after();
                chunk(2 * (1 - it.dh) + j, j, false);
              }
              if (!ok) break;
              for (int j = 0; j < C::kOhSlots; ++j) mma_commit(BAR(C::BAR_QEMPTY + j));
              if (!(ok = mbar_wait(BAR(C::BAR_QFULL + slot1), (s1 / C::kDhSlots) & 1, ab))) break;
              tc_fence_after();
              chunk(2 * it.dh + 1, slot1, false);
              mma_commit(BAR(C::BAR_SDPFULL));
            }
          } else {
          if constexpr (C::kD64) {
            // K (S^T warp) or V (dP^T warp) of the item into TMEM, after this
            // warp's products of the previous item, which read them there
            tc_fence_after();
            const uint64_t a0 = dp ? dV_kmaj : dK_kmaj;
            const uint32_t ta = tmem + (dp ? C::kTmemVA : C::kTmemKA);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) tmem_cp_128x256b(ta + 8 * kk, adv(a0, kk * 32));
          }
          for (int i = 0; i < it.ntiles && ok; ++i) {
            const int gg = g + i;
            const int st = gg % STAGES;
            if (!(ok = mbar_wait(BAR(C::BAR_QFULL + st), (gg / STAGES) & 1, ab))) break;
            // S and dP are free once both warpgroups have read the previous tile's.
            if (gg >= 1 && !(ok = mbar_wait(BAR(C::BAR_SDPFREE), (gg - 1) & 1, ab))) break;
            tc_fence_after();
            const uint32_t st_off = st * C::kQBytes;
            // S^T = K Q^T (warp 9) or dP^T = V dO^T (warp 11).
            const uint32_t acc = dp ? C::kTmemDP : C::kTmemS;
            const uint64_t a0 = dp ? dV_kmaj : dK_kmaj;
            const uint64_t b0 = dp ? dO_kmaj : dQ_kmaj;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
              const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
              if constexpr (C::kD64)
                mma_ts(tmem + acc, tmem + (dp ? C::kTmemVA : C::kTmemKA) + 8 * kk,
                       adv(b0, st_off + qoff), kIdS, kk > 0 ? 1u : 0u);
              else
                mma_ss(tmem + acc, adv(a0, koff), adv(b0, st_off + qoff), kIdS, kk > 0 ? 1u : 0u);
            }
            mma_commit(BAR(C::BAR_SDPFULL));
          }
          }
          g += it.ntiles;
          ++k;
        }
      } else {
        while (ok) {
          if (!(ok = mbar_wait(BAR(C::BAR_ITEMFULL + (k & 3)), (k >> 2) & 1, ab))) break;
          const Bwd2Item it = *ring(k & 3);
          if (it.v < 0) break;
          // The head-dim half dh starts at 64-wide chunk 2 dh of K, Q and dO.
          const uint64_t dK_mn =
              sdesc_sw128(sbase + C::kOffK + (k % C::KVBUF) * C::kKVBytes + it.dh * 2 * (BN * 128),
                          BN * 128, 1024);
          const uint64_t dQ_mn =
              sdesc_sw128(sbase + C::kOffQ + it.dh * 2 * (BMQ * 128), BMQ * 128, 1024);
          const uint64_t dO_mn =
              sdesc_sw128(sbase + C::kOffDO + it.dh * 2 * (BMQ * 128), BMQ * 128, 1024);
          // dK / dV of the previous item must be read out before they restart
          // (waited for every item, so that ITEMDONE(k) always follows
          // ACCFREE(k - 1)).
          if (k >= 1 && !(ok = mbar_wait(BAR(C::BAR_ACCFREE), (k - 1) & 1, ab))) break;
          for (int i = 0; i < it.ntiles && ok; ++i) {
            // dV, dK, dQ of tile gg once its P^T / dS^T are in place: P^T in
            // TMEM buffer gg % 2 (the A operand of dV += P^T dO), dS^T in
            // shared tile gg % kDSBufs, as a K-major A operand (dK += dS^T Q)
            // and an MN-major B operand (dQ^T = K^T dS^T).
            const int gg = g + i;
            const uint32_t st_off = (gg % STAGES) * C::kQBytes;
            if (!(ok = mbar_wait(BAR(C::BAR_PDSFULL + (gg & 1)), (gg >> 1) & 1, ab))) break;
            tc_fence_after();
            const uint32_t ds_base = sbase + C::kOffDS + (gg % C::kDSBufs) * C::kDSBytes;
            const uint64_t dDS_mn = sdesc_sw128(ds_base, BN * 128, 1024);
            if constexpr (C::kChunkRing) {
              // dV, dK of the item's head-dim half, 64 dims (one chunk of dO
              // and of Q, in its ring slot) at a time; each slot is released
              // once its own products complete (the next tile's second chunk
              // goes into the first one's slot).
              constexpr uint32_t kIdKV64 = idesc_bf16(BN, 64, false, true);
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int slot = C::kOhSlots + (2 * gg + j) % C::kDhSlots;
                const uint32_t slot_base = sbase + C::kOffQ + slot * C::kSlotBytes;
                const uint64_t q_mn = sdesc_sw128(slot_base, BMQ * 128, 1024);
                const uint64_t o_mn = sdesc_sw128(slot_base + BMQ * 128, BMQ * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < BMQ / 16; ++kk) {
                  // queries [16kk, 16kk+16): chunk kk/2, P^T first 16 columns, dS^T last 16
                  const uint32_t col = tmem + C::kTmemP + 32 * (kk >> 1) + 8 * (kk & 1);
                  const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                  mma_ts(tmem + C::kTmemDV + 64 * j, col, adv(o_mn, kk * 16 * 128), kIdKV64, acc);
                  mma_ts(tmem + C::kTmemDK + 64 * j, col + 16, adv(q_mn, kk * 16 * 128), kIdKV64,
                         acc);
                }
                mma_commit(BAR(C::BAR_QEMPTY + slot));
              }
            } else if constexpr (C::kD64) {
              // P^T / dS^T of tile gg in TMEM buffer gg % 2: chunk kk / 2,
              // P^T in its first 16 columns, dS^T in the last 16
              const uint32_t pbase = tmem + C::kTmemP + 64 * (gg & 1);
#pragma unroll
              for (int kk = 0; kk < BMQ / 16; ++kk) {
                const uint32_t col = pbase + 32 * (kk >> 1) + 8 * (kk & 1);
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                mma_ts(tmem + C::kTmemDV, col, adv(dO_mn, st_off + kk * 16 * 128), kIdKV, acc);
                mma_ts(tmem + C::kTmemDK, col + 16, adv(dQ_mn, st_off + kk * 16 * 128), kIdKV,
                       acc);
              }
              mma_commit(BAR(C::BAR_QEMPTY + (gg % STAGES)));
            } else {
              const uint32_t pcol = tmem + C::kTmemP + 32 * (gg & 1);
              const uint64_t dDS_k = sdesc_sw128(ds_base, 16, 1024);
#pragma unroll
              for (int kk = 0; kk < BMQ / 16; ++kk) {
                // queries [16kk, 16kk+16): 8 columns of P^T, 32 bytes of each dS^T row
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                mma_ts(tmem + C::kTmemDV, pcol + 8 * kk, adv(dO_mn, st_off + kk * 16 * 128), kIdKV,
                       acc);
                mma_ss(tmem + C::kTmemDK, adv(dDS_k, kk * 32), adv(dQ_mn, st_off + kk * 16 * 128),
                       kIdKV, acc);
              }
              // dQ^T reads no Q / dO: the stage is free once dV / dK are done.
              mma_commit(BAR(C::BAR_QEMPTY + (gg % STAGES)));
            }
            // The DQ columns still hold dQ of tile gg-1 until it has been read out.
            if (gg >= 1 && !(ok = mbar_wait(BAR(C::BAR_DQFREE), (gg - 1) & 1, ab))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ss(tmem + C::kTmemDQ, adv(dK_mn, kk * 16 * 128), adv(dDS_mn, kk * 16 * 128),
                     kIdDQ, kk > 0 ? 1u : 0u);
            mma_commit(BAR(C::BAR_MMA2 + gg % C::kDSBufs));
          }
          if (!ok) break;
          mma_commit(BAR(C::BAR_ITEMDONE + k % C::KVBUF));
          g += it.ntiles;
          ++k;
        }
      }
      mma_commit(BAR(C::BAR_ALL));
    }
    __syncwarp();
   }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegCompute));
    // ------------------------------------------------------------ compute
    // Both warpgroups work on every query tile: warpgroup wg takes query
    // columns [32 wg, 32 wg + 32) of S^T, dP^T, P^T / dS^T and dQ^T.  The dQ
    // of a tile is read out of TMEM in the next tile's turn, after that
    // tile's P^T / dS^T are handed over, so no warpgroup waits for the dV,
    // dK, dQ products of the tile it has just finished.
    constexpr int HC = C::HC;                // query columns per warpgroup
    const int wg = warp >> 2;
    const int c0 = wg * HC;                  // first column of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // key row of the tile / TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    const uint64_t scale2 = f2_pack(sl2, sl2);
    const uint64_t dscale2 = f2_pack(p.scale, p.scale);
    const size_t dq_stride = static_cast<size_t>(p.H) * D;
    // Headdim 64: dQ^T (M = 64) has head dims 16 q .. 16 q + 15 in lanes
    // 32 q .. 32 q + 15 of lane quarter q = warp % 4, read with the 16-lane
    // shape: thread t holds head dim 16 q + t % 16 of the warpgroup's queries
    // c0 + 16 (t / 16) + [0, 16).
    auto drain_dq64 = [&](const Bwd2Item& it, int h, int qh, int qs) -> bool {
      constexpr int QC = HC / 2;  // queries per thread
      uint32_t dq[QC];
      tmem_ld_half<QC, QC>(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::kTmemDQ + c0,
                           dq);
      tmem_wait_ld();
      tmem_pin<QC>(dq);
      tc_fence_before();
      mbar_arrive_warp(BAR(C::BAR_DQFREE));
      const int n = VARLEN ? it.n : p.n;
      const int up = lane >> 4;
      if constexpr (!DET) {
        // The warp's HC queries x 16 head dims (float32, 64-byte rows: the
        // box of its bulk reduce) in its own staging tile; the upper half of
        // the warp writes its queries one step later, so that the two halves
        // of a store fall in different banks.
        const uint32_t stg = sbase + C::kOffDQS + warp * C::kDQSBytes;
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < QC; ++c) {
          const int cq = up ? ((c + 1) & (QC - 1)) : c;
          const uint32_t v = up ? dq[(c + 1) & (QC - 1)] : dq[c];
          st_shared_f32(stg + (QC * up + cq) * 64 + (lane & 15) * 4, __uint_as_float(v));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && qs + c0 < n) {
          const CUtensorMap* mdq = VARLEN ? &p.vl_maps[it.slot].dq : &p.tm_dq;
          const HalfRows dr = in_rows<VARLEN>(it.wi.b, qh);
          if (p.pass == 2)  // noisy-diagonal pass: the rows' first contribution
            tma_store_5d(mdq, stg, 16 * (warp & 3), h, dr.base + qs + c0, dr.c3, dr.c4);
          else
            tma_reduce_add_5d(mdq, stg, 16 * (warp & 3), h, dr.base + qs + c0, dr.c3, dr.c4);
          bulk_commit_group();
        }
        return true;
      } else {
        const size_t first = VARLEN ? static_cast<size_t>(it.row0)
                                    : static_cast<size_t>(it.wi.b) * 2 * static_cast<size_t>(p.n);
        // after the contributions of the key tiles the work order takes earlier
        const int ord = dq_ordinal(p.mode, n, VARLEN ? it.bs : p.bs, BMQ, BN, qh, qs / BMQ,
                                   it.wi.half, it.wi.tile);
        unsigned* sem = p.dq_sem + static_cast<size_t>(h) * p.sem_rows + first +
                        static_cast<size_t>(qh) * n + qs;
        if (!sem_wait_warp(sem, static_cast<unsigned>(C::kComputeWarps * ord), ab)) return false;
        const int qo = c0 + QC * up;  // the thread's first query of the tile
        float* ptr = p.dq_acc + ((first + static_cast<size_t>(qh) * n + qs + qo) * p.H + h) * D +
                     16 * (warp & 3) + (lane & 15);
        const int qmax = n - qs - qo;
#pragma unroll
        for (int c = 0; c < QC; ++c) {
          if (c < qmax) {
            if (p.pass == 2)
              *ptr = __uint_as_float(dq[c]);
            else
              red_add_f32(ptr, __uint_as_float(dq[c]));
          }
          ptr += dq_stride;
        }
        sem_signal_warp(sem);
        return true;
      }
    };
    // dQ^T of the tile whose products completed last: TMEM lane = head dim
    // `row`, columns = queries; added into the float32 accumulator.
    auto drain_dq = [&](const Bwd2Item& it, int h, int qh, int qs) -> bool {
      if constexpr (C::kD64) return drain_dq64(it, h, qh, qs);
      uint32_t dq[HC];
      tmem_ld_cols<HC>(t_lane + C::kTmemDQ + c0, dq);
      tmem_wait_ld();
      tmem_pin<HC>(dq);
      tc_fence_before();
      mbar_arrive_warp(BAR(C::BAR_DQFREE));
      if constexpr (C::kTmaDQ && !DET) {
        // Stage the warp's HC queries x 32 head dims (scaled) in its own
        // shared tile and let the copy engine add them into the accumulator.
        // Lane 0 issues the reduce; before the warp rewrites the tile it
        // waits until lane 0's previous reduce has read it.
        const uint32_t stg = sbase + C::kOffDQS + warp * C::kDQSBytes;
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < HC; ++c)
          st_shared_f32(stg + c * 128 + lane * 4, __uint_as_float(dq[c]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && qs + c0 < (VARLEN ? it.n : p.n)) {
          // Varlen: through the sample's own map, so that rows of the box
          // past the half are skipped rather than added to the next sample.
          const CUtensorMap* mdq = VARLEN ? &p.vl_maps[it.slot].dq : &p.tm_dq;
          const HalfRows dr = in_rows<VARLEN>(it.wi.b, qh);
          if (p.pass == 2)  // noisy-diagonal pass: the rows' first contribution
            tma_store_5d(mdq, stg, it.dh * DH + 32 * (warp & 3), h, dr.base + qs + c0, dr.c3,
                         dr.c4);
          else
            tma_reduce_add_5d(mdq, stg, it.dh * DH + 32 * (warp & 3), h, dr.base + qs + c0, dr.c3,
                              dr.c4);
          bulk_commit_group();
        }
        return true;
      }
      const int n = VARLEN ? it.n : p.n;
      const size_t first = VARLEN ? static_cast<size_t>(it.row0)
                                  : static_cast<size_t>(it.wi.b) * 2 * static_cast<size_t>(p.n);
      unsigned* sem = nullptr;
      if constexpr (DET) {
        // This item's contribution to the query tile comes after those of
        // the key tiles the work order takes earlier: wait for them.
        const int ord = dq_ordinal(p.mode, n, VARLEN ? it.bs : p.bs, BMQ, BN, qh, qs / BMQ,
                                   it.wi.half, it.wi.tile);
        sem = p.dq_sem + (static_cast<size_t>(it.dh) * p.H + h) * p.sem_rows + first +
              static_cast<size_t>(qh) * n + qs;
        if (!sem_wait_warp(sem, static_cast<unsigned>(C::kComputeWarps * ord), ab)) return false;
      }
      float* ptr = p.dq_acc + ((first + static_cast<size_t>(qh) * n + qs + c0) * p.H + h) * D +
                   it.dh * DH + row;
      const int qmax = n - qs - c0;
      if (p.pass == 2) {
        // noisy-diagonal pass: this item's contribution is the rows' first
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          if (c < qmax) *ptr = __uint_as_float(dq[c]);
          ptr += dq_stride;
        }
      } else if (qmax >= HC) {
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          red_add_f32(ptr, __uint_as_float(dq[c]));
          ptr += dq_stride;
        }
      } else {
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          if (c < qmax) red_add_f32(ptr, __uint_as_float(dq[c]));
          ptr += dq_stride;
        }
      }
      if constexpr (DET) sem_signal_warp(sem);
      return true;
    };
    bool ok = true;
    int g = 0, k = 0;
    while (ok) {
      if (!(ok = mbar_wait_warp(BAR(C::BAR_ITEMFULL + (k & 3)), (k >> 2) & 1, ab))) break;
      const Bwd2Item it = *ring(k & 3);
      if (it.v < 0) break;
      if constexpr (VARLEN && C::kTmaDQ) {
        // this launch's dq, dk, dv maps of the item's sample, as memory
        // holds them (headdim 64: dq only)
        if (lane == 0) {
          if constexpr (!DET) tensormap_acquire(&p.vl_maps[it.slot].dq);
          if constexpr (!C::kD64) {
            tensormap_acquire(&p.vl_maps[it.slot].dk);
            tensormap_acquire(&p.vl_maps[it.slot].dv);
          }
        }
      }
      const int ks = it.wi.tile * BN;
      const int j = ks + row;  // key inside its half
      // Query rows that see key j, per segment of the item: computed once,
      // so a tile needs no division and no per-tile visibility test (a tile
      // the mask does not cut gives the full column mask below).
      const int n = VARLEN ? it.n : p.n;
      const int bs = VARLEN ? it.bs : p.bs;
      const Interval iv0 = query_interval(it.rule0, j, n, bs);
      const Interval iv1 = query_interval(it.rule1, j, n, bs);
      // dQ of tile t: query head, half and first row
      auto drain_tile = [&](int t) -> bool {
        int hh, l;
        it.template split<GQA>(t, hh, l);
        return drain_dq(it, it.h0 + hh, it.lhalf(l), it.ltile(l) * BMQ);
      };
      for (int i = 0; i < it.ntiles && ok; ++i) {
        const int gg = g + i;
        const int st = C::kChunkRing ? (gg & 1) : gg % STAGES;  // -LSE, -D buffer
        int hh, l;
        it.template split<GQA>(i, hh, l);
        const int qs = it.ltile(l) * BMQ;
        const bool seg0 = l < it.n0;
        if (!(ok = mbar_wait_warp(BAR(C::BAR_SDPFULL), gg & 1, ab))) break;
        tc_fence_after();
        uint32_t sr[HC], dpr[HC];
        tmem_ld_cols<HC>(t_lane + C::kTmemS + c0, sr);
        tmem_ld_cols<HC>(t_lane + C::kTmemDP + c0, dpr);
        tmem_wait_ld();
        tmem_pin<HC>(sr);
        tmem_pin<HC>(dpr);
        tc_fence_before();
        mbar_arrive_warp(BAR(C::BAR_SDPFREE));

        const uint32_t nlse_s = sbase + C::kOffLSE + 4 * (st * BMQ + c0);
        const uint32_t ndel_s = sbase + C::kOffDEL + 4 * (st * BMQ + c0);
        // Columns (queries) of this warpgroup that see key j, as a mask:
        // those in [clo, chi) (all of them on a tile the mask does not cut).
        uint32_t keep;
        {
          const Interval iv = seg0 ? iv0 : iv1;
          const int lo = iv.lo - qs - c0, hi = iv.hi - qs - c0;
          const int clo = lo < 0 ? 0 : (lo > HC ? HC : lo);
          const int chi = hi < clo ? clo : (hi > HC ? HC : hi);
          const uint32_t below_hi = chi >= 32 ? 0xffffffffu : ((1u << chi) - 1u);
          const uint32_t below_lo = clo >= 32 ? 0xffffffffu : ((1u << clo) - 1u);
          keep = below_hi & ~below_lo;
        }
        // P^T and dS^T in packed pairs: x = s * sl2 - lse2, p = 2^x,
        // ds = p * (dp - D) * scale.  On a tile the mask cuts, a hidden
        // pair's p is cleared by AND with its column's mask bit spread to a
        // word; -LSE and -D of four columns come in one shared load.
        uint32_t wp[HC / 2], wd[HC / 2];
        auto pds = [&](auto masked) {
#pragma unroll
          for (int e4 = 0; e4 < HC / 4; ++e4) {
            uint32_t la, lb, lc, ld, da, db, dc, dd4;
            ld_shared_v4(nlse_s + 16 * e4, la, lb, lc, ld);
            ld_shared_v4(ndel_s + 16 * e4, da, db, dc, dd4);
            const uint32_t nl[4] = {la, lb, lc, ld};
            const uint32_t nd[4] = {da, db, dc, dd4};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 2 * e4 + h;
              const uint64_t x = f2_fma(
                  f2_pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), scale2,
                  f2_pack(__uint_as_float(nl[2 * h]), __uint_as_float(nl[2 * h + 1])));
              float x0, x1;
              f2_unpack(x, x0, x1);
              float p0 = ex2_approx(x0);
              float p1 = ex2_approx(x1);
              if constexpr (decltype(masked)::value) {
                p0 = __uint_as_float(__float_as_uint(p0) & bit_spread(keep, 2 * e));
                p1 = __uint_as_float(__float_as_uint(p1) & bit_spread(keep, 2 * e + 1));
              }
              // (dP - D) * scale: dS carries the softmax scale, so dQ and dK
              // need no scaling afterwards
              const uint64_t dd = f2_fma(
                  f2_pack(__uint_as_float(dpr[2 * e]), __uint_as_float(dpr[2 * e + 1])), dscale2,
                  f2_pack(__uint_as_float(nd[2 * h]), __uint_as_float(nd[2 * h + 1])));
              float d0, d1;
              f2_unpack(f2_mul(f2_pack(p0, p1), dd), d0, d1);
              wp[e] = pack_bf16x2(p0, p1);
              wd[e] = pack_bf16x2(d0, d1);
            }
          }
        };
        if (__all_sync(0xffffffffu, keep == 0xffffffffu))
          pds(std::false_type{});
        else
          pds(std::true_type{});
        // P^T buffer gg % 2 and dS^T tile gg % kDSBufs still feed the
        // products of tile gg - kDSBufs (headdim 128: the tile before the
        // previous one) until they complete.
        if (gg >= C::kDSBufs &&
            !(ok = mbar_wait_warp(BAR(C::BAR_MMA2 + (gg % C::kDSBufs)),
                                  ((gg / C::kDSBufs) - 1) & 1, ab)))
          break;
        tc_fence_after();
        if constexpr (C::kChunkRing) {
          // chunk c0 / 32: P^T in its first 16 columns, dS^T in the last 16;
          // this warpgroup's HC / 2 words of each start at word (c0 % 32) / 2
          const uint32_t pds_col = C::kTmemP + 32 * (c0 / 32) + (c0 % 32) / 2;
          tmem_st_cols<HC / 2>(t_lane + pds_col, wp);
          tmem_st_cols<HC / 2>(t_lane + pds_col + 16, wd);
        } else if constexpr (C::kD64) {
          // buffer gg % 2, chunk c0 / 32 (HC = 32: the warpgroup's whole chunk)
          static_assert(HC == 32, "one 32-query chunk per warpgroup");
          const uint32_t pds_col = C::kTmemP + 64 * (gg & 1) + c0;
          tmem_st_cols<16>(t_lane + pds_col, wp);
          tmem_st_cols<16>(t_lane + pds_col + 16, wd);
        } else {
          // this warpgroup's HC queries: HC / 2 words of P^T from column c0 / 2
          tmem_st_cols<HC / 2>(t_lane + C::kTmemP + 32 * (gg & 1) + c0 / 2, wp);
        }
        // dS^T row `row` of the shared tile: 16-byte units c0 / 8 onwards.
        const uint32_t ds_s = sbase + C::kOffDS + (gg % C::kDSBufs) * C::kDSBytes;
#pragma unroll
        for (int u4 = 0; u4 < HC / 8; ++u4) {
          const int u = c0 / 8 + u4;
          const uint32_t off = row * 128 + ((u ^ (row & 7)) << 4);
          st_shared_v4(ds_s + off, wd[4 * u4], wd[4 * u4 + 1], wd[4 * u4 + 2], wd[4 * u4 + 3]);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive_warp(BAR(C::BAR_PDSFULL + (gg & 1)));
        // The previous tile's dQ, once its products are complete (with one
        // dS^T tile that was waited for above).
        if (i >= 1) {
          if (C::kDSBufs == 2 &&
              !(ok = mbar_wait_warp(BAR(C::BAR_MMA2 + ((gg - 1) & 1)), ((gg - 1) >> 1) & 1, ab)))
            break;
          tc_fence_after();
          if (!(ok = drain_tile(i - 1))) break;
        }
      }
      if (!ok) break;

      // -------------------------------------------------------- item epilogue
      // The first half of the warpgroups writes dV, the second dK, each
      // warpgroup DW head dims of it, once the item's MMAs are done; TMEM is
      // released as soon as all have read their part.  Then the dQ of the
      // item's last tile.
      if (!(ok = mbar_wait_warp(BAR(C::BAR_ITEMDONE + k % C::KVBUF), (k / C::KVBUF) & 1, ab)))
        break;
      tc_fence_after();
      constexpr int PER = C::NWG / 2;  // warpgroups per accumulator
      constexpr int DW = DH / PER;     // head dims per warpgroup
      const bool is_v = wg < PER;
      const int d0 = (wg % PER) * DW;
      const uint32_t col = (is_v ? C::kTmemDV : C::kTmemDK) + d0;
      uint32_t o[DW];
      if (it.ntiles > 0) {
#pragma unroll
        for (int c = 0; c < DW / 32; ++c) tmem_ld32(t_lane + col + 32 * c, o + 32 * c);
        tmem_wait_ld();
        tmem_pin<DW>(o);
      } else {
#pragma unroll
        for (int e = 0; e < DW; ++e) o[e] = 0u;
      }
      tc_fence_before();
      mbar_arrive_warp(BAR(C::BAR_ACCFREE));
      const size_t first = VARLEN ? static_cast<size_t>(it.row0)
                                  : static_cast<size_t>(it.wi.b) * 2 * static_cast<size_t>(p.n);
      if constexpr (C::kTmaDQ && C::kDQSBytes >= 4096) {
        // The warp's 32 key rows (dK needs no scale: it is already in dS),
        // 64 head dims at a time through the warp's staging tile (once the
        // copy before has read it), in the 128-byte-swizzled layout of a TMA
        // box, and out with a bulk tensor store: rows past the half are
        // dropped by the copy, and the warp does not wait for the stores.
        static_assert(DW % 64 == 0, "whole 64-dim boxes");
        const uint32_t stg = sbase + C::kOffDQS + warp * C::kDQSBytes;
        const CUtensorMap* mkv = VARLEN ? (is_v ? &p.vl_maps[it.slot].dv : &p.vl_maps[it.slot].dk)
                                        : (is_v ? &p.tm_dv : &p.tm_dk);
        const HalfRows kr = in_rows<VARLEN>(it.wi.b, it.wi.half);
#pragma unroll
        for (int rd = 0; rd < DW / 64; ++rd) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int e0 = 64 * rd + 8 * u;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[e0 + 2 * e]), __uint_as_float(o[e0 + 2 * e + 1]));
            st_shared_v4(stg + lane * 128 + ((u ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_5d(mkv, stg, it.dh * DH + d0 + 64 * rd, it.wi.h,
                         kr.base + ks + (warp & 3) * 32, kr.c3, kr.c4);
            bulk_commit_group();
          }
        }
      } else if (j < n) {
        // headdim 256 (no staging tile left) or a staging tile too small for
        // a box: each thread its own row
        const size_t pos = static_cast<size_t>(it.wi.half) * n + j;
        const size_t off = ((first + pos) * p.Hk + it.wi.h) * D + it.dh * DH + d0;
        __nv_bfloat16* dst = (is_v ? p.dv : p.dk) + off;
#pragma unroll
        for (int g8 = 0; g8 < DW / 8; ++g8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[g8 * 8 + 2 * e]),
                               __uint_as_float(o[g8 * 8 + 2 * e + 1]));
          st_global_v4(dst + 8 * g8, w[0], w[1], w[2], w[3]);
        }
      }
      if (it.ntiles > 0 && !(ok = drain_tile(it.ntiles - 1))) break;
      g += it.ntiles;
      ++k;
    }
    // The last bulk reduce-adds must be complete before the CTA exits.
    if constexpr (C::kTmaDQ) {
      if (lane == 0) bulk_wait_all();
    }
  }
#undef BAR

  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpS) {
    if (lane == 0) mbar_wait_limited(sbase + C::kOffBar + 8 * C::BAR_ALL, 0, 1000000000ull);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0) sched_finish(p.sched);
}

template <int D, int STAGES, int NWG, int KVBUF, bool GQA, bool VARLEN, bool DET = false>
static cudaError_t launch_bwd2_impl(const BwdParams& p, cudaStream_t stream) {
  using C = Bwd2Cfg<D, STAGES, NWG, KVBUF>;
  auto kern = dfa_bwd2_kernel<D, STAGES, NWG, KVBUF, GQA, VARLEN, DET>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The setmaxnreg split must fit the registers the kernel is launched with,
  // or the compute warps' increase would never be granted: refuse to launch.
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs * C::kThreads < C::kRegCtl * 128 + C::kRegCompute * 128 * C::NWG)
    return cudaErrorInvalidConfiguration;
  const long long items =
      (VARLEN  ? static_cast<long long>(p.units)
       : p.pass ? static_cast<long long>(p.B) * p.Hk * p.k_tiles  // one key half per pass
                : pass_items(p.mode, p.B, p.Hk, p.k_tiles)) *
      C::NDH;
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

cudaError_t launch_backward_d128(const BwdParams& p, cudaStream_t stream) {
  // Grouped key/value heads get their own instantiation, so that the
  // multi-head kernel keeps its tile loop free of head bookkeeping.
  constexpr int W = kBwd2WarpgroupsD128;
  // Deterministic mode: its own instantiations (grouped heads, both layouts).
  if (p.dq_sem)
    return p.vl ? launch_bwd2_impl<128, 3, W, 1, true, true, true>(p, stream)
                : launch_bwd2_impl<128, 3, W, 1, true, false, true>(p, stream);
  if (p.vl) return launch_bwd2_impl<128, 3, W, 1, true, true>(p, stream);
  return p.kv_group > 1 ? launch_bwd2_impl<128, 3, W, 1, true, false>(p, stream)
                        : launch_bwd2_impl<128, 3, W, 1, false, false>(p, stream);
}

// Headdim 64: 64-query tiles, the same pipeline as headdim 128 (P^T / dS^T
// double-buffered in TMEM, S^T / dP^T released once read), four Q / dO
// stages of 16 KB.
cudaError_t launch_backward_d64(const BwdParams& p, cudaStream_t stream) {
  if (p.dq_sem)
    return p.vl ? launch_bwd2_impl<64, 4, 2, 1, true, true, true>(p, stream)
                : launch_bwd2_impl<64, 4, 2, 1, true, false, true>(p, stream);
  if (p.vl) return launch_bwd2_impl<64, 4, 2, 1, true, true>(p, stream);
  return p.kv_group > 1 ? launch_bwd2_impl<64, 4, 2, 1, true, false>(p, stream)
                        : launch_bwd2_impl<64, 4, 2, 1, false, false>(p, stream);
}

cudaError_t launch_backward_d256(const BwdParams& p, cudaStream_t stream);

cudaError_t launch_backward(const BwdParams& p, int headdim, cudaStream_t stream) {
  switch (headdim) {
    case 64: return launch_backward_d64(p, stream);
    case 128: return launch_backward_d128(p, stream);
    case 256: return launch_backward_d256(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_backward_d256(const BwdParams& p, cudaStream_t stream) {
  if (p.dq_sem)
    return p.vl ? launch_bwd2_impl<256, 1, 2, 1, true, true, true>(p, stream)
                : launch_bwd2_impl<256, 1, 2, 1, true, false, true>(p, stream);
  if (p.vl) return launch_bwd2_impl<256, 1, 2, 1, true, true>(p, stream);
  return p.kv_group > 1 ? launch_bwd2_impl<256, 1, 2, 1, true, false>(p, stream)
                        : launch_bwd2_impl<256, 1, 2, 1, false, false>(p, stream);
}

}  // namespace dfa
