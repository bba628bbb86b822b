// Persistent forward kernel of block-diffusion attention (headdim 64, 128).
//
// One CTA per SM takes work items from a work counter until none are left,
// one item being one 128-row query tile of one half of one (batch, head)
// (items ordered longest first inside groups of heads that share L2, the
// shortest of all heads last).  For its item it visits
// exactly the key tiles the mask reaches ("Fast Diffusion Attention", "Visit
// only the visible tiles") and runs the loop of "FlashAttention: Exact
// Attention Without Materialization", section 5.1, with the online softmax of
// section 4.2.
//
// Eight softmax warps share every key tile of the item, each on 16 of its
// 128 rows: TMEM is read and written in the 16-lane shape, which gives
// thread t of the warp row t % 16 of the warp's 16 and key columns
// [64 (t / 16), 64 (t / 16) + 64) of it, so the two halves of a row sit in
// threads t and t ^ 16 of one warp and their maxima and sums meet in one
// shuffle.  Every row's reference maximum is thus common to both halves,
// the probabilities of the whole tile feed a single output accumulator O in
// TMEM and nothing is merged at the end of an item.  Scores S = Q K^T land
// in one of three TMEM buffers, so the
// scores of the next two tiles are computed while the softmax of this one
// runs (a tile's products and softmax form a chain of about three times the
// tensor-core time of a tile, most of it latency);
// the probabilities of each half row go as bf16 back into the first half of
// that half's columns of the buffer, where O += P V reads them as the MMA's
// A operand.  A row's reference maximum is only moved (O and the sum
// rescaled) when a tile maximum exceeds it by more than 2^8: exact in real
// arithmetic, and probabilities stay below 256.  With headdim 64 O is also
// double-buffered by item, so the next item's first products need not wait
// for the read-out of this one.
//
// The K/V ring, the query double buffer and all barrier phases run on across
// items, so the loads and S products of the next item overlap the read-out
// and stores of the current one.
// The softmax warps first; then one warp takes the items and loads Q, K and
// V, one issues O += P V and one S = Q K^T, and one stores the out tiles (staged
// by the softmax warps in the item's query buffer) with TMA and zeroes
// the backward's float32 dq accumulator when the caller asks for it.
// The load/MMA warpgroup hands registers to the softmax warps (setmaxnreg):
// launched with 168 per thread, it drops to 56 and the softmax warps rise to
// 224.  256 * (224 - 168) == 128 * (168 - 56): the pool balances.
#include <cuda_bf16.h>

#include "geometry.cuh"
#include "params.cuh"
#include "sm100.cuh"

namespace dfa {

// FP8: q, k, v in e4m3 (the FP8 forward of "Fast Diffusion Attention"):
// 128-byte rows hold 128 elements, a K step of the products is 32 elements,
// P goes to TMEM as four e4m3 per column; out stays bf16, staged in the
// query buffer, which keeps the bf16 tile's size.
// STAGES K tiles and VSTAGES V tiles in flight (a K tile is needed first,
// by S, a V tile a softmax later, by P V).
// Eight softmax warps, each thread on kCols = 64 key columns of a row of
// every tile and kDCols = D / 2 head dims of its row of O.
template <int D, int STAGES, int VSTAGES, bool FP8 = false>
struct Fwd2Cfg {
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int kCols = BN / 2;
  static constexpr int kDCols = D / 2;
  static constexpr int kSoftWarps = 8;
  static constexpr int kWarpLoad = kSoftWarps;       // items, Q / K / V loads
  static constexpr int kWarpPV = kSoftWarps + 1;     // O += P V; owns TMEM
  static constexpr int kWarpS = kSoftWarps + 2;      // S = Q K^T
  static constexpr int kWarpStore = kSoftWarps + 3;  // out stores, dq zeroing
  static constexpr int kThreads = 32 * (kSoftWarps + 4);
  // setmaxnreg split within the launch's pool: the load / MMA / store warps
  // drop to kRegCtl, the softmax warps rise to kRegSoft.
  static constexpr int kRegLaunch = 168;
  static constexpr int kRegCtl = 56;
  static constexpr int kRegSoft = 224;
  static_assert(kRegCtl * 128 + kRegSoft * 32 * kSoftWarps <= kRegLaunch * kThreads,
                "register split exceeds the launch pool");
  static_assert(kCols % 32 == 0 && kDCols % 16 == 0, "column split");
  static constexpr int ES = FP8 ? 1 : 2;           // bytes per q / k / v element
  static constexpr int kChunkElems = 128 / ES;     // elements per 128-byte row
  static constexpr int kChunks = D / kChunkElems;  // 128-byte chunks of q, k, v rows
  static constexpr int kOutChunks = D / 64;        // 128-byte chunks of a bf16 out row
  static constexpr int kKSteps = D * ES / 32;      // K steps of S = Q K^T (32 bytes each)
  static constexpr int kPVKeys = 32 / ES;          // keys per step of O += P V
  static constexpr int kQLoadBytes = BM * D * ES;
  static constexpr int kQBytes = BM * D * 2;       // query buffer: also the bf16 out tile
  static constexpr int kKVBytes = BN * D * ES;
  static constexpr int kOffQ = 0;  // 2 buffers
  static constexpr int kOffK = kOffQ + 2 * kQBytes;
  static constexpr int kOffV = kOffK + STAGES * kKVBytes;  // [VSTAGES]
  // TMEM buffers of S (tiles in flight between the S product and P V)
  static constexpr int kSBufs = 3;
  static constexpr int kOffBar = kOffV + VSTAGES * kKVBytes;
  enum {
    BAR_QFULL = 0,                    // [2]
    BAR_QEMPTY = BAR_QFULL + 2,       // [2]
    BAR_KFULL = BAR_QEMPTY + 2,        // [STAGES]
    BAR_KEMPTY = BAR_KFULL + STAGES,   // [STAGES]
    BAR_VFULL = BAR_KEMPTY + STAGES,   // [VSTAGES]
    BAR_VEMPTY = BAR_VFULL + VSTAGES,  // [VSTAGES]
    BAR_SFULL = BAR_VEMPTY + VSTAGES,   // [kSBufs] per S buffer: S of its tile complete
    BAR_PFULL = BAR_SFULL + kSBufs,     // [kSBufs] per S buffer: P of its tile written (8 warps)
    BAR_SFREE = BAR_PFULL + kSBufs,     // [kSBufs] per S buffer: P V of its tile complete
    BAR_OFREE = BAR_SFREE + kSBufs,     // [2] per O buffer: read out (8 warps)
    BAR_ITEMFULL = BAR_OFREE + 2,     // [4] item published
    BAR_OSTAGED = BAR_ITEMFULL + 4,   // [2] per query buffer: the item's out tile staged in it
    BAR_ALL = BAR_OSTAGED + 2,        // every MMA of the CTA complete
    NUM_BARS = BAR_ALL + 1
  };
  static constexpr int kOffItem = kOffBar + NUM_BARS * 8;  // 4 decoded items (ItemGeom)
  static constexpr int kOffTmemSlot = kOffItem + 4 * 128;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  // The dynamic shared memory starts 1024-byte aligned (the kernel checks
  // this, for the 128-byte swizzle of the TMA boxes and MMA operands).
  static constexpr int kSmemBytes = kOffAbort + 4;
  // S[b] at b * BN (tile g in buffer g % kSBufs); P of key columns
  // [64 h, 64 h + 64) in its columns [64 h, 64 h + 32).  O[item % kOBufs]
  // after the S buffers.
  static constexpr int kTmemS = 0;
  static constexpr int kTmemO = kSBufs * BN;
  static constexpr int kOBufs = kSBufs * BN + 2 * D <= 512 ? 2 : 1;
  static constexpr int kTmemCols = 512;
  static constexpr float kRescaleThreshold = 8.0f;  // log2 units
  static_assert(kTmemO + kOBufs * D <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// One work item: query tile and the key tiles it visits (at most two
// segments, kept in scalars so that nothing is indexed dynamically).  The
// producer decodes each item once and publishes the decoded form to the other
// roles through a ring in shared memory; item < 0 means no work is left.
struct ItemGeom {
  int item;
  WorkItem wi;
  int n0, ntiles, qs;
  int half0, rule0, tb0, half1, rule1, tb1;
  int n, row0;  // varlen: the sample's half length and first row
  int slot;     // varlen: the sample's slot (its tensor maps)
  __device__ __forceinline__ int ktile(int j) const { return j < n0 ? tb0 + j : tb1 + (j - n0); }
  __device__ __forceinline__ int khalf(int j) const { return j < n0 ? half0 : half1; }
};

static_assert(sizeof(ItemGeom) <= 128, "item ring slot");

template <bool VARLEN>
__device__ __forceinline__ void item_geom(const FwdParams& p, int item, int bm, int bn,
                                          ItemGeom* g) {
  g->item = item;
  if (item < 0) return;
  int n = p.n, bs = p.bs;
  if constexpr (VARLEN) {
    g->slot = varlen_slot(p.vl, p.vl_slots, item);
    const VarlenSlot sl = p.vl[g->slot];
    n = sl.n;
    bs = imin(p.bs, n);
    g->wi = fwd_work(item - sl.off, MODE_DIFFUSION, 1, p.H, cdiv(n, bm), sl.group);
    g->wi.b = sl.b;
    g->n = n;
    g->row0 = sl.row0;
  } else {
    g->wi = fwd_work(item, p.mode, p.B, p.H, p.q_tiles, p.group);
    g->slot = 0;
  }
  Segment seg[2] = {{0, RULE_NONE, 0, 0}, {0, RULE_NONE, 0, 0}};
  const int nseg = fwd_segments(p.mode, n, bs, bm, bn, g->wi.half, g->wi.tile, seg);
  g->n0 = nseg > 0 ? seg[0].t_end - seg[0].t_begin : 0;
  g->ntiles = g->n0 + (nseg > 1 ? seg[1].t_end - seg[1].t_begin : 0);
  g->half0 = seg[0].half;
  g->rule0 = seg[0].rule;
  g->tb0 = seg[0].t_begin;
  g->half1 = seg[1].half;
  g->rule1 = seg[1].rule;
  g->tb1 = seg[1].t_begin;
  g->qs = g->wi.tile * bm;
}

template <int D, int STAGES, int VSTAGES, bool VARLEN, bool FP8 = false>
__global__ void __launch_bounds__(Fwd2Cfg<D, STAGES, VSTAGES, FP8>::kThreads, 1)
    dfa_fwd2_kernel(const __grid_constant__ FwdParams p) {
  using C = Fwd2Cfg<D, STAGES, VSTAGES, FP8>;
  constexpr int BM = C::BM;
  constexpr int BN = C::BN;
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
  // Slot s of the item ring; written by the load warp before it arrives on
  // ITEMFULL[s] (release), read by the other roles after their wait (acquire).
  auto ring = [&](int s) { return reinterpret_cast<ItemGeom*>(smem + C::kOffItem + 128 * s); };
  const AbortFlag ab{abort_flag, p.status};
  const int num_items = VARLEN ? p.items : static_cast<int>(pass_items(p.mode, p.B, p.H, p.q_tiles));
#define BAR(i) (sbase + C::kOffBar + 8 * (i))

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(C::BAR_QFULL + b), 1);
      mbar_init(BAR(C::BAR_QEMPTY + b), 1);
      mbar_init(BAR(C::BAR_OFREE + b), C::kSoftWarps);
      mbar_init(BAR(C::BAR_OSTAGED + b), C::kSoftWarps);
    }
    for (int b = 0; b < C::kSBufs; ++b) {
      mbar_init(BAR(C::BAR_SFULL + b), 1);
      mbar_init(BAR(C::BAR_PFULL + b), C::kSoftWarps);
      mbar_init(BAR(C::BAR_SFREE + b), 1);
    }
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(BAR(C::BAR_KFULL + s), 1);
      mbar_init(BAR(C::BAR_KEMPTY + s), 1);
    }
    for (int s = 0; s < VSTAGES; ++s) {
      mbar_init(BAR(C::BAR_VFULL + s), 1);
      mbar_init(BAR(C::BAR_VEMPTY + s), 1);
    }
    for (int s = 0; s < 4; ++s) mbar_init(BAR(C::BAR_ITEMFULL + s), 1);
    mbar_init(BAR(C::BAR_ALL), 2);  // both MMA-issuing warps
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kWarpPV) {
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

  if (warp >= C::kSoftWarps) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegCtl));
   if (warp == C::kWarpLoad) {
    // ------------------------------------------------------------ producer
    // Takes items, publishes them and loads Q and the K and V rings.  The V
    // load of a tile is issued after the K load of the next one, so that a K
    // tile (needed first, by S) never waits behind a V slot.
    if (lane == 0) {
      if constexpr (!VARLEN) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
      }
      bool ok = true;
      int g = 0;  // K/V ring position across items
      // The V tile still to be loaded: ring position vg (< 0: none), its
      // tensor map and coordinates.
      int vg = -1, vh = 0, vc2 = 0, vc3 = 0, vc4 = 0;
      const CUtensorMap* vmap = &p.tm_v;
      auto load_v = [&]() -> bool {
        const int st = vg % VSTAGES;
        const int round = vg / VSTAGES;
        if (round > 0 && !mbar_wait(BAR(C::BAR_VEMPTY + st), (round - 1) & 1, ab)) return false;
        mbar_arrive_expect_tx(BAR(C::BAR_VFULL + st), C::kKVBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          if constexpr (FP8)  // V^T (n, half, headdim, heads, batch): keys innermost;
                              // vc3 = 2 * batch + half (batched coordinates)
            tma_load_5d(sbase + C::kOffV + st * C::kKVBytes, &p.tm_v, BAR(C::BAR_VFULL + st), vc2,
                        vc3 & 1, 0, vh, vc3 >> 1);
          else
            tma_load_5d(sbase + C::kOffV + st * C::kKVBytes + c * BN * 128, vmap,
                        BAR(C::BAR_VFULL + st), C::kChunkElems * c, vh, vc2, vc3, vc4);
        vg = -1;
        return true;
      };
      for (int k = 0; ok; ++k) {
        // Items come from the work counter and are published, decoded, to the
        // other roles through slot k % 4 of the item ring.  The slot last held
        // item k - 4, whose readers are all done: for item k - 1's query
        // buffer this loader has already waited until the store warp stored item
        // k - 3's out tile, which exists only after every role has read item
        // k - 4's slot.
        ItemGeom ig;
        item_geom<VARLEN>(p, sched_next(p.sched, num_items), BM, BN, &ig);
        *ring(k & 3) = ig;
        mbar_arrive(BAR(C::BAR_ITEMFULL + (k & 3)));
        if (ig.item < 0) break;
        const int qb = k & 1;
        if (k >= 2 && !(ok = mbar_wait(BAR(C::BAR_QEMPTY + qb), ((k >> 1) - 1) & 1, ab))) break;
        // Varlen: the sample's own maps (rows past its halves read zero).
        const CUtensorMap* mq = &p.tm_q;
        const CUtensorMap* mk = &p.tm_k;
        const CUtensorMap* mv = &p.tm_v;
        if constexpr (VARLEN) {
          mq = &p.vl_maps[ig.slot].q;
          mk = &p.vl_maps[ig.slot].k;
          mv = &p.vl_maps[ig.slot].v;
          tensormap_acquire(mq);
          tensormap_acquire(mk);
          tensormap_acquire(mv);
        }
        mbar_arrive_expect_tx(BAR(C::BAR_QFULL + qb), C::kQLoadBytes);
        const HalfRows qr = in_rows<VARLEN>(ig.wi.b, ig.wi.half);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_5d(sbase + C::kOffQ + qb * C::kQBytes + c * BM * 128, mq,
                      BAR(C::BAR_QFULL + qb), C::kChunkElems * c, ig.wi.h, qr.base + ig.qs, qr.c3,
                      qr.c4);
        // key/value head of query head wi.h (grouped heads: kv_group > 1)
        const int hk = p.kv_group == 1 ? ig.wi.h : ig.wi.h / p.kv_group;
        for (int j = 0; j < ig.ntiles; ++j, ++g) {
          const int st = g % STAGES;
          const int round = g / STAGES;
          if (round > 0 && !(ok = mbar_wait(BAR(C::BAR_KEMPTY + st), (round - 1) & 1, ab))) break;
          mbar_arrive_expect_tx(BAR(C::BAR_KFULL + st), C::kKVBytes);
          const HalfRows kr = in_rows<VARLEN>(ig.wi.b, ig.khalf(j));
          const int krow = kr.base + ig.ktile(j) * BN;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_5d(sbase + C::kOffK + st * C::kKVBytes + c * BN * 128, mk,
                        BAR(C::BAR_KFULL + st), C::kChunkElems * c, hk, krow, kr.c3, kr.c4);
          if (vg >= 0 && !(ok = load_v())) break;
          vg = g;
          vmap = mv;
          vh = hk;
          vc2 = krow;
          vc3 = kr.c3;
          vc4 = kr.c4;
        }
      }
      if (ok && vg >= 0) ok = load_v();
      if (!ok) {
        // Unwinding: give the copies already issued time to land.
        const unsigned long long t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 20000000ull) {
        }
      }
    }
    __syncwarp();
   } else if (warp == C::kWarpPV || warp == C::kWarpS) {
    // ------------------------------------------------------------ MMA issuers
    // One warp issues S = Q K^T, another O += P V.  Issued from one warp, the
    // products slow down while the softmax warps that share its scheduler are
    // busy; from two warps on two schedulers they keep the tensor pipe fed.
    // The two streams meet only through barriers: S of tile g goes into
    // buffer g % kSBufs once P V of tile g - kSBufs (whose P it held) has
    // completed (SFREE); P V of a tile waits for all softmax warps' P (PFULL),
    // and the first P V of an item for the read-out of the O buffer it reuses
    // (OFREE).
    if (lane == 0) {
      const bool s_warp = warp == C::kWarpS;
      constexpr uint32_t kIdS =
          FP8 ? idesc_e4m3(BM, BN, false, false) : idesc_bf16(BM, BN, false, false);
      constexpr uint32_t kIdPV =
          FP8 ? idesc_e4m3(BM, D, false, false) : idesc_bf16(BM, D, false, true);
      constexpr int kPVSteps = BN / C::kPVKeys;
      const uint64_t dQ = sdesc_sw128(sbase + C::kOffQ, 16, 1024);
      const uint64_t dK = sdesc_sw128(sbase + C::kOffK, 16, 1024);
      // V: MN-major (keys = K in rows); FP8 reads V^T, K-major (128 keys a row)
      const uint64_t dV = FP8 ? sdesc_sw128(sbase + C::kOffV, 16, 1024)
                              : sdesc_sw128(sbase + C::kOffV, BN * 128, 1024);
      auto adv = [](uint64_t d, uint32_t bytes) { return d + static_cast<uint64_t>(bytes >> 4); };
      bool ok = true;
      int g = 0;  // tiles of earlier items (K/V ring and S buffer position)
      for (int k = 0; ok; ++k) {
        if (!(ok = mbar_wait(BAR(C::BAR_ITEMFULL + (k & 3)), (k >> 2) & 1, ab))) break;
        const ItemGeom ig = *ring(k & 3);
        if (ig.item < 0) break;
        const int qb = k & 1;
        const int ob = k % C::kOBufs;
        if (s_warp) {
          if (!(ok = mbar_wait(BAR(C::BAR_QFULL + qb), (k >> 1) & 1, ab))) break;
        } else {
          // O buffer ob still holds item k - kOBufs until it is read out.
          if (k >= C::kOBufs &&
              !(ok = mbar_wait(BAR(C::BAR_OFREE + ob), ((k / C::kOBufs) - 1) & 1, ab)))
            break;
        }
        tc_fence_after();
        for (int j = 0; j < ig.ntiles && ok; ++j) {
          const int gg = g + j;
          const int st = gg % STAGES;
          const int sb = gg % C::kSBufs;
          const int su = gg / C::kSBufs;  // earlier tiles in buffer sb
          if (s_warp) {
            if (!(ok = mbar_wait(BAR(C::BAR_KFULL + st), (gg / STAGES) & 1, ab))) break;
            if (su >= 1 && !(ok = mbar_wait(BAR(C::BAR_SFREE + sb), (su - 1) & 1, ab))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < C::kKSteps; ++kk) {
              const uint64_t a = adv(dQ, qb * C::kQBytes + (kk >> 2) * (BM * 128) + (kk & 3) * 32);
              const uint64_t b = adv(dK, st * C::kKVBytes + (kk >> 2) * (BN * 128) + (kk & 3) * 32);
              if constexpr (FP8)
                mma_ss_f8(tmem + C::kTmemS + sb * BN, a, b, kIdS, kk > 0 ? 1u : 0u);
              else
                mma_ss(tmem + C::kTmemS + sb * BN, a, b, kIdS, kk > 0 ? 1u : 0u);
            }
            mma_commit(BAR(C::BAR_SFULL + sb));
            mma_commit(BAR(C::BAR_KEMPTY + st));
          } else {
            if (!(ok = mbar_wait(BAR(C::BAR_PFULL + sb), su & 1, ab))) break;
            const int vs = gg % VSTAGES;
            if (!(ok = mbar_wait(BAR(C::BAR_VFULL + vs), (gg / VSTAGES) & 1, ab))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kPVSteps; ++kk) {
              // P of keys [kPVKeys kk, kPVKeys (kk + 1)): in the columns of the
              // row half that holds them, 8 columns per step (bf16 pairs or
              // e4m3 quadruples); V: 16 key rows of 128 bytes, or (V^T) 32
              // bytes of 128-key rows
              constexpr int kStepsPerHalf = C::kCols / C::kPVKeys;
              const uint32_t pcol =
                  C::kTmemS + sb * BN + C::kCols * (kk / kStepsPerHalf) + 8 * (kk % kStepsPerHalf);
              const uint64_t b =
                  adv(dV, vs * C::kKVBytes + (FP8 ? kk * 32 : kk * C::kPVKeys * 128));
              const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
              if constexpr (FP8)
                mma_ts_f8(tmem + C::kTmemO + ob * D, tmem + pcol, b, kIdPV, acc);
              else
                mma_ts(tmem + C::kTmemO + ob * D, tmem + pcol, b, kIdPV, acc);
            }
            mma_commit(BAR(C::BAR_VEMPTY + vs));
            mma_commit(BAR(C::BAR_SFREE + sb));
          }
        }
        if (!ok) break;
        g += ig.ntiles;
      }
      mma_commit(BAR(C::BAR_ALL));
    }
    __syncwarp();
   } else {
    // ------------------------------------------------------------ out stores
    // Warp 11 stores each item's out tile, which the softmax warps stage
    // (bf16, 128-byte swizzled) in the item's query buffer, with TMA, and
    // then hands the buffer back to the producer.  Between items it zeroes
    // the backward's dq accumulator when asked, paced by the work counter so
    // that the stores spread over the launch.
    // Ring slots and staging barriers cannot run two phases ahead of this
    // warp: the producer publishes item k + 4, and the softmax warps
    // stage item k + 2, only after this warp has released item k's buffer.
    ZeroShare zs;
    if (p.zero_dst != nullptr) zs.init(p.zero_dst, p.zero_groups);
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int qb = k & 1;
      if (!(ok = mbar_wait_warp(BAR(C::BAR_ITEMFULL + (k & 3)), (k >> 2) & 1, ab))) break;
      const ItemGeom ig = *ring(k & 3);
      if (ig.item < 0) break;
      if (!(ok = mbar_wait_warp(BAR(C::BAR_OSTAGED + qb), (k >> 1) & 1, ab))) break;
      const uint32_t stage = sbase + C::kOffQ + qb * C::kQBytes;
      const HalfRows orr = half_rows<VARLEN>(ig.wi.b, ig.wi.half, ig.n, ig.row0);
      if (!VARLEN || ig.qs + BM <= ig.n) {
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < C::kOutChunks; ++c)
            tma_store_5d(&p.tm_o, stage + c * BM * 128, 64 * c, ig.wi.h, orr.base + ig.qs, orr.c3,
                         orr.c4);
          bulk_commit_group();
          bulk_wait_read_all();
          mbar_arrive(BAR(C::BAR_QEMPTY + qb));
        }
      } else {
        // Varlen, last tile of a half: a box store would run into the next
        // rows of the packed tensor, so the warp copies the half's rows out
        // of the staged (swizzled) tile with 16-byte stores.
        constexpr int kUnits = D / 8;  // 16-byte units per row
        const int rows = ig.n - ig.qs;
        __nv_bfloat16* dst0 = p.out + (static_cast<size_t>(orr.base + ig.qs) * p.H + ig.wi.h) * D;
        for (int idx = lane; idx < rows * kUnits; idx += 32) {
          const int r = idx / kUnits;
          const int u = idx - r * kUnits;
          uint32_t w0, w1, w2, w3;
          ld_shared_v4(stage + (u >> 3) * (BM * 128) + r * 128 + (((u & 7) ^ (r & 7)) << 4), w0,
                       w1, w2, w3);
          st_global_v4(dst0 + static_cast<size_t>(r) * p.H * D + 8 * u, w0, w1, w2, w3);
        }
        // The producer's next TMA load into this buffer follows these reads.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::BAR_QEMPTY + qb));
      }
      __syncwarp();
      if (p.zero_dst != nullptr) {
        unsigned taken = 0;
        if (lane == 0) taken = *reinterpret_cast<const volatile unsigned*>(p.sched);
        taken = __shfl_sync(0xffffffffu, taken, 0);
        zs.upto(static_cast<long long>(taken) + gridDim.x, num_items, lane);
      }
    }
    if (p.zero_dst != nullptr) zs.upto(1, 1, lane);
    if (lane == 0) bulk_wait_all();
    __syncwarp();
   }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegSoft));
    // ------------------------------------------------------------ softmax
    // Warp `warp`: rows [lb, lb + 16) of every tile of the item, lb = 32
    // (warp % 4) + 16 (warp / 4), the TMEM lanes of the half of its quarter;
    // thread t: row lb + t % 16, key columns [kCols h, kCols (h + 1)) of each
    // tile and head dims [kDCols h, kDCols (h + 1)) of O, h = t / 16.
    constexpr int KC = C::kCols;
    constexpr int DC = C::kDCols;
    const int w = lane >> 4;  // column half of the thread's row
    const int lb = (warp & 3) * 32 + (warp >> 2) * 16;
    const int row = lb + (lane & 15);
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(lb) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g = 0;  // tiles of earlier items
    for (int k = 0; ok; ++k) {
      if (!(ok = mbar_wait_warp(BAR(C::BAR_ITEMFULL + (k & 3)), (k >> 2) & 1, ab))) break;
      const ItemGeom ig = *ring(k & 3);
      if (ig.item < 0) break;
      const int qb = k & 1;  // query buffer of the item
      const int ob = k % C::kOBufs;
      const int qs = ig.qs;
      const int r = qs + row;  // row inside the half
      // Keys visible to row r, per segment of the item: computed once, so a
      // tile needs no division (rows past the end of the half see nothing).
      const int n = VARLEN ? ig.n : p.n;
      const int bs = VARLEN ? imin(p.bs, n) : p.bs;
      const Interval kv0 = key_interval(ig.rule0, r, n, bs);
      const Interval kv1 = key_interval(ig.rule1, r, n, bs);
      const uint32_t o_col = t_lane + C::kTmemO + ob * D;  // + DC w, through the split
      float m_ref = -INFINITY;  // reference maximum, scaled log2 units
      float l_run = 0.f;        // running sum of 2^(s * sl2 - m_ref) over this half's keys
      for (int j = 0; j < ig.ntiles; ++j) {
        const int gg = g + j;
        const int sb = gg % C::kSBufs;
        const int seg = j < ig.n0 ? 0 : 1;
        const int kt = ig.ktile(j);
        const uint32_t s_col = t_lane + C::kTmemS + sb * BN;  // + KC w, through the split
        if (!(ok = mbar_wait_warp(BAR(C::BAR_SFULL + sb), (gg / C::kSBufs) & 1, ab))) break;
        tc_fence_after();
        const int ks = kt * BN + KC * w;
        const Interval iv = seg ? kv1 : kv0;
        const int clo = iv.lo - ks, chi = iv.hi - ks;
        // The warp masks element by element only if one of its rows needs it.
        const bool full = __all_sync(0xffffffffu, clo <= 0 && chi >= KC);
        // The thread's half of the score row in registers; hidden keys ->
        // -inf, so they drop out of the maximum and get probability 0.
        uint32_t sr[KC];
#pragma unroll
        for (int c = 0; c < KC / 32; ++c) tmem_ld_half<32, KC>(s_col + 32 * c, sr + 32 * c);
        tmem_wait_ld();
        tmem_pin<KC>(sr);
        if (!full) {
          // Keys [clo, chi) of the part are visible to row r: a 32-bit mask
          // per 32 columns, hidden scores set to -inf with one AND / OR each,
          // in straight-line code.
#pragma unroll
          for (int c32 = 0; c32 < KC / 32; ++c32) {
            const int lo = clo - 32 * c32 < 0 ? 0 : (clo - 32 * c32 > 32 ? 32 : clo - 32 * c32);
            const int hi = chi - 32 * c32 < lo ? lo : (chi - 32 * c32 > 32 ? 32 : chi - 32 * c32);
            const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
            const uint32_t below_lo = lo >= 32 ? 0xffffffffu : ((1u << lo) - 1u);
            const uint32_t keep = below_hi & ~below_lo;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const uint32_t m = bit_spread(keep, e);
              sr[32 * c32 + e] = (sr[32 * c32 + e] & m) | (0xff800000u & ~m);
            }
          }
        }
        // The row's tile maximum over both halves: the two threads of the
        // row then take the same decision on the common reference maximum.
        const float mh = max_tree<KC>(sr);
        const float mall = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 16));
        const float m_tile = mall * sl2;
        const bool move = m_tile > m_ref + C::kRescaleThreshold;
        float corr = 1.f;
        if (move) {
          corr = ex2_approx(m_ref - m_tile);  // 0 while m_ref = -inf
          l_run *= corr;
          m_ref = m_tile;
        }
        // O holds the item's products of tiles 0 .. j - 1; once the last of
        // them has completed, each thread rescales its DC head dims of the
        // row (the row's other thread, deciding alike, takes the others).
        if (j >= 1 && __any_sync(0xffffffffu, move)) {
          const int gp = gg - 1;
          if (!(ok = mbar_wait_warp(BAR(C::BAR_SFREE + gp % C::kSBufs), (gp / C::kSBufs) & 1, ab)))
            break;
          tc_fence_after();
          constexpr int OW = DC < 32 ? DC : 32;  // columns per TMEM access
#pragma unroll
          for (int c = 0; c < DC / OW; ++c) {
            uint32_t o[OW];
            tmem_ld_half<OW, DC>(o_col + OW * c, o);
            tmem_wait_ld();
            tmem_pin<OW>(o);
#pragma unroll
            for (int e = 0; e < OW; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st_half<OW, DC>(o_col + OW * c, o);
          }
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        // Probabilities 2^(s * sl2 - m_use), two lanes per instruction for
        // the scaling and the sums (four independent pair accumulators),
        // written back as bf16 pairs (e4m3 quadruples) into the first half of
        // the columns of the thread's half row -- the scores there are
        // already in registers.
        const uint64_t scale2 = f2_pack(sl2, sl2);
        const uint64_t neg_m2 = f2_pack(-m_use, -m_use);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < KC / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[32 * c + 2 * e]),
                                              __uint_as_float(sr[32 * c + 2 * e + 1])),
                                      scale2, neg_m2);
            float x0, x1;
            f2_unpack(x, x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            acc[e & 3] = f2_add(acc[e & 3], f2_pack(p0, p1));
            if constexpr (FP8) {
              const uint32_t h = pack_e4m3x2(p0, p1);
              pk[e >> 1] = (e & 1) ? (pk[e >> 1] | (h << 16)) : h;
            } else {
              pk[e] = pack_bf16x2(p0, p1);
            }
          }
          if constexpr (FP8)
            tmem_st_half<8, KC>(s_col + 8 * c, pk);
          else
            tmem_st_half<16, KC>(s_col + 16 * c, pk);
        }
        float a0, a1, b0, b1;
        f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
        f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
        l_run += (a0 + a1) + (b0 + b1);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(BAR(C::BAR_PFULL + sb));
      }
      if (!ok) break;
      // ---------------------------------------------------------- read-out
      // Once the item's last P V has completed: the row sum of both halves,
      // then the thread's half of the head dims of its row of O, normalised,
      // as bf16 into the item's query buffer (its last S product has
      // completed) in the 128-byte-swizzled layout of a TMA box, for the
      // store warp; rows past the end of the half are dropped by the copy.
      if (ig.ntiles > 0) {
        const int gl = g + ig.ntiles - 1;
        if (!(ok = mbar_wait_warp(BAR(C::BAR_SFREE + gl % C::kSBufs), (gl / C::kSBufs) & 1, ab)))
          break;
      }
      tc_fence_after();
      const float lsum = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
      // FP8: out = (P V8) * v_descale / l
      const float inv = lsum > 0.f ? (FP8 ? p.out_scale : 1.f) / lsum : 0.f;
      const uint32_t stage = sbase + C::kOffQ + qb * C::kQBytes;
      constexpr int RW = DC < 32 ? DC : 32;  // columns per TMEM read
#pragma unroll
      for (int c = 0; c < DC / RW; ++c) {
        const int col = w * DC + RW * c;
        uint32_t oa[RW];
        tmem_ld_half<RW, DC>(o_col + RW * c, oa);
        tmem_wait_ld();
        tmem_pin<RW>(oa);
#pragma unroll
        for (int gq = 0; gq < RW / 8; ++gq) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = lsum > 0.f ? __uint_as_float(oa[gq * 8 + 2 * e]) * inv : 0.f;
            const float x1 = lsum > 0.f ? __uint_as_float(oa[gq * 8 + 2 * e + 1]) * inv : 0.f;
            wv[e] = pack_bf16x2(x0, x1);
          }
          const int unit = col / 8 + gq;  // 16-byte unit of the row
          st_shared_v4(stage + (unit >> 3) * (BM * 128) + row * 128 +
                           (((unit & 7) ^ (row & 7)) << 4),
                       wv[0], wv[1], wv[2], wv[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(BAR(C::BAR_OSTAGED + qb));
      if (r < n && w == 0) {
        const float lse =
            lsum > 0.f ? (m_ref + lg2_approx(lsum)) * 0.69314718055994531f : -INFINITY;
        if constexpr (VARLEN)
          p.lse[static_cast<size_t>(ig.wi.h) * p.rows + ig.row0 + ig.wi.half * ig.n + r] = lse;
        else
          p.lse[lse_offset(p.mode, ig.wi.b, ig.wi.h, ig.wi.half, r, p.H, p.n)] = lse;
      }
      tc_fence_before();
      mbar_arrive_warp(BAR(C::BAR_OFREE + ob));
      g += ig.ntiles;
    }
  }
#undef BAR

  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpPV) {
    if (lane == 0) mbar_wait_limited(sbase + C::kOffBar + 8 * C::BAR_ALL, 0, 1000000000ull);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0) sched_finish(p.sched);
}

template <int D, int STAGES, int VSTAGES, bool VARLEN, bool FP8 = false>
static cudaError_t launch_fwd2_impl(const FwdParams& p, cudaStream_t stream) {
  using C = Fwd2Cfg<D, STAGES, VSTAGES, FP8>;
  auto kern = dfa_fwd2_kernel<D, STAGES, VSTAGES, VARLEN, FP8>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The setmaxnreg split must fit the registers the kernel is launched with,
  // or the softmax warps' increase would never be granted: refuse to launch.
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs * C::kThreads < C::kRegCtl * 128 + C::kRegSoft * 32 * C::kSoftWarps)
    return cudaErrorInvalidConfiguration;
  const long long items = VARLEN ? p.items : pass_items(p.mode, p.B, p.H, p.q_tiles);
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const long long grid = items < sms ? items : sms;
  return launch_chained(kern, dim3(static_cast<unsigned>(grid)), dim3(C::kThreads), C::kSmemBytes,
                        stream, p);
}

// FP8 (e4m3) q, k, v, headdim 128: smaller K / V tiles, so more stages.
cudaError_t launch_forward_fp8(const FwdParams& p, int headdim, cudaStream_t stream) {
  if (headdim != 128 || p.vl) return cudaErrorInvalidValue;
  return launch_fwd2_impl<128, 5, 4, false, true>(p, stream);
}

// K / V stages per head dimension: as many K tiles in flight as the shared
// memory holds beside two query tiles and the V ring.
cudaError_t launch_forward_persistent(const FwdParams& p, int headdim, cudaStream_t stream) {
  switch (headdim) {
    case 64:
      return p.vl ? launch_fwd2_impl<64, 6, 4, true>(p, stream)
                  : launch_fwd2_impl<64, 6, 4, false>(p, stream);
    case 128:
      return p.vl ? launch_fwd2_impl<128, 3, 2, true>(p, stream)
                  : launch_fwd2_impl<128, 3, 2, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfa
