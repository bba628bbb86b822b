// Backward kernel of block-diffusion attention on sm_103a.
//
// Recompute-based backward of "FlashAttention: Exact Attention Without
// Materialization", section 4.5: from q, k, v, dout, the forward's
// log-sum-exp and D = rowsum(dout * out), recompute the probabilities on
// chip and accumulate the gradients.  Key-tile major: one CTA owns one
// 128-key tile of one half of one (batch, head), keeps its K and V in shared
// memory and its dK and dV accumulators in TMEM, and walks exactly the query
// tiles that see it ("Fast Diffusion Attention", "Visit only the visible
// tiles"): a clean key tile is seen by the clean queries of its block onward
// and by the noisy queries of the later blocks; a noisy key tile only by the
// noisy queries of its own blocks.
//
// Per query tile i (tensor cores, accumulators in TMEM), b = i % 2:
//   S^T  = K Q^T                    -> TMEM S[b]
//   dP^T = V dO^T                   -> TMEM dP[b] (one buffer for d = 64)
//   P^T  = exp(scale S^T - LSE)  (0 on hidden pairs), dS^T = P^T (dP^T - D)
//        written back as bf16 into the columns of dP, dS^T also to shared
//   dV  += P^T dO,  dK += dS^T Q    (A operand read from TMEM)
//   dQ   = dS K                     -> TMEM S[b] (S is consumed by then),
//        then added to a float32 accumulator in device memory.
// Warp roles (384 threads): two compute warpgroups, warpgroup b handling the
// query tiles i with i % 2 == b (thread t of a warpgroup owns key row t of
// the tile, TMEM lane t), so that the MMAs of one tile overlap the
// softmax-gradient work of the other; warp 8 loads (TMA for Q/dO, plain loads
// for LSE/D); warp 9 issues the MMAs; warps 10-11 idle.  The load/MMA
// warpgroup drops to 72 registers and the compute warpgroups rise to 216
// (setmaxnreg; launched with 168: 256 * 48 == 128 * 96), so a 64-query
// slice of S^T and dP^T is read from TMEM in one batch.
#include <cuda_bf16.h>

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
  // dP^T is double-buffered when TMEM has room (headdim 128); with headdim
  // 64 the 128-query tiles leave room for one buffer only.
  static constexpr int kDPBufs = (2 * BMQ + 2 * BMQ + 2 * D <= 512) ? 2 : 1;
  enum {
    BAR_KV = 0,
    BAR_QFULL = 1,
    BAR_QEMPTY = BAR_QFULL + STAGES,
    BAR_SFULL = BAR_QEMPTY + STAGES,  // [2] per tile parity
    BAR_DPFULL = BAR_SFULL + 2,       // [2]
    BAR_PDS = BAR_DPFULL + 2,         // [2]
    BAR_MMA2 = BAR_PDS + 2,           // [2]
    BAR_DQFREE = BAR_MMA2 + 2,        // [2]
    BAR_ALL = BAR_DQFREE + 2,         // every MMA done (epilogue, drain)
    NUM_BARS = BAR_ALL + 1
  };
  static constexpr int kOffTmemSlot = kOffBar + NUM_BARS * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;
  // dQ is computed transposed (rows = head dims) when headdim = 128, so that
  // each warp's float atomics cover 32 consecutive head dims of one query;
  // with headdim 64 it is computed as (queries x head dims).
  static constexpr bool kDqTransposed = (D == 128);
  static constexpr int kTmemS = 0;                     // S[b] at b * BMQ
  static constexpr int kTmemDP = 2 * BMQ;              // dP[b] at kTmemDP + b * BMQ
  static constexpr int kTmemDK = kTmemDP + kDPBufs * BMQ;
  static constexpr int kTmemDV = kTmemDK + D;
  static constexpr int kDqCols = kDqTransposed ? BMQ : D;
  static constexpr int kTmemCols = 512;
  static constexpr int kThreads = 384;
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;
  static_assert(kTmemDV + D <= kTmemCols, "TMEM budget");
  static_assert(kDqCols <= BMQ, "dQ must fit in an S buffer");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kDqTransposed ? (D == 128) : (BMQ == 128), "dQ MMA needs M = 128");
  static_assert(BMQ % 32 == 0, "query tile");
};

template <int D, int BMQ>
__global__ void __launch_bounds__(384, 1) dfa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D, BMQ>;
  constexpr int BN = C::BN;
  constexpr int STAGES = C::STAGES;
  constexpr int DPB = C::kDPBufs;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  const AbortFlag ab{abort_flag, p.status};
#define BAR(i) (sbase + C::kOffBar + 8 * (i))

  const WorkItem wi = bwd_work(blockIdx.x, p.mode, p.B, p.H, p.k_tiles, p.group);
  Segment seg[2];
  const int nseg = bwd_segments(p.mode, p.n, p.bs, BMQ, BN, wi.half, wi.tile, seg);
  const int n0 = nseg > 0 ? seg[0].t_end - seg[0].t_begin : 0;
  const int ntiles = n0 + (nseg > 1 ? seg[1].t_end - seg[1].t_begin : 0);
  const int ks = wi.tile * BN;
  const size_t L = 2 * static_cast<size_t>(p.n);

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::BAR_KV), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(BAR(C::BAR_QFULL + s), 1);
      mbar_init(BAR(C::BAR_QEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(C::BAR_SFULL + b), 1);
      mbar_init(BAR(C::BAR_DPFULL + b), 1);
      mbar_init(BAR(C::BAR_PDS + b), 128);
      mbar_init(BAR(C::BAR_MMA2 + b), 1);
      mbar_init(BAR(C::BAR_DQFREE + b), 128);
    }
    mbar_init(BAR(C::BAR_ALL), 1);
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

  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
   if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(BAR(C::BAR_KV), 2 * C::kKVBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_5d(sbase + C::kOffK + c * BN * 128, &p.tm_k, BAR(C::BAR_KV), 64 * c, wi.h, ks,
                    wi.half, wi.b);
        tma_load_5d(sbase + C::kOffV + c * BN * 128, &p.tm_v, BAR(C::BAR_KV), 64 * c, wi.h, ks,
                    wi.half, wi.b);
      }
    }
    __syncwarp();
    const float* del_bh = p.delta + (static_cast<size_t>(wi.b) * p.H + wi.h) * L;
    // LSE and D of a query tile are read into registers one tile ahead, so
    // that their latency overlaps the wait for a free stage.
    constexpr int kPerLane = BMQ / 32;
    float lse_r[kPerLane], del_r[kPerLane];
    auto load_rows = [&](int it) {
      const int s = it < n0 ? 0 : 1;
      const int qt = seg[s].t_begin + (s ? it - n0 : it);
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) {
        const int q = qt * BMQ + lane + 32 * e;
        const bool valid = q < p.n;
        const size_t pos = static_cast<size_t>(seg[s].half) * p.n + q;
        // Stored negated: -LSE * log2(e) and -D, the addends of the packed
        // arithmetic below.  Rows past the half: probability 0.
        lse_r[e] = valid ? p.lse[lse_offset(p.mode, wi.b, wi.h, seg[s].half, q, p.H, p.n)] *
                               -1.4426950408889634f
                         : -INFINITY;
        del_r[e] = valid ? -del_bh[pos] : 0.f;
      }
    };
    if (ntiles > 0) load_rows(0);
    bool ok = true;
    int i = 0;
    for (; i < ntiles && ok; ++i) {
      const int s = i < n0 ? 0 : 1;
      const int qt = seg[s].t_begin + (s ? i - n0 : i);
      const int st = i % STAGES;
      const int round = i / STAGES;
      if (round > 0) {
        int w = 0;
        if (lane == 0) w = mbar_wait(BAR(C::BAR_QEMPTY + st), (round - 1) & 1, ab) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        if (!ok) break;
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
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_5d(sbase + C::kOffQ + st * C::kQBytes + c * BMQ * 128, &p.tm_q,
                      BAR(C::BAR_QFULL + st), 64 * c, wi.h, qt * BMQ, seg[s].half, wi.b);
          tma_load_5d(sbase + C::kOffDO + st * C::kQBytes + c * BMQ * 128, &p.tm_do,
                      BAR(C::BAR_QFULL + st), 64 * c, wi.h, qt * BMQ, seg[s].half, wi.b);
        }
      }
      __syncwarp();
      if (i + 1 < ntiles) load_rows(i + 1);
    }
    if (!ok && lane == 0) {
      mbar_wait_limited(BAR(C::BAR_KV), 0, 100000000ull);
      for (int t = (i > STAGES ? i - STAGES : 0); t < i; ++t)
        mbar_wait_limited(BAR(C::BAR_QFULL + t % STAGES), (t / STAGES) & 1, 100000000ull);
    }
    __syncwarp();
   } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(BN, BMQ, false, false);      // K Q^T, V dO^T
      constexpr uint32_t kIdKV = idesc_bf16(BN, D, false, true);        // P^T dO, dS^T Q
      constexpr uint32_t kIdDQ = C::kDqTransposed ? idesc_bf16(D, BMQ, true, true)   // K^T dS^T
                                                  : idesc_bf16(BMQ, D, true, true);  // dS K
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
      bool ok = mbar_wait(BAR(C::BAR_KV), 0, ab);

      auto issue_dp = [&](int i) {
        const uint32_t st_off = (i % STAGES) * C::kQBytes;
        const uint32_t d_dp = tmem + C::kTmemDP + (DPB == 2 ? (i & 1) * BMQ : 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
          mma_ss(d_dp, adv(dV_kmaj, koff), adv(dO_kmaj, st_off + qoff), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(C::BAR_DPFULL + (i & 1)));
      };
      // dV, dK and dQ of tile j, once its P^T / dS^T are in place.
      auto issue_second = [&](int j) -> bool {
        const int b = j & 1;
        const uint32_t st_off = (j % STAGES) * C::kQBytes;
        if (!mbar_wait(BAR(C::BAR_PDS + b), (j >> 1) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t pds = tmem + C::kTmemDP + (DPB == 2 ? b * BMQ : 0);
#pragma unroll
        for (int kk = 0; kk < BMQ / 16; ++kk) {
          // P^T / dS^T of queries [16kk, 16kk+16): columns of 32-query chunk
          // kk/2, P^T in its first 16 columns, dS^T in its last 16.
          const uint32_t col = 32 * (kk >> 1) + 8 * (kk & 1);
          const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tmem + C::kTmemDV, pds + col, adv(dO_mn, st_off + kk * 16 * 128), kIdKV, acc);
          mma_ts(tmem + C::kTmemDK, pds + col + 16, adv(dQ_mn, st_off + kk * 16 * 128), kIdKV,
                 acc);
        }
        const uint32_t ds_off = b * C::kDSBytes;
        const uint32_t d_dq = tmem + C::kTmemS + b * BMQ;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t kdesc = adv(dK_mn, kk * 16 * 128);
          const uint64_t sdesc = adv(dDS_mn, ds_off + kk * 16 * 128);
          if (C::kDqTransposed)
            mma_ss(d_dq, kdesc, sdesc, kIdDQ, kk > 0 ? 1u : 0u);
          else
            mma_ss(d_dq, sdesc, kdesc, kIdDQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(C::BAR_MMA2 + b));
        mma_commit(BAR(C::BAR_QEMPTY + (j % STAGES)));
        return true;
      };

      for (int i = 0; i < ntiles && ok; ++i) {
        const int b = i & 1;
        const int st = i % STAGES;
        if (!(ok = mbar_wait(BAR(C::BAR_QFULL + st), (i / STAGES) & 1, ab))) break;
        // S[b] held dQ of tile i-2: wait until it has been read out.
        if (i >= 2 && !(ok = mbar_wait(BAR(C::BAR_DQFREE + b), ((i - 2) >> 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t st_off = st * C::kQBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
          mma_ss(tmem + C::kTmemS + b * BMQ, adv(dK_kmaj, koff), adv(dQ_kmaj, st_off + qoff), kIdS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(C::BAR_SFULL + b));
        if (DPB == 2) {
          issue_dp(i);
          if (i >= 1 && !(ok = issue_second(i - 1))) break;
        } else {
          // One dP buffer: it still holds P^T / dS^T of tile i-1 until the
          // dV / dK products of tile i-1 have been issued.
          if (i >= 1 && !(ok = issue_second(i - 1))) break;
          issue_dp(i);
        }
      }
      if (ok && ntiles > 0) issue_second(ntiles - 1);
      // Every MMA is complete when BAR_ALL fires (epilogue; TMEM release).
      mma_commit(BAR(C::BAR_ALL));
    }
    __syncwarp();
   }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;");
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2;            // this warpgroup handles tiles i % 2 == wg
    const int row = (warp & 3) * 32 + lane;  // key row of the tile / TMEM lane
    const int j = ks + row;                  // key inside its half
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;

    // Read dQ of tile `it` out of TMEM S[it%2] and add it to dq_acc.
    auto drain_dq = [&](int it) -> bool {
      const int b = it & 1;
      if (!mbar_wait_warp(BAR(C::BAR_MMA2 + b), (it >> 1) & 1, ab)) return false;
      tc_fence_after();
      const int s = it < n0 ? 0 : 1;
      const int qt = seg[s].t_begin + (s ? it - n0 : it);
      const int qh = seg[s].half;
      const int qs = qt * BMQ;
      const uint32_t src = t_lane + C::kTmemS + b * BMQ;
      if (C::kDqTransposed) {
        // TMEM lane = head dim `row`; columns = queries of the tile.
        uint32_t dq[BMQ];
#pragma unroll
        for (int c = 0; c < BMQ / 32; ++c) tmem_ld32(src + 32 * c, dq + 32 * c);
        tmem_wait_ld();
        tmem_pin<BMQ>(dq);
        tc_fence_before();
        mbar_arrive(BAR(C::BAR_DQFREE + b));
        const size_t stride = static_cast<size_t>(p.H) * D;
        float* ptr = p.dq_acc + ((static_cast<size_t>(wi.b) * L + static_cast<size_t>(qh) * p.n +
                                  qs) * p.H + wi.h) * D + row;
        if (qs + BMQ <= p.n) {
#pragma unroll
          for (int c = 0; c < BMQ; ++c) {
            red_add_f32(ptr, __uint_as_float(dq[c]) * p.scale);
            ptr += stride;
          }
        } else {
          const int qmax = p.n - qs;
#pragma unroll
          for (int c = 0; c < BMQ; ++c) {
            if (c < qmax) red_add_f32(ptr, __uint_as_float(dq[c]) * p.scale);
            ptr += stride;
          }
        }
      } else {
        // TMEM lane = query `row` of the tile; columns = head dims.
        uint32_t dq[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(src + 32 * c, dq + 32 * c);
        tmem_wait_ld();
        tmem_pin<D>(dq);
        tc_fence_before();
        mbar_arrive(BAR(C::BAR_DQFREE + b));
        const int q = qs + row;
        if (q < p.n) {
          float* dst = p.dq_acc + ((static_cast<size_t>(wi.b) * L + static_cast<size_t>(qh) * p.n +
                                    q) * p.H + wi.h) * D;
#pragma unroll
          for (int c = 0; c < D; c += 4)
            red_add_v4_f32(dst + c, __uint_as_float(dq[c]) * p.scale,
                           __uint_as_float(dq[c + 1]) * p.scale,
                           __uint_as_float(dq[c + 2]) * p.scale,
                           __uint_as_float(dq[c + 3]) * p.scale);
        }
      }
      return true;
    };

    // P^T and dS^T of one 64-query slice h: S^T and dP^T in (one batch of
    // TMEM loads), bf16 P^T / dS^T back into the dP columns of each 32-query
    // chunk (P^T in its first 16 columns, dS^T in its last 16), dS^T also into
    // the swizzled shared tile.  Pairs of columns go through packed f32x2
    // arithmetic: x = s * sl2 - lse2, p = 2^x, ds = p * (dp - D).
    auto slice = [&](auto masked, int h, uint32_t s_col, uint32_t dp_col, uint32_t ds_s,
                     const float* nlse_s, const float* ndel_s, int qs, Interval iv) {
      uint32_t sr[64], dpr[64];
      tmem_ld32(s_col + 64 * h, sr);
      tmem_ld32(s_col + 64 * h + 32, sr + 32);
      tmem_ld32(dp_col + 64 * h, dpr);
      tmem_ld32(dp_col + 64 * h + 32, dpr + 32);
      tmem_wait_ld();
      tmem_pin<64>(sr);
      tmem_pin<64>(dpr);
      const uint64_t scale2 = f2_pack(sl2, sl2);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int cbase = 64 * h + 32 * cc;  // first query column of the chunk
        uint32_t wp[16], wd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int cl = 32 * cc + 2 * e;  // column inside the slice
          const float2 nl = *reinterpret_cast<const float2*>(nlse_s + cbase + 2 * e);
          const float2 nd = *reinterpret_cast<const float2*>(ndel_s + cbase + 2 * e);
          const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[cl]), __uint_as_float(sr[cl + 1])),
                                    scale2, f2_pack(nl.x, nl.y));
          float x0, x1;
          f2_unpack(x, x0, x1);
          float p0 = ex2_approx(x0);
          float p1 = ex2_approx(x1);
          if (decltype(masked)::value) {
            const int q = qs + cbase + 2 * e;
            if (q < iv.lo || q >= iv.hi) p0 = 0.f;
            if (q + 1 < iv.lo || q + 1 >= iv.hi) p1 = 0.f;
          }
          const uint64_t pp = f2_pack(p0, p1);
          const uint64_t dd =
              f2_add(f2_pack(__uint_as_float(dpr[cl]), __uint_as_float(dpr[cl + 1])),
                     f2_pack(nd.x, nd.y));
          float d0, d1;
          f2_unpack(f2_mul(pp, dd), d0, d1);
          wp[e] = pack_bf16x2(p0, p1);
          wd[e] = pack_bf16x2(d0, d1);
        }
        const int chunk = 2 * h + cc;
        tmem_st16(dp_col + 32 * chunk, wp);
        tmem_st16(dp_col + 32 * chunk + 16, wd);
        const int a = chunk >> 1;  // 64-column swizzle atom
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const int u = (chunk & 1) * 4 + u4;  // 16-byte unit inside the row
          const uint32_t off = a * (BN * 128) + row * 128 + ((u ^ (row & 7)) << 4);
          st_shared_v4(ds_s + off, wd[4 * u4], wd[4 * u4 + 1], wd[4 * u4 + 2], wd[4 * u4 + 3]);
        }
      }
    };

    for (int i = wg; i < ntiles && ok; i += 2) {
      const int s = i < n0 ? 0 : 1;
      const int qt = seg[s].t_begin + (s ? i - n0 : i);
      const int st = i % STAGES;
      const int b = i & 1;
      const int dpb = DPB == 2 ? b : 0;
      if (!(ok = mbar_wait_warp(BAR(C::BAR_SFULL + b), (i >> 1) & 1, ab))) break;
      if (!(ok = mbar_wait_warp(BAR(C::BAR_DPFULL + b), (i >> 1) & 1, ab))) break;
      tc_fence_after();

      const float* lse_s = reinterpret_cast<const float*>(smem + C::kOffLSE) + st * BMQ;
      const float* del_s = reinterpret_cast<const float*>(smem + C::kOffDEL) + st * BMQ;
      const int qs = qt * BMQ;
      const bool full = tile_full(seg[s].rule, p.n, p.bs, qs, BMQ, ks, BN);
      const Interval iv = query_interval(seg[s].rule, j, p.n, p.bs);
      const uint32_t s_col = t_lane + C::kTmemS + b * BMQ;
      const uint32_t dp_col = t_lane + C::kTmemDP + dpb * BMQ;
      const uint32_t ds_s = sbase + C::kOffDS + b * C::kDSBytes;
      if (full) {
#pragma unroll 1
        for (int h = 0; h < BMQ / 64; ++h)
          slice(std::false_type{}, h, s_col, dp_col, ds_s, lse_s, del_s, qs, iv);
      } else {
#pragma unroll 1
        for (int h = 0; h < BMQ / 64; ++h)
          slice(std::true_type{}, h, s_col, dp_col, ds_s, lse_s, del_s, qs, iv);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(C::BAR_PDS + b));

      if (!(ok = drain_dq(i))) break;
    }

    // ------------------------------------------------------------ epilogue
    // Warpgroup 0 writes dV, warpgroup 1 writes dK, once every MMA is done.
    if (ok) ok = mbar_wait_warp(BAR(C::BAR_ALL), 0, ab);
    tc_fence_after();
    if (ok) {
      const bool valid = j < p.n;
      const size_t pos = static_cast<size_t>(wi.half) * p.n + j;
      const size_t off = ((static_cast<size_t>(wi.b) * L + pos) * p.H + wi.h) * D;
      __nv_bfloat16* dst = (wg == 0 ? p.dv : p.dk) + off;
      const float mul = wg == 0 ? 1.f : p.scale;
      const uint32_t col = wg == 0 ? C::kTmemDV : C::kTmemDK;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (ntiles > 0) {
          tmem_ld32(t_lane + col + 32 * c, o);
          tmem_wait_ld();
          tmem_pin<32>(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[g * 8 + 2 * e]) * mul,
                                 __uint_as_float(o[g * 8 + 2 * e + 1]) * mul);
            st_global_v4(dst + 32 * c + 8 * g, w[0], w[1], w[2], w[3]);
          }
        }
      }
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
}

template <int D, int BMQ>
static cudaError_t launch_bwd_impl(const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D, BMQ>;
  auto kern = dfa_bwd_kernel<D, BMQ>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long blocks = 2LL * p.B * p.H * p.k_tiles;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(blocks), C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_backward(const BwdParams& p, int headdim, cudaStream_t stream) {
  switch (headdim) {
    case 64: return launch_bwd_impl<64, 128>(p, stream);
    case 128: return launch_backward_d128(p, stream);
    case 256: return launch_backward_d256(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfa
