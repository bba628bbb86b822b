// Backward kernel of block-diffusion attention, headdim 128 and 256, on sm_103a.
//
// Recompute-based backward of "FlashAttention: Exact Attention Without
// Materialization", section 4.5.  Key-tile major: one CTA owns one 128-key
// tile of one half of one (batch, head), keeps K and V in shared memory and
// the dK and dV accumulators in TMEM, and walks exactly the 64-query tiles
// that see it ("Fast Diffusion Attention", "Visit only the visible tiles").
//
// Per query tile i (tensor cores, accumulators in TMEM):
//   S^T  = K Q^T     -> TMEM S        dP^T = V dO^T   -> TMEM dP
//   P^T  = exp(scale S^T - LSE) (0 on hidden pairs),  dS^T = P^T (dP^T - D)
//        bf16 P^T / dS^T -> TMEM PdS, dS^T also -> shared memory
//   dV  += P^T dO,  dK += dS^T Q       (A operand read from TMEM PdS)
//   dQ^T = K^T dS^T  -> TMEM DQ, then added to a float32 accumulator in
//        device memory (each warp covers 32 consecutive head dims of a query)
// TMEM (512 columns): S 64 | dP 64 | PdS 64 | DQ 64 | dK 128 | dV 128.
// With headdim 256 the dK and dV accumulators of all head dims would need
// every TMEM column, so each CTA takes one 128-wide half of the head
// dimension of its key tile: it recomputes S^T and dP^T in full (their
// contraction runs over all 256 dims) and accumulates dK, dV and dQ for its
// half only; the two halves of a key tile are neighbouring CTAs.  K and V
// (128 KB) then leave room for a single Q / dO stage.
// Two compute warpgroups take alternate query tiles.  A warpgroup releases S
// and dP as soon as it has read them into registers, so the scores of the
// next tile are computed while it works; P^T / dS^T and dQ have TMEM columns
// of their own, so no product waits for a read-out it does not need.
// Warps 0-7 compute, warp 8 loads, warp 9 issues MMAs, warps 10-11 idle; the
// load/MMA warpgroup drops to 136 registers and the compute warpgroups rise
// to 184 (setmaxnreg; launched with 168: 256 * 16 == 128 * 32).
#include <cuda_bf16.h>

#include "geometry.cuh"
#include "params.cuh"
#include "sm100.cuh"

namespace dfa {

template <int D_, int STAGES_>
struct Bwd2Cfg {
  static constexpr int D = D_;
  static constexpr int DH = 128;       // head dims accumulated per CTA
  static constexpr int NDH = D / DH;   // CTAs per key tile
  static constexpr int BN = 128;  // keys per tile (MMA M)
  static constexpr int BMQ = 64;  // queries per tile
  static constexpr int STAGES = STAGES_;
  static constexpr int kChunks = D / 64;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kQBytes = BMQ * D * 2;
  static constexpr int kDSBytes = BN * BMQ * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVBytes;
  static constexpr int kOffQ = kOffV + kKVBytes;
  static constexpr int kOffDO = kOffQ + STAGES * kQBytes;
  static constexpr int kOffDS = kOffDO + STAGES * kQBytes;
  static constexpr int kOffLSE = kOffDS + kDSBytes;           // STAGES x BMQ floats
  static constexpr int kOffDEL = kOffLSE + STAGES * BMQ * 4;  // STAGES x BMQ floats
  static constexpr int kOffBar = kOffDEL + STAGES * BMQ * 4;
  enum {
    BAR_KV = 0,
    BAR_QFULL = 1,
    BAR_QEMPTY = BAR_QFULL + STAGES,
    // S^T and dP^T of a tile computed; one barrier per warpgroup, so that a
    // warpgroup never waits for a phase two ahead of the last one it saw.
    BAR_SDPFULL = BAR_QEMPTY + STAGES,  // [2]
    BAR_SDPFREE = BAR_SDPFULL + 2,      // S^T / dP^T read into registers
    BAR_PDSFULL = BAR_SDPFREE + 1,      // P^T / dS^T of a tile in place
    BAR_MMA2 = BAR_PDSFULL + 1,         // dV, dK, dQ of a tile done
    BAR_DQFREE = BAR_MMA2 + 1,          // dQ of a tile read out of TMEM
    BAR_ALL = BAR_DQFREE + 1,           // every MMA of the CTA done
    NUM_BARS = BAR_ALL + 1
  };
  static constexpr int kOffTmemSlot = kOffBar + NUM_BARS * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;
  static constexpr int kTmemS = 0;
  static constexpr int kTmemDP = 64;
  static constexpr int kTmemPDS = 128;
  static constexpr int kTmemDQ = 192;
  static constexpr int kTmemDK = 256;
  static constexpr int kTmemDV = 384;
  static constexpr int kTmemCols = 512;
  static constexpr int kThreads = 384;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int D_, int STAGES_>
__global__ void __launch_bounds__(384, 1) dfa_bwd2_kernel(const __grid_constant__ BwdParams p) {
  using C = Bwd2Cfg<D_, STAGES_>;
  constexpr int DH = C::DH;
  constexpr int D = C::D;
  constexpr int BN = C::BN;
  constexpr int BMQ = C::BMQ;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  const AbortFlag ab{abort_flag, p.status};
#define BAR(i) (sbase + C::kOffBar + 8 * (i))

  const int dh = blockIdx.x % C::NDH;  // head-dim half of this CTA
  const WorkItem wi = bwd_work(blockIdx.x / C::NDH, p.mode, p.B, p.H, p.k_tiles, p.group);
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
    mbar_init(BAR(C::BAR_SDPFULL), 1);
    mbar_init(BAR(C::BAR_SDPFULL + 1), 1);
    mbar_init(BAR(C::BAR_SDPFREE), 128);
    mbar_init(BAR(C::BAR_PDSFULL), 128);
    mbar_init(BAR(C::BAR_MMA2), 1);
    mbar_init(BAR(C::BAR_DQFREE), 128);
    mbar_init(BAR(C::BAR_ALL), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(sbase + C::kOffTmemSlot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::kOffTmemSlot);

  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 136;");
   if (warp == 8) {
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
    // -LSE * log2(e) and -D of a query tile, read one tile ahead.
    float lse_r[2], del_r[2];
    auto load_rows = [&](int it) {
      const int s = it < n0 ? 0 : 1;
      const int qt = seg[s].t_begin + (s ? it - n0 : it);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int q = qt * BMQ + lane + 32 * e;
        const bool valid = q < p.n;
        const size_t pos = static_cast<size_t>(seg[s].half) * p.n + q;
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
      for (int e = 0; e < 2; ++e) {
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
   } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(BN, BMQ, false, false);  // K Q^T, V dO^T
      constexpr uint32_t kIdKV = idesc_bf16(BN, DH, false, true);   // P^T dO, dS^T Q
      constexpr uint32_t kIdDQ = idesc_bf16(DH, BMQ, true, true);   // K^T dS^T
      const uint64_t dK_kmaj = sdesc_sw128(sbase + C::kOffK, 16, 1024);
      const uint64_t dV_kmaj = sdesc_sw128(sbase + C::kOffV, 16, 1024);
      // The head-dim half dh starts at 64-wide chunk 2 dh of K, Q and dO.
      const uint64_t dK_mn = sdesc_sw128(sbase + C::kOffK + dh * 2 * (BN * 128), BN * 128, 1024);
      const uint64_t dQ_kmaj = sdesc_sw128(sbase + C::kOffQ, 16, 1024);
      const uint64_t dO_kmaj = sdesc_sw128(sbase + C::kOffDO, 16, 1024);
      const uint64_t dQ_mn =
          sdesc_sw128(sbase + C::kOffQ + dh * 2 * (BMQ * 128), BMQ * 128, 1024);
      const uint64_t dO_mn =
          sdesc_sw128(sbase + C::kOffDO + dh * 2 * (BMQ * 128), BMQ * 128, 1024);
      const uint64_t dDS_mn = sdesc_sw128(sbase + C::kOffDS, BN * 128, 1024);
      auto adv = [](uint64_t d, uint32_t bytes) { return d + static_cast<uint64_t>(bytes >> 4); };
      bool ok = mbar_wait(BAR(C::BAR_KV), 0, ab);

      // dV, dK, dQ of tile j, once its P^T / dS^T are in place.
      auto issue_second = [&](int j) -> bool {
        const uint32_t st_off = (j % STAGES) * C::kQBytes;
        if (!mbar_wait(BAR(C::BAR_PDSFULL), j & 1, ab)) return false;
        tc_fence_after();
        const uint32_t pds = tmem + C::kTmemPDS;
#pragma unroll
        for (int kk = 0; kk < BMQ / 16; ++kk) {
          // queries [16kk, 16kk+16): chunk kk/2, P^T first 16 columns, dS^T last 16
          const uint32_t col = 32 * (kk >> 1) + 8 * (kk & 1);
          const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tmem + C::kTmemDV, pds + col, adv(dO_mn, st_off + kk * 16 * 128), kIdKV, acc);
          mma_ts(tmem + C::kTmemDK, pds + col + 16, adv(dQ_mn, st_off + kk * 16 * 128), kIdKV,
                 acc);
        }
        // The DQ columns still hold dQ of tile j-1 until it has been read out.
        if (j >= 1 && !mbar_wait(BAR(C::BAR_DQFREE), (j - 1) & 1, ab)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ss(tmem + C::kTmemDQ, adv(dK_mn, kk * 16 * 128), adv(dDS_mn, kk * 16 * 128), kIdDQ,
                 kk > 0 ? 1u : 0u);
        mma_commit(BAR(C::BAR_MMA2));
        mma_commit(BAR(C::BAR_QEMPTY + (j % STAGES)));
        return true;
      };

      for (int i = 0; i < ntiles && ok; ++i) {
        const int st = i % STAGES;
        // With a single Q / dO stage, tile i can only be loaded once the
        // products of tile i-1 (the stage's last readers) are issued.
        if (STAGES == 1 && i >= 1 && !(ok = issue_second(i - 1))) break;
        if (!(ok = mbar_wait(BAR(C::BAR_QFULL + st), (i / STAGES) & 1, ab))) break;
        // S and dP are free once the previous tile's warpgroup has read them.
        if (i >= 1 && !(ok = mbar_wait(BAR(C::BAR_SDPFREE), (i - 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t st_off = st * C::kQBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
          mma_ss(tmem + C::kTmemS, adv(dK_kmaj, koff), adv(dQ_kmaj, st_off + qoff), kIdS,
                 kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
          mma_ss(tmem + C::kTmemDP, adv(dV_kmaj, koff), adv(dO_kmaj, st_off + qoff), kIdS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(C::BAR_SDPFULL + (i & 1)));
        if (STAGES > 1 && i >= 1 && !(ok = issue_second(i - 1))) break;
      }
      if (ok && ntiles > 0) issue_second(ntiles - 1);
      mma_commit(BAR(C::BAR_ALL));
    }
    __syncwarp();
   }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2;                // this warpgroup handles tiles i % 2 == wg
    const int row = (warp & 3) * 32 + lane;  // key row of the tile / TMEM lane
    const int j = ks + row;                  // key inside its half
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    const uint64_t scale2 = f2_pack(sl2, sl2);
    bool ok = true;
    for (int i = wg; i < ntiles && ok; i += 2) {
      const int s = i < n0 ? 0 : 1;
      const int qt = seg[s].t_begin + (s ? i - n0 : i);
      const int qh = seg[s].half;
      const int st = i % STAGES;
      const int qs = qt * BMQ;
      if (!(ok = mbar_wait_warp(BAR(C::BAR_SDPFULL + (i & 1)), (i >> 1) & 1, ab))) break;
      tc_fence_after();
      uint32_t sr[BMQ], dpr[BMQ];
      tmem_ld32(t_lane + C::kTmemS, sr);
      tmem_ld32(t_lane + C::kTmemS + 32, sr + 32);
      tmem_ld32(t_lane + C::kTmemDP, dpr);
      tmem_ld32(t_lane + C::kTmemDP + 32, dpr + 32);
      tmem_wait_ld();
      tmem_pin<BMQ>(sr);
      tmem_pin<BMQ>(dpr);
      tc_fence_before();
      mbar_arrive(BAR(C::BAR_SDPFREE));

      const float* nlse_s = reinterpret_cast<const float*>(smem + C::kOffLSE) + st * BMQ;
      const float* ndel_s = reinterpret_cast<const float*>(smem + C::kOffDEL) + st * BMQ;
      const bool full = tile_full(seg[s].rule, p.n, p.bs, qs, BMQ, ks, BN);
      const Interval iv = query_interval(seg[s].rule, j, p.n, p.bs);
      // P^T and dS^T in packed pairs: x = s * sl2 - lse2, p = 2^x,
      // ds = p * (dp - D); bf16 pairs packed two chunks of 16 words each.
      uint32_t wp[BMQ / 2], wd[BMQ / 2];
#pragma unroll
      for (int e = 0; e < BMQ / 2; ++e) {
        const float2 nl = *reinterpret_cast<const float2*>(nlse_s + 2 * e);
        const float2 nd = *reinterpret_cast<const float2*>(ndel_s + 2 * e);
        const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])),
                                  scale2, f2_pack(nl.x, nl.y));
        float x0, x1;
        f2_unpack(x, x0, x1);
        float p0 = ex2_approx(x0);
        float p1 = ex2_approx(x1);
        if (!full) {
          const int q = qs + 2 * e;
          if (q < iv.lo || q >= iv.hi) p0 = 0.f;
          if (q + 1 < iv.lo || q + 1 >= iv.hi) p1 = 0.f;
        }
        const uint64_t dd = f2_add(
            f2_pack(__uint_as_float(dpr[2 * e]), __uint_as_float(dpr[2 * e + 1])),
            f2_pack(nd.x, nd.y));
        float d0, d1;
        f2_unpack(f2_mul(f2_pack(p0, p1), dd), d0, d1);
        wp[e] = pack_bf16x2(p0, p1);
        wd[e] = pack_bf16x2(d0, d1);
      }
      // PdS (TMEM) and the dS^T shared tile still feed the previous tile's
      // products until they complete.
      if (i >= 1 && !(ok = mbar_wait_warp(BAR(C::BAR_MMA2), (i - 1) & 1, ab))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < BMQ / 32; ++c) {
        tmem_st16(t_lane + C::kTmemPDS + 32 * c, wp + 16 * c);
        tmem_st16(t_lane + C::kTmemPDS + 32 * c + 16, wd + 16 * c);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t off = row * 128 + ((u ^ (row & 7)) << 4);
        st_shared_v4(sbase + C::kOffDS + off, wd[4 * u], wd[4 * u + 1], wd[4 * u + 2],
                     wd[4 * u + 3]);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(C::BAR_PDSFULL));

      // dQ of this tile: TMEM lane = head dim `row`, columns = queries.
      if (!(ok = mbar_wait_warp(BAR(C::BAR_MMA2), i & 1, ab))) break;
      tc_fence_after();
      uint32_t dq[BMQ];
      tmem_ld32(t_lane + C::kTmemDQ, dq);
      tmem_ld32(t_lane + C::kTmemDQ + 32, dq + 32);
      tmem_wait_ld();
      tmem_pin<BMQ>(dq);
      tc_fence_before();
      mbar_arrive(BAR(C::BAR_DQFREE));
      const size_t stride = static_cast<size_t>(p.H) * D;
      float* ptr = p.dq_acc +
                   ((static_cast<size_t>(wi.b) * L + static_cast<size_t>(qh) * p.n + qs) * p.H +
                    wi.h) * D + dh * DH + row;
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
    }

    // ------------------------------------------------------------ epilogue
    // Warpgroup 0 writes dV, warpgroup 1 writes dK, once every MMA is done.
    if (ok) ok = mbar_wait_warp(BAR(C::BAR_ALL), 0, ab);
    tc_fence_after();
    if (ok) {
      const bool valid = j < p.n;
      const size_t pos = static_cast<size_t>(wi.half) * p.n + j;
      const size_t off = ((static_cast<size_t>(wi.b) * L + pos) * p.H + wi.h) * D + dh * DH;
      __nv_bfloat16* dst = (wg == 0 ? p.dv : p.dk) + off;
      const float mul = wg == 0 ? 1.f : p.scale;
      const uint32_t col = wg == 0 ? C::kTmemDV : C::kTmemDK;
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
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
  if (warp == 9) {
    if (lane == 0) mbar_wait_limited(sbase + C::kOffBar + 8 * C::BAR_ALL, 0, 1000000000ull);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int STAGES>
static cudaError_t launch_bwd2_impl(const BwdParams& p, cudaStream_t stream) {
  using C = Bwd2Cfg<D, STAGES>;
  auto kern = dfa_bwd2_kernel<D, STAGES>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long blocks = 2LL * p.B * p.H * p.k_tiles * C::NDH;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(blocks), C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_backward_d128(const BwdParams& p, cudaStream_t stream) {
  return launch_bwd2_impl<128, 3>(p, stream);
}

cudaError_t launch_backward_d256(const BwdParams& p, cudaStream_t stream) {
  return launch_bwd2_impl<256, 1>(p, stream);
}

}  // namespace dfa
