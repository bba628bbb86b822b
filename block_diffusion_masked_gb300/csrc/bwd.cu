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
// Per query tile (all on tcgen05 tensor cores, accumulators in TMEM):
//   S^T  = K Q^T          dP^T = V dO^T
//   P^T  = exp(scale S^T - LSE)   (0 on hidden pairs)
//   dS^T = P^T * (dP^T - D)
//   dV  += P^T dO         dK  += dS^T Q
//   dQ   = dS K  (added to a float32 accumulator in device memory)
// Warp roles (192 threads): warps 0-3 compute (thread t owns key row t of the
// tile, TMEM lane t), warp 4 loads (TMA for Q/dO, plain loads for LSE/D),
// warp 5 issues the MMAs.
#include <cuda_bf16.h>

#include "geometry.cuh"
#include "params.cuh"
#include "sm100.cuh"

namespace dfa {

template <int D, int BMQ>
struct BwdCfg {
  static constexpr int BN = 128;  // keys per tile (MMA M)
  static constexpr int STAGES = 2;
  static constexpr int kChunks = D / 64;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kQBytes = BMQ * D * 2;
  static constexpr int kPBytes = BN * BMQ * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVBytes;
  static constexpr int kOffQ = kOffV + kKVBytes;
  static constexpr int kOffDO = kOffQ + STAGES * kQBytes;
  static constexpr int kOffP = kOffDO + STAGES * kQBytes;
  static constexpr int kOffDS = kOffP + kPBytes;
  static constexpr int kOffLSE = kOffDS + kPBytes;           // STAGES x BMQ floats
  static constexpr int kOffDEL = kOffLSE + STAGES * BMQ * 4;  // STAGES x BMQ floats
  static constexpr int kOffBar = kOffDEL + STAGES * BMQ * 4;
  enum {
    BAR_KV = 0,
    BAR_QFULL = 1,
    BAR_QEMPTY = BAR_QFULL + STAGES,
    BAR_SDP = BAR_QEMPTY + STAGES,
    BAR_PDS = BAR_SDP + 1,
    BAR_MMA2 = BAR_PDS + 1,
    BAR_DQFREE = BAR_MMA2 + 1,
    BAR_DRAIN = BAR_DQFREE + 1,
    NUM_BARS = BAR_DRAIN + 1
  };
  static constexpr int kOffTmemSlot = kOffBar + NUM_BARS * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;
  // dQ is computed transposed (rows = head dims) when headdim = 128, so that
  // each warp's float atomics cover 32 consecutive head dims of one query;
  // with headdim 64 it is computed as (queries x head dims).
  static constexpr bool kDqTransposed = (D == 128);
  static constexpr int kTmemS = 0;
  static constexpr int kTmemDP = BMQ;
  static constexpr int kTmemDV = 2 * BMQ;
  static constexpr int kTmemDK = 2 * BMQ + D;
  static constexpr int kTmemDQ = 2 * BMQ + 2 * D;
  static constexpr int kDqCols = kDqTransposed ? BMQ : D;
  static constexpr int kTmemCols = 512;
  static constexpr int kThreads = 192;
  static_assert(kTmemDQ + kDqCols <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kDqTransposed ? (D == 128) : (BMQ == 128), "dQ MMA needs M = 128");
};

template <int D, int BMQ>
__global__ void __launch_bounds__(192, 1) dfa_bwd_kernel(const __grid_constant__ BwdParams p) {
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
  const AbortFlag ab{abort_flag, p.status};
#define BAR(i) (sbase + C::kOffBar + 8 * (i))

  const WorkItem wi = bwd_work(blockIdx.x, p.mode, p.B, p.H, p.k_tiles);
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
    mbar_init(BAR(C::BAR_SDP), 1);
    mbar_init(BAR(C::BAR_PDS), 128);
    mbar_init(BAR(C::BAR_MMA2), 1);
    mbar_init(BAR(C::BAR_DQFREE), 128);
    mbar_init(BAR(C::BAR_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(sbase + C::kOffTmemSlot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::kOffTmemSlot);

  if (warp == 4) {
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
      for (int c = lane; c < BMQ; c += 32) {
        const int q = qt * BMQ + c;
        const bool valid = q < p.n;
        const size_t pos = static_cast<size_t>(seg[s].half) * p.n + q;
        lse_s[c] = valid ? p.lse[lse_offset(p.mode, wi.b, wi.h, seg[s].half, q, p.H, p.n)] *
                               1.4426950408889634f
                         : INFINITY;
        del_s[c] = valid ? del_bh[pos] : 0.f;
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
    }
    if (!ok && lane == 0) {
      mbar_wait_limited(BAR(C::BAR_KV), 0, 100000000ull);
      for (int t = (i > STAGES ? i - STAGES : 0); t < i; ++t)
        mbar_wait_limited(BAR(C::BAR_QFULL + t % STAGES), (t / STAGES) & 1, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(BN, BMQ, false, false);      // K Q^T, V dO^T
      constexpr uint32_t kIdKV = idesc_bf16(BN, D, false, true);        // P^T dO, dS^T Q
      constexpr uint32_t kIdDQ = C::kDqTransposed ? idesc_bf16(D, BMQ, true, true)   // K^T dS^T
                                                  : idesc_bf16(BMQ, D, true, true);  // dS K
      bool ok = mbar_wait(BAR(C::BAR_KV), 0, ab);
      for (int i = 0; i < ntiles && ok; ++i) {
        const int st = i % STAGES;
        if (!(ok = mbar_wait(BAR(C::BAR_QFULL + st), (i / STAGES) & 1, ab))) break;
        tc_fence_after();
        const uint32_t q_s = sbase + C::kOffQ + st * C::kQBytes;
        const uint32_t do_s = sbase + C::kOffDO + st * C::kQBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
          mma_ss(tmem + C::kTmemS, sdesc_sw128(sbase + C::kOffK + koff, 16, 1024),
                 sdesc_sw128(q_s + qoff, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (BMQ * 128) + (kk & 3) * 32;
          mma_ss(tmem + C::kTmemDP, sdesc_sw128(sbase + C::kOffV + koff, 16, 1024),
                 sdesc_sw128(do_s + qoff, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(C::BAR_SDP));
        if (!(ok = mbar_wait(BAR(C::BAR_PDS), i & 1, ab))) break;
        if (i > 0 && !(ok = mbar_wait(BAR(C::BAR_DQFREE), (i - 1) & 1, ab))) break;
        tc_fence_after();
        // dV += P^T dO ; dK += dS^T Q   (M = keys, N = head dims, K = queries)
#pragma unroll
        for (int kk = 0; kk < BMQ / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          mma_ss(tmem + C::kTmemDV, sdesc_sw128(sbase + C::kOffP + poff, 16, 1024),
                 sdesc_sw128(do_s + kk * 16 * 128, BMQ * 128, 1024), kIdKV, acc);
          mma_ss(tmem + C::kTmemDK, sdesc_sw128(sbase + C::kOffDS + poff, 16, 1024),
                 sdesc_sw128(q_s + kk * 16 * 128, BMQ * 128, 1024), kIdKV, acc);
        }
        // dQ (transposed or not), K = keys
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t kdesc = sdesc_sw128(sbase + C::kOffK + kk * 16 * 128, BN * 128, 1024);
          const uint64_t sdesc = sdesc_sw128(sbase + C::kOffDS + kk * 16 * 128, BN * 128, 1024);
          if (C::kDqTransposed)
            mma_ss(tmem + C::kTmemDQ, kdesc, sdesc, kIdDQ, kk > 0 ? 1u : 0u);
          else
            mma_ss(tmem + C::kTmemDQ, sdesc, kdesc, kIdDQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(C::BAR_MMA2));
        mma_commit(BAR(C::BAR_QEMPTY + st));
      }
      mma_commit(BAR(C::BAR_DRAIN));
      mbar_wait_limited(BAR(C::BAR_DRAIN), 0, 1000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute
    const int row = warp * 32 + lane;  // key row of the tile / TMEM lane
    const int j = ks + row;            // key inside its half
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int s = i < n0 ? 0 : 1;
      const int qt = seg[s].t_begin + (s ? i - n0 : i);
      const int qh = seg[s].half;
      const int st = i % STAGES;
      if (!(ok = mbar_wait_warp(BAR(C::BAR_SDP), i & 1, ab))) break;
      tc_fence_after();

      const float* lse_s = reinterpret_cast<const float*>(smem + C::kOffLSE) + st * BMQ;
      const float* del_s = reinterpret_cast<const float*>(smem + C::kOffDEL) + st * BMQ;
      const int qs = qt * BMQ;
      const bool full = tile_full(seg[s].rule, p.n, p.bs, qs, BMQ, ks, BN);
      const Interval iv = query_interval(seg[s].rule, j, p.n, p.bs);
      // 32 query columns at a time: S^T and dP^T chunks, then P^T and dS^T
      // rows into the swizzled shared tiles (4 x 16 bytes each per chunk).
#pragma unroll 1
      for (int cc = 0; cc < BMQ / 32; ++cc) {
        uint32_t sr[32], dpr[32];
        tmem_ld32(t_lane + C::kTmemS + 32 * cc, sr);
        tmem_ld32(t_lane + C::kTmemDP + 32 * cc, dpr);
        tmem_wait_ld();
        tmem_pin<32>(sr);
        tmem_pin<32>(dpr);
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          uint32_t wp[4], wd[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pv[2], dv[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int cl = u4 * 8 + 2 * e + h2;  // column inside the chunk
              const int c = cc * 32 + cl;          // column inside the tile
              float pr = ex2_approx(fmaf(__uint_as_float(sr[cl]), sl2, -lse_s[c]));
              if (!full) {
                const int q = qs + c;
                if (q < iv.lo || q >= iv.hi) pr = 0.f;
              }
              pv[h2] = pr;
              dv[h2] = pr * (__uint_as_float(dpr[cl]) - del_s[c]);
            }
            wp[e] = pack_bf16x2(pv[0], pv[1]);
            wd[e] = pack_bf16x2(dv[0], dv[1]);
          }
          const int a = cc >> 1;                   // 64-column swizzle atom
          const int u = (cc & 1) * 4 + u4;         // 16-byte unit inside the row
          const uint32_t off = a * (BN * 128) + row * 128 + ((u ^ (row & 7)) << 4);
          st_shared_v4(sbase + C::kOffP + off, wp[0], wp[1], wp[2], wp[3]);
          st_shared_v4(sbase + C::kOffDS + off, wd[0], wd[1], wd[2], wd[3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(BAR(C::BAR_PDS));

      // dQ of this query tile: read it from TMEM and add it to the float32
      // accumulator in device memory.
      if (!(ok = mbar_wait_warp(BAR(C::BAR_MMA2), i & 1, ab))) break;
      tc_fence_after();
      if (C::kDqTransposed) {
        // TMEM lane = head dim `row`; columns = queries of the tile.
        uint32_t dq[BMQ];
#pragma unroll
        for (int c = 0; c < BMQ / 32; ++c) tmem_ld32(t_lane + C::kTmemDQ + 32 * c, dq + 32 * c);
        tmem_wait_ld();
        tmem_pin<BMQ>(dq);
        tc_fence_before();
        mbar_arrive(BAR(C::BAR_DQFREE));
        float* base = p.dq_acc + ((static_cast<size_t>(wi.b) * L + static_cast<size_t>(qh) * p.n) *
                                      p.H + wi.h) * D + row;
        const int qmax = p.n - qs;
#pragma unroll
        for (int c = 0; c < BMQ; ++c) {
          if (c < qmax)
            red_add_f32(base + (static_cast<size_t>(qs + c) * p.H) * D,
                        __uint_as_float(dq[c]) * p.scale);
        }
      } else {
        // TMEM lane = query `row` of the tile; columns = head dims.
        uint32_t dq[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(t_lane + C::kTmemDQ + 32 * c, dq + 32 * c);
        tmem_wait_ld();
        tmem_pin<D>(dq);
        tc_fence_before();
        mbar_arrive(BAR(C::BAR_DQFREE));
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
    }

    // ------------------------------------------------------------ epilogue
    if (ok) {
      const bool valid = j < p.n;
      const size_t pos = static_cast<size_t>(wi.half) * p.n + j;
      const size_t off = ((static_cast<size_t>(wi.b) * L + pos) * p.H + wi.h) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = (which == 0 ? p.dv : p.dk) + off;
        const float mul = which == 0 ? 1.f : p.scale;
        const uint32_t col = which == 0 ? C::kTmemDV : C::kTmemDK;
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
  }
#undef BAR

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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
    case 128: return launch_bwd_impl<128, 64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfa
