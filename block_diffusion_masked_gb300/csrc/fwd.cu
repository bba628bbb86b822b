// Forward kernel of block-diffusion attention on sm_103a.
//
// One CTA computes one 128-row query tile of one half of one (batch, head).
// It visits exactly the key tiles the mask reaches ("Fast Diffusion
// Attention", "Visit only the visible tiles"): for a clean query tile the
// clean key tiles up to its own block, for a noisy query tile the clean key
// tiles before its blocks and then the noisy key tiles of its blocks.  Per
// key tile it runs the loop of "FlashAttention: Exact Attention Without
// Materialization", section 5.1: S = Q K^T, running max and sum (section
// 4.2), O += P V; only O and the log-sum-exp reach device memory.
//
// Warp roles (224 threads):
//   warps 0-3  softmax: thread t owns query row t of the tile (TMEM lane t);
//              on request they first zero their CTA's share of the
//              backward's float32 dq accumulator;
//   warp 4     TMA producer: Q once, then K/V tiles through a STAGES-deep ring;
//   warp 5     MMA issuer of S = Q K^T into one of two TMEM score buffers;
//   warp 6     MMA issuer of O += P V into a TMEM accumulator (two issuing
//              warps on two schedulers: one alone is slowed by the busy
//              softmax warp that shares its scheduler).
// Scores live in TMEM, probabilities in a 128-byte-swizzled shared tile.
#include <cuda_bf16.h>

#include "geometry.cuh"
#include "params.cuh"
#include "sm100.cuh"

namespace dfa {

template <int D, int BN, int STAGES>
struct FwdCfg {
  static constexpr int BM = 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kPBytes = BM * BN * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + STAGES * kKVBytes;
  static constexpr int kOffP = kOffV + STAGES * kKVBytes;
  static constexpr int kOffBar = kOffP + kPBytes;
  enum {
    BAR_Q = 0,
    BAR_KFULL = 1,
    BAR_KEMPTY = BAR_KFULL + STAGES,
    BAR_VFULL = BAR_KEMPTY + STAGES,
    BAR_VEMPTY = BAR_VFULL + STAGES,
    BAR_SFULL = BAR_VEMPTY + STAGES,
    BAR_SFREE = BAR_SFULL + 2,
    BAR_PFULL = BAR_SFREE + 2,
    BAR_PVDONE = BAR_PFULL + 1,
    BAR_DRAIN = BAR_PVDONE + 1,
    NUM_BARS = BAR_DRAIN + 1
  };
  static constexpr int kOffTmemSlot = kOffBar + NUM_BARS * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + base alignment slack
  static constexpr int kTmemS0 = 0;
  static constexpr int kTmemS1 = BN;
  static constexpr int kTmemO = 2 * BN;
  static constexpr int kTmemCols = 512;
  static constexpr int kThreads = 224;
  static_assert(2 * BN + D <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(BN % 64 == 0 && D % 64 == 0, "tile shape");
};

template <int D, int BN, int STAGES, bool VARLEN>
__global__ void __launch_bounds__(224, 1) dfa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D, BN, STAGES>;
  constexpr int BM = C::BM;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  const AbortFlag ab{abort_flag, p.status};
#define BAR(i) (sbase + C::kOffBar + 8 * (i))

  // The CTA's item.  A varlen item is decoded from the slot table, which
  // may only be read after grid_dependency_wait below.
  WorkItem wi;
  Segment seg[2];
  int n = p.n, bs = p.bs, row0 = 0, n0 = 0, ntiles = 0, qs = 0, hk = 0, slot = 0;
  auto decode = [&]() {
    if constexpr (VARLEN) {
      slot = varlen_slot(p.vl, p.vl_slots, blockIdx.x);
      const VarlenSlot sl = p.vl[slot];
      n = sl.n;
      bs = imin(p.bs, n);
      row0 = sl.row0;
      wi = fwd_work(blockIdx.x - sl.off, MODE_DIFFUSION, 1, p.H, cdiv(n, BM), sl.group);
      wi.b = sl.b;
    } else {
      wi = fwd_work(blockIdx.x, p.mode, p.B, p.H, p.q_tiles, p.group);
    }
    const int nseg = fwd_segments(p.mode, n, bs, BM, BN, wi.half, wi.tile, seg);
    n0 = nseg > 0 ? seg[0].t_end - seg[0].t_begin : 0;
    ntiles = n0 + (nseg > 1 ? seg[1].t_end - seg[1].t_begin : 0);
    qs = wi.tile * BM;
    hk = wi.h / p.kv_group;  // key/value head
  };
  if constexpr (!VARLEN) decode();

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::BAR_Q), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(BAR(C::BAR_KFULL + s), 1);
      mbar_init(BAR(C::BAR_KEMPTY + s), 1);
      mbar_init(BAR(C::BAR_VFULL + s), 1);
      mbar_init(BAR(C::BAR_VEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(C::BAR_SFULL + b), 1);
      mbar_init(BAR(C::BAR_SFREE + b), 128);
    }
    mbar_init(BAR(C::BAR_PFULL), 128);
    mbar_init(BAR(C::BAR_PVDONE), 1);
    mbar_init(BAR(C::BAR_DRAIN), 2);  // both MMA-issuing warps
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
  // The prologue above touches only shared memory and TMEM; global memory
  // waits for the stream's previous kernel.
  grid_dependency_wait();
  if constexpr (VARLEN) decode();

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Varlen: the sample's own maps (rows past its halves read zero).
      const CUtensorMap* mq = &p.tm_q;
      const CUtensorMap* mk = &p.tm_k;
      const CUtensorMap* mv = &p.tm_v;
      if constexpr (VARLEN) {
        mq = &p.vl_maps[slot].q;
        mk = &p.vl_maps[slot].k;
        mv = &p.vl_maps[slot].v;
        tensormap_acquire(mq);
        tensormap_acquire(mk);
        tensormap_acquire(mv);
      }
      tma_prefetch_desc(mq);
      tma_prefetch_desc(mk);
      tma_prefetch_desc(mv);
      mbar_arrive_expect_tx(BAR(C::BAR_Q), C::kQBytes);
      const HalfRows qr = in_rows<VARLEN>(wi.b, wi.half);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_5d(sbase + C::kOffQ + c * BM * 128, mq, BAR(C::BAR_Q), 64 * c, wi.h,
                    qr.base + qs, qr.c3, qr.c4);
      bool ok = true;
      int j = 0;
      for (; j < ntiles && ok; ++j) {
        const int s = j < n0 ? 0 : 1;
        const int kt = seg[s].t_begin + (s ? j - n0 : j);
        const int st = j % STAGES;
        const int round = j / STAGES;
        if (round > 0 && !(ok = mbar_wait(BAR(C::BAR_KEMPTY + st), (round - 1) & 1, ab))) break;
        mbar_arrive_expect_tx(BAR(C::BAR_KFULL + st), C::kKVBytes);
        const HalfRows kr = in_rows<VARLEN>(wi.b, seg[s].half);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_5d(sbase + C::kOffK + st * C::kKVBytes + c * BN * 128, mk,
                      BAR(C::BAR_KFULL + st), 64 * c, hk, kr.base + kt * BN, kr.c3, kr.c4);
        if (round > 0 && !(ok = mbar_wait(BAR(C::BAR_VEMPTY + st), (round - 1) & 1, ab))) {
          // K of this stage is in flight; account for it while unwinding.
          ++j;
          break;
        }
        mbar_arrive_expect_tx(BAR(C::BAR_VFULL + st), C::kKVBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_5d(sbase + C::kOffV + st * C::kKVBytes + c * BN * 128, mv,
                      BAR(C::BAR_VFULL + st), 64 * c, hk, kr.base + kt * BN, kr.c3, kr.c4);
      }
      if (!ok) {
        // Unwinding: let the copies already issued land before the CTA exits.
        mbar_wait_limited(BAR(C::BAR_Q), 0, 100000000ull);
        for (int t = (j > STAGES ? j - STAGES : 0); t < j; ++t) {
          mbar_wait_limited(BAR(C::BAR_KFULL + t % STAGES), (t / STAGES) & 1, 100000000ull);
          mbar_wait_limited(BAR(C::BAR_VFULL + t % STAGES), (t / STAGES) & 1, 100000000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5 || warp == 6) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 5 issues S = Q K^T, warp 6 O += P V; the two streams share no
    // operand (S double-buffered in TMEM, P in shared memory), so each only
    // waits for the softmax warps, and they issue from two schedulers.
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(BM, BN, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(BM, D, false, true);
      bool ok = true;
      if (warp == 6) {
        for (int i = 0; i < ntiles && ok; ++i) {
          const int st = i % STAGES;
          if (!(ok = mbar_wait(BAR(C::BAR_PFULL), i & 1, ab))) break;
          if (!(ok = mbar_wait(BAR(C::BAR_VFULL + st), (i / STAGES) & 1, ab))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t a = sdesc_sw128(
                sbase + C::kOffP + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t b =
                sdesc_sw128(sbase + C::kOffV + st * C::kKVBytes + kk * 16 * 128, BN * 128, 1024);
            mma_ss(tmem + C::kTmemO, a, b, kIdPV, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(BAR(C::BAR_PVDONE));
          mma_commit(BAR(C::BAR_VEMPTY + st));
        }
      } else {
        ok = mbar_wait(BAR(C::BAR_Q), 0, ab);
        tc_fence_after();
        for (int j = 0; j < ntiles && ok; ++j) {
          const int st = j % STAGES;
          const int buf = j & 1;
          if (!(ok = mbar_wait(BAR(C::BAR_KFULL + st), (j / STAGES) & 1, ab))) break;
          if (j >= 2 && !(ok = mbar_wait(BAR(C::BAR_SFREE + buf), ((j - 2) >> 1) & 1, ab))) break;
          tc_fence_after();
          const uint32_t d_s = tmem + (buf ? C::kTmemS1 : C::kTmemS0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = sdesc_sw128(
                sbase + C::kOffQ + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(
                sbase + C::kOffK + st * C::kKVBytes + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16,
                1024);
            mma_ss(d_s, a, b, kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(BAR(C::BAR_SFULL + buf));
          mma_commit(BAR(C::BAR_KEMPTY + st));
        }
      }
      // Every MMA must be complete before the TMEM is released.
      mma_commit(BAR(C::BAR_DRAIN));
      mbar_wait_limited(BAR(C::BAR_DRAIN), 0, 1000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // The backward's dq accumulator, if the caller asks for it, is zeroed
    // here while the first scores are computed: this CTA's share of the
    // stores, issued and left to drain.
    if (p.zero_dst != nullptr) grid_zero16(p.zero_dst, p.zero_groups, threadIdx.x, 128);
    const int row = warp * 32 + lane;
    const int r = qs + row;  // row inside the half
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;  // running max, in scaled log2 units
    float l_run = 0.f;        // running sum of 2^(s*sl2 - m_run)
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int s = j < n0 ? 0 : 1;
      const int kt = seg[s].t_begin + (s ? j - n0 : j);
      const int buf = j & 1;
      if (!(ok = mbar_wait_warp(BAR(C::BAR_SFULL + buf), (j >> 1) & 1, ab))) break;
      tc_fence_after();
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(t_lane + (buf ? C::kTmemS1 : C::kTmemS0) + 32 * c, sr + 32 * c);
      tmem_wait_ld();
      tmem_pin<BN>(sr);
      tc_fence_before();
      mbar_arrive(BAR(C::BAR_SFREE + buf));

      const int ks = kt * BN;
      if (!tile_full(seg[s].rule, n, bs, qs, BM, ks, BN)) {
        const Interval iv = key_interval(seg[s].rule, r, n, bs);
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int key = ks + c;
          if (key < iv.lo || key >= iv.hi) sr[c] = __float_as_uint(-INFINITY);
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      const float m_new = fmaxf(m_run, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2_approx(m_run - m_use);

      // P buffer and O accumulator are shared with the previous PV product.
      if (j > 0) {
        if (!(ok = mbar_wait_warp(BAR(C::BAR_PVDONE), (j - 1) & 1, ab))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, corr != 1.0f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(t_lane + C::kTmemO + 32 * c, o);
            tmem_wait_ld();
            tmem_pin<32>(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st32(t_lane + C::kTmemO + 32 * c, o);
          }
          tmem_wait_st();
        }
      }
      float rs = 0.f;
#pragma unroll
      for (int a = 0; a < BN / 64; ++a) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = a * 64 + u * 8 + 2 * e;
            const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, -m_use));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), sl2, -m_use));
            rs += p0 + p1;
            w[e] = pack_bf16x2(p0, p1);
          }
          st_shared_v4(sbase + C::kOffP + a * (BM * 128) + row * 128 + ((u ^ (row & 7)) << 4),
                       w[0], w[1], w[2], w[3]);
        }
      }
      l_run = l_run * corr + rs;
      m_run = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(C::BAR_PFULL));
    }

    // ------------------------------------------------------------ epilogue
    if (ok && ntiles > 0) ok = mbar_wait_warp(BAR(C::BAR_PVDONE), (ntiles - 1) & 1, ab);
    tc_fence_after();
    if (ok) {
      const size_t pos = static_cast<size_t>(wi.half) * n + r;
      const size_t first =
          VARLEN ? static_cast<size_t>(row0) : wi.b * 2 * static_cast<size_t>(n);
      __nv_bfloat16* orow = p.out + ((first + pos) * p.H + wi.h) * D;
      const bool valid = r < n;
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (ntiles > 0) {
          tmem_ld32(t_lane + C::kTmemO + 32 * c, o);
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
              w[e] = pack_bf16x2(__uint_as_float(o[g * 8 + 2 * e]) * inv_l,
                                 __uint_as_float(o[g * 8 + 2 * e + 1]) * inv_l);
            st_global_v4(orow + 32 * c + 8 * g, w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (valid) {
        const float lse = l_run > 0.f ? (m_run + lg2_approx(l_run)) * 0.69314718055994531f
                                      : -INFINITY;
        if constexpr (VARLEN)
          p.lse[static_cast<size_t>(wi.h) * p.rows + row0 + pos] = lse;
        else
          p.lse[lse_offset(p.mode, wi.b, wi.h, wi.half, r, p.H, p.n)] = lse;
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

template <int D, int BN, int STAGES, bool VARLEN>
static cudaError_t launch_fwd_impl(const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D, BN, STAGES>;
  auto kern = dfa_fwd_kernel<D, BN, STAGES, VARLEN>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long blocks = VARLEN ? p.items : pass_items(p.mode, p.B, p.H, p.q_tiles);
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_chained(kern, dim3(static_cast<unsigned>(blocks)), dim3(C::kThreads),
                        C::kSmemBytes, stream, p);
}

cudaError_t launch_forward(const FwdParams& p, int headdim, cudaStream_t stream) {
  switch (headdim) {
    case 64:
    case 128: return launch_forward_persistent(p, headdim, stream);
    case 256:
      return p.vl ? launch_fwd_impl<256, 64, 2, true>(p, stream)
                  : launch_fwd_impl<256, 64, 2, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfa
