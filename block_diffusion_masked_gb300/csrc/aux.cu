// Memory-bound helpers of the backward pass.
//
// preprocess: D_i = sum_d dout_i,d * out_i,d for every row (the term of the
// softmax gradient that "FlashAttention: Exact Attention Without
// Materialization", section 4.5, recomputes instead of storing P), and zero
// the float32 dQ accumulator unless the forward did.  The rows' out/dout
// bytes are read once, coalesced, 16 bytes per lane.
//
// convert: dq = bf16(dq_acc), round to nearest even, 8 elements per thread.
#include <cuda_bf16.h>

#include "params.cuh"
#include "sm100.cuh"

namespace dfa {

// Each lane reads 16 bytes of out and of dout (8 elements), D / 8 lanes per
// row; a warp takes kUnroll row groups of consecutive positions of one
// (batch, head) and issues all their loads before any reduction, so that
// enough bytes are in flight to cover the memory latency.  Grid: x = chunks
// of 8 * kRowsPerPass positions, y = (batch, head) pairs (strided when there
// are more than the grid's y extent).  dq_acc may be null: then only D is
// computed (the forward zeroed the accumulator).
template <int D>
__global__ void __launch_bounds__(256) dfa_bwd_preprocess_kernel(
    const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
    float* __restrict__ delta, float* __restrict__ dq_acc, int L, int H, int BH) {
  constexpr int kLanesPerRow = D / 8;             // 8, 16 or 32
  constexpr int kRowsPerGroup = 32 / kLanesPerRow;  // rows one warp load covers
  constexpr int kUnroll = 4;
  constexpr int kRowsPerPass = kRowsPerGroup * kUnroll;
  grid_dependency_wait();  // out and dout come from the kernels before this one
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow;  // row of the group
  const int col = (lane % kLanesPerRow) * 8;
  const long long p0 =
      (static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kRowsPerPass;
  if (p0 >= L) return;  // warp-uniform
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    const int b = bh / H;
    const int h = bh - b * H;
    uint4 o[kUnroll], g[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long pos = p0 + u * kRowsPerGroup + sub;
      if (pos < L) {
        const size_t base = ((static_cast<size_t>(b) * L + pos) * H + h) * D + col;
        o[u] = *reinterpret_cast<const uint4*>(out + base);
        g[u] = *reinterpret_cast<const uint4*>(dout + base);
      } else {
        o[u] = make_uint4(0u, 0u, 0u, 0u);
        g[u] = o[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long pos = p0 + u * kRowsPerGroup + sub;
      const uint32_t ow[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
      const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
        const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
        acc = fmaf(of.x, gf.x, acc);
        acc = fmaf(of.y, gf.y, acc);
      }
#pragma unroll
      for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (pos < L) {
        if (dq_acc != nullptr) {
          float4* z = reinterpret_cast<float4*>(
              dq_acc + ((static_cast<size_t>(b) * L + pos) * H + h) * D + col);
          z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
          z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // delta is laid out (b, head, position)
        if (lane % kLanesPerRow == 0) delta[static_cast<size_t>(bh) * L + pos] = acc;
      }
    }
  }
}

__global__ void __launch_bounds__(256) dfa_dq_convert_kernel(const float4* __restrict__ src,
                                                             uint4* __restrict__ dst,
                                                             long long groups) {
  grid_dependency_wait();  // dq_acc comes from the kernel before this one
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
       g += stride) {
    const float4 a = src[2 * g];
    const float4 b = src[2 * g + 1];
    uint4 w;
    __nv_bfloat162 t;
    t = __floats2bfloat162_rn(a.x, a.y);
    w.x = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(a.z, a.w);
    w.y = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(b.x, b.y);
    w.z = *reinterpret_cast<uint32_t*>(&t);
    t = __floats2bfloat162_rn(b.z, b.w);
    w.w = *reinterpret_cast<uint32_t*>(&t);
    dst[g] = w;
  }
}

// FP8 forward: V^T.  vt[b][h][c][half][j] = v[b][half * n + j][h][c] for
// e4m3 v (B, 2n, H, 128), with vt rows of n_pad >= n keys, so that the
// P V product reads V with the keys contiguous (the K-major operand layout).
// One block per (128 keys of one half, head, batch): the 128 x 128-byte
// tile goes through shared memory, read and written in 16-byte units.
__global__ void __launch_bounds__(256) dfa_fp8_v_transpose_kernel(const uint8_t* __restrict__ v,
                                                                   uint8_t* __restrict__ vt, int n,
                                                                   int n_pad, int H) {
  // tile[r][w]: bytes 4w..4w+3 of the head dims of key r (rows padded by a
  // word against bank conflicts)
  __shared__ uint32_t tile[128][33];
  grid_dependency_wait();
  const int per_half = gridDim.x >> 1;  // 128-key chunks per half
  const int half = blockIdx.x >= per_half ? 1 : 0;
  const int jh = (blockIdx.x - half * per_half) * 128;  // first key of the block in its half
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  for (int u = threadIdx.x; u < 128 * 8; u += blockDim.x) {
    const int r = u >> 3, c16 = u & 7;  // key row, 16-byte unit of the head dims
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (jh + r < n)
      w = *reinterpret_cast<const uint4*>(
          v + ((static_cast<size_t>(b) * 2 * n + static_cast<size_t>(half) * n + jh + r) * H + h) *
                  128 + 16 * c16);
    tile[r][4 * c16 + 0] = w.x;
    tile[r][4 * c16 + 1] = w.y;
    tile[r][4 * c16 + 2] = w.z;
    tile[r][4 * c16 + 3] = w.w;
  }
  __syncthreads();
  // 4 x 4 byte blocks: keys 4m..4m+3 x head dims 4c4..4c4+3.  A warp takes
  // the 32 key groups of one head-dim group, so each of its four output
  // rows is written as 128 contiguous bytes.
  const int m = threadIdx.x & 31;
  for (int c4 = threadIdx.x >> 5; c4 < 32; c4 += blockDim.x >> 5) {
    const uint32_t w0 = tile[4 * m + 0][c4], w1 = tile[4 * m + 1][c4];
    const uint32_t w2 = tile[4 * m + 2][c4], w3 = tile[4 * m + 3][c4];
    const uint32_t t0 = __byte_perm(w0, w1, 0x5140), t1 = __byte_perm(w2, w3, 0x5140);
    const uint32_t t2 = __byte_perm(w0, w1, 0x7362), t3 = __byte_perm(w2, w3, 0x7362);
    const uint32_t o[4] = {__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632),
                           __byte_perm(t2, t3, 0x5410), __byte_perm(t2, t3, 0x7632)};
    if (jh + 4 * m < n_pad) {
#pragma unroll
      for (int jd = 0; jd < 4; ++jd) {
        const int c = 4 * c4 + jd;  // head dim = output row
        *reinterpret_cast<uint32_t*>(
            vt + (((static_cast<size_t>(b) * H + h) * 128 + c) * 2 + half) * n_pad + jh + 4 * m) =
            o[jd];
      }
    }
  }
}

cudaError_t launch_fp8_v_transpose(const uint8_t* v, uint8_t* vt, int B, int n, int n_pad, int H,
                                   cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  // blocks along x: the 128-key chunks of the noisy half, then the clean
  const int per_half = (n_pad + 127) / 128;
  const dim3 grid(static_cast<unsigned>(2 * per_half), static_cast<unsigned>(H),
                  static_cast<unsigned>(B));
  return launch_chained(dfa_fp8_v_transpose_kernel, grid, dim3(256), 0, stream, v, vt, n, n_pad,
                        H);
}

// Failure-detection self-test: one warp waits, through the same bounded
// wait the attention kernels use, on an mbarrier that nothing arrives on.
// The wait gives up after `limit_ns`, records the timeout in the status word
// and the kernel returns normally.
__global__ void dfa_selftest_wait_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const AbortFlag ab{&abort_flag, status};
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, ab, limit_ns);
  __syncwarp();
}

cudaError_t launch_selftest_wait(unsigned* status, unsigned long long limit_ns,
                                 cudaStream_t stream) {
  dfa_selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

static int grid_for(long long work, int per_block) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(sms) * 8;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_bwd_preprocess(const __nv_bfloat16* out, const __nv_bfloat16* dout,
                                  float* delta, float* dq_acc, int B, int L, int H, int d,
                                  cudaStream_t stream) {
  const long long bh = static_cast<long long>(B) * H;
  if (bh == 0 || L == 0) return cudaSuccess;
  if (bh > 0x7fffffffLL) return cudaErrorInvalidValue;
  // 8 warps of 1024 / d positions each per block
  const long long per_block = 8192 / d;
  const long long chunks = (L + per_block - 1) / per_block;
  if (chunks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(bh < 65535 ? bh : 65535));
  const int BH = static_cast<int>(bh);
  switch (d) {
    case 64:
      return launch_chained(dfa_bwd_preprocess_kernel<64>, grid, dim3(256), 0, stream, out, dout,
                            delta, dq_acc, L, H, BH);
    case 128:
      return launch_chained(dfa_bwd_preprocess_kernel<128>, grid, dim3(256), 0, stream, out, dout,
                            delta, dq_acc, L, H, BH);
    case 256:
      return launch_chained(dfa_bwd_preprocess_kernel<256>, grid, dim3(256), 0, stream, out, dout,
                            delta, dq_acc, L, H, BH);
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* dq_acc, __nv_bfloat16* dq, long long count,
                              cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const long long groups = count / 8;  // count is a multiple of 64 (headdim)
  return launch_chained(dfa_dq_convert_kernel, dim3(grid_for(groups, 256)), dim3(256), 0, stream,
                        reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint4*>(dq),
                        groups);
}

}  // namespace dfa
