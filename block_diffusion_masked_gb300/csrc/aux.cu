// Memory-bound helpers of the backward pass.
//
// preprocess: D_i = sum_d dout_i,d * out_i,d for every row (the term of the
// softmax gradient that "FlashAttention: Exact Attention Without
// Materialization", section 4.5, recomputes instead of storing P), and zero
// the float32 dQ accumulator.  One warp per (batch, position, head) row; the
// row's out/dout bytes are read once, coalesced.
//
// convert: dq = bf16(dq_acc), round to nearest even, 8 elements per thread.
#include <cuda_bf16.h>

#include "params.cuh"
#include "sm100.cuh"

namespace dfa {

template <int D>
__global__ void __launch_bounds__(256) dfa_bwd_preprocess_kernel(
    const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
    float* __restrict__ delta, float* __restrict__ dq_acc, int B, int L, int H) {
  constexpr int PER_LANE = D / 32;  // 2, 4 or 8 elements
  const long long rows = static_cast<long long>(B) * L * H;
  const int lane = threadIdx.x & 31;
  const long long warps_total = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += warps_total) {
    const size_t base = static_cast<size_t>(r) * D + lane * PER_LANE;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < PER_LANE; e += 2) {
      const __nv_bfloat162 o = *reinterpret_cast<const __nv_bfloat162*>(out + base + e);
      const __nv_bfloat162 g = *reinterpret_cast<const __nv_bfloat162*>(dout + base + e);
      const float2 of = __bfloat1622float2(o);
      const float2 gf = __bfloat1622float2(g);
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
#pragma unroll
    for (int e = 0; e < PER_LANE; ++e) dq_acc[base + e] = 0.f;
    if (lane == 0) {
      // r enumerates (b, position, head); delta is laid out (b, head, position).
      const long long h = r % H;
      const long long bp = r / H;
      const long long pos = bp % L;
      const long long b = bp / L;
      delta[(b * H + h) * L + pos] = acc;
    }
  }
}

__global__ void __launch_bounds__(256) dfa_dq_convert_kernel(const float4* __restrict__ src,
                                                             uint4* __restrict__ dst,
                                                             long long groups) {
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
  const long long rows = static_cast<long long>(B) * L * H;
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows, 8);
  switch (d) {
    case 64:
      dfa_bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(out, dout, delta, dq_acc, B, L, H);
      break;
    case 128:
      dfa_bwd_preprocess_kernel<128><<<grid, 256, 0, stream>>>(out, dout, delta, dq_acc, B, L, H);
      break;
    case 256:
      dfa_bwd_preprocess_kernel<256><<<grid, 256, 0, stream>>>(out, dout, delta, dq_acc, B, L, H);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* dq_acc, __nv_bfloat16* dq, long long count,
                              cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const long long groups = count / 8;  // count is a multiple of 64 (headdim)
  dfa_dq_convert_kernel<<<grid_for(groups, 256), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint4*>(dq), groups);
  return cudaGetLastError();
}

}  // namespace dfa
