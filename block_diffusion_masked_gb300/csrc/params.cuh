// Parameter blocks handed from the C ABI layer to the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace dfa {

// Device status bits, OR-ed into the status word a kernel receives.
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusIndex = 2u;

// Packed batches of samples of different lengths ("Fast Diffusion
// Attention": varlen batches, scheduled longest first).  Sample b occupies
// rows [row0, row0 + 2n) of the packed (rows, heads, headdim) tensors, its
// noisy half first.  The host lists the non-empty samples longest first, one
// slot each; `off` counts the work units of the slots before it (units: the
// items of a pass without the backward's head-dim split).
struct VarlenSlot {
  int b;      // sample index (order of the packed tensors)
  int n;      // length of each half
  int row0;   // first row of the sample
  int group;  // heads per L2 scheduling group inside the sample
  int off;    // first work unit of the slot
};

// Varlen: tensor maps of one sample (rows [row0, row0 + 2n) of the packed
// tensors) viewed as (headdim, heads, n, 2, 1) -- the batched view of a
// batch of one -- so that rows past the end of either half read as zeros
// instead of the next sample's rows, and reduce-adds skip them: no value of
// one sample, finite or not, reaches another sample's tiles or results.
// The forward uses q, k, v; the backward q, k, v, dout and (headdim 128)
// dq, the float32 accumulator.
struct VarlenMaps {  // CUtensorMap carries its own (128-byte) alignment
  CUtensorMap q, k, v, dout, dq, dk, dv;
};

// Forward kernel parameters.  Batched: tensor maps view q/k/v as 5-D arrays
// (headdim, heads, n, halves, 1), halves = 2 * batch (sample b's noisy half
// is half 2b, its clean half 2b + 1; in the causal mode every sequence is
// one half), so that a tile never crosses the noisy/clean boundary and rows
// past the end of a half read as zeros.
// Varlen: q, k, v are read through per-sample maps (VarlenMaps); tm_o is a
// map of the packed output, (headdim, heads, rows, 1, 1).
struct FwdParams {
  CUtensorMap tm_q;  // box (64, 1, block_m, 1, 1)
  CUtensorMap tm_k;  // box (64, 1, block_n, 1, 1)
  CUtensorMap tm_v;  // box (64, 1, block_n, 1, 1)
  CUtensorMap tm_o;  // out, box (64, 1, block_m, 1, 1) (persistent forward's stores)
  __nv_bfloat16* out;
  float* lse;
  unsigned* status;
  int B, n, H, bs, mode;
  int kv_group;      // query heads per key/value head (1: multi-head)
  int q_tiles;       // tiles per half along the queries
  int group;         // (batch, head) pairs per scheduling group
  float scale_log2;  // softmax scale * log2(e)
  unsigned* sched;   // work counter of a persistent launch (see sched_next)
  // Optional: the backward's float32 dq accumulator, zeroed by the forward
  // launch alongside its tensor-core work (zero_groups 16-byte groups).
  float4* zero_dst;
  long long zero_groups;
  // Varlen only (vl == nullptr for a batched launch): the slot table, its
  // length, the rows of the packed tensors (lse is (heads, rows)) and the
  // work units of the launch.
  const VarlenSlot* vl;
  const VarlenMaps* vl_maps;  // one per slot
  int vl_slots;
  int rows;
  int items;
  float out_scale;  // FP8 forward: v's descale, applied to out
};

struct BwdParams {
  CUtensorMap tm_q;   // box (64, 1, block_m, 1, 1)
  CUtensorMap tm_do;  // box (64, 1, block_m, 1, 1)
  CUtensorMap tm_k;   // box (64, 1, block_n, 1, 1)
  CUtensorMap tm_v;   // box (64, 1, block_n, 1, 1)
  CUtensorMap tm_dq;  // float32 dq_acc, box (32, 1, query columns per warpgroup, 1, 1); headdim 128
  CUtensorMap tm_dk;  // dk, box (64, 1, 32, 1, 1): one warp's key rows; headdim 128
  CUtensorMap tm_dv;  // dv, the same
  const float* lse;   // (B, H, 2n)
  const float* delta; // (B, H, 2n): rowsum(dout * out)
  float* dq_acc;      // (B, 2n, H, d) fp32, zeroed before the kernel
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  unsigned* status;
  int B, n, H, bs, mode;
  int Hk;             // key/value heads (dk, dv are (B, 2n, Hk, d))
  int kv_group;       // query heads per key/value head, H / Hk
  int k_tiles;        // tiles per half along the keys
  int group;          // (batch, key/value head) pairs per scheduling group
  float scale;        // softmax scale
  float scale_log2;   // scale * log2(e)
  unsigned* sched;    // work counter of a persistent launch (see sched_next)
  int items;          // work items of the launch
  // Varlen only (vl == nullptr for a batched launch): the slot table, its
  // length and the rows of the packed tensors (lse, delta are (heads, rows)).
  const VarlenSlot* vl;
  const VarlenMaps* vl_maps;  // one per slot
  int vl_slots;
  int rows;
  int units;          // work units (items without the head-dim split)
  // Deterministic mode only (null otherwise): one counter per (head-dim
  // part, head, first row of a query tile), zero before the launch; rows =
  // the rows of q (batch * 2n, or the packed rows).
  unsigned* dq_sem;
  int sem_rows;
  // Passes of the noisy-diagonal specialisation (diffusion mode, batched):
  // 0 every key tile; 1 clean key tiles only; 2 noisy key tiles only, dQ
  // stored into the accumulator (each noisy query row gets its one noisy
  // diagonal contribution) instead of added.
  int pass;
};

#if defined(__CUDACC__)
// Work counter of a persistent launch, two words zero before the launch:
// sched[0] hands out item indices in order, sched[1] counts CTAs that have
// finished.  The last CTA to finish sets both back to zero, so the next
// launch on the same stream finds them zero again.
__device__ __forceinline__ int sched_next(unsigned* sched, int items) {
  const unsigned w = atomicAdd(sched, 1u);
  return w < static_cast<unsigned>(items) ? static_cast<int>(w) : -1;
}
// Slot of work unit u of a varlen launch: the last slot whose first unit is
// at most u (binary search over the slots' `off`, ascending).
__device__ __forceinline__ int varlen_slot(const VarlenSlot* vl, int slots, int u) {
  int lo = 0, hi = slots - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (vl[mid].off <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Tensor-map coordinates (c2, c3, c4) of row `base + r` of one half: batched
// maps are (headdim, heads, n, halves, 1), packed varlen maps (the output
// and dq maps) (headdim, heads, rows, 1, 1).
struct HalfRows {
  int base, c3, c4;
};
template <bool VARLEN>
__device__ __forceinline__ HalfRows half_rows(int b, int half, int n, int row0) {
  if constexpr (VARLEN) return {row0 + half * n, 0, 0};
  else return {0, 2 * b + half, 0};
}
// Coordinates of the input maps (q, k, v, dout): batched maps as above;
// varlen inputs are read through the sample's own maps (VarlenMaps), whose
// half index is the half itself.
template <bool VARLEN>
__device__ __forceinline__ HalfRows in_rows(int b, int half) {
  if constexpr (VARLEN) return {0, half, 0};
  else return {0, 2 * b + half, 0};
}

// One thread per CTA, after the CTA's last sched_next.
__device__ __forceinline__ void sched_finish(unsigned* sched) {
  __threadfence();
  if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
    atomicExch(sched, 0u);
    atomicExch(sched + 1, 0u);
  }
}
#endif

// Launch with programmatic stream serialization: the kernel may be launched
// while the kernel before it in the stream is still running, and waits for
// it (griddepcontrol.wait, grid_dependency_wait) before touching global
// memory, so that its launch and prologue overlap the predecessor's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Host helpers of the C ABI layer (api.cu) for the other translation units.
// check_device: the per-device set-up and architecture check every entry
// point runs first (DFA_OK, DFA_EUNSUPPORTED or DFA_ECUDA); *ctx_id receives
// the id of the device's current context, which changes when the context is
// destroyed and re-created.  record_cuda_failure: remember a failing CUDA
// call for dfa_last_cuda_error and return DFA_ECUDA.  check_backward_args:
// the shape checks of dfa_backward.
int check_device(unsigned long long* ctx_id);
int record_cuda_failure(cudaError_t e);
int check_backward_args(int B, int n, int H, int d, int bs);

// Launchers (one per translation unit).  Return a cudaError_t.
cudaError_t launch_forward(const FwdParams& p, int headdim, cudaStream_t stream);
cudaError_t launch_forward_persistent(const FwdParams& p, int headdim, cudaStream_t stream);
cudaError_t launch_forward_fp8(const FwdParams& p, int headdim, cudaStream_t stream);
cudaError_t launch_backward(const BwdParams& p, int headdim, cudaStream_t stream);
cudaError_t launch_backward_d128(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_backward_d256(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_backward_d64(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const __nv_bfloat16* out, const __nv_bfloat16* dout,
                                  float* delta, float* dq_acc, int B, int L, int H, int d,
                                  cudaStream_t stream);
cudaError_t launch_selftest_wait(unsigned* status, unsigned long long limit_ns,
                                 cudaStream_t stream);
cudaError_t launch_dq_convert(const float* dq_acc, __nv_bfloat16* dq, long long count,
                              cudaStream_t stream);
cudaError_t launch_fp8_v_transpose(const uint8_t* v, uint8_t* vt, int B, int n, int n_pad, int H,
                                   cudaStream_t stream);

// Compute warpgroups of the headdim-128 backward kernel; each takes
// 64 / this query columns of a tile and stages that many rows of dQ.
constexpr int kBwd2WarpgroupsD128 = 2;

// Tile shapes per head dimension.
struct TileShape {
  int fwd_bm, fwd_bn, bwd_bn, bwd_bm;
};
inline bool tile_shape_for(int d, TileShape* t) {
  switch (d) {
    case 64: *t = {128, 128, 128, 64}; return true;
    case 128: *t = {128, 128, 128, 64}; return true;
    case 256: *t = {128, 64, 128, 64}; return true;  // backward: 128 keys x 64 queries
    default: return false;
  }
}

}  // namespace dfa
