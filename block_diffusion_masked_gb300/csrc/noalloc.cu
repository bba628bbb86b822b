// Backward pass that allocates no device memory.
//
// dfa_backward takes its float32 scratch (the dq accumulator and the row
// vector D = rowsum(dout * out)) from the stream-ordered allocator.  Some
// callers cannot let a library allocate: a framework whose caching allocator
// must own every byte of device memory (so that its accounting and its
// out-of-memory handling stay right), or a latency-critical step where an
// allocation could block or fail half-way through.  dfa_backward_noalloc runs
// the same three steps with the scratch in a fixed array that lives in this
// file, so the call itself never allocates.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kNoallocScratchBytes) until the process exits.  Host code
// must not use the array's name as an address (on the host it only names a
// stand-in); its device address is fetched with cudaGetSymbolAddress, with
// the device current, on the first call there, and fetched again if the
// device's context has been destroyed and re-created since (for instance by
// cudaDeviceReset), because the old address then belongs to a dead context.
#include <cuda_runtime.h>

#include <mutex>

#include "dfa.h"
#include "params.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr size_t kNoallocScratchFloats = kNoallocScratchBytes / sizeof(float);
constexpr int kMaxDevices = 64;

struct NoallocSlot {
  float* ptr = nullptr;
  unsigned long long ctx_id = 0;  // context `ptr` was looked up in
};

std::mutex g_noalloc_mu;
NoallocSlot g_noalloc[kMaxDevices];

}  // namespace

static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

extern "C" int dfa_backward_noalloc(const void* q, const void* k, const void* v, const void* out,
                                    const void* dout, const float* lse, void* dq, void* dk,
                                    void* dv, int batch, int n, int heads, int headdim,
                                    int block_size, dfa_stream_t stream) {
  // The checks of dfa_backward come first, in its order: arguments, then
  // the device (an unsupported device is DFA_EUNSUPPORTED, as there).
  int rc = dfa::check_backward_args(batch, n, heads, headdim, block_size);
  if (rc) return rc;
  if (batch == 0) return DFA_OK;
  // Scratch: dq_acc (batch * 2n * heads * headdim floats), then delta
  // (batch * heads * 2n floats).  headdim is a multiple of 64, so delta
  // starts 256-byte aligned.
  const size_t rows = static_cast<size_t>(batch) * heads * 2 * static_cast<size_t>(n);
  const size_t elems = rows * static_cast<size_t>(headdim);
  if (elems + rows > kNoallocScratchFloats) return DFA_EINVAL;
  unsigned long long ctx = 0;
  if ((rc = dfa::check_device(&ctx))) return rc;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFA_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return DFA_EUNSUPPORTED;
  float* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot& slot = g_noalloc[dev];
    if (!slot.ptr || slot.ctx_id != ctx) {
      void* addr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
      if (e != cudaSuccess) return dfa::record_cuda_failure(e);
      if (addr == nullptr) return DFA_ECUDA;
      slot.ptr = static_cast<float*>(addr);
      slot.ctx_id = ctx;
    }
    base = slot.ptr;
  }
  float* dq_acc = base;
  float* delta = base + elems;
  // The preprocess step zeroes dq_acc, so a previous call's contents never
  // leak into this one.
  rc = dfa_bwd_preprocess(out, dout, delta, dq_acc, batch, n, heads, headdim, stream);
  if (rc) return rc;
  rc = dfa_bwd_main(q, k, v, dout, lse, delta, dq_acc, dk, dv, batch, n, heads, headdim,
                    block_size, DFA_MODE_DIFFUSION, stream);
  if (rc) return rc;
  return dfa_bwd_dq_convert(dq_acc, dq, batch, n, heads, headdim, stream);
}
