// C ABI of libdfa: argument checks, tensor maps, scratch, launches.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <initializer_list>
#include <mutex>
#include <cstring>
#include <vector>

#include "dfa.h"
#include "geometry.cuh"
#include "params.cuh"

// Device status word: kernels OR error bits into it, dfa_status() reads and
// clears it.  Host code reaches it through cudaGetSymbolAddress.
static __device__ unsigned g_dfa_status;

// Work counters of the persistent kernels: one pair of words per slot, a
// slot per stream (see sched_for_stream).  Zero at load; every launch leaves
// its slot zero again when its last CTA finishes.
constexpr int kSchedSlots = 256;
static __device__ unsigned g_dfa_sched[kSchedSlots * 8];

namespace dfa {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  unsigned long long ctx_id = 0;  // context the addresses below belong to
  unsigned* status = nullptr;
  unsigned* sched = nullptr;  // kSchedSlots slots of 8 words
  long long l2_bytes = 0;
  const void* slot_key[kSchedSlots] = {};
  int slots_used = 0;
  int slot_next = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
thread_local cudaError_t t_last_error = cudaSuccess;

// Remember a failing CUDA call's code for dfa_last_cuda_error().
int cuda_fail(cudaError_t e) {
  t_last_error = e;
  return DFA_ECUDA;
}
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

// Driver entry points, resolved once (caller holds g_mu).
bool resolve_driver() {
  if (g_encode && g_ctx_current && g_ctx_get_id) return true;
  auto get = [](const char* name, int version, void** fn) {
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion(name, fn, version, cudaEnableDefault, &q) ==
               cudaSuccess &&
           q == cudaDriverEntryPointSuccess && *fn != nullptr;
  };
  void* a = nullptr;
  void* b = nullptr;
  void* c = nullptr;
  if (!get("cuTensorMapEncodeTiled", 12000, &a) || !get("cuCtxGetCurrent", 4000, &b) ||
      !get("cuCtxGetId", 12000, &c))
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(a);
  g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(b);
  g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(c);
  return true;
}

// Process-unique id of the calling thread's current context, 0 if there is
// none yet.  cudaDeviceReset destroys a device's primary context; the one
// the runtime creates next has a new id, and device addresses looked up in
// the old one are stale.
unsigned long long ctx_id_now() {
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!g_ctx_current || g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (!g_ctx_get_id || g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Per-device set-up on first use, and again whenever the device's context
// has changed: check the architecture (the library holds sm_103a code only)
// and find the device addresses of the status word and the work counters.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFA_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return DFA_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!resolve_driver()) return DFA_ECUDA;
  DeviceState& s = g_dev[dev];
  if (s.ready && s.supported) {
    // The context may not be current on this thread yet: a symbol lookup
    // makes the runtime bind its primary context.
    unsigned long long id = ctx_id_now();
    if (id == 0) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_dfa_status) != cudaSuccess) return DFA_ECUDA;
      id = ctx_id_now();
    }
    if (id != s.ctx_id) s = DeviceState();  // a new context: set up again
  }
  if (!s.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return DFA_ECUDA;
    s.supported = (major == 10 && minor == 3);
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return DFA_ECUDA;
    s.l2_bytes = l2;
    if (s.supported) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_dfa_status) != cudaSuccess) return DFA_ECUDA;
      s.status = static_cast<unsigned*>(addr);
      if (cudaGetSymbolAddress(&addr, g_dfa_sched) != cudaSuccess) return DFA_ECUDA;
      s.sched = static_cast<unsigned*>(addr);
      s.ctx_id = ctx_id_now();
    }
    s.ready = true;
  }
  if (!s.supported) return DFA_EUNSUPPORTED;
  *out = &s;
  return DFA_OK;
}

// Work counter for a launch on `stream`.  Launches on one stream run one
// after another, so they can share a counter (each leaves it zero); launches
// on different streams may run at the same time and get different slots.
// The per-thread default stream has one handle for many streams, so it is
// keyed by the calling thread.  Past kSchedSlots streams the oldest slot is
// reused.
thread_local char t_stream_key;
unsigned* sched_for_stream(DeviceState* s, cudaStream_t stream) {
  const void* key = stream == cudaStreamPerThread ? static_cast<const void*>(&t_stream_key)
                                                  : static_cast<const void*>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < s->slots_used; ++i)
    if (s->slot_key[i] == key) return s->sched + 8 * i;
  int i;
  if (s->slots_used < kSchedSlots) {
    i = s->slots_used++;
  } else {
    i = s->slot_next;
    s->slot_next = (s->slot_next + 1) % kSchedSlots;
  }
  s->slot_key[i] = key;
  return s->sched + 8 * i;
}

// View a bf16 tensor of `halves` consecutive halves of n rows, (halves * n,
// H, d), as 5-D (d, H, n, halves, 1) -- strides increasing -- and load boxes
// of (64, 1, rows, 1, 1) with 128-byte swizzle: `rows` consecutive positions
// of one half of one head, 64 head dims each.  Rows past the end of a half
// read zero.  A (B, 2n, H, d) diffusion tensor has 2B halves (sample b's are
// 2b and 2b + 1); a causal (Bc, n, H, d) tensor has Bc, one per sequence.
int make_map(CUtensorMap* map, const void* base, long long halves, int n, int H, int d, int rows,
             bool packed = false) {
  // packed (varlen): n is the number of rows of the packed tensor, viewed as
  // (d, H, rows, 1, 1)
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(n),
                              packed ? 1u : static_cast<cuuint64_t>(halves), 1u};
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(H) * d * 2;
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(d) * 2, row_bytes, row_bytes * n,
                                 row_bytes * n * (packed ? 1 : static_cast<cuuint64_t>(halves))};
  const cuuint32_t box[5] = {64, 1, static_cast<cuuint32_t>(rows), 1, 1};
  const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFA_OK : DFA_ECUDA;
}

// An e4m3 (one byte per element) (B, 2n, H, d) tensor as 5-D (d, H, n,
// 2B, 1) with boxes of (128, 1, rows, 1, 1), 128-byte swizzle: rows of
// 128 head dims, the same 128-byte rows as the bf16 maps' 64.
int make_map_u8(CUtensorMap* map, const void* base, int B, int n, int H, int d, int rows) {
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(n), 2 * static_cast<cuuint64_t>(B), 1};
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(H) * d;
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(d), row_bytes, row_bytes * n,
                                 row_bytes * 2 * n * B};
  const cuuint32_t box[5] = {128, 1, static_cast<cuuint32_t>(rows), 1, 1};
  const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFA_OK : DFA_ECUDA;
}

// The FP8 forward's V^T, (B, H, 128, 2, n_pad) bytes, as 5-D (n, half,
// 128, H, B) with boxes of (128, 1, 128, 1, 1): 128 keys of one half for
// all 128 head dims, 128-byte swizzle; keys past n read zero.
int make_map_vt(CUtensorMap* map, const void* base, int B, int n, int n_pad, int H) {
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(n), 2, 128, static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t np = static_cast<cuuint64_t>(n_pad);
  const cuuint64_t strides[4] = {np, 2 * np, 256 * np, 256 * np * H};
  const cuuint32_t box[5] = {128, 1, 128, 1, 1};
  const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFA_OK : DFA_ECUDA;
}

// The float32 dQ accumulator, laid out as q, as 5-D (d, H, n, halves, 1)
// with boxes of (32, 1, rows, 1, 1), no swizzle: the target of the
// backward's bulk reduce-add of one warp's part of a query tile's dQ (rows
// past the end of a half are skipped by the copy engine).
int make_map_f32(CUtensorMap* map, const void* base, long long halves, int n, int H, int d,
                 int rows, bool packed = false, int inner = 32) {
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(n),
                              packed ? 1u : static_cast<cuuint64_t>(halves), 1u};
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(H) * d * 4;
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(d) * 4, row_bytes, row_bytes * n,
                                 row_bytes * n * (packed ? 1 : static_cast<cuuint64_t>(halves))};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(inner), 1, static_cast<cuuint32_t>(rows), 1,
                             1};
  const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFA_OK : DFA_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int n, int H, int d, int bs) {
  if (B < 0 || n < 1 || H < 1 || bs < 1) return DFA_EINVAL;
  if (d != 64 && d != 128 && d != 256) return DFA_EUNSUPPORTED;
  // Index arithmetic inside the kernels uses 64-bit offsets; tile counts and
  // the grid use 32-bit integers.
  if (static_cast<long long>(n) * 2 > (1LL << 30)) return DFA_EINVAL;
  return DFA_OK;
}

// Query heads per key/value head, or 0 when Hk does not divide H.
int kv_group_of(int H, int Hk) { return Hk >= 1 && Hk <= H && H % Hk == 0 ? H / Hk : 0; }

int forward_impl(int mode, const void* q, const void* k, const void* v, void* out, float* lse,
                 float* dq_acc, int B, int n, int H, int Hk, int d, int bs, cudaStream_t stream) {
  int rc = check_common(B, n, H, d, bs);
  if (rc) return rc;
  const int G = kv_group_of(H, Hk);
  if (G == 0) return DFA_EINVAL;
  if (B == 0) return DFA_OK;
  if (!q || !k || !v || !out || !lse) return DFA_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (dq_acc && !aligned16(dq_acc)))
    return DFA_EINVAL;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds))) return rc;
  TileShape ts;
  tile_shape_for(d, &ts);
  // Diffusion: B samples of two halves; causal: B sequences of n rows.
  const long long halves = launch_halves(mode, B);
  FwdParams p{};
  if ((rc = make_map(&p.tm_q, q, halves, n, H, d, ts.fwd_bm))) return rc;
  if ((rc = make_map(&p.tm_k, k, halves, n, Hk, d, ts.fwd_bn))) return rc;
  if ((rc = make_map(&p.tm_v, v, halves, n, Hk, d, ts.fwd_bn))) return rc;
  if ((rc = make_map(&p.tm_o, out, halves, n, H, d, ts.fwd_bm))) return rc;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = ds->status;
  p.B = B;
  p.n = n;
  p.H = H;
  p.kv_group = G;
  p.bs = bs < n ? bs : n;
  p.mode = mode;
  p.q_tiles = cdiv(n, ts.fwd_bm);
  // q, k, v and out of one (batch, head), or of one (sequence, head)
  p.group = l2_group(8LL * (mode == MODE_CAUSAL ? 1 : 2) * n * d, ds->l2_bytes, B * H);
  p.sched = sched_for_stream(ds, stream);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  p.zero_dst = reinterpret_cast<float4*>(dq_acc);
  // halves * n * H * d floats, d a multiple of 64: whole 16-byte groups
  p.zero_groups = dq_acc ? halves * n * H * d / 4 : 0;
  const cudaError_t e = launch_forward(p, d, stream);
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

// FP8 forward: q, k, v e4m3 with per-tensor descales (x = x8 * x_descale);
// out bf16, lse as dfa_forward's.  Headdim 128.
// vt_in: V^T already in the layout dfa_fp8_transpose_v writes (v unused),
// or null: V^T goes through stream-ordered scratch.
int forward_fp8_impl(const void* q, const void* k, const void* v, void* out, float* lse,
                     float q_descale, float k_descale, float v_descale, int B, int n, int H,
                     int Hk, int d, int bs, cudaStream_t stream, const void* vt_in = nullptr) {
  int rc = check_common(B, n, H, d, bs);
  if (rc) return rc;
  if (d != 128) return DFA_EUNSUPPORTED;
  const int G = kv_group_of(H, Hk);
  if (G == 0) return DFA_EINVAL;
  if (!(q_descale > 0.f) || !(k_descale > 0.f) || !(v_descale > 0.f) ||
      !std::isfinite(q_descale) || !std::isfinite(k_descale) || !std::isfinite(v_descale))
    return DFA_EINVAL;
  if (B == 0) return DFA_OK;
  const void* vsrc = vt_in ? vt_in : v;
  if (!q || !k || !vsrc || !out || !lse) return DFA_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vsrc) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return DFA_EINVAL;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds))) return rc;
  TileShape ts;
  tile_shape_for(d, &ts);
  // V^T (given, or in stream-ordered scratch), keys padded to 16 (TMA row
  // strides)
  const int n_pad = (n + 15) / 16 * 16;
  uint8_t* vt = nullptr;
  const size_t vt_bytes = static_cast<size_t>(B) * Hk * 128 * 2 * n_pad;
  FwdParams p{};
  if ((rc = make_map_u8(&p.tm_q, q, B, n, H, d, ts.fwd_bm))) return rc;
  if ((rc = make_map_u8(&p.tm_k, k, B, n, Hk, d, ts.fwd_bn))) return rc;
  if ((rc = make_map(&p.tm_o, out, 2LL * B, n, H, d, ts.fwd_bm))) return rc;
  if (vt_in) {
    if ((rc = make_map_vt(&p.tm_v, vt_in, B, n, n_pad, Hk))) return rc;
  } else {
    if (cudaMallocAsync(reinterpret_cast<void**>(&vt), vt_bytes, stream) != cudaSuccess)
      return DFA_ECUDA;
    if ((rc = make_map_vt(&p.tm_v, vt, B, n, n_pad, Hk))) {
      cudaFreeAsync(vt, stream);
      return rc;
    }
  }
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = ds->status;
  p.B = B;
  p.n = n;
  p.H = H;
  p.kv_group = G;
  p.bs = bs < n ? bs : n;
  p.mode = MODE_DIFFUSION;
  p.q_tiles = cdiv(n, ts.fwd_bm);
  // q, k, v (one byte) and out (two) of one (batch, head)
  p.group = l2_group(5LL * 2 * n * d, ds->l2_bytes, B * H);
  p.sched = sched_for_stream(ds, stream);
  const double scale = static_cast<double>(q_descale) * k_descale / std::sqrt(static_cast<double>(d));
  p.scale_log2 = static_cast<float>(1.4426950408889634 * scale);
  p.out_scale = v_descale;
  cudaError_t e = cudaSuccess;
  if (!vt_in) e = launch_fp8_v_transpose(static_cast<const uint8_t*>(v), vt, B, n, n_pad, Hk, stream);
  if (e == cudaSuccess) e = launch_forward_fp8(p, d, stream);
  if (vt) cudaFreeAsync(vt, stream);
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

bool aligned_all(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p || !aligned16(p)) return false;
  return true;
}

// The tensor-core backward step alone: caller-owned delta and dq_acc.
int bwd_main_impl(int mode, const void* q, const void* k, const void* v, const void* dout,
                  const float* lse, const float* delta, float* dq_acc, void* dk, void* dv, int B,
                  int n, int H, int Hk, int d, int bs, cudaStream_t stream,
                  unsigned* dq_sem = nullptr, int pass = 0) {
  int rc = check_common(B, n, H, d, bs);
  if (rc) return rc;
  const int G = kv_group_of(H, Hk);
  if (G == 0) return DFA_EINVAL;
  if (B == 0) return DFA_OK;
  if (!aligned_all({q, k, v, dout, dq_acc, dk, dv}) || !lse || !delta ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(delta) & 3u))
    return DFA_EINVAL;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds))) return rc;
  TileShape ts;
  tile_shape_for(d, &ts);
  const long long halves = launch_halves(mode, B);
  BwdParams p{};
  if ((rc = make_map(&p.tm_q, q, halves, n, H, d, ts.bwd_bm))) return rc;
  if ((rc = make_map(&p.tm_do, dout, halves, n, H, d, ts.bwd_bm))) return rc;
  if ((rc = make_map(&p.tm_k, k, halves, n, Hk, d, ts.bwd_bn))) return rc;
  if ((rc = make_map(&p.tm_v, v, halves, n, Hk, d, ts.bwd_bn))) return rc;
  // dq accumulator boxes of the bulk reduce-adds, one per warp: a
  // warpgroup's queries of a tile x 32 head dims (headdim 128) or 16 (64)
  if ((d == 128 || d == 64) &&
      (rc = make_map_f32(&p.tm_dq, dq_acc, halves, n, H, d, ts.bwd_bm / kBwd2WarpgroupsD128,
                         false, d == 64 ? 16 : 32)))
    return rc;
  if (d == 128 && ((rc = make_map(&p.tm_dk, dk, halves, n, Hk, d, 32)) ||
                   (rc = make_map(&p.tm_dv, dv, halves, n, Hk, d, 32))))
    return rc;
  p.lse = lse;
  p.delta = delta;
  p.dq_acc = dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.status = ds->status;
  p.B = B;
  p.n = n;
  p.H = H;
  p.Hk = Hk;
  p.kv_group = G;
  p.bs = bs < n ? bs : n;
  p.mode = mode;
  p.k_tiles = cdiv(n, ts.bwd_bn);
  // per (batch, key/value head), or (sequence, key/value head): k, v (bf16)
  // and, for each of its G query heads, q, dout (bf16) and the float32 dq
  // accumulator
  p.group = l2_group((4LL + 8LL * G) * (mode == MODE_CAUSAL ? 1 : 2) * n * d, ds->l2_bytes,
                     B * Hk);
  p.sched = sched_for_stream(ds, stream);
  p.items = 0;  // set by the launcher
  p.dq_sem = dq_sem;
  p.sem_rows = static_cast<int>(halves * n);
  p.pass = pass;
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  const cudaError_t e = launch_backward(p, d, stream);
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

// delta = rowsum(dout * out) over B groups of `rows` rows, laid out (B, H,
// rows): rows = 2n for diffusion samples, n for causal sequences.
int check_rows(int B, int rows, int H, int d) {
  if (B < 0 || rows < 1 || rows > (1 << 30) || H < 1) return DFA_EINVAL;
  if (d != 64 && d != 128 && d != 256) return DFA_EUNSUPPORTED;
  return DFA_OK;
}

// The tensor-core backward step, with the noisy-diagonal specialisation
// when asked and applicable (diffusion mode, no block crossing a key tile):
// the pass over the noisy key tiles, which stores the noisy queries' first
// dQ contribution, then the pass over the clean key tiles; otherwise the
// single pass over every key tile.
int bwd_main_passes(int mode, const void* q, const void* k, const void* v, const void* dout,
                    const float* lse, const float* delta, float* dq_acc, void* dk, void* dv,
                    int B, int n, int H, int Hk, int d, int bs, cudaStream_t stream, bool diag,
                    unsigned* dq_sem = nullptr) {
  TileShape ts;
  if (diag && !dq_sem && mode == MODE_DIFFUSION && n >= 1 && bs >= 1 && tile_shape_for(d, &ts) &&
      diag_pass_applies(n, bs < n ? bs : n, ts.bwd_bn)) {
    int rc = bwd_main_impl(mode, q, k, v, dout, lse, delta, dq_acc, dk, dv, B, n, H, Hk, d, bs,
                           stream, nullptr, 2);
    if (rc) return rc;
    return bwd_main_impl(mode, q, k, v, dout, lse, delta, dq_acc, dk, dv, B, n, H, Hk, d, bs,
                         stream, nullptr, 1);
  }
  return bwd_main_impl(mode, q, k, v, dout, lse, delta, dq_acc, dk, dv, B, n, H, Hk, d, bs, stream,
                       dq_sem, 0);
}

int preprocess_impl(const void* out, const void* dout, float* delta, float* dq_acc, int B,
                    int rows, int H, int d, cudaStream_t stream) {
  int rc = check_rows(B, rows, H, d);
  if (rc) return rc;
  if (B == 0) return DFA_OK;
  if (!aligned_all({out, dout}) || (dq_acc && !aligned16(dq_acc)) || !delta ||
      (reinterpret_cast<uintptr_t>(delta) & 3u))
    return DFA_EINVAL;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds))) return rc;
  const cudaError_t e =
      launch_bwd_preprocess(static_cast<const __nv_bfloat16*>(out),
                            static_cast<const __nv_bfloat16*>(dout), delta, dq_acc, B, rows, H, d,
                            stream);
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

// dq = bf16(dq_acc) over B groups of `rows` rows of H * d elements.
int convert_impl(const float* dq_acc, void* dq, int B, int rows, int H, int d,
                 cudaStream_t stream) {
  int rc = check_rows(B, rows, H, d);
  if (rc) return rc;
  if (B == 0) return DFA_OK;
  if (!aligned_all({dq_acc, dq})) return DFA_EINVAL;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds))) return rc;
  const long long elems = static_cast<long long>(B) * rows * H * d;
  const cudaError_t e = launch_dq_convert(dq_acc, static_cast<__nv_bfloat16*>(dq), elems, stream);
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

// Full backward: stream-ordered scratch, then the three steps.
// Counters of the deterministic mode: one per (head-dim part, head, row),
// zero, stream-ordered.
int alloc_dq_sem(size_t head_rows, cudaStream_t stream, unsigned** sem) {
  const size_t bytes = 2 * head_rows * sizeof(unsigned);
  if (cudaMallocAsync(reinterpret_cast<void**>(sem), bytes, stream) != cudaSuccess)
    return DFA_ECUDA;
  if (cudaMemsetAsync(*sem, 0, bytes, stream) != cudaSuccess) {
    cudaFreeAsync(*sem, stream);
    return DFA_ECUDA;
  }
  return DFA_OK;
}

int backward_impl(int mode, const void* q, const void* k, const void* v, const void* out,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int n,
                  int H, int Hk, int d, int bs, cudaStream_t stream, bool det = false,
                  bool diag = false) {
  int rc = check_common(B, n, H, d, bs);
  if (rc) return rc;
  if (kv_group_of(H, Hk) == 0) return DFA_EINVAL;
  if (B == 0) return DFA_OK;
  if (!aligned_all({q, k, v, out, dout, dq, dk, dv}) || !lse ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return DFA_EINVAL;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds))) return rc;
  // rows per sample (two halves) or, causal, per sequence
  const int L = mode == MODE_CAUSAL ? n : 2 * n;
  const size_t elems = static_cast<size_t>(B) * L * H * d;
  const size_t rows = static_cast<size_t>(B) * H * L;
  float* dq_acc = nullptr;
  float* delta = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&dq_acc), elems * sizeof(float), stream) !=
      cudaSuccess)
    return DFA_ECUDA;
  if (cudaMallocAsync(reinterpret_cast<void**>(&delta), rows * sizeof(float), stream) !=
      cudaSuccess) {
    cudaFreeAsync(dq_acc, stream);
    return DFA_ECUDA;
  }
  unsigned* sem = nullptr;
  if (det && (rc = alloc_dq_sem(rows, stream, &sem))) {
    cudaFreeAsync(delta, stream);
    cudaFreeAsync(dq_acc, stream);
    return rc;
  }
  rc = preprocess_impl(out, dout, delta, dq_acc, B, L, H, d, stream);
  if (!rc)
    rc = bwd_main_passes(mode, q, k, v, dout, lse, delta, dq_acc, dk, dv, B, n, H, Hk, d, bs,
                         stream, diag, sem);
  if (!rc) rc = convert_impl(dq_acc, dq, B, L, H, d, stream);
  if (sem) cudaFreeAsync(sem, stream);
  cudaFreeAsync(delta, stream);
  cudaFreeAsync(dq_acc, stream);
  return rc;
}

// ------------------------------------------------------------ varlen
// Packed batches: sample b is rows [cu[b], cu[b+1]) of the packed tensors,
// its noisy half first, so every length cu[b+1] - cu[b] is even.  The
// non-empty samples are scheduled longest first ("Fast Diffusion
// Attention": varlen batches), one slot each.

// Check cu_seqlens (host, batch + 1 entries) and return the packed rows.
int varlen_rows(const int* cu, int batch, int* rows) {
  if (!cu || batch < 0 || cu[0] != 0) return DFA_EINVAL;
  for (int b = 0; b < batch; ++b) {
    const long long len = static_cast<long long>(cu[b + 1]) - cu[b];
    if (len < 0 || (len & 1)) return DFA_EINVAL;
  }
  if (cu[batch] > (1 << 30)) return DFA_EINVAL;
  *rows = cu[batch];
  return DFA_OK;
}

// Slots of the non-empty samples, longest first (ties in sample order), for
// a pass whose work unit is (head, half, tile of `tile` rows): 2 * heads *
// cdiv(n, tile) units per sample.  `bytes_per_pos` is what one position of
// one head brings into L2, for the L2 head groups inside a sample.
int varlen_schedule(const int* cu, int batch, int heads, int tile, long long bytes_per_pos,
                    long long l2_bytes, std::vector<VarlenSlot>* slots, int* units) {
  std::vector<int> order;
  for (int b = 0; b < batch; ++b)
    if (cu[b + 1] > cu[b]) order.push_back(b);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    return cu[a + 1] - cu[a] > cu[b + 1] - cu[b];
  });
  slots->clear();
  long long off = 0;
  for (int b : order) {
    const int n = (cu[b + 1] - cu[b]) / 2;
    VarlenSlot sl;
    sl.b = b;
    sl.n = n;
    sl.row0 = cu[b];
    sl.group = l2_group(bytes_per_pos * 2 * n, l2_bytes, heads);
    sl.off = static_cast<int>(off);
    slots->push_back(sl);
    off += 2LL * heads * cdiv(n, tile);
    if (off > 0x7fffffffLL) return DFA_EINVAL;
  }
  *units = static_cast<int>(off);
  return DFA_OK;
}

// Tensor maps of every slot's sample: (d, H, n, 2, 1) views starting at
// the sample's first row, so that rows past the end of a half read zero.
// Forward: q (box bm rows), k, v (box bn rows); backward also dout (bm) and,
// if dq_acc is given, the float32 accumulator (box dq_rows rows of 32); if
// dk / dv are given, those (box 32 rows), which the stores go through.
int varlen_maps(const std::vector<VarlenSlot>& slots, const void* q, const void* k,
                const void* v, const void* dout, int H, int Hk, int d, int bm, int bn,
                std::vector<VarlenMaps>* maps, const float* dq_acc = nullptr, int dq_rows = 0,
                const void* dk = nullptr, const void* dv = nullptr, int dq_inner = 32) {
  maps->assign(slots.size(), VarlenMaps{});
  const size_t qrow = static_cast<size_t>(H) * d * 2, krow = static_cast<size_t>(Hk) * d * 2;
  for (size_t i = 0; i < slots.size(); ++i) {
    const VarlenSlot& sl = slots[i];
    VarlenMaps& m = (*maps)[i];
    const char* qb = static_cast<const char*>(q) + sl.row0 * qrow;
    int rc;
    if ((rc = make_map(&m.q, qb, 2, sl.n, H, d, bm))) return rc;
    if ((rc = make_map(&m.k, static_cast<const char*>(k) + sl.row0 * krow, 2, sl.n, Hk, d, bn)))
      return rc;
    if ((rc = make_map(&m.v, static_cast<const char*>(v) + sl.row0 * krow, 2, sl.n, Hk, d, bn)))
      return rc;
    if (dout &&
        (rc = make_map(&m.dout, static_cast<const char*>(dout) + sl.row0 * qrow, 2, sl.n, H, d,
                       bm)))
      return rc;
    if (dq_acc && (rc = make_map_f32(&m.dq, dq_acc + static_cast<size_t>(sl.row0) * H * d, 2,
                                     sl.n, H, d, dq_rows, false, dq_inner)))
      return rc;
    if (dk && (rc = make_map(&m.dk, static_cast<const char*>(dk) + sl.row0 * krow, 2, sl.n, Hk,
                             d, 32)))
      return rc;
    if (dv && (rc = make_map(&m.dv, static_cast<const char*>(dv) + sl.row0 * krow, 2, sl.n, Hk,
                             d, 32)))
      return rc;
  }
  return DFA_OK;
}

// Copy the slot table and the slots' tensor maps to stream-ordered device
// memory: maps first (at the allocation's 256-byte aligned start), then the table.  One allocation,
// freed by the caller with cudaFreeAsync(*dmaps) after the launch that reads
// it.
int upload_slots(const std::vector<VarlenSlot>& slots, const std::vector<VarlenMaps>& maps,
                 cudaStream_t stream, VarlenMaps** dmaps, VarlenSlot** dslots) {
  const size_t mbytes = maps.size() * sizeof(VarlenMaps);
  const size_t sbytes = slots.size() * sizeof(VarlenSlot);
  std::vector<char> host(mbytes + sbytes);
  std::memcpy(host.data(), maps.data(), mbytes);
  std::memcpy(host.data() + mbytes, slots.data(), sbytes);
  void* d = nullptr;
  if (cudaMallocAsync(&d, host.size(), stream) != cudaSuccess) return DFA_ECUDA;
  if (cudaMemcpyAsync(d, host.data(), host.size(), cudaMemcpyHostToDevice, stream) !=
      cudaSuccess) {
    cudaFreeAsync(d, stream);
    return DFA_ECUDA;
  }
  // From pageable memory the copy has staged the host buffer by the time it
  // returns, so the buffer may go out of scope now.
  *dmaps = static_cast<VarlenMaps*>(d);
  *dslots = reinterpret_cast<VarlenSlot*>(static_cast<char*>(d) + mbytes);
  return DFA_OK;
}

int check_varlen(int H, int Hk, int d, int bs) {
  if (H < 1 || bs < 1) return DFA_EINVAL;
  if (d != 64 && d != 128 && d != 256) return DFA_EUNSUPPORTED;
  if (kv_group_of(H, Hk) == 0) return DFA_EINVAL;
  return DFA_OK;
}

int forward_varlen_impl(const void* q, const void* k, const void* v, void* out, float* lse,
                        const int* cu, int batch, int H, int Hk, int d, int bs,
                        cudaStream_t stream) {
  int rc = check_varlen(H, Hk, d, bs);
  if (rc) return rc;
  int rows = 0;
  if ((rc = varlen_rows(cu, batch, &rows))) return rc;
  if (rows == 0) return DFA_OK;
  if (!q || !k || !v || !out || !lse) return DFA_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return DFA_EINVAL;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds))) return rc;
  TileShape ts;
  tile_shape_for(d, &ts);
  std::vector<VarlenSlot> slots;
  int units = 0;
  // q, k, v and out of one head
  if ((rc = varlen_schedule(cu, batch, H, ts.fwd_bm, 8LL * d, ds->l2_bytes, &slots, &units)))
    return rc;
  // q, k, v through per-sample maps; out through a map of the packed tensor
  std::vector<VarlenMaps> maps;
  if ((rc = varlen_maps(slots, q, k, v, nullptr, H, Hk, d, ts.fwd_bm, ts.fwd_bn, &maps)))
    return rc;
  FwdParams p{};
  if ((rc = make_map(&p.tm_o, out, 1, rows, H, d, ts.fwd_bm, true))) return rc;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = ds->status;
  p.B = 1;
  p.n = 1;  // per sample: the slot table
  p.H = H;
  p.kv_group = H / Hk;
  p.bs = bs;  // clamped per sample by the kernels
  p.mode = MODE_DIFFUSION;
  p.q_tiles = 1;
  p.group = 1;
  p.sched = sched_for_stream(ds, stream);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  p.vl_slots = static_cast<int>(slots.size());
  p.rows = rows;
  p.items = units;
  VarlenSlot* dslots = nullptr;
  VarlenMaps* dmaps = nullptr;
  if ((rc = upload_slots(slots, maps, stream, &dmaps, &dslots))) return rc;
  p.vl = dslots;
  p.vl_maps = dmaps;
  const cudaError_t e = launch_forward(p, d, stream);
  cudaFreeAsync(dmaps, stream);
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

int backward_varlen_impl(const void* q, const void* k, const void* v, const void* out,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         const int* cu, int batch, int H, int Hk, int d, int bs,
                         cudaStream_t stream, bool det = false) {
  int rc = check_varlen(H, Hk, d, bs);
  if (rc) return rc;
  int rows = 0;
  if ((rc = varlen_rows(cu, batch, &rows))) return rc;
  if (rows == 0) return DFA_OK;
  if (!aligned_all({q, k, v, out, dout, dq, dk, dv}) || !lse ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return DFA_EINVAL;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds))) return rc;
  const int G = H / Hk;
  TileShape ts;
  tile_shape_for(d, &ts);
  std::vector<VarlenSlot> slots;
  int units = 0;
  // per key/value head: k, v and, for each of its G query heads, q, dout
  // (bf16) and the float32 dq accumulator
  if ((rc = varlen_schedule(cu, batch, Hk, ts.bwd_bn, (4LL + 8LL * G) * d, ds->l2_bytes, &slots,
                            &units)))
    return rc;
  const size_t elems = static_cast<size_t>(rows) * H * d;
  float* dq_acc = nullptr;
  float* delta = nullptr;
  VarlenSlot* dslots = nullptr;
  VarlenMaps* dmaps = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&dq_acc), elems * sizeof(float), stream) !=
      cudaSuccess)
    return DFA_ECUDA;
  if (cudaMallocAsync(reinterpret_cast<void**>(&delta),
                      static_cast<size_t>(rows) * H * sizeof(float), stream) != cudaSuccess) {
    cudaFreeAsync(dq_acc, stream);
    return DFA_ECUDA;
  }
  // q, dout, k, v, the dq accumulator (headdim 64, 128) and (128) dk, dv through
  // per-sample maps (rows past a half read zero; reduce-adds and stores past
  // a half are skipped)
  std::vector<VarlenMaps> maps;
  if ((rc = varlen_maps(slots, q, k, v, dout, H, Hk, d, ts.bwd_bm, ts.bwd_bn, &maps,
                        d == 128 || d == 64 ? dq_acc : nullptr,
                        ts.bwd_bm / kBwd2WarpgroupsD128, d == 128 ? dk : nullptr,
                        d == 128 ? dv : nullptr, d == 64 ? 16 : 32)) ||
      (rc = upload_slots(slots, maps, stream, &dmaps, &dslots))) {
    cudaFreeAsync(delta, stream);
    cudaFreeAsync(dq_acc, stream);
    return rc;
  }
  unsigned* sem = nullptr;
  if (det && (rc = alloc_dq_sem(static_cast<size_t>(rows) * H, stream, &sem))) {
    cudaFreeAsync(dmaps, stream);
    cudaFreeAsync(delta, stream);
    cudaFreeAsync(dq_acc, stream);
    return rc;
  }
  // delta = rowsum(dout * out) as (heads, rows), the layout of lse; dq_acc = 0
  cudaError_t e = launch_bwd_preprocess(static_cast<const __nv_bfloat16*>(out),
                                        static_cast<const __nv_bfloat16*>(dout), delta, dq_acc,
                                        1, rows, H, d, stream);
  if (e == cudaSuccess) {
    BwdParams p{};
    p.lse = lse;
    p.delta = delta;
    p.dq_acc = dq_acc;
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.status = ds->status;
    p.B = 1;
    p.n = 1;  // per sample: the slot table
    p.H = H;
    p.Hk = Hk;
    p.kv_group = G;
    p.bs = bs;  // clamped per sample by the kernels
    p.mode = MODE_DIFFUSION;
    p.k_tiles = 1;
    p.group = 1;
    p.sched = sched_for_stream(ds, stream);
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    p.vl = dslots;
    p.vl_maps = dmaps;
    p.vl_slots = static_cast<int>(slots.size());
    p.rows = rows;
    p.units = units;
    p.dq_sem = sem;
    p.sem_rows = rows;
    e = launch_backward(p, d, stream);
  }
  if (e == cudaSuccess)
    e = launch_dq_convert(dq_acc, static_cast<__nv_bfloat16*>(dq), static_cast<long long>(elems),
                          stream);
  if (sem) cudaFreeAsync(sem, stream);
  cudaFreeAsync(dmaps, stream);
  cudaFreeAsync(delta, stream);
  cudaFreeAsync(dq_acc, stream);
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

}  // namespace

// For the other translation units of the library (see params.cuh).
int check_device(unsigned long long* ctx_id) {
  DeviceState* ds = nullptr;
  const int rc = device_state(&ds);
  if (rc) return rc;
  if (ctx_id) *ctx_id = ds->ctx_id;
  return DFA_OK;
}

int record_cuda_failure(cudaError_t e) { return cuda_fail(e); }

int check_backward_args(int B, int n, int H, int d, int bs) { return check_common(B, n, H, d, bs); }

}  // namespace dfa

using namespace dfa;

extern "C" {

int dfa_version(void) { return 100; }

const char* dfa_error_string(int code) {
  switch (code) {
    case DFA_OK: return "ok";
    case DFA_EINVAL: return "invalid argument";
    case DFA_EUNSUPPORTED: return "unsupported head dimension or device";
    case DFA_ECUDA: return "CUDA call failed";
    case DFA_ETIMEOUT: return "a kernel wait timed out";
    case DFA_EDEVICE: return "a kernel index check failed";
    default: return "unknown error";
  }
}

int dfa_forward(const void* q, const void* k, const void* v, void* out, float* lse, int batch,
                int n, int heads, int headdim, int block_size, dfa_stream_t stream) {
  return forward_impl(MODE_DIFFUSION, q, k, v, out, lse, nullptr, batch, n, heads, heads, headdim,
                      block_size, static_cast<cudaStream_t>(stream));
}

int dfa_forward_gqa(const void* q, const void* k, const void* v, void* out, float* lse, int batch,
                    int n, int heads, int kv_heads, int headdim, int block_size,
                    dfa_stream_t stream) {
  return forward_impl(MODE_DIFFUSION, q, k, v, out, lse, nullptr, batch, n, heads, kv_heads,
                      headdim, block_size, static_cast<cudaStream_t>(stream));
}

int dfa_backward(const void* q, const void* k, const void* v, const void* out, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int batch, int n, int heads,
                 int headdim, int block_size, dfa_stream_t stream) {
  return backward_impl(MODE_DIFFUSION, q, k, v, out, dout, lse, dq, dk, dv, batch, n, heads,
                       heads, headdim, block_size, static_cast<cudaStream_t>(stream));
}

int dfa_backward_gqa(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv, int batch,
                     int n, int heads, int kv_heads, int headdim, int block_size,
                     dfa_stream_t stream) {
  return backward_impl(MODE_DIFFUSION, q, k, v, out, dout, lse, dq, dk, dv, batch, n, heads,
                       kv_heads, headdim, block_size, static_cast<cudaStream_t>(stream));
}

int dfa_forward_varlen(const void* q, const void* k, const void* v, void* out, float* lse,
                       const int* cu_seqlens, int batch, int heads, int kv_heads, int headdim,
                       int block_size, dfa_stream_t stream) {
  return forward_varlen_impl(q, k, v, out, lse, cu_seqlens, batch, heads, kv_heads, headdim,
                             block_size, static_cast<cudaStream_t>(stream));
}

int dfa_backward_varlen(const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        const int* cu_seqlens, int batch, int heads, int kv_heads, int headdim,
                        int block_size, dfa_stream_t stream) {
  return backward_varlen_impl(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens, batch, heads,
                              kv_heads, headdim, block_size, static_cast<cudaStream_t>(stream));
}

int dfa_forward_fp8(const void* q, const void* k, const void* v, void* out, float* lse,
                    float q_descale, float k_descale, float v_descale, int batch, int n,
                    int heads, int kv_heads, int headdim, int block_size, dfa_stream_t stream) {
  return forward_fp8_impl(q, k, v, out, lse, q_descale, k_descale, v_descale, batch, n, heads,
                          kv_heads, headdim, block_size, static_cast<cudaStream_t>(stream));
}

long long dfa_fp8_vt_bytes(int batch, int n, int kv_heads, int headdim) {
  if (batch < 0 || n < 1 || kv_heads < 1 || headdim != 128) return DFA_EINVAL;
  return static_cast<long long>(batch) * kv_heads * 128 * 2 * ((n + 15) / 16 * 16);
}

int dfa_fp8_transpose_v(const void* v, void* vt, int batch, int n, int kv_heads, int headdim,
                        dfa_stream_t stream) {
  if (dfa_fp8_vt_bytes(batch, n, kv_heads, headdim) < 0) return DFA_EINVAL;
  if (batch == 0) return DFA_OK;
  if (!v || !vt || !aligned16(v) || !aligned16(vt)) return DFA_EINVAL;
  DeviceState* ds = nullptr;
  const int rc = device_state(&ds);
  if (rc) return rc;
  const cudaError_t e =
      launch_fp8_v_transpose(static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), batch, n,
                             (n + 15) / 16 * 16, kv_heads, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

int dfa_forward_fp8_vt(const void* q, const void* k, const void* vt, void* out, float* lse,
                       float q_descale, float k_descale, float v_descale, int batch, int n,
                       int heads, int kv_heads, int headdim, int block_size,
                       dfa_stream_t stream) {
  if (!vt) return DFA_EINVAL;
  return forward_fp8_impl(q, k, nullptr, out, lse, q_descale, k_descale, v_descale, batch, n,
                          heads, kv_heads, headdim, block_size,
                          static_cast<cudaStream_t>(stream), vt);
}

int dfa_backward_ex(const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv,
                    const int* cu_seqlens, int batch, int n, int heads, int kv_heads, int headdim,
                    int block_size, int flags, dfa_stream_t stream) {
  if (flags & ~(DFA_DETERMINISTIC | DFA_NOISY_DIAG_PASS)) return DFA_EINVAL;
  const bool det = (flags & DFA_DETERMINISTIC) != 0;
  const bool diag = (flags & DFA_NOISY_DIAG_PASS) != 0;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cu_seqlens)
    return backward_varlen_impl(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens, batch, heads,
                                kv_heads, headdim, block_size, s, det);
  return backward_impl(MODE_DIFFUSION, q, k, v, out, dout, lse, dq, dk, dv, batch, n, heads,
                       kv_heads, headdim, block_size, s, det, diag);
}

// Causal attention on (batch, seqlen, heads, headdim): the diffusion kernels
// in their causal mode, every sequence one "half" of seqlen rows that
// attends causally to itself.
int dfa_causal_forward(const void* q, const void* k, const void* v, void* out, float* lse,
                       int batch, int seqlen, int heads, int headdim, dfa_stream_t stream) {
  if (batch < 0 || seqlen < 1) return DFA_EINVAL;
  return forward_impl(MODE_CAUSAL, q, k, v, out, lse, nullptr, batch, seqlen, heads, heads,
                      headdim, 1, static_cast<cudaStream_t>(stream));
}

int dfa_causal_backward(const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        int batch, int seqlen, int heads, int headdim, dfa_stream_t stream) {
  if (batch < 0 || seqlen < 1) return DFA_EINVAL;
  return backward_impl(MODE_CAUSAL, q, k, v, out, dout, lse, dq, dk, dv, batch, seqlen, heads,
                       heads, headdim, 1, static_cast<cudaStream_t>(stream));
}

int dfa_fwd_main(const void* q, const void* k, const void* v, void* out, float* lse,
                 float* dq_acc, int batch, int n, int heads, int headdim, int block_size, int mode,
                 dfa_stream_t stream) {
  if (mode != MODE_DIFFUSION && mode != MODE_CAUSAL) return DFA_EINVAL;
  return forward_impl(mode, q, k, v, out, lse, dq_acc, batch, n, heads, heads, headdim,
                      mode == MODE_CAUSAL ? 1 : block_size, static_cast<cudaStream_t>(stream));
}

int dfa_fwd_main_gqa(const void* q, const void* k, const void* v, void* out, float* lse,
                     float* dq_acc, int batch, int n, int heads, int kv_heads, int headdim,
                     int block_size, int mode, dfa_stream_t stream) {
  if (mode != MODE_DIFFUSION && mode != MODE_CAUSAL) return DFA_EINVAL;
  return forward_impl(mode, q, k, v, out, lse, dq_acc, batch, n, heads, kv_heads, headdim,
                      mode == MODE_CAUSAL ? 1 : block_size, static_cast<cudaStream_t>(stream));
}

int dfa_bwd_main_ex(const void* q, const void* k, const void* v, const void* dout,
                    const float* lse, const float* delta, float* dq_acc, void* dk, void* dv,
                    int batch, int n, int heads, int kv_heads, int headdim, int block_size,
                    int mode, int flags, dfa_stream_t stream) {
  if (mode != MODE_DIFFUSION && mode != MODE_CAUSAL) return DFA_EINVAL;
  if (flags & ~DFA_NOISY_DIAG_PASS) return DFA_EINVAL;
  return bwd_main_passes(mode, q, k, v, dout, lse, delta, dq_acc, dk, dv, batch, n, heads,
                         kv_heads, headdim, mode == MODE_CAUSAL ? 1 : block_size,
                         static_cast<cudaStream_t>(stream), (flags & DFA_NOISY_DIAG_PASS) != 0);
}

int dfa_bwd_main_gqa(const void* q, const void* k, const void* v, const void* dout,
                     const float* lse, const float* delta, float* dq_acc, void* dk, void* dv,
                     int batch, int n, int heads, int kv_heads, int headdim, int block_size,
                     int mode, dfa_stream_t stream) {
  if (mode != MODE_DIFFUSION && mode != MODE_CAUSAL) return DFA_EINVAL;
  return bwd_main_impl(mode, q, k, v, dout, lse, delta, dq_acc, dk, dv, batch, n, heads,
                       kv_heads, headdim, mode == MODE_CAUSAL ? 1 : block_size,
                       static_cast<cudaStream_t>(stream));
}

int dfa_bwd_preprocess(const void* out, const void* dout, float* delta, float* dq_acc, int batch,
                       int n, int heads, int headdim, dfa_stream_t stream) {
  if (n < 1 || n > (1 << 29)) return DFA_EINVAL;
  return preprocess_impl(out, dout, delta, dq_acc, batch, 2 * n, heads, headdim,
                         static_cast<cudaStream_t>(stream));
}

int dfa_bwd_preprocess_ex(const void* out, const void* dout, float* delta, float* dq_acc,
                          int batch, int n, int heads, int headdim, int mode,
                          dfa_stream_t stream) {
  if (mode != MODE_DIFFUSION && mode != MODE_CAUSAL) return DFA_EINVAL;
  if (n < 1 || n > (1 << 29)) return DFA_EINVAL;
  return preprocess_impl(out, dout, delta, dq_acc, batch, mode == MODE_CAUSAL ? n : 2 * n, heads,
                         headdim, static_cast<cudaStream_t>(stream));
}

int dfa_bwd_main(const void* q, const void* k, const void* v, const void* dout, const float* lse,
                 const float* delta, float* dq_acc, void* dk, void* dv, int batch, int n,
                 int heads, int headdim, int block_size, int mode, dfa_stream_t stream) {
  if (mode != MODE_DIFFUSION && mode != MODE_CAUSAL) return DFA_EINVAL;
  return bwd_main_impl(mode, q, k, v, dout, lse, delta, dq_acc, dk, dv, batch, n, heads, heads,
                       headdim, mode == MODE_CAUSAL ? 1 : block_size,
                       static_cast<cudaStream_t>(stream));
}

int dfa_bwd_dq_convert(const float* dq_acc, void* dq, int batch, int n, int heads, int headdim,
                       dfa_stream_t stream) {
  if (n < 1 || n > (1 << 29)) return DFA_EINVAL;
  return convert_impl(dq_acc, dq, batch, 2 * n, heads, headdim, static_cast<cudaStream_t>(stream));
}

int dfa_bwd_dq_convert_ex(const float* dq_acc, void* dq, int batch, int n, int heads,
                          int headdim, int mode, dfa_stream_t stream) {
  if (mode != MODE_DIFFUSION && mode != MODE_CAUSAL) return DFA_EINVAL;
  if (n < 1 || n > (1 << 29)) return DFA_EINVAL;
  return convert_impl(dq_acc, dq, batch, mode == MODE_CAUSAL ? n : 2 * n, heads, headdim,
                      static_cast<cudaStream_t>(stream));
}

int dfa_selftest_wait_timeout(int limit_us, dfa_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return DFA_EINVAL;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc) return rc;
  const cudaError_t e = launch_selftest_wait(ds->status, 1000ull * limit_us,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DFA_OK : cuda_fail(e);
}

const char* dfa_last_cuda_error(void) { return cudaGetErrorString(t_last_error); }

int dfa_status(dfa_stream_t stream) {
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DFA_ECUDA;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_dfa_status, sizeof(word)) != cudaSuccess) return DFA_ECUDA;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_dfa_status, &zero, sizeof(zero)) != cudaSuccess) return DFA_ECUDA;
  if (word & kStatusTimeout) return DFA_ETIMEOUT;
  if (word & kStatusIndex) return DFA_EDEVICE;
  return DFA_OK;
}

static int encode_segments(const Segment* seg, int cnt, int* out) {
  for (int i = 0; i < cnt; ++i) {
    out[4 * i + 0] = seg[i].half;
    out[4 * i + 1] = seg[i].rule;
    out[4 * i + 2] = seg[i].t_begin;
    out[4 * i + 3] = seg[i].t_end;
  }
  return cnt;
}

static bool geom_args_ok(int mode, int n, int bs, int bm, int bn, int half) {
  return (mode == MODE_DIFFUSION || mode == MODE_CAUSAL) && n >= 1 && bs >= 1 && bm >= 1 &&
         bn >= 1 && (half == 0 || half == 1);
}

int dfa_fwd_segments(int mode, int n, int block_size, int block_m, int block_n, int q_half,
                     int q_tile, int* seg) {
  if (!seg || !geom_args_ok(mode, n, block_size, block_m, block_n, q_half) || q_tile < 0)
    return DFA_EINVAL;
  Segment s[2];
  const int cnt = fwd_segments(mode, n, block_size < n ? block_size : n, block_m, block_n, q_half,
                               q_tile, s);
  return encode_segments(s, cnt, seg);
}

int dfa_bwd_segments(int mode, int n, int block_size, int block_m, int block_n, int k_half,
                     int k_tile, int* seg) {
  if (!seg || !geom_args_ok(mode, n, block_size, block_m, block_n, k_half) || k_tile < 0)
    return DFA_EINVAL;
  Segment s[2];
  const int cnt = bwd_segments(mode, n, block_size < n ? block_size : n, block_m, block_n, k_half,
                               k_tile, s);
  return encode_segments(s, cnt, seg);
}

int dfa_tile_full(int rule, int n, int block_size, int q_start, int block_m, int k_start,
                  int block_n) {
  if (n < 1 || block_size < 1 || block_m < 1 || block_n < 1) return DFA_EINVAL;
  return tile_full(rule, n, block_size < n ? block_size : n, q_start, block_m, k_start, block_n)
             ? 1
             : 0;
}

long long dfa_tile_visits(int mode, int n, int block_size, int block_m, int block_n, int pass) {
  if (!geom_args_ok(mode, n, block_size, block_m, block_n, 0) || (pass != 0 && pass != 1))
    return DFA_EINVAL;
  const int bs = block_size < n ? block_size : n;
  long long total = 0;
  const int tiles = cdiv(n, pass == 0 ? block_m : block_n);
  for (int half = 0; half < 2; ++half)
    for (int t = 0; t < tiles; ++t) {
      Segment s[2];
      const int cnt = pass == 0 ? fwd_segments(mode, n, bs, block_m, block_n, half, t, s)
                                : bwd_segments(mode, n, bs, block_m, block_n, half, t, s);
      for (int i = 0; i < cnt; ++i) total += s[i].t_end - s[i].t_begin;
    }
  return total;
}

int dfa_work_item(int pass, int mode, int w, int batch, int heads, int tiles, int group,
                  int* item) {
  if (pass < 0 || pass > 3 || (mode != MODE_DIFFUSION && mode != MODE_CAUSAL) || batch < 1 ||
      heads < 1 || tiles < 1 || group < 1 || !item)
    return DFA_EINVAL;
  if (pass >= 2 && mode != MODE_DIFFUSION) return DFA_EINVAL;
  const long long items = pass >= 2 ? static_cast<long long>(batch) * heads * tiles
                                    : pass_items(mode, batch, heads, tiles);
  if (items > 0x7fffffffLL || w < 0 || w >= items) return DFA_EINVAL;
  const WorkItem it = pass == 0   ? fwd_work(w, mode, batch, heads, tiles, group)
                      : pass == 1 ? bwd_work(w, mode, batch, heads, tiles, group)
                                  : bwd_work_pass(w, pass - 1, batch, heads, tiles, group);
  item[0] = it.b;
  item[1] = it.h;
  item[2] = it.half;
  item[3] = it.tile;
  return DFA_OK;
}

int dfa_tile_shape(int headdim, int* fwd_block_m, int* fwd_block_n, int* bwd_block_n,
                   int* bwd_block_m) {
  TileShape t;
  if (!tile_shape_for(headdim, &t)) return DFA_EUNSUPPORTED;
  if (fwd_block_m) *fwd_block_m = t.fwd_bm;
  if (fwd_block_n) *fwd_block_n = t.fwd_bn;
  if (bwd_block_n) *bwd_block_n = t.bwd_bn;
  if (bwd_block_m) *bwd_block_m = t.bwd_bm;
  return DFA_OK;
}

}  // extern "C"
