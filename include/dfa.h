/*
 * dfa.h - C ABI of libdfa: exact softmax attention under the block-diffusion
 * mask, forward and backward, on NVIDIA GB300 (sm_103a).
 *
 * The operation.  A sample is the concatenation [noisy | clean] of two halves
 * of n tokens ("Fast Diffusion Attention", section "Block diffusion in one
 * picture").  Positions inside a half are cut into blocks of block_size
 * tokens, starting at the first position of the half (the last block is
 * short when block_size does not divide n; block_size > n gives one block
 * per half).  With blk(p) the block of position p inside its half:
 *   noisy query i, noisy key j : visible iff blk(j) == blk(i)
 *   noisy query i, clean key j : visible iff blk(j) <  blk(i)
 *   clean query i, clean key j : visible iff blk(j) <= blk(i)
 *   clean query i, noisy key j : never visible.
 * out = softmax(scale * q k^T restricted to visible pairs) v, scale =
 * 1/sqrt(headdim); lse is the natural-log log-sum-exp of the scaled visible
 * scores of each row, kept for the recompute-based backward ("FlashAttention:
 * Exact Attention Without Materialization", section 4.5).  No score or
 * probability matrix is ever written to device memory.
 *
 * Layout.  Every q/k/v/out/dout/dq/dk/dv tensor is a contiguous row-major
 * bfloat16 array of shape (batch, 2n, heads, headdim): positions [0, n) are
 * the noisy half, [n, 2n) the clean half.  lse is a contiguous float32 array
 * of shape (batch, heads, 2n).  Every base pointer must be 16-byte aligned.
 * headdim must be 64, 128 or 256.
 *
 * Pointers.  All tensor pointers are DEVICE pointers on the current CUDA
 * device, owned by the caller; the library never frees or retains them.
 * `stream` is a cudaStream_t passed as an opaque pointer (NULL = the legacy
 * default stream).  All calls are asynchronous on that stream: a return of
 * DFA_OK means the work was enqueued.
 *
 * Concurrency.  The persistent kernels draw work items from a counter the
 * library keeps in device memory, one per stream (up to 256 streams per
 * device; past that the least recently added stream's counter is shared).
 * Each launch leaves its counter zero when it finishes, so launches on one
 * stream never interfere, and launches on different streams use different
 * counters.  A CUDA graph captured from a stream keeps that stream's counter:
 * do not replay it while other work of the same stream, or another replay
 * of it, is running.
 *
 * Errors.  Functions return 0 (DFA_OK) or a negative code below; nothing
 * else crosses the ABI.  Argument errors are detected on the host before any
 * launch.  Kernels never trap: every wait inside a kernel is bounded, and a
 * kernel that gives up records DFA_ETIMEOUT in a device status word that
 * dfa_status() reads.
 */
#ifndef DFA_H_
#define DFA_H_

#ifdef __cplusplus
extern "C" {
#endif

#define DFA_OK 0
#define DFA_EINVAL (-1)        /* bad shape, null or misaligned pointer      */
#define DFA_EUNSUPPORTED (-2)  /* headdim not supported, or device not sm_103 */
#define DFA_ECUDA (-3)         /* a CUDA runtime/driver call failed           */
#define DFA_ETIMEOUT (-4)      /* a kernel's bounded wait gave up             */
#define DFA_EDEVICE (-5)       /* a kernel's own index check failed           */

#define DFA_MODE_DIFFUSION 0   /* block-diffusion mask over [noisy | clean]   */
#define DFA_MODE_CAUSAL 1      /* causal mask inside each half (yardstick)    */

typedef void *dfa_stream_t;

/* Library version as 10000*major + 100*minor + patch. */
int dfa_version(void);

/* Human-readable name of a return code (static storage, never NULL). */
const char *dfa_error_string(int code);

/* Description of the CUDA error behind the calling thread's last DFA_ECUDA
 * from a kernel launch (static storage, never NULL). */
const char *dfa_last_cuda_error(void);

/*
 * Forward pass ("Fast Diffusion Attention", "Visit only the visible tiles";
 * "FlashAttention: Exact Attention Without Materialization", sections 4.1-4.2
 * and 5.1).  Reads q, k, v; writes out (batch, 2n, heads, headdim) bf16 and
 * lse (batch, heads, 2n) fp32.  n >= 1, block_size >= 1.  Allocates nothing.
 */
int dfa_forward(const void *q, const void *k, const void *v, void *out, float *lse,
                int batch, int n, int heads, int headdim, int block_size,
                dfa_stream_t stream);

/*
 * Backward pass ("FlashAttention: Exact Attention Without Materialization",
 * section 4.5; the key-tile enumeration of "Visit only the visible tiles").
 * Given q, k, v, the forward's out and lse, and dout, writes dq, dk, dv
 * (batch, 2n, heads, headdim) bf16: the gradients of sum(dout * out).
 * Scratch: a float32 dq accumulator of the shape of q and a float32 row
 * vector D = rowsum(dout * out) of the shape of lse are allocated and freed
 * stream-ordered on `stream` (cudaMallocAsync / cudaFreeAsync).
 */
int dfa_backward(const void *q, const void *k, const void *v, const void *out,
                 const void *dout, const float *lse, void *dq, void *dk, void *dv,
                 int batch, int n, int heads, int headdim, int block_size,
                 dfa_stream_t stream);

/*
 * Grouped key/value heads (multi-query and grouped-query attention, which
 * "Fast Diffusion Attention" lists among the supported shapes, with a
 * "GQA-grouped backward"): k and v (and dk, dv) are (batch, 2n, kv_heads,
 * headdim) bf16 while q, out, dout, dq are (batch, 2n, heads, headdim) and
 * lse (batch, heads, 2n).  Query head h reads key/value head
 * h / (heads / kv_heads) (integer division: consecutive query heads share a
 * key/value head).  kv_heads must divide heads (1 <= kv_heads <= heads),
 * otherwise DFA_EINVAL.  dk and dv of a key/value head are the sums of the
 * gradients through all of its query heads, accumulated on chip (a work
 * item of the backward walks the query tiles of every query head of its
 * group).  kv_heads == heads is dfa_forward / dfa_backward.  Scratch and
 * errors as for dfa_forward / dfa_backward.
 */
int dfa_forward_gqa(const void *q, const void *k, const void *v, void *out, float *lse,
                    int batch, int n, int heads, int kv_heads, int headdim, int block_size,
                    dfa_stream_t stream);
int dfa_backward_gqa(const void *q, const void *k, const void *v, const void *out,
                     const void *dout, const float *lse, void *dq, void *dk, void *dv,
                     int batch, int n, int heads, int kv_heads, int headdim, int block_size,
                     dfa_stream_t stream);

/*
 * Packed batches of samples of different lengths ("Fast Diffusion
 * Attention": varlen batches, the second API, modeled on FlashAttention's
 * varlen call).  cu_seqlens is a HOST array of batch + 1 int32 prefix sums
 * (cu_seqlens[0] == 0, non-decreasing): sample b is rows
 * [cu_seqlens[b], cu_seqlens[b+1]) of the packed tensors, [noisy | clean],
 * so its length 2 n_b must be even; zero-length samples are allowed.
 * rows = cu_seqlens[batch] <= 2^30.  Layouts: q, out, dout, dq are
 * (rows, heads, headdim) bf16, k, v, dk, dv (rows, kv_heads, headdim) bf16
 * (kv_heads divides heads, as for dfa_forward_gqa), lse (heads, rows)
 * float32.  block_size applies to every sample (clamped to each n_b).  The
 * non-empty samples run in one launch per pass, longest first.  Every
 * sample is read through tensor maps of its own, so rows past the end of a
 * half read as zeros: no value of one sample -- finite or not -- reaches
 * another sample's results.  The schedule (20 bytes and four 128-byte
 * tensor maps per sample) is copied to stream-ordered device memory on
 * `stream` (cudaMallocAsync, cudaMemcpyAsync from a host array,
 * cudaFreeAsync);
 * dfa_backward_varlen also takes the scratch of dfa_backward.  Errors:
 * DFA_EINVAL for a bad cu_seqlens (odd or negative length, cu_seqlens[0] !=
 * 0, NULL) or head counts, otherwise as dfa_forward / dfa_backward.
 */
int dfa_forward_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                       const int *cu_seqlens, int batch, int heads, int kv_heads, int headdim,
                       int block_size, dfa_stream_t stream);
int dfa_backward_varlen(const void *q, const void *k, const void *v, const void *out,
                        const void *dout, const float *lse, void *dq, void *dk, void *dv,
                        const int *cu_seqlens, int batch, int heads, int kv_heads,
                        int headdim, int block_size, dfa_stream_t stream);

/*
 * FP8 forward ("Fast Diffusion Attention" lists an FP8 forward): q, k, v
 * are e4m3 (one byte per element; q (batch, 2n, heads, 128), k, v (batch,
 * 2n, kv_heads, 128)) with per-tensor descales: the attention is that of
 * q8 * q_descale, k8 * k_descale, v8 * v_descale (descales finite, > 0).
 * S = Q K^T and O = P V run on the e4m3 tensor-core path with float32
 * accumulation; P is rounded to e4m3 (round to nearest even) for P V, while
 * the row sums and lse use the unrounded probabilities, so |out - exact|
 * <= 2^-4 * max|v| per element, plus the underflow of probabilities below
 * e4m3's smallest subnormal.  out bf16 (batch, 2n, heads, 128), lse as
 * dfa_forward.  headdim 128 only (DFA_EUNSUPPORTED otherwise).
 */
int dfa_forward_fp8(const void *q, const void *k, const void *v, void *out, float *lse,
                    float q_descale, float k_descale, float v_descale, int batch, int n,
                    int heads, int kv_heads, int headdim, int block_size, dfa_stream_t stream);

/*
 * The FP8 forward in two steps, for callers that produce V^T once (e.g.
 * while quantising V) and reuse it: dfa_fp8_transpose_v writes the V^T that
 * dfa_forward_fp8 builds internally -- e4m3 bytes laid out (batch,
 * kv_heads, 128, 2, n_pad), n_pad = n rounded up to 16, element
 * [b][h][c][half][j] = v[b][half * n + j][h][c]; keys j >= n unspecified --
 * into dfa_fp8_vt_bytes(batch, n, kv_heads, 128) bytes of device memory,
 * and dfa_forward_fp8_vt runs the forward on it (no scratch).  Results as
 * dfa_forward_fp8.
 */
long long dfa_fp8_vt_bytes(int batch, int n, int kv_heads, int headdim);
int dfa_fp8_transpose_v(const void *v, void *vt, int batch, int n, int kv_heads, int headdim,
                        dfa_stream_t stream);
int dfa_forward_fp8_vt(const void *q, const void *k, const void *vt, void *out, float *lse,
                       float q_descale, float k_descale, float v_descale, int batch, int n,
                       int heads, int kv_heads, int headdim, int block_size,
                       dfa_stream_t stream);

/*
 * The backward with options.  cu_seqlens == NULL: the batched layout of
 * dfa_backward_gqa (batch, n); otherwise the packed layout of
 * dfa_backward_varlen (n ignored).  flags: 0, DFA_DETERMINISTIC,
 * DFA_NOISY_DIAG_PASS, or both (then DFA_DETERMINISTIC alone applies).
 *
 * DFA_DETERMINISTIC (the deterministic mode of "Fast Diffusion Attention",
 * where semaphores fix the order of the dQ sums): the key tiles that reach
 * a query tile add their share of dQ one after another, in the order the
 * work counter hands them out, through one counter per (head-dim part,
 * head, query tile) in global memory; the results are then bitwise the
 * same from run to run.  dK and dV are summed inside one work item in a
 * fixed order in every mode (with grouped heads too), so only dQ needs the
 * counters.  Extra scratch: 2 * heads * rows uint32 counters (rows = batch
 * * 2n, or the packed rows), zeroed stream-ordered.  Every wait is bounded;
 * a wait that gives up sets DFA_ETIMEOUT in the status word.  Unknown flag
 * bits: DFA_EINVAL.
 */
#define DFA_DETERMINISTIC 1
/*
 * DFA_NOISY_DIAG_PASS (the dedicated noisy-diagonal pass of the backward,
 * "Fast Diffusion Attention", "Hopper: the FlashAttention-3 generation"):
 * the tensor-core backward runs as two launches on `stream`, first over the
 * noisy key tiles only -- the complete dK / dV of the noisy keys, and the
 * noisy queries' dQ from their own block STORED into the accumulator --
 * then over the clean key tiles, which add the rest of dQ.  It applies to
 * the batched layout when the block size divides the 128-key tile or a
 * half fits in one tile (min(block_size, n) divides 128, or n <= 128), so
 * that every noisy query row meets the noisy keys of one key tile only; in
 * every other case (varlen, DFA_DETERMINISTIC, other block sizes) the
 * single launch runs.  Results equal the single launch's up to the order
 * of float32 dQ additions; dK and dV are bitwise the same.
 */
#define DFA_NOISY_DIAG_PASS 2
int dfa_backward_ex(const void *q, const void *k, const void *v, const void *out,
                    const void *dout, const float *lse, void *dq, void *dk, void *dv,
                    const int *cu_seqlens, int batch, int n, int heads, int kv_heads,
                    int headdim, int block_size, int flags, dfa_stream_t stream);

/*
 * The yardstick of "Fast Diffusion Attention", section "The right yardstick":
 * causal attention on `batch` (>= 0, any number) independent sequences of
 * length `seqlen` (>= 1), same layout (batch, seqlen, heads, headdim), lse
 * (batch, heads, seqlen), run by the same kernels with causal tile
 * enumeration: each sequence takes the place of one half of a sample.
 * Viewing a (B, 2n, H, d) tensor as (2B, n, H, d) gives causal attention on
 * the 2B halves.  Scratch of dfa_causal_backward as for dfa_backward (delta
 * laid out (batch, heads, seqlen)).
 */
int dfa_causal_forward(const void *q, const void *k, const void *v, void *out, float *lse,
                       int batch, int seqlen, int heads, int headdim, dfa_stream_t stream);
int dfa_causal_backward(const void *q, const void *k, const void *v, const void *out,
                        const void *dout, const float *lse, void *dq, void *dk, void *dv,
                        int batch, int seqlen, int heads, int headdim, dfa_stream_t stream);

/*
 * The forward and the three steps dfa_backward runs, for callers that own
 * the scratch or time the steps one by one.  `mode` is DFA_MODE_DIFFUSION or
 * DFA_MODE_CAUSAL.  Diffusion: tensors (batch, 2n, heads, headdim), lse and
 * delta (batch, heads, 2n).  Causal: `batch` sequences of length n, tensors
 * (batch, n, heads, headdim), lse and delta (batch, heads, n), block_size
 * ignored -- dfa_causal_forward / dfa_causal_backward in steps.
 *   dfa_fwd_main: dfa_forward (or, in the causal mode, dfa_causal_forward);
 *     if dq_acc is not NULL the same launch also sets dq_acc (float32, shape
 *     of q) to zero, with stores issued alongside the tensor-core work by
 *     warps that are not on its critical path, so that the backward needs no
 *     separate pass over it.
 *   dfa_bwd_preprocess: delta = rowsum(dout * out), float32 (batch, heads, 2n);
 *     dq_acc (float32, shape of q) set to zero unless dq_acc is NULL (then
 *     the caller zeroed it, e.g. through dfa_fwd_main).
 *     dfa_bwd_preprocess_ex: the same with `mode` (causal: rows of n).
 *   dfa_bwd_main: the tensor-core backward: writes dk, dv (bf16) and adds
 *     dq (already scaled) into dq_acc (float32 atomics or bulk reduce-adds).
 *   dfa_bwd_dq_convert: dq = bf16(dq_acc), round to nearest even.
 *     dfa_bwd_dq_convert_ex: the same with `mode` (causal: rows of n).
 *   dfa_bwd_main_ex: dfa_bwd_main_gqa with flags, 0 or DFA_NOISY_DIAG_PASS
 *     (see dfa_backward_ex; causal mode: the flag is ignored).  Where the
 *     noisy-diagonal pass applies, the noisy rows of dq_acc are overwritten
 *     rather than added to: their prior contents do not matter.
 * dq_acc and delta are device buffers the caller allocated (16-byte aligned).
 */
int dfa_fwd_main(const void *q, const void *k, const void *v, void *out, float *lse,
                 float *dq_acc, int batch, int n, int heads, int headdim, int block_size,
                 int mode, dfa_stream_t stream);
int dfa_bwd_preprocess(const void *out, const void *dout, float *delta, float *dq_acc,
                       int batch, int n, int heads, int headdim, dfa_stream_t stream);
int dfa_bwd_main(const void *q, const void *k, const void *v, const void *dout,
                 const float *lse, const float *delta, float *dq_acc, void *dk, void *dv,
                 int batch, int n, int heads, int headdim, int block_size, int mode,
                 dfa_stream_t stream);
int dfa_bwd_dq_convert(const float *dq_acc, void *dq, int batch, int n, int heads,
                       int headdim, dfa_stream_t stream);
int dfa_bwd_preprocess_ex(const void *out, const void *dout, float *delta, float *dq_acc,
                          int batch, int n, int heads, int headdim, int mode,
                          dfa_stream_t stream);
int dfa_bwd_dq_convert_ex(const float *dq_acc, void *dq, int batch, int n, int heads,
                          int headdim, int mode, dfa_stream_t stream);
/*
 * dfa_fwd_main and dfa_bwd_main with grouped key/value heads: k, v, dk, dv
 * have kv_heads heads (a divisor of heads), as for dfa_forward_gqa; q, out,
 * dout, lse, delta and dq_acc keep `heads`.  kv_heads == heads is
 * dfa_fwd_main / dfa_bwd_main.
 */
int dfa_fwd_main_gqa(const void *q, const void *k, const void *v, void *out, float *lse,
                     float *dq_acc, int batch, int n, int heads, int kv_heads, int headdim,
                     int block_size, int mode, dfa_stream_t stream);
int dfa_bwd_main_gqa(const void *q, const void *k, const void *v, const void *dout,
                     const float *lse, const float *delta, float *dq_acc, void *dk, void *dv,
                     int batch, int n, int heads, int kv_heads, int headdim, int block_size,
                     int mode, dfa_stream_t stream);
int dfa_bwd_main_ex(const void *q, const void *k, const void *v, const void *dout,
                    const float *lse, const float *delta, float *dq_acc, void *dk, void *dv,
                    int batch, int n, int heads, int kv_heads, int headdim, int block_size,
                    int mode, int flags, dfa_stream_t stream);

/*
 * dfa_backward without any allocation.  No passage of the pages has a
 * counterpart: this entry point exists for callers that cannot let a library
 * allocate device memory -- a framework whose own caching allocator must
 * account for every byte, or a latency-critical step where an allocation
 * could block or fail part-way.  Same arguments, results and errors as
 * dfa_backward, but the float32 scratch (dq accumulator and D) lives in one
 * fixed 32 MiB array inside the library that every GPU loading the library
 * holds until the process exits.  The problem must fit it:
 *   batch * heads * 2n * (headdim + 1) * 4 bytes <= 32 MiB,
 * otherwise DFA_EINVAL is returned before any work is enqueued.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All
 * calls share the one array and it keeps the last call's contents (the dq
 * accumulator is zeroed at the start of every call): calls whose work
 * overlaps on the GPU -- on different streams, or from different threads --
 * race on it and must be serialised by the caller.
 */
int dfa_backward_noalloc(const void *q, const void *k, const void *v, const void *out,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv,
                         int batch, int n, int heads, int headdim, int block_size,
                         dfa_stream_t stream);

/*
 * Synchronise `stream`, then return and clear the device status word of the
 * current device: DFA_OK, DFA_ETIMEOUT or DFA_EDEVICE (or DFA_ECUDA if the
 * synchronisation itself failed).
 */
int dfa_status(dfa_stream_t stream);

/*
 * Failure-detection self-test.  Launches one warp that waits, through the
 * same bounded wait the attention kernels use, on an mbarrier that nothing
 * ever arrives on.  After limit_us microseconds (1 .. 1,000,000) the wait
 * gives up, DFA_ETIMEOUT is recorded in the device status word and the
 * kernel returns; the next dfa_status() reports it and the context stays
 * usable.  No passage of the pages has a counterpart: it checks the guard
 * that turns a kernel-side hang into an error code.
 */
int dfa_selftest_wait_timeout(int limit_us, dfa_stream_t stream);

/*
 * Tile geometry, host side, for tests and schedulers.  mode is one of
 * DFA_MODE_*; halves are 0 (noisy) and 1 (clean); tiles are block_m query
 * rows by block_n keys, counted inside a half.
 *
 * dfa_fwd_segments: key tiles visited by query tile q_tile of half q_half.
 * Writes up to 2 segments as 4 ints each (key_half, rule, first_tile,
 * end_tile) into seg[8] and returns their number (or a negative code).
 *
 * dfa_bwd_segments: query tiles that see key tile k_tile of half k_half,
 * same encoding with the query half in place of the key half.
 *
 * dfa_tile_full: 1 if every (query, key) pair of the tile is visible under
 * `rule` (so the kernels skip per-element masking), else 0.
 *
 * dfa_tile_visits: total tile visits per (batch, head) of the forward
 * (pass 0) or backward (pass 1) enumeration.
 */
int dfa_fwd_segments(int mode, int n, int block_size, int block_m, int block_n,
                     int q_half, int q_tile, int *seg);
int dfa_bwd_segments(int mode, int n, int block_size, int block_m, int block_n,
                     int k_half, int k_tile, int *seg);
int dfa_tile_full(int rule, int n, int block_size, int q_start, int block_m,
                  int k_start, int block_n);
long long dfa_tile_visits(int mode, int n, int block_size, int block_m, int block_n, int pass);

/*
 * Work order of the kernels, host side, for tests and schedulers: the w-th
 * work item (0 <= w < 2 * batch * heads * tiles; causal mode: batch counts
 * sequences, w < batch * heads * tiles) of the forward (pass 0, one item per
 * query tile) or backward (pass 1, one item per key tile) enumeration, for
 * `tiles` tiles per half and scheduling groups of `group` (batch, head)
 * pairs ((sequence, head) pairs in the causal mode).  Writes (batch, head,
 * half, tile) into item[4]; in the causal mode sequence s is reported as
 * (s / 2, head, s % 2, tile).
 * Passes 2 and 3 (diffusion mode only, w < batch * heads * tiles) are the
 * two launches of DFA_NOISY_DIAG_PASS: 2 the clean key tiles, 3 the noisy
 * key tiles.
 * Inside a group the items of a (batch, head) go longest first; the
 * shortest ones of all pairs come last ("Fast Diffusion Attention",
 * "Hopper" and "Ampere and Ada": longest-first, L2-aware order).  The
 * persistent kernels hand the items out in this order from a work counter.
 */
int dfa_work_item(int pass, int mode, int w, int batch, int heads, int tiles, int group,
                  int *item);

/*
 * Tile shapes the kernels use for a head dimension: forward query rows and
 * keys per tile, backward keys and query rows per tile.  Returns DFA_OK or
 * DFA_EUNSUPPORTED.
 */
int dfa_tile_shape(int headdim, int *fwd_block_m, int *fwd_block_n,
                   int *bwd_block_n, int *bwd_block_m);

#ifdef __cplusplus
}
#endif
#endif /* DFA_H_ */
