/*
 * libqkvfront: the decode-batch attention front on one GB300 (sm_103a).
 *
 * Defined by the API pages of vllm.models.muse_spark.nvidia.specialized_decode:
 *   "cutedsl.attention.qkv_front" (module docstring; functions qkv_front,
 *   launch, unsupported, prepare, variant, hidden_rows_ok,
 *   kv_cache_layout_ok, supports_shape) and "runtime.cute_ops" (split_qkv,
 *   supports_call, unsupported_projection, attn2 paragraph for the cache).
 *
 * For 1 <= M <= 16 tokens one launch computes
 *     out[M, N] = bf16( x[M, 8192] @ W[N, 8192]^T )       (FP32 accumulation)
 * over packed rows [q | k | v | gate] (8 q heads, 1 k head, 1 v head and 8
 * gate heads of 64 columns per KV head, so N = 1152 * num_kv_heads), then for
 * each 64-wide q and k head the weightless RMS norm (eps 1e-6) and the
 * interleaved RoPE (pairs 2i, 2i+1; cos in table column i, sin in 32 + i) of
 * the token's position, stores the row in `out`, and writes each token's
 * k head g into the K half (elements 0..63) and v head g into the V half
 * (64..127) of cache slot `slots[t]` (page slot / 16, offset slot % 16) of KV
 * head g.  v and gate columns of `out` hold the rounded projection.
 *
 * Conventions of every entry point below:
 *   - bf16 arrays are passed as uint16_t bit patterns; all arrays are
 *     row-major and contiguous; all pointers are DEVICE pointers owned by the
 *     caller and must be 16-byte aligned;
 *   - the library allocates no device memory per call and keeps no state
 *     across calls except a device status word (qkv_front_status);
 *   - per device it caches, on first use, the kernels' attributes and the
 *     device address of its no-allocation array (attn2_split_kv_noalloc);
 *     after cudaDeviceReset on a device, do not call the library on that
 *     device again in the same process;
 *   - `stream` is a cudaStream_t (NULL: the legacy default stream); calls are
 *     asynchronous on it.  The kernel is launched with programmatic stream
 *     serialization (PDL): it may start while the previous kernel on the
 *     stream runs, reads only W before it waits for that kernel, and reads
 *     x / positions / slots / cos_sin and writes out / kv_cache after;
 *     so W must not be written by a kernel that may still be running when
 *     the call is launched (weights are written at load time only);
 *   - return value 0 (QKVF_OK) or a QKVF_ERR_* code; nothing is launched
 *     when a code is returned.  qkv_front_strerror gives its text.
 */
#ifndef QKVFRONT_H
#define QKVFRONT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes -------------------------------------------------------- */
#define QKVF_OK 0
#define QKVF_ERR_TOKENS 1        /* M outside 0..16 */
#define QKVF_ERR_SHAPE 2         /* num_kv_heads < 1 or N != 1152 * num_kv_heads */
#define QKVF_ERR_NULL 3          /* a required pointer is NULL */
#define QKVF_ERR_ALIGN 4         /* a pointer is not 16-byte aligned */
#define QKVF_ERR_DEVICE 5        /* the current device is not compute capability 10.3 */
#define QKVF_ERR_CUDA 6          /* a CUDA runtime/driver call failed */
#define QKVF_ERR_SIZES 7         /* cos_sin_rows < 1, num_pages < 1, or too large */
#define QKVF_ERR_VARIANT 8       /* an explicit variant that this shape cannot use */
#define QKVF_ERR_ARG 9           /* any other bad argument */

/* ---- device status bits (qkv_front_status) ------------------------------- */
#define QKVF_STATUS_BAD_SLOT 1u      /* a slot >= num_pages * 16: that token's insert skipped */
#define QKVF_STATUS_BAD_POSITION 2u  /* a position outside [0, cos_sin_rows): its q/k heads and insert skipped */
#define QKVF_STATUS_WAIT_TIMEOUT 4u  /* a bounded wait in the kernel gave up: outputs of that call are invalid */
#define QKVF_STATUS_BAD_REQUEST 8u   /* attn2: a request with L < 8, L beyond its table, or a page outside the cache: its rows skipped */

/*
 * qkv_front: check the call, then launch the fused front.
 *   x          [M, 8192] bf16 bits.  The attention input.
 *   W          [N, 8192] bf16 bits.  Unquantized, bias-free QKV + o-gate weight.
 *   positions  [M] int64.  Token positions; each must be in [0, cos_sin_rows).
 *   slots      [M] int64.  Cache slot of each token (page * 16 + offset);
 *              a negative slot means "no insert" (padding token); a slot
 *              >= num_pages * 16 is skipped and flagged QKVF_STATUS_BAD_SLOT.
 *   cos_sin    [cos_sin_rows, 64] fp32.  Row p: cos(p f_i) in column i,
 *              sin(p f_i) in column 32 + i (interleaved, not neox style).
 *   out        [M, N] bf16 bits, written.
 *   kv_cache   [num_pages, num_kv_heads, 16, 128] bf16 bits; only the named
 *              slots change.
 *   M          0..16 tokens (M == 0 launches nothing and returns QKVF_OK).
 *   N          1152 * num_kv_heads.
 * Tokens must name distinct slots (two tokens writing one slot race).
 * x, W and cos_sin must not overlap out or kv_cache.
 */
int qkv_front(const uint16_t *x, const uint16_t *W, const int64_t *positions,
              const int64_t *slots, const float *cos_sin, int64_t cos_sin_rows,
              uint16_t *out, uint16_t *kv_cache, int64_t num_pages, int M, int N,
              int num_kv_heads, void *stream);

/*
 * qkv_front_unsupported: why qkv_front would refuse this call, or NULL when
 * it takes it (page qkv_front, function unsupported).  Host-only checks, no
 * CUDA call except the device query.  Returns a static string.
 */
const char *qkv_front_unsupported(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                                  const int64_t *slots, const float *cos_sin,
                                  int64_t cos_sin_rows, uint16_t *out, uint16_t *kv_cache,
                                  int64_t num_pages, int M, int N, int num_kv_heads);

/*
 * qkv_front_launch: qkv_front without its argument checks, for a call that
 * qkv_front_unsupported already accepted (page qkv_front, function launch).
 * Out-of-contract arguments here are undefined behaviour.
 */
int qkv_front_launch(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                     const int64_t *slots, const float *cos_sin, int64_t cos_sin_rows,
                     uint16_t *out, uint16_t *kv_cache, int64_t num_pages, int M, int N,
                     int num_kv_heads, void *stream);

/* ---- contraction engines (qkv_front_variant, qkv_front_launch_variant) --- */
#define QKVF_CONSUMER_DEFAULT 0   /* the library's choice */
#define QKVF_CONSUMER_MMA_SYNC 1  /* mma.sync m16n8k16 in four consumer warps */
#define QKVF_CONSUMER_TCGEN05 2   /* tcgen05.mma M=64 into tensor memory, one issuing thread */
#define QKVF_CONSUMER_RESIDENT 3  /* mma.sync with the CTA's whole W share on chip (shared memory and
                                     registers) before the PDL wait, partials pushed to the owner
                                     rank with st.async: splits 8, kb 4, stages 4 only */

/*
 * qkv_front_variant: the launch shape qkv_front uses for N columns and M
 * tokens on the current device (page qkv_front, function variant):
 *   *tiles    8-token column tiles (1 or 2),
 *   *stages   depth of the shared-memory weight ring,
 *   *splits   CTAs per head (the cluster size; K is split cyclically among them),
 *   *kb       64-wide K boxes per ring stage (1, 2 or 4),
 *   *consumer QKVF_CONSUMER_MMA_SYNC, QKVF_CONSUMER_TCGEN05 or
 *             QKVF_CONSUMER_RESIDENT (chosen when splits is 8: N = 1152).
 * Any output pointer may be NULL.  The result depends on the launch shape:
 * `splits` and `kb` fix how K is divided among CTAs, and the consumer fixes
 * the order inside one CTA; `stages` never changes it.
 */
int qkv_front_variant(int N, int M, int *tiles, int *stages, int *splits, int *kb, int *consumer);

/*
 * qkv_front_launch_variant: qkv_front (with its checks) at an explicit
 * variant, for tests and tuning.  splits in {1, 2, 4, 8, 16}; kb in {1, 2, 4}
 * (0: the default) with splits * kb <= 128; stages >= 2 within the
 * shared-memory limit; consumer one of QKVF_CONSUMER_* (the resident engine
 * takes splits 8, kb 4 or 0, stages 4).  Otherwise QKVF_ERR_VARIANT.
 */
int qkv_front_launch_variant(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                             const int64_t *slots, const float *cos_sin,
                             int64_t cos_sin_rows, uint16_t *out, uint16_t *kv_cache,
                             int64_t num_pages, int M, int N, int num_kv_heads, int splits,
                             int stages, int kb, int consumer, void *stream);

/*
 * qkv_front_prepare: set the kernel attributes (dynamic shared memory,
 * non-portable cluster size) of the variants that N columns take, so that
 * later calls can be captured in a CUDA graph (page qkv_front, function
 * prepare).  Calls made without it prepare themselves on first use.
 */
int qkv_front_prepare(int N, int num_kv_heads);

/*
 * qkv_front_status: copy the device status word (an OR of QKVF_STATUS_* bits
 * raised by calls since the last read) into *bits and clear it.
 * Synchronizes the current device.
 */
int qkv_front_status(unsigned int *bits);

/*
 * qkv_front_from_host: the whole call for a caller whose tokens live in host
 * memory.  On `stream`, asynchronously: x [M, 8192], positions [M] and slots
 * [M] go from host memory into the caller's device `staging` buffer, qkv_front
 * runs on them, and out [M, N] goes back to `out_host`.  Pinned (page-locked,
 * device-mapped) host buffers are read by a staging kernel over the host link,
 * PDL-linked to the front so that its weight stream starts while x arrives,
 * and a pinned out_host is written by the front directly; pageable buffers go
 * through copies on the stream instead.  Host buffers must stay valid and
 * unchanged until the stream passes the call.  W, cos_sin and kv_cache are
 * device pointers as for qkv_front.
 *   staging        device buffer, 256-byte aligned, at least
 *                  qkv_front_staging_bytes(M, N) bytes; owned by the caller;
 *                  the call overwrites it (two calls in flight on different
 *                  streams need two buffers).
 * Same checks and codes as qkv_front, plus QKVF_ERR_SIZES when staging is too
 * small and QKVF_ERR_ALIGN when it is not 256-byte aligned.  The library
 * allocates nothing.
 */
int qkv_front_from_host(const uint16_t *x_host, const int64_t *positions_host,
                        const int64_t *slots_host, uint16_t *out_host, const uint16_t *W,
                        const float *cos_sin, int64_t cos_sin_rows, uint16_t *kv_cache,
                        int64_t num_pages, void *staging, uint64_t staging_bytes, int M, int N,
                        int num_kv_heads, void *stream);

/* Device staging bytes qkv_front_from_host needs for M tokens and N columns. */
uint64_t qkv_front_staging_bytes(int M, int N);

/*
 * qknorm_rope_kv_insert: the unfused epilogue on its own, for any number of
 * tokens (fused_muse_spark_qknorm_rope_kv_insert, the kernel the fused front
 * replaces: page qkv_front, module docstring; page cute_ops, qkv_front
 * paragraph).  In place on a BF16 projection output:
 *   qkv        [T, N] bf16 bits, rows [q | k | v | gate]; every q and k head
 *              is normed and rotated (same arithmetic as qkv_front), v and
 *              gate heads are not touched.
 *   positions, slots, cos_sin, cos_sin_rows, kv_cache, num_pages, N,
 *   num_kv_heads: as for qkv_front, with T entries in positions and slots.
 *   T          0 .. 2^24 tokens (0: no launch).
 * Each token's k head g goes to the K half and v head g to the V half of its
 * slot.  Out-of-range positions and slots follow qkv_front's rules and raise
 * the same status bits.  Launched with PDL like qkv_front (it waits for the
 * previous kernel before reading anything).  Allocates nothing.
 */
int qknorm_rope_kv_insert(uint16_t *qkv, const int64_t *positions, const int64_t *slots,
                          const float *cos_sin, int64_t cos_sin_rows, uint16_t *kv_cache,
                          int64_t num_pages, int T, int N, int num_kv_heads, void *stream);

/* Why qknorm_rope_kv_insert would refuse this call, or NULL (host checks only). */
const char *qknorm_rope_kv_insert_unsupported(uint16_t *qkv, const int64_t *positions,
                                              const int64_t *slots, const float *cos_sin,
                                              int64_t cos_sin_rows, uint16_t *kv_cache,
                                              int64_t num_pages, int T, int N, int num_kv_heads);

/*
 * layer_front: the kernel before the QKV front in the first decoder layer
 * (page layer_front, class LayerFront, run): for each of `rows` rows of
 * 8192 values,
 *   stream = x as FP32 (the residual stream), aux = stream (if aux is not
 *   NULL), out = bf16((stream * r) * w), r = 1 / sqrt(mean(stream^2) + eps),
 *   w the BF16 weight widened to FP32 (out = bf16(stream * r) when weight is
 *   NULL) — the attention input the QKV front reads as x.
 *   x          [rows, 8192], bf16 bits (x_is_f32 = 0) or fp32 (x_is_f32 = 1).
 *   weight     [8192] bf16 bits, or NULL.
 *   stream, aux [rows, 8192] fp32 (aux may be NULL); out [rows, 8192] bf16 bits.
 *   rows       0 .. 2^20 (0: no launch); eps in (0, 1].
 * All arrays are device pointers, 16-byte aligned; outputs must not overlap
 * each other or the inputs.  Launched with PDL: it waits for the previous
 * kernel, then at once lets the next kernel on the stream start, so a
 * qkv_front call issued after it streams its weights while this runs.
 */
int layer_front(const void *x, int x_is_f32, const uint16_t *weight, float *stream, float *aux,
                uint16_t *out, int rows, float eps, void *cuda_stream);

/*
 * attn2: paged decode attention of the 8-token verify step fused with the
 * output's weightless RMS norm and sigmoid gate — the o_proj input (page
 * cute_ops, attn2 paragraph).  For each request r (query rows 8r .. 8r+7 of
 * qkv, row i the token at position L_r - 8 + i):
 *   out[8r+i, head h] = bf16( o / sqrt(mean(o^2) + eps) * sigmoid(gate) ),
 *   o = softmax(scale * q K^T) V over keys j <= L_r - 8 + i (and, with a
 *   window W > 0, j > L_r - 8 + i - W); q = q head h of the row, gate = gate
 *   head h of the row, K and V from KV head h / 8 of the cache.
 *   qkv          [8 R, N] bf16 bits, rows [q | k | v | gate] (the front's out).
 *   kv_cache     [num_pages, num_kv_heads, 16, 128] bf16 bits (K | V per slot).
 *   block_table  [R, max_blocks] int32: key j of request r is slot j % 16 of
 *                page block_table[r][j / 16].
 *   context_lens [R] int32, each >= 8.
 *   out          [8 R, 512 num_kv_heads] bf16 bits.
 *   window       0 (none) or W >= 1; scale > 0 (1/8 for head_dim 64);
 *   eps in (0, 1].  num_reqs 0 .. 65535.
 * A request whose length is < 8 or needs more than max_blocks pages, or
 * whose table names a page outside the cache, is skipped (its rows left as
 * they were) and raises QKVF_STATUS_BAD_REQUEST.  Long contexts are split
 * over up to 8 CTAs of a cluster (attn2_launch_splits reaches 16), chosen
 * from num_reqs, num_kv_heads, max_blocks and window (not from the lengths,
 * which stay on the device): doubled while num_reqs * num_kv_heads * splits
 * stays within the SM count and each split keeps two or more of the pages a
 * row can see; the split partials are merged through distributed shared
 * memory in a fixed order.
 * Allocates nothing; launched with PDL like qkv_front.
 */
int attn2(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
          const int32_t *block_table, int max_blocks, const int32_t *context_lens, int num_reqs,
          int N, int num_kv_heads, int window, float scale, float eps, uint16_t *out,
          void *stream);

/*
 * attn2_unsupported: why attn2 (and attn2_split_kv / _noalloc, given a valid
 * workspace and split) would refuse this call, or NULL when it takes it
 * (page cute_ops, unsupported_attn2).  Host-only checks, no CUDA call except
 * the device query; returns a static string.  Of the page's refusals, the
 * layout ones are fixed by this ABI: head_dim 64 and 8 q heads per KV head
 * are implied by N = 1152 * num_kv_heads, and a layer without the o-norm and
 * sigmoid gate has nothing to call here (the Python binding's
 * unsupported_attn2 refuses such a layer).  The page's kernel is built for
 * one softmax scale and one o-norm eps, whose values the page does not
 * print; this kernel takes both per call and refuses only scale <= 0 and eps
 * outside (0, 1].
 */
const char *attn2_unsupported(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                              const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                              int num_reqs, int N, int num_kv_heads, int window, float scale, float eps,
                              uint16_t *out);

/* attn2 at an explicit split (1, 2, 4, 8 or 16 CTAs per request and KV head;
 * otherwise QKVF_ERR_VARIANT), for tests and tuning. */
int attn2_launch_splits(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                        const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                        int num_reqs, int N, int num_kv_heads, int window, float scale, float eps,
                        uint16_t *out, int splits, void *stream);

/* The split attn2 uses for this shape (window 0: none) on the current device
 * (0 on bad input). */
int attn2_splits(int num_reqs, int num_kv_heads, int max_blocks, int window);

/*
 * attn2, split-KV engine: the same result as attn2 (same arguments, readings
 * and bad-request rule) with the pages a row sees split over `splits` CTAs
 * per (request, KV head) without clusters, so that few requests can still
 * cover every SM.  Two grids on the stream (the second PDL-linked when the
 * first leaves SMs idle): the first writes each CTA's partial (row maxima,
 * sums and unnormalised O, FP32) to its slot of the caller's workspace; the
 * second merges a row's slots in split order (a fixed `splits` gives the
 * same bits every time) and finishes the rows.
 *   splits          1 .. 256, or 0 for attn2_split_kv_splits' choice;
 *                   otherwise QKVF_ERR_VARIANT.
 *   workspace       device memory, 256-byte aligned, at least
 *                   attn2_split_kv_workspace_bytes(num_reqs, num_kv_heads,
 *                   splits) bytes, owned by the caller, overlapping no other
 *                   argument, no initial contents needed; one workspace serves
 *                   one stream at a time.
 * With splits == 1 the call runs one grid (each CTA finishes its own rows)
 * and leaves the workspace untouched.
 * Returns QKVF_ERR_NULL / _ALIGN / _SIZES / _ARG for a missing, misaligned,
 * short or overlapping workspace, else as attn2.
 */
int attn2_split_kv(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                   const int32_t *block_table, int max_blocks, const int32_t *context_lens, int num_reqs,
                   int N, int num_kv_heads, int window, float scale, float eps, uint16_t *out, int splits,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes attn2_split_kv needs (0 on bad input): num_reqs *
 * num_kv_heads * splits slots of 17152 bytes. */
size_t attn2_split_kv_workspace_bytes(int num_reqs, int num_kv_heads, int splits);

/* The split attn2_split_kv picks for splits == 0 on the current device: the
 * grid covers the SMs once (num_reqs * num_kv_heads * splits <= SM count) and
 * each split keeps two or more of the pages a row can see; 0 on bad input. */
int attn2_split_kv_splits(int num_reqs, int num_kv_heads, int max_blocks, int window);

/*
 * attn2_split_kv for callers that cannot allocate device memory: a plugin
 * whose host process owns every device allocation through its own pool, or
 * a decode step that must not risk cudaMalloc's implicit synchronisation or
 * a failed allocation mid-step.  The pages have no counterpart of this entry
 * point.  Same arguments and result as attn2_split_kv without the workspace:
 * the partials go to a file-scope device array of the library, 256 slots of
 * 17152 bytes (4,390,912 bytes), which every GPU that loads the library holds
 * until the process exits.  The call allocates nothing.
 *   When splits (after splits == 0 is resolved as attn2_split_kv_splits
 *   does) is above 1, num_reqs * num_kv_heads * splits must be <= 256, else
 *   QKVF_ERR_SIZES.  At one split the call runs the direct path (each CTA
 *   finishes its own rows), touches no array slot and takes any num_reqs.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The array needs no clearing: a call reads only slots it wrote.
 * Every call shares it, so calls that overlap on the GPU (other streams,
 * other host threads) race; run them one after another.
 */
int attn2_split_kv_noalloc(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                           const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                           int num_reqs, int N, int num_kv_heads, int window, float scale, float eps,
                           uint16_t *out, int splits, void *stream);


/* Static text of a QKVF_* return code. */
const char *qkv_front_strerror(int code);

/*
 * qkv_front_selftest_wait: launch a one-CTA kernel that waits, through the
 * same bounded shared-memory barrier wait the front uses, on a barrier that
 * nothing completes, for at most timeout_ns nanoseconds (1..10^9); it then
 * raises QKVF_STATUS_WAIT_TIMEOUT and returns.  Tests that the kernel's waits
 * end without hanging the GPU.
 */
int qkv_front_selftest_wait(int64_t timeout_ns, void *stream);

/*
 * qkv_front_set_pdl: launch this library's kernels with programmatic stream
 * serialization (enable = 1, the default) or as plain stream-ordered launches
 * (0).  With PDL a kernel may start while the previous kernel on its stream
 * still runs and streams its weights before waiting for it; turn it off when
 * a kernel that may still be running writes W (or, for measurement, to see
 * what the overlap gains).  Other values: QKVF_ERR_ARG.  Applies to launches
 * made after the call, on every device.
 */
int qkv_front_set_pdl(int enable);

/* Bounded-wait limit of the front's barrier waits in nanoseconds
 * (default 2e9); values outside 1e3..1e10 are refused with QKVF_ERR_ARG. */
int qkv_front_set_wait_limit(int64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* QKVFRONT_H */
