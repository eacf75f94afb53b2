/*
 * nsp.h -- C ABI of the GB300 (sm_103a) varlen attention hot path.
 *
 * One GPU, caller-owned device memory, caller stream.  The library computes:
 *
 *   - document-masked ("varlen") causal self-attention over a packed token
 *     stream, forward and backward, with grouped-query heads;
 *   - the chunk-partial attention of ring-style sequence parallelism (a query
 *     range against a key range) and the log-sum-exp merge of such partials;
 *   - the Ulysses seq-sharded -> head-sharded layout permutation.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts (row-major, innermost last):
 *   q, out, dout, dq : [tokens, Hq,  d]      k, v, dk, dv : [tokens, Hkv, d]
 *   lse              : [Hq, tokens] float32 (natural log of the scaled scores)
 *   cu_seqlens       : int32 [ndoc + 1], device memory, cu[0] = 0,
 *                      non-decreasing, cu[ndoc] = total tokens of the stream.
 *                      Zero-length documents are allowed.
 * Element types: NSP_BF16 inputs are computed with float32 accumulation;
 *   NSP_F32 inputs with true float32 arithmetic (no TF32).
 * Ownership: the caller allocates and frees every buffer, including the
 *   workspace.  The library allocates no device or host memory, never
 *   synchronises the stream (except nsp_status_query) and enqueues all work
 *   on `stream`.  Calls on different streams with different workspaces may
 *   run concurrently.
 * Alignment: every device pointer must be 16-byte aligned; the bf16 outputs
 * of attention (out of a forward, dq / dk / dv of a backward) must be
 * 32-byte aligned (they are written as 32-byte vectors).
 * Errors: scalar, alignment and size errors are detected on the host and
 *   returned before anything is enqueued.  Errors in device data (a bad
 *   cu_seqlens) are detected by the first kernel, recorded in the status word
 *   at the start of the workspace, and make every later kernel of the call a
 *   no-op; nsp_status_query() returns that word.  A CUDA launch failure
 *   returns NSP_ERR_CUDA.  Every device-side wait is bounded: if a bound
 *   expires the kernel records NSP_ERR_TIMEOUT and returns (it never traps).
 *
 * Pages the operations come from (cited by title and section):
 *   [NSP]  "NSP: Accelerating Variable-Length LLM Training via Nested Sequence
 *          Parallelism" -- Sec. 2.2 Sequence Packing, Sec. 2.3 recomputation.
 *   [BASP] "BASP: Communication-Efficient Batch-Aware Sequence Parallelism for
 *          LLM Training" -- Sec. II-A Scaled Dot-Product Attention, Sec. II-C
 *          DeepSpeed Ulysses.
 *   [HSAP] "HSAP: A Hierachical Sequence-aware Parallelism for Hybrid-Context
 *          Generative Models" -- Sec. 2.1 Sequence Packing (cu_len),
 *          Sec. 2.2.1 InterSP (ring, online accumulation), Sec. 2.2.2 IntraSP
 *          (all-to-all), Sec. 3.2 attention-block patterns, Limitations
 *          (fusing copy and rescale).
 */
#ifndef NSP_H_
#define NSP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* nsp_stream_t;

typedef enum {
  NSP_OK = 0,
  NSP_ERR_INVALID = 1,      /* bad scalar argument or bad cu_seqlens contents */
  NSP_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d not 64/128)  */
  NSP_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required     */
  NSP_ERR_CUDA = 4,         /* a CUDA call or launch failed                   */
  NSP_ERR_TIMEOUT = 5,      /* a bounded device-side wait expired             */
  NSP_ERR_ALIGN = 6         /* a pointer is not 16 (bf16 outputs: 32)-byte aligned */
} nsp_status;

typedef enum { NSP_F32 = 0, NSP_BF16 = 1 } nsp_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* nsp_status_str(int32_t status);

/* Library version string, e.g. "nsp 0.1 sm_103a". */
const char* nsp_version(void);

/* Number of kernels this library has launched in this process so far (all
 * devices, all streams; a relaxed atomic counter).  Lets callers and
 * benchmarks count the library's own launches. */
int64_t nsp_kernel_launches(void);

/* Number of attention kernels (forward, dK/dV and dQ kernels) this library
 * has launched in this process on the tensor-core path (tensor_core = 1:
 * tcgen05, TMEM, TMA) or on the CUDA-core path (tensor_core = 0: float32
 * I/O, or no tensor-map support in the driver).
 * Lets a caller see which path its calls took. */
int64_t nsp_path_launches(int32_t tensor_core);

/* Bound, in GPU clock cycles, of every wait inside the tensor-core attention
 * kernels (a thread waiting for a copy, a product or another role of its
 * block).  When a wait runs longer, the kernel records NSP_ERR_TIMEOUT in the
 * workspace status word (read it with nsp_status_query), every role of the
 * block stops, waits for the copies and products it already issued, frees its
 * tensor memory and returns: the context stays usable and the next call on
 * the same workspace starts afresh.  The outputs of the failed call are
 * unspecified.
 *
 * It makes the kernels' failure detection testable: the default (cycles < 0
 * restores it) is 4e9 cycles, about 2 s,
 * far beyond any legitimate wait; a tiny bound (0 to a few hundred cycles)
 * makes a call's first wait that is not already satisfied expire.
 * Process-wide; applies to calls issued after it returns (not to calls
 * already enqueued).  Returns the previous bound.  No counterpart on the
 * pages, which describe no device-side failure handling. */
int64_t nsp_set_wait_timeout_cycles(int64_t cycles);

/* ------------------------------------------------------------------------
 * Varlen attention forward  ([BASP] Sec. II-A; [HSAP] Sec. 2.1, 2.2.1).
 *
 * For every query row t in [q_start, q_start + q_len) of the packed stream,
 * every query head h and g = h / (Hq / Hkv):
 *   J(t)  = keys of t's document, restricted to positions <= t if causal,
 *           intersected with [kv_start, kv_start + kv_len);
 *   x_j   = scale * <q[t,h], k[j,g]>,   lse[h,t] = ln sum_{j in J(t)} exp(x_j),
 *   out[t,h] = sum_{j in J(t)} exp(x_j - lse[h,t]) v[j,g].
 * A row with empty J(t) gets out = 0 and lse = -inf.
 *
 * Whole-stream attention: q_start = kv_start = 0, q_len = kv_len = T.
 * Ring chunk partial ([HSAP] Sec. 2.2.1 / 3.2): `q` points at the first row
 * of the query shard ([q_len, Hq, d]) and `k`, `v` at the first row of the
 * key shard ([kv_len, Hkv, d]); q_start / kv_start are the shards' global
 * token offsets, used only to compare positions with cu_seqlens.  Request
 * out_dtype = NSP_F32 for partials that will be merged.
 *
 * Arguments: q, k, v device, io_dtype; cu_seqlens device int32 [ndoc+1];
 *   Hq % Hkv == 0; d in {64, 128}; scale > 0 and finite; causal 0/1; out device [q_len, Hq, d] of
 *   out_dtype (NSP_F32 or io_dtype); lse device float32 [Hq, q_len] (may be
 *   NULL when not needed); workspace device, at least
 *   nsp_attn_fwd_workspace_size(...) bytes, contents need no initialisation.
 *
 * Kernel choice: bf16 (d = 128 or 64) runs on the tensor cores (tcgen05,
 * TMEM, TMA), any Hq / Hkv (an even ratio pairs two query heads of a KV
 * group per work item, an odd one, multi-head attention among them, pairs
 * two adjacent query tiles of one head).  float32 I/O runs on the CUDA
 * cores: a correct but much slower path (nsp_path_launches tells which
 * ran).
 * ---------------------------------------------------------------------- */
size_t nsp_attn_fwd_workspace_size(int64_t q_len, int64_t kv_len, int32_t Hq, int32_t Hkv,
                                   int32_t d);

int32_t nsp_attn_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                     int32_t ndoc, int64_t q_start, int64_t q_len, int64_t kv_start,
                     int64_t kv_len, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                     int32_t causal, int32_t io_dtype, void* out, int32_t out_dtype,
                     float* lse, void* workspace, size_t workspace_bytes, nsp_stream_t stream);

/* Host-only argument check of nsp_attn_fwd (no CUDA call): returns the
 * status nsp_attn_fwd would return before enqueuing anything. */
int32_t nsp_attn_fwd_validate(const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens, int32_t ndoc, int64_t q_start,
                              int64_t q_len, int64_t kv_start, int64_t kv_len, int32_t Hq,
                              int32_t Hkv, int32_t d, int32_t causal, int32_t io_dtype,
                              const void* out, int32_t out_dtype, const void* workspace,
                              size_t workspace_bytes);

/* ------------------------------------------------------------------------
 * Ring partial accumulated in place: the partial block of nsp_attn_fwd
 * merged into a running result inside the attention kernel itself (the
 * running result enters the online softmax as one more weighted term).
 * This is the ring's online accumulation (HSAP Sec. 2.2.1) with the
 * receive-side rescale fused into the attention computation, as HSAP's
 * Limitations section proposes; nsp_lse_merge is the same combine as a
 * separate pass.  Results agree with partials + nsp_lse_merge to well
 * inside the stated tolerances, not bit for bit (P is rounded to bf16
 * against a different reference maximum).
 *
 * For the query rows [q_start, q_start + q_len) against the keys
 * [kv_start, kv_start + kv_len) (global token ids, checked against
 * cu_seqlens exactly as in nsp_attn_fwd) it forms the partial (o_p, lse_p)
 * and updates, per (row t, head h):
 *   lse' = log(exp(lse_acc) + exp(lse_p)),
 *   acc' = exp(lse_acc - lse') acc + exp(lse_p - lse') o_p.
 * Rows that see no key of the range (lse_p = -inf) are left unchanged.
 *   q, k, v, cu_seqlens, ndoc, ranges, Hq, Hkv, d, scale, causal, io_dtype,
 *     workspace: as nsp_attn_fwd (workspace sized by
 *     nsp_attn_fwd_workspace_size(q_len, kv_len, ...)).
 *   acc: device float32 [q_len, Hq, d], read and written.
 *   lse_acc: device float32 [Hq, q_len] (natural log), read and written;
 *     required.
 * Start a ring with lse_acc = -inf and acc = 0 everywhere; after the last
 * block acc holds the attention output and lse_acc its log-sum-exp (a row
 * that never saw a key keeps acc = 0, lse_acc = -inf).  Blocks may come in
 * any order.  Errors: as nsp_attn_fwd (with out_dtype = NSP_F32); a NULL
 * lse_acc is NSP_ERR_INVALID.
 * ---------------------------------------------------------------------- */
int32_t nsp_attn_fwd_accumulate(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens, int32_t ndoc, int64_t q_start,
                                int64_t q_len, int64_t kv_start, int64_t kv_len, int32_t Hq,
                                int32_t Hkv, int32_t d, float scale, int32_t causal,
                                int32_t io_dtype, float* acc, float* lse_acc, void* workspace,
                                size_t workspace_bytes, nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Whole-stream forward with q and out in the head-group-major layout an
 * Ulysses-style all-to-all delivers ([HSAP] Sec. 2.2.2: IntraSP moves
 * R^{n x H x d} per rank to R^{N x h x d}, h = H / P; [BASP] Sec. II-C):
 *   q, out: device [P][T][Hq / P][d] (group g holds query heads
 *     g Hq/P .. (g + 1) Hq/P - 1 of every token, i.e.
 *     nsp_seq2head_permute's output);
 *   k, v: device [T][Hkv][d] (the packed layout, not permuted: a group's
 *     query heads find their key/value head as h / (Hq / Hkv));
 *   lse: device float32 [Hq, T] or NULL.
 * The result equals nsp_attn_fwd on the packed layout followed by
 * nsp_seq2head_permute of out, bit for bit (same kernels, same order of
 * arithmetic), without either permutation pass: the kernels address the
 * grouped rows directly (TMA coordinates of a [P T, (Hq/P) d] map).
 * P must divide Hq; P T must fit in int32.  Kernel choice as nsp_attn_fwd
 * (tensor cores for bf16; CUDA cores for float32 I/O).
 * Other arguments and errors: as nsp_attn_fwd
 * with q_start = kv_start = 0, q_len = kv_len = T (workspace sized by
 * nsp_attn_fwd_workspace_size(T, T, ...)); a bad P is NSP_ERR_INVALID.
 * ---------------------------------------------------------------------- */
int32_t nsp_attn_fwd_headgroups(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens, int32_t ndoc, int64_t T, int32_t Hq,
                                int32_t Hkv, int32_t d, int32_t P, float scale, int32_t causal,
                                int32_t io_dtype, void* out, int32_t out_dtype, float* lse,
                                void* workspace, size_t workspace_bytes, nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Batched ring blocks: several (query range, key range) blocks of the same
 * packed stream in one call ([HSAP] Sec. 2.2.1, InterSP: each rank's query
 * shard meets every key/value shard; Sec. 3.2, attention blocks A1-A5).  On
 * one GPU holding every shard, a ring step (or a whole ring) is one schedule
 * and one persistent launch instead of one call per block.
 *
 *   q: device [T][Hq][d], k, v: device [T][Hkv][d]: the whole packed stream;
 *      a block's rows are addressed by global token ids.
 *   blocks: host array of nblocks (1..64) descriptors, read during the call:
 *      q_start, q_len: the block's query rows; kv_start, kv_len: its keys;
 *      out: device float32 [q_len][Hq][d]; lse: device float32 [Hq][q_len]
 *      (required when accumulate = 1, else optional).
 *   accumulate = 0: each block's out / lse are written with the partial of
 *      its rows against its keys, exactly as nsp_attn_fwd with out_dtype =
 *      NSP_F32, q / k / v pointing at the block's rows and
 *      q_start / kv_start as given (bit-identical results).
 *   accumulate = 1: each block's partial is merged into its out / lse in
 *      place, as nsp_attn_fwd_accumulate does.
 * The blocks' outputs must not share bytes (NSP_ERR_INVALID otherwise): a
 * ring step's blocks have distinct query shards.  Rows of a block that see
 * no key of it get out = 0, lse = -inf (accumulate: left unchanged).
 * Workspace: at least nsp_attn_fwd_blocks_workspace_size(nblocks, blocks,
 * ...) bytes.  Other arguments, kernel choice and errors as nsp_attn_fwd;
 * ranges outside [0, T) are NSP_ERR_INVALID.
 * ---------------------------------------------------------------------- */
typedef struct {
  int64_t q_start, q_len, kv_start, kv_len;
  void* out;
  float* lse;
} nsp_block_t;

size_t nsp_attn_fwd_blocks_workspace_size(int32_t nblocks, const nsp_block_t* blocks, int32_t Hq,
                                          int32_t Hkv, int32_t d);

int32_t nsp_attn_fwd_blocks(const void* q, const void* k, const void* v,
                            const int32_t* cu_seqlens, int32_t ndoc, int64_t T, int32_t nblocks,
                            const nsp_block_t* blocks, int32_t Hq, int32_t Hkv, int32_t d,
                            float scale, int32_t causal, int32_t io_dtype, int32_t accumulate,
                            void* workspace, size_t workspace_bytes, nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Batched ring-block backward: the gradient contributions of many
 * (query range, key range) blocks of one packed stream, as
 * nsp_attn_bwd_accumulate computes them for each block (full-row
 * probabilities and delta, sums restricted to the block; [HSAP] Sec. 2.2.1
 * ring InterSP, Sec. 3.2 blocks), in one schedule and one launch of each
 * backward kernel: a whole ring's backward as one call.
 *
 *   q, out, dout: device [T][Hq][d]; k, v: device [T][Hkv][d]: the whole
 *     stream, rows addressed by global token ids; lse: device float32 [Hq][T],
 *     the rows' final lse (the forward's over all keys).
 *   ranges: host array of nranges (1..64) {q_start, q_len, kv_start, kv_len},
 *     read during the call; blocks may share rows or overlap.
 *   dq_acc: device float32 [T][Hq][d]; dk_acc, dv_acc: device float32
 *     [T][Hkv][d]: every block's contributions are ADDED at global rows with
 *     float atomics (the caller zeroes them first; the order of the
 *     additions, hence the last bits, may vary between runs).
 * Tensor cores only: bf16 with d = 128 or 64 (float32: NSP_ERR_UNSUPPORTED;
 * use nsp_attn_bwd_accumulate per block).  Every q_start must be a multiple
 * of 4 (NSP_ERR_UNSUPPORTED otherwise).  Workspace: at least
 * nsp_attn_bwd_blocks_workspace_size(T, nranges, ranges, Hq, Hkv, d) bytes;
 * bytes past it (from the next 1024-byte boundary) are a dS cache as for
 * nsp_attn_bwd, used when it holds every visible tile pair of every block
 * (nsp_attn_bwd_blocks_ds_cache_size bytes).
 * Other arguments and errors as nsp_attn_bwd_accumulate.
 * ---------------------------------------------------------------------- */
typedef struct {
  int64_t q_start, q_len, kv_start, kv_len;
} nsp_range_t;

size_t nsp_attn_bwd_blocks_workspace_size(int64_t T, int32_t nranges, const nsp_range_t* ranges,
                                          int32_t Hq, int32_t Hkv, int32_t d);

/* Bytes of dS cache that let nsp_attn_bwd_blocks compute dq from cached
 * tiles: Hq x (visible 128 x 128 tile pairs of every block, tiles aligned to
 * the block's q_start and kv_start) x 32768, from HOST cu_seqlens [ndoc + 1].
 * 0 for a bad argument. */
size_t nsp_attn_bwd_blocks_ds_cache_size(const int32_t* cu_seqlens_host, int32_t ndoc,
                                         int32_t nranges, const nsp_range_t* ranges, int32_t Hq,
                                         int32_t causal);

int32_t nsp_attn_bwd_blocks(const void* q, const void* k, const void* v, const void* out,
                            const void* dout, const float* lse, const int32_t* cu_seqlens,
                            int32_t ndoc, int64_t T, int32_t nranges, const nsp_range_t* ranges,
                            int32_t Hq, int32_t Hkv, int32_t d, float scale, int32_t causal,
                            int32_t io_dtype, float* dq_acc, float* dk_acc, float* dv_acc,
                            void* workspace, size_t workspace_bytes, nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * nsp_attn_fwd without a workspace argument.  No page has a counterpart of
 * this entry point: it exists for callers that cannot allocate device
 * memory where they run attention (code inside a custom allocator or
 * memory-pool callback, plugins whose host framework owns every device
 * allocation, processes that must keep a fixed footprint after start-up).
 *
 * Same arguments, semantics, layouts and results as nsp_attn_fwd, minus
 * workspace / workspace_bytes.  The scheduler scratch lives in a 1 MiB
 * static __device__ array of the library instead, present on every GPU that
 * loads the library until the process exits; nothing is allocated (no
 * cudaMalloc, cudaFree or allocating library call).
 *   Limit: nsp_attn_fwd_workspace_size(q_len, kv_len, ...) must not exceed
 *   1 MiB (about 8.3 million query tokens when q_len = kv_len); larger
 *   problems return NSP_ERR_WORKSPACE before anything is enqueued.
 *   device_status: optional device int32; receives (stream-ordered) the
 *   status word the kernels recorded (NSP_OK, NSP_ERR_INVALID for a bad
 *   cu_seqlens, NSP_ERR_TIMEOUT); NULL to skip.
 *   The first call on each device looks up the array's device address with
 *   cudaGetSymbolAddress (with that device current) and caches it; make that
 *   first call before any stream capture.
 *   Every call shares the one array per device: calls whose kernels overlap
 *   on the GPU (other streams, other host threads) race and must be
 *   serialised by the caller.  Each call rewrites all the scratch it reads.
 * ---------------------------------------------------------------------- */
int32_t nsp_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                             const int32_t* cu_seqlens, int32_t ndoc, int64_t q_start,
                             int64_t q_len, int64_t kv_start, int64_t kv_len, int32_t Hq,
                             int32_t Hkv, int32_t d, float scale, int32_t causal,
                             int32_t io_dtype, void* out, int32_t out_dtype, float* lse,
                             int32_t* device_status, nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Varlen attention backward over the whole stream ([NSP] Sec. 2.3: the
 * backward recomputes attention; only out and lse are kept).
 *
 * Gradients of L = sum(dout * out) for the forward above (q_start =
 * kv_start = 0, q_len = kv_len = T):
 *   delta_t = <dout[t,h], out[t,h]>,  p_tj = exp(x_tj - lse[h,t]),
 *   dS_tj = p_tj (<dout[t,h], v[j,g]> - delta_t),
 *   dq[t,h] = scale sum_j dS_tj k[j,g],
 *   dk[j,g] = scale sum_{h in g} sum_t dS_tj q[t,h],
 *   dv[j,g] = sum_{h in g} sum_t p_tj dout[t,h].
 * out and lse must be the forward's results for the same inputs.
 * dq, dk, dv are written (not accumulated) in io_dtype.  The workspace (at
 * least nsp_attn_bwd_workspace_size bytes for the same T, heads, d and
 * io_dtype) holds the tile schedules, delta and lse * log2(e); its contents
 * need no initialisation.  bf16 (d = 128 or 64) runs on the tensor cores
 * (dq, dk, dv each written once, deterministic); float32 runs on CUDA cores,
 * whose dq is summed with float atomics in a float32 accumulator that the
 * workspace then also holds (last bits may vary).
 *
 * dS cache (tensor-core path only; storing instead of recomputing, the
 * trade NSP Sec. 2.3 weighs for attention's backward).  Workspace bytes past
 * nsp_attn_bwd_workspace_size (from the next 1024-byte boundary on) are a
 * cache for dS = P (dP - delta), the probabilities' gradient: when it holds
 * every visible (128-row query tile, 128-key tile) pair of every query head
 * (nsp_attn_bwd_ds_cache_size bytes), the dK/dV kernel copies each dS tile
 * it builds into the cache and dq is computed from the cached tiles (one
 * 128 x 128 x 128 product per pair instead of recomputing S and dP: three).
 * Otherwise, or with no such bytes, dq recomputes them.  The decision is
 * taken on the device from cu_seqlens; results agree within rounding (dq
 * then uses the dS rounded to bf16 that dk uses; deterministic either way).
 * ---------------------------------------------------------------------- */
size_t nsp_attn_bwd_workspace_size(int64_t T, int32_t Hq, int32_t Hkv, int32_t d,
                                   int32_t io_dtype);

/* Bytes of dS cache that let nsp_attn_bwd / nsp_attn_bwd_headgroups compute
 * dq from cached tiles: Hq x (visible 128 x 128 tile pairs) x 32768, from
 * HOST cu_seqlens [ndoc + 1] (int32, non-decreasing from 0).  Pass at least
 * nsp_attn_bwd_workspace_size rounded up to 1024, plus this, as the
 * workspace.  0 for a bad argument. */
size_t nsp_attn_bwd_ds_cache_size(const int32_t* cu_seqlens_host, int32_t ndoc, int32_t Hq,
                                  int32_t causal);

/* Whether the last backward on this workspace computed dq from the dS cache:
 * *used = 1 or 0, read from the workspace header (a copy to the host on
 * stream, then a synchronisation of stream).  NSP_ERR_INVALID for a NULL
 * argument, NSP_ERR_CUDA if the copy fails. */
int32_t nsp_bwd_ds_cache_used(const void* workspace, int32_t* used, nsp_stream_t stream);

int32_t nsp_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, const int32_t* cu_seqlens,
                     int32_t ndoc, int64_t T, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                     int32_t causal, int32_t io_dtype, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, nsp_stream_t stream);

int32_t nsp_attn_bwd_validate(const void* q, const void* k, const void* v, const void* out,
                              const void* dout, const float* lse, const int32_t* cu_seqlens,
                              int32_t ndoc, int64_t T, int32_t Hq, int32_t Hkv, int32_t d,
                              int32_t causal, int32_t io_dtype, const void* dq,
                              const void* dk, const void* dv, const void* workspace,
                              size_t workspace_bytes);

/* ------------------------------------------------------------------------
 * Whole-stream backward in the Ulysses receive layout, the backward of
 * nsp_attn_fwd_headgroups ([HSAP] Sec. 2.2.2; [BASP] Sec. II-C):
 *   q, out, dout, dq: device [P][T][Hq / P][d] (head-group-major);
 *   k, v, dk, dv: device [T][Hkv][d] (packed);
 *   lse: device float32 [Hq, T].
 * The gradients equal nsp_attn_bwd on the packed layout with dq moved by
 * nsp_seq2head_permute, bit for bit, without the permutation passes.
 * P must divide Hq; P T must fit in int32.  Other arguments, workspace
 * (nsp_attn_bwd_workspace_size(T, ...)) and errors: as nsp_attn_bwd; a bad P
 * is NSP_ERR_INVALID.
 * ---------------------------------------------------------------------- */
int32_t nsp_attn_bwd_headgroups(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse,
                                const int32_t* cu_seqlens, int32_t ndoc, int64_t T, int32_t Hq,
                                int32_t Hkv, int32_t d, int32_t P, float scale, int32_t causal,
                                int32_t io_dtype, void* dq, void* dk, void* dv, void* workspace,
                                size_t workspace_bytes, nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Ring-block backward: one (query range, key range) block's share of the
 * gradients, added into float32 accumulators.  In ring-style InterSP
 * ([HSAP] Sec. 2.2.1) each rank keeps its query shard and the key/value
 * blocks circulate; the backward meets every block once, adds the block's
 * dq into its own accumulator and sends the block's dk/dv contribution on
 * with the block.  Summing the blocks of any chunking of queries and keys
 * gives nsp_attn_bwd's gradients.
 *
 * For the query rows [q_start, q_start + q_len) and the keys
 * [kv_start, kv_start + kv_len) (global token ids, checked against
 * cu_seqlens as in nsp_attn_fwd), with p_tj and delta_t those of the whole
 * row (lse and out are the row's final results over all its keys):
 *   dq_acc[t - q_start, h] += scale sum_{j in block} dS_tj k[j, g],
 *   dk_acc[j - kv_start, g] += scale sum_{t in block, h in g} dS_tj q[t, h],
 *   dv_acc[j - kv_start, g] += sum_{t in block, h in g} p_tj dout[t, h].
 *   q, out, dout: device io_dtype [q_len, Hq, d] (the query shard, its final
 *     attention output and the output gradient).
 *   lse: device float32 [Hq, q_len], the rows' final log-sum-exp.
 *   k, v: device io_dtype [kv_len, Hkv, d] (the key/value block).
 *   dq_acc: device float32 [q_len, Hq, d]; dk_acc, dv_acc: device float32
 *     [kv_len, Hkv, d]; read and written (start them at zero).
 *   workspace: device, at least nsp_attn_bwd_accumulate_workspace_size(q_len,
 *     kv_len, ...) bytes, no initialisation.
 * Pairs no query of the block can see add nothing; a block with no visible
 * pair leaves the accumulators unchanged.  bf16 (d = 128 or 64) runs on the
 * tensor cores (each accumulator element read and written once per call);
 * float32 runs on CUDA cores (dq_acc summed with float atomics).
 * Errors: as nsp_attn_bwd (NULL or misaligned buffers, bad scalars before
 * any launch; a bad cu_seqlens through the workspace status word).
 * ---------------------------------------------------------------------- */
size_t nsp_attn_bwd_accumulate_workspace_size(int64_t q_len, int64_t kv_len, int32_t Hq,
                                              int32_t Hkv, int32_t d, int32_t io_dtype);

int32_t nsp_attn_bwd_accumulate(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse,
                                const int32_t* cu_seqlens, int32_t ndoc, int64_t q_start,
                                int64_t q_len, int64_t kv_start, int64_t kv_len, int32_t Hq,
                                int32_t Hkv, int32_t d, float scale, int32_t causal,
                                int32_t io_dtype, float* dq_acc, float* dk_acc, float* dv_acc,
                                void* workspace, size_t workspace_bytes, nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Log-sum-exp merge of n partials of the same T query rows over disjoint
 * key sets ([HSAP] Sec. 2.2.1 online accumulation; Limitations "rescale"):
 *   m = max_i lse_i;  m = -inf -> out = 0, lse = -inf;  otherwise
 *   lse = m + ln sum_i exp(lse_i - m),  out = sum_i exp(lse_i - lse) out_i.
 *
 * outs, lses: HOST arrays of n DEVICE pointers (1 <= n <= 64); outs[i] is
 *   float32 [T, H, d], lses[i] float32 [H, T].  out: device [T, H, d] of
 *   out_dtype (NSP_F32 or NSP_BF16, round-to-nearest-even); lse: device
 *   float32 [H, T] (may be NULL).  out and lse must not overlap any input.
 * ---------------------------------------------------------------------- */
int32_t nsp_lse_merge(const float* const* outs, const float* const* lses, int32_t n,
                      int64_t T, int32_t H, int32_t d, void* out, int32_t out_dtype,
                      float* lse, nsp_stream_t stream);

int32_t nsp_lse_merge_validate(const float* const* outs, const float* const* lses, int32_t n,
                               int64_t T, int32_t H, int32_t d, const void* out,
                               int32_t out_dtype, const float* lse);

/* ------------------------------------------------------------------------
 * Several independent LSE merges in one launch: segment g combines its
 * counts[g] partials into out[g] / lse[g], exactly as nsp_lse_merge would
 * (same arithmetic, same results).  For a ring on one GPU this merges every
 * query shard at once ([HSAP] Sec. 2.2.1), so the launch ramps up and
 * drains once instead of once per shard.
 *   nseg: 1 .. 16 segments, each of T tokens, H heads, head dim d.
 *   counts: HOST int32 [nseg], each >= 1, sum <= 64.
 *   outs, lses: HOST arrays of sum(counts) device pointers, segment after
 *     segment (layouts as in nsp_lse_merge).
 *   out: HOST array of nseg device pointers [T, H, d] (out_dtype);
 *   lse: HOST array of nseg device pointers [H, T] (entries may be NULL),
 *     or NULL.
 * Errors: as nsp_lse_merge, per segment; bad nseg / counts are
 * NSP_ERR_INVALID.
 * ---------------------------------------------------------------------- */
int32_t nsp_lse_merge_batch(int32_t nseg, const int32_t* counts, const float* const* outs,
                            const float* const* lses, int64_t T, int32_t H, int32_t d,
                            void* const* out, int32_t out_dtype, float* const* lse,
                            nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Ulysses seq -> head permutation ([HSAP] Sec. 2.2.2: blocks in
 * R^{n x H x d} per group become R^{N x h x d}, h = H / P; [BASP] Sec. II-C).
 * With the P sequence shards stacked on this device as in = [T, H, d]:
 *   inverse = 0:  out[g][t][j][:] = in[t][g*h + j][:]    out = [P, T, h, d]
 *   inverse = 1:  out[t][g*h + j][:] = in[g][t][j][:]    (head -> seq)
 * Elements are elem_bytes wide (1, 2, 4 or 8) and copied bit-exactly.
 * H % P == 0; in and out must not overlap.
 * ---------------------------------------------------------------------- */
int32_t nsp_seq2head_permute(const void* in, void* out, int64_t T, int32_t H, int32_t d,
                             int32_t P, int32_t elem_bytes, int32_t inverse,
                             nsp_stream_t stream);

int32_t nsp_seq2head_permute_validate(const void* in, const void* out, int64_t T, int32_t H,
                                      int32_t d, int32_t P, int32_t elem_bytes);

/* ------------------------------------------------------------------------
 * Batch-aware subgroup all-to-all layout ([BASP] Sec. IV, "Batch-aware
 * group formation", "Batch Aware Sequence Partitioning" (Alg. 2),
 * "Subgroup all-to-all"): a micro-batch of B sequences of L tokens on
 * N = B K ranks, where each sequence is sharded over its own group of K ranks
 * and each group runs an independent K-way all-to-all.  With the batch
 * stacked on one device, the receive side of all B groups:
 *   inverse = 0:  out[b][g][t][j][:] = in[b L + t][g H/K + j][:]
 *   inverse = 1:  in[b L + t][g H/K + j][:] = out[b][g][t][j][:] (roles of
 *                 the buffers swapped: `in` is [B][K][L][H/K][d])
 *   in:  device [B L][H][d] elements of elem_bytes (1, 2, 4 or 8 bytes);
 *   out: device [B][K][L][H/K][d].
 * Each group's block is the nsp_seq2head_permute of its own sequence with
 * P = K (B = 1 is exactly that call); no data crosses sequences.  Bit-exact
 * data movement, one launch for all B groups.  Errors as
 * nsp_seq2head_permute on the whole [B L, H, d] batch (K must divide H;
 * in, out 16-byte aligned, not overlapping); B < 1 or L < 0 is
 * NSP_ERR_INVALID.
 * ---------------------------------------------------------------------- */
int32_t nsp_seq2head_permute_groups(const void* in, void* out, int32_t B, int64_t L, int32_t H,
                                    int32_t d, int32_t K, int32_t elem_bytes, int32_t inverse,
                                    nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Status word of the last call that used `workspace`.  Synchronises `stream`
 * first (the only synchronising call).  Returns NSP_OK, the recorded device
 * error (NSP_ERR_INVALID for bad cu_seqlens, NSP_ERR_TIMEOUT), or
 * NSP_ERR_CUDA if the synchronisation itself failed.
 * ---------------------------------------------------------------------- */
int32_t nsp_status_query(const void* workspace, nsp_stream_t stream);

/* ------------------------------------------------------------------------
 * Useful work of a whole-stream causal/bidirectional attention, from a HOST
 * copy of cu_seqlens (NSP's cost model takes "attention FLOPs" of the routed
 * inputs, [NSP] Sec. 4.1): pairs = allowed (query, key) pairs per query head.
 * Writes *pairs; returns NSP_ERR_INVALID for a malformed cu_seqlens.
 * ---------------------------------------------------------------------- */
int32_t nsp_attn_pairs(const int32_t* cu_seqlens_host, int32_t ndoc, int32_t causal,
                       double* pairs);

/* ------------------------------------------------------------------------
 * Cost of one attention call, from a HOST copy of cu_seqlens: the hook a
 * planner that balances attention work over ranks or pipelines needs (NSP
 * Sec. 4.1: the backend reports the attention FLOPs of the inputs routed to
 * it; HSAP Sec. 3.2 balances ranks by attention block counts).  For the
 * query rows [q_start, q_start + q_len) against the keys
 * [kv_start, kv_start + kv_len) (the whole stream: 0, T, 0, T):
 *   pairs      allowed (query, key) pairs per query head;
 *   fwd_flop   4 d Hq pairs (Q K^T and P V);
 *   bwd_flop   10 d Hq pairs (the recomputed Q K^T, dOut V^T, P^T dOut,
 *              dS^T Q, dS K);
 *   tiles      (128-row query tile, 128-key tile) pairs holding at least one
 *              allowed pair: the tiles the kernels schedule, per query head
 *              (executed tensor-core work is 4 d Hq 128^2 tiles forward);
 *   fwd_bytes  compulsory HBM bytes of nsp_attn_fwd: q, k, v read, out
 *              written in io_dtype, lse written (float32);
 *   bwd_bytes  compulsory HBM bytes of nsp_attn_bwd: q, k, v, out, dout and
 *              lse read, dq, dk, dv written.
 * Returns NSP_ERR_INVALID for a malformed cu_seqlens, ranges outside it or
 * bad head counts; *cost is written only on NSP_OK.  No device work.
 * ---------------------------------------------------------------------- */
typedef struct {
  double pairs, fwd_flop, bwd_flop, tiles, fwd_bytes, bwd_bytes;
} nsp_attn_cost_t;

int32_t nsp_attn_cost(const int32_t* cu_seqlens_host, int32_t ndoc, int64_t q_start,
                      int64_t q_len, int64_t kv_start, int64_t kv_len, int32_t Hq, int32_t Hkv,
                      int32_t d, int32_t causal, int32_t io_dtype, nsp_attn_cost_t* cost);

#ifdef __cplusplus
}
#endif

#endif /* NSP_H_ */
