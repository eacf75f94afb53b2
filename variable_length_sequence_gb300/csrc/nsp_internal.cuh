// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "nsp.h"

namespace nsp {

// Fixed-size header at the start of every attention workspace.
struct WsHeader {
  int32_t status;       // nsp_status recorded by device code (0 = OK)
  int32_t counter;      // dynamic work-fetch counter (reset by the prep kernel)
  int32_t n_items;      // number of scheduled work items
  int32_t max_cost;     // largest per-q-tile KV-tile count
  int32_t counter2;     // second work counter (backward dK/dV)
  int32_t n_items2;
  int32_t n_nonempty;   // query tiles that see a key (listed first in the order)
  int32_t ds_on;        // backward: dS of every visible tile pair fits the cache
  int64_t ds_pairs;     // backward: visible (query tile, key tile) pairs per head
  int32_t pad[54];      // header is 256 bytes
};
static_assert(sizeof(WsHeader) == 256, "workspace header must stay 256 bytes");

constexpr int kTileM = 128;        // query rows per tile (tcgen05 M)
constexpr int kTileN = 128;        // keys per KV tile

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The softmax scale must be a positive finite number (a temperature).
inline bool scale_ok(float scale) { return scale > 0.f && scale <= 3.0e38f; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Forward workspace layout (all offsets from the workspace base).  The
// scheduled query tiles are tile_rows = 128 rows, or 256 when the
// tensor-core forward pairs two 128-row tiles of one head per work item
// (fwd_tile_rows); the size of the 128-row layout bounds both.
struct FwdWsLayout {
  size_t tiles;        // int2 [n_qtiles]: first/last KV tile of each query tile
  size_t order;        // int32 [n_qtiles]: query tiles, most KV tiles first
  size_t hist;         // int32 [n_kvtiles + 2]: counting-sort buckets
  size_t total;
  int64_t n_qtiles, n_kvtiles;
  int32_t tile_rows;
};

// Rows of a scheduled forward query tile: 256 when the tensor-core forward
// takes the problem (bf16, d = 128 or 64) with an odd number of query heads per
// KV head (multi-head attention among them): a work item is then two
// adjacent 128-row tiles of one head, which read the same K/V tiles; 128
// otherwise (a work item is one tile and two heads of a KV group).
inline int32_t fwd_tile_rows(int32_t io_dtype, int32_t d, int32_t Hq, int32_t Hkv) {
  return (io_dtype == NSP_BF16 && (d == 128 || d == 64) && Hkv > 0 && ((Hq / Hkv) & 1)) ? 2 * kTileM
                                                                                  : kTileM;
}

// One (query range, key range) block of a forward call, and the table of a
// call's blocks, passed to the schedule and attention kernels by value.
// The single-range entry points use one block whose q / k / v pointers are
// the block's own first rows (global_rows = 0); the batched entry point
// (nsp_attn_fwd_blocks) addresses whole-stream q / k / v by global token ids
// (global_rows = 1).  Token ids fit in int32 (at most 2^30 tokens).
constexpr int kMaxBlocks = 64;
struct FwdBlock {
  int32_t q_start, q_len, kv_start, kv_len;   // global token ids
  int32_t tile0;                              // first scheduled query tile of the block
  int32_t ktile0;                             // first scheduled key tile (backward)
  void* out;                                  // [q_len, Hq, d]
  float* lse;                                 // [Hq, q_len] or null
};
struct FwdBlocks {
  int32_t n;
  int32_t global_rows;
  FwdBlock b[kMaxBlocks];
};

inline FwdWsLayout fwd_ws_layout(int64_t q_len, int64_t kv_len, int32_t tile_rows = kTileM) {
  FwdWsLayout L;
  L.tile_rows = tile_rows;
  L.n_qtiles = ceil_div(q_len, tile_rows);
  L.n_kvtiles = ceil_div(kv_len, kTileN);
  size_t off = sizeof(WsHeader);
  L.tiles = off;  off = align_up(off + sizeof(int2) * (size_t)L.n_qtiles, 256);
  L.order = off;  off = align_up(off + sizeof(int32_t) * (size_t)L.n_qtiles, 256);
  L.hist = off;   off = align_up(off + sizeof(int32_t) * (size_t)(L.n_kvtiles + 2), 256);
  L.total = off;
  return L;
}

// Layout of a batched forward: the query tiles of every block, one sort;
// fills in each block's tile0.
inline FwdWsLayout fwd_ws_layout_blocks(FwdBlocks& B, int32_t tile_rows) {
  int64_t n_q = 0, max_kv = 0;
  for (int i = 0; i < B.n; ++i) {
    B.b[i].tile0 = (int32_t)n_q;
    n_q += ceil_div(B.b[i].q_len, tile_rows);
    max_kv = B.b[i].kv_len > max_kv ? B.b[i].kv_len : max_kv;
  }
  FwdWsLayout L = fwd_ws_layout(n_q * tile_rows, max_kv, tile_rows);
  return L;
}

// Backward workspace: header; schedule of 128-row query tiles listing
// 128-key tiles (dQ kernel) and of 128-key tiles listing 128-row query tiles
// (dK/dV kernel); delta and lse * log2(e) [Hq, Tp] f32 (rows padded to whole
// 128-row tiles, padding zeroed); and, for the CUDA-core path of the
// whole-stream backward only, a float32 dq accumulator [q_len, Hq, d].
// A ring block (nsp_attn_bwd_accumulate) has q_len query rows and kv_len keys;
// the whole-stream backward is q_len = kv_len = T.
constexpr int kBwdSub = 128;       // tile granularity listed by the backward schedules

struct BwdWsLayout {
  size_t qtiles, qorder, qhist;    // int2 [n_qtiles], int32 [n_qtiles], int32 [n_qhist]
  size_t ktiles, korder, khist;    // int2 [n_ktiles], int32 [n_ktiles], int32 [n_khist]
  size_t delta;                    // float [Hq, Tp]
  size_t nlse2;                     // float [Hq, Tp]
  size_t dq_acc;                   // float [q_len, Hq, d] (CUDA-core path)
  size_t qoff;                     // int64 [n_qtiles]: first dS slot of each query tile
  size_t total;
  // dS cache (tensor-core backward of the whole stream or of a table of
  // blocks): the workspace bytes past total, from ds_cache on (0 bytes: dQ
  // recomputes S and dP)
  size_t ds_cache = 0, ds_cache_bytes = 0;
  int64_t Tp, n_qtiles, n_ktiles;
  int64_t n_qhist, n_khist;        // counting-sort buckets of the two schedules
};

inline BwdWsLayout bwd_ws_layout(int64_t q_len, int64_t kv_len, int32_t Hq, int32_t d,
                                 bool need_dq_acc) {
  BwdWsLayout L;
  L.n_qtiles = ceil_div(q_len, kTileM);
  L.n_ktiles = ceil_div(kv_len, kTileN);
  L.Tp = L.n_qtiles * kTileM;
  L.n_qhist = L.n_ktiles + 2;
  L.n_khist = L.n_qtiles + 2;
  size_t off = sizeof(WsHeader);
  L.qtiles = off; off = align_up(off + sizeof(int2) * (size_t)L.n_qtiles, 256);
  L.qorder = off; off = align_up(off + sizeof(int32_t) * (size_t)L.n_qtiles, 256);
  L.qhist = off;  off = align_up(off + sizeof(int32_t) * (size_t)L.n_qhist, 256);
  L.ktiles = off; off = align_up(off + sizeof(int2) * (size_t)L.n_ktiles, 256);
  L.korder = off; off = align_up(off + sizeof(int32_t) * (size_t)L.n_ktiles, 256);
  L.khist = off;  off = align_up(off + sizeof(int32_t) * (size_t)L.n_khist, 256);
  L.delta = off;  off = align_up(off + sizeof(float) * (size_t)Hq * (size_t)L.Tp, 256);
  L.nlse2 = off;   off = align_up(off + sizeof(float) * (size_t)Hq * (size_t)L.Tp, 256);
  L.dq_acc = off;
  if (need_dq_acc)
    off = align_up(off + sizeof(float) * (size_t)q_len * (size_t)Hq * (size_t)d, 256);
  L.qoff = off;   off = align_up(off + sizeof(int64_t) * (size_t)L.n_qtiles, 256);
  L.total = off;
  return L;
}

// Backward of a table of blocks over a whole stream of T tokens: the query
// tiles and the key tiles of every block, one sort each; delta and -lse
// log2(e) over the whole stream [Hq, Tp].  Fills in each block's tile0 and
// ktile0.
inline BwdWsLayout bwd_ws_layout_blocks(FwdBlocks& B, int64_t T, int32_t Hq) {
  int64_t nq = 0, nk = 0, max_q = 0, max_k = 0;
  for (int i = 0; i < B.n; ++i) {
    B.b[i].tile0 = (int32_t)nq;
    B.b[i].ktile0 = (int32_t)nk;
    const int64_t q = ceil_div(B.b[i].q_len, kTileM), k = ceil_div(B.b[i].kv_len, kTileN);
    nq += q; nk += k;
    max_q = q > max_q ? q : max_q;
    max_k = k > max_k ? k : max_k;
  }
  BwdWsLayout L;
  L.n_qtiles = nq;
  L.n_ktiles = nk;
  // one spare tile of (zeroed) padding: the dK/dV kernel copies the values
  // of whole 128-row tiles starting at a block's q_start, which need not be
  // a multiple of 128, so the last copy may run up to 127 rows past T
  L.Tp = (ceil_div(T, kTileM) + 1) * kTileM;
  L.n_qhist = max_k + 2;
  L.n_khist = max_q + 2;
  size_t off = sizeof(WsHeader);
  L.qtiles = off; off = align_up(off + sizeof(int2) * (size_t)nq, 256);
  L.qorder = off; off = align_up(off + sizeof(int32_t) * (size_t)nq, 256);
  L.qhist = off;  off = align_up(off + sizeof(int32_t) * (size_t)L.n_qhist, 256);
  L.ktiles = off; off = align_up(off + sizeof(int2) * (size_t)nk, 256);
  L.korder = off; off = align_up(off + sizeof(int32_t) * (size_t)nk, 256);
  L.khist = off;  off = align_up(off + sizeof(int32_t) * (size_t)L.n_khist, 256);
  L.delta = off;  off = align_up(off + sizeof(float) * (size_t)Hq * (size_t)L.Tp, 256);
  L.nlse2 = off;  off = align_up(off + sizeof(float) * (size_t)Hq * (size_t)L.Tp, 256);
  L.dq_acc = off;
  L.qoff = off;   off = align_up(off + sizeof(int64_t) * (size_t)nq, 256);
  L.total = off;
  return L;
}

// Bytes of one cached dS tile: 128 x 128 bf16.
constexpr size_t kDsTileBytes = 128 * 128 * 2;

// Problem description passed by value to kernels.
struct AttnProblem {
  const void* q; const void* k; const void* v;
  const int32_t* cu; int32_t ndoc;
  int64_t q_start, q_len, kv_start, kv_len;
  int32_t Hq, Hkv, d;
  float scale;
  int32_t causal;
  int32_t io_dtype, out_dtype;
  void* out; float* lse;
  WsHeader* hdr;
  // Forward: accumulate into a running ring result instead of writing the
  // partial: out is then the float32 accumulator and lse its log-sum-exp
  // (both read and written; rows that see no key of the range are left
  // unchanged).  Backward: add the block's dq/dk/dv into float32
  // accumulators instead of writing io-typed gradients.
  int32_t accumulate = 0;
  // Query-side layout (q, out, dout, dq): 1 = [q_len, Hq, d]; P > 1 = the
  // head-group-major [P][q_len][Hq / P][d] layout an all-to-all delivers.
  int32_t q_groups = 1;
  // Cycles a bounded device wait may last before the kernel records
  // NSP_ERR_TIMEOUT and leaves (set by the launchers from
  // nsp_set_wait_timeout_cycles).
  int64_t wait_budget = 4000000000LL;
};

// ---- launchers implemented in the .cu files (return cudaError_t) ----
// The forward's blocks: `blocks` (n >= 1), or when null the one block
// [q_start, +q_len) x [kv_start, +kv_len) of p with p's out and lse.
cudaError_t launch_fwd_schedule(const AttnProblem& p, const FwdWsLayout& L, char* ws,
                                cudaStream_t s, const FwdBlocks* blocks = nullptr);
// The backward's blocks: `blocks` (tile0 and ktile0 filled in), or when
// null the one range of p.
cudaError_t launch_bwd_schedules(const AttnProblem& p, const BwdWsLayout& L, char* ws,
                                 cudaStream_t s, const FwdBlocks* blocks = nullptr);
cudaError_t launch_attn_fwd_simt(const AttnProblem& p, cudaStream_t s);
cudaError_t launch_attn_fwd_tc(const AttnProblem& p, const FwdWsLayout& L, char* ws,
                               cudaStream_t s, bool* launched, const FwdBlocks* blocks = nullptr);
// The single block of a single-range call.
FwdBlocks single_block(const AttnProblem& p);
cudaError_t launch_attn_bwd_simt(const AttnProblem& p, const void* out, const void* dout,
                                 const float* lse, void* dq, void* dk, void* dv,
                                 const BwdWsLayout& L, char* ws, cudaStream_t s);
// True when the tensor-core backward takes this problem (bf16, d = 128 or
// 64, Hq a multiple of Hkv).
bool bwd_tc_eligible(int32_t io_dtype, int32_t d, int32_t Hq, int32_t Hkv);
// With `blocks`: every block's contributions added into whole-stream float32
// dq / dk / dv (global rows) with atomics; p covers the whole stream.
cudaError_t launch_attn_bwd_tc(const AttnProblem& p, const void* out, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv,
                               const BwdWsLayout& L, char* ws, cudaStream_t s,
                               const FwdBlocks* blocks = nullptr);
cudaError_t launch_bwd_delta(const void* out, const void* dout, const float* lse, float* delta,
                             float* nlse2, int64_t T, int64_t Tp, int Hq, int d, int io_dtype,
                             int P, WsHeader* hdr, cudaStream_t s);
cudaError_t launch_dq_convert(const float* acc, void* dq, int64_t n, int io_dtype,
                              WsHeader* hdr, cudaStream_t s);
cudaError_t launch_lse_merge(const float* const* outs, const float* const* lses, int n,
                             int64_t T, int H, int d, void* out, int out_dtype, float* lse,
                             cudaStream_t s);
cudaError_t launch_lse_merge_segments(int nseg, const int* counts, const float* const* outs,
                                      const float* const* lses, int64_t T, int H, int d,
                                      void* const* dst, int out_dtype, float* const* dst_lse,
                                      cudaStream_t s);
cudaError_t launch_permute(const void* in, void* out, int64_t T, int H, int d, int P,
                           int elem_bytes, int inverse, cudaStream_t s);
// nb independent permutations of T-token groups stacked in memory.
cudaError_t launch_permute_groups(const void* in, void* out, int64_t nb, int64_t T, int H, int d,
                                  int P, int elem_bytes, int inverse, cudaStream_t s);

// Number of SMs of the current device (cached per device).
int num_sms();

// Grid of the persistent attention kernels (num_sms(), or fewer CTAs when
// the environment variable NSP_PERSISTENT_CTAS asks for it).
int persistent_grid();

// Adds n to the library-wide count of kernels launched (nsp_kernel_launches).
void count_launches(int n);

// Counts one attention kernel launch on the tensor-core path (true) or the
// CUDA-core path (false) (nsp_path_launches).
void count_path(bool tensor_core);

// The process-wide bound of device waits (nsp_set_wait_timeout_cycles).
int64_t wait_budget_cycles();

}  // namespace nsp

// ---- device helpers ----
#ifdef __CUDACC__
namespace nsp {

__device__ __forceinline__ float ld_in(const float* p) { return *p; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ void st_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Index of the document holding global token t: the last b with cu[b] <= t
// (binary search over cu[0..ndoc]); zero-length documents are never returned.
__device__ __forceinline__ int doc_of(const int32_t* __restrict__ cu, int ndoc, int64_t t) {
  int lo = 0, hi = ndoc;            // answer in [0, ndoc - 1]
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Element offset of (range-relative row, query head h) in q / out: the
// packed [rows, Hq, d] layout, or the head-group-major [P][rows][Hq/P][d]
// layout when p.q_groups = P > 1.
__device__ __forceinline__ int64_t qo_offset(const AttnProblem& p, int64_t row, int h) {
  if (p.q_groups <= 1) return (row * p.Hq + h) * p.d;
  const int hpg = p.Hq / p.q_groups;
  const int g = h / hpg;
  return (((int64_t)g * p.q_len + row) * hpg + (h - g * hpg)) * p.d;
}

__device__ __forceinline__ bool status_bad(const WsHeader* hdr) {
  return *((volatile const int32_t*)&hdr->status) != 0;
}

// Programmatic dependent launch.  A kernel launched with launch_dependent may
// start while the kernel before it in the stream is still running, as soon as
// every CTA of that kernel has executed grid_dep_trigger() (or exited); it
// must execute grid_dep_wait() before it reads anything that kernel (or one
// before it) wrote: the wait returns once that kernel has completed and its
// writes are visible.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace nsp
#endif
