// C ABI entry points: host-side validation, workspace carving and dispatch.
// Nothing here allocates memory or synchronises (except nsp_status_query).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "nsp_internal.cuh"

namespace nsp {

std::atomic<long long> g_kernel_launches{0};

void count_launches(int n) { g_kernel_launches.fetch_add(n, std::memory_order_relaxed); }

std::atomic<long long> g_path_launches[2] = {{0}, {0}};

void count_path(bool tensor_core) {
  g_path_launches[tensor_core ? 1 : 0].fetch_add(1, std::memory_order_relaxed);
}

constexpr long long kDefaultWaitBudget = 4000000000LL;     // about 2 s at 2 GHz
std::atomic<long long> g_wait_budget{kDefaultWaitBudget};

int64_t wait_budget_cycles() { return g_wait_budget.load(std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

// CTAs of the persistent attention kernels: one per SM, or the positive
// integer in the environment variable NSP_PERSISTENT_CTAS (read at every
// launch, capped at the SM count).  Each work item is computed whole by one
// CTA, so results do not depend on the grid (tests run several grids and
// compare bits to expose scheduling races), with one exception: the
// ring-block backward (nsp_attn_bwd_accumulate) splits its dK/dV items over
// query-head subsets when the block has few key tiles for the grid, and the
// subsets add into the float32 accumulators with atomics, so its dk/dv may
// differ in the last bits between grids.
int persistent_grid() {
  const int n = num_sms();
  const char* e = std::getenv("NSP_PERSISTENT_CTAS");
  if (e != nullptr && *e != 0) {
    char* end = nullptr;
    const long v = std::strtol(e, &end, 10);
    if (end != nullptr && *end == 0 && v > 0) return (int)std::min<long>(v, n);
  }
  return n;
}

}  // namespace nsp

using namespace nsp;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// bf16 outputs of the attention kernels are written as 32-byte vectors (a
// whole sector per lane), so their base must be 32-byte aligned
inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
inline bool dtype_ok(int32_t t) { return t == NSP_F32 || t == NSP_BF16; }

constexpr int64_t kMaxTokens = (int64_t)1 << 30;   // keeps tile counts in int32

int32_t check_common(int32_t ndoc, int32_t Hq, int32_t Hkv, int32_t d, int32_t causal,
                     int32_t io_dtype) {
  if (ndoc < 1) return NSP_ERR_INVALID;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return NSP_ERR_INVALID;
  if (causal != 0 && causal != 1) return NSP_ERR_INVALID;
  if (!dtype_ok(io_dtype)) return NSP_ERR_INVALID;
  if (d != 64 && d != 128) return NSP_ERR_UNSUPPORTED;
  return NSP_OK;
}

}  // namespace

extern "C" {

const char* nsp_status_str(int32_t status) {
  switch (status) {
    case NSP_OK: return "NSP_OK";
    case NSP_ERR_INVALID: return "NSP_ERR_INVALID: invalid argument or cu_seqlens contents";
    case NSP_ERR_UNSUPPORTED: return "NSP_ERR_UNSUPPORTED: valid but unsupported shape or type";
    case NSP_ERR_WORKSPACE: return "NSP_ERR_WORKSPACE: workspace missing or too small";
    case NSP_ERR_CUDA: return "NSP_ERR_CUDA: a CUDA call or kernel launch failed";
    case NSP_ERR_TIMEOUT: return "NSP_ERR_TIMEOUT: a bounded device-side wait expired";
    case NSP_ERR_ALIGN: return "NSP_ERR_ALIGN: a pointer is not 16-byte aligned";
    default: return "NSP_ERR_UNKNOWN";
  }
}

const char* nsp_version(void) { return "nsp 0.1 sm_103a"; }

int64_t nsp_kernel_launches(void) { return (int64_t)g_kernel_launches.load(); }

int64_t nsp_path_launches(int32_t tensor_core) {
  return (int64_t)g_path_launches[tensor_core ? 1 : 0].load();
}

int64_t nsp_set_wait_timeout_cycles(int64_t cycles) {
  const long long v = cycles < 0 ? kDefaultWaitBudget : (long long)cycles;
  return (int64_t)g_wait_budget.exchange(v);
}

size_t nsp_attn_fwd_workspace_size(int64_t q_len, int64_t kv_len, int32_t Hq, int32_t Hkv,
                                   int32_t d) {
  (void)Hq; (void)Hkv; (void)d;
  if (q_len < 0 || kv_len < 0) return 0;
  return fwd_ws_layout(q_len, kv_len).total;
}

int32_t nsp_attn_fwd_validate(const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens, int32_t ndoc, int64_t q_start,
                              int64_t q_len, int64_t kv_start, int64_t kv_len, int32_t Hq,
                              int32_t Hkv, int32_t d, int32_t causal, int32_t io_dtype,
                              const void* out, int32_t out_dtype, const void* workspace,
                              size_t workspace_bytes) {
  int32_t st = check_common(ndoc, Hq, Hkv, d, causal, io_dtype);
  if (st != NSP_OK) return st;
  if (q_start < 0 || q_len < 0 || kv_start < 0 || kv_len < 0) return NSP_ERR_INVALID;
  if (q_start + q_len > kMaxTokens || kv_start + kv_len > kMaxTokens) return NSP_ERR_UNSUPPORTED;
  if (out_dtype != NSP_F32 && out_dtype != io_dtype) return NSP_ERR_INVALID;
  // Buffers of zero elements may be NULL (empty tensors have no storage).
  if (!cu_seqlens || (q_len > 0 && (!q || !out)) || (kv_len > 0 && (!k || !v)))
    return NSP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(cu_seqlens))
    return NSP_ERR_ALIGN;
  if (out_dtype == NSP_BF16 && !aligned32(out)) return NSP_ERR_ALIGN;
  if (!workspace || workspace_bytes < fwd_ws_layout(q_len, kv_len).total)
    return NSP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NSP_ERR_ALIGN;
  return NSP_OK;
}

int32_t nsp_attn_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                     int32_t ndoc, int64_t q_start, int64_t q_len, int64_t kv_start,
                     int64_t kv_len, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                     int32_t causal, int32_t io_dtype, void* out, int32_t out_dtype,
                     float* lse, void* workspace, size_t workspace_bytes,
                     nsp_stream_t stream) {
  int32_t st = nsp_attn_fwd_validate(q, k, v, cu_seqlens, ndoc, q_start, q_len, kv_start,
                                     kv_len, Hq, Hkv, d, causal, io_dtype, out, out_dtype,
                                     workspace, workspace_bytes);
  if (st != NSP_OK) return st;
  if (!scale_ok(scale)) return NSP_ERR_INVALID;
  if (lse && !aligned16(lse)) return NSP_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  const FwdWsLayout L = fwd_ws_layout(q_len, kv_len, fwd_tile_rows(io_dtype, d, Hq, Hkv));
  AttnProblem p;
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = q_start; p.q_len = q_len; p.kv_start = kv_start; p.kv_len = kv_len;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = out_dtype; p.out = out; p.lse = lse;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  if (launch_fwd_schedule(p, L, ws, s) != cudaSuccess) return NSP_ERR_CUDA;
  if (q_len == 0) return NSP_OK;
  bool launched = false;
  if (launch_attn_fwd_tc(p, L, ws, s, &launched) != cudaSuccess) return NSP_ERR_CUDA;
  if (!launched && launch_attn_fwd_simt(p, s) != cudaSuccess) return NSP_ERR_CUDA;
  return NSP_OK;
}

int32_t nsp_attn_fwd_headgroups(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens, int32_t ndoc, int64_t T, int32_t Hq,
                                int32_t Hkv, int32_t d, int32_t P, float scale, int32_t causal,
                                int32_t io_dtype, void* out, int32_t out_dtype, float* lse,
                                void* workspace, size_t workspace_bytes, nsp_stream_t stream) {
  int32_t st = nsp_attn_fwd_validate(q, k, v, cu_seqlens, ndoc, 0, T, 0, T, Hq, Hkv, d, causal,
                                     io_dtype, out, out_dtype, workspace, workspace_bytes);
  if (st != NSP_OK) return st;
  if (P < 1 || Hq % P != 0) return NSP_ERR_INVALID;
  if ((int64_t)P * T > (int64_t)INT32_MAX) return NSP_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return NSP_ERR_INVALID;
  if (lse && !aligned16(lse)) return NSP_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  const FwdWsLayout L = fwd_ws_layout(T, T, fwd_tile_rows(io_dtype, d, Hq, Hkv));
  AttnProblem p;
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = 0; p.q_len = T; p.kv_start = 0; p.kv_len = T;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = out_dtype; p.out = out; p.lse = lse;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.q_groups = P;
  if (launch_fwd_schedule(p, L, ws, s) != cudaSuccess) return NSP_ERR_CUDA;
  if (T == 0) return NSP_OK;
  bool launched = false;
  if (launch_attn_fwd_tc(p, L, ws, s, &launched) != cudaSuccess) return NSP_ERR_CUDA;
  if (!launched && launch_attn_fwd_simt(p, s) != cudaSuccess) return NSP_ERR_CUDA;
  return NSP_OK;
}

int32_t nsp_attn_fwd_accumulate(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens, int32_t ndoc, int64_t q_start,
                                int64_t q_len, int64_t kv_start, int64_t kv_len, int32_t Hq,
                                int32_t Hkv, int32_t d, float scale, int32_t causal,
                                int32_t io_dtype, float* acc, float* lse_acc, void* workspace,
                                size_t workspace_bytes, nsp_stream_t stream) {
  int32_t st = nsp_attn_fwd_validate(q, k, v, cu_seqlens, ndoc, q_start, q_len, kv_start,
                                     kv_len, Hq, Hkv, d, causal, io_dtype, acc, NSP_F32,
                                     workspace, workspace_bytes);
  if (st != NSP_OK) return st;
  if (!scale_ok(scale)) return NSP_ERR_INVALID;
  if (q_len > 0 && !lse_acc) return NSP_ERR_INVALID;
  if (!aligned16(lse_acc)) return NSP_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  const FwdWsLayout L = fwd_ws_layout(q_len, kv_len, fwd_tile_rows(io_dtype, d, Hq, Hkv));
  AttnProblem p;
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = q_start; p.q_len = q_len; p.kv_start = kv_start; p.kv_len = kv_len;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = NSP_F32; p.out = acc; p.lse = lse_acc;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.accumulate = 1;
  if (launch_fwd_schedule(p, L, ws, s) != cudaSuccess) return NSP_ERR_CUDA;
  if (q_len == 0) return NSP_OK;
  bool launched = false;
  if (launch_attn_fwd_tc(p, L, ws, s, &launched) != cudaSuccess) return NSP_ERR_CUDA;
  if (!launched && launch_attn_fwd_simt(p, s) != cudaSuccess) return NSP_ERR_CUDA;
  return NSP_OK;
}

namespace {

// Host checks of a batched forward's block table: sizes, ranges inside
// [0, T), aligned outputs, and no two blocks writing the same bytes.
int32_t check_blocks(int64_t T, int32_t nblocks, const nsp_block_t* blocks, int32_t Hq,
                     int32_t d, int32_t accumulate) {
  if (nblocks < 1 || nblocks > kMaxBlocks || !blocks) return NSP_ERR_INVALID;
  for (int32_t i = 0; i < nblocks; ++i) {
    const nsp_block_t& b = blocks[i];
    if (b.q_start < 0 || b.q_len < 0 || b.kv_start < 0 || b.kv_len < 0) return NSP_ERR_INVALID;
    if (b.q_start + b.q_len > T || b.kv_start + b.kv_len > T) return NSP_ERR_INVALID;
    if (b.q_len > 0 && (!b.out || (accumulate && !b.lse))) return NSP_ERR_INVALID;
    if (!aligned16(b.out) || !aligned16(b.lse)) return NSP_ERR_ALIGN;
  }
  auto overlap = [](const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
  };
  for (int32_t i = 0; i < nblocks; ++i)
    for (int32_t j = i + 1; j < nblocks; ++j) {
      const nsp_block_t &a = blocks[i], &b = blocks[j];
      const size_t oa = (size_t)a.q_len * Hq * d * 4, ob = (size_t)b.q_len * Hq * d * 4;
      const size_t la = a.lse ? (size_t)a.q_len * Hq * 4 : 0, lb = b.lse ? (size_t)b.q_len * Hq * 4 : 0;
      if (overlap(a.out, oa, b.out, ob) || overlap(a.lse, la, b.lse, lb) ||
          overlap(a.out, oa, b.lse, lb) || overlap(a.lse, la, b.out, ob))
        return NSP_ERR_INVALID;
    }
  return NSP_OK;
}

FwdBlocks table_of(int32_t nblocks, const nsp_block_t* blocks) {
  FwdBlocks B;
  B.n = nblocks;
  B.global_rows = 1;
  for (int32_t i = 0; i < nblocks; ++i) {
    B.b[i].q_start = (int32_t)blocks[i].q_start; B.b[i].q_len = (int32_t)blocks[i].q_len;
    B.b[i].kv_start = (int32_t)blocks[i].kv_start; B.b[i].kv_len = (int32_t)blocks[i].kv_len;
    B.b[i].tile0 = 0; B.b[i].ktile0 = 0;
    B.b[i].out = blocks[i].out; B.b[i].lse = blocks[i].lse;
  }
  return B;
}

}  // namespace

size_t nsp_attn_fwd_blocks_workspace_size(int32_t nblocks, const nsp_block_t* blocks, int32_t Hq,
                                          int32_t Hkv, int32_t d) {
  (void)Hq; (void)Hkv; (void)d;
  if (nblocks < 1 || nblocks > kMaxBlocks || !blocks) return 0;
  for (int32_t i = 0; i < nblocks; ++i)
    if (blocks[i].q_len < 0 || blocks[i].kv_len < 0 || blocks[i].q_len > kMaxTokens ||
        blocks[i].kv_len > kMaxTokens)
      return 0;
  FwdBlocks B = table_of(nblocks, blocks);
  return fwd_ws_layout_blocks(B, kTileM).total;
}

int32_t nsp_attn_fwd_blocks(const void* q, const void* k, const void* v,
                            const int32_t* cu_seqlens, int32_t ndoc, int64_t T, int32_t nblocks,
                            const nsp_block_t* blocks, int32_t Hq, int32_t Hkv, int32_t d,
                            float scale, int32_t causal, int32_t io_dtype, int32_t accumulate,
                            void* workspace, size_t workspace_bytes, nsp_stream_t stream) {
  int32_t st = check_common(ndoc, Hq, Hkv, d, causal, io_dtype);
  if (st != NSP_OK) return st;
  if (T < 0 || (accumulate != 0 && accumulate != 1)) return NSP_ERR_INVALID;
  if (T > kMaxTokens) return NSP_ERR_UNSUPPORTED;
  if (!scale_ok(scale) || !cu_seqlens) return NSP_ERR_INVALID;
  if (T > 0 && (!q || !k || !v)) return NSP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(cu_seqlens)) return NSP_ERR_ALIGN;
  st = check_blocks(T, nblocks, blocks, Hq, d, accumulate);
  if (st != NSP_OK) return st;
  if (!workspace ||
      workspace_bytes < nsp_attn_fwd_blocks_workspace_size(nblocks, blocks, Hq, Hkv, d))
    return NSP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NSP_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  FwdBlocks B = table_of(nblocks, blocks);
  const FwdWsLayout L = fwd_ws_layout_blocks(B, fwd_tile_rows(io_dtype, d, Hq, Hkv));
  AttnProblem p;                       // whole-stream q / k / v; ranges and outputs per block
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = 0; p.q_len = T; p.kv_start = 0; p.kv_len = T;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = NSP_F32; p.out = nullptr; p.lse = nullptr;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.accumulate = accumulate;
  if (launch_fwd_schedule(p, L, ws, s, &B) != cudaSuccess) return NSP_ERR_CUDA;
  if (T == 0) return NSP_OK;
  bool launched = false;
  if (launch_attn_fwd_tc(p, L, ws, s, &launched, &B) != cudaSuccess) return NSP_ERR_CUDA;
  if (launched) return NSP_OK;
  // CUDA-core path (float32 I/O): one launch per block, on pointers
  // to the block's own rows
  const size_t es = io_dtype == NSP_BF16 ? 2 : 4;
  for (int32_t i = 0; i < nblocks; ++i) {
    const nsp_block_t& b = blocks[i];
    if (b.q_len == 0) continue;
    AttnProblem pb = p;
    pb.q = reinterpret_cast<const char*>(q) + (size_t)b.q_start * Hq * d * es;
    pb.k = reinterpret_cast<const char*>(k) + (size_t)b.kv_start * Hkv * d * es;
    pb.v = reinterpret_cast<const char*>(v) + (size_t)b.kv_start * Hkv * d * es;
    pb.q_start = b.q_start; pb.q_len = b.q_len; pb.kv_start = b.kv_start; pb.kv_len = b.kv_len;
    pb.out = b.out; pb.lse = b.lse;
    if (launch_attn_fwd_simt(pb, s) != cudaSuccess) return NSP_ERR_CUDA;
  }
  return NSP_OK;
}

namespace {

FwdBlocks range_table(int32_t nranges, const nsp_range_t* ranges) {
  FwdBlocks B;
  B.n = nranges;
  B.global_rows = 1;
  for (int32_t i = 0; i < nranges; ++i) {
    B.b[i].q_start = (int32_t)ranges[i].q_start; B.b[i].q_len = (int32_t)ranges[i].q_len;
    B.b[i].kv_start = (int32_t)ranges[i].kv_start; B.b[i].kv_len = (int32_t)ranges[i].kv_len;
    B.b[i].tile0 = 0; B.b[i].ktile0 = 0;
    B.b[i].out = nullptr; B.b[i].lse = nullptr;
  }
  return B;
}

bool ranges_ok(int64_t T, int32_t nranges, const nsp_range_t* ranges) {
  if (nranges < 1 || nranges > kMaxBlocks || !ranges) return false;
  for (int32_t i = 0; i < nranges; ++i) {
    const nsp_range_t& r = ranges[i];
    if (r.q_start < 0 || r.q_len < 0 || r.kv_start < 0 || r.kv_len < 0) return false;
    if (r.q_start + r.q_len > T || r.kv_start + r.kv_len > T) return false;
  }
  return true;
}

}  // namespace

// Workspace bytes past the layout, from the next 1024-byte boundary, are the
// whole-stream tensor-core backward's dS cache.
static void attach_ds_cache(BwdWsLayout& L, size_t workspace_bytes) {
  const size_t base = align_up(L.total, 1024);
  if (workspace_bytes >= base + kDsTileBytes) {
    L.ds_cache = base;
    L.ds_cache_bytes = workspace_bytes - base;
  }
}

// Visible (128-row query tile, 128-key tile) pairs of the query rows
// [qs, qs + ql) against the keys [ks, ks + kl), tiles aligned to qs and ks
// (the backward schedule's rule: query tile [r0, r1] sees the key tiles from
// its first row's document start to r1 (causal) or to the end of its last
// row's document, clipped to the key range).  cu validated by the caller.
static int64_t visible_tile_pairs(const int32_t* cu, int32_t ndoc, int64_t qs, int64_t ql,
                                  int64_t ks, int64_t kl, int32_t causal) {
  int64_t pairs = 0;
  int32_t b0 = 0;
  for (int64_t r0 = qs; r0 < qs + ql; r0 += kTileM) {
    const int64_t r1 = (r0 + kTileM < qs + ql ? r0 + kTileM : qs + ql) - 1;
    while (cu[b0 + 1] <= r0) ++b0;
    int32_t b1 = b0;
    while (cu[b1 + 1] <= r1) ++b1;
    int64_t lo = cu[b0], hi = causal ? r1 + 1 : (int64_t)cu[b1 + 1];
    lo = lo > ks ? lo : ks;
    hi = hi < ks + kl ? hi : ks + kl;
    if (hi > lo) pairs += (hi - 1 - ks) / kBwdSub - (lo - ks) / kBwdSub + 1;
  }
  (void)ndoc;
  return pairs;
}

static bool cu_host_ok(const int32_t* cu, int32_t ndoc) {
  if (cu == nullptr || ndoc < 1 || cu[0] != 0) return false;
  for (int32_t b = 0; b < ndoc; ++b)
    if (cu[b] > cu[b + 1]) return false;
  return true;
}

size_t nsp_attn_bwd_ds_cache_size(const int32_t* cu, int32_t ndoc, int32_t Hq, int32_t causal) {
  if (!cu_host_ok(cu, ndoc) || Hq < 1) return 0;
  const int64_t T = cu[ndoc];
  return (size_t)visible_tile_pairs(cu, ndoc, 0, T, 0, T, causal) * (size_t)Hq * kDsTileBytes;
}

size_t nsp_attn_bwd_blocks_ds_cache_size(const int32_t* cu, int32_t ndoc, int32_t nranges,
                                         const nsp_range_t* ranges, int32_t Hq, int32_t causal) {
  if (!cu_host_ok(cu, ndoc) || Hq < 1) return 0;
  const int64_t T = cu[ndoc];
  if (!ranges_ok(T, nranges, ranges)) return 0;
  int64_t pairs = 0;
  for (int32_t i = 0; i < nranges; ++i)
    pairs += visible_tile_pairs(cu, ndoc, ranges[i].q_start, ranges[i].q_len, ranges[i].kv_start,
                                ranges[i].kv_len, causal);
  return (size_t)pairs * (size_t)Hq * kDsTileBytes;
}

int32_t nsp_bwd_ds_cache_used(const void* workspace, int32_t* used, nsp_stream_t stream) {
  if (!workspace || !used) return NSP_ERR_INVALID;
  const WsHeader* hdr = reinterpret_cast<const WsHeader*>(workspace);
  int32_t v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, &hdr->ds_on, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return NSP_ERR_CUDA;
  *used = v;
  return NSP_OK;
}

size_t nsp_attn_bwd_blocks_workspace_size(int64_t T, int32_t nranges, const nsp_range_t* ranges,
                                          int32_t Hq, int32_t Hkv, int32_t d) {
  (void)Hkv; (void)d;
  if (T < 0 || T > kMaxTokens || Hq < 1 || !ranges_ok(T, nranges, ranges)) return 0;
  FwdBlocks B = range_table(nranges, ranges);
  return bwd_ws_layout_blocks(B, T, Hq).total;
}

int32_t nsp_attn_bwd_blocks(const void* q, const void* k, const void* v, const void* out,
                            const void* dout, const float* lse, const int32_t* cu_seqlens,
                            int32_t ndoc, int64_t T, int32_t nranges, const nsp_range_t* ranges,
                            int32_t Hq, int32_t Hkv, int32_t d, float scale, int32_t causal,
                            int32_t io_dtype, float* dq_acc, float* dk_acc, float* dv_acc,
                            void* workspace, size_t workspace_bytes, nsp_stream_t stream) {
  int32_t st = check_common(ndoc, Hq, Hkv, d, causal, io_dtype);
  if (st != NSP_OK) return st;
  if (T < 0) return NSP_ERR_INVALID;
  if (T > kMaxTokens) return NSP_ERR_UNSUPPORTED;
  if (!scale_ok(scale) || !cu_seqlens) return NSP_ERR_INVALID;
  if (!ranges_ok(T, nranges, ranges)) return NSP_ERR_INVALID;
  if (!bwd_tc_eligible(io_dtype, d, Hq, Hkv)) return NSP_ERR_UNSUPPORTED;
  for (int32_t i = 0; i < nranges; ++i)     // whole-stream lse / delta rows are bulk-copied
    if (ranges[i].q_start % 4 != 0) return NSP_ERR_UNSUPPORTED;
  if (T > 0 && (!q || !k || !v || !out || !dout || !lse || !dq_acc || !dk_acc || !dv_acc))
    return NSP_ERR_INVALID;
  const void* ptrs[] = {q, k, v, out, dout, lse, cu_seqlens, dq_acc, dk_acc, dv_acc};
  for (const void* x : ptrs)
    if (!aligned16(x)) return NSP_ERR_ALIGN;
  FwdBlocks B = range_table(nranges, ranges);
  BwdWsLayout L = bwd_ws_layout_blocks(B, T, Hq);
  if (!workspace || workspace_bytes < L.total) return NSP_ERR_WORKSPACE;
  attach_ds_cache(L, workspace_bytes);
  if (!aligned16(workspace)) return NSP_ERR_ALIGN;
  if (T == 0) return NSP_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  AttnProblem p;                       // whole stream; ranges per block
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = 0; p.q_len = T; p.kv_start = 0; p.kv_len = T;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = NSP_F32; p.out = nullptr; p.lse = nullptr;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.accumulate = 1;
  if (launch_bwd_schedules(p, L, ws, s, &B) != cudaSuccess) return NSP_ERR_CUDA;
  return launch_attn_bwd_tc(p, out, dout, lse, dq_acc, dk_acc, dv_acc, L, ws, s, &B) ==
                 cudaSuccess
             ? NSP_OK
             : NSP_ERR_CUDA;
}

size_t nsp_attn_bwd_workspace_size(int64_t T, int32_t Hq, int32_t Hkv, int32_t d,
                                   int32_t io_dtype) {
  if (T < 0 || Hq < 1 || Hkv < 1 || d < 1) return 0;
  return bwd_ws_layout(T, T, Hq, d, !bwd_tc_eligible(io_dtype, d, Hq, Hkv)).total;
}

int32_t nsp_attn_bwd_validate(const void* q, const void* k, const void* v, const void* out,
                              const void* dout, const float* lse, const int32_t* cu_seqlens,
                              int32_t ndoc, int64_t T, int32_t Hq, int32_t Hkv, int32_t d,
                              int32_t causal, int32_t io_dtype, const void* dq,
                              const void* dk, const void* dv, const void* workspace,
                              size_t workspace_bytes) {
  int32_t st = check_common(ndoc, Hq, Hkv, d, causal, io_dtype);
  if (st != NSP_OK) return st;
  if (T < 0) return NSP_ERR_INVALID;
  if (T > kMaxTokens) return NSP_ERR_UNSUPPORTED;
  if (!cu_seqlens) return NSP_ERR_INVALID;
  if (T > 0 && (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv))
    return NSP_ERR_INVALID;
  const void* ptrs[] = {q, k, v, out, dout, lse, cu_seqlens, dq, dk, dv};
  for (const void* x : ptrs)
    if (!aligned16(x)) return NSP_ERR_ALIGN;
  if (io_dtype == NSP_BF16 && (!aligned32(dq) || !aligned32(dk) || !aligned32(dv)))
    return NSP_ERR_ALIGN;
  if (!workspace ||
      workspace_bytes < bwd_ws_layout(T, T, Hq, d, !bwd_tc_eligible(io_dtype, d, Hq, Hkv)).total)
    return NSP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NSP_ERR_ALIGN;
  return NSP_OK;
}

int32_t nsp_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, const int32_t* cu_seqlens,
                     int32_t ndoc, int64_t T, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                     int32_t causal, int32_t io_dtype, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, nsp_stream_t stream) {
  int32_t st = nsp_attn_bwd_validate(q, k, v, out, dout, lse, cu_seqlens, ndoc, T, Hq, Hkv, d,
                                     causal, io_dtype, dq, dk, dv, workspace, workspace_bytes);
  if (st != NSP_OK) return st;
  if (!scale_ok(scale)) return NSP_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  const bool tc = bwd_tc_eligible(io_dtype, d, Hq, Hkv);
  BwdWsLayout L = bwd_ws_layout(T, T, Hq, d, !tc);
  if (tc) attach_ds_cache(L, workspace_bytes);
  AttnProblem p;
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = 0; p.q_len = T; p.kv_start = 0; p.kv_len = T;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = io_dtype; p.out = nullptr; p.lse = nullptr;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  if (launch_bwd_schedules(p, L, ws, s) != cudaSuccess) return NSP_ERR_CUDA;
  if (T == 0) return NSP_OK;
  const cudaError_t e = tc ? launch_attn_bwd_tc(p, out, dout, lse, dq, dk, dv, L, ws, s)
                           : launch_attn_bwd_simt(p, out, dout, lse, dq, dk, dv, L, ws, s);
  return e == cudaSuccess ? NSP_OK : NSP_ERR_CUDA;
}

int32_t nsp_attn_bwd_headgroups(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse,
                                const int32_t* cu_seqlens, int32_t ndoc, int64_t T, int32_t Hq,
                                int32_t Hkv, int32_t d, int32_t P, float scale, int32_t causal,
                                int32_t io_dtype, void* dq, void* dk, void* dv, void* workspace,
                                size_t workspace_bytes, nsp_stream_t stream) {
  int32_t st = nsp_attn_bwd_validate(q, k, v, out, dout, lse, cu_seqlens, ndoc, T, Hq, Hkv, d,
                                     causal, io_dtype, dq, dk, dv, workspace, workspace_bytes);
  if (st != NSP_OK) return st;
  if (P < 1 || Hq % P != 0) return NSP_ERR_INVALID;
  if ((int64_t)P * T > (int64_t)INT32_MAX) return NSP_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return NSP_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  const bool tc = bwd_tc_eligible(io_dtype, d, Hq, Hkv);
  BwdWsLayout L = bwd_ws_layout(T, T, Hq, d, !tc);
  if (tc) attach_ds_cache(L, workspace_bytes);
  AttnProblem p;
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = 0; p.q_len = T; p.kv_start = 0; p.kv_len = T;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = io_dtype; p.out = nullptr; p.lse = nullptr;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.q_groups = P;
  if (launch_bwd_schedules(p, L, ws, s) != cudaSuccess) return NSP_ERR_CUDA;
  if (T == 0) return NSP_OK;
  const cudaError_t e = tc ? launch_attn_bwd_tc(p, out, dout, lse, dq, dk, dv, L, ws, s)
                           : launch_attn_bwd_simt(p, out, dout, lse, dq, dk, dv, L, ws, s);
  return e == cudaSuccess ? NSP_OK : NSP_ERR_CUDA;
}

size_t nsp_attn_bwd_accumulate_workspace_size(int64_t q_len, int64_t kv_len, int32_t Hq,
                                              int32_t Hkv, int32_t d, int32_t io_dtype) {
  (void)Hkv; (void)io_dtype;
  if (q_len < 0 || kv_len < 0 || Hq < 1 || d < 1) return 0;
  return bwd_ws_layout(q_len, kv_len, Hq, d, false).total;
}

int32_t nsp_attn_bwd_accumulate(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse,
                                const int32_t* cu_seqlens, int32_t ndoc, int64_t q_start,
                                int64_t q_len, int64_t kv_start, int64_t kv_len, int32_t Hq,
                                int32_t Hkv, int32_t d, float scale, int32_t causal,
                                int32_t io_dtype, float* dq_acc, float* dk_acc, float* dv_acc,
                                void* workspace, size_t workspace_bytes, nsp_stream_t stream) {
  int32_t st = check_common(ndoc, Hq, Hkv, d, causal, io_dtype);
  if (st != NSP_OK) return st;
  if (q_start < 0 || q_len < 0 || kv_start < 0 || kv_len < 0) return NSP_ERR_INVALID;
  if (q_start + q_len > kMaxTokens || kv_start + kv_len > kMaxTokens) return NSP_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return NSP_ERR_INVALID;
  if (!cu_seqlens) return NSP_ERR_INVALID;
  if (q_len > 0 && (!q || !out || !dout || !lse || !dq_acc)) return NSP_ERR_INVALID;
  if (kv_len > 0 && (!k || !v || !dk_acc || !dv_acc)) return NSP_ERR_INVALID;
  const void* ptrs[] = {q, k, v, out, dout, lse, cu_seqlens, dq_acc, dk_acc, dv_acc};
  for (const void* x : ptrs)
    if (!aligned16(x)) return NSP_ERR_ALIGN;
  const BwdWsLayout L = bwd_ws_layout(q_len, kv_len, Hq, d, false);
  if (!workspace || workspace_bytes < L.total) return NSP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NSP_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  AttnProblem p;
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = q_start; p.q_len = q_len; p.kv_start = kv_start; p.kv_len = kv_len;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = NSP_F32; p.out = nullptr; p.lse = nullptr;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.accumulate = 1;
  if (q_len == 0 || kv_len == 0) return NSP_OK;        // an empty block adds nothing
  if (launch_bwd_schedules(p, L, ws, s) != cudaSuccess) return NSP_ERR_CUDA;
  const cudaError_t e =
      bwd_tc_eligible(io_dtype, d, Hq, Hkv)
          ? launch_attn_bwd_tc(p, out, dout, lse, dq_acc, dk_acc, dv_acc, L, ws, s)
          : launch_attn_bwd_simt(p, out, dout, lse, dq_acc, dk_acc, dv_acc, L, ws, s);
  return e == cudaSuccess ? NSP_OK : NSP_ERR_CUDA;
}

int32_t nsp_lse_merge_validate(const float* const* outs, const float* const* lses, int32_t n,
                               int64_t T, int32_t H, int32_t d, const void* out,
                               int32_t out_dtype, const float* lse) {
  if (n < 1 || n > 64 || T < 0 || H < 1 || d < 4 || d % 4 != 0) return NSP_ERR_INVALID;
  if (!dtype_ok(out_dtype)) return NSP_ERR_INVALID;
  if (!outs || !lses) return NSP_ERR_INVALID;
  if (T == 0) return NSP_OK;
  if (!out) return NSP_ERR_INVALID;
  for (int i = 0; i < n; ++i) {
    if (!outs[i] || !lses[i]) return NSP_ERR_INVALID;
    if (!aligned16(outs[i]) || !aligned16(lses[i])) return NSP_ERR_ALIGN;
  }
  if (!aligned16(out) || (lse && !aligned16(lse))) return NSP_ERR_ALIGN;
  return NSP_OK;
}

int32_t nsp_lse_merge(const float* const* outs, const float* const* lses, int32_t n,
                      int64_t T, int32_t H, int32_t d, void* out, int32_t out_dtype,
                      float* lse, nsp_stream_t stream) {
  int32_t st = nsp_lse_merge_validate(outs, lses, n, T, H, d, out, out_dtype, lse);
  if (st != NSP_OK) return st;
  if (T == 0) return NSP_OK;
  if (launch_lse_merge(outs, lses, n, T, H, d, out, out_dtype, lse,
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NSP_ERR_CUDA;
  return NSP_OK;
}

int32_t nsp_lse_merge_batch(int32_t nseg, const int32_t* counts, const float* const* outs,
                            const float* const* lses, int64_t T, int32_t H, int32_t d,
                            void* const* out, int32_t out_dtype, float* const* lse,
                            nsp_stream_t stream) {
  if (nseg < 1 || nseg > 16 || !counts || !out) return NSP_ERR_INVALID;
  int total = 0;
  for (int g = 0; g < nseg; ++g) {
    if (counts[g] < 1) return NSP_ERR_INVALID;
    total += counts[g];
  }
  if (total > 64) return NSP_ERR_INVALID;
  int first = 0;
  for (int g = 0; g < nseg; ++g) {     // each segment: the checks of nsp_lse_merge
    const int32_t st = nsp_lse_merge_validate(outs ? outs + first : nullptr,
                                              lses ? lses + first : nullptr, counts[g], T, H, d,
                                              out[g], out_dtype, lse ? lse[g] : nullptr);
    if (st != NSP_OK) return st;
    first += counts[g];
  }
  if (T == 0) return NSP_OK;
  if (launch_lse_merge_segments(nseg, counts, outs, lses, T, H, d, out, out_dtype, lse,
                                reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NSP_ERR_CUDA;
  return NSP_OK;
}

int32_t nsp_seq2head_permute_validate(const void* in, const void* out, int64_t T, int32_t H,
                                      int32_t d, int32_t P, int32_t elem_bytes) {
  if (T < 0 || H < 1 || d < 1 || P < 1 || H % P != 0) return NSP_ERR_INVALID;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return NSP_ERR_INVALID;
  if (T == 0) return NSP_OK;
  if (!in || !out) return NSP_ERR_INVALID;
  if (!aligned16(in) || !aligned16(out)) return NSP_ERR_ALIGN;
  const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
  const uintptr_t n = (uintptr_t)T * H * d * elem_bytes;
  if (T > 0 && a < b + n && b < a + n) return NSP_ERR_INVALID;     // overlap
  return NSP_OK;
}

int32_t nsp_seq2head_permute(const void* in, void* out, int64_t T, int32_t H, int32_t d,
                             int32_t P, int32_t elem_bytes, int32_t inverse,
                             nsp_stream_t stream) {
  int32_t st = nsp_seq2head_permute_validate(in, out, T, H, d, P, elem_bytes);
  if (st != NSP_OK) return st;
  if (inverse != 0 && inverse != 1) return NSP_ERR_INVALID;
  if (T == 0) return NSP_OK;
  if (launch_permute(in, out, T, H, d, P, elem_bytes, inverse,
                     reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NSP_ERR_CUDA;
  return NSP_OK;
}

int32_t nsp_seq2head_permute_groups(const void* in, void* out, int32_t B, int64_t L, int32_t H,
                                    int32_t d, int32_t K, int32_t elem_bytes, int32_t inverse,
                                    nsp_stream_t stream) {
  if (B < 1 || L < 0) return NSP_ERR_INVALID;
  if ((int64_t)B * L > ((int64_t)1 << 40)) return NSP_ERR_UNSUPPORTED;
  // the checks of the whole batch as one [B L, H, d] permutation
  int32_t st = nsp_seq2head_permute_validate(in, out, (int64_t)B * L, H, d, K, elem_bytes);
  if (st != NSP_OK) return st;
  if (inverse != 0 && inverse != 1) return NSP_ERR_INVALID;
  if (L == 0) return NSP_OK;
  if (launch_permute_groups(in, out, B, L, H, d, K, elem_bytes, inverse,
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NSP_ERR_CUDA;
  return NSP_OK;
}

int32_t nsp_status_query(const void* workspace, nsp_stream_t stream) {
  if (!workspace) return NSP_ERR_INVALID;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NSP_ERR_CUDA;
  int32_t st = 0;
  if (cudaMemcpy(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return NSP_ERR_CUDA;
  return st;
}

int32_t nsp_attn_pairs(const int32_t* cu_seqlens_host, int32_t ndoc, int32_t causal,
                       double* pairs) {
  if (!cu_seqlens_host || !pairs || ndoc < 1 || cu_seqlens_host[0] != 0) return NSP_ERR_INVALID;
  double acc = 0.0;
  for (int i = 0; i < ndoc; ++i) {
    const int64_t L = (int64_t)cu_seqlens_host[i + 1] - cu_seqlens_host[i];
    if (L < 0) return NSP_ERR_INVALID;
    acc += causal ? 0.5 * (double)L * (double)(L + 1) : (double)L * (double)L;
  }
  *pairs = acc;
  return NSP_OK;
}

int32_t nsp_attn_cost(const int32_t* cu, int32_t ndoc, int64_t q_start, int64_t q_len,
                      int64_t kv_start, int64_t kv_len, int32_t Hq, int32_t Hkv, int32_t d,
                      int32_t causal, int32_t io_dtype, nsp_attn_cost_t* cost) {
  if (!cu || !cost || ndoc < 1 || cu[0] != 0) return NSP_ERR_INVALID;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d < 1 || !dtype_ok(io_dtype)) return NSP_ERR_INVALID;
  if ((causal != 0 && causal != 1) || q_start < 0 || q_len < 0 || kv_start < 0 || kv_len < 0)
    return NSP_ERR_INVALID;
  for (int32_t i = 0; i < ndoc; ++i)
    if (cu[i + 1] < cu[i]) return NSP_ERR_INVALID;
  const int64_t T = cu[ndoc];
  if (q_start + q_len > T || kv_start + kv_len > T) return NSP_ERR_INVALID;
  const int64_t qa = q_start, qb = q_start + q_len, ka = kv_start, kb = kv_start + kv_len;
  // allowed pairs, per document: rows t in [t0, t1) see keys [lo, hi(t))
  double pairs = 0.0;
  for (int32_t b = 0; b < ndoc; ++b) {
    const int64_t s = cu[b], e = cu[b + 1];
    const int64_t t0 = std::max(s, qa), t1 = std::min(e, qb);
    const int64_t lo = std::max(s, ka);
    if (t1 <= t0) continue;
    if (!causal) {
      const int64_t w = std::min(e, kb) - lo;
      if (w > 0) pairs += (double)w * (double)(t1 - t0);
      continue;
    }
    // rows with t + 1 <= kb see t + 1 - lo keys (when positive), the rest kb - lo
    const int64_t a0 = std::max(t0, lo), a1 = std::min(t1, kb);
    if (a1 > a0)      // sum over t in [a0, a1) of (t + 1 - lo)
      pairs += 0.5 * (double)(a1 - a0) * (double)((a0 + 1 - lo) + (a1 - lo));
    const int64_t b0 = std::max(t0, kb);
    if (t1 > b0 && kb > lo) pairs += (double)(t1 - b0) * (double)(kb - lo);
  }
  // scheduled tiles: per 128-row query tile, the contiguous 128-key tiles
  // from its first row's document start to its last row's last visible key
  double tiles = 0.0;
  for (int64_t r0 = qa; r0 < qb; r0 += kTileM) {
    const int64_t r1 = std::min(r0 + kTileM, qb) - 1;
    const int32_t* it0 = std::upper_bound(cu, cu + ndoc + 1, (int32_t)r0);
    const int32_t* it1 = std::upper_bound(cu, cu + ndoc + 1, (int32_t)r1);
    const int64_t b0 = (it0 - cu) - 1, b1 = (it1 - cu) - 1;
    const int64_t lo = std::max((int64_t)cu[b0], ka);
    const int64_t hi = std::min(causal ? r1 + 1 : (int64_t)cu[b1 + 1], kb);
    if (hi > lo) tiles += (double)((hi - 1 - ka) / kTileN - (lo - ka) / kTileN + 1);
  }
  const double e = io_dtype == NSP_BF16 ? 2.0 : 4.0;
  const double qo = (double)q_len * Hq * d * e;        // one [q_len, Hq, d] tensor
  const double kv = (double)kv_len * Hkv * d * e;      // one [kv_len, Hkv, d] tensor
  const double ls = 4.0 * (double)Hq * (double)q_len;  // lse
  cost->pairs = pairs;
  cost->fwd_flop = 4.0 * d * Hq * pairs;
  cost->bwd_flop = 10.0 * d * Hq * pairs;
  cost->tiles = tiles;
  cost->fwd_bytes = 2.0 * qo + 2.0 * kv + ls;                // q, k, v in; out, lse out
  cost->bwd_bytes = 3.0 * qo + 2.0 * kv + ls + qo + 2.0 * kv;  // q, out, dout, k, v, lse; dq, dk, dv
  return NSP_OK;
}

}  // extern "C"
