// Forward attention without a caller-provided workspace.
//
// nsp_attn_fwd needs a small device workspace (status word, tile ranges and
// tile order of the scheduler).  Some callers cannot allocate device memory
// at the point where they run attention: code inside a custom allocator or
// memory-pool callback, plugins of a host framework that owns all device
// allocations, or a process that must keep its footprint fixed after
// start-up.  nsp_attn_fwd_noalloc serves them: it runs the same kernels with
// that scratch in a statically sized __device__ array of this library, so it
// calls no cudaMalloc, cudaFree or allocating routine.
//
// The array is 1 MiB, allocated on every GPU that loads the library, for the
// life of the process.  It holds the scheduler state of the call (header,
// per-tile KV ranges, tile order, histogram); the schedule kernel rewrites
// every byte a call uses (status, counters and histogram included) before
// the attention kernel reads it, so nothing carries over between calls.
// Because all calls share the array, calls whose kernels overlap on the GPU
// (different streams, or different host threads) race; serialise them.
#include <mutex>

#include "nsp_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

}  // namespace

// File-scope scratch, one copy per device.  In host code this name is only a
// host-side stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char nsp_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
int32_t scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NSP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NSP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, nsp_noalloc_scratch) != cudaSuccess || p == nullptr)
      return NSP_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return NSP_OK;
}

}  // namespace

using namespace nsp;

extern "C" int32_t nsp_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                        const int32_t* cu_seqlens, int32_t ndoc, int64_t q_start,
                                        int64_t q_len, int64_t kv_start, int64_t kv_len,
                                        int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                        int32_t causal, int32_t io_dtype, void* out,
                                        int32_t out_dtype, float* lse, int32_t* device_status,
                                        nsp_stream_t stream) {
  // The host checks of nsp_attn_fwd, with a placeholder standing for the
  // static scratch and its size as the workspace size: they bound the sizes
  // first and return NSP_ERR_WORKSPACE when the call's scheduler state would
  // not fit, so every error code matches nsp_attn_fwd's.
  int32_t st = nsp_attn_fwd_validate(q, k, v, cu_seqlens, ndoc, q_start, q_len, kv_start, kv_len,
                                     Hq, Hkv, d, causal, io_dtype, out, out_dtype,
                                     reinterpret_cast<const void*>(uintptr_t(256)),
                                     kNoAllocScratchBytes);
  if (st != NSP_OK) return st;
  if (!scale_ok(scale)) return NSP_ERR_INVALID;
  if ((lse && (reinterpret_cast<uintptr_t>(lse) & 15u)) ||
      (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)))
    return NSP_ERR_ALIGN;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != NSP_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(scratch);
  const FwdWsLayout L = fwd_ws_layout(q_len, kv_len, fwd_tile_rows(io_dtype, d, Hq, Hkv));
  AttnProblem p;
  p.q = q; p.k = k; p.v = v; p.cu = cu_seqlens; p.ndoc = ndoc;
  p.q_start = q_start; p.q_len = q_len; p.kv_start = kv_start; p.kv_len = kv_len;
  p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.scale = scale; p.causal = causal;
  p.io_dtype = io_dtype; p.out_dtype = out_dtype; p.out = out; p.lse = lse;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  if (launch_fwd_schedule(p, L, ws, s) != cudaSuccess) return NSP_ERR_CUDA;
  if (q_len > 0) {
    bool launched = false;
    if (launch_attn_fwd_tc(p, L, ws, s, &launched) != cudaSuccess) return NSP_ERR_CUDA;
    if (!launched && launch_attn_fwd_simt(p, s) != cudaSuccess) return NSP_ERR_CUDA;
  }
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess)
    return NSP_ERR_CUDA;
  return NSP_OK;
}
