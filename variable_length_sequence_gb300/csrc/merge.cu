// Log-sum-exp merge of ring-attention partials (HSAP, Sec. 2.2.1: the
// key/value blocks circulate and each rank accumulates its queries' partial
// results online; HSAP's Limitations call this step the "rescale").
//
// For each (token t, head h), given n partials (out_i, lse_i) over disjoint
// key sets:  m = max_i lse_i;  if m = -inf the row saw no key: out = 0 and
// lse = -inf;  else lse = m + ln sum_i exp(lse_i - m) and
// out = sum_i exp(lse_i - lse) out_i.
//
// HBM-bound: every partial row is read once (float4 per lane), the merged
// row written once.  A warp walks 32 consecutive tokens of one head so the
// lse reads ([H, T] layout) are warp-coalesced and reused from L1; it loads
// 4 row groups of every partial before combining them, so each lane keeps
// several independent loads in flight.
//
// One launch can merge several independent segments (e.g. every query shard
// of a ring on one GPU): the work items of all segments share one grid, so
// the launch ramps up and drains once.
#include "nsp_internal.cuh"

namespace nsp {
namespace {

constexpr int kMaxPartials = 64;
constexpr int kMaxSegments = 16;
constexpr int kMergeThreads = 256;

struct MergePtrs {
  const float* out[kMaxPartials];       // partials, segment after segment
  const float* lse[kMaxPartials];
  void* dst[kMaxSegments];              // merged out of each segment
  float* dst_lse[kMaxSegments];         // merged lse of each segment (may be null)
  int first[kMaxSegments];              // first partial of each segment
  int count[kMaxSegments];              // partials of each segment
  int nseg;
};

__device__ __forceinline__ float4 ld_stream4(const float* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p));
  return r;
}

template <typename TO>
__device__ __forceinline__ void st4(TO* p, float4 v);
template <>
__device__ __forceinline__ void st4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void st4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

template <typename TO>
__global__ void __launch_bounds__(kMergeThreads, 4) lse_merge_kernel(const __grid_constant__
                                                                     MergePtrs segs,
                                                                     int64_t T, int H, int d) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kMergeThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kMergeThreads) >> 5;
  const int64_t tgroups = (T + 31) / 32;
  const int64_t per_seg = tgroups * H;
  const int d4 = d / 4;
  for (int64_t wj = warp; wj < per_seg * segs.nseg; wj += nwarps) {
    const int sg = (int)(wj / per_seg);
    const int64_t wi = wj - sg * per_seg;
    const int h = (int)(wi / tgroups);
    const int64_t t0 = (wi % tgroups) * 32;
    const int n = segs.count[sg];
    const float* const* p_out = segs.out + segs.first[sg];
    const float* const* p_lse = segs.lse + segs.first[sg];
    TO* __restrict__ out = reinterpret_cast<TO*>(segs.dst[sg]);
    float* __restrict__ lse_out = segs.dst_lse[sg];
    // lane l: merged lse of token t0 + l
    const int64_t tl = t0 + lane;
    float m = -INFINITY;
    if (tl < T)
      for (int i = 0; i < n; ++i) m = fmaxf(m, __ldg(p_lse[i] + (int64_t)h * T + tl));
    float L = -INFINITY;
    if (m != -INFINITY) {
      float s = 0.f;
      for (int i = 0; i < n; ++i) s += expf(__ldg(p_lse[i] + (int64_t)h * T + tl) - m);
      L = m + logf(s);
    }
    if (tl < T && lse_out != nullptr) lse_out[(int64_t)h * T + tl] = L;
    const int rows = (int)min((int64_t)32, T - t0);
    if (32 % d4 == 0) {
      // 32 / d4 rows per warp load; RB of those loads per partial in flight
      constexpr int RB = 4;
      const int rpi = 32 / d4;
      const int sub = lane / d4, c = lane % d4;
      for (int r0 = 0; r0 < rows; r0 += RB * rpi) {
        float4 acc[RB];
        float Lr[RB];
        int64_t off[RB];
        int rr[RB];
#pragma unroll
        for (int k = 0; k < RB; ++k) {
          rr[k] = r0 + k * rpi + sub;
          Lr[k] = __shfl_sync(0xffffffffu, L, rr[k] & 31);
          if (rr[k] >= rows) Lr[k] = -INFINITY;
          off[k] = ((t0 + rr[k]) * H + h) * (int64_t)d + 4 * c;
          acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 1
        for (int i = 0; i < n; ++i) {
          const float* lsei = p_lse[i] + (int64_t)h * T + t0;
          const float* oi = p_out[i];
          float4 o[RB];
          float li[RB];
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            li[k] = -INFINITY;
            o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (Lr[k] != -INFINITY) {
              li[k] = __ldg(lsei + rr[k]);
              o[k] = ld_stream4(oi + off[k]);
            }
          }
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            const float w = Lr[k] != -INFINITY ? expf(li[k] - Lr[k]) : 0.f;
            acc[k].x = fmaf(w, o[k].x, acc[k].x);
            acc[k].y = fmaf(w, o[k].y, acc[k].y);
            acc[k].z = fmaf(w, o[k].z, acc[k].z);
            acc[k].w = fmaf(w, o[k].w, acc[k].w);
          }
        }
#pragma unroll
        for (int k = 0; k < RB; ++k)
          if (rr[k] < rows) st4<TO>(out + off[k], acc[k]);
      }
      continue;
    }
    for (int r = 0; r < rows; ++r) {
      const float Lr = __shfl_sync(0xffffffffu, L, r);
      const int64_t t = t0 + r;
      const int64_t off = (t * H + h) * (int64_t)d;
      for (int c = lane; c < d4; c += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Lr != -INFINITY) {
          for (int i = 0; i < n; ++i) {
            const float li = __ldg(p_lse[i] + (int64_t)h * T + t);
            const float w = expf(li - Lr);
            const float4 o = ld_stream4(p_out[i] + off + 4 * c);
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
          }
        }
        st4<TO>(out + off + 4 * c, acc);
      }
    }
  }
}

}  // namespace

cudaError_t launch_lse_merge_segments(int nseg, const int* counts, const float* const* outs,
                                      const float* const* lses, int64_t T, int H, int d,
                                      void* const* dst, int out_dtype, float* const* dst_lse,
                                      cudaStream_t s) {
  MergePtrs segs = {};
  int total = 0;
  for (int g = 0; g < nseg; ++g) {
    segs.first[g] = total;
    segs.count[g] = counts[g];
    segs.dst[g] = dst[g];
    segs.dst_lse[g] = dst_lse ? dst_lse[g] : nullptr;
    for (int i = 0; i < counts[g]; ++i) {
      segs.out[total + i] = outs[total + i];
      segs.lse[total + i] = lses[total + i];
    }
    total += counts[g];
  }
  segs.nseg = nseg;
  const int64_t work = ((T + 31) / 32) * H * nseg;
  int64_t blocks = ceil_div(work, (int64_t)(kMergeThreads / 32));
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (out_dtype == NSP_BF16)
    lse_merge_kernel<__nv_bfloat16><<<(unsigned)blocks, kMergeThreads, 0, s>>>(segs, T, H, d);
  else
    lse_merge_kernel<float><<<(unsigned)blocks, kMergeThreads, 0, s>>>(segs, T, H, d);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const float* const* outs, const float* const* lses, int n,
                             int64_t T, int H, int d, void* out, int out_dtype, float* lse,
                             cudaStream_t s) {
  void* dst[1] = {out};
  float* dl[1] = {lse};
  return launch_lse_merge_segments(1, &n, outs, lses, T, H, d, dst, out_dtype, dl, s);
}

}  // namespace nsp
