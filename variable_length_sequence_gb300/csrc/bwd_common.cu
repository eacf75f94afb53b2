// Kernels shared by both backward paths: delta = rowsum(dOut * Out) before
// the main backward kernel, and the float32 dQ accumulator converted to the
// I/O type after it.  Both are HBM-bound streaming kernels with 16-byte
// vector loads.
#include "nsp_internal.cuh"

namespace nsp {
namespace {

template <typename TI>
__device__ __forceinline__ void load8(const TI* p, float (&x)[16 / sizeof(TI)]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&x)[4]) {
  const float4 u = __ldg(reinterpret_cast<const float4*>(p));
  x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
}

// delta[h, t] = <dout[t, h, :], out[t, h, :]> and nlse2[h, t] = -lse[h, t] log2(e),
// both with row stride Tp (rows padded to whole tiles, padding set to 0);
// TPR threads share one (t, h) row.  Rows are walked in memory order: the
// packed [T, Hq, d] layout (P = 1) or the head-group-major [P][T][Hq/P][d].
template <typename TI, int D, bool GROUPED>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const TI* __restrict__ out,
                                                        const TI* __restrict__ dout,
                                                        const float* __restrict__ lse,
                                                        float* __restrict__ delta,
                                                        float* __restrict__ nlse2, int64_t T,
                                                        int64_t Tp, int Hq, int P,
                                                        const WsHeader* hdr) {
  constexpr int VEC = 16 / sizeof(TI);
  constexpr int TPR = D / VEC;                  // 16 (bf16, d=128) ... 32 (f32, d=128)
  constexpr int RPW = 32 / TPR;                 // rows per warp step
  static_assert(TPR <= 32 && 32 % TPR == 0, "row split");
  grid_dep_trigger();                       // the dK/dV kernel may launch (it waits)
  if (status_bad(hdr)) return;
  const int lane = threadIdx.x & 31;
  const int sub = lane / TPR, part = lane % TPR;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t rows = T * Hq;
  for (int64_t r0 = warp * RPW; r0 < rows; r0 += nwarps * RPW) {
    const int64_t rr = r0 + sub;
    float acc = 0.f;
    if (rr < rows) {
      float a[VEC], b[VEC];
      load8<TI>(out + rr * D + part * VEC, a);
      load8<TI>(dout + rr * D + part * VEC, b);
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc = fmaf(a[i], b[i], acc);
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (rr < rows && part == 0) {
      int64_t t;
      int h;
      if constexpr (!GROUPED) {
        t = rr / Hq;
        h = (int)(rr - t * Hq);
      } else {                              // rr = (g T + t) (Hq/P) + j, h = g (Hq/P) + j
        const int hpg = Hq / P;
        const int64_t gt = rr / hpg;
        const int64_t g = gt / T;
        t = gt - g * T;
        h = (int)(g * hpg + (rr - gt * hpg));
      }
      delta[(int64_t)h * Tp + t] = acc;
      nlse2[(int64_t)h * Tp + t] = lse[(int64_t)h * T + t] * -1.4426950408889634f;
    }
  }
  // zero the padding columns [T, Tp) of every head row
  const int64_t pad = Tp - T;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = gtid; e < pad * Hq; e += nthreads) {
    const int64_t h = e / pad, t = T + e % pad;
    delta[h * Tp + t] = 0.f;
    nlse2[h * Tp + t] = 0.f;
  }
}

template <typename TO>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         TO* __restrict__ dq, int64_t n4,
                                                         const WsHeader* hdr) {
  if (status_bad(hdr)) return;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(acc) + i);
    if constexpr (sizeof(TO) == 2) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
      const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&a);
      u.y = *reinterpret_cast<const uint32_t*>(&b);
      reinterpret_cast<uint2*>(dq)[i] = u;
    } else {
      reinterpret_cast<float4*>(dq)[i] = v;
    }
  }
}

}  // namespace

cudaError_t launch_bwd_delta(const void* out, const void* dout, const float* lse, float* delta,
                             float* nlse2, int64_t T, int64_t Tp, int Hq, int d, int io_dtype,
                             int P, WsHeader* hdr, cudaStream_t s) {
  const int blocks = num_sms() * 8;
  const bool g = P > 1;
  auto go = [&](auto kern, const auto* o, const auto* dq) {
    kern<<<blocks, 256, 0, s>>>(o, dq, lse, delta, nlse2, T, Tp, Hq, P, hdr);
  };
  using bf = __nv_bfloat16;
  const bf* ob = reinterpret_cast<const bf*>(out);
  const bf* db = reinterpret_cast<const bf*>(dout);
  const float* of = reinterpret_cast<const float*>(out);
  const float* df = reinterpret_cast<const float*>(dout);
  // the packed layout's instantiation has no head-group arithmetic at all
  if (io_dtype == NSP_BF16 && d == 128)
    g ? go(bwd_delta_kernel<bf, 128, true>, ob, db) : go(bwd_delta_kernel<bf, 128, false>, ob, db);
  else if (io_dtype == NSP_BF16)
    g ? go(bwd_delta_kernel<bf, 64, true>, ob, db) : go(bwd_delta_kernel<bf, 64, false>, ob, db);
  else if (d == 128)
    g ? go(bwd_delta_kernel<float, 128, true>, of, df)
      : go(bwd_delta_kernel<float, 128, false>, of, df);
  else
    g ? go(bwd_delta_kernel<float, 64, true>, of, df)
      : go(bwd_delta_kernel<float, 64, false>, of, df);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* acc, void* dq, int64_t n, int io_dtype,
                              WsHeader* hdr, cudaStream_t s) {
  const int blocks = num_sms() * 8;
  if (io_dtype == NSP_BF16)
    dq_convert_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        acc, reinterpret_cast<__nv_bfloat16*>(dq), n / 4, hdr);
  else
    dq_convert_kernel<float><<<blocks, 256, 0, s>>>(acc, reinterpret_cast<float*>(dq), n / 4, hdr);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace nsp
