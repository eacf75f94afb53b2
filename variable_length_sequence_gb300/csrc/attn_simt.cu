// CUDA-core (FP32 FMA) varlen attention, forward and backward.
//
// This is the path for float32 inputs (computed in true float32, no TF32)
// and for shapes the tensor-core kernels do not take.  It computes the same
// definition as the tcgen05 path: scaled dot-product attention (BASP,
// Sec. II-A) restricted to each packed document (HSAP, Sec. 2.1, cu_len),
// causal within the document, optionally restricted to a query range and a
// key range (ring-style partial blocks, HSAP Sec. 2.2.1).
//
// Every query row t sees a single contiguous key interval [lo_t, hi_t):
// its document's start (clipped to the key range) up to itself (causal) or
// to the document's end.  Masking is a per-row interval test, so a tile that
// spans several short documents is handled without a doc-id per key.
#include "nsp_internal.cuh"

namespace nsp {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- forward
// Block: 64 query rows of one head; 2 threads per row, each owning half of
// the head dimension.  K/V tiles of 32 keys are staged in shared memory as
// float32; the second half of every row is shifted by 4 floats so that the
// two distinct addresses of a warp-wide load fall in different banks.
constexpr int kFwdBM = 64, kFwdBN = 32, kFwdThreads = 128;

template <int D>
struct FwdSmem {
  static constexpr int DH = D / 2;
  static constexpr int ROW = D + 8;
  float k[kFwdBN][ROW];
  float v[kFwdBN][ROW];
};

template <int D>
__device__ __forceinline__ int smem_col(int c) { return c + (c >= D / 2 ? 4 : 0); }

template <typename TI, typename TO, int D>
__global__ void __launch_bounds__(kFwdThreads) attn_fwd_simt_kernel(AttnProblem p) {
  constexpr int DH = D / 2;
  __shared__ __align__(16) FwdSmem<D> sm;
  __shared__ int s_klo, s_khi;
  if (status_bad(p.hdr)) return;

  const int tid = threadIdx.x;
  const int r = tid >> 1, half = tid & 1;
  const int h = blockIdx.y;
  const int g = h / (p.Hq / p.Hkv);
  const int64_t row = (int64_t)blockIdx.x * kFwdBM + r;       // shard-relative
  const bool valid = row < p.q_len;
  const int64_t t = p.q_start + row;                           // global
  const int64_t kv_end = p.kv_start + p.kv_len;

  // This row's allowed key interval, shard-relative: [lo, hi).
  int64_t lo = 0, hi = 0;
  if (valid) {
    const int b = doc_of(p.cu, p.ndoc, t);
    const int64_t glo = max((int64_t)p.cu[b], p.kv_start);
    const int64_t ghi = min(p.causal ? t + 1 : (int64_t)p.cu[b + 1], kv_end);
    lo = glo - p.kv_start;
    hi = max(ghi - p.kv_start, lo);
  }
  if (tid == 0) { s_klo = INT_MAX; s_khi = 0; }
  __syncthreads();
  if (valid && hi > lo) { atomicMin(&s_klo, (int)lo); atomicMax(&s_khi, (int)hi); }
  __syncthreads();
  const int klo = s_klo, khi = s_khi;

  const TI* Q = reinterpret_cast<const TI*>(p.q);
  const TI* K = reinterpret_cast<const TI*>(p.k);
  const TI* V = reinterpret_cast<const TI*>(p.v);
  float qr[DH];
  const float sl2 = p.scale * kLog2e;
#pragma unroll
  for (int c = 0; c < DH; ++c)
    qr[c] = valid ? ld_in(Q + qo_offset(p, row, h) + half * DH + c) * sl2 : 0.f;

  float o[DH];
#pragma unroll
  for (int c = 0; c < DH; ++c) o[c] = 0.f;
  float m = -INFINITY, l = 0.f;

  for (int j0 = (klo == INT_MAX ? khi : (klo / kFwdBN) * kFwdBN); j0 < khi; j0 += kFwdBN) {
    __syncthreads();
    for (int e = tid; e < kFwdBN * D; e += kFwdThreads) {
      const int jj = e / D, c = e % D;
      const int64_t key = j0 + jj;
      float kv = 0.f, vv = 0.f;
      if (key < p.kv_len) {
        kv = ld_in(K + (key * p.Hkv + g) * D + c);
        vv = ld_in(V + (key * p.Hkv + g) * D + c);
      }
      sm.k[jj][smem_col<D>(c)] = kv;
      sm.v[jj][smem_col<D>(c)] = vv;
    }
    __syncthreads();

    float s[kFwdBN];
    float mt = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < kFwdBN; ++jj) {
      const float4* kr = reinterpret_cast<const float4*>(&sm.k[jj][half * (DH + 4)]);
      float acc = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < DH / 4; ++c4) {
        const float4 kk = kr[c4];
        acc = fmaf(qr[4 * c4 + 0], kk.x, acc);
        acc = fmaf(qr[4 * c4 + 1], kk.y, acc);
        acc = fmaf(qr[4 * c4 + 2], kk.z, acc);
        acc = fmaf(qr[4 * c4 + 3], kk.w, acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      const int64_t key = j0 + jj;
      s[jj] = (key >= lo && key < hi) ? acc : -INFINITY;     // log2-domain score
      mt = fmaxf(mt, s[jj]);
    }
    const float m_new = fmaxf(m, mt);
    if (m_new == -INFINITY) continue;                          // nothing allowed yet
    const float corr = exp2f(m - m_new);                       // 0 when m = -inf
    l *= corr;
#pragma unroll
    for (int c = 0; c < DH; ++c) o[c] *= corr;
#pragma unroll
    for (int jj = 0; jj < kFwdBN; ++jj) {
      const float pj = exp2f(s[jj] - m_new);
      l += pj;
      const float4* vr = reinterpret_cast<const float4*>(&sm.v[jj][half * (DH + 4)]);
#pragma unroll
      for (int c4 = 0; c4 < DH / 4; ++c4) {
        const float4 vv = vr[c4];
        o[4 * c4 + 0] = fmaf(pj, vv.x, o[4 * c4 + 0]);
        o[4 * c4 + 1] = fmaf(pj, vv.y, o[4 * c4 + 1]);
        o[4 * c4 + 2] = fmaf(pj, vv.z, o[4 * c4 + 2]);
        o[4 * c4 + 3] = fmaf(pj, vv.w, o[4 * c4 + 3]);
      }
    }
    m = m_new;
  }

  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (p.accumulate) {
    // merge this partial into the running result (both threads of the row
    // read the old lse before the first one writes the new one)
    const float lp = (valid && l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
    float la = -INFINITY;
    if (lp != -INFINITY) la = p.lse[(int64_t)h * p.q_len + row];
    __syncwarp();
    if (lp == -INFINITY) return;
    const float mx = fmaxf(la, lp);
    const float L = mx + logf(expf(la - mx) + expf(lp - mx));
    const float wa = expf(la - L), wp = expf(lp - L) * inv;
    float* A = reinterpret_cast<float*>(p.out) + qo_offset(p, row, h) + half * DH;
#pragma unroll
    for (int c = 0; c < DH; ++c) A[c] = fmaf(wa, A[c], wp * o[c]);
    if (half == 0) p.lse[(int64_t)h * p.q_len + row] = L;
    return;
  }
  if (!valid) return;
  TO* O = reinterpret_cast<TO*>(p.out);
#pragma unroll
  for (int c = 0; c < DH; ++c) st_out(O + qo_offset(p, row, h) + half * DH + c, o[c] * inv);
  if (half == 0 && p.lse != nullptr)
    p.lse[(int64_t)h * p.q_len + row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// ---------------------------------------------------------------- backward
// Key-stationary dK/dV: a block owns 32 keys of one KV head, loops over the
// query heads of the group and over every query tile whose rows can see its
// keys, recomputing p from lse; dQ partial sums go to a float32 accumulator
// with atomics.  4 threads per key, each owning a quarter of the head dim.
constexpr int kBwdBK = 32, kBwdBM = 32, kBwdThreads = 128;

template <int D>
struct BwdSmem {
  float q[kBwdBM][D + 4];
  float dO[kBwdBM][D + 4];
  float k[kBwdBK][D + 4];
  float ds[kBwdBM][kBwdBK + 1];
  float lse[kBwdBM];
  float delta[kBwdBM];
  int64_t lo[kBwdBM];
  int64_t hi[kBwdBM];
};

template <typename TI, int D>
__global__ void __launch_bounds__(kBwdThreads) attn_bwd_dkdv_simt_kernel(
    AttnProblem p, const TI* __restrict__ dout, const float* __restrict__ lse,
    const float* __restrict__ delta, int64_t delta_stride, float* __restrict__ dq_acc,
    TI* __restrict__ dk, TI* __restrict__ dv, float* __restrict__ dk_acc32,
    float* __restrict__ dv_acc32) {
  constexpr int DQ = D / 4;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
  if (status_bad(p.hdr)) return;

  const int tid = threadIdx.x;
  const int j = tid >> 2, qtr = tid & 3;
  const int g = blockIdx.y;
  const int G = p.Hq / p.Hkv;
  const int64_t T = p.q_len;                      // query rows of the range
  const int64_t NK = p.kv_len;                    // keys of the range
  const int64_t key0 = (int64_t)blockIdx.x * kBwdBK;
  const int64_t key = key0 + j;
  const int64_t key_g = p.kv_start + key;         // global token id of this thread's key
  const bool kvalid = key < NK;
  const int64_t key_last = min(key0 + kBwdBK, NK) - 1;

  const TI* Q = reinterpret_cast<const TI*>(p.q);
  const TI* K = reinterpret_cast<const TI*>(p.k);
  const TI* V = reinterpret_cast<const TI*>(p.v);

  float kr[DQ], vr[DQ], dk_acc[DQ], dv_acc[DQ];
#pragma unroll
  for (int c = 0; c < DQ; ++c) {
    kr[c] = kvalid ? ld_in(K + (key * p.Hkv + g) * D + qtr * DQ + c) : 0.f;
    vr[c] = kvalid ? ld_in(V + (key * p.Hkv + g) * D + qtr * DQ + c) : 0.f;
    dk_acc[c] = 0.f;
    dv_acc[c] = 0.f;
  }
  for (int e = tid; e < kBwdBK * D; e += kBwdThreads) {
    const int jj = e / D, c = e % D;
    const int64_t kk = key0 + jj;
    sm.k[jj][c] = kk < NK ? ld_in(K + (kk * p.Hkv + g) * D + c) : 0.f;
  }
  // Query rows (relative to the query range) that can see any key of this block.
  const int64_t k0g = p.kv_start + key0, klg = p.kv_start + key_last;
  const int b0 = doc_of(p.cu, p.ndoc, k0g), b1 = doc_of(p.cu, p.ndoc, klg);
  const int64_t r_lo = max(p.causal ? k0g : (int64_t)p.cu[b0], p.q_start) - p.q_start;
  const int64_t r_hi = min((int64_t)p.cu[b1 + 1], p.q_start + T) - p.q_start;
  const float sl2 = p.scale * kLog2e;

  for (int hh = 0; hh < G; ++hh) {
    const int h = g * G + hh;
    for (int64_t t0 = r_lo; t0 < r_hi; t0 += kBwdBM) {
      __syncthreads();
      for (int e = tid; e < kBwdBM * D; e += kBwdThreads) {
        const int rr = e / D, c = e % D;
        const int64_t t = t0 + rr;
        const bool ok = t < r_hi;
        sm.q[rr][c] = ok ? ld_in(Q + qo_offset(p, t, h) + c) : 0.f;
        sm.dO[rr][c] = ok ? ld_in(dout + qo_offset(p, t, h) + c) : 0.f;
      }
      if (tid < kBwdBM) {
        const int64_t t = t0 + tid;
        if (t < r_hi) {
          const int64_t tg = p.q_start + t;
          const int b = doc_of(p.cu, p.ndoc, tg);
          sm.lo[tid] = p.cu[b];
          sm.hi[tid] = p.causal ? tg + 1 : (int64_t)p.cu[b + 1];
          sm.lse[tid] = lse[(int64_t)h * T + t];
          sm.delta[tid] = delta[(int64_t)h * delta_stride + t];
        } else {
          sm.lo[tid] = 0; sm.hi[tid] = 0; sm.lse[tid] = 0.f; sm.delta[tid] = 0.f;
        }
      }
      __syncthreads();
      for (int rr = 0; rr < kBwdBM; ++rr) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < DQ; ++c) {
          s = fmaf(sm.q[rr][qtr * DQ + c], kr[c], s);
          dp = fmaf(sm.dO[rr][qtr * DQ + c], vr[c], dp);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        dp += __shfl_xor_sync(0xffffffffu, dp, 1);
        dp += __shfl_xor_sync(0xffffffffu, dp, 2);
        const bool allowed = kvalid && key_g >= sm.lo[rr] && key_g < sm.hi[rr];
        const float pr = allowed ? exp2f(s * sl2 - sm.lse[rr] * kLog2e) : 0.f;
        const float ds = pr * (dp - sm.delta[rr]);
#pragma unroll
        for (int c = 0; c < DQ; ++c) {
          dv_acc[c] = fmaf(pr, sm.dO[rr][qtr * DQ + c], dv_acc[c]);
          dk_acc[c] = fmaf(ds, sm.q[rr][qtr * DQ + c], dk_acc[c]);
        }
        if (qtr == 0) sm.ds[rr][j] = ds;
      }
      __syncthreads();
      // dQ[t, h, c] += scale * sum_j ds[t][j] k[j][c]
      for (int e = tid; e < kBwdBM * D; e += kBwdThreads) {
        const int rr = e / D, c = e % D;
        const int64_t t = t0 + rr;
        if (t >= r_hi) continue;
        float acc = 0.f;
#pragma unroll 8
        for (int jj = 0; jj < kBwdBK; ++jj) acc = fmaf(sm.ds[rr][jj], sm.k[jj][c], acc);
        if (acc != 0.f) atomicAdd(dq_acc + qo_offset(p, t, h) + c, acc * p.scale);
      }
    }
  }
  if (!kvalid) return;
  if (p.accumulate) {
    // ring block: add into the float32 accumulators (one thread per element)
#pragma unroll
    for (int c = 0; c < DQ; ++c) {
      dk_acc32[(key * p.Hkv + g) * D + qtr * DQ + c] += dk_acc[c] * p.scale;
      dv_acc32[(key * p.Hkv + g) * D + qtr * DQ + c] += dv_acc[c];
    }
    return;
  }
#pragma unroll
  for (int c = 0; c < DQ; ++c) {
    st_out(dk + (key * p.Hkv + g) * D + qtr * DQ + c, dk_acc[c] * p.scale);
    st_out(dv + (key * p.Hkv + g) * D + qtr * DQ + c, dv_acc[c]);
  }
}

template <typename TI, typename TO, int D>
cudaError_t fwd_dispatch(const AttnProblem& p, cudaStream_t s) {
  dim3 grid((unsigned)ceil_div(p.q_len, kFwdBM), (unsigned)p.Hq);
  attn_fwd_simt_kernel<TI, TO, D><<<grid, kFwdThreads, 0, s>>>(p); count_launches(1);
  count_path(false);
  return cudaGetLastError();
}

template <typename TI, int D>
cudaError_t bwd_dispatch(const AttnProblem& p, const void* out, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, const BwdWsLayout& L,
                         char* ws, cudaStream_t s) {
  const int64_t T = p.q_len;
  float* delta = reinterpret_cast<float*>(ws + L.delta);
  // a ring block adds dQ straight into the caller's float32 accumulator
  float* dq_acc = p.accumulate ? reinterpret_cast<float*>(dq)
                               : reinterpret_cast<float*>(ws + L.dq_acc);
  cudaError_t e = cudaSuccess;
  if (!p.accumulate) e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)T * p.Hq * D, s);
  if (e != cudaSuccess) return e;
  e = launch_bwd_delta(out, dout, lse, delta, reinterpret_cast<float*>(ws + L.nlse2), T, L.Tp,
                       p.Hq, D, p.io_dtype, p.q_groups, p.hdr, s);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(BwdSmem<D>);
  e = cudaFuncSetAttribute(attn_bwd_dkdv_simt_kernel<TI, D>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ceil_div(p.kv_len, kBwdBK), (unsigned)p.Hkv);
  attn_bwd_dkdv_simt_kernel<TI, D><<<grid, kBwdThreads, smem, s>>>(
      p, reinterpret_cast<const TI*>(dout), lse, delta, L.Tp, dq_acc, reinterpret_cast<TI*>(dk),
      reinterpret_cast<TI*>(dv), reinterpret_cast<float*>(dk), reinterpret_cast<float*>(dv));
  count_launches(1);
  count_path(false);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.accumulate) return e;
  return launch_dq_convert(dq_acc, dq, T * p.Hq * D, p.io_dtype, p.hdr, s);
}

}  // namespace

cudaError_t launch_attn_fwd_simt(const AttnProblem& p, cudaStream_t s) {
  const bool bf = p.io_dtype == NSP_BF16;
  const bool of = p.out_dtype == NSP_F32;
  if (p.d == 128) {
    if (bf) return of ? fwd_dispatch<__nv_bfloat16, float, 128>(p, s)
                      : fwd_dispatch<__nv_bfloat16, __nv_bfloat16, 128>(p, s);
    return fwd_dispatch<float, float, 128>(p, s);
  }
  if (bf) return of ? fwd_dispatch<__nv_bfloat16, float, 64>(p, s)
                    : fwd_dispatch<__nv_bfloat16, __nv_bfloat16, 64>(p, s);
  return fwd_dispatch<float, float, 64>(p, s);
}

cudaError_t launch_attn_bwd_simt(const AttnProblem& p, const void* out, const void* dout,
                                 const float* lse, void* dq, void* dk, void* dv,
                                 const BwdWsLayout& L, char* ws, cudaStream_t s) {
  const bool bf = p.io_dtype == NSP_BF16;
  if (p.d == 128)
    return bf ? bwd_dispatch<__nv_bfloat16, 128>(p, out, dout, lse, dq, dk, dv, L, ws, s)
              : bwd_dispatch<float, 128>(p, out, dout, lse, dq, dk, dv, L, ws, s);
  return bf ? bwd_dispatch<__nv_bfloat16, 64>(p, out, dout, lse, dq, dk, dv, L, ws, s)
            : bwd_dispatch<float, 64>(p, out, dout, lse, dq, dk, dv, L, ws, s);
}

}  // namespace nsp
