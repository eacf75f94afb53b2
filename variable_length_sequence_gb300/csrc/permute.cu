// Ulysses seq -> head layout permutation (HSAP, Sec. 2.2.2 "Intra-group
// Sequence Parallelism": R^{n x H x d} per group -> R^{N x h x d}, h = H/P;
// BASP, Sec. II-C "DeepSpeed Ulysses").
//
// With the P sequence shards stacked as in = [T, H, d], the head group g of
// token t, in[t][g*h .. g*h+h)[:], is one contiguous chunk of h*d elements,
// and it lands as one contiguous chunk at out[g][t].  So the permutation is
// a transpose of a [T][P] grid of chunks into a [P][T] grid (the inverse
// transposes back).  BASP's subgroup all-to-all (Sec. IV: B sequences of L
// tokens, each exchanged among its own K ranks) is the same transpose done
// independently for each sequence: B stacked [L][K] grids become B stacked
// [K][L] grids, at the same offsets.  It is pure data movement, bound by HBM bandwidth: each
// warp moves whole chunks with 16-byte vector loads and stores, several in
// flight per thread, neither reads nor writes allocated in L1.
#include "nsp_internal.cuh"

namespace nsp {
namespace {

constexpr int kPermThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Vector path: chunk size (in 16-byte words) cw; for each of nb stacked
// grids, chunk (a, b) of the source grid [A][B] goes to (b, a) of the
// destination grid [B][A].  Each warp takes kUnroll destination chunks per
// step and issues all their loads before the stores.
__global__ void __launch_bounds__(kPermThreads) permute_vec_kernel(const uint4* __restrict__ in,
                                                                   uint4* __restrict__ out,
                                                                   int64_t A, int64_t B,
                                                                   int64_t cw, int64_t nb) {
  const int lane = threadIdx.x & 31;
  const int64_t grid = A * B;
  const int64_t nchunks = grid * nb;
  const int64_t warp = ((int64_t)blockIdx.x * kPermThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kPermThreads) >> 5;
  for (int64_t c0 = warp * kUnroll; c0 < nchunks; c0 += nwarps * kUnroll) {
    const uint4* src[kUnroll];
    uint4* dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = c0 + u;                 // destination chunk = z grid + b A + a
      const int64_t z = c / grid, loc = c - z * grid;
      const int64_t a = loc % A, b = loc / A;
      src[u] = in + (z * grid + a * B + b) * cw;
      dst[u] = out + c * cw;
    }
    for (int64_t x = lane; x < cw; x += 32) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (c0 + u < nchunks) v[u] = ld_stream(src[u] + x);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (c0 + u < nchunks) st_stream(dst[u] + x, v[u]);
    }
  }
}

// Element path for chunk sizes that are not a multiple of 16 bytes.
template <typename E>
__global__ void __launch_bounds__(kPermThreads) permute_elem_kernel(const E* __restrict__ in,
                                                                    E* __restrict__ out,
                                                                    int64_t A, int64_t B,
                                                                    int64_t ce, int64_t nb) {
  const int lane = threadIdx.x & 31;
  const int64_t grid = A * B;
  const int64_t nchunks = grid * nb;
  const int64_t warp = ((int64_t)blockIdx.x * kPermThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kPermThreads) >> 5;
  for (int64_t c = warp; c < nchunks; c += nwarps) {
    const int64_t z = c / grid, loc = c - z * grid;
    const int64_t a = loc % A, b = loc / A;
    const E* src = in + (z * grid + a * B + b) * ce;
    E* dst = out + c * ce;
    for (int64_t x = lane; x < ce; x += 32) dst[x] = src[x];
  }
}

}  // namespace

cudaError_t launch_permute(const void* in, void* out, int64_t T, int H, int d, int P,
                           int elem_bytes, int inverse, cudaStream_t s) {
  return launch_permute_groups(in, out, 1, T, H, d, P, elem_bytes, inverse, s);
}

cudaError_t launch_permute_groups(const void* in, void* out, int64_t nb, int64_t T, int H, int d,
                                  int P, int elem_bytes, int inverse, cudaStream_t s) {
  const int64_t h = H / P;
  const int64_t chunk_bytes = h * d * elem_bytes;
  // per group of T tokens, seq2head: source grid [T][P] -> destination
  // [P][T]; inverse: [P][T] -> [T][P].
  const int64_t A = inverse ? P : T;
  const int64_t B = inverse ? T : P;
  const int nsm = num_sms();
  if (chunk_bytes % 16 == 0) {
    const int64_t cw = chunk_bytes / 16;
    int64_t blocks = ceil_div(A * B * nb, (int64_t)(kPermThreads / 32) * kUnroll);
    blocks = blocks < (int64_t)nsm * 8 ? blocks : (int64_t)nsm * 8;
    if (blocks < 1) blocks = 1;
    permute_vec_kernel<<<(unsigned)blocks, kPermThreads, 0, s>>>(
        reinterpret_cast<const uint4*>(in), reinterpret_cast<uint4*>(out), A, B, cw, nb); count_launches(1);
    return cudaGetLastError();
  }
  const int64_t ce = h * d;
  int64_t blocks = ceil_div(A * B * nb, (int64_t)(kPermThreads / 32));
  blocks = blocks < (int64_t)nsm * 8 ? blocks : (int64_t)nsm * 8;
  if (blocks < 1) blocks = 1;
  switch (elem_bytes) {
    case 1: permute_elem_kernel<uint8_t><<<(unsigned)blocks, kPermThreads, 0, s>>>(
                reinterpret_cast<const uint8_t*>(in), reinterpret_cast<uint8_t*>(out), A, B, ce, nb); count_launches(1);
            break;
    case 2: permute_elem_kernel<uint16_t><<<(unsigned)blocks, kPermThreads, 0, s>>>(
                reinterpret_cast<const uint16_t*>(in), reinterpret_cast<uint16_t*>(out), A, B, ce, nb); count_launches(1);
            break;
    case 4: permute_elem_kernel<uint32_t><<<(unsigned)blocks, kPermThreads, 0, s>>>(
                reinterpret_cast<const uint32_t*>(in), reinterpret_cast<uint32_t*>(out), A, B, ce, nb); count_launches(1);
            break;
    default: permute_elem_kernel<uint64_t><<<(unsigned)blocks, kPermThreads, 0, s>>>(
                reinterpret_cast<const uint64_t*>(in), reinterpret_cast<uint64_t*>(out), A, B, ce, nb); count_launches(1);
            break;
  }
  return cudaGetLastError();
}

}  // namespace nsp
