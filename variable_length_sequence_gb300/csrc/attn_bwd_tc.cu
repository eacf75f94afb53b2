// Varlen attention backward on the tcgen05 tensor cores, bf16 inputs,
// float32 accumulation, d = 128.
//
// Gradients of L = sum(dOut * out) for document-masked attention (BASP
// Sec. II-A, HSAP Sec. 2.1), recomputing the probabilities from the saved
// lse instead of storing them (the recomputation NSP Sec. 2.3 discusses):
//   P = exp(scale Q K^T - lse),  dP = dOut V^T,  dS = P (dP - delta),
//   dV = P^T dOut,  dK = scale dS^T Q,  dQ = scale dS K,
// delta = rowsum(dOut * out) (computed by bwd_delta_kernel beforehand).
//
// Work item: one 128-key tile of one KV head.  It walks every (query head
// of the group, 128-row query tile that can see the keys) pair; the key
// tile's dK and dV accumulate in TMEM over the whole walk, so they are
// written once, without atomics.  dQ of each step is added to a float32
// accumulator with vector reductions (red.global.add.v4.f32).
//
// Per step (keys are the M dimension of the transposed products):
//   S^T  = K Q^T          TMEM R0 [0,128)     (A = K, B = Q, both K-major smem)
//   dP^T = V dOut^T       TMEM R1 [128,256)   (A = V, B = dOut, K-major)
//   softmax warps: P^T = 2^(S^T scale log2e - lse log2e), dS^T = P^T (dP^T - delta),
//     P^T (bf16) written over S^T in TMEM, dS^T (bf16) to shared memory in a
//     128-byte-swizzled [q-block][key][64] layout
//   dV  += P^T dOut       TMEM R2 [256,384)   (A = P^T from TMEM, B = dOut MN-major)
//   dK  += dS^T Q         TMEM R3 [384,512)   (A = dS^T smem K-major, B = Q MN-major)
//   dQ   = dS K           TMEM R1             (A = dS smem MN-major, B = K MN-major)
//   epilogue warps: dQ rows (TMEM lane = query row) -> scale -> red.add to global
// The next step's S^T is issued right after this step's dQ (the tensor core
// executes its MMAs in order, so S^T never overwrites P^T before dV read it);
// its dP^T waits until the dQ rows have been read out of R1.
//
// CTA roles (320 threads): warps 0-3 and 4-7 each own half of the query
// columns of the softmax and half of the head dimension of the dQ epilogue
// (TMEM lanes 0-127 each); warp 8 is the TMA producer; warp 9 allocates TMEM
// and one of its threads issues every MMA.  All waits are bounded.
#include <cudaTypedefs.h>

#include "tc_ptx.cuh"

namespace nsp {
namespace {

using namespace tc;

constexpr int BK = 128, BQ = 128, HD = 128;
constexpr int kThreads = 320;
constexpr int kWarpProducer = 8, kWarpMma = 9;
constexpr uint32_t kColBlockBytes = 128 * 64 * 2;
constexpr uint32_t kTileBytes = 2 * kColBlockBytes;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdItem {
  int ktile;      // 128-key tile
  int g;          // key/value head
  int i_lo;       // first query tile that sees the keys
  int n_q;        // number of query tiles
  int steps;      // G * n_q (-1: stop)
  int pad[3];
};

struct __align__(1024) Smem {
  uint8_t k[kTileBytes];
  uint8_t v[kTileBytes];
  uint8_t q[2][kTileBytes];
  uint8_t dout[2][kTileBytes];
  uint8_t ds[kTileBytes];
  float lse2[2][BQ];           // lse * log2(e) of the stage's query rows
  float delta[2][BQ];
  uint64_t kv_full, kv_empty;
  uint64_t qdo_full[2], qdo_empty[2];
  uint64_t s_full, ds_full, dq_full, dq_empty, dkv_full, dkv_empty;
  uint64_t item_full[2], item_empty[2];
  BwdItem items[2];
  uint32_t tmem_base;
  int abort_flag;
};

// Dynamic shared memory: the tile set plus whatever alignment slack still
// fits under the 227 KB limit; the kernel checks at run time that the
// 1024-byte-aligned tile set fits (the base is 1024-aligned in practice).
constexpr size_t kSmemLimit = 232448;
static_assert(sizeof(Smem) <= kSmemLimit, "backward tile set exceeds 227 KB of shared memory");
constexpr size_t kSmemBytes =
    sizeof(Smem) + 1024 <= kSmemLimit ? sizeof(Smem) + 1024 : kSmemLimit;

// D (+)= A B^T with both operands K-major, 128-byte swizzle (as the forward QK^T).
__device__ __forceinline__ void mma_kk(uint32_t d_tmem, uint32_t a_saddr, uint32_t b_saddr,
                                       bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
  const uint64_t ad = smem_desc_sw128(a_saddr, 16, 1024);
  const uint64_t bd = smem_desc_sw128(b_saddr, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = ((kk >> 2) * kColBlockBytes + (kk & 3) * 32) >> 4;
    mma_ss(d_tmem, ad + off, bd + off, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <typename TO>
__device__ __forceinline__ void store_row32(TO* dst, const uint32_t (&v)[32], float scale) {
  if constexpr (sizeof(TO) == 2) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * scale, __uint_as_float(v[2 * i + 1]) * scale);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  } else {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      d4[i] = make_float4(__uint_as_float(v[4 * i]) * scale, __uint_as_float(v[4 * i + 1]) * scale,
                          __uint_as_float(v[4 * i + 2]) * scale,
                          __uint_as_float(v[4 * i + 3]) * scale);
  }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles) return;
  }
}

struct BwdArgs {
  AttnProblem p;
  const float* lse2;      // [Hq, Tp] lse * log2(e), padded rows
  const float* delta;     // [Hq, Tp]
  int64_t Tp;
  float* dq_acc;          // [T, Hq, d] float32, zeroed
  __nv_bfloat16* dk;      // [T, Hkv, d]
  __nv_bfloat16* dv;
  const int2* ktiles;     // per key tile: first/last query tile
  const int* korder;      // key tiles, most query tiles first
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const BwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const AttnProblem& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = p.hdr;
  if (status_bad(hdr)) return;
  {
    uint32_t dyn_bytes;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
    const uint32_t base = smem_u32(smem_raw);
    if (((base + 1023u) & ~1023u) - base + sizeof(Smem) > dyn_bytes) {
      if (threadIdx.x == 0) atomicExch(&hdr->status, (int)NSP_ERR_UNSUPPORTED);
      return;
    }
  }
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));

  if (threadIdx.x == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.qdo_full[s], 1);
      mbar_init(&sm.qdo_empty[s], 1);
      mbar_init(&sm.item_full[s], 1);
      mbar_init(&sm.item_empty[s], 1 + 8);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.ds_full, 256);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_empty, 256);
    mbar_init(&sm.dkv_full, 1);
    mbar_init(&sm.dkv_empty, 256);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  const int G = p.Hq / p.Hkv;
  const int64_t T = p.q_len;
  const int n_items = hdr->n_items2 * p.Hkv;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it_count = 0, kv_count = 0, qc = 0;
      bool ok = true;
      while (ok) {
        const int idx = atomicAdd(&hdr->counter2, 1);
        BwdItem it;
        it.ktile = 0; it.g = 0; it.i_lo = 0; it.n_q = 0; it.steps = -1;
        if (idx < n_items) {
          const int kt = a.korder[idx / p.Hkv];
          const int2 tr = a.ktiles[kt];
          it.ktile = kt;
          it.g = idx - (idx / p.Hkv) * p.Hkv;
          it.i_lo = tr.x;
          it.n_q = tr.y - tr.x + 1;
          it.steps = G * it.n_q;
        }
        const uint32_t slot = it_count & 1;
        if (it_count >= 2 &&
            !mbar_wait(&sm.item_empty[slot], ((it_count >> 1) - 1) & 1, abort_flag, hdr)) {
          ok = false;
          break;
        }
        sm.items[slot] = it;
        mbar_arrive(&sm.item_full[slot]);
        ++it_count;
        if (it.steps < 0) break;
        if (kv_count >= 1 && !mbar_wait(&sm.kv_empty, (kv_count - 1) & 1, abort_flag, hdr)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          tma_load_2d(sm.k + cb * kColBlockBytes, &tm_k, &sm.kv_full, it.g * HD + cb * 64,
                      it.ktile * BK);
          tma_load_2d(sm.v + cb * kColBlockBytes, &tm_v, &sm.kv_full, it.g * HD + cb * 64,
                      it.ktile * BK);
        }
        ++kv_count;
        for (int n = 0; n < it.steps; ++n) {
          const int h = it.g * G + n / it.n_q;
          const int i = it.i_lo + n % it.n_q;
          const uint32_t st = qc & 1, use = qc >> 1;
          if (use >= 1 && !mbar_wait(&sm.qdo_empty[st], (use - 1) & 1, abort_flag, hdr)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.qdo_full[st], 2 * kTileBytes + 2 * BQ * sizeof(float));
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) {
            tma_load_2d(sm.q[st] + cb * kColBlockBytes, &tm_q, &sm.qdo_full[st], h * HD + cb * 64,
                        i * BQ);
            tma_load_2d(sm.dout[st] + cb * kColBlockBytes, &tm_do, &sm.qdo_full[st],
                        h * HD + cb * 64, i * BQ);
          }
          const int64_t row = (int64_t)h * a.Tp + (int64_t)i * BQ;
          bulk_load(sm.lse2[st], a.lse2 + row, BQ * sizeof(float), &sm.qdo_full[st]);
          bulk_load(sm.delta[st], a.delta + row, BQ * sizeof(float), &sm.qdo_full[st]);
          ++qc;
        }
      }
      if (!ok) {
        if (kv_count >= 1) drain_wait(&sm.kv_full, (kv_count - 1) & 1);
        for (uint32_t s = 0; s < 2 && s < qc; ++s) {
          const uint32_t last = qc - 1 - ((qc - 1 - s) & 1);
          drain_wait(&sm.qdo_full[last & 1], (last >> 1) & 1);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, true, false);   // B MN-major
      constexpr uint32_t idesc_dq = idesc_bf16_f32(128, 128, true, true);    // A, B MN-major
      const uint32_t k_s = smem_u32(sm.k), v_s = smem_u32(sm.v), ds_s = smem_u32(sm.ds);
      uint32_t it_count = 0, items_done = 0, qc = 0;
      bool ok = true;
      while (ok) {
        const uint32_t slot = it_count & 1;
        if (!mbar_wait(&sm.item_full[slot], (it_count >> 1) & 1, abort_flag, hdr)) break;
        const BwdItem it = sm.items[slot];
        mbar_arrive(&sm.item_empty[slot]);
        ++it_count;
        if (it.steps < 0) break;
        if (!mbar_wait(&sm.kv_full, items_done & 1, abort_flag, hdr)) break;
        for (int n = 0; n < it.steps && ok; ++n) {
          const uint32_t st = qc & 1;
          const uint32_t q_s = smem_u32(sm.q[st]), do_s = smem_u32(sm.dout[st]);
          if (n == 0) {
            if (!mbar_wait(&sm.qdo_full[st], (qc >> 1) & 1, abort_flag, hdr)) { ok = false; break; }
            tc_fence_after();
            mma_kk(tmem + kColS, k_s, q_s, false);                 // S^T = K Q^T
          }
          if (qc > 0 && !mbar_wait(&sm.dq_empty, (qc - 1) & 1, abort_flag, hdr)) { ok = false; break; }
          tc_fence_after();
          mma_kk(tmem + kColDP, v_s, do_s, false);                 // dP^T = V dOut^T
          mma_commit(&sm.s_full);
          if (!mbar_wait(&sm.ds_full, qc & 1, abort_flag, hdr)) { ok = false; break; }
          tc_fence_after();
          if (n == 0 && items_done > 0 &&
              !mbar_wait(&sm.dkv_empty, (items_done - 1) & 1, abort_flag, hdr)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool acc = n > 0;
          {
            // dV += P^T dOut: P^T columns of query rows 0-63 at [0,32), 64-127 at [64,96)
            const uint64_t bd = smem_desc_sw128(do_s, kColBlockBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t a_col = kColS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
              mma_ts(tmem + kColDV, tmem + a_col, bd + ((kk * 2048) >> 4), idesc_pv,
                     (acc || kk > 0) ? 1u : 0u);
            }
          }
          {
            // dK += dS^T Q: A = dS^T K-major (rows = keys), B = Q MN-major
            const uint64_t ad = smem_desc_sw128(ds_s, 16, 1024);
            const uint64_t bd = smem_desc_sw128(q_s, kColBlockBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t aoff = ((kk >> 2) * kColBlockBytes + (kk & 3) * 32) >> 4;
              mma_ss(tmem + kColDK, ad + aoff, bd + ((kk * 2048) >> 4), idesc_pv,
                     (acc || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(&sm.qdo_empty[st]);
          {
            // dQ = dS K: A = dS MN-major (M = query rows), B = K MN-major
            const uint64_t ad = smem_desc_sw128(ds_s, kColBlockBytes, 1024);
            const uint64_t bd = smem_desc_sw128(k_s, kColBlockBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + kColDP, ad + ((kk * 2048) >> 4), bd + ((kk * 2048) >> 4), idesc_dq,
                     kk > 0 ? 1u : 0u);
          }
          mma_commit(&sm.dq_full);
          if (n + 1 < it.steps) {
            const uint32_t stn = (qc + 1) & 1;
            if (!mbar_wait(&sm.qdo_full[stn], ((qc + 1) >> 1) & 1, abort_flag, hdr)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_kk(tmem + kColS, k_s, smem_u32(sm.q[stn]), false);
          }
          ++qc;
        }
        if (!ok) break;
        mma_commit(&sm.dkv_full);
        mma_commit(&sm.kv_empty);
        ++items_done;
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + epilogues
    const int wg = warp >> 2;                 // 0: query columns / head dims 0-63; 1: 64-127
    const int wq = warp & 3;
    const int r = wq * 32 + lane;             // TMEM lane: key row (S^T, dV, dK) or query row (dQ)
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float sl2 = p.scale * kLog2e;
    const uint32_t ds_row = smem_u32(sm.ds) + wg * kColBlockBytes + r * 128;
    uint32_t it_count = 0, items_done = 0, qc = 0;
    bool ok = true;
    while (ok) {
      const uint32_t slot = it_count & 1;
      if (!mbar_wait(&sm.item_full[slot], (it_count >> 1) & 1, abort_flag, hdr)) break;
      const BwdItem it = sm.items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.item_empty[slot]);
      ++it_count;
      if (it.steps < 0) break;
      // this thread's key and the query interval [qlo, qhi) that sees it
      const int64_t key = (int64_t)it.ktile * BK + r;
      int64_t qlo = 0, qhi = 0;
      if (key < T) {
        const int b = doc_of(p.cu, p.ndoc, key);
        qlo = p.causal ? key : (int64_t)__ldg(p.cu + b);
        qhi = (int64_t)__ldg(p.cu + b + 1);
      }
      for (int n = 0; n < it.steps && ok; ++n) {
        const int h = it.g * G + n / it.n_q;
        const int64_t q0 = (int64_t)(it.i_lo + n % it.n_q) * BQ;
        const uint32_t st = qc & 1;
        // the stage's lse2 / delta rows arrive with its Q and dOut tiles
        if (!mbar_wait(&sm.qdo_full[st], (qc >> 1) & 1, abort_flag, hdr)) { ok = false; break; }
        const float* lse2s = sm.lse2[st];
        const float* deltas = sm.delta[st];
        if (!mbar_wait(&sm.s_full, qc & 1, abort_flag, hdr)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col0 = wg * 64 + c * 32;
          uint32_t s[32], dp[32];
          tmem_ld32(tmem + lane_base + kColS + col0, s);
          tmem_ld32(tmem + lane_base + kColDP + col0, dp);
          tmem_wait_ld();
          const int64_t qg0 = q0 + col0;
          // visible query columns of this key, clipped to the chunk: [loc, hic)
          const int loc = (int)min(max(qlo - qg0, (int64_t)0), (int64_t)32);
          const int hic = (int)min(max(qhi - qg0, (int64_t)0), (int64_t)32);
          const uint32_t span = (uint32_t)(hic - loc);
          const bool full_w = __all_sync(0xffffffffu, qlo <= qg0 && qg0 + 32 <= qhi);
          uint32_t pk[16], dk[16];
          if (full_w) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int cc = col0 + 2 * e;
              const float p0 = ex2(fmaf(__uint_as_float(s[2 * e]), sl2, -lse2s[cc]));
              const float p1 = ex2(fmaf(__uint_as_float(s[2 * e + 1]), sl2, -lse2s[cc + 1]));
              pk[e] = pack_bf16x2(p0, p1);
              dk[e] = pack_bf16x2(p0 * (__uint_as_float(dp[2 * e]) - deltas[cc]),
                                  p1 * (__uint_as_float(dp[2 * e + 1]) - deltas[cc + 1]));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int cc = col0 + 2 * e;
              const bool v0 = (uint32_t)(2 * e - loc) < span;
              const bool v1 = (uint32_t)(2 * e + 1 - loc) < span;
              const float x0 = fmaf(__uint_as_float(s[2 * e]), sl2, -lse2s[cc]);
              const float x1 = fmaf(__uint_as_float(s[2 * e + 1]), sl2, -lse2s[cc + 1]);
              const float p0 = ex2(v0 ? x0 : -INFINITY);
              const float p1 = ex2(v1 ? x1 : -INFINITY);
              const float d0 = v0 ? __uint_as_float(dp[2 * e]) - deltas[cc] : 0.f;
              const float d1 = v1 ? __uint_as_float(dp[2 * e + 1]) - deltas[cc + 1] : 0.f;
              pk[e] = pack_bf16x2(p0, p1);
              dk[e] = pack_bf16x2(p0 * d0, p1 * d1);
            }
          }
          tmem_st16(tmem + lane_base + kColS + wg * 64 + c * 16, pk);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int chunk = c * 4 + u;                     // 8 query columns per 16 bytes
            st_shared_v4(ds_row + ((chunk ^ (r & 7)) << 4), dk[4 * u], dk[4 * u + 1],
                         dk[4 * u + 2], dk[4 * u + 3]);
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.ds_full);
        // dQ rows of this step: TMEM lane = query row, my half of the head dimension
        if (!mbar_wait(&sm.dq_full, qc & 1, abort_flag, hdr)) { ok = false; break; }
        tc_fence_after();
        {
          const int64_t qrow = q0 + r;
          float* dst = a.dq_acc + (qrow * p.Hq + h) * HD + wg * 64;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kColDP + wg * 64 + c * 32, v);
            tmem_wait_ld();
            if (qrow < T) {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                red_add_v4(dst + c * 32 + 4 * u, __uint_as_float(v[4 * u]) * p.scale,
                           __uint_as_float(v[4 * u + 1]) * p.scale,
                           __uint_as_float(v[4 * u + 2]) * p.scale,
                           __uint_as_float(v[4 * u + 3]) * p.scale);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.dq_empty);
        ++qc;
      }
      if (!ok) break;
      // item epilogue: dV (warps 0-3) and dK (warps 4-7), TMEM lane = key row
      if (!mbar_wait(&sm.dkv_full, items_done & 1, abort_flag, hdr)) break;
      tc_fence_after();
      {
        const uint32_t col = wg == 0 ? kColDV : kColDK;
        const float sc = wg == 0 ? 1.f : p.scale;
        __nv_bfloat16* dst = (wg == 0 ? a.dv : a.dk) + (key * p.Hkv + it.g) * HD;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + col + c * 32, v);
          tmem_wait_ld();
          if (key < T) store_row32<__nv_bfloat16>(dst + c * 32, v, sc);
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.dkv_empty);
      ++items_done;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * 2)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const AttnProblem& p, const void* out, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv,
                               const BwdWsLayout& L, char* ws, cudaStream_t s, bool* launched) {
  *launched = false;
  if (p.io_dtype != NSP_BF16 || p.d != HD || p.q_len <= 0) return cudaSuccess;
  const int64_t T = p.q_len;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map(&mq, p.q, T, (int64_t)p.Hq * HD) || !make_map(&mdo, dout, T, (int64_t)p.Hq * HD) ||
      !make_map(&mk, p.k, T, (int64_t)p.Hkv * HD) || !make_map(&mv, p.v, T, (int64_t)p.Hkv * HD))
    return cudaSuccess;
  *launched = true;
  float* delta = reinterpret_cast<float*>(ws + L.delta);
  float* lse2 = reinterpret_cast<float*>(ws + L.lse2);
  float* dq_acc = reinterpret_cast<float*>(ws + L.dq_acc);
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)T * p.Hq * HD, s);
  if (e != cudaSuccess) return e;
  e = launch_bwd_delta(out, dout, lse, delta, lse2, T, L.Tp, p.Hq, HD, p.io_dtype, p.hdr, s);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  BwdArgs a;
  a.p = p;
  a.lse2 = lse2;
  a.delta = delta;
  a.Tp = L.Tp;
  a.dq_acc = dq_acc;
  a.dk = reinterpret_cast<__nv_bfloat16*>(dk);
  a.dv = reinterpret_cast<__nv_bfloat16*>(dv);
  a.ktiles = reinterpret_cast<const int2*>(ws + L.ktiles);
  a.korder = reinterpret_cast<const int*>(ws + L.korder);
  attn_bwd_tc_kernel<<<num_sms(), kThreads, kSmemBytes, s>>>(mq, mk, mv, mdo, a);
  count_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_dq_convert(dq_acc, dq, T * p.Hq * HD, p.io_dtype, p.hdr, s);
}

}  // namespace nsp
