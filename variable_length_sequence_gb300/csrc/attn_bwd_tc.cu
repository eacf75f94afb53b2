// Varlen attention backward on the tcgen05 tensor cores, bf16 inputs,
// float32 accumulation, d = 128: two persistent kernels, no atomics.
//
// Gradients of L = sum(dOut * out) for document-masked attention (BASP
// Sec. II-A, HSAP Sec. 2.1), recomputing the probabilities from the saved
// lse instead of storing them (the recomputation NSP Sec. 2.3 discusses):
//   P = exp(scale Q K^T - lse),  dP = dOut V^T,  dS = P (dP - delta),
//   dV = P^T dOut,  dK = scale dS^T Q,  dQ = scale dS K,
// with delta = rowsum(dOut * out) and lse * log2(e) prepared by
// bwd_delta_kernel in padded [Hq, Tp] rows.
//
// dK/dV kernel (key-stationary).  Work item: one 128-key tile of one KV
// head.  It walks every 64-row query sub-tile that can see the keys, for
// the query heads of the group taken two at a time; the two heads are two
// chains that ping-pong on the tensor core (one chain's softmax overlaps
// the other chain's MMAs) and accumulate into the same dV and dK in TMEM:
//   S^T  = K Q^T      (M = 128 keys, N = 64 queries)   TMEM [128X, 128X+64)
//   dP^T = V dOut^T                                     TMEM [128X+64, 128X+128)
//   P^T and dS^T (bf16) are written back over S^T and dP^T by the softmax
//   dV  += P^T dOut   (A = P^T from TMEM, B = dOut MN-major)   TMEM [256, 384)
//   dK  += dS^T Q     (A = dS^T from TMEM, B = Q MN-major)     TMEM [384, 512)
// dK and dV are written once per item, in bf16.
//
// dQ kernel (query-stationary, the shape of the forward).  Work item: one
// 128-row query tile for a pair of query heads of one KV group; it walks the
// 64-key sub-tiles the rows can see; the two heads ping-pong:
//   S  = Q K^T        (M = 128 queries, N = 64 keys)   TMEM [256X, 256X+64)
//   dP = dOut V^T                                       TMEM [256X+64, 256X+128)
//   dS (bf16) is written back over S
//   dQ += dS K        (A = dS from TMEM, B = K MN-major)   TMEM [256X+128, 256X+256)
// dQ is scaled and written once per item, in bf16.
//
// Roles (320 threads): warps 0-3 run chain / head 0, warps 4-7 chain / head
// 1 (one TMEM lane each), warp 8 is the TMA producer and work fetcher, warp
// 9 allocates TMEM and one of its threads issues every MMA.  Masking is one
// unsigned compare per element against the row's (or key's) visible
// interval, skipped for fully visible chunks.  All waits are bounded.
#include <cudaTypedefs.h>

#include "tc_ptx.cuh"

namespace nsp {
namespace {

using namespace tc;

constexpr int HD = 128;
constexpr int SUB = kBwdSub;                          // 64
constexpr int kThreads = 320;
constexpr int kWarpProducer = 8, kWarpMma = 9;
constexpr uint32_t kBlk128 = 128 * 64 * 2;            // 128 rows x 64 bf16 column block
constexpr uint32_t kBlk64 = 64 * 64 * 2;              // 64 rows x 64 bf16 column block
constexpr uint32_t kTile128 = 2 * kBlk128;            // 128 x 128 bf16
constexpr uint32_t kTile64 = 2 * kBlk64;              // 64 x 128 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr size_t kSmemLimit = 232448;

// ---------------------------------------------------------------- MMA helpers

// D = A B^T, A and B K-major (128-byte swizzle), K = 128 (head dim).
// a_blk / b_blk: byte distance between the two 64-wide column blocks.
__device__ __forceinline__ void mma_k128(uint32_t d_tmem, uint32_t a_saddr, uint32_t a_blk,
                                         uint32_t b_saddr, uint32_t b_blk, uint32_t idesc) {
  const uint64_t ad = smem_desc_sw128(a_saddr, 16, 1024);
  const uint64_t bd = smem_desc_sw128(b_saddr, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t ao = ((kk >> 2) * a_blk + (kk & 3) * 32) >> 4;
    const uint32_t bo = ((kk >> 2) * b_blk + (kk & 3) * 32) >> 4;
    mma_ss(d_tmem, ad + ao, bd + bo, idesc, kk > 0 ? 1u : 0u);
  }
}

// D (+)= A[tmem] B, K = 64 (4 steps of 16, 8 TMEM columns each); B is
// MN-major with K along its rows (16 rows = 2048 B per step) and its two
// 64-wide N blocks b_blk bytes apart.
__device__ __forceinline__ void mma_tk64(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_saddr,
                                         uint32_t b_blk, uint32_t idesc, bool accumulate) {
  const uint64_t bd = smem_desc_sw128(b_saddr, b_blk, 1024);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts(d_tmem, a_tmem + kk * 8, bd + ((kk * 2048) >> 4), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles) return;
  }
}

__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32],
                                                 float scale) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    w[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * scale, __uint_as_float(v[2 * i + 1]) * scale);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// 1024-aligned view of dynamic shared memory, or nullptr (error recorded)
// when the aligned structure would not fit in the launch's allocation.
template <typename S>
__device__ __forceinline__ S* smem_view(uint8_t* raw, WsHeader* hdr) {
  uint32_t dyn_bytes;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
  const uint32_t base = smem_u32(raw);
  if (((base + 1023u) & ~1023u) - base + sizeof(S) > dyn_bytes) {
    if (threadIdx.x == 0) atomicExch(&hdr->status, (int)NSP_ERR_UNSUPPORTED);
    return nullptr;
  }
  return reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                              ~static_cast<uintptr_t>(1023));
}

template <typename S>
constexpr size_t smem_bytes() {
  return sizeof(S) + 1024 <= kSmemLimit ? sizeof(S) + 1024 : kSmemLimit;
}

struct BwdArgs {
  AttnProblem p;
  const float* lse2;      // [Hq, Tp] lse * log2(e)
  const float* delta;     // [Hq, Tp]
  int64_t Tp;
  __nv_bfloat16* dq;      // [T, Hq, d]
  __nv_bfloat16* dk;      // [T, Hkv, d]
  __nv_bfloat16* dv;
  const int2* qtiles;     // per 128-row query tile: first/last 64-key sub-tile
  const int* qorder;
  const int2* ktiles;     // per 128-key tile: first/last 64-row query sub-tile
  const int* korder;
};

// ================================================================ dK / dV

constexpr int KV_NS = 2;

struct KvItem {
  int ktile, g, i_lo, n_q, steps, pad[3];   // steps = (G / 2) * n_q; -1 stops
};

struct __align__(1024) SmemKV {
  uint8_t k[kTile128];
  uint8_t v[kTile128];
  uint8_t q[2][KV_NS][kTile64];
  uint8_t dout[2][KV_NS][kTile64];
  float lse2[2][KV_NS][SUB];
  float delta[2][KV_NS][SUB];
  uint64_t kv_full, kv_empty;
  uint64_t qdo_full[2][KV_NS], qdo_empty[2][KV_NS];
  uint64_t s_full[2], p_full[2];
  uint64_t dkv_full, dkv_empty;
  uint64_t item_full[2], item_empty[2];
  KvItem items[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SmemKV) <= kSmemLimit, "dK/dV tile set exceeds shared memory");

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q64,
                            const __grid_constant__ CUtensorMap tm_do64,
                            const __grid_constant__ CUtensorMap tm_k128,
                            const __grid_constant__ CUtensorMap tm_v128, const BwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const AttnProblem& p = a.p;
  WsHeader* hdr = p.hdr;
  if (status_bad(hdr)) return;
  SmemKV* smp = smem_view<SmemKV>(smem_raw, hdr);
  if (smp == nullptr) return;
  SmemKV& sm = *smp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int x = 0; x < 2; ++x) {
      for (int s = 0; s < KV_NS; ++s) {
        mbar_init(&sm.qdo_full[x][s], 1);
        mbar_init(&sm.qdo_empty[x][s], 1);
      }
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.p_full[x], 128);
      mbar_init(&sm.item_full[x], 1);
      mbar_init(&sm.item_empty[x], 1 + 8);
    }
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
    tma_prefetch_desc(&tm_q64);
    tma_prefetch_desc(&tm_do64);
    tma_prefetch_desc(&tm_k128);
    tma_prefetch_desc(&tm_v128);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  const int G = p.Hq / p.Hkv;
  const int npair = G >> 1;
  const int64_t T = p.q_len;
  const int n_items = hdr->n_items2 * p.Hkv;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it_count = 0, kv_count = 0, qc = 0;
      bool ok = true;
      while (ok) {
        const int idx = atomicAdd(&hdr->counter2, 1);
        KvItem it;
        it.ktile = 0; it.g = 0; it.i_lo = 0; it.n_q = 0; it.steps = -1;
        if (idx < n_items) {
          const int kt = a.korder[idx / p.Hkv];
          const int2 tr = a.ktiles[kt];
          it.ktile = kt;
          it.g = idx - (idx / p.Hkv) * p.Hkv;
          it.i_lo = tr.x;
          it.n_q = tr.y - tr.x + 1;
          it.steps = npair * it.n_q;
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
        mbar_arrive_expect_tx(&sm.kv_full, 2 * kTile128);
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          tma_load_2d(sm.k + cb * kBlk128, &tm_k128, &sm.kv_full, it.g * HD + cb * 64,
                      it.ktile * 128);
          tma_load_2d(sm.v + cb * kBlk128, &tm_v128, &sm.kv_full, it.g * HD + cb * 64,
                      it.ktile * 128);
        }
        ++kv_count;
        for (int n = 0; n < it.steps && ok; ++n) {
          const int pair = n / it.n_q;
          const int i = it.i_lo + (n - pair * it.n_q);
          const uint32_t st = qc % KV_NS, use = qc / KV_NS;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok) continue;
            const int h = it.g * G + 2 * pair + x;
            if (use >= 1 &&
                !mbar_wait(&sm.qdo_empty[x][st], (use - 1) & 1, abort_flag, hdr)) {
              ok = false;
              continue;
            }
            mbar_arrive_expect_tx(&sm.qdo_full[x][st], 2 * kTile64 + 2 * SUB * sizeof(float));
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
              tma_load_2d(sm.q[x][st] + cb * kBlk64, &tm_q64, &sm.qdo_full[x][st],
                          h * HD + cb * 64, i * SUB);
              tma_load_2d(sm.dout[x][st] + cb * kBlk64, &tm_do64, &sm.qdo_full[x][st],
                          h * HD + cb * 64, i * SUB);
            }
            const int64_t row = (int64_t)h * a.Tp + (int64_t)i * SUB;
            bulk_load(sm.lse2[x][st], a.lse2 + row, SUB * sizeof(float), &sm.qdo_full[x][st]);
            bulk_load(sm.delta[x][st], a.delta + row, SUB * sizeof(float), &sm.qdo_full[x][st]);
          }
          if (ok) ++qc;
        }
      }
      if (!ok) {
        // abort: every copy issued so far completes on its stage barrier
        if (kv_count >= 1) drain_wait(&sm.kv_full, (kv_count - 1) & 1);
        for (uint32_t j = (qc > KV_NS ? qc - KV_NS : 0); j <= qc; ++j)
          for (int x = 0; x < 2; ++x) drain_wait(&sm.qdo_full[x][j % KV_NS], (j / KV_NS) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, SUB, false, false);   // S^T, dP^T
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, HD, true, false);   // dV, dK
      const uint32_t k_s = smem_u32(sm.k), v_s = smem_u32(sm.v);
      uint32_t it_count = 0, items_done = 0, qc = 0;
      uint32_t pc[2] = {0, 0};
      bool ok = true;
      while (ok) {
        const uint32_t slot = it_count & 1;
        if (!mbar_wait(&sm.item_full[slot], (it_count >> 1) & 1, abort_flag, hdr)) break;
        const KvItem it = sm.items[slot];
        mbar_arrive(&sm.item_empty[slot]);
        ++it_count;
        if (it.steps < 0) break;
        if (!mbar_wait(&sm.kv_full, items_done & 1, abort_flag, hdr)) break;
        for (int n = 0; n < it.steps && ok; ++n) {
          const uint32_t st = qc % KV_NS;
          if (n == 0) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (!ok) continue;
              if (!mbar_wait(&sm.qdo_full[x][st], (qc / KV_NS) & 1, abort_flag, hdr)) {
                ok = false;
                continue;
              }
              tc_fence_after();
              mma_k128(tmem + 128 * x, k_s, kBlk128, smem_u32(sm.q[x][st]), kBlk64, idesc_s);
              mma_k128(tmem + 128 * x + 64, v_s, kBlk128, smem_u32(sm.dout[x][st]), kBlk64,
                       idesc_s);
              mma_commit(&sm.s_full[x]);
            }
            if (!ok) break;
          }
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok) continue;
            if (!mbar_wait(&sm.p_full[x], pc[x] & 1, abort_flag, hdr)) { ok = false; continue; }
            ++pc[x];
            const bool first = (n == 0 && x == 0);
            if (first && items_done > 0 &&
                !mbar_wait(&sm.dkv_empty, (items_done - 1) & 1, abort_flag, hdr)) {
              ok = false;
              continue;
            }
            tc_fence_after();
            mma_tk64(tmem + 256, tmem + 128 * x, smem_u32(sm.dout[x][st]), kBlk64, idesc_acc,
                     !first);
            mma_tk64(tmem + 384, tmem + 128 * x + 64, smem_u32(sm.q[x][st]), kBlk64, idesc_acc,
                     !first);
            mma_commit(&sm.qdo_empty[x][st]);
            if (n + 1 < it.steps) {
              const uint32_t stn = (qc + 1) % KV_NS;
              if (!mbar_wait(&sm.qdo_full[x][stn], ((qc + 1) / KV_NS) & 1, abort_flag, hdr)) {
                ok = false;
                continue;
              }
              tc_fence_after();
              mma_k128(tmem + 128 * x, k_s, kBlk128, smem_u32(sm.q[x][stn]), kBlk64, idesc_s);
              mma_k128(tmem + 128 * x + 64, v_s, kBlk128, smem_u32(sm.dout[x][stn]), kBlk64,
                       idesc_s);
              mma_commit(&sm.s_full[x]);
            }
          }
          if (ok) ++qc;
        }
        if (!ok) break;
        mma_commit(&sm.dkv_full);
        mma_commit(&sm.kv_empty);
        ++items_done;
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + dK/dV epilogue
    const int x = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;                          // TMEM lane = key row
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + 128 * x;
    const uint32_t dp_tm = s_tm + 64;
    const float sl2 = p.scale * kLog2e;
    uint32_t it_count = 0, items_done = 0, qc = 0, sc = 0;
    bool ok = true;
    while (ok) {
      const uint32_t slot = it_count & 1;
      if (!mbar_wait(&sm.item_full[slot], (it_count >> 1) & 1, abort_flag, hdr)) break;
      const KvItem it = sm.items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.item_empty[slot]);
      ++it_count;
      if (it.steps < 0) break;
      const int64_t key = (int64_t)it.ktile * 128 + r;
      int64_t qlo = 0, qhi = 0;                             // queries that see this key
      if (key < T) {
        const int b = doc_of(p.cu, p.ndoc, key);
        qlo = p.causal ? key : (int64_t)__ldg(p.cu + b);
        qhi = (int64_t)__ldg(p.cu + b + 1);
      }
      for (int n = 0; n < it.steps && ok; ++n) {
        const int pair = n / it.n_q;
        const int64_t q0 = (int64_t)(it.i_lo + (n - pair * it.n_q)) * SUB;
        const uint32_t st = qc % KV_NS;
        if (!mbar_wait(&sm.qdo_full[x][st], (qc / KV_NS) & 1, abort_flag, hdr)) { ok = false; break; }
        if (!mbar_wait(&sm.s_full[x], sc & 1, abort_flag, hdr)) { ok = false; break; }
        ++sc;
        tc_fence_after();
        const float* lse2s = sm.lse2[x][st];
        const float* deltas = sm.delta[x][st];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t s[32], dp[32];
          tmem_ld32(s_tm + c * 32, s);
          tmem_ld32(dp_tm + c * 32, dp);
          tmem_wait_ld();
          const int64_t qg0 = q0 + c * 32;
          const int loc = (int)min(max(qlo - qg0, (int64_t)0), (int64_t)32);
          const int hic = (int)min(max(qhi - qg0, (int64_t)0), (int64_t)32);
          const uint32_t span = (uint32_t)(hic - loc);
          const bool full_w = __all_sync(0xffffffffu, loc == 0 && hic == 32);
          uint32_t pk[16], dk[16];
          if (full_w) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int cc = c * 32 + 2 * e;
              const float p0 = ex2(fmaf(__uint_as_float(s[2 * e]), sl2, -lse2s[cc]));
              const float p1 = ex2(fmaf(__uint_as_float(s[2 * e + 1]), sl2, -lse2s[cc + 1]));
              pk[e] = pack_bf16x2(p0, p1);
              dk[e] = pack_bf16x2(p0 * (__uint_as_float(dp[2 * e]) - deltas[cc]),
                                  p1 * (__uint_as_float(dp[2 * e + 1]) - deltas[cc + 1]));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int cc = c * 32 + 2 * e;
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
          tmem_st16(s_tm + c * 16, pk);       // P^T over S^T (columns already read)
          tmem_st16(dp_tm + c * 16, dk);      // dS^T over dP^T
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm.p_full[x]);
        ++qc;
      }
      if (!ok) break;
      // item epilogue: dV (warps 0-3) and dK (warps 4-7), TMEM lane = key row
      if (!mbar_wait(&sm.dkv_full, items_done & 1, abort_flag, hdr)) break;
      tc_fence_after();
      {
        const uint32_t col = x == 0 ? 256u : 384u;
        const float scale = x == 0 ? 1.f : p.scale;
        __nv_bfloat16* dst = (x == 0 ? a.dv : a.dk) + (key * p.Hkv + it.g) * HD;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + col + c * 32, v);
          tmem_wait_ld();
          if (key < T) store_row32_bf16(dst + c * 32, v, scale);
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

// ================================================================ dQ

constexpr int Q_NS = 3;

struct QItem {
  int qtile, h0, g, j_lo, n_kv, pad[3];     // n_kv 64-key sub-tiles; -1 stops
};

struct __align__(1024) SmemQ {
  uint8_t q[2][kTile128];
  uint8_t dout[2][kTile128];
  uint8_t k[Q_NS][kTile64];
  uint8_t v[Q_NS][kTile64];
  uint64_t qdo_full, qdo_empty;
  uint64_t k_full[Q_NS], k_empty[Q_NS], v_full[Q_NS], v_empty[Q_NS];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t item_full[2], item_empty[2];
  QItem items[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SmemQ) <= kSmemLimit, "dQ tile set exceeds shared memory");

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q128,
                          const __grid_constant__ CUtensorMap tm_do128,
                          const __grid_constant__ CUtensorMap tm_k64,
                          const __grid_constant__ CUtensorMap tm_v64, const BwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const AttnProblem& p = a.p;
  WsHeader* hdr = p.hdr;
  if (status_bad(hdr)) return;
  SmemQ* smp = smem_view<SmemQ>(smem_raw, hdr);
  if (smp == nullptr) return;
  SmemQ& sm = *smp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&sm.qdo_full, 1);
    mbar_init(&sm.qdo_empty, 1);
    for (int s = 0; s < Q_NS; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.p_full[x], 128);
      mbar_init(&sm.o_full[x], 1);
      mbar_init(&sm.item_full[x], 1);
      mbar_init(&sm.item_empty[x], 1 + 8);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    tma_prefetch_desc(&tm_q128);
    tma_prefetch_desc(&tm_do128);
    tma_prefetch_desc(&tm_k64);
    tma_prefetch_desc(&tm_v64);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  const int n_pairs = p.Hq >> 1;
  const int G = p.Hq / p.Hkv;
  const int64_t T = p.q_len;
  const int n_items = hdr->n_items * n_pairs;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it_count = 0, q_count = 0, kv_count = 0;
      bool ok = true;
      while (ok) {
        const int idx = atomicAdd(&hdr->counter, 1);
        QItem it;
        it.qtile = 0; it.h0 = 0; it.g = 0; it.j_lo = 0; it.n_kv = -1;
        if (idx < n_items) {
          const int qt = a.qorder[idx / n_pairs];
          const int pair = idx - (idx / n_pairs) * n_pairs;
          const int2 tr = a.qtiles[qt];
          it.qtile = qt;
          it.h0 = 2 * pair;
          it.g = (2 * pair) / G;
          it.j_lo = tr.x;
          it.n_kv = tr.y - tr.x + 1;
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
        if (it.n_kv <= 0) {
          if (it.n_kv < 0) break;
          continue;
        }
        if (q_count >= 1 && !mbar_wait(&sm.qdo_empty, (q_count - 1) & 1, abort_flag, hdr)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm.qdo_full, 4 * kTile128);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) {
            tma_load_2d(sm.q[x] + cb * kBlk128, &tm_q128, &sm.qdo_full, (it.h0 + x) * HD + cb * 64,
                        it.qtile * 128);
            tma_load_2d(sm.dout[x] + cb * kBlk128, &tm_do128, &sm.qdo_full,
                        (it.h0 + x) * HD + cb * 64, it.qtile * 128);
          }
        ++q_count;
        for (int jj = 0; jj < it.n_kv; ++jj) {
          const uint32_t st = kv_count % Q_NS, use = kv_count / Q_NS;
          const int key0 = (it.j_lo + jj) * SUB;
          if (use >= 1 && !mbar_wait(&sm.k_empty[st], (use - 1) & 1, abort_flag, hdr)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.k_full[st], kTile64);
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
            tma_load_2d(sm.k[st] + cb * kBlk64, &tm_k64, &sm.k_full[st], it.g * HD + cb * 64, key0);
          if (use >= 1 && !mbar_wait(&sm.v_empty[st], (use - 1) & 1, abort_flag, hdr)) {
            drain_wait(&sm.k_full[st], use & 1);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.v_full[st], kTile64);
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
            tma_load_2d(sm.v[st] + cb * kBlk64, &tm_v64, &sm.v_full[st], it.g * HD + cb * 64, key0);
          ++kv_count;
        }
      }
      if (!ok) {
        if (q_count >= 1) drain_wait(&sm.qdo_full, (q_count - 1) & 1);
        for (uint32_t j = (kv_count > Q_NS ? kv_count - Q_NS : 0); j < kv_count; ++j) {
          drain_wait(&sm.k_full[j % Q_NS], (j / Q_NS) & 1);
          drain_wait(&sm.v_full[j % Q_NS], (j / Q_NS) & 1);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, SUB, false, false);   // S, dP
      constexpr uint32_t idesc_dq = idesc_bf16_f32(128, HD, true, false);    // dQ
      uint32_t it_count = 0, q_count = 0, kv_count = 0;
      uint32_t pc[2] = {0, 0};
      bool ok = true;
      while (ok) {
        const uint32_t slot = it_count & 1;
        if (!mbar_wait(&sm.item_full[slot], (it_count >> 1) & 1, abort_flag, hdr)) break;
        const QItem it = sm.items[slot];
        mbar_arrive(&sm.item_empty[slot]);
        ++it_count;
        if (it.n_kv < 0) break;
        if (it.n_kv == 0) continue;
        if (!mbar_wait(&sm.qdo_full, q_count & 1, abort_flag, hdr)) break;
        ++q_count;
        {
          const uint32_t st = kv_count % Q_NS, use = kv_count / Q_NS;
          if (!mbar_wait(&sm.k_full[st], use & 1, abort_flag, hdr)) break;
          if (!mbar_wait(&sm.v_full[st], use & 1, abort_flag, hdr)) break;
          tc_fence_after();
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            mma_k128(tmem + 256 * x, smem_u32(sm.q[x]), kBlk128, smem_u32(sm.k[st]), kBlk64,
                     idesc_s);
            mma_k128(tmem + 256 * x + 64, smem_u32(sm.dout[x]), kBlk128, smem_u32(sm.v[st]),
                     kBlk64, idesc_s);
            mma_commit(&sm.s_full[x]);
          }
          mma_commit(&sm.v_empty[st]);
          if (it.n_kv == 1) mma_commit(&sm.qdo_empty);
        }
        for (int jj = 0; jj < it.n_kv && ok; ++jj) {
          const uint32_t st = (kv_count + jj) % Q_NS;
          const bool has_next = jj + 1 < it.n_kv;
          const uint32_t stn = (kv_count + jj + 1) % Q_NS, usen = (kv_count + jj + 1) / Q_NS;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok) continue;
            if (!mbar_wait(&sm.p_full[x], pc[x] & 1, abort_flag, hdr)) { ok = false; continue; }
            ++pc[x];
            tc_fence_after();
            mma_tk64(tmem + 256 * x + 128, tmem + 256 * x, smem_u32(sm.k[st]), kBlk64, idesc_dq,
                     jj > 0);
            if (x == 1) mma_commit(&sm.k_empty[st]);
            if (!has_next) {
              mma_commit(&sm.o_full[x]);
              continue;
            }
            if (x == 0) {
              if (!mbar_wait(&sm.k_full[stn], usen & 1, abort_flag, hdr) ||
                  !mbar_wait(&sm.v_full[stn], usen & 1, abort_flag, hdr)) {
                ok = false;
                continue;
              }
              tc_fence_after();
            }
            mma_k128(tmem + 256 * x, smem_u32(sm.q[x]), kBlk128, smem_u32(sm.k[stn]), kBlk64,
                     idesc_s);
            mma_k128(tmem + 256 * x + 64, smem_u32(sm.dout[x]), kBlk128, smem_u32(sm.v[stn]),
                     kBlk64, idesc_s);
            mma_commit(&sm.s_full[x]);
            if (x == 1) {
              mma_commit(&sm.v_empty[stn]);
              if (jj + 2 == it.n_kv) mma_commit(&sm.qdo_empty);
            }
          }
        }
        if (!ok) break;
        kv_count += it.n_kv;
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + dQ epilogue
    const int x = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;                          // TMEM lane = query row
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + 256 * x;
    const uint32_t dp_tm = s_tm + 64;
    const uint32_t dq_tm = s_tm + 128;
    const float sl2 = p.scale * kLog2e;
    uint32_t it_count = 0, sc = 0, oc = 0;
    bool ok = true;
    while (ok) {
      const uint32_t slot = it_count & 1;
      if (!mbar_wait(&sm.item_full[slot], (it_count >> 1) & 1, abort_flag, hdr)) break;
      const QItem it = sm.items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.item_empty[slot]);
      ++it_count;
      if (it.n_kv < 0) break;
      const int h = it.h0 + x;
      const int64_t row = (int64_t)it.qtile * 128 + r;
      const bool valid = row < T;
      int lo = 0, hi = 0;                                    // visible keys [lo, hi)
      float lse2r = 0.f, deltar = 0.f;
      if (valid) {
        const int b = doc_of(p.cu, p.ndoc, row);
        lo = __ldg(p.cu + b);
        hi = p.causal ? (int)row + 1 : __ldg(p.cu + b + 1);
        lse2r = __ldg(a.lse2 + (int64_t)h * a.Tp + row);
        deltar = __ldg(a.delta + (int64_t)h * a.Tp + row);
      }
      for (int jj = 0; jj < it.n_kv && ok; ++jj) {
        if (!mbar_wait(&sm.s_full[x], sc & 1, abort_flag, hdr)) { ok = false; break; }
        ++sc;
        tc_fence_after();
        const int key0 = (it.j_lo + jj) * SUB;
        const int aa = lo - key0;
        const uint32_t span = (uint32_t)(hi - lo);
        const bool full_w = __all_sync(0xffffffffu, lo <= key0 && key0 + SUB <= hi);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t s[32], dp[32];
          tmem_ld32(s_tm + c * 32, s);
          tmem_ld32(dp_tm + c * 32, dp);
          tmem_wait_ld();
          uint32_t dk[16];
          if (full_w) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p0 = ex2(fmaf(__uint_as_float(s[2 * e]), sl2, -lse2r));
              const float p1 = ex2(fmaf(__uint_as_float(s[2 * e + 1]), sl2, -lse2r));
              dk[e] = pack_bf16x2(p0 * (__uint_as_float(dp[2 * e]) - deltar),
                                  p1 * (__uint_as_float(dp[2 * e + 1]) - deltar));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int col = c * 32 + 2 * e;
              const bool v0 = (uint32_t)(col - aa) < span;
              const bool v1 = (uint32_t)(col + 1 - aa) < span;
              const float p0 = ex2(v0 ? fmaf(__uint_as_float(s[2 * e]), sl2, -lse2r) : -INFINITY);
              const float p1 =
                  ex2(v1 ? fmaf(__uint_as_float(s[2 * e + 1]), sl2, -lse2r) : -INFINITY);
              const float d0 = v0 ? __uint_as_float(dp[2 * e]) - deltar : 0.f;
              const float d1 = v1 ? __uint_as_float(dp[2 * e + 1]) - deltar : 0.f;
              dk[e] = pack_bf16x2(p0 * d0, p1 * d1);
            }
          }
          tmem_st16(s_tm + c * 16, dk);       // dS over S (columns already read)
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm.p_full[x]);
      }
      if (!ok) break;
      // epilogue: dQ = scale * accumulated dS K, written once in bf16
      __nv_bfloat16* dst = a.dq + (row * p.Hq + h) * HD;
      if (it.n_kv > 0) {
        if (!mbar_wait(&sm.o_full[x], oc & 1, abort_flag, hdr)) break;
        ++oc;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(dq_tm + c * 32, v);
          tmem_wait_ld();
          if (valid) store_row32_bf16(dst + c * 32, v, p.scale);
        }
      } else if (valid) {
        uint32_t z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) store_row32_bf16(dst + c * 32, z, 0.f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================ host

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

// [rows, cols] bf16 row-major; box = 64 columns x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * 2)};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool bwd_tc_eligible(int32_t io_dtype, int32_t d, int32_t Hq, int32_t Hkv) {
  return io_dtype == NSP_BF16 && d == HD && Hkv > 0 && Hq % Hkv == 0 && (Hq / Hkv) % 2 == 0;
}

cudaError_t launch_attn_bwd_tc(const AttnProblem& p, const void* out, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv,
                               const BwdWsLayout& L, char* ws, cudaStream_t s) {
  const int64_t T = p.q_len;
  CUtensorMap mq128, mdo128, mk128, mv128, mq64, mdo64, mk64, mv64;
  const int64_t qc = (int64_t)p.Hq * HD, kc = (int64_t)p.Hkv * HD;
  if (!make_map(&mq128, p.q, T, qc, 128) || !make_map(&mdo128, dout, T, qc, 128) ||
      !make_map(&mk128, p.k, T, kc, 128) || !make_map(&mv128, p.v, T, kc, 128) ||
      !make_map(&mq64, p.q, T, qc, 64) || !make_map(&mdo64, dout, T, qc, 64) ||
      !make_map(&mk64, p.k, T, kc, 64) || !make_map(&mv64, p.v, T, kc, 64))
    return cudaErrorNotSupported;
  float* delta = reinterpret_cast<float*>(ws + L.delta);
  float* lse2 = reinterpret_cast<float*>(ws + L.lse2);
  cudaError_t e = launch_bwd_delta(out, dout, lse, delta, lse2, T, L.Tp, p.Hq, HD, p.io_dtype,
                                   p.hdr, s);
  if (e != cudaSuccess) return e;
  BwdArgs a;
  a.p = p;
  a.lse2 = lse2;
  a.delta = delta;
  a.Tp = L.Tp;
  a.dq = reinterpret_cast<__nv_bfloat16*>(dq);
  a.dk = reinterpret_cast<__nv_bfloat16*>(dk);
  a.dv = reinterpret_cast<__nv_bfloat16*>(dv);
  a.qtiles = reinterpret_cast<const int2*>(ws + L.qtiles);
  a.qorder = reinterpret_cast<const int*>(ws + L.qorder);
  a.ktiles = reinterpret_cast<const int2*>(ws + L.ktiles);
  a.korder = reinterpret_cast<const int*>(ws + L.korder);
  const int grid = num_sms();
  constexpr size_t kv_bytes = smem_bytes<SmemKV>();
  constexpr size_t q_bytes = smem_bytes<SmemQ>();
  e = cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kv_bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)q_bytes);
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_tc_kernel<<<grid, kThreads, kv_bytes, s>>>(mq64, mdo64, mk128, mv128, a);
  count_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_dq_tc_kernel<<<grid, kThreads, q_bytes, s>>>(mq128, mdo128, mk64, mv64, a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace nsp
