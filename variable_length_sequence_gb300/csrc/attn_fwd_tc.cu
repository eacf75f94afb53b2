// Varlen attention forward on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA loads), bf16 inputs, float32 accumulation, head
// dimension 128 or 64.
//
// What it computes is the definition of the CUDA-core path (scaled
// dot-product attention inside each packed document, BASP Sec. II-A, HSAP
// Sec. 2.1 cu_len; optionally a ring partial block, HSAP Sec. 2.2.1), with
// the blockwise online softmax (Milakov and Gimelshein, cited by HSAP
// Sec. 2.2.1) so no score matrix is ever stored.
//
// Work decomposition.  The schedule kernel lists, per 128-row query tile
// (aligned to the start of the query range), the contiguous range of
// 128-key tiles its rows may see, and orders the query tiles by that count,
// longest first.  A work item is (query tile, pair of query heads of one
// KV group): both heads read the same K/V tiles, so every K/V tile loaded
// into shared memory feeds two 128x128x128 QK^T and two PV products.  With
// an odd number of query heads per KV head (multi-head attention among
// them) a work item is instead (two adjacent 128-row query tiles, one
// head): the scheduler lists 256-row tiles, whose key range is the union of
// its two halves', and the two halves take the two softmax roles (a half
// whose rows cannot see a key tile gets P = 0 there).  A persistent grid of
// one CTA per SM takes items from an atomic counter.
//
// CTA roles (384 threads, three warpgroups):
//   warps 0-3  softmax for head h0 (TMEM lanes 0-127, one query row each)
//   warps 4-7  softmax for head h0+1
//   warp 8     TMA producer and work fetch
//   warp 9     TMEM allocation and the single MMA-issuing thread
//   warps 10-11 idle (they complete the control warpgroup)
// Registers: launched at 168 per thread (384 x 168 = 64512); inside its role
// branch the control warpgroup gives back to 112 and each softmax warpgroup
// grows to 192 (256 x 192 + 128 x 112 = 63488), enough to hold a whole
// 128-column S row so S is read from TMEM once per tile.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512);
// P (bf16, two per 32-bit cell) is written over the first 64 columns of S
// and read from TMEM by the PV product.  The tensor core alternates
// between the two heads, so one head's softmax overlaps the other head's
// MMAs.  The running output is rescaled only when a row's maximum grows
// by more than 2^8 (the result is exact either way: numerator and
// denominator share the same reference maximum).
//
// Masking: every query row sees one contiguous key interval [lo, hi) (its
// document's start up to itself, clipped to the key range), so a KV tile
// is either fully visible to a row or masked per column by two compares;
// tiles no row can see are never scheduled.
//
// Ring accumulation (p.accumulate, float32 out): the row's running output
// and lse enter the online softmax as one more term (O preloaded at the
// item's start, m = running lse, l = 1), so the plain epilogue writes the
// merged result.  Head groups (p.q_groups = P > 1): q and out are
// [P][q_len][Hq/P][d]; the Q map is [P q_len, (Hq/P) d] and a head's tile
// sits at row block (h / (Hq/P)) q_len, column block h % (Hq/P).
#include <cudaTypedefs.h>

#include <type_traits>

#include "tc_ptx.cuh"

namespace nsp {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 128, HD = 128;
constexpr int NSTAGE = 2;
constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 192, kRegsControl = 112;
constexpr int kWarpProducer = 8, kWarpMma = 9;
constexpr uint32_t kColBlockBytes = 128 * 64 * 2;        // 128 rows x 64 bf16 (one swizzle span)
constexpr uint32_t kTileBytes = 2 * kColBlockBytes;      // 128 x 128 bf16
// TMEM columns of S (and P) and O for the two query heads of an item.
__host__ __device__ constexpr uint32_t col_s(int t) { return t == 0 ? 0u : 128u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return t == 0 ? 256u : 384u; }
constexpr float kRescaleThreshold = 8.0f;                 // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Item {
  int qtile;      // scheduled query tile (-1: none): 128 rows, or 256 with paired tiles
  int h0;         // first of the two query heads (paired tiles: the one head)
  int g;          // key/value head
  int j_lo;       // first KV tile
  int n_kv;       // number of KV tiles (0: no key visible; -1: stop)
  int blk;        // block of the call (batched forward; 0 otherwise)
  int pad[2];
};

// Block of scheduled tile t: the largest index whose tile0 <= t (a block
// without tiles shares tile0 with the next one).
__device__ __forceinline__ int block_of(const FwdBlocks& B, int t) {
  int lo = 0, hi = B.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (B.b[mid].tile0 <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct __align__(1024) Smem {
  uint8_t q[2][kTileBytes];
  uint8_t k[NSTAGE][kTileBytes];
  uint8_t v[NSTAGE][kTileBytes];
  uint64_t q_full, q_empty;
  uint64_t k_full[NSTAGE], k_empty[NSTAGE], v_full[NSTAGE], v_empty[NSTAGE];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t item_full[2], item_empty[2];
  Item items[2];
  uint64_t mma_drain_bar;
  uint32_t tmem_base;
  WaitCtl wait;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;      // + alignment slack

// S = Q K^T: D / 16 MMAs of K = 16 over the head dimension D.  Both operands
// are K-major with 128-byte swizzle; stepping K by 16 elements moves the
// start address by 32 bytes inside a swizzle span, and the second 64-wide
// half of the head dimension (D = 128) lives in the next 16 KB column block.  The start
// address field holds address >> 4 and never carries (shared memory <
// 256 KB), so descriptors are advanced by adding offset >> 4.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_saddr, uint32_t k_saddr) {
  constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false);
  const uint64_t qd = smem_desc_sw128(q_saddr, 16, 1024);
  const uint64_t kd = smem_desc_sw128(k_saddr, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kColBlockBytes + (kk & 3) * 32) >> 4;
    mma_ss(d_tmem, qd + off, kd + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V: P (bf16) from TMEM, 8 columns per K = 16 keys; V is MN-major
// (keys are K, the head dimension is N = D): 16 keys = two 8-row groups
// (SBO = 1024 B), the two 64-wide halves of N (D = 128) are one column block
// apart (LBO = 16 KB).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_saddr,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(BM, D, true);
  const uint64_t vd = smem_desc_sw128(v_saddr, kColBlockBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    mma_ts(d_tmem, p_tmem + kk * 8, vd + ((kk * 2048) >> 4), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

// Store 32 consecutive output elements of one row (raw float32 bits in v),
// 32 bytes per instruction and lane (whole sectors); dst is 32-byte aligned
// (rows are 256 or 512 bytes, chunks 64 or 128).
template <typename TO>
__device__ __forceinline__ void store_row_chunk(TO* dst, const uint32_t (&v)[32], float scale);

template <>
__device__ __forceinline__ void store_row_chunk<__nv_bfloat16>(__nv_bfloat16* dst,
                                                               const uint32_t (&v)[32],
                                                               float scale) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    w[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * scale, __uint_as_float(v[2 * i + 1]) * scale);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    st_global_v8(dst + 16 * i, w[8 * i], w[8 * i + 1], w[8 * i + 2], w[8 * i + 3], w[8 * i + 4],
                 w[8 * i + 5], w[8 * i + 6], w[8 * i + 7]);
}

template <>
__device__ __forceinline__ void store_row_chunk<float>(float* dst, const uint32_t (&v)[32],
                                                       float scale) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__uint_as_float(v[8 * i + k]) * scale);
    st_global_v8(dst + 8 * i, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
  }
}

// PAIR: an item is two adjacent tiles of one head (odd Hq / Hkv) instead of
// one tile and two heads.  MULTI: the batched call, ranges and outputs per
// block of the table and q / k / v rows addressed by global token ids;
// otherwise the single range and outputs of p.  ACC: ring accumulation in
// place (float32 out only).  All three are compile-time so the common cases
// (one range, head pairs, written output) carry none of the others'
// bookkeeping or registers.  D: the head dimension, 128 or 64 (Q, K, V
// tiles of 64 columns use the first column block of each tile buffer, and O
// the first 64 of its TMEM columns).
template <typename TO, bool PAIR, bool MULTI, bool ACC, int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnProblem p,
                       const int2* __restrict__ tiles, const int* __restrict__ order,
                       const __grid_constant__ FwdBlocks blks) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = p.hdr;
  grid_dep_wait();                          // the schedule kernel's lists and status
  if (status_bad(hdr)) return;

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], 128);
      mbar_init(&sm.o_full[t], 1);
      mbar_init(&sm.item_full[t], 1);
      mbar_init(&sm.item_empty[t], 1 + 8);
    }
    mbar_init(&sm.mma_drain_bar, 1);
    wait_ctl_init(&sm.wait, p.wait_budget);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = sm.tmem_base;
  WaitCtl* const wc = &sm.wait;
  const int G = p.Hq / p.Hkv;
  // odd G (multi-head attention among them): an item is two adjacent
  // 128-row tiles of one head instead of one tile and two heads
  constexpr bool pair_tiles = PAIR;
  const int per_tile = pair_tiles ? p.Hq : (p.Hq >> 1);         // items per scheduled tile
  constexpr int tile_rows = pair_tiles ? 2 * BM : BM;
  // query tiles no key of the range reaches are not work items: the softmax
  // warps zero-fill them up front (or, accumulating, leave them alone)
  const int n_items = hdr->n_nonempty * per_tile;
  constexpr int kBlocks = D / 64;                               // 64-column blocks of a row
  constexpr uint32_t kLoadBytes = kBlocks * kColBlockBytes;     // one Q, K or V tile

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it_count = 0, q_count = 0, kv_count = 0;
      bool ok = true;
      while (ok) {
        const int idx = atomicAdd(&hdr->counter, 1);
        Item it;
        it.qtile = -1; it.h0 = 0; it.g = 0; it.j_lo = 0; it.n_kv = -1; it.blk = 0;
        if (idx < n_items) {
          const int qt = order[idx / per_tile];
          const int sub = idx - (idx / per_tile) * per_tile;
          const int2 tr = tiles[qt];
          if constexpr (MULTI) {
            it.blk = block_of(blks, qt);
            it.qtile = qt - blks.b[it.blk].tile0;           // tile within its block
          } else {
            it.qtile = qt;
          }
          it.h0 = pair_tiles ? sub : 2 * sub;
          it.g = it.h0 / G;
          it.j_lo = tr.x;
          it.n_kv = tr.y - tr.x + 1;
        }
        const uint32_t slot = it_count & 1;
        if (it_count >= 2 &&
            !mbar_wait(&sm.item_empty[slot], ((it_count >> 1) - 1) & 1, wc, hdr)) {
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
        if (q_count >= 1 && !mbar_wait(&sm.q_empty, (q_count - 1) & 1, wc, hdr)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm.q_full, 2 * kLoadBytes);
        // packed layout: map [q_len, Hq d]; head groups: map [P q_len, (Hq/P) d],
        // head h at column block h % (Hq/P) of rows (h / (Hq/P)) q_len + row;
        // a batched call's maps span the whole stream (rows = global ids)
        const int q_row_base = MULTI ? blks.b[it.blk].q_start : 0;
        const int k_row_base = MULTI ? blks.b[it.blk].kv_start : 0;
        const int q_len_b = MULTI ? blks.b[it.blk].q_len : (int)p.q_len;
        const int hpg = p.Hq / p.q_groups;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          // role t: head h0 + t of the tile, or (paired tiles) half t of the
          // 256-row tile for head h0 (a half past the range reads rows that
          // are never stored)
          const int head = pair_tiles ? it.h0 : it.h0 + t;
          const int grp = head / hpg;
          const int row0 = q_row_base + grp * q_len_b + it.qtile * tile_rows +
                           (pair_tiles ? t * BM : 0);
#pragma unroll
          for (int cb = 0; cb < kBlocks; ++cb)
            tma_load_2d(sm.q[t] + cb * kColBlockBytes, &tm_q, &sm.q_full,
                        (head - grp * hpg) * D + cb * 64, row0);
        }
        ++q_count;
        for (int jj = 0; jj < it.n_kv; ++jj) {
          const uint32_t st = kv_count % NSTAGE, use = kv_count / NSTAGE;
          const int key0 = k_row_base + (it.j_lo + jj) * BN;
          if (use >= 1 && !mbar_wait(&sm.k_empty[st], (use - 1) & 1, wc, hdr)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.k_full[st], kLoadBytes);
#pragma unroll
          for (int cb = 0; cb < kBlocks; ++cb)
            tma_load_2d(sm.k[st] + cb * kColBlockBytes, &tm_k, &sm.k_full[st], it.g * D + cb * 64,
                        key0);
          if (use >= 1 && !mbar_wait(&sm.v_empty[st], (use - 1) & 1, wc, hdr)) {
            // the K copy just issued is in flight: drain it before leaving
            drain_wait(&sm.k_full[st], use & 1);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.v_full[st], kLoadBytes);
#pragma unroll
          for (int cb = 0; cb < kBlocks; ++cb)
            tma_load_2d(sm.v[st] + cb * kColBlockBytes, &tm_v, &sm.v_full[st], it.g * D + cb * 64,
                        key0);
          ++kv_count;
        }
      }
      {
        // Leaving, normally or on an abort: wait (bounded) for every copy still
        // in flight to land (after a normal end these phases completed long ago).
        if (q_count >= 1) drain_wait(&sm.q_full, (q_count - 1) & 1);
        for (uint32_t s = 0; s < NSTAGE && s < kv_count; ++s) {
          const uint32_t last = kv_count - 1 - ((kv_count - 1 - s) % NSTAGE);
          drain_wait(&sm.k_full[last % NSTAGE], (last / NSTAGE) & 1);
          drain_wait(&sm.v_full[last % NSTAGE], (last / NSTAGE) & 1);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it_count = 0, q_count = 0, kv_count = 0;
      uint32_t p_count[2] = {0, 0};
      const uint32_t q_saddr[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
      while (true) {
        const uint32_t slot = it_count & 1;
        if (!mbar_wait(&sm.item_full[slot], (it_count >> 1) & 1, wc, hdr)) break;
        const Item it = sm.items[slot];
        mbar_arrive(&sm.item_empty[slot]);
        ++it_count;
        if (it.n_kv < 0) break;
        if (it.n_kv == 0) continue;
        if (!mbar_wait(&sm.q_full, q_count & 1, wc, hdr)) break;
        ++q_count;
        bool ok = true;
        {
          const uint32_t st = kv_count % NSTAGE, use = kv_count / NSTAGE;
          if (!mbar_wait(&sm.k_full[st], use & 1, wc, hdr)) break;
          tc_fence_after();
          const uint32_t ks = smem_u32(sm.k[st]);
          issue_qk<D>(tmem + col_s(0), q_saddr[0], ks);
          mma_commit(&sm.s_full[0]);
          issue_qk<D>(tmem + col_s(1), q_saddr[1], ks);
          mma_commit(&sm.s_full[1]);
          mma_commit(&sm.k_empty[st]);
          if (it.n_kv == 1) mma_commit(&sm.q_empty);
        }
        for (int jj = 0; jj < it.n_kv && ok; ++jj) {
          const uint32_t st = (kv_count + jj) % NSTAGE, use = (kv_count + jj) / NSTAGE;
          const bool has_next = jj + 1 < it.n_kv;
          const uint32_t stn = (kv_count + jj + 1) % NSTAGE, usen = (kv_count + jj + 1) / NSTAGE;
          if (!mbar_wait(&sm.v_full[st], use & 1, wc, hdr)) { ok = false; break; }
          const uint32_t vs = smem_u32(sm.v[st]);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok) continue;
            if (!mbar_wait(&sm.p_full[t], p_count[t] & 1, wc, hdr)) { ok = false; continue; }
            ++p_count[t];
            tc_fence_after();
            // a ring accumulation's O starts as the preloaded running output
            issue_pv<D>(tmem + col_o(t), tmem + col_s(t), vs, jj > 0 || ACC);
            if (t == 1) mma_commit(&sm.v_empty[st]);
            if (!has_next) {
              mma_commit(&sm.o_full[t]);
              continue;
            }
            if (t == 0) {
              if (!mbar_wait(&sm.k_full[stn], usen & 1, wc, hdr)) { ok = false; continue; }
              tc_fence_after();
            }
            issue_qk<D>(tmem + col_s(t), q_saddr[t], smem_u32(sm.k[stn]));
            mma_commit(&sm.s_full[t]);
            if (t == 1) {
              mma_commit(&sm.k_empty[stn]);
              if (jj + 2 == it.n_kv) mma_commit(&sm.q_empty);
            }
          }
        }
        if (!ok) break;
        kv_count += it.n_kv;
      }
      mma_drain(&sm.mma_drain_bar);        // every product done before TMEM is freed
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + col_s(t);
    const uint32_t o_tm = tmem + lane_base + col_o(t);
    const float sl2 = p.scale * kLog2e;
    uint32_t it_count = 0, s_count = 0, o_count = 0;
    if (!ACC) {
      // Query tiles that see no key of the range (listed last by the
      // schedule): out = 0 and lse = -inf, written by the softmax warps of
      // every CTA in a grid-stride loop over (tile, head, 32-row group), one
      // whole row per 16-byte lane group, before the first work item.
      const int n_empty = hdr->n_items - hdr->n_nonempty;
      const int groups = tile_rows / 32;                        // 32-row groups per tile
      const int64_t units = (int64_t)n_empty * p.Hq * groups;
      constexpr int kLanesPerRow = D * (int)sizeof(TO) / 16;    // 32, 16 or 8
      constexpr int kRowsPerPass = 32 / kLanesPerRow;
      const int sub = lane / kLanesPerRow, part = lane % kLanesPerRow;
      for (int64_t u = (int64_t)blockIdx.x * 8 + warp; u < units; u += (int64_t)gridDim.x * 8) {
        const int e = (int)(u / (p.Hq * groups));
        const int rem = (int)(u - (int64_t)e * p.Hq * groups);
        const int hz = rem / groups;
        const int tile = order[hdr->n_nonempty + e];
        const int bz = MULTI ? block_of(blks, tile) : 0;
        TO* const out = reinterpret_cast<TO*>(MULTI ? blks.b[bz].out : p.out);
        float* const lse_z = MULTI ? blks.b[bz].lse : p.lse;
        const int64_t q_len_z = MULTI ? (int64_t)blks.b[bz].q_len : p.q_len;
        const int64_t r0 = (int64_t)(tile - (MULTI ? blks.b[bz].tile0 : 0)) * tile_rows +
                           (rem % groups) * 32;
#pragma unroll 4
        for (int rr = 0; rr < 32; rr += kRowsPerPass) {
          const int64_t grow = r0 + rr + sub;
          if (grow < q_len_z)
            reinterpret_cast<uint4*>(out + qo_offset(p, grow, hz))[part] = make_uint4(0, 0, 0, 0);
        }
        if (lse_z != nullptr && r0 + lane < q_len_z)
          lse_z[(int64_t)hz * q_len_z + r0 + lane] = -INFINITY;
      }
    }
    while (true) {
      const uint32_t slot = it_count & 1;
      if (!mbar_wait_warp(&sm.item_full[slot], (it_count >> 1) & 1, wc, hdr)) break;
      const Item it = sm.items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.item_empty[slot]);
      ++it_count;
      if (it.n_kv < 0) break;
      // the item's ranges (global ids) and outputs: its block's (batched
      // call) or the call's, read where they are used (kernel parameters,
      // so no register holds them across the tile loop)
      // (a batched call copies its block's entry once per item; a single
      // range reads the kernel parameter p at each use)
      FwdBlock mb{};
      if constexpr (MULTI) mb = blks.b[it.blk];
#define NSP_BLK(field, whole) (MULTI ? (int64_t)mb.field : (int64_t)p.whole)
#define NSP_OUT (reinterpret_cast<TO*>(MULTI ? mb.out : p.out))
#define NSP_LSE (MULTI ? mb.lse : p.lse)
      const int h = pair_tiles ? it.h0 : it.h0 + t;
      // first row of this role's 128-row tile, query-range relative
      const int64_t tile_base = (int64_t)it.qtile * tile_rows + (pair_tiles ? t * BM : 0);
      const int64_t row = tile_base + r;
      const bool valid = row < NSP_BLK(q_len, q_len);
      int lo = 0, hi = 0;                                      // key-range relative [lo, hi)
      if (valid) {
        const int64_t kv_start = NSP_BLK(kv_start, kv_start);
        const int64_t kv_end = kv_start + NSP_BLK(kv_len, kv_len);
        const int64_t tg = NSP_BLK(q_start, q_start) + row;
        const int b = doc_of(p.cu, p.ndoc, tg);
        const int64_t glo = max((int64_t)__ldg(p.cu + b), kv_start);
        const int64_t ghi = min(p.causal ? tg + 1 : (int64_t)__ldg(p.cu + b + 1), kv_end);
        lo = (int)(glo - kv_start);
        hi = (int)max(ghi - kv_start, glo - kv_start);
      }
      float m = -INFINITY, l = 0.f;
      // Ring accumulation: a row that sees a key of this block (acc_row)
      // enters the online softmax with its running result as one more
      // weighted term: O starts as the running output acc, with weight 1 at
      // the reference maximum m = lse_acc (log2 units), so at the end O / l
      // and m + log2 l are the merged output and lse (the rescaling of O and
      // l as the maximum grows covers acc too).  The preload runs while the
      // item's first S is computed; the block's first P V then accumulates
      // onto it.  Every other row starts from O = 0 and is not written.
      const bool acc_row = ACC && valid && hi > lo;
      if constexpr (sizeof(TO) == 4) {
        if (ACC && it.n_kv > 0) {
          float la2 = -INFINITY;
          if (acc_row) la2 = NSP_LSE[(int64_t)h * NSP_BLK(q_len, q_len) + row] * kLog2e;
          const float4* arow = reinterpret_cast<const float4*>(NSP_OUT + qo_offset(p, row, h));
          {
            // the whole row (4 D bytes) in flight at once (one DRAM round
            // trip; S's registers are not live yet)
            uint32_t v[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c)
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 x = la2 != -INFINITY ? __ldcg(arow + c * 8 + i)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                v[c][4 * i] = __float_as_uint(x.x);
                v[c][4 * i + 1] = __float_as_uint(x.y);
                v[c][4 * i + 2] = __float_as_uint(x.z);
                v[c][4 * i + 3] = __float_as_uint(x.w);
              }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_st32(o_tm + c * 32, v[c]);
          }
          tmem_wait_st();              // before a first-tile rescale reads O back
          if (la2 != -INFINITY) {
            m = la2;
            l = 1.f;
          }
        }
      }
      bool ok = true;
      for (int jj = 0; jj < it.n_kv; ++jj) {
        if (!mbar_wait_warp(&sm.s_full[t], s_count & 1, wc, hdr)) { ok = false; break; }
        ++s_count;
        tc_fence_after();
        const int key0 = (it.j_lo + jj) * BN;
        // visible columns are [a, b): one unsigned compare per column; a
        // warp whose rows all see the whole tile skips the mask entirely
        const int a = lo - key0;
        const uint32_t span = (uint32_t)(hi - lo);
        const bool full_w = __all_sync(0xffffffffu, lo <= key0 && key0 + BN <= hi);
        // S row -> registers (one TMEM round trip); masked columns -> -inf
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_tm + c * 32, sr[c]);
        tmem_wait_ld();
        if (!full_w) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if ((uint32_t)(c * 32 + i - a) >= span) sr[c][i] = 0xff800000u;   // -inf
        }
        // row maximum: 8 independent chains, then a small tree
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          mx[u] = fmaxf(__uint_as_float(sr[0][u]), __uint_as_float(sr[0][u + 8]));
#pragma unroll
        for (int u = 0; u < 8; ++u)
          mx[u] = fmaxf(mx[u], fmaxf(__uint_as_float(sr[0][u + 16]), __uint_as_float(sr[0][u + 24])));
#pragma unroll
        for (int c = 1; c < 4; ++c)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            mx[u] = fmaxf(fmaxf(mx[u], fmaxf(__uint_as_float(sr[c][u]), __uint_as_float(sr[c][u + 8]))),
                          fmaxf(__uint_as_float(sr[c][u + 16]), __uint_as_float(sr[c][u + 24])));
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_new = fmaxf(m, mt * sl2);
        // the running output is rescaled only when the maximum grew a lot
        const bool need = (m != -INFINITY) && (m_new > m + kRescaleThreshold);
        const float corr = need ? ex2(m - m_new) : 1.f;
        if (need || m == -INFINITY) m = m_new;
        const float mb = (m == -INFINITY) ? 0.f : m;
        // p = 2^(s * scale * log2 e - m) from registers, bf16 P over S, row sum
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = ex2(fmaf(__uint_as_float(sr[c][2 * i]), sl2, -mb));
            const float p1 = ex2(fmaf(__uint_as_float(sr[c][2 * i + 1]), sl2, -mb));
            ls[i & 3] += p0 + p1;
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(s_tm + c * 16, pk);
        }
        l = l * corr + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orow[32];
            tmem_ld32(o_tm + c * 32, orow);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * corr);
            tmem_st32(o_tm + c * 32, orow);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm.p_full[t]);
      }
      if (!ok) break;
      // ---- epilogue: out = O / l, lse = (m + log2 l) ln 2
      const float inv = l > 0.f ? 1.f / l : 0.f;
      TO* dst = NSP_OUT + qo_offset(p, row, h);
      if (it.n_kv > 0) {
        if (!mbar_wait_warp(&sm.o_full[t], o_count & 1, wc, hdr)) break;
        ++o_count;
        tc_fence_after();
        if constexpr (sizeof(TO) == 4) {
          // float32 rows: read O as 16-lane fragments so that the four lanes
          // of a row write 32 contiguous bytes and consecutive stores of a
          // warp continue the same 8 rows; thread t holds rows 8 i + t/4 of
          // the warp's 32 (i = 0..3)
          // (ring accumulation: rows that saw no key of the block keep their
          // running output, so they are skipped)
          const float wp = (ACC && !acc_row) ? 0.f : inv;
          float wpr[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) wpr[i] = __shfl_sync(0xffffffffu, wp, 8 * i + (lane >> 2));
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t x[32];
            tmem_ld16x256_x4(o_tm + c * 32, x);
            tmem_ld16x256_x4(o_tm + (16u << 16) + c * 32, x + 16);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int i = 2 * (k >> 3) + (k & 1);
              const int64_t grow = tile_base + wq * 32 + 8 * i + (lane >> 2);
              if (grow < NSP_BLK(q_len, q_len) && (!ACC || wpr[i] != 0.f))
                *reinterpret_cast<float2*>(NSP_OUT + qo_offset(p, grow, h) + c * 32 +
                                           8 * ((k >> 1) & 3) + 2 * (lane & 3)) =
                    make_float2(__uint_as_float(x[2 * k]) * wpr[i],
                                __uint_as_float(x[2 * k + 1]) * wpr[i]);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orow[32];
            tmem_ld32(o_tm + c * 32, orow);
            tmem_wait_ld();
            if (valid) store_row_chunk<TO>(dst + c * 32, orow, inv);
          }
        }
      } else if (!ACC) {
        // no key of the range is visible to any row of the tile: zero rows,
        // each written whole by a warp (16-byte lanes, full sectors)
        constexpr int kLanesPerRow = D * (int)sizeof(TO) / 16;    // 32, 16 or 8
        constexpr int kRowsPerPass = 32 / kLanesPerRow;
        const int sub = lane / kLanesPerRow, part = lane % kLanesPerRow;
#pragma unroll 4
        for (int rr = 0; rr < 32; rr += kRowsPerPass) {
          const int64_t grow = tile_base + wq * 32 + rr + sub;
          if (grow < NSP_BLK(q_len, q_len))
            reinterpret_cast<uint4*>(NSP_OUT + qo_offset(p, grow, h))[part] = make_uint4(0, 0, 0, 0);
        }
      }
      if (valid && NSP_LSE != nullptr && (!ACC || acc_row))
        NSP_LSE[(int64_t)h * NSP_BLK(q_len, q_len) + row] =
            l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
#undef NSP_BLK
#undef NSP_OUT
#undef NSP_LSE
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
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

// [rows, cols] bf16 row-major, box = 64 columns x 128 rows, 128-byte swizzle.
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

template <typename TO, bool PAIR, bool MULTI, bool ACC, int D>
cudaError_t launch_typed(const AttnProblem& p, const FwdWsLayout& L, char* ws, cudaStream_t s,
                         const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const FwdBlocks& B) {
  auto kern = attn_fwd_tc_kernel<TO, PAIR, MULTI, ACC, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid();
  e = launch_dependent(kern, dim3(grid), dim3(kThreads), kSmemBytes, s, mq, mk, mv, p,
                       reinterpret_cast<const int2*>(ws + L.tiles),
                       reinterpret_cast<const int*>(ws + L.order), B);
  count_launches(1);
  count_path(true);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Every variant of one head dimension D.
template <int D>
cudaError_t launch_d(const AttnProblem& pk, const FwdWsLayout& L, char* ws, cudaStream_t s,
                     const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     const FwdBlocks& B, bool batched) {
  const bool pair = ((pk.Hq / pk.Hkv) & 1) != 0;
  const bool acc = pk.accumulate != 0;                // (float32 out only)
  // batched blocks: float32 partials or accumulators
  auto f32 = [&](auto pair_c, auto multi_c) {
    constexpr bool P = decltype(pair_c)::value, M = decltype(multi_c)::value;
    return acc ? launch_typed<float, P, M, true, D>(pk, L, ws, s, mq, mk, mv, B)
               : launch_typed<float, P, M, false, D>(pk, L, ws, s, mq, mk, mv, B);
  };
  using T_ = std::true_type;
  using F_ = std::false_type;
  if (batched) return pair ? f32(T_{}, T_{}) : f32(F_{}, T_{});
  if (pk.out_dtype == NSP_F32) return pair ? f32(T_{}, F_{}) : f32(F_{}, F_{});
  return pair ? launch_typed<__nv_bfloat16, true, false, false, D>(pk, L, ws, s, mq, mk, mv, B)
              : launch_typed<__nv_bfloat16, false, false, false, D>(pk, L, ws, s, mq, mk, mv, B);
}

}  // namespace

cudaError_t launch_attn_fwd_tc(const AttnProblem& p, const FwdWsLayout& L, char* ws,
                               cudaStream_t s, bool* launched, const FwdBlocks* blocks) {
  *launched = false;
  if (p.io_dtype != NSP_BF16 || (p.d != 128 && p.d != 64)) return cudaSuccess;
  if (p.q_len <= 0 || p.kv_len <= 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.q_len * p.q_groups, (int64_t)(p.Hq / p.q_groups) * p.d) ||
      !make_map(&mk, p.k, p.kv_len, (int64_t)p.Hkv * p.d) ||
      !make_map(&mv, p.v, p.kv_len, (int64_t)p.Hkv * p.d))
    return cudaSuccess;                       // no tensor-map support: CUDA-core path
  *launched = true;
  AttnProblem pk = p;
  pk.wait_budget = wait_budget_cycles();
  const FwdBlocks B = blocks ? *blocks : single_block(p);
  return p.d == 128 ? launch_d<128>(pk, L, ws, s, mq, mk, mv, B, blocks != nullptr)
                    : launch_d<64>(pk, L, ws, s, mq, mk, mv, B, blocks != nullptr);
}

}  // namespace nsp
