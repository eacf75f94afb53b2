// Varlen tile scheduler: from cu_seqlens (device) build, for every 128-row
// query tile, the contiguous range of 128-key tiles it must visit, and the
// order in which persistent CTAs should take the tiles (most KV tiles first,
// longest-processing-time order).  Fully masked KV tiles are never listed.
//
// The block patterns come from HSAP ("Sequence-aware Parallelism", Sec. 3.2,
// "Partition attention computation blocks"): for a causally masked packed
// sequence, a (query block, key block) pair is either empty, causal
// (diagonal), a full cross block, or a block cut by a document edge.  Here
// the "empty" blocks are dropped at schedule time and the cut blocks are
// masked per row inside the attention kernels.  Balancing by block count
// mirrors SAP's regional load balancing (same section) on one GPU.
//
// Mode 0 (forward / backward dQ view): tile i covers query rows
//   [q_start + 128 i, ...) and lists the key sub-tiles j (keys
//   [kv_start + gran j, ...), gran = 128) its rows see.
// Mode 1 (backward dK/dV view): tile j covers keys [kv_start + 128 j, ...)
//   and lists the query sub-tiles (rows [q_start + gran i, ...)) whose rows
//   can see any of those keys.
// A tile that sees nothing of the other range gets the empty list
// (first = 0, last = -1): it happens only for ring blocks, never for the
// whole stream (every key and query sees itself).
//
// One block of 1024 threads; the first mode-0 launch of a call validates
// cu_seqlens and resets the workspace status word.  The counting-sort
// histogram lives in shared memory when it fits (it almost always does), and
// the descending-cost scan is a warp-shuffle scan: the kernel is a handful of
// block barriers long.
#include "nsp_internal.cuh"

namespace nsp {
namespace {

constexpr int kSchedThreads = 1024;
constexpr int kSmemBuckets = 12 * 1024;    // 48 KB of counting-sort buckets in shared memory

struct SchedArgs {
  const int32_t* cu;
  int32_t ndoc;
  int64_t q_start, q_len, kv_start, kv_len;
  int32_t causal;
  int32_t mode;        // 0: query tiles list KV tiles; 1: key tiles list query tiles
  int32_t validate;
  int2* tiles;
  int32_t* order;
  int32_t* hist;       // n_buckets ints
  int32_t n_tiles;     // tiles to schedule
  int32_t n_buckets;   // max cost + 1 (cost = number of listed tiles)
  int32_t gran;        // granularity (rows or keys) of the listed tiles
  int32_t tile_rows;   // mode 0: rows of a scheduled query tile (128 or 256)
  WsHeader* hdr;
  int32_t second;      // write counters into counter2 / n_items2
  // the blocks whose tiles are listed: mode 0 tile i belongs to the block
  // with the largest tile0 <= i, mode 1 tile i (use_blocks) to the block
  // with the largest ktile0 <= i (the range fields above are then unused)
  FwdBlocks blks;
  int32_t use_blocks;  // mode 1: take the key tiles of blks instead of the range fields
  // mode 0 of a whole-stream backward with a dS cache: per query tile, the
  // first of its dS slots (an exclusive prefix sum of the listed counts, in
  // tile order); the header records whether Hq heads' slots fit the cache
  int64_t* qoff;
  int64_t ds_cache_bytes;
  int32_t Hq;
};

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const __grid_constant__ SchedArgs a) {
  extern __shared__ int s_hist_dyn[];       // n_buckets ints when they fit
  __shared__ int s_bad;
  __shared__ int s_max;
  __shared__ int s_warp[kSchedThreads / 32];
  __shared__ long long s_warp64[kSchedThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int* const hist = a.n_buckets <= kSmemBuckets ? s_hist_dyn : a.hist;
  grid_dep_trigger();                       // the attention kernel may launch (it waits)
  if (tid == 0) { s_bad = 0; s_max = 0; }
  __syncthreads();

  if (a.validate) {
    if (tid == 0) {
      if (a.ndoc < 1 || a.cu[0] != 0) s_bad = 1;
      const int64_t total = a.cu[a.ndoc];
      if (a.mode == 0 || a.use_blocks) {
        for (int bi = 0; bi < a.blks.n; ++bi) {
          const FwdBlock& B = a.blks.b[bi];
          if (total < (int64_t)B.q_start + B.q_len || total < (int64_t)B.kv_start + B.kv_len)
            s_bad = 1;
        }
      } else if (total < a.q_start + a.q_len || total < a.kv_start + a.kv_len) {
        s_bad = 1;
      }
    }
    for (int i = tid; i < a.ndoc; i += kSchedThreads)
      if (a.cu[i] > a.cu[i + 1]) s_bad = 1;
    __syncthreads();
    if (s_bad) {
      if (tid == 0) {
        a.hdr->status = NSP_ERR_INVALID;
        a.hdr->n_items = 0; a.hdr->counter = 0;
        a.hdr->n_items2 = 0; a.hdr->counter2 = 0;
        a.hdr->max_cost = 0; a.hdr->n_nonempty = 0;
        a.hdr->ds_on = 0; a.hdr->ds_pairs = 0;
      }
      return;
    }
    if (tid == 0) a.hdr->status = NSP_OK;
  } else if (status_bad(a.hdr)) {
    if (tid == 0) { a.hdr->n_items2 = 0; a.hdr->counter2 = 0; }
    return;
  }

  for (int i = tid; i < a.n_buckets; i += kSchedThreads) hist[i] = 0;
  __syncthreads();

  const int64_t q_end = a.q_start + a.q_len, kv_end = a.kv_start + a.kv_len;
  for (int i = tid; i < a.n_tiles; i += kSchedThreads) {
    int lo_t = 0, hi_t = -1;
    if (a.mode == 0) {
      // the block of tile i: the largest index whose tile0 <= i (blocks
      // without tiles share tile0 with the next one)
      int bl = 0, bh = a.blks.n - 1;
      while (bl < bh) {
        const int mid = (bl + bh + 1) >> 1;
        if (a.blks.b[mid].tile0 <= i) bl = mid; else bh = mid - 1;
      }
      const FwdBlock& B = a.blks.b[bl];
      const int64_t ks = B.kv_start, ke = (int64_t)B.kv_start + B.kv_len;
      const int64_t r0 = (int64_t)B.q_start + (int64_t)(i - B.tile0) * a.tile_rows;
      const int64_t r1 = min(r0 + a.tile_rows, (int64_t)B.q_start + B.q_len) - 1;  // last row
      const int b0 = doc_of(a.cu, a.ndoc, r0), b1 = doc_of(a.cu, a.ndoc, r1);
      const int64_t lo = max((int64_t)a.cu[b0], ks);
      const int64_t hi = min(a.causal ? r1 + 1 : (int64_t)a.cu[b1 + 1], ke);  // exclusive
      if (hi > lo) {
        lo_t = (int)((lo - ks) / a.gran);
        hi_t = (int)((hi - 1 - ks) / a.gran);
      }
    } else {
      int64_t ks = a.kv_start, ke = kv_end, qs = a.q_start, qe = q_end, k0 = a.kv_start;
      if (a.use_blocks) {
        int bl = 0, bh = a.blks.n - 1;
        while (bl < bh) {
          const int mid = (bl + bh + 1) >> 1;
          if (a.blks.b[mid].ktile0 <= i) bl = mid; else bh = mid - 1;
        }
        const FwdBlock& B = a.blks.b[bl];
        ks = B.kv_start; ke = (int64_t)B.kv_start + B.kv_len;
        qs = B.q_start; qe = (int64_t)B.q_start + B.q_len;
        k0 = ks + (int64_t)(i - B.ktile0) * kTileN;
      } else {
        k0 = a.kv_start + (int64_t)i * kTileN;
      }
      const int64_t k1 = min(k0 + kTileN, ke) - 1;               // last key of the tile
      const int b0 = doc_of(a.cu, a.ndoc, k0), b1 = doc_of(a.cu, a.ndoc, k1);
      const int64_t lo = max(a.causal ? k0 : (int64_t)a.cu[b0], qs);
      const int64_t hi = min((int64_t)a.cu[b1 + 1], qe);         // exclusive
      if (hi > lo) {
        lo_t = (int)((lo - qs) / a.gran);
        hi_t = (int)((hi - 1 - qs) / a.gran);
      }
    }
    a.tiles[i] = make_int2(lo_t, hi_t);
    const int cost = hi_t - lo_t + 1;
    atomicAdd(&hist[cost], 1);
    atomicMax(&s_max, cost);
  }
  __syncthreads();

  if (a.mode == 0 && !a.second) {
    // dS slots: thread t owns a contiguous run of tiles; block-wide scan of
    // the runs' listed counts
    const int per_t = (a.n_tiles + kSchedThreads - 1) / kSchedThreads;
    const int t_begin = min(tid * per_t, a.n_tiles), t_end = min(t_begin + per_t, a.n_tiles);
    long long cnt = 0;
    for (int i = t_begin; i < t_end; ++i) cnt += a.tiles[i].y - a.tiles[i].x + 1;
    long long xs = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, xs, o);
      if (lane >= o) xs += y;
    }
    if (lane == 31) s_warp64[wid] = xs;
    __syncthreads();
    if (wid == 0) {
      long long w = s_warp64[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_warp64[lane] = w;
    }
    __syncthreads();
    if (a.qoff != nullptr) {
      long long run = xs - cnt + (wid > 0 ? s_warp64[wid - 1] : 0);
      for (int i = t_begin; i < t_end; ++i) {
        a.qoff[i] = run;
        run += a.tiles[i].y - a.tiles[i].x + 1;
      }
    }
    if (tid == 0) {
      const long long pairs = s_warp64[kSchedThreads / 32 - 1];
      const long long cap = a.qoff != nullptr && a.Hq > 0
                                ? a.ds_cache_bytes / ((long long)a.Hq * (long long)kDsTileBytes)
                                : -1;
      a.hdr->ds_pairs = pairs;
      a.hdr->ds_on = pairs <= cap ? 1 : 0;
    }
  }

  // Exclusive scan in descending cost order: start[c] = sum_{c' > c} hist[c'].
  // Thread t owns a contiguous run of reversed bucket indices.
  const int per = (a.n_buckets + kSchedThreads - 1) / kSchedThreads;
  const int r_begin = tid * per, r_end = min(r_begin + per, a.n_buckets);
  int local = 0;
  for (int r = r_begin; r < r_end; ++r) local += hist[a.n_buckets - 1 - r];
  // block-wide inclusive scan of `local`: within warps, then over warp totals
  int x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  int run = x - local + (wid > 0 ? s_warp[wid - 1] : 0);   // exclusive prefix of my run
  for (int r = r_begin; r < r_end; ++r) {
    const int c = a.n_buckets - 1 - r;
    const int h = hist[c];
    hist[c] = run;
    run += h;
  }
  __syncthreads();
  // the empty tiles (cost 0) come last: hist[0] is where they start
  if (tid == 0 && !a.second) a.hdr->n_nonempty = hist[0];

  for (int i = tid; i < a.n_tiles; i += kSchedThreads) {
    const int2 t = a.tiles[i];
    const int pos = atomicAdd(&hist[t.y - t.x + 1], 1);
    a.order[pos] = i;
  }
  if (tid == 0) {
    if (a.second) { a.hdr->counter2 = 0; a.hdr->n_items2 = a.n_tiles; }
    else { a.hdr->counter = 0; a.hdr->n_items = a.n_tiles; a.hdr->max_cost = s_max; }
  }
}

size_t sched_smem(const SchedArgs& a) {
  return a.n_buckets <= kSmemBuckets ? sizeof(int) * (size_t)a.n_buckets : 0;
}

}  // namespace

FwdBlocks single_block(const AttnProblem& p) {
  FwdBlocks B;
  B.n = 1;
  B.global_rows = 0;
  B.b[0].q_start = (int32_t)p.q_start; B.b[0].q_len = (int32_t)p.q_len;
  B.b[0].kv_start = (int32_t)p.kv_start; B.b[0].kv_len = (int32_t)p.kv_len;
  B.b[0].tile0 = 0; B.b[0].ktile0 = 0;
  B.b[0].out = p.out; B.b[0].lse = p.lse;
  return B;
}

cudaError_t launch_fwd_schedule(const AttnProblem& p, const FwdWsLayout& L, char* ws,
                                cudaStream_t s, const FwdBlocks* blocks) {
  SchedArgs a;
  a.blks = blocks ? *blocks : single_block(p);
  a.use_blocks = 0;
  a.gran = kTileN;
  a.tile_rows = L.tile_rows;
  a.cu = p.cu; a.ndoc = p.ndoc;
  a.q_start = p.q_start; a.q_len = p.q_len; a.kv_start = p.kv_start; a.kv_len = p.kv_len;
  a.causal = p.causal; a.mode = 0; a.validate = 1;
  a.tiles = reinterpret_cast<int2*>(ws + L.tiles);
  a.order = reinterpret_cast<int32_t*>(ws + L.order);
  a.hist = reinterpret_cast<int32_t*>(ws + L.hist);
  a.n_tiles = (int32_t)L.n_qtiles;
  a.n_buckets = (int32_t)L.n_kvtiles + 2;
  a.hdr = p.hdr; a.second = 0;
  a.qoff = nullptr; a.ds_cache_bytes = 0; a.Hq = p.Hq;
  schedule_kernel<<<1, kSchedThreads, sched_smem(a), s>>>(a); count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_bwd_schedules(const AttnProblem& p, const BwdWsLayout& L, char* ws,
                                 cudaStream_t s, const FwdBlocks* blocks) {
  // query tiles of 128 rows listing 128-key tiles (validates cu_seqlens)
  SchedArgs a;
  a.cu = p.cu; a.ndoc = p.ndoc;
  a.q_start = p.q_start; a.q_len = p.q_len; a.kv_start = p.kv_start; a.kv_len = p.kv_len;
  a.causal = p.causal; a.mode = 0; a.validate = 1; a.gran = kBwdSub; a.tile_rows = kTileM;
  a.blks = blocks ? *blocks : single_block(p);
  a.use_blocks = 0;
  a.tiles = reinterpret_cast<int2*>(ws + L.qtiles);
  a.order = reinterpret_cast<int32_t*>(ws + L.qorder);
  a.hist = reinterpret_cast<int32_t*>(ws + L.qhist);
  a.n_tiles = (int32_t)L.n_qtiles;
  a.n_buckets = (int32_t)L.n_qhist;
  a.hdr = p.hdr; a.second = 0;
  // the dS cache serves the whole-stream backward and the batched blocks (not
  // a single accumulated ring block)
  const bool cache = (blocks != nullptr || !p.accumulate) && L.ds_cache_bytes > 0;
  a.qoff = cache ? reinterpret_cast<int64_t*>(ws + L.qoff) : nullptr;
  a.ds_cache_bytes = cache ? (int64_t)L.ds_cache_bytes : 0;
  a.Hq = p.Hq;
  schedule_kernel<<<1, kSchedThreads, sched_smem(a), s>>>(a); count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // key tiles of 128 keys listing 128-row query tiles
  a.mode = 1; a.validate = 0; a.use_blocks = blocks != nullptr;
  a.tiles = reinterpret_cast<int2*>(ws + L.ktiles);
  a.order = reinterpret_cast<int32_t*>(ws + L.korder);
  a.hist = reinterpret_cast<int32_t*>(ws + L.khist);
  a.n_tiles = (int32_t)L.n_ktiles;
  a.n_buckets = (int32_t)L.n_khist;
  a.hdr = p.hdr; a.second = 1;
  schedule_kernel<<<1, kSchedThreads, sched_smem(a), s>>>(a); count_launches(1);
  return cudaGetLastError();
}

}  // namespace nsp
