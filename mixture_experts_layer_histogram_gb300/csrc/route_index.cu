// Routing (top-k + renormalised softmax), token counting and index generation.
//   routing kernel : one thread per token, a sorted top-k list in registers (route_token).
//
// "Scalable Pretraining of Large MoE LMs on Aurora", brief, section 核心方法: FastSparseMoE counts
// the tokens of each expert and generates their indices with GPU kernels before the grouped GEMM.
// Here that is a stable counting sort of the T*k routing slots by expert id:
//   count kernel : warp-aggregated (match.any) shared-memory histograms, one global atomic per
//                  (block, expert); the last block to finish scans counts into offsets and tile offsets.
//   index kernel : every block ranks its chunk of slots stably (each warp counts its own 128
//                  consecutive slots per expert with match.any, then adds the earlier warps'), then
//                  finds, per expert, how many earlier slots went to that expert with a decoupled
//                  look-back over the preceding blocks (one 64-bit flag|value word per block and
//                  expert), and scatters row_of_slot / token_of_row.
//   route_count_index kernel : the routing, count and index kernels' work in one launch (each block
//                  routes the tokens of its slots, two lanes per token, ranks its slots and publishes
//                  its per-expert counts; the blocks meet once, when all have published, and then each
//                  block scans the totals and sums its predecessors' counts itself and scatters).
#include <math.h>

#include "common.cuh"

namespace moe {

constexpr int kRouteThreads = 128;               // tokens (threads) per routing block
constexpr int kIdxThreads = 256;                 // 8 warps
constexpr int kIdxItems = 4;                     // slots per thread
constexpr int kIdxChunk = kIdxThreads * kIdxItems;
// The fused routing kernel's blocks own kIdxThreads * ITEMS slots, ITEMS = 2 (twice the index
// kernel's blocks, so twice the SMs route) while that is at most one block per SM, else 4. Its
// per-block count table ([blocks][E] int32) lives in the index kernel's look-back words
// ([blocks][E] uint64 at kIdxChunk slots per block), which it fits for ITEMS >= kIdxItems / 2.

// look-back word: flag in the high 32 bits, value in the low 32 bits; a look-back reads this many
// predecessors' words per round
constexpr int kLookWindow = 8;
constexpr uint64_t kFlagAggregate = 1ull << 32;
constexpr uint64_t kFlagPrefix = 2ull << 32;

// ---------------------------------------------------------------------------------------------
// top-k routing: one thread per token. The thread reads its row of logits 64 at a time (16 vector
// loads issued before any is used, so one memory latency per 64 experts), walks it in increasing
// expert id inserting into a sorted top-k list held in registers (value desc, id asc: an equal
// value never displaces a lower id; -0 == +0), then takes the softmax of the selected logits.
template <int KMAX>
__device__ __forceinline__ void route_token(const float *__restrict__ logits, int64_t t, int E, int k,
                                            int (&ti)[KMAX], float (&w)[KMAX]) {
  const float *row = logits + t * E;
  const bool vec = (E & 3) == 0;   // rows then start on 16-byte boundaries
  float tv[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    tv[j] = -INFINITY;
    ti[j] = 0;
  }
  for (int e0 = 0; e0 < E; e0 += 64) {
    float v[64];
    if (vec) {
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 f = e0 + 4 * q < E ? __ldg(reinterpret_cast<const float4 *>(row + e0) + q)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = e0 + i < E ? __ldg(row + e0 + i) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) {   // leave at the row's end: predicated-off insertions still issue
      if (e0 + i >= E) break;
      topk_insert<KMAX>(tv, ti, v[i], e0 + i);
    }
  }
  const float m = tv[0];
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    w[j] = j < k ? expf(tv[j] - m) : 0.0f;
    s += w[j];
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j) w[j] = w[j] / s;
}

template <int KMAX>
__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(const float *__restrict__ logits, int T, int E,
                                                                   int k, int32_t *__restrict__ topk_idx,
                                                                   float *__restrict__ topk_w) {
  const int64_t t = (int64_t)blockIdx.x * kRouteThreads + threadIdx.x;
  if (t >= T) return;
  int ti[KMAX];
  float w[KMAX];
  route_token<KMAX>(logits, t, E, k, ti, w);
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (j < k) {
      topk_idx[t * k + j] = ti[j];
      topk_w[t * k + j] = w[j];
    }
}

// ---------------------------------------------------------------------------------------------
// count kernel
struct IndexWs {
  WsHeader hdr;   // tickets[0]: count blocks done, tickets[1]: index block ticket
};

__device__ __forceinline__ int slot_key(const int32_t *__restrict__ idx, int64_t s, int64_t n, int E, WsHeader *hdr) {
  if (s >= n) return -1;
  int e = __ldg(idx + s);
  if ((unsigned)e >= (unsigned)E) {
    report(hdr, MOE_ERR_BAD_INDEX, (int)s);
    return -1;
  }
  return e;
}

// Exclusive scans of the per-expert totals in acc: counts, offsets (scan of counts) and tile_offsets
// (scan of ceil(counts / BM)). One warp, 8 experts per lane (E <= 256).
__device__ __forceinline__ void scan_counts(int32_t *acc, int E, int BM, int32_t *__restrict__ counts,
                                            int32_t *__restrict__ offsets, int32_t *__restrict__ tile_offsets) {
  const int lane = threadIdx.x & 31;
  int c[8], tl[8], sc = 0, st = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    int e = lane * 8 + q;
    c[q] = e < E ? atomicAdd(acc + e, 0) : 0;
    tl[q] = (c[q] + BM - 1) / BM;
    sc += c[q];
    st += tl[q];
  }
  int ic = sc, it = st;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int a = __shfl_up_sync(0xffffffffu, ic, off), b = __shfl_up_sync(0xffffffffu, it, off);
    if (lane >= off) { ic += a; it += b; }
  }
  int rc = ic - sc, rt = it - st;   // exclusive prefix of this lane's first expert
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    int e = lane * 8 + q;
    if (e < E) {
      counts[e] = c[q];
      offsets[e] = rc;
      tile_offsets[e] = rt;
    }
    rc += c[q];
    rt += tl[q];
  }
  if (lane == 31) {
    offsets[E] = ic;
    tile_offsets[E] = it;
  }
}

__global__ void __launch_bounds__(kIdxThreads) count_kernel(const int32_t *__restrict__ idx, int64_t n, int E, int BM,
                                                            WsHeader *hdr, int32_t *__restrict__ acc, int32_t *hook,
                                                            uint64_t *__restrict__ lookback, int32_t *__restrict__ counts,
                                                            int32_t *__restrict__ offsets,
                                                            int32_t *__restrict__ tile_offsets) {
  __shared__ int hist[MOE_MAX_EXPERTS];
  __shared__ bool is_last;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += kIdxThreads) {
    hist[e] = 0;
    lookback[(size_t)blockIdx.x * E + e] = 0;   // reset this block's look-back words for the index kernel
  }
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kIdxChunk;
#pragma unroll
  for (int i = 0; i < kIdxItems; ++i) {
    int key = slot_key(idx, base + i * kIdxThreads + tid, n, E, hdr);
    unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[key], __popc(peers));
  }
  __syncthreads();
  for (int e = tid; e < E; e += kIdxThreads)
    if (hist[e]) atomicAdd(acc + e, hist[e]);
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(&hdr->tickets[0], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (tid == 0) {   // arm (or disarm) the look-back fault hook for the index kernel, then clear it
    hdr->armed = *hook;
    *hook = 0;
  }
  if (tid < 32) scan_counts(acc, E, BM, counts, offsets, tile_offsets);
}

// ---------------------------------------------------------------------------------------------
// Stable ranks of a block's slots within their expert and the block's per-expert totals. Warp w
// owns the block's slots [32 ITEMS w, 32 ITEMS (w + 1)): key[i] is the expert of its slot
// 32 ITEMS w + 32 i + lane (-1: none). A warp counts its slots per expert as it goes (match.any per
// round of 32, no block barrier between rounds); the counts of the block's earlier warps are added
// at the end. On return rank[i] counts the block's earlier slots (in slot order) with the same
// expert and run[e] holds the block's count of expert e. warp_cnt must be all zero on entry; it is
// left holding each warp's exclusive offsets.
template <int ITEMS>
__device__ __forceinline__ void warp_ranks(const int (&key)[ITEMS], int (&rank)[ITEMS],
                                           int (*warp_cnt)[MOE_MAX_EXPERTS], int *run, int E) {
  constexpr int kWarps = kIdxThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const unsigned peers = __match_any_sync(0xffffffffu, key[i]);
    const int before = key[i] >= 0 ? warp_cnt[warp][key[i]] : 0;
    rank[i] = before + __popc(peers & lt_mask);
    __syncwarp();
    if (key[i] >= 0 && lane == __ffs(peers) - 1) warp_cnt[warp][key[i]] = before + __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = tid; e < E; e += kIdxThreads) {   // exclusive scan over the warps
    int r = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = warp_cnt[w][e];
      warp_cnt[w][e] = r;
      r += c;
    }
    run[e] = r;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < ITEMS; ++i)
    if (key[i] >= 0) rank[i] += warp_cnt[warp][key[i]];
}

// Decoupled look-back: publish block b's per-expert aggregate run[e], walk back over the preceding
// blocks' words, kLookWindow per round (an aggregate adds and continues, an inclusive prefix adds
// and stops, a word not yet published is waited for, at most about 0.2 s in all), set excl[e] to
// the number of slots of expert e in blocks 0..b-1 and publish block b's inclusive prefix.
// `withhold` leaves this block's words unpublished (the fault hook of moe_count_index).
__device__ __forceinline__ void block_lookback(int b, int E, const int *run, int *excl, uint64_t *lookback,
                                               WsHeader *hdr, bool withhold) {
  for (int e = threadIdx.x; e < E; e += kIdxThreads) {
    const uint32_t agg = (uint32_t)run[e];
    volatile uint64_t *mine = lookback + (size_t)b * E + e;
    if (b == 0) {
      if (!withhold) *mine = kFlagPrefix | agg;
      excl[e] = 0;
      continue;
    }
    if (!withhold) *mine = kFlagAggregate | agg;
    uint32_t sum = 0;
    int p = b - 1;
    uint64_t t0 = 0;
    while (p >= 0) {
      // the next kLookWindow predecessors' words at once, nearest first (before block 0: a zero
      // prefix), then consumed in order up to the first prefix or the first word not yet published
      uint64_t w[kLookWindow];
#pragma unroll
      for (int j = 0; j < kLookWindow; ++j)
        w[j] = p - j >= 0 ? (uint64_t)*(volatile uint64_t *)(lookback + (size_t)(p - j) * E + e)
                          : (uint64_t)kFlagPrefix;
      int used = 0;
      bool stop = false, stalled = false;
#pragma unroll
      for (int j = 0; j < kLookWindow; ++j) {
        const uint64_t flag = w[j] & 0xffffffff00000000ull;
        if (stop || stalled) continue;
        if (flag == 0) {
          stalled = true;
          continue;
        }
        sum += (uint32_t)w[j];
        ++used;
        stop = flag == kFlagPrefix;
      }
      if (stop) break;
      p -= used;
      if (stalled) {
        const uint64_t now = global_ns();
        if (t0 == 0) t0 = now;
        if (now - t0 > kWaitLimitNs) {
          report(hdr, MOE_ERR_DEVICE_TIMEOUT, b);
          break;
        }
        __nanosleep(64);
      }
    }
    excl[e] = (int)sum;
    if (!withhold) *mine = kFlagPrefix | (sum + agg);
  }
}

// ---------------------------------------------------------------------------------------------
// index kernel: stable ranks + per-expert decoupled look-back + scatter
__global__ void __launch_bounds__(kIdxThreads) index_kernel(const int32_t *__restrict__ idx, int64_t n, int k, int E,
                                                            int BM, WsHeader *hdr, uint64_t *__restrict__ lookback,
                                                            const int32_t *__restrict__ counts,
                                                            const int32_t *__restrict__ tile_offsets,
                                                            int32_t *__restrict__ row_of_slot,
                                                            int32_t *__restrict__ token_of_row) {
  __shared__ int warp_cnt[kIdxThreads / 32][MOE_MAX_EXPERTS];
  __shared__ int run[MOE_MAX_EXPERTS];
  __shared__ int excl[MOE_MAX_EXPERTS];
  __shared__ int row_base[MOE_MAX_EXPERTS];
  __shared__ int bid_s;
  const int tid = threadIdx.x;
  if (tid == 0) bid_s = (int)atomicAdd(&hdr->tickets[1], 1u);   // dynamic block id: predecessors already run
  for (int i = tid; i < (kIdxThreads / 32) * MOE_MAX_EXPERTS; i += kIdxThreads) (&warp_cnt[0][0])[i] = 0;
  for (int e = tid; e < E; e += kIdxThreads) {
    run[e] = 0;
    row_base[e] = tile_offsets[e] * BM;
  }
  __syncthreads();
  const int b = bid_s;
  const int64_t base = (int64_t)b * kIdxChunk + (tid >> 5) * (32 * kIdxItems) + (tid & 31);   // slot of item 0
  int key[kIdxItems], rank[kIdxItems];
#pragma unroll
  for (int i = 0; i < kIdxItems; ++i) key[i] = slot_key(idx, base + 32 * i, n, E, nullptr);
  warp_ranks<kIdxItems>(key, rank, warp_cnt, run, E);
  block_lookback(b, E, run, excl, lookback, hdr, b == hdr->armed - 1);
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kIdxItems; ++i) {
    const int64_t s = base + 32 * i;
    if (s >= n) continue;
    if (key[i] < 0) {
      row_of_slot[s] = -1;
      continue;
    }
    const int row = row_base[key[i]] + excl[key[i]] + rank[i];
    row_of_slot[s] = row;
    token_of_row[row] = (int)s / k;   // s < T*k < 2^31
  }
  // padding rows of the grouped layout
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    int start = tile_offsets[e] * BM + counts[e], end = tile_offsets[e + 1] * BM;
    for (int r = start + tid; r < end; r += kIdxThreads) token_of_row[r] = -1;
  }
}

// ---------------------------------------------------------------------------------------------
// Routing, counting and index generation in one kernel (moe_route_count_index). Block b owns the
// C = kIdxThreads * ITEMS slots [b C, (b + 1) C).
//   1. Routing: each token of the block's slots is routed by a pair of adjacent lanes, each lane
//      keeping the top-k of one half of the experts; the lower lane merges the upper lane's list
//      into its own (route_token_pair). A token whose slots straddle two blocks is routed by both,
//      identically; the block holding its first slot writes topk_idx / topk_w.
//   2. Ranks: warp w owns slots [32 ITEMS w, 32 ITEMS (w + 1)) of the chunk, ITEMS rounds of 32;
//      a slot's rank within its expert is the warp's running count (match.any per round, no block
//      barrier), plus the slots of that expert in the block's earlier warps.
//   3. The block publishes its per-expert counts (one row of agg) and adds them to the totals acc,
//      then counts itself in. Once all blocks have (a bounded wait of about 0.2 s), every block
//      reads the totals and its predecessors' rows from L2, scans the totals itself, and scatters
//      row_of_slot / token_of_row; block 0 writes counts, offsets and tile_offsets.
// The blocks wait for one another, so all of them must be resident at once: the host launches the
// kernel cooperatively, and only when the whole grid fits on the GPU.
template <int KMAX>
__device__ __forceinline__ void route_token_pair(const float *__restrict__ logits, int64_t t, bool active, int E,
                                                 int k, int (&ti)[KMAX], float (&w)[KMAX]) {
  const int h = threadIdx.x & 1;
  const int split = min(E, ((E + 1) / 2 + 3) & ~3);   // the upper half starts on a 16-byte boundary
  const int lo = h ? split : 0, hi = h ? E : split;
  const float *row = logits + t * E;
  const bool vec = (E & 3) == 0;
  float tv[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    tv[j] = -INFINITY;
    ti[j] = 0;
  }
  if (active) {
    for (int e0 = lo; e0 < hi; e0 += 64) {
      float v[64];
      if (vec) {
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float4 f = e0 + 4 * q < hi ? __ldg(reinterpret_cast<const float4 *>(row + e0) + q)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
          v[4 * q] = f.x;
          v[4 * q + 1] = f.y;
          v[4 * q + 2] = f.z;
          v[4 * q + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = e0 + i < hi ? __ldg(row + e0 + i) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) {   // leave at the half's end: predicated-off insertions still issue
        if (e0 + i >= hi) break;
        topk_insert<KMAX>(tv, ti, v[i], e0 + i);
      }
    }
  }
  // The upper lane's entries all carry higher ids than the lower lane's and arrive in their list
  // order (value desc, id asc), which is the order topk_insert requires.
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const float pv = __shfl_xor_sync(0xffffffffu, tv[j], 1);
    const int pi = __shfl_xor_sync(0xffffffffu, ti[j], 1);
    if (h == 0 && j < k) topk_insert<KMAX>(tv, ti, pv, pi);
  }
  const float m = tv[0];
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    w[j] = j < k ? expf(tv[j] - m) : 0.0f;
    s += w[j];
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j) w[j] = w[j] / s;
}

template <int KMAX, int ITEMS>
__global__ void __launch_bounds__(kIdxThreads) route_count_index_kernel(
    const float *__restrict__ logits, int T, int E, int k, int BM, WsHeader *hdr, int32_t *acc,
    int32_t *agg, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ tile_offsets, int32_t *__restrict__ row_of_slot,
    int32_t *__restrict__ token_of_row) {
  static_assert(2 * ITEMS >= kIdxItems, "the count table must fit the look-back words");
  constexpr int kWarps = kIdxThreads / 32, kWarpSlots = 32 * ITEMS, kRciChunk = kIdxThreads * ITEMS;
  __shared__ int sk[kRciChunk];                            // experts of this block's slots, slot order
  __shared__ int warp_cnt[kWarps][MOE_MAX_EXPERTS];
  __shared__ int run[MOE_MAX_EXPERTS];                     // this block's slots per expert
  __shared__ int excl[MOE_MAX_EXPERTS];                    // slots of each expert in blocks 0..b-1
  __shared__ int cnt[MOE_MAX_EXPERTS];                     // totals
  __shared__ int tile_first[MOE_MAX_EXPERTS + 1];          // exclusive scan of the tiles per expert
  __shared__ __align__(16) int part[4 * kIdxThreads];
  __shared__ int wsum_c[kWarps], wsum_t[kWarps];
  __shared__ bool ready;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int64_t n = (int64_t)T * k;
  const int64_t base = (int64_t)b * kRciChunk;
  const int64_t send = base + kRciChunk < n ? base + kRciChunk : n;   // this block's slots: [base, send)
  for (int i = tid; i < kWarps * MOE_MAX_EXPERTS; i += kIdxThreads) (&warp_cnt[0][0])[i] = 0;
  // 1. route the tokens of slots [base, send), a pair of lanes per token
  const int64_t t_first = base / k, t_last = (send - 1) / k;
  for (int64_t t0 = t_first; t0 <= t_last; t0 += kIdxThreads / 2) {   // the same trip count in every lane
    const int64_t t = t0 + (tid >> 1);
    const bool active = t <= t_last;
    int ti[KMAX];
    float w[KMAX];
    route_token_pair<KMAX>(logits, t, active, E, k, ti, w);
    if (active && (tid & 1) == 0) {
      const bool owner = t * k >= base;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) {
          const int64_t s = t * k + j;
          if (s >= base && s < send) sk[s - base] = ti[j];
          if (owner) {
            topk_idx[s] = ti[j];
            topk_w[s] = w[j];
          }
        }
    }
  }
  __syncthreads();
  // 2. stable ranks: a warp's running count per expert, then the earlier warps' counts
  int key[ITEMS], rank[ITEMS];
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int64_t s = base + warp * kWarpSlots + i * 32 + lane;
    key[i] = s < send ? sk[s - base] : -1;
  }
  warp_ranks<ITEMS>(key, rank, warp_cnt, run, E);
  // 3. publish: the block's row of agg, the totals
  for (int e = tid; e < E; e += kIdxThreads) {
    const int r = run[e];
    agg[(size_t)b * E + e] = r;
    if (r) atomicAdd(acc + e, r);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {   // count in, then wait (bounded) for every block to have done the same
    atomicAdd(&hdr->tickets[0], 1u);
    bool ok = true;
    const uint64_t t0 = global_ns();
    while (*reinterpret_cast<volatile uint32_t *>(&hdr->tickets[0]) < gridDim.x) {
      if (global_ns() - t0 > kWaitLimitNs) {
        report(hdr, MOE_ERR_DEVICE_TIMEOUT, b);
        ok = false;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    ready = ok;
  }
  __syncthreads();
  if (!ready) return;
  // totals (threads 0..E-1) and this block's offset per expert: a row of the count table is read by
  // Q threads (16-byte loads of four experts when E % 4 == 0, else one expert each); thread
  // (eq, q) sums the rows of the blocks p < b with p = q mod parts, eight loads in flight, into
  // part[q * E + expert]
  const bool vec4 = (E & 3) == 0;   // rows then start on 16-byte boundaries
  const int Q = vec4 ? E / 4 : E;
  const int parts = kIdxThreads / Q;   // E <= MOE_MAX_EXPERTS == kIdxThreads
  const int eq = tid % Q, q = tid / Q;
  const int c = tid < E ? __ldcg(acc + tid) : 0;
  if (q < parts) {
    if (vec4) {
      int4 sum = make_int4(0, 0, 0, 0);
      for (int p0 = q; p0 < b; p0 += 8 * parts) {
        int4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int p = p0 + j * parts;
          v[j] = p < b ? __ldcg(reinterpret_cast<const int4 *>(agg + (size_t)p * E) + eq) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sum.x += v[j].x;
          sum.y += v[j].y;
          sum.z += v[j].z;
          sum.w += v[j].w;
        }
      }
      reinterpret_cast<int4 *>(part)[tid] = sum;   // part[q * E + 4 eq + 0..3]
    } else {
      int sum = 0;
      for (int p0 = q; p0 < b; p0 += 8 * parts) {
        int v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int p = p0 + j * parts;
          v[j] = p < b ? __ldcg(agg + (size_t)p * E + eq) : 0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) sum += v[j];
      }
      part[tid] = sum;   // part[q * E + eq]
    }
  }
  // exclusive scans of the totals and of their tile counts over the experts
  const int tl = (c + BM - 1) / BM;
  int ic = c, it = tl;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, off), d = __shfl_up_sync(0xffffffffu, it, off);
    if (lane >= off) {
      ic += a;
      it += d;
    }
  }
  if (lane == 31) {
    wsum_c[warp] = ic;
    wsum_t[warp] = it;
  }
  __syncthreads();
  if (tid < E) {
    int pc = 0, pt = 0;
    for (int w = 0; w < warp; ++w) {
      pc += wsum_c[w];
      pt += wsum_t[w];
    }
    const int oc = pc + ic - c, ot = pt + it - tl;
    int x = 0;
    for (int j = 0; j < parts; ++j) x += part[j * E + tid];
    excl[tid] = x;
    cnt[tid] = c;
    tile_first[tid] = ot;
    if (tid == E - 1) tile_first[E] = ot + tl;
    if (b == 0) {
      counts[tid] = c;
      offsets[tid] = oc;
      tile_offsets[tid] = ot;
      if (tid == E - 1) {
        offsets[E] = oc + c;
        tile_offsets[E] = ot + tl;
      }
    }
  }
  __syncthreads();
  // 4. scatter
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int64_t s = base + warp * kWarpSlots + i * 32 + lane;
    if (s >= send || key[i] < 0) continue;
    const int row = tile_first[key[i]] * BM + excl[key[i]] + rank[i];
    row_of_slot[s] = row;
    token_of_row[row] = (int)s / k;   // s < T*k < 2^31
  }
  for (int e = b; e < E; e += gridDim.x) {   // padding rows of the grouped layout
    const int start = tile_first[e] * BM + cnt[e], end = tile_first[e + 1] * BM;
    for (int r = start + tid; r < end; r += kIdxThreads) token_of_row[r] = -1;
  }
}

}  // namespace moe

using namespace moe;

extern "C" int moe_route_topk(const float *logits, int T, int E, int k, int32_t *topk_idx, float *topk_w,
                              moe_stream_t stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E || k > MOE_MAX_TOPK) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  const int blocks = (int)(((int64_t)T + kRouteThreads - 1) / kRouteThreads);
  cudaStream_t s = (cudaStream_t)stream;
#define MOE_ROUTE(KM) route_topk_kernel<KM><<<blocks, kRouteThreads, 0, s>>>(logits, T, E, k, topk_idx, topk_w)
  if (k <= 2) MOE_ROUTE(2);
  else if (k <= 4) MOE_ROUTE(4);
  else if (k <= 8) MOE_ROUTE(8);
  else MOE_ROUTE(16);
#undef MOE_ROUTE
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" int64_t moe_grouped_rows_max(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return -1;
  int64_t r = (int64_t)T * k + (int64_t)E * (MOE_GROUP_ROWS - 1);
  return (r + MOE_GROUP_ROWS - 1) / MOE_GROUP_ROWS * MOE_GROUP_ROWS;
}

static int64_t index_blocks(int T, int k) { return ((int64_t)T * k + kIdxChunk - 1) / kIdxChunk; }

// layout: [IndexWs header][acc: E int32, padded to 256 B][fault hook int32, padded to 256 B]
//         [lookback: blocks * E uint64]
static size_t acc_bytes(int E) { return ((size_t)E * 4 + 255) / 256 * 256; }
constexpr size_t kHookBytes = 256;

extern "C" size_t moe_count_index_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  int64_t nb = index_blocks(T, k);
  if (nb < 1) nb = 1;
  return sizeof(IndexWs) + acc_bytes(E) + kHookBytes + (size_t)nb * E * sizeof(uint64_t);
}

extern "C" int moe_count_index(const int32_t *topk_idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                               int32_t *tile_offsets, int32_t *row_of_slot, int32_t *token_of_row, void *ws,
                               size_t ws_bytes, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_TOPK) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * k >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !tile_offsets || !token_of_row || !ws) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !row_of_slot)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_count_index_workspace_size(T, k, E)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char *w = static_cast<char *>(ws);
  IndexWs *iw = reinterpret_cast<IndexWs *>(w);
  int32_t *acc = reinterpret_cast<int32_t *>(w + sizeof(IndexWs));
  uint64_t *lookback = reinterpret_cast<uint64_t *>(w + sizeof(IndexWs) + acc_bytes(E) + kHookBytes);
  // One memset resets the status word, the tickets and the histogram accumulator; the fault hook
  // lives after them and is consumed (read and cleared) by the count kernel's last block.
  MOE_TRY_CUDA(cudaMemsetAsync(w, 0, sizeof(IndexWs) + acc_bytes(E), s));
  int32_t *hook = reinterpret_cast<int32_t *>(w + sizeof(IndexWs) + acc_bytes(E));
  const int64_t n = (int64_t)T * k;
  const int nb = (int)(n > 0 ? index_blocks(T, k) : 1);
  count_kernel<<<nb, kIdxThreads, 0, s>>>(topk_idx, n, E, MOE_GROUP_ROWS, &iw->hdr, acc, hook, lookback, counts,
                                          offsets, tile_offsets);
  MOE_CHECK_LAUNCH();
  index_kernel<<<nb, kIdxThreads, 0, s>>>(topk_idx, n, k, E, MOE_GROUP_ROWS, &iw->hdr, lookback, counts,
                                          tile_offsets, row_of_slot, token_of_row);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

// Launch route_count_index_kernel<KMAX, ITEMS> if its whole grid fits on the GPU at once; *launched
// tells whether it did (if not, nothing was enqueued).
template <int KMAX, int ITEMS>
static int launch_rci(const float *logits, int T, int E, int k, int32_t *topk_idx, float *topk_w, int32_t *counts,
                      int32_t *offsets, int32_t *tile_offsets, int32_t *row_of_slot, int32_t *token_of_row, void *ws,
                      cudaStream_t s, bool *launched) {
  *launched = false;
  const int64_t chunk = (int64_t)kIdxThreads * ITEMS;
  const int64_t nb = ((int64_t)T * k + chunk - 1) / chunk;
  int per_sm = 0;   // every block must be resident at once (each waits until all have published)
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_count_index_kernel<KMAX, ITEMS>, kIdxThreads,
                                                    0) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_OK;
  }
  if ((int64_t)per_sm * sm_count() < nb) return MOE_OK;
  char *w = static_cast<char *>(ws);
  IndexWs *iw = reinterpret_cast<IndexWs *>(w);
  int32_t *acc = reinterpret_cast<int32_t *>(w + sizeof(IndexWs));
  // the blocks' per-expert counts, [nb][E] int32, in the look-back words' space (every block writes
  // its whole row before any block reads it, so the rows need no reset)
  int32_t *agg = reinterpret_cast<int32_t *>(w + sizeof(IndexWs) + acc_bytes(E) + kHookBytes);
  // status, tickets and totals start at zero (the fault hook is cleared too)
  MOE_TRY_CUDA(cudaMemsetAsync(w, 0, sizeof(IndexWs) + acc_bytes(E) + kHookBytes, s));
  // A cooperative launch: CUDA starts the grid only when all of its blocks can be resident together,
  // also while kernels from other streams (another layer, even another fused call) hold SMs, so the
  // blocks' meeting point cannot wait on a block that is still queued.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nb, 1, 1);
  cfg.blockDim = dim3(kIdxThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, route_count_index_kernel<KMAX, ITEMS>, logits, T, E, k,
                                           (int)MOE_GROUP_ROWS, &iw->hdr, acc, agg, topk_idx, topk_w, counts,
                                           offsets, tile_offsets, row_of_slot, token_of_row);
  if (e == cudaErrorCooperativeLaunchTooLarge) {   // the grid cannot be resident at once
    (void)cudaGetLastError();
    return MOE_OK;
  }
  MOE_TRY_CUDA(e);
  *launched = true;
  return MOE_OK;
}

// 512 slots per block while that is at most one block per SM (more blocks than SMs route no faster
// and lengthen every block's sum over its predecessors' counts), else 1024.
template <int KMAX>
static int launch_route_count_index(const float *logits, int T, int E, int k, int32_t *topk_idx, float *topk_w,
                                    int32_t *counts, int32_t *offsets, int32_t *tile_offsets, int32_t *row_of_slot,
                                    int32_t *token_of_row, void *ws, cudaStream_t s, bool *launched) {
  const int64_t nb512 = ((int64_t)T * k + 2 * kIdxThreads - 1) / (2 * kIdxThreads);
  if (nb512 <= sm_count())
    return launch_rci<KMAX, 2>(logits, T, E, k, topk_idx, topk_w, counts, offsets, tile_offsets, row_of_slot,
                               token_of_row, ws, s, launched);
  return launch_rci<KMAX, 4>(logits, T, E, k, topk_idx, topk_w, counts, offsets, tile_offsets, row_of_slot,
                             token_of_row, ws, s, launched);
}

extern "C" int moe_route_count_index(const float *logits, int T, int E, int k, int32_t *topk_idx, float *topk_w,
                                     int32_t *counts, int32_t *offsets, int32_t *tile_offsets,
                                     int32_t *row_of_slot, int32_t *token_of_row, void *ws, size_t ws_bytes,
                                     moe_stream_t stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E || k > MOE_MAX_TOPK) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * k >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !tile_offsets || !token_of_row || !ws) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_idx || !topk_w || !row_of_slot)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_count_index_workspace_size(T, k, E)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  bool launched = false;
  int rc = MOE_OK;
  if (T > 0) {
    if (k <= 2) rc = launch_route_count_index<2>(logits, T, E, k, topk_idx, topk_w, counts, offsets, tile_offsets,
                                                 row_of_slot, token_of_row, ws, s, &launched);
    else if (k <= 4) rc = launch_route_count_index<4>(logits, T, E, k, topk_idx, topk_w, counts, offsets,
                                                      tile_offsets, row_of_slot, token_of_row, ws, s, &launched);
    else if (k <= 8) rc = launch_route_count_index<8>(logits, T, E, k, topk_idx, topk_w, counts, offsets,
                                                      tile_offsets, row_of_slot, token_of_row, ws, s, &launched);
    else rc = launch_route_count_index<16>(logits, T, E, k, topk_idx, topk_w, counts, offsets, tile_offsets,
                                           row_of_slot, token_of_row, ws, s, &launched);
  }
  if (rc || launched) return rc;
  // too many blocks to be resident at once (or T = 0): the two calls, same results
  if ((rc = moe_route_topk(logits, T, E, k, topk_idx, topk_w, stream))) return rc;
  return moe_count_index(topk_idx, T, k, E, counts, offsets, tile_offsets, row_of_slot, token_of_row, ws, ws_bytes,
                         stream);
}

extern "C" size_t moe_count_index_hook_offset(int E) {
  if (E < 1) return 0;
  return sizeof(IndexWs) + acc_bytes(E);
}

// ---------------------------------------------------------------------------------------------
// Allocation-free variant of moe_count_index.
//
// Some callers cannot allocate device memory at all: a plugin inside a host framework that owns
// every device allocation and hands the plugin only its input and output buffers, or a service
// that forbids allocation once it has started. They cannot provide the workspace that
// moe_count_index needs, so this variant keeps that scratch in a fixed array in the library's own
// device memory. The array exists on every GPU that loads the library, for the life of the
// process, and is shared by all calls on that GPU.
static __device__ __align__(256) unsigned char g_count_index_scratch[MOE_STATIC_SCRATCH_BYTES];

#include <mutex>

// The array's name is only a host-side stand-in, not a device address; each device's address is
// looked up once (with that device current) and cached for the life of the process. A reset of the
// device's primary context (cudaDeviceReset) reloads the module at a new address, which this cache
// does not follow: the header tells callers not to use this entry point after such a reset.
static int static_scratch_address(void **out) {
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_count_index_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return MOE_OK;
}

extern "C" int moe_count_index_static(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                                      int32_t *offsets, int32_t *tile_offsets, int32_t *row_of_slot,
                                      int32_t *token_of_row, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_TOPK) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * k >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !tile_offsets || !token_of_row) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !row_of_slot)) return MOE_ERR_INVALID_ARG;
  if (moe_count_index_workspace_size(T, k, E) > (size_t)MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  int rc = static_scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  char *w = static_cast<char *>(scratch);
  IndexWs *iw = reinterpret_cast<IndexWs *>(w);
  int32_t *acc = reinterpret_cast<int32_t *>(w + sizeof(IndexWs));
  int32_t *hook = reinterpret_cast<int32_t *>(w + sizeof(IndexWs) + acc_bytes(E));
  uint64_t *lookback = reinterpret_cast<uint64_t *>(w + sizeof(IndexWs) + acc_bytes(E) + kHookBytes);
  // The array keeps the previous call's contents: reset the status word, tickets, histogram
  // accumulator and fault hook here; the count kernel resets the look-back words it uses.
  MOE_TRY_CUDA(cudaMemsetAsync(w, 0, sizeof(IndexWs) + acc_bytes(E) + kHookBytes, s));
  const int64_t n = (int64_t)T * k;
  const int nb = (int)(n > 0 ? index_blocks(T, k) : 1);
  count_kernel<<<nb, kIdxThreads, 0, s>>>(topk_idx, n, E, MOE_GROUP_ROWS, &iw->hdr, acc, hook, lookback, counts,
                                          offsets, tile_offsets);
  MOE_CHECK_LAUNCH();
  index_kernel<<<nb, kIdxThreads, 0, s>>>(topk_idx, n, k, E, MOE_GROUP_ROWS, &iw->hdr, lookback, counts,
                                          tile_offsets, row_of_slot, token_of_row);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
