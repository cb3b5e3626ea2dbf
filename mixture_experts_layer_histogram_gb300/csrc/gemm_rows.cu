// Row-grouped kinds of the grouped SwiGLU GEMM on CTA pairs, with the weights as the MMA's A operand
// and the tokens as its B operand (sm_103a, tcgen05.mma.cta_group::2).
//
// "Scalable Pretraining of Large MoE LMs on Aurora", brief, section 核心方法: the experts'
// computation is merged into one grouped GEMM; summary page, section 关键设计: with optimised
// matrix multiplication and activation. The four kinds whose output rows are grouped tokens:
//   GATEUP  [a | b] = x_perm Wgu[e]^T, epilogue writes a, b and h = silu(a) * b
//   DOWN    y = h Wd[e]^T
//   DH      dh = dy Wd[e], epilogue reads a, b and writes da, db (the SwiGLU backward)
//   DGRAD   dx = dab Wgu[e]
//
// Why the weights are A. In a CTA-pair MMA (M = 256) each CTA supplies 128 rows of A and half of
// B, and both CTAs multiply by the whole of B. With tokens as A, the two CTAs must take two row
// tiles of one expert, so an expert with an odd number of 128-row tiles computes a discarded tile,
// and every expert computes its padding up to a multiple of 128 rows. With the weights as A (256
// output features per pair, 128 per CTA) and the tokens as B, a tile's token count is the MMA's N,
// which may be any multiple of 16 up to 256. Expert e's c_e rows fill ceil(c_e / 256) tiles: full
// ones of 256 tokens, then the rest rounded up to a multiple of 32, so the pair computes at most 31
// rows past an expert's last token: no discarded tile, no padding beyond the next multiple of 32.
// The tile count is the same as with tokens as A (ceil(ceil(c_e / 128) / 2) = ceil(c_e / 256)
// pairs), and a tile's time is set mostly by its ring stages, not by its N, so the gain is the
// tensor work (and power) of the rows no longer computed, plus a cheaper epilogue.
// Every tile loads full 128-row token boxes: loading only the rows a short tile uses took more,
// smaller TMA requests and was slower.
//
// The accumulator is then transposed relative to the output: TMEM lane = output feature, TMEM
// column = token. The epilogue reads it with tcgen05.ld.16x256b, whose register layout is that of
// an mma fragment (thread T: lanes T/4 and T/4 + 8, columns 2 (T % 4) + {0, 1}), converts to bf16
// and writes token-major blocks to shared memory with stmatrix .trans; a TMA bulk tensor store
// writes each block out. DH works the other way round as well: it copies its saved a, b blocks in
// with cp.async and ldmatrix .trans, and writes da, db with plain coalesced stores (its TMA copies
// queued behind the ring's loads in the SM's TMA unit). GATEUP's A holds each group of 8 gate rows next to the same features' 8 up
// rows (a 5D tensor map), so one thread receives a (lane T/4) and b (lane T/4 + 8) of the same
// feature and token and computes h in registers.
//
// Warp roles per CTA (both CTAs of the pair):
//   warp 0      TMA producer: 128 weight rows and 128 token rows per k-block into a shared-memory
//               ring of six 64-deep stages (DH five: its epilogue buffers take the sixth); the whole
//               warp polls the ring, one elected lane issues
//   warp 1      TMEM allocation (512 columns, two accumulators of up to 256 tokens); in the leader
//               CTA the converged warp issues the MMAs from one elected lane and commits to both
//               CTAs' barriers
// Each role walks the cluster's tiles incrementally (TileWalker): no division or search at a tile
// boundary, the next tile's offsets loaded while the current one runs.
//   warps 2..9  epilogue: two warps per 32-lane TMEM quarter, each taking every second 32-token chunk
// Padding rows (from the last computed token of an expert up to its group's multiple of 128) are
// written with zeros by the expert's last tile. Every wait is bounded (0.2 s): on timeout the kernel
// records MOE_ERR_DEVICE_TIMEOUT in the workspace status word and leaves.
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace moe {
namespace tc {
namespace rows {

enum Kind { GATEUP = 0, DOWN = 1, DH = 2, DGRAD = 3 };

constexpr int LANES = 128;            // weight rows (output features) per CTA = TMEM lanes
constexpr int NT_MAX = 256;           // tokens per tile: the MMA's N
constexpr int TOK_ROWS = NT_MAX / 2;  // token rows per CTA in one B box
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int LOADER_WARPS = 2;                       // gathering GATEUP: warps per loader set, ...
constexpr int LOADER_SETS = 3;                        // ... one set per ring slot
constexpr int THREADS_G = THREADS + 32 * LOADER_WARPS * LOADER_SETS;
constexpr int TMEM_COLS = 2 * NT_MAX;
constexpr int MAX_E = MOE_MAX_EXPERTS;

// The ring: 64-deep stages, as many as fit beside the epilogue's staging buffers (a load's latency
// under full load is about as long for a 32 KB stage as for a 64 KB one, so more, smaller stages
// keep more of it covered). Gathering GATEUP (G) keeps three 128-deep stages, one per loader set.
// (Deeper rings for the gathering kind measured no faster: its loaders set its pace.)
template <int K, bool G = false> struct Cfg {
  static constexpr int BKP = G ? 128 : 64;                   // k depth of one ring stage
  static constexpr int KA = BKP / 64;                        // 128-byte swizzle atoms along k per stage
  static constexpr int A_BYTES = LANES * BKP * 2;
  static constexpr int B_BYTES = TOK_ROWS * BKP * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = G ? 3 : (K == DH ? 5 : 6);
  static constexpr int BUF_BYTES = K == GATEUP ? 1024 : 2048;   // one 32-token staging block
  static constexpr int NBUF = K == DOWN || K == DGRAD ? 2 : 4;   // per warp (DH: two chunks of a + b)
  static constexpr int EPI_BYTES = EPI_WARPS * NBUF * BUF_BYTES;
  static constexpr int NBARS = 2 * STAGES + 5;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 8 * NBARS + 16 + (MAX_E + 1) * 4;
  static_assert(SMEM <= 232448, "row-grouped GEMM shared memory exceeds 227 KB");
  static_assert(A_BYTES == B_BYTES, "A and B atoms share one k-offset table");
};

struct Params {
  const int32_t *tile_offsets;   // [E+1] 128-row groups
  const int32_t *offsets;        // [E+1] exclusive scan of the routed row counts
  WsHeader *hdr;
  int E;
  int n_ft;                      // feature tiles per expert
  int num_kb;                    // ring stages per tile (K / BKP)
  int a_rows_e;                  // rows of the weight's 2D view per expert (DOWN, DH, DGRAD)
  int f;                         // GATEUP, DH: column of b in ab / dab
  int64_t rows_max;              // rows of every grouped buffer (bounds the zero-padding writes)
  __nv_bfloat16 *out0;           // zero padding rows: GATEUP ab (null: a, b not stored), DOWN y, DH dab, DGRAD dx
  int64_t ld0;
  __nv_bfloat16 *out1;           // GATEUP h
  int64_t ld1;
  const __nv_bfloat16 *gx;       // gathering GATEUP: the token rows x [ntok, ldgx] ...
  const int32_t *tor;            // ... and the token of each grouped row (-1 on padding rows)
  const __nv_bfloat16 *in0;      // DH: the saved a, b [rows, 2f] (row stride ld0)
  int64_t ldgx;
  int ntok;
};

// Tile = (expert e, token tile i, feature tile ft). Expert e's c rows fill n = ceil(c / 256) token
// tiles: n - 1 full ones of 256 tokens, then the rest rounded up to a multiple of 32.
struct Tile {
  int index;      // position in the kernel's tile list
  int e, ft;
  int start;      // first grouped row of the tile
  int nt;         // tokens (the MMA's N): a multiple of 32, at most 256
  int zero_end;   // rows [start + nt, zero_end) get zeros (the expert's padding; last tile only)
  bool ok;        // debug build: the tile passed its consistency checks (always true otherwise)
};

// One cluster's tiles in order: first, first + step, ... (tile = token tile gt * n_ft + feature
// tile ft). Token tiles only grow along the walk, so each tile's expert (the last one whose first
// token tile is <= gt; experts without rows are skipped) is found by stepping forward from the
// previous tile's, and the division by n_ft happens once. The expert's offsets are loaded from
// global memory one tile ahead, while the current tile runs: a tile boundary costs the ring only
// the few shared-memory steps of the walk.
struct TileWalker {
  int tile, step, num_tiles;
  int gt, ft, dgt, dft, e;
  int o0, o1, g0, g1;   // offsets[e], offsets[e + 1], tile_offsets[e], tile_offsets[e + 1] of `tile`

  __device__ __forceinline__ TileWalker(int first, int step_, int n, const Params &p, const int *ttoff)
      : tile(first), step(step_), num_tiles(n) {
    gt = first / p.n_ft;
    ft = first - gt * p.n_ft;
    dgt = step_ / p.n_ft;
    dft = step_ - dgt * p.n_ft;
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ttoff[mid] <= gt) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    load(p);
  }
  __device__ __forceinline__ void load(const Params &p) {
    if (tile >= num_tiles) return;
    o0 = p.offsets[e];
    o1 = p.offsets[e + 1];
    g0 = p.tile_offsets[e];
    g1 = p.tile_offsets[e + 1];
  }
  // The walk's next tile into t; false past the last.
  __device__ __forceinline__ bool next(Tile &t, const Params &p, const int *ttoff) {
    if (tile >= num_tiles) return false;
    t.index = tile;
    t.e = e;
    t.ft = ft;
    const int i = gt - ttoff[e];
    const int c = o1 - o0;
    const int nt = (c + NT_MAX - 1) / NT_MAX;
    const bool last = i == nt - 1;
    t.nt = last ? ((c - NT_MAX * i + 31) & ~31) : NT_MAX;
    t.start = g0 * 128 + NT_MAX * i;
    t.zero_end = last ? g1 * 128 : t.start + t.nt;
#if MOE_CHECKS
    // the expert's routed rows fit its 128-row group, and the group lies inside the buffers
    t.ok = c > 0 && g0 <= g1 && ((c + 31) & ~31) <= (g1 - g0) * 128 && (int64_t)g1 * 128 <= p.rows_max;
#else
    t.ok = true;
#endif
    tile += step;
    gt += dgt;
    ft += dft;
    if (ft >= p.n_ft) {
      ft -= p.n_ft;
      ++gt;
    }
    if (tile < num_tiles) {
      while (e + 1 < p.E && ttoff[e + 1] <= gt) ++e;
      load(p);
    }
    return true;
  }
};

// Instruction descriptor, kind::f16: D fp32, A and B bf16, B K-major, A MN-major when a_mn,
// M = 256 (the pair), N = nt.
__device__ __forceinline__ uint32_t idesc(bool a_mn, int nt) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((uint32_t)(nt >> 3) << 17) |
         ((uint32_t)(256 >> 4) << 24);
}

__device__ __forceinline__ void bulk_store(const CUtensorMap *map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}

// Zero 32 rows x `cols` bf16 columns (cols = 16 or 32) of a row-major output: lane = row.
__device__ __forceinline__ void zero_rows(__nv_bfloat16 *out, int64_t ld, int row0, int col0, int cols, int lane) {
  uint4 *dst = reinterpret_cast<uint4 *>(out + (int64_t)(row0 + lane) * ld + col0);
  for (int i = 0; i < cols / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
}

// G (GATEUP only): the token operand is gathered from x by token_of_row with cp.async by loader
// warps, instead of being read from the permuted x_perm by TMA (the permutation fused into the load).
template <int K, bool G>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(G ? THREADS_G : THREADS, 1)
    rows_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1, const Params p) {
  using C = Cfg<K, G>;
  constexpr bool A_MN = (K == DH || K == DGRAD);
  constexpr int PS = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *epi_smem = smem + PS * C::STAGE_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(epi_smem + C::EPI_BYTES);
  // bars: full[PS], empty[PS], tfull[2], tempty[2], mma_done, (DH) two a/b load barriers per epilogue warp
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + C::NBARS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  int *ttoff = reinterpret_cast<int *>(tmem_holder + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (PS + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * PS + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * PS + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * PS + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < PS; ++s) {
      // gathering: the leader's expect_tx plus one arrival per loader warp of both CTAs
      mbar_init(full_bar(s), G ? 1 + 2 * LOADER_WARPS : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * EPI_WARPS);   // one arrival per epilogue warp of both CTAs
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    if (!G) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 0) {   // ttoff = exclusive scan of the token tiles per expert, ceil(rows / 256)
    int c[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane * 8 + q;
      c[q] = e < p.E ? (p.offsets[e + 1] - p.offsets[e] + NT_MAX - 1) / NT_MAX : 0;
      sum += c[q];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane * 8 + q;
      if (e < p.E) ttoff[e] = run;
      run += c[q];
    }
    if (lane == 31) ttoff[p.E] = incl;
  }
  if (warp == 1) {   // collective TMEM allocation by one warp of each CTA of the pair
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"((uint32_t)TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();   // both CTAs: barriers initialised, ttoff written, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int num_tiles = ttoff[p.E] * p.n_ft;
  const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    // The whole warp runs the loop and waits, converged; one elected lane issues the copies.
    int stage = 0;
    uint32_t phase = 0;
    TileWalker walk(cluster_id, num_clusters, num_tiles, p, ttoff);
    for (Tile t; walk.next(t, p, ttoff);) {
      if (!t.ok) {   // debug build: every role skips the tile; the producer reports it
        if (lane == 0) report(p.hdr, MOE_ERR_CHECK_FAILED, t.index);
        continue;
      }
      const int brow = t.start + (int)rank * (t.nt >> 1);   // this CTA's half of the tile's tokens
      const int frow = t.ft * (K == GATEUP ? 128 : 256) + (int)rank * (K == GATEUP ? 64 : 128);
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!mbar_spin_cluster(empty_bar(stage), phase ^ 1u, abort_flag, p.hdr, 21)) { ok = false; break; }
        if (elect_one()) {
        const uint32_t sA = sbase + stage * C::STAGE_BYTES, sB = sA + C::A_BYTES;
        const uint32_t fb = mapa_shared(full_bar(stage), 0);   // the leader's full barrier
        if (leader) mbar_expect_tx(full_bar(stage), 2 * (G ? C::A_BYTES : C::STAGE_BYTES));
        const int kx = kb * C::BKP;
        if (!G) {
#pragma unroll
          for (int a = 0; a < C::KA; ++a) tma_load_2d_pair(sB + a * (TOK_ROWS * 128), &tmB, kx + 64 * a, brow, fb);
        }
        if (K == GATEUP) {
#pragma unroll
          for (int a = 0; a < C::KA; ++a)
            tma_load_5d_pair(sA + a * (LANES * 128), &tmA, kx + 64 * a, 0, 0, frow >> 3, t.e, fb);
        } else if (K == DOWN) {
#pragma unroll
          for (int a = 0; a < C::KA; ++a)
            tma_load_2d_pair(sA + a * (LANES * 128), &tmA, kx + 64 * a, t.e * p.a_rows_e + frow, fb);
        } else {   // DH, DGRAD: MN-major A, two 64-feature boxes of BKP k rows
#pragma unroll
          for (int q = 0; q < 2; ++q)
            tma_load_2d_pair(sA + q * (C::BKP * 128), &tmA, frow + 64 * q, t.e * p.a_rows_e + kx, fb);
        }
        }
        __syncwarp();
        if (++stage == PS) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
  } else if (warp == 1 && leader) {
    // ------------------------------------------------------------------ MMA issuer (leader only)
    // The whole warp runs the loop and waits, converged; one elected lane issues the MMAs. The
    // operand descriptors are formed once: every shared-memory address here lies below 256 KB, so a
    // stage's or a k step's offset adds to the descriptor's start-address field without carry.
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool issued_any = false;
    const uint64_t desc_a0 = A_MN ? sdesc(sbase, C::BKP * 128, 1024) : sdesc(sbase, 16, 1024);
    const uint64_t desc_b0 = sdesc(sbase + C::A_BYTES, 16, 1024);
    TileWalker walk(cluster_id, num_clusters, num_tiles, p, ttoff);
    for (Tile t; walk.next(t, p, ttoff);) {
      if (!t.ok) continue;
      if (!mbar_ready_cluster(tempty_bar(acc), acc_phase ^ 1u) &&
          !mbar_wait_cluster(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.hdr, 22))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NT_MAX);
      const uint32_t id = idesc(A_MN, t.nt);
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!mbar_spin_cluster(full_bar(stage), phase, abort_flag, p.hdr, 23)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t so = (uint32_t)(stage * C::STAGE_BYTES) >> 4;
#pragma unroll
          for (int kk = 0; kk < C::BKP / 16; ++kk) {
            // K-major: atom kk/4 (128 rows x 128 B each), 32 B per 16-deep step inside the atom.
            // MN-major A: 2048 B per 16 k-rows; its two 64-feature blocks are BKP * 128 B apart.
            const uint32_t koff = (uint32_t)((kk >> 2) * (LANES * 128) + (kk & 3) * 32) >> 4;
            const uint64_t ad = desc_a0 + so + (A_MN ? (uint32_t)(kk * 2048 >> 4) : koff);
            const uint64_t bd = desc_b0 + so + koff;
            mma_bf16_pair(d_tmem, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit_pair(empty_bar(stage), 0x3);   // frees this stage in both CTAs
        }
        __syncwarp();
        issued_any = true;
        if (++stage == PS) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) mma_commit_pair(tfull_bar(acc), 0x3);   // both CTAs' accumulators are ready
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (issued_any) {
      if (elect_one()) mma_commit_pair(mma_done_bar, 0x1);
      __syncwarp();
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(mma_done_bar, 0) && global_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (G && warp >= 2 + EPI_WARPS) {
    // ------------------------------------------------------------------ token-row gather (both CTAs)
    // Loader set q (two warps) fills ring slot q: every third fill. Each thread copies one 16-byte
    // chunk (lane % 8) of 16 of the CTA's token rows per 64-deep atom into the 128-byte-swizzled
    // K-major layout the TMA would have written; a padding row (token -1) is filled with zeros.
    static_assert(!G || PS == LOADER_SETS, "one loader set per ring slot");
    const int lw = warp - (2 + EPI_WARPS);
    const int q = lw / LOADER_WARPS;
    const int chunk = lane & 7;
    const int rsub = (lw % LOADER_WARPS) * 4 + (lane >> 3);   // rows rsub, rsub + 8, ..., rsub + 120
    int fill = 0;                             // fills of the ring so far (all slots)
    uint32_t phase = 0;                       // parity of slot q's next fill
    bool ok = true;
    TileWalker walk(cluster_id, num_clusters, num_tiles, p, ttoff);
    for (Tile t; ok && walk.next(t, p, ttoff);) {
      if (!t.ok) continue;
      const int brow = t.start + (int)rank * (t.nt >> 1), nrows = t.nt >> 1;
      int tok[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int row = 8 * j + rsub;
        const int tk = row < nrows ? p.tor[brow + row] : -2;   // -2: the MMA reads no such row
        tok[j] = tk >= p.ntok ? -1 : tk;                       // an index past the tokens reads as padding
      }
      for (int kb = 0; kb < p.num_kb; ++kb, ++fill) {
        if (fill % PS != q) continue;
        if (!mbar_spin_cluster(empty_bar(q), phase ^ 1u, abort_flag, p.hdr, 26)) { ok = false; break; }
        phase ^= 1u;
        gather_rows<C::KA>(sbase + q * C::STAGE_BYTES + C::A_BYTES, TOK_ROWS * 128, p.gx, p.ldgx, tok, rsub, chunk,
                           kb * C::BKP);
        gather_done(full_bar(q), lane);
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;             // TMEM lanes 32 quarter .. 32 quarter + 31
    const int hh = (warp - 2) >> 2;           // this warp takes the tile's 32-token chunks j = hh, hh + 2, ...
    const uint32_t wbuf = smem_u32(epi_smem) + (uint32_t)(warp - 2) * (C::NBUF * C::BUF_BYTES);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int mi = lane >> 3, mrow = lane & 7;   // stmatrix / ldmatrix: matrix and row this lane addresses
    int bi = 0;                               // next staging buffer (GATEUP, DOWN, DGRAD)
    // DH: the saved a, b of a chunk arrive two chunks ahead into one of two buffer pairs, copied by
    // the warp itself with cp.async (one commit group per chunk): TMA copies would queue behind the
    // ring's loads in the SM's TMA unit, and the warp would stall issuing them.
    // DH load cursor: chunk lj of tile lt is the next of this warp's chunks to bring in
    TileWalker lwalk(cluster_id, num_clusters, num_tiles, p, ttoff);
    Tile lt{};
    int lj = hh, lchunks = 0;
    bool lvalid = false;
    if (K == DH) {
      lvalid = lwalk.next(lt, p, ttoff);
      lchunks = lvalid && lt.ok ? lt.nt >> 5 : 0;
    }
    auto cursor_norm = [&]() {                // move the cursor to a chunk that exists
      while (lvalid && lj >= lchunks) {
        lvalid = lwalk.next(lt, p, ttoff);
        lchunks = lvalid && lt.ok ? lt.nt >> 5 : 0;
        lj = hh;
      }
    };
    auto issue_load = [&](int b) {   // DH: one commit group, empty past the last chunk
      if (K != DH) return;
      if (lvalid) {
        // lane: 16-byte column q of token rows lane / 4 + 8 i, into the 64-byte-swizzled layout
        const uint32_t dst = wbuf + (uint32_t)b * (2 * C::BUF_BYTES);
        const int x = lt.ft * 256 + (int)rank * 128 + quarter * 32, y = lt.start + 32 * lj, q = lane & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = (lane >> 2) + 8 * i;
          const uint32_t so = (uint32_t)t * 64 + ((uint32_t)(q ^ ((t >> 1) & 3)) << 4);
          if (y + t < p.rows_max) {
            const __nv_bfloat16 *src = p.in0 + (int64_t)(y + t) * p.ld0 + x + 8 * q;
            cp_async16(dst + so, src);
            cp_async16(dst + C::BUF_BYTES + so, src + p.f);
          }
        }
        lj += 2;
        cursor_norm();
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (K == DH) {
      cursor_norm();
      issue_load(0);
      issue_load(1);
    }
    int acc = 0;
    uint32_t acc_phase = 0;
    TileWalker walk(cluster_id, num_clusters, num_tiles, p, ttoff);
    for (Tile t; walk.next(t, p, ttoff);) {
      if (!t.ok) continue;
      if (!mbar_wait_cluster(tfull_bar(acc), acc_phase, abort_flag, p.hdr, 24)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + (uint32_t)(acc * NT_MAX);
      const int fcol = t.ft * (K == GATEUP ? 128 : 256) + (int)rank * (K == GATEUP ? 64 : 128) +
                       quarter * (K == GATEUP ? 16 : 32);   // first output feature of this warp
      bool ok = true;
#pragma unroll 1
      for (int j = hh; j < (t.nt >> 5); j += 2) {
        const int y = t.start + 32 * j;
        uint32_t r0[16], r1[16];
        tmem_ld16x256b_x4(tacc + 32u * j, r0);                    // lanes +0..15 of the quarter
        tmem_ld16x256b_x4(tacc + (16u << 16) + 32u * j, r1);      // lanes +16..31
        if (K == GATEUP) {
          // r0: features 16 quarter + T/4 (a: regs 4c, 4c+1; b: 4c+2, 4c+3); r1: features + 8
          tmem_ld_wait();
          uint32_t pa[2][4], pb[2][4], ph[2][4];   // [s][c]: fragments of the 8 x 8 blocks
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              const uint32_t *r = s ? r1 : r0;
              const float a0 = __uint_as_float(r[4 * c]), a1 = __uint_as_float(r[4 * c + 1]);
              const float b0 = __uint_as_float(r[4 * c + 2]), b1 = __uint_as_float(r[4 * c + 3]);
              pa[s][c] = pack_bf16x2(a0, a1);
              pb[s][c] = pack_bf16x2(b0, b1);
              ph[s][c] = pack_bf16x2(a0 * sigmoidf_(a0) * b0, a1 * sigmoidf_(a1) * b1);
            }
          }
          // three [32 tokens][16 features] blocks (32-byte rows, 32-byte swizzle); a and b only when
          // they are stored
          const uint32_t(*blk[3])[4] = {pa, pb, ph};
#pragma unroll
          for (int o = 0; o < 3; ++o) {
            if (o < 2 && p.out0 == nullptr) continue;
            const uint32_t buf = wbuf + (uint32_t)bi * C::BUF_BYTES;
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");   // buf's last store read it
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 2; ++u) {   // matrices (s, c) = (mi & 1, 2u + (mi >> 1))
              const int t = 8 * (2 * u + (mi >> 1)) + mrow, s = mi & 1;
              const uint32_t addr = buf + (uint32_t)t * 32 + ((uint32_t)(s ^ ((t >> 2) & 1)) << 4);
              stmatrix_t4(addr, blk[o][0][2 * u], blk[o][1][2 * u], blk[o][0][2 * u + 1], blk[o][1][2 * u + 1]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              const int x = o == 0 ? fcol : (o == 1 ? p.f + fcol : fcol);
              bulk_store(o == 2 ? &tmC1 : &tmC0, x, y, buf);
              asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            bi = (bi + 1) & (C::NBUF - 1);
          }
        } else if (K == DH) {
          asm volatile("cp.async.wait_group 1;" ::: "memory");   // this chunk's group; the next one may be in flight
          __syncwarp();
          const uint32_t abuf = wbuf + (uint32_t)bi * (2 * C::BUF_BYTES), bbuf = abuf + C::BUF_BYTES;
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int t = 8 * c + mrow;
            const uint32_t off = (uint32_t)t * 64 + ((uint32_t)(mi ^ ((t >> 1) & 3)) << 4);
            uint32_t qa[4], qb[4], da[4], db[4];
            ldmatrix_t4(abuf + off, qa);   // group g = features 8 g + T/4 of the warp
            ldmatrix_t4(bbuf + off, qb);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t *r = (g >> 1) ? r1 : r0;
              float av[2], bv[2], dd[2], de[2];
              av[0] = __uint_as_float(qa[g] << 16);
              av[1] = __uint_as_float(qa[g] & 0xffff0000u);
              bv[0] = __uint_as_float(qb[g] << 16);
              bv[1] = __uint_as_float(qb[g] & 0xffff0000u);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const float dh = __uint_as_float(r[4 * c + 2 * (g & 1) + h]), a = av[h], sg = sigmoidf_(a);
                dd[h] = dh * bv[h] * sg * (1.0f + a * (1.0f - sg));
                de[h] = dh * a * sg;
              }
              da[g] = pack_bf16x2(dd[0], dd[1]);
              db[g] = pack_bf16x2(de[0], de[1]);
            }
            stmatrix_t4(abuf + off, da[0], da[1], da[2], da[3]);
            stmatrix_t4(bbuf + off, db[0], db[1], db[2], db[3]);
          }
          __syncwarp();
          // da, db out with plain 16-byte stores (lane: 16-byte column q of token rows lane / 4 + 8 i),
          // so the buffer pair is free as soon as the warp has read it: a TMA store would hold it
          // until the SM's TMA unit, busy with the ring's loads, got round to reading it.
          {
            const int q = lane & 3;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int t = (lane >> 2) + 8 * i;
              const uint32_t so = (uint32_t)t * 64 + ((uint32_t)(q ^ ((t >> 1) & 3)) << 4);
              const uint4 va = ld_shared_v4(abuf + so), vb = ld_shared_v4(bbuf + so);
              if (y + t < p.rows_max) {
                __nv_bfloat16 *dst = p.out0 + (int64_t)(y + t) * p.ld0 + fcol + 8 * q;
                *reinterpret_cast<uint4 *>(dst) = va;
                *reinterpret_cast<uint4 *>(dst + p.f) = vb;
              }
            }
          }
          __syncwarp();
          issue_load(bi);   // the chunk two ahead reuses this buffer pair
          __syncwarp();
          bi ^= 1;
        } else {   // DOWN, DGRAD
          const uint32_t buf = wbuf + (uint32_t)bi * C::BUF_BYTES;
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          __syncwarp();
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int t = 8 * c + mrow;
            const uint32_t addr = buf + (uint32_t)t * 64 + ((uint32_t)(mi ^ ((t >> 1) & 3)) << 4);
            stmatrix_t4(addr, pack_bf16x2(__uint_as_float(r0[4 * c]), __uint_as_float(r0[4 * c + 1])),
                        pack_bf16x2(__uint_as_float(r0[4 * c + 2]), __uint_as_float(r0[4 * c + 3])),
                        pack_bf16x2(__uint_as_float(r1[4 * c]), __uint_as_float(r1[4 * c + 1])),
                        pack_bf16x2(__uint_as_float(r1[4 * c + 2]), __uint_as_float(r1[4 * c + 3])));
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            bulk_store(&tmC0, fcol, y, buf);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
          bi ^= 1;
        }
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      // the expert's padding rows after its last computed token: zeros, 32 rows per step
      const int zend = (int64_t)t.zero_end < p.rows_max ? t.zero_end : (int)p.rows_max;
      for (int y = t.start + t.nt + 32 * hh; y + 32 <= zend; y += 64) {
        if (K == GATEUP) {
          if (p.out0) {
            zero_rows(p.out0, p.ld0, y, fcol, 16, lane);
            zero_rows(p.out0, p.ld0, y, p.f + fcol, 16, lane);
          }
          zero_rows(p.out1, p.ld1, y, fcol, 16, lane);
        } else if (K == DH) {
          zero_rows(p.out0, p.ld0, y, fcol, 32, lane);
          zero_rows(p.out0, p.ld0, y, p.f + fcol, 32, lane);
        } else {
          zero_rows(p.out0, p.ld0, y, fcol, 32, lane);
        }
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (K == DH) asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();   // no CTA leaves while its peer may still signal its barriers or use its TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)TMEM_COLS)
                 : "memory");
  }
}

// A persistent grid of as many CTA pairs as can be resident at once (at most one per tile).
template <int K, bool G = false>
static int launch(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c0, const CUtensorMap &c1,
                  const Params &p, int64_t max_tiles, cudaStream_t s) {
  constexpr int smem = Cfg<K, G>::SMEM;
  constexpr int threads = G ? THREADS_G : THREADS;
  MOE_TRY_CUDA(cudaFuncSetAttribute(rows_kernel<K, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  int resident = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count() / 2 * 2), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  if (cudaOccupancyMaxActiveClusters(&resident, rows_kernel<K, G>, &cfg) != cudaSuccess || resident < 1) {
    (void)cudaGetLastError();
    resident = sm_count() / 2;
  }
  int64_t clusters = resident;
  if (max_tiles < clusters) clusters = max_tiles;
  if (clusters < 1) clusters = 1;
  rows_kernel<K, G><<<(int)(2 * clusters), threads, smem, s>>>(a, b, c0, c1, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // namespace rows
}  // namespace tc

// Host entry points used by gemm_tc.cu. The token tiles of one launch number at most
// sum_e ceil(c_e / 256) <= rows_max / 128.
int rows_gateup(const void *x_perm, const void *wgu, const int32_t *tile_offsets, const int32_t *offsets, int E, int d,
                int f, int64_t rows_max, void *ab, void *h, WsHeader *hdr, cudaStream_t s) {
  using namespace tc;
  using namespace tc::rows;
  CUtensorMap mA, mB, mC0, mC1;   // ab == nullptr: a, b are not stored (mC0 is then a stand-in, unused)
  if (!make_gateup_map(&mA, wgu, E, f, d) || !make_map(&mB, x_perm, rows_max, d, TOK_ROWS) ||
      !(ab ? make_store_map16(&mC0, ab, rows_max, 2 * f) : make_store_map16(&mC0, h, rows_max, f)) ||
      !make_store_map16(&mC1, h, rows_max, f))
    return MOE_ERR_CUDA;
  rows::Params p{};
  p.tile_offsets = tile_offsets;
  p.offsets = offsets;
  p.hdr = hdr;
  p.E = E;
  p.rows_max = rows_max;
  p.n_ft = f / 128;
  p.num_kb = d / Cfg<GATEUP>::BKP;
  p.f = f;
  p.out0 = (__nv_bfloat16 *)ab;
  p.ld0 = 2 * (int64_t)f;
  p.out1 = (__nv_bfloat16 *)h;
  p.ld1 = f;
  return launch<GATEUP>(mA, mB, mC0, mC1, p, (rows_max / 128) * p.n_ft, s);
}

// GEMM1 with the permutation fused into its token-operand load: rows of x [T, d] gathered by
// token_of_row (grouped row -> token, -1 on padding rows) instead of read from x_perm.
int rows_gateup_gather(const void *x, const int32_t *token_of_row, int T, const void *wgu, const int32_t *tile_offsets,
                       const int32_t *offsets, int E, int d, int f, int64_t rows_max, void *ab, void *h, WsHeader *hdr,
                       cudaStream_t s) {
  using namespace tc;
  using namespace tc::rows;
  CUtensorMap mA, mC0, mC1;   // ab == nullptr: a, b are not stored (mC0 is then a stand-in, unused)
  if (!make_gateup_map(&mA, wgu, E, f, d) ||
      !(ab ? make_store_map16(&mC0, ab, rows_max, 2 * f) : make_store_map16(&mC0, h, rows_max, f)) ||
      !make_store_map16(&mC1, h, rows_max, f))
    return MOE_ERR_CUDA;
  rows::Params p{};
  p.tile_offsets = tile_offsets;
  p.offsets = offsets;
  p.hdr = hdr;
  p.E = E;
  p.rows_max = rows_max;
  p.n_ft = f / 128;
  p.num_kb = d / Cfg<GATEUP, true>::BKP;
  p.f = f;
  p.out0 = (__nv_bfloat16 *)ab;
  p.ld0 = 2 * (int64_t)f;
  p.out1 = (__nv_bfloat16 *)h;
  p.ld1 = f;
  p.gx = (const __nv_bfloat16 *)x;
  p.tor = token_of_row;
  p.ldgx = d;
  p.ntok = T;
  return launch<GATEUP, true>(mA, mA, mC0, mC1, p, (rows_max / 128) * p.n_ft, s);
}

int rows_down(const void *h, const void *wd, const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f,
              int64_t rows_max, void *y, WsHeader *hdr, cudaStream_t s) {
  using namespace tc;
  using namespace tc::rows;
  CUtensorMap mA, mB, mC;
  if (!make_map(&mA, wd, (uint64_t)E * d, f, LANES) || !make_map(&mB, h, rows_max, f, TOK_ROWS) ||
      !make_store_map(&mC, y, rows_max, d))
    return MOE_ERR_CUDA;
  rows::Params p{};
  p.tile_offsets = tile_offsets;
  p.offsets = offsets;
  p.hdr = hdr;
  p.E = E;
  p.rows_max = rows_max;
  p.n_ft = d / 256;
  p.num_kb = f / Cfg<DOWN>::BKP;
  p.a_rows_e = d;
  p.out0 = (__nv_bfloat16 *)y;
  p.ld0 = d;
  return launch<DOWN>(mA, mB, mC, mC, p, (rows_max / 128) * p.n_ft, s);
}

int rows_dh(const void *dy, const void *wd, const void *ab, const int32_t *tile_offsets, const int32_t *offsets, int E,
            int d, int f, int64_t rows_max, void *dab, WsHeader *hdr, cudaStream_t s) {
  using namespace tc;
  using namespace tc::rows;
  CUtensorMap mA, mB, mC, mAB;
  if (!make_map(&mA, wd, (uint64_t)E * d, f, Cfg<DH>::BKP) || !make_map(&mB, dy, rows_max, d, TOK_ROWS) ||
      !make_store_map(&mC, dab, rows_max, 2 * f) || !make_store_map(&mAB, ab, rows_max, 2 * f))
    return MOE_ERR_CUDA;
  rows::Params p{};
  p.tile_offsets = tile_offsets;
  p.offsets = offsets;
  p.hdr = hdr;
  p.E = E;
  p.rows_max = rows_max;
  p.n_ft = f / 256;
  p.num_kb = d / Cfg<DH>::BKP;
  p.a_rows_e = d;
  p.f = f;
  p.out0 = (__nv_bfloat16 *)dab;
  p.ld0 = 2 * (int64_t)f;
  p.in0 = (const __nv_bfloat16 *)ab;
  return launch<DH>(mA, mB, mC, mAB, p, (rows_max / 128) * p.n_ft, s);
}

int rows_dgrad(const void *dab, const void *wgu, const int32_t *tile_offsets, const int32_t *offsets, int E, int d,
               int f, int64_t rows_max, void *dx, WsHeader *hdr, cudaStream_t s) {
  using namespace tc;
  using namespace tc::rows;
  CUtensorMap mA, mB, mC;
  if (!make_map(&mA, wgu, (uint64_t)E * 2 * f, d, Cfg<DGRAD>::BKP) || !make_map(&mB, dab, rows_max, 2 * f, TOK_ROWS) ||
      !make_store_map(&mC, dx, rows_max, d))
    return MOE_ERR_CUDA;
  rows::Params p{};
  p.tile_offsets = tile_offsets;
  p.offsets = offsets;
  p.hdr = hdr;
  p.E = E;
  p.rows_max = rows_max;
  p.n_ft = d / 256;
  p.num_kb = 2 * f / Cfg<DGRAD>::BKP;
  p.a_rows_e = 2 * f;
  p.out0 = (__nv_bfloat16 *)dx;
  p.ld0 = d;
  return launch<DGRAD>(mA, mB, mC, mC, p, (rows_max / 128) * p.n_ft, s);
}

}  // namespace moe
