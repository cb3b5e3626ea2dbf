// Grouped GEMMs on the 5th-generation tensor cores (sm_103a) whose reduction runs over the rows of
// a group: the expert weight gradients, and the router's backward.
//
// "Scalable Pretraining of Large MoE LMs on Aurora", brief, section 核心方法: the experts'
// computation is merged into one grouped GEMM, and (sections 为什么值得记录 / 关键结果) the module is
// measured on the forward-backward pass. The kinds whose output rows are grouped tokens (GATEUP,
// DOWN, DH, DGRAD) live in gemm_rows.cu; this file holds the rest, in two persistent,
// warp-specialised kernels:
//   WGRAD   dW[e] = act1_e^T act2_e over expert e's rows (A and B read MN-major, K = the expert's
//           padded row count; experts without rows get zero gradients without touching TMEM), on
//           the CTA-pair kernel (tcgen05.mma.cta_group::2, 256 x 256 tiles, the pairs run along the
//           weight rows, six 64-deep ring stages; the epilogue writes dW with plain coalesced
//           stores from a staging buffer)
//   RDX     dx (+)= dL Wr (B read MN-major; the epilogue adds the previous dx when asked), and
//   RDW     fp32 partial dWr = dL_g^T x_g over token range g (A and B MN-major), plain fp32 stores,
//           the router backward's two kinds, on the single-CTA kernel (one "group" = all tokens for
//           RDX, one token range per group for RDW):
//
//   warp 0      TMA producer: 128B-swizzled tiles of A and B into a shared-memory ring (the whole
//               warp polls, one elected lane issues)
//   warp 1      allocates the 512 TMEM columns, issues tcgen05.mma from one elected lane of the
//               converged warp, commits to barriers
//   warps 2..9  epilogue: tcgen05.ld of the fp32 accumulator (double-buffered in TMEM, 2 x 256
//               columns) -> bf16 or fp32 -> global; two warps share each 32-lane TMEM quarter and
//               take one half of the tile's columns each
//
// Every wait is bounded (0.2 s); on timeout the kernel records MOE_ERR_DEVICE_TIMEOUT in the
// workspace status word, lets in-flight copies and MMAs land, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = BN * BK * 2;        // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;                // two warps per TMEM lane quarter, each drains half the columns
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int THREADS = 64 + EPI_THREADS;
constexpr int TMEM_COLS = 2 * BN;           // two fp32 accumulators of 128 lanes x 256 columns
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 32 * 32 * 2 * 2 * EPI_WARPS + 1024 + 256;

// (the values name the kernel instantiations; the row-grouped kinds 0..3 are in gemm_rows.cu)
enum Kind { WGRAD = 4, RDX = 5, RDW = 6 };
// kinds whose tiles reduce over the rows of one group (A and B read MN-major)
__host__ __device__ constexpr bool row_reduce(int kind) { return kind == WGRAD || kind == RDW; }
// 16-byte vectors an epilogue thread of RDX loads before its accumulator is ready: its row's whole
// addend (128 columns)
constexpr int PRE = 16;

struct Params {
  const int32_t *tile_offsets;
  const int32_t *offsets;   // WGRAD: [E+1] exclusive scan of the routed row counts
  WsHeader *hdr;
  int E, d, f;
  int n_tiles;        // output tiles along N
  int m_tiles;        // WGRAD: output tiles along M' per expert
  int num_kb;         // RDX: K / BK
  __nv_bfloat16 *out0;
  int64_t ld0;
  const __nv_bfloat16 *aux;
  int64_t ld_aux;
  int64_t out_e_stride;
  const __nv_bfloat16 *gx;   // WGRAD gathering: B rows are the tokens x [ntok, ldgx] of ...
  const int32_t *tor;        // ... each grouped row (-1 on padding rows) instead of rows of x_perm
  int64_t ldgx;
  int ntok;
  float *outf;        // RDW: fp32 partials [groups, rows_valid, ldf]
  int64_t ldf;
  int rows_valid;     // RDX: rows of dx (tokens); RDW: rows of dWr (experts)
  int64_t rows_max;   // WGRAD: rows of the grouped operands (debug-build bound on the rows read)
};

// Instruction descriptor, kind::f16: D fp32, A and B bf16, M = 128, N = 256, K-major unless *_mn.
__host__ __device__ constexpr uint32_t idesc_bf16(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// ----------------------------------------------------------------------------- scheduling ------
struct Tile {
  int e;       // expert
  int m0;      // RDX: first token row; WGRAD, RDW: first row of the weight gradient
  int n0;      // first output column
  int kb;      // number of BK blocks
  int krow0;   // WGRAD, RDW: first grouped row of the group
  bool ok;     // debug build (WGRAD): the tile passed its consistency checks (always true otherwise)
};

template <int KIND>
__device__ __forceinline__ Tile decode(int tile, const Params &p, const int *toff) {
  Tile t;
  if (row_reduce(KIND)) {
    const int per = p.m_tiles * p.n_tiles;
    t.e = tile / per;
    const int r = tile - t.e * per;
    t.m0 = (r / p.n_tiles) * BM;
    t.n0 = (r % p.n_tiles) * BN;
    t.krow0 = toff[t.e] * BM;
    t.kb = (toff[t.e + 1] - toff[t.e]) * (BM / BK);
  } else {
    const int rt = tile / p.n_tiles;
    const int nt = tile - rt * p.n_tiles;
    int lo = 0, hi = p.E - 1;   // last expert whose first row tile is <= rt
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (toff[mid] <= rt) lo = mid;
      else hi = mid - 1;
    }
    t.e = lo;
    t.m0 = rt * BM;
    t.n0 = nt * BN;
    t.kb = p.num_kb;
    t.krow0 = 0;
  }
  return t;
}

// ----------------------------------------------------------------------------- epilogues -------
// Output path: each epilogue warp converts 32 rows x 32 columns to bf16, writes them into one of
// its two 2 KB shared-memory buffers (64-byte swizzle: 16-byte chunk c of row r goes to chunk
// c ^ ((r >> 1) & 3), which keeps the 32 lanes' writes free of bank conflicts), and one lane
// stores the block with a TMA bulk tensor store. The L2 then sees whole-line writes instead of
// one 16-byte partial-sector request per thread and row.
constexpr int EPI_BUF_BYTES = 32 * 32 * 2;                 // one 32 x 32 bf16 block
constexpr int EPI_STAGE_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;

struct EpiStore {
  uint32_t buf;   // this warp's two buffers (shared::cta address, 1024-aligned region)
  int bi;
  int lane;
  __device__ __forceinline__ void put(const CUtensorMap *map, int x, int y, const float *v) {
    const uint32_t b = buf + (uint32_t)bi * EPI_BUF_BYTES;
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");   // b's previous store has read it
    __syncwarp();
    const uint32_t row = b + (uint32_t)lane * 64, sw = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 q = pack_bf16x8(v + 8 * c);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c ^ sw) << 4)), "r"(q.x), "r"(q.y), "r"(q.z),
                   "r"(q.w)
                   : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the TMA (async proxy)
    __syncwarp();
    if (lane == 0) {
      asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                       reinterpret_cast<uint64_t>(map)),
                   "r"(x), "r"(y), "r"(b)
                   : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    bi ^= 1;
  }
  // The same 32 x 32 block written with plain 16-byte stores from the staging buffer (four lanes per
  // 64-byte row, eight rows per instruction): block row i goes to out + (y + i) ld + x. In the
  // weight-gradient kernel TMA stores queued with the ring's operand loads in the SM's TMA unit and
  // left the MMA waiting for data; these stores do not.
  __device__ __forceinline__ void put_plain(__nv_bfloat16 *out, int64_t ld, int x, int y, const float *v) {
    const uint32_t b = buf;
    const uint32_t row = b + (uint32_t)lane * 64, sw = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 q = pack_bf16x8(v + 8 * c);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c ^ sw) << 4)), "r"(q.x), "r"(q.y), "r"(q.z),
                   "r"(q.w)
                   : "memory");
    }
    __syncwarp();
    const int q = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rr = (lane >> 2) + 8 * i;
      uint4 val;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                   : "r"(b + (uint32_t)rr * 64 + (((uint32_t)q ^ (((uint32_t)rr >> 1) & 3u)) << 4))
                   : "memory");
      *reinterpret_cast<uint4 *>(out + (int64_t)(y + rr) * ld + x + 8 * q) = val;
    }
    __syncwarp();   // the buffer is rewritten by the next block
  }
  __device__ __forceinline__ void drain() {
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }
};

// Columns [c0, c0 + BN / 2) of the accumulator for the warp's 32 rows; `row` is this thread's row
// in the tile, `yrow` the global row (in the output map) of the warp's first row.
template <int KIND>
__device__ __forceinline__ void epilogue_tile(const Tile &t, const Params &p, uint32_t tbase, int row, int yrow, int c0,
                                              const uint4 (&pre)[PRE], EpiStore &es, const CUtensorMap *mc0) {
  float v[32];
  uint32_t r[32];
  if (KIND == RDW) {
    // fp32 partial of token range t.e; rows are experts, stored for the first rows_valid only
    const int er = t.m0 + row;
    float *dst = p.outf + ((int64_t)t.e * p.rows_valid + er) * p.ldf + t.n0;
#pragma unroll 1
    for (int c = c0; c < c0 + BN / 2; c += 32) {
      tmem_ld32(tbase + c, r);
      tmem_ld_wait();
      if (er < p.rows_valid) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (t.n0 + c + 4 * q < p.d)
            *reinterpret_cast<float4 *>(dst + c + 4 * q) =
                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
                            __uint_as_float(r[4 * q + 3]));
      }
    }
  } else {
    // RDX: with an addend, this row's previous dx, loaded in full (pre) before the accumulator was
    // ready (zeros past the tokens and past d)
    const bool add = p.aux != nullptr;
#pragma unroll
    for (int cc = 0; cc < BN / 64; ++cc) {
      const int c = c0 + 32 * cc;
      tmem_ld32(tbase + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      if (add) {
        float av[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) unpack_bf16x8(pre[4 * cc + i], av + 8 * i);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += av[i];
      }
      es.put(mc0, t.n0 + c, yrow, v);
    }
  }
}

// Global row (in the output tensor map) of the first of the 32 rows a warp stores.
template <int KIND>
__device__ __forceinline__ int epi_yrow(const Tile &t, const Params &p, int quarter) {
  return KIND == WGRAD ? t.e * (p.m_tiles * BM) + t.m0 + quarter * 32 : t.m0 + quarter * 32;
}

// ----------------------------------------------------------------------------- the kernel ------
template <int KIND>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC0, const Params p) {
  static_assert(KIND == RDX || KIND == RDW, "the single-CTA kernel runs the router's kinds");
  constexpr bool A_MN = row_reduce(KIND);
  constexpr bool B_MN = true;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *epi_smem = smem + STAGES * STAGE_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(epi_smem + EPI_STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], mma_done
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  const int *toff = p.tile_offsets;   // read through L1; shared memory goes to the ring

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), EPI_THREADS);
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"((uint32_t)TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int num_tiles = row_reduce(KIND) ? p.E * p.m_tiles * p.n_tiles : toff[p.E] * p.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp runs the loop and polls the ring, converged; one elected lane issues.
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;   // bit s: stage s has a load whose completion nobody has waited for yet
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const Tile t = decode<KIND>(tile, p, toff);
      bool ok = true;
      for (int kb = 0; kb < t.kb; ++kb) {
        if (!mbar_spin_cluster(empty_bar(stage), phase ^ 1u, abort_flag, p.hdr, 1)) { ok = false; break; }
        if (elect_one()) {
          const uint32_t sA = sbase + stage * STAGE_BYTES, sB = sA + A_BYTES, fb = full_bar(stage);
          mbar_expect_tx(fb, STAGE_BYTES);
          const int kx = kb * BK;
          if (KIND == RDX) {   // K-major A (dL rows), MN-major B (Wr; rows past E read as zero)
            tma_load_2d(sA, &tmA, kx, t.m0, fb);
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) tma_load_2d(sB + q * 8192, &tmB, t.n0 + 64 * q, kx, fb);
          } else {   // RDW
#pragma unroll
            for (int q = 0; q < BM / 64; ++q) tma_load_2d(sA + q * 8192, &tmA, t.m0 + 64 * q, t.krow0 + kx, fb);
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) tma_load_2d(sB + q * 8192, &tmB, t.n0 + 64 * q, t.krow0 + kx, fb);
          }
        }
        __syncwarp();
        issued |= 1u << stage;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    // Let every copy this thread issued land before the CTA can exit: wait for the last phase of
    // each used stage (normally already complete, since the MMA consumed it).
    for (int s = 0; s < STAGES; ++s) {
      if (!((issued >> s) & 1u)) continue;
      // stage s was last filled in phase `phase` if s < stage, else in phase ^ 1
      uint32_t ph = (s < stage) ? phase : (phase ^ 1u);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(full_bar(s), ph) && global_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp polls, one elected lane issues; the descriptors are formed once
    // (shared-memory addresses below 256 KB: an offset adds to the start-address field without carry).
    constexpr uint32_t idesc = idesc_bf16(A_MN, B_MN);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool issued_any = false;
    const uint64_t desc_a0 = A_MN ? sdesc(sbase, 8192, 1024) : sdesc(sbase, 16, 1024);
    const uint64_t desc_b0 = B_MN ? sdesc(sbase + A_BYTES, 8192, 1024) : sdesc(sbase + A_BYTES, 16, 1024);
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const Tile t = decode<KIND>(tile, p, toff);
      if (t.kb == 0) continue;
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.hdr, 2)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      bool ok = true;
      for (int kb = 0; kb < t.kb; ++kb) {
        if (!mbar_spin_cluster(full_bar(stage), phase, abort_flag, p.hdr, 3)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t so = (uint32_t)(stage * STAGE_BYTES) >> 4;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t ka = A_MN ? (uint32_t)(kk * 2048 >> 4) : (uint32_t)(kk * 32 >> 4);
            const uint32_t kb_ = B_MN ? (uint32_t)(kk * 2048 >> 4) : (uint32_t)(kk * 32 >> 4);
            mma_bf16(d_tmem, desc_a0 + so + ka, desc_b0 + so + kb_, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(empty_bar(stage));   // frees the smem stage once these MMAs have read it
        }
        __syncwarp();
        issued_any = true;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) mma_commit(tfull_bar(acc));   // accumulator ready for the epilogue
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (issued_any) {   // every MMA must have completed before TMEM is released
      if (elect_one()) mma_commit(mma_done_bar);
      __syncwarp();
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(mma_done_bar, 0) && global_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                       // TMEM lanes this warp may access: 32 * quarter ...
    const int half = (warp - 2) >> 2;                   // which half of the tile's columns
    const int row_in_tile = quarter * 32 + lane;
    const int c0 = half * (BN / 2);
    EpiStore es{smem_u32(epi_smem) + (uint32_t)(warp - 2) * 2 * EPI_BUF_BYTES, 0, lane};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const Tile t = decode<KIND>(tile, p, toff);
      if (t.kb == 0) {   // RDW, a token range with no rows: its partial is zero
        const int er = t.m0 + row_in_tile;
        if (er < p.rows_valid) {
          float *dst = p.outf + ((int64_t)t.e * p.rows_valid + er) * p.ldf + t.n0 + c0;
          for (int i = 0; i < BN / 2; i += 4)
            if (t.n0 + c0 + i < p.d) *reinterpret_cast<float4 *>(dst + i) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        continue;
      }
      uint4 pre[PRE];
      if (KIND == RDX && p.aux != nullptr) {   // the addend row: independent of the MMA, load before waiting
        const bool live = t.m0 + row_in_tile < p.rows_valid;
        const __nv_bfloat16 *arow = p.aux + (int64_t)(live ? t.m0 + row_in_tile : 0) * p.ld_aux + t.n0 + c0;
#pragma unroll
        for (int i = 0; i < PRE; ++i)
          pre[i] = (live && t.n0 + c0 + 8 * i < p.d) ? reinterpret_cast<const uint4 *>(arow)[i] : make_uint4(0, 0, 0, 0);
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.hdr, 4)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      epilogue_tile<KIND>(t, p, tbase, row_in_tile, epi_yrow<KIND>(t, p, quarter), c0, pre, es, &tmC0);
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    es.drain();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)TMEM_COLS)
                 : "memory");
  }
}

// ----------------------------------------------------------------------------- CTA-pair kernel --
// The weight gradients on a cluster of two CTAs (one TPC): tcgen05.mma.cta_group::2 computes a
// 256 x 256 tile of dW[e]; CTA r holds rows [128 r, 128 r + 128) of A (weight rows m0 + 128 r) and
// half r of B (N rows [128 r, 128 r + 128)) in its own shared memory, and receives its 128 rows x
// 256 columns of the accumulator in its own TMEM. Each SM therefore loads 32 KB per 64-deep k-block
// instead of 48 KB for the same MMA work. The leader (rank 0) issues the MMAs; both CTAs' TMA loads
// complete on the leader's full barrier; the MMA commits multicast to both CTAs' empty /
// accumulator-full barriers; both epilogues arrive on the leader's accumulator-empty barrier. The
// pairs run along the weight rows, so no tile is discarded; K is the expert's padded row count.
// Tile order. A tile's time grows with its expert's rows, which vary up to about 8x the mean under
// skewed routing. The tiles are therefore taken in order of decreasing K (experts sorted by row
// count, ties to the lower expert id; an expert's tiles stay adjacent, so the clusters that share
// its activations run together) and dealt to the clusters in a snake: round r gives position p to
// cluster p on even rounds and to cluster C - 1 - p on odd ones, a static form of
// longest-first scheduling.
// The ring has six 64-deep stages of 32 KB: a load's latency under full load is about as long for
// 32 KB as for 64 KB, so six small stages keep more of it covered than three large ones. Gathering
// (G) keeps three 128-deep stages, one per loader set.
template <bool G> struct PairCfg {
  static constexpr int BKP = G ? 128 : 64;                // k depth of one ring stage
  static constexpr int A_BYTES = BM * BKP * 2;            // this CTA's 128 rows of A
  static constexpr int B_BYTES = (BN / 2) * BKP * 2;      // this CTA's half of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = G ? 3 : 6;
  static constexpr int EPI_BYTES = EPI_STAGE_BYTES;
  static constexpr int NBARS = 2 * STAGES + 5;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 8 * NBARS + 16 + MOE_MAX_EXPERTS * 4;
  static_assert(EPI_BYTES >= MOE_MAX_EXPERTS * 4, "the set-up borrows the epilogue buffers");
  static_assert(SMEM <= 232448, "pair kernel shared memory exceeds 227 KB");
};

// Instruction descriptor for the pair MMA: M = 256 (128 rows per CTA), N = 256, A and B MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16_pair_mn() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)((2 * BM) >> 4) << 24);
}

// Tile position of round r for cluster c of C (the snake), or -1 past the last tile.
__device__ __forceinline__ int snake_tile(int r, int c, int C, int num_tiles) {
  const int s = r * C + ((r & 1) ? C - 1 - c : c);
  return s < num_tiles ? s : -1;
}

// a / b for a >= 0 and b > 0, given rb = 1 / b in float: below 2^22 the float quotient is within
// one of the true one; the remainder steps correct it (exactly, for any a).
__device__ __forceinline__ int div_small(int a, int b, float rb) {
  int q = __float2int_rz(__int2float_rn(a) * rb);
  int r = a - q * b;
  while (r < 0) {
    --q;
    r += b;
  }
  while (r >= b) {
    ++q;
    r -= b;
  }
  return q;
}

// The weight-gradient tiles a cluster runs, in its snake order, decoded one ahead: the expert's group
// offsets are loaded from global memory while the previous tile runs, so a tile boundary costs the
// ring only a few instructions. Tile s (in order of decreasing K) is expert order[s / per], row pair
// and N tile of s % per, seen from CTA `rank`; t.kb counts ring stages of bkp rows.
struct WgradWalker {
  int r, cluster, clusters, num_tiles, per, rank, bkp;
  float rper, rnt;
  int s, e, k0, k1, c;   // the next tile, its expert's toff[e], toff[e + 1] and routed row count
  const int *toff, *order, *offs;

  __device__ __forceinline__ WgradWalker(int cluster_, int clusters_, int num_tiles_, const Params &p,
                                         const int *toff_, const int *order_, int rank_, int bkp_)
      : r(0), cluster(cluster_), clusters(clusters_), num_tiles(num_tiles_), rank(rank_), bkp(bkp_), toff(toff_),
        order(order_), offs(p.offsets) {
    per = (p.m_tiles / 2) * p.n_tiles;
    rper = 1.0f / (float)per;
    rnt = 1.0f / (float)p.n_tiles;
    load();
  }
  __device__ __forceinline__ void load() {
    s = snake_tile(r, cluster, clusters, num_tiles);
    if (s < 0) return;
    e = order[div_small(s, per, rper)];
    k0 = toff[e];
    k1 = toff[e + 1];
    c = offs[e + 1] - offs[e];
  }
  __device__ __forceinline__ bool next(Tile &t, const Params &p) {
    if (s < 0) return false;
    t.e = e;
    const int q = s - div_small(s, per, rper) * per;
    const int m = div_small(q, p.n_tiles, rnt);
    t.m0 = m * (2 * BM) + rank * BM;
    t.n0 = (q - m * p.n_tiles) * BN;
    t.krow0 = k0 * BM;
    t.kb = (c + bkp - 1) / bkp;   // up to the last k-block that holds a routed row; the rest is zero padding
#if MOE_CHECKS
    // the expert's group is non-empty-or-empty in order, its routed rows fit it, and the rows it
    // reduces over lie inside the buffers
    t.ok = k0 <= k1 && c >= 0 && c <= (k1 - k0) * BM && (int64_t)k1 * BM <= p.rows_max;
    if (!t.ok) t.kb = 0;
#else
    t.ok = true;
#endif
    ++r;
    load();
    return true;
  }
};

// G: B (x_perm for dW_gate_up) is gathered from x by token_of_row with cp.async by loader warps
// instead of loaded by TMA (the permutation fused into the operand load): three sets of two warps,
// one set per ring slot.
constexpr int LOADER_WARPS = 2, LOADER_SETS = 3;
template <bool G>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(G ? THREADS + 32 * LOADER_WARPS * LOADER_SETS : THREADS, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC0, const Params p) {
  using Cfg = PairCfg<G>;
  constexpr int PS = Cfg::STAGES;
  constexpr int P_BK = Cfg::BKP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *epi_smem = smem + PS * Cfg::STAGE_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(epi_smem + Cfg::EPI_BYTES);
  // bars: full[PS], empty[PS], tfull[2], tempty[2], mma_done
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + Cfg::NBARS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  int *order = reinterpret_cast<int *>(tmem_holder + 4);   // experts by decreasing row count
  int *kbs = reinterpret_cast<int *>(epi_smem);            // row tiles of each expert (set-up only)
  const int *toff = p.tile_offsets;   // read through L1; shared memory goes to the ring

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
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) kbs[e] = toff[e + 1] - toff[e];
  __syncthreads();
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {   // rank of e: experts with more rows, or as many and a lower id
    const int k = kbs[e];
    int rk = 0;
    for (int j = 0; j < p.E; ++j) rk += (kbs[j] > k) || (kbs[j] == k && j < e);
    order[rk] = e;
  }
  __syncthreads();
  if (warp == 1) {   // collective TMEM allocation by one warp of each CTA of the pair
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"((uint32_t)TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();   // both CTAs: barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int num_tiles = p.E * (p.m_tiles / 2) * p.n_tiles;
  const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    // The whole warp runs the loop and waits, converged; one elected lane issues the copies.
    int stage = 0;
    uint32_t phase = 0;
    WgradWalker walk(cluster_id, num_clusters, num_tiles, p, toff, order, (int)rank, P_BK);
    for (Tile t; walk.next(t, p);) {
      const int bn = t.n0 + (int)rank * (BN / 2);   // this CTA's half of B
      bool ok = true;
      for (int kb = 0; kb < t.kb; ++kb) {
        if (!mbar_spin_cluster(empty_bar(stage), phase ^ 1u, abort_flag, p.hdr, 11)) { ok = false; break; }
        if (elect_one()) {
          const uint32_t sA = sbase + stage * Cfg::STAGE_BYTES, sB = sA + Cfg::A_BYTES;
          const uint32_t fb = mapa_shared(full_bar(stage), 0);   // the leader's full barrier
          if (leader) mbar_expect_tx(full_bar(stage), 2 * (G ? Cfg::A_BYTES : Cfg::STAGE_BYTES));
          const int ky = t.krow0 + kb * P_BK;
#pragma unroll
          for (int q = 0; q < 2; ++q) tma_load_2d_pair(sA + q * (P_BK * 128), &tmA, t.m0 + 64 * q, ky, fb);
          if (!G) {
#pragma unroll
            for (int q = 0; q < 2; ++q) tma_load_2d_pair(sB + q * (P_BK * 128), &tmB, bn + 64 * q, ky, fb);
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
    constexpr uint32_t idesc = idesc_bf16_pair_mn();
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool issued_any = false;
    const uint64_t desc_a0 = sdesc(sbase, P_BK * 128, 1024);
    const uint64_t desc_b0 = sdesc(sbase + Cfg::A_BYTES, P_BK * 128, 1024);
    WgradWalker walk(cluster_id, num_clusters, num_tiles, p, toff, order, 0, P_BK);
    for (Tile t; walk.next(t, p);) {
      if (!t.ok || t.kb == 0) continue;
      if (!mbar_ready_cluster(tempty_bar(acc), acc_phase ^ 1u) &&
          !mbar_wait_cluster(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.hdr, 12))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      bool ok = true;
      for (int kb = 0; kb < t.kb; ++kb) {
        if (!mbar_spin_cluster(full_bar(stage), phase, abort_flag, p.hdr, 13)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t so = (uint32_t)(stage * Cfg::STAGE_BYTES) >> 4;
#pragma unroll
          for (int kk = 0; kk < P_BK / 16; ++kk) {
            // MN-major: 2048 B per 16 k-rows; the two 64-wide MN blocks are P_BK * 128 B apart.
            const uint32_t ko = (uint32_t)(kk * 2048) >> 4;
            mma_bf16_pair(d_tmem, desc_a0 + so + ko, desc_b0 + so + ko, idesc, (kb | kk) != 0 ? 1u : 0u);
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
    // B's k rows are the expert's grouped rows: loader set q (two warps) fills ring slot q, every
    // third fill, with the x rows of the stage's 128 k rows, 128 columns from this CTA's half of the
    // N tile, two boxes of 64 (see gather_rows).
    static_assert(!G || (Cfg::STAGES == LOADER_SETS && P_BK == 128), "one loader set of 128 rows per ring slot");
    const int lw = warp - (2 + EPI_WARPS);
    const int q = lw / LOADER_WARPS;
    const int chunk = lane & 7;
    const int rsub = (lw % LOADER_WARPS) * 4 + (lane >> 3);
    int fill = 0;
    uint32_t phase = 0;
    bool ok = true;
    WgradWalker walk(cluster_id, num_clusters, num_tiles, p, toff, order, (int)rank, P_BK);
    for (Tile t; ok && walk.next(t, p);) {
      if (!t.ok) continue;
      const int bn = t.n0 + (int)rank * (BN / 2);
      for (int kb = 0; kb < t.kb; ++kb, ++fill) {
        if (fill % PS != q) continue;
        int tok[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tk = p.tor[t.krow0 + kb * P_BK + 8 * j + rsub];
          tok[j] = tk >= p.ntok ? -1 : tk;   // an index past the tokens reads as padding
        }
        if (!mbar_spin_cluster(empty_bar(q), phase ^ 1u, abort_flag, p.hdr, 15)) { ok = false; break; }
        phase ^= 1u;
        gather_rows<2>(sbase + q * Cfg::STAGE_BYTES + Cfg::A_BYTES, P_BK * 128, p.gx, p.ldgx, tok, rsub, chunk, bn);
        gather_done(full_bar(q), lane);
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = quarter * 32 + lane;
    const int c0 = half * (BN / 2);
    EpiStore es{smem_u32(epi_smem) + (uint32_t)(warp - 2) * 2 * EPI_BUF_BYTES, 0, lane};
    int acc = 0;
    uint32_t acc_phase = 0;
    WgradWalker walk(cluster_id, num_clusters, num_tiles, p, toff, order, (int)rank, P_BK);
    for (Tile t; walk.next(t, p);) {
      if (!t.ok) continue;
      if (t.kb == 0) {   // an expert with no rows: its gradient is zero
        __nv_bfloat16 *dst =
            p.out0 + (int64_t)t.e * p.out_e_stride + (int64_t)(t.m0 + row_in_tile) * p.ld0 + t.n0 + c0;
        uint4 *q = reinterpret_cast<uint4 *>(dst);
        for (int i = 0; i < BN / 16; ++i) q[i] = make_uint4(0, 0, 0, 0);
        continue;
      }
      uint4 pre[PRE];   // unused by this kind
      if (!mbar_wait_cluster(tfull_bar(acc), acc_phase, abort_flag, p.hdr, 14)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      {   // dW blocks through the staging buffer with plain coalesced stores (see put_plain)
        const int yrow = epi_yrow<WGRAD>(t, p, quarter);
#pragma unroll 1
        for (int c = c0; c < c0 + BN / 2; c += 32) {
          uint32_t r[32];
          tmem_ld32(tbase + c, r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          es.put_plain(p.out0, p.ld0, t.n0 + c, yrow, v);
        }
        (void)pre;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    es.drain();
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

// ----------------------------------------------------------------------------- host side -------
// The single-CTA kernel (router kinds) on a persistent grid of min(SMs, max_tiles) CTAs.
template <int KIND>
static int launch_single(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c0, const Params &p,
                         int64_t max_tiles, cudaStream_t s) {
  MOE_TRY_CUDA(cudaFuncSetAttribute(tc_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
  int64_t grid = sm_count();
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  tc_gemm_kernel<KIND><<<(int)grid, THREADS, SMEM_BYTES, s>>>(a, b, c0, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

// The weight-gradient kind on a persistent grid of as many CTA pairs as can be resident at once.
template <bool G>
static int launch_wgrad(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c0, const Params &p,
                        int64_t max_pair_tiles, cudaStream_t s) {
  constexpr int smem = PairCfg<G>::SMEM;
  constexpr int threads = G ? THREADS + 32 * LOADER_WARPS * LOADER_SETS : THREADS;
  MOE_TRY_CUDA(cudaFuncSetAttribute(tc_pair_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  int resident = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count() / 2 * 2), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  if (cudaOccupancyMaxActiveClusters(&resident, tc_pair_kernel<G>, &cfg) != cudaSuccess || resident < 1) {
    (void)cudaGetLastError();
    resident = sm_count() / 2;
  }
  int64_t clusters = resident;
  if (max_pair_tiles < clusters) clusters = max_pair_tiles;
  if (clusters < 1) clusters = 1;
  tc_pair_kernel<G><<<(int)(2 * clusters), threads, smem, s>>>(a, b, c0, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // namespace tc

// Row-grouped kinds (gemm_rows.cu): weights as A, tokens as B, on CTA pairs.
int rows_gateup(const void *x_perm, const void *wgu, const int32_t *tile_offsets, const int32_t *offsets, int E, int d,
                int f, int64_t rows_max, void *ab, void *h, WsHeader *hdr, cudaStream_t s);
int rows_gateup_gather(const void *x, const int32_t *token_of_row, int T, const void *wgu, const int32_t *tile_offsets,
                       const int32_t *offsets, int E, int d, int f, int64_t rows_max, void *ab, void *h, WsHeader *hdr,
                       cudaStream_t s);
int rows_down(const void *h, const void *wd, const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f,
              int64_t rows_max, void *y, WsHeader *hdr, cudaStream_t s);
int rows_dh(const void *dy, const void *wd, const void *ab, const int32_t *tile_offsets, const int32_t *offsets, int E,
            int d, int f, int64_t rows_max, void *dab, WsHeader *hdr, cudaStream_t s);
int rows_dgrad(const void *dab, const void *wgu, const int32_t *tile_offsets, const int32_t *offsets, int E, int d,
               int f, int64_t rows_max, void *dx, WsHeader *hdr, cudaStream_t s);

// Entry points used by the C ABI (api.cu). The tokens come either permuted (x = x_perm [rows_max, d],
// token_of_row = nullptr) or in token order (x [T, d] and token_of_row): then GEMM1 and the gate/up
// weight gradient gather their token rows themselves and x_perm is never formed.
int tc_grouped_ffn_fwd(const void *x, const int32_t *token_of_row, int T, const void *wgu, const void *wd,
                       const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f, int64_t rows_max,
                       void *ab, void *h, void *y, WsHeader *hdr, cudaStream_t s) {
  // GEMM1: [a | b] = x_perm Wgu^T, SwiGLU epilogue
  int rc = token_of_row
               ? rows_gateup_gather(x, token_of_row, T, wgu, tile_offsets, offsets, E, d, f, rows_max, ab, h, hdr, s)
               : rows_gateup(x, wgu, tile_offsets, offsets, E, d, f, rows_max, ab, h, hdr, s);
  if (rc || y == nullptr) return rc;   // y == nullptr: GEMM1 only (recompute of ab, h)
  // GEMM2: y = h Wd^T
  return rows_down(h, wd, tile_offsets, offsets, E, d, f, rows_max, y, hdr, s);
}

int tc_grouped_ffn_bwd(const void *dy, const void *x, const int32_t *token_of_row, int T, const void *ab, const void *h,
                       const void *wgu, const void *wd, const int32_t *tile_offsets, const int32_t *offsets, int E, int d,
                       int f, int64_t rows_max, void *dab, void *dx, void *dwgu, void *dwd, WsHeader *hdr,
                       cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB, mC;
  Params p{};
  p.tile_offsets = tile_offsets;
  p.offsets = offsets;
  p.hdr = hdr;
  p.E = E;
  p.d = d;
  p.f = f;
  p.rows_max = rows_max;
  int rc;
  // dh = dy Wd[e] (Wd read MN-major), SwiGLU backward epilogue -> dab
  if ((rc = rows_dh(dy, wd, ab, tile_offsets, offsets, E, d, f, rows_max, dab, hdr, s))) return rc;
  // dWd[e] = dy_e^T h_e (the weight-gradient kind runs on the CTA-pair kernel, whose stage depth its maps take)
  if (!make_map(&mA, dy, rows_max, d, PairCfg<false>::BKP) || !make_map(&mB, h, rows_max, f, PairCfg<false>::BKP) ||
      !make_store_map(&mC, dwd, (uint64_t)E * d, f))
    return MOE_ERR_CUDA;
  p.m_tiles = d / BM;
  p.n_tiles = f / BN;
  p.out0 = (__nv_bfloat16 *)dwd;
  p.ld0 = f;
  p.out_e_stride = (int64_t)d * f;
  if ((rc = launch_wgrad<false>(mA, mB, mC, p, (int64_t)E * (p.m_tiles / 2) * p.n_tiles, s)))
    return rc;
  // dx_perm = dab Wgu[e] (Wgu read MN-major)
  if ((rc = rows_dgrad(dab, wgu, tile_offsets, offsets, E, d, f, rows_max, dx, hdr, s))) return rc;
  // dWgu[e] = dab_e^T x_perm_e (x_perm's rows gathered from x when token_of_row is given)
  const int bkp = token_of_row ? PairCfg<true>::BKP : PairCfg<false>::BKP;
  if (!make_map(&mA, dab, rows_max, 2 * f, bkp) || !make_store_map(&mC, dwgu, (uint64_t)E * 2 * f, d))
    return MOE_ERR_CUDA;
  if (!token_of_row && !make_map(&mB, x, rows_max, d, bkp)) return MOE_ERR_CUDA;
  p.m_tiles = 2 * f / BM;
  p.n_tiles = d / BN;
  p.out0 = (__nv_bfloat16 *)dwgu;
  p.ld0 = d;
  p.out_e_stride = (int64_t)2 * f * d;
  const int64_t pair_tiles = (int64_t)E * (p.m_tiles / 2) * p.n_tiles;
  if (token_of_row) {
    p.gx = (const __nv_bfloat16 *)x;
    p.tor = token_of_row;
    p.ldgx = d;
    p.ntok = T;
    return launch_wgrad<true>(mA, mA, mC, p, pair_tiles, s);
  }
  return launch_wgrad<false>(mA, mB, mC, p, pair_tiles, s);
}

// Router backward GEMMs (router.cu prepares dl16, the bf16 copy of d_logits [t_pad, ek] with zero
// padding, and the group offsets in 128-row tiles).
// dx (+)= dL Wr: one group of t_pad / 128 row tiles; B = Wr [E, d] read MN-major (rows >= E read as 0).
int tc_router_dx(const void *dl16, int64_t t_pad, int ek, const void *wr, int E, int d, int T,
                 const int32_t *toff, void *dx, bool accumulate, WsHeader *hdr, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB, mC;
  if (!make_map(&mA, dl16, t_pad, ek, 128) || !make_map(&mB, wr, E, d, BK) || !make_store_map(&mC, dx, T, d))
    return MOE_ERR_CUDA;
  Params p{};
  p.tile_offsets = toff;
  p.hdr = hdr;
  p.E = 1;
  p.d = d;
  p.n_tiles = (d + BN - 1) / BN;
  p.num_kb = ek / BK;
  p.out0 = (__nv_bfloat16 *)dx;
  p.ld0 = d;
  p.aux = accumulate ? (const __nv_bfloat16 *)dx : nullptr;
  p.ld_aux = d;
  p.rows_valid = T;
  return launch_single<RDX>(mA, mB, mC, p, (t_pad / BM) * p.n_tiles, s);
}

// fp32 partials part[g] = dL_g^T x_g for the G token ranges of toff_split (in 128-row tiles).
int tc_router_dw(const void *dl16, int64_t t_pad, int ek, const void *x, int T, int d, int E,
                 const int32_t *toff_split, int G, float *part, WsHeader *hdr, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB;
  if (!make_map(&mA, dl16, t_pad, ek, BK) || !make_map(&mB, x, T, d, BK)) return MOE_ERR_CUDA;
  Params p{};
  p.tile_offsets = toff_split;
  p.hdr = hdr;
  p.E = G;
  p.d = d;
  p.m_tiles = (E + BM - 1) / BM;
  p.n_tiles = (d + BN - 1) / BN;
  p.outf = part;
  p.ldf = d;
  p.rows_valid = E;
  return launch_single<RDW>(mA, mB, mA, p, (int64_t)G * p.m_tiles * p.n_tiles, s);
}

}  // namespace moe
