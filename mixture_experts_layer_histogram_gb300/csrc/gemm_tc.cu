// Grouped GEMM over every expert's SwiGLU FFN on the 5th-generation tensor cores (sm_103a).
//
// "Scalable Pretraining of Large MoE LMs on Aurora", brief, section 核心方法: the experts'
// computation is merged into one grouped GEMM; summary page, section 关键设计: with optimised
// matrix multiplication and activation. Here one persistent, warp-specialised kernel per GEMM:
//
//   warp 0      TMA producer: 128B-swizzled tiles of A and B into a 4-stage shared-memory ring
//   warp 1      allocates the 512 TMEM columns, issues tcgen05.mma (one thread), commits to barriers
//   warps 2..9  epilogue: tcgen05.ld of the fp32 accumulator (double-buffered in TMEM, 2 x 256
//               columns) -> fused SwiGLU / SwiGLU-backward / plain -> bf16 -> global; two warps
//               share each 32-lane TMEM quarter and take one half of the tile's columns each
//
// Tile 128 x 256 x 64 (bf16 in, fp32 accumulate). Every expert's row group is padded to 128 rows,
// so every tile belongs to one expert and is full; the tile scheduler walks the flattened tile
// list with a static stride of gridDim.x and finds the expert of a row tile by binary search over
// tile_offsets. Five kinds share the kernel:
//   GATEUP  [a | b] = x_perm Wgu[e]^T  (B = 128 gate rows + the matching 128 up rows), epilogue
//           writes a, b and h = silu(a) * b
//   DOWN    y = h Wd[e]^T
//   DH      dh = dy Wd[e]  (B read MN-major), epilogue reads a, b and writes da, db
//   DGRAD   dx = dab Wgu[e] (B read MN-major)
//   WGRAD   dW[e] = act1_e^T act2_e over expert e's rows (A and B read MN-major, K = rows of e)
// Every wait is bounded (0.2 s); on timeout the kernel records MOE_ERR_DEVICE_TIMEOUT in the
// workspace status word, lets in-flight copies and MMAs land, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"

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
constexpr int MAX_E = MOE_MAX_EXPERTS;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256 + (MAX_E + 1) * 4;

enum Kind { GATEUP = 0, DOWN = 1, DH = 2, DGRAD = 3, WGRAD = 4 };

struct Params {
  const int32_t *tile_offsets;
  WsHeader *hdr;
  int E, d, f;
  int n_tiles;        // output tiles along N
  int m_tiles;        // WGRAD: output tiles along M' per expert
  int num_kb;         // row-grouped kinds: K / BK
  int b_rows_e;       // rows of the weight's 2D view per expert
  __nv_bfloat16 *out0;
  int64_t ld0;
  __nv_bfloat16 *out1;
  int64_t ld1;
  const __nv_bfloat16 *aux;
  int64_t ld_aux;
  int64_t out_e_stride;
};

// ----------------------------------------------------------------------------- PTX wrappers ----
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with parity `parity` of barrier `bar`. False = gave up (timeout or abort).
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, WsHeader *hdr,
                                       int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      report(hdr, MOE_ERR_DEVICE_TIMEOUT, where);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05), 128-byte swizzle, SM100 descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, M = 128, N = 256, K-major unless *_mn.
__host__ __device__ constexpr uint32_t idesc_bf16(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// ----------------------------------------------------------------------------- scheduling ------
struct Tile {
  int e;       // expert
  int m0;      // first grouped row (row-grouped kinds) or first row of dW[e] (WGRAD)
  int n0;      // first output column (GATEUP: first gate column)
  int kb;      // number of BK blocks
  int krow0;   // WGRAD: first grouped row of expert e
};

template <int KIND>
__device__ __forceinline__ Tile decode(int tile, const Params &p, const int *toff) {
  Tile t;
  if (KIND == WGRAD) {
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
    t.n0 = nt * (KIND == GATEUP ? BN / 2 : BN);
    t.kb = p.num_kb;
    t.krow0 = 0;
  }
  return t;
}

// ----------------------------------------------------------------------------- epilogues -------
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16 *dst, const float *v) {   // 32 values, 64 B
  uint4 *q = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = pack_bf16x8(v + 8 * i);
}

// Columns [c0, c0 + cols) of the accumulator (GATEUP: of each half) for one row of the tile.
template <int KIND>
__device__ __forceinline__ void epilogue_tile(const Tile &t, const Params &p, uint32_t tbase, int row_in_tile,
                                              int c0, const uint4 (&pre)[8]) {
  float v[32];
  uint32_t r[32];
  if (KIND == GATEUP) {
    const int64_t grow = t.m0 + row_in_tile;
    __nv_bfloat16 *ab = p.out0 + grow * p.ld0;
    __nv_bfloat16 *h = p.out1 + grow * p.ld1;
#pragma unroll 1
    for (int c = c0; c < c0 + BN / 4; c += 32) {
      uint32_t rb[32];
      tmem_ld32(tbase + c, r);
      tmem_ld32(tbase + BN / 2 + c, rb);
      tmem_ld_wait();
      float hv[32], bv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a = __uint_as_float(r[i]), b = __uint_as_float(rb[i]);
        v[i] = a;
        bv[i] = b;
        hv[i] = a * sigmoidf_(a) * b;
      }
      store_row_bf16(ab + t.n0 + c, v);
      store_row_bf16(ab + p.f + t.n0 + c, bv);
      store_row_bf16(h + t.n0 + c, hv);
    }
  } else if (KIND == DH) {
    // a and b of the current 32 columns arrive one chunk ahead (the first chunk was loaded
    // before the accumulator was ready): the loads' latency overlaps the previous chunk's work.
    const int64_t grow = t.m0 + row_in_tile;
    const __nv_bfloat16 *abrow = p.aux + grow * p.ld_aux;
    __nv_bfloat16 *dab = p.out0 + grow * p.ld0;
    uint4 cur[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cur[i] = pre[i];
#pragma unroll 1
    for (int c = c0; c < c0 + BN / 2; c += 32) {
      uint4 nxt[8];
      if (c + 32 < c0 + BN / 2) {
        const uint4 *qa = reinterpret_cast<const uint4 *>(abrow + t.n0 + c + 32);
        const uint4 *qb = reinterpret_cast<const uint4 *>(abrow + p.f + t.n0 + c + 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          nxt[i] = qa[i];
          nxt[4 + i] = qb[i];
        }
      }
      tmem_ld32(tbase + c, r);
      float av[32], bv[32], db[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        unpack_bf16x8(cur[i], av + 8 * i);
        unpack_bf16x8(cur[4 + i], bv + 8 * i);
      }
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float dh = __uint_as_float(r[i]), a = av[i], s = sigmoidf_(a);
        v[i] = dh * bv[i] * s * (1.0f + a * (1.0f - s));
        db[i] = dh * a * s;
      }
      store_row_bf16(dab + t.n0 + c, v);
      store_row_bf16(dab + p.f + t.n0 + c, db);
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
    }
  } else {
    __nv_bfloat16 *dst;
    if (KIND == WGRAD) dst = p.out0 + (int64_t)t.e * p.out_e_stride + (int64_t)(t.m0 + row_in_tile) * p.ld0 + t.n0;
    else dst = p.out0 + (int64_t)(t.m0 + row_in_tile) * p.ld0 + t.n0;
#pragma unroll 1
    for (int c = c0; c < c0 + BN / 2; c += 32) {
      tmem_ld32(tbase + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      store_row_bf16(dst + c, v);
    }
  }
}

// ----------------------------------------------------------------------------- the kernel ------
template <int KIND>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
  constexpr bool A_MN = (KIND == WGRAD);
  constexpr bool B_MN = (KIND == DH || KIND == DGRAD || KIND == WGRAD);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], mma_done
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  int *toff = reinterpret_cast<int *>(tmem_holder + 4);

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
  for (int i = threadIdx.x; i <= p.E; i += THREADS) toff[i] = p.tile_offsets[i];
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

  const int num_tiles = (KIND == WGRAD) ? p.E * p.m_tiles * p.n_tiles : toff[p.E] * p.n_tiles;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;   // bit s: stage s has a load whose completion nobody has waited for yet
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const Tile t = decode<KIND>(tile, p, toff);
      bool ok = true;
      for (int kb = 0; kb < t.kb; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.hdr, 1)) { ok = false; break; }
        const uint32_t sA = sbase + stage * STAGE_BYTES, sB = sA + A_BYTES, fb = full_bar(stage);
        mbar_expect_tx(fb, STAGE_BYTES);
        issued |= 1u << stage;
        const int kx = kb * BK;
        if (KIND == GATEUP) {
          tma_load_2d(sA, &tmA, kx, t.m0, fb);
          tma_load_2d(sB, &tmB, kx, t.e * p.b_rows_e + t.n0, fb);
          tma_load_2d(sB + B_BYTES / 2, &tmB, kx, t.e * p.b_rows_e + p.f + t.n0, fb);
        } else if (KIND == DOWN) {
          tma_load_2d(sA, &tmA, kx, t.m0, fb);
          tma_load_2d(sB, &tmB, kx, t.e * p.b_rows_e + t.n0, fb);
          tma_load_2d(sB + B_BYTES / 2, &tmB, kx, t.e * p.b_rows_e + t.n0 + BN / 2, fb);
        } else if (KIND == DH || KIND == DGRAD) {
          tma_load_2d(sA, &tmA, kx, t.m0, fb);
#pragma unroll
          for (int q = 0; q < BN / 64; ++q) tma_load_2d(sB + q * 8192, &tmB, t.n0 + 64 * q, t.e * p.b_rows_e + kx, fb);
        } else {   // WGRAD
#pragma unroll
          for (int q = 0; q < BM / 64; ++q) tma_load_2d(sA + q * 8192, &tmA, t.m0 + 64 * q, t.krow0 + kx, fb);
#pragma unroll
          for (int q = 0; q < BN / 64; ++q) tma_load_2d(sB + q * 8192, &tmB, t.n0 + 64 * q, t.krow0 + kx, fb);
        }
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
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16(A_MN, B_MN);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool issued_any = false;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const Tile t = decode<KIND>(tile, p, toff);
      if (t.kb == 0) continue;
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.hdr, 2)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      bool ok = true;
      for (int kb = 0; kb < t.kb; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.hdr, 3)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sA = sbase + stage * STAGE_BYTES, sB = sA + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = A_MN ? sdesc(sA + kk * 2048, 8192, 1024) : sdesc(sA + kk * 32, 16, 1024);
          const uint64_t bd = B_MN ? sdesc(sB + kk * 2048, 8192, 1024) : sdesc(sB + kk * 32, 16, 1024);
          mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        issued_any = true;
        mma_commit(empty_bar(stage));   // frees the smem stage once these MMAs have read it
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      mma_commit(tfull_bar(acc));       // accumulator ready for the epilogue
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (issued_any) {   // every MMA must have completed before TMEM is released
      mma_commit(mma_done_bar);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(mma_done_bar, 0) && global_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                       // TMEM lanes this warp may access: 32 * quarter ...
    const int half = (warp - 2) >> 2;                   // which half of the tile's columns
    const int row_in_tile = quarter * 32 + lane;
    const int c0 = half * (KIND == GATEUP ? BN / 4 : BN / 2);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const Tile t = decode<KIND>(tile, p, toff);
      if (t.kb == 0) {   // WGRAD of an expert with no rows: the gradient is zero
        __nv_bfloat16 *dst =
            p.out0 + (int64_t)t.e * p.out_e_stride + (int64_t)(t.m0 + row_in_tile) * p.ld0 + t.n0 + c0;
        uint4 *q = reinterpret_cast<uint4 *>(dst);
        for (int i = 0; i < BN / 16; ++i) q[i] = make_uint4(0, 0, 0, 0);
        continue;
      }
      uint4 pre[8];
      if (KIND == DH) {   // first chunk of a, b: independent of the MMA, load before waiting
        const __nv_bfloat16 *abrow = p.aux + (int64_t)(t.m0 + row_in_tile) * p.ld_aux + t.n0 + c0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pre[i] = reinterpret_cast<const uint4 *>(abrow)[i];
          pre[4 + i] = reinterpret_cast<const uint4 *>(abrow + p.f)[i];
        }
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.hdr, 4)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      epilogue_tile<KIND>(t, p, tbase, row_in_tile, c0, pre);
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)TMEM_COLS)
                 : "memory");
  }
}

// ----------------------------------------------------------------------------- host side -------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2D bf16 row-major [rows, cols], box = 64 columns (128 B, the swizzle span) x box_rows rows.
static bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND>
static int launch(const CUtensorMap &a, const CUtensorMap &b, const Params &p, int64_t max_tiles, cudaStream_t s) {
  MOE_TRY_CUDA(cudaFuncSetAttribute(tc_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
  int64_t grid = sm_count();
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  tc_gemm_kernel<KIND><<<(int)grid, THREADS, SMEM_BYTES, s>>>(a, b, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // namespace tc

// Entry points used by the C ABI (gemm_api.cu).
int tc_grouped_ffn_fwd(const void *x_perm, const void *wgu, const void *wd, const int32_t *tile_offsets, int E, int d,
                       int f, int64_t rows_max, void *ab, void *h, void *y, WsHeader *hdr, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB;
  Params p{};
  p.tile_offsets = tile_offsets;
  p.hdr = hdr;
  p.E = E;
  p.d = d;
  p.f = f;
  const int64_t row_tiles = rows_max / BM;
  // GEMM1: [a | b] = x_perm Wgu^T, SwiGLU epilogue
  if (!make_map(&mA, x_perm, rows_max, d, 128) || !make_map(&mB, wgu, (uint64_t)E * 2 * f, d, 128))
    return MOE_ERR_CUDA;
  p.n_tiles = f / (BN / 2);
  p.num_kb = d / BK;
  p.b_rows_e = 2 * f;
  p.out0 = (__nv_bfloat16 *)ab;
  p.ld0 = 2 * (int64_t)f;
  p.out1 = (__nv_bfloat16 *)h;
  p.ld1 = f;
  int rc = launch<GATEUP>(mA, mB, p, row_tiles * p.n_tiles, s);
  if (rc) return rc;
  // GEMM2: y = h Wd^T
  if (!make_map(&mA, h, rows_max, f, 128) || !make_map(&mB, wd, (uint64_t)E * d, f, 128)) return MOE_ERR_CUDA;
  p.n_tiles = d / BN;
  p.num_kb = f / BK;
  p.b_rows_e = d;
  p.out0 = (__nv_bfloat16 *)y;
  p.ld0 = d;
  p.out1 = nullptr;
  return launch<DOWN>(mA, mB, p, row_tiles * p.n_tiles, s);
}

int tc_grouped_ffn_bwd(const void *dy, const void *x_perm, const void *ab, const void *h, const void *wgu,
                       const void *wd, const int32_t *tile_offsets, int E, int d, int f, int64_t rows_max, void *dab,
                       void *dx, void *dwgu, void *dwd, WsHeader *hdr, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB;
  Params p{};
  p.tile_offsets = tile_offsets;
  p.hdr = hdr;
  p.E = E;
  p.d = d;
  p.f = f;
  const int64_t row_tiles = rows_max / BM;
  int rc;
  // dh = dy Wd[e] (Wd read MN-major), SwiGLU backward epilogue -> dab
  if (!make_map(&mA, dy, rows_max, d, 128) || !make_map(&mB, wd, (uint64_t)E * d, f, 64)) return MOE_ERR_CUDA;
  p.n_tiles = f / BN;
  p.num_kb = d / BK;
  p.b_rows_e = d;
  p.out0 = (__nv_bfloat16 *)dab;
  p.ld0 = 2 * (int64_t)f;
  p.aux = (const __nv_bfloat16 *)ab;
  p.ld_aux = 2 * (int64_t)f;
  if ((rc = launch<DH>(mA, mB, p, row_tiles * p.n_tiles, s))) return rc;
  // dWd[e] = dy_e^T h_e
  if (!make_map(&mA, dy, rows_max, d, 64) || !make_map(&mB, h, rows_max, f, 64)) return MOE_ERR_CUDA;
  p.m_tiles = d / BM;
  p.n_tiles = f / BN;
  p.out0 = (__nv_bfloat16 *)dwd;
  p.ld0 = f;
  p.out_e_stride = (int64_t)d * f;
  p.aux = nullptr;
  if ((rc = launch<WGRAD>(mA, mB, p, (int64_t)E * p.m_tiles * p.n_tiles, s))) return rc;
  // dx_perm = dab Wgu[e] (Wgu read MN-major)
  if (!make_map(&mA, dab, rows_max, 2 * f, 128) || !make_map(&mB, wgu, (uint64_t)E * 2 * f, d, 64))
    return MOE_ERR_CUDA;
  p.n_tiles = d / BN;
  p.num_kb = 2 * f / BK;
  p.b_rows_e = 2 * f;
  p.out0 = (__nv_bfloat16 *)dx;
  p.ld0 = d;
  if ((rc = launch<DGRAD>(mA, mB, p, row_tiles * p.n_tiles, s))) return rc;
  // dWgu[e] = dab_e^T x_perm_e
  if (!make_map(&mA, dab, rows_max, 2 * f, 64) || !make_map(&mB, x_perm, rows_max, d, 64)) return MOE_ERR_CUDA;
  p.m_tiles = 2 * f / BM;
  p.n_tiles = d / BN;
  p.out0 = (__nv_bfloat16 *)dwgu;
  p.ld0 = d;
  p.out_e_stride = (int64_t)2 * f * d;
  return launch<WGRAD>(mA, mB, p, (int64_t)E * p.m_tiles * p.n_tiles, s);
}

}  // namespace moe
