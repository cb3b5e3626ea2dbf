// Router: logits L = x Wr^T with the top-k selection and renormalised softmax fused into the
// GEMM's epilogue, and the router's backward (dx (+)= dL Wr, dWr = dL^T x).
//
// "Scalable Pretraining of Large MoE LMs on Aurora", summary page, section 关键设计: expert
// selection ahead of the token counting; brief, section 核心方法: the FastSparseMoE module, of
// which routing is the first step.
//
// bf16 forward, one tcgen05 kernel (router_fwd_kernel):
//   warp 0      TMA producer: 128-token x 64 tiles of x and all E rows x 64 of Wr (128B swizzle),
//               a ring of up to 8 stages
//   warp 1      allocates TMEM (two accumulators of 128 lanes x E columns), issues tcgen05.mma
//               with M = 128 tokens, N = E rounded up to 16 (rows of Wr past E read as zero)
//   warps 2..9  epilogue, two threads per token (warps 2..5 and 6..9 share the TMEM lane quarters
//               and split the columns): tcgen05.ld of the token's logits, 32 at a time, optional
//               store of the fp32 logits, insertion into a sorted top-k list held in registers
//               (value desc, id asc); the two lists merge through shared memory, then the softmax
//               of the selected logits
// When there are fewer token tiles than SMs, S (<= 4) CTAs share a tile, each over 1/S of d: each
// writes fp32 partial logits to the workspace and the last one to finish (an atomic count per tile)
// adds the S partials in split order (deterministic) and selects. x is read once either way; Wr
// stays in L2.
//
// bf16 backward: router_prep_kernel writes dl16 = bf16(dL) [t_pad, ek] with zero padding and the
// group offsets; the single-CTA grouped-GEMM kernel runs its RDX kind (dx (+)= dl16 Wr) and its
// RDW kind (fp32 partial dWr per token range); router_reduce_kernel sums the partials in a fixed
// order and writes dWr in bf16.
//
// fp32: SIMT FFMA kernels (router_simt_kernel) and the moe_route_topk kernel.
#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace moe {
int tc_router_dx(const void *dl16, int64_t t_pad, int ek, const void *wr, int E, int d, int T, const int32_t *toff,
                 void *dx, bool accumulate, WsHeader *hdr, cudaStream_t s);
int tc_router_dw(const void *dl16, int64_t t_pad, int ek, const void *x, int T, int d, int E,
                 const int32_t *toff_split, int G, float *part, WsHeader *hdr, cudaStream_t s);

namespace router {
using namespace tc;

constexpr int RBM = 128;                 // tokens per tile (TMEM lanes)
constexpr int RBK = 64;                  // k depth of one stage (128 B of bf16: the swizzle span)
constexpr int R_THREADS = 320;           // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int R_EPI_THREADS = 256;       // two threads per token: each takes half of the experts
constexpr int R_A_BYTES = RBM * RBK * 2; // 16 KB
constexpr int R_RING_BYTES = 192 * 1024;
constexpr int R_MAX_STAGES = 8;
constexpr int R_MERGE_BYTES = RBM * MOE_MAX_TOPK * 8;   // upper-half top-k lists handed to the lower half
constexpr int R_SMEM = R_RING_BYTES + R_MERGE_BYTES + 1024 + 8 * (2 * R_MAX_STAGES + 5) + 16;
constexpr int kSplitTarget = 152;        // RDW: aim for about one output tile per SM
constexpr int kMaxSplits = 64;

struct FwdParams {
  WsHeader *hdr;
  int T, E, k;
  int n_mma;       // MMA N: E rounded up to 16
  int acc_cols;    // TMEM columns per accumulator (power of two >= 32 and >= E rounded up to 32)
  int stages;
  int stage_bytes;
  int num_kb;      // ceil(d / 64)
  int num_tiles;   // ceil(T / 128)
  int splits;      // S: CTAs that share one token tile, each over kb_split k-blocks of d
  int kb_split;
  float *partial;          // S > 1: fp32 partial logits [S, T, E]
  uint32_t *tile_count;    // S > 1: per-tile count of finished splits (zero at launch)
  float *logits;   // may be null
  int32_t *topk_idx;
  float *topk_w;
};

// True on every epilogue thread (the 256 threads of warps 2..9) if `v` holds on any of them.
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(R_EPI_THREADS)
      : "memory");
  return r != 0;
}

// One token's logits for columns [c0, c0 + 32): optional store of the fp32 logits, then insertion
// into the top-k list.
template <int KMAX>
__device__ __forceinline__ void take_chunk(const float (&v)[32], int c0, int E, bool live, float *lrow, bool vec,
                                           float (&tv)[KMAX], int (&ti)[KMAX]) {
  if (live && lrow) {
    if (vec) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c0 + 4 * q < E)
          *reinterpret_cast<float4 *>(lrow + c0 + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c0 + i < E) lrow[c0 + i] = v[i];
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) {   // leave at the row's end: predicated-off insertions still issue
    if (c0 + i >= E) break;
    topk_insert<KMAX>(tv, ti, v[i], c0 + i);
  }
}

template <int KMAX>
__global__ void __launch_bounds__(R_THREADS, 1)
    router_fwd_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  float *merge_v = reinterpret_cast<float *>(smem + R_RING_BYTES);            // [MOE_MAX_TOPK][RBM]
  int *merge_i = reinterpret_cast<int *>(smem + R_RING_BYTES + R_MERGE_BYTES / 2);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + R_RING_BYTES + R_MERGE_BYTES);
  // bars: full[S], empty[S], tfull[2], tempty[2], mma_done
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * R_MAX_STAGES + 5);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  volatile int *last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (R_MAX_STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * R_MAX_STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * R_MAX_STAGES + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * R_MAX_STAGES + 4);
  const uint32_t tmem_cols = 2u * (uint32_t)p.acc_cols;
  const int splits = p.splits;
  const int num_units = p.num_tiles * splits;   // unit u: tile u / splits, split u % splits

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), R_EPI_THREADS);
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    *last_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp runs the loop and polls the ring, converged; one elected lane issues. Each
    // stage carries little tensor work here, so the hand-off per stage sets the kernel's pace.
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const int tile = u / splits, kb0 = (u - tile * splits) * p.kb_split;
      const int kb1 = min(p.num_kb, kb0 + p.kb_split);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_spin_cluster(empty_bar(stage), phase ^ 1u, abort_flag, p.hdr, 11)) { ok = false; break; }
        if (elect_one()) {
          const uint32_t sA = sbase + stage * p.stage_bytes, fb = full_bar(stage);
          mbar_expect_tx(fb, p.stage_bytes);
          tma_load_2d(sA, &tmX, kb * RBK, tile * RBM, fb);
          tma_load_2d(sA + R_A_BYTES, &tmW, kb * RBK, 0, fb);
        }
        __syncwarp();
        issued |= 1u << stage;
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
    for (int s = 0; s < S; ++s) {   // every issued copy lands before the CTA may exit
      if (!((issued >> s) & 1u)) continue;
      const uint32_t ph = (s < stage) ? phase : (phase ^ 1u);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(full_bar(s), ph) && global_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // kind::f16, D fp32, A and B bf16 K-major, M = 128, N = n_mma. The whole warp polls, one
    // elected lane issues; the descriptors are formed once (shared-memory addresses below 256 KB:
    // a stage's or k step's offset adds to the start-address field without carry).
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(p.n_mma >> 3) << 17) |
                           ((uint32_t)(RBM >> 4) << 24);
    const uint64_t desc_a0 = sdesc(sbase, 16, 1024), desc_b0 = sdesc(sbase + R_A_BYTES, 16, 1024);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool issued_any = false, ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const int tile = u / splits, kb0 = (u - tile * splits) * p.kb_split;
      const int kb1 = min(p.num_kb, kb0 + p.kb_split);
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.hdr, 12)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.acc_cols);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_spin_cluster(full_bar(stage), phase, abort_flag, p.hdr, 13)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t so = (uint32_t)(stage * p.stage_bytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < RBK / 16; ++kk)
            mma_bf16(d_tmem, desc_a0 + so + (uint32_t)(kk * 2), desc_b0 + so + (uint32_t)(kk * 2), idesc,
                     (kb != kb0 || kk != 0) ? 1u : 0u);
          mma_commit(empty_bar(stage));
        }
        __syncwarp();
        issued_any = true;
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) mma_commit(tfull_bar(acc));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (issued_any) {
      if (elect_one()) mma_commit(mma_done_bar);
      __syncwarp();
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(mma_done_bar, 0) && global_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue: two threads per token
    // Warps 2..5 (half 0) and 6..9 (half 1) share the TMEM lane quarters; in each pair the thread
    // of half h takes the 32-column chunks [h * nc0, ...) of its token's logits, keeps its own
    // top-k list, and half 1 hands its list to half 0 through shared memory for the final merge.
    const int quarter = warp & 3;   // TMEM lanes 32 * quarter ... 32 * quarter + 31
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const int E = p.E, k = p.k;
    const int nc = (E + 31) / 32, nc0 = (nc + 1) / 2;
    const int cbeg = half ? nc0 * 32 : 0, cend = half ? E : (nc0 * 32 < E ? nc0 * 32 : E);
    const bool vec = (E & 3) == 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const int tile = u / splits, split = u - tile * splits;
      const bool got = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.hdr, 14);
      if (epi_any(!got)) break;   // all epilogue threads leave together: they meet at named barriers
      tc_fence_after();
      const int t = tile * RBM + row;
      const bool live = t < p.T;
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * p.acc_cols);
      float *lrow = p.logits ? p.logits + (int64_t)t * E : nullptr;
      float tv[KMAX];
      int ti[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        tv[j] = -INFINITY;
        ti[j] = 0;
      }
      bool last = true;
      if (splits == 1) {
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
          uint32_t r[32];
          float v[32];
          tmem_ld32(tbase + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          take_chunk<KMAX>(v, c0, E, live, lrow, vec, tv, ti);
        }
        tc_fence_before();
        mbar_arrive(tempty_bar(acc));
      } else {
        // this split's partial logits -> global; the last split of the tile to finish adds all
        // partials in split order and selects
        float *prow = p.partial + ((int64_t)split * p.T + t) * E;
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tbase + c0, r);
          tmem_ld_wait();
          if (live) {
            if (vec) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                if (c0 + 4 * q < E)
                  *reinterpret_cast<float4 *>(prow + c0 + 4 * q) =
                      make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                  __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c0 + i < E) prow[c0 + i] = __uint_as_float(r[i]);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(tempty_bar(acc));
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"n"(R_EPI_THREADS) : "memory");
        if (warp == 2 && lane == 0) {
          const unsigned old = atomicAdd(p.tile_count + tile, 1u);
          __threadfence();
          *last_flag = old == (unsigned)(splits - 1);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(R_EPI_THREADS) : "memory");
        last = *last_flag != 0;
        if (last) {
#pragma unroll 1
          for (int c0 = cbeg; c0 < cend; c0 += 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            if (live) {
              if (vec) {
#pragma unroll
                for (int q = 0; q < 4; ++q)   // at most 4 splits; the loads of all of them can be in flight
                  if (q < splits) {
                    const float4 *src = reinterpret_cast<const float4 *>(p.partial + ((int64_t)q * p.T + t) * E + c0);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                      if (c0 + 4 * j < E) {
                        const float4 f = __ldcg(src + j);
                        v[4 * j] += f.x;
                        v[4 * j + 1] += f.y;
                        v[4 * j + 2] += f.z;
                        v[4 * j + 3] += f.w;
                      }
                  }
              } else {
                for (int q = 0; q < splits; ++q) {
                  const float *src = p.partial + ((int64_t)q * p.T + t) * E + c0;
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    if (c0 + i < E) v[i] += __ldcg(src + i);
                }
              }
            }
            take_chunk<KMAX>(v, c0, E, live, lrow, vec, tv, ti);
          }
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      if (!last) continue;   // uniform across the epilogue threads
      // merge: half 1 hands its list to half 0 (its experts have the higher ids, and its list is in
      // (value desc, id asc) order, so inserting it entry by entry keeps the tie rule)
      if (half == 1) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          merge_v[j * RBM + row] = tv[j];
          merge_i[j * RBM + row] = ti[j];
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(R_EPI_THREADS) : "memory");
      if (half == 0) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) topk_insert<KMAX>(tv, ti, merge_v[j * RBM + row], merge_i[j * RBM + row]);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(R_EPI_THREADS) : "memory");   // merge buffer free again
      if (half == 0 && live) {
        const float m = tv[0];
        float ex[KMAX], s = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          ex[j] = j < k ? expf(tv[j] - m) : 0.0f;
          s += ex[j];
        }
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) {
            p.topk_idx[(int64_t)t * k + j] = ti[j];
            p.topk_w[(int64_t)t * k + j] = ex[j] / s;
          }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(tmem_cols) : "memory");
  }
}

// ---------------------------------------------------------------------------------------------
// Backward preparation: dl16[t, e] = bf16(dL[t, e]) for t < T, e < E, zero elsewhere in
// [t_pad, ek]; toff_dx = {0, t_pad / 128}; toff_dw[g] = floor(g * tiles / G) (token ranges).
__global__ void __launch_bounds__(256) router_prep_kernel(const float *__restrict__ dl, int T, int E, int64_t t_pad,
                                                          int ek, __nv_bfloat16 *__restrict__ dl16, int32_t *toff_dx,
                                                          int32_t *toff_dw, int G) {
  const int64_t groups = t_pad * (ek / 8);   // 8 bf16 (16 B) per thread and step
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < groups; i += stride) {
    const int64_t t = i / (ek / 8);
    const int e0 = (int)(i - t * (ek / 8)) * 8;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (t < T && e0 + j < E) ? __ldg(dl + t * E + e0 + j) : 0.0f;
    *reinterpret_cast<uint4 *>(dl16 + t * ek + e0) = pack_bf16x8(v);
  }
  if (blockIdx.x == 0) {
    const int tiles = (int)(t_pad / RBM);
    if (threadIdx.x == 0) {
      toff_dx[0] = 0;
      toff_dx[1] = tiles;
    }
    for (int g = threadIdx.x; g <= G; g += blockDim.x) toff_dw[g] = (int)((int64_t)g * tiles / G);
  }
}

// dWr[e, c] = sum_g part[g][e][c], g ascending, fp32 -> bf16 (G = 0 writes zeros).
__global__ void __launch_bounds__(256) router_reduce_kernel(const float *__restrict__ part, int G, int E, int d,
                                                            __nv_bfloat16 *__restrict__ dw) {
  const int64_t n4 = (int64_t)E * d / 4;   // d % 8 == 0
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t plane = (int64_t)E * d;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g0 = 0; g0 < G; g0 += 8) {   // eight partials' loads in flight, added in split order
      float4 q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        q[j] = g0 + j < G ? __ldg(reinterpret_cast<const float4 *>(part + (g0 + j) * plane) + i)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (g0 + j < G) {
          s.x += q[j].x;
          s.y += q[j].y;
          s.z += q[j].z;
          s.w += q[j].w;
        }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y), hi = __floats2bfloat162_rn(s.z, s.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&lo);
    o.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(dw)[i] = o;
  }
}

// ---------------------------------------------------------------------------------------------
// fp32: C[m, n] (+)= sum_k A(m, k) B(n, k) through (row, k) strides; 32 x 32 tiles, 256 threads,
// 4 outputs per thread. C may be the addend itself (each element is read and written by one thread).
constexpr int ST = 32;
__global__ void __launch_bounds__(256) router_simt_kernel(const float *__restrict__ A, int64_t sAm, int64_t sAk,
                                                          const float *__restrict__ B, int64_t sBn, int64_t sBk, int M,
                                                          int N, int K, float *C, int64_t ldc, bool accumulate) {
  __shared__ float As[ST][ST + 1], Bs[ST][ST + 1];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int m0 = blockIdx.y * ST, n0 = blockIdx.x * ST;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < K; k0 += ST) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = ty + 8 * i, kk = k0 + tx;
      As[r][tx] = (m0 + r < M && kk < K) ? A[(int64_t)(m0 + r) * sAm + (int64_t)kk * sAk] : 0.0f;
      Bs[r][tx] = (n0 + r < N && kk < K) ? B[(int64_t)(n0 + r) * sBn + (int64_t)kk * sBk] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < ST; ++kk) {
      const float b = Bs[tx][kk];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = fmaf(As[ty + 8 * i][kk], b, acc[i]);
    }
    __syncthreads();
  }
  const int n = n0 + tx;
  if (n >= N) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 8 * i;
    if (m >= M) continue;
    float *c = C + (int64_t)m * ldc + n;
    *c = accumulate ? *c + acc[i] : acc[i];
  }
}

static int simt_gemm(const float *A, int64_t sAm, int64_t sAk, const float *B, int64_t sBn, int64_t sBk, int M, int N,
                     int K, float *C, int64_t ldc, bool accumulate, cudaStream_t s) {
  if (M == 0 || N == 0) return MOE_OK;
  dim3 grid((N + ST - 1) / ST, (M + ST - 1) / ST);
  router_simt_kernel<<<grid, 256, 0, s>>>(A, sAm, sAk, B, sBn, sBk, M, N, K, C, ldc, accumulate);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

// ---------------------------------------------------------------------------------------------
// Workspace layout (bf16): [header 256 B][toff_dx: 4 int32][toff_dw: kMaxSplits + 1 int32]
//                          (padded to 1 KB)[dl16: t_pad x ek bf16][part: G x E x d fp32]
//                  (fp32): [header 256 B][logits scratch: T x E fp32]
constexpr size_t kHdrBytes = 256;
constexpr size_t kToffBytes = 768;

static int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
static int64_t t_pad_of(int T) { return round_up(T, RBM); }
static int ek_of(int E) { return (int)round_up(E, RBK); }
static int splits_of(int T, int d, int E) {
  const int64_t tiles = t_pad_of(T) / RBM;
  if (tiles == 0) return 0;
  const int64_t per = ((E + RBM - 1) / RBM) * ((d + 255) / 256);   // output tiles of one split
  int64_t g = (kSplitTarget + per - 1) / per;
  if (g > tiles) g = tiles;
  if (g > kMaxSplits) g = kMaxSplits;
  return (int)(g < 1 ? 1 : g);
}
static size_t dl16_bytes(int T, int E) { return (size_t)round_up((int64_t)t_pad_of(T) * ek_of(E) * 2, 256); }

// Forward: S CTAs share a token tile when there are few tiles, so that about one CTA per SM streams
// x (S <= 4, each split at least one 64-wide k-block). Depends on the shape only.
constexpr int kFwdCtaTarget = 152;
static void fwd_splits(int T, int d, int *splits, int *kb_split) {
  const int tiles = (int)(t_pad_of(T) / RBM), num_kb = (d + RBK - 1) / RBK;
  int S = tiles > 0 ? kFwdCtaTarget / tiles : 1;
  if (S > 4) S = 4;
  if (S > num_kb) S = num_kb;
  if (S < 1) S = 1;
  const int kbs = (num_kb + S - 1) / S;
  *kb_split = kbs;
  *splits = (num_kb + kbs - 1) / kbs;
}
// forward scratch: [header 256 B][tile counters, padded to 256 B][partials S x T x E fp32]
static size_t fwd_count_bytes(int T) { return (size_t)round_up(t_pad_of(T) / RBM * 4, 256); }
static size_t fwd_ws_bytes(int T, int d, int E) {
  int S, kbs;
  fwd_splits(T, d, &S, &kbs);
  return kHdrBytes + fwd_count_bytes(T) + (S > 1 ? (size_t)S * T * E * 4 : 0);
}

}  // namespace router
}  // namespace moe

using namespace moe;
using namespace moe::router;

extern "C" size_t moe_router_workspace_size(int T, int d, int E, int dtype) {
  if (T < 0 || d < 1 || E < 1) return 0;
  if (dtype == MOE_F32) return kHdrBytes + (size_t)round_up((int64_t)T * E * 4, 256);
  const size_t bwd = kHdrBytes + kToffBytes + dl16_bytes(T, E) + (size_t)splits_of(T, d, E) * E * d * 4;
  const size_t fwd = fwd_ws_bytes(T, d, E);
  return bwd > fwd ? bwd : fwd;
}

static int check_router(const void *x, const void *wr, int T, int d, int E, int dtype, const void *ws,
                        size_t ws_bytes) {
  if (T < 0 || d < 1 || E < 1 || E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < moe_router_workspace_size(T, d, E, dtype))
    return MOE_ERR_INVALID_ARG;
  if (!wr || !aligned16(wr)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !aligned16(x))) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * (d > E ? d : E) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_BF16 && d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

template <int KMAX>
static int launch_fwd(const CUtensorMap &mx, const CUtensorMap &mw, const FwdParams &p, cudaStream_t s) {
  MOE_TRY_CUDA(cudaFuncSetAttribute(router_fwd_kernel<KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, R_SMEM));
  int grid = sm_count();
  if (p.num_tiles * p.splits < grid) grid = p.num_tiles * p.splits;
  router_fwd_kernel<KMAX><<<grid, R_THREADS, R_SMEM, s>>>(mx, mw, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" int moe_router_fwd(const void *x, const void *w_router, int T, int d, int E, int k, int dtype,
                              float *logits, int32_t *topk_idx, float *topk_w, void *ws, size_t ws_bytes,
                              moe_stream_t stream) {
  int rc = check_router(x, w_router, T, d, E, dtype, ws, ws_bytes);
  if (rc) return rc;
  if (k < 1 || k > E || k > MOE_MAX_TOPK) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (logits && !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  WsHeader *hdr = static_cast<WsHeader *>(ws);
  // status word and (bf16) the per-tile split counters start at zero
  MOE_TRY_CUDA(cudaMemsetAsync(hdr, 0, dtype == MOE_F32 ? sizeof(WsHeader) : kHdrBytes + fwd_count_bytes(T), s));
  if (T == 0) return MOE_OK;
  if (dtype == MOE_F32) {
    float *L = logits ? logits : reinterpret_cast<float *>(static_cast<char *>(ws) + kHdrBytes);
    if ((rc = simt_gemm((const float *)x, d, 1, (const float *)w_router, d, 1, T, E, d, L, E, false, s))) return rc;
    return moe_route_topk(L, T, E, k, topk_idx, topk_w, stream);
  }
  FwdParams p{};
  p.hdr = hdr;
  p.T = T;
  p.E = E;
  p.k = k;
  p.n_mma = (int)round_up(E, 16);
  const int e32 = (int)round_up(E, 32);
  p.acc_cols = 32;
  while (p.acc_cols < e32) p.acc_cols *= 2;
  p.stage_bytes = R_A_BYTES + p.n_mma * RBK * 2;
  p.stages = R_RING_BYTES / p.stage_bytes;
  if (p.stages > R_MAX_STAGES) p.stages = R_MAX_STAGES;
  p.num_kb = (d + RBK - 1) / RBK;
  p.num_tiles = (int)(t_pad_of(T) / RBM);
  fwd_splits(T, d, &p.splits, &p.kb_split);
  p.tile_count = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + kHdrBytes);
  p.partial = reinterpret_cast<float *>(static_cast<char *>(ws) + kHdrBytes + fwd_count_bytes(T));
  p.logits = logits;
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  CUtensorMap mx, mw;
  if (!make_map(&mx, x, T, d, RBM) || !make_map(&mw, w_router, E, d, p.n_mma)) return MOE_ERR_CUDA;
  if (k <= 2) return launch_fwd<2>(mx, mw, p, s);
  if (k <= 4) return launch_fwd<4>(mx, mw, p, s);
  if (k <= 8) return launch_fwd<8>(mx, mw, p, s);
  return launch_fwd<16>(mx, mw, p, s);
}

extern "C" int moe_router_bwd(const void *x, const void *w_router, const float *d_logits, int T, int d, int E,
                              int dtype, int accumulate_dx, void *dx, void *dw_router, void *ws, size_t ws_bytes,
                              moe_stream_t stream) {
  int rc = check_router(x, w_router, T, d, E, dtype, ws, ws_bytes);
  if (rc) return rc;
  if (!dw_router || !aligned16(dw_router)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!d_logits || !dx || !aligned16(dx))) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char *w = static_cast<char *>(ws);
  WsHeader *hdr = reinterpret_cast<WsHeader *>(w);
  MOE_TRY_CUDA(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s));
  if (dtype == MOE_F32) {
    if (T == 0) {
      MOE_TRY_CUDA(cudaMemsetAsync(dw_router, 0, (size_t)E * d * 4, s));
      return MOE_OK;
    }
    // dx (+)= dL Wr: A(t, e) = dL[t, e], B(c, e) = Wr[e, c]
    if ((rc = simt_gemm(d_logits, E, 1, (const float *)w_router, 1, d, T, d, E, (float *)dx, d, accumulate_dx != 0,
                        s)))
      return rc;
    // dWr = dL^T x: A(e, t) = dL[t, e], B(c, t) = x[t, c]
    return simt_gemm(d_logits, 1, E, (const float *)x, 1, d, E, d, T, (float *)dw_router, d, false, s);
  }
  const int G = splits_of(T, d, E);
  const int64_t t_pad = t_pad_of(T);
  const int ek = ek_of(E);
  int32_t *toff_dx = reinterpret_cast<int32_t *>(w + kHdrBytes);
  int32_t *toff_dw = toff_dx + 4;
  __nv_bfloat16 *dl16 = reinterpret_cast<__nv_bfloat16 *>(w + kHdrBytes + kToffBytes);
  float *part = reinterpret_cast<float *>(w + kHdrBytes + kToffBytes + dl16_bytes(T, E));
  if (T > 0) {
    const int64_t groups = t_pad * (ek / 8);
    int blocks = (int)((groups + 255) / 256);
    if (blocks > 4 * sm_count()) blocks = 4 * sm_count();
    router_prep_kernel<<<blocks, 256, 0, s>>>(d_logits, T, E, t_pad, ek, dl16, toff_dx, toff_dw, G);
    MOE_CHECK_LAUNCH();
    if ((rc = tc_router_dx(dl16, t_pad, ek, w_router, E, d, T, toff_dx, dx, accumulate_dx != 0, hdr, s))) return rc;
    if ((rc = tc_router_dw(dl16, t_pad, ek, x, T, d, E, toff_dw, G, part, hdr, s))) return rc;
  }
  const int64_t n4 = (int64_t)E * d / 4;
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > 4 * sm_count()) blocks = 4 * sm_count();
  router_reduce_kernel<<<blocks, 256, 0, s>>>(part, G, E, d, (__nv_bfloat16 *)dw_router);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
