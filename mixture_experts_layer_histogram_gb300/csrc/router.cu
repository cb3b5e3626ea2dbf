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
//   warps 2..5  epilogue, one thread per token: tcgen05.ld of the token's E logits, 32 at a time,
//               optional store of the fp32 logits, insertion into a sorted top-k list held in
//               registers (value desc, id asc), softmax of the selected logits
// The logits never make a round trip through HBM (x is read once, Wr stays in L2).
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
constexpr int R_THREADS = 192;           // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int R_EPI_THREADS = 128;
constexpr int R_A_BYTES = RBM * RBK * 2; // 16 KB
constexpr int R_RING_BYTES = 192 * 1024;
constexpr int R_MAX_STAGES = 8;
constexpr int R_SMEM = R_RING_BYTES + 1024 + 8 * (2 * R_MAX_STAGES + 5) + 16;
constexpr int kSplitTarget = 296;        // RDW: aim for about this many output tiles (2 per SM)
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
  float *logits;   // may be null
  int32_t *topk_idx;
  float *topk_w;
};

// Insert (v, e) into the list tv/ti (k entries, sorted by value desc then id asc). Ids arrive in
// increasing order, so an equal value goes after the entries already present; every entry after
// the insertion point shifts down one place and the last one drops out.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&tv)[KMAX], int (&ti)[KMAX], int k, float v, int e) {
  float cv = v;
  int ci = e;
  bool shifting = false;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const bool take = j < k && (shifting || cv > tv[j]);
    const float ov = tv[j];
    const int oi = ti[j];
    tv[j] = take ? cv : ov;
    ti[j] = take ? ci : oi;
    cv = take ? ov : cv;
    ci = take ? oi : ci;
    shifting = shifting || take;
  }
}

template <int KMAX>
__global__ void __launch_bounds__(R_THREADS, 1)
    router_fwd_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + R_RING_BYTES);
  // bars: full[S], empty[S], tfull[2], tempty[2], mma_done
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * R_MAX_STAGES + 5);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (R_MAX_STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * R_MAX_STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * R_MAX_STAGES + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * R_MAX_STAGES + 4);
  const uint32_t tmem_cols = 2u * (uint32_t)p.acc_cols;

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

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.hdr, 11)) { ok = false; break; }
        const uint32_t sA = sbase + stage * p.stage_bytes, fb = full_bar(stage);
        mbar_expect_tx(fb, p.stage_bytes);
        issued |= 1u << stage;
        tma_load_2d(sA, &tmX, kb * RBK, tile * RBM, fb);
        tma_load_2d(sA + R_A_BYTES, &tmW, kb * RBK, 0, fb);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
    for (int s = 0; s < S; ++s) {   // every issued copy lands before the CTA may exit
      if (!((issued >> s) & 1u)) continue;
      const uint32_t ph = (s < stage) ? phase : (phase ^ 1u);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(full_bar(s), ph) && global_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    // kind::f16, D fp32, A and B bf16 K-major, M = 128, N = n_mma
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(p.n_mma >> 3) << 17) |
                           ((uint32_t)(RBM >> 4) << 24);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool issued_any = false, ok = true;
    for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.hdr, 12)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.acc_cols);
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.hdr, 13)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sA = sbase + stage * p.stage_bytes, sB = sA + R_A_BYTES;
#pragma unroll
        for (int kk = 0; kk < RBK / 16; ++kk)
          mma_bf16(d_tmem, sdesc(sA + kk * 32, 16, 1024), sdesc(sB + kk * 32, 16, 1024), idesc,
                   (kb | kk) != 0 ? 1u : 0u);
        issued_any = true;
        mma_commit(empty_bar(stage));
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      mma_commit(tfull_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (issued_any) {
      mma_commit(mma_done_bar);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(mma_done_bar, 0) && global_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue: one token per thread
    const int quarter = warp & 3;   // TMEM lanes 32 * quarter ... 32 * quarter + 31
    const int row = quarter * 32 + lane;
    const int E = p.E, k = p.k;
    const bool vec = (E & 3) == 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.hdr, 14)) break;
      tc_fence_after();
      const int t = tile * RBM + row;
      const bool live = t < p.T;
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * p.acc_cols);
      float tv[KMAX];
      int ti[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        tv[j] = -INFINITY;
        ti[j] = 0;
      }
      float *lrow = p.logits ? p.logits + (int64_t)t * E : nullptr;
#pragma unroll 1
      for (int c0 = 0; c0 < E; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tbase + c0, r);
        tmem_ld_wait();
        if (live && lrow) {
          if (vec) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (c0 + 4 * q < E)
                *reinterpret_cast<float4 *>(lrow + c0 + 4 * q) =
                    make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c0 + i < E) lrow[c0 + i] = __uint_as_float(r[i]);
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < E) topk_insert<KMAX>(tv, ti, k, __uint_as_float(r[i]), c0 + i);
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      if (live) {
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
    for (int g = 0; g < G; ++g) {
      const float4 q = __ldg(reinterpret_cast<const float4 *>(part + g * plane) + i);
      s.x += q.x;
      s.y += q.y;
      s.z += q.z;
      s.w += q.w;
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

}  // namespace router
}  // namespace moe

using namespace moe;
using namespace moe::router;

extern "C" size_t moe_router_workspace_size(int T, int d, int E, int dtype) {
  if (T < 0 || d < 1 || E < 1) return 0;
  if (dtype == MOE_F32) return kHdrBytes + (size_t)round_up((int64_t)T * E * 4, 256);
  return kHdrBytes + kToffBytes + dl16_bytes(T, E) + (size_t)splits_of(T, d, E) * E * d * 4;
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
  if (p.num_tiles < grid) grid = p.num_tiles;
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
  MOE_TRY_CUDA(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s));
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
