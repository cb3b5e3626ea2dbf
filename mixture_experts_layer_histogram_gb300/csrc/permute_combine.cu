// Token permutation into the grouped layout, the weighted combine back to token order, and the
// combine/routing backward. All three are HBM-bound row copies: a warp per token (per 2 KB segment
// of a token's row in the combine), 16-byte vectors per lane, fp32 accumulation, the k row indices
// of a token held in lanes 0..k-1; every lane issues the loads of all k rows of a chunk before it
// uses any of them.
//
// "Scalable Pretraining of Large MoE LMs on Aurora", brief, section 核心方法: the generated indices
// feed the grouped GEMM (permute) and the experts' outputs return to token order (combine); the
// backward of both is part of the module's forward-backward pass (sections 为什么值得记录 / 关键结果).
#include "common.cuh"

namespace moe {

constexpr int kRowThreads = 256;   // 8 warps, one work unit (token or row segment) per warp per iteration
constexpr int kUnroll = 8;         // 16-byte vectors in flight per lane (a 4 KB row in one round trip)
constexpr int kSegVecs = 128;      // combine: 16-byte vectors of a row per work unit (2 KB)

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void unpack(const uint4 &q, float *v) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y); v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
  static __device__ __forceinline__ uint4 pack(const float *v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
  }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void unpack(const uint4 &q, float *v) { unpack_bf16x8(q, v); }
  static __device__ __forceinline__ uint4 pack(const float *v) { return pack_bf16x8(v); }
};

// Zero the padding rows of expert e: [tile_offsets[e]*BM + counts[e], tile_offsets[e+1]*BM).
__device__ __forceinline__ void zero_padding_rows(uint4 *dst, int64_t row_vecs, int e, const int32_t *counts,
                                                  const int32_t *tile_offsets, int BM, int64_t rows_max) {
  int64_t start = (int64_t)tile_offsets[e] * BM + counts[e];
  int64_t end = (int64_t)tile_offsets[e + 1] * BM;
  if (end > rows_max) end = rows_max;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t i = start * row_vecs + threadIdx.x; i < end * row_vecs; i += blockDim.x) dst[i] = z;
}

__device__ __forceinline__ int load_row(const int32_t *row_of_slot, int64_t t, int k, int lane, int64_t rows_max) {
  int r = -1;
  if (lane < k) {
    r = __ldg(row_of_slot + t * k + lane);
    if (r < 0 || r >= rows_max) r = -1;
  }
  return r;
}

// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kRowThreads) permute_kernel(const uint4 *__restrict__ x, int64_t T, int64_t row_vecs,
                                                              int k, const int32_t *__restrict__ row_of_slot,
                                                              const int32_t *__restrict__ counts,
                                                              const int32_t *__restrict__ tile_offsets, int BM,
                                                              int64_t rows_max, int token_blocks,
                                                              uint4 *__restrict__ xp) {
  if ((int)blockIdx.x >= token_blocks) {
    zero_padding_rows(xp, row_vecs, blockIdx.x - token_blocks, counts, tile_offsets, BM, rows_max);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)token_blocks * (kRowThreads / 32);
  for (int64_t t = (int64_t)blockIdx.x * (kRowThreads / 32) + (threadIdx.x >> 5); t < T; t += nw) {
    const int myrow = load_row(row_of_slot, t, k, lane, rows_max);
    const uint4 *src = x + t * row_vecs;
    for (int64_t v0 = 0; v0 < row_vecs; v0 += 32 * kUnroll) {
      uint4 buf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        int64_t v = v0 + u * 32 + lane;
        if (v < row_vecs) buf[u] = ld_stream(src + v);
      }
      for (int j = 0; j < k; ++j) {
        int r = __shfl_sync(0xffffffffu, myrow, j);
        if (r < 0) continue;
        uint4 *dst = xp + (int64_t)r * row_vecs;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          int64_t v = v0 + u * 32 + lane;
          if (v < row_vecs) dst[v] = buf[u];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------------------
// KMAX: compile-time upper bound on k. Per 512-byte chunk of the output row every lane first issues
// the loads of all k expert rows, then accumulates them in slot order (fp32), so a warp waits for
// one memory latency per chunk rather than one per slot.
template <typename T, bool WEIGHTED, int KMAX>
__global__ void __launch_bounds__(kRowThreads) combine_kernel(const uint4 *__restrict__ y, const float *__restrict__ w,
                                                              const int32_t *__restrict__ row_of_slot, int64_t Tn,
                                                              int64_t row_vecs, int k, int64_t rows_max,
                                                              uint4 *__restrict__ out) {
  constexpr int N = Elem<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * (kRowThreads / 32);
  // work unit: one kSegVecs-vector segment of one token's row (finer units balance the last wave)
  const int64_t nseg = (row_vecs + kSegVecs - 1) / kSegVecs;
  for (int64_t u = (int64_t)blockIdx.x * (kRowThreads / 32) + (threadIdx.x >> 5); u < Tn * nseg; u += nw) {
    const int64_t t = u / nseg;
    const int64_t vbeg = (u - t * nseg) * kSegVecs;
    const int64_t vend = vbeg + kSegVecs < row_vecs ? vbeg + kSegVecs : row_vecs;
    const int myrow = load_row(row_of_slot, t, k, lane, rows_max);
    const float myw = (WEIGHTED && lane < k) ? __ldg(w + t * k + lane) : 1.0f;
    int rows[KMAX];
    float ws[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      rows[j] = j < k ? __shfl_sync(0xffffffffu, myrow, j) : -1;
      ws[j] = j < k ? __shfl_sync(0xffffffffu, myw, j) : 0.0f;
    }
    // warp-uniform loop: loads and stores are predicated per lane
    for (int64_t v0 = vbeg; v0 < vend; v0 += 32) {
      const int64_t v = v0 + lane;
      const bool act = v < vend;
      uint4 q[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (rows[j] >= 0 && act) q[j] = ld_stream(y + (int64_t)rows[j] * row_vecs + v);
      float acc[N];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (rows[j] < 0 || !act) continue;
        float val[N];
        Elem<T>::unpack(q[j], val);
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = WEIGHTED ? fmaf(ws[j], val[i], acc[i]) : acc[i] + val[i];
      }
      if (act) out[t * row_vecs + v] = Elem<T>::pack(acc);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// KMAX: compile-time upper bound on k (the per-slot arrays live in registers)
template <typename T, int KMAX>
__global__ void __launch_bounds__(kRowThreads) combine_bwd_kernel(
    const uint4 *__restrict__ g, const uint4 *__restrict__ y, const float *__restrict__ w,
    const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ row_of_slot, const int32_t *__restrict__ counts,
    const int32_t *__restrict__ tile_offsets, int BM, int64_t Tn, int64_t row_vecs, int k, int E, int64_t rows_max,
    int token_blocks, uint4 *__restrict__ dy, float *__restrict__ d_topk_w, float *__restrict__ d_logits) {
  if ((int)blockIdx.x >= token_blocks) {
    zero_padding_rows(dy, row_vecs, blockIdx.x - token_blocks, counts, tile_offsets, BM, rows_max);
    return;
  }
  constexpr int N = Elem<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)token_blocks * (kRowThreads / 32);
  for (int64_t t = (int64_t)blockIdx.x * (kRowThreads / 32) + (threadIdx.x >> 5); t < Tn; t += nw) {
    const int myrow = load_row(row_of_slot, t, k, lane, rows_max);
    const float myw = lane < k ? __ldg(w + t * k + lane) : 0.0f;
    const int mye = lane < k ? __ldg(topk_idx + t * k + lane) : -1;
    float part[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) part[j] = 0.0f;
    int rows[KMAX];
    float ws[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      rows[j] = j < k ? __shfl_sync(0xffffffffu, myrow, j) : -1;
      ws[j] = j < k ? __shfl_sync(0xffffffffu, myw, j) : 0.0f;
    }
    // warp-uniform loop over 512-byte chunks of the row; per chunk all k expert rows are loaded
    // before any dy row is stored, so the k loads are in flight together
    for (int64_t v0 = 0; v0 < row_vecs; v0 += 32) {
      const int64_t v = v0 + lane;
      const bool act = v < row_vecs;
      uint4 gq = make_uint4(0, 0, 0, 0), yq[KMAX];
      if (act) gq = ld_stream(g + t * row_vecs + v);
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k && act && rows[j] >= 0) yq[j] = ld_stream(y + (int64_t)rows[j] * row_vecs + v);
      float gv[N];
      Elem<T>::unpack(gq, gv);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j >= k) break;
        if (!act || rows[j] < 0) continue;
        float yv[N], o[N];
        Elem<T>::unpack(yq[j], yv);
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < N; ++i) {
          s = fmaf(gv[i], yv[i], s);
          o[i] = ws[j] * gv[i];
        }
        part[j] += s;
        dy[(int64_t)rows[j] * row_vecs + v] = Elem<T>::pack(o);
      }
    }
    // d_topk_w[t, j] = <g, y_j>: reduce each partial over the warp; lane j keeps slot j
    float dw = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j >= k) break;
      float s = part[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane == j) dw = s;
    }
    float sw = lane < k ? myw * dw : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, off);
    const float dl = myw * (dw - sw);
    if (lane < k) d_topk_w[t * k + lane] = dw;
    for (int e0 = 0; e0 < E; e0 += 32) {
      int e = e0 + lane;
      float val = 0.0f;
      for (int j = 0; j < k; ++j) {
        int ej = __shfl_sync(0xffffffffu, mye, j);
        float dj = __shfl_sync(0xffffffffu, dl, j);
        if (ej == e) val = dj;
      }
      if (e < E) d_logits[t * E + e] = val;
    }
  }
}

static int row_blocks(int64_t T) {
  int64_t b = (T + (kRowThreads / 32) - 1) / (kRowThreads / 32);
  int64_t cap = (int64_t)sm_count() * 8;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace moe

using namespace moe;

static bool valid_dtype(int dtype) { return dtype == MOE_F32 || dtype == MOE_BF16; }

extern "C" int moe_permute(const void *x, int dtype, int T, int d, int k, int E, const int32_t *row_of_slot,
                           const int32_t *counts, const int32_t *tile_offsets, int64_t rows_max, void *x_perm,
                           moe_stream_t stream) {
  if (!valid_dtype(dtype) || T < 0 || d < 1 || k < 1 || k > MOE_MAX_TOPK || E < 1 || E > MOE_MAX_EXPERTS)
    return MOE_ERR_INVALID_ARG;
  const size_t row_bytes = (size_t)d * dtype_size(dtype);
  if (row_bytes % 16) return MOE_ERR_UNSUPPORTED;
  if (rows_max < moe_grouped_rows_max(T, k, E)) return MOE_ERR_INVALID_ARG;
  if (!x_perm || !counts || !tile_offsets || (T > 0 && (!x || !row_of_slot))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  const int tb = row_blocks(T);
  permute_kernel<<<tb + E, kRowThreads, 0, (cudaStream_t)stream>>>(
      (const uint4 *)x, T, (int64_t)(row_bytes / 16), k, row_of_slot, counts, tile_offsets, MOE_GROUP_ROWS, rows_max,
      tb, (uint4 *)x_perm);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" int moe_combine_fwd(const void *y_perm, const float *topk_w, const int32_t *row_of_slot, int T, int d,
                               int k, int64_t rows_max, int dtype, void *out, moe_stream_t stream) {
  if (!valid_dtype(dtype) || T < 0 || d < 1 || k < 1 || k > MOE_MAX_TOPK || rows_max < 0) return MOE_ERR_INVALID_ARG;
  const size_t row_bytes = (size_t)d * dtype_size(dtype);
  if (row_bytes % 16) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_perm || !row_of_slot || !out || !aligned16(y_perm) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const int64_t rv = (int64_t)(row_bytes / 16);
  const int nb = row_blocks((int64_t)T * ((rv + kSegVecs - 1) / kSegVecs));   // one warp per row segment
  cudaStream_t s = (cudaStream_t)stream;
  const uint4 *y = (const uint4 *)y_perm;
  uint4 *o = (uint4 *)out;
#define MOE_COMBINE(TYPE, W, KM) combine_kernel<TYPE, W, KM><<<nb, kRowThreads, 0, s>>>(y, topk_w, row_of_slot, T, rv, k, rows_max, o)
#define MOE_COMBINE_K(TYPE, W)                     \
  do {                                             \
    if (k <= 2) MOE_COMBINE(TYPE, W, 2);           \
    else if (k <= 4) MOE_COMBINE(TYPE, W, 4);      \
    else if (k <= 8) MOE_COMBINE(TYPE, W, 8);      \
    else MOE_COMBINE(TYPE, W, 16);                 \
  } while (0)
  if (dtype == MOE_BF16) {
    if (topk_w) MOE_COMBINE_K(__nv_bfloat16, true);
    else MOE_COMBINE_K(__nv_bfloat16, false);
  } else {
    if (topk_w) MOE_COMBINE_K(float, true);
    else MOE_COMBINE_K(float, false);
  }
#undef MOE_COMBINE_K
#undef MOE_COMBINE
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

extern "C" int moe_combine_bwd(const void *grad_out, const void *y_perm, const float *topk_w, const int32_t *topk_idx,
                               const int32_t *row_of_slot, const int32_t *counts, const int32_t *tile_offsets, int T,
                               int d, int k, int E, int64_t rows_max, int dtype, void *dy_perm, float *d_topk_w,
                               float *d_logits, moe_stream_t stream) {
  if (!valid_dtype(dtype) || T < 0 || d < 1 || k < 1 || k > MOE_MAX_TOPK || E < 1 || E > MOE_MAX_EXPERTS || k > E)
    return MOE_ERR_INVALID_ARG;
  const size_t row_bytes = (size_t)d * dtype_size(dtype);
  if (row_bytes % 16) return MOE_ERR_UNSUPPORTED;
  if (rows_max < moe_grouped_rows_max(T, k, E)) return MOE_ERR_INVALID_ARG;
  if (!dy_perm || !counts || !tile_offsets || !aligned16(dy_perm)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!grad_out || !y_perm || !topk_w || !topk_idx || !row_of_slot || !d_topk_w || !d_logits ||
                !aligned16(grad_out) || !aligned16(y_perm)))
    return MOE_ERR_INVALID_ARG;
  const int64_t rv = (int64_t)(row_bytes / 16);
  const int tb = row_blocks(T);
  cudaStream_t s = (cudaStream_t)stream;
#define MOE_COMBINE_BWD(TYPE, KM)                                                                               \
  combine_bwd_kernel<TYPE, KM><<<tb + E, kRowThreads, 0, s>>>(                                                  \
      (const uint4 *)grad_out, (const uint4 *)y_perm, topk_w, topk_idx, row_of_slot, counts, tile_offsets,     \
      MOE_GROUP_ROWS, T, rv, k, E, rows_max, tb, (uint4 *)dy_perm, d_topk_w, d_logits)
  if (dtype == MOE_BF16) {
    if (k <= 2) MOE_COMBINE_BWD(__nv_bfloat16, 2);
    else if (k <= 4) MOE_COMBINE_BWD(__nv_bfloat16, 4);
    else if (k <= 8) MOE_COMBINE_BWD(__nv_bfloat16, 8);
    else MOE_COMBINE_BWD(__nv_bfloat16, 16);
  } else {
    if (k <= 2) MOE_COMBINE_BWD(float, 2);
    else if (k <= 4) MOE_COMBINE_BWD(float, 4);
    else if (k <= 8) MOE_COMBINE_BWD(float, 8);
    else MOE_COMBINE_BWD(float, 16);
  }
#undef MOE_COMBINE_BWD
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
