// Grouped expert FFN in true fp32 (FFMA on the CUDA cores) for fp32 layers.
//
// Same five GEMM kinds and the same padded grouped layout as the tensor-core path; tf32 tensor
// cores would not hold fp32 accuracy, so fp32 layers take this path. Tile 32 x 32 x 32 through
// shared memory, 256 threads, 4 outputs per thread. Operands are addressed through (row, k)
// strides, which covers K-major and MN-major reads alike.
#include "common.cuh"

namespace moe {
namespace simt {

enum Kind { GATEUP = 0, DOWN = 1, DH = 2, DGRAD = 3, WGRAD = 4 };
constexpr int TS = 32;

struct Args {
  const float *A;
  int64_t sAm, sAk;
  const float *B;
  int64_t sBn, sBk, sBe;   // sBe: per-expert offset (row-grouped kinds)
  int64_t up_off;          // GATEUP: offset of the up projection rows
  int N, K, E, BM;
  int64_t rows_max;
  const int32_t *toff;
  float *C;
  int64_t ldc, sCe;
  float *C2;               // GATEUP: h
  int64_t ldc2;
  const float *aux;        // DH: ab
  int64_t ld_aux;
  int f;
  int Mw;                  // WGRAD: rows of dW[e]
  const int32_t *gA;       // GATEUP gathering: A row m is token gA[m] of A (-1: zero row)
  const int32_t *gB;       // WGRAD gathering: B's k row r (a grouped row) is token gB[r] of B (-1: zero)
  int ntok;                // tokens of the gathered operand (indices past it read as zero rows)
};

template <int KIND>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const Args p) {
  __shared__ float As[TS][TS + 1], Bs[TS][TS + 1], Bs2[TS][TS + 1];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int n0 = blockIdx.x * TS;
  int m0 = blockIdx.y * TS, e, K, M;
  const float *A = p.A, *B = p.B;
  if (KIND == WGRAD) {
    e = blockIdx.z;
    const int64_t r0 = (int64_t)p.toff[e] * p.BM;
    K = (p.toff[e + 1] - p.toff[e]) * p.BM;
    A += r0 * p.sAk;
    B += r0 * p.sBk;
    M = p.Mw;
  } else {
    M = p.toff[p.E] * p.BM;
    if (m0 >= M) return;
    const int rt = m0 / p.BM;
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (p.toff[mid] <= rt) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    K = p.K;
    B += (int64_t)e * p.sBe;
  }
  float acc[4] = {0, 0, 0, 0}, acc2[4] = {0, 0, 0, 0};
  for (int k0 = 0; k0 < K; k0 += TS) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = ty + 8 * i, kk = k0 + tx;
      if (KIND == GATEUP && p.gA) {
        const int tk = (m0 + r < M && kk < K) ? p.gA[m0 + r] : -1;
        As[r][tx] = (tk >= 0 && tk < p.ntok) ? A[(int64_t)tk * p.sAm + (int64_t)kk * p.sAk] : 0.0f;
      } else {
        As[r][tx] = (m0 + r < M && kk < K) ? A[(int64_t)(m0 + r) * p.sAm + (int64_t)kk * p.sAk] : 0.0f;
      }
      const bool nb = n0 + r < p.N && kk < K;
      if (KIND == WGRAD && p.gB) {
        const int tk = nb ? p.gB[(int64_t)p.toff[e] * p.BM + kk] : -1;
        Bs[r][tx] = (tk >= 0 && tk < p.ntok) ? p.B[(int64_t)(n0 + r) * p.sBn + (int64_t)tk * p.sBk] : 0.0f;
      } else {
        Bs[r][tx] = nb ? B[(int64_t)(n0 + r) * p.sBn + (int64_t)kk * p.sBk] : 0.0f;
      }
      if (KIND == GATEUP) Bs2[r][tx] = nb ? B[p.up_off + (int64_t)(n0 + r) * p.sBn + (int64_t)kk * p.sBk] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < TS; ++kk) {
      const float b = Bs[tx][kk];
      const float b2 = (KIND == GATEUP) ? Bs2[tx][kk] : 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i] = fmaf(As[ty + 8 * i][kk], b, acc[i]);
        if (KIND == GATEUP) acc2[i] = fmaf(As[ty + 8 * i][kk], b2, acc2[i]);
      }
    }
    __syncthreads();
  }
  const int n = n0 + tx;
  if (n >= p.N) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty + 8 * i;
    if (m >= M) continue;
    if (KIND == GATEUP) {
      const float a = acc[i], b = acc2[i];
      if (p.C) {   // null: a, b are not stored
        p.C[m * p.ldc + n] = a;
        p.C[m * p.ldc + p.f + n] = b;
      }
      p.C2[m * p.ldc2 + n] = a / (1.0f + expf(-a)) * b;
    } else if (KIND == DH) {
      const float dh = acc[i], a = p.aux[m * p.ld_aux + n], b = p.aux[m * p.ld_aux + p.f + n];
      const float s = 1.0f / (1.0f + expf(-a));
      p.C[m * p.ldc + n] = dh * b * s * (1.0f + a * (1.0f - s));
      p.C[m * p.ldc + p.f + n] = dh * a * s;
    } else if (KIND == WGRAD) {
      p.C[(int64_t)e * p.sCe + m * p.ldc + n] = acc[i];
    } else {
      p.C[m * p.ldc + n] = acc[i];
    }
  }
}

template <int KIND>
static int launch(const Args &a, int64_t m_rows, int n, int gz, cudaStream_t s) {
  dim3 grid((n + TS - 1) / TS, (unsigned)((m_rows + TS - 1) / TS), gz);
  simt_gemm_kernel<KIND><<<grid, 256, 0, s>>>(a);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // namespace simt

// x is x_perm [rows_max, d], or with token_of_row the tokens [T, d] in token order (gathered).
int simt_grouped_ffn_fwd(const float *x, const int32_t *token_of_row, int T, const float *wgu, const float *wd,
                         const int32_t *toff, int E, int d, int f, int64_t rows_max, float *ab, float *h, float *y,
                         cudaStream_t s) {
  using namespace simt;
  Args a{};
  a.gA = token_of_row;
  a.ntok = T;
  a.toff = toff;
  a.E = E;
  a.BM = MOE_GROUP_ROWS;
  a.rows_max = rows_max;
  a.f = f;
  // [a | b] = x Wgu^T, h = silu(a) * b
  a.A = x; a.sAm = d; a.sAk = 1;
  a.B = wgu; a.sBn = d; a.sBk = 1; a.sBe = (int64_t)2 * f * d; a.up_off = (int64_t)f * d;
  a.N = f; a.K = d;
  a.C = ab; a.ldc = 2 * (int64_t)f; a.C2 = h; a.ldc2 = f;
  int rc = launch<GATEUP>(a, rows_max, f, 1, s);
  if (rc || y == nullptr) return rc;   // y == nullptr: GEMM1 only (recompute of ab, h)
  // y = h Wd^T
  a.A = h; a.sAm = f; a.sAk = 1;
  a.B = wd; a.sBn = f; a.sBk = 1; a.sBe = (int64_t)d * f; a.up_off = 0;
  a.N = d; a.K = f;
  a.C = y; a.ldc = d; a.C2 = nullptr;
  a.gA = nullptr;
  return launch<DOWN>(a, rows_max, d, 1, s);
}

int simt_grouped_ffn_bwd(const float *dy, const float *x, const int32_t *token_of_row, int T, const float *ab,
                         const float *h, const float *wgu, const float *wd, const int32_t *toff, int E, int d, int f,
                         int64_t rows_max, float *dab, float *dx, float *dwgu, float *dwd, cudaStream_t s) {
  using namespace simt;
  Args a{};
  a.ntok = T;
  a.toff = toff;
  a.E = E;
  a.BM = MOE_GROUP_ROWS;
  a.rows_max = rows_max;
  a.f = f;
  int rc;
  // dh = dy Wd[e]: B(n=j, k=c) = Wd[e][c][j]
  a.A = dy; a.sAm = d; a.sAk = 1;
  a.B = wd; a.sBn = 1; a.sBk = f; a.sBe = (int64_t)d * f;
  a.N = f; a.K = d;
  a.C = dab; a.ldc = 2 * (int64_t)f; a.aux = ab; a.ld_aux = 2 * (int64_t)f;
  if ((rc = launch<DH>(a, rows_max, f, 1, s))) return rc;
  // dx = dab Wgu[e]: B(n=c, k=i) = Wgu[e][i][c]
  a.A = dab; a.sAm = 2 * (int64_t)f; a.sAk = 1;
  a.B = wgu; a.sBn = 1; a.sBk = d; a.sBe = (int64_t)2 * f * d;
  a.N = d; a.K = 2 * f;
  a.C = dx; a.ldc = d; a.aux = nullptr;
  if ((rc = launch<DGRAD>(a, rows_max, d, 1, s))) return rc;
  // dWd[e][c][j] = sum_r dy[r][c] h[r][j]
  a.A = dy; a.sAm = 1; a.sAk = d;
  a.B = h; a.sBn = 1; a.sBk = f; a.sBe = 0;
  a.N = f; a.Mw = d;
  a.C = dwd; a.ldc = f; a.sCe = (int64_t)d * f;
  if ((rc = launch<WGRAD>(a, d, f, E, s))) return rc;
  // dWgu[e][i][c] = sum_r dab[r][i] x[r][c] (x's rows gathered from the tokens when token_of_row is given)
  a.A = dab; a.sAm = 1; a.sAk = 2 * (int64_t)f;
  a.B = x; a.sBn = 1; a.sBk = d;
  a.gB = token_of_row;
  a.N = d; a.Mw = 2 * f;
  a.C = dwgu; a.ldc = d; a.sCe = (int64_t)2 * f * d;
  return launch<WGRAD>(a, 2 * f, d, E, s);
}

}  // namespace moe
