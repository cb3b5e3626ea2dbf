// C-ABI entry points of the grouped expert FFN, plus status and version helpers.
// Argument validation happens here, before anything is enqueued.
#include "common.cuh"

namespace moe {
int tc_grouped_ffn_fwd(const void *x, const int32_t *token_of_row, int T, const void *wgu, const void *wd,
                       const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f, int64_t rows_max,
                       void *ab, void *h, void *y, WsHeader *hdr, cudaStream_t s);
int tc_grouped_ffn_bwd(const void *dy, const void *x, const int32_t *token_of_row, int T, const void *ab, const void *h,
                       const void *wgu, const void *wd, const int32_t *tile_offsets, const int32_t *offsets, int E, int d,
                       int f, int64_t rows_max, void *dab, void *dx, void *dwgu, void *dwd, WsHeader *hdr,
                       cudaStream_t s);
int simt_grouped_ffn_fwd(const float *x, const int32_t *token_of_row, int T, const float *wgu, const float *wd,
                         const int32_t *toff, int E, int d, int f, int64_t rows_max, float *ab, float *h, float *y,
                         cudaStream_t s);
int simt_grouped_ffn_bwd(const float *dy, const float *x, const int32_t *token_of_row, int T, const float *ab,
                         const float *h, const float *wgu, const float *wd, const int32_t *toff, int E, int d, int f,
                         int64_t rows_max, float *dab, float *dx, float *dwgu, float *dwd, cudaStream_t s);
}  // namespace moe

using namespace moe;

static int check_ffn_shape(int E, int d, int f, int64_t rows_max, int dtype, const void *ws, size_t ws_bytes) {
  if (E < 1 || E > MOE_MAX_EXPERTS || d < 1 || f < 1 || rows_max < 0 || rows_max % MOE_GROUP_ROWS)
    return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < moe_grouped_ffn_workspace_size(E, d, f, rows_max, dtype, 1))
    return MOE_ERR_INVALID_ARG;
  if (rows_max >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_BF16 && (d % 256 != 0 || f % 256 != 0)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The token operand: x_perm [rows_max, d] (token_of_row == nullptr), or x [T, d] in token order with
// token_of_row [rows_max] (gathered by the GEMMs).
static int check_tokens(const void *x, const int32_t *token_of_row, bool gather, int T) {
  if (!x || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  if (gather && (!token_of_row || T < 0)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

extern "C" size_t moe_grouped_ffn_workspace_size(int E, int d, int f, int64_t rows_max, int dtype, int backward) {
  (void)E; (void)d; (void)f; (void)rows_max; (void)dtype; (void)backward;
  return 256;   // the device status word; the GEMM schedulers need no scratch memory
}

static int ffn_fwd(const void *x, const int32_t *tor, int T, bool gather, const void *w_gate_up, const void *w_down,
                   const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f, int64_t rows_max, int dtype,
                   void *ab, void *h, void *y_perm, void *ws, size_t ws_bytes, moe_stream_t stream) {
  int rc = check_ffn_shape(E, d, f, rows_max, dtype, ws, ws_bytes);
  if (rc) return rc;
  if (rows_max == 0) return MOE_OK;
  if ((rc = check_tokens(x, tor, gather, T))) return rc;
  const void *ptrs[] = {w_gate_up, w_down, h, y_perm};
  for (const void *q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (ab && !aligned16(ab)) return MOE_ERR_INVALID_ARG;   // null: a, b are not stored
  if (!tile_offsets || !offsets) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == MOE_F32)
    return simt_grouped_ffn_fwd((const float *)x, tor, T, (const float *)w_gate_up, (const float *)w_down, tile_offsets,
                                E, d, f, rows_max, (float *)ab, (float *)h, (float *)y_perm, s);
  return tc_grouped_ffn_fwd(x, tor, T, w_gate_up, w_down, tile_offsets, offsets, E, d, f, rows_max, ab, h, y_perm,
                            static_cast<WsHeader *>(ws), s);
}

static int ffn_bwd(const void *dy_perm, const void *x, const int32_t *tor, int T, bool gather, const void *ab,
                   const void *h, const void *w_gate_up, const void *w_down, const int32_t *tile_offsets,
                   const int32_t *offsets, int E, int d, int f, int64_t rows_max, int dtype, void *dab, void *dx_perm,
                   void *dw_gate_up, void *dw_down, void *ws, size_t ws_bytes, moe_stream_t stream) {
  int rc = check_ffn_shape(E, d, f, rows_max, dtype, ws, ws_bytes);
  if (rc) return rc;
  const void *ptrs[] = {dy_perm, ab, h, w_gate_up, w_down, dab, dx_perm, dw_gate_up, dw_down};
  if (rows_max > 0) {
    for (const void *q : ptrs)
      if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if ((rc = check_tokens(x, tor, gather, T))) return rc;
  }
  if (!tile_offsets || !offsets) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == MOE_F32)
    return simt_grouped_ffn_bwd((const float *)dy_perm, (const float *)x, tor, T, (const float *)ab, (const float *)h,
                                (const float *)w_gate_up, (const float *)w_down, tile_offsets, E, d, f, rows_max,
                                (float *)dab, (float *)dx_perm, (float *)dw_gate_up, (float *)dw_down, s);
  return tc_grouped_ffn_bwd(dy_perm, x, tor, T, ab, h, w_gate_up, w_down, tile_offsets, offsets, E, d, f, rows_max, dab,
                            dx_perm, dw_gate_up, dw_down, static_cast<WsHeader *>(ws), s);
}

static int ffn_bwd_recompute(const void *dy_perm, const void *x, const int32_t *tor, int T, bool gather, void *ab,
                             void *h, const void *w_gate_up, const void *w_down, const int32_t *tile_offsets,
                             const int32_t *offsets, int E, int d, int f, int64_t rows_max, int dtype, void *dab,
                             void *dx_perm, void *dw_gate_up, void *dw_down, void *ws, size_t ws_bytes,
                             moe_stream_t stream) {
  int rc = check_ffn_shape(E, d, f, rows_max, dtype, ws, ws_bytes);
  if (rc) return rc;
  const void *ptrs[] = {dy_perm, ab, h, w_gate_up, w_down, dab, dx_perm, dw_gate_up, dw_down};
  if (rows_max > 0) {
    for (const void *q : ptrs)
      if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if ((rc = check_tokens(x, tor, gather, T))) return rc;
  }
  if (!tile_offsets || !offsets) return MOE_ERR_INVALID_ARG;
  if (rows_max == 0) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  // 1. a, b and h again from the tokens (the forward's GEMM1 with its SwiGLU epilogue)
  if (dtype == MOE_F32)
    rc = simt_grouped_ffn_fwd((const float *)x, tor, T, (const float *)w_gate_up, (const float *)w_down, tile_offsets,
                              E, d, f, rows_max, (float *)ab, (float *)h, nullptr, s);
  else
    rc = tc_grouped_ffn_fwd(x, tor, T, w_gate_up, w_down, tile_offsets, offsets, E, d, f, rows_max, ab, h, nullptr,
                            static_cast<WsHeader *>(ws), s);
  if (rc) return rc;
  // 2. the backward on the recomputed activations
  return ffn_bwd(dy_perm, x, tor, T, gather, ab, h, w_gate_up, w_down, tile_offsets, offsets, E, d, f, rows_max, dtype,
                 dab, dx_perm, dw_gate_up, dw_down, ws, ws_bytes, stream);
}

extern "C" int moe_grouped_ffn_fwd(const void *x_perm, const void *w_gate_up, const void *w_down,
                                   const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f,
                                   int64_t rows_max, int dtype, void *ab, void *h, void *y_perm, void *ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  return ffn_fwd(x_perm, nullptr, 0, false, w_gate_up, w_down, tile_offsets, offsets, E, d, f, rows_max, dtype, ab, h,
                 y_perm, ws, ws_bytes, stream);
}

extern "C" int moe_grouped_ffn_fwd_gather(const void *x, const int32_t *token_of_row, int T, const void *w_gate_up,
                                          const void *w_down, const int32_t *tile_offsets, const int32_t *offsets,
                                          int E, int d, int f, int64_t rows_max, int dtype, void *ab, void *h,
                                          void *y_perm, void *ws, size_t ws_bytes, moe_stream_t stream) {
  return ffn_fwd(x, token_of_row, T, true, w_gate_up, w_down, tile_offsets, offsets, E, d, f, rows_max, dtype, ab, h,
                 y_perm, ws, ws_bytes, stream);
}

extern "C" int moe_grouped_ffn_bwd(const void *dy_perm, const void *x_perm, const void *ab, const void *h,
                                   const void *w_gate_up, const void *w_down, const int32_t *tile_offsets,
                                   const int32_t *offsets, int E, int d, int f, int64_t rows_max, int dtype, void *dab,
                                   void *dx_perm, void *dw_gate_up, void *dw_down, void *ws, size_t ws_bytes,
                                   moe_stream_t stream) {
  return ffn_bwd(dy_perm, x_perm, nullptr, 0, false, ab, h, w_gate_up, w_down, tile_offsets, offsets, E, d, f, rows_max,
                 dtype, dab, dx_perm, dw_gate_up, dw_down, ws, ws_bytes, stream);
}

extern "C" int moe_grouped_ffn_bwd_gather(const void *dy_perm, const void *x, const int32_t *token_of_row, int T,
                                          const void *ab, const void *h, const void *w_gate_up, const void *w_down,
                                          const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f,
                                          int64_t rows_max, int dtype, void *dab, void *dx_perm, void *dw_gate_up,
                                          void *dw_down, void *ws, size_t ws_bytes, moe_stream_t stream) {
  return ffn_bwd(dy_perm, x, token_of_row, T, true, ab, h, w_gate_up, w_down, tile_offsets, offsets, E, d, f, rows_max,
                 dtype, dab, dx_perm, dw_gate_up, dw_down, ws, ws_bytes, stream);
}

extern "C" int moe_grouped_ffn_bwd_recompute(const void *dy_perm, const void *x_perm, void *ab, void *h,
                                             const void *w_gate_up, const void *w_down, const int32_t *tile_offsets,
                                             const int32_t *offsets, int E, int d, int f, int64_t rows_max, int dtype,
                                             void *dab, void *dx_perm, void *dw_gate_up, void *dw_down, void *ws,
                                             size_t ws_bytes, moe_stream_t stream) {
  return ffn_bwd_recompute(dy_perm, x_perm, nullptr, 0, false, ab, h, w_gate_up, w_down, tile_offsets, offsets, E, d,
                           f, rows_max, dtype, dab, dx_perm, dw_gate_up, dw_down, ws, ws_bytes, stream);
}

extern "C" int moe_grouped_ffn_bwd_recompute_gather(const void *dy_perm, const void *x, const int32_t *token_of_row,
                                                    int T, void *ab, void *h, const void *w_gate_up,
                                                    const void *w_down, const int32_t *tile_offsets,
                                                    const int32_t *offsets, int E, int d, int f, int64_t rows_max,
                                                    int dtype, void *dab, void *dx_perm, void *dw_gate_up,
                                                    void *dw_down, void *ws, size_t ws_bytes, moe_stream_t stream) {
  return ffn_bwd_recompute(dy_perm, x, token_of_row, T, true, ab, h, w_gate_up, w_down, tile_offsets, offsets, E, d, f,
                           rows_max, dtype, dab, dx_perm, dw_gate_up, dw_down, ws, ws_bytes, stream);
}

extern "C" int moe_read_status(const void *ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  int32_t st = 0;
  MOE_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  MOE_TRY_CUDA(cudaMemcpy(&st, ws, sizeof(st), cudaMemcpyDeviceToHost));
  return st;
}

extern "C" const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_BAD_INDEX: return "expert index out of range";
    case MOE_ERR_CHECK_FAILED: return "consistency check failed (debug build)";
    default: return "unknown status";
  }
}

extern "C" int moe_version(void) { return MOE_VERSION; }
