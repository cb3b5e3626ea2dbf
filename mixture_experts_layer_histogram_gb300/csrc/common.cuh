// Shared device/host helpers of libmoe (sm_103a). Nothing here is visible through the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

#define MOE_TRY_CUDA(expr)                 \
  do {                                     \
    cudaError_t err__ = (expr);            \
    if (err__ != cudaSuccess) {            \
      (void)cudaGetLastError();            \
      return MOE_ERR_CUDA;                 \
    }                                      \
  } while (0)

#define MOE_CHECK_LAUNCH() MOE_TRY_CUDA(cudaGetLastError())

// The debug build (-DMOE_CHECKS=1) compiles device-side consistency checks into the GEMM kernels;
// a failed check records MOE_ERR_CHECK_FAILED and skips the work instead of trapping.
#ifndef MOE_CHECKS
#define MOE_CHECKS 0
#endif

namespace moe {

// Every workspace starts with this header (the device status word first).
struct WsHeader {
  int32_t status;        // first device-detected error (0 = none)
  int32_t detail;        // extra information about it (e.g. the block that timed out)
  int32_t armed;         // moe_count_index: look-back fault hook as consumed for this call (0 = off)
  int32_t pad0;
  uint32_t tickets[4];   // self-managed counters (reset by the call that uses them)
  uint32_t pad1[8];
};
static_assert(sizeof(WsHeader) == 64, "workspace header is 64 bytes");

constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;   // bounded device waits: 0.2 s

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Record the first error only.
__device__ __forceinline__ void report(WsHeader *ws, int code, int detail) {
  if (ws == nullptr) return;
  if (atomicCAS(&ws->status, 0, code) == 0) ws->detail = detail;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // round to nearest even
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 &q, float *v) {
  v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
  v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
  v[4] = __uint_as_float(q.z << 16); v[5] = __uint_as_float(q.z & 0xffff0000u);
  v[6] = __uint_as_float(q.w << 16); v[7] = __uint_as_float(q.w & 0xffff0000u);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float *v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {   // read-once data: skip L1
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Logistic sigmoid for the bf16 tensor-core epilogues: __expf, then the approximate reciprocal
// (one MUFU op, at most 1 ulp of fp32 error) instead of an IEEE-rounded divide, whose multi-
// instruction sequence made the SwiGLU-backward epilogue noticeably slower. The inputs here are
// bf16 and so are the results: one fp32 ulp (2^-23 relative) is far below bf16 rounding (2^-9).
// 1 + exp(-z) >= 1, so flushing subnormal inputs changes nothing; z -> -inf gives exp = inf and a
// result of 0.
__device__ __forceinline__ float sigmoidf_(float z) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + __expf(-z)));
  return r;
}

// Insert (v, e) into the list tv/ti (sorted by value desc, then id asc). Ids arrive in increasing
// order, so v goes after every entry >= v, the entries after it shift down one place and the last
// one drops out. Every slot's new content is computed from the old list at once (one comparison
// per slot), which keeps the dependent chain per insertion short.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&tv)[KMAX], int (&ti)[KMAX], float v, int e) {
  bool ge[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) ge[j] = tv[j] >= v;
#pragma unroll
  for (int j = KMAX - 1; j >= 0; --j) {
    const bool prev_ge = j == 0 ? true : ge[j > 0 ? j - 1 : 0];
    const float pv = j == 0 ? v : tv[j > 0 ? j - 1 : 0];
    const int pi = j == 0 ? e : ti[j > 0 ? j - 1 : 0];
    tv[j] = ge[j] ? tv[j] : (prev_ge ? v : pv);
    ti[j] = ge[j] ? ti[j] : (prev_ge ? e : pi);
  }
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

inline size_t dtype_size(int dtype) { return dtype == MOE_F32 ? 4 : 2; }

}  // namespace moe
