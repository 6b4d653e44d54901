// tc_common.cuh -- constants and helpers shared by the tensor-core kernels
// and the device status word (included only by tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace fmca {

// Device-side status: the first bounded wait that ran out (code, where).
// This header is included by exactly one translation unit (tc.cu).
__device__ int g_fmca_status = 0;
__device__ int g_fmca_where = 0;

namespace {

constexpr int kStatusTimeout = 7;                 // FMCA_ERR_TIMEOUT
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

__device__ __forceinline__ void record_timeout(int where) {
  if (atomicCAS(&g_fmca_status, 0, kStatusTimeout) == 0) atomicExch(&g_fmca_where, where);
}

constexpr int S_DIM = 128;     // attention width s handled by this path
constexpr int E_TILE = 256;    // e columns per accumulator tile
constexpr int KEY_STAGE = 64;  // keys (or state rows) per pipeline stage
constexpr int ROW_TILE = 128;  // rows per MMA tile (tcgen05 M)

// 8 consecutive floats (32-byte aligned) through the read-only cache.
__device__ __forceinline__ void load8(const float *__restrict__ p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// In place over one 16-byte chunk (8 bf16): x -> x * g + b, rounded to bf16.
__device__ __forceinline__ uint4 affine8(uint4 v, const float (&g)[8], const float (&b)[8]) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = pack_bf16x2(bf16_lo(w[i]) * g[2 * i] + b[2 * i],
                       bf16_hi(w[i]) * g[2 * i + 1] + b[2 * i + 1]);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// affine8 followed by a scale w of the 8 results, before rounding.
__device__ __forceinline__ uint4 affine8_scaled(uint4 v, const float (&g)[8], const float (&b)[8],
                                                float w) {
  uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    x[i] = pack_bf16x2((bf16_lo(x[i]) * g[2 * i] + b[2 * i]) * w,
                       (bf16_hi(x[i]) * g[2 * i + 1] + b[2 * i + 1]) * w);
  return make_uint4(x[0], x[1], x[2], x[3]);
}

}  // namespace
}  // namespace fmca
