// tc_scan.cuh -- the chunk-axis prefix of the per-chunk linear-attention
// states ("FLASH: Possibly the Most Interesting Efficient Transformer Design
// Recently", section "Mixed Chunk": the sum over all chunks of K^lin_h^T V_h,
// or its cumsum over the chunks before g for a decoder), scaled by 1/n.
// Device code of the tensor-core path, included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

// =====================================================================
// tc_state_scan: prefix (or total) over chunks of the bf16 states, in fp32,
// scaled by the global-term divisor's inverse (1/n by default; 1/(g*C) for
// causal chunk g with the tokens-summed divisor; 1 with the per-position
// divisor, which the T2 rows carry instead) and rounded to bf16.  The thread count is a multiple of 32
// for every shape this path takes (B * s * e / 8).
// =====================================================================
// LIN_NORM: the global-term divisor (kLinNorm*), one instantiation each, so
// that the default one is the plain 1/n scan.
template <int LIN_NORM>
__global__ void __launch_bounds__(256)
    tc_state_scan(const __nv_bfloat16 *__restrict__ S, __nv_bfloat16 *__restrict__ P, int B,
                  int G, int64_t se, float inv_n, int causal, int C) {
  // launched as a dependent of the prep kernel: wait for its states; let the
  // attention kernel start launching (it waits for this grid in turn)
  griddep_wait();
  griddep_launch_dependents();
  if (LIN_NORM == kLinNormNone) return;  // no global term: nothing to sum
  const int64_t per_b = se / 8;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * per_b) return;
  const int64_t b = t / per_b, x = (t % per_b) * 8;
  const __nv_bfloat16 *src = S + b * G * se + x;
  __nv_bfloat16 *dst = P + (causal ? b * G * se : b * se) + x;
  float run[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) run[i] = 0.f;
  const float keep = LIN_NORM == kLinNormPosition ? 1.0f : inv_n;  // all but summed+causal
  constexpr int U = 8;
  for (int g0 = 0; g0 < G; g0 += U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (g0 + u < G) v[u] = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)(g0 + u) * se));
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (g0 + u < G) {
        if (causal) {
          const int g = g0 + u;
          const float f = LIN_NORM != kLinNormSummed ? keep
                          : (g > 0 ? 1.0f / ((float)g * (float)C) : 0.0f);
          uint4 o;
          o.x = pack_bf16x2(run[0] * f, run[1] * f);
          o.y = pack_bf16x2(run[2] * f, run[3] * f);
          o.z = pack_bf16x2(run[4] * f, run[5] * f);
          o.w = pack_bf16x2(run[6] * f, run[7] * f);
          *reinterpret_cast<uint4 *>(dst + (int64_t)(g0 + u) * se) = o;
        }
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          run[2 * i] += bf16_lo(w[i]);
          run[2 * i + 1] += bf16_hi(w[i]);
        }
      }
    }
    // The states are dead once read: drop their lines from L2 so they are
    // never written back (eight lanes share a 128-byte line; every lane's
    // load has returned once the sums above used it).
    __syncwarp();
    if ((x & 63) == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (g0 + u < G) discard_l2_line(src + (int64_t)(g0 + u) * se);
    }
  }
  if (!causal) {
    uint4 o;
    o.x = pack_bf16x2(run[0] * keep, run[1] * keep);
    o.y = pack_bf16x2(run[2] * keep, run[3] * keep);
    o.z = pack_bf16x2(run[4] * keep, run[5] * keep);
    o.w = pack_bf16x2(run[6] * keep, run[7] * keep);
    *reinterpret_cast<uint4 *>(dst) = o;
  }
}

}  // namespace
}  // namespace fmca
