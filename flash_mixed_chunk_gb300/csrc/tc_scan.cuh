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
// divisor, which the T2 rows carry instead) and rounded to bf16.  One thread
// per 4 columns (8-byte accesses: more threads, so more loads in flight, for
// the same bytes), the chunks of its column in rounds of kScanU loads; the
// states are read once with evict-first loads.  The thread count is a
// multiple of 32 for every shape this path takes (B * s * e / 4).
// =====================================================================
constexpr int kScanCols = 4;
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
  const int64_t per_b = se / kScanCols;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * per_b) return;
  const int64_t b = t / per_b, x = (t % per_b) * kScanCols;
  const __nv_bfloat16 *src = S + b * G * se + x;
  __nv_bfloat16 *dst = P + (causal ? b * G * se : b * se) + x;
  float run[4] = {0.f, 0.f, 0.f, 0.f};
  const float keep = LIN_NORM == kLinNormPosition ? 1.0f : inv_n;  // all but summed+causal
  constexpr int kScanU = 8;
  for (int g0 = 0; g0 < G; g0 += kScanU) {
    uint2 v[kScanU];
#pragma unroll
    for (int u = 0; u < kScanU; ++u)
      if (g0 + u < G) v[u] = __ldcs(reinterpret_cast<const uint2 *>(src + (int64_t)(g0 + u) * se));
#pragma unroll
    for (int u = 0; u < kScanU; ++u) {
      if (g0 + u < G) {
        if (causal) {
          const int g = g0 + u;
          const float f = LIN_NORM != kLinNormSummed ? keep
                          : (g > 0 ? 1.0f / ((float)g * (float)C) : 0.0f);
          uint2 o;
          o.x = pack_bf16x2(run[0] * f, run[1] * f);
          o.y = pack_bf16x2(run[2] * f, run[3] * f);
          *reinterpret_cast<uint2 *>(dst + (int64_t)g * se) = o;
        }
        run[0] += bf16_lo(v[u].x);
        run[1] += bf16_hi(v[u].x);
        run[2] += bf16_lo(v[u].y);
        run[3] += bf16_hi(v[u].y);
      }
    }
  }
  if (!causal) {
    uint2 o;
    o.x = pack_bf16x2(run[0] * keep, run[1] * keep);
    o.y = pack_bf16x2(run[2] * keep, run[3] * keep);
    *reinterpret_cast<uint2 *>(dst) = o;
  }
}

// Segmented form of the scan for long chunk axes (G >= kScanSegMinG), where
// one thread per 8 columns walking all G chunks is a long chain of dependent
// rounds: a block is 64 column groups x kScanSeg segments of the chunk axis.
// Pass 1: each thread sums its segment's states; the segment totals meet in
// shared memory.  Pass 2 (causal): each thread starts from the sum of the
// segments before its own and rescans its segment, writing the scaled
// exclusive prefixes; the states are read again (from L2) and their lines
// dropped after this last read.  Bidirectional: segment 0's thread writes the
// scaled total.  Same factors and fp32 sums as tc_state_scan, in a different
// order of addition.
constexpr int kScanSeg = 4;
constexpr int kScanSegMinG = 64;
template <int LIN_NORM>
__global__ void __launch_bounds__(256)
    tc_state_scan_seg(const __nv_bfloat16 *__restrict__ S, __nv_bfloat16 *__restrict__ P, int B,
                      int G, int64_t se, float inv_n, int causal, int C) {
  griddep_wait();
  griddep_launch_dependents();
  if (LIN_NORM == kLinNormNone) return;
  __shared__ float tot[kScanSeg][64][9];  // [segment][column group][8 sums], padded
  const int xi = threadIdx.x % 64, sg = threadIdx.x / 64;
  const int64_t per_b = se / 8;
  const int64_t colg = (int64_t)blockIdx.x * 64 + xi;  // column group over all sequences
  const bool active = colg < (int64_t)B * per_b;
  const int64_t b = active ? colg / per_b : 0, x = active ? (colg % per_b) * 8 : 0;
  const int glen = (G + kScanSeg - 1) / kScanSeg;
  const int g_lo = sg * glen < G ? sg * glen : G, g_hi = g_lo + glen < G ? g_lo + glen : G;
  const __nv_bfloat16 *src = S + b * G * se + x;
  const float keep = LIN_NORM == kLinNormPosition ? 1.0f : inv_n;  // all but summed+causal
  constexpr int U = 8;
  float run[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) run[i] = 0.f;
  // pass 1: this segment's sum (the lines stay in L2 for pass 2 when causal)
  if (active) {
    for (int g0 = g_lo; g0 < g_hi; g0 += U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (g0 + u < g_hi) v[u] = *reinterpret_cast<const uint4 *>(src + (int64_t)(g0 + u) * se);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (g0 + u < g_hi) {
          const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            run[2 * i] += bf16_lo(w[i]);
            run[2 * i + 1] += bf16_hi(w[i]);
          }
        }
      if (!causal) {  // the last read of these states
        __syncwarp();
        if ((x & 63) == 0) {
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (g0 + u < g_hi) discard_l2_line(src + (int64_t)(g0 + u) * se);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) tot[sg][xi][i] = run[i];
  __syncthreads();
  if (!active) return;
  if (!causal) {
    if (sg == 0) {
      float t[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        t[i] = 0.f;
        for (int q = 0; q < kScanSeg; ++q) t[i] += tot[q][xi][i];
      }
      uint4 o;
      o.x = pack_bf16x2(t[0] * keep, t[1] * keep);
      o.y = pack_bf16x2(t[2] * keep, t[3] * keep);
      o.z = pack_bf16x2(t[4] * keep, t[5] * keep);
      o.w = pack_bf16x2(t[6] * keep, t[7] * keep);
      *reinterpret_cast<uint4 *>(P + b * se + x) = o;
    }
    return;
  }
  // pass 2: the segments before this one, then the exclusive scan of this one
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    run[i] = 0.f;
    for (int q = 0; q < sg; ++q) run[i] += tot[q][xi][i];
  }
  __nv_bfloat16 *dst = P + b * G * se + x;
  for (int g0 = g_lo; g0 < g_hi; g0 += U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (g0 + u < g_hi) v[u] = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)(g0 + u) * se));
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (g0 + u < g_hi) {
        const int g = g0 + u;
        const float f = LIN_NORM != kLinNormSummed ? keep
                        : (g > 0 ? 1.0f / ((float)g * (float)C) : 0.0f);
        uint4 o;
        o.x = pack_bf16x2(run[0] * f, run[1] * f);
        o.y = pack_bf16x2(run[2] * f, run[3] * f);
        o.z = pack_bf16x2(run[4] * f, run[5] * f);
        o.w = pack_bf16x2(run[6] * f, run[7] * f);
        *reinterpret_cast<uint4 *>(dst + (int64_t)g * se) = o;
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          run[2 * i] += bf16_lo(w[i]);
          run[2 * i + 1] += bf16_hi(w[i]);
        }
      }
    }
    __syncwarp();
    if ((x & 63) == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (g0 + u < g_hi) discard_l2_line(src + (int64_t)(g0 + u) * se);
    }
  }
}

}  // namespace
}  // namespace fmca
