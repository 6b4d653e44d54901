// tc_bwd.cuh -- the elementwise steps of the tensor-core backward pass
// (the products run in tc_bgemm; launch_tc_backward in tc_backward.cuh gives
// the order).  The forward kernels, fed dO in place of U, give dU = dO * Y
// directly; the rest:
//   dY = dO * U;  T0, T1, T3 rows in bf16;
//   the reverse chunk scan of d(prefix): dS_h = sum_{g>h} f_g dP_g;
//   dZ = sum_k dT_k * gamma_k with per-block dgamma/dbeta partials.
// Row-wise kernels move 8 bf16 (16 bytes) per thread.  Included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

__device__ __forceinline__ float bf(const __nv_bfloat16 &x) { return __bfloat162float(x); }
__device__ __forceinline__ __nv_bfloat16 tob(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ void unpack8(const uint4 &v, float *f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}
__device__ __forceinline__ uint4 pack8(const float *f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// dY = dO * U over [rows][e] (bf16), 8 elements per thread; count8 = count / 8
__global__ void tcb_gate_dy(const uint4 *__restrict__ dO, const uint4 *__restrict__ U,
                            uint4 *__restrict__ dY, int64_t count8) {
  griddep_wait();  // launched as a dependent of the previous step
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count8) return;
  float g[8], u[8];
  unpack8(__ldcs(dO + i), g);
  unpack8(__ldcs(U + i), u);
#pragma unroll
  for (int k = 0; k < 8; ++k) g[k] *= u[k];
  dY[i] = pack8(g);
}

// T0, T1, T3 = Z * gamma_k + beta_k over [rows][s] (bf16), 8 columns per
// thread; gamma, beta [4][s] read as float4 (s % 8 == 0).
__global__ void tcb_affine_rows(const uint4 *__restrict__ Z, const float4 *__restrict__ gamma,
                                const float4 *__restrict__ beta, uint4 *__restrict__ T0,
                                uint4 *__restrict__ T1, uint4 *__restrict__ T3, int64_t count8,
                                int s) {
  griddep_wait();  // launched as a dependent of the previous step
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count8) return;
  const int a4 = (int)(i % (s / 8)) * 2;  // float4 index of the first column
  float z[8], t[8];
  unpack8(__ldcs(Z + i), z);
  uint4 *const out[3] = {T0, T1, T3};
  const int ks[3] = {0, 1, 3};
#pragma unroll
  for (int m = 0; m < 3; ++m) {
    const int o = ks[m] * (s / 4) + a4;
    const float4 g0 = __ldg(gamma + o), g1 = __ldg(gamma + o + 1);
    const float4 b0 = __ldg(beta + o), b1 = __ldg(beta + o + 1);
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = fmaf(z[k], g[k], b[k]);
    out[m][i] = pack8(t);
  }
}

// Reverse scan over chunks of d(prefix) [B][G][s][e] (bf16, in place, fp32
// sums), 8 columns per thread: causal dS_h = sum_{g>h} f_g dP_g; bidirectional
// slot (b, 0) gets f * sum_g dP_g (every chunk of the sequence reads it).
// f_g is the divisor's inverse that the forward scan applied to chunk g's
// prefix (1 with the per-position divisor, which the T2 rows carry).
__global__ void tcb_reverse_scan(uint4 *__restrict__ dP, int B, int G, int64_t se8, int n, int C,
                                 int causal, int lin_norm) {
  griddep_wait();  // launched as a dependent of the previous step
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * se8) return;
  const int64_t b = t / se8, x = t % se8;
  uint4 *p = dP + b * G * se8 + x;
  auto factor = [&](int g) -> float {
    if (lin_norm == kLinNormPosition) return 1.f;
    if (lin_norm == kLinNormSummed && causal) return g > 0 ? 1.f / ((float)g * (float)C) : 0.f;
    return 1.f / (float)n;
  };
  float run[8], v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) run[k] = 0.f;
  constexpr int UN = 8;
  if (causal) {
    for (int g1 = G; g1 > 0; g1 -= UN) {  // chunks g1-1 down to g1-UN
      uint4 in[UN];
#pragma unroll
      for (int u = 0; u < UN; ++u)
        if (g1 - 1 - u >= 0) in[u] = p[(int64_t)(g1 - 1 - u) * se8];
#pragma unroll
      for (int u = 0; u < UN; ++u) {
        const int g = g1 - 1 - u;
        if (g >= 0) {
          p[(int64_t)g * se8] = pack8(run);
          unpack8(in[u], v);
          const float f = factor(g);
#pragma unroll
          for (int k = 0; k < 8; ++k) run[k] = fmaf(f, v[k], run[k]);
        }
      }
    }
  } else {
    for (int g0 = 0; g0 < G; g0 += UN) {
      uint4 in[UN];
#pragma unroll
      for (int u = 0; u < UN; ++u)
        if (g0 + u < G) in[u] = p[(int64_t)(g0 + u) * se8];
#pragma unroll
      for (int u = 0; u < UN; ++u)
        if (g0 + u < G) {
          unpack8(in[u], v);
#pragma unroll
          for (int k = 0; k < 8; ++k) run[k] += v[k];
        }
    }
    const float f = factor(0);
#pragma unroll
    for (int k = 0; k < 8; ++k) run[k] *= f;
    p[0] = pack8(run);
  }
}

__device__ __forceinline__ void unpack4(const uint2 &v, float *f) {
  f[0] = bf16_lo(v.x);
  f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y);
  f[3] = bf16_hi(v.y);
}

// dZ = sum_k dT_k gamma_k over kTcbAffRows token rows per block, and the
// block's partial sums of dgamma_k = sum_t dT_k z and dbeta_k = sum_t dT_k.
// Block (s / 4, kTcbAffLanes): thread (x, y) takes columns 4x .. 4x + 3 of
// rows y, y + kTcbAffLanes, ...; the row lanes' sums are then added in lane
// order through shared memory, one of the eight quantities at a time.  dT2
// holds the gradient of the lin_q rows as the kernels used them (times
// 1/(t+1) with the per-position divisor), so that row factor is applied here.
constexpr int kTcbAffLanes = 8;
__global__ void tcb_affine_reduce(const uint2 *__restrict__ Z, const float *__restrict__ gamma,
                                  const uint2 *__restrict__ dT0, const uint2 *__restrict__ dT1,
                                  const uint2 *__restrict__ dT2, const uint2 *__restrict__ dT3,
                                  uint2 *__restrict__ dZ, float *__restrict__ part, int64_t rows,
                                  int n, int s, int lin_norm, int global) {
  griddep_wait();  // launched as a dependent of the previous step
  extern __shared__ float red[];  // [kTcbAffLanes][s]
  const int x = threadIdx.x, y = threadIdx.y, s4 = s / 4;
  const int64_t t0 = (int64_t)blockIdx.x * kTcbAffRows;
  float g[4][4], pg[4][4], pb[4][4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      g[k][c] = gamma[k * s + 4 * x + c];
      pg[k][c] = 0.f;
      pb[k][c] = 0.f;
    }
#pragma unroll 2
  for (int r = y; r < kTcbAffRows; r += kTcbAffLanes) {
    const int64_t t = t0 + r;
    if (t >= rows) break;
    const int64_t o = t * s4 + x;
    float z[4], d[4][4];
    unpack4(__ldcs(Z + o), z);
    unpack4(__ldcs(dT0 + o), d[0]);
    unpack4(__ldcs(dT1 + o), d[1]);
    if (global) {
      unpack4(__ldcs(dT2 + o), d[2]);
      unpack4(__ldcs(dT3 + o), d[3]);
      if (lin_norm == kLinNormPosition) {
        const float f = 1.f / (float)(t % n + 1);
#pragma unroll
        for (int c = 0; c < 4; ++c) d[2][c] *= f;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) d[2][c] = d[3][c] = 0.f;
    }
    float dz[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      dz[c] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        dz[c] = fmaf(d[k][c], g[k][c], dz[c]);
        pg[k][c] = fmaf(d[k][c], z[c], pg[k][c]);
        pb[k][c] += d[k][c];
      }
    }
    dZ[o] = make_uint2(pack_bf16x2(dz[0], dz[1]), pack_bf16x2(dz[2], dz[3]));
  }
  float *pp = part + (int64_t)blockIdx.x * 8 * s;
  const int tid = y * s4 + x, nthr = s4 * kTcbAffLanes;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float *v = q < 4 ? pg[q] : pb[q - 4];
#pragma unroll
    for (int c = 0; c < 4; ++c) red[y * s + 4 * x + c] = v[c];
    __syncthreads();
    for (int a = tid; a < s; a += nthr) {
      float tot = 0.f;
      for (int l = 0; l < kTcbAffLanes; ++l) tot += red[l * s + a];
      pp[q * s + a] = tot;
    }
    __syncthreads();
  }
}

// Sum of the nblk partials of each of the 8 s outputs (dgamma, then dbeta),
// in a fixed order: thread (x, y) of a (32, 32) block adds partials y, y+32,
// ...; the 32 sums are then added in y order.  grid ceil(8 s / 32).
__global__ void tcb_gamma_beta(const float *__restrict__ part, int nblk, int s,
                               float *__restrict__ dgamma, float *__restrict__ dbeta) {
  griddep_wait();  // launched as a dependent of the previous step
  __shared__ float acc[32][33];
  const int x = blockIdx.x * 32 + threadIdx.x, y = threadIdx.y;
  float v = 0.f;
  if (x < 8 * s)
    for (int i = y; i < nblk; i += 32) v += part[(int64_t)i * 8 * s + x];
  acc[y][threadIdx.x] = v;
  __syncthreads();
  if (y == 0 && x < 8 * s) {
    float tot = 0.f;
    for (int k = 0; k < 32; ++k) tot += acc[k][threadIdx.x];
    if (x < 4 * s)
      dgamma[x] = tot;
    else
      dbeta[x - 4 * s] = tot;
  }
}

}  // namespace
}  // namespace fmca
