// tc_bwd.cuh -- the elementwise steps of the tensor-core backward pass
// (the products run in tc_bgemm; see launch_tc_backward in tc.cu for the
// order).  With Y = quad + glob recomputed by the forward kernels:
//   dY = dO * U, dU = dO * Y;  T0, T1, T3 rows in bf16;
//   dS_ij = dw_ij * 2 a relu(a S_ij), with relu(a S_ij) = sqrt(w_ij) taken
//   from the stored weights w = relu(a S)^2 (0 where masked), plus the
//   per-chunk transposes of dS and w;
//   the reverse chunk scan of d(prefix): dS_h = sum_{g>h} f_g dP_g;
//   dZ = sum_k dT_k * gamma_k with per-block dgamma/dbeta partials.
// Included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

__device__ __forceinline__ float bf(const __nv_bfloat16 &x) { return __bfloat162float(x); }
__device__ __forceinline__ __nv_bfloat16 tob(float x) { return __float2bfloat16_rn(x); }

// dY = dO * U and dU = dO * Y over [rows][e] (bf16)
__global__ void tcb_gate_grads(const __nv_bfloat16 *__restrict__ dO,
                               const __nv_bfloat16 *__restrict__ U,
                               const __nv_bfloat16 *__restrict__ Y, __nv_bfloat16 *__restrict__ dY,
                               __nv_bfloat16 *__restrict__ dU, int64_t count) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const float g = bf(dO[i]);
  dY[i] = tob(g * bf(U[i]));
  dU[i] = tob(g * bf(Y[i]));
}

// T0, T1, T3 = Z * gamma_k + beta_k over [rows][s] (bf16)
__global__ void tcb_affine_rows(const __nv_bfloat16 *__restrict__ Z, const float *__restrict__ gamma,
                                const float *__restrict__ beta, __nv_bfloat16 *__restrict__ T0,
                                __nv_bfloat16 *__restrict__ T1, __nv_bfloat16 *__restrict__ T3,
                                int64_t count, int s) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const int a = (int)(i % s);
  const float z = bf(Z[i]);
  T0[i] = tob(z * gamma[a] + beta[a]);
  T1[i] = tob(z * gamma[s + a] + beta[s + a]);
  T3[i] = tob(z * gamma[3 * s + a] + beta[3 * s + a]);
}

// One 32 x 32 tile (query rows i, keys j) of chunk bg: dS = dw * 2 a sqrt(w)
// in place over dw, and the transposes dSt[j][i], Wt[j][i].  Causal: keys
// j > i are masked (the forward pass never writes those weights: they are
// not read, and the gradients there are 0).
// grid (B*G, C/32, C/32); block (32, 8).
__global__ void tcb_score_grads(__nv_bfloat16 *__restrict__ dw, const __nv_bfloat16 *__restrict__ W,
                                __nv_bfloat16 *__restrict__ dSt, __nv_bfloat16 *__restrict__ Wt,
                                int C, float quad_a, int causal) {
  __shared__ float ts[32][33], tw[32][33];
  const int64_t base = (int64_t)blockIdx.x * C * C;  // chunk bg: rows bg*C.. of [rows][C]
  const int i0 = blockIdx.y * 32, j0 = blockIdx.z * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int r = ty; r < 32; r += 8) {
    const int64_t o = base + (int64_t)(i0 + r) * C + j0 + tx;
    const bool keep = !causal || j0 + tx <= i0 + r;
    const float w = keep ? bf(W[o]) : 0.f;
    const float d = keep ? bf(dw[o]) * 2.f * quad_a * sqrtf(w) : 0.f;
    dw[o] = tob(d);
    ts[r][tx] = d;
    tw[r][tx] = w;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int64_t o = base + (int64_t)(j0 + r) * C + i0 + tx;
    dSt[o] = tob(ts[tx][r]);
    Wt[o] = tob(tw[tx][r]);
  }
}

// Reverse scan over chunks of d(prefix) [B][G][s][e] (bf16, in place, fp32
// sums): causal dS_h = sum_{g>h} f_g dP_g; bidirectional slot (b, 0) gets
// f * sum_g dP_g (every chunk of the sequence reads it).
__global__ void tcb_reverse_scan(__nv_bfloat16 *__restrict__ dP, int B, int G, int64_t se, int n,
                                 int C, int causal, int lin_norm) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * se) return;
  const int64_t b = t / se, x = t % se;
  __nv_bfloat16 *p = dP + b * G * se + x;
  auto factor = [&](int g) -> float {
    if (lin_norm == kLinNormPosition) return 1.f;
    if (lin_norm == kLinNormSummed && causal) return g > 0 ? 1.f / ((float)g * (float)C) : 0.f;
    return 1.f / (float)n;
  };
  if (causal) {
    float run = 0.f;
    for (int g = G - 1; g >= 0; --g) {
      const float v = bf(p[(int64_t)g * se]);
      p[(int64_t)g * se] = tob(run);
      run += factor(g) * v;
    }
  } else {
    float tot = 0.f;
    for (int g = 0; g < G; ++g) tot += bf(p[(int64_t)g * se]);
    p[0] = tob(tot * factor(0));
  }
}

// dV = dVq + dVl (bf16)
__global__ void tcb_add(const __nv_bfloat16 *__restrict__ a, const __nv_bfloat16 *__restrict__ b,
                        __nv_bfloat16 *__restrict__ out, int64_t count) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) out[i] = tob(bf(a[i]) + bf(b[i]));
}

// 64 token rows per block, one thread per column a (blockDim = s): dZ and
// per-block partial sums of dgamma_k, dbeta_k; dT2 holds the gradient of the
// lin_q rows as the kernels used them (times 1/(t+1) with the per-position
// divisor), so its row factor is applied here.
constexpr int kTcbAffRows = 64;
__global__ void tcb_affine_reduce(const __nv_bfloat16 *__restrict__ Z,
                                  const float *__restrict__ gamma,
                                  const __nv_bfloat16 *__restrict__ dT0,
                                  const __nv_bfloat16 *__restrict__ dT1,
                                  const __nv_bfloat16 *__restrict__ dT2,
                                  const __nv_bfloat16 *__restrict__ dT3,
                                  __nv_bfloat16 *__restrict__ dZ, float *__restrict__ part,
                                  int64_t rows, int n, int s, int lin_norm, int global) {
  const int a = threadIdx.x;
  const int64_t t0 = (int64_t)blockIdx.x * kTcbAffRows;
  float g[4], pg[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k) g[k] = gamma[k * s + a];
  for (int64_t t = t0; t < t0 + kTcbAffRows && t < rows; ++t) {
    const int64_t o = t * s + a;
    const float z = bf(Z[o]);
    float d[4];
    d[0] = bf(dT0[o]);
    d[1] = bf(dT1[o]);
    d[2] = global ? bf(dT2[o]) : 0.f;
    d[3] = global ? bf(dT3[o]) : 0.f;
    if (lin_norm == kLinNormPosition) d[2] *= 1.f / (float)(t % n + 1);
    float dz = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      dz = fmaf(d[k], g[k], dz);
      pg[k] = fmaf(d[k], z, pg[k]);
      pb[k] += d[k];
    }
    dZ[o] = tob(dz);
  }
  float *pp = part + (int64_t)blockIdx.x * 8 * s;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    pp[k * s + a] = pg[k];
    pp[(4 + k) * s + a] = pb[k];
  }
}

__global__ void tcb_gamma_beta(const float *__restrict__ part, int nblk, int s,
                               float *__restrict__ dgamma, float *__restrict__ dbeta) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= 8 * s) return;
  float acc = 0.f;
  for (int i = 0; i < nblk; ++i) acc += part[(int64_t)i * 8 * s + x];
  if (x < 4 * s)
    dgamma[x] = acc;
  else
    dbeta[x - 4 * s] = acc;
}

}  // namespace
}  // namespace fmca
