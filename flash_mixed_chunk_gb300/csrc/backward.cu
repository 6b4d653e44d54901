// backward.cu -- gradients of the mixed-chunk attention core on the CUDA
// cores (fp32).  The pages ("FLASH: Possibly the Most Interesting Efficient
// Transformer Design Recently", section "Mixed Chunk") give the forward pass;
// with Y = quad + glob and O = U * Y, calculus gives, for an incoming dO:
//
//   dU = dO * Y,  dY = dO * U
//   quad: w_ij = relu(a T0_i . T1_j)^2 (masked), a = sqrt(quad_scale)
//         dV_j  += sum_i w_ij dY_i
//         dS_ij  = (dY_i . V_j) * 2 a relu(a T0_i . T1_j)
//         dT0_i  = sum_j dS_ij T1_j,  dT1_j = sum_i dS_ij T0_i
//   glob: P~_g = f_g * sum_{h<g (or all h)} T3_h^T V_h, glob_t = w_t T2_t . P~_g
//         dT2_t  = w_t dY_t P~_g^T
//         dP~_g  = sum_{t in g} w_t T2_t^T dY_t
//         dS_h   = sum_{g>h} f_g dP~_g   (causal; every h: f sum_g dP~_g otherwise)
//         dT3_t  = V_t dS_h^T,  dV_t += T3_t dS_h
//   affine maps: dZ = sum_k dT_k * gamma_k, dgamma_k = sum_t dT_k * Z, dbeta_k = sum_t dT_k
//
// f_g and w_t are the global-term divisor's inverse (1/n; 1/(g C) for the
// tokens-summed divisor; w_t = 1/(t+1) for the per-position one; 0 without a
// global term).  Reductions have a fixed order (no atomics): the gradients are
// deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"

namespace fmca {
namespace {

template <typename T>
__device__ __forceinline__ float bw_f(T v);
template <>
__device__ __forceinline__ float bw_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float bw_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T>
__device__ __forceinline__ T bw_t(float v);
template <>
__device__ __forceinline__ float bw_t<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 bw_t<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

constexpr int kBR = 32;    // rows (tokens, state rows or keys) per block
constexpr int kBC = 64;    // e columns per block
constexpr int kBK = 32;    // keys per inner block
constexpr int kBT = 256;   // threads
constexpr int kBP = kBR * kBC / kBT;  // 8 outputs per thread

// inverse divisor of chunk g's global sum; 1 for the per-position divisor
// (the rows carry it), 0 without a global term
__device__ __forceinline__ float chunk_factor(int g, int n, int C, int causal, int lin_norm) {
  if (lin_norm == kLinNormNone) return 0.f;
  if (lin_norm == kLinNormPosition) return 1.f;
  if (lin_norm == kLinNormSummed && causal) return g > 0 ? 1.f / ((float)g * (float)C) : 0.f;
  return 1.f / (float)n;
}
__device__ __forceinline__ float row_factor(int t, int lin_norm) {
  return lin_norm == kLinNormPosition ? 1.f / (float)(t + 1) : 1.f;
}

// out[bg][a][c] = sum_{j in chunk g} L_j[a] R_j[c], L = (Z gamma_k + beta_k) (times
// the row factor when row_scaled), R = a row-major [B*n][e] matrix.
// grid (B*G, ceil(e/64), ceil(s/32)); block 256.
template <typename T, typename RT>
__global__ void __launch_bounds__(kBT)
    bwd_chunk_outer(const T *__restrict__ Z, const RT *__restrict__ R,
                    const float *__restrict__ gamma, const float *__restrict__ beta, int k,
                    int row_scaled, int lin_norm, float *__restrict__ out, int n, int s, int e,
                    int C, int G) {
  __shared__ float lt[kBK][kBR + 1];
  __shared__ float rb[kBK][kBC];
  const int bg = blockIdx.x, b = bg / G, g = bg % G;
  const int c0 = blockIdx.y * kBC, a0 = blockIdx.z * kBR;
  const int tid = threadIdx.x, col = tid % kBC, rbase = tid / kBC;
  const int64_t row0 = (int64_t)b * n + (int64_t)g * C;
  float acc[kBP];
#pragma unroll
  for (int i = 0; i < kBP; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < C; j0 += kBK) {
    for (int x = tid; x < kBK * kBR; x += kBT) {
      const int j = x / kBR, a = x % kBR;
      float v = 0.f;
      if (j0 + j < C && a0 + a < s) {
        v = bw_f(Z[(row0 + j0 + j) * s + a0 + a]) * gamma[k * s + a0 + a] + beta[k * s + a0 + a];
        if (row_scaled) v *= row_factor(g * C + j0 + j, lin_norm);
      }
      lt[j][a] = v;
    }
    for (int x = tid; x < kBK * kBC; x += kBT) {
      const int j = x / kBC, c = x % kBC;
      rb[j][c] = (j0 + j < C && c0 + c < e) ? bw_f(R[(row0 + j0 + j) * e + c0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kBK; ++j) {
      const float rv = rb[j][col];
#pragma unroll
      for (int i = 0; i < kBP; ++i) acc[i] = fmaf(lt[j][rbase + 4 * i], rv, acc[i]);
    }
    __syncthreads();
  }
  if (c0 + col < e) {
    float *dst = out + (int64_t)bg * s * e;
#pragma unroll
    for (int i = 0; i < kBP; ++i) {
      const int a = a0 + rbase + 4 * i;
      if (a < s) dst[(int64_t)a * e + c0 + col] = acc[i];
    }
  }
}

// P~[b][g] = f_g sum_{h<g} S[b][h] (causal) or P~[b][0] = f sum_h S[b][h]
__global__ void bwd_prefix(const float *__restrict__ S, float *__restrict__ P, int B, int G,
                           int64_t se, int n, int C, int causal, int lin_norm) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * se) return;
  const int64_t b = t / se, x = t % se;
  const float *src = S + b * G * se + x;
  float run = 0.f;
  if (causal) {
    float *dst = P + b * G * se + x;
    for (int g = 0; g < G; ++g) {
      dst[(int64_t)g * se] = run * chunk_factor(g, n, C, causal, lin_norm);
      run += src[(int64_t)g * se];
    }
  } else {
    for (int g = 0; g < G; ++g) run += src[(int64_t)g * se];
    P[b * se + x] = run * chunk_factor(0, n, C, causal, lin_norm);
  }
}

// dS[b][h] = sum_{g>h} f_g dP[b][g] in place (causal); dS[b][0] = f sum_g dP[b][g]
// (non-causal: every chunk reads slot 0)
__global__ void bwd_reverse_scan(float *__restrict__ dP, int B, int G, int64_t se, int n, int C,
                                 int causal, int lin_norm) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * se) return;
  const int64_t b = t / se, x = t % se;
  float *p = dP + b * G * se + x;
  if (causal) {
    float run = 0.f;
    for (int g = G - 1; g >= 0; --g) {
      const float v = p[(int64_t)g * se];
      p[(int64_t)g * se] = run;
      run += chunk_factor(g, n, C, causal, lin_norm) * v;
    }
  } else {
    float tot = 0.f;
    for (int g = 0; g < G; ++g) tot += p[(int64_t)g * se];
    p[0] = tot * chunk_factor(0, n, C, causal, lin_norm);
  }
}

// dY = dO * U (fp32), elementwise over [B*n][e].
template <typename T>
__global__ void bwd_dy(const T *__restrict__ dO, const T *__restrict__ U, float *__restrict__ dY,
                       int64_t count) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) dY[i] = bw_f(dO[i]) * bw_f(U[i]);
}

// Rows [r0, r0+32) of chunk bg, columns [c0, c0+64): Y = quad + glob from the
// stored relu^2 weights W and the scaled prefix; dU = dO * Y.
// grid (B*G*ceil(C/32), ceil(e/64)); dynamic smem (32*s + 32*33 + 32*64) floats.
template <typename T>
__global__ void __launch_bounds__(kBT)
    bwd_rows(const T *__restrict__ Z, const T *__restrict__ V, const T *__restrict__ dO,
             const float *__restrict__ gamma, const float *__restrict__ beta,
             const float *__restrict__ W, const float *__restrict__ P, T *__restrict__ dU, int n,
             int s, int e, int C, int G, int causal, int lin_norm) {
  extern __shared__ float sm[];
  float *t2 = sm;                      // [32][s] lin_q rows
  float *w = t2 + kBR * s;             // [32][33] weights
  float *vb = w + kBR * (kBK + 1);     // [32][64]
  const int nrb = (C + kBR - 1) / kBR;
  const int bg = blockIdx.x / nrb, rbk = blockIdx.x % nrb;
  const int b = bg / G, g = bg % G;
  const int c0 = blockIdx.y * kBC;
  const int tid = threadIdx.x, col = tid % kBC, rbase = tid / kBC;
  const int64_t chunk0 = (int64_t)b * n + (int64_t)g * C;
  const int r0 = rbk * kBR;
  const float *Wb = W + (int64_t)bg * C * C;
  float acc[kBP];
#pragma unroll
  for (int i = 0; i < kBP; ++i) acc[i] = 0.f;
  const int kb_end = causal ? rbk : nrb - 1;
  for (int kb = 0; kb <= kb_end; ++kb) {
    const int k0 = kb * kBK;
    __syncthreads();
    for (int x = tid; x < kBR * kBK; x += kBT) {
      const int r = x / kBK, j = x % kBK;
      w[r * (kBK + 1) + j] = (r0 + r < C && k0 + j < C) ? Wb[(int64_t)(r0 + r) * C + k0 + j] : 0.f;
    }
    for (int x = tid; x < kBK * kBC; x += kBT) {
      const int j = x / kBC, c = x % kBC;
      vb[x] = (k0 + j < C && c0 + c < e) ? bw_f(V[(chunk0 + k0 + j) * e + c0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kBK; ++j) {
      const float vv = vb[j * kBC + col];
#pragma unroll
      for (int i = 0; i < kBP; ++i) acc[i] = fmaf(w[(rbase + 4 * i) * (kBK + 1) + j], vv, acc[i]);
    }
  }
  if (lin_norm != kLinNormNone) {
    __syncthreads();
    for (int x = tid; x < kBR * s; x += kBT) {
      const int r = x / s, a = x % s;
      const float z = (r0 + r < C) ? bw_f(Z[(chunk0 + r0 + r) * s + a]) : 0.f;
      t2[x] = (z * gamma[2 * s + a] + beta[2 * s + a]) * row_factor(g * C + r0 + r, lin_norm);
    }
    const float *pg = P + (int64_t)(causal ? bg : b) * s * e;
    for (int a0 = 0; a0 < s; a0 += kBK) {
      __syncthreads();
      for (int x = tid; x < kBK * kBC; x += kBT) {
        const int a = x / kBC, c = x % kBC;
        vb[x] = (a0 + a < s && c0 + c < e) ? pg[(int64_t)(a0 + a) * e + c0 + c] : 0.f;
      }
      __syncthreads();
      const int amax = min(kBK, s - a0);
      for (int a = 0; a < amax; ++a) {
        const float pv = vb[a * kBC + col];
#pragma unroll
        for (int i = 0; i < kBP; ++i) acc[i] = fmaf(t2[(rbase + 4 * i) * s + a0 + a], pv, acc[i]);
      }
    }
  }
  if (c0 + col < e) {
#pragma unroll
    for (int i = 0; i < kBP; ++i) {
      const int r = r0 + rbase + 4 * i;
      if (r < C) {
        const int64_t off = (chunk0 + r) * e + c0 + col;
        dU[off] = bw_t<T>(bw_f(dO[off]) * acc[i]);
      }
    }
  }
}

// Row block rb (32 query rows i) of chunk bg: for every key block, the relu^2
// weights w_ij and score gradients dS_ij = (dY_i . V_j) 2 a relu(a S_ij), both
// stored [bg][C][C]; dT0_i = sum_j dS_ij T1_j written to dT0.
// grid B*G*ceil(C/32); dynamic smem (32*s + 32*(s+1) + 32*64 + 32*65 + 2*32*33)
// floats (key rows padded to odd strides: no bank conflicts across the keys).
template <typename T>
__global__ void __launch_bounds__(kBT)
    bwd_quad_scores(const T *__restrict__ Z, const T *__restrict__ V,
                    const float *__restrict__ dY, const float *__restrict__ gamma,
                    const float *__restrict__ beta, float *__restrict__ W, float *__restrict__ dS,
                    float *__restrict__ dT0, int n, int s, int e, int C, int G, int causal,
                    float quad_a) {
  extern __shared__ float sm[];
  float *t0 = sm;                 // [32][s]
  float *t1 = t0 + kBR * s;       // [32][s + 1]
  float *yr = t1 + kBK * (s + 1); // [32][64] dY rows
  float *vk = yr + kBR * kBC;     // [32][65] V keys
  float *dw = vk + kBK * (kBC + 1);  // [32][33]
  float *ds = dw + kBR * (kBK + 1);  // [32][33]
  const int nrb = (C + kBR - 1) / kBR;
  const int bg = blockIdx.x / nrb, rbk = blockIdx.x % nrb;
  const int b = bg / G, g = bg % G;
  const int tid = threadIdx.x;
  const int64_t chunk0 = (int64_t)b * n + (int64_t)g * C;
  const int r0 = rbk * kBR;
  for (int x = tid; x < kBR * s; x += kBT) {
    const int r = x / s, a = x % s;
    const float z = (r0 + r < C) ? bw_f(Z[(chunk0 + r0 + r) * s + a]) : 0.f;
    t0[x] = z * gamma[a] + beta[a];
  }
  // dT0 accumulators: thread owns (row, a) pairs x = tid + 256 q
  constexpr int kMaxQ = (kBR * 256 + kBT - 1) / kBT;  // s <= 256
  float dacc[kMaxQ];
#pragma unroll
  for (int q = 0; q < kMaxQ; ++q) dacc[q] = 0.f;
  const int kb_end = causal ? rbk : nrb - 1;
  float *Wb = W + (int64_t)bg * C * C, *dSb = dS + (int64_t)bg * C * C;
  for (int kb = 0; kb <= kb_end; ++kb) {
    const int k0 = kb * kBK;
    __syncthreads();
    for (int x = tid; x < kBK * s; x += kBT) {
      const int j = x / s, a = x % s;
      const float z = (k0 + j < C) ? bw_f(Z[(chunk0 + k0 + j) * s + a]) : 0.f;
      t1[j * (s + 1) + a] = z * gamma[s + a] + beta[s + a];
    }
    // dw_ij = dY_i . V_j over e, in 64-column slabs; thread owns 4 (i, j)
    float dacc_ij[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c0 = 0; c0 < e; c0 += kBC) {
      __syncthreads();
      for (int x = tid; x < kBR * kBC; x += kBT) {
        const int r = x / kBC, c = x % kBC;
        yr[x] = (r0 + r < C && c0 + c < e) ? dY[(chunk0 + r0 + r) * e + c0 + c] : 0.f;
        vk[r * (kBC + 1) + c] =
            (k0 + r < C && c0 + c < e) ? bw_f(V[(chunk0 + k0 + r) * e + c0 + c]) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int x = tid + kBT * q, r = x / kBK, j = x % kBK;
        float d = dacc_ij[q];
#pragma unroll 8
        for (int c = 0; c < kBC; ++c) d = fmaf(yr[r * kBC + c], vk[j * (kBC + 1) + c], d);
        dacc_ij[q] = d;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int x = tid + kBT * q, r = x / kBK, j = x % kBK;
      float sc = 0.f;
      for (int a = 0; a < s; ++a) sc = fmaf(t0[r * s + a], t1[j * (s + 1) + a], sc);
      const float rl = fmaxf(sc * quad_a, 0.f);
      const bool valid = (r0 + r < C) && (k0 + j < C) && (!causal || k0 + j <= r0 + r);
      const float wv = valid ? rl * rl : 0.f;
      const float dv = valid ? dacc_ij[q] * 2.f * quad_a * rl : 0.f;
      ds[r * (kBK + 1) + j] = dv;
      if (r0 + r < C && k0 + j < C) {
        Wb[(int64_t)(r0 + r) * C + k0 + j] = wv;
        dSb[(int64_t)(r0 + r) * C + k0 + j] = dv;
      }
    }
    __syncthreads();
    // dT0[r][a] += sum_j ds[r][j] t1[j][a]
#pragma unroll
    for (int q = 0; q < kMaxQ; ++q) {
      const int x = tid + kBT * q;
      if (x < kBR * s) {
        const int r = x / s, a = x % s;
        float d = dacc[q];
        for (int j = 0; j < kBK; ++j) d = fmaf(ds[r * (kBK + 1) + j], t1[j * (s + 1) + a], d);
        dacc[q] = d;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kMaxQ; ++q) {
    const int x = tid + kBT * q;
    if (x < kBR * s) {
      const int r = x / s, a = x % s;
      if (r0 + r < C) dT0[(chunk0 + r0 + r) * s + a] = dacc[q];
    }
  }
}

// Key block kb (32 keys j) of chunk bg: dT1_j = sum_i dS_ij T0_i over the rows
// that see key j.  grid B*G*ceil(C/32); dynamic smem (32*s + 32*33) floats.
template <typename T>
__global__ void __launch_bounds__(kBT)
    bwd_quad_keys(const T *__restrict__ Z, const float *__restrict__ gamma,
                  const float *__restrict__ beta, const float *__restrict__ dS,
                  float *__restrict__ dT1, int n, int s, int C, int G, int causal) {
  extern __shared__ float sm[];
  float *t0 = sm;             // [32][s] query rows
  float *ds = t0 + kBR * s;   // [32 i][33]
  const int nrb = (C + kBR - 1) / kBR;
  const int bg = blockIdx.x / nrb, kbk = blockIdx.x % nrb;
  const int b = bg / G, g = bg % G;
  const int tid = threadIdx.x;
  const int64_t chunk0 = (int64_t)b * n + (int64_t)g * C;
  const int k0 = kbk * kBK;
  constexpr int kMaxQ = (kBK * 256 + kBT - 1) / kBT;
  float acc[kMaxQ];
#pragma unroll
  for (int q = 0; q < kMaxQ; ++q) acc[q] = 0.f;
  const float *dSb = dS + (int64_t)bg * C * C;
  for (int rb = causal ? kbk : 0; rb < nrb; ++rb) {
    const int r0 = rb * kBR;
    __syncthreads();
    for (int x = tid; x < kBR * s; x += kBT) {
      const int r = x / s, a = x % s;
      const float z = (r0 + r < C) ? bw_f(Z[(chunk0 + r0 + r) * s + a]) : 0.f;
      t0[x] = z * gamma[a] + beta[a];
    }
    for (int x = tid; x < kBR * kBK; x += kBT) {
      const int r = x / kBK, j = x % kBK;
      ds[r * (kBK + 1) + j] =
          (r0 + r < C && k0 + j < C) ? dSb[(int64_t)(r0 + r) * C + k0 + j] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kMaxQ; ++q) {
      const int x = tid + kBT * q;
      if (x < kBK * s) {
        const int j = x / s, a = x % s;
        float d = acc[q];
        for (int r = 0; r < kBR; ++r) d = fmaf(ds[r * (kBK + 1) + j], t0[r * s + a], d);
        acc[q] = d;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kMaxQ; ++q) {
    const int x = tid + kBT * q;
    if (x < kBK * s) {
      const int j = x / s, a = x % s;
      if (k0 + j < C) dT1[(chunk0 + k0 + j) * s + a] = acc[q];
    }
  }
}

// Rows [r0, r0+32) of chunk bg, state rows [a0, a0+32):
//   dT2[t][a] = w_t sum_c dY[t][c] P~[g][a][c],  dT3[t][a] = sum_c V[t][c] dS[h][a][c]
// grid (B*G*ceil(C/32), ceil(s/32)); static smem.
template <typename T>
__global__ void __launch_bounds__(kBT)
    bwd_lin_rows(const T *__restrict__ V, const float *__restrict__ dY,
                 const float *__restrict__ P, const float *__restrict__ dSt,
                 float *__restrict__ dT2, float *__restrict__ dT3, int n, int s, int e, int C,
                 int G, int causal, int lin_norm) {
  __shared__ float yr[kBR][kBC + 1], vr[kBR][kBC + 1], pt[kBR][kBC + 1], st[kBR][kBC + 1];
  const int nrb = (C + kBR - 1) / kBR;
  const int bg = blockIdx.x / nrb, rbk = blockIdx.x % nrb;
  const int b = bg / G, g = bg % G;
  const int a0 = blockIdx.y * kBR;
  const int tid = threadIdx.x;
  const int64_t chunk0 = (int64_t)b * n + (int64_t)g * C;
  const int r0 = rbk * kBR;
  const float *pg = P + (int64_t)(causal ? bg : b) * s * e;
  const float *sg = dSt + (int64_t)(causal ? bg : (int64_t)b * G) * s * e;
  // thread owns (r, a) pairs x = tid + 256 q, q < 4
  float a2[4] = {0.f, 0.f, 0.f, 0.f}, a3[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c0 = 0; c0 < e; c0 += kBC) {
    __syncthreads();
    for (int x = tid; x < kBR * kBC; x += kBT) {
      const int r = x / kBC, c = x % kBC;
      const bool ok = r0 + r < C && c0 + c < e;
      yr[r][c] = ok ? dY[(chunk0 + r0 + r) * e + c0 + c] : 0.f;
      vr[r][c] = ok ? bw_f(V[(chunk0 + r0 + r) * e + c0 + c]) : 0.f;
      const bool oka = a0 + r < s && c0 + c < e;
      pt[r][c] = oka ? pg[(int64_t)(a0 + r) * e + c0 + c] : 0.f;
      st[r][c] = oka ? sg[(int64_t)(a0 + r) * e + c0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int x = tid + kBT * q, r = x / kBR, a = x % kBR;
      float d2 = a2[q], d3 = a3[q];
#pragma unroll 8
      for (int c = 0; c < kBC; ++c) {
        d2 = fmaf(yr[r][c], pt[a][c], d2);
        d3 = fmaf(vr[r][c], st[a][c], d3);
      }
      a2[q] = d2;
      a3[q] = d3;
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int x = tid + kBT * q, r = x / kBR, a = x % kBR;
    if (r0 + r < C && a0 + a < s) {
      const int64_t o = (chunk0 + r0 + r) * s + a0 + a;
      dT2[o] = a2[q] * row_factor(g * C + r0 + r, lin_norm);
      dT3[o] = a3[q];
    }
  }
}

// Key rows [k0, k0+32) of chunk bg, columns [c0, c0+64):
//   dV_j = sum_{i sees j} W_ij dY_i + sum_a T3_j[a] dS[h][a][c]
// grid (B*G*ceil(C/32), ceil(e/64)); dynamic smem (32*s + 32*33 + 32*64) floats.
template <typename T>
__global__ void __launch_bounds__(kBT)
    bwd_dv(const T *__restrict__ Z, const float *__restrict__ gamma,
           const float *__restrict__ beta, const float *__restrict__ W,
           const float *__restrict__ dY, const float *__restrict__ dSt, T *__restrict__ dV, int n,
           int s, int e, int C, int G, int causal, int lin_norm) {
  extern __shared__ float sm[];
  float *t3 = sm;                 // [32][s]
  float *wt = t3 + kBK * s;       // [32 i][33 j]
  float *vb = wt + kBR * (kBK + 1);  // [32][64]
  const int nrb = (C + kBR - 1) / kBR;
  const int bg = blockIdx.x / nrb, kbk = blockIdx.x % nrb;
  const int b = bg / G, g = bg % G;
  const int c0 = blockIdx.y * kBC;
  const int tid = threadIdx.x, col = tid % kBC, jbase = tid / kBC;
  const int64_t chunk0 = (int64_t)b * n + (int64_t)g * C;
  const int k0 = kbk * kBK;
  float acc[kBP];
#pragma unroll
  for (int q = 0; q < kBP; ++q) acc[q] = 0.f;
  const float *Wb = W + (int64_t)bg * C * C;
  for (int rb = causal ? kbk : 0; rb < nrb; ++rb) {
    const int r0 = rb * kBR;
    __syncthreads();
    for (int x = tid; x < kBR * kBK; x += kBT) {
      const int r = x / kBK, j = x % kBK;
      wt[r * (kBK + 1) + j] = (r0 + r < C && k0 + j < C) ? Wb[(int64_t)(r0 + r) * C + k0 + j] : 0.f;
    }
    for (int x = tid; x < kBR * kBC; x += kBT) {
      const int r = x / kBC, c = x % kBC;
      vb[x] = (r0 + r < C && c0 + c < e) ? dY[(chunk0 + r0 + r) * e + c0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int r = 0; r < kBR; ++r) {
      const float yv = vb[r * kBC + col];
#pragma unroll
      for (int q = 0; q < kBP; ++q) acc[q] = fmaf(wt[r * (kBK + 1) + jbase + 4 * q], yv, acc[q]);
    }
  }
  if (lin_norm != kLinNormNone) {
    const float *sg = dSt + (int64_t)(causal ? bg : (int64_t)b * G) * s * e;
    for (int x = tid; x < kBK * s; x += kBT) {
      const int j = x / s, a = x % s;
      const float z = (k0 + j < C) ? bw_f(Z[(chunk0 + k0 + j) * s + a]) : 0.f;
      t3[x] = z * gamma[3 * s + a] + beta[3 * s + a];
    }
    for (int a0 = 0; a0 < s; a0 += kBK) {
      __syncthreads();
      for (int x = tid; x < kBK * kBC; x += kBT) {
        const int a = x / kBC, c = x % kBC;
        vb[x] = (a0 + a < s && c0 + c < e) ? sg[(int64_t)(a0 + a) * e + c0 + c] : 0.f;
      }
      __syncthreads();
      const int amax = min(kBK, s - a0);
      for (int a = 0; a < amax; ++a) {
        const float sv = vb[a * kBC + col];
#pragma unroll
        for (int q = 0; q < kBP; ++q) acc[q] = fmaf(t3[(jbase + 4 * q) * s + a0 + a], sv, acc[q]);
      }
    }
  }
  if (c0 + col < e) {
#pragma unroll
    for (int q = 0; q < kBP; ++q) {
      const int j = k0 + jbase + 4 * q;
      if (j < C) dV[(chunk0 + j) * e + c0 + col] = bw_t<T>(acc[q]);
    }
  }
}

// 64 token rows per block, one thread per column a (blockDim = s):
// dZ[t][a] = sum_k dT_k[t][a] gamma_k[a]; per-block partial sums of
// dgamma_k[a] = sum_t dT_k[t][a] Z[t][a] and dbeta_k[a] = sum_t dT_k[t][a].
constexpr int kAffRows = 64;
template <typename T>
__global__ void bwd_affine(const T *__restrict__ Z, const float *__restrict__ gamma,
                           const float *__restrict__ dT, T *__restrict__ dZ,
                           float *__restrict__ part, int64_t rows, int s) {
  const int a = threadIdx.x;
  const int64_t t0 = (int64_t)blockIdx.x * kAffRows;
  float g[4], pg[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k) g[k] = gamma[k * s + a];
  for (int64_t t = t0; t < t0 + kAffRows && t < rows; ++t) {
    const float z = bw_f(Z[t * s + a]);
    float dz = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float d = dT[((int64_t)k * rows + t) * s + a];
      dz = fmaf(d, g[k], dz);
      pg[k] = fmaf(d, z, pg[k]);
      pb[k] += d;
    }
    dZ[t * s + a] = bw_t<T>(dz);
  }
  float *pp = part + (int64_t)blockIdx.x * 8 * s;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    pp[k * s + a] = pg[k];
    pp[(4 + k) * s + a] = pb[k];
  }
}

// dgamma / dbeta = the partials summed over blocks in block order.
__global__ void bwd_gamma_beta(const float *__restrict__ part, int nblk, int s,
                               float *__restrict__ dgamma, float *__restrict__ dbeta) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;  // over 8*s
  if (x >= 8 * s) return;
  float acc = 0.f;
  for (int i = 0; i < nblk; ++i) acc += part[(int64_t)i * 8 * s + x];
  if (x < 4 * s)
    dgamma[x] = acc;
  else
    dbeta[x - 4 * s] = acc;
}

template <typename T>
int launch_backward_impl(const void *Zv, const void *Vv, const void *Uv, const float *gamma,
                         const float *beta, const void *dOv, void *dZv, void *dVv, void *dUv,
                         float *dgamma, float *dbeta, int B, int n, int s, int e, int C,
                         int causal, const Variant &var, void *workspace, cudaStream_t stream) {
  const BackwardLayout L = backward_layout(B, n, s, e, C, causal);
  char *ws = static_cast<char *>(workspace);
  float *S = reinterpret_cast<float *>(ws + L.states);
  float *P = reinterpret_cast<float *>(ws + L.prefix);
  float *dP = reinterpret_cast<float *>(ws + L.dprefix);
  float *dY = reinterpret_cast<float *>(ws + L.dY);
  float *W = reinterpret_cast<float *>(ws + L.W);
  float *dS = reinterpret_cast<float *>(ws + L.dS);
  float *dT = reinterpret_cast<float *>(ws + L.dT);
  float *part = reinterpret_cast<float *>(ws + L.part);
  const T *Z = static_cast<const T *>(Zv);
  const T *V = static_cast<const T *>(Vv);
  const T *U = static_cast<const T *>(Uv);
  const T *dO = static_cast<const T *>(dOv);
  T *dZ = static_cast<T *>(dZv);
  T *dV = static_cast<T *>(dVv);
  T *dU = static_cast<T *>(dUv);
  const int G = n / C;
  const int64_t rows = (int64_t)B * n;
  const int64_t se = (int64_t)s * e;
  const int nrb = (C + kBR - 1) / kBR;
  const bool glob = var.lin_norm != kLinNormNone;
  const int lanes_blocks = (int)((B * se + 255) / 256);
  // forward pieces: chunk states and their (scaled) prefix
  if (glob) {
    dim3 g1(B * G, (e + kBC - 1) / kBC, (s + kBR - 1) / kBR);
    bwd_chunk_outer<T, T><<<g1, kBT, 0, stream>>>(Z, V, gamma, beta, 3, 0, var.lin_norm, S, n, s,
                                                   e, C, G);
    bwd_prefix<<<lanes_blocks, 256, 0, stream>>>(S, P, B, G, se, n, C, causal, var.lin_norm);
  }
  // dY = dO * U; the intra-chunk weights and score gradients (dT0); then Y and dU
  const int64_t cnt = rows * e;
  bwd_dy<T><<<(unsigned)((cnt + 255) / 256), 256, 0, stream>>>(dO, U, dY, cnt);
  const size_t sm_sc = sizeof(float) * ((size_t)kBR * s + kBK * ((size_t)s + 1) + kBR * kBC +
                                         kBK * (kBC + 1) + 2 * kBR * (kBK + 1));
  if (cudaFuncSetAttribute(bwd_quad_scores<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sm_sc) != cudaSuccess)
    return 1;
  bwd_quad_scores<T><<<B * G * nrb, kBT, sm_sc, stream>>>(Z, V, dY, gamma, beta, W, dS, dT, n, s,
                                                          e, C, G, causal, var.quad_a);
  const size_t sm_rows = sizeof(float) * ((size_t)kBR * s + kBR * (kBK + 1) + kBK * kBC);
  dim3 g3(B * G * nrb, (e + kBC - 1) / kBC);
  bwd_rows<T><<<g3, kBT, sm_rows, stream>>>(Z, V, dO, gamma, beta, W, P, dU, n, s, e, C, G,
                                            causal, var.lin_norm);
  const size_t sm_k = sizeof(float) * ((size_t)kBR * s + kBR * (kBK + 1));
  bwd_quad_keys<T><<<B * G * nrb, kBT, sm_k, stream>>>(Z, gamma, beta, dS, dT + rows * s, n, s, C,
                                                       G, causal);
  // the global term
  float *dT2 = dT + 2 * rows * s, *dT3 = dT + 3 * rows * s;
  if (glob) {
    dim3 g4(B * G, (e + kBC - 1) / kBC, (s + kBR - 1) / kBR);
    bwd_chunk_outer<T, float><<<g4, kBT, 0, stream>>>(Z, dY, gamma, beta, 2, 1, var.lin_norm, dP,
                                                       n, s, e, C, G);
    bwd_reverse_scan<<<lanes_blocks, 256, 0, stream>>>(dP, B, G, se, n, C, causal, var.lin_norm);
    dim3 g5(B * G * nrb, (s + kBR - 1) / kBR);
    bwd_lin_rows<T><<<g5, kBT, 0, stream>>>(V, dY, P, dP, dT2, dT3, n, s, e, C, G, causal,
                                            var.lin_norm);
  } else if (cudaMemsetAsync(dT2, 0, sizeof(float) * 2 * rows * s, stream) != cudaSuccess) {
    return 1;
  }
  const size_t sm_dv = sizeof(float) * ((size_t)kBK * s + kBR * (kBK + 1) + kBR * kBC);
  dim3 g6(B * G * nrb, (e + kBC - 1) / kBC);
  bwd_dv<T><<<g6, kBT, sm_dv, stream>>>(Z, gamma, beta, W, dY, dP, dV, n, s, e, C, G, causal,
                                        var.lin_norm);
  // the affine maps
  const int nblk = (int)((rows + kAffRows - 1) / kAffRows);
  bwd_affine<T><<<nblk, s, 0, stream>>>(Z, gamma, dT, dZ, part, rows, s);
  bwd_gamma_beta<<<(8 * s + 255) / 256, 256, 0, stream>>>(part, nblk, s, dgamma, dbeta);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace

int launch_backward(const void *Z, const void *V, const void *U, const float *gamma,
                    const float *beta, const void *dO, void *dZ, void *dV, void *dU,
                    float *dgamma, float *dbeta, int B, int n, int s, int e, int C, int causal,
                    int dtype_bf16, const Variant &var, void *workspace, cudaStream_t stream) {
  if (dtype_bf16)
    return launch_backward_impl<__nv_bfloat16>(Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma,
                                               dbeta, B, n, s, e, C, causal, var, workspace,
                                               stream);
  return launch_backward_impl<float>(Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma, dbeta, B, n,
                                     s, e, C, causal, var, workspace, stream);
}

}  // namespace fmca
