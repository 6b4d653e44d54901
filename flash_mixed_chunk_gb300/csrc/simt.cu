// simt.cu -- CUDA-core (fp32 FMA) kernels of the mixed-chunk attention forward
// core.  They cover every supported shape and both element types; they carry
// the fp32 mode (where tensor-core tf32/bf16 products would not meet the fp32
// tolerance) and any bf16 shape the tensor-core path does not take.
//
// Three launches per call, following "FLASH: Possibly the Most Interesting
// Efficient Transformer Design Recently", section "Mixed Chunk":
//   simt_chunk_state  state_g = T3_g^T V_g            (per chunk, s x e, fp32)
//   simt_chunk_scan   P_g = sum_{h<g} state_h / n      (causal, exclusive)
//                     P   = sum_h state_h / n          (bidirectional)
//   simt_chunk_output O_g = U_g * (relu(T0_g T1_g^T / C)^2 V_g  [masked]
//                                  + T2_g P_g)
// (scale and divisor as the caller's variant chooses: 1/C and n by default).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"

namespace fmca {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

constexpr int kRows = 32;   // rows (tokens or state rows) per block
constexpr int kCols = 64;   // e columns per block
constexpr int kKeys = 32;   // keys per inner block
constexpr int kThreads = 256;
constexpr int kPerThread = kRows * kCols / kThreads;  // 8

// state_g[a][c] = sum_{j in chunk g} (Z[j][a] * gamma3[a] + beta3[a]) * V[j][c]
// grid: (B*G, ceil(e/64), ceil(s/32)); block 256.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    simt_chunk_state(const T *__restrict__ Z, const T *__restrict__ V,
                     const float *__restrict__ gamma, const float *__restrict__ beta,
                     float *__restrict__ S, int n, int s, int e, int C, int G) {
  __shared__ float t3[kKeys][kRows + 1];
  __shared__ float vb[kKeys][kCols];
  const int bg = blockIdx.x;
  const int b = bg / G, g = bg % G;
  const int c0 = blockIdx.y * kCols, a0 = blockIdx.z * kRows;
  const int tid = threadIdx.x;
  const int col = tid % kCols;
  const int rbase = tid / kCols;  // rows rbase + 4*i
  const int64_t row0 = (int64_t)b * n + (int64_t)g * C;
  float acc[kPerThread];
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < C; j0 += kKeys) {
    for (int x = tid; x < kKeys * kRows; x += kThreads) {
      int j = x / kRows, a = x % kRows;
      float v = 0.f;
      if (j0 + j < C && a0 + a < s)
        v = to_f(Z[(row0 + j0 + j) * s + a0 + a]) * gamma[3 * s + a0 + a] + beta[3 * s + a0 + a];
      t3[j][a] = v;
    }
    for (int x = tid; x < kKeys * kCols; x += kThreads) {
      int j = x / kCols, c = x % kCols;
      float v = 0.f;
      if (j0 + j < C && c0 + c < e) v = to_f(V[(row0 + j0 + j) * e + c0 + c]);
      vb[j][c] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kKeys; ++j) {
      float vv = vb[j][col];
#pragma unroll
      for (int i = 0; i < kPerThread; ++i) acc[i] = fmaf(t3[j][rbase + 4 * i], vv, acc[i]);
    }
    __syncthreads();
  }
  if (c0 + col < e) {
    float *dst = S + (int64_t)bg * s * e;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      int a = a0 + rbase + 4 * i;
      if (a < s) dst[(int64_t)a * e + c0 + col] = acc[i];
    }
  }
}

// causal: P[b][g][x] = sum_{h<g} S[b][h][x] * f(g) ; else P[b][x] = sum_h S * f
// with f the inverse of the global-term divisor: 1/n by default; 1/(g*C) for
// causal chunk g with the tokens-summed divisor; 1 with the per-position
// divisor (the T2 rows carry 1/(t+1) instead).
__global__ void simt_chunk_scan(const float *__restrict__ S, float *__restrict__ P, int B, int G,
                                int64_t se, float inv_n, int causal, int C, int lin_norm) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * se) return;
  const int64_t b = t / se, x = t % se;
  const float *src = S + b * G * se + x;
  const float keep = lin_norm == kLinNormPosition ? 1.0f : (lin_norm == kLinNormNone ? 0.0f : inv_n);
  float run = 0.f;
  if (causal) {
    float *dst = P + b * G * se + x;
    for (int g = 0; g < G; ++g) {
      const float f = lin_norm != kLinNormSummed ? keep
                      : (g > 0 ? 1.0f / ((float)g * (float)C) : 0.0f);
      dst[(int64_t)g * se] = run * f;
      run += src[(int64_t)g * se];
    }
  } else {
    for (int g = 0; g < G; ++g) run += src[(int64_t)g * se];
    P[b * se + x] = run * keep;
  }
}

// O rows [r0, r0+32) of chunk g, columns [c0, c0+64).
// grid: (B*G*ceil(C/32), ceil(e/64)); block 256; dynamic smem (3*32*s + ...)*4.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    simt_chunk_output(const T *__restrict__ Z, const T *__restrict__ V, const T *__restrict__ U,
                      const float *__restrict__ gamma, const float *__restrict__ beta,
                      const float *__restrict__ P, T *__restrict__ O, int n, int s, int e, int C,
                      int G, int causal, float quad_a, int lin_norm) {
  extern __shared__ float sm[];
  float *t0 = sm;                      // [32][s]  quad_q rows
  float *t2 = t0 + kRows * s;          // [32][s]  lin_q rows
  float *t1 = t2 + kRows * s;          // [32][s+1] quad_k keys (odd stride: the
                                       // 32 lanes of a warp read 32 banks)
  float *w = t1 + kKeys * (s + 1);     // [32][33] relu^2 weights
  float *vb = w + kRows * (kKeys + 1); // [32][64] V keys / P rows
  const int nrb = (C + kRows - 1) / kRows;
  const int bg = blockIdx.x / nrb, rb = blockIdx.x % nrb;
  const int b = bg / G, g = bg % G;
  const int c0 = blockIdx.y * kCols;
  const int tid = threadIdx.x, col = tid % kCols, rbase = tid / kCols;
  const int64_t chunk0 = (int64_t)b * n + (int64_t)g * C;
  const int r0 = rb * kRows;

  for (int x = tid; x < kRows * s; x += kThreads) {
    int r = x / s, a = x % s;
    float z = (r0 + r < C) ? to_f(Z[(chunk0 + r0 + r) * s + a]) : 0.f;
    t0[x] = z * gamma[a] + beta[a];
    // per-position divisor: the lin_q row of token t carries 1/(t+1)
    const float w = lin_norm == kLinNormPosition ? 1.0f / (float)(g * C + r0 + r + 1) : 1.0f;
    t2[x] = (z * gamma[2 * s + a] + beta[2 * s + a]) * w;
  }
  float acc[kPerThread];
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) acc[i] = 0.f;

  // intra-chunk relu^2 attention over key blocks (causal: blocks up to rb)
  const int kb_end = causal ? rb : nrb - 1;
  for (int kb = 0; kb <= kb_end; ++kb) {
    const int k0 = kb * kKeys;
    __syncthreads();
    for (int x = tid; x < kKeys * s; x += kThreads) {
      int j = x / s, a = x % s;
      float z = (k0 + j < C) ? to_f(Z[(chunk0 + k0 + j) * s + a]) : 0.f;
      t1[j * (s + 1) + a] = z * gamma[s + a] + beta[s + a];
    }
    for (int x = tid; x < kKeys * kCols; x += kThreads) {
      int j = x / kCols, c = x % kCols;
      float v = 0.f;
      if (k0 + j < C && c0 + c < e) v = to_f(V[(chunk0 + k0 + j) * e + c0 + c]);
      vb[x] = v;
    }
    __syncthreads();
    for (int x = tid; x < kRows * kKeys; x += kThreads) {
      int r = x / kKeys, j = x % kKeys;
      float dotv = 0.f;
      const float *q = t0 + r * s, *k = t1 + j * (s + 1);
      for (int a = 0; a < s; ++a) dotv = fmaf(q[a], k[a], dotv);
      float rl = fmaxf(dotv * quad_a, 0.f);
      float wt = rl * rl;
      bool valid = (r0 + r < C) && (k0 + j < C) && (!causal || k0 + j <= r0 + r);
      w[r * (kKeys + 1) + j] = valid ? wt : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < kKeys; ++j) {
      float vv = vb[j * kCols + col];
#pragma unroll
      for (int i = 0; i < kPerThread; ++i)
        acc[i] = fmaf(w[(rbase + 4 * i) * (kKeys + 1) + j], vv, acc[i]);
    }
  }
  // global linear term: T2 rows . P_g  (P_g already scaled by the divisor)
  const float *pg = P + (int64_t)(causal ? bg : b) * s * e;
  for (int a0 = 0; a0 < s; a0 += kKeys) {
    __syncthreads();
    for (int x = tid; x < kKeys * kCols; x += kThreads) {
      int a = x / kCols, c = x % kCols;
      float v = 0.f;
      if (a0 + a < s && c0 + c < e) v = pg[(int64_t)(a0 + a) * e + c0 + c];
      vb[x] = v;
    }
    __syncthreads();
    const int amax = min(kKeys, s - a0);
    for (int a = 0; a < amax; ++a) {
      float pv = vb[a * kCols + col];
#pragma unroll
      for (int i = 0; i < kPerThread; ++i) acc[i] = fmaf(t2[(rbase + 4 * i) * s + a0 + a], pv, acc[i]);
    }
  }
  if (c0 + col < e) {
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      int r = r0 + rbase + 4 * i;
      if (r < C) {
        int64_t off = (chunk0 + r) * e + c0 + col;
        O[off] = from_f<T>(to_f(U[off]) * acc[i]);
      }
    }
  }
}

size_t output_smem_bytes(int s) {
  return sizeof(float) * ((size_t)kRows * s * 2 + (size_t)kKeys * (s + 1) +
                          kRows * (kKeys + 1) + kKeys * kCols);
}

template <typename T>
int launch_simt_impl(const void *Z, const void *V, const void *U, const float *gamma,
                     const float *beta, void *O, int B, int n, int s, int e, int C, int causal,
                     const Variant &var, float *states, float *prefix, cudaStream_t stream,
                     cudaEvent_t const *events) {
  const int G = n / C;
  const T *z = static_cast<const T *>(Z);
  const T *v = static_cast<const T *>(V);
  const T *u = static_cast<const T *>(U);
  T *o = static_cast<T *>(O);
  dim3 g1(B * G, (e + kCols - 1) / kCols, (s + kRows - 1) / kRows);
  if (!record_event(events, 0, stream)) return 1;
  simt_chunk_state<T><<<g1, kThreads, 0, stream>>>(z, v, gamma, beta, states, n, s, e, C, G);
  if (cudaGetLastError() != cudaSuccess || !record_event(events, 1, stream)) return 1;
  const int64_t se = (int64_t)s * e;
  const int64_t lanes = (int64_t)B * se;
  simt_chunk_scan<<<(unsigned)((lanes + 255) / 256), 256, 0, stream>>>(states, prefix, B, G, se,
                                                                         1.0f / (float)n, causal, C,
                                                                         var.lin_norm);
  if (cudaGetLastError() != cudaSuccess || !record_event(events, 2, stream)) return 1;
  const size_t smem = output_smem_bytes(s);
  if (cudaFuncSetAttribute(simt_chunk_output<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return 1;
  dim3 g3(B * G * ((C + kRows - 1) / kRows), (e + kCols - 1) / kCols);
  simt_chunk_output<T><<<g3, kThreads, smem, stream>>>(z, v, u, gamma, beta, prefix, o, n, s, e,
                                                       C, G, causal, var.quad_a, var.lin_norm);
  if (cudaGetLastError() != cudaSuccess || !record_event(events, 3, stream)) return 1;
  return 0;
}

}  // namespace

int launch_simt_forward(const void *Z, const void *V, const void *U, const float *gamma,
                        const float *beta, void *O, int B, int n, int s, int e, int C,
                        int causal, int dtype_bf16, const Variant &var, void *workspace,
                        cudaStream_t stream, cudaEvent_t const *events) {
  const SimtLayout L = simt_layout(B, n, s, e, C, causal);
  float *states = reinterpret_cast<float *>(static_cast<char *>(workspace) + L.states);
  float *prefix = reinterpret_cast<float *>(static_cast<char *>(workspace) + L.prefix);
  if (dtype_bf16)
    return launch_simt_impl<__nv_bfloat16>(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, var,
                                           states, prefix, stream, events);
  return launch_simt_impl<float>(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, var, states,
                                 prefix, stream, events);
}

}  // namespace fmca
