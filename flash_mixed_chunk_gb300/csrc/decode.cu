// decode.cu -- one autoregressive step of the causal mixed-chunk attention
// core in its recurrent form ("FLASH: Possibly the Most Interesting Efficient
// Transformer Design Recently", section "Mixed Chunk": the decoder's cumsum
// form of V-hat^lin_g and the masked intra-chunk term; "大模型训练之加速篇
// -attention优化", section 1.4: linear attention as a recurrence over a
// carried state).
//
// The token at position t (chunk g = t / C, index i = t % C in its chunk) gets
//   o_t = u_t * ( sum_{j <= i} quad_scale * relu(T0_t . T1_j)^2 v_j
//               + T2_t . P_g / d(t) )
// where j runs over the tokens of chunk g up to t, P_g is the sum of
// T3_h^T V_h over the completed chunks h < g, and d(t) is the global-term
// divisor (n, the g*C tokens P_g covers, or t+1).  This is row t of the causal
// forward pass over the whole sequence, computed from a carried state instead
// of the sequence:
//   P      fp32 [B][s][e]   sum of T3^T V over completed chunks
//   Zc     [B][C][s]        Z rows of the current chunk's tokens so far
//   Vc     [B][C][e]        their V rows
// Each step appends its token to the chunk cache; the last token of a chunk
// also folds the cached chunk into P (a second launch).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include <cstdint>

#include "launch.h"

namespace fmca {
namespace {

template <typename T>
__device__ __forceinline__ float dec_f(T v);
template <>
__device__ __forceinline__ float dec_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float dec_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T>
__device__ __forceinline__ T dec_t(float v);
template <>
__device__ __forceinline__ float dec_t<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 dec_t<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

constexpr int kDecThreads = 256;  // eight warps
constexpr int kDecWarps = kDecThreads / 32;

// grid (B, ceil(e / (32 K))); dynamic smem: q0[s] q2[s] w[C] part[8][32 K]
// floats.  The block's rows -- the chunk's cached keys j <= i (weights w_j,
// rows of V) and the state rows a < s (weights T2_t[a] / d, rows of P) -- are
// split over the eight warps; lane l owns columns l + 32 k (k < K); partial
// sums meet in shared memory.  Every block computes the i+1 key weights of its
// sequence, so K (the block's width) trades that repeated work against the
// number of blocks.
template <typename T, int K>
__global__ void __launch_bounds__(kDecThreads)
    decode_token(const T *__restrict__ z, const T *__restrict__ v, const T *__restrict__ u,
                 const float *__restrict__ gamma, const float *__restrict__ beta,
                 T *__restrict__ o, const T *__restrict__ P, T *__restrict__ Zc,
                 T *__restrict__ Vc, int s, int e, int C, int i, float quad_a, float lin_f,
                 float t2_w) {
  extern __shared__ float dsm[];
  float *q0 = dsm;
  float *q2 = q0 + s;
  float *w = q2 + s;
  float *part = w + C;  // [kDecWarps][32 K]
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c0 = blockIdx.y * 32 * K + lane;
  const T *zt = z + (int64_t)b * s;
  const T *vt = v + (int64_t)b * e;
  // quad_q row, and the lin_q row with the divisor's inverse folded in
  for (int a = tid; a < s; a += kDecThreads) {
    const float zz = dec_f(zt[a]);
    q0[a] = zz * gamma[a] + beta[a];
    q2[a] = (zz * gamma[2 * s + a] + beta[2 * s + a]) * t2_w * lin_f;
  }
  __syncthreads();
  // relu^2 weights of the chunk's keys j <= i: each warp takes eight keys at a
  // time, so that eight rows' loads are in flight together
  constexpr int KJ = 8;
  for (int j0 = warp * KJ; j0 <= i; j0 += kDecWarps * KJ) {
    float dot[KJ];
#pragma unroll
    for (int q = 0; q < KJ; ++q) dot[q] = 0.f;
    for (int a = lane; a < s; a += 32) {
      const float qa = q0[a], g1 = gamma[s + a], b1 = beta[s + a];
#pragma unroll
      for (int q = 0; q < KJ; ++q) {
        const int j = j0 + q;
        if (j <= i) {
          const T *zj = j < i ? Zc + ((int64_t)b * C + j) * s : zt;
          dot[q] = fmaf(qa, dec_f(zj[a]) * g1 + b1, dot[q]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < KJ; ++q) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot[q] += __shfl_xor_sync(0xffffffffu, dot[q], off);
    }
    if (lane < KJ && j0 + lane <= i) {
      float d = dot[0];
#pragma unroll
      for (int q = 1; q < KJ; ++q)
        if (lane == q) d = dot[q];
      const float r = fmaxf(d * quad_a, 0.f);
      w[j0 + lane] = r * r;
    }
  }
  __syncthreads();
  float acc[K];
#pragma unroll
  for (int k = 0; k < K; ++k) acc[k] = 0.f;
  const T *vcb = Vc + (int64_t)b * C * e;
  const T *pb = P + (int64_t)b * s * e;
  // intra-chunk keys: cached rows j < i, this token's row j = i
#pragma unroll 8
  for (int j = warp; j < i; j += kDecWarps) {
    const float wj = w[j];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int c = c0 + 32 * k;
      if (c < e) acc[k] = fmaf(wj, dec_f(vcb[(int64_t)j * e + c]), acc[k]);
    }
  }
  if (warp == i % kDecWarps) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int c = c0 + 32 * k;
      if (c < e) acc[k] = fmaf(w[i], dec_f(vt[c]), acc[k]);
    }
  }
  // global term: rows of the carried state
#pragma unroll 8
  for (int a = warp; a < s; a += kDecWarps) {
    const float qa = q2[a];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int c = c0 + 32 * k;
      if (c < e) acc[k] = fmaf(qa, dec_f(pb[(int64_t)a * e + c]), acc[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < K; ++k) part[warp * 32 * K + 32 * k + lane] = acc[k];
  __syncthreads();
  if (warp < K) {
    // warp k sums column group k over the eight warps' partials
    const int c = c0 + 32 * warp;
    if (c < e) {
      float out = 0.f;
#pragma unroll
      for (int r = 0; r < kDecWarps; ++r) out += part[r * 32 * K + 32 * warp + lane];
      o[(int64_t)b * e + c] = dec_t<T>(dec_f(u[(int64_t)b * e + c]) * out);
      // append this token to the chunk cache (slot i; this launch reads only
      // slots j < i)
      Vc[((int64_t)b * C + i) * e + c] = vt[c];
    }
  }
  if (blockIdx.y == 0)
    for (int a = tid; a < s; a += kDecThreads) Zc[((int64_t)b * C + i) * s + a] = zt[a];
}

// Eight consecutive elements, loaded raw (one 16-byte load for bf16, two for
// fp32) so that a batch of rows is in flight before any is used, then
// widened to floats.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 r;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
    r = __ldg(reinterpret_cast<const uint4 *>(p));
  }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = __ldg(reinterpret_cast<const float4 *>(p));
    b = __ldg(reinterpret_cast<const float4 *>(p + 4));
  }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
  }
};

// The same step with 16-byte loads, for s and e multiples of 8: grid (B,
// ceil(e / W)); a block is one sequence and W columns (W = 256, 128 or 64).
// W / 8 lanes cover a row, eight columns each, so a warp takes 256 / W rows
// at a time and the block's 8 * 256 / W row slots split the rows (cached
// keys, then state rows); each thread forms the relu^2 weight of its own
// keys (one key a thread for chunks of up to 256).  dynamic smem: q0[s]
// q2[s] g1[s] b1[s] w[C] part[2048] floats.
template <typename T, int W>
__global__ void __launch_bounds__(kDecThreads)
    decode_token_v8(const T *__restrict__ z, const T *__restrict__ v, const T *__restrict__ u,
                    const float *__restrict__ gamma, const float *__restrict__ beta,
                    T *__restrict__ o, const T *__restrict__ P, T *__restrict__ Zc,
                    T *__restrict__ Vc, int s, int e, int C, int i, float quad_a, float lin_f,
                    float t2_w) {
  extern __shared__ float dsm[];
  float *q0 = dsm;
  float *q2 = q0 + s;
  float *g1 = q2 + s;
  float *b1 = g1 + s;
  float *w = b1 + s;
  constexpr int kL = W / 8;                // lanes a row
  constexpr int kSlots = kDecWarps * (32 / kL);  // rows in flight a block
  float *part = w + C;  // [kSlots][W]
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = warp * (32 / kL) + lane / kL;
  const int c = blockIdx.y * W + 8 * (lane % kL);  // this lane's first column
  const T *zt = z + (int64_t)b * s;
  const T *vt = v + (int64_t)b * e;
  for (int a = tid; a < s; a += kDecThreads) {
    const float zz = dec_f(zt[a]);
    q0[a] = zz * gamma[a] + beta[a];
    q2[a] = (zz * gamma[2 * s + a] + beta[2 * s + a]) * t2_w * lin_f;
    g1[a] = gamma[s + a];
    b1[a] = beta[s + a];
  }
  __syncthreads();
  // relu^2 weights of the chunk's keys j <= i, a key a thread (its row's
  // 16-byte pieces eight at a time in flight)
  constexpr int kR = 8;
  for (int j = tid; j <= i; j += kDecThreads) {
    const T *zj = j < i ? Zc + ((int64_t)b * C + j) * s : zt;
    float dot = 0.f;
    for (int a0 = 0; a0 < s; a0 += 8 * kR) {
      Raw8<T> raw[kR];
#pragma unroll
      for (int q = 0; q < kR; ++q)
        if (a0 + 8 * q < s) raw[q].load(zj + a0 + 8 * q);
#pragma unroll
      for (int q = 0; q < kR; ++q)
        if (a0 + 8 * q < s) {
          float f[8];
          raw[q].get(f);
          const int a = a0 + 8 * q;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dot = fmaf(q0[a + k], fmaf(f[k], g1[a + k], b1[a + k]), dot);
        }
    }
    const float r = fmaxf(dot * quad_a, 0.f);
    w[j] = r * r;
  }
  __syncthreads();
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  if (c < e) {
    const T *vcb = Vc + (int64_t)b * C * e + c;
    const T *pb = P + (int64_t)b * s * e + c;
    // intra-chunk keys: cached rows j < i (eight of this warp's rows in
    // flight), this token's row j = i
    for (int j0 = slot; j0 < i; j0 += kR * kSlots) {
      Raw8<T> raw[kR];
#pragma unroll
      for (int q = 0; q < kR; ++q)
        if (j0 + q * kSlots < i) raw[q].load(vcb + (int64_t)(j0 + q * kSlots) * e);
#pragma unroll
      for (int q = 0; q < kR; ++q)
        if (j0 + q * kSlots < i) {
          float f[8];
          raw[q].get(f);
          const float wj = w[j0 + q * kSlots];
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[k] = fmaf(wj, f[k], acc[k]);
        }
    }
    if (slot == i % kSlots) {
      Raw8<T> raw;
      raw.load(vt + c);
      float f[8];
      raw.get(f);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = fmaf(w[i], f[k], acc[k]);
    }
    // global term: rows of the carried state
    for (int a0 = slot; a0 < s; a0 += kR * kSlots) {
      Raw8<T> raw[kR];
#pragma unroll
      for (int q = 0; q < kR; ++q)
        if (a0 + q * kSlots < s) raw[q].load(pb + (int64_t)(a0 + q * kSlots) * e);
#pragma unroll
      for (int q = 0; q < kR; ++q)
        if (a0 + q * kSlots < s) {
          float f[8];
          raw[q].get(f);
          const float qa = q2[a0 + q * kSlots];
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[k] = fmaf(qa, f[k], acc[k]);
        }
    }
  }
  float4 *pp = reinterpret_cast<float4 *>(part + slot * W + 8 * (lane % kL));
  pp[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  pp[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  // thread tid < W: column blockIdx.y * W + tid, summed over the row slots
  const int cc = blockIdx.y * W + tid;
  if (tid < W && cc < e) {
    float out = 0.f;
#pragma unroll
    for (int r = 0; r < kSlots; ++r) out += part[r * W + tid];
    o[(int64_t)b * e + cc] = dec_t<T>(dec_f(u[(int64_t)b * e + cc]) * out);
    // append this token to the chunk cache (slot i; this launch reads only
    // slots j < i)
    Vc[((int64_t)b * C + i) * e + cc] = vt[cc];
  }
  if (blockIdx.y == 0)
    for (int a = tid; a < s; a += kDecThreads) Zc[((int64_t)b * C + i) * s + a] = zt[a];
}

// P[b] += sum_{j < C} T3(Zc[b][j])^T Vc[b][j] : the finished chunk joins the
// carried state (and, for bf16 I/O, its bf16 copy Pb the token kernel reads).
// grid (B, ceil(s / 32), ceil(e / 128)); smem T3 tile [C][32].
constexpr int kFoldThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kFoldThreads)
    decode_fold(float *__restrict__ P, T *__restrict__ Pb, const T *__restrict__ Zc,
                const T *__restrict__ Vc,
                const float *__restrict__ gamma, const float *__restrict__ beta, int s, int e,
                int C) {
  extern __shared__ float t3[];  // [C][32]
  const int b = blockIdx.x, a0 = blockIdx.y * 32;
  const int c = blockIdx.z * kFoldThreads + threadIdx.x;
  for (int x = threadIdx.x; x < C * 32; x += kFoldThreads) {
    const int j = x / 32, a = x % 32;
    float val = 0.f;
    if (a0 + a < s)
      val = dec_f(Zc[((int64_t)b * C + j) * s + a0 + a]) * gamma[3 * s + a0 + a] +
            beta[3 * s + a0 + a];
    t3[x] = val;
  }
  __syncthreads();
  if (c >= e) return;
  float acc[32];
#pragma unroll
  for (int a = 0; a < 32; ++a) acc[a] = 0.f;
  for (int j = 0; j < C; ++j) {
    const float vv = dec_f(Vc[((int64_t)b * C + j) * e + c]);
#pragma unroll
    for (int a = 0; a < 32; ++a) acc[a] = fmaf(t3[j * 32 + a], vv, acc[a]);
  }
  float *pb = P + (int64_t)b * s * e + c;
#pragma unroll
  for (int a = 0; a < 32; ++a)
    if (a0 + a < s) {
      const float nv = pb[(int64_t)(a0 + a) * e] + acc[a];
      pb[(int64_t)(a0 + a) * e] = nv;
      if (std::is_same<T, __nv_bfloat16>::value)
        Pb[(int64_t)b * s * e + c + (int64_t)(a0 + a) * e] = dec_t<T>(nv);
    }
}

template <typename T>
int launch_decode_impl(const void *z, const void *v, const void *u, const float *gamma,
                       const float *beta, void *o, int B, int s, int e, int C, int t, int n_norm,
                       const Variant &var, void *state, cudaStream_t stream) {
  const DecodeStateLayout L = decode_state_layout(B, s, e, C, sizeof(T));
  char *st = static_cast<char *>(state);
  float *P = reinterpret_cast<float *>(st + L.P);
  // the rows the token kernel reads: P itself, or its bf16 copy
  T *Pr = std::is_same<T, __nv_bfloat16>::value ? reinterpret_cast<T *>(st + L.Pb)
                                                : reinterpret_cast<T *>(P);
  T *Zc = reinterpret_cast<T *>(st + L.Zc);
  T *Vc = reinterpret_cast<T *>(st + L.Vc);
  const int g = t / C, i = t % C;
  // the global term's divisor: n, the g*C tokens P_g covers, or t+1 (carried
  // by the lin_q row)
  float lin_f = 1.0f / (float)n_norm, t2_w = 1.0f;  // t2_w * lin_f scales the lin_q row
  if (var.lin_norm == kLinNormSummed) lin_f = g > 0 ? 1.0f / ((float)g * (float)C) : 0.0f;
  if (var.lin_norm == kLinNormPosition) {
    lin_f = 1.0f;
    t2_w = 1.0f / (float)(t + 1);
  }
  if (var.lin_norm == kLinNormNone) lin_f = 0.0f;
  // 16-byte rows for s and e multiples of 8: the widest block (256, 128 or
  // 64 columns) that still gives at least one block per SM, else 64 columns
  auto blocks = [&](int w) { return (int64_t)B * ((e + w - 1) / w); };
  const int W = blocks(256) >= 152 ? 256 : (blocks(128) >= 152 ? 128 : 64);
  if (s % 8 == 0 && e % 8 == 0) {
    dim3 g1(B, (e + W - 1) / W);
    const size_t smem1 = sizeof(float) * (4 * (size_t)s + (size_t)C + 2048);
    auto *kern = W == 256 ? decode_token_v8<T, 256>
                          : (W == 128 ? decode_token_v8<T, 128> : decode_token_v8<T, 64>);
    kern<<<g1, kDecThreads, smem1, stream>>>(
        static_cast<const T *>(z), static_cast<const T *>(v), static_cast<const T *>(u), gamma,
        beta, static_cast<T *>(o), Pr, Zc, Vc, s, e, C, i, var.quad_a, lin_f, t2_w);
  } else {
    // other widths, a column a lane: 32 columns while that leaves fewer than
    // about three blocks per SM, wider (fewer repeats of the key weights)
    // beyond
    const int64_t blocks32 = (int64_t)B * ((e + 31) / 32);
    const int K = blocks32 >= 12 * 152 ? 4 : (blocks32 >= 6 * 152 ? 2 : 1);
    dim3 g1(B, (e + 32 * K - 1) / (32 * K));
    const size_t smem1 = sizeof(float) * (2 * (size_t)s + (size_t)C + kDecWarps * 32 * K);
    auto *kern = K == 4 ? decode_token<T, 4> : (K == 2 ? decode_token<T, 2> : decode_token<T, 1>);
    kern<<<g1, kDecThreads, smem1, stream>>>(
        static_cast<const T *>(z), static_cast<const T *>(v), static_cast<const T *>(u), gamma,
        beta, static_cast<T *>(o), Pr, Zc, Vc, s, e, C, i, var.quad_a, lin_f, t2_w);
  }
  if (cudaGetLastError() != cudaSuccess) return 1;
  if (i == C - 1) {
    const size_t smem2 = sizeof(float) * (size_t)C * 32;
    if (smem2 > 48 * 1024 &&
        cudaFuncSetAttribute(decode_fold<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem2) != cudaSuccess)
      return 1;
    dim3 g2(B, (s + 31) / 32, (e + kFoldThreads - 1) / kFoldThreads);
    decode_fold<T><<<g2, kFoldThreads, smem2, stream>>>(P, Pr, Zc, Vc, gamma, beta, s, e, C);
    if (cudaGetLastError() != cudaSuccess) return 1;
  }
  return 0;
}

}  // namespace

int launch_decode_step(const void *z, const void *v, const void *u, const float *gamma,
                       const float *beta, void *o, int B, int s, int e, int C, int t, int n_norm,
                       int dtype_bf16, const Variant &var, void *state, cudaStream_t stream) {
  if (dtype_bf16)
    return launch_decode_impl<__nv_bfloat16>(z, v, u, gamma, beta, o, B, s, e, C, t, n_norm, var,
                                             state, stream);
  return launch_decode_impl<float>(z, v, u, gamma, beta, o, B, s, e, C, t, n_norm, var, state,
                                   stream);
}

}  // namespace fmca
