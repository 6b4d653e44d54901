// tc.cu -- tensor-core path of the mixed-chunk attention forward core
// (sm_103a: tcgen05 MMA into TMEM, TMA-staged 128-byte-swizzled bf16 tiles,
// mbarrier pipelines) for bf16 I/O, s = 128, C in {128, 256}, e % 256 == 0.
//
// Per call: one memset of the two work counters and three kernels
// ("FLASH: Possibly the Most Interesting Efficient Transformer Design
// Recently", sections "Weak Attention" and "Mixed Chunk"):
//
//   tc_chunk_prep    state_g = T3_g^T V_g per chunk and 256-column slice of e
//                    (bf16), P = relu(T0 T1^T / C)^2 (masked) and T2 rows
//                    (bf16), as one persistent stream of work units
//   tc_state_scan    exclusive prefix over chunks (causal) or total
//                    (bidirectional) of the states, times 1/n, to bf16
//   tc_chunk_attn    O = U * (P V_g + T2 prefix_g) per (chunk, row tile,
//                    e tile), both products accumulated in TMEM
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "ptx.cuh"

#include "tc_common.cuh"
#include "tc_prep.cuh"
#include "tc_scan.cuh"
#include "tc_attn.cuh"
#include "tc_gemm.cuh"
#include "tc_bgemm.cuh"
#include "tc_bwd.cuh"

namespace fmca {
namespace {

// A kernel whose only wait can never complete: exercises the bounded-wait
// exit path (records a timeout, returns) without hanging the GPU.
__global__ void tc_timeout_selftest(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, limit_ns)) record_timeout(900);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [rows][cols] matrix, 128-byte swizzle by
// default (the box's rows must then be 128 bytes; 64 for the 64-byte swizzle).
bool make_map_bf16(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Streaming multiprocessors of the current device (one persistent CTA each).
int num_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 148;
  return sms;
}

}  // namespace

bool tc_supported(int B, int n, int s, int e, int C) {
  if (s != S_DIM) return false;
  if (C % ROW_TILE) return false;  // whole 128-row tiles (C = n: FLASH-Quad)
  if (e % E_TILE) return false;
  if (n % C) return false;
  (void)B;
  return true;
}

int tc_launch_count() { return 3; }

int launch_tc_forward(const void *Z, const void *V, const void *U, const float *gamma,
                      const float *beta, void *O, int B, int n, int s, int e, int C, int causal,
                      const Variant &var, void *workspace, cudaStream_t stream,
                      cudaEvent_t const *events) {
  const int G = n / C;
  const int R = C / ROW_TILE;
  const int64_t se = (int64_t)s * e;
  const int Gp = causal ? G : 1;
  const WorkspaceLayout L = workspace_layout(B, n, s, e, C, causal);
  char *ws = static_cast<char *>(workspace);
  __nv_bfloat16 *states = reinterpret_cast<__nv_bfloat16 *>(ws + L.states);
  __nv_bfloat16 *prefix = reinterpret_cast<__nv_bfloat16 *>(ws + L.prefix);
  void *pw = ws + L.scores;
  void *t2 = ws + L.lin_q;
  unsigned int *sched = reinterpret_cast<unsigned int *>(ws + L.sched);

  CUtensorMap mZ64, mZ128, mVs, mSt, mPw, mT2, mV, mS, mU, mO;
  const uint64_t rows = (uint64_t)B * n;
  if (!make_map_bf16(&mZ64, Z, s, rows, 64, 64) || !make_map_bf16(&mZ128, Z, s, rows, 64, 128) ||
      !make_map_bf16(&mVs, V, e, rows, 64, 64) ||
      !make_map_bf16(&mSt, states, e, (uint64_t)B * G * s, 64, 128) ||
      !make_map_bf16(&mPw, pw, C, rows, 64, 128) || !make_map_bf16(&mT2, t2, s, rows, 64, 128) ||
      !make_map_bf16(&mV, V, e, rows, 64, 64) ||
      !make_map_bf16(&mS, prefix, e, (uint64_t)B * Gp * s, 64, 64) ||
      !make_map_bf16(&mU, U, e, rows, 64, 128) || !make_map_bf16(&mO, O, e, rows, 64, 128))
    return 2;

  static bool attrs = false;
  if (!attrs) {
    if (cudaFuncSetAttribute(tc_chunk_prep<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)PREP_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(tc_chunk_prep<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)PREP_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(tc_chunk_attn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)AT_SMEM) != cudaSuccess)
      return 1;
    attrs = true;
  }
  if (!record_event(events, 0, stream)) return 1;
  // sched[0]: work counter of tc_chunk_prep; sched[1]: of tc_chunk_attn
  if (cudaMemsetAsync(sched, 0, 2 * sizeof(unsigned int), stream) != cudaSuccess) return 1;
  // without a global term (FMCA_LIN_NORM_NONE) there are no chunk states, the
  // scan has nothing to do and the attention units have no lin_q items
  const bool no_global = var.lin_norm == kLinNormNone;
  const int n_state = no_global ? 0 : B * G * (e / E_TILE);
  const int n_score = B * G * (causal ? R * (R + 1) : R * (C / KEY_STAGE));
  const int n_prep = n_state + n_score;
  auto *prep = var.lin_norm == kLinNormPosition ? tc_chunk_prep<true> : tc_chunk_prep<false>;
  prep<<<n_prep < num_sms() ? n_prep : num_sms(), PREP_THREADS, PREP_SMEM, stream>>>(
      mZ64, mZ128, mVs, mSt, mPw, gamma, beta, reinterpret_cast<__nv_bfloat16 *>(t2), sched, n, e,
      C, G, causal, n_state, n_score, var.quad_a);
  if (cudaGetLastError() != cudaSuccess || !record_event(events, 1, stream)) return 1;
  // The scan and the attention kernel are launched as programmatic dependents
  // of the kernel before them: each may start launching (and run its
  // prologue) while its predecessor drains, and waits (griddepcontrol.wait)
  // for it to complete before reading what it wrote.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  const int64_t lanes = (int64_t)B * se / 8;
  cfg.gridDim = dim3(no_global ? 1u : (unsigned)((lanes + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  auto *scan = var.lin_norm == kLinNormSummed     ? tc_state_scan<kLinNormSummed>
               : var.lin_norm == kLinNormPosition ? tc_state_scan<kLinNormPosition>
               : no_global                        ? tc_state_scan<kLinNormNone>
                                                  : tc_state_scan<kLinNormN>;
  if (cudaLaunchKernelEx(&cfg, scan, (const __nv_bfloat16 *)states, prefix, B, G, se,
                         1.0f / (float)n, causal, C) != cudaSuccess ||
      !record_event(events, 2, stream))
    return 1;
  const int n_units = B * G * R * (e / E_TILE);
  cfg.gridDim = dim3(n_units < num_sms() ? n_units : num_sms());
  cfg.blockDim = dim3(AT_THREADS);
  cfg.dynamicSmemBytes = AT_SMEM;
  if (cudaLaunchKernelEx(&cfg, tc_chunk_attn, mPw, mT2, mV,
                         mS, mU, mO, sched + 1, n, e, C, G,
                         causal, n_units, no_global ? 0 : S_DIM / KEY_STAGE) != cudaSuccess ||
      !record_event(events, 3, stream))
    return 1;
  return 0;
}

int launch_gemm(const void *A, const void *B, int M, int N, int K, void *D0, void *D1,
                void *D2, int n0, int n1, int silu, cudaStream_t stream) {
  CUtensorMap mA, mB, m0, m1, m2;
  if (!make_map_bf16(&mA, A, K, M, 64, 128) || !make_map_bf16(&mB, B, K, N, 64, GM_TILE_N) ||
      !make_map_bf16(&m0, D0, n0, M, 64, 128))
    return 2;
  m1 = m0;
  m2 = m0;
  if (n1 > n0 && !make_map_bf16(&m1, D1, n1 - n0, M, 64, 128)) return 2;
  if (N > n1 && !make_map_bf16(&m2, D2, N - n1, M, 64, 128)) return 2;
  static bool attrs = false;
  if (!attrs) {
    if (cudaFuncSetAttribute(tc_gemm<GEMM_ACT_NONE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)GEMM_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm<GEMM_ACT_SILU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)GEMM_SMEM) != cudaSuccess)
      return 1;
    attrs = true;
  }
  const int units = ((M + 127) / 128) * ((N + GM_TILE_N - 1) / GM_TILE_N);
  const int sms = num_sms();
  auto *kern = silu ? tc_gemm<GEMM_ACT_SILU> : tc_gemm<GEMM_ACT_NONE>;
  kern<<<units < sms ? units : sms, GEMM_THREADS, GEMM_SMEM, stream>>>(mA, mB, m0, m1, m2, M, N,
                                                                      K, n0, n1);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

namespace {

// A row-major bf16 operand [rows][cols] of tc_bgemm.
struct BgOperand {
  const void *p = nullptr;
  uint64_t cols = 0, rows = 0;
};

// One product of a tc_bgemm launch (fields as in BgProblem).
struct BgSpec {
  BgOperand A, B, A2, B2;  // A2/B2 used when K2 > 0
  void *D = nullptr;
  const void *w = nullptr;
  float alpha = 1.f;
  int M = 0, N = 0, K = 0, K2 = 0, batches = 0, nt = 128;
  int a_rpb = 0, a_div = 1, b_rpb = 0, b_div = 1, a2_rpb = 0, a2_div = 1, b2_rpb = 0, b2_div = 1;
  bool a_mn = false, b_mn = false, a2_mn = false, b2_mn = false;
  int krange = BG_K_FULL;
  bool skip_upper = false, causal = false;
  int epi = BG_EPI_STORE;
};

bool fill_problem(BgProblem &p, const BgSpec &s) {
  const BgOperand &a2 = s.K2 > 0 ? s.A2 : s.A, &b2 = s.K2 > 0 ? s.B2 : s.B;
  const bool a2_mn = s.K2 > 0 ? s.a2_mn : s.a_mn, b2_mn = s.K2 > 0 ? s.b2_mn : s.b_mn;
  if (!make_map_bf16(&p.A, s.A.p, s.A.cols, s.A.rows, 64, s.a_mn ? 64 : 128) ||
      !make_map_bf16(&p.B, s.B.p, s.B.cols, s.B.rows, 64, s.b_mn ? 64 : s.nt) ||
      !make_map_bf16(&p.A2, a2.p, a2.cols, a2.rows, 64, a2_mn ? 64 : 128) ||
      !make_map_bf16(&p.B2, b2.p, b2.cols, b2.rows, 64, b2_mn ? 64 : s.nt) ||
      !make_map_bf16(&p.D, s.D, (uint64_t)s.N, (uint64_t)s.batches * s.M, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B))
    return false;
  p.w = static_cast<const __nv_bfloat16 *>(s.w);
  p.alpha = s.alpha;
  p.M = s.M, p.N = s.N, p.K = s.K, p.K2 = s.K2, p.batches = s.batches, p.nt = s.nt;
  p.a_rpb = s.a_rpb, p.a_div = s.a_div, p.b_rpb = s.b_rpb, p.b_div = s.b_div;
  p.a2_rpb = s.a2_rpb, p.a2_div = s.a2_div, p.b2_rpb = s.b2_rpb, p.b2_div = s.b2_div;
  p.a_mn = s.a_mn, p.b_mn = s.b_mn, p.a2_mn = a2_mn, p.b2_mn = b2_mn;
  p.krange = s.krange, p.skip_upper = s.skip_upper, p.epi = s.epi, p.causal = s.causal;
  p.units = s.batches * (s.M / 128) * (s.N / s.nt);
  return true;
}

// One tc_bgemm launch over n (1..3) independent products.
int launch_bgemm(const BgSpec *specs, int n, cudaStream_t stream) {
  BgParams P;
  P.n_problems = n;
  int units = 0;
  for (int i = 0; i < n; ++i) {
    if (!fill_problem(P.p[i], specs[i])) return 2;
    units += P.p[i].units;
  }
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(tc_bgemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)BGEMM_SMEM) != cudaSuccess)
      return 1;
    attr = true;
  }
  const int sms = num_sms();
  tc_bgemm<<<units < sms ? units : sms, BGEMM_THREADS, BGEMM_SMEM, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

unsigned blocks_for(int64_t count) { return (unsigned)((count + 255) / 256); }

}  // namespace

// The backward pass on the tensor cores (bf16, shapes of the tensor-core
// forward path).  The forward kernels run once more with dO in place of U:
// their gated output is dU = dO * (quad + glob), and they leave the relu^2
// weights W (0 past the causal diagonal within each 128-row tile), the lin_q
// rows T2 and the scaled prefix P~ in their workspace.  Then, per chunk, in
// three grouped product launches around the reverse scan:
//   dY = dO * U
//   [dS = (dY V^T) 2a sqrt(W),  dT2 = dY P~^T]
//   [d(prefix) = T2^T dY,  dT0 = dS T1,  dT1 = dS^T T0]
//   reverse scan of d(prefix) -> dS_h
//   [dT3 = V dS_h^T,  dV = W^T dY + T3 dS_h]
// and finally dZ, dgamma, dbeta from dT0..dT3.  Causal chunks compute only
// the tiles and k ranges on or below the diagonal.
int launch_tc_backward(const void *Z, const void *V, const void *U, const float *gamma,
                       const float *beta, const void *dO, void *dZ, void *dV, void *dU,
                       float *dgamma, float *dbeta, int B, int n, int s, int e, int C, int causal,
                       const Variant &var, void *workspace, cudaStream_t stream) {
  const TcBackwardLayout L = tc_backward_layout(B, n, s, e, C, causal);
  const WorkspaceLayout FL = workspace_layout(B, n, s, e, C, causal);
  char *ws = static_cast<char *>(workspace);
  typedef __nv_bfloat16 bf16;
  auto at = [&](size_t off) { return reinterpret_cast<bf16 *>(ws + off); };
  bf16 *dY = at(L.dY), *T0 = at(L.T0), *T1 = at(L.T1), *T3 = at(L.T3), *dS = at(L.dS);
  bf16 *dP = at(L.dP);
  bf16 *dT0 = at(L.dT0), *dT1 = at(L.dT1), *dT2 = at(L.dT2), *dT3 = at(L.dT3);
  const bf16 *prefix = at(L.fwd + FL.prefix), *W = at(L.fwd + FL.scores);
  const bf16 *T2 = at(L.fwd + FL.lin_q);
  float *part = reinterpret_cast<float *>(ws + L.part);
  const int G = n / C, Gp = causal ? G : 1, BG = B * G;
  const uint64_t rows = (uint64_t)B * n;
  const bool glob = var.lin_norm != kLinNormNone;
  // dU = dO * (quad + glob), and the forward workspace
  if (launch_tc_forward(Z, V, dO, gamma, beta, dU, B, n, s, e, C, causal, var, ws + L.fwd,
                        stream) != 0)
    return 1;
  const int64_t ne8 = (int64_t)rows * e / 8, ns8 = (int64_t)rows * s / 8;
  tcb_gate_dy<<<blocks_for(ne8), 256, 0, stream>>>(static_cast<const uint4 *>(dO),
                                                   static_cast<const uint4 *>(U),
                                                   reinterpret_cast<uint4 *>(dY), ne8);
  tcb_affine_rows<<<blocks_for(ns8), 256, 0, stream>>>(
      static_cast<const uint4 *>(Z), reinterpret_cast<const float4 *>(gamma),
      reinterpret_cast<const float4 *>(beta), reinterpret_cast<uint4 *>(T0),
      reinterpret_cast<uint4 *>(T1), reinterpret_cast<uint4 *>(T3), ns8, s);
  if (cudaGetLastError() != cudaSuccess) return 1;
  const BgOperand oY{dY, (uint64_t)e, rows}, oV{V, (uint64_t)e, rows};
  const BgOperand oT0{T0, (uint64_t)s, rows}, oT1{T1, (uint64_t)s, rows};
  const BgOperand oT2{T2, (uint64_t)s, rows}, oT3{T3, (uint64_t)s, rows};
  const BgOperand odS{dS, (uint64_t)C, rows}, oW{W, (uint64_t)C, rows};
  const BgOperand oP{prefix, (uint64_t)e, (uint64_t)B * Gp * s};
  const BgOperand odP{dP, (uint64_t)e, (uint64_t)BG * s};
  // chunk h's state gradient dS_h: its own slot (causal) or the sequence's
  const int h_rpb = causal ? s : G * s, h_div = causal ? 1 : G;
  BgSpec sp[3];
  int np = 0, rc = 0;
  {  // dS = (dY V^T) 2a sqrt(W) (C x C, K = e); dT2 = dY P~^T (C x s, K = e)
    BgSpec &a = sp[np++];
    a.A = oY, a.B = oV, a.D = dS, a.M = C, a.N = C, a.K = e, a.batches = BG;
    a.nt = C % 256 == 0 ? 256 : 128, a.a_rpb = C, a.b_rpb = C;
    a.epi = BG_EPI_SCORE, a.w = W, a.alpha = var.quad_a, a.causal = causal;
    a.skip_upper = causal;
    if (glob) {
      BgSpec &b = sp[np++];
      b.A = oY, b.B = oP, b.D = dT2, b.M = C, b.N = s, b.K = e, b.batches = BG, b.nt = 128;
      b.a_rpb = C, b.b_rpb = s, b.b_div = causal ? 1 : G;
    }
    rc |= launch_bgemm(sp, np, stream);
  }
  np = 0;
  {  // d(prefix) = T2^T dY (s x e, K = C); dT0 = dS T1, dT1 = dS^T T0 (C x s, K = C)
    if (glob) {
      BgSpec &c = sp[np++];
      c = BgSpec();
      c.A = oT2, c.a_mn = true, c.B = oY, c.b_mn = true, c.D = dP, c.M = s, c.N = e, c.K = C;
      c.batches = BG, c.nt = 256, c.a_rpb = C, c.b_rpb = C;
    }
    BgSpec &a = sp[np++];
    a = BgSpec();
    a.A = odS, a.B = oT1, a.b_mn = true, a.D = dT0, a.M = C, a.N = s, a.K = C, a.batches = BG;
    a.a_rpb = C, a.b_rpb = C, a.krange = causal ? BG_K_TO_M : BG_K_FULL;
    BgSpec &b = sp[np++];
    b = BgSpec();
    b.A = odS, b.a_mn = true, b.B = oT0, b.b_mn = true, b.D = dT1, b.M = C, b.N = s, b.K = C;
    b.batches = BG, b.a_rpb = C, b.b_rpb = C, b.krange = causal ? BG_K_FROM_M : BG_K_FULL;
    rc |= launch_bgemm(sp, np, stream);
  }
  if (glob) {
    const int64_t se8 = (int64_t)s * e / 8;
    tcb_reverse_scan<<<blocks_for((int64_t)B * se8), 256, 0, stream>>>(
        reinterpret_cast<uint4 *>(dP), B, G, se8, n, C, causal, var.lin_norm);
  }
  np = 0;
  {  // dT3 = V dS_h^T (C x s, K = e); dV = W^T dY [+ T3 dS_h] (C x e, K = C [+ s])
    if (glob) {
      BgSpec &c = sp[np++];
      c = BgSpec();
      c.A = oV, c.B = odP, c.D = dT3, c.M = C, c.N = s, c.K = e, c.batches = BG, c.nt = 128;
      c.a_rpb = C, c.b_rpb = h_rpb, c.b_div = h_div;
    }
    BgSpec &a = sp[np++];
    a = BgSpec();
    a.A = oW, a.a_mn = true, a.B = oY, a.b_mn = true, a.D = dV, a.M = C, a.N = e, a.K = C;
    a.batches = BG, a.nt = 256, a.a_rpb = C, a.b_rpb = C;
    a.krange = causal ? BG_K_FROM_M : BG_K_FULL;
    if (glob) {
      a.A2 = oT3, a.B2 = odP, a.b2_mn = true, a.K2 = s;
      a.a2_rpb = C, a.b2_rpb = h_rpb, a.b2_div = h_div;
    }
    rc |= launch_bgemm(sp, np, stream);
  }
  if (rc) return 1;
  const int nblk = (int)((rows + kTcbAffRows - 1) / kTcbAffRows);
  auto u2 = [](const void *p) { return static_cast<const uint2 *>(p); };
  tcb_affine_reduce<<<nblk, dim3(s / 4, kTcbAffLanes), sizeof(float) * kTcbAffLanes * s,
                      stream>>>(u2(Z), gamma, u2(dT0), u2(dT1), u2(dT2), u2(dT3),
                                static_cast<uint2 *>(dZ), part, (int64_t)rows, n, s,
                                var.lin_norm, glob ? 1 : 0);
  tcb_gamma_beta<<<(8 * s + 31) / 32, dim3(32, 32), 0, stream>>>(part, nblk, s, dgamma, dbeta);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int read_and_clear_device_status(cudaStream_t stream, int32_t *where) {
  int st = 0, wh = 0;
  const int zero = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(&st, g_fmca_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(&wh, g_fmca_where, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_fmca_status, &zero, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_fmca_where, &zero, sizeof(int)) != cudaSuccess) return -1;
  if (where) *where = wh;
  return st;
}

int launch_timeout_selftest(int limit_us, cudaStream_t stream) {
  tc_timeout_selftest<<<1, 32, 0, stream>>>((uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace fmca
