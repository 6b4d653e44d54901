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

// 2-D bf16 map over a row-major [rows][cols] matrix, 128-byte swizzle.
bool make_map_bf16(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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
  const void *p;
  uint64_t cols, rows;
};

// D_b = alpha (A_b B_b [+ A2_b B2_b]) on the tensor cores (see tc_bgemm.cuh);
// A and B are read K-major or MN-major, A2 and B2 (used when sh.K2 > 0) the
// same way.
template <bool A_MN, bool B_MN, int NT>
int bgemm(const BgOperand &A, const BgOperand &Bm, void *D, const BgShape &sh,
          cudaStream_t stream, const BgOperand *A2 = nullptr, const BgOperand *B2 = nullptr) {
  CUtensorMap mA, mB, mD, mA2, mB2;
  const BgOperand &a2 = A2 ? *A2 : A, &b2 = B2 ? *B2 : Bm;
  if (!make_map_bf16(&mA, A.p, A.cols, A.rows, 64, A_MN ? 64 : 128) ||
      !make_map_bf16(&mB, Bm.p, Bm.cols, Bm.rows, 64, B_MN ? 64 : NT) ||
      !make_map_bf16(&mA2, a2.p, a2.cols, a2.rows, 64, A_MN ? 64 : 128) ||
      !make_map_bf16(&mB2, b2.p, b2.cols, b2.rows, 64, B_MN ? 64 : NT) ||
      !make_map_bf16(&mD, D, (uint64_t)sh.N, (uint64_t)sh.batches * sh.M, 64, 128))
    return 2;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(tc_bgemm<A_MN, B_MN, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)BGEMM_SMEM) != cudaSuccess)
      return 1;
    attr = true;
  }
  const int units = sh.batches * (sh.M / 128) * (sh.N / NT);
  const int sms = num_sms();
  tc_bgemm<A_MN, B_MN, NT><<<units < sms ? units : sms, BGEMM_THREADS, BGEMM_SMEM, stream>>>(
      mA, mB, mD, mA2, mB2, sh);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

unsigned blocks_for(int64_t count) { return (unsigned)((count + 255) / 256); }

}  // namespace

// The backward pass on the tensor cores (bf16, shapes of the tensor-core
// forward path).  The forward kernels run once more with dO in place of U:
// their gated output is dU = dO * (quad + glob), and they leave the relu^2
// weights W, the lin_q rows T2 and the scaled prefix P~ in their workspace.
// Then, per chunk:
//   dY = dO * U,  dw = dY V^T,  dS = dw 2a sqrt(W),  dT0 = dS T1,
//   dT1 = dS^T T0,  dP~ = T2^T dY -> reverse scan -> dS_h,  dT2 = dY P~^T,
//   dT3 = V dS_h^T,  dV = W^T dY + T3 dS_h (one product of depth C + s),
// and finally dZ, dgamma, dbeta from dT0..dT3.
int launch_tc_backward(const void *Z, const void *V, const void *U, const float *gamma,
                       const float *beta, const void *dO, void *dZ, void *dV, void *dU,
                       float *dgamma, float *dbeta, int B, int n, int s, int e, int C, int causal,
                       const Variant &var, void *workspace, cudaStream_t stream) {
  const TcBackwardLayout L = tc_backward_layout(B, n, s, e, C, causal);
  const WorkspaceLayout FL = workspace_layout(B, n, s, e, C, causal);
  char *ws = static_cast<char *>(workspace);
  typedef __nv_bfloat16 bf16;
  auto at = [&](size_t off) { return reinterpret_cast<bf16 *>(ws + off); };
  bf16 *dY = at(L.dY), *T0 = at(L.T0), *T1 = at(L.T1), *T3 = at(L.T3);
  bf16 *dw = at(L.dw), *dSt = at(L.dSt), *Wt = at(L.Wt), *dP = at(L.dP);
  bf16 *dT0 = at(L.dT0), *dT1 = at(L.dT1), *dT2 = at(L.dT2), *dT3 = at(L.dT3);
  const bf16 *prefix = at(L.fwd + FL.prefix), *W = at(L.fwd + FL.scores);
  const bf16 *T2 = at(L.fwd + FL.lin_q);
  float *part = reinterpret_cast<float *>(ws + L.part);
  const int G = n / C, Gp = causal ? G : 1;
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
      static_cast<const uint4 *>(Z), gamma, beta, reinterpret_cast<uint4 *>(T0),
      reinterpret_cast<uint4 *>(T1), reinterpret_cast<uint4 *>(T3), ns8, s);
  if (cudaGetLastError() != cudaSuccess) return 1;
  const int BG = B * G;
  const BgOperand oY{dY, (uint64_t)e, rows}, oV{V, (uint64_t)e, rows};
  const BgOperand oT0{T0, (uint64_t)s, rows}, oT1{T1, (uint64_t)s, rows};
  const BgOperand oT2{T2, (uint64_t)s, rows}, oT3{T3, (uint64_t)s, rows};
  const BgOperand odS{dw, (uint64_t)C, rows}, odSt{dSt, (uint64_t)C, rows};
  const BgOperand oWt{Wt, (uint64_t)C, rows};
  const BgOperand oP{prefix, (uint64_t)e, (uint64_t)B * Gp * s};
  const BgOperand odP{dP, (uint64_t)e, (uint64_t)BG * s};
  int rc = 0;
  // dw = dY V^T per chunk (C x C, K = e)
  const BgShape s_dw{C, C, e, BG, C, 1, C, 1, 1.f};
  rc |= C % 256 == 0 ? bgemm<false, false, 256>(oY, oV, dw, s_dw, stream)
                     : bgemm<false, false, 128>(oY, oV, dw, s_dw, stream);
  tcb_score_grads<<<dim3(BG, C / 32, C / 32), dim3(32, 8), 0, stream>>>(dw, W, dSt, Wt, C,
                                                                        var.quad_a, causal);
  // dT0 = dS T1, dT1 = dS^T T0 (C x s, K = C)
  const BgShape s_t{C, s, C, BG, C, 1, C, 1, 1.f};
  rc |= bgemm<false, true, 128>(odS, oT1, dT0, s_t, stream);
  rc |= bgemm<false, true, 128>(odSt, oT0, dT1, s_t, stream);
  // the chunk states' sources dS_h = d(state_h); the global term's pair of dV
  const int h_rpb = causal ? s : G * s, h_div = causal ? 1 : G;
  if (glob) {
    // d(prefix) per chunk = T2^T dY (s x e, K = C), then the reverse scan
    const BgShape s_dp{s, e, C, BG, C, 1, C, 1, 1.f};
    rc |= bgemm<true, true, 256>(oT2, oY, dP, s_dp, stream);
    const int64_t se8 = (int64_t)s * e / 8;
    tcb_reverse_scan<<<blocks_for((int64_t)B * se8), 256, 0, stream>>>(
        reinterpret_cast<uint4 *>(dP), B, G, se8, n, C, causal, var.lin_norm);
    // dT2 = dY P~^T (C x s, K = e); P~ per chunk, or one per sequence
    const BgShape s_t2{C, s, e, BG, C, 1, s, causal ? 1 : G, 1.f};
    rc |= bgemm<false, false, 128>(oY, oP, dT2, s_t2, stream);
    // dT3 = V dS_h^T (C x s, K = e)
    const BgShape s_t3{C, s, e, BG, C, 1, h_rpb, h_div, 1.f};
    rc |= bgemm<false, false, 128>(oV, odP, dT3, s_t3, stream);
  }
  // dV = W^T dY (C x e, K = C) [+ T3 dS_h (K = s)]
  BgShape s_v{C, e, C, BG, C, 1, C, 1, 1.f};
  if (glob) {
    s_v.K2 = s;
    s_v.a2_rpb = C;
    s_v.b2_rpb = h_rpb;
    s_v.b2_div = h_div;
  }
  rc |= bgemm<false, true, 256>(oWt, oY, dV, s_v, stream, &oT3, &odP);
  if (rc) return 1;
  const int nblk = (int)((rows + kTcbAffRows - 1) / kTcbAffRows);
  tcb_affine_reduce<<<nblk, s, 0, stream>>>(static_cast<const bf16 *>(Z), gamma, dT0, dT1, dT2,
                                            dT3, static_cast<bf16 *>(dZ), part, (int64_t)rows, n,
                                            s, var.lin_norm, glob ? 1 : 0);
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
