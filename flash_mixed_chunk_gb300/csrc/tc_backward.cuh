// tc_backward.cuh -- host side of the tensor-core backward pass: the
// grouped product launches of tc_bgemm and the order of the backward steps.
// Included at the end of tc.cu, so that its kernels share the translation
// unit's device status with the forward kernels.
#pragma once

#include <utility>

#include "tc_bgemm.cuh"
#include "tc_bwd.cuh"

namespace fmca {

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

// Launches `kernel` as a programmatic dependent of the work before it on
// `stream`: it may start launching (and run its prologue) while its
// predecessor drains.  Every kernel of the backward pass waits
// (griddepcontrol.wait) for its predecessor to complete before it reads, so
// each one's completion implies all earlier ones'.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
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
  static OncePerDevice attr;
  if (!attr.run([] {
        return cudaFuncSetAttribute(tc_bgemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)BGEMM_SMEM) == cudaSuccess;
      }))
    return 1;
  const int sms = num_sms();
  return launch_dependent(tc_bgemm, dim3(units < sms ? units : sms), dim3(BGEMM_THREADS),
                          BGEMM_SMEM, stream, P) == cudaSuccess
             ? 0
             : 1;
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
                       const Variant &var, void *workspace, cudaStream_t stream, bool saved) {
  const TcBackwardLayout L = tc_backward_layout(B, n, s, e, C, causal);
  const TcLayout FL = tc_layout(B, n, s, e, C, causal, true);
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
  // dU = dO * (quad + glob), and the forward workspace (with `saved`, the
  // chunk states and prefix are the ones the forward pass left there)
  if (launch_tc_forward_materialised(Z, V, dO, gamma, beta, dU, B, n, s, e, C, causal, var,
                                     ws + L.fwd, stream, !saved) != 0)
    return 1;
  const int64_t ne8 = (int64_t)rows * e / 8, ns8 = (int64_t)rows * s / 8;
  if (launch_dependent(tcb_gate_dy, dim3(blocks_for(ne8)), dim3(256), 0, stream,
                       static_cast<const uint4 *>(dO), static_cast<const uint4 *>(U),
                       reinterpret_cast<uint4 *>(dY), ne8) != cudaSuccess ||
      launch_dependent(tcb_affine_rows, dim3(blocks_for(ns8)), dim3(256), 0, stream,
                       static_cast<const uint4 *>(Z), reinterpret_cast<const float4 *>(gamma),
                       reinterpret_cast<const float4 *>(beta), reinterpret_cast<uint4 *>(T0),
                       reinterpret_cast<uint4 *>(T1), reinterpret_cast<uint4 *>(T3), ns8,
                       s) != cudaSuccess)
    return 1;
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
    if (launch_dependent(tcb_reverse_scan, dim3(blocks_for((int64_t)B * se8)), dim3(256), 0,
                         stream, reinterpret_cast<uint4 *>(dP), B, G, se8, n, C, causal,
                         var.lin_norm) != cudaSuccess)
      return 1;
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
  if (launch_dependent(tcb_affine_reduce, dim3(nblk), dim3(s / 4, kTcbAffLanes),
                       sizeof(float) * kTcbAffLanes * s, stream, u2(Z), gamma, u2(dT0), u2(dT1),
                       u2(dT2), u2(dT3), static_cast<uint2 *>(dZ), part, (int64_t)rows, n, s,
                       var.lin_norm, glob ? 1 : 0) != cudaSuccess ||
      launch_dependent(tcb_gamma_beta, dim3((8 * s + 31) / 32), dim3(32, 32), 0, stream, part,
                       nblk, s, dgamma, dbeta) != cudaSuccess)
    return 1;
  return 0;
}

}  // namespace fmca
