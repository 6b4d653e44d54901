// launch.h -- host-side declarations shared by the C-ABI layer and the kernel
// translation units (launchers, workspace layout, device status).
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include <cstddef>
#include <cstdint>

namespace fmca {

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the CUDA-core (SIMT) forward path, fp32, each region 256-byte
// aligned:
//   states  per-chunk states [B][G][s][e]
//   prefix  their prefix sums (causal: Gp = G chunks) or total (Gp = 1) / n
struct SimtLayout {
  size_t states, prefix, total;
};
inline SimtLayout simt_layout(int B, int n, int s, int e, int C, int causal) {
  const size_t G = (size_t)(n / C), se = (size_t)s * (size_t)e, Gp = causal ? G : 1;
  SimtLayout L;
  L.states = 0;
  L.prefix = align256(sizeof(float) * (size_t)B * G * se);
  L.total = L.prefix + align256(sizeof(float) * (size_t)B * Gp * se);
  return L;
}

// Segments of the chunk axis for the chunk walkers: about kWalkUnits units
// (sequence, 256 e columns, segment) in all, as few segments as give that,
// every one non-empty; L chunks each.
constexpr int kWalkUnits = 144;
struct WalkSplit {
  int S, L;
};
inline WalkSplit walk_split(int B, int n, int e, int C) {
  const int G = n / C;
  const int slices = B * ((e + 255) / 256);
  int S = slices > 0 ? kWalkUnits / slices : 1;
  S = S < 1 ? 1 : (S > G ? G : S);
  const int L = (G + S - 1) / S;
  return WalkSplit{(G + L - 1) / L, L};
}

// Workspace of the tensor-core forward path, each region 256-byte aligned:
//   local   bf16 sums of the states of a segment's chunks before each chunk
//           [B][G][s][e] (causal only)
//   seg     bf16 segment totals, then carries (the sum of the segments
//           before; bidirectional: the total, in slot 0) [B][S][s][e]
//   sched   the work counters
//   trows   bf16 rows T0, T1, T2 [3][B*n][s] (T2 carrying the global term's
//           divisor), the fused output kernel's operands
// and, only in the form the backward pass runs (materialised = true):
//   prefix  bf16 scaled prefix (causal: Gp = G chunks) or total (Gp = 1)
//   scores  bf16 intra-chunk relu^2 weights [B*n][C]
//   lin_q   bf16 T2 = Z * gamma2 + beta2 rows [B*n][s]
// The first four regions sit at the same offsets in both forms (the backward
// pass that keeps the forward pass's intermediates reads local and seg).
struct TcLayout {
  size_t local, seg, sched, trows, prefix, scores, lin_q, total;
};
inline size_t tc_sched_bytes() { return 256; }
inline TcLayout tc_layout(int B, int n, int s, int e, int C, int causal, bool materialised) {
  const size_t G = (size_t)(n / C), se = (size_t)s * (size_t)e, Gp = causal ? G : 1;
  const WalkSplit ws = walk_split(B, n, e, C);
  TcLayout L;
  L.local = 0;
  L.seg = causal ? align256(2 * (size_t)B * G * se) : 0;
  L.sched = L.seg + align256(2 * (size_t)B * ws.S * se);
  L.trows = L.sched + tc_sched_bytes();
  L.prefix = L.trows + align256(3 * 2 * (size_t)B * n * (size_t)s);
  L.scores = L.prefix + (materialised ? align256(2 * (size_t)B * Gp * se) : 0);
  L.lin_q = L.scores + (materialised ? align256(2 * (size_t)B * n * (size_t)C) : 0);
  L.total = L.lin_q + (materialised ? align256(2 * (size_t)B * n * (size_t)s) : 0);
  return L;
}

// flash_mca_workspace_bytes: enough for either forward path, so that a
// workspace sized for a shape serves every path a call may pick.
inline size_t workspace_bytes(int B, int n, int s, int e, int C, int causal) {
  const size_t a = simt_layout(B, n, s, e, C, causal).total;
  size_t b = tc_layout(B, n, s, e, C, causal, false).total;
  // chunks longer than 256 tokens: the quadratic-only model keeps its relu^2
  // weights in the workspace (tc_layout with the intermediates)
  if (C > 256) {
    const size_t bm = tc_layout(B, n, s, e, C, causal, true).total;
    if (bm > b) b = bm;
  }
  return a > b ? a : b;
}

// Scale and normalisation variants (flash_mca_forward_ex): intra-chunk weights
// relu(x * quad_a)^2 (quad_a = sqrt(quad_scale); 1/C by default), global-term
// divisor lin_norm (FMCA_LIN_NORM_*).
struct Variant {
  float quad_a;
  int lin_norm;
};
constexpr int kLinNormN = 0, kLinNormSummed = 1, kLinNormPosition = 2, kLinNormNone = 3;
inline Variant default_variant(int C) { return Variant{1.0f / (float)C, kLinNormN}; }

// `events` (may be NULL) holds launch-count + 1 cudaEvent_t handles recorded
// before the first kernel and after each kernel.
int launch_simt_forward(const void *Z, const void *V, const void *U, const float *gamma,
                        const float *beta, void *O, int B, int n, int s, int e, int C,
                        int causal, int dtype_bf16, const Variant &var, void *workspace,
                        cudaStream_t stream, cudaEvent_t const *events = nullptr);

// The tensor-core forward pass (workspace: tc_layout(..., false); without a
// global term and with C > 256 it runs the kernels of
// launch_tc_forward_materialised and needs tc_layout(..., true)).
// A call on one piece of longer causal sequences (flash_mca_forward_seq):
// state_in (fp32 [B][s][e], or null) is the sum of the states T3^T V of the
// sequences' chunks before the piece, state_out (or null) receives that sum
// with the piece's chunks added; tok0 is the piece's first token in its
// sequence (a multiple of C) and n_norm the length the divisor 1/n uses.
struct SeqCarry {
  const float *state_in = nullptr;
  float *state_out = nullptr;
  int tok0 = 0;
  int n_norm = 0;
};
int launch_tc_forward(const void *Z, const void *V, const void *U, const float *gamma,
                      const float *beta, void *O, int B, int n, int s, int e, int C, int causal,
                      const Variant &var, void *workspace, cudaStream_t stream,
                      cudaEvent_t const *events = nullptr, const SeqCarry *carry = nullptr);
// Kernels one launch_tc_forward queues (the memset of its counters not
// counted).
int tc_launch_count(int B, int n, int e, int C, int causal, const Variant &var);
// kernels of launch_tc_forward_materialised (with_states: it forms the local
// sums and carries itself, as the forward pass does)
int tc_materialised_launch_count(int B, int n, int e, int C, int causal, const Variant &var,
                                 bool with_states);

// The forward pass as the backward pass needs it (workspace:
// tc_layout(..., true)): besides O it leaves the relu^2 weights, the lin_q
// rows and the scaled prefix in the workspace.  with_states = false: the
// chunk states and prefix are taken as an earlier launch_tc_forward with the
// same inputs left them in the workspace; only the relu^2 weights, lin_q rows
// and the output are computed.
int launch_tc_forward_materialised(const void *Z, const void *V, const void *U,
                                   const float *gamma, const float *beta, void *O, int B, int n,
                                   int s, int e, int C, int causal, const Variant &var,
                                   void *workspace, cudaStream_t stream, bool with_states,
                                   cudaEvent_t const *events = nullptr);

// Runs a setup step (kernel attributes) once per device and process, safely
// when several host threads make their first call at the same time; later
// calls return the first run's result.
struct OncePerDevice {
  static constexpr int kMaxDevices = 64;
  std::once_flag flags[kMaxDevices];
  bool ok[kMaxDevices] = {};
  template <typename F>
  bool run(F &&setup) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::call_once(flags[dev], [&] { ok[dev] = setup(); });
    return ok[dev];
  }
};

inline bool record_event(cudaEvent_t const *events, int i, cudaStream_t stream) {
  return events == nullptr || cudaEventRecord(events[i], stream) == cudaSuccess;
}

// Decode state (caller-owned, flash_mca_decode_state_bytes), each region
// 256-byte aligned:
//   P   fp32 [B][s][e]   sum of T3^T V over the completed chunks
//   Pb  bf16 [B][s][e]   P rounded to bf16 at each fold, read by the bf16
//                        token kernel (bf16 I/O only; the forward pass also
//                        reads its prefix in bf16)
//   Zc  [B][C][s]        Z rows of the current chunk's tokens (I/O type)
//   Vc  [B][C][e]        their V rows (I/O type)
struct DecodeStateLayout {
  size_t P, Pb, Zc, Vc, total;
};
inline DecodeStateLayout decode_state_layout(int B, int s, int e, int C, size_t elem) {
  DecodeStateLayout L;
  L.P = 0;
  L.Pb = align256(sizeof(float) * (size_t)B * s * e);
  L.Zc = L.Pb + (elem == 2 ? align256(2 * (size_t)B * s * e) : 0);
  L.Vc = L.Zc + align256(elem * (size_t)B * C * s);
  L.total = L.Vc + align256(elem * (size_t)B * C * e);
  return L;
}
constexpr int kDecodeMaxC = 1024;  // chunk length the decode kernels take

// One decode step for the token at position t (launches 1 kernel, or 2 at
// the last token of a chunk).
int launch_decode_step(const void *z, const void *v, const void *u, const float *gamma,
                       const float *beta, void *o, int B, int s, int e, int C, int t, int n_norm,
                       int dtype_bf16, const Variant &var, void *state, cudaStream_t stream);

// Backward workspace (flash_mca_backward_workspace_bytes), fp32, each region
// 256-byte aligned:
//   states   [B][G][s][e]   chunk states (recomputed)
//   prefix   [B][Gp][s][e]  their scaled prefix / total (recomputed)
//   dprefix  [B][G][s][e]   d(prefix) per chunk, then the chunk-state gradients
//   dY       [B*n][e]       dO * U
//   W, dS    [B][G][C][C]   relu^2 weights and score gradients
//   dT       [4][B*n][s]    gradients of the four affine maps
//   part     [ceil(B*n/64)][8][s]  per-block partial sums of dgamma, dbeta
struct BackwardLayout {
  size_t states, prefix, dprefix, dY, W, dS, dT, part, total;
};
inline BackwardLayout backward_layout(int B, int n, int s, int e, int C, int causal) {
  const size_t G = (size_t)(n / C), se = (size_t)s * (size_t)e, rows = (size_t)B * n;
  const size_t Gp = causal ? G : 1;
  BackwardLayout L;
  L.states = 0;
  L.prefix = L.states + align256(4 * (size_t)B * G * se);
  L.dprefix = L.prefix + align256(4 * (size_t)B * Gp * se);
  L.dY = L.dprefix + align256(4 * (size_t)B * G * se);
  L.W = L.dY + align256(4 * rows * (size_t)e);
  L.dS = L.W + align256(4 * (size_t)B * G * (size_t)C * (size_t)C);
  L.dT = L.dS + align256(4 * (size_t)B * G * (size_t)C * (size_t)C);
  L.part = L.dT + align256(4 * 4 * rows * (size_t)s);
  L.total = L.part + align256(4 * 8 * (size_t)s * ((rows + 63) / 64));
  return L;
}

int launch_backward(const void *Z, const void *V, const void *U, const float *gamma,
                    const float *beta, const void *dO, void *dZ, void *dV, void *dU,
                    float *dgamma, float *dbeta, int B, int n, int s, int e, int C, int causal,
                    int dtype_bf16, const Variant &var, void *workspace, cudaStream_t stream);
constexpr int kBackwardLaunches = 12;  // kernels + memsets one backward call queues (at most)

// D = act(A B^T) on the tensor cores: A [M][K], B [N][K] bf16; D's columns
// [0, n0) go to D0 [M][n0], [n0, n1) to D1, [n1, N) to D2 (bf16, row-major).
int launch_gemm(const void *A, const void *B, int M, int N, int K, void *D0, void *D1,
                void *D2, int n0, int n1, int silu, cudaStream_t stream);

// Workspace of the tensor-core backward (bf16 unless noted), each region
// 256-byte aligned: the materialised forward workspace (chunk states, scaled
// prefix, work counters, relu^2 weights, lin_q rows), then dY [B*n][e], T0, T1, T3
// [B*n][s], dS [B*n][C], dT0..dT3 [B*n][s], d(prefix) [B][G][s][e], and fp32
// per-block dgamma/dbeta partials.
constexpr int kTcbAffRows = 64;  // token rows per block of the dZ/dgamma/dbeta reduction
struct TcBackwardLayout {
  size_t fwd, dY, T0, T1, T3, dS, dT0, dT1, dT2, dT3, dP, part, total;
};
inline TcBackwardLayout tc_backward_layout(int B, int n, int s, int e, int C, int causal) {
  const size_t rows = (size_t)B * n, G = (size_t)(n / C);
  TcBackwardLayout L;
  L.fwd = 0;
  L.dY = align256(tc_layout(B, n, s, e, C, causal, true).total);
  L.T0 = L.dY + align256(2 * rows * e);
  L.T1 = L.T0 + align256(2 * rows * s);
  L.T3 = L.T1 + align256(2 * rows * s);
  L.dS = L.T3 + align256(2 * rows * s);
  L.dT0 = L.dS + align256(2 * rows * C);
  L.dT1 = L.dT0 + align256(2 * rows * s);
  L.dT2 = L.dT1 + align256(2 * rows * s);
  L.dT3 = L.dT2 + align256(2 * rows * s);
  L.dP = L.dT3 + align256(2 * rows * s);
  L.part = L.dP + align256(2 * (size_t)B * G * s * e);
  L.total = L.part + align256(4 * 8 * (size_t)s * ((rows + kTcbAffRows - 1) / kTcbAffRows));
  return L;
}
// saved: the workspace already holds the forward pass's intermediates (an
// earlier flash_mca_forward with the same inputs, options and workspace).
int launch_tc_backward(const void *Z, const void *V, const void *U, const float *gamma,
                       const float *beta, const void *dO, void *dZ, void *dV, void *dU,
                       float *dgamma, float *dbeta, int B, int n, int s, int e, int C, int causal,
                       const Variant &var, void *workspace, cudaStream_t stream,
                       bool saved = false);

// Shapes the tensor-core path covers.
bool tc_supported(int B, int n, int s, int e, int C);  // every tensor-core kernel (e % 256)
bool tc_forward_supported(int B, int n, int s, int e, int C, int lin_norm);  // the forward pass
constexpr int kSimtLaunches = 3;

// Device-side status word (tensor-core kernels' bounded waits).
int read_and_clear_device_status(cudaStream_t stream, int32_t *where);
int launch_timeout_selftest(int limit_us, cudaStream_t stream);

}  // namespace fmca
