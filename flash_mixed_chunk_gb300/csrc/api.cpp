// api.cpp -- the C ABI declared in include/flash_mca.h: argument checks,
// workspace sizing, dispatch between the tensor-core and SIMT kernels, and
// the host-buffer end-to-end entry point.  No allocation happens here.
#include "flash_mca.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "launch.h"

using namespace fmca;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

fmca_status check_sizes(int B, int n, int s, int e, int C, int causal, fmca_dtype dtype) {
  (void)causal;
  if (B <= 0 || n <= 0 || s <= 0 || e <= 0 || C <= 0) return FMCA_ERR_INVALID_ARG;
  if (dtype != FMCA_F32 && dtype != FMCA_BF16) return FMCA_ERR_INVALID_ARG;
  if (C > n || n % C != 0) return FMCA_ERR_SHAPE;
  if (s > 256) return FMCA_ERR_UNSUPPORTED;
  const int64_t big = (int64_t)B * n * (s > e ? s : e);
  if (big >= ((int64_t)1 << 31)) return FMCA_ERR_UNSUPPORTED;
  // the state tensor [B][G][s][e] must be indexable as well
  if ((int64_t)B * (n / C) * s * (int64_t)e >= ((int64_t)1 << 31)) return FMCA_ERR_UNSUPPORTED;
  return FMCA_OK;
}

// the forward pass on the tensor cores (lin_norm: the call's global-term
// divisor, which selects the stored-weights form for chunks over 256 tokens
// without a global term)
bool want_tc(int B, int n, int s, int e, int C, fmca_dtype dtype, int lin_norm = kLinNormN) {
  return dtype == FMCA_BF16 && tc_forward_supported(B, n, s, e, C, lin_norm);
}

size_t elem_size(fmca_dtype dtype) { return dtype == FMCA_BF16 ? 2 : 4; }

// The kernels' form of the options: relu(x * quad_a)^2 with quad_a =
// sqrt(quad_scale).  The defaults give exactly quad_a = 1/C.
fmca_status to_variant(const fmca_options *opts, int C, Variant *v) {
  *v = default_variant(C);
  if (!opts) return FMCA_OK;
  const float q = opts->quad_scale;
  if (!std::isfinite(q) || q < 0.0f) return FMCA_ERR_INVALID_ARG;
  if (opts->lin_norm != FMCA_LIN_NORM_N && opts->lin_norm != FMCA_LIN_NORM_SUMMED &&
      opts->lin_norm != FMCA_LIN_NORM_POSITION && opts->lin_norm != FMCA_LIN_NORM_NONE)
    return FMCA_ERR_INVALID_ARG;
  const double dq = (double)q, dflt = 1.0 / ((double)C * (double)C);
  if ((float)dflt != q) v->quad_a = (float)std::sqrt(dq);
  v->lin_norm = opts->lin_norm;
  return FMCA_OK;
}

fmca_status forward_impl(const void *Z, const void *V, const void *U, const float *gamma,
                         const float *beta, void *O, int B, int n, int s, int e, int C,
                         int causal, fmca_dtype dtype, void *workspace, size_t workspace_bytes_,
                         fmca_path path, const fmca_options *opts, void *const *events,
                         int n_events, fmca_stream_t stream, const fmca_seq *seq = nullptr);

}  // namespace

extern "C" {

fmca_status flash_mca_default_options(int C, fmca_options *opts) {
  if (C <= 0 || !opts) return FMCA_ERR_INVALID_ARG;
  opts->quad_scale = (float)(1.0 / ((double)C * (double)C));
  opts->lin_norm = FMCA_LIN_NORM_N;
  return FMCA_OK;
}

size_t flash_mca_workspace_bytes(int B, int n, int s, int e, int C, int causal,
                                 fmca_dtype dtype) {
  if (check_sizes(B, n, s, e, C, causal, dtype) != FMCA_OK) return 0;
  return workspace_bytes(B, n, s, e, C, causal);
}

int flash_mca_auto_path(int B, int n, int s, int e, int C, int causal, fmca_dtype dtype) {
  if (check_sizes(B, n, s, e, C, causal, dtype) != FMCA_OK) return -1;
  return want_tc(B, n, s, e, C, dtype) ? FMCA_PATH_TCGEN05 : FMCA_PATH_SIMT;
}

int flash_mca_launch_count_ex(int B, int n, int s, int e, int C, int causal, fmca_dtype dtype,
                              fmca_path path, const fmca_options *opts) {
  if (check_sizes(B, n, s, e, C, causal, dtype) != FMCA_OK) return 0;
  Variant var;
  if (to_variant(opts, C, &var) != FMCA_OK) return 0;
  if (path == FMCA_PATH_AUTO)
    path = want_tc(B, n, s, e, C, dtype, var.lin_norm) ? FMCA_PATH_TCGEN05 : FMCA_PATH_SIMT;
  if (path == FMCA_PATH_TCGEN05)
    return want_tc(B, n, s, e, C, dtype, var.lin_norm) ? tc_launch_count(B, n, e, C, causal, var)
                                                       : 0;
  if (path == FMCA_PATH_SIMT) return kSimtLaunches;
  return 0;
}

int flash_mca_launch_count(int B, int n, int s, int e, int C, int causal, fmca_dtype dtype,
                           fmca_path path) {
  return flash_mca_launch_count_ex(B, n, s, e, C, causal, dtype, path, nullptr);
}

fmca_status flash_mca_forward_timed(const void *Z, const void *V, const void *U,
                                    const float *gamma, const float *beta, void *O, int B,
                                    int n, int s, int e, int C, int causal, fmca_dtype dtype,
                                    void *workspace, size_t workspace_bytes_, fmca_path path,
                                    const fmca_options *opts, void *const *events, int n_events,
                                    fmca_stream_t stream) {
  return forward_impl(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, dtype, workspace,
                      workspace_bytes_, path, opts, events, n_events, stream);
}

size_t flash_mca_decode_state_bytes(int B, int s, int e, int C, fmca_dtype dtype) {
  if (B <= 0 || s <= 0 || e <= 0 || C <= 0) return 0;
  if (dtype != FMCA_F32 && dtype != FMCA_BF16) return 0;
  if (s > 256 || C > kDecodeMaxC) return 0;
  if ((int64_t)B * s * e >= ((int64_t)1 << 31) || (int64_t)B * C * (s > e ? s : e) >= ((int64_t)1 << 31))
    return 0;
  return decode_state_layout(B, s, e, C, elem_size(dtype)).total;
}

fmca_status flash_mca_decode_reset(void *state, size_t state_bytes, int B, int s, int e, int C,
                                   fmca_dtype dtype, fmca_stream_t stream) {
  const size_t need = flash_mca_decode_state_bytes(B, s, e, C, dtype);
  if (need == 0) return FMCA_ERR_INVALID_ARG;
  if (!state || state_bytes < need) return FMCA_ERR_WORKSPACE;
  if (!aligned256(state)) return FMCA_ERR_ALIGN;
  // only the carried sum must start at zero; cache slots are written before
  // they are read
  const DecodeStateLayout L = decode_state_layout(B, s, e, C, elem_size(dtype));
  return cudaMemsetAsync(state, 0, L.Zc - L.P, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FMCA_OK
             : FMCA_ERR_CUDA;
}

fmca_status flash_mca_decode_step(const void *z, const void *v, const void *u,
                                  const float *gamma, const float *beta, void *o, int B, int s,
                                  int e, int C, int t, int n_norm, fmca_dtype dtype,
                                  const fmca_options *opts, void *state, size_t state_bytes,
                                  fmca_stream_t stream) {
  const size_t need = flash_mca_decode_state_bytes(B, s, e, C, dtype);
  if (need == 0 || t < 0) return FMCA_ERR_INVALID_ARG;
  if (!z || !v || !u || !gamma || !beta || !o) return FMCA_ERR_INVALID_ARG;
  Variant var;
  fmca_status st = to_variant(opts, C, &var);
  if (st != FMCA_OK) return st;
  if (var.lin_norm == FMCA_LIN_NORM_N && n_norm <= t) return FMCA_ERR_INVALID_ARG;
  if (!aligned16(z) || !aligned16(v) || !aligned16(u) || !aligned16(o) || !aligned16(gamma) ||
      !aligned16(beta))
    return FMCA_ERR_ALIGN;
  if (!state || state_bytes < need) return FMCA_ERR_WORKSPACE;
  if (!aligned256(state)) return FMCA_ERR_ALIGN;
  {  // o must not overlap the inputs or the state
    const size_t es = elem_size(dtype);
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(o), o1 = o0 + (size_t)B * e * es;
    auto overlaps = [&](const void *p, size_t bytes) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), a1 = a0 + bytes;
      return a0 < o1 && o0 < a1;
    };
    if (overlaps(z, (size_t)B * s * es) || overlaps(v, (size_t)B * e * es) ||
        overlaps(u, (size_t)B * e * es) || overlaps(state, state_bytes))
      return FMCA_ERR_INVALID_ARG;
  }
  return launch_decode_step(z, v, u, gamma, beta, o, B, s, e, C, t, n_norm,
                            dtype == FMCA_BF16 ? 1 : 0, var, state,
                            reinterpret_cast<cudaStream_t>(stream)) == 0
             ? FMCA_OK
             : FMCA_ERR_CUDA;
}

// bf16 shapes of the tensor-core forward path run the tensor-core backward;
// everything else the CUDA-core one.
static bool tc_backward(int B, int n, int s, int e, int C, fmca_dtype dtype) {
  return dtype == FMCA_BF16 && tc_supported(B, n, s, e, C);
}
static size_t backward_bytes(int B, int n, int s, int e, int C, int causal, fmca_dtype dtype) {
  return tc_backward(B, n, s, e, C, dtype) ? tc_backward_layout(B, n, s, e, C, causal).total
                                           : backward_layout(B, n, s, e, C, causal).total;
}

size_t flash_mca_backward_workspace_bytes(int B, int n, int s, int e, int C, int causal,
                                          fmca_dtype dtype) {
  if (check_sizes(B, n, s, e, C, causal, dtype) != FMCA_OK) return 0;
  return backward_bytes(B, n, s, e, C, causal, dtype);
}

static fmca_status backward_impl(const void *Z, const void *V, const void *U, const float *gamma,
                                 const float *beta, const void *dO, void *dZ, void *dV, void *dU,
                                 float *dgamma, float *dbeta, int B, int n, int s, int e, int C,
                                 int causal, fmca_dtype dtype, const fmca_options *opts,
                                 void *workspace, size_t workspace_bytes_, fmca_stream_t stream,
                                 bool saved) {
  fmca_status st = check_sizes(B, n, s, e, C, causal, dtype);
  if (st != FMCA_OK) return st;
  if (saved && !tc_backward(B, n, s, e, C, dtype)) return FMCA_ERR_UNSUPPORTED;
  if (!Z || !V || !U || !gamma || !beta || !dO || !dZ || !dV || !dU || !dgamma || !dbeta)
    return FMCA_ERR_INVALID_ARG;
  Variant var;
  st = to_variant(opts, C, &var);
  if (st != FMCA_OK) return st;
  const void *ptrs[] = {Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma, dbeta};
  for (const void *p : ptrs)
    if (!aligned16(p)) return FMCA_ERR_ALIGN;
  if (!workspace) return FMCA_ERR_WORKSPACE;
  if (!aligned256(workspace)) return FMCA_ERR_ALIGN;
  if (workspace_bytes_ < backward_bytes(B, n, s, e, C, causal, dtype)) return FMCA_ERR_WORKSPACE;
  {  // outputs must not overlap the inputs or the workspace
    const size_t es = elem_size(dtype), zb = (size_t)B * n * s * es, vb = (size_t)B * n * e * es;
    const size_t gb = sizeof(float) * 4 * (size_t)s;
    struct Span { const void *p; size_t n; };
    const Span outs[] = {{dZ, zb}, {dV, vb}, {dU, vb}, {dgamma, gb}, {dbeta, gb}};
    const Span ins[] = {{Z, zb}, {V, vb}, {U, vb}, {dO, vb}, {gamma, gb}, {beta, gb},
                        {workspace, workspace_bytes_}};
    auto overlap = [](const Span &a, const Span &b) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
      return a0 < b0 + b.n && b0 < a0 + a.n;
    };
    for (const Span &o : outs) {
      for (const Span &i : ins)
        if (overlap(o, i)) return FMCA_ERR_INVALID_ARG;
      for (const Span &o2 : outs)
        if (&o2 != &o && overlap(o, o2)) return FMCA_ERR_INVALID_ARG;
    }
  }
  if (tc_backward(B, n, s, e, C, dtype))
    return launch_tc_backward(Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma, dbeta, B, n, s, e, C,
                              causal ? 1 : 0, var, workspace,
                              reinterpret_cast<cudaStream_t>(stream), saved) == 0
               ? FMCA_OK
               : FMCA_ERR_CUDA;
  return launch_backward(Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma, dbeta, B, n, s, e, C,
                         causal ? 1 : 0, dtype == FMCA_BF16 ? 1 : 0, var, workspace,
                         reinterpret_cast<cudaStream_t>(stream)) == 0
             ? FMCA_OK
             : FMCA_ERR_CUDA;
}

fmca_status flash_mca_backward(const void *Z, const void *V, const void *U, const float *gamma,
                               const float *beta, const void *dO, void *dZ, void *dV, void *dU,
                               float *dgamma, float *dbeta, int B, int n, int s, int e, int C,
                               int causal, fmca_dtype dtype, const fmca_options *opts,
                               void *workspace, size_t workspace_bytes_, fmca_stream_t stream) {
  return backward_impl(Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma, dbeta, B, n, s, e, C, causal,
                       dtype, opts, workspace, workspace_bytes_, stream, false);
}

int flash_mca_backward_launch_count(int B, int n, int s, int e, int C, int causal,
                                    fmca_dtype dtype, const fmca_options *opts, int saved) {
  if (check_sizes(B, n, s, e, C, causal, dtype) != FMCA_OK) return 0;
  Variant var;
  if (to_variant(opts, C, &var) != FMCA_OK) return 0;
  const int glob = var.lin_norm != kLinNormNone ? 1 : 0;
  if (tc_backward(B, n, s, e, C, dtype))
    // forward kernels (with `saved`: without the chunk walkers), dY and the
    // T rows, three product launches, the reverse scan, dZ with its partials
    // and their sum
    return tc_materialised_launch_count(B, n, e, C, causal, var, !saved) + 2 + 3 + glob + 2;
  if (saved) return 0;
  // CUDA cores: the chunk states and prefix, dY, score gradients, dU, key
  // gradients, the d(prefix) outer products, reverse scan and lin rows, dV,
  // dZ with its partials and their sum
  return glob ? 12 : 7;
}

fmca_status flash_mca_backward_saved(const void *Z, const void *V, const void *U,
                                     const float *gamma, const float *beta, const void *dO,
                                     void *dZ, void *dV, void *dU, float *dgamma, float *dbeta,
                                     int B, int n, int s, int e, int C, int causal,
                                     fmca_dtype dtype, const fmca_options *opts, void *workspace,
                                     size_t workspace_bytes_, fmca_stream_t stream) {
  return backward_impl(Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma, dbeta, B, n, s, e, C, causal,
                       dtype, opts, workspace, workspace_bytes_, stream, true);
}

fmca_status flash_mca_gau_project(const void *X, const void *Wt, void *U, void *V, void *Z,
                                  int M, int d, int e, int s, fmca_stream_t stream) {
  if (!X || !Wt || !U || !V || !Z || M <= 0 || d <= 0 || e <= 0 || s <= 0)
    return FMCA_ERR_INVALID_ARG;
  if (d % 8 || e % 64 || s % 64) return FMCA_ERR_UNSUPPORTED;
  if ((int64_t)M * (2 * (int64_t)e + s) >= ((int64_t)1 << 31) ||
      (int64_t)M * d >= ((int64_t)1 << 31))
    return FMCA_ERR_UNSUPPORTED;
  const void *ptrs[] = {X, Wt, U, V, Z};
  for (const void *p : ptrs)
    if (!aligned16(p)) return FMCA_ERR_ALIGN;
  {
    struct Span { const void *p; size_t n; };
    const Span ins[] = {{X, 2 * (size_t)M * d}, {Wt, 2 * (size_t)(2 * e + s) * d}};
    const Span outs[] = {{U, 2 * (size_t)M * e}, {V, 2 * (size_t)M * e}, {Z, 2 * (size_t)M * s}};
    auto overlap = [](const Span &a, const Span &b) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
      return a0 < b0 + b.n && b0 < a0 + a.n;
    };
    for (const Span &o : outs) {
      for (const Span &i : ins)
        if (overlap(o, i)) return FMCA_ERR_INVALID_ARG;
      for (const Span &o2 : outs)
        if (&o2 != &o && overlap(o, o2)) return FMCA_ERR_INVALID_ARG;
    }
  }
  return launch_gemm(X, Wt, M, 2 * e + s, d, U, V, Z, e, 2 * e, 1,
                     reinterpret_cast<cudaStream_t>(stream)) == 0
             ? FMCA_OK
             : FMCA_ERR_CUDA;
}

fmca_status flash_mca_gau_output(const void *Y, const void *Wo_t, void *Out, int M, int e, int d,
                                 fmca_stream_t stream) {
  if (!Y || !Wo_t || !Out || M <= 0 || d <= 0 || e <= 0) return FMCA_ERR_INVALID_ARG;
  if (e % 8 || d % 64) return FMCA_ERR_UNSUPPORTED;
  if ((int64_t)M * (e > d ? e : d) >= ((int64_t)1 << 31)) return FMCA_ERR_UNSUPPORTED;
  if (!aligned16(Y) || !aligned16(Wo_t) || !aligned16(Out)) return FMCA_ERR_ALIGN;
  {
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(Out), o1 = o0 + 2 * (size_t)M * d;
    auto overlaps = [&](const void *p, size_t bytes) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), a1 = a0 + bytes;
      return a0 < o1 && o0 < a1;
    };
    if (overlaps(Y, 2 * (size_t)M * e) || overlaps(Wo_t, 2 * (size_t)d * e))
      return FMCA_ERR_INVALID_ARG;
  }
  return launch_gemm(Y, Wo_t, M, d, e, Out, Out, Out, d, d, 0,
                     reinterpret_cast<cudaStream_t>(stream)) == 0
             ? FMCA_OK
             : FMCA_ERR_CUDA;
}

fmca_status flash_mca_forward_ex(const void *Z, const void *V, const void *U,
                                 const float *gamma, const float *beta, void *O, int B, int n,
                                 int s, int e, int C, int causal, fmca_dtype dtype,
                                 void *workspace, size_t workspace_bytes_, fmca_path path,
                                 const fmca_options *opts, fmca_stream_t stream) {
  return forward_impl(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, dtype, workspace,
                      workspace_bytes_, path, opts, nullptr, 0, stream);
}

fmca_status flash_mca_forward_seq(const void *Z, const void *V, const void *U,
                                  const float *gamma, const float *beta, void *O, int B, int n,
                                  int s, int e, int C, int causal, fmca_dtype dtype,
                                  void *workspace, size_t workspace_bytes_,
                                  const fmca_options *opts, const fmca_seq *seq,
                                  fmca_stream_t stream) {
  return forward_impl(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, dtype, workspace,
                      workspace_bytes_, FMCA_PATH_AUTO, opts, nullptr, 0, stream, seq);
}

}  // extern "C"

namespace {

fmca_status forward_impl(const void *Z, const void *V, const void *U, const float *gamma,
                         const float *beta, void *O, int B, int n, int s, int e, int C,
                         int causal, fmca_dtype dtype, void *workspace, size_t workspace_bytes_,
                         fmca_path path, const fmca_options *opts, void *const *events,
                         int n_events, fmca_stream_t stream, const fmca_seq *seq) {
  fmca_status st = check_sizes(B, n, s, e, C, causal, dtype);
  if (st != FMCA_OK) return st;
  Variant var;
  st = to_variant(opts, C, &var);
  if (st != FMCA_OK) return st;
  if (!Z || !V || !U || !gamma || !beta || !O) return FMCA_ERR_INVALID_ARG;
  if (path != FMCA_PATH_AUTO && path != FMCA_PATH_SIMT && path != FMCA_PATH_TCGEN05)
    return FMCA_ERR_INVALID_ARG;
  if (!aligned16(Z) || !aligned16(V) || !aligned16(U) || !aligned16(O) || !aligned16(gamma) ||
      !aligned16(beta))
    return FMCA_ERR_ALIGN;
  if (!workspace) return FMCA_ERR_WORKSPACE;
  if (!aligned256(workspace)) return FMCA_ERR_ALIGN;
  if (workspace_bytes_ < workspace_bytes(B, n, s, e, C, causal)) return FMCA_ERR_WORKSPACE;
  // O must not overlap the inputs or the workspace
  {
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(O);
    const uintptr_t o1 = o0 + (size_t)B * n * e * elem_size(dtype);
    auto overlaps = [&](const void *p, size_t bytes) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), a1 = a0 + bytes;
      return a0 < o1 && o0 < a1;
    };
    const size_t es = elem_size(dtype);
    if (overlaps(Z, (size_t)B * n * s * es) || overlaps(V, (size_t)B * n * e * es) ||
        overlaps(U, (size_t)B * n * e * es) || overlaps(workspace, workspace_bytes_))
      return FMCA_ERR_INVALID_ARG;
  }
  const bool tc_ok = want_tc(B, n, s, e, C, dtype, var.lin_norm);
  if (path == FMCA_PATH_TCGEN05 && !tc_ok) return FMCA_ERR_UNSUPPORTED;
  // a piece of longer sequences: causal, the tensor-core path, a global term
  SeqCarry carry;
  if (seq != nullptr) {
    if (!causal || !tc_ok || var.lin_norm == kLinNormNone) return FMCA_ERR_UNSUPPORTED;
    if (seq->token_offset < 0 || seq->token_offset % C != 0 || seq->n_norm < 0 ||
        seq->token_offset + (int64_t)n >= ((int64_t)1 << 31) || seq->n_norm >= ((int64_t)1 << 31))
      return FMCA_ERR_INVALID_ARG;
    if (!aligned16(seq->state_in) || !aligned16(seq->state_out)) return FMCA_ERR_ALIGN;
    if (seq->state_out != nullptr) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(seq->state_out);
      const uintptr_t a1 = a0 + sizeof(float) * (size_t)B * s * e;
      auto hits = [&](const void *p, size_t bytes) {
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(p), b1 = b0 + bytes;
        return b0 < a1 && a0 < b1;
      };
      const size_t es = elem_size(dtype);
      if (hits(Z, (size_t)B * n * s * es) || hits(V, (size_t)B * n * e * es) ||
          hits(U, (size_t)B * n * e * es) || hits(O, (size_t)B * n * e * es) ||
          hits(workspace, workspace_bytes_))
        return FMCA_ERR_INVALID_ARG;
    }
    carry.state_in = seq->state_in;
    carry.state_out = seq->state_out;
    carry.tok0 = (int)seq->token_offset;
    carry.n_norm = (int)seq->n_norm;
  }
  const bool use_tc = (path == FMCA_PATH_TCGEN05) || (path == FMCA_PATH_AUTO && tc_ok);
  const int nlaunch = use_tc ? tc_launch_count(B, n, e, C, causal, var) : kSimtLaunches;
  if (events != nullptr) {
    if (n_events != nlaunch + 1) return FMCA_ERR_INVALID_ARG;
    for (int i = 0; i < n_events; ++i)
      if (events[i] == nullptr) return FMCA_ERR_INVALID_ARG;
  }
  cudaEvent_t const *ev = reinterpret_cast<cudaEvent_t const *>(events);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int rc;
  if (use_tc)
    rc = launch_tc_forward(Z, V, U, gamma, beta, O, B, n, s, e, C, causal ? 1 : 0, var,
                           workspace, cs, ev, seq != nullptr ? &carry : nullptr);
  else
    rc = launch_simt_forward(Z, V, U, gamma, beta, O, B, n, s, e, C, causal ? 1 : 0,
                             dtype == FMCA_BF16 ? 1 : 0, var, workspace, cs, ev);
  return rc == 0 ? FMCA_OK : FMCA_ERR_CUDA;
}

// Pieces of the host-buffer pipeline: with at least two sequences and 96 MB
// of inputs and output, up to four pieces of whole sequences (their copies
// overlap the passes); smaller problems keep one stream (their passes and
// copies are too short for the overlap to pay for its extra launches).  Fewer
// than four causal sequences of 96 MB or more on the tensor cores run pieces
// of every sequence's tokens instead (flash_mca_forward_host).
constexpr size_t kHostPipelineBytes = (size_t)96 << 20;
int host_pipeline_pieces(int B, size_t bytes) {
  if (B < 2 || bytes < kHostPipelineBytes) return 1;
  return B < 4 ? B : 4;
}

// The host-buffer pipeline's copy streams and events, one set per device,
// created on first use; a call holds the set's mutex while it queues.
constexpr int kMaxHostPieces = 4;
struct HostStreams {
  std::mutex mutex;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, out_done = nullptr;
  cudaEvent_t in_done[kMaxHostPieces] = {}, pass_done[kMaxHostPieces] = {};
  bool ready = false;
};
constexpr int kMaxHostDevices = 64;
HostStreams g_host_streams[kMaxHostDevices];
std::mutex g_host_streams_init;

HostStreams *host_streams() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxHostDevices) return nullptr;
  HostStreams &h = g_host_streams[dev];
  std::lock_guard<std::mutex> lock(g_host_streams_init);
  if (!h.ready) {
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.start, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.out_done, ef) == cudaSuccess;
    for (int k = 0; ok && k < kMaxHostPieces; ++k)
      ok = cudaEventCreateWithFlags(&h.in_done[k], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&h.pass_done[k], ef) == cudaSuccess;
    if (!ok) return nullptr;
    h.ready = true;
  }
  return &h;
}

}  // namespace

extern "C" {


fmca_status flash_mca_forward_path(const void *Z, const void *V, const void *U,
                                   const float *gamma, const float *beta, void *O, int B,
                                   int n, int s, int e, int C, int causal, fmca_dtype dtype,
                                   void *workspace, size_t workspace_bytes_, fmca_path path,
                                   fmca_stream_t stream) {
  return flash_mca_forward_timed(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, dtype,
                                 workspace, workspace_bytes_, path, nullptr, nullptr, 0, stream);
}

fmca_status flash_mca_forward(const void *Z, const void *V, const void *U, const float *gamma,
                              const float *beta, void *O, int B, int n, int s, int e, int C,
                              int causal, fmca_dtype dtype, void *workspace,
                              size_t workspace_bytes_, fmca_stream_t stream) {
  return flash_mca_forward_path(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, dtype, workspace,
                                workspace_bytes_, FMCA_PATH_AUTO, stream);
}

// Arena layout for the host-buffer entry point: Z | V | U | gamma | beta | O |
// workspace, each 256-byte aligned.
size_t flash_mca_host_arena_bytes(int B, int n, int s, int e, int C, int causal,
                                  fmca_dtype dtype) {
  if (check_sizes(B, n, s, e, C, causal, dtype) != FMCA_OK) return 0;
  const size_t es = elem_size(dtype);
  return align256((size_t)B * n * s * es) + 3 * align256((size_t)B * n * e * es) +
         2 * align256(sizeof(float) * 4 * (size_t)s) + workspace_bytes(B, n, s, e, C, causal) +
         align256(sizeof(float) * (size_t)B * s * e);  // the carried state of token pieces
}

fmca_status flash_mca_forward_host(const void *hZ, const void *hV, const void *hU,
                                   const float *hgamma, const float *hbeta, void *hO, int B,
                                   int n, int s, int e, int C, int causal, fmca_dtype dtype,
                                   void *device_arena, size_t arena_bytes,
                                   fmca_stream_t stream) {
  fmca_status st = check_sizes(B, n, s, e, C, causal, dtype);
  if (st != FMCA_OK) return st;
  if (!hZ || !hV || !hU || !hgamma || !hbeta || !hO) return FMCA_ERR_INVALID_ARG;
  if (!device_arena) return FMCA_ERR_WORKSPACE;
  if (!aligned256(device_arena)) return FMCA_ERR_ALIGN;
  if (arena_bytes < flash_mca_host_arena_bytes(B, n, s, e, C, causal, dtype))
    return FMCA_ERR_WORKSPACE;
  const size_t es = elem_size(dtype);
  const size_t zb = (size_t)B * n * s * es, vb = (size_t)B * n * e * es;
  const size_t gbytes = sizeof(float) * 4 * (size_t)s;
  char *p = static_cast<char *>(device_arena);
  char *dZ = p;
  p += align256(zb);
  char *dV = p;
  p += align256(vb);
  char *dU = p;
  p += align256(vb);
  float *dg = reinterpret_cast<float *>(p);
  p += align256(gbytes);
  float *db = reinterpret_cast<float *>(p);
  p += align256(gbytes);
  char *dO = p;
  p += align256(vb);
  void *ws = p;
  const size_t wsb = workspace_bytes(B, n, s, e, C, causal);
  p += align256(wsb);
  float *dstate = reinterpret_cast<float *>(p);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int pieces = host_pipeline_pieces(B, zb + 3 * vb);
  // Fewer than four sequences, causal, on the tensor cores: pieces of every
  // sequence's tokens instead (a quarter or a half of each), run in order
  // with the chunk-state sum carried from piece to piece (flash_mca_forward_seq),
  // so that the last piece's pass and copy out are short.
  int parts = 1;
  if (zb + 3 * vb >= kHostPipelineBytes && B < 4 && causal && want_tc(B, n, s, e, C, dtype))
    for (int p2 : {4, 2})
      if (n % p2 == 0 && (n / p2) % C == 0) {
        parts = p2;
        break;
      }
  if (parts > 1) {
    HostStreams *hs = host_streams();
    if (hs == nullptr) return FMCA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(hs->mutex);
    const int np = n / parts;
    const size_t zr = (size_t)np * s * es, vr = (size_t)np * e * es;  // one sequence's part
    const size_t zpiece = (size_t)B * zr, vpiece = (size_t)B * vr;     // a piece, all sequences
    if (cudaEventRecord(hs->start, cs) != cudaSuccess ||
        cudaStreamWaitEvent(hs->in, hs->start, 0) != cudaSuccess ||
        cudaMemcpyAsync(dg, hgamma, gbytes, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
        cudaMemcpyAsync(db, hbeta, gbytes, cudaMemcpyHostToDevice, hs->in) != cudaSuccess)
      return FMCA_ERR_CUDA;
    for (int k = 0; k < parts; ++k) {
      // piece k: tokens [k np, (k + 1) np) of every sequence, gathered into a
      // contiguous [B][np][.] block of the arena (one strided copy each)
      char *pz = dZ + k * zpiece, *pv = dV + k * vpiece, *pu = dU + k * vpiece;
      char *po = dO + k * vpiece;
      if (cudaMemcpy2DAsync(pz, zr, static_cast<const char *>(hZ) + k * zr, (size_t)n * s * es,
                            zr, B, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
          cudaMemcpy2DAsync(pv, vr, static_cast<const char *>(hV) + k * vr, (size_t)n * e * es,
                            vr, B, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
          cudaMemcpy2DAsync(pu, vr, static_cast<const char *>(hU) + k * vr, (size_t)n * e * es,
                            vr, B, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
          cudaEventRecord(hs->in_done[k], hs->in) != cudaSuccess ||
          cudaStreamWaitEvent(cs, hs->in_done[k], 0) != cudaSuccess)
        return FMCA_ERR_CUDA;
      fmca_seq seq;
      seq.state_in = k > 0 ? dstate : nullptr;
      seq.state_out = dstate;
      seq.token_offset = (int64_t)k * np;
      seq.n_norm = n;
      st = flash_mca_forward_seq(pz, pv, pu, dg, db, po, B, np, s, e, C, causal, dtype, ws, wsb,
                                 nullptr, &seq, stream);
      if (st != FMCA_OK) return st;
      if (cudaEventRecord(hs->pass_done[k], cs) != cudaSuccess ||
          cudaStreamWaitEvent(hs->out, hs->pass_done[k], 0) != cudaSuccess ||
          cudaMemcpy2DAsync(static_cast<char *>(hO) + k * vr, (size_t)n * e * es, po, vr, vr, B,
                            cudaMemcpyDeviceToHost, hs->out) != cudaSuccess)
        return FMCA_ERR_CUDA;
    }
    if (cudaEventRecord(hs->out_done, hs->out) != cudaSuccess ||
        cudaStreamWaitEvent(cs, hs->out_done, 0) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess)
      return FMCA_ERR_CUDA;
    return FMCA_OK;
  }
  if (pieces <= 1) {
    // one stream: copies in, the pass, the copy out
    if (cudaMemcpyAsync(dZ, hZ, zb, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(dV, hV, vb, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(dU, hU, vb, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(dg, hgamma, gbytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(db, hbeta, gbytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
      return FMCA_ERR_CUDA;
    st = flash_mca_forward(dZ, dV, dU, dg, db, dO, B, n, s, e, C, causal, dtype, ws, wsb, stream);
    if (st != FMCA_OK) return st;
    if (cudaMemcpyAsync(hO, dO, vb, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
      return FMCA_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return FMCA_ERR_CUDA;
    return FMCA_OK;
  }
  // Pieces of whole sequences: piece k's copies in (copy-in stream) overlap
  // piece k-1's pass (the caller's stream) and its copy out (copy-out
  // stream).  Each piece runs as a batch of its own through one workspace.
  HostStreams *hs = host_streams();
  if (hs == nullptr) return FMCA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(hs->mutex);
  const size_t zrow = (size_t)n * s * es, vrow = (size_t)n * e * es;  // one sequence
  if (cudaEventRecord(hs->start, cs) != cudaSuccess ||
      cudaStreamWaitEvent(hs->in, hs->start, 0) != cudaSuccess ||
      cudaMemcpyAsync(dg, hgamma, gbytes, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
      cudaMemcpyAsync(db, hbeta, gbytes, cudaMemcpyHostToDevice, hs->in) != cudaSuccess)
    return FMCA_ERR_CUDA;
  for (int k = 0; k < pieces; ++k) {
    const int b0 = (int)((int64_t)B * k / pieces), b1 = (int)((int64_t)B * (k + 1) / pieces);
    const size_t bp = (size_t)(b1 - b0);
    const char *hz = static_cast<const char *>(hZ) + b0 * zrow;
    const char *hv = static_cast<const char *>(hV) + b0 * vrow;
    const char *hu = static_cast<const char *>(hU) + b0 * vrow;
    if (cudaMemcpyAsync(dZ + b0 * zrow, hz, bp * zrow, cudaMemcpyHostToDevice, hs->in) !=
            cudaSuccess ||
        cudaMemcpyAsync(dV + b0 * vrow, hv, bp * vrow, cudaMemcpyHostToDevice, hs->in) !=
            cudaSuccess ||
        cudaMemcpyAsync(dU + b0 * vrow, hu, bp * vrow, cudaMemcpyHostToDevice, hs->in) !=
            cudaSuccess ||
        cudaEventRecord(hs->in_done[k], hs->in) != cudaSuccess ||
        cudaStreamWaitEvent(cs, hs->in_done[k], 0) != cudaSuccess)
      return FMCA_ERR_CUDA;
    st = flash_mca_forward(dZ + b0 * zrow, dV + b0 * vrow, dU + b0 * vrow, dg, db,
                           dO + b0 * vrow, (int)bp, n, s, e, C, causal, dtype, ws, wsb, stream);
    if (st != FMCA_OK) return st;
    if (cudaEventRecord(hs->pass_done[k], cs) != cudaSuccess ||
        cudaStreamWaitEvent(hs->out, hs->pass_done[k], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char *>(hO) + b0 * vrow, dO + b0 * vrow, bp * vrow,
                        cudaMemcpyDeviceToHost, hs->out) != cudaSuccess)
      return FMCA_ERR_CUDA;
  }
  if (cudaEventRecord(hs->out_done, hs->out) != cudaSuccess ||
      cudaStreamWaitEvent(cs, hs->out_done, 0) != cudaSuccess ||
      cudaStreamSynchronize(cs) != cudaSuccess)
    return FMCA_ERR_CUDA;
  return FMCA_OK;
}

fmca_status flash_mca_device_status(fmca_stream_t stream, int32_t *where) {
  int st = read_and_clear_device_status(reinterpret_cast<cudaStream_t>(stream), where);
  if (st < 0) return FMCA_ERR_CUDA;
  return st;
}

fmca_status flash_mca_selftest_timeout(int limit_us, fmca_stream_t stream) {
  if (limit_us <= 0 || limit_us > 10 * 1000 * 1000) return FMCA_ERR_INVALID_ARG;
  return launch_timeout_selftest(limit_us, reinterpret_cast<cudaStream_t>(stream)) == 0
             ? FMCA_OK
             : FMCA_ERR_CUDA;
}

const char *flash_mca_status_string(fmca_status status) {
  switch (status) {
    case FMCA_OK: return "FMCA_OK";
    case FMCA_ERR_INVALID_ARG: return "FMCA_ERR_INVALID_ARG: NULL pointer, non-positive size or bad enum";
    case FMCA_ERR_SHAPE: return "FMCA_ERR_SHAPE: C must divide n and C <= n";
    case FMCA_ERR_UNSUPPORTED: return "FMCA_ERR_UNSUPPORTED: shape outside what the kernels support";
    case FMCA_ERR_ALIGN: return "FMCA_ERR_ALIGN: pointer not aligned (16 B data, 256 B workspace)";
    case FMCA_ERR_WORKSPACE: return "FMCA_ERR_WORKSPACE: workspace missing or too small";
    case FMCA_ERR_CUDA: return "FMCA_ERR_CUDA: a CUDA launch or copy failed";
    case FMCA_ERR_TIMEOUT: return "FMCA_ERR_TIMEOUT: a bounded device-side wait ran out";
    default: return "unknown fmca status";
  }
}

const char *flash_mca_version(void) { return "0.1.0"; }

}  // extern "C"
