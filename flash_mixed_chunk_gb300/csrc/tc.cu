// tc.cu -- tensor-core path of the mixed-chunk attention forward core
// (sm_103a: tcgen05 MMA into TMEM, TMA-staged 128-byte-swizzled bf16 tiles,
// mbarrier pipelines) for bf16 I/O, s = 128, C % 128 == 0, e % 64 == 0 (the
// stored-weights form and the backward pass: e % 256 == 0).
//
// Per call ("FLASH: Possibly the Most Interesting Efficient Transformer
// Design Recently", sections "Weak Attention" and "Mixed Chunk"):
//
//   tc_chunk_walk    segment walkers: per (segment of the chunk axis,
//                    sequence, 256-column slice of e), the segment's chunks
//                    in order: state_g = T3_g^T V_g in TMEM, the running sum
//                    (fp32, TMEM) out as each chunk's local sum and the
//                    segment's total (bf16), and the rows T0, T1, T2 (T2
//                    carrying the global term's divisor)
//   tc_chunk_pair    chunks of 256: the segment carries (bidirectional: the
//                    total) from the walkers' totals, then per (chunk, run
//                    of e tiles) the relu^2 weights in TMEM and O = U * (P V_g
//                    + T2 (local + carry)) (bidirectional: + T2 total) for
//                    both row tiles; a programmatic dependent of the walkers
//   tc_seg_carry +   chunks of 128 or over 256 tokens: the carries (or the
//   tc_chunk_fused   total) in a launch of their own, then the same per
//                    (chunk, row tile, e tiles)
//
// Without a global term: tc_affine_rows (T0, T1) and the fused kernel, or,
// for chunks over 256 tokens, the stored-weights form below.  The backward
// pass runs that stored-weights form (launch_tc_forward_materialised):
// tc_chunk_prep writes the relu^2 weights P and the T2 rows to the workspace
// and tc_chunk_attn forms O = U * (P V_g + T2 prefix_g) from them, leaving P
// and T2 for the gradient products.
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
#include "tc_attn.cuh"
#include "tc_fused.cuh"
#include "tc_pair.cuh"
#include "tc_gemm.cuh"

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

// 3-D bf16 map viewing a row-major [rows][cols] matrix (cols % 64 == 0) as
// (64 inner columns, rows, cols / 64 column blocks), 128-byte swizzle: a box
// {64, box_rows, box_blocks} lands as box_blocks consecutive [box_rows][64]
// tiles (see tma_load_3d).
bool make_map3_bf16(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                    uint32_t box_rows, uint32_t box_blocks) {
  EncodeTiledFn enc = get_encode();
  if (!enc || cols % 64) return false;
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_blocks};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
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

// The forward pass's own forms take e in 64-column steps (the output
// kernels' e tiles are 128 columns, the last may be 64; the walkers' last
// slice may be 64 or 128 of its 256), except the
// stored-weights form (no global term, chunks over 256 tokens), whose output
// kernel takes 256-column tiles.
bool tc_forward_supported(int B, int n, int s, int e, int C, int lin_norm) {
  if (s != S_DIM || C % ROW_TILE || n % C || e % (FU_ET / 2)) return false;
  if (lin_norm == kLinNormNone && C > 2 * ROW_TILE && e % E_TILE) return false;
  (void)B;
  return true;
}

// The row-pair output kernel (tc_chunk_pair): chunks of two 128-row tiles
// with a global term, causal or bidirectional.  It forms the segment carries
// (or the total) itself.
static bool use_pair_kernel(int C, int causal, bool lin) {
  (void)causal;
  return lin && C == 2 * ROW_TILE;
}

int tc_launch_count(int B, int n, int e, int C, int causal, const Variant &var) {
  if (var.lin_norm == kLinNormNone) return 2;  // T0 / T1 rows, fused kernel
  if (use_pair_kernel(C, causal, true)) return 2;  // walkers, row-pair kernel
  const WalkSplit sp = walk_split(B, n, e, C);
  return (sp.S > 1 || !causal) ? 3 : 2;  // walkers, [carries], fused kernel
}

int tc_materialised_launch_count(int B, int n, int e, int C, int causal, const Variant &var,
                                 bool with_states) {
  if (var.lin_norm == kLinNormNone) return 2;  // relu^2 weights, output kernel
  const WalkSplit sp = walk_split(B, n, e, C);
  // [walkers, [carries]], scaled prefix, relu^2 weights, output kernel
  return (with_states ? 1 + ((sp.S > 1 || !causal) ? 1 : 0) : 0) + 3;
}

namespace {


// Tiles of the fused kernel: (batch x chunk, row tile, e tile).
FusedGrid fused_grid(int B, int n, int e, int C, int causal, bool lin) {
  FusedGrid g;
  g.n = n;
  g.C = C;
  g.G = n / C;
  g.causal = causal;
  g.lin = lin ? 1 : 0;
  g.R = C / ROW_TILE;
  g.n_et = (e + FU_ET - 1) / FU_ET;  // the last e tile may be 64 columns
  g.n_tiles = B * g.G * g.R * g.n_et;
  g.S = 1;
  g.L = g.G;
  g.rows_early = 0;
  g.carry_all = 0;
  return g;
}

// Launch configuration of a programmatic dependent of the work before it on
// the stream: it may start launching (and run its prologue) while its
// predecessor drains, and waits (griddepcontrol.wait) before it reads what
// the predecessor wrote.
struct PdlConfig {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg;
  PdlConfig(cudaStream_t stream, bool dependent) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg = cudaLaunchConfig_t{};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
  }
};

}  // namespace

int launch_tc_forward(const void *Z, const void *V, const void *U, const float *gamma,
                      const float *beta, void *O, int B, int n, int s, int e, int C, int causal,
                      const Variant &var, void *workspace, cudaStream_t stream,
                      cudaEvent_t const *events, const SeqCarry *carry) {
  // Without a global term and with chunks longer than 256 tokens (the
  // quadratic-only model), a row tile's relu^2 weights do not fit in TMEM
  // beside its accumulators: the chunk kernel would form them again for every
  // e tile.  Those go through HBM once instead (bf16 [B n][C]).
  if (var.lin_norm == kLinNormNone && C > 2 * ROW_TILE)
    return launch_tc_forward_materialised(Z, V, U, gamma, beta, O, B, n, s, e, C, causal, var,
                                          workspace, stream, false, events);
  const int G = n / C;
  const int64_t se = (int64_t)s * e;
  const TcLayout L = tc_layout(B, n, s, e, C, causal, false);
  const WalkSplit sp = walk_split(B, n, e, C);
  char *ws = static_cast<char *>(workspace);
  __nv_bfloat16 *local = reinterpret_cast<__nv_bfloat16 *>(ws + L.local);
  __nv_bfloat16 *seg = reinterpret_cast<__nv_bfloat16 *>(ws + L.seg);
  __nv_bfloat16 *trows = reinterpret_cast<__nv_bfloat16 *>(ws + L.trows);
  const uint64_t rows = (uint64_t)B * n;
  const int64_t plane = (int64_t)rows * s;  // elements of one T-row plane

  // walkers: Z keys and V slices as one 3-D box each (64 keys), sums out as
  // [128 rows][64 cols] tiles; fused kernel: 3-D boxes of 128 rows x two
  // 64-column blocks (32 KB) for every operand
  CUtensorMap mZw, mVw, mL, mT, mT0, mT1, mT2, mV, mLoc, mCy, mU3;
  const uint64_t lrows = causal ? (uint64_t)B * G * s : (uint64_t)s;  // (unused if bidirectional)
  if (!make_map3_bf16(&mZw, Z, s, rows, 64, 2) || !make_map3_bf16(&mVw, V, e, rows, 64, 4) ||
      !make_map_bf16(&mL, local, e, lrows, 64, 128) ||
      !make_map_bf16(&mT, seg, e, (uint64_t)B * sp.S * s, 64, 128) ||
      !make_map3_bf16(&mT0, trows, s, rows, 128, 2) ||
      !make_map3_bf16(&mT1, trows + plane, s, rows, 128, 2) ||
      !make_map3_bf16(&mT2, trows + 2 * plane, s, rows, 128, 2) ||
      !make_map3_bf16(&mV, V, e, rows, 128, 2) ||
      !make_map3_bf16(&mLoc, local, e, lrows, 128, 2) ||
      !make_map3_bf16(&mCy, seg, e, (uint64_t)B * sp.S * s, 128, 2) ||
      !make_map3_bf16(&mU3, U, e, rows, 128, 2))
    return 2;

  static OncePerDevice attrs;
  if (!attrs.run([] {
        return cudaFuncSetAttribute(tc_chunk_walk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)WALK_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(tc_chunk_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)FUSED_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(tc_chunk_pair<false, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)PAIR_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(tc_chunk_pair<true, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)PAIR_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(tc_chunk_pair<false, false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)PAIR_SMEM) == cudaSuccess;
      }))
    return 1;
  if (!record_event(events, 0, stream)) return 1;
  const int sms = num_sms();
  const bool no_global = var.lin_norm == kLinNormNone;
  // the row-pair kernel forms the segment carries itself (counted in
  // sched[2], which the walkers clear)
  const bool pair = use_pair_kernel(C, causal, !no_global);
  const SeqCarry sq = carry != nullptr ? *carry : SeqCarry{};
  const bool with_state = causal && (sq.state_in != nullptr || sq.state_out != nullptr);
  const int n_norm = sq.n_norm > 0 ? sq.n_norm : n;
  unsigned int *carried = reinterpret_cast<unsigned int *>(ws + L.sched) + 2;
  FusedGrid fg = fused_grid(B, n, e, C, causal, !no_global);
  fg.S = sp.S;
  fg.L = sp.L;
  fg.rows_early = 0;
  fg.carry_all = causal && sq.state_in != nullptr ? 1 : 0;
  int ev = 1;
  if (!no_global) {
    // the segment walkers: local sums, segment totals and the T rows
    const int units = B * ((e + WK_ET - 1) / WK_ET) * sp.S;
    tc_chunk_walk<<<units < sms ? units : sms, WK_THREADS, WALK_SMEM, stream>>>(
        mZw, mVw, mL, mT, gamma, beta, trows, plane, B, n, e, C, causal, var.lin_norm, sp.S, sp.L,
        carried, pair ? 0 : 1, sq.tok0, n_norm);
    if (cudaGetLastError() != cudaSuccess || !record_event(events, ev++, stream)) return 1;
    if ((sp.S > 1 || !causal || with_state) && !pair) {
      // totals -> carries (bidirectional: the total), a programmatic
      // dependent of the walkers
      PdlConfig cc(stream, true);
      const int64_t lanes = (int64_t)B * se / 8;
      cc.cfg.gridDim = dim3((unsigned)((lanes + 255) / 256));
      cc.cfg.blockDim = dim3(256);
      cc.cfg.dynamicSmemBytes = 0;
      if (cudaLaunchKernelEx(&cc.cfg, tc_seg_carry, seg, B, sp.S, se, causal, sq.state_in,
                             sq.state_out) != cudaSuccess ||
          !record_event(events, ev++, stream))
        return 1;
      fg.rows_early = 1;
    }
  } else {
    // without a global term: the T0 and T1 rows only
    const int64_t n_vec = plane / 8;
    tc_affine_rows<<<(unsigned)((n_vec + 255) / 256), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(Z), gamma, beta, trows, plane, n_vec);
    if (cudaGetLastError() != cudaSuccess || !record_event(events, ev++, stream)) return 1;
  }
  PdlConfig fc(stream, true);
  if (pair) {
    // both row tiles of a chunk per unit (the e tile's operands serve both)
    PairGrid pg;
    pg.n = n;
    pg.G = G;
    pg.n_et = (e + FU_ET - 1) / FU_ET;
    pg.n_tiles = B * G * pg.n_et;
    pg.S = sp.S;
    pg.L = sp.L;
    pg.rows_early = 0;  // no kernel between: the T rows wait for the walkers too
    pg.B = B;
    pg.carries = sp.S > 1 || with_state;
    pg.carry_all = sq.state_in != nullptr ? 1 : 0;
    fc.cfg.gridDim = dim3(pg.n_tiles < sms ? pg.n_tiles : sms);
    fc.cfg.blockDim = dim3(PAIR_THREADS);
    fc.cfg.dynamicSmemBytes = PAIR_SMEM;
    auto *pair_kernel = !causal      ? tc_chunk_pair<false, false>
                        : with_state ? tc_chunk_pair<true, true>
                                     : tc_chunk_pair<false, true>;
    if (cudaLaunchKernelEx(&fc.cfg, pair_kernel, mT0, mT1, mT2, mV, mLoc, mCy, mU3,
                           static_cast<const __nv_bfloat16 *>(U), static_cast<__nv_bfloat16 *>(O),
                           pg, e, var.quad_a, seg, carried, sq.state_in, sq.state_out) !=
                               cudaSuccess ||
        !record_event(events, ev++, stream))
      return 1;
    return 0;
  }
  fc.cfg.gridDim = dim3(fg.n_tiles < sms ? fg.n_tiles : sms);
  fc.cfg.blockDim = dim3(FUSED_THREADS);
  fc.cfg.dynamicSmemBytes = FUSED_SMEM;
  if (cudaLaunchKernelEx(&fc.cfg, tc_chunk_fused, mT0, mT1, mT2, mV, mLoc, mCy, mU3,
                         static_cast<const __nv_bfloat16 *>(U), static_cast<__nv_bfloat16 *>(O),
                         fg, e, var.quad_a) != cudaSuccess ||
      !record_event(events, ev++, stream))
    return 1;
  return 0;
}

int launch_tc_forward_materialised(const void *Z, const void *V, const void *U,
                                   const float *gamma, const float *beta, void *O, int B, int n,
                                   int s, int e, int C, int causal, const Variant &var,
                                   void *workspace, cudaStream_t stream, bool with_states,
                                   cudaEvent_t const *events) {
  const int G = n / C;
  const int R = C / ROW_TILE;
  const int64_t se = (int64_t)s * e;
  const int Gp = causal ? G : 1;
  const TcLayout L = tc_layout(B, n, s, e, C, causal, true);
  const WalkSplit sp = walk_split(B, n, e, C);
  char *ws = static_cast<char *>(workspace);
  __nv_bfloat16 *local = reinterpret_cast<__nv_bfloat16 *>(ws + L.local);
  __nv_bfloat16 *seg = reinterpret_cast<__nv_bfloat16 *>(ws + L.seg);
  __nv_bfloat16 *trows = reinterpret_cast<__nv_bfloat16 *>(ws + L.trows);
  __nv_bfloat16 *prefix = reinterpret_cast<__nv_bfloat16 *>(ws + L.prefix);
  void *pw = ws + L.scores;
  void *t2 = ws + L.lin_q;
  unsigned int *sched = reinterpret_cast<unsigned int *>(ws + L.sched);
  const uint64_t rows = (uint64_t)B * n;
  const int64_t plane = (int64_t)rows * s;

  CUtensorMap mZ64, mZ128, mZw, mVw, mL, mT, mPw, mT2, mV, mS, mU, mO;
  const uint64_t lrows = causal ? (uint64_t)B * G * s : (uint64_t)s;
  if (!make_map_bf16(&mZ64, Z, s, rows, 64, 64) || !make_map_bf16(&mZ128, Z, s, rows, 64, 128) ||
      !make_map3_bf16(&mZw, Z, s, rows, 64, 2) || !make_map3_bf16(&mVw, V, e, rows, 64, 4) ||
      !make_map_bf16(&mL, local, e, lrows, 64, 128) ||
      !make_map_bf16(&mT, seg, e, (uint64_t)B * sp.S * s, 64, 128) ||
      !make_map_bf16(&mPw, pw, C, rows, 64, 128) || !make_map_bf16(&mT2, t2, s, rows, 64, 128) ||
      !make_map_bf16(&mV, V, e, rows, 64, 64) ||
      !make_map_bf16(&mS, prefix, e, (uint64_t)B * Gp * s, 64, 64) ||
      !make_map_bf16(&mU, U, e, rows, 64, 128) || !make_map_bf16(&mO, O, e, rows, 64, 128))
    return 2;

  static OncePerDevice attrs;
  if (!attrs.run([] {
        return cudaFuncSetAttribute(tc_chunk_prep<false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)PREP_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(tc_chunk_prep<true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)PREP_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(tc_chunk_walk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)WALK_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(tc_chunk_attn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)AT_SMEM) == cudaSuccess;
      }))
    return 1;
  // sched[0]: work counter of tc_chunk_prep; sched[1]: of tc_chunk_attn
  if (cudaMemsetAsync(sched, 0, 2 * sizeof(unsigned int), stream) != cudaSuccess) return 1;
  if (!record_event(events, 0, stream)) return 1;
  int ev = 1;
  // without a global term (FMCA_LIN_NORM_NONE) there is no prefix and the
  // attention units have no lin_q items
  const bool no_global = var.lin_norm == kLinNormNone;
  const int sms = num_sms();
  // the relu^2 weights P and the T2 rows (score units only) first: they need
  // nothing of the global term, and the kernels after it chain on it by
  // programmatic dependent launch (each waits for the one before)
  const int n_score = B * G * score_units_per_chunk(C, causal);
  auto *prep = var.lin_norm == kLinNormPosition ? tc_chunk_prep<true> : tc_chunk_prep<false>;
  prep<<<n_score < sms ? n_score : sms, PREP_THREADS, PREP_SMEM, stream>>>(
      mZ64, mZ128, mZw, mVw, mL, mPw, gamma, beta, reinterpret_cast<__nv_bfloat16 *>(t2),
      nullptr, 0, sched, n, e, C, G, causal, 0, n_score, var.quad_a);
  if (cudaGetLastError() != cudaSuccess || !record_event(events, ev++, stream)) return 1;
  if (!no_global) {
    if (with_states) {
      // the local sums and carries exactly as the forward pass forms them
      // (the walkers end only after the weight kernel has)
      const int units = B * ((e + WK_ET - 1) / WK_ET) * sp.S;
      PdlConfig wc(stream, true);
      wc.cfg.gridDim = dim3(units < sms ? units : sms);
      wc.cfg.blockDim = dim3(WK_THREADS);
      wc.cfg.dynamicSmemBytes = WALK_SMEM;
      if (cudaLaunchKernelEx(&wc.cfg, tc_chunk_walk, mZw, mVw, mL, mT, gamma, beta, trows, plane,
                             B, n, e, C, causal, var.lin_norm, sp.S, sp.L,
                             static_cast<unsigned int *>(nullptr), 1, 0, n) != cudaSuccess ||
          !record_event(events, ev++, stream))
        return 1;
      if (sp.S > 1 || !causal) {
        const int64_t lanes = (int64_t)B * se / 8;
        PdlConfig cc(stream, true);
        cc.cfg.gridDim = dim3((unsigned)((lanes + 255) / 256));
        cc.cfg.blockDim = dim3(256);
        if (cudaLaunchKernelEx(&cc.cfg, tc_seg_carry, seg, B, sp.S, se, causal,
                               static_cast<const float *>(nullptr),
                               static_cast<float *>(nullptr)) != cudaSuccess ||
            !record_event(events, ev++, stream))
          return 1;
      }
    }
    // the scaled prefix of the attention kernel (unscaled T2 rows)
    const int64_t lanes = (int64_t)B * Gp * se / 8;
    PdlConfig fc(stream, true);
    fc.cfg.gridDim = dim3((unsigned)((lanes + 255) / 256));
    fc.cfg.blockDim = dim3(256);
    if (cudaLaunchKernelEx(&fc.cfg, tc_prefix_fixup, static_cast<const __nv_bfloat16 *>(local),
                           static_cast<const __nv_bfloat16 *>(seg), prefix, B, G, sp.S, sp.L, se,
                           causal, n, C, var.lin_norm) != cudaSuccess ||
        !record_event(events, ev++, stream))
      return 1;
  }
  // O = U * (P V_g + T2 prefix_g).  With a global term, a programmatic
  // dependent of the prefix fix-up, whose grid ends after the weight kernel's
  // (through the chain above): the weights and T2 rows are final when it
  // starts, and only its prefix loads wait.  Without one, an ordinary launch
  // after the weight kernel.
  const int n_units = B * G * R * (e / E_TILE);
  PdlConfig ac(stream, !no_global);
  ac.cfg.gridDim = dim3(n_units < sms ? n_units : sms);
  ac.cfg.blockDim = dim3(AT_THREADS);
  ac.cfg.dynamicSmemBytes = AT_SMEM;
  if (cudaLaunchKernelEx(&ac.cfg, tc_chunk_attn, mPw, mT2, mV, mS, mU, mO, sched + 1, n, e, C, G,
                         causal, n_units, no_global ? 0 : S_DIM / KEY_STAGE) != cudaSuccess ||
      !record_event(events, ev++, stream))
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
  static OncePerDevice attrs;
  if (!attrs.run([] {
        return cudaFuncSetAttribute(tc_gemm<GEMM_ACT_NONE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)GEMM_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(tc_gemm<GEMM_ACT_SILU>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)GEMM_SMEM) == cudaSuccess;
      }))
    return 1;
  const int units = ((M + 127) / 128) * ((N + GM_TILE_N - 1) / GM_TILE_N);
  const int sms = num_sms();
  auto *kern = silu ? tc_gemm<GEMM_ACT_SILU> : tc_gemm<GEMM_ACT_NONE>;
  kern<<<units < sms ? units : sms, GEMM_THREADS, GEMM_SMEM, stream>>>(mA, mB, m0, m1, m2, M, N,
                                                                      K, n0, n1);
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

// The tensor-core backward pass (same translation unit: one device status).
#include "tc_backward.cuh"

