// tc_bgemm.cuh -- batched products of the backward pass on the tensor cores.
//
//   D_b = alpha * (A_b B_b [+ A2_b B2_b])   for b < batches,
//   bf16 in, fp32 accumulate in TMEM, bf16 out
//
// with A_b [M][K] and B_b [K][N] read from row-major bf16 arrays either
// K-major (A stored [m][k], B stored [n][k]) or MN-major (A stored [k][m], B
// stored [k][n]), chosen per operand at run time.  Operand rows of batch b
// start at (b / div) * rows_per_batch (div > 1 lets consecutive batches share
// an operand, e.g. every chunk of a sequence reading one state matrix); D_b
// occupies rows b * M .. of D [rows][N].  The optional second pair (depth K2)
// accumulates into the same tile.  M and K are multiples of 128 and 64, N a
// multiple of the N tile (128 or 256), so that no tile reaches into another
// batch's rows.
//
// One launch runs up to three independent problems: their tiles are numbered
// one after the other and dealt round-robin to the persistent CTAs (one per
// SM).  Causal chunks of the backward pass need only part of each product, so
// a problem may restrict the first pair's k range by the tile's m rows (k up
// to the tile's last row, or from its first row) and skip tiles whose first
// column lies past the tile's last row.  The epilogue either scales and
// stores, or forms the score gradient dS = D * 2a sqrt(w) from the stored
// relu^2 weights w (0 past the causal diagonal) before it stores.
//
// Per CTA: K streamed in 64-deep stages through a four-slot ring [A 16 KB |
// B NT x 128 B], 128-byte swizzle; MMA M = 128, N = NT into one of two TMEM
// accumulators; eight epilogue warps each round a 32 x 32 box to bf16 into
// their own swizzled staging buffer and TMA-store it.  Warps: 0 scheduler + TMA, 1 MMA
// issuer, 2-9 epilogue.  Every barrier has one consumer; every wait is
// bounded.  Included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

constexpr int BG_RING = 4;
constexpr uint32_t BG_A_BYTES = 128 * 64 * 2;   // 16 KB
constexpr uint32_t BG_SLOT = 49152;
constexpr uint32_t BG_WSTAGE_BYTES = 32 * 32 * 2;  // one warp's 32 x 32 output box
constexpr uint32_t BG_OFF_STAGE = BG_RING * BG_SLOT;
constexpr int BG_QUEUE = 2;
constexpr int BG_EPI_WARPS = 8;
constexpr int BGEMM_THREADS = 64 + 32 * BG_EPI_WARPS;
constexpr uint32_t BGEMM_SMEM = BG_OFF_STAGE + BG_EPI_WARPS * 2 * BG_WSTAGE_BYTES + 1024;
constexpr int BG_MAX_PROBLEMS = 3;
static_assert(BGEMM_SMEM + 1024 <= 232448, "tc_bgemm exceeds 227 KB of shared memory");

// k range of the first operand pair for m tile mt
constexpr int BG_K_FULL = 0;     // all of K
constexpr int BG_K_TO_M = 1;     // k < 128 (mt + 1): keys up to the tile's last query
constexpr int BG_K_FROM_M = 2;   // k >= 128 mt: queries from the tile's first key
// epilogue
constexpr int BG_EPI_STORE = 0;  // D = alpha acc
constexpr int BG_EPI_SCORE = 1;  // D = acc * 2 alpha sqrt(w), w [batches*M][N]

struct BgProblem {
  CUtensorMap A, B, A2, B2, D;   // K-major A box {64, 128}, MN-major {64, 64};
                                 // K-major B box {64, nt}, MN-major {64, 64};
                                 // D [batches*M][N] box {32, 32}, 64-byte swizzle
  const __nv_bfloat16 *w;        // BG_EPI_SCORE weights (row-major like D)
  float alpha;
  int M, N, K, K2, batches, nt;
  int a_rpb, a_div, b_rpb, b_div, a2_rpb, a2_div, b2_rpb, b2_div;
  int a_mn, b_mn, a2_mn, b2_mn;
  int krange, skip_upper, epi, causal;
  int units;                     // batches * (M / 128) * (N / nt)
};
struct BgParams {
  BgProblem p[BG_MAX_PROBLEMS];
  int n_problems;
};

struct BgUnit {
  int pi, bt, mt, nt, k1_lo, n1, n_ks;
  bool skip;
};

// Unit u of the launch: its problem, batch, tiles and k steps; false past the end.
__device__ __forceinline__ bool bg_unit(const BgParams &P, int u, BgUnit &o) {
  int pi = 0;
  while (pi < P.n_problems && u >= P.p[pi].units) u -= P.p[pi++].units;
  if (pi >= P.n_problems) return false;
  const BgProblem &p = P.p[pi];
  const int n_nt = p.N / p.nt, per_batch = (p.M / 128) * n_nt;
  o.pi = pi;
  o.bt = u / per_batch;
  const int w = u % per_batch;
  o.mt = w / n_nt;
  o.nt = w % n_nt;
  int lo = 0, hi = p.K / 64;
  if (p.krange == BG_K_TO_M) hi = min(hi, 2 * (o.mt + 1));
  if (p.krange == BG_K_FROM_M) lo = 2 * o.mt;
  o.k1_lo = lo;
  o.n1 = hi > lo ? hi - lo : 0;
  o.n_ks = o.n1 + p.K2 / 64;
  o.skip = (p.skip_upper && o.nt * p.nt > o.mt * 128 + 127) || o.n_ks == 0;
  return true;
}

__global__ void __launch_bounds__(BGEMM_THREADS, 1) tc_bgemm(const __grid_constant__ BgParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[BG_RING], empty[BG_RING];
  __shared__ __align__(8) uint64_t q_full[BG_QUEUE], q_empty[BG_QUEUE];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ int q_unit[BG_QUEUE], acc_unit[2];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < BG_RING; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < BG_QUEUE; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 2);
      mbar_init(&acc_empty[i], BG_EPI_WARPS);
    }
    mbar_init(&mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  // launched as a programmatic dependent: the set-up above overlapped the
  // previous kernel's tail; nothing below runs before it has completed
  griddep_wait();

  if (warp == 0) {
    // =========================== scheduler + TMA producer
    if (lane == 0) {
      for (int i = 0; i < P.n_problems; ++i) {
        tma_prefetch_desc(&P.p[i].A);
        tma_prefetch_desc(&P.p[i].B);
        if (P.p[i].K2 > 0) {
          tma_prefetch_desc(&P.p[i].A2);
          tma_prefetch_desc(&P.p[i].B2);
        }
      }
      int it = 0, j = 0;
      bool ok = true;
      for (int c = 0; ok; ++c) {
        const int u = (int)blockIdx.x + c * (int)gridDim.x;
        BgUnit un;
        const bool valid = bg_unit(P, u, un);
        if (valid && un.skip) continue;
        const int qs = j % BG_QUEUE;
        if (j >= BG_QUEUE && !mbar_wait(&q_empty[qs], ((j / BG_QUEUE) - 1) & 1, kWaitLimitNs)) {
          record_timeout(700);
          break;
        }
        q_unit[qs] = valid ? u : -1;
        mbar_arrive(&q_full[qs]);
        ++j;
        if (!valid) break;
        const BgProblem &p = P.p[un.pi];
        const uint32_t bytes = BG_A_BYTES + (uint32_t)p.nt * 128u;
        const int a_row1 = (un.bt / p.a_div) * p.a_rpb, b_row1 = (un.bt / p.b_div) * p.b_rpb;
        const int a_row2 = (un.bt / p.a2_div) * p.a2_rpb, b_row2 = (un.bt / p.b2_div) * p.b2_rpb;
        for (int ks = 0; ks < un.n_ks; ++ks, ++it) {
          const int slot = it % BG_RING;
          if (it >= BG_RING && !mbar_wait(&empty[slot], ((it / BG_RING) - 1) & 1, kWaitLimitNs)) {
            record_timeout(701);
            ok = false;
            break;
          }
          const bool second = ks >= un.n1;
          const CUtensorMap *mA = second ? &p.A2 : &p.A, *mB = second ? &p.B2 : &p.B;
          const int kr = (second ? ks - un.n1 : un.k1_lo + ks) * 64;
          const int a_row0 = second ? a_row2 : a_row1, b_row0 = second ? b_row2 : b_row1;
          const bool a_mn = second ? p.a2_mn : p.a_mn, b_mn = second ? p.b2_mn : p.b_mn;
          uint8_t *sz = smem + slot * BG_SLOT;
          mbar_arrive_expect_tx(&full[slot], bytes);
          if (a_mn) {  // rows k, columns m: two 64-column boxes
            tma_load_2d(sz, mA, &full[slot], un.mt * 128, a_row0 + kr);
            tma_load_2d(sz + 8192, mA, &full[slot], un.mt * 128 + 64, a_row0 + kr);
          } else {     // rows m, columns k
            tma_load_2d(sz, mA, &full[slot], kr, a_row0 + un.mt * 128);
          }
          uint8_t *sb = sz + BG_A_BYTES;
          if (b_mn) {  // rows k, columns n: nt / 64 boxes of 64 columns
            for (int q = 0; q < p.nt / 64; ++q)
              tma_load_2d(sb + q * 8192, mB, &full[slot], un.nt * p.nt + 64 * q, b_row0 + kr);
          } else {     // rows n, columns k
            tma_load_2d(sb, mB, &full[slot], kr, b_row0 + un.nt * p.nt);
          }
        }
      }
      for (int q = (it > BG_RING ? it - BG_RING : 0); q < it; ++q)
        if (!mbar_wait(&full[q % BG_RING], (q / BG_RING) & 1, kWaitLimitNs)) record_timeout(702);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      int it = 0, j = 0;
      bool ok = true;
      for (;; ++j) {
        const int qs = j % BG_QUEUE;
        if (!mbar_wait(&q_full[qs], (j / BG_QUEUE) & 1, kWaitLimitNs)) {
          record_timeout(710);
          ok = false;
          break;
        }
        const int u = q_unit[qs];
        mbar_arrive(&q_empty[qs]);
        const int buf = j & 1, use = j >> 1;
        if (use >= 1 && !mbar_wait(&acc_empty[buf], (use - 1) & 1, kWaitLimitNs)) {
          record_timeout(711);
          ok = false;
          break;
        }
        if (u < 0) break;
        BgUnit un;
        bg_unit(P, u, un);
        const BgProblem &p = P.p[un.pi];
        const uint32_t id1 = idesc_bf16_f32(128, p.nt, p.a_mn, p.b_mn);
        const uint32_t id2 = idesc_bf16_f32(128, p.nt, p.a2_mn, p.b2_mn);
        tc_fence_after();
        const uint32_t dcol = tbase + (uint32_t)buf * 256u;
        for (int ks = 0; ks < un.n_ks; ++ks, ++it) {
          const int slot = it % BG_RING;
          if (!mbar_wait(&full[slot], (it / BG_RING) & 1, kWaitLimitNs)) {
            record_timeout(712);
            ok = false;
            break;
          }
          tc_fence_after();
          const bool second = ks >= un.n1;
          const bool a_mn = second ? p.a2_mn : p.a_mn, b_mn = second ? p.b2_mn : p.b_mn;
          const uint32_t idesc = second ? id2 : id1;
          const uint32_t sa = smem_u32(smem + slot * BG_SLOT);
          const uint32_t sb = sa + BG_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // K-major: the next 16 k are 32 bytes further along each 128-byte
            // row; MN-major: 16 k rows further, 2048 bytes (LBO: the stride
            // between 64-column boxes)
            const uint64_t ad = a_mn ? smem_desc_sw128(sa + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = b_mn ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 16, 1024);
            mma_bf16_ss(dcol, ad, bd, idesc, (ks | kk) != 0);
          }
          mma_commit(&empty[slot]);
        }
        if (!ok) break;
        acc_unit[buf] = u;
        mbar_arrive(&acc_full[buf]);
        mma_commit(&acc_full[buf]);
      }
      if (ok) {
        const int buf = j & 1;
        acc_unit[buf] = -1;
        mbar_arrive(&acc_full[buf]);
        mma_commit(&acc_full[buf]);
      }
      mma_commit(&mma_done);
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(713);
    }
  } else {
    // =========================== epilogue warps (256 threads)
    // Warp w reads TMEM lanes 32 (w % 4) .. (its 32 rows of the tile); the two
    // warps of each lane quarter take the two 32-column halves of every
    // 64-column piece.  Each warp stages its own 32 x 32 box (64-byte swizzle,
    // two buffers) and stores it with TMA itself: no barrier across warps.
    const int ew = warp - 2;  // 0..7
    const int quad = warp & 3, half = ew / 4;
    const int row = quad * 32 + lane;
    uint8_t *wst = smem + BG_OFF_STAGE + ew * 2 * BG_WSTAGE_BYTES;
    int nst = 0;
    for (int j = 0;; ++j) {
      const int buf = j & 1, use = j >> 1;
      const bool got = mbar_wait(&acc_full[buf], use & 1, kWaitLimitNs);
      if (!got) {
        if (lane == 0) record_timeout(720);
        break;
      }
      const int u = acc_unit[buf];
      if (u < 0) break;
      tc_fence_after();
      BgUnit un;
      bg_unit(P, u, un);
      const BgProblem &p = P.p[un.pi];
      const bool score = p.epi == BG_EPI_SCORE;
      const int qi = un.mt * 128 + row;  // query row within the chunk (score epilogue)
      const __nv_bfloat16 *wrow = p.w + ((int64_t)un.bt * p.M + qi) * p.N;
      const float two_a = 2.f * p.alpha;
      const uint32_t dcol =
          tbase + (uint32_t)buf * 256u + (uint32_t)(half * 32) + ((uint32_t)(quad * 32) << 16);
      const int nq = p.nt / 64;
      const int drow = un.bt * p.M + un.mt * 128 + quad * 32;
      for (int q = 0; q < nq; ++q, ++nst) {
        uint8_t *sb = wst + (nst & 1) * BG_WSTAGE_BYTES;
        if (nst >= 2) {  // the store from this buffer two pieces ago has read it
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
        }
        uint32_t r[32];
        tmem_ld32(dcol + q * 64, r);
        const int j0 = un.nt * p.nt + q * 64 + half * 32;  // first column of this box
        uint4 wv[4];
        const bool any = score && (!p.causal || j0 <= qi);
        if (any) {
#pragma unroll
          for (int v = 0; v < 4; ++v) wv[v] = __ldg(reinterpret_cast<const uint4 *>(wrow + j0) + v);
        }
        tmem_ld_wait();
        if (q == nq - 1) {  // this warp's last read of the accumulator
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const uint32_t *v = r + 8 * j4;
          float x[8];
          if (score) {
            const uint4 w4 = any ? wv[j4] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int key = j0 + 8 * j4 + i;
              const float wt = (i & 1) ? bf16_hi(ww[i / 2]) : bf16_lo(ww[i / 2]);
              // sqrt(w) = w * w^-1/2 for w > 0 (relu^2 weights are >= 0)
              const bool keep = any && wt > 0.f && (!p.causal || key <= qi);
              x[i] = keep ? __uint_as_float(v[i]) * two_a * (wt * rsqrtf(wt)) : 0.f;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = p.alpha * __uint_as_float(v[i]);
          }
          *reinterpret_cast<uint4 *>(sb + sw64_offset(lane, 16 * j4)) =
              make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                         pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.D, sb, j0, drow);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }
  // the single-lane roles (TMA producer, MMA issuer) rejoin their warps
  // before the block-wide barrier, which counts converged warps
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace
}  // namespace fmca
