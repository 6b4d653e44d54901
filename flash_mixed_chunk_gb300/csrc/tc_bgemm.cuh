// tc_bgemm.cuh -- batched products of the backward pass on the tensor cores.
//
//   D_b = alpha * A_b B_b   for b < batches, bf16 in, fp32 accumulate, bf16 out
//
// with A_b [M][K] and B_b [K][N] read from row-major bf16 arrays either
// K-major (A stored [m][k], B stored [n][k]) or MN-major (A stored [k][m], B
// stored [k][n]).  Operand rows of batch b start at (b / div) * rows_per_batch
// (div > 1 lets consecutive batches share an operand, e.g. every chunk of a
// sequence reading one state matrix); D_b occupies rows b * M .. of D [rows][N].
// M and K are multiples of 128 and 64, N a multiple of the N tile, so that no
// tile reaches into another batch's rows.  A second operand pair (A2 [M][K2],
// B2 [K2][N], same majorness) may extend the contraction:
// D_b = alpha (A_b B_b + A2_b B2_b), one accumulator for both.
//
// Persistent kernel, one CTA per SM, tiles (batch, 128-row tile, NT-column
// tile) dealt round-robin; K streamed in 64-deep stages through a four-slot
// ring [A 16 KB | B NT x 128 B], 128-byte swizzle; MMA M = 128, N = NT into one
// of two TMEM accumulators; four epilogue warps scale, round to bf16 into a
// swizzled staging tile and TMA-store 64-column pieces.  Warps: 0 scheduler +
// TMA, 1 MMA issuer, 2-5 epilogue.  Every barrier has one consumer; every wait
// is bounded.  Included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

constexpr int BG_RING = 4;
constexpr uint32_t BG_A_BYTES = 128 * 64 * 2;   // 16 KB
constexpr uint32_t BG_SLOT = 49152;
constexpr int BG_STAGE_BUFS = 2;
constexpr uint32_t BG_STAGE_BYTES = 128 * 64 * 2;
constexpr uint32_t BG_OFF_STAGE = BG_RING * BG_SLOT;
constexpr uint32_t BGEMM_SMEM = BG_OFF_STAGE + BG_STAGE_BUFS * BG_STAGE_BYTES + 1024;
constexpr int BG_QUEUE = 2;
constexpr int BGEMM_THREADS = 192;
static_assert(BGEMM_SMEM + 1024 <= 232448, "tc_bgemm exceeds 227 KB of shared memory");

struct BgShape {
  int M, N, K, batches;
  int a_rpb, a_div;   // operand rows per batch step and batch divisor
  int b_rpb, b_div;
  float alpha;
  int K2 = 0;         // depth of the second operand pair (0: none)
  int a2_rpb = 0, a2_div = 1, b2_rpb = 0, b2_div = 1;
};

template <bool A_MN, bool B_MN, int NT>
__global__ void __launch_bounds__(BGEMM_THREADS, 1)
    tc_bgemm(const __grid_constant__ CUtensorMap mapA,  // K-major: box {64, 128}; MN: {64, 64}
             const __grid_constant__ CUtensorMap mapB,  // K-major: box {64, NT}; MN: {64, 64}
             const __grid_constant__ CUtensorMap mapD,  // D [batches*M][N], box {64, 128}
             const __grid_constant__ CUtensorMap mapA2,  // as mapA, for k >= K
             const __grid_constant__ CUtensorMap mapB2,  // as mapB, for k >= K
             const BgShape sh) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[BG_RING], empty[BG_RING];
  __shared__ __align__(8) uint64_t q_full[BG_QUEUE], q_empty[BG_QUEUE];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ int q_unit[BG_QUEUE], acc_unit[2];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_mt = sh.M / 128, n_nt = sh.N / NT;
  const int per_batch = n_mt * n_nt;
  const int n_units = sh.batches * per_batch;
  const int n_k1 = sh.K / 64, n_ks = n_k1 + sh.K2 / 64;

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
      mbar_init(&acc_empty[i], 1);
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

  if (warp == 0) {
    // =========================== scheduler + TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapB);
      if (sh.K2 > 0) {
        tma_prefetch_desc(&mapA2);
        tma_prefetch_desc(&mapB2);
      }
      int it = 0;
      bool ok = true;
      constexpr uint32_t B_BYTES = NT * 64 * 2;
      for (int i = 0; ok; ++i) {
        const int u = (int)blockIdx.x + i * (int)gridDim.x;
        const int uu = u < n_units ? u : -1;
        const int qs = i % BG_QUEUE;
        if (i >= BG_QUEUE && !mbar_wait(&q_empty[qs], ((i / BG_QUEUE) - 1) & 1, kWaitLimitNs)) {
          record_timeout(700);
          break;
        }
        q_unit[qs] = uu;
        mbar_arrive(&q_full[qs]);
        if (uu < 0) break;
        const int bt = uu / per_batch, w = uu % per_batch;
        const int mt = w / n_nt, nt = w % n_nt;
        const int a_row1 = (bt / sh.a_div) * sh.a_rpb, b_row1 = (bt / sh.b_div) * sh.b_rpb;
        const int a_row2 = (bt / sh.a2_div) * sh.a2_rpb, b_row2 = (bt / sh.b2_div) * sh.b2_rpb;
        for (int ks = 0; ks < n_ks; ++ks, ++it) {
          const bool second = ks >= n_k1;
          const CUtensorMap *mA = second ? &mapA2 : &mapA, *mB = second ? &mapB2 : &mapB;
          const int kr = (second ? ks - n_k1 : ks) * 64;
          const int a_row0 = second ? a_row2 : a_row1, b_row0 = second ? b_row2 : b_row1;
          const int slot = it % BG_RING;
          if (it >= BG_RING && !mbar_wait(&empty[slot], ((it / BG_RING) - 1) & 1, kWaitLimitNs)) {
            record_timeout(701);
            ok = false;
            break;
          }
          uint8_t *sz = smem + slot * BG_SLOT;
          mbar_arrive_expect_tx(&full[slot], BG_A_BYTES + B_BYTES);
          if (A_MN) {  // rows k, columns m: two 64-column boxes
            tma_load_2d(sz, mA, &full[slot], mt * 128, a_row0 + kr);
            tma_load_2d(sz + 8192, mA, &full[slot], mt * 128 + 64, a_row0 + kr);
          } else {     // rows m, columns k
            tma_load_2d(sz, mA, &full[slot], kr, a_row0 + mt * 128);
          }
          uint8_t *sb = sz + BG_A_BYTES;
          if (B_MN) {  // rows k, columns n: NT / 64 boxes of 64 columns
            for (int j = 0; j < NT / 64; ++j)
              tma_load_2d(sb + j * 8192, mB, &full[slot], nt * NT + 64 * j, b_row0 + kr);
          } else {     // rows n, columns k
            tma_load_2d(sb, mB, &full[slot], kr, b_row0 + nt * NT);
          }
        }
      }
      for (int q = (it > BG_RING ? it - BG_RING : 0); q < it; ++q)
        if (!mbar_wait(&full[q % BG_RING], (q / BG_RING) & 1, kWaitLimitNs)) record_timeout(702);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NT, A_MN, B_MN);
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
        tc_fence_after();
        const uint32_t dcol = tbase + (uint32_t)buf * 256u;
        for (int ks = 0; ks < n_ks; ++ks, ++it) {
          const int slot = it % BG_RING;
          if (!mbar_wait(&full[slot], (it / BG_RING) & 1, kWaitLimitNs)) {
            record_timeout(712);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + slot * BG_SLOT);
          const uint32_t sb = sa + BG_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // K-major: the next 16 k are 32 bytes further along each 128-byte
            // row; MN-major: 16 k rows further, 2048 bytes (LBO: the stride
            // between 64-column boxes)
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
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
    // =========================== epilogue warps (128 threads)
    const int mt_ = threadIdx.x - 64;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    uint8_t *stage = smem + BG_OFF_STAGE;
    int nst = 0;
    for (int j = 0;; ++j) {
      const int buf = j & 1, use = j >> 1;
      const bool got = mbar_wait(&acc_full[buf], use & 1, kWaitLimitNs);
      const int u = got ? acc_unit[buf] : -1;
      if (!named_bar_and(1, 128, u >= 0)) {
        if (!got && mt_ == 0) record_timeout(720);
        break;
      }
      tc_fence_after();
      const int bt = u / per_batch, w = u % per_batch;
      const int mt = w / n_nt, nt = w % n_nt;
      const uint32_t dcol = tbase + (uint32_t)buf * 256u + ((uint32_t)(quad * 32) << 16);
      for (int q = 0; q < NT / 64; ++q, ++nst) {
        uint8_t *sb = stage + (nst % BG_STAGE_BUFS) * BG_STAGE_BYTES;
        if (mt_ == 0 && nst >= BG_STAGE_BUFS) bulk_wait_group_read<BG_STAGE_BUFS - 1>();
        named_bar_sync(1, 128);
        uint32_t r[2][32];
        tmem_ld32(dcol + q * 64, r[0]);
        tmem_ld32(dcol + q * 64 + 32, r[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const uint32_t *v = r[c2] + 8 * j4;
            const float a = sh.alpha;
            *reinterpret_cast<uint4 *>(sb + sw128_offset(row, c2 * 64 + 16 * j4)) = make_uint4(
                pack_bf16x2(a * __uint_as_float(v[0]), a * __uint_as_float(v[1])),
                pack_bf16x2(a * __uint_as_float(v[2]), a * __uint_as_float(v[3])),
                pack_bf16x2(a * __uint_as_float(v[4]), a * __uint_as_float(v[5])),
                pack_bf16x2(a * __uint_as_float(v[6]), a * __uint_as_float(v[7])));
          }
        fence_proxy_async_smem();
        if (q == NT / 64 - 1) tc_fence_before();
        named_bar_sync(1, 128);
        if (mt_ == 0) {
          tma_store_2d(&mapD, sb, nt * NT + q * 64, bt * sh.M + mt * 128);
          bulk_commit_group();
          if (q == NT / 64 - 1) mbar_arrive(&acc_empty[buf]);
        }
        __syncwarp();
      }
    }
    if (mt_ == 0) bulk_wait_group<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace
}  // namespace fmca
