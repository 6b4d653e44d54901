// tc_gemm.cuh -- the dense projections around the attention core ("FLASH:
// Possibly the Most Interesting Efficient Transformer Design Recently":
// section "Initial Power", U = phi(X W_u), V = phi(X W_v) with phi = Swish;
// section "Weak Attention", Z = phi(X W_z); section "Strong Combination",
// eq. mix, the layer output (U * A V) W_o):
//
//   D = act(A B^T), A [M][K] bf16, B [N][K] bf16 (one row per output
//   feature), act = SiLU or identity, D's columns split over up to three
//   row-major bf16 outputs by column range.
//
// Persistent kernel, one CTA per SM; a unit is a 128 x 256 tile of D, dealt
// round-robin (CTA c takes tiles c, c + grid, ...: the tiles are uniform, and
// no scratch memory is needed).  Each unit streams K in
// 64-element stages through a four-slot ring of 48 KB items [A: 128 rows x 64
// (16 KB) | B: 256 rows x 64 (32 KB)], both operands K-major with the 128-byte
// swizzle, and accumulates D into one of two TMEM accumulators (M = 128,
// N = 256); four epilogue warps apply the activation, round to bf16 into a
// swizzled staging tile and store each 64-column piece with TMA into the
// output its columns belong to.  Warps: 0 scheduler + TMA, 1 MMA issuer, 2-5
// epilogue.  Every barrier has one consumer; every wait is bounded.
// Included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

constexpr int GM_RING = 4;
constexpr uint32_t GM_A_BYTES = 128 * 64 * 2;   // 16 KB
constexpr uint32_t GM_SLOT = 49152;             // A | B (32 KB)
constexpr int GM_STAGE_BUFS = 2;
constexpr uint32_t GM_STAGE_BYTES = 128 * 64 * 2;
constexpr uint32_t GM_OFF_STAGE = GM_RING * GM_SLOT;
constexpr uint32_t GEMM_SMEM = GM_OFF_STAGE + GM_STAGE_BUFS * GM_STAGE_BYTES + 1024;
constexpr int GM_QUEUE = 2;
constexpr int GEMM_THREADS = 192;
constexpr int GM_TILE_N = 256;
static_assert(GEMM_SMEM + 1024 <= 232448, "tc_gemm exceeds 227 KB of shared memory");

enum : int { GEMM_ACT_NONE = 0, GEMM_ACT_SILU = 1 };

// x * sigmoid(x), with the fast exponential and division intrinsics (the
// epilogue runs one per output element and must keep pace with the MMAs)
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

template <int ACT>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    tc_gemm(const __grid_constant__ CUtensorMap mapA,   // A [M][K], box {64, 128}
            const __grid_constant__ CUtensorMap mapB,   // B [N][K], box {64, 256}
            const __grid_constant__ CUtensorMap mapD0,  // columns [0, n0), box {64, 128}
            const __grid_constant__ CUtensorMap mapD1,  // columns [n0, n1)
            const __grid_constant__ CUtensorMap mapD2,  // columns [n1, N)
            int M, int N, int K, int n0, int n1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[GM_RING], empty[GM_RING];
  __shared__ __align__(8) uint64_t q_full[GM_QUEUE], q_empty[GM_QUEUE];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ int q_unit[GM_QUEUE], acc_unit[2];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_mt = (M + 127) / 128, n_nt = (N + GM_TILE_N - 1) / GM_TILE_N;
  const int n_units = n_mt * n_nt;
  const int n_ks = (K + 63) / 64;

  if (threadIdx.x == 0) {
    for (int i = 0; i < GM_RING; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < GM_QUEUE; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 2);  // tcgen05.commit + the MMA thread's arrive
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
      int it = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int u = (int)blockIdx.x + i * (int)gridDim.x;
        const int uu = u < n_units ? u : -1;
        const int qs = i % GM_QUEUE;
        if (i >= GM_QUEUE && !mbar_wait(&q_empty[qs], ((i / GM_QUEUE) - 1) & 1, kWaitLimitNs)) {
          record_timeout(600);
          break;
        }
        q_unit[qs] = uu;
        mbar_arrive(&q_full[qs]);
        if (uu < 0) break;
        const int mt = uu / n_nt, nt = uu % n_nt;
        for (int ks = 0; ks < n_ks; ++ks, ++it) {
          const int slot = it % GM_RING;
          if (it >= GM_RING && !mbar_wait(&empty[slot], ((it / GM_RING) - 1) & 1, kWaitLimitNs)) {
            record_timeout(601);
            ok = false;
            break;
          }
          uint8_t *sz = smem + slot * GM_SLOT;
          // out-of-range rows and K columns arrive as zeros; the full boxes count
          mbar_arrive_expect_tx(&full[slot], GM_SLOT);
          tma_load_2d(sz, &mapA, &full[slot], ks * 64, mt * 128);
          tma_load_2d(sz + GM_A_BYTES, &mapB, &full[slot], ks * 64, nt * GM_TILE_N);
        }
      }
      // wait (bounded) for the last copy issued into each slot
      for (int q = (it > GM_RING ? it - GM_RING : 0); q < it; ++q)
        if (!mbar_wait(&full[q % GM_RING], (q / GM_RING) & 1, kWaitLimitNs)) record_timeout(602);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      // D[128][256] += A[128][k] B[256][k]^T, both K-major
      constexpr uint32_t idesc = idesc_bf16_f32(128, GM_TILE_N, false, false);
      int it = 0, j = 0;
      bool ok = true;
      for (;; ++j) {
        const int qs = j % GM_QUEUE;
        if (!mbar_wait(&q_full[qs], (j / GM_QUEUE) & 1, kWaitLimitNs)) {
          record_timeout(610);
          ok = false;
          break;
        }
        const int u = q_unit[qs];
        mbar_arrive(&q_empty[qs]);
        const int buf = j & 1, use = j >> 1;
        if (use >= 1 && !mbar_wait(&acc_empty[buf], (use - 1) & 1, kWaitLimitNs)) {
          record_timeout(611);
          ok = false;
          break;
        }
        if (u < 0) break;
        tc_fence_after();
        const uint32_t dcol = tbase + (uint32_t)buf * 256u;
        for (int ks = 0; ks < n_ks; ++ks, ++it) {
          const int slot = it % GM_RING;
          if (!mbar_wait(&full[slot], (it / GM_RING) & 1, kWaitLimitNs)) {
            record_timeout(612);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + slot * GM_SLOT);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(sa + GM_A_BYTES + kk * 32, 16, 1024);
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
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(613);
    }
  } else {
    // =========================== epilogue warps (128 threads)
    const int mt_ = threadIdx.x - 64;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // TMEM lane = tile row
    uint8_t *stage = smem + GM_OFF_STAGE;
    int nst = 0;
    for (int j = 0;; ++j) {
      const int buf = j & 1, use = j >> 1;
      const bool got = mbar_wait(&acc_full[buf], use & 1, kWaitLimitNs);
      const int u = got ? acc_unit[buf] : -1;
      if (!named_bar_and(1, 128, u >= 0)) {
        if (!got && mt_ == 0) record_timeout(620);
        break;
      }
      tc_fence_after();
      const int mt = u / n_nt, nt = u % n_nt;
      const uint32_t dcol = tbase + (uint32_t)buf * 256u + ((uint32_t)(quad * 32) << 16);
      for (int q = 0; q < GM_TILE_N / 64; ++q) {
        const int col = nt * GM_TILE_N + q * 64;
        if (col >= N) {  // past the last output column (uniform across the warps)
          if (q == GM_TILE_N / 64 - 1 || col + 64 >= N) {
            tc_fence_before();
            named_bar_sync(1, 128);
            if (mt_ == 0) mbar_arrive(&acc_empty[buf]);
            break;
          }
          continue;
        }
        uint8_t *sb = stage + (nst % GM_STAGE_BUFS) * GM_STAGE_BYTES;
        if (mt_ == 0 && nst >= GM_STAGE_BUFS) bulk_wait_group_read<GM_STAGE_BUFS - 1>();
        named_bar_sync(1, 128);
        uint32_t r[2][32];
        tmem_ld32(dcol + q * 64, r[0]);
        tmem_ld32(dcol + q * 64 + 32, r[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float x = __uint_as_float(r[c2][8 * j4 + i]);
              v[i] = ACT == GEMM_ACT_SILU ? silu_f(x) : x;
            }
            *reinterpret_cast<uint4 *>(sb + sw128_offset(row, c2 * 64 + 16 * j4)) =
                make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                           pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
          }
        fence_proxy_async_smem();
        const bool last = q == GM_TILE_N / 64 - 1 || col + 64 >= N;
        if (last) tc_fence_before();
        named_bar_sync(1, 128);
        if (mt_ == 0) {
          if (col < n0)
            tma_store_2d(&mapD0, sb, col, mt * 128);
          else if (col < n1)
            tma_store_2d(&mapD1, sb, col - n0, mt * 128);
          else
            tma_store_2d(&mapD2, sb, col - n1, mt * 128);
          bulk_commit_group();
          if (last) mbar_arrive(&acc_empty[buf]);
        }
        __syncwarp();
        ++nst;
        if (last) break;
      }
    }
    if (mt_ == 0) bulk_wait_group<0>();
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
