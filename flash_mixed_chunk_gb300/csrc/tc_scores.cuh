// tc_scores.cuh -- intra-chunk relu^2 weights and the lin_q rows, per
// (chunk, 128-row tile):
//     P  = relu(T0 T1^T / C)^2, strict upper triangle masked in causal mode
//     T2 = Z * gamma[2] + beta[2]
// ("FLASH: Possibly the Most Interesting Efficient Transformer Design Recently",
// section "Weak Attention" for the affine maps, section "Mixed Chunk" for the
// intra-chunk weights and the decoder mask.)  Both are written to the
// workspace in bf16 -- P as [B*n rows][C keys] (query row-major), T2 as
// [B*n][s] -- for the streaming attention kernel.  Included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

// shared memory: [0, 64K) Z tile of the chunk's keys (K-major, atom a = s
// columns 64a..64a+63 at a*32K, 256 rows x 128 B), turned into T1 in place,
// then overwritten by P (key atom k at k*16K, 128 rows x 128 B);
// [64K, 96K) T0 rows; [96K, 128K) T2 rows.
constexpr uint32_t SC_OFF_T0 = 65536, SC_OFF_T2 = 98304;
constexpr uint32_t SC_SMEM = 131072 + 1024;
constexpr int SC_THREADS = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 math

__global__ void __launch_bounds__(SC_THREADS, 1)
    tc_chunk_scores(const __grid_constant__ CUtensorMap mapZ,   // Z [B*n][s], box {64,128}
                    const __grid_constant__ CUtensorMap mapPw,  // P [B*n][C], box {64,128}
                    const __grid_constant__ CUtensorMap mapT2,  // T2 [B*n][s], box {64,128}
                    const float *__restrict__ gamma, const float *__restrict__ beta,
                    unsigned int *__restrict__ state_sched, int n, int C, int G, int causal) {
  // the state kernel that follows on the stream hands out work from here
  if (blockIdx.x == 0 && threadIdx.x == 0) *state_sched = 0u;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t zfull, tready, sfull;
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int R = C / ROW_TILE;
  const int rt = blockIdx.x % R;
  const int bg = blockIdx.x / R;
  const int b = bg / G, g = bg % G;
  const int keys_n = causal ? (rt + 1) * ROW_TILE : C;
  const int chunk_row = b * n + g * C;
  const int row0 = chunk_row + rt * ROW_TILE;

  if (threadIdx.x == 0) {
    mbar_init(&zfull, 1);
    mbar_init(&tready, 1);
    mbar_init(&sfull, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  uint8_t *zt = smem;
  uint8_t *t0 = smem + SC_OFF_T0;
  uint8_t *t2 = smem + SC_OFF_T2;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mapZ);
      mbar_arrive_expect_tx(&zfull, (uint32_t)keys_n * S_DIM * 2);
      for (int kh = 0; kh < keys_n / ROW_TILE; ++kh)
        for (int a = 0; a < 2; ++a)
          tma_load_2d(zt + a * 32768 + kh * 16384, &mapZ, &zfull, 64 * a,
                      chunk_row + ROW_TILE * kh);
      if (!mbar_wait(&zfull, 0, kWaitLimitNs)) record_timeout(301);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (mbar_wait(&tready, 0, kWaitLimitNs)) {
        tc_fence_after();
        // S[128 rows][keys] = T0 T1^T, both K-major, K = s
        const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)keys_n, false, false);
        const uint32_t a0 = smem_u32(t0), b0 = smem_u32(zt);
        for (int j = 0; j < S_DIM / 16; ++j) {
          const uint64_t ad = smem_desc_sw128(a0 + (j >> 2) * 16384 + (j & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(b0 + (j >> 2) * 32768 + (j & 3) * 32, 16, 1024);
          mma_bf16_ss(tbase, ad, bd, idesc, j > 0);
        }
      } else {
        record_timeout(302);
      }
      // sfull completes once every MMA issued above has finished (also on
      // the timeout path, where none was issued), so TMEM may be released
      mma_commit(&sfull);
      if (!mbar_wait(&sfull, 0, kWaitLimitNs)) record_timeout(303);
    }
  } else {
    // ---------------- math warps: affine maps, then P
    const int mt = threadIdx.x - 64;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int ro = rt * ROW_TILE;
    // every 16-byte chunk this thread touches sits at physical chunk position
    // p = mt % 8 of rows r with r % 8 = (mt / 8) % 8, so it covers logical
    // columns c_a = 64 a + 8 (p ^ (r % 8)) for the two atoms a = 0, 1
    const int p = mt & 7, rbase = mt >> 3;
    const int cl = ((p ^ (rbase & 7)) << 3);
    float g0[2][8], b0[2][8], g1[2][8], b1[2][8], g2[2][8], b2[2][8];
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      load8(gamma + a * 64 + cl, g0[a]);
      load8(beta + a * 64 + cl, b0[a]);
      load8(gamma + S_DIM + a * 64 + cl, g1[a]);
      load8(beta + S_DIM + a * 64 + cl, b1[a]);
      load8(gamma + 2 * S_DIM + a * 64 + cl, g2[a]);
      load8(beta + 2 * S_DIM + a * 64 + cl, b2[a]);
    }
    bool got = mbar_wait(&zfull, 0, kWaitLimitNs);
    if (got) {
#pragma unroll
      for (int a = 0; a < 2; ++a)
        for (int i = 0; i < ROW_TILE / 16; ++i) {
          const int r = rbase + 16 * i;
          const uint4 v = *reinterpret_cast<const uint4 *>(zt + a * 32768 + (ro + r) * 128 + p * 16);
          *reinterpret_cast<uint4 *>(t0 + a * 16384 + r * 128 + p * 16) = affine8(v, g0[a], b0[a]);
          *reinterpret_cast<uint4 *>(t2 + a * 16384 + r * 128 + p * 16) = affine8(v, g2[a], b2[a]);
        }
    }
    bool ok = named_bar_and(1, 128, got);
    if (ok) {
      // T1 in place over the keys (after every thread has read its T0/T2 rows)
#pragma unroll
      for (int a = 0; a < 2; ++a)
        for (int i = 0; i < keys_n / 16; ++i) {
          uint4 *ptr = reinterpret_cast<uint4 *>(zt + a * 32768 + (rbase + 16 * i) * 128 + p * 16);
          *ptr = affine8(*ptr, g1[a], b1[a]);
        }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (mt == 0) {
        mbar_arrive(&tready);
        // T2 rows out (generic-proxy writes fenced above)
        for (int a = 0; a < 2; ++a) tma_store_2d(&mapT2, t2 + a * 16384, 64 * a, row0);
        bulk_commit_group();
      }
      __syncwarp();
      got = mbar_wait(&sfull, 0, kWaitLimitNs);
      if (got) {
        tc_fence_after();
        const float inv_c = 1.0f / (float)C;
        const int qpos = ro + row;  // this row's position among the chunk's keys
        for (int kc = 0; kc < keys_n / 32; ++kc) {
          uint32_t r[32];
          tmem_ld32(tbase + ((uint32_t)(quad * 32) << 16) + kc * 32, r);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int k0 = kc * 32 + 2 * i;
            float x0 = fmaxf(__uint_as_float(r[2 * i]) * inv_c, 0.f);
            float x1 = fmaxf(__uint_as_float(r[2 * i + 1]) * inv_c, 0.f);
            x0 = x0 * x0;
            x1 = x1 * x1;
            if (causal) {
              if (k0 > qpos) x0 = 0.f;
              if (k0 + 1 > qpos) x1 = 0.f;
            }
            pk[i] = pack_bf16x2(x0, x1);
          }
          uint8_t *patom = zt + (kc >> 1) * 16384;
          const uint32_t byte0 = (kc & 1) * 64;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4 *>(patom + sw128_offset(row, byte0 + 16 * q)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      ok = named_bar_and(1, 128, got);
      if (mt == 0) {
        if (ok) {
          for (int ka = 0; ka < keys_n / 64; ++ka)
            tma_store_2d(&mapPw, zt + ka * 16384, 64 * ka, row0);
          bulk_commit_group();
        } else {
          record_timeout(304);
        }
        bulk_wait_group<0>();
      }
      __syncwarp();
    } else if (mt == 0) {
      record_timeout(305);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 256);
}

}  // namespace
}  // namespace fmca
