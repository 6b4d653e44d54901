// tc_state.cuh -- per-chunk linear-attention states and their chunk-axis
// prefix (included by tc.cu; device code of the tensor-core path).
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

// =====================================================================
// tc_chunk_state: one CTA per (b, g, 256-column slice of e)
// =====================================================================
// shared memory: NSLOT_STATE slots of [Z: 64 keys x 128 s (2 boxes of 8 KB)]
//                                   + [V: 64 keys x 256 e (4 boxes of 8 KB)]
constexpr int STATE_NSLOT = 2;
constexpr uint32_t STATE_Z_BYTES = KEY_STAGE * S_DIM * 2;      // 16 KB
constexpr uint32_t STATE_V_BYTES = KEY_STAGE * E_TILE * 2;     // 32 KB
constexpr uint32_t STATE_SLOT = STATE_Z_BYTES + STATE_V_BYTES; // 48 KB
constexpr uint32_t STATE_SMEM = STATE_NSLOT * STATE_SLOT + 1024;
constexpr int STATE_THREADS = 192;  // warp0 TMA, warp1 MMA, warps 2-5 math

__global__ void __launch_bounds__(STATE_THREADS, 1)
    tc_chunk_state(const __grid_constant__ CUtensorMap mapZ,   // box {64, 64}
                   const __grid_constant__ CUtensorMap mapV,   // box {64, 64}
                   const float *__restrict__ gamma, const float *__restrict__ beta,
                   float *__restrict__ states, int n, int e, int C, int G) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[STATE_NSLOT], tready[STATE_NSLOT], empty[STATE_NSLOT];
  __shared__ __align__(8) uint64_t dfull, mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ float g3[S_DIM], b3[S_DIM];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_es = e / E_TILE;
  const int es = blockIdx.x % n_es;
  const int bg = blockIdx.x / n_es;
  const int b = bg / G, g = bg % G;
  const int e0 = es * E_TILE;
  const int row0 = b * n + g * C;
  const int nstage = C / KEY_STAGE;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STATE_NSLOT; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&tready[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&dfull, 1);
    mbar_init(&mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i < S_DIM; i += STATE_THREADS) {
    g3[i] = gamma[3 * S_DIM + i];
    b3[i] = beta[3 * S_DIM + i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mapZ);
      tma_prefetch_desc(&mapV);
      int issued = 0;
      for (int q = 0; q < nstage; ++q) {
        const int slot = q % STATE_NSLOT;
        if (q >= STATE_NSLOT) {
          if (!mbar_wait(&empty[slot], ((q / STATE_NSLOT) - 1) & 1, kWaitLimitNs)) {
            record_timeout(101);
            break;
          }
        }
        uint8_t *sz = smem + slot * STATE_SLOT;
        uint8_t *sv = sz + STATE_Z_BYTES;
        mbar_arrive_expect_tx(&full[slot], STATE_SLOT);
        const int y = row0 + q * KEY_STAGE;
        tma_load_2d(sz, &mapZ, &full[slot], 0, y);
        tma_load_2d(sz + 8192, &mapZ, &full[slot], 64, y);
        for (int i = 0; i < 4; ++i) tma_load_2d(sv + i * 8192, &mapV, &full[slot], e0 + 64 * i, y);
        issued = q + 1;
      }
      // drain: every issued stage has landed before this CTA may exit
      for (int q = (issued > STATE_NSLOT ? issued - STATE_NSLOT : 0); q < issued; ++q)
        if (!mbar_wait(&full[q % STATE_NSLOT], (q / STATE_NSLOT) & 1, kWaitLimitNs))
          record_timeout(102);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      // D_h^T[e][s] += V^T[e][k] * T3[k][s]   (A: V tile, MN-major;
      // B: T3 tile, MN-major), M = 128 (e), N = 128 (s), K = 16 keys per op.
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, true, true);
      bool ok = true;
      for (int q = 0; q < nstage && ok; ++q) {
        const int slot = q % STATE_NSLOT;
        if (!mbar_wait(&tready[slot], (q / STATE_NSLOT) & 1, kWaitLimitNs)) {
          record_timeout(103);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sz = smem_u32(smem + slot * STATE_SLOT);
        const uint32_t sv = sz + STATE_Z_BYTES;
        for (int kk = 0; kk < KEY_STAGE / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(sz + kk * 2048, 8192, 1024);
          for (int h = 0; h < 2; ++h) {
            const uint64_t adesc = smem_desc_sw128(sv + h * 16384 + kk * 2048, 8192, 1024);
            mma_bf16_ss(tbase + h * 128, adesc, bdesc, idesc, (q | kk) != 0);
          }
        }
        mma_commit(&empty[slot]);
      }
      mma_commit(&dfull);
      // every MMA has finished before TMEM is released
      mma_commit(&mma_done);
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(106);
    }
  } else {
    // ---------------- math warps: T3 in place, then the epilogue
    const int mt = threadIdx.x - 64;  // 0..127
    bool ok = true;
    for (int q = 0; q < nstage; ++q) {
      const int slot = q % STATE_NSLOT;
      const bool got = mbar_wait(&full[slot], (q / STATE_NSLOT) & 1, kWaitLimitNs);
      if (got) {
        uint8_t *sz = smem + slot * STATE_SLOT;
        // 2 boxes x 64 rows x 8 chunks of 16 B = 1024 chunks
        for (int x = mt; x < 1024; x += 128) {
          const int box = x >> 9, r = (x >> 3) & 63, p = x & 7;
          uint4 *ptr = reinterpret_cast<uint4 *>(sz + box * 8192 + r * 128 + p * 16);
          uint4 v = *ptr;
          const int c = box * 64 + ((p ^ (r & 7)) << 3);
          uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float lo = bf16_lo(w[i]) * g3[c + 2 * i] + b3[c + 2 * i];
            float hi = bf16_hi(w[i]) * g3[c + 2 * i + 1] + b3[c + 2 * i + 1];
            w[i] = pack_bf16x2(lo, hi);
          }
          *ptr = make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
      }
      ok = named_bar_and(1, 128, got);
      if (!ok) {
        if (mt == 0) record_timeout(104);
        break;
      }
      if (mt == 0) mbar_arrive(&tready[slot]);
    }
    // epilogue: thread = e row of D^T, 2 halves x 4 chunks of 32 s columns
    if (ok && mbar_wait(&dfull, 0, kWaitLimitNs)) {
      tc_fence_after();
      const int quad = warp & 3;
      const int e_idx = e0 + quad * 32 + lane;
      float *dst = states + (size_t)bg * S_DIM * e;
      for (int h = 0; h < 2; ++h) {
        for (int c = 0; c < S_DIM / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tbase + ((uint32_t)(quad * 32) << 16) + h * 128 + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            dst[(size_t)(c * 32 + i) * e + e_idx + h * 128] = __uint_as_float(r[i]);
        }
      }
    } else if (ok) {
      record_timeout(105);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 256);
}

// =====================================================================
// tc_state_scan: prefix (or total) over chunks, scaled by 1/n, to bf16
// =====================================================================
__global__ void __launch_bounds__(256)
    tc_state_scan(const float *__restrict__ S, __nv_bfloat16 *__restrict__ P, int B, int G,
                  int64_t se, float inv_n, int causal, unsigned int *__restrict__ sched) {
  // the attention kernel that follows on the stream hands out work from here
  if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0u;
  const int64_t per_b = se / 8;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * per_b) return;
  const int64_t b = t / per_b, x = (t % per_b) * 8;
  const float *src = S + b * G * se + x;
  float run[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) run[i] = 0.f;
  constexpr int U = 4;
  if (causal) {
    __nv_bfloat16 *dst = P + b * G * se + x;
    for (int g0 = 0; g0 < G; g0 += U) {
      float4 v[U][2];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (g0 + u < G) {
          const float4 *p4 = reinterpret_cast<const float4 *>(src + (int64_t)(g0 + u) * se);
          v[u][0] = __ldcs(p4);
          v[u][1] = __ldcs(p4 + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (g0 + u < G) {
          uint4 o;
          o.x = pack_bf16x2(run[0] * inv_n, run[1] * inv_n);
          o.y = pack_bf16x2(run[2] * inv_n, run[3] * inv_n);
          o.z = pack_bf16x2(run[4] * inv_n, run[5] * inv_n);
          o.w = pack_bf16x2(run[6] * inv_n, run[7] * inv_n);
          *reinterpret_cast<uint4 *>(dst + (int64_t)(g0 + u) * se) = o;
          run[0] += v[u][0].x; run[1] += v[u][0].y; run[2] += v[u][0].z; run[3] += v[u][0].w;
          run[4] += v[u][1].x; run[5] += v[u][1].y; run[6] += v[u][1].z; run[7] += v[u][1].w;
        }
      }
    }
  } else {
    for (int g0 = 0; g0 < G; g0 += U) {
      float4 v[U][2];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (g0 + u < G) {
          const float4 *p4 = reinterpret_cast<const float4 *>(src + (int64_t)(g0 + u) * se);
          v[u][0] = __ldcs(p4);
          v[u][1] = __ldcs(p4 + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (g0 + u < G) {
          run[0] += v[u][0].x; run[1] += v[u][0].y; run[2] += v[u][0].z; run[3] += v[u][0].w;
          run[4] += v[u][1].x; run[5] += v[u][1].y; run[6] += v[u][1].z; run[7] += v[u][1].w;
        }
      }
    }
    uint4 o;
    o.x = pack_bf16x2(run[0] * inv_n, run[1] * inv_n);
    o.y = pack_bf16x2(run[2] * inv_n, run[3] * inv_n);
    o.z = pack_bf16x2(run[4] * inv_n, run[5] * inv_n);
    o.w = pack_bf16x2(run[6] * inv_n, run[7] * inv_n);
    *reinterpret_cast<uint4 *>(P + b * se + x) = o;
  }
}

}  // namespace
}  // namespace fmca
