// tc_state.cuh -- per-chunk linear-attention states and their chunk-axis
// prefix ("FLASH: Possibly the Most Interesting Efficient Transformer Design
// Recently", section "Mixed Chunk": the summands K^lin_h^T V_h of V-hat^lin_g
// and their sum over all chunks, or cumsum over the chunks before g for a
// decoder).  Device code of the tensor-core path, included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

// =====================================================================
// tc_chunk_state: state_h = T3_h^T V_h, T3 = Z * gamma3 + beta3
// =====================================================================
// Persistent: one CTA per SM takes units (chunk h, 256-column slice of e)
// from a counter (zeroed by tc_chunk_scores, which runs first).  A unit
// streams C/64 items [Z: 64 keys x 128 s (16 KB) | V: 64 keys x 256 e (32 KB)]
// through a four-slot ring.  Four transform warps turn each item's Z part into
// T3 in place; the MMA warp accumulates D[s][e] = T3^T V over the unit's keys
// in TMEM (A = the T3 tile as an MN-major operand, B = the V tile, both
// MN-major); four epilogue warps round D to bf16 into a swizzled staging tile
// that a TMA store writes to the workspace.  The accumulator is
// double-buffered so a unit's epilogue overlaps the next unit's MMAs.  Each
// barrier has a single consumer.
constexpr int ST_RING = 4;
constexpr uint32_t ST_Z_BYTES = KEY_STAGE * S_DIM * 2;   // 16 KB
constexpr uint32_t ST_SLOT = ST_Z_BYTES + KEY_STAGE * E_TILE * 2;  // 48 KB
constexpr int ST_STAGE_BUFS = 2;                         // epilogue staging buffers
constexpr uint32_t ST_STAGE_BYTES = 128 * 64 * 2;        // [128 s][64 e] bf16, 16 KB
constexpr uint32_t ST_OFF_STAGE = ST_RING * ST_SLOT;
constexpr uint32_t STATE_SMEM = ST_OFF_STAGE + ST_STAGE_BUFS * ST_STAGE_BYTES + 1024;
constexpr int ST_QUEUE = 2;
// warp 0: scheduler + TMA; warp 1: MMA; warps 2-5: T3 transform;
// warps 6-9: epilogue
constexpr int STATE_THREADS = 320;
static_assert(STATE_SMEM + 1024 <= 232448, "tc_chunk_state exceeds 227 KB of shared memory");

__global__ void __launch_bounds__(STATE_THREADS, 1)
    tc_chunk_state(const __grid_constant__ CUtensorMap mapZ,   // Z [B*n][s], box {64, 64}
                   const __grid_constant__ CUtensorMap mapV,   // V [B*n][e], box {64, 64}
                   const __grid_constant__ CUtensorMap mapSt,  // states [B*G*s][e], box {64, 128}
                   const float *__restrict__ gamma, const float *__restrict__ beta,
                   unsigned int *__restrict__ sched, int n, int e, int C, int G, int n_units) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[ST_RING], tready[ST_RING], empty[ST_RING];
  __shared__ __align__(8) uint64_t q_full[ST_QUEUE], q_empty[ST_QUEUE];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ int q_unit[ST_QUEUE], acc_unit[2], slot_valid[ST_RING];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_es = e / E_TILE;
  const int nstage = C / KEY_STAGE;

  if (threadIdx.x == 0) {
    for (int i = 0; i < ST_RING; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&tready[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < ST_QUEUE; ++i) {
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
      tma_prefetch_desc(&mapZ);
      tma_prefetch_desc(&mapV);
      int it = 0;
      bool ok = true, ended = false;
      // the next unit is fetched one unit ahead, so the atomic's latency
      // overlaps the current unit's copies
      int u_next = (int)atomicAdd(sched, 1u);
      for (int i = 0; ok; ++i) {
        const int u = u_next;
        const int uu = u < n_units ? u : -1;
        if (uu >= 0) u_next = (int)atomicAdd(sched, 1u);
        const int qs = i % ST_QUEUE;
        if (i >= ST_QUEUE && !mbar_wait(&q_empty[qs], ((i / ST_QUEUE) - 1) & 1, kWaitLimitNs)) {
          record_timeout(500);
          break;
        }
        q_unit[qs] = uu;
        mbar_arrive(&q_full[qs]);
        // one more ring item than real work: an empty one tells the
        // transform warps that the stream has ended
        const int es = uu < 0 ? 0 : uu % n_es;
        const int hb = uu < 0 ? 0 : uu / n_es;  // b*G + h
        const int row0 = (hb / G) * n + (hb % G) * C;
        const int items = uu < 0 ? 1 : nstage;
        for (int k = 0; k < items; ++k, ++it) {
          const int slot = it % ST_RING;
          if (it >= ST_RING &&
              !mbar_wait(&empty[slot], ((it / ST_RING) - 1) & 1, kWaitLimitNs)) {
            record_timeout(501);
            ok = false;
            break;
          }
          if (uu < 0) {
            slot_valid[slot] = 0;
            mbar_arrive(&full[slot]);
            ended = true;
            break;
          }
          slot_valid[slot] = 1;
          uint8_t *sz = smem + slot * ST_SLOT;
          mbar_arrive_expect_tx(&full[slot], ST_SLOT);
          const int y = row0 + k * KEY_STAGE;
          tma_load_2d(sz, &mapZ, &full[slot], 0, y);
          tma_load_2d(sz + 8192, &mapZ, &full[slot], 64, y);
          for (int j = 0; j < 4; ++j)
            tma_load_2d(sz + ST_Z_BYTES + j * 8192, &mapV, &full[slot], es * E_TILE + 64 * j, y);
        }
        if (uu < 0) break;
      }
      // After a normal end the transform warps have waited on every item, so
      // every copy has landed.  After a timeout, wait (bounded) for the last
      // copy issued into each slot.  (Not after a normal end: the end marker
      // moved one slot's barrier a phase further.)
      if (!ended)
        for (int q = (it > ST_RING ? it - ST_RING : 0); q < it; ++q)
          if (!mbar_wait(&full[q % ST_RING], (q / ST_RING) & 1, kWaitLimitNs)) record_timeout(502);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      // D[s][e] += T3^T[s][k] V[k][e]: M = 128 (s), N = 256 (e), K = 16 keys per op
      constexpr uint32_t idesc = idesc_bf16_f32(128, E_TILE, true, true);
      int it = 0, j = 0;
      bool ok = true;
      for (;; ++j) {
        const int qs = j % ST_QUEUE;
        if (!mbar_wait(&q_full[qs], (j / ST_QUEUE) & 1, kWaitLimitNs)) {
          record_timeout(510);
          ok = false;
          break;
        }
        const int u = q_unit[qs];
        mbar_arrive(&q_empty[qs]);
        const int buf = j & 1, use = j >> 1;
        if (use >= 1 && !mbar_wait(&acc_empty[buf], (use - 1) & 1, kWaitLimitNs)) {
          record_timeout(511);
          ok = false;
          break;
        }
        if (u < 0) break;
        tc_fence_after();
        const uint32_t dcol = tbase + (uint32_t)buf * 256u;
        for (int k = 0; k < nstage; ++k, ++it) {
          const int slot = it % ST_RING;
          if (!mbar_wait(&tready[slot], (it / ST_RING) & 1, kWaitLimitNs)) {
            record_timeout(512);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sz = smem_u32(smem + slot * ST_SLOT);
#pragma unroll
          for (int kk = 0; kk < KEY_STAGE / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(sz + kk * 2048, 8192, 1024);
            const uint64_t bd = smem_desc_sw128(sz + ST_Z_BYTES + kk * 2048, 8192, 1024);
            mma_bf16_ss(dcol, ad, bd, idesc, (k | kk) != 0);
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
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(513);
    }
  } else if (warp < 6) {
    // =========================== T3 transform warps (128 threads)
    const int mt = threadIdx.x - 64;
    // chunk x = mt + 128 i of a Z stage: box i / 4, row (mt / 8 + 16 i) % 64,
    // physical 16-byte chunk mt % 8, i.e. logical columns 64 box + cl .. + 7
    const int p = mt & 7, rb = mt >> 3;
    const int cl = (p ^ (rb & 7)) << 3;
    float g3[2][8], b3[2][8];
#pragma unroll
    for (int bx = 0; bx < 2; ++bx) {
      load8(gamma + 3 * S_DIM + bx * 64 + cl, g3[bx]);
      load8(beta + 3 * S_DIM + bx * 64 + cl, b3[bx]);
    }
    for (int it = 0;; ++it) {
      const int slot = it % ST_RING;
      const bool got = mbar_wait(&full[slot], (it / ST_RING) & 1, kWaitLimitNs);
      const bool valid = got && slot_valid[slot] != 0;
      if (valid) {
        uint8_t *sz = smem + slot * ST_SLOT;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int bx = i >> 2, r = (rb + 16 * i) & 63;
          uint4 *ptr = reinterpret_cast<uint4 *>(sz + bx * 8192 + r * 128 + p * 16);
          *ptr = affine8(*ptr, g3[bx], b3[bx]);
        }
        fence_proxy_async_smem();
      }
      if (!named_bar_and(1, 128, valid)) {
        if (!got && mt == 0) record_timeout(520);
        break;
      }
      if (mt == 0) mbar_arrive(&tready[slot]);
      __syncwarp();
    }
  } else {
    // =========================== epilogue warps (128 threads)
    const int mt = threadIdx.x - 192;
    const int quad = warp & 3;
    const int srow = quad * 32 + lane;  // accumulator row = state row s
    uint8_t *stage = smem + ST_OFF_STAGE;
    int nst = 0;  // staging tiles written so far
    for (int j = 0;; ++j) {
      const int buf = j & 1, use = j >> 1;
      const bool got = mbar_wait(&acc_full[buf], use & 1, kWaitLimitNs);
      const int u = got ? acc_unit[buf] : -1;
      if (!named_bar_and(2, 128, u >= 0)) {
        if (!got && mt == 0) record_timeout(530);
        break;
      }
      tc_fence_after();
      const int es = u % n_es, hb = u / n_es;
      const uint32_t dcol = tbase + (uint32_t)buf * 256u + ((uint32_t)(quad * 32) << 16);
      for (int q = 0; q < E_TILE / 64; ++q, ++nst) {
        uint8_t *sb = stage + (nst % ST_STAGE_BUFS) * ST_STAGE_BYTES;
        // the TMA store that last read this staging tile has finished reading it
        if (mt == 0 && nst >= ST_STAGE_BUFS) bulk_wait_group_read<ST_STAGE_BUFS - 1>();
        named_bar_sync(2, 128);
        uint32_t r[2][32];
        tmem_ld32(dcol + q * 64, r[0]);
        tmem_ld32(dcol + q * 64 + 32, r[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const uint32_t *v = r[c2] + 8 * j4;
            *reinterpret_cast<uint4 *>(sb + sw128_offset(srow, c2 * 64 + 16 * j4)) =
                make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                           pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                           pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                           pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
          }
        fence_proxy_async_smem();
        if (q == E_TILE / 64 - 1) tc_fence_before();
        named_bar_sync(2, 128);
        if (mt == 0) {
          tma_store_2d(&mapSt, sb, es * E_TILE + 64 * q, hb * S_DIM);
          bulk_commit_group();
          // every epilogue thread has read this unit's accumulator
          if (q == E_TILE / 64 - 1) mbar_arrive(&acc_empty[buf]);
        }
        __syncwarp();
      }
    }
    if (mt == 0) bulk_wait_group<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// =====================================================================
// tc_state_scan: prefix (or total) over chunks of the bf16 states, in fp32,
// scaled by 1/n and rounded to bf16; also zeroes the attention kernel's work
// counter (it runs right after on the same stream).  The thread count is a
// multiple of 32 for every shape this path takes (B * s * e / 8).
// =====================================================================
__global__ void __launch_bounds__(256)
    tc_state_scan(const __nv_bfloat16 *__restrict__ S, __nv_bfloat16 *__restrict__ P, int B,
                  int G, int64_t se, float inv_n, int causal, unsigned int *__restrict__ sched) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0u;
  const int64_t per_b = se / 8;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * per_b) return;
  const int64_t b = t / per_b, x = (t % per_b) * 8;
  const __nv_bfloat16 *src = S + b * G * se + x;
  __nv_bfloat16 *dst = P + (causal ? b * G * se : b * se) + x;
  float run[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) run[i] = 0.f;
  constexpr int U = 8;
  for (int g0 = 0; g0 < G; g0 += U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (g0 + u < G) v[u] = __ldcs(reinterpret_cast<const uint4 *>(src + (int64_t)(g0 + u) * se));
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (g0 + u < G) {
        if (causal) {
          uint4 o;
          o.x = pack_bf16x2(run[0] * inv_n, run[1] * inv_n);
          o.y = pack_bf16x2(run[2] * inv_n, run[3] * inv_n);
          o.z = pack_bf16x2(run[4] * inv_n, run[5] * inv_n);
          o.w = pack_bf16x2(run[6] * inv_n, run[7] * inv_n);
          *reinterpret_cast<uint4 *>(dst + (int64_t)(g0 + u) * se) = o;
        }
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          run[2 * i] += bf16_lo(w[i]);
          run[2 * i + 1] += bf16_hi(w[i]);
        }
      }
    }
    // The states are dead once read: drop their lines from L2 so they are
    // never written back (eight lanes share a 128-byte line; every lane's
    // load has returned once the sums above used it).
    __syncwarp();
    if ((x & 63) == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (g0 + u < G) discard_l2_line(src + (int64_t)(g0 + u) * se);
    }
  }
  if (!causal) {
    uint4 o;
    o.x = pack_bf16x2(run[0] * inv_n, run[1] * inv_n);
    o.y = pack_bf16x2(run[2] * inv_n, run[3] * inv_n);
    o.z = pack_bf16x2(run[4] * inv_n, run[5] * inv_n);
    o.w = pack_bf16x2(run[6] * inv_n, run[7] * inv_n);
    *reinterpret_cast<uint4 *>(dst) = o;
  }
}

}  // namespace
}  // namespace fmca
