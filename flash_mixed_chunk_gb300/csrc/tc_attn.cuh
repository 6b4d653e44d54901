// tc_attn.cuh -- the output of the mixed-chunk attention core:
//     O = U * (P V_g + T2 P_g)
// with P = relu(T0 T1^T / C)^2 (masked) and T2 rows from tc_chunk_scores, and
// P_g the chunk-state prefix (or total) / n from tc_state_scan ("FLASH:
// Possibly the Most Interesting Efficient Transformer Design Recently",
// section "Mixed Chunk": V-hat^quad_g + V-hat^lin_g, gated by U_g).  Both
// products run on the tensor cores into one TMEM accumulator.  Included by
// tc.cu.
//
// Persistent kernel: one CTA per SM takes work units from a global counter.
// A unit is (chunk, 128-row tile, 256-column e tile); it streams
//   nkv items  (P rows x 64 keys [16 KB], V 64 keys x 256 e [32 KB])
//   2 items    (T2 rows x 64 s [16 KB], prefix 64 s rows x 256 e [32 KB])
// through ring A (three slots; the MMA warp's only input: every operand is
// used once per unit, so nothing stays resident across units), and its U tile
// in four 64-column quarters through ring B (four slots, so a unit's U tile
// can be in flight while the previous unit's epilogue runs; turned into O in
// place and stored with TMA).  The accumulator is double-buffered in TMEM, so
// the epilogue of one unit overlaps the MMAs of the next.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

constexpr int AT_RING_A = 3;
constexpr uint32_t AT_A_BYTES = 16384;               // A operand part of an item
constexpr uint32_t AT_SLOT_A = AT_A_BYTES + 32768;   // + B operand part
constexpr int AT_RING_B = 4;
constexpr uint32_t AT_SLOT_B = 16384;
constexpr int AT_QUEUE = 2;                          // unit-id queue depth
constexpr uint32_t AT_OFF_B = AT_RING_A * AT_SLOT_A;
constexpr uint32_t AT_SMEM = AT_OFF_B + AT_RING_B * AT_SLOT_B + 1024;
// warp 0: scheduler + ring A loads; warp 1: MMA; warp 2: ring B loads;
// warps 3-6: epilogue
constexpr int AT_THREADS = 224;
static_assert(AT_SMEM + 1024 <= 232448, "tc_chunk_attn exceeds 227 KB of shared memory");

struct AttnUnit {
  int row0;   // first token row of the tile in [B*n]
  int crow;   // first token row of its chunk
  int prow;   // first prefix row of its chunk in [B*Gp*s]
  int e0;     // first e column
  int nkv;    // V / P stages (64 keys each)
};

__device__ __forceinline__ AttnUnit decode_unit(int u, int n, int e, int C, int G, int causal,
                                                int n_units) {
  const int R = C / ROW_TILE;
  const int n_et = e / E_TILE;
  int rt, t;
  if (causal && R >= 4) {
    // long causal chunks: row tile rt reads 2 (rt + 1) key stages, so the
    // units are numbered row tile major and (taken from the top) longest
    // first, which keeps a long unit out of the tail
    const int per_rt = n_units / R;
    rt = u / per_rt;
    t = u % per_rt;
  } else {
    rt = u % R;  // row tiles of one chunk and e tile are adjacent (V reuse in L2)
    t = u / R;
  }
  const int et = t % n_et;
  const int bg = t / n_et;
  const int b = bg / G, g = bg % G;
  AttnUnit a;
  a.crow = b * n + g * C;
  a.row0 = a.crow + rt * ROW_TILE;
  a.prow = (causal ? bg : b) * S_DIM;
  a.e0 = et * E_TILE;
  a.nkv = (causal ? (rt + 1) * ROW_TILE : C) / KEY_STAGE;
  return a;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    tc_chunk_attn(const __grid_constant__ CUtensorMap mapPr,  // P [B*n][C], box {64,128}
                  const __grid_constant__ CUtensorMap mapT2,  // T2 [B*n][s], box {64,128}
                  const __grid_constant__ CUtensorMap mapV,   // V [B*n][e], box {64,64}
                  const __grid_constant__ CUtensorMap mapS,   // prefix [B*Gp*s][e], box {64,64}
                  const __grid_constant__ CUtensorMap mapU,   // U [B*n][e], box {64,128}
                  const __grid_constant__ CUtensorMap mapO,   // O [B*n][e], box {64,128}
                  unsigned int *__restrict__ sched, int n, int e, int C, int G, int causal,
                  int n_units, int lin_items) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t fullA[AT_RING_A], emptyA[AT_RING_A];
  __shared__ __align__(8) uint64_t fullB[AT_RING_B], emptyB[AT_RING_B];
  __shared__ __align__(8) uint64_t qm_full[AT_QUEUE], qm_empty[AT_QUEUE];
  __shared__ __align__(8) uint64_t qb_full[AT_QUEUE], qb_empty[AT_QUEUE];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ int qm_unit[AT_QUEUE], qb_unit[AT_QUEUE], acc_unit[2];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < AT_RING_A; ++i) {
      mbar_init(&fullA[i], 1);
      mbar_init(&emptyA[i], 1);
    }
    for (int i = 0; i < AT_RING_B; ++i) {
      mbar_init(&fullB[i], 1);
      mbar_init(&emptyB[i], 1);
    }
    for (int i = 0; i < AT_QUEUE; ++i) {
      mbar_init(&qm_full[i], 1);
      mbar_init(&qm_empty[i], 1);
      mbar_init(&qb_full[i], 1);
      mbar_init(&qb_empty[i], 1);
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
  uint8_t *ringA = smem;
  uint8_t *ringB = smem + AT_OFF_B;
  // Launched as a dependent of the scan, which itself started only after the
  // prep kernel had finished and flushed: the relu^2 weights and the lin_q
  // rows are final already, so only the loads of the scan's prefix rows wait
  // for the scan (griddepcontrol.wait in the ring A producer, before its first
  // prefix load); the quad items and U tiles of the first units overlap the
  // scan's tail.

  if (warp == 0) {
    // =========================== scheduler + ring A producer
    if (lane == 0) {
      tma_prefetch_desc(&mapPr);
      tma_prefetch_desc(&mapT2);
      tma_prefetch_desc(&mapV);
      tma_prefetch_desc(&mapS);
      int ia = 0;
      bool ok = true, scan_done = false;
      // the next unit is fetched one unit ahead, so the atomic's latency
      // overlaps the current unit's copies
      int u_next = (int)atomicAdd(sched, 1u);
      for (int i = 0; ok; ++i) {
        // units are taken last chunk first: the prep kernel streamed V in
        // chunk order, so the chunks it read last are the likeliest to still
        // be in L2 (and the longer causal row tiles go before the short ones)
        const int u = u_next;
        const int uu = u < n_units ? n_units - 1 - u : -1;
        if (uu >= 0) u_next = (int)atomicAdd(sched, 1u);
        // hand the unit to the MMA warp and to the ring B producer
        const int qs = i % AT_QUEUE;
        if (i >= AT_QUEUE) {
          if (!mbar_wait(&qm_empty[qs], ((i / AT_QUEUE) - 1) & 1, kWaitLimitNs) ||
              !mbar_wait(&qb_empty[qs], ((i / AT_QUEUE) - 1) & 1, kWaitLimitNs)) {
            record_timeout(400);
            break;
          }
        }
        qm_unit[qs] = uu;
        qb_unit[qs] = uu;
        mbar_arrive(&qm_full[qs]);
        mbar_arrive(&qb_full[qs]);
        if (uu < 0) break;
        const AttnUnit a = decode_unit(uu, n, e, C, G, causal, n_units);
        const int items = a.nkv + lin_items;
        for (int k = 0; k < items; ++k, ++ia) {
          const int slot = ia % AT_RING_A;
          if (ia >= AT_RING_A &&
              !mbar_wait(&emptyA[slot], ((ia / AT_RING_A) - 1) & 1, kWaitLimitNs)) {
            record_timeout(401);
            ok = false;
            break;
          }
          uint8_t *dst = ringA + slot * AT_SLOT_A;
          mbar_arrive_expect_tx(&fullA[slot], AT_SLOT_A);
          if (k < a.nkv) {  // P rows x keys [64k, 64k+64) ; V keys [64k, +64) x e [e0, e0+256)
            tma_load_2d(dst, &mapPr, &fullA[slot], 64 * k, a.row0);
            const int y = a.crow + k * KEY_STAGE;
            for (int j = 0; j < 4; ++j)
              tma_load_2d(dst + AT_A_BYTES + j * 8192, &mapV, &fullA[slot], a.e0 + 64 * j, y);
          } else {  // T2 rows x s [64q, 64q+64) ; prefix rows [64q, +64) x e [e0, e0+256)
            if (!scan_done) {
              griddep_wait();
              scan_done = true;
            }
            const int q = k - a.nkv;
            tma_load_2d(dst, &mapT2, &fullA[slot], 64 * q, a.row0);
            const int y = a.prow + q * KEY_STAGE;
            for (int j = 0; j < 4; ++j)
              tma_load_2d(dst + AT_A_BYTES + j * 8192, &mapS, &fullA[slot], a.e0 + 64 * j, y);
          }
        }
      }
      // drain: the last load issued into every slot has landed
      for (int q = (ia > AT_RING_A ? ia - AT_RING_A : 0); q < ia; ++q)
        if (!mbar_wait(&fullA[q % AT_RING_A], (q / AT_RING_A) & 1, kWaitLimitNs)) record_timeout(402);
    }
  } else if (warp == 2) {
    // =========================== ring B producer (U tiles)
    if (lane == 0) {
      tma_prefetch_desc(&mapU);
      // U is read once: keep it from displacing V and the workspace in L2
      const uint64_t stream_policy = policy_evict_first();
      int ib = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int qs = i % AT_QUEUE;
        if (!mbar_wait(&qb_full[qs], (i / AT_QUEUE) & 1, kWaitLimitNs)) {
          record_timeout(403);
          break;
        }
        const int u = qb_unit[qs];
        mbar_arrive(&qb_empty[qs]);
        if (u < 0) break;
        const AttnUnit a = decode_unit(u, n, e, C, G, causal, n_units);
        for (int q = 0; q < E_TILE / 64; ++q, ++ib) {
          const int slot = ib % AT_RING_B;
          if (ib >= AT_RING_B &&
              !mbar_wait(&emptyB[slot], ((ib / AT_RING_B) - 1) & 1, kWaitLimitNs)) {
            record_timeout(404);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&fullB[slot], AT_SLOT_B);
          tma_load_2d_hint(ringB + slot * AT_SLOT_B, &mapU, &fullB[slot], a.e0 + 64 * q, a.row0,
                           stream_policy);
        }
      }
      for (int q = (ib > AT_RING_B ? ib - AT_RING_B : 0); q < ib; ++q)
        if (!mbar_wait(&fullB[q % AT_RING_B], (q / AT_RING_B) & 1, kWaitLimitNs)) record_timeout(405);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      // acc[rows][256 e] = P V + T2 prefix  (A K-major, B MN-major)
      constexpr uint32_t idesc = idesc_bf16_f32(128, E_TILE, false, true);
      int ia = 0, j = 0;
      bool ok = true;
      for (;; ++j) {
        const int qs = j % AT_QUEUE;
        if (!mbar_wait(&qm_full[qs], (j / AT_QUEUE) & 1, kWaitLimitNs)) {
          record_timeout(410);
          ok = false;
          break;
        }
        const int u = qm_unit[qs];
        mbar_arrive(&qm_empty[qs]);
        const int buf = j & 1, use = j >> 1;
        // the epilogue has drained this accumulator (its previous unit)
        if (use >= 1 && !mbar_wait(&acc_empty[buf], (use - 1) & 1, kWaitLimitNs)) {
          record_timeout(412);
          ok = false;
          break;
        }
        if (u < 0) break;
        tc_fence_after();
        const AttnUnit a = decode_unit(u, n, e, C, G, causal, n_units);
        const int items = a.nkv + lin_items;
        const uint32_t dcol = tbase + (uint32_t)buf * 256u;
        for (int k = 0; k < items; ++k, ++ia) {
          const int slot = ia % AT_RING_A;
          if (!mbar_wait(&fullA[slot], (ia / AT_RING_A) & 1, kWaitLimitNs)) {
            record_timeout(413);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ringA + slot * AT_SLOT_A);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(sa + AT_A_BYTES + kk * 2048, 8192, 1024);
            mma_bf16_ss(dcol, ad, bd, idesc, (k | kk) != 0);
          }
          mma_commit(&emptyA[slot]);
        }
        if (!ok) break;
        acc_unit[buf] = u;
        mbar_arrive(&acc_full[buf]);
        mma_commit(&acc_full[buf]);
      }
      // tell the epilogue there is no further unit (in the buffer it waits on next)
      if (ok) {
        const int buf = j & 1;
        acc_unit[buf] = -1;
        mbar_arrive(&acc_full[buf]);
        mma_commit(&acc_full[buf]);
      }
      // every MMA has finished before TMEM is released
      mma_commit(&mma_done);
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(414);
    }
  } else {
    // =========================== epilogue warps (128 threads)
    const int mt = threadIdx.x - 96;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int ib = 0;
    // O is written once and read by nobody here: first out of L2
    const uint64_t out_policy = policy_evict_first();
    // Each O store is committed as its own bulk group; a U slot is released
    // once the store after it has been issued (wait_group.read 1), so the
    // store's shared-memory read overlaps the next quarter's work.
    for (int j = 0;; ++j) {
      const int buf = j & 1, use = j >> 1;
      const bool acc_ok = mbar_wait(&acc_full[buf], use & 1, kWaitLimitNs);
      const int u = acc_ok ? acc_unit[buf] : -1;
      // every epilogue thread leaves together (end of work or a timeout)
      if (!named_bar_and(1, 128, u >= 0)) {
        if (!acc_ok && mt == 0) record_timeout(420);
        break;
      }
      tc_fence_after();
      const AttnUnit a = decode_unit(u, n, e, C, G, causal, n_units);
      const uint32_t dcol = tbase + (uint32_t)buf * 256u + ((uint32_t)(quad * 32) << 16);
      bool ok = true;
      for (int q = 0; q < E_TILE / 64; ++q, ++ib) {
        const int slot = ib % AT_RING_B;
        const bool got = mbar_wait(&fullB[slot], (ib / AT_RING_B) & 1, kWaitLimitNs);
        uint8_t *us = ringB + slot * AT_SLOT_B;
        if (got) {
          uint32_t r[2][32];
          tmem_ld32(dcol + q * 64, r[0]);
          tmem_ld32(dcol + q * 64 + 32, r[1]);
          tmem_ld_wait();
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              uint4 *ptr = reinterpret_cast<uint4 *>(us + sw128_offset(row, c2 * 64 + 16 * j4));
              const uint4 uv = *ptr;
              const uint32_t w[4] = {uv.x, uv.y, uv.z, uv.w};
              uint32_t o[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int jj = 8 * j4 + 2 * i;
                o[i] = pack_bf16x2(bf16_lo(w[i]) * __uint_as_float(r[c2][jj]),
                                   bf16_hi(w[i]) * __uint_as_float(r[c2][jj + 1]));
              }
              *ptr = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
          fence_proxy_async_smem();
        }
        if (q == E_TILE / 64 - 1) tc_fence_before();
        ok = named_bar_and(1, 128, got);
        if (!ok) {
          if (mt == 0) record_timeout(421);
          break;
        }
        if (mt == 0) {
          tma_store_2d_hint(&mapO, us, a.e0 + 64 * q, a.row0, out_policy);
          bulk_commit_group();
          if (ib > 0) {
            bulk_wait_group_read<1>();  // the previous quarter's store has read its slot
            mbar_arrive(&emptyB[(ib - 1) % AT_RING_B]);
          }
          // all 128 threads have read this unit's accumulator
          if (q == E_TILE / 64 - 1) mbar_arrive(&acc_empty[buf]);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    if (mt == 0) {
      bulk_wait_group<0>();
      if (ib > 0) mbar_arrive(&emptyB[(ib - 1) % AT_RING_B]);  // nobody waits on it; keeps the count even
    }
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
