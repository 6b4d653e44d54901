// tc_prep.cuh -- everything the output kernel needs besides the inputs, in one
// persistent kernel ("FLASH: Possibly the Most Interesting Efficient
// Transformer Design Recently", sections "Weak Attention" and "Mixed Chunk"):
//
//   state units  (chunk h, 256-column slice of e):
//                state_h = T3_h^T V_h, T3 = Z * gamma3 + beta3, bf16 [B*G*s][e]
//   score units  (chunk, 128-row tile, block of up to two 64-key stages):
//                P = relu(T0 T1^T / C)^2, strict upper triangle masked in causal
//                mode, bf16 [B*n][C]; the first block of each row tile also
//                writes T2 = Z * gamma2 + beta2, bf16 [B*n][s]
//
// One CTA per SM: the small, latency-bound score units first, dealt
// round-robin over the CTAs, so that their chains overlap the state units
// streaming behind them; then the state units, from a work counter (zeroed
// before the launch).  Every unit streams 48 KB items through one
// four-slot ring:
//   state item [Z: 64 keys x 128 s (16 KB) | V: 64 keys x 256 e (32 KB)]
//   score item [Z: 128 query rows x 128 s (32 KB) | Z: 64 keys x 128 s (16 KB)]
//              for the block's first stage, [- | Z: 64 keys x 128 s] for the
//              others, whose products read the query rows from the first
//              item's slot (released only after the block's last product)
// Four transform warps form T3 (state) or T0, T1 and T2 (score) in place; the
// MMA warp accumulates D = T3^T V (M = s, N = 256; both operands MN-major) or
// S = T0 T1^T (M = 128 rows, N = 64 keys per stage; both K-major) into one of
// two TMEM accumulators; four epilogue warps round D (or relu(S/C)^2) to bf16 into a
// swizzled staging tile that a TMA store writes out.  Every barrier has one
// consumer.  Included by tc.cu.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

constexpr int PR_RING = 4;
constexpr uint32_t PR_SLOT = 49152;                      // 48 KB items
constexpr uint32_t PR_ST_Z = KEY_STAGE * S_DIM * 2;      // state: Z part, 16 KB
constexpr uint32_t PR_SC_K = 128 * S_DIM * 2;            // score: offset of the key part
constexpr int PR_STAGE_BUFS = 2;
constexpr uint32_t PR_STAGE_BYTES = 128 * 64 * 2;        // [128 rows][64 cols] bf16
constexpr uint32_t PR_OFF_STAGE = PR_RING * PR_SLOT;
constexpr uint32_t PREP_SMEM = PR_OFF_STAGE + PR_STAGE_BUFS * PR_STAGE_BYTES + 1024;
constexpr int PR_QUEUE = 2;
// warp 0: scheduler + TMA; warp 1: MMA; warps 2-5: transform; warps 6-9: epilogue
constexpr int PREP_THREADS = 320;
static_assert(PREP_SMEM + 1024 <= 232448, "tc_chunk_prep exceeds 227 KB of shared memory");

enum : int { KIND_END = 0, KIND_STATE = 1, KIND_SCORE = 2 };

struct PrepUnit {
  int kind;
  // state: hb = b*G + h, es = 256-column slice
  int hb, es;
  // score: rows [row0, row0+128) of the chunk starting at crow; key stages
  // ks .. ks + nks - 1
  int crow, row0, rt, ks, nks;
};

// Key stages per score unit (at most the ring's slots: the first item's slot
// is held until the block's last product).  Measured on long_causal, gau_base
// and flash_quad: two beat one (the query rows loaded and transformed once per
// stage) and four (fewer, longer chains to overlap).
constexpr int PR_SCORE_BLOCK = 2;
static_assert(PR_SCORE_BLOCK <= PR_RING, "a score block holds its first slot");

// Score units per chunk: row tile rt reads 2 (rt + 1) key stages (causal) or
// C / 64 (bidirectional), in blocks of PR_SCORE_BLOCK stages.
__host__ __device__ __forceinline__ int score_blocks(int rt, int C, int causal) {
  const int stages = causal ? 2 * (rt + 1) : C / KEY_STAGE;
  return (stages + PR_SCORE_BLOCK - 1) / PR_SCORE_BLOCK;
}
__host__ __device__ __forceinline__ int score_units_per_chunk(int C, int causal) {
  int u = 0;
  for (int rt = 0; rt < C / ROW_TILE; ++rt) u += score_blocks(rt, C, causal);
  return u;
}

__device__ __forceinline__ PrepUnit decode_prep(int u, int n_state, int n_score, int n, int e,
                                                int C, int G, int causal) {
  PrepUnit p;
  p.kind = KIND_END;
  p.hb = p.es = p.crow = p.row0 = p.rt = p.ks = p.nks = 0;
  if (u < 0 || u >= n_state + n_score) return p;
  if (u >= n_score) {
    u -= n_score;
    const int n_es = e / E_TILE;
    p.kind = KIND_STATE;
    p.es = u % n_es;
    p.hb = u / n_es;
    return p;
  }
  const int R = C / ROW_TILE;
  // causal: row tile rt covers keys [0, 128 (rt+1)); otherwise all C keys
  // the row tile: a short walk over the chunk's row tiles (their block
  // counts differ in causal mode)
  const int per_chunk = score_units_per_chunk(C, causal);
  const int bg = u / per_chunk;
  int w = u % per_chunk, rt = 0;
  for (; rt < R - 1; ++rt) {
    const int nb = score_blocks(rt, C, causal);
    if (w < nb) break;
    w -= nb;
  }
  const int stages = causal ? 2 * (rt + 1) : C / KEY_STAGE;
  const int ks = w * PR_SCORE_BLOCK;
  const int nks = min(PR_SCORE_BLOCK, stages - ks);
  p.kind = KIND_SCORE;
  p.crow = (bg / G) * n + (bg % G) * C;
  p.rt = rt;
  p.row0 = p.crow + rt * ROW_TILE;
  p.ks = ks;
  p.nks = nks;
  return p;
}

// BY_POSITION: the lin_q rows carry the per-position divisor 1/(t+1) of the
// global term (a separate instantiation, so that the default one carries no
// code for it).
template <bool BY_POSITION>
__global__ void __launch_bounds__(PREP_THREADS, 1)
    tc_chunk_prep(const __grid_constant__ CUtensorMap mapZ64,   // Z [B*n][s], box {64, 64}
                  const __grid_constant__ CUtensorMap mapZ128,  // Z [B*n][s], box {64, 128}
                  const __grid_constant__ CUtensorMap mapZ3,    // Z 3-D, box {64, 64, 2}
                  const __grid_constant__ CUtensorMap mapV3,    // V 3-D, box {64, 64, 4}
                  const __grid_constant__ CUtensorMap mapSt,    // states [B*G*s][e], box {64, 128}
                  const __grid_constant__ CUtensorMap mapPw,    // P [B*n][C], box {64, 128}
                  const float *__restrict__ gamma, const float *__restrict__ beta,
                  __nv_bfloat16 *__restrict__ t2out, __nv_bfloat16 *__restrict__ trows,
                  int64_t rows_plane, unsigned int *__restrict__ sched, int n, int e, int C,
                  int G, int causal, int n_state, int n_score, float quad_a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[PR_RING], tready[PR_RING], empty[PR_RING];
  __shared__ __align__(8) uint64_t q_full[PR_QUEUE], q_empty[PR_QUEUE];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ int q_unit[PR_QUEUE], acc_unit[2], slot_unit[PR_RING], slot_item[PR_RING];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_units = n_state + n_score;

  if (threadIdx.x == 0) {
    for (int i = 0; i < PR_RING; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&tready[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < PR_QUEUE; ++i) {
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
      tma_prefetch_desc(&mapZ64);
      tma_prefetch_desc(&mapZ128);
      tma_prefetch_desc(&mapZ3);
      tma_prefetch_desc(&mapV3);
      int it = 0;
      bool ok = true, ended = false;
      // Score units are dealt round-robin (CTA c takes c, c + grid, ...): they
      // come first and are short, so an atomic per unit would cost more than
      // the unit.  State units come from the work counter, fetched one unit
      // ahead so that the atomic's latency overlaps the current unit's copies.
      int k_static = 0;
      auto next_unit = [&]() -> int {
        const int us = (int)blockIdx.x + k_static * (int)gridDim.x;
        if (us < n_score) {
          ++k_static;
          return us;
        }
        return n_score + (int)atomicAdd(sched, 1u);
      };
      int u_next = next_unit();
      for (int i = 0; ok; ++i) {
        const int uu = u_next < n_units ? u_next : -1;
        if (uu >= 0) u_next = next_unit();
        // This CTA has taken its last unit: the scan kernel may start launching
        // once every CTA is this far (it waits for this grid to finish before
        // reading).  Triggered no earlier, so that its blocks do not sit on the
        // SMs beside this kernel's CTAs for their whole run.
        if (u_next >= n_units) griddep_launch_dependents();
        const int qs = i % PR_QUEUE;
        if (i >= PR_QUEUE && !mbar_wait(&q_empty[qs], ((i / PR_QUEUE) - 1) & 1, kWaitLimitNs)) {
          record_timeout(500);
          break;
        }
        q_unit[qs] = uu;
        mbar_arrive(&q_full[qs]);
        const PrepUnit p = decode_prep(uu, n_state, n_score, n, e, C, G, causal);
        // state: C/64 items; score: one per key stage of the block; end: one
        // empty item that tells the transform warps the stream is over
        const int items = p.kind == KIND_STATE ? C / KEY_STAGE
                          : p.kind == KIND_SCORE ? p.nks
                                                 : 1;
        for (int k = 0; k < items; ++k, ++it) {
          const int slot = it % PR_RING;
          if (it >= PR_RING && !mbar_wait(&empty[slot], ((it / PR_RING) - 1) & 1, kWaitLimitNs)) {
            record_timeout(501);
            ok = false;
            break;
          }
          slot_unit[slot] = uu;
          slot_item[slot] = k;
          if (p.kind == KIND_END) {
            mbar_arrive(&full[slot]);
            ended = true;
            break;
          }
          uint8_t *sz = smem + slot * PR_SLOT;
          // a score block's later items carry only their keys
          mbar_arrive_expect_tx(&full[slot], p.kind == KIND_SCORE && k > 0
                                                 ? (uint32_t)(KEY_STAGE * S_DIM * 2)
                                                 : PR_SLOT);
          if (p.kind == KIND_STATE) {
            // Z keys [64 rows][2 x 64 s] and V [64 rows][4 x 64 e], one 3-D box each
            const int y = (p.hb / G) * n + (p.hb % G) * C + k * KEY_STAGE;
            tma_load_3d(sz, &mapZ3, &full[slot], 0, y, 0);
            tma_load_3d(sz + PR_ST_Z, &mapV3, &full[slot], 0, y, p.es * (E_TILE / 64));
          } else {
            if (k == 0) {  // the query rows, for the whole block
              tma_load_2d(sz, &mapZ128, &full[slot], 0, p.row0);
              tma_load_2d(sz + 16384, &mapZ128, &full[slot], 64, p.row0);
            }
            const int y = p.crow + (p.ks + k) * KEY_STAGE;
            tma_load_2d(sz + PR_SC_K, &mapZ64, &full[slot], 0, y);
            tma_load_2d(sz + PR_SC_K + 8192, &mapZ64, &full[slot], 64, y);
          }
        }
        if (ended) break;
      }
      // After a normal end the transform warps have waited on every item, so
      // every copy has landed; after a timeout, wait (bounded) for the last
      // copy issued into each slot.
      if (!ended)
        for (int q = (it > PR_RING ? it - PR_RING : 0); q < it; ++q)
          if (!mbar_wait(&full[q % PR_RING], (q / PR_RING) & 1, kWaitLimitNs)) record_timeout(502);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      // state: D[s][e] += T3^T[s][k] V[k][e], M = 128 (s), N = 256, MN-major A and B
      constexpr uint32_t idesc_st = idesc_bf16_f32(128, E_TILE, true, true);
      // score: S[rows][keys] = T0 T1^T, M = 128, N = 64, K-major A and B
      constexpr uint32_t idesc_sc = idesc_bf16_f32(128, KEY_STAGE, false, false);
      int it = 0, j = 0;
      bool ok = true;
      for (;; ++j) {
        const int qs = j % PR_QUEUE;
        if (!mbar_wait(&q_full[qs], (j / PR_QUEUE) & 1, kWaitLimitNs)) {
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
        const PrepUnit p = decode_prep(u, n_state, n_score, n, e, C, G, causal);
        const uint32_t dcol = tbase + (uint32_t)buf * 256u;
        const int items = p.kind == KIND_STATE ? C / KEY_STAGE : p.nks;
        int slot0 = 0;  // a score block's first item: its slot holds the query rows
        for (int k = 0; k < items; ++k, ++it) {
          const int slot = it % PR_RING;
          if (!mbar_wait(&tready[slot], (it / PR_RING) & 1, kWaitLimitNs)) {
            record_timeout(512);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sz = smem_u32(smem + slot * PR_SLOT);
          if (p.kind == KIND_STATE) {
#pragma unroll
            for (int kk = 0; kk < KEY_STAGE / 16; ++kk) {
              const uint64_t ad = smem_desc_sw128(sz + kk * 2048, 8192, 1024);
              const uint64_t bd = smem_desc_sw128(sz + PR_ST_Z + kk * 2048, 8192, 1024);
              mma_bf16_ss(dcol, ad, bd, idesc_st, (k | kk) != 0);
            }
            mma_commit(&empty[slot]);
          } else {
            // S[:, 64k .. 64k+63] = T0 (first item's slot) T1_k (this item's slot)
            if (k == 0) slot0 = slot;
            const uint32_t sq = smem_u32(smem + slot0 * PR_SLOT);
#pragma unroll
            for (int kk = 0; kk < S_DIM / 16; ++kk) {
              const uint64_t ad = smem_desc_sw128(sq + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
              const uint64_t bd =
                  smem_desc_sw128(sz + PR_SC_K + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
              mma_bf16_ss(dcol + (uint32_t)(KEY_STAGE * k), ad, bd, idesc_sc, kk != 0);
            }
            if (k > 0) mma_commit(&empty[slot]);
            // the query rows' slot goes back once the block's last product is done
            if (k == items - 1) mma_commit(&empty[slot0]);
          }
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
    // =========================== transform warps (128 threads)
    const int mt = threadIdx.x - 64;
    // Thread mt owns physical 16-byte chunk p = mt % 8 of the rows r with
    // r % 8 = (mt / 8) % 8 in 64-column atom a = mt / 64 of every operand box:
    // under the 128-byte swizzle those are logical columns a*64 + cl .. + 7 in
    // every such row, so the thread needs gamma/beta of only those 8 columns
    // for each of the four transforms, kept in registers for the whole kernel.
    const int a = mt >> 6, p = mt & 7, rb = (mt >> 3) & 7;
    const int cl = a * 64 + ((p ^ rb) << 3);
    float g0[8], b0[8], g1[8], b1[8], g2[8], b2[8], g3[8], b3[8];
    load8(gamma + cl, g0);
    load8(beta + cl, b0);
    load8(gamma + S_DIM + cl, g1);
    load8(beta + S_DIM + cl, b1);
    load8(gamma + 2 * S_DIM + cl, g2);
    load8(beta + 2 * S_DIM + cl, b2);
    load8(gamma + 3 * S_DIM + cl, g3);
    load8(beta + 3 * S_DIM + cl, b3);
    for (int it = 0;; ++it) {
      const int slot = it % PR_RING;
      const bool got = mbar_wait(&full[slot], (it / PR_RING) & 1, kWaitLimitNs);
      const PrepUnit pu =
          decode_prep(got ? slot_unit[slot] : -1, n_state, n_score, n, e, C, G, causal);
      uint8_t *sz = smem + slot * PR_SLOT;
      if (pu.kind == KIND_STATE) {
        // T3 in place over the Z part (atom a: 64 key rows); the units of the
        // first e slice also write the rows T0, T1, T2 of these keys for the
        // fused output kernel (trows: [3][B*n][s], if given)
        const bool rows_out = trows != nullptr && pu.es == 0;
        const int row_base = (pu.hb / G) * n + (pu.hb % G) * C + slot_item[slot] * KEY_STAGE;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = rb + 8 * i;
          uint4 *ptr = reinterpret_cast<uint4 *>(sz + a * 8192 + r * 128 + p * 16);
          const uint4 z = *ptr;
          if (rows_out) {
            __nv_bfloat16 *dst = trows + (size_t)(row_base + r) * S_DIM + cl;
            *reinterpret_cast<uint4 *>(dst) = affine8(z, g0, b0);
            *reinterpret_cast<uint4 *>(dst + rows_plane) = affine8(z, g1, b1);
            if (BY_POSITION)  // row t of its sequence carries 1/(t+1)
              *reinterpret_cast<uint4 *>(dst + 2 * rows_plane) =
                  affine8_scaled(z, g2, b2, 1.0f / (float)((row_base + r) % n + 1));
            else
              *reinterpret_cast<uint4 *>(dst + 2 * rows_plane) = affine8(z, g2, b2);
          }
          *ptr = affine8(z, g3, b3);
        }
        fence_proxy_async_smem();
      } else if (pu.kind == KIND_SCORE) {
        // query rows (atom a: 128 rows), in the block's first item only: T0 in
        // place; T2 to global from the same Z values, once per row tile (by
        // its first block)
        const int tpos0 = BY_POSITION ? pu.row0 % n : 0;  // position of the tile's first row
        if (slot_item[slot] == 0) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int r = rb + 8 * i;
            uint4 *ptr = reinterpret_cast<uint4 *>(sz + a * 16384 + r * 128 + p * 16);
            const uint4 z = *ptr;
            if (pu.ks == 0) {
              uint4 *t2p =
                  reinterpret_cast<uint4 *>(t2out + (size_t)(pu.row0 + r) * S_DIM + cl);
              if (BY_POSITION)  // row t of its sequence carries 1/(t+1)
                *t2p = affine8_scaled(z, g2, b2, 1.0f / (float)(tpos0 + r + 1));
              else
                *t2p = affine8(z, g2, b2);
            }
            *ptr = affine8(z, g0, b0);
          }
        }
        // keys (atom a: 64 rows): T1 in place
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 *ptr =
              reinterpret_cast<uint4 *>(sz + PR_SC_K + a * 8192 + (rb + 8 * i) * 128 + p * 16);
          *ptr = affine8(*ptr, g1, b1);
        }
        fence_proxy_async_smem();
      }
      const bool valid = pu.kind != KIND_END;
      if (!named_bar_and(1, 128, valid)) {
        if (!got && mt == 0) record_timeout(520);
        break;
      }
      if (mt == 0) mbar_arrive(&tready[slot]);
      __syncwarp();
    }
  } else if (warp < 10) {
    // =========================== epilogue warps (128 threads)
    const int mt = threadIdx.x - 192;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // accumulator row (state row s or query row)
    uint8_t *stage = smem + PR_OFF_STAGE;
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
      const PrepUnit p = decode_prep(u, n_state, n_score, n, e, C, G, causal);
      const uint32_t dcol = tbase + (uint32_t)buf * 256u + ((uint32_t)(quad * 32) << 16);
      const int nq = p.kind == KIND_STATE ? E_TILE / 64 : p.nks;
      for (int q = 0; q < nq; ++q, ++nst) {
        uint8_t *sb = stage + (nst % PR_STAGE_BUFS) * PR_STAGE_BYTES;
        // the TMA store that last read this staging tile has finished reading it
        if (mt == 0 && nst >= PR_STAGE_BUFS) bulk_wait_group_read<PR_STAGE_BUFS - 1>();
        named_bar_sync(2, 128);
        uint32_t r[2][32];
        tmem_ld32(dcol + q * 64, r[0]);
        tmem_ld32(dcol + q * 64 + 32, r[1]);
        tmem_ld_wait();
        if (p.kind == KIND_SCORE) {
          // relu(S * quad_a)^2 (quad_a = 1/C by default); causal: key position >
          // query position -> 0
          const int qpos = p.rt * ROW_TILE + row;
          const int kbase = (p.ks + q) * KEY_STAGE;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float x = fmaxf(__uint_as_float(r[c2][i]) * quad_a, 0.f);
              x = x * x;
              if (causal && kbase + c2 * 32 + i > qpos) x = 0.f;
              r[c2][i] = __float_as_uint(x);
            }
        }
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const uint32_t *v = r[c2] + 8 * j4;
            *reinterpret_cast<uint4 *>(sb + sw128_offset(row, c2 * 64 + 16 * j4)) =
                make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                           pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                           pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                           pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
          }
        fence_proxy_async_smem();
        if (q == nq - 1) tc_fence_before();
        named_bar_sync(2, 128);
        if (mt == 0) {
          if (p.kind == KIND_STATE)
            tma_store_2d(&mapSt, sb, p.es * E_TILE + 64 * q, p.hb * S_DIM);
          else
            tma_store_2d(&mapPw, sb, (p.ks + q) * KEY_STAGE, p.row0);
          bulk_commit_group();
          // every epilogue thread has read this unit's accumulator
          if (q == nq - 1) mbar_arrive(&acc_empty[buf]);
        }
        __syncwarp();
      }
    }
    if (mt == 0) bulk_wait_group<0>();
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
