// tc_fused.cuh -- the chunk-local kernel of the mixed-chunk attention core:
//     O = U * (relu(T0 T1^T * a)^2 V_g + T2 prefix_g)
// with the relu^2 weights produced and consumed on chip ("FLASH: Possibly the
// Most Interesting Efficient Transformer Design Recently", section "Mixed
// Chunk": V-hat^quad_g with the upper triangle masked for a decoder, plus
// V-hat^lin_g from the chunk-state prefix, gated by U_g).  T0, T1, T2 (the
// affine maps of "Weak Attention") come as bf16 rows from the state kernel.
// Included by tc.cu.
//
// Persistent kernel, one CTA per SM.  The (chunk, 128-row tile, 128-column
// e tile) tiles, ordered chunk, row tile, e tile, are split into one
// contiguous range per CTA of about equal cost (bytes streamed: V and, where
// the weights are recomputed, T1 per key stage; U, O and the prefix), so
// every CTA finishes at about the same time with one or two units.  A unit
// is the run of one row tile's e tiles in a CTA's range:
//   S_k = T0 T1_k^T        64 keys per stage k, M = 128, N = 64, K = s = 128,
//                          into one of two TMEM S slots
//   P_k = relu(S_k a)^2    masked (key > query -> 0) in registers by four
//                          "relu" warps and stored back to TMEM as bf16 (the A
//                          operand of the next product) in one of four P slots
//   per e tile:
//     O  = sum_k P_k V_k   M = 128, N = 128, K = 64 per stage, A from TMEM
//     O += T2 local_g      K = s = 128 (causal: the sum of the states of the
//                          chunk's segment before it)
//     O += T2 carry        K = s = 128 (causal: the sum of the segments
//                          before the chunk's, past the first; bidirectional:
//                          the total); T2 carries the global term's divisor
//     out = U * O          four epilogue warps, in place in the U tile, one
//                          TMA store
// A row tile with at most four key stages (every chunk of 256) keeps its
// P_k resident in TMEM and computes them once for all e tiles of the unit;
// longer rows (FLASH-Quad) recompute them per e tile in blocks of four
// stages.  The S, P and O tiles never leave the SM.
//
// Every copy is one TMA instruction of 32 KB (a 3-D box of two 64-column
// blocks, see tma_load_3d): an issuing thread pays a few hundred cycles per
// instruction whatever its size, so the items are made large.  Shared memory
// holds only the products' operands, so that as many bytes as possible are in
// flight (the kernel streams from HBM):
//   A        T0 rows of the tile        [2][128][64] bf16 (score products)
//   B        T2 rows of the tile        [2][128][64] bf16 (global products)
//   ring     5 x 32 KB items, the MMA warp's only input:
//              keys   T1 rows of 128 keys   [2][128][64] (two stages)
//              V      128 keys x 128 e      [2][128][64]
//              local or carry 128 s x 128 e [2][128][64]
// The epilogue warps read U and write O with 16-byte loads and stores, one
// tile row per thread; a tile's U is loaded while its products run.
// TMEM (512 columns): O [0, 256) as two 128-column buffers (the epilogue of
// one e tile overlaps the products of the next), S [256, 384), P [384, 512).
#pragma once

#include "tc_common.cuh"
#include "tc_walk.cuh"

namespace fmca {
namespace {

constexpr int FU_ET = 128;                            // e columns per O tile
constexpr int FU_KI = 128;                            // keys per ring item (two stages)
constexpr uint32_t FU_ITEM = 32768;                   // ring item bytes
constexpr int FU_RING = 5;
constexpr uint32_t FU_AB_BYTES = 32768;               // T0 / T2 tile
constexpr uint32_t FU_OFF_A = FU_RING * FU_ITEM;
constexpr uint32_t FU_OFF_B = FU_OFF_A + FU_AB_BYTES;
constexpr uint32_t FUSED_SMEM = FU_OFF_B + FU_AB_BYTES + 1024;
constexpr int FU_QUEUE = 2;        // unit-id queue depth
constexpr int FU_SSLOTS = 2;       // S slots (64 columns each)
constexpr int FU_PSLOTS = 4;       // P slots (32 columns each): a key block
constexpr uint32_t FU_COL_S = 256, FU_COL_P = 384;
// warp 0: scheduler + ring, A and B loads; warp 1: MMA; warps 2-3: idle;
// warps 4-7: relu^2; warps 8-11: epilogue
constexpr int FUSED_THREADS = 384;
static_assert(FUSED_SMEM + 1024 <= 232448, "tc_chunk_fused exceeds 227 KB of shared memory");

struct FusedUnit {
  int g;      // chunk within its sequence
  int row0;   // first token row of the tile in [B*n]
  int crow;   // first token row of its chunk
  int lrow;   // first row of the chunk's local sums in [B*G*s]
  int crow2;  // first row of its carry in [B*S*s] (its total when bidirectional)
  bool carry; // a carry product (causal: past the first segment)
  int rt;     // row tile within the chunk
  int et0;    // first 128-column e tile
  int net;    // e tiles in the unit
  int nkv;    // 64-key stages of the row tile (even)
};

// The tiles: t = (bg * R + rt) * n_et + et for sequence-chunk bg (of B * G),
// row tile rt (of R = C / 128) and e tile et (of n_et = ceil(e / 128); the
// last may be 64 columns).
struct FusedGrid {
  int n, C, G, causal, lin, R, n_et, n_tiles;
  int S, L;        // segments of the chunk axis, chunks each
  int rows_early;  // the T rows may be read before the grid-dependency wait
  int carry_all;   // a carried-in state: every causal chunk has a carry
};

// 64-key stages of row tile rt
__device__ __forceinline__ int fused_nkv(int rt, const FusedGrid &g) {
  return (g.causal ? (rt + 1) * ROW_TILE : g.C) / KEY_STAGE;
}
// the cost of one tile of row tile rt, in KB streamed: 16 per key stage of V,
// 16 more of T1 where the relu^2 weights are recomputed per e tile (more than
// FU_PSLOTS stages), 32 each of U and O, 32 of the prefix
__device__ __forceinline__ int64_t fused_tile_cost(int rt, const FusedGrid &g) {
  const int nkv = fused_nkv(rt, g);
  return (int64_t)nkv * (nkv <= FU_PSLOTS ? 16 : 32) + 64 +
         (g.lin ? (g.causal && g.S > 1 ? 64 : 32) : 0);
}
// the tile that holds cost position x (the tiles laid end to end in order)
__device__ __forceinline__ int fused_tile_at(int64_t x, const FusedGrid &g) {
  int64_t per_bg = 0;
  for (int r = 0; r < g.R; ++r) per_bg += (int64_t)g.n_et * fused_tile_cost(r, g);
  const int64_t bg = x / per_bg;
  if (bg * g.R * g.n_et >= g.n_tiles) return g.n_tiles;
  int64_t rem = x - bg * per_bg;
  int rt = 0;
  for (; rt < g.R - 1; ++rt) {
    const int64_t w = (int64_t)g.n_et * fused_tile_cost(rt, g);
    if (rem < w) break;
    rem -= w;
  }
  int et = (int)(rem / fused_tile_cost(rt, g));
  if (et >= g.n_et) et = g.n_et - 1;
  return (int)((bg * g.R + rt) * g.n_et + et);
}
// CTA c's tiles: [fused_range_start(c), fused_range_start(c + 1))
__device__ __forceinline__ int fused_range_start(int c, int grid_size, const FusedGrid &g) {
  if (c <= 0) return 0;
  if (c >= grid_size) return g.n_tiles;
  int64_t per_bg = 0;
  for (int r = 0; r < g.R; ++r) per_bg += (int64_t)g.n_et * fused_tile_cost(r, g);
  const int64_t total = per_bg * (g.n_tiles / (g.R * g.n_et));
  return fused_tile_at(total * c / grid_size, g);
}

// The unit of net tiles from tile t (all of one row tile)
__device__ __forceinline__ FusedUnit decode_fused(int t, int net, const FusedGrid &g) {
  const int et = t % g.n_et;
  const int rt = (t / g.n_et) % g.R;
  const int bg = t / (g.n_et * g.R);
  const int b = bg / g.G, c = bg % g.G;
  FusedUnit f;
  f.g = c;
  f.crow = b * g.n + c * g.C;
  f.row0 = f.crow + rt * ROW_TILE;
  f.lrow = bg * S_DIM;
  f.crow2 = (b * g.S + (g.causal ? c / g.L : 0)) * S_DIM;
  f.carry = !g.causal || g.carry_all || c / g.L > 0;
  f.rt = rt;
  f.et0 = et;
  f.net = net;
  f.nkv = fused_nkv(rt, g);
  return f;
}

// Key blocks: FU_PSLOTS stages (two ring items) each; a row tile of at most
// one block keeps its relu^2 weights resident for all its e tiles.
__device__ __forceinline__ int block_stages(const FusedUnit &f, int kb) {
  return min(FU_PSLOTS, f.nkv - kb * FU_PSLOTS);
}
__device__ __forceinline__ bool p_resident(const FusedUnit &f) { return f.nkv <= FU_PSLOTS; }

__global__ void __launch_bounds__(FUSED_THREADS, 1)
    tc_chunk_fused(const __grid_constant__ CUtensorMap mapT0,  // T0 rows, 3-D box {64, 128, 2}
                   const __grid_constant__ CUtensorMap mapT1,  // T1 rows, 3-D box {64, 128, 2}
                   const __grid_constant__ CUtensorMap mapT2,  // T2 rows, 3-D box {64, 128, 2}
                   const __grid_constant__ CUtensorMap mapV,   // V 3-D, box {64, 128, 2}
                   const __grid_constant__ CUtensorMap mapS,   // local sums 3-D, box {64, 128, 2}
                   const __grid_constant__ CUtensorMap mapCy,  // carries 3-D, box {64, 128, 2}
                   const __grid_constant__ CUtensorMap mapU,   // U 3-D, box {64, 128, 2} (L2 prefetch)
                   const __nv_bfloat16 *__restrict__ U,        // [B*n][e]
                   __nv_bfloat16 *__restrict__ O,              // [B*n][e]
                   FusedGrid grid, int e, float quad_a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t uq_full[FU_QUEUE], uq_empty[FU_QUEUE];
  __shared__ __align__(8) uint64_t a_full, a_empty, b_full, b_empty;
  __shared__ __align__(8) uint64_t full[FU_RING], empty[FU_RING];
  __shared__ __align__(8) uint64_t s_full[FU_SSLOTS], s_empty[FU_SSLOTS];
  __shared__ __align__(8) uint64_t p_full[FU_PSLOTS], p_empty[FU_PSLOTS];
  __shared__ __align__(8) uint64_t o_full[2], o_empty[2], mma_done;
  __shared__ int uq_unit[FU_QUEUE], uq_net[FU_QUEUE];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const bool lin = grid.lin != 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < FU_QUEUE; ++i) {
      mbar_init(&uq_full[i], 1);
      mbar_init(&uq_empty[i], 3);  // MMA issuer, relu^2 warps, epilogue warps
    }
    mbar_init(&a_full, 1);
    mbar_init(&a_empty, 1);
    mbar_init(&b_full, 1);
    mbar_init(&b_empty, 1);
    for (int i = 0; i < FU_RING; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < FU_SSLOTS; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 1);
    }
    for (int i = 0; i < FU_PSLOTS; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_full[i], 1);  // tcgen05.commit
      mbar_init(&o_empty[i], 1);
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
  uint8_t *ring = smem;
  uint8_t *abuf = smem + FU_OFF_A;
  uint8_t *bbuf = smem + FU_OFF_B;

  if (warp == 0) {
    // =========================== scheduler + ring, A and B producer
    if (lane == 0) {
      tma_prefetch_desc(&mapT0);
      tma_prefetch_desc(&mapT1);
      tma_prefetch_desc(&mapT2);
      tma_prefetch_desc(&mapV);
      tma_prefetch_desc(&mapS);
      tma_prefetch_desc(&mapCy);
      tma_prefetch_desc(&mapU);
      int it = 0;
      bool ok = true, rows_ready = false, prefix_ready = false;
      // one ring item: waits for its slot, then one 32 KB box
      auto issue = [&](const CUtensorMap *map, int y, int z) -> bool {
        const int slot = it % FU_RING;
        if (it >= FU_RING && !mbar_wait(&empty[slot], ((it / FU_RING) - 1) & 1, kWaitLimitNs)) {
          record_timeout(602);
          return false;
        }
        mbar_arrive_expect_tx(&full[slot], FU_ITEM);
        tma_load_3d(ring + slot * FU_ITEM, map, &full[slot], 0, y, z);
        ++it;
        return true;
      };
      // this CTA's tiles, one unit per row tile they touch
      int t = fused_range_start((int)blockIdx.x, (int)gridDim.x, grid);
      const int t_end = fused_range_start((int)blockIdx.x + 1, (int)gridDim.x, grid);
      for (int j = 0; ok; ++j) {
        const int uu = t < t_end ? t : -1;
        const int et = t % grid.n_et;
        const int net = uu >= 0 ? min(grid.n_et - et, t_end - t) : 0;
        t += net;
        const int qs = j % FU_QUEUE;
        if (j >= FU_QUEUE && !mbar_wait(&uq_empty[qs], ((j / FU_QUEUE) - 1) & 1, kWaitLimitNs)) {
          record_timeout(600);
          break;
        }
        uq_unit[qs] = uu;
        uq_net[qs] = net;
        mbar_arrive(&uq_full[qs]);
        if (uu < 0) break;
        const FusedUnit f = decode_fused(uu, net, grid);
        // The T rows: with the carry kernel between their writer and this
        // grid, the writer had completed before it let this grid launch (it
        // waits for it first); otherwise they come from the kernel just
        // before: wait here.
        if (!grid.rows_early && !rows_ready) {
          griddep_wait();
          rows_ready = true;
        }
        // A (T0): the previous unit's score products are done with it
        if (j >= 1 && !mbar_wait(&a_empty, (j - 1) & 1, kWaitLimitNs)) {
          record_timeout(601);
          break;
        }
        mbar_arrive_expect_tx(&a_full, FU_AB_BYTES);
        tma_load_3d(abuf, &mapT0, &a_full, 0, f.row0, 0);
        const bool res = p_resident(f);
        const int nkb = (f.nkv + FU_PSLOTS - 1) / FU_PSLOTS;
        for (int x = 0; x < f.net && ok; ++x) {
          const int eb = (f.et0 + x) * (FU_ET / 64);  // first 64-column block of the tile
          // the epilogue's U rows of this tile, into L2 ahead of its loads
          tma_prefetch_l2_3d(&mapU, 0, f.row0, eb);
          for (int kb = 0; kb < nkb && ok; ++kb) {
            const int ni = block_stages(f, kb) / 2;   // items of 128 keys
            const int key0 = f.crow + kb * FU_PSLOTS * KEY_STAGE;
            if (x == 0 || !res)  // T1 rows of the block's keys
              for (int i = 0; i < ni && ok; ++i) ok = issue(&mapT1, key0 + i * FU_KI, 0);
            for (int i = 0; i < ni && ok; ++i)  // V rows of the block's keys, e tile x
              ok = issue(&mapV, key0 + i * FU_KI, eb);
          }
          if (!ok || !lin) continue;
          if (x == 0) {
            // B (T2): the previous unit's global products are done with it
            if (j >= 1 && !mbar_wait(&b_empty, (j - 1) & 1, kWaitLimitNs)) {
              record_timeout(604);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&b_full, FU_AB_BYTES);
            tma_load_3d(bbuf, &mapT2, &b_full, 0, f.row0, 0);
          }
          // the local sums and carries come from the kernels before: wait
          // once, before the first such load (the unit's rows, scores,
          // weights and first products overlap their tail)
          if (!prefix_ready) {
            griddep_wait();
            prefix_ready = true;
          }
          if (grid.causal) ok = issue(&mapS, f.lrow, eb);  // local sums, e tile x
          if (ok && f.carry) ok = issue(&mapCy, f.crow2, eb);
        }
      }
      // drain: the last load issued into every ring slot has landed
      for (int q = (it > FU_RING ? it - FU_RING : 0); q < it; ++q)
        if (!mbar_wait(&full[q % FU_RING], (q / FU_RING) & 1, kWaitLimitNs)) record_timeout(603);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      // S = T0 T1^T: M = 128 rows, N = 64 keys, A and B K-major
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, KEY_STAGE, false, false);
      // O += P V (A from TMEM) and O += T2 prefix (A K-major); B MN-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, FU_ET, false, true);
      const uint32_t aaddr = smem_u32(abuf), baddr = smem_u32(bbuf);
      int it = 0, sc = 0, pc = 0, oc = 0, j = 0;
      bool ok = true;
      auto wait_item = [&](int item) -> bool {
        if (!mbar_wait(&full[item % FU_RING], (item / FU_RING) & 1, kWaitLimitNs)) {
          record_timeout(624);
          return false;
        }
        return true;
      };
      for (;; ++j) {
        const int qs = j % FU_QUEUE;
        if (!mbar_wait(&uq_full[qs], (j / FU_QUEUE) & 1, kWaitLimitNs)) {
          record_timeout(620);
          ok = false;
          break;
        }
        const int u = uq_unit[qs], unet = uq_net[qs];
        mbar_arrive(&uq_empty[qs]);
        if (u < 0) break;
        const FusedUnit f = decode_fused(u, unet, grid);
        const bool res = p_resident(f);
        const int nkb = (f.nkv + FU_PSLOTS - 1) / FU_PSLOTS;
        if (!mbar_wait(&a_full, j & 1, kWaitLimitNs)) {
          record_timeout(621);
          ok = false;
          break;
        }
        tc_fence_after();
        int pbase = pc;  // P slot counter of stage 0 of the current key block
        for (int x = 0; x < f.net && ok; ++x, ++oc) {
          const int ob = oc & 1;
          const uint32_t ocol = tbase + (uint32_t)(ob * FU_ET);
          bool first = true;  // the next product into O starts the tile
          for (int kb = 0; kb < nkb && ok; ++kb) {
            const int ns = block_stages(f, kb), ni = ns / 2;
            const bool need_s = x == 0 || !res;
            const bool last_use = !res || x == f.net - 1;
            if (need_s) pbase = pc;
            const int t1_item = it, v_item = it + (need_s ? ni : 0);
            // O += P_k V_k, the stages of one V item (128 keys)
            auto pv_item = [&](int i) -> bool {
              const int item = v_item + i;
              if (!wait_item(item)) return false;
              for (int h = 0; h < 2; ++h) {
                const int k = 2 * i + h, ps = (pbase + k) % FU_PSLOTS;
                if (need_s &&
                    !mbar_wait(&p_full[ps], ((pbase + k) / FU_PSLOTS) & 1, kWaitLimitNs)) {
                  record_timeout(622);
                  return false;
                }
                // the epilogue has drained this O buffer (two e tiles ago)
                if (first && oc >= 2 &&
                    !mbar_wait(&o_empty[ob], ((oc >> 1) - 1) & 1, kWaitLimitNs)) {
                  record_timeout(623);
                  return false;
                }
                tc_fence_after();
                const uint32_t vb = smem_u32(ring + (item % FU_RING) * FU_ITEM) + h * 8192;
                const uint32_t pa = tbase + FU_COL_P + (uint32_t)(32 * ps);
#pragma unroll
                for (int kk = 0; kk < KEY_STAGE / 16; ++kk)
                  mma_bf16_ts(ocol, pa + 8 * kk, smem_desc_sw128(vb + kk * 2048, 16384, 1024),
                              idesc_o, (first && kk == 0) ? 0u : 1u);
                first = false;
                if (last_use) mma_commit(&p_empty[ps]);
              }
              mma_commit(&empty[item % FU_RING]);
              return true;
            };
            if (need_s) {
              for (int i = 0; i < ni && ok; ++i) {
                const int item = t1_item + i, slot = item % FU_RING;
                if (!wait_item(item)) {
                  ok = false;
                  break;
                }
                const uint32_t kaddr = smem_u32(ring + slot * FU_ITEM);
                for (int h = 0; h < 2 && ok; ++h) {  // the two 64-key stages of the item
                  const int ss = sc % FU_SSLOTS;
                  if (sc >= FU_SSLOTS &&
                      !mbar_wait(&s_empty[ss], ((sc / FU_SSLOTS) - 1) & 1, kWaitLimitNs)) {
                    record_timeout(626);
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  const uint32_t sd = tbase + FU_COL_S + (uint32_t)(KEY_STAGE * ss);
#pragma unroll
                  for (int kk = 0; kk < S_DIM / 16; ++kk) {
                    const uint64_t ad =
                        smem_desc_sw128(aaddr + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(
                        kaddr + (kk >> 2) * 16384 + h * 8192 + (kk & 3) * 32, 16, 1024);
                    mma_bf16_ss(sd, ad, bd, idesc_s, kk != 0);
                  }
                  mma_commit(&s_full[ss]);
                  ++sc;
                  ++pc;
                }
                mma_commit(&empty[slot]);  // T1 of the item consumed
                // A goes back after the unit's last score product
                if (i == ni - 1 && kb == nkb - 1 && (res || x == f.net - 1)) mma_commit(&a_empty);
                // the products of the previous item's stages, while this one's
                // relu^2 weights are formed
                if (ok && i >= 1 && !pv_item(i - 1)) ok = false;
              }
              if (ok && !pv_item(ni - 1)) ok = false;
            } else {
              for (int i = 0; i < ni && ok; ++i)
                if (!pv_item(i)) ok = false;
            }
            it = v_item + ni;
          }
          if (!ok) break;
          if (lin) {
            if (x == 0 && !mbar_wait(&b_full, j & 1, kWaitLimitNs)) {
              record_timeout(627);
              ok = false;
              break;
            }
            // O += T2 local_g (causal), then O += T2 carry (when present)
            const int n_glob = (grid.causal ? 1 : 0) + (f.carry ? 1 : 0);
            for (int gi = 0; gi < n_glob && ok; ++gi) {
              if (!wait_item(it)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t pb = smem_u32(ring + (it % FU_RING) * FU_ITEM);
#pragma unroll
              for (int kk = 0; kk < S_DIM / 16; ++kk) {
                const uint64_t ad =
                    smem_desc_sw128(baddr + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                const uint64_t bd = smem_desc_sw128(pb + kk * 2048, 16384, 1024);
                mma_bf16_ss(ocol, ad, bd, idesc_o, 1u);
              }
              mma_commit(&empty[it % FU_RING]);
              ++it;
            }
            if (!ok) break;
            if (x == f.net - 1) mma_commit(&b_empty);  // B goes back after the unit
          }
          mma_commit(&o_full[ob]);
        }
        if (!ok) break;
      }
      // every MMA has finished before TMEM is released
      mma_commit(&mma_done);
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(629);
    }
  } else if (warp >= 4 && warp < 8) {
    // =========================== relu^2 warps (128 threads): S -> P in TMEM
    const int mt = threadIdx.x - 128;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // query row within the tile (TMEM lane)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int sc = 0, pc = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      const int qs = j % FU_QUEUE;
      const bool got = mbar_wait(&uq_full[qs], (j / FU_QUEUE) & 1, kWaitLimitNs);
      const int u = got ? uq_unit[qs] : -1, unet = got ? uq_net[qs] : 0;
      const bool more = named_bar_and(2, 128, u >= 0);
      if (mt == 0 && got) mbar_arrive(&uq_empty[qs]);
      if (!more) {
        if (!got && mt == 0) record_timeout(640);
        break;
      }
      const FusedUnit f = decode_fused(u, unet, grid);
      const bool res = p_resident(f);
      const int nkb = (f.nkv + FU_PSLOTS - 1) / FU_PSLOTS;
      const int qpos = f.rt * ROW_TILE + row;  // query position within the chunk
      for (int x = 0; x < (res ? 1 : f.net) && ok; ++x) {
        for (int kb = 0; kb < nkb && ok; ++kb) {
          const int ns = block_stages(f, kb);
          for (int k = 0; k < ns; ++k, ++sc, ++pc) {
            const int ss = sc % FU_SSLOTS, ps = pc % FU_PSLOTS;
            bool w = mbar_wait(&s_full[ss], (sc / FU_SSLOTS) & 1, kWaitLimitNs);
            // the last product that read this P slot has completed
            if (w && pc >= FU_PSLOTS)
              w = mbar_wait(&p_empty[ps], ((pc / FU_PSLOTS) - 1) & 1, kWaitLimitNs);
            if (w) {
              tc_fence_after();
              uint32_t r[2][32];
              const uint32_t sa = tbase + lane_off + FU_COL_S + (uint32_t)(KEY_STAGE * ss);
              tmem_ld32(sa, r[0]);
              tmem_ld32(sa + 32, r[1]);
              tmem_ld_wait();
              // relu(S a)^2 (a = 1/C by default); causal: key position > query
              // position -> 0; two keys a column, the lower key in the low half
              const int kbase = (kb * FU_PSLOTS + k) * KEY_STAGE;
              uint32_t pk[32];
#pragma unroll
              for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int key = kbase + c2 * 32 + 2 * i;
                  float x0 = fmaxf(__uint_as_float(r[c2][2 * i]) * quad_a, 0.f);
                  float x1 = fmaxf(__uint_as_float(r[c2][2 * i + 1]) * quad_a, 0.f);
                  x0 *= x0;
                  x1 *= x1;
                  if (grid.causal) {
                    if (key > qpos) x0 = 0.f;
                    if (key + 1 > qpos) x1 = 0.f;
                  }
                  pk[c2 * 16 + i] = pack_bf16x2(x0, x1);
                }
              tmem_st32(tbase + lane_off + FU_COL_P + (uint32_t)(32 * ps), pk);
              tmem_st_wait();
              tc_fence_before();
            }
            ok = named_bar_and(2, 128, w);
            if (!ok) {
              if (mt == 0) record_timeout(641);
              break;
            }
            if (mt == 0) {
              mbar_arrive(&s_empty[ss]);  // every thread has read this S slot
              mbar_arrive(&p_full[ps]);
            }
          }
        }
      }
    }
  } else if (warp >= 8) {
    // =========================== epilogue warps (128 threads)
    const int mt = threadIdx.x - 256;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // tile row (TMEM lane)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int oc = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      const int qs = j % FU_QUEUE;
      const bool got = mbar_wait(&uq_full[qs], (j / FU_QUEUE) & 1, kWaitLimitNs);
      const int u = got ? uq_unit[qs] : -1, unet = got ? uq_net[qs] : 0;
      const bool more = named_bar_and(3, 128, u >= 0);
      if (mt == 0 && got) mbar_arrive(&uq_empty[qs]);
      if (!more) {
        if (!got && mt == 0) record_timeout(650);
        break;
      }
      const FusedUnit f = decode_fused(u, unet, grid);
      const size_t roff = (size_t)(f.row0 + row) * (size_t)e;
      for (int x = 0; x < f.net && ok; ++x, ++oc) {
        const int ob = oc & 1;
        const int e0 = (f.et0 + x) * FU_ET;
        // this thread's row of the U tile, loaded while the products run
        u32x8 uv[FU_ET / 16];
        const __nv_bfloat16 *usrc = U + roff + e0;
#pragma unroll
        for (int c = 0; c < FU_ET / 16; ++c)
          if (e0 + 16 * c < e) uv[c] = ldg_stream(usrc + 16 * c);  // a 64-column last tile
        const bool w = mbar_wait(&o_full[ob], (oc >> 1) & 1, kWaitLimitNs);
        if (w) {
          tc_fence_after();
          __nv_bfloat16 *odst = O + roff + e0;
#pragma unroll
          for (int q = 0; q < FU_ET / 32; ++q) {  // 32 columns at a time
            if (e0 + 32 * q >= e) break;
            uint32_t r[32];
            tmem_ld32(tbase + lane_off + (uint32_t)(ob * FU_ET + 32 * q), r);
            tmem_ld_wait();
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {  // 16 columns per 32-byte access
              const u32x8 &uu = uv[2 * q + c2];
              const uint32_t wv[8] = {uu.lo.x, uu.lo.y, uu.lo.z, uu.lo.w,
                                      uu.hi.x, uu.hi.y, uu.hi.z, uu.hi.w};
              uint32_t o[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int jj = 16 * c2 + 2 * i;
                o[i] = pack_bf16x2(bf16_lo(wv[i]) * __uint_as_float(r[jj]),
                                   bf16_hi(wv[i]) * __uint_as_float(r[jj + 1]));
              }
              u32x8 ov;
              ov.lo = make_uint4(o[0], o[1], o[2], o[3]);
              ov.hi = make_uint4(o[4], o[5], o[6], o[7]);
              stg_stream(odst + 32 * q + 16 * c2, ov);
            }
          }
          tc_fence_before();
        }
        ok = named_bar_and(3, 128, w);
        if (!ok) {
          if (mt == 0) record_timeout(651);
          break;
        }
        // all 128 threads have read this tile's accumulator
        if (mt == 0) mbar_arrive(&o_empty[ob]);
      }
    }
  }
  // the single-lane roles (TMA producer, MMA issuer) rejoin their warps
  // before the block-wide barrier, which counts converged warps
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// T0 and T1 rows for the fused kernel when there is no global term (no state
// kernel to write them): one thread per 8 consecutive elements of Z.
__global__ void __launch_bounds__(256)
    tc_affine_rows(const __nv_bfloat16 *__restrict__ Z, const float *__restrict__ gamma,
                   const float *__restrict__ beta, __nv_bfloat16 *__restrict__ trows,
                   int64_t rows_plane, int64_t n_vec) {
  // the fused kernel may start its prologue; it waits for this grid to
  // complete before it reads the rows
  griddep_launch_dependents();
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n_vec) return;
  const int col = (int)(t % (S_DIM / 8)) * 8;
  float g0[8], b0[8], g1[8], b1[8];
  load8(gamma + col, g0);
  load8(beta + col, b0);
  load8(gamma + S_DIM + col, g1);
  load8(beta + S_DIM + col, b1);
  const uint4 z = __ldg(reinterpret_cast<const uint4 *>(Z) + t);
  reinterpret_cast<uint4 *>(trows)[t] = affine8(z, g0, b0);
  reinterpret_cast<uint4 *>(trows + rows_plane)[t] = affine8(z, g1, b1);
}

}  // namespace
}  // namespace fmca
