// tc_pair.cuh -- the chunk-local kernel of the mixed-chunk attention core for
// chunks of 256 tokens with a global term, both 128-row tiles of a chunk in
// one unit:
//     causal:         O = U * (relu(T0 T1^T * a)^2 V_g + T2 local_g + T2 carry)
//     bidirectional:  O = U * (relu(T0 T1^T * a)^2 V_g + T2 total)
// ("FLASH: Possibly the Most Interesting Efficient Transformer Design
// Recently", section "Mixed Chunk": V-hat^quad_g, with the upper triangle
// masked when causal, plus V-hat^lin_g from the chunk walkers' local sums and
// carries, or the sum of all chunks' states when bidirectional, gated by
// U_g).  Included by tc.cu.
//
// At its start every CTA turns its share of the walkers' segment totals into
// carries (bidirectional: the total of each sequence, in its first segment's
// slot; warps 2-3, otherwise unused, and 8-11, idle until the first output
// tile) and
// counts itself on a grid counter; the producer loads no carry before every
// CTA is counted.  Causal: a segment's first chunk has no local-sum item (its
// local sum is zero and the walkers do not store it), a sequence's first
// chunk no global product at all.  Bidirectional: every chunk's one global
// item is its sequence's total.
//
// The chunk-local kernel streams V, the local sums and the carries once per
// e tile; with one row tile per unit (tc_chunk_fused) both row tiles of a
// chunk load them.  Here a unit is (chunk, run of 128-column e tiles) and
// each e tile's operands serve both row tiles, about 40% fewer bytes through
// an SM, which is what bounds the kernel (its loads take microseconds to
// land, so the bytes each SM can have in flight set the rate).
//   S   = T0_r T1^T      once per unit in stages of 128 keys (M = 128, N =
//                        128, K = s; an N = 64 product costs more than half
//                        of an N = 128 one): row tile 1 with keys 0-127 and
//                        128-255, then row tile 0 with keys 0-127 (and,
//                        bidirectional, 128-255), into the drained
//                        accumulators' columns
//   P   = relu(S a)^2    (causal: key > query -> 0) by four relu^2 warps, 64
//                        keys at a time, bf16 in TMEM, resident for the unit
//                        (causal 2 + 4 slots, bidirectional 4 + 4)
//   per e tile, r = 1 then 0:
//     O_r  = sum_k P_rk V_k + T2_r local_g + T2_r carry   (A of the first
//            from TMEM; M = 128, N = 128; the local sums and the carry are
//            two products into the same accumulator: cheaper than adding the
//            two tiles in shared memory first, which the MMA issuer would
//            wait for)
//     out  = U * O_r      eight warps (the epilogue warps columns 0-63, the
//                         relu^2 warps, idle once a unit's weights are formed,
//                         columns 64-127); O_1 drains while O_0 forms and the
//                         reverse, so each accumulator buffers the other
// Row tile 1 goes first.  Causal, it alone reads the keys 128-255, whose V
// item then goes back early for the next e tile's copies; bidirectional,
// both row tiles read the keys 128-255 first and row tile 0 frees them.
// Shared memory: a ring of 5 items of 32 KB (3-D TMA boxes of 128 rows x two
// 64-column blocks): T0 of each row tile, T1 of keys 0-127 and 128-255 (unit
// start), then per e tile V of keys 128-255 and 0-127, the local sums and the
// carry (bidirectional: the total); and the T2 rows of both row tiles (64
// KB) for the unit.
// TMEM (512 columns): O_0 [0, 128), O_1 [128, 256), P [320, 512) (causal) or
// [256, 512) (bidirectional); the score stages use [0, 128), [128, 256), then
// the same columns again once the stage before is read, all before the
// unit's first products there.
#pragma once

#include "tc_common.cuh"
#include "tc_fused.cuh"

namespace fmca {
namespace {

constexpr int PA_RING = 5;
constexpr uint32_t PA_ITEM = 32768;
constexpr uint32_t PA_OFF_B = PA_RING * PA_ITEM;   // T2 rows of both row tiles
constexpr uint32_t PAIR_SMEM = PA_OFF_B + 2 * PA_ITEM + 1024;
// relu^2 weight slots (32 TMEM columns, 64 keys each) and their first
// column: causal, row tile 0 reads keys 0-127 only (2 + 4 slots in [320,
// 512)); bidirectional, both row tiles read all 256 keys (4 + 4 in [256, 512))
template <bool kCausal>
__host__ __device__ constexpr int pair_pslots() { return kCausal ? 6 : 8; }
template <bool kCausal>
__host__ __device__ constexpr uint32_t pair_col_p() { return kCausal ? 320u : 256u; }
// warps: 0 producer, 1 MMA, 2-3 the start's carries only, 4-7 relu^2 then
// the epilogue of columns 64-127, 8-11 epilogue (columns 0-63)
constexpr int PAIR_THREADS = 384;
static_assert(PAIR_SMEM <= 232448, "tc_chunk_pair exceeds 227 KB of shared memory");

// 64-key stages of row tile r, and the P slot of its stage k
template <bool kCausal>
__device__ __forceinline__ int pair_stages(int r) {
  return kCausal && r == 0 ? 2 : 4;
}
template <bool kCausal>
__device__ __forceinline__ int pair_pslot(int r, int k) {
  return kCausal ? (r == 0 ? k : 2 + k) : (r == 1 ? k : 4 + k);
}
// Score stages (128 keys each): 0 row tile 1 keys 0-127, 1 row tile 1 keys
// 128-255, 2 row tile 0 keys 0-127, and bidirectional 3 row tile 0 keys
// 128-255; stage st is in TMEM columns [128 (st & 1), + 128)
template <bool kCausal>
__host__ __device__ constexpr int pair_sstages() { return kCausal ? 3 : 4; }
__device__ __forceinline__ int pair_srow(int st) { return st < 2 ? 1 : 0; }
__device__ __forceinline__ uint32_t pair_scol(int st) { return (uint32_t)(st & 1) * 128u; }

// Tiles t = bg * n_et + et; CTA c takes [c T / grid, (c + 1) T / grid) (equal
// cost per tile); a unit is the run of one chunk's e tiles in that range.
struct PairGrid {
  int n, G, n_et, n_tiles;
  int S, L;        // segments of the chunk axis, chunks each
  int rows_early;  // the T rows may be read before the grid-dependency wait
  int B;
  int carries;     // form the segment carries here before the first carry load
  int carry_all;   // a carried-in state: every chunk has a carry
};

struct PairUnit {
  int crow;   // first token row of the chunk in [B*n]
  int lrow;   // first row of its local sums in [B*G*s]
  int crow2;  // first row of its carry in [B*S*s]
  bool local; // not its segment's first chunk (whose local sums are zero and not stored)
  bool carry; // past the first segment
  int et0, net;
};

template <bool kState, bool kCausal>
__device__ __forceinline__ PairUnit decode_pair(int t, int net, const PairGrid &g) {
  const int bg = t / g.n_et;
  const int b = bg / g.G, c = bg % g.G;
  PairUnit f;
  f.crow = b * g.n + c * 256;
  f.lrow = bg * S_DIM;
  if (kCausal) {
    f.crow2 = (b * g.S + c / g.L) * S_DIM;
    f.local = c % g.L != 0;
    f.carry = (kState && g.carry_all) || c / g.L > 0;
  } else {
    // every chunk: the sequence's total, in its first segment's slot
    f.crow2 = b * g.S * S_DIM;
    f.local = false;
    f.carry = true;
  }
  f.et0 = t % g.n_et;
  f.net = net;
  return f;
}

// out = U * O for 64 columns of this thread's row: uv the U values (already
// loaded), taddr the TMEM address of the accumulator's columns, roff the
// element offset of the row's columns in O.
__device__ __forceinline__ void pair_gate64(const u32x8 (&uv)[4], __nv_bfloat16 *__restrict__ O,
                                            size_t roff, uint32_t taddr) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {  // 32 columns at a time
    uint32_t o32[32];
    tmem_ld32(taddr + 32 * q, o32);
    tmem_ld_wait();
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {  // 16 columns per 32-byte access
      const u32x8 &uu = uv[2 * q + c2];
      const uint32_t wv[8] = {uu.lo.x, uu.lo.y, uu.lo.z, uu.lo.w, uu.hi.x, uu.hi.y, uu.hi.z, uu.hi.w};
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int jj = 16 * c2 + 2 * i;
        o[i] = pack_bf16x2(bf16_lo(wv[i]) * __uint_as_float(o32[jj]),
                           bf16_hi(wv[i]) * __uint_as_float(o32[jj + 1]));
      }
      u32x8 ov;
      ov.lo = make_uint4(o[0], o[1], o[2], o[3]);
      ov.hi = make_uint4(o[4], o[5], o[6], o[7]);
      stg_stream(O + roff + 32 * q + 16 * c2, ov);
    }
  }
}

// kState: a carried-in state or a state out (flash_mca_forward_seq); the
// plain forward pass compiles without that code.  kCausal: causal chunks
// (masked scores, prefix sums); otherwise bidirectional (every key, the
// sequence's total).
template <bool kState, bool kCausal>
__global__ void __launch_bounds__(PAIR_THREADS, 1)
    tc_chunk_pair(const __grid_constant__ CUtensorMap mapT0,  // T0 rows, 3-D box {64, 128, 2}
                  const __grid_constant__ CUtensorMap mapT1,  // T1 rows, 3-D box {64, 128, 2}
                  const __grid_constant__ CUtensorMap mapT2,  // T2 rows, 3-D box {64, 128, 2}
                  const __grid_constant__ CUtensorMap mapV,   // V 3-D, box {64, 128, 2}
                  const __grid_constant__ CUtensorMap mapS,   // local sums 3-D, box {64, 128, 2}
                  const __grid_constant__ CUtensorMap mapCy,  // carries 3-D, box {64, 128, 2}
                  const __grid_constant__ CUtensorMap mapU,   // U 3-D, box {64, 128, 2} (L2 prefetch)
                  const __nv_bfloat16 *__restrict__ U,        // [B*n][e]
                  __nv_bfloat16 *__restrict__ O,              // [B*n][e]
                  PairGrid grid, int e, float quad_a,
                  __nv_bfloat16 *__restrict__ seg,  // segment totals -> carries, in place
                  unsigned int *__restrict__ carried,  // CTAs done with their carries
                  const float *__restrict__ state_in,  // carried-in state, or null
                  float *__restrict__ state_out) {     // the state after this call, or null
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t uq_full[FU_QUEUE], uq_empty[FU_QUEUE];
  __shared__ __align__(8) uint64_t b_full, b_empty;
  __shared__ __align__(8) uint64_t full[PA_RING], empty[PA_RING];
  constexpr int kSS = pair_sstages<kCausal>(), kPS = pair_pslots<kCausal>();
  constexpr uint32_t kColP = pair_col_p<kCausal>();
  __shared__ __align__(8) uint64_t s_full[kSS];  // stage st's scores are in TMEM
  __shared__ __align__(8) uint64_t p_full[kPS], p_empty[kPS];
  __shared__ __align__(8) uint64_t o_full[2], o_empty[2], mma_done;
  __shared__ int uq_unit[FU_QUEUE], uq_net[FU_QUEUE];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < FU_QUEUE; ++i) {
      mbar_init(&uq_full[i], 1);
      mbar_init(&uq_empty[i], 3);  // MMA issuer, relu^2 and epilogue warps
    }
    mbar_init(&b_full, 1);
    mbar_init(&b_empty, 1);
    for (int i = 0; i < PA_RING; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kSS; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < kPS; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_full[i], 1);   // tcgen05.commit
      mbar_init(&o_empty[i], 2);  // both column halves drained
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
  uint8_t *bbuf = smem + PA_OFF_B;

  // The segment carries, formed while the unit's rows, scores and weights
  // come in: warps 2-3 and 8-11 (idle until the first output tile)
  // turn this CTA's share of the column groups' totals into carries, then
  // the CTA is counted; the producer loads no carry before every CTA is.
  if (grid.carries && (warp == 2 || warp == 3 || warp >= 8)) {
    const int ct = (warp < 8 ? warp - 2 : warp - 6) * 32 + lane;  // 0 .. 191
    griddep_wait();  // the walkers' totals
    const int64_t se = (int64_t)S_DIM * e;
    const int64_t groups = (int64_t)grid.B * (se / 8);
    for (int64_t t = (int64_t)blockIdx.x * 192 + ct; t < groups; t += (int64_t)gridDim.x * 192)
      seg_carry_group(seg, grid.S, se, kCausal ? 1 : 0, t, kState ? state_in : nullptr,
                      kState ? state_out : nullptr);
    named_bar_sync(5, 192);
    // every thread's carries are stored (the barrier orders them before the
    // release)
    if (ct == 0) red_release_add_gpu(carried, 1u);
  }

  if (warp == 0) {
    // =========================== producer: unit queue, ring, T2 rows
    if (lane == 0) {
      tma_prefetch_desc(&mapT0);
      tma_prefetch_desc(&mapT1);
      tma_prefetch_desc(&mapT2);
      tma_prefetch_desc(&mapV);
      tma_prefetch_desc(&mapS);
      tma_prefetch_desc(&mapCy);
      tma_prefetch_desc(&mapU);
      int it = 0;
      bool ok = true, rows_ready = false, sums_ready = false;
      const uint64_t pol_first = policy_evict_first();
      // one ring item: waits for its slot, then one 32 KB box
      auto issue = [&](const CUtensorMap *map, int y, int z, bool last_use = false) -> bool {
        const int slot = it % PA_RING;
        if (it >= PA_RING && !mbar_wait(&empty[slot], ((it / PA_RING) - 1) & 1, kWaitLimitNs)) {
          record_timeout(802);
          return false;
        }
        mbar_arrive_expect_tx(&full[slot], PA_ITEM);
        if (last_use)
          tma_load_3d_hint(ring + slot * PA_ITEM, map, &full[slot], 0, y, z, pol_first);
        else
          tma_load_3d(ring + slot * PA_ITEM, map, &full[slot], 0, y, z);
        ++it;
        return true;
      };
      int t = (int)(((int64_t)blockIdx.x * grid.n_tiles) / gridDim.x);
      const int t_end = (int)(((int64_t)(blockIdx.x + 1) * grid.n_tiles) / gridDim.x);
      for (int j = 0; ok; ++j) {
        const int uu = t < t_end ? t : -1;
        const int net = uu >= 0 ? min(grid.n_et - t % grid.n_et, t_end - t) : 0;
        t += net;
        const int qs = j % FU_QUEUE;
        if (j >= FU_QUEUE && !mbar_wait(&uq_empty[qs], ((j / FU_QUEUE) - 1) & 1, kWaitLimitNs)) {
          record_timeout(800);
          break;
        }
        uq_unit[qs] = uu;
        uq_net[qs] = net;
        mbar_arrive(&uq_full[qs]);
        if (uu < 0) break;
        const PairUnit f = decode_pair<kState, kCausal>(uu, net, grid);
        // the T rows: with the carry kernel between their writer and this
        // grid, the writer had completed before this grid launched; otherwise
        // wait for the kernel before
        if (!grid.rows_early && !rows_ready) {
          griddep_wait();
          rows_ready = true;
        }
        // T0 of row tile 1, T1 of keys 0-127, T1 of keys 128-255, T0 of row
        // tile 0, in the order the score products use them
        ok = issue(&mapT0, f.crow + 128, 0) && issue(&mapT1, f.crow, 0) &&
             issue(&mapT1, f.crow + 128, 0) && issue(&mapT0, f.crow, 0);
        if (!ok) break;
        // T2 of both row tiles: the previous unit's global products are done
        if (j >= 1 && !mbar_wait(&b_empty, (j - 1) & 1, kWaitLimitNs)) {
          record_timeout(804);
          break;
        }
        mbar_arrive_expect_tx(&b_full, 2 * PA_ITEM);
        tma_load_3d(bbuf, &mapT2, &b_full, 0, f.crow, 0);
        tma_load_3d(bbuf + PA_ITEM, &mapT2, &b_full, 0, f.crow + 128, 0);
        for (int x = 0; x < f.net && ok; ++x) {
          const int eb = (f.et0 + x) * 2;  // first 64-column block of the e tile
          // V's last read: it may leave L2 first.  Keys 128-255 first: row
          // tile 1's first products read them
          ok = issue(&mapV, f.crow + 128, eb, true) && issue(&mapV, f.crow, eb, true);
          // the epilogue's U rows of this e tile, into L2 ahead of its loads
          // (their latency from DRAM otherwise sets the pace)
          tma_prefetch_l2_3d(&mapU, 0, f.crow + 128, eb);
          tma_prefetch_l2_3d(&mapU, 0, f.crow, eb);
          // the local sums and carries come from the kernels before: wait
          // once, before the first such load
          if (ok && !sums_ready && (f.local || f.carry)) {
            griddep_wait();
            // every CTA has formed its share of the carries
            if (grid.carries) {
              if (!wait_count_geq(carried, gridDim.x, kWaitLimitNs)) {
                record_timeout(805);
                ok = false;
                break;
              }
              fence_proxy_async_global();  // read next through the async proxy
            }
            sums_ready = true;
          }
          if (ok && f.local) ok = issue(&mapS, f.lrow, eb);
          if (ok && f.carry) ok = issue(&mapCy, f.crow2, eb);
        }
      }
      // drain: the last load issued into every ring slot has landed
      for (int q = (it > PA_RING ? it - PA_RING : 0); q < it; ++q)
        if (!mbar_wait(&full[q % PA_RING], (q / PA_RING) & 1, kWaitLimitNs)) record_timeout(803);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      // S = T0 T1^T: M = 128 rows, N = 128 keys, A and B K-major
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      // O += P V (A from TMEM) and O += T2 (local | carry) (A K-major); B MN-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, FU_ET, false, true);
      const uint32_t baddr = smem_u32(bbuf);
      int it = 0, tcnt = 0;
      bool ok = true;
      auto wait_item = [&](int item) -> bool {
        if (!mbar_wait(&full[item % PA_RING], (item / PA_RING) & 1, kWaitLimitNs)) {
          record_timeout(824);
          return false;
        }
        return true;
      };
      auto slot_addr = [&](int item) -> uint32_t {
        return smem_u32(ring + (item % PA_RING) * PA_ITEM);
      };
      for (int j = 0;; ++j) {
        const int qs = j % FU_QUEUE;
        if (!mbar_wait(&uq_full[qs], (j / FU_QUEUE) & 1, kWaitLimitNs)) {
          record_timeout(820);
          ok = false;
          break;
        }
        const int u = uq_unit[qs], unet = uq_net[qs];
        mbar_arrive(&uq_empty[qs]);
        if (u < 0) break;
        const PairUnit f = decode_pair<kState, kCausal>(u, unet, grid);
        // ---- scores, once per unit, into the accumulators' columns: the
        // previous unit's last tile has been drained from both
        const int i_a1 = it, i_k0 = it + 1, i_k1 = it + 2, i_a0 = it + 3;
        it += 4;
        if (tcnt >= 1) {
          for (int r = 0; r < 2 && ok; ++r)
            if (!mbar_wait(&o_empty[r], (tcnt - 1) & 1, kWaitLimitNs)) {
              record_timeout(825);
              ok = false;
            }
          if (!ok) break;
        }
        for (int st = 0; st < kSS && ok; ++st) {
          const int i_a = st < 2 ? i_a1 : i_a0, i_k = (st & 1) ? i_k1 : i_k0;
          if (!wait_item(i_a) || !wait_item(i_k)) {
            ok = false;
            break;
          }
          // stages 2 and 3 reuse the columns of stages 0 and 1 (row tile 1's):
          // the relu^2 warps have read them
          if (st >= 2 &&
              (!mbar_wait(&p_full[pair_pslot<kCausal>(1, (st & 1) * 2)], j & 1, kWaitLimitNs) ||
               !mbar_wait(&p_full[pair_pslot<kCausal>(1, (st & 1) * 2 + 1)], j & 1, kWaitLimitNs))) {
            record_timeout(826);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aaddr = slot_addr(i_a), kaddr = slot_addr(i_k);
          const uint32_t sd = tbase + pair_scol(st);
#pragma unroll
          for (int kk = 0; kk < S_DIM / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(sd, smem_desc_sw128(aaddr + off, 16, 1024),
                        smem_desc_sw128(kaddr + off, 16, 1024), idesc_s, kk != 0);
          }
          mma_commit(&s_full[st]);
          // the items go back after their last score product (bidirectional:
          // row tile 0 reads the keys 128-255 too)
          if (st == 1) {
            if (kCausal) mma_commit(&empty[i_k1 % PA_RING]);
            mma_commit(&empty[i_a1 % PA_RING]);
          }
          if (st == 2) {
            if (kCausal) mma_commit(&empty[i_a0 % PA_RING]);
            mma_commit(&empty[i_k0 % PA_RING]);
          }
          if (st == 3) {
            mma_commit(&empty[i_a0 % PA_RING]);
            mma_commit(&empty[i_k1 % PA_RING]);
          }
        }
        if (!ok) break;
        // ---- e tiles: row tile 1 (stages 2, 3 then 0, 1), then row tile 0
        // (stages 0, 1); O_r = sum_k P_rk V_k + T2_r (local + carry)
        for (int x = 0; x < f.net && ok; ++x, ++tcnt) {
          // il: the local sums, or the carry alone in a segment's first chunk
          const int iv1 = it, iv0 = it + 1, il = it + 2;
          const int nglob = (int)f.local + (int)f.carry;
          it += 2 + nglob;
          for (int rr = 0; rr < 2 && ok; ++rr) {
            const int r = 1 - rr;
            // the epilogue has drained O_r (the previous e tile's)
            if (tcnt >= 1 && !mbar_wait(&o_empty[r], (tcnt - 1) & 1, kWaitLimitNs)) {
              record_timeout(823);
              ok = false;
              break;
            }
            const uint32_t ocol = tbase + (uint32_t)(r * FU_ET);
            const int ns = pair_stages<kCausal>(r);
            // the unit's first tile: every score stage in the columns O_r
            // reuses has been read in full before the first product
            // overwrites them (causal: the row tile's own weights are formed;
            // bidirectional, where both row tiles' stages share the columns:
            // all weights, before the first product)
            for (int k = 0; x == 0 && (kCausal || r == 1) && k < (kCausal ? ns : kPS) && ok; ++k)
              if (!mbar_wait(&p_full[kCausal ? pair_pslot<kCausal>(r, k) : k], j & 1,
                             kWaitLimitNs)) {
                record_timeout(822);
                ok = false;
              }
            if (!ok) break;
            tc_fence_after();
            for (int q = 0; q < ns && ok; ++q) {
              // keys 128-255 first (causal row tile 0 reads keys 0-127 only)
              const int k = (r == 1 || !kCausal) ? (q + 2) % 4 : q;
              const int iv = k < 2 ? iv0 : iv1, ps = pair_pslot<kCausal>(r, k);
              if (!wait_item(iv)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t vb = slot_addr(iv) + (k & 1) * 8192;
              const uint32_t pa = tbase + kColP + (uint32_t)(32 * ps);
#pragma unroll
              for (int kk = 0; kk < KEY_STAGE / 16; ++kk)
                mma_bf16_ts(ocol, pa + 8 * kk, smem_desc_sw128(vb + kk * 2048, 16384, 1024),
                            idesc_o, (q == 0 && kk == 0) ? 0u : 1u);
              // keys 128-255 are read last by row tile 1 (causal) or row tile
              // 0 (bidirectional)
              if (k == 3 && r == (kCausal ? 1 : 0)) mma_commit(&empty[iv1 % PA_RING]);
            }
            if (!ok) break;
            if (r == 0) mma_commit(&empty[iv0 % PA_RING]);  // row tile 0 read keys 0-127 last
            if (x == 0 && r == 1 && !mbar_wait(&b_full, j & 1, kWaitLimitNs)) {
              record_timeout(827);
              ok = false;
              break;
            }
            // the global items (the local sums and the carry, each its own
            // product into the same accumulator) have landed
            if (r == 1 && nglob > 0 &&
                (!wait_item(il) || (nglob == 2 && !wait_item(il + 1)))) {
              record_timeout(828);
              ok = false;
              break;
            }
            tc_fence_after();
            for (int gi = 0; gi < nglob; ++gi) {
              const uint32_t pb = slot_addr(il + gi);
              const uint32_t ab = baddr + (uint32_t)r * PA_ITEM;
#pragma unroll
              for (int kk = 0; kk < S_DIM / 16; ++kk) {
                const uint64_t ad =
                    smem_desc_sw128(ab + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                const uint64_t bd = smem_desc_sw128(pb + kk * 2048, 16384, 1024);
                mma_bf16_ss(ocol, ad, bd, idesc_o, 1u);
              }
              if (r == 0) mma_commit(&empty[(il + gi) % PA_RING]);  // its last read
            }
            mma_commit(&o_full[r]);
          }
        }
        if (!ok) break;
        // the unit's relu^2 weights and T2 rows are done with
        for (int ps = 0; ps < kPS; ++ps) mma_commit(&p_empty[ps]);
        mma_commit(&b_empty);
      }
      // every MMA has finished before TMEM is released
      mma_commit(&mma_done);
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(829);
    }
  } else if (warp >= 4 && warp < 8) {
    // =========================== relu^2 warps (128 threads): S -> P in TMEM
    const int mt = threadIdx.x - 128;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // query row within its row tile (TMEM lane)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int tcnt = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      const int qs = j % FU_QUEUE;
      const bool got = mbar_wait(&uq_full[qs], (j / FU_QUEUE) & 1, kWaitLimitNs);
      const int u = got ? uq_unit[qs] : -1, unet = got ? uq_net[qs] : 0;
      const bool more = named_bar_and(2, 128, u >= 0);
      if (mt == 0 && got) mbar_arrive(&uq_empty[qs]);
      if (!more) {
        if (!got && mt == 0) record_timeout(840);
        break;
      }
      // the score stages in order, 64 keys at a time (one P slot each)
      for (int st = 0; st < kSS && ok; ++st) {
        const int r = pair_srow(st);
        const int qpos = r * ROW_TILE + row;  // query position within the chunk
        const bool got_s = mbar_wait(&s_full[st], j & 1, kWaitLimitNs);
        for (int h = 0; h < 2; ++h) {
          const int k = (st & 1) * 2 + h;  // 64-key stage within the row tile
          const int ps = pair_pslot<kCausal>(r, k);
          bool w = got_s;
          // the previous unit's last product that read this P slot has completed
          if (w && j >= 1) w = mbar_wait(&p_empty[ps], (j - 1) & 1, kWaitLimitNs);
          if (w) {
            uint32_t sv[2][32];
            tc_fence_after();
            const uint32_t sa = tbase + lane_off + pair_scol(st) + (uint32_t)(64 * h);
            tmem_ld32(sa, sv[0]);
            tmem_ld32(sa + 32, sv[1]);
            tmem_ld_wait();
            // relu(S a)^2 (a = 1/C by default); causal, key position > query
            // position -> 0; two keys a column, the lower key in the low half
            const int kbase = k * KEY_STAGE;
            uint32_t pk[32];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int key = kbase + c2 * 32 + 2 * i;
                float x0 = fmaxf(__uint_as_float(sv[c2][2 * i]) * quad_a, 0.f);
                float x1 = fmaxf(__uint_as_float(sv[c2][2 * i + 1]) * quad_a, 0.f);
                x0 *= x0;
                x1 *= x1;
                if (kCausal && key > qpos) x0 = 0.f;
                if (kCausal && key + 1 > qpos) x1 = 0.f;
                pk[c2 * 16 + i] = pack_bf16x2(x0, x1);
              }
            tmem_st32(tbase + lane_off + kColP + (uint32_t)(32 * ps), pk);
            tmem_st_wait();
            tc_fence_before();
          }
          ok = named_bar_and(2, 128, w);
          if (!ok) {
            if (mt == 0) record_timeout(841);
            break;
          }
          if (mt == 0) mbar_arrive(&p_full[ps]);
        }
      }
      // then columns 64-127 of the unit's output tiles (the epilogue warps
      // take 0-63)
      const PairUnit f = decode_pair<kState, kCausal>(u, unet, grid);
      for (int x = 0; x < f.net && ok; ++x, ++tcnt) {
        for (int rr = 0; rr < 2 && ok; ++rr) {
          const int r = 1 - rr;
          const size_t roff =
              (size_t)(f.crow + r * ROW_TILE + row) * (size_t)e + (f.et0 + x) * FU_ET + 64;
          // a 64-column last e tile has no upper half
          const bool live = (f.et0 + x) * FU_ET + 64 < e;
          u32x8 uv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (live) uv[c] = ldg_stream(U + roff + 16 * c);
          const bool w = mbar_wait(&o_full[r], tcnt & 1, kWaitLimitNs);
          if (w && live) {
            tc_fence_after();
            pair_gate64(uv, O, roff, tbase + lane_off + (uint32_t)(r * FU_ET + 64));
            tc_fence_before();
          }
          ok = named_bar_and(2, 128, w);
          if (!ok) {
            if (mt == 0) record_timeout(852);
            break;
          }
          if (mt == 0) mbar_arrive(&o_empty[r]);
        }
      }
    }
  } else if (warp >= 8) {
    // =========================== epilogue warps (128 threads)
    const int mt = threadIdx.x - 256;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // tile row (TMEM lane)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int tcnt = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      const int qs = j % FU_QUEUE;
      const bool got = mbar_wait(&uq_full[qs], (j / FU_QUEUE) & 1, kWaitLimitNs);
      const int u = got ? uq_unit[qs] : -1, unet = got ? uq_net[qs] : 0;
      const bool more = named_bar_and(3, 128, u >= 0);
      if (mt == 0 && got) mbar_arrive(&uq_empty[qs]);
      if (!more) {
        if (!got && mt == 0) record_timeout(850);
        break;
      }
      const PairUnit f = decode_pair<kState, kCausal>(u, unet, grid);
      for (int x = 0; x < f.net && ok; ++x, ++tcnt) {
        for (int rr = 0; rr < 2 && ok; ++rr) {
          const int r = 1 - rr;  // the order the accumulators are formed in
          // columns 0-63 of the e tile (the relu^2 warps take 64-127)
          const size_t roff = (size_t)(f.crow + r * ROW_TILE + row) * (size_t)e + (f.et0 + x) * FU_ET;
          u32x8 uv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) uv[c] = ldg_stream(U + roff + 16 * c);
          const bool w = mbar_wait(&o_full[r], tcnt & 1, kWaitLimitNs);
          if (w) {
            tc_fence_after();
            pair_gate64(uv, O, roff, tbase + lane_off + (uint32_t)(r * FU_ET));
            tc_fence_before();
          }
          ok = named_bar_and(3, 128, w);
          if (!ok) {
            if (mt == 0) record_timeout(851);
            break;
          }
          if (mt == 0) mbar_arrive(&o_empty[r]);  // this half of O_r is drained
        }
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

}  // namespace
}  // namespace fmca
