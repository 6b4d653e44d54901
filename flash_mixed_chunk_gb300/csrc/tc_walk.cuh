// tc_walk.cuh -- the chunk-state sums of the mixed-chunk attention forward
// pass, formed in TMEM while the chunks stream past, never written as
// per-chunk states ("FLASH: Possibly the Most Interesting Efficient
// Transformer Design Recently", section "Mixed Chunk": the decoder's
// cumulative sum of K^lin_h^T V_h over the chunks h < g, or the sum over all
// chunks without a mask).  Included by tc.cu.
//
// The chunk axis of a sequence is cut into S segments of L chunks.  A walker
// unit (segment sg, sequence b, 256 e columns) walks its segment's chunks in
// order:
//   R += T3_g^T V_g[:, slice]      M = 128 (s), N = 256, K = C keys, both
//                                  operands MN-major, accumulated in TMEM
//                                  (R = the fp32 sum of the segment's states
//                                  up to g; the first chunk's products start
//                                  it afresh)
//   causal: after chunk g, local_{g+1} = R, stored as bf16 (the segment's
//           first chunk's local sums are zero: stored as zeros only for the
//           output kernels that read them, not the row-pair one)
//   after the segment's last chunk: its total R, stored as bf16
// The epilogue reads R once per chunk and releases it to the next chunk's
// products as soon as it is read, before its stores; bidirectional walkers
// read it once per segment.
// The chunk states are never rounded; the sums are fp32 sums of the fp32
// products.  seg_carry_group (run by the row-pair kernel's idle warps, or as
// the launch tc_seg_carry) then turns the segment totals into carries (the
// sum of the segments before each, from a carried-in state when the call is
// one piece of longer sequences; the total of all when bidirectional), so that
//   prefix_g = carry_sg(g) + local_g     (causal)
//   total    = carry_0                   (bidirectional)
// which the output kernel forms as two products of the same T2 rows.  The
// global term's divisor is carried by the T2 rows (1/n; 1/(t+1) per
// position; 1/(g C) for causal chunk g with the tokens-summed divisor), which
// the walker of e slice g % ceil(e / 256) writes with T0 and T1.
//
// A unit takes 256 e columns, so each Z chunk it loads serves twice the
// columns of a 128-column slice.  The MMA issuer waits for the epilogue's read
// of R between chunks; that read, not the copies, is the kernel's chain.
// Warp roles (352 threads): 0 and 10 TMA producers (Z and V: one thread
// issues a copy every few hundred cycles, so the two streams issue in
// parallel), 1 MMA issuer, 2-5 transform (T3 = Z gamma_3 + beta_3 in place;
// T rows), 6-9 epilogue (R out as bf16 sums through a staging tile and TMA
// stores).
// Shared memory: a ring of 4 items of 48 KB (64 keys: Z [2][64][64] and V
// [4][64][64], 128-byte swizzled), one 32 KB staging tile.  TMEM: R in
// [256, 512) of the 512 columns allocated; the next chunk's products wait
// until the epilogue has read R.
#pragma once

#include "tc_common.cuh"

namespace fmca {
namespace {

constexpr int WK_THREADS = 352;
constexpr int WK_RING = 4;
constexpr int WK_KEYS = 64;            // keys per item
constexpr uint32_t WK_ITEM = 49152;
constexpr uint32_t WK_ITEM_V = 16384;  // offset of the V part of an item (after Z)
constexpr uint32_t WK_ATOM = 8192;     // one 64-column block of 64 rows
constexpr int WK_ET = 256;             // e columns per slice
constexpr uint32_t WK_OFF_STAGE = WK_RING * WK_ITEM;
constexpr uint32_t WK_STAGE_TILE = 128 * 64 * 2;  // [128 rows][64 cols] bf16
constexpr uint32_t WALK_SMEM = WK_OFF_STAGE + 2 * WK_STAGE_TILE + 1024;
constexpr uint32_t WK_COL_R = 256;
static_assert(WALK_SMEM <= 232448, "tc_chunk_walk exceeds 227 KB of shared memory");

// The T2 row weight of the global term's divisor: row t (position in its
// sequence) of chunk g.
__device__ __forceinline__ float t2_weight(int lin_norm, int causal, int t, int g, int n, int C) {
  if (lin_norm == kLinNormPosition) return 1.0f / (float)(t + 1);
  if (lin_norm == kLinNormSummed && causal) return g > 0 ? 1.0f / ((float)g * (float)C) : 0.0f;
  return 1.0f / (float)n;
}

// Units u = sg * (B * e/128) + b * e/128 + es; walker CTA w takes w, w + W, ...
__global__ void __launch_bounds__(WK_THREADS, 1)
    tc_chunk_walk(const __grid_constant__ CUtensorMap mapZ3,  // Z 3-D, box {64, 64, 2}
                  const __grid_constant__ CUtensorMap mapV3,  // V 3-D, box {64, 64, 4}
                  const __grid_constant__ CUtensorMap mapL,   // local [B*G*s][e], box {64, 128}
                  const __grid_constant__ CUtensorMap mapT,   // totals [B*S*s][e], box {64, 128}
                  const float *__restrict__ gamma, const float *__restrict__ beta,
                  __nv_bfloat16 *__restrict__ trows, int64_t rows_plane, int B, int n, int e,
                  int C, int causal, int lin_norm, int S, int L,
                  unsigned int *__restrict__ zero_count,  // cleared here if not null
                  int store_first_local,  // 0: a segment's first chunk (zero sums) is not stored
                  int tok0, int n_norm) {  // the call's first token in its sequence; divisor length
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[WK_RING], tready[WK_RING], empty[WK_RING];
  __shared__ __align__(8) uint64_t acc_full, acc_empty, mma_done;
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = n / C;
  const int n_es = (e + WK_ET - 1) / WK_ET;  // the last slice may be narrower
  const int n_slices = B * n_es;
  const int n_units = n_slices * S;
  const int W = (int)gridDim.x;
  const int items = C / WK_KEYS;  // items per chunk
  // the chunks of unit u
  auto unit_range = [&](int u, int &b, int &es, int &sg, int &g0, int &g1) {
    sg = u / n_slices;
    const int sl = u % n_slices;
    b = sl / n_es;
    es = sl % n_es;
    g0 = sg * L;
    g1 = g0 + L < G ? g0 + L : G;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < WK_RING; ++i) {
      mbar_init(&full[i], 2);  // the Z and the V producer
      mbar_init(&tready[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&acc_full, 1);  // tcgen05.commit
    mbar_init(&acc_empty, 1);
    mbar_init(&mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  // the next kernel's CTAs may take the SMs this grid leaves free, and each
  // SM as its walker ends; they read nothing of ours before their
  // grid-dependency wait.  Its counter starts at zero.
  if (threadIdx.x == 0 && blockIdx.x == 0 && zero_count != nullptr) *zero_count = 0u;
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;

  if (warp == 0 || warp == 10) {
    // =========================== TMA producers (warp 0: Z, warp 10: V)
    if (lane == 0) {
      const bool zp = warp == 0;
      tma_prefetch_desc(zp ? &mapZ3 : &mapV3);
      // V stays in L2 for the output kernel's second read where it fits; Z
      // is not read again (the T rows go out from here)
      const uint64_t pol_v = policy_evict_last(), pol_z = policy_evict_first();
      int it = 0;
      bool ok = true;
      for (int u = (int)blockIdx.x; u < n_units && ok; u += W) {
        int b, es, sg, g0, g1;
        unit_range(u, b, es, sg, g0, g1);
        for (int g = g0; g < g1 && ok; ++g)
          for (int k = 0; k < items; ++k, ++it) {
            const int slot = it % WK_RING;
            if (it >= WK_RING &&
                !mbar_wait(&empty[slot], ((it / WK_RING) - 1) & 1, kWaitLimitNs)) {
              record_timeout(700);
              ok = false;
              break;
            }
            uint8_t *sz = smem + slot * WK_ITEM;
            mbar_arrive_expect_tx(&full[slot], zp ? WK_ITEM_V : WK_ITEM - WK_ITEM_V);
            const int y = b * n + g * C + k * WK_KEYS;
            if (zp)
              tma_load_3d_hint(sz, &mapZ3, &full[slot], 0, y, 0, pol_z);
            else
              tma_load_3d_hint(sz + WK_ITEM_V, &mapV3, &full[slot], 0, y, es * (WK_ET / 64), pol_v);
          }
      }
      // the last copy issued into each slot has landed
      for (int q = (it > WK_RING ? it - WK_RING : 0); q < it; ++q)
        if (!mbar_wait(&full[q % WK_RING], (q / WK_RING) & 1, kWaitLimitNs)) record_timeout(701);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      // D[s][e] = T3^T[s][k] V[k][e]: M = 128 (s), N = 256, A and B MN-major
      constexpr uint32_t idesc = idesc_bf16_f32(128, WK_ET, true, true);
      int it = 0, j = 0;
      bool ok = true;
      for (int u = (int)blockIdx.x; u < n_units && ok; u += W) {
        int b, es, sg, g0, g1;
        unit_range(u, b, es, sg, g0, g1);
        for (int g = g0; g < g1 && ok; ++g, ++j) {
          if (j >= 1 && !mbar_wait(&acc_empty, (j - 1) & 1, kWaitLimitNs)) {
            record_timeout(710);
            ok = false;
            break;
          }
          tc_fence_after();
          // R += T3_g^T V_g: the segment's running sum, fresh at its first chunk
          const uint32_t rcol = tbase + WK_COL_R;
          const bool first = g == g0;
          for (int k = 0; k < items; ++k, ++it) {
            const int slot = it % WK_RING;
            if (!mbar_wait(&tready[slot], (it / WK_RING) & 1, kWaitLimitNs)) {
              record_timeout(711);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sz = smem_u32(smem + slot * WK_ITEM);
            // K = 16 keys per product: 16 rows of every 64-column block
#pragma unroll
            for (int kk = 0; kk < WK_KEYS / 16; ++kk) {
              const uint64_t ad = smem_desc_sw128(sz + kk * 2048, WK_ATOM, 1024);
              const uint64_t bd = smem_desc_sw128(sz + WK_ITEM_V + kk * 2048, WK_ATOM, 1024);
              mma_bf16_ss(rcol, ad, bd, idesc, (!first || (k | kk) != 0) ? 1u : 0u);
            }
            mma_commit(&empty[slot]);
          }
          if (!ok) break;
          mma_commit(&acc_full);
        }
      }
      mma_commit(&mma_done);
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(712);
    }
  } else if (warp < 6) {
    // =========================== transform warps (128 threads)
    // Thread mt owns physical 16-byte chunk p = mt % 8 of the rows r with
    // r % 8 = (mt / 8) % 8 in 64-column atom a = mt / 64 of the Z box: under
    // the 128-byte swizzle those are logical columns a*64 + cl .. + 7 of every
    // such row, so it keeps gamma/beta of only those 8 columns.
    const int mt = threadIdx.x - 64;
    const int a = mt >> 6, p = mt & 7, rb = (mt >> 3) & 7;
    const int cl = a * 64 + ((p ^ rb) << 3);
    float g0v[8], b0v[8], g1v[8], b1v[8], g2v[8], b2v[8], g3v[8], b3v[8];
    load8(gamma + cl, g0v);
    load8(beta + cl, b0v);
    load8(gamma + S_DIM + cl, g1v);
    load8(beta + S_DIM + cl, b1v);
    load8(gamma + 2 * S_DIM + cl, g2v);
    load8(beta + 2 * S_DIM + cl, b2v);
    load8(gamma + 3 * S_DIM + cl, g3v);
    load8(beta + 3 * S_DIM + cl, b3v);
    const int g_off = tok0 / C;  // the call's first chunk in its sequence
    int it = 0;
    bool ok = true;
    for (int u = (int)blockIdx.x; u < n_units && ok; u += W) {
      int b, es, sg, g0, g1;
      unit_range(u, b, es, sg, g0, g1);
      for (int g = g0; g < g1 && ok; ++g) {
        const bool rows_out = g % n_es == es;  // this unit writes the chunk's T rows
        for (int k = 0; k < items; ++k, ++it) {
          const int slot = it % WK_RING;
          const bool got = mbar_wait(&full[slot], (it / WK_RING) & 1, kWaitLimitNs);
          if (got) {
            uint8_t *sz = smem + slot * WK_ITEM;
            const int row_base = b * n + g * C + k * WK_KEYS;
#pragma unroll 4
            for (int i = 0; i < WK_KEYS / 8; ++i) {
              const int r = rb + 8 * i;
              uint4 *ptr = reinterpret_cast<uint4 *>(sz + a * WK_ATOM + r * 128 + p * 16);
              const uint4 z = *ptr;
              if (rows_out) {
                __nv_bfloat16 *dst = trows + (size_t)(row_base + r) * S_DIM + cl;
                *reinterpret_cast<uint4 *>(dst) = affine8(z, g0v, b0v);
                *reinterpret_cast<uint4 *>(dst + rows_plane) = affine8(z, g1v, b1v);
                const int t = g * C + k * WK_KEYS + r;  // position in the sequence
                *reinterpret_cast<uint4 *>(dst + 2 * rows_plane) =
                    affine8_scaled(z, g2v, b2v,
                                   t2_weight(lin_norm, causal, tok0 + t, g_off + g, n_norm, C));
              }
              *ptr = affine8(z, g3v, b3v);
            }
            fence_proxy_async_smem();
          }
          ok = named_bar_and(1, 128, got);
          if (!ok) {
            if (mt == 0) record_timeout(720);
            break;
          }
          if (mt == 0) mbar_arrive(&tready[slot]);
        }
      }
    }
  } else {
    // =========================== epilogue warps (128 threads)
    const int mt = threadIdx.x - 192;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // state row s (TMEM lane)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    uint8_t *stage = smem + WK_OFF_STAGE;
    const uint32_t rcol = tbase + lane_off + WK_COL_R;
    int j = 0;
    bool ok = true;
    // R (or zeros) out as bf16: 128 columns at a time through the staging
    // tile, two [128][64] TMA stores at (col0 + 128 h, prow) each; release:
    // R goes back to the MMA issuer once every thread has read its last
    // columns, before their stores
    auto pass = [&](bool zero, const CUtensorMap *map, int col0, int prow, bool release) {
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (mt == 0) bulk_wait_group_read<0>();  // the previous stores have read the tile
        named_bar_sync(2, 128);
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          const uint32_t c = (uint32_t)(32 * (4 * h + q));
          uint32_t r[32];
          if (zero) {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          } else {
            tmem_ld32(rcol + c, r);
            tmem_ld_wait();
          }
          uint8_t *sb = stage + (q >> 1) * WK_STAGE_TILE;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const uint32_t *v = r + 8 * c4;
            *reinterpret_cast<uint4 *>(sb + sw128_offset(row, (q & 1) * 64 + 16 * c4)) =
                make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                           pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                           pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                           pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
          }
        }
        fence_proxy_async_smem();
        if (release && h == 1) tc_fence_before();
        named_bar_sync(2, 128);
        if (mt == 0) {
          if (release && h == 1) mbar_arrive(&acc_empty);
          // a narrower last slice: the columns past e (zeros) are not stored
          if (col0 + 128 * h < e) tma_store_2d(map, stage, col0 + 128 * h, prow);
          if (col0 + 128 * h + 64 < e)
            tma_store_2d(map, stage + WK_STAGE_TILE, col0 + 128 * h + 64, prow);
          bulk_commit_group();
        }
      }
    };
    for (int u = (int)blockIdx.x; u < n_units && ok; u += W) {
      int b, es, sg, g0, g1;
      unit_range(u, b, es, sg, g0, g1);
      for (int g = g0; g < g1 && ok; ++g, ++j) {
        const bool got = mbar_wait(&acc_full, j & 1, kWaitLimitNs);
        if (!named_bar_and(2, 128, got)) {
          if (mt == 0) record_timeout(730);
          ok = false;
          break;
        }
        tc_fence_after();
        // R = the segment's sum up to and including chunk g: the next chunk's
        // local sums (causal), or after the segment's last chunk its total.
        // A segment's first chunk has zero local sums, stored only when the
        // output kernel reads them (not the row-pair one).
        if (causal && g == g0 && store_first_local)
          pass(true, &mapL, es * WK_ET, (b * G + g) * S_DIM, false);
        if (g == g1 - 1) {
          pass(false, &mapT, es * WK_ET, (b * S + sg) * S_DIM, true);
        } else if (causal) {
          pass(false, &mapL, es * WK_ET, (b * G + g + 1) * S_DIM, true);
        } else {
          // nothing of R read for this chunk
          named_bar_sync(2, 128);
          if (mt == 0) mbar_arrive(&acc_empty);
        }
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
  // launched as a programmatic dependent of the relu^2-weight kernel (the
  // stored-weights forward pass): this grid ends only after that one, so the
  // kernels after it may take its outputs as final
  griddep_wait();
}

// Segment totals -> carries for one group of 8 columns (t of B * s * e / 8),
// in place in T [B][S][s][e] (bf16): causal, carry_sg = the sum of the
// totals before segment sg (carry_0 = 0); bidirectional, the sum of all of
// them, in slot 0.  fp32 sums.
// With a carried-in state (causal: the sum of the states of the sequence's
// chunks before this call, fp32 [B][s][e]) the running sum starts from it, so
// every carry includes it; with state_out the sum of the state and all the
// totals (the state after this call) is written there, fp32.
__device__ __forceinline__ void seg_carry_group(__nv_bfloat16 *__restrict__ T, int S, int64_t se,
                                                int causal, int64_t t,
                                                const float *__restrict__ state_in,
                                                float *__restrict__ state_out) {
  const int64_t per_b = se / 8;
  const int64_t b = t / per_b, x = (t % per_b) * 8;
  __nv_bfloat16 *p = T + b * S * se + x;
  float run[8];
  if (state_in != nullptr) {
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(state_in + b * se + x));
    const float4 c = __ldcg(reinterpret_cast<const float4 *>(state_in + b * se + x + 4));
    run[0] = a.x, run[1] = a.y, run[2] = a.z, run[3] = a.w;
    run[4] = c.x, run[5] = c.y, run[6] = c.z, run[7] = c.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) run[i] = 0.f;
  }
  auto put = [&](__nv_bfloat16 *dst) {
    *reinterpret_cast<uint4 *>(dst) =
        make_uint4(pack_bf16x2(run[0], run[1]), pack_bf16x2(run[2], run[3]),
                   pack_bf16x2(run[4], run[5]), pack_bf16x2(run[6], run[7]));
  };
  // 16 segments' loads in flight before any of their carries is stored (the
  // stores go to the same slots): one round trip for up to 16 segments
  constexpr int kBatch = 16;
  for (int s0 = 0; s0 < S; s0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (s0 + k < S) v[k] = __ldcg(reinterpret_cast<const uint4 *>(p + (s0 + k) * se));
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (s0 + k < S) {
        if (causal) put(p + (s0 + k) * se);
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          run[2 * i] += bf16_lo(w[i]);
          run[2 * i + 1] += bf16_hi(w[i]);
        }
      }
    }
  }
  if (!causal) put(p);
  if (state_out != nullptr) {
    float4 *q = reinterpret_cast<float4 *>(state_out + b * se + x);
    q[0] = make_float4(run[0], run[1], run[2], run[3]);
    q[1] = make_float4(run[4], run[5], run[6], run[7]);
  }
}

// tc_seg_carry: seg_carry_group over all column groups, one thread each; a
// programmatic dependent of the walkers.
__global__ void __launch_bounds__(256)
    tc_seg_carry(__nv_bfloat16 *__restrict__ T, int B, int S, int64_t se, int causal,
                 const float *__restrict__ state_in, float *__restrict__ state_out) {
  griddep_wait();  // the walkers' totals
  griddep_launch_dependents();
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * (se / 8)) return;
  seg_carry_group(T, S, se, causal, t, state_in, state_out);
}

// tc_prefix_fixup (the form the backward pass runs): the scaled prefix
//   causal: prefix_g = f(g) (local_g + carry_{g / L}),   bidirectional: f carry_0
// bf16 [B][Gp][s][e], with f the global term's divisor as the unscaled T2 rows
// of the backward pass need it (1/n; 1 per position; 1/(g C), 0 at g = 0, for
// causal chunk g with the tokens-summed divisor).  One thread per 8 columns.
__global__ void __launch_bounds__(256)
    tc_prefix_fixup(const __nv_bfloat16 *__restrict__ local, const __nv_bfloat16 *__restrict__ carry,
                    __nv_bfloat16 *__restrict__ prefix, int B, int G, int S, int L, int64_t se,
                    int causal, int n, int C, int lin_norm) {
  const int Gp = causal ? G : 1;
  const int64_t per = se / 8;
  griddep_wait();  // the carries (or, with the states kept, the kernel before)
  griddep_launch_dependents();
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * Gp * per) return;
  const int64_t bg = t / per, x = (t % per) * 8;
  const int b = (int)(bg / Gp), g = (int)(bg % Gp);
  float f = lin_norm == kLinNormPosition ? 1.0f : 1.0f / (float)n;
  if (causal && lin_norm == kLinNormSummed) f = g > 0 ? 1.0f / ((float)g * (float)C) : 0.0f;
  const int sg = causal ? g / L : 0;
  float v[8];
  const uint4 c = *reinterpret_cast<const uint4 *>(carry + ((int64_t)b * S + sg) * se + x);
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = sg > 0 || !causal ? bf16_lo(cw[i]) : 0.f;
    v[2 * i + 1] = sg > 0 || !causal ? bf16_hi(cw[i]) : 0.f;
  }
  if (causal && g % L != 0) {  // a segment's first chunk: zero local sums, maybe not stored
    const uint4 l = *reinterpret_cast<const uint4 *>(local + ((int64_t)b * G + g) * se + x);
    const uint32_t lw[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] += bf16_lo(lw[i]);
      v[2 * i + 1] += bf16_hi(lw[i]);
    }
  }
  *reinterpret_cast<uint4 *>(prefix + bg * se + x) =
      make_uint4(pack_bf16x2(v[0] * f, v[1] * f), pack_bf16x2(v[2] * f, v[3] * f),
                 pack_bf16x2(v[4] * f, v[5] * f), pack_bf16x2(v[6] * f, v[7] * f));
}

}  // namespace
}  // namespace fmca
