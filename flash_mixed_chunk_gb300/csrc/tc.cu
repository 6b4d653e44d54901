// tc.cu -- tensor-core path (sm_103a: tcgen05 MMA into TMEM, TMA-staged
// 128-byte-swizzled bf16 tiles, mbarrier pipelines) of the mixed-chunk
// attention forward core for bf16 I/O, s = 128, C in {128, 256}, e % 256 == 0.
//
// Three kernels per call ("FLASH: Possibly the Most Interesting Efficient
// Transformer Design Recently", section "Mixed Chunk"):
//
//   tc_chunk_state   state_g^T = V_g^T T3_g for every chunk g and 256-column
//                    slice of e; fp32 [B][G][s][e].  T3 = Z*gamma3 + beta3 is
//                    formed in shared memory on the loaded Z tile.
//   tc_state_scan    exclusive prefix over chunks (causal) or total
//                    (bidirectional) of the states, times 1/n, rounded to
//                    bf16 [B][Gp][s][e] -- the B operand of the global term.
//   tc_chunk_attn    per (chunk, 128-row tile, e slice): T0/T2 rows and T1
//                    keys formed in shared memory from one Z tile; S = T0 T1^T
//                    into TMEM; P = relu(S/C)^2 (masked) to shared memory as
//                    bf16; then for each 256-wide e tile the accumulator
//                    P V_g + T2 P_g builds up in TMEM (double-buffered), and
//                    the epilogue forms O = U * acc in the U tile's shared
//                    memory and stores it with TMA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "ptx.cuh"

namespace fmca {

// Device-side status: first bounded wait that ran out (code, where).
__device__ int g_fmca_status = 0;
__device__ int g_fmca_where = 0;

namespace {

constexpr int kStatusTimeout = 7;  // FMCA_ERR_TIMEOUT
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

__device__ __forceinline__ void record_timeout(int where) {
  if (atomicCAS(&g_fmca_status, 0, kStatusTimeout) == 0) atomicExch(&g_fmca_where, where);
}

constexpr int S_DIM = 128;     // attention width s handled by this path

// 8 consecutive floats (32-byte aligned) through the read-only cache.
__device__ __forceinline__ void load8(const float *__restrict__ p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
constexpr int E_TILE = 256;    // e columns per accumulator tile
constexpr int KEY_STAGE = 64;  // keys (or state rows) per pipeline stage

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
                  int64_t se, float inv_n, int causal) {
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

// =====================================================================
// tc_chunk_attn: one CTA per (b, g, e group, 128-row tile)
// =====================================================================
// shared memory (offsets from the 1024-aligned base):
//   [0,   64K)  Z tile of the chunk's keys, K-major (atom a = s cols 64a..64a+63
//               at a*32K, 256 rows x 128 B); turned into T1 in place; after the
//               score MMA it holds P (bf16 [128 rows][keys], key atom k at k*16K)
//   [64K, 96K)  T0 rows (2 atoms x 16K); after the score MMA: ring B, 2 slots
//               of U / O tiles (128 rows x 64 e, 16 KB)
//   [96K,128K)  T2 rows (2 atoms x 16K)
//   [128K, 224K) ring A, 3 x 32 KB slots: V stages (64 keys x 256 e) and state
//               prefix stages (64 s rows x 256 e)
// Each ring has exactly one consumer (ring A: the MMA warp; ring B: the
// epilogue warps), so a consumer never waits on a slot whose previous phase
// belongs to another consumer.
constexpr int RING_A = 3;
constexpr uint32_t SLOT_A = 32768;
constexpr int RING_B = 2;
constexpr uint32_t SLOT_B = 16384;
constexpr uint32_t OFF_T0 = 65536, OFF_T2 = 98304, OFF_RING = 131072;
constexpr uint32_t OFF_RING_B = OFF_T0;
constexpr uint32_t ATTN_SMEM = OFF_RING + RING_A * SLOT_A + 1024;
constexpr int ATTN_THREADS = 192;
static_assert(ATTN_SMEM + 512 <= 232448, "tc_chunk_attn exceeds 227 KB of shared memory");
static_assert(RING_B * SLOT_B <= OFF_T2 - OFF_T0, "ring B must fit in the T0 region");

__global__ void __launch_bounds__(ATTN_THREADS, 1)
    tc_chunk_attn(const __grid_constant__ CUtensorMap mapZ,   // box {64, 128}
                  const __grid_constant__ CUtensorMap mapV,   // box {64, 64}
                  const __grid_constant__ CUtensorMap mapP,   // box {64, 64}
                  const __grid_constant__ CUtensorMap mapU,   // box {64, 128}
                  const __grid_constant__ CUtensorMap mapO,   // box {64, 128}
                  const float *__restrict__ gamma, const float *__restrict__ beta, int n,
                  int e, int C, int G, int causal, int n_et) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t fullA[RING_A], emptyA[RING_A], fullB[RING_B], emptyB[RING_B];
  __shared__ __align__(8) uint64_t zfull, tready, sfull, pready, acc_full[2], acc_empty[2];
  __shared__ __align__(8) uint64_t mma_done;
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int R = C / 128;
  const int n_eg = e / (E_TILE * n_et);
  const int rt = blockIdx.x % R;
  int t1 = blockIdx.x / R;
  const int eg = t1 % n_eg;
  const int bg = t1 / n_eg;
  const int b = bg / G, g = bg % G;
  const int keys_n = causal ? (rt + 1) * 128 : C;
  const int nkv = keys_n / KEY_STAGE;  // V stages per e tile
  const int chunk_row = b * n + g * C;
  const int prow = (causal ? bg : b) * S_DIM;  // first row of this chunk's prefix in [.., e]
  const int a_per_et = nkv + 2;                // ring A items per e tile: V stages, 2 prefix stages
  constexpr int B_PER_ET = E_TILE / 64;        // ring B items per e tile: U quarters

  if (threadIdx.x == 0) {
    for (int i = 0; i < RING_A; ++i) {
      mbar_init(&fullA[i], 1);
      mbar_init(&emptyA[i], 1);
    }
    for (int i = 0; i < RING_B; ++i) {
      mbar_init(&fullB[i], 1);
      mbar_init(&emptyB[i], 1);
    }
    mbar_init(&zfull, 1);
    mbar_init(&tready, 1);
    mbar_init(&sfull, 1);
    mbar_init(&pready, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
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
  uint8_t *zt = smem;
  uint8_t *t0 = smem + OFF_T0;
  uint8_t *t2 = smem + OFF_T2;
  uint8_t *ringA = smem + OFF_RING;
  uint8_t *ringB = smem + OFF_RING_B;

  if (warp == 0) {
    // =========================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mapZ);
      tma_prefetch_desc(&mapV);
      tma_prefetch_desc(&mapP);
      tma_prefetch_desc(&mapU);
      mbar_arrive_expect_tx(&zfull, (uint32_t)keys_n * S_DIM * 2);
      for (int kh = 0; kh < keys_n / 128; ++kh)
        for (int a = 0; a < 2; ++a)
          tma_load_2d(zt + a * 32768 + kh * 16384, &mapZ, &zfull, 64 * a, chunk_row + 128 * kh);
      int ia = 0, ib = 0;
      bool ok = true;
      for (int et = 0; et < n_et && ok; ++et) {
        const int e0 = (eg * n_et + et) * E_TILE;
        for (int k = 0; k < a_per_et; ++k, ++ia) {
          const int slot = ia % RING_A;
          if (ia >= RING_A &&
              !mbar_wait(&emptyA[slot], ((ia / RING_A) - 1) & 1, kWaitLimitNs)) {
            record_timeout(201);
            ok = false;
            break;
          }
          uint8_t *dst = ringA + slot * SLOT_A;
          mbar_arrive_expect_tx(&fullA[slot], SLOT_A);
          if (k < nkv) {  // V keys [64k, 64k+64) x e cols [e0, e0+256)
            const int y = chunk_row + k * KEY_STAGE;
            for (int i = 0; i < 4; ++i) tma_load_2d(dst + i * 8192, &mapV, &fullA[slot], e0 + 64 * i, y);
          } else {  // prefix rows [64q, 64q+64) x [e0, e0+256)
            const int y = prow + (k - nkv) * KEY_STAGE;
            for (int i = 0; i < 4; ++i) tma_load_2d(dst + i * 8192, &mapP, &fullA[slot], e0 + 64 * i, y);
          }
        }
        if (!ok) break;
        // ring B lives over T0, which is free once the score MMA has retired
        if (et == 0 && !mbar_wait(&sfull, 0, kWaitLimitNs)) {
          record_timeout(204);
          ok = false;
          break;
        }
        for (int q = 0; q < B_PER_ET; ++q, ++ib) {
          const int slot = ib % RING_B;
          if (ib >= RING_B &&
              !mbar_wait(&emptyB[slot], ((ib / RING_B) - 1) & 1, kWaitLimitNs)) {
            record_timeout(205);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&fullB[slot], SLOT_B);
          tma_load_2d(ringB + slot * SLOT_B, &mapU, &fullB[slot], e0 + 64 * q, chunk_row + rt * 128);
        }
      }
      // drain: the last load issued into every slot has landed
      for (int q = (ia > RING_A ? ia - RING_A : 0); q < ia; ++q)
        if (!mbar_wait(&fullA[q % RING_A], (q / RING_A) & 1, kWaitLimitNs)) record_timeout(202);
      for (int q = (ib > RING_B ? ib - RING_B : 0); q < ib; ++q)
        if (!mbar_wait(&fullB[q % RING_B], (q / RING_B) & 1, kWaitLimitNs)) record_timeout(206);
      if (!mbar_wait(&zfull, 0, kWaitLimitNs)) record_timeout(203);
    }
  } else if (warp == 1) {
    // =========================== MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(&tready, 0, kWaitLimitNs);
      if (!ok) record_timeout(211);
      if (ok) {
        tc_fence_after();
        // S[128 rows][keys] = T0 * T1^T, both K-major, K = s
        const uint32_t idesc_s = idesc_bf16_f32(128, (uint32_t)keys_n, false, false);
        const uint32_t a0 = smem_u32(t0), b0 = smem_u32(zt);
        for (int j = 0; j < S_DIM / 16; ++j) {
          const uint64_t ad = smem_desc_sw128(a0 + (j >> 2) * 16384 + (j & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(b0 + (j >> 2) * 32768 + (j & 3) * 32, 16, 1024);
          mma_bf16_ss(tbase, ad, bd, idesc_s, j > 0);
        }
        mma_commit(&sfull);
        ok = mbar_wait(&pready, 0, kWaitLimitNs);
        if (!ok) record_timeout(212);
      }
      // acc[rows][256 e] = P * V (A K-major, B MN-major) + T2 * Pg (same)
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, E_TILE, false, true);
      const uint32_t pbase = smem_u32(zt), t2base = smem_u32(t2);
      int ia = 0;
      for (int et = 0; et < n_et && ok; ++et) {
        const int buf = (et & 1) ? 0 : 1;  // tile 0 -> cols 256.., tile 1 -> cols 0..
        const int use = et >> 1;
        if (use >= 1 && !mbar_wait(&acc_empty[buf], (use - 1) & 1, kWaitLimitNs)) {
          record_timeout(213);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dcol = tbase + (buf ? 256u : 0u);
        for (int k = 0; k < a_per_et; ++k, ++ia) {
          const int slot = ia % RING_A;
          if (!mbar_wait(&fullA[slot], (ia / RING_A) & 1, kWaitLimitNs)) {
            record_timeout(214);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = smem_u32(ringA + slot * SLOT_A);
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = smem_desc_sw128(sb + kk * 2048, 8192, 1024);
            uint64_t ad;
            if (k < nkv)
              ad = smem_desc_sw128(pbase + k * 16384 + kk * 32, 16, 1024);
            else
              ad = smem_desc_sw128(t2base + (k - nkv) * 16384 + kk * 32, 16, 1024);
            mma_bf16_ss(dcol, ad, bd, idesc_o, (k | kk) != 0);
          }
          mma_commit(&emptyA[slot]);
        }
        if (!ok) break;
        mma_commit(&acc_full[buf]);
      }
      // every MMA has finished before TMEM is released
      mma_commit(&mma_done);
      if (!mbar_wait(&mma_done, 0, kWaitLimitNs)) record_timeout(215);
    }
  } else {
    // =========================== math warps (128 threads)
    // Every named barrier below is a consensus barrier, so the four warps
    // always take the same path even when a bounded wait runs out.
    const int mt = threadIdx.x - 64;
    const int quad = warp & 3;            // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;     // accumulator row = TMEM lane
    const int ro = rt * 128;              // first row of this tile inside the Z tile
    bool got = mbar_wait(&zfull, 0, kWaitLimitNs);
    // ---- T0 and T2 from the tile's rows (same swizzle position: ro % 8 == 0)
    if (got) {
      for (int x = mt; x < 2048; x += 128) {
        const int a = x >> 10, r = (x >> 3) & 127, p = x & 7;
        const uint4 v = *reinterpret_cast<const uint4 *>(zt + a * 32768 + (ro + r) * 128 + p * 16);
        const int c = a * 64 + ((p ^ (r & 7)) << 3);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float g0[8], b0[8], g2[8], b2[8];
        load8(gamma + c, g0);
        load8(beta + c, b0);
        load8(gamma + 2 * S_DIM + c, g2);
        load8(beta + 2 * S_DIM + c, b2);
        uint32_t o0[4], o2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
          o0[i] = pack_bf16x2(lo * g0[2 * i] + b0[2 * i], hi * g0[2 * i + 1] + b0[2 * i + 1]);
          o2[i] = pack_bf16x2(lo * g2[2 * i] + b2[2 * i], hi * g2[2 * i + 1] + b2[2 * i + 1]);
        }
        *reinterpret_cast<uint4 *>(t0 + a * 16384 + r * 128 + p * 16) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
        *reinterpret_cast<uint4 *>(t2 + a * 16384 + r * 128 + p * 16) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
      }
    }
    bool ok = named_bar_and(1, 128, got);
    if (!ok && mt == 0) record_timeout(221);
    // ---- T1 in place over the keys
    if (ok) {
      const int nch = keys_n * 16;  // 2 atoms x keys_n rows x 8 chunks
      for (int x = mt; x < nch; x += 128) {
        const int a = x / (keys_n * 8), rem = x % (keys_n * 8);
        const int r = rem >> 3, p = rem & 7;
        uint4 *ptr = reinterpret_cast<uint4 *>(zt + a * 32768 + r * 128 + p * 16);
        const uint4 v = *ptr;
        const int c = a * 64 + ((p ^ (r & 7)) << 3);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float g1[8], b1[8];
        load8(gamma + S_DIM + c, g1);
        load8(beta + S_DIM + c, b1);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = pack_bf16x2(bf16_lo(w[i]) * g1[2 * i] + b1[2 * i],
                             bf16_hi(w[i]) * g1[2 * i + 1] + b1[2 * i + 1]);
        *ptr = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (mt == 0) mbar_arrive(&tready);
      __syncwarp();
    }
    // ---- P = relu(S / C)^2 (masked) as bf16 over the Z tile
    if (ok) {
      got = mbar_wait(&sfull, 0, kWaitLimitNs);
      if (got) {
        tc_fence_after();
        const float inv_c = 1.0f / (float)C;
        const int qpos = ro + row;  // position of this row inside the chunk's key range
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
        if (ok) mbar_arrive(&pready);
        else record_timeout(222);
      }
      __syncwarp();
    }
    // ---- epilogue per e tile: O = U * acc in ring B, TMA store per 64 columns
    int ib = 0;
    for (int et = 0; et < n_et && ok; ++et) {
      const int e0 = (eg * n_et + et) * E_TILE;
      const int buf = (et & 1) ? 0 : 1;
      const int use = et >> 1;
      const bool acc_ok = mbar_wait(&acc_full[buf], use & 1, kWaitLimitNs);
      if (acc_ok) tc_fence_after();
      const uint32_t dcol = tbase + (buf ? 256u : 0u) + ((uint32_t)(quad * 32) << 16);
      for (int q = 0; q < B_PER_ET; ++q, ++ib) {
        const int slot = ib % RING_B;
        got = acc_ok && mbar_wait(&fullB[slot], (ib / RING_B) & 1, kWaitLimitNs);
        uint8_t *us = ringB + slot * SLOT_B;
        if (got) {
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t r[32];
            tmem_ld32(dcol + q * 64 + c2 * 32, r);
            tmem_ld_wait();
            const uint32_t byte0 = c2 * 64;
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              uint4 *ptr = reinterpret_cast<uint4 *>(us + sw128_offset(row, byte0 + 16 * j4));
              const uint4 uv = *ptr;
              const uint32_t w[4] = {uv.x, uv.y, uv.z, uv.w};
              uint32_t o[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int j = 8 * j4 + 2 * i;
                o[i] = pack_bf16x2(bf16_lo(w[i]) * __uint_as_float(r[j]),
                                   bf16_hi(w[i]) * __uint_as_float(r[j + 1]));
              }
              *ptr = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
          fence_proxy_async_smem();
        }
        ok = named_bar_and(1, 128, got);
        if (!ok) {
          if (mt == 0) record_timeout(224);
          break;
        }
        if (mt == 0) {
          tma_store_2d(&mapO, us, e0 + 64 * q, chunk_row + rt * 128);
          bulk_commit_group();
          bulk_wait_group_read<0>();
          mbar_arrive(&emptyB[slot]);
        }
        __syncwarp();
      }
      if (!ok) break;
      tc_fence_before();
      named_bar_sync(1, 128);
      if (mt == 0) mbar_arrive(&acc_empty[buf]);
      __syncwarp();
    }
    if (mt == 0) bulk_wait_group<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// A kernel whose only wait can never complete: exercises the bounded-wait
// exit path (records a timeout, returns) without hanging the GPU.
__global__ void tc_timeout_selftest(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, limit_ns)) record_timeout(900);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [rows][cols] matrix, 128-byte swizzle.
bool make_map_bf16(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e tiles per attention CTA: enough CTAs to cover the SMs at least twice, else 1.
int pick_n_et(int B, int G, int R, int e) {
  const int n_tiles = e / E_TILE;
  int best = 1;
  for (int d = 1; d <= n_tiles; ++d) {
    if (n_tiles % d) continue;
    const long ctas = (long)B * G * R * (n_tiles / d);
    if (ctas >= 2 * 148) best = d;
  }
  return best;
}

}  // namespace

bool tc_supported(int B, int n, int s, int e, int C) {
  if (s != S_DIM) return false;
  if (C != 128 && C != 256) return false;
  if (e % E_TILE) return false;
  if (n % C) return false;
  (void)B;
  return true;
}

int tc_launch_count() { return 3; }

int launch_tc_forward(const void *Z, const void *V, const void *U, const float *gamma,
                      const float *beta, void *O, int B, int n, int s, int e, int C, int causal,
                      void *workspace, cudaStream_t stream, cudaEvent_t const *events) {
  const int G = n / C;
  const int R = C / 128;
  const int64_t se = (int64_t)s * e;
  float *states = static_cast<float *>(workspace);
  __nv_bfloat16 *prefix = reinterpret_cast<__nv_bfloat16 *>(
      static_cast<char *>(workspace) + align256(sizeof(float) * (size_t)B * G * se));
  const int Gp = causal ? G : 1;

  CUtensorMap mZs, mVs, mZ, mV, mP, mU, mO;
  const uint64_t rows = (uint64_t)B * n;
  if (!make_map_bf16(&mZs, Z, s, rows, 64, 64) || !make_map_bf16(&mVs, V, e, rows, 64, 64) ||
      !make_map_bf16(&mZ, Z, s, rows, 64, 128) || !make_map_bf16(&mV, V, e, rows, 64, 64) ||
      !make_map_bf16(&mP, prefix, e, (uint64_t)B * Gp * s, 64, 64) ||
      !make_map_bf16(&mU, U, e, rows, 64, 128) || !make_map_bf16(&mO, O, e, rows, 64, 128))
    return 2;

  static bool attrs = false;
  if (!attrs) {
    if (cudaFuncSetAttribute(tc_chunk_state, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)STATE_SMEM) != cudaSuccess)
      return 1;
    if (cudaFuncSetAttribute(tc_chunk_attn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ATTN_SMEM) != cudaSuccess)
      return 1;
    attrs = true;
  }
  if (!record_event(events, 0, stream)) return 1;
  tc_chunk_state<<<B * G * (e / E_TILE), STATE_THREADS, STATE_SMEM, stream>>>(
      mZs, mVs, gamma, beta, states, n, e, C, G);
  if (cudaGetLastError() != cudaSuccess || !record_event(events, 1, stream)) return 1;
  const int64_t lanes = (int64_t)B * se / 8;
  tc_state_scan<<<(unsigned)((lanes + 255) / 256), 256, 0, stream>>>(states, prefix, B, G, se,
                                                                     1.0f / (float)n, causal);
  if (cudaGetLastError() != cudaSuccess || !record_event(events, 2, stream)) return 1;
  const int n_et = pick_n_et(B, G, R, e);
  const int n_eg = e / (E_TILE * n_et);
  tc_chunk_attn<<<B * G * R * n_eg, ATTN_THREADS, ATTN_SMEM, stream>>>(
      mZ, mV, mP, mU, mO, gamma, beta, n, e, C, G, causal, n_et);
  if (cudaGetLastError() != cudaSuccess || !record_event(events, 3, stream)) return 1;
  return 0;
}

int read_and_clear_device_status(cudaStream_t stream, int32_t *where) {
  int st = 0, wh = 0;
  const int zero = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(&st, g_fmca_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(&wh, g_fmca_where, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_fmca_status, &zero, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_fmca_where, &zero, sizeof(int)) != cudaSuccess) return -1;
  if (where) *where = wh;
  return st;
}

int launch_timeout_selftest(int limit_us, cudaStream_t stream) {
  tc_timeout_selftest<<<1, 32, 0, stream>>>((uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace fmca
