// bf16 backward on the 5th-generation tensor cores: a dK/dV kernel and a dQ
// kernel (mosaic_backward.py make_mosaic_backward_dkv_kernel and
// make_mosaic_backward_dq_kernel, restated for tcgen05 / TMEM), after the
// delta pre-pass.
//
// Per live pair (query i, key j), with x = temp_i * cap(s_ij) * log2(e):
//   P_ij  = 2^(x - LSE_i * log2(e))                       (0 when masked)
//   dX_ij = sm_scale * temp_i * cap'(s_ij) * P_ij * (dP_ij - delta_i + z * LSE_i)
//
// dK/dV: one CTA per (batch, KV head, 128-key tile).  K and V stay in shared
// memory; the CTA loops over the query heads of its GQA group and the query
// tiles of the tile's visit map, accumulating dK and dV in TMEM (the group sum
// happens in place, no reduction pass).  Per step:
//   S^T  = K Q^T, dP^T = V dO^T            (SS MMAs, M = keys, N = queries)
//   elementwise, in two halves of 64 query columns: P^T and dX^T written back
//   into TMEM as packed bf16 over the consumed columns
//   dV += P^T dO, dK += dX^T Q             (TS MMAs, K = 64 per half)
// so the tensor pipe runs the first half's dV / dK while the second half is
// computed.  TMEM: S^T [0,128), dP^T [128,256), dV [256,384), dK [384,512).
//
// dQ: one CTA per (batch, query head, 128-query tile), looping over the KV tiles
// of its visit map.  S = Q K^T, dP = dO V^T, then dQ += dX K in two halves.
// TMEM: S [0,128), dP [128,256), dQ [256,384).
//
// Warp roles in both kernels: warp 0 TMA producer, warp 1 TMEM allocator and
// MMA issuer, warps 2..5 elementwise (one TMEM lane = one tile row each).
#include <math.h>

#include "cap_math.cuh"
#include "capattn_internal.h"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

constexpr int HD = 128;
constexpr int BT = 128;                       // tile rows (queries and keys)
constexpr int SLAB = 128 * 64 * 2;
constexpr int TILE = 2 * SLAB;
constexpr int NSTAGE = 2;
constexpr int NTHREADS = 192;
constexpr int SMEM_BYTES = 2 * TILE + NSTAGE * 2 * TILE + 1024;

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32], float scale) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * scale, __uint_as_float(v[2 * e + 1]) * scale);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
}

__device__ __forceinline__ void store_zero_bf16(__nv_bfloat16* dst) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < 4; ++e) d4[e] = make_uint4(0u, 0u, 0u, 0u);
}

// ======================================================================= dK / dV
template <int METHOD>
__global__ void __launch_bounds__(NTHREADS, 1)
dkv_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
              const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[16];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ __align__(16) float4 colc[2][BT];  // per query column: lse2, rowadd, c1, tl
  __shared__ __align__(16) int4 coli[2][BT];    // per query column: live span (lo, hi, e)

  const int gb = blockIdx.x;
  const int g = gb % p.Hkv, b = gb / p.Hkv;
  const int kt = blockIdx.y;
  const int k0 = kt * BT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base, sV = base + TILE;
  const uint32_t sQD = base + 2 * TILE;  // stage s: Q at sQD + s*2*TILE, dO at + TILE

  const uint32_t bar_kv = smem_u32(&bars[0]);
  const uint32_t bar_full = smem_u32(&bars[1]);    // + s*8 (Q and dO)
  const uint32_t bar_empty = smem_u32(&bars[3]);   // + s*8
  const uint32_t bar_sdp = smem_u32(&bars[5]);
  const uint32_t bar_ew = smem_u32(&bars[6]);      // + half*8
  const uint32_t bar_final = smem_u32(&bars[8]);
  const uint32_t bar_cfull = smem_u32(&bars[9]);   // + cb*8: column constants written
  const uint32_t bar_cfree = smem_u32(&bars[11]);  // + cb*8: column constants consumed

  const uint32_t* map = p.kmap + ((size_t)b * p.nk + kt) * p.wq;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_kv, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_sdp, 1);
    mbar_init(bar_ew, 4);
    mbar_init(bar_ew + 8, 4);
    mbar_init(bar_final, 1);
    for (int c = 0; c < 2; ++c) {
      mbar_init(bar_cfull + 8 * c, 128);
      mbar_init(bar_cfree + 8 * c, 128);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int ntiles = count_tiles(map, p.wq);
  const int n = ntiles * p.G;  // steps: (query head of the group) x (visited query tile)

  if (warp == 0) {
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mdo);
      mbar_expect_tx(bar_kv, 2 * TILE);
      tma_load_4d(sK, &mk, bar_kv, 0, g, k0, b);
      tma_load_4d(sK + SLAB, &mk, bar_kv, 64, g, k0, b);
      tma_load_4d(sV, &mv, bar_kv, 0, g, k0, b);
      tma_load_4d(sV + SLAB, &mv, bar_kv, 64, g, k0, b);
      int j = 0;
      for (int hh = 0; hh < p.G && !abort_flag; ++hh) {
        const int h = g * p.G + hh;
        TileIter it(map, p.wq);
        int qt;
        while (it.next(qt)) {
          const int s = j % NSTAGE, u = j / NSTAGE;
          if (u > 0 && !mbar_wait(bar_empty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) break;
          const uint32_t sQ = sQD + s * 2 * TILE, sO = sQ + TILE;
          mbar_expect_tx(bar_full + 8 * s, 2 * TILE);
          tma_load_4d(sQ, &mq, bar_full + 8 * s, 0, h, qt * BT, b);
          tma_load_4d(sQ + SLAB, &mq, bar_full + 8 * s, 64, h, qt * BT, b);
          tma_load_4d(sO, &mdo, bar_full + 8 * s, 0, h, qt * BT, b);
          tma_load_4d(sO + SLAB, &mdo, bar_full + 8 * s, 64, h, qt * BT, b);
          ++j;
        }
      }
      drain_wait(bar_kv, 0);
      for (int jj = (j > NSTAGE ? j - NSTAGE : 0); jj < j; ++jj)
        drain_wait(bar_full + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BT, BT, 0, 0);
      constexpr uint32_t idesc_g = idesc_bf16(BT, HD, 0, 1);
      bool ok = mbar_wait(bar_kv, 0, p.status, &abort_flag);
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (!mbar_wait(bar_full + 8 * s, u & 1, p.status, &abort_flag)) break;
        tc_fence_after();
        const uint32_t sQ = sQD + s * 2 * TILE, sO = sQ + TILE;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
          mma_ss(tmem, smem_desc(sK + off, 16, 1024), smem_desc(sQ + off, 16, 1024), idesc_s, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
          mma_ss(tmem + 128u, smem_desc(sV + off, 16, 1024), smem_desc(sO + off, 16, 1024), idesc_s,
                 ks > 0);
        }
        mma_commit(bar_sdp);
        for (int half = 0; half < 2; ++half) {
          if (!mbar_wait(bar_ew + 8 * half, j & 1, p.status, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int ks = half * 4 + kk;
            const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
            mma_ts(tmem + 256u, tmem + (uint32_t)(ks * 8), smem_desc(sO + ks * 2048, SLAB, 1024),
                   idesc_g, acc);
            mma_ts(tmem + 384u, tmem + 128u + (uint32_t)(ks * 8),
                   smem_desc(sQ + ks * 2048, SLAB, 1024), idesc_g, acc);
          }
        }
        if (!ok) break;
        mma_commit(bar_empty + 8 * s);
      }
      mma_commit(bar_final);
      drain_wait(bar_final, 0);
    }
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row within the tile (TMEM lane)
    const int jrow = k0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const float zw = p.z_loss_weight;
    bool aborted = false;
    int step = 0;
    for (int hh = 0; hh < p.G && !aborted; ++hh) {
      const int h = g * p.G + hh;
      TileIter it(map, p.wq);
      int qt;
      while (it.next(qt)) {
        const int q0 = qt * BT;
        const int cb = step & 1;
        const int cu = step >> 1;
        {  // column constants of this query tile (thread r loads query row q0 + r)
          if (step >= 2 && !mbar_wait(bar_cfree + 8 * cb, (cu - 1) & 1, p.status, &abort_flag)) {
            aborted = true;
            break;
          }
          const int i = q0 + r;
          const bool valid = i < p.L;
          const size_t rr = ((size_t)b * p.Hq + h) * p.L + i;
          const float lse = valid ? p.lse[rr] : -INFINITY;
          const float dl = valid ? p.delta[rr] : 0.f;
          const float temp = (p.temp && valid) ? p.temp[(size_t)b * p.L + i] : 1.f;
          const bool fin = isfinite(lse);
          colc[cb][r] = make_float4(fin ? lse * kLog2e : 0.f, -dl + (fin ? zw * lse : 0.f),
                                    p.sm_scale * temp, temp * kLog2e);
          coli[cb][r] = valid ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
          mbar_arrive(bar_cfull + 8 * cb);
          // Every pair of the tile is live when kt lies in the query tile's full range.
          const int2 fr = p.qfull[(size_t)b * p.nq + qt];
          const bool tile_full = (kt >= fr.x) && (kt < fr.y);
          if (!mbar_wait(bar_cfull + 8 * cb, cu & 1, p.status, &abort_flag) ||
              !mbar_wait(bar_sdp, step & 1, p.status, &abort_flag)) {
            aborted = true;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t sv[64], dp[64];
            tmem_ld32(lane_base + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
            tmem_ld32(lane_base + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
            tmem_ld32(lane_base + 128u + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
            tmem_ld32(lane_base + 128u + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
            tmem_wait_ld();
            uint32_t pp[32], px[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float pv[2], xv[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int c = half * 64 + 2 * e + u;
                const float4 cc = colc[cb][c];
                float dc;
                const float cv = cap_value_grad<METHOD>(__uint_as_float(sv[2 * e + u]) * p.sm_scale,
                                                        p.cap, &dc);
                bool lv = true;
                if (!tile_full) {
                  const int4 ci = coli[cb][c];
                  lv = (jrow >= ci.x && jrow < ci.y) || jrow == ci.z;
                }
                const float P = lv ? ex2_approx(fmaf(cv, cc.w, -cc.x)) : 0.f;
                pv[u] = P;
                xv[u] = cc.z * dc * P * (__uint_as_float(dp[2 * e + u]) + cc.y);
              }
              pp[e] = pack_bf16x2(pv[0], pv[1]);
              px[e] = pack_bf16x2(xv[0], xv[1]);
            }
            tmem_st32(lane_base + half * 32, pp);
            tmem_st32(lane_base + 128u + half * 32, px);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ew + 8 * half);
          }
          mbar_arrive(bar_cfree + 8 * cb);
        }
        ++step;
      }
    }
    // ---------------------------------------------------------- epilogue
    bool have = false;
    if (n > 0 && !aborted) {
      have = mbar_wait(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
    }
    if (have || n == 0 || aborted) {
      __nv_bfloat16* dvg = static_cast<__nv_bfloat16*>(p.dv) + ((size_t)(b * p.L + jrow) * p.Hkv + g) * HD;
      __nv_bfloat16* dkg = static_cast<__nv_bfloat16*>(p.dk) + ((size_t)(b * p.L + jrow) * p.Hkv + g) * HD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (have) {
          uint32_t v[32], k[32];
          tmem_ld32(lane_base + 256u + c * 32, v);
          tmem_ld32(lane_base + 384u + c * 32, k);
          tmem_wait_ld();
          if (jrow < p.L) {
            store_row_bf16(dvg + c * 32, v, 1.f);
            store_row_bf16(dkg + c * 32, k, 1.f);
          }
        } else if (jrow < p.L) {
          store_zero_bf16(dvg + c * 32);
          store_zero_bf16(dkg + c * 32);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================= dQ
template <int METHOD>
__global__ void __launch_bounds__(NTHREADS, 1)
dq_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
             const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[16];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int hb = blockIdx.x;
  const int h = hb % p.Hq, b = hb / p.Hq;
  const int qt = p.nq - 1 - (int)blockIdx.y;
  const int g = h / p.G;
  const int q0 = qt * BT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base, sO = base + TILE;
  const uint32_t sKV = base + 2 * TILE;  // stage s: K at sKV + s*2*TILE, V at + TILE

  const uint32_t bar_q = smem_u32(&bars[0]);
  const uint32_t bar_full = smem_u32(&bars[1]);    // + s*8
  const uint32_t bar_empty = smem_u32(&bars[3]);   // + s*8
  const uint32_t bar_sdp = smem_u32(&bars[5]);
  const uint32_t bar_ew = smem_u32(&bars[6]);      // + half*8
  const uint32_t bar_final = smem_u32(&bars[8]);

  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_sdp, 1);
    mbar_init(bar_ew, 4);
    mbar_init(bar_ew + 8, 4);
    mbar_init(bar_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int n = count_tiles(map, p.wk);

  if (warp == 0) {
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      mbar_expect_tx(bar_q, 2 * TILE);
      tma_load_4d(sQ, &mq, bar_q, 0, h, q0, b);
      tma_load_4d(sQ + SLAB, &mq, bar_q, 64, h, q0, b);
      tma_load_4d(sO, &mdo, bar_q, 0, h, q0, b);
      tma_load_4d(sO + SLAB, &mdo, bar_q, 64, h, q0, b);
      TileIter it(map, p.wk);
      int t, j = 0;
      while (it.next(t)) {
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (u > 0 && !mbar_wait(bar_empty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) break;
        const uint32_t sK = sKV + s * 2 * TILE, sV = sK + TILE;
        mbar_expect_tx(bar_full + 8 * s, 2 * TILE);
        tma_load_4d(sK, &mk, bar_full + 8 * s, 0, g, t * BT, b);
        tma_load_4d(sK + SLAB, &mk, bar_full + 8 * s, 64, g, t * BT, b);
        tma_load_4d(sV, &mv, bar_full + 8 * s, 0, g, t * BT, b);
        tma_load_4d(sV + SLAB, &mv, bar_full + 8 * s, 64, g, t * BT, b);
        ++j;
      }
      drain_wait(bar_q, 0);
      for (int jj = (j > NSTAGE ? j - NSTAGE : 0); jj < j; ++jj)
        drain_wait(bar_full + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BT, BT, 0, 0);
      constexpr uint32_t idesc_g = idesc_bf16(BT, HD, 0, 1);
      bool ok = mbar_wait(bar_q, 0, p.status, &abort_flag);
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (!mbar_wait(bar_full + 8 * s, u & 1, p.status, &abort_flag)) break;
        tc_fence_after();
        const uint32_t sK = sKV + s * 2 * TILE, sV = sK + TILE;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
          mma_ss(tmem, smem_desc(sQ + off, 16, 1024), smem_desc(sK + off, 16, 1024), idesc_s, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
          mma_ss(tmem + 128u, smem_desc(sO + off, 16, 1024), smem_desc(sV + off, 16, 1024), idesc_s,
                 ks > 0);
        }
        mma_commit(bar_sdp);
        for (int half = 0; half < 2; ++half) {
          if (!mbar_wait(bar_ew + 8 * half, j & 1, p.status, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int ks = half * 4 + kk;
            mma_ts(tmem + 256u, tmem + (uint32_t)(ks * 8), smem_desc(sK + ks * 2048, SLAB, 1024),
                   idesc_g, (j > 0 || ks > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        mma_commit(bar_empty + 8 * s);
      }
      mma_commit(bar_final);
      drain_wait(bar_final, 0);
    }
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int i = q0 + r;
    const bool valid = i < p.L;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int4 ri = valid ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
    const float temp = (p.temp && valid) ? p.temp[(size_t)b * p.L + i] : 1.f;
    const size_t rr = ((size_t)b * p.Hq + h) * p.L + i;
    const float lse = valid ? p.lse[rr] : -INFINITY;
    const float dl = valid ? p.delta[rr] : 0.f;
    const bool fin = isfinite(lse);
    const float lse2 = fin ? lse * kLog2e : 0.f;
    const float rowadd = -dl + (fin ? p.z_loss_weight * lse : 0.f);
    const float c1 = p.sm_scale * temp;
    const float tl = temp * kLog2e;
    bool aborted = false;
    TileIter it(map, p.wk);
    for (int j = 0; j < n; ++j) {
      int t;
      it.next(t);
      const int k0 = t * BT;
      const bool full = (ri.x <= k0) && (ri.y >= k0 + BT);
      if (!mbar_wait(bar_sdp, j & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[64], dp[64];
        tmem_ld32(lane_base + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(lane_base + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld32(lane_base + 128u + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_ld32(lane_base + 128u + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        tmem_wait_ld();
        uint32_t px[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float xv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = half * 64 + 2 * e + u;
            float dc;
            const float cv = cap_value_grad<METHOD>(__uint_as_float(sv[2 * e + u]) * p.sm_scale, p.cap, &dc);
            const int jj = k0 + c;
            const bool lv = full || (jj >= ri.x && jj < ri.y) || jj == ri.z;
            const float P = lv ? ex2_approx(fmaf(cv, tl, -lse2)) : 0.f;
            xv[u] = c1 * dc * P * (__uint_as_float(dp[2 * e + u]) + rowadd);
          }
          px[e] = pack_bf16x2(xv[0], xv[1]);
        }
        tmem_st32(lane_base + half * 32, px);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ew + 8 * half);
      }
    }
    bool have = false;
    if (n > 0 && !aborted) {
      have = mbar_wait(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
    }
    __nv_bfloat16* dqg = static_cast<__nv_bfloat16*>(p.dq) + ((size_t)(b * p.L + i) * p.Hq + h) * HD;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (have) {
        uint32_t v[32];
        tmem_ld32(lane_base + 256u + c * 32, v);
        tmem_wait_ld();
        if (valid) store_row_bf16(dqg + c * 32, v, 1.f);
      } else if (valid) {
        store_zero_bf16(dqg + c * 32);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int METHOD>
struct BwdTcLaunch {
  static cudaError_t run(const Params& p, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mdo;
    cudaError_t e = make_bhld_map(&mq, p.q, p.B, p.L, p.Hq, HD, BT);
    if (e == cudaSuccess) e = make_bhld_map(&mk, p.k, p.B, p.L, p.Hkv, HD, BT);
    if (e == cudaSuccess) e = make_bhld_map(&mv, p.v, p.B, p.L, p.Hkv, HD, BT);
    if (e == cudaSuccess) e = make_bhld_map(&mdo, p.dO, p.B, p.L, p.Hq, HD, BT);
    if (e != cudaSuccess) return e;
    auto kdkv = dkv_tc_kernel<METHOD>;
    e = cudaFuncSetAttribute(kdkv, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prof_begin(CAPATTN_KERNEL_DKV, s);
    prof_count(CAPATTN_KERNEL_DKV, 1);
    kdkv<<<dim3(p.Hkv * p.B, p.nk), NTHREADS, SMEM_BYTES, s>>>(mq, mk, mv, mdo, p);
    prof_end(CAPATTN_KERNEL_DKV, s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kdq = dq_tc_kernel<METHOD>;
    e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prof_begin(CAPATTN_KERNEL_DQ, s);
    prof_count(CAPATTN_KERNEL_DQ, 1);
    kdq<<<dim3(p.Hq * p.B, p.nq), NTHREADS, SMEM_BYTES, s>>>(mq, mk, mv, mdo, p);
    prof_end(CAPATTN_KERNEL_DQ, s);
    return cudaGetLastError();
  }
};

}  // namespace

cudaError_t launch_bwd_bf16(const Params& p, cudaStream_t s) {
  return dispatch_cap<BwdTcLaunch>(p.cap.method, p, s);
}

}  // namespace capattn
