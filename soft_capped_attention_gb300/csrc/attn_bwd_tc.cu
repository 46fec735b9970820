// bf16 backward on the 5th-generation tensor cores: a dK/dV kernel and a dQ
// kernel (mosaic_backward.py make_mosaic_backward_dkv_kernel and
// make_mosaic_backward_dq_kernel, restated for tcgen05 / TMEM), after the
// delta pre-pass.
//
// Per live pair (query i, key j), with x = temp_i * cap(s_ij) * log2(e):
//   P_ij  = 2^(x - LSE_i * log2(e))                       (0 when masked)
//   dX_ij = sm_scale * temp_i * cap'(s_ij) * P_ij * (dP_ij - delta_i + z * LSE_i + dLSE_i)
// (dLSE: an optional upstream gradient of the forward's LSE, 0 without one)
//
// Both kernels work in 128 x 128 steps with four tcgen05 phases per step:
// score MMAs (S and dP, N = 128, separately committed), the elementwise pass,
// and the accumulation MMAs, handed over in 16-column chunks as the
// elementwise warps finish them.  The elementwise warps copy their S columns
// to registers first and release them, so the next step's S MMAs run during
// this step's elementwise pass; P / dX are packed to bf16 over the dP columns
// already read, and the next step's dP MMAs follow the last chunk.
//
// dK/dV: one CTA per (batch, KV head, 128-key tile).  K and V stay in shared
// memory; the CTA loops over the query heads of its GQA group and the query
// tiles of the tile's visit map, accumulating dK and dV in TMEM (the group sum
// happens in place): S^T = K Q^T, dP^T = V dO^T (SS MMAs, M = keys); dV += P^T
// dO, dK += dX^T Q (TS MMAs).  TMEM: S^T [0, 128), dP^T [128, 256), dV
// [256, 384), dK [384, 512).
//
// dQ: one CTA per (batch, query head, 128-query tile), looping over the KV
// tiles of its visit map: S = Q K^T, dP = dO V^T; dQ += dX K (TS MMAs).  TMEM:
// S [0, 128), dP [128, 256), dQ [256, 384).
//
// Warp roles in both kernels (10 warps): warp 0 TMA producer, warp 1 TMEM
// allocator and MMA issuer (both run their loops warp-wide; one elected lane
// issues), warps 2..5 and 6..9 the two elementwise warpgroups (one TMEM lane =
// one tile row each; each warpgroup owns 64 columns).
#include <math.h>

#include "cap_math.cuh"
#include "capattn_internal.h"
#include "row_span.h"
#include "softmax_elem.cuh"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

constexpr int BT = 128;                       // tile rows (queries and keys)
constexpr int SLAB = 128 * 64 * 2;
// A 128-row tile of head dim HD (64 or 128) is HD / 64 slabs.
template <int HD>
constexpr int tile_bytes() { return (HD / 64) * SLAB; }
constexpr int NSTAGE = 2;
constexpr int NTHREADS = 320;
template <int HD>
constexpr int smem_bytes() { return 2 * tile_bytes<HD>() + NSTAGE * 2 * tile_bytes<HD>() + 1024; }


// 32 fp32 values of row r as bf16 into 16-byte chunks q0 .. q0 + 3 of a
// swizzled [128][64] bf16 slab (the layout the TMA store reads).
__device__ __forceinline__ void st_row32_swz(uint32_t slab, int r, int q0, const uint32_t (&v)[32]) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
#pragma unroll
  for (int e = 0; e < 4; ++e) st_swz_chunk(slab, r, q0 + e, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
}

// Steps of the dK/dV kernel: (query head of the group) x (visited query tile).
struct StepIter {
  const uint32_t* map;
  int nwords, G, hh;
  TileIter it;
  __device__ StepIter(const uint32_t* m, int n, int g) : map(m), nwords(n), G(g), hh(0), it(m, n) {}
  __device__ bool next(int& h_out, int& qt) {
    while (hh < G) {
      if (it.next(qt)) {
        h_out = hh;
        return true;
      }
      ++hh;
      it = TileIter(map, nwords);
    }
    return false;
  }
};

// Raw per-query-column inputs of one step, loaded ahead of use and left
// untouched until then (arithmetic on them here would stall on the loads).
struct ColRaw {
  float lse, dl, gl, temp;  // gl: upstream gradient of the LSE (0 without one)
  int4 ri;
};

__device__ __forceinline__ ColRaw load_col_raw(const Params& p, int b, int h, int qt, int c, bool active) {
  ColRaw r;
  r.lse = -INFINITY;
  r.dl = 0.f;
  r.gl = 0.f;
  r.temp = 1.f;
  r.ri = make_int4(0, 0, -1, 0);
  const int i = qt * BT + c;
  if (active && i < p.L) {
    const size_t rr = ((size_t)b * p.Hq + h) * p.L + i;
    r.lse = p.lse[rr];
    r.dl = p.delta[rr];
    if (p.dlse) r.gl = p.dlse[rr];
    if (p.temp) r.temp = p.temp[(size_t)b * p.L + i];
    r.ri = p.rowinfo[(size_t)b * p.L + i];
  }
  return r;
}

// ======================================================================= dK / dV
// Score MMAs of a whole step: D[128 x 128] = A[128 x 128] B^T, both K-major,
// from the tiles' descriptors.
template <int HD>
__device__ __forceinline__ void issue_scores(uint32_t d, uint64_t dA, uint64_t dB) {
  constexpr uint32_t idesc = idesc_bf16(BT, BT, 0, 0);
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
    mma_ss(d, desc_add(dA, off), desc_add(dB, off), idesc, ks > 0 ? 1u : 0u);
  }
}

// Per-step constants of a pair of query columns (c, c + 1), each half of a float4
// being one packed f32x2 operand:
//   a = (mul_c, mul_c+1, addl_c, addl_c+1)         x = mul * f + addl  (log2 domain, LSE folded in)
//   b = (ndsc_c, ndsc_c+1, ndr_c, ndr_c+1)         ndsc = -dscale, ndr = -dscale * radd
struct ColPair {
  float4 a, b;
};

// P and dX of one pair of scores of a key row, packed to bf16:
//   P  = 2^(mul f(X) + addl)                        (0 where masked)
//   dX = dscale f'(X) P (dP + radd) = (-f') P (ndsc dP + ndr)
// For the tanh cap, -f' = f^2 - 1; with POLY, tanh runs on the FMA pipe through
// the polynomial with the argument scale folded in (the caller guarantees
// |X in| <= 0.5 and usable coefficients for the whole warp).
// Temperature gradient terms of a row (dQ kernel): dT = P (dP + radd) and the
// capped score c = kc f + bc, accumulated as sum dT c.
struct DtempRow {
  F2 radd, kc, bc;
};

template <int METHOD, bool POLY, bool DT = false>
__device__ __forceinline__ void dkv_pair(float X0, float X1, float dp0, float dp1, const Xf& xf,
                                         const TanhFold& tf, const ColPair& c, bool l0, bool l1,
                                         uint32_t& pk, uint32_t& xk, const DtempRow* dr = nullptr,
                                         F2* dacc = nullptr, const CapConsts* cap = nullptr) {
  F2 f, e;
  if constexpr (METHOD == CAPATTN_CAP_ALSC && POLY) {
    // the sigmoid on the FMA pipe (the caller checked |X| <= alsc_xmax for the
    // warp); -f' = f^2 - f
    f = f2_add(f2(cap->alsc_sb, cap->alsc_sb), alsc_poly2(f2(X0, X1), *cap));
    e = f2_mul(f, f2_add(f, f2(-1.f, -1.f)));
  } else if constexpr (METHOD == CAPATTN_CAP_TANH) {
    if constexpr (POLY) {
      f = tanh_fold_eval(f2(X0, X1), tf, f2(0.f, 0.f));   // tanh(in X) = X Q(X^2)
    } else {
      float a, b;
      f2_split(f2_mul(f2(X0, X1), f2(xf.in, xf.in)), a, b);
      f = f2(tanh_approx(a), tanh_approx(b));
    }
    e = f2_fma(f, f, f2(-1.f, -1.f));
  } else {
    float d0, d1;
    const float f0 = cap_f_d<METHOD>(X0, xf, &d0);
    const float f1 = cap_f_d<METHOD>(X1, xf, &d1);
    f = f2(f0, f1);
    e = f2(-d0, -d1);
  }
  float x0, x1;
  f2_split(f2_fma(f2(c.a.x, c.a.y), f, f2(c.a.z, c.a.w)), x0, x1);
  const float P0 = l0 ? ex2_approx(x0) : 0.f;
  const float P1 = l1 ? ex2_approx(x1) : 0.f;
  const F2 h = f2_fma(f2(dp0, dp1), f2(c.b.x, c.b.y), f2(c.b.z, c.b.w));
  float g0, g1;
  f2_split(f2_mul(e, f2_mul(f2(P0, P1), h)), g0, g1);
  pk = pack_bf16x2(P0, P1);
  xk = pack_bf16x2(g0, g1);
  if constexpr (DT) {
    const F2 dT = f2_mul(f2(P0, P1), f2_add(f2(dp0, dp1), dr->radd));
    *dacc = f2_fma(dT, f2_fma(dr->kc, f, dr->bc), *dacc);
  }
}

constexpr int kDkvPolyPairs = 5;  // of the 8 column pairs of a chunk: tanh on the FMA pipe

// One 16-column chunk (columns 16 C .. 16 C + 15 of the warpgroup's 64) of a key
// row: S values from the row's register copy, dP from dp.
template <int METHOD, bool MASKED, bool POLY, int C>
__device__ __forceinline__ void dkv_chunk(const uint32_t (&s)[64], const uint32_t (&dp)[16],
                                          const ColPair* cp, const int4* ci, int jrow, const Xf& xf,
                                          const TanhFold& tf, const CapConsts& cap, uint32_t (&pk)[8],
                                          uint32_t (&xk)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const ColPair c = cp[8 * C + e];
    bool l0 = true, l1 = true;
    if constexpr (MASKED) {
      const int4 a = ci[16 * C + 2 * e], b = ci[16 * C + 2 * e + 1];
      l0 = (jrow >= a.x && jrow < a.y) || jrow == a.z;
      l1 = (jrow >= b.x && jrow < b.y) || jrow == b.z;
    }
    const float X0 = __uint_as_float(s[16 * C + 2 * e]), X1 = __uint_as_float(s[16 * C + 2 * e + 1]);
    const float d0 = __uint_as_float(dp[2 * e]), d1 = __uint_as_float(dp[2 * e + 1]);
    if (POLY && (METHOD == CAPATTN_CAP_ALSC || e < kDkvPolyPairs))
      dkv_pair<METHOD, true>(X0, X1, d0, d1, xf, tf, c, l0, l1, pk[e], xk[e], nullptr, nullptr, &cap);
    else
      dkv_pair<METHOD, false>(X0, X1, d0, d1, xf, tf, c, l0, l1, pk[e], xk[e]);
  }
}

// The warpgroup's 64 columns of one step, chunk by chunk: dP of chunk C + 1 is
// loaded while chunk C is computed; the packed P^T and dX^T of chunk C overwrite
// its dP columns ([16 C, 16 C + 8) and [16 C + 8, 16 C + 16) of the warpgroup's
// range) and the chunk is handed to the MMA issuer.
// Stored-dX backward (dxo != kNoDx): after chunk C's hand-off (whose release
// would otherwise wait for the store), the thread writes its 16 dX values of
// the chunk, 32 bytes, at 32-byte unit dxo + 128 C of the pool.  The pool
// keeps each tile in the layout of a 32-byte-swizzled MN-major MMA operand:
// eight blocks of 16 query columns, each 128 key rows of 32 bytes, with the
// two 16-byte halves of rows 4..7 of every 8 swapped (the swizzle).  A warp's
// store then covers 1 KB of consecutive bytes.
constexpr uint32_t kNoDx = 0xFFFFFFFFu;
template <int METHOD, bool MASKED, bool POLY, bool DX>
__device__ __forceinline__ void dkv_step(const uint32_t (&s)[64], uint32_t dp_base, const ColPair* cp,
                                         const int4* ci, int jrow, const Xf& xf, const TanhFold& tf,
                                         const CapConsts& cap, uint32_t bar_chunk0, int lane, char* pool,
                                         uint32_t dxo) {
  uint32_t da[16], db[16], pk[8], xk[8];
  tmem_ld16(dp_base, da);
  tmem_wait_ld();
#define CAPATTN_DKV_CHUNK(C, CUR, NXT)                                                     \
  {                                                                                       \
    if (C < 3) tmem_ld16(dp_base + 16 * (C + 1), NXT);                                    \
    dkv_chunk<METHOD, MASKED, POLY, C>(s, CUR, cp, ci, jrow, xf, tf, cap, pk, xk);        \
    __syncwarp();                                                                         \
    tmem_st8(dp_base + 16 * C, pk);                                                       \
    tmem_st8(dp_base + 16 * C + 8, xk);                                                   \
    tmem_wait_st();                                                                       \
    if (C < 3) tmem_wait_ld();                                                            \
    tc_fence_before();                                                                    \
    __syncwarp();                                                                         \
    if (lane == 0) mbar_arrive(bar_chunk0 + 8 * C);                                       \
    if (DX && dxo != kNoDx) {                                                             \
      const bool sw = (lane >> 2) & 1;                                                    \
      st_global_v8(pool + 32 * (size_t)(dxo + 128u * C), sw ? xk[4] : xk[0],               \
                   sw ? xk[5] : xk[1], sw ? xk[6] : xk[2], sw ? xk[7] : xk[3],            \
                   sw ? xk[0] : xk[4], sw ? xk[1] : xk[5], sw ? xk[2] : xk[6],            \
                   sw ? xk[3] : xk[7]);                                                   \
    }                                                                                     \
  }
  CAPATTN_DKV_CHUNK(0, da, db)
  CAPATTN_DKV_CHUNK(1, db, da)
  CAPATTN_DKV_CHUNK(2, da, db)
  CAPATTN_DKV_CHUNK(3, db, da)
#undef CAPATTN_DKV_CHUNK
}

// dK/dV: one CTA per (batch, KV head, 128-key tile).  K and V stay in shared
// memory; the CTA loops over the query heads of its GQA group and the query tiles
// of the tile's visit map ("steps"), accumulating dK and dV in TMEM (the group
// sum happens in place).  Per step j (M = keys, N = queries, K-dim = head dim):
//   S^T = K Q_j^T and dP^T = V dO_j^T   (SS MMAs, N = 128, separate commits)
//   dV += P^T dO_j, dK += dX^T Q_j      (TS MMAs, 16 query rows per chunk)
// TMEM: S^T [0, 128), dP^T [128, 256), dV [256, 384), dK [384, 512).  Each
// elementwise warpgroup owns 64 query columns: it copies its S^T columns to
// registers and releases them at once (the MMA issuer then computes S^T of step
// j + 1 while step j's elementwise work runs), and packs P^T / dX^T over its dP^T
// columns chunk by chunk; dP^T of step j + 1 is issued once every chunk's MMAs
// are.
template <int METHOD, int HD, bool DX>
__global__ void __launch_bounds__(NTHREADS, 1)
dkv_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
              const __grid_constant__ CUtensorMap mdk, const __grid_constant__ CUtensorMap mdv,
              const Params p) {
  constexpr int TILE = tile_bytes<HD>();
  constexpr int NSLAB = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[26];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ __align__(16) ColPair colc[2][BT / 2];  // per query column pair (double-buffered)
  __shared__ __align__(16) int4 coli[2][BT];         // per query column: live span (lo, hi, e)

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
  const uint32_t bar_s = smem_u32(&bars[5]);       // S^T of the step complete
  const uint32_t bar_dp = smem_u32(&bars[6]);      // dP^T of the step complete
  const uint32_t bar_sfree = smem_u32(&bars[7]);   // S^T copied to registers (8 warps)
  const uint32_t bar_chunk = smem_u32(&bars[8]);   // + c*8: chunk c packed by both warpgroups (8 warps)
  const uint32_t bar_final = smem_u32(&bars[16]);
  const uint32_t bar_cfull = smem_u32(&bars[17]);  // + (2*wg + cb)*8: column constants written
  const uint32_t bar_cfree = smem_u32(&bars[21]);  // + (2*wg + cb)*8: column constants consumed

  const uint32_t* map = p.kmap + ((size_t)b * p.nk + kt) * p.wq;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_kv, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_sfree, 8);
    for (int c = 0; c < 4; ++c) mbar_init(bar_chunk + 8 * c, 8);
    mbar_init(bar_final, 1);
    for (int c = 0; c < 4; ++c) {
      mbar_init(bar_cfull + 8 * c, 128);
      mbar_init(bar_cfree + 8 * c, 128);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  // the setup above overlaps the previous kernel's tail; global memory only after it
  pdl_trigger();
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int ntiles = count_tiles(map, p.wq);
  const int n = ntiles * p.G;  // steps: (query head of the group) x (visited query tile)

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (n > 0) {
      const bool leader = elect_one_sync();
      if (leader) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mdo);
        tma_prefetch_desc(&mdk);
        tma_prefetch_desc(&mdv);
        mbar_expect_tx(bar_kv, 2 * TILE);
        for (int sl = 0; sl < NSLAB; ++sl) {
          tma_load_4d(sK + sl * SLAB, &mk, bar_kv, 64 * sl, g, k0, b);
          tma_load_4d(sV + sl * SLAB, &mv, bar_kv, 64 * sl, g, k0, b);
        }
      }
      __syncwarp();
      StepIter st(map, p.wq, p.G);
      int hh, qt, j = 0;
      while (!__any_sync(0xFFFFFFFFu, abort_flag != 0) && st.next(hh, qt)) {
        const int h = g * p.G + hh;
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (u > 0 && !mbar_wait_warp(bar_empty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) break;
        if (leader) {
          const uint32_t sQ = sQD + s * 2 * TILE, sO = sQ + TILE;
          mbar_expect_tx(bar_full + 8 * s, 2 * TILE);
          for (int sl = 0; sl < NSLAB; ++sl) {
            tma_load_4d(sQ + sl * SLAB, &mq, bar_full + 8 * s, 64 * sl, h, qt * BT, b);
            tma_load_4d(sO + sl * SLAB, &mdo, bar_full + 8 * s, 64 * sl, h, qt * BT, b);
          }
        }
        __syncwarp();
        ++j;
      }
      if (leader) {
        drain_wait(bar_kv, 0);
        for (int jj = (j > NSTAGE ? j - NSTAGE : 0); jj < j; ++jj)
          drain_wait(bar_full + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      const bool leader = elect_one_sync();
      constexpr uint32_t idesc_acc = idesc_bf16(BT, HD, 0, 1);
      const uint64_t dK = smem_desc(sK, 16, 1024), dV = smem_desc(sV, 16, 1024);
      const uint64_t dQD = smem_desc(sQD, 16, 1024);        // Q / dO stages, K-major
      const uint64_t dQDmn = smem_desc(sQD, SLAB, 1024);    // the same, MN-major
      bool ok = mbar_wait_warp(bar_kv, 0, p.status, &abort_flag) &&
                mbar_wait_warp(bar_full, 0, p.status, &abort_flag);
      if (ok) {
        tc_fence_after();
        if (leader) {
          issue_scores<HD>(tmem, dK, dQD);                          // S^T  = K Q^T
          mma_commit(bar_s);
          issue_scores<HD>(tmem + 128u, dV, desc_add(dQD, TILE));   // dP^T = V dO^T
          mma_commit(bar_dp);
        }
        __syncwarp();
      }
      for (int j = 0; ok && j < n; ++j) {
        const uint32_t so = (uint32_t)((j % NSTAGE) * 2 * TILE);
        const uint32_t son = (uint32_t)(((j + 1) % NSTAGE) * 2 * TILE);
        const bool more = j + 1 < n;
        if (!mbar_wait_warp(bar_sfree, j & 1, p.status, &abort_flag)) break;
        if (more) {
          if (!mbar_wait_warp(bar_full + 8 * ((j + 1) % NSTAGE), ((j + 1) / NSTAGE) & 1, p.status,
                              &abort_flag))
            break;
          tc_fence_after();
          if (leader) {
            issue_scores<HD>(tmem, dK, desc_add(dQD, son));
            mma_commit(bar_s);
          }
          __syncwarp();
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (ok && !mbar_wait_warp(bar_chunk + 8 * c, j & 1, p.status, &abort_flag)) ok = false;
          if (ok) {
            tc_fence_after();
            if (leader) {
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                const uint32_t q0 = (uint32_t)(64 * w + 16 * c);
                const uint32_t acc = (j == 0 && c == 0 && w == 0) ? 0u : 1u;
                mma_ts(tmem + 256u, tmem + 128u + q0, desc_add(dQDmn, so + TILE + q0 * 128), idesc_acc,
                       acc);                                                 // dV += P^T dO
                mma_ts(tmem + 384u, tmem + 128u + q0 + 8, desc_add(dQDmn, so + q0 * 128), idesc_acc,
                       acc);                                                 // dK += dX^T Q
              }
            }
            __syncwarp();
          }
        }
        if (!ok) break;
        if (leader) {
          mma_commit(bar_empty + 8 * (j % NSTAGE));
          if (more) {
            issue_scores<HD>(tmem + 128u, dV, desc_add(dQD, son + TILE));
            mma_commit(bar_dp);
          }
        }
        __syncwarp();
      }
      // No wait for this commit here: the consumer warps wait for it, and
      // warp 1 re-checks it before freeing TMEM.
      if (leader) mma_commit(bar_final);
      __syncwarp();
    }
  } else {
    const int wg = (warp - 2) >> 2;        // query columns [64 wg, 64 wg + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;     // key row within the tile (TMEM lane)
    const int tid = (warp - 2 - 4 * wg) * 32 + lane;  // 0..127 within the warpgroup
    const int jrow = k0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_cols = lane_base + 64u * wg, dp_cols = lane_base + 128u + 64u * wg;
    const Xf xf = make_xf<METHOD>(p.cap, p.sm_scale);
    TanhFold tf{};
    if constexpr (METHOD == CAPATTN_CAP_TANH) tf = tanh_fold(xf.in, 1.f);
    const int my_col = 64 * wg + tid;      // query column whose constants this thread loads
    bool aborted = false;
    // Per-step column constants go through a double buffer one step ahead of
    // use, and their global inputs (and the tile's fully-live flag) are loaded
    // two steps ahead, so that no global load sits between two steps.
    auto put = [&](int buf, const ColRaw& r) {
      if (tid < 64) {
        const bool fin = isfinite(r.lse);
        const float lse2 = fin ? r.lse * kL2E : 0.f;
        const float radd = -r.dl + (fin ? p.z_loss_weight * r.lse + r.gl : 0.f);
        float mul, add;
        row_consts<METHOD>(p.cap, p.sm_scale, r.temp, &mul, &add);
        const float dsc = row_dscale<METHOD>(p.cap, p.sm_scale, r.temp);
        float* cf = reinterpret_cast<float*>(&colc[buf][my_col >> 1]);
        const int o = my_col & 1;
        cf[0 + o] = mul;
        cf[2 + o] = add - lse2;
        cf[4 + o] = -dsc;
        cf[6 + o] = -dsc * radd;
        coli[buf][my_col] = r.ri;
      }
    };
    // fully-live query-tile range of a step's query tile (raw; compared at use)
    auto qfull_of = [&](bool have, int qt) {
      return have ? p.qfull[(size_t)b * p.nq + qt] : make_int2(0, 0x7fffffff);
    };
    StepIter nx(map, p.wq, p.G);
    int nh = 0, nqt = 0;
    const bool have0 = nx.next(nh, nqt);
    const ColRaw r0 = load_col_raw(p, b, g * p.G + nh, nqt, my_col, have0 && tid < 64);
    int2 fr_cur = qfull_of(have0, nqt);
    int2 hq_cur = make_int2(g * p.G + nh, nqt);  // (query head, query tile) of the step
    const bool have1 = nx.next(nh, nqt);
    ColRaw r1 = load_col_raw(p, b, g * p.G + nh, nqt, my_col, have1 && tid < 64);
    int2 fr_nxt = qfull_of(have1, nqt);
    int2 hq_nxt = make_int2(g * p.G + nh, nqt);
    // stored-dX backward: this thread's first 32-byte unit in the step's dX^T
    // tile (1024 units per tile; the pool is at most 16 GiB = 2^29 units, so
    // units fit 32 bits):
    // block 4 wg (query columns 64 wg ..), key row r
    auto dx_unit = [&](int2 hq) -> uint32_t {
      if (!DX) return kNoDx;
      const int lo = p.dx_c >= 0 ? imax32(0, hq.y - p.dx_c) : 0;
      const int d = kt - lo;
      if (d < 0 || d >= p.dx_wmax) {
        atomicOr(p.status, kStatusBandBit);
        return kNoDx;
      }
      const uint32_t slot = ((uint32_t)(b * p.Hq + hq.x) * (uint32_t)p.nq + (uint32_t)hq.y) *
                                (uint32_t)p.dx_wmax + (uint32_t)d;
      return slot * 1024u + (uint32_t)(wg * 512 + r);
    };
    put(0, r0);
    mbar_arrive(bar_cfull + 8 * (2 * wg));
    for (int step = 0; step < n; ++step) {
      const int cb = step & 1, cu = step >> 1;
      const uint32_t my_cfull = bar_cfull + 8 * (2 * wg + cb);
      const uint32_t my_cfree = bar_cfree + 8 * (2 * wg + cb);
      if (step + 1 < n) {
        // constants of step + 1 into the other buffer (last used by step - 1)
        const int nb = cb ^ 1, nu = (step + 1) >> 1;
        if (step >= 1 &&
            !mbar_wait_warp(bar_cfree + 8 * (2 * wg + nb), (nu - 1) & 1, p.status, &abort_flag)) {
          aborted = true;
          break;
        }
        put(nb, r1);
        mbar_arrive(bar_cfull + 8 * (2 * wg + nb));
      }
      const bool have2 = nx.next(nh, nqt);
      const ColRaw r2 = load_col_raw(p, b, g * p.G + nh, nqt, my_col, have2 && tid < 64);
      const int2 fr2 = qfull_of(have2, nqt);
      const int2 hq2 = make_int2(g * p.G + nh, nqt);
      const uint32_t dxo = dx_unit(hq_cur);
      const bool tile_full = (kt >= fr_cur.x) && (kt < fr_cur.y);
      if (!mbar_wait_warp(my_cfull, cu & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      // S^T of this warpgroup's columns to registers; the columns are then free
      if (!mbar_wait_warp(bar_s, step & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld16(s_cols, *reinterpret_cast<uint32_t(*)[16]>(&sv[0]));
      tmem_ld16(s_cols + 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[16]));
      tmem_ld16(s_cols + 32, *reinterpret_cast<uint32_t(*)[16]>(&sv[32]));
      tmem_ld16(s_cols + 48, *reinterpret_cast<uint32_t(*)[16]>(&sv[48]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sfree);
      bool poly = false;
      if constexpr (METHOD == CAPATTN_CAP_TANH || METHOD == CAPATTN_CAP_ALSC) {
        float am = 0.f;
#pragma unroll
        for (int e = 0; e < 64; e += 2) am = fmax3_abs(am, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
        if constexpr (METHOD == CAPATTN_CAP_TANH)
          poly = __all_sync(0xFFFFFFFFu, tf.ok && am * fabsf(xf.in) <= kTanhPolyMaxU);
        else
          poly = __all_sync(0xFFFFFFFFu, am <= p.cap.alsc_xmax);  // the sigmoid on the FMA pipe
      }
      if (!mbar_wait_warp(bar_dp, step & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const ColPair* cp = &colc[cb][32 * wg];
      const int4* ci = &coli[cb][64 * wg];
      if (tile_full) {
        if (poly)
          dkv_step<METHOD, false, true, DX>(sv, dp_cols, cp, ci, jrow, xf, tf, p.cap, bar_chunk, lane, static_cast<char*>(p.dx_pool), dxo);
        else
          dkv_step<METHOD, false, false, DX>(sv, dp_cols, cp, ci, jrow, xf, tf, p.cap, bar_chunk, lane, static_cast<char*>(p.dx_pool), dxo);
      } else {
        if (poly)
          dkv_step<METHOD, true, true, DX>(sv, dp_cols, cp, ci, jrow, xf, tf, p.cap, bar_chunk, lane, static_cast<char*>(p.dx_pool), dxo);
        else
          dkv_step<METHOD, true, false, DX>(sv, dp_cols, cp, ci, jrow, xf, tf, p.cap, bar_chunk, lane, static_cast<char*>(p.dx_pool), dxo);
      }
      mbar_arrive(my_cfree);
      r1 = r2;
      fr_cur = fr_nxt;
      fr_nxt = fr2;
      hq_cur = hq_nxt;
      hq_nxt = hq2;
    }
    // ---------------------------------------------------------- epilogue
    bool have = false;
    if (n > 0 && !aborted) {
      have = mbar_wait_warp(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
    }
    // Warpgroup 0 writes dV, warpgroup 1 dK, each through the shared memory of
    // the V or K tile (free once every MMA has completed) in the swizzled
    // layout, then two TMA stores of 64 columns (rows past L are clipped).
    const uint32_t oslab = wg == 0 ? sV : sK;
    const uint32_t acc = lane_base + (wg == 0 ? 256u : 384u);
#pragma unroll 1
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(acc + c * 32, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      st_row32_swz(oslab + (uint32_t)(c >> 1) * SLAB, r, 4 * (c & 1), v);
    }
    fence_async_smem();
    named_bar_sync(1 + wg, 128);  // the warpgroup's rows are in shared memory
    if (tid == 0) {
      const CUtensorMap* mo = wg == 0 ? &mdv : &mdk;
      for (int sl = 0; sl < NSLAB; ++sl) tma_store_4d(mo, oslab + sl * SLAB, 64 * sl, g, k0, b);
      bulk_commit();
      bulk_wait_read0();
    }
  }
  __syncwarp();  // warps 0 and 1 reach the CTA barrier converged
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // Every MMA has completed before TMEM is released (normally already
    // observed by the consumer warps; bounded non-suspending poll).
    if (lane == 0 && n > 0) mbar_poll(bar_final, 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================= dQ
// One 16-column chunk (key columns 16 C .. 16 C + 15 of the warpgroup's 64) of a
// query row: dX packed to bf16.  Row constants in rc (both halves equal).
template <int METHOD, bool MASKED, bool POLY, int C, bool DT>
__device__ __forceinline__ void dq_chunk(const uint32_t (&s)[64], const uint32_t (&dp)[16],
                                         const ColPair& rc, int4 ri, int j0, const Xf& xf,
                                         const TanhFold& tf, uint32_t (&xk)[8], const DtempRow& dr,
                                         F2& dacc) {
  const uint32_t live = MASKED ? live_bits16(ri, j0 + 16 * C) : 0xFFFFu;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const bool l0 = (live >> (2 * e)) & 1u, l1 = (live >> (2 * e + 1)) & 1u;
    const float X0 = __uint_as_float(s[16 * C + 2 * e]), X1 = __uint_as_float(s[16 * C + 2 * e + 1]);
    const float d0 = __uint_as_float(dp[2 * e]), d1 = __uint_as_float(dp[2 * e + 1]);
    uint32_t pk;
    if (POLY && e < kDkvPolyPairs)
      dkv_pair<METHOD, METHOD == CAPATTN_CAP_TANH, DT>(X0, X1, d0, d1, xf, tf, rc, l0, l1, pk, xk[e], &dr, &dacc);
    else
      dkv_pair<METHOD, false, DT>(X0, X1, d0, d1, xf, tf, rc, l0, l1, pk, xk[e], &dr, &dacc);
  }
}

// The warpgroup's 64 key columns of one step: dX of chunk C is packed over the
// first 8 of its 16 dP columns and handed to the MMA issuer.
template <int METHOD, bool MASKED, bool POLY, bool DT>
__device__ __forceinline__ void dq_step(const uint32_t (&s)[64], uint32_t dp_base, const ColPair& rc,
                                        int4 ri, int j0, const Xf& xf, const TanhFold& tf,
                                        uint32_t bar_chunk0, int lane, const DtempRow& dr, F2& dacc) {
  uint32_t da[16], db[16], xk[8];
  tmem_ld16(dp_base, da);
  tmem_wait_ld();
#define CAPATTN_DQ_CHUNK(C, CUR, NXT)                                                      \
  {                                                                                       \
    if (C < 3) tmem_ld16(dp_base + 16 * (C + 1), NXT);                                    \
    dq_chunk<METHOD, MASKED, POLY, C, DT>(s, CUR, rc, ri, j0, xf, tf, xk, dr, dacc);      \
    __syncwarp();                                                                         \
    tmem_st8(dp_base + 16 * C, xk);                                                       \
    tmem_wait_st();                                                                       \
    if (C < 3) tmem_wait_ld();                                                            \
    tc_fence_before();                                                                    \
    __syncwarp();                                                                         \
    if (lane == 0) mbar_arrive(bar_chunk0 + 8 * C);                                       \
  }
  CAPATTN_DQ_CHUNK(0, da, db)
  CAPATTN_DQ_CHUNK(1, db, da)
  CAPATTN_DQ_CHUNK(2, da, db)
  CAPATTN_DQ_CHUNK(3, db, da)
#undef CAPATTN_DQ_CHUNK
}

// dQ: one CTA per (batch, query head, 128-query tile), looping over the KV tiles
// of its visit map.  Per step j (M = queries, N = keys, K-dim = head dim):
//   S = Q K_j^T and dP = dO V_j^T   (SS MMAs, N = 128, separately committed)
//   dQ += dX K_j                    (TS MMAs, 16 keys per chunk)
// TMEM: S [0, 128), dP of even steps [128, 256), dP of odd steps [256, 384),
// dQ [384, 512).  K and V have their own two-stage rings: V_j is read only by
// dP_j, so its stage is free as soon as dP_j has run, and dP of step j + 2 is
// computed (into the buffer step j used) right after step j's accumulation
// MMAs; it is ready long before step j + 2 starts.  S of step j + 1 goes into
// the S buffer once the elementwise warps have copied step j's S to registers
// (at the start of step j) and K_{j+1} has landed.  The elementwise warpgroups
// own 64 key columns each and pack dX over the step's dP columns chunk by chunk.
template <int METHOD, bool DT, int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
dq_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
             const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
             const __grid_constant__ CUtensorMap mdq, const Params p) {
  constexpr int TILE = tile_bytes<HD>();
  constexpr int NSLAB = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[24];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float dxch[2][BT];   // half-row sums of O * dO (delta), one per warpgroup

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
  const uint32_t bar_kfull = smem_u32(&bars[1]);   // + s*8: K of stage s landed
  const uint32_t bar_vfull = smem_u32(&bars[3]);   // + s*8: V of stage s landed
  const uint32_t bar_kempty = smem_u32(&bars[5]);  // + s*8: K of stage s no longer read
  const uint32_t bar_vempty = smem_u32(&bars[7]);  // + s*8: V of stage s no longer read
  const uint32_t bar_s = smem_u32(&bars[9]);       // S of the step complete
  const uint32_t bar_sfree = smem_u32(&bars[10]);  // S copied to registers (8 warps)
  const uint32_t bar_dp = smem_u32(&bars[11]);     // + x*8: dP in buffer x complete
  // + (4 * (j & 1) + c) * 8: chunk c of step j packed by both warpgroups.  The
  // elementwise warps may run a step ahead of the issuer (dP of the next step is
  // ready early), so even and odd steps use separate barriers: a barrier then
  // never completes a phase the issuer has not waited for yet.
  const uint32_t bar_chunk = smem_u32(&bars[13]);
  const uint32_t bar_final = smem_u32(&bars[21]);
  const uint32_t bar_dx = smem_u32(&bars[22]);     // both warpgroups wrote their delta halves

  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
      mbar_init(bar_vempty + 8 * s, 1);
      mbar_init(bar_dp + 8 * s, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_sfree, 8);
    for (int c = 0; c < 8; ++c) mbar_init(bar_chunk + 8 * c, 8);
    mbar_init(bar_final, 1);
    mbar_init(bar_dx, 8);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  // the setup above overlaps the previous kernel's tail; global memory only after it
  pdl_trigger();
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int n = count_tiles(map, p.wk);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (n > 0) {
      const bool leader = elect_one_sync();
      if (leader) {
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&mdq);
        mbar_expect_tx(bar_q, 2 * TILE);
        for (int sl = 0; sl < NSLAB; ++sl) {
          tma_load_4d(sQ + sl * SLAB, &mq, bar_q, 64 * sl, h, q0, b);
          tma_load_4d(sO + sl * SLAB, &mdo, bar_q, 64 * sl, h, q0, b);
        }
      }
      __syncwarp();
      // V of step j as soon as dP of step j - 2 has read its stage, then K of
      // step j once step j - 2's accumulation MMAs have
      TileIter it(map, p.wk);
      int t, j = 0;
      while (!__any_sync(0xFFFFFFFFu, abort_flag != 0) && it.next(t)) {
        const int s = j % NSTAGE, u = j / NSTAGE;
        const uint32_t sK = sKV + s * 2 * TILE, sV = sK + TILE;
        if (u > 0 && !mbar_wait_warp(bar_vempty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) break;
        if (leader) {
          mbar_expect_tx(bar_vfull + 8 * s, TILE);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sV + sl * SLAB, &mv, bar_vfull + 8 * s, 64 * sl, g, t * BT, b);
        }
        __syncwarp();
        if (u > 0 && !mbar_wait_warp(bar_kempty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) {
          ++j;  // V of this step is in flight: drained below
          break;
        }
        if (leader) {
          mbar_expect_tx(bar_kfull + 8 * s, TILE);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sK + sl * SLAB, &mk, bar_kfull + 8 * s, 64 * sl, g, t * BT, b);
        }
        __syncwarp();
        ++j;
      }
      if (leader) {
        // (on an early exit the last step's K may not have been issued; its
        // barrier then never completes and the bounded wait just runs out)
        drain_wait(bar_q, 0);
        for (int jj = (j > NSTAGE ? j - NSTAGE : 0); jj < j; ++jj) {
          drain_wait(bar_vfull + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
          drain_wait(bar_kfull + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
        }
      }
      __syncwarp();
    }
    // Key-tile visit map for the dK/dV kernel (launched after this grid
    // completes): query tile qt's bit in the word of every KV tile it visits.
    // One head per (b, qt) writes; rowmap_kernel cleared the words.
    if (h == 0) {
      for (int w = lane; w < p.wk; w += 32) {
        uint32_t bits = map[w];
        while (bits) {
          const int kt = 32 * w + __ffs(bits) - 1;
          bits &= bits - 1u;
          atomicOr(&p.kmap[((size_t)b * p.nk + kt) * p.wq + (qt >> 5)], 1u << (qt & 31));
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      const bool leader = elect_one_sync();
      constexpr uint32_t idesc_acc = idesc_bf16(BT, HD, 0, 1);
      const uint64_t dQ = smem_desc(sQ, 16, 1024), dO = smem_desc(sO, 16, 1024);
      const uint64_t dKV = smem_desc(sKV, 16, 1024);        // K / V stages, K-major
      const uint64_t dKVmn = smem_desc(sKV, SLAB, 1024);    // the same, MN-major
      // S of step j into the S buffer (step j - 1's S has been copied out)
      auto issue_s = [&](int j) -> bool {
        if (!mbar_wait_warp(bar_kfull + 8 * (j % NSTAGE), (j / NSTAGE) & 1, p.status, &abort_flag))
          return false;
        tc_fence_after();
        if (leader) {
          issue_scores<HD>(tmem, dQ, desc_add(dKV, (uint32_t)((j % NSTAGE) * 2 * TILE)));
          mma_commit(bar_s);
        }
        __syncwarp();
        return true;
      };
      // dP of step j into buffer j & 1 (step j - 2's accumulation MMAs, which
      // read that buffer, were issued before); V's stage is then free
      auto issue_dp = [&](int j) -> bool {
        if (!mbar_wait_warp(bar_vfull + 8 * (j % NSTAGE), (j / NSTAGE) & 1, p.status, &abort_flag))
          return false;
        tc_fence_after();
        if (leader) {
          issue_scores<HD>(tmem + 128u + 128u * (uint32_t)(j & 1), dO,
                       desc_add(dKV, (uint32_t)((j % NSTAGE) * 2 * TILE + TILE)));
          mma_commit(bar_dp + 8 * (j & 1));
          mma_commit(bar_vempty + 8 * (j % NSTAGE));
        }
        __syncwarp();
        return true;
      };
      bool ok = mbar_wait_warp(bar_q, 0, p.status, &abort_flag);
      tc_fence_after();
      ok = ok && issue_s(0) && issue_dp(0) && (n < 2 || issue_dp(1));
      for (int j = 0; ok && j < n; ++j) {
        const uint32_t so = (uint32_t)((j % NSTAGE) * 2 * TILE);
        const uint32_t xo = 128u + 128u * (uint32_t)(j & 1);
        // S of step j + 1 once step j's S is out of TMEM and K_{j+1} has landed
        // (the elementwise warps need it first; this step's accumulation MMAs
        // can follow later)
        if (j + 1 < n) {
          if (!mbar_wait_warp(bar_sfree, j & 1, p.status, &abort_flag) || !issue_s(j + 1)) break;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (ok && !mbar_wait_warp(bar_chunk + 8 * (4 * (j & 1) + c), (j >> 1) & 1, p.status, &abort_flag))
            ok = false;
          if (ok) {
            tc_fence_after();
            if (leader) {
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                const uint32_t k0c = (uint32_t)(64 * w + 16 * c);
                mma_ts(tmem + 384u, tmem + xo + k0c, desc_add(dKVmn, so + k0c * 128), idesc_acc,
                       (j == 0 && c == 0 && w == 0) ? 0u : 1u);     // dQ += dX K
              }
            }
            __syncwarp();
          }
        }
        if (!ok) break;
        if (leader) mma_commit(bar_kempty + 8 * (j % NSTAGE));
        __syncwarp();
        if (j + 2 < n && !issue_dp(j + 2)) break;
      }
      if (leader) mma_commit(bar_final);
      __syncwarp();
    }
  } else {
    const int wg = (warp - 2) >> 2;        // key columns [64 wg, 64 wg + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int i = q0 + r;
    const bool valid = i < p.L;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_cols = lane_base + 64u * wg;
    const int4 ri = valid ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
    const float temp = (p.temp && valid) ? p.temp[(size_t)b * p.L + i] : 1.f;
    const size_t rr = ((size_t)b * p.Hq + h) * p.L + i;
    const float lse = valid ? p.lse[rr] : -INFINITY;
    const float gl = (p.dlse && valid) ? p.dlse[rr] : 0.f;
    bool aborted = false;
    // delta_i = rowsum(O * dO) (the pre-pass of the backward), computed here for
    // the tile's rows: each warpgroup sums its 64 dims, O from global memory and
    // dO from the tile staged for the dP MMAs (128-byte swizzle: the 16-byte
    // chunk c of row r sits at chunk c ^ (r % 8)); the halves add through shared
    // memory.  A tile with no visited KV tile has only fully masked rows, whose
    // O and delta are 0.
    float dl = 0.f;
    {
      float dpart = 0.f;
      if (n > 0) {
        // O is loaded first, so that its latency overlaps the wait for the tiles
        constexpr int NCH = HD / 8;       // 16-byte chunks (8 bf16) of a row; each warpgroup takes half
        uint4 orow_g[NCH / 2];
        if (valid) {
          const uint4* og = reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(p.o) + ((size_t)(b * p.L + i) * p.Hq + h) * HD + (HD / 2) * wg);
#pragma unroll
          for (int c = 0; c < NCH / 2; ++c) orow_g[c] = og[c];
        }
        if (!mbar_wait_warp(bar_q, 0, p.status, &abort_flag)) aborted = true;
        if (valid && !aborted) {
#pragma unroll
          for (int c = 0; c < NCH / 2; ++c) {
            const int gc = (NCH / 2) * wg + c;   // chunk of the row: slab gc / 8, chunk gc % 8
            const uint8_t* orow = smem_raw + (sO - smem_u32(smem_raw)) + (gc >> 3) * SLAB + r * 128;
            const uint4 a = orow_g[c];
            const uint4 d = *reinterpret_cast<const uint4*>(orow + (((gc & 7) ^ (r & 7)) << 4));
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, dv4[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
              const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dv4[e]));
              dpart = fmaf(x.x, y.x, dpart);
              dpart = fmaf(x.y, y.y, dpart);
            }
          }
        }
        dxch[wg][r] = dpart;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dx);
        if (!mbar_wait_warp(bar_dx, 0, p.status, &abort_flag)) aborted = true;
        dl = dpart + dxch[wg ^ 1][r];
      }
      if (wg == 0 && valid) p.delta[rr] = dl;
    }
    const bool fin = isfinite(lse);
    const Xf xf = make_xf<METHOD>(p.cap, p.sm_scale);
    TanhFold tf{};
    if constexpr (METHOD == CAPATTN_CAP_TANH) tf = tanh_fold(xf.in, 1.f);
    ColPair rc;
    DtempRow dr;
    {
      // capped score c = kc f + bc in terms of the cap's shape f
      float kc = p.cap.cap, bc = 0.f;
      if constexpr (METHOD == CAPATTN_CAP_ALSC) {
        kc = p.cap.alsc_out;
        bc = -p.cap.alsc_out * p.cap.alsc_sb;
      } else if constexpr (METHOD == CAPATTN_CAP_NONE) {
        kc = p.sm_scale;
      }
      dr.kc = f2(kc, kc);
      dr.bc = f2(bc, bc);
    }
    {
      float mul, add;
      row_consts<METHOD>(p.cap, p.sm_scale, temp, &mul, &add);
      const float addl = add - (fin ? lse * kL2E : 0.f);
      const float dsc = row_dscale<METHOD>(p.cap, p.sm_scale, temp);
      const float radd = -dl + (fin ? p.z_loss_weight * lse + gl : 0.f);
      rc.a = make_float4(mul, mul, addl, addl);
      rc.b = make_float4(-dsc, -dsc, -dsc * radd, -dsc * radd);
      dr.radd = f2(radd, radd);
    }
    F2 dacc = f2(0.f, 0.f);
    TileIter it(map, p.wk);
    for (int j = 0; j < n; ++j) {
      int t;
      it.next(t);
      const int k0 = t * BT;
      const bool full = __all_sync(0xFFFFFFFFu, (ri.x <= k0) && (ri.y >= k0 + BT));
      if (!mbar_wait_warp(bar_s, j & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld16(s_cols, *reinterpret_cast<uint32_t(*)[16]>(&sv[0]));
      tmem_ld16(s_cols + 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[16]));
      tmem_ld16(s_cols + 32, *reinterpret_cast<uint32_t(*)[16]>(&sv[32]));
      tmem_ld16(s_cols + 48, *reinterpret_cast<uint32_t(*)[16]>(&sv[48]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sfree);
      bool poly = false;
      if constexpr (METHOD == CAPATTN_CAP_TANH) {
        float am = 0.f;
#pragma unroll
        for (int e = 0; e < 64; e += 2) am = fmax3_abs(am, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
        poly = __all_sync(0xFFFFFFFFu, tf.ok && am * fabsf(xf.in) <= kTanhPolyMaxU);
      }
      if (!mbar_wait_warp(bar_dp + 8 * (j & 1), (j >> 1) & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const int j0 = k0 + 64 * wg;
      const uint32_t dp_cols = lane_base + 128u + 128u * (uint32_t)(j & 1) + 64u * wg;
      const uint32_t chunk_bars = bar_chunk + 32u * (uint32_t)(j & 1);
      if (full) {
        if (poly)
          dq_step<METHOD, false, true, DT>(sv, dp_cols, rc, ri, j0, xf, tf, chunk_bars, lane, dr, dacc);
        else
          dq_step<METHOD, false, false, DT>(sv, dp_cols, rc, ri, j0, xf, tf, chunk_bars, lane, dr, dacc);
      } else {
        if (poly)
          dq_step<METHOD, true, true, DT>(sv, dp_cols, rc, ri, j0, xf, tf, chunk_bars, lane, dr, dacc);
        else
          dq_step<METHOD, true, false, DT>(sv, dp_cols, rc, ri, j0, xf, tf, chunk_bars, lane, dr, dacc);
      }
    }
    bool have = false;
    if (n > 0 && !aborted) {
      have = mbar_wait_warp(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
    }
    if constexpr (DT) {
      // this warpgroup's part of sum over the row's keys of dT c, one slot per
      // (head, row, warpgroup); the slots are added in a fixed order afterwards
      float a0, a1;
      f2_split(dacc, a0, a1);
      if (valid) p.dtemp_part[2 * rr + wg] = aborted ? 0.f : a0 + a1;
    }
    // Warpgroup wg writes dQ columns [64 wg, 64 wg + 64) through slab wg of
    // the Q tile's shared memory (free once every MMA has completed) and one
    // TMA store (rows past L are clipped).
    // HD = 128: warpgroup wg fills slab wg; HD = 64: the two warpgroups fill
    // the two halves (16-byte chunks [0, 4) and [4, 8)) of the one slab.
    const uint32_t oslab = sQ + (HD == 128 ? (uint32_t)wg * SLAB : 0u);
    const int chunk0 = HD == 128 ? 0 : 4 * wg;
#pragma unroll 1
    for (int c = 0; c < HD / 64; ++c) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(lane_base + 384u + (HD / 2) * wg + 32 * c, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      st_row32_swz(oslab, r, chunk0 + 4 * c, v);
    }
    fence_async_smem();
    if constexpr (HD == 128) {
      named_bar_sync(1 + wg, 128);  // the warpgroup's rows are in shared memory
      if (warp == 2 + 4 * wg && lane == 0) {
        tma_store_4d(&mdq, oslab, 64 * wg, h, q0, b);
        bulk_commit();
        bulk_wait_read0();
      }
    } else {
      named_bar_sync(1, 256);       // both warpgroups' halves are in shared memory
      if (warp == 2 && lane == 0) {
        tma_store_4d(&mdq, oslab, 0, h, q0, b);
        bulk_commit();
        bulk_wait_read0();
      }
    }
  }
  __syncwarp();  // warps 0 and 1 reach the CTA barrier converged
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0 && n > 0) mbar_poll(bar_final, 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int METHOD, int HD>
cudaError_t launch_bwd_hd(const Params& p, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  cudaError_t e = make_bhld_map(&mq, p.q, p.B, p.L, p.Hq, HD, BT);
  if (e == cudaSuccess) e = make_bhld_map(&mk, p.k, p.B, p.Lk, p.Hkv, HD, BT);
  if (e == cudaSuccess) e = make_bhld_map(&mv, p.v, p.B, p.Lk, p.Hkv, HD, BT);
  if (e == cudaSuccess) e = make_bhld_map(&mdo, p.dO, p.B, p.L, p.Hq, HD, BT);
  if (e == cudaSuccess) e = make_bhld_map(&mdq, p.dq, p.B, p.L, p.Hq, HD, BT);
  if (e == cudaSuccess) e = make_bhld_map(&mdk, p.dk, p.B, p.Lk, p.Hkv, HD, BT);
  if (e == cudaSuccess) e = make_bhld_map(&mdv, p.dv, p.B, p.Lk, p.Hkv, HD, BT);
  if (e != cudaSuccess) return e;
  constexpr int SMEM_BYTES = smem_bytes<HD>();
  if (p.dx_pool) {
    // stored-dX backward: delta (and the key-tile map), then dK/dV (which also
    // stores dX), then dQ as a GEMM over the stored tiles
    e = launch_delta_bf16(p, s);
    if (e != cudaSuccess) return e;
  } else {
    // dQ first: it also computes delta, which the dK/dV kernel reads.
    auto kdq = p.dtemp ? dq_tc_kernel<METHOD, true, HD> : dq_tc_kernel<METHOD, false, HD>;
    e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prof_begin(CAPATTN_KERNEL_DQ, s);
    prof_count(CAPATTN_KERNEL_DQ, 1);
    e = launch_pdl(kdq, dim3(p.Hq * p.B, p.nq), dim3(NTHREADS), SMEM_BYTES, s, mq, mk, mv, mdo, mdq, p);
    if (e != cudaSuccess) return e;
    prof_end(CAPATTN_KERNEL_DQ, s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto kdkv = p.dx_pool ? dkv_tc_kernel<METHOD, HD, true> : dkv_tc_kernel<METHOD, HD, false>;
  e = cudaFuncSetAttribute(kdkv, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  prof_begin(CAPATTN_KERNEL_DKV, s);
  prof_count(CAPATTN_KERNEL_DKV, 1);
  e = launch_pdl(kdkv, dim3(p.Hkv * p.B, p.nk), dim3(NTHREADS), SMEM_BYTES, s, mq, mk, mv, mdo, mdk, mdv, p);
  if (e != cudaSuccess) return e;
  prof_end(CAPATTN_KERNEL_DKV, s);
  e = cudaGetLastError();
  if (e != cudaSuccess || !p.dx_pool) return e;
  return launch_dq_gemm(p, s);
}

template <int METHOD>
struct BwdTcLaunch {
  static cudaError_t run(const Params& p, cudaStream_t s) {
    return p.D == 64 ? launch_bwd_hd<METHOD, 64>(p, s) : launch_bwd_hd<METHOD, 128>(p, s);
  }
};

}  // namespace

cudaError_t launch_bwd_bf16(const Params& p, cudaStream_t s) {
  return dispatch_cap<BwdTcLaunch>(p.cap.method, p, s);
}

}  // namespace capattn
