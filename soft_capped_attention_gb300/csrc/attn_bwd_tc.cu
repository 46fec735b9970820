// bf16 backward on the 5th-generation tensor cores: a dK/dV kernel and a dQ
// kernel (mosaic_backward.py make_mosaic_backward_dkv_kernel and
// make_mosaic_backward_dq_kernel, restated for tcgen05 / TMEM), after the
// delta pre-pass.
//
// Per live pair (query i, key j), with x = temp_i * cap(s_ij) * log2(e):
//   P_ij  = 2^(x - LSE_i * log2(e))                       (0 when masked)
//   dX_ij = sm_scale * temp_i * cap'(s_ij) * P_ij * (dP_ij - delta_i + z * LSE_i)
//
// Both kernels cut every 128 x 128 step into two halves of 64 columns ("parts")
// with their own TMEM buffers, so that one part's score MMAs of the next step
// run on the tensor pipe while the elementwise warps work on the other part:
//   MMA order:  ... | acc(j, 0)  S/dP(j+1, 0) | acc(j, 1)  S/dP(j+1, 1) | ...
//   elementwise:        part 1 of step j       |   part 0 of step j+1
// TMEM: part 0 scores [0, 64), part 0 dP [64, 128), part 1 scores [128, 192),
// part 1 dP [192, 256), accumulators from 256.  Each elementwise warpgroup
// owns 32 columns of a part; its packed bf16 results overwrite score / dP
// columns it has already read, and the part is handed to the MMA issuer once
// both warpgroups arrive.
//
// dK/dV: one CTA per (batch, KV head, 128-key tile).  K and V stay in shared
// memory; the CTA loops over the query heads of its GQA group and the query
// tiles of the tile's visit map, accumulating dK and dV in TMEM (the group sum
// happens in place).  Per part: S^T = K Q_part^T, dP^T = V dO_part^T (SS MMAs,
// M = keys, N = 64 queries); dV += P^T dO_part, dK += dX^T Q_part (TS MMAs,
// K = 64).  TMEM: dV [256, 384), dK [384, 512).
//
// dQ: one CTA per (batch, query head, 128-query tile), looping over the KV
// tiles of its visit map.  Per part: S = Q K_part^T, dP = dO V_part^T (N = 64
// keys); dQ += dX K_part (K = 64).  TMEM: dQ [256, 384).
//
// Warp roles in both kernels (10 warps): warp 0 TMA producer, warp 1 TMEM
// allocator and MMA issuer, warps 2..5 and 6..9 the two elementwise
// warpgroups (one TMEM lane = one tile row each).
#include <math.h>

#include "cap_math.cuh"
#include "capattn_internal.h"
#include "softmax_elem.cuh"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

constexpr int HD = 128;
constexpr int BT = 128;                       // tile rows (queries and keys)
constexpr int SLAB = 128 * 64 * 2;
constexpr int TILE = 2 * SLAB;
constexpr int NSTAGE = 2;
constexpr int NTHREADS = 320;
constexpr int SMEM_BYTES = 2 * TILE + NSTAGE * 2 * TILE + 1024;
constexpr int kBwdPolyPairs = 10;  // of 16 column pairs in a dQ chunk: tanh on the FMA pipe
constexpr int kDkvPolyPairs = 5;   // of 8 column pairs in a dK/dV sub-chunk

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32]) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
}

__device__ __forceinline__ void store_zero_bf16(__nv_bfloat16* dst) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < 4; ++e) d4[e] = make_uint4(0u, 0u, 0u, 0u);
}

// Scores of one part: D[128 x 64] = A[128 x 128] B_part^T, both K-major; the
// part's 64 rows of B start at row 64 * part of the staged tile.
__device__ __forceinline__ void issue_scores_part(uint32_t d, uint32_t sA, uint32_t sB, int part) {
  constexpr uint32_t idesc = idesc_bf16(BT, 64, 0, 0);
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
    mma_ss(d, smem_desc(sA + off, 16, 1024), smem_desc(sB + off + part * 64 * 128, 16, 1024), idesc,
           ks > 0);
  }
}

// TMEM column (within a part's score or dP buffer) of the packed bf16 values
// for the part's columns [16 ks, 16 ks + 16): warpgroup ks / 2, sub-chunk ks % 2.
__device__ __forceinline__ uint32_t packed_col(int ks) { return (uint32_t)(32 * (ks >> 1) + 8 * (ks & 1)); }

// D[128 x 128] += A (packed bf16 in TMEM, 64 columns of the part) x B rows
// [64 part, 64 part + 64) (MN-major, N = 128).
__device__ __forceinline__ void issue_acc_part(uint32_t d, uint32_t a_base, uint32_t sB, int part, bool first) {
  constexpr uint32_t idesc = idesc_bf16(BT, HD, 0, 1);
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
    mma_ts(d, a_base + packed_col(ks), smem_desc(sB + (64 * part + 16 * ks) * 128, SLAB, 1024), idesc,
           (first && ks == 0) ? 0u : 1u);
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

// Raw per-query-column inputs of one step (loaded ahead of use).
struct ColRaw {
  float lse2, radd, temp;
  int4 ri;
};

__device__ __forceinline__ ColRaw load_col_raw(const Params& p, int b, int h, int qt, int c, bool active) {
  ColRaw r;
  r.lse2 = 0.f;
  r.radd = 0.f;
  r.temp = 1.f;
  r.ri = make_int4(0, 0, -1, 0);
  const int i = qt * BT + c;
  if (active && i < p.L) {
    const size_t rr = ((size_t)b * p.Hq + h) * p.L + i;
    const float lse = p.lse[rr];
    const float dl = p.delta[rr];
    const bool fin = isfinite(lse);
    r.lse2 = fin ? lse * kL2E : 0.f;
    r.radd = -dl + (fin ? p.z_loss_weight * lse : 0.f);
    if (p.temp) r.temp = p.temp[(size_t)b * p.L + i];
    r.ri = p.rowinfo[(size_t)b * p.L + i];
  }
  return r;
}

// Backward elementwise on a pair of scores: P = 2^(mul * f + add) (0 when
// masked) and dX = dscale * f' * P * (dP + radd), with packed fp32x2 math.  For
// the tanh cap with POLY, tanh is evaluated on the FMA pipe (the caller
// guarantees |X * in| <= 0.5 for the whole warp).
template <int METHOD, bool POLY>
__device__ __forceinline__ void bwd_pair(float X0, float X1, float dp0, float dp1, const Xf& xf,
                                         F2 mul, F2 add, F2 dsc, F2 radd, bool l0, bool l1,
                                         float& P0, float& P1, float& dX0, float& dX1) {
  F2 f, d;
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    const F2 u = f2_mul(f2(X0, X1), f2(xf.in, xf.in));
    if constexpr (POLY) {
      f = tanh_poly2(u);
    } else {
      float a, b;
      f2_split(u, a, b);
      f = f2(tanh_approx(a), tanh_approx(b));
    }
    d = f2_fma(f2_mul(f, f2(-1.f, -1.f)), f, f2(1.f, 1.f));
  } else {
    float d0, d1;
    const float f0 = cap_f_d<METHOD>(X0, xf, &d0);
    const float f1 = cap_f_d<METHOD>(X1, xf, &d1);
    f = f2(f0, f1);
    d = f2(d0, d1);
  }
  float x0, x1;
  f2_split(f2_fma(mul, f, add), x0, x1);
  P0 = l0 ? ex2_approx(x0) : 0.f;
  P1 = l1 ? ex2_approx(x1) : 0.f;
  const F2 g = f2_mul(f2(P0, P1), f2_add(f2(dp0, dp1), radd));
  f2_split(f2_mul(f2_mul(dsc, d), g), dX0, dX1);
}

// dK/dV elementwise on 16 query columns (col0 .. col0 + 15) of key row jrow:
// P^T and dX^T packed to bf16 and stored at TMEM addresses p_dst and x_dst.
template <int METHOD, bool MASKED, bool POLY>
__device__ __forceinline__ void dkv_sub_impl(const uint32_t (&sv)[16], const uint32_t (&dp)[16],
                                             const float4* colc, const int4* coli, int col0,
                                             int jrow, const Xf& xf, uint32_t p_dst, uint32_t x_dst) {
  uint32_t pp[8], px[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int cc = col0 + 2 * e;
    const float4 ka = colc[cc], kb = colc[cc + 1];
    bool l0 = true, l1 = true;
    if constexpr (MASKED) {
      const int4 ca = coli[cc], cb = coli[cc + 1];
      l0 = (jrow >= ca.x && jrow < ca.y) || jrow == ca.z;
      l1 = (jrow >= cb.x && jrow < cb.y) || jrow == cb.z;
    }
    float P0, P1, x0, x1;
    const float X0 = __uint_as_float(sv[2 * e]), X1 = __uint_as_float(sv[2 * e + 1]);
    const float d0 = __uint_as_float(dp[2 * e]), d1 = __uint_as_float(dp[2 * e + 1]);
    if (POLY && e < kDkvPolyPairs)
      bwd_pair<METHOD, true>(X0, X1, d0, d1, xf, f2(ka.x, kb.x), f2(ka.y, kb.y), f2(ka.z, kb.z),
                             f2(ka.w, kb.w), l0, l1, P0, P1, x0, x1);
    else
      bwd_pair<METHOD, false>(X0, X1, d0, d1, xf, f2(ka.x, kb.x), f2(ka.y, kb.y), f2(ka.z, kb.z),
                              f2(ka.w, kb.w), l0, l1, P0, P1, x0, x1);
    pp[e] = pack_bf16x2(P0, P1);
    px[e] = pack_bf16x2(x0, x1);
  }
  tmem_st8(p_dst, pp);
  tmem_st8(x_dst, px);
}

// dK/dV elementwise on 16 query columns (col0 .. col0 + 15) of key row jrow:
// P^T and dX^T packed to bf16 and stored at TMEM addresses p_dst and x_dst.
// For the tanh cap the warp votes on whether all its arguments are small enough
// for the FMA-pipe polynomial.
template <int METHOD, bool MASKED>
__device__ __forceinline__ void dkv_sub(const uint32_t (&sv)[16], const uint32_t (&dp)[16],
                                        const float4* colc, const int4* coli, int col0, int jrow,
                                        const Xf& xf, uint32_t p_dst, uint32_t x_dst) {
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) am = fmaxf(am, fabsf(__uint_as_float(sv[e])));
    if (__all_sync(0xFFFFFFFFu, am * fabsf(xf.in) <= kTanhPolyMaxU)) {
      dkv_sub_impl<METHOD, MASKED, true>(sv, dp, colc, coli, col0, jrow, xf, p_dst, x_dst);
      return;
    }
  }
  dkv_sub_impl<METHOD, MASKED, false>(sv, dp, colc, coli, col0, jrow, xf, p_dst, x_dst);
}

// One warpgroup's 32 columns of one part: two sub-chunks of 16, the second
// one's TMEM loads in flight while the first is computed.
template <int METHOD, bool MASKED>
__device__ __forceinline__ void dkv_part(const float4* colc, const int4* coli, int wg, int part,
                                         int jrow, const Xf& xf, uint32_t lane_base) {
  const uint32_t sbuf = lane_base + 128u * part, dbuf = sbuf + 64u;
  const int pc0 = 32 * wg;              // first column within the part
  const int col0 = 64 * part + pc0;     // first query column within the tile
  uint32_t sa[16], da[16], sb[16], db[16];
  tmem_ld16(sbuf + pc0, sa);
  tmem_ld16(dbuf + pc0, da);
  tmem_wait_ld();
  tmem_ld16(sbuf + pc0 + 16, sb);
  tmem_ld16(dbuf + pc0 + 16, db);
  dkv_sub<METHOD, MASKED>(sa, da, colc, coli, col0, jrow, xf, sbuf + pc0, dbuf + pc0);
  tmem_wait_ld();
  dkv_sub<METHOD, MASKED>(sb, db, colc, coli, col0 + 16, jrow, xf, sbuf + pc0 + 8, dbuf + pc0 + 8);
  tmem_wait_st();
}

// dQ elementwise on 32 key columns (absolute j0 .. j0 + 31) of query row (span
// ri): dX packed to bf16 into px.  (No TMEM access: callers branch per row.)
// With POLY (tanh cap), column pairs [0, poly_pairs) use the FMA-pipe tanh.
template <int METHOD, bool MASKED, bool POLY>
__device__ __forceinline__ void dq_chunk(const uint32_t (&sv)[32], const uint32_t (&dp)[32], int j0,
                                         int4 ri, const Xf& xf, float mul, float addl, float dscale,
                                         float radd, uint32_t (&px)[16]) {
  const F2 mul2 = f2(mul, mul), add2 = f2(addl, addl), dsc2 = f2(dscale, dscale),
           radd2 = f2(radd, radd);
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    bool l0 = true, l1 = true;
    if constexpr (MASKED) {
      const int ja = j0 + 2 * e, jb = ja + 1;
      l0 = (ja >= ri.x && ja < ri.y) || ja == ri.z;
      l1 = (jb >= ri.x && jb < ri.y) || jb == ri.z;
    }
    float P0, P1, x0, x1;
    const float X0 = __uint_as_float(sv[2 * e]), X1 = __uint_as_float(sv[2 * e + 1]);
    const float d0 = __uint_as_float(dp[2 * e]), d1 = __uint_as_float(dp[2 * e + 1]);
    if (POLY && e < kBwdPolyPairs)
      bwd_pair<METHOD, true>(X0, X1, d0, d1, xf, mul2, add2, dsc2, radd2, l0, l1, P0, P1, x0, x1);
    else
      bwd_pair<METHOD, false>(X0, X1, d0, d1, xf, mul2, add2, dsc2, radd2, l0, l1, P0, P1, x0, x1);
    px[e] = pack_bf16x2(x0, x1);
  }
}

// Chooses the dQ chunk variant: masked or not (per row), FMA-pipe tanh when the
// whole warp's arguments are in range (warp vote).
template <int METHOD>
__device__ __forceinline__ void dq_dispatch(bool full, const uint32_t (&sv)[32], const uint32_t (&dp)[32],
                                            int j0, int4 ri, const Xf& xf, float mul, float addl,
                                            float dscale, float radd, uint32_t (&px)[16]) {
  bool poly = false;
  if constexpr (METHOD == CAPATTN_CAP_TANH) {
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) am = fmaxf(am, fabsf(__uint_as_float(sv[e])));
    poly = __all_sync(0xFFFFFFFFu, am * fabsf(xf.in) <= kTanhPolyMaxU);
  }
  if (poly) {
    if (full)
      dq_chunk<METHOD, false, true>(sv, dp, j0, ri, xf, mul, addl, dscale, radd, px);
    else
      dq_chunk<METHOD, true, true>(sv, dp, j0, ri, xf, mul, addl, dscale, radd, px);
  } else {
    if (full)
      dq_chunk<METHOD, false, false>(sv, dp, j0, ri, xf, mul, addl, dscale, radd, px);
    else
      dq_chunk<METHOD, true, false>(sv, dp, j0, ri, xf, mul, addl, dscale, radd, px);
  }
}

// ======================================================================= dK / dV
template <int METHOD>
__global__ void __launch_bounds__(NTHREADS, 1)
dkv_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
              const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[24];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ __align__(16) float4 colc[2][BT];  // per query column: mul, add - lse2, dscale, radd
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
  const uint32_t bar_sdp = smem_u32(&bars[5]);     // + part*8: scores of the part ready
  const uint32_t bar_ew = smem_u32(&bars[7]);      // + part*8: part's P / dX written
  const uint32_t bar_final = smem_u32(&bars[10]);
  const uint32_t bar_cfull = smem_u32(&bars[11]);  // + (2*wg + cb)*8: column constants written
  const uint32_t bar_cfree = smem_u32(&bars[15]);  // + (2*wg + cb)*8: column constants consumed

  const uint32_t* map = p.kmap + ((size_t)b * p.nk + kt) * p.wq;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_kv, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(bar_sdp + 8 * c, 1);
      mbar_init(bar_ew + 8 * c, 8);
    }
    for (int c = 0; c < 4; ++c) {
      mbar_init(bar_cfull + 8 * c, 128);
      mbar_init(bar_cfree + 8 * c, 128);
    }
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
      StepIter st(map, p.wq, p.G);
      int hh, qt, j = 0;
      while (!abort_flag && st.next(hh, qt)) {
        const int h = g * p.G + hh;
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
      drain_wait(bar_kv, 0);
      for (int jj = (j > NSTAGE ? j - NSTAGE : 0); jj < j; ++jj)
        drain_wait(bar_full + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && n > 0) {
      // scores of part `part` of step j into that part's TMEM buffer
      auto scores = [&](int j, int part) {
        const uint32_t sQ = sQD + (j % NSTAGE) * 2 * TILE, sO = sQ + TILE;
        issue_scores_part(tmem + 128u * part, sK, sQ, part);         // S^T  = K Q^T
        issue_scores_part(tmem + 128u * part + 64u, sV, sO, part);   // dP^T = V dO^T
        mma_commit(bar_sdp + 8 * part);
      };
      bool ok = mbar_wait(bar_kv, 0, p.status, &abort_flag) &&
                mbar_wait(bar_full, 0, p.status, &abort_flag);
      if (ok) {
        tc_fence_after();
        scores(0, 0);
        scores(0, 1);
      }
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % NSTAGE;
        const uint32_t sQ = sQD + s * 2 * TILE, sO = sQ + TILE;
        const bool more = j + 1 < n;
        for (int part = 0; part < 2; ++part) {
          if (!mbar_wait(bar_ew + 8 * part, j & 1, p.status, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool first = (j == 0) && (part == 0);
          issue_acc_part(tmem + 256u, tmem + 128u * part, sO, part, first);         // dV += P^T dO
          issue_acc_part(tmem + 384u, tmem + 128u * part + 64u, sQ, part, first);   // dK += dX^T Q
          if (part == 1) mma_commit(bar_empty + 8 * s);
          if (more) {
            if (part == 0 &&
                !mbar_wait(bar_full + 8 * ((j + 1) % NSTAGE), ((j + 1) / NSTAGE) & 1, p.status,
                           &abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            scores(j + 1, part);
          }
        }
      }
      // No wait for this commit here: the consumer warps wait for it, and
      // warp 1 re-checks it before freeing TMEM.
      mma_commit(bar_final);
    }
  } else {
    const int wg = (warp - 2) >> 2;        // 32 columns of each part
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;     // key row within the tile (TMEM lane)
    const int tid = (warp - 2 - 4 * wg) * 32 + lane;  // 0..127 within the warpgroup
    const int jrow = k0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const Xf xf = make_xf<METHOD>(p.cap, p.sm_scale);
    // query column whose constants this thread loads: the warpgroup's 32
    // columns of part 0 and of part 1
    const int my_col = (tid < 32) ? 32 * wg + tid : 64 + 32 * wg + (tid - 32);
    bool aborted = false;
    StepIter nx(map, p.wq, p.G);
    int nh = 0, nqt = 0;
    bool have_next = nx.next(nh, nqt);
    ColRaw cur = load_col_raw(p, b, g * p.G + nh, nqt, my_col, have_next && tid < 64);
    int cur_qt = nqt;
    for (int step = 0; step < n && have_next; ++step) {
      const int cb = step & 1, cu = step >> 1;
      const uint32_t my_cfull = bar_cfull + 8 * (2 * wg + cb);
      const uint32_t my_cfree = bar_cfree + 8 * (2 * wg + cb);
      if (step >= 2 && !mbar_wait_warp(my_cfree, (cu - 1) & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      if (tid < 64) {
        float mul, add;
        row_consts<METHOD>(p.cap, p.sm_scale, cur.temp, &mul, &add);
        colc[cb][my_col] = make_float4(mul, add - cur.lse2,
                                       row_dscale<METHOD>(p.cap, p.sm_scale, cur.temp), cur.radd);
        coli[cb][my_col] = cur.ri;
      }
      mbar_arrive(my_cfull);
      const int2 fr = p.qfull[(size_t)b * p.nq + cur_qt];
      const bool tile_full = (kt >= fr.x) && (kt < fr.y);
      have_next = nx.next(nh, nqt);
      const ColRaw nxt = load_col_raw(p, b, g * p.G + nh, nqt, my_col, have_next && tid < 64);
      if (!mbar_wait_warp(my_cfull, cu & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      for (int part = 0; part < 2; ++part) {
        if (!mbar_wait_warp(bar_sdp + 8 * part, step & 1, p.status, &abort_flag)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        if (tile_full)
          dkv_part<METHOD, false>(colc[cb], coli[cb], wg, part, jrow, xf, lane_base);
        else
          dkv_part<METHOD, true>(colc[cb], coli[cb], wg, part, jrow, xf, lane_base);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ew + 8 * part);
      }
      if (aborted) break;
      mbar_arrive(my_cfree);
      cur = nxt;
      cur_qt = nqt;
    }
    // ---------------------------------------------------------- epilogue
    bool have = false;
    if (n > 0 && !aborted) {
      have = mbar_wait_warp(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
    }
    // warpgroup 0 writes dV, warpgroup 1 writes dK
    void* outp = wg == 0 ? p.dv : p.dk;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(outp) + ((size_t)(b * p.L + jrow) * p.Hkv + g) * HD;
    const uint32_t acc = lane_base + (wg == 0 ? 256u : 384u);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      if (have) {
        uint32_t v[32];
        tmem_ld32(acc + c * 32, v);
        tmem_wait_ld();
        if (jrow < p.L) store_row_bf16(dst + c * 32, v);
      } else if (jrow < p.L) {
        store_zero_bf16(dst + c * 32);
      }
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
  const uint32_t bar_sdp = smem_u32(&bars[5]);     // + part*8
  const uint32_t bar_ew = smem_u32(&bars[7]);      // + part*8
  const uint32_t bar_final = smem_u32(&bars[10]);

  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(bar_sdp + 8 * c, 1);
      mbar_init(bar_ew + 8 * c, 8);
    }
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
      auto scores = [&](int j, int part) {
        const uint32_t sK = sKV + (j % NSTAGE) * 2 * TILE, sV = sK + TILE;
        issue_scores_part(tmem + 128u * part, sQ, sK, part);         // S  = Q K^T
        issue_scores_part(tmem + 128u * part + 64u, sO, sV, part);   // dP = dO V^T
        mma_commit(bar_sdp + 8 * part);
      };
      bool ok = mbar_wait(bar_q, 0, p.status, &abort_flag) &&
                mbar_wait(bar_full, 0, p.status, &abort_flag);
      if (ok) {
        tc_fence_after();
        scores(0, 0);
        scores(0, 1);
      }
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % NSTAGE;
        const uint32_t sK = sKV + s * 2 * TILE;
        const bool more = j + 1 < n;
        for (int part = 0; part < 2; ++part) {
          if (!mbar_wait(bar_ew + 8 * part, j & 1, p.status, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_acc_part(tmem + 256u, tmem + 128u * part + 64u, sK, part, (j == 0) && (part == 0));
          if (part == 1) mma_commit(bar_empty + 8 * s);
          if (more) {
            if (part == 0 &&
                !mbar_wait(bar_full + 8 * ((j + 1) % NSTAGE), ((j + 1) / NSTAGE) & 1, p.status,
                           &abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            scores(j + 1, part);
          }
        }
      }
      mma_commit(bar_final);
    }
  } else {
    const int wg = (warp - 2) >> 2;        // 32 key columns of each part
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
    const Xf xf = make_xf<METHOD>(p.cap, p.sm_scale);
    float mul, add;
    row_consts<METHOD>(p.cap, p.sm_scale, temp, &mul, &add);
    const float addl = add - (fin ? lse * kL2E : 0.f);
    const float dscale = row_dscale<METHOD>(p.cap, p.sm_scale, temp);
    const float radd = -dl + (fin ? p.z_loss_weight * lse : 0.f);
    bool aborted = false;
    TileIter it(map, p.wk);
    for (int j = 0; j < n && !aborted; ++j) {
      int t;
      it.next(t);
      const int k0 = t * BT;
      const bool full = (ri.x <= k0) && (ri.y >= k0 + BT);
      for (int part = 0; part < 2; ++part) {
        if (!mbar_wait_warp(bar_sdp + 8 * part, j & 1, p.status, &abort_flag)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t sbuf = lane_base + 128u * part, dbuf = sbuf + 64u;
        const int pc0 = 32 * wg;
        uint32_t sv[32], dp[32], px[16];
        tmem_ld32(sbuf + pc0, sv);
        tmem_ld32(dbuf + pc0, dp);
        tmem_wait_ld();
        dq_dispatch<METHOD>(full, sv, dp, k0 + 64 * part + pc0, ri, xf, mul, addl, dscale, radd, px);
        __syncwarp();
        // packed dX of columns [pc0, pc0 + 32): 16 columns at dbuf + pc0
        tmem_st16(dbuf + pc0, px);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ew + 8 * part);
      }
    }
    bool have = false;
    if (n > 0 && !aborted) {
      have = mbar_wait_warp(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
    }
    // warpgroup wg writes dQ columns [64 wg, 64 wg + 64)
    __nv_bfloat16* dqg = static_cast<__nv_bfloat16*>(p.dq) + ((size_t)(b * p.L + i) * p.Hq + h) * HD;
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      const int col = 64 * wg + 32 * c;
      if (have) {
        uint32_t v[32];
        tmem_ld32(lane_base + 256u + col, v);
        tmem_wait_ld();
        if (valid) store_row_bf16(dqg + col, v);
      } else if (valid) {
        store_zero_bf16(dqg + col);
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
