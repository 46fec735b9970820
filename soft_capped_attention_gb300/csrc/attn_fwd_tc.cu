// bf16 forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: triton_kernels.py make_triton_forward_kernel (scores, cap,
// temperature, masks, online softmax with the l / m residuals), with the cap
// forms of mosaic_backward.py _apply_cap_mosaic, the ranker mask of
// ranker_mask_mosaic_kv_q (transposed) and an exp2-domain softmax as in the
// Mosaic kernels.
//
// One CTA owns two 128-row query tiles (Q0, Q1) of one (batch, head) and walks
// the union of their KV visit maps.  Warp roles (18 warps):
//   warp 0       TMA producer: Q0, Q1 once, then K_j / V_j into a 2-stage ring;
//   warp 1       TMEM allocator and MMA issuer (warp-wide loop, one elected
//                lane issues), ping-ponging the two tiles so that one tile's
//                softmax overlaps the other tile's MMAs:
//                  S0_j S1_j | PV0_j S0_{j+1} | PV1_j S1_{j+1} | ...
//                  S_t = Q_t K_j^T  (SS MMA, M = N = 128)
//                  O_t += P_t V_j   (TS MMA: P_t read from TMEM as bf16)
//   warps 2..9   softmax of tile 0, warps 10..17 softmax of tile 1.  Each row
//                (TMEM lane) is shared by two threads, one per half of the
//                step's 128 key columns (warps 2..5 / 10..13 the first half).
//                Pass 1 takes the range of the half-row's raw scores; the two
//                halves exchange it through shared memory (every cap is
//                increasing, so the logit maximum is the transformed raw
//                maximum); pass 2 applies sm_scale, cap, temperature and the
//                row's live span and writes P = 2^(x - m) as packed bf16 over
//                the first 32 columns of the half; each half keeps its part of
//                l.  The running max is only moved (and O rescaled in TMEM, each
//                half its 64 columns of O) when it grows by more than 2^8;
//                otherwise P stays <= 256.
// A tile's S_{j+1} is issued after its PV_j, so when the softmax sees S_{j+1}
// complete, PV_j is complete too and O may be rescaled in place.
// TMEM: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512); packed P of a
// tile's key columns [0, 64) at S [0, 32), of [64, 128) at S [64, 96).
// At the end each (tile, half) group writes its normalised O as bf16 into its
// slab of the tile's Q in shared memory and one thread stores the slab by TMA.
#include "fwd_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

using namespace fwdtc;

constexpr int NSTAGE = 2;
template <int HD>
constexpr int smem_bytes() { return 2 * tile_bytes<HD>() + NSTAGE * 2 * tile_bytes<HD>() + 1024; }
constexpr int NTHREADS = 576;


// Iterates the union of two rows of a visit bitmap, reporting per tile which
// of the two query tiles is live in it.
struct PairIter {
  const uint32_t* m0;
  const uint32_t* m1;  // null when the second tile does not exist
  int nwords, w;
  uint32_t b0, b1;
  __device__ PairIter(const uint32_t* a, const uint32_t* c, int n) : m0(a), m1(c), nwords(n), w(0) {
    b0 = n > 0 ? a[0] : 0u;
    b1 = (n > 0 && c) ? c[0] : 0u;
  }
  __device__ bool next(int& t, bool& a0, bool& a1) {
    while ((b0 | b1) == 0u) {
      if (++w >= nwords) return false;
      b0 = m0[w];
      b1 = m1 ? m1[w] : 0u;
    }
    const uint32_t u = b0 | b1;
    const int bit = __ffs(u) - 1;
    const uint32_t mask = 1u << bit;
    a0 = (b0 & mask) != 0u;
    a1 = (b1 & mask) != 0u;
    b0 &= ~mask;
    b1 &= ~mask;
    t = w * 32 + bit;
    return true;
  }
};

__device__ __forceinline__ int count_union(const uint32_t* a, const uint32_t* c, int n) {
  int s = 0;
  for (int w = 0; w < n; ++w) s += __popc(a[w] | (c ? c[w] : 0u));
  return s;
}


template <int METHOD, int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
              const Params p) {
  constexpr int TILE = tile_bytes<HD>();
  constexpr int NSLAB = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[16];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  // half-row partial results exchanged between the two halves of a row:
  // [step parity][tile][half][row] = (max, min) of the half's raw scores,
  // and at the end (l of the half, unused)
  __shared__ float2 xch[2][2][2][BM];

  const int hb = blockIdx.x;
  const int h = hb % p.Hq, b = hb / p.Hq;
  const int npair = (p.nq + 1) >> 1;
  const int pr = npair - 1 - (int)blockIdx.y;  // heaviest (latest) query tiles first
  const int qt0 = 2 * pr;
  const bool has1 = qt0 + 1 < p.nq;
  const int g = h / p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ0 = base, sQ1 = base + TILE;
  const uint32_t sKV = base + 2 * TILE;  // stage s: K at sKV + s*2*TILE, V at + TILE

  const uint32_t bar_q = smem_u32(&bars[0]);
  const uint32_t bar_kfull = smem_u32(&bars[1]);   // + s*8
  const uint32_t bar_vfull = smem_u32(&bars[3]);   // + s*8
  const uint32_t bar_empty = smem_u32(&bars[5]);   // + s*8
  const uint32_t bar_sfull = smem_u32(&bars[7]);   // + tile*8
  const uint32_t bar_pfull = smem_u32(&bars[9]);   // + tile*8
  const uint32_t bar_final = smem_u32(&bars[11]);
  const uint32_t bar_xch = smem_u32(&bars[12]);    // + tile*8: both halves of the rows wrote xch

  const uint32_t* map0 = p.qmap + ((size_t)b * p.nq + qt0) * p.wk;
  const uint32_t* map1 = has1 ? map0 + p.wk : nullptr;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_sfull + 8 * t, 1);
      mbar_init(bar_pfull + 8 * t, 8);
      mbar_init(bar_xch + 8 * t, 8);
    }
    mbar_init(bar_final, 1);
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
  const int n = count_union(map0, map1, p.wk);

  // Softmax rows (warps 2..17): per-row constants, and whether every row of the
  // CTA can use a fixed reference instead of the running max (capped method,
  // logit window <= kSpanMax, and the running max m / sum l not requested).
  const int sw = warp - 2;                     // 0..15 for softmax warps
  const int tsel = (sw >> 3) & 1;              // query tile 0 or 1
  const int half = (sw >> 2) & 1;              // key columns [64 half, 64 half + 64) of each step
  const int r = (warp & 3) * 32 + lane;
  const int i = (qt0 + tsel) * BM + r;
  const bool valid = warp >= 2 && i < p.L;
  const float temp = (p.temp && valid) ? p.temp[(size_t)b * p.L + i] : 1.f;
  float rmul, radd;
  row_consts<METHOD>(p.cap, p.sm_scale, temp, &rmul, &radd);
  float x_hi = 0.f, span = 0.f;
  if constexpr (METHOD == CAPATTN_CAP_TANH || METHOD == CAPATTN_CAP_SOFT_SIGN) {
    x_hi = fabsf(rmul);
    span = 2.f * fabsf(rmul);
  } else if constexpr (METHOD == CAPATTN_CAP_ALSC) {
    x_hi = fmaxf(radd, rmul + radd);
    span = fabsf(rmul);
  }
  const bool fixed_ref = (METHOD != CAPATTN_CAP_NONE) && p.m == nullptr && p.l == nullptr &&
                         __syncthreads_and(warp < 2 || span <= kSpanMax);
  const float m_fixed = fixed_reference(x_hi, span);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (n > 0) {
      const bool leader = elect_one_sync();
      if (leader) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&mo);
        mbar_expect_tx(bar_q, 2 * TILE);
        for (int sl = 0; sl < NSLAB; ++sl) {
          tma_load_4d(sQ0 + sl * SLAB, &mq, bar_q, 64 * sl, h, qt0 * BM, b);
          tma_load_4d(sQ1 + sl * SLAB, &mq, bar_q, 64 * sl, h, qt0 * BM + BM, b);
        }
      }
      __syncwarp();
      PairIter it(map0, map1, p.wk);
      int t, j = 0;
      bool a0, a1;
      while (it.next(t, a0, a1)) {
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (u > 0 && !mbar_wait_warp(bar_empty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) break;
        if (leader) {
          const uint32_t sK = sKV + s * 2 * TILE, sV = sK + TILE;
          mbar_expect_tx(bar_kfull + 8 * s, TILE);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sK + sl * SLAB, &mk, bar_kfull + 8 * s, 64 * sl, g, t * BN, b);
          mbar_expect_tx(bar_vfull + 8 * s, TILE);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sV + sl * SLAB, &mv, bar_vfull + 8 * s, 64 * sl, g, t * BN, b);
        }
        __syncwarp();
        ++j;
      }
      if (leader) {
        drain_wait(bar_q, 0);
        for (int jj = (j > NSTAGE ? j - NSTAGE : 0); jj < j; ++jj) {
          drain_wait(bar_kfull + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
          drain_wait(bar_vfull + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      const bool leader = elect_one_sync();
      const uint64_t dQ0 = smem_desc(sQ0, 16, 1024), dQ1 = smem_desc(sQ1, 16, 1024);
      const uint64_t dKV = smem_desc(sKV, 16, 1024);      // K / V stages, K-major
      const uint64_t dKVmn = smem_desc(sKV, SLAB, 1024);  // the same, MN-major
      bool ok = mbar_wait_warp(bar_q, 0, p.status, &abort_flag);
      tc_fence_after();
      PairIter it(map0, map1, p.wk);
      int t;
      bool c0 = false, c1 = false;  // activity of the current tile
      bool n0 = false, n1 = false;  // activity of the next tile
      it.next(t, c0, c1);
      int pc0 = 0, pc1 = 0;         // p_full phases consumed per query tile
      uint32_t started0 = 0, started1 = 0;
      if (ok) ok = mbar_wait_warp(bar_kfull, 0, p.status, &abort_flag);
      if (ok) {
        tc_fence_after();
        if (leader) {
          if (c0) { issue_s<HD>(tmem, dQ0, dKV); mma_commit(bar_sfull); }
          if (c1) { issue_s<HD>(tmem + 128u, dQ1, dKV); mma_commit(bar_sfull + 8); }
        }
        __syncwarp();
      }
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % NSTAGE;
        const uint32_t vo = (uint32_t)(s * 2 * TILE + TILE);
        n0 = n1 = false;
        const bool more = (j + 1 < n) && it.next(t, n0, n1);
        const int s1 = (j + 1) % NSTAGE;
        const uint32_t ko = (uint32_t)(s1 * 2 * TILE);
        if (!mbar_wait_warp(bar_vfull + 8 * s, (j / NSTAGE) & 1, p.status, &abort_flag)) break;
        if (c0) {
          if (!mbar_wait_warp(bar_pfull, pc0 & 1, p.status, &abort_flag)) break;
          ++pc0;
          tc_fence_after();
          if (leader) issue_pv<HD>(tmem + 256u, tmem, desc_add(dKVmn, vo), started0);
          __syncwarp();
          started0 = 1;
        }
        if (more) {
          if (!mbar_wait_warp(bar_kfull + 8 * s1, ((j + 1) / NSTAGE) & 1, p.status, &abort_flag)) break;
          tc_fence_after();
          if (n0 && leader) { issue_s<HD>(tmem, dQ0, desc_add(dKV, ko)); mma_commit(bar_sfull); }
          __syncwarp();
        }
        if (c1) {
          if (!mbar_wait_warp(bar_pfull + 8, pc1 & 1, p.status, &abort_flag)) break;
          ++pc1;
          tc_fence_after();
          if (leader) issue_pv<HD>(tmem + 384u, tmem + 128u, desc_add(dKVmn, vo), started1);
          __syncwarp();
          started1 = 1;
        }
        if (leader) {
          mma_commit(bar_empty + 8 * s);
          if (more && n1) { issue_s<HD>(tmem + 128u, dQ1, desc_add(dKV, ko)); mma_commit(bar_sfull + 8); }
        }
        __syncwarp();
        c0 = n0;
        c1 = n1;
      }
      // The MMA thread does not wait for its own commit here: the consumer
      // warps wait for it, and warp 1 re-checks it before freeing TMEM.
      if (leader) mma_commit(bar_final);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_base = tmem + lane_off + (uint32_t)tsel * 128u + 64u * (uint32_t)half;
    // this half's HD / 2 columns of the tile's O
    const uint32_t o_base = tmem + lane_off + 256u + (uint32_t)tsel * 128u + (uint32_t)(HD / 2) * half;
    const uint32_t my_sfull = bar_sfull + 8 * tsel, my_pfull = bar_pfull + 8 * tsel;
    const uint32_t my_xch = bar_xch + 8 * tsel;
    const int4 ri = valid ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
    const bool neg = temp < 0.f;
    // the row minimum is needed for a negative temperature and for the range
    // check of the tanh polynomial
    const bool need_min = (METHOD == CAPATTN_CAP_TANH) || __any_sync(0xFFFFFFFFu, neg);
    const Xf xf = make_xf<METHOD>(p.cap, p.sm_scale);
    TanhFold tf{};
    if constexpr (METHOD == CAPATTN_CAP_TANH) tf = tanh_fold(xf.in, rmul);
    float m_use = fixed_ref ? m_fixed : -INFINITY, m_true = -INFINITY, lsum = 0.f;
    int cnt = 0;
    bool aborted = false;
    PairIter it(map0, map1, p.wk);
    int t;
    bool a0, a1;
    while (it.next(t, a0, a1)) {
      if (!(tsel == 0 ? a0 : a1)) continue;
      const int k0 = t * BN;
      const int c0 = k0 + 64 * half;           // first key column of this half
      if (!mbar_wait_warp(my_sfull, cnt & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const bool full = (ri.x <= k0) && (ri.y >= k0 + BN);
      const bool warp_partial = __any_sync(0xFFFFFFFFu, !full);
      float alpha = 1.f;
      bool poly = false;
      if (!fixed_ref) {
      // ---- pass 1: range of the half-row's live raw scores, kept in registers
      uint32_t v[64];
      tmem_ld32(s_base, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(s_base + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_wait_ld();
      float vmax, vmin;
      if (!full)
        row_range<true, 64>(v, c0, ri, vmax, vmin);
      else if (need_min)
        row_range_full<true, 64>(v, vmax, vmin);
      else
        row_range_full<false, 64>(v, vmax, vmin);
      // ---- combine with the other half of the row
      xch[cnt & 1][tsel][half][r] = make_float2(vmax, vmin);
      __syncwarp();
      if (lane == 0) mbar_arrive(my_xch);
      if (!mbar_wait_warp(my_xch, cnt & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      {
        const float2 other = xch[cnt & 1][tsel][half ^ 1][r];
        vmax = fmaxf(vmax, other.x);
        vmin = fminf(vmin, other.y);
      }
      // Every cap is increasing: the logit maximum is the transform of the raw
      // maximum (of the minimum for a negative temperature).
      const float xsel = neg ? vmin : vmax;
      const float x_max =
          (vmax == -INFINITY) ? -INFINITY : fmaf(rmul, cap_f<METHOD>(xsel, xf), radd);
      // tanh on the FMA pipe when the whole warp's arguments are in range (the
      // two halves of a row see the same range, so they decide alike)
      if constexpr (METHOD == CAPATTN_CAP_TANH)
        poly = __all_sync(0xFFFFFFFFu, tf.ok && fmaxf(vmax, -vmin) * fabsf(xf.in) <= kTanhPolyMaxU);
      m_true = fmaxf(m_true, x_max);
      const float m_new = fmaxf(m_use, x_max);
      const bool resc = m_new > m_use + kRescaleThreshold;
      if (resc) {
        alpha = ex2_approx(m_use - m_new);
        m_use = m_new;
      }
      // ---- O rescale of this half's 64 columns (PV of the previous live tile is complete)
      if (cnt > 0 && __any_sync(0xFFFFFFFFu, resc)) {
#pragma unroll 1
        for (int c = 0; c < HD / 64; ++c) {
          uint32_t o[32];
          tmem_ld32(o_base + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(o_base + c * 32, o);
        }
      }
      }  // !fixed_ref
      // ---- pass 2: P = 2^(x - m_use), packed bf16 over this half's columns [0, 32)
      const bool any = m_use != -INFINITY;
      const float addm = radd - (any ? m_use : 0.f);
      const bool fast = full && any;
      // Sub-chunk c (16 columns) is reloaded from TMEM (the next one's load in
      // flight while it is computed) and packed over columns [8 c, 8 c + 8).
      float psum = 0.f;
      {
        uint32_t va[16], vb[16], pk[8];
        tmem_ld16(s_base, va);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
          tmem_ld16(s_base + 16 * (c + 1), vb);
          // (warp-wide vote, taken only in steps with partially masked rows)
          if (warp_partial && sub_dead(ri, c0 + 16 * c)) {
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = 0u;
          } else {
            if (fixed_ref) poly = sub_poly<METHOD>(va, tf, xf);
            psum += p_dispatch<METHOD>(fast, poly, va, pk, xf, tf, rmul, addm, c0 + 16 * c, ri, any);
          }
          __syncwarp();
          tmem_st8(s_base + 8 * c, pk);
          tmem_wait_ld();
          if (c + 2 < 4) tmem_ld16(s_base + 16 * (c + 2), va);
          // (warp-wide vote, taken only in steps with partially masked rows)
          if (warp_partial && sub_dead(ri, c0 + 16 * (c + 1))) {
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = 0u;
          } else {
            if (fixed_ref) poly = sub_poly<METHOD>(vb, tf, xf);
            psum += p_dispatch<METHOD>(fast, poly, vb, pk, xf, tf, rmul, addm, c0 + 16 * (c + 1), ri, any);
          }
          __syncwarp();
          tmem_st8(s_base + 8 * (c + 1), pk);
          if (c + 2 < 4) tmem_wait_ld();
        }
      }
      lsum = lsum * alpha + psum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(my_pfull);
      ++cnt;
    }
    // ---------------------------------------------------------- epilogue
    // l of the whole row: the two halves add their parts (one more exchange;
    // with the running max every step used one exchange phase, with the fixed
    // reference none did)
    float l_row = lsum;
    if (cnt > 0 && !aborted) {
      const int xp = fixed_ref ? 0 : (cnt & 1);
      xch[xp][tsel][half][r] = make_float2(lsum, 0.f);
      __syncwarp();
      if (lane == 0) mbar_arrive(my_xch);
      if (mbar_wait_warp(my_xch, xp, p.status, &abort_flag))
        l_row = lsum + xch[xp][tsel][half ^ 1][r].x;
      else
        aborted = true;
    }
    // Every MMA has completed before O is read and before Q's shared memory
    // takes O: also for a tile with no live step in a CTA that has some (its Q
    // was loaded; writing O over it before that load lands would lose O).
    bool have_o = false;
    if (n > 0 && !aborted) {
      const bool done = mbar_wait_warp(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
      have_o = done && cnt > 0;
    }
    const bool live = l_row > 0.f;
    const float inv = live ? 1.f / l_row : 0.f;
    // O leaves through shared memory: once every MMA has completed, this
    // half's slab of the tile's Q is free and takes the rows' 64 bf16 values in
    // the swizzled layout; one TMA store per (tile, half) writes the slab (rows
    // past L are clipped by the tensor map).
    // HD = 128: each half fills its own slab; HD = 64: the two halves fill the
    // two halves (16-byte chunks [0, 4) and [4, 8)) of the tile's one slab.
    const uint32_t tile_smem = tsel ? sQ1 : sQ0;
    const uint32_t oslab = tile_smem + (HD == 128 ? (uint32_t)half * SLAB : 0u);
    const int chunk0 = HD == 128 ? 0 : 4 * half;
#pragma unroll 1
    for (int c = 0; c < HD / 64; ++c) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(o_base + c * 32, o);
        tmem_wait_ld();
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float a = (have_o && live) ? __uint_as_float(o[2 * e]) * inv : 0.f;
        const float bb = (have_o && live) ? __uint_as_float(o[2 * e + 1]) * inv : 0.f;
        pk[e] = pack_bf16x2(a, bb);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e)
        st_swz_chunk(oslab, r, chunk0 + 4 * c + e, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
    }
    fence_async_smem();
    if constexpr (HD == 128) {
      named_bar_sync(1 + (sw >> 2), 128);  // the four warps of this (tile, half)
      if ((sw & 3) == 0 && lane == 0 && (tsel == 0 || has1)) {
        tma_store_4d(&mo, oslab, 64 * half, h, (qt0 + tsel) * BM, b);
        bulk_commit();
        bulk_wait_read0();
      }
    } else {
      named_bar_sync(1 + tsel, 256);       // the eight warps of this tile
      if ((sw & 7) == 0 && lane == 0 && (tsel == 0 || has1)) {
        tma_store_4d(&mo, tile_smem, 0, h, (qt0 + tsel) * BM, b);
        bulk_commit();
        bulk_wait_read0();
      }
    }
    if (valid && half == 0) {
      const size_t rr = ((size_t)b * p.Hq + h) * p.L + i;
      p.lse[rr] = live ? (m_use + log2f(l_row)) * kLn2 : -INFINITY;
      if (p.m) p.m[rr] = live ? m_true * kLn2 : -INFINITY;
      if (p.l) p.l[rr] = live ? l_row * ex2_approx(m_use - m_true) : 0.f;
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

template <int METHOD, int HD>
cudaError_t launch_fwd_hd(const Params& p, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mo;
  cudaError_t e = make_bhld_map(&mq, p.q, p.B, p.L, p.Hq, HD, BM);
  if (e == cudaSuccess) e = make_bhld_map(&mk, p.k, p.B, p.Lk, p.Hkv, HD, BN);
  if (e == cudaSuccess) e = make_bhld_map(&mv, p.v, p.B, p.Lk, p.Hkv, HD, BN);
  if (e == cudaSuccess) e = make_bhld_map(&mo, p.o, p.B, p.L, p.Hq, HD, BM);
  if (e != cudaSuccess) return e;
  auto kern = fwd_tc_kernel<METHOD, HD>;
  constexpr int SMEM_BYTES = smem_bytes<HD>();
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  prof_begin(CAPATTN_KERNEL_FWD, s);
  prof_count(CAPATTN_KERNEL_FWD, 1);
  e = launch_pdl(kern, dim3(p.Hq * p.B, (p.nq + 1) / 2), dim3(NTHREADS), SMEM_BYTES, s, mq, mk, mv, mo, p);
  if (e != cudaSuccess) return e;
  prof_end(CAPATTN_KERNEL_FWD, s);
  return cudaGetLastError();
}

template <int METHOD>
struct FwdTcLaunch {
  static cudaError_t run(const Params& p, cudaStream_t s) {
    return p.D == 64 ? launch_fwd_hd<METHOD, 64>(p, s) : launch_fwd_hd<METHOD, 128>(p, s);
  }
};

}  // namespace

// Whether every row can use the fixed reference (the persistent forward's
// only mode): a cap, no temperature, m and l not requested, and the capped
// logits' window (the same for every row without a temperature) within
// kSpanMax, checked here with a margin so that the device's fp32 test agrees.
static bool fixed_reference_everywhere(const Params& p) {
  if (p.cap.method == CAPATTN_CAP_NONE || p.m != nullptr || p.l != nullptr || p.temp != nullptr)
    return false;
  const double l2e = 1.4426950408889634;
  const double span = p.cap.method == CAPATTN_CAP_ALSC ? fabs((double)p.cap.alsc_out * l2e)
                                                       : 2.0 * fabs((double)p.cap.cap * l2e);
  return span <= 0.999 * (double)kSpanMax;
}

// Four forward kernels, chosen from the configuration alone by what measured
// fastest on GB300 (forward times against this file's two-tile kernel):
//  * the fixed reference everywhere, any mask: the persistent kernel
//    (attn_fwd3_tc.cu);
//  * otherwise, a sliding window or segment ids: one tile per CTA, two CTAs
//    per SM (attn_fwd1_tc.cu; -9 % on a 1024-key window and on packed
//    documents, where a CTA visits few key tiles and the CTAs' fixed costs
//    dominate);
//  * otherwise, ranker bounds: this file's two tiles per CTA (the others were
//    +4 % and +12 % on ranker histories);
//  * otherwise (causal or unmasked): one tile per CTA with two score buffers
//    (attn_fwd2_tc.cu; -3 % causal over 2048 keys, -7 % on 8192 unmasked keys).
cudaError_t launch_fwd_bf16(const Params& p, cudaStream_t s) {
  if (fixed_reference_everywhere(p)) return launch_fwd3_bf16(p, s);
  if (p.window_len > 0 || p.seg != nullptr) return launch_fwd1_bf16(p, s);
  if (p.bounds != nullptr) return dispatch_cap<FwdTcLaunch>(p.cap.method, p, s);
  return launch_fwd2_bf16(p, s);
}

}  // namespace capattn
