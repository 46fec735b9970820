// bf16 forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: triton_kernels.py make_triton_forward_kernel (scores, cap,
// temperature, masks, online softmax with the l / m residuals), with the cap
// forms of mosaic_backward.py _apply_cap_mosaic, the ranker mask of
// ranker_mask_mosaic_kv_q (transposed) and an exp2-domain softmax as in the
// Mosaic kernels.
//
// One CTA owns one 128-row query tile of one (batch, head) and walks the
// tile's KV visit map; two CTAs share an SM (half its TMEM and under half its
// shared memory each), so one CTA's softmax overlaps the other's MMAs and one
// CTA's prologue and epilogue overlap the other's steps.  Warp roles (10 warps):
//   warp 0      TMA producer: Q once, then K_j and V_j, each into its own
//               buffer as soon as the previous step's S (K) or PV (V) has read it;
//   warp 1      TMEM allocator and MMA issuer (warp-wide loop, one elected lane
//               issues):  S_0 | PV_0 S_1 | PV_1 S_2 | ...
//                 S = Q K_j^T   (SS MMA, M = N = 128)
//                 O += P V_j    (TS MMA: P read from TMEM as bf16)
//   warps 2..9  softmax.  Each row (TMEM lane) is shared by two threads, one
//               per half of the step's 128 key columns (warps 2..5 the first
//               half).  With a running max, pass 1 takes the range of the
//               half-row's raw scores and the two halves exchange it through
//               shared memory (every cap is increasing, so the logit maximum
//               is the transformed raw maximum); with the fixed reference (any
//               cap, m and l not requested) there is no pass 1.  Pass 2
//               applies sm_scale, cap, temperature and the row's live span and
//               writes P = 2^(x - m) as packed bf16 over the first 32 columns
//               of the half; each half keeps its part of l.  The running max
//               is only moved (and O rescaled in TMEM, each half its columns)
//               when it grows by more than 2^8; otherwise P stays <= 256.
// S_{j+1} is issued after PV_j, so when the softmax sees S_{j+1} complete,
// PV_j is complete too and O may be rescaled in place.
// TMEM (256 columns): S [0,128), O [128, 128 + HD); packed P of the key
// columns [0, 64) at S [0, 32), of [64, 128) at S [64, 96).
// At the end each half writes its normalised O as bf16 into its slab of Q in
// shared memory and one thread stores the slab by TMA.
#include "fwd_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

using namespace fwdtc;

// Q, K and V tiles
template <int HD>
constexpr int smem_bytes() { return 3 * tile_bytes<HD>() + 1024; }
constexpr int NTHREADS = 320;

template <int METHOD, int HD>
__global__ void __launch_bounds__(NTHREADS, 2)
fwd1_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
              const Params p) {
  constexpr int TILE = tile_bytes<HD>();
  constexpr int NSLAB = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[10];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  // half-row partial results exchanged between the two halves of a row:
  // [step parity][half][row] = (max, min) of the half's raw scores, and at the
  // end (l of the half, unused)
  __shared__ float2 xch[2][2][BM];

  const int hb = blockIdx.x;
  const int h = hb % p.Hq, b = hb / p.Hq;
  const int qt = p.nq - 1 - (int)blockIdx.y;  // heaviest (latest) query tiles first
  const int g = h / p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base, sK = base + TILE, sV = base + 2 * TILE;

  const uint32_t bar_q = smem_u32(&bars[0]);
  const uint32_t bar_kfull = smem_u32(&bars[1]);
  const uint32_t bar_kempty = smem_u32(&bars[2]);  // S of the step complete: K no longer read
  const uint32_t bar_vfull = smem_u32(&bars[3]);
  const uint32_t bar_vempty = smem_u32(&bars[4]);  // PV of the step complete: V no longer read
  const uint32_t bar_sfull = smem_u32(&bars[5]);
  const uint32_t bar_pfull = smem_u32(&bars[6]);   // P written by the 8 softmax warps
  const uint32_t bar_final = smem_u32(&bars[7]);
  const uint32_t bar_xch = smem_u32(&bars[8]);     // both halves of the rows wrote xch

  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    mbar_init(bar_kfull, 1);
    mbar_init(bar_kempty, 1);
    mbar_init(bar_vfull, 1);
    mbar_init(bar_vempty, 1);
    mbar_init(bar_sfull, 1);
    mbar_init(bar_pfull, 8);
    mbar_init(bar_final, 1);
    mbar_init(bar_xch, 8);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 256);
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

  // Softmax rows (warps 2..9): per-row constants, and whether every row of the
  // CTA can use a fixed reference instead of the running max (capped method,
  // logit window <= kSpanMax, and the running max m / sum l not requested).
  const int sw = warp - 2;                     // 0..7 for softmax warps
  const int half = (sw >> 2) & 1;              // key columns [64 half, 64 half + 64) of each step
  const int r = (warp & 3) * 32 + lane;
  const int i = qt * BM + r;
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
        mbar_expect_tx(bar_q, TILE);
        for (int sl = 0; sl < NSLAB; ++sl) tma_load_4d(sQ + sl * SLAB, &mq, bar_q, 64 * sl, h, qt * BM, b);
      }
      __syncwarp();
      // K_j once S_{j-1} has read K_{j-1}; V_j once PV_{j-1} has read V_{j-1}
      TileIter it(map, p.wk);
      int t, jk = 0, jv = 0;
      while (it.next(t)) {
        if (jk > 0 && !mbar_wait_warp(bar_kempty, (jk - 1) & 1, p.status, &abort_flag)) break;
        if (leader) {
          mbar_expect_tx(bar_kfull, TILE);
          for (int sl = 0; sl < NSLAB; ++sl) tma_load_4d(sK + sl * SLAB, &mk, bar_kfull, 64 * sl, g, t * BN, b);
        }
        __syncwarp();
        ++jk;
        if (jv > 0 && !mbar_wait_warp(bar_vempty, (jv - 1) & 1, p.status, &abort_flag)) break;
        if (leader) {
          mbar_expect_tx(bar_vfull, TILE);
          for (int sl = 0; sl < NSLAB; ++sl) tma_load_4d(sV + sl * SLAB, &mv, bar_vfull, 64 * sl, g, t * BN, b);
        }
        __syncwarp();
        ++jv;
      }
      if (leader) {
        // (on an early exit the loads in flight land before the CTA ends)
        drain_wait(bar_q, 0);
        if (jk > 0) drain_wait(bar_kfull, (jk - 1) & 1);
        if (jv > 0) drain_wait(bar_vfull, (jv - 1) & 1);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    //   S_0 | PV_0 S_1 | PV_1 S_2 | ...
    // S_{j+1} is issued after PV_j (which reads P_j from S's columns), and the
    // softmax seeing S_{j+1} complete knows PV_j is complete (in-order MMAs).
    if (n > 0) {
      const bool leader = elect_one_sync();
      const uint64_t dQ = smem_desc(sQ, 16, 1024);
      const uint64_t dK = smem_desc(sK, 16, 1024);
      const uint64_t dVmn = smem_desc(sV, SLAB, 1024);
      bool ok = mbar_wait_warp(bar_q, 0, p.status, &abort_flag) &&
                mbar_wait_warp(bar_kfull, 0, p.status, &abort_flag);
      if (ok) {
        tc_fence_after();
        if (leader) {
          issue_s<HD>(tmem, dQ, dK);
          mma_commit(bar_sfull);
          mma_commit(bar_kempty);
        }
        __syncwarp();
      }
      for (int j = 0; ok && j < n; ++j) {
        if (!mbar_wait_warp(bar_pfull, j & 1, p.status, &abort_flag)) break;
        if (!mbar_wait_warp(bar_vfull, j & 1, p.status, &abort_flag)) break;
        tc_fence_after();
        if (leader) {
          issue_pv<HD>(tmem + 128u, tmem, dVmn, j > 0 ? 1u : 0u);
          mma_commit(bar_vempty);
        }
        __syncwarp();
        if (j + 1 < n) {
          if (!mbar_wait_warp(bar_kfull, (j + 1) & 1, p.status, &abort_flag)) break;
          tc_fence_after();
          if (leader) {
            issue_s<HD>(tmem, dQ, dK);
            mma_commit(bar_sfull);
            mma_commit(bar_kempty);
          }
          __syncwarp();
        }
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
    const uint32_t s_base = tmem + lane_off + 64u * (uint32_t)half;
    // this half's HD / 2 columns of O
    const uint32_t o_base = tmem + lane_off + 128u + (uint32_t)(HD / 2) * half;
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
    TileIter it(map, p.wk);
    int t;
    while (it.next(t)) {
      const int k0 = t * BN;
      const int c0 = k0 + 64 * half;           // first key column of this half
      if (!mbar_wait_warp(bar_sfull, cnt & 1, p.status, &abort_flag)) {
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
      xch[cnt & 1][half][r] = make_float2(vmax, vmin);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_xch);
      if (!mbar_wait_warp(bar_xch, cnt & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      {
        const float2 other = xch[cnt & 1][half ^ 1][r];
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
      // ALSC's sigmoid on the FMA pipe when every live score is in the polynomial's range
      if constexpr (METHOD == CAPATTN_CAP_ALSC)
        poly = __all_sync(0xFFFFFFFFu, fmaxf(vmax, -vmin) <= p.cap.alsc_xmax);
      m_true = fmaxf(m_true, x_max);
      const float m_new = fmaxf(m_use, x_max);
      const bool resc = m_new > m_use + kRescaleThreshold;
      if (resc) {
        alpha = ex2_approx(m_use - m_new);
        m_use = m_new;
      }
      // ---- O rescale of this half's columns (PV of the previous live tile is complete)
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
            if (fixed_ref)
              poly = METHOD == CAPATTN_CAP_ALSC ? sub_alsc_poly(va, p.cap.alsc_xmax) : sub_poly<METHOD>(va, tf, xf);
            psum += p_dispatch<METHOD>(fast, poly, va, pk, xf, tf, rmul, addm, c0 + 16 * c, ri, any, &p.cap);
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
            if (fixed_ref)
              poly = METHOD == CAPATTN_CAP_ALSC ? sub_alsc_poly(vb, p.cap.alsc_xmax) : sub_poly<METHOD>(vb, tf, xf);
            psum += p_dispatch<METHOD>(fast, poly, vb, pk, xf, tf, rmul, addm, c0 + 16 * (c + 1), ri, any, &p.cap);
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
      if (lane == 0) mbar_arrive(bar_pfull);
      ++cnt;
    }
    // ---------------------------------------------------------- epilogue
    // l of the whole row: the two halves add their parts (one more exchange;
    // with the running max every step used one exchange phase, with the fixed
    // reference none did)
    float l_row = lsum;
    if (cnt > 0 && !aborted) {
      const int xp = fixed_ref ? 0 : (cnt & 1);
      xch[xp][half][r] = make_float2(lsum, 0.f);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_xch);
      if (mbar_wait_warp(bar_xch, xp, p.status, &abort_flag))
        l_row = lsum + xch[xp][half ^ 1][r].x;
      else
        aborted = true;
    }
    // Every MMA (and so the Q load) has completed before O is read and before
    // Q's shared memory takes O.
    bool have_o = false;
    if (n > 0 && !aborted) {
      const bool done = mbar_wait_warp(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
      have_o = done && cnt > 0;
    }
    const bool live = l_row > 0.f;
    const float inv = live ? 1.f / l_row : 0.f;
    // O leaves through shared memory: once every MMA has completed, this
    // half's slab of Q is free and takes the rows' 64 bf16 values in the
    // swizzled layout; one TMA store per half writes the slab (rows past L are
    // clipped by the tensor map).
    // HD = 128: each half fills its own slab; HD = 64: the two halves fill the
    // two halves (16-byte chunks [0, 4) and [4, 8)) of the tile's one slab.
    const uint32_t oslab = sQ + (HD == 128 ? (uint32_t)half * SLAB : 0u);
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
      named_bar_sync(1 + half, 128);  // the four warps of this half
      if ((sw & 3) == 0 && lane == 0) {
        tma_store_4d(&mo, oslab, 64 * half, h, qt * BM, b);
        bulk_commit();
        bulk_wait_read0();
      }
    } else {
      named_bar_sync(1, 256);         // the eight softmax warps
      if (sw == 0 && lane == 0) {
        tma_store_4d(&mo, sQ, 0, h, qt * BM, b);
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
    tmem_dealloc(tmem, 256);
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
  auto kern = fwd1_tc_kernel<METHOD, HD>;
  constexpr int SMEM_BYTES = smem_bytes<HD>();
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  prof_begin(CAPATTN_KERNEL_FWD, s);
  prof_count(CAPATTN_KERNEL_FWD, 1);
  e = launch_pdl(kern, dim3(p.Hq * p.B, p.nq), dim3(NTHREADS), SMEM_BYTES, s, mq, mk, mv, mo, p);
  if (e != cudaSuccess) return e;
  prof_end(CAPATTN_KERNEL_FWD, s);
  return cudaGetLastError();
}

template <int METHOD>
struct Fwd1TcLaunch {
  static cudaError_t run(const Params& p, cudaStream_t s) {
    return p.D == 64 ? launch_fwd_hd<METHOD, 64>(p, s) : launch_fwd_hd<METHOD, 128>(p, s);
  }
};

}  // namespace

cudaError_t launch_fwd1_bf16(const Params& p, cudaStream_t s) {
  return dispatch_cap<Fwd1TcLaunch>(p.cap.method, p, s);
}

}  // namespace capattn
