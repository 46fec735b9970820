// bf16 forward on the 5th-generation tensor cores with two score buffers.
//
// What it computes: triton_kernels.py make_triton_forward_kernel (scores, cap,
// temperature, masks, online softmax with the l / m residuals), with the cap
// forms of mosaic_backward.py _apply_cap_mosaic, the ranker mask of
// ranker_mask_mosaic_kv_q (transposed) and an exp2-domain softmax as in the
// Mosaic kernels.
//
// One CTA owns one 128-row query tile of one (batch, head) and walks the
// tile's KV visit map.  Each row (TMEM lane) is shared by four threads, one per
// quarter of the step's 128 key columns, and TMEM holds two score buffers, so
// the MMA issuer computes S of step j + 2 while the softmax works on step j + 1:
// the tensor pipe does not wait for the softmax, and the softmax finds the next
// scores ready when it finishes a step.  With the fixed reference (any cap, m
// and l not requested) a step needs no exchange between the four threads of a
// row; with the running max they exchange their quarter's range through shared
// memory, and before O is rescaled the softmax waits for the previous step's
// PV (the scores it sees complete are two steps ahead of its own PV).
// Warp roles (18 warps):
//   warp 0       TMA producer: lane 0 loads Q once and then K_j into a
//                three-stage ring (a stage is free once S_j has read it),
//                lane 1 loads V_j into a two-stage ring (free once PV_j has);
//   warp 1       TMEM allocator and MMA issuer (warp-wide loop, one elected
//                lane issues):  S_0 S_1 | PV_0 S_2 | PV_1 S_3 | ...
//                  S_j = Q K_j^T  into buffer j & 1 (SS MMA, M = N = 128)
//                  O += P_j V_j   (TS MMA: P_j read from buffer j & 1)
//   warps 2..17  softmax: warp w takes TMEM lanes 32 (w % 4) .. + 31 and key
//                columns [32 c, 32 c + 32) of each step, c = (w - 2) / 4; it
//                writes its P (bf16) over the first 16 of its own 32 columns.
// TMEM (512 columns): S buffers [0,128) and [128,256), O [256, 256 + HD).
// At the end each thread writes its quarter of the row's normalised O as bf16
// into Q's shared memory and one thread stores the tile by TMA.
#include "fwd_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

using namespace fwdtc;

constexpr int KST = 3;  // K stages
constexpr int VST = 2;  // V stages
// Q, KST K tiles, VST V tiles
template <int HD>
constexpr int smem_bytes() { return (1 + KST + VST) * tile_bytes<HD>() + 1024; }
constexpr int NTHREADS = 576;

// O += P V with P (bf16) in TMEM packed per 32-key quarter: keys
// [32 c, 32 c + 32) at pt + 32 c + [0, 16); V's MN-major descriptor (N = HD).
template <int HD>
__device__ __forceinline__ void issue_pv4(uint32_t d, uint32_t pt, uint64_t dV, uint32_t acc0) {
  constexpr uint32_t idesc = idesc_bf16(BM, HD, 0, 1);
#pragma unroll
  for (int ks = 0; ks < BN / 16; ++ks)
    mma_ts(d, pt + 32 * (ks >> 1) + 8 * (ks & 1), desc_add(dV, ks * 2048), idesc, (acc0 || ks > 0) ? 1u : 0u);
}

template <int METHOD, int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
fwd2_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
               const Params p) {
  constexpr int TILE = tile_bytes<HD>();
  constexpr int NSLAB = HD / 64;
  constexpr int OQ = HD / 4;  // O columns per thread (a quarter of the row)
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[1 + 2 * KST + 2 * VST + 8];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  // quarter-row partial results exchanged among the four threads of a row:
  // [step parity][quarter][row] = (max, min) of the quarter's raw scores, and
  // at the end (l of the quarter, unused)
  __shared__ float2 xch[2][4][BM];

  const int hb = blockIdx.x;
  const int h = hb % p.Hq, b = hb / p.Hq;
  const int qt = p.nq - 1 - (int)blockIdx.y;  // heaviest (latest) query tiles first
  const int g = h / p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK = base + TILE;                  // stage s at + s * TILE
  const uint32_t sV = base + (1 + KST) * TILE;      // stage s at + s * TILE

  const uint32_t bar_q = smem_u32(&bars[0]);
  const uint32_t bar_kfull = smem_u32(&bars[1]);             // + s*8
  const uint32_t bar_kempty = bar_kfull + 8 * KST;           // + s*8: S of the stage's step complete
  const uint32_t bar_vfull = bar_kempty + 8 * KST;           // + s*8
  const uint32_t bar_vempty = bar_vfull + 8 * VST;           // + s*8: PV of the stage's step complete
  const uint32_t bar_sfull = bar_vempty + 8 * VST;           // + x*8: S in buffer x complete
  const uint32_t bar_pfull = bar_sfull + 16;                 // + x*8: P in buffer x written (16 warps)
  const uint32_t bar_pvdone = bar_pfull + 16;                // one phase per PV
  const uint32_t bar_final = bar_pvdone + 8;
  const uint32_t bar_xch = bar_final + 8;                    // the four quarters of the rows wrote xch

  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_vempty + 8 * s, 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar_sfull + 8 * x, 1);
      mbar_init(bar_pfull + 8 * x, 16);
    }
    mbar_init(bar_pvdone, 1);
    mbar_init(bar_final, 1);
    mbar_init(bar_xch, 16);
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

  // Softmax rows (warps 2..17): per-row constants, and whether every row of the
  // CTA can use a fixed reference instead of the running max (capped method,
  // logit window <= kSpanMax, and the running max m / sum l not requested).
  const int sw = warp - 2;                     // 0..15 for softmax warps
  const int cq = sw >> 2;                      // key columns [32 cq, 32 cq + 32) of each step
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
    // Two independent loops in two lanes (each waits on its own ring).
    if (n > 0 && lane < 2) {
      bool ok = true;
      int j = 0;
      if (lane == 0) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mo);
        mbar_expect_tx(bar_q, TILE);
        for (int sl = 0; sl < NSLAB; ++sl) tma_load_4d(sQ + sl * SLAB, &mq, bar_q, 64 * sl, h, qt * BM, b);
        TileIter it(map, p.wk);
        int t;
        while (ok && it.next(t)) {
          const int s = j % KST, u = j / KST;
          if (u > 0 && !mbar_wait(bar_kempty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar_kfull + 8 * s, TILE);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sK + s * TILE + sl * SLAB, &mk, bar_kfull + 8 * s, 64 * sl, g, t * BN, b);
          ++j;
        }
        // (on an early exit the loads in flight land before the CTA ends)
        drain_wait(bar_q, 0);
        for (int jj = (j > KST ? j - KST : 0); jj < j; ++jj)
          drain_wait(bar_kfull + 8 * (jj % KST), (jj / KST) & 1);
      } else {
        tma_prefetch_desc(&mv);
        TileIter it(map, p.wk);
        int t;
        while (ok && it.next(t)) {
          const int s = j % VST, u = j / VST;
          if (u > 0 && !mbar_wait(bar_vempty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar_vfull + 8 * s, TILE);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sV + s * TILE + sl * SLAB, &mv, bar_vfull + 8 * s, 64 * sl, g, t * BN, b);
          ++j;
        }
        for (int jj = (j > VST ? j - VST : 0); jj < j; ++jj)
          drain_wait(bar_vfull + 8 * (jj % VST), (jj / VST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      const bool leader = elect_one_sync();
      const uint64_t dQ = smem_desc(sQ, 16, 1024);
      const uint64_t dK = smem_desc(sK, 16, 1024);
      const uint64_t dVmn = smem_desc(sV, SLAB, 1024);
      // S of step jj into buffer jj & 1; its K stage is free once it completes
      auto issue_scores = [&](int jj) -> bool {
        const int s = jj % KST;
        if (!mbar_wait_warp(bar_kfull + 8 * s, (jj / KST) & 1, p.status, &abort_flag)) return false;
        tc_fence_after();
        if (leader) {
          issue_s<HD>(tmem + 128u * (uint32_t)(jj & 1), dQ, desc_add(dK, (uint32_t)(s * TILE)));
          mma_commit(bar_sfull + 8 * (jj & 1));
          mma_commit(bar_kempty + 8 * s);
        }
        __syncwarp();
        return true;
      };
      bool ok = mbar_wait_warp(bar_q, 0, p.status, &abort_flag) && issue_scores(0);
      if (ok && n > 1) ok = issue_scores(1);
      for (int j = 0; ok && j < n; ++j) {
        const int x = j & 1, s = j % VST;
        if (!mbar_wait_warp(bar_pfull + 8 * x, (j >> 1) & 1, p.status, &abort_flag)) break;
        if (!mbar_wait_warp(bar_vfull + 8 * s, (j / VST) & 1, p.status, &abort_flag)) break;
        tc_fence_after();
        if (leader) {
          issue_pv4<HD>(tmem + 256u, tmem + 128u * (uint32_t)x, desc_add(dVmn, (uint32_t)(s * TILE)),
                        j > 0 ? 1u : 0u);
          mma_commit(bar_vempty + 8 * s);
          mma_commit(bar_pvdone);
        }
        __syncwarp();
        // S of step j + 2 overwrites P_j's buffer after PV_j (in-order MMAs)
        if (j + 2 < n && !issue_scores(j + 2)) break;
      }
      // The MMA thread does not wait for its own commit here: the consumer
      // warps wait for it, and warp 1 re-checks it before freeing TMEM.
      if (leader) mma_commit(bar_final);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_quarter = tmem + lane_off + 32u * (uint32_t)cq;   // + 128 x: buffer x
    const uint32_t o_base = tmem + lane_off + 256u + (uint32_t)(OQ * cq);
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
      const int c0 = k0 + 32 * cq;             // first key column of this quarter
      const uint32_t sb = s_quarter + 128u * (uint32_t)(cnt & 1);
      if (!mbar_wait_warp(bar_sfull + 8 * (cnt & 1), (cnt >> 1) & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const bool full = (ri.x <= k0) && (ri.y >= k0 + BN);
      const bool warp_partial = __any_sync(0xFFFFFFFFu, !full);
      // the quarter-row's 32 raw scores, read once for both passes
      uint32_t v[32];
      tmem_ld32(sb, v);
      tmem_wait_ld();
      float alpha = 1.f;
      bool poly = false;
      if (!fixed_ref) {
        // ---- pass 1: range of the quarter-row's live raw scores
        float vmax, vmin;
        if (!full)
          row_range<true, 32>(v, c0, ri, vmax, vmin);
        else if (need_min)
          row_range_full<true, 32>(v, vmax, vmin);
        else
          row_range_full<false, 32>(v, vmax, vmin);
        // ---- combine the four quarters of the row
        xch[cnt & 1][cq][r] = make_float2(vmax, vmin);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_xch);
        if (!mbar_wait_warp(bar_xch, cnt & 1, p.status, &abort_flag)) {
          aborted = true;
          break;
        }
#pragma unroll
        for (int o = 1; o < 4; ++o) {
          const float2 other = xch[cnt & 1][(cq + o) & 3][r];
          vmax = fmaxf(vmax, other.x);
          vmin = fminf(vmin, other.y);
        }
        // Every cap is increasing: the logit maximum is the transform of the raw
        // maximum (of the minimum for a negative temperature).
        const float xsel = neg ? vmin : vmax;
        const float x_max =
            (vmax == -INFINITY) ? -INFINITY : fmaf(rmul, cap_f<METHOD>(xsel, xf), radd);
        // tanh on the FMA pipe when the whole warp's arguments are in range (the
        // four quarters of a row see the same range, so they decide alike)
        if constexpr (METHOD == CAPATTN_CAP_TANH)
          poly = __all_sync(0xFFFFFFFFu, tf.ok && fmaxf(vmax, -vmin) * fabsf(xf.in) <= kTanhPolyMaxU);
        m_true = fmaxf(m_true, x_max);
        const float m_new = fmaxf(m_use, x_max);
        const bool resc = m_new > m_use + kRescaleThreshold;
        if (resc) {
          alpha = ex2_approx(m_use - m_new);
          m_use = m_new;
        }
        // ---- O rescale of this quarter's columns, once the previous step's PV
        // (the last one issued) has completed
        if (cnt > 0 && __any_sync(0xFFFFFFFFu, resc)) {
          if (!mbar_wait_warp(bar_pvdone, (cnt - 1) & 1, p.status, &abort_flag)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          if constexpr (OQ == 32) {
            uint32_t o[32];
            tmem_ld32(o_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(o_base, o);
          } else {
            uint32_t o[16];
            tmem_ld16(o_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(o_base, o);
          }
        }
      }  // !fixed_ref
      // ---- pass 2: P = 2^(x - m_use), packed bf16 over the quarter's columns [0, 16)
      const bool any = m_use != -INFINITY;
      const float addm = radd - (any ? m_use : 0.f);
      const bool fast = full && any;
      float psum = 0.f;
      {
        uint32_t pk[16];
        // (warp-wide vote, taken only in steps with partially masked rows)
        if (warp_partial && quarter_dead(ri, c0)) {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = 0u;
        } else {
          if (fixed_ref) poly = quarter_poly<METHOD>(v, tf, xf);
          psum = p_dispatch32<METHOD>(fast, poly, v, pk, xf, tf, rmul, addm, c0, ri, any);
        }
        __syncwarp();
        tmem_st16(sb, pk);
      }
      lsum = lsum * alpha + psum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfull + 8 * (cnt & 1));
      ++cnt;
    }
    // ---------------------------------------------------------- epilogue
    // l of the whole row: the four quarters add their parts (one more
    // exchange; with the running max every step used one exchange phase, with
    // the fixed reference none did)
    float l_row = lsum;
    if (cnt > 0 && !aborted) {
      const int xp = fixed_ref ? 0 : (cnt & 1);
      xch[xp][cq][r] = make_float2(lsum, 0.f);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_xch);
      if (mbar_wait_warp(bar_xch, xp, p.status, &abort_flag)) {
        l_row = 0.f;
#pragma unroll
        for (int o = 0; o < 4; ++o) l_row += xch[xp][o][r].x;
      } else {
        aborted = true;
      }
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
    // O leaves through Q's shared memory (free once every MMA has completed) in
    // the swizzled layout of the loads: this thread's OQ columns are 16-byte
    // chunks [OQ / 8 cq, OQ / 8 (cq + 1)) of the row across the tile's slabs.
    uint32_t o[OQ];
    if (have_o) {
      if constexpr (OQ == 32) tmem_ld32(o_base, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
      else tmem_ld16(o_base, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
      tmem_wait_ld();
    }
    uint32_t pk[OQ / 2];
#pragma unroll
    for (int e = 0; e < OQ / 2; ++e) {
      const float a = (have_o && live) ? __uint_as_float(o[2 * e]) * inv : 0.f;
      const float bb = (have_o && live) ? __uint_as_float(o[2 * e + 1]) * inv : 0.f;
      pk[e] = pack_bf16x2(a, bb);
    }
#pragma unroll
    for (int e = 0; e < OQ / 8; ++e) {
      const int chunk = (OQ / 8) * cq + e;   // 16-byte chunk of the row (0 .. HD / 8 - 1)
      st_swz_chunk(sQ + (uint32_t)(chunk >> 3) * SLAB, r, chunk & 7, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2],
                   pk[4 * e + 3]);
    }
    fence_async_smem();
    named_bar_sync(1, 512);  // the sixteen softmax warps
    if (sw == 0 && lane == 0) {
      for (int sl = 0; sl < NSLAB; ++sl) tma_store_4d(&mo, sQ + sl * SLAB, 64 * sl, h, qt * BM, b);
      bulk_commit();
      bulk_wait_read0();
    }
    if (valid && cq == 0) {
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
  auto kern = fwd2_tc_kernel<METHOD, HD>;
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
struct Fwd2TcLaunch {
  static cudaError_t run(const Params& p, cudaStream_t s) {
    return p.D == 64 ? launch_fwd_hd<METHOD, 64>(p, s) : launch_fwd_hd<METHOD, 128>(p, s);
  }
};

}  // namespace

cudaError_t launch_fwd2_bf16(const Params& p, cudaStream_t s) {
  return dispatch_cap<Fwd2TcLaunch>(p.cap.method, p, s);
}

}  // namespace capattn
