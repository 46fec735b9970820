// Persistent bf16 forward with the fixed reference, on the 5th-generation
// tensor cores.
//
// What it computes: triton_kernels.py make_triton_forward_kernel (scores, cap,
// masks, softmax with its log-sum-exp) with the cap forms of
// mosaic_backward.py _apply_cap_mosaic and an exp2-domain softmax, for the
// configurations where every row can use the fixed reference of the capped
// logits (a cap, no temperature tensor, m and l not requested, logit window
// <= kSpanMax), with any of the masks: each step is one pass over the scores,
// with no row maximum.  The key tiles of an item are the pre-pass's visit set
// of its query tile; each row's live keys are its pre-pass span (in closed form
// when the mask is causal or none).
//
// One CTA per SM takes work items (batch, head, 128-row query tile) from a
// counter, heaviest (latest) query tiles first; an item without a live key
// tile only writes its zero rows.  The steps of one item run as in the
// two-buffer forward (attn_fwd2_tc.cu): four threads per row, 32 key columns
// each, two TMEM score buffers so S of step j + 2 is computed while the
// softmax works on step j + 1.  Across items, Q and O are double-buffered (two
// Q tiles in shared memory, two O accumulators in TMEM), so the next item's Q
// is loaded ahead and its first scores are computed while the softmax warps
// finish the current item; they take the row's l at once and drain the item's
// O (out of TMEM, straight to global memory) after handing over the next
// item's first P, by which time the item's last P V has completed.
// Warp roles (20 warps):
//   warp 19      fetches the items (a two-slot ring in shared memory, each slot
//                with the item's key-tile count and the first word of its
//                visit bitmap, so that no reader waits on that load) and
//                loads each item's Q into buffer x, running up to two items
//                ahead; warps 0 and 18 follow the items and load the K and V
//                tiles into two-stage rings;
//   warp 1       TMEM allocator and MMA issuer: per item S_0 S_1 | PV_0 S_2 |
//                PV_1 S_3 | ..., O of item k in accumulator x (k's use of the
//                buffers: items without steps take none);
//   warps 2..17  softmax and epilogue, as in the two-buffer forward.
// TMEM (512 columns): S buffers [0,128) and [128,256), O accumulators
// [256, 256 + HD) and [384, 384 + HD).
// No role waits on a CTA-wide or warpgroup barrier inside its loop.
#include "fwd_common.cuh"
#include "row_span.h"
#include "tma_maps.h"

namespace capattn {

namespace {

using namespace fwdtc;

constexpr int KST = 2;  // K stages (two Q tiles and the l exchange leave no room for a third)
constexpr int VST = 2;  // V stages
// two Q tiles, KST K tiles, VST V tiles, the l exchange [2][4][128] floats
template <int HD>
constexpr int smem_bytes() { return (2 + KST + VST) * tile_bytes<HD>() + 4096 + 1024; }
constexpr int NTHREADS = 640;

template <int HD>
__device__ __forceinline__ void issue_pv4(uint32_t d, uint32_t pt, uint64_t dV, uint32_t acc0) {
  constexpr uint32_t idesc = idesc_bf16(BM, HD, 0, 1);
#pragma unroll
  for (int ks = 0; ks < BN / 16; ++ks)
    mma_ts(d, pt + 32 * (ks >> 1) + 8 * (ks & 1), desc_add(dV, ks * 2048), idesc, (acc0 || ks > 0) ? 1u : 0u);
}

struct Item {
  int b, h, qt;
};

__device__ __forceinline__ Item decode_item(const Params& p, int it) {
  const int planes = p.B * p.Hq;
  Item r;
  r.qt = p.nq - 1 - it / planes;
  const int hb = it % planes;
  r.h = hb % p.Hq;
  r.b = hb / p.Hq;
  return r;
}

// SPANS: the rows' live keys come from the pre-pass (a window, segment ids or
// ranker bounds); otherwise they are computed in closed form.
template <int METHOD, int HD, bool SPANS>
__global__ void __launch_bounds__(NTHREADS, 1)
fwd3_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const Params p) {
  constexpr int TILE = tile_bytes<HD>();
  constexpr int NSLAB = HD / 64;
  constexpr int OQ = HD / 4;  // O columns per thread (a quarter of the row)
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * 2 + 2 * KST + 2 * VST + 2 * 2 + 2 * 2 + 2 * 2 + 2];
  // item slots: (item, key tiles it visits, first word of its visit bitmap);
  // the publisher reads the bitmap, so that no reader waits on that load
  __shared__ int4 items[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nitems = p.B * p.Hq * p.nq;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;                         // buffer x at + x * TILE
  const uint32_t sK = base + 2 * TILE;              // stage s at + s * TILE
  const uint32_t sV = base + (2 + KST) * TILE;      // stage s at + s * TILE
  // the l exchange: [2][4][BM] floats (item parity, quarter, row)
  float* xch = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)) + (2 + KST + VST) * TILE);

  const uint32_t bar_qfull = smem_u32(&bars[0]);             // + x*8
  const uint32_t bar_qempty = bar_qfull + 16;                // + x*8: the item's last S complete
  const uint32_t bar_kfull = bar_qempty + 16;                // + s*8
  const uint32_t bar_kempty = bar_kfull + 8 * KST;           // + s*8
  const uint32_t bar_vfull = bar_kempty + 8 * KST;           // + s*8
  const uint32_t bar_vempty = bar_vfull + 8 * VST;           // + s*8
  const uint32_t bar_sfull = bar_vempty + 8 * VST;           // + x*8: S in buffer x complete
  const uint32_t bar_pfull = bar_sfull + 16;                 // + x*8: P in buffer x written (16 warps)
  const uint32_t bar_ofull = bar_pfull + 16;                 // + x*8: the item's last PV complete
  const uint32_t bar_oempty = bar_ofull + 16;                // + x*8: O read by the 16 softmax warps
  const uint32_t bar_ifull = bar_oempty + 16;                // + x*8: item slot x written
  const uint32_t bar_iempty = bar_ifull + 16;                // + x*8: item slot x read (19 readers)
  const uint32_t bar_xch = bar_iempty + 16;                  // the four quarters of the rows wrote l
  const uint32_t bar_final = bar_xch + 8;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar_qfull + 8 * x, 1);
      mbar_init(bar_qempty + 8 * x, 1);
      mbar_init(bar_sfull + 8 * x, 1);
      mbar_init(bar_pfull + 8 * x, 16);
      mbar_init(bar_ofull + 8 * x, 1);
      mbar_init(bar_oempty + 8 * x, 16);
      mbar_init(bar_ifull + 8 * x, 1);
      mbar_init(bar_iempty + 8 * x, 19);
    }
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_vempty + 8 * s, 1);
    }
    mbar_init(bar_xch, 16);
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

  if (warp == 0 || warp >= 18) {
    // ------------------------------------------------------------ TMA producers
    // warp 19 fetches the items and loads their Q tiles (running up to two
    // items ahead); warps 0 and 18 follow the items and load the K and V tiles.
    // Each runs its loop warp-wide; one elected lane issues the copies.
    const bool leader = elect_one_sync();
    const int role = warp == 19 ? 2 : (warp == 0 ? 0 : 1);
    if (leader) tma_prefetch_desc(role == 2 ? &mq : (role == 0 ? &mk : &mv));
    __syncwarp();
    int j = 0;                 // steps loaded so far (ring position)
    int qu0 = 0, qu1 = 0;      // items loaded into each Q buffer so far
    for (int k = 0;; ++k) {
      int4 slot;
      if (role == 2) {
        int it = 0;
        if (lane == 0) it = (int)atomicAdd(p.fwd_work, 1u);
        it = __shfl_sync(0xFFFFFFFFu, it, 0);
        slot = make_int4(-1, 0, 0, 0);
        if (it < nitems) {
          const Item w = decode_item(p, it);
          const uint32_t* map = p.qmap + ((size_t)w.b * p.nq + w.qt) * p.wk;
          slot = make_int4(it, count_tiles(map, p.wk), (int)map[0], 0);
        }
        if (k >= 2 && !mbar_wait_warp(bar_iempty + 8 * (k & 1), ((k >> 1) - 1) & 1, p.status, &abort_flag))
          break;
        if (lane == 0) {
          items[k & 1] = slot;
          mbar_arrive(bar_ifull + 8 * (k & 1));
        }
        __syncwarp();
      } else {
        if (!mbar_wait_warp(bar_ifull + 8 * (k & 1), (k >> 1) & 1, p.status, &abort_flag)) break;
        slot = items[k & 1];  // (the wait above is a compiler memory barrier)
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_iempty + 8 * (k & 1));
      }
      const int it = slot.x;
      if (it < 0) break;
      const Item w = decode_item(p, it);
      const uint32_t* map = p.qmap + ((size_t)w.b * p.nq + w.qt) * p.wk;
      if (slot.y == 0) continue;
      if (role == 2) {
        const int x = k & 1;
        const int uq = x ? qu1++ : qu0++;
        if (uq > 0 && !mbar_wait_warp(bar_qempty + 8 * x, (uq - 1) & 1, p.status, &abort_flag)) break;
        if (leader) {
          mbar_expect_tx(bar_qfull + 8 * x, TILE);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sQ + x * TILE + sl * SLAB, &mq, bar_qfull + 8 * x, 64 * sl, w.h, w.qt * BM, w.b);
        }
        __syncwarp();
        continue;
      }
      const int g = w.h / p.G;
      bool ok = true;
      TileIter ti(map, p.wk, (uint32_t)slot.z);
      int t;
      while (ti.next(t)) {
        const int nst = role == 0 ? KST : VST;
        const int s = j % nst, u = j / nst;
        const uint32_t empty = (role == 0 ? bar_kempty : bar_vempty) + 8 * s;
        const uint32_t full = (role == 0 ? bar_kfull : bar_vfull) + 8 * s;
        if (u > 0 && !mbar_wait_warp(empty, (u - 1) & 1, p.status, &abort_flag)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_expect_tx(full, TILE);
          const uint32_t dst = (role == 0 ? sK : sV) + s * TILE;
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(dst + sl * SLAB, role == 0 ? &mk : &mv, full, 64 * sl, g, t * BN, w.b);
        }
        __syncwarp();
        ++j;
      }
      if (!ok) break;
    }
    // (on an early exit the copies in flight land before the CTA ends)
    if (leader) {
      if (role == 2) {
        for (int x = 0; x < 2; ++x) {
          const int uq = x ? qu1 : qu0;
          if (uq > 0) drain_wait(bar_qfull + 8 * x, (uq - 1) & 1);
        }
      } else {
        const int nst = role == 0 ? KST : VST;
        const uint32_t full = role == 0 ? bar_kfull : bar_vfull;
        for (int jj = (j > nst ? j - nst : 0); jj < j; ++jj)
          drain_wait(full + 8 * (jj % nst), (jj / nst) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one_sync();
    const uint64_t dQ = smem_desc(sQ, 16, 1024);
    const uint64_t dK = smem_desc(sK, 16, 1024);
    const uint64_t dVmn = smem_desc(sV, SLAB, 1024);
    int g = 0;                 // steps issued so far (ring and score-buffer position)
    int qu0 = 0, qu1 = 0;      // items in each Q buffer so far
    int ou0 = 0, ou1 = 0;      // items in each O accumulator so far
    for (int k = 0;; ++k) {
      if (!mbar_wait_warp(bar_ifull + 8 * (k & 1), (k >> 1) & 1, p.status, &abort_flag)) break;
      const int4 slot = items[k & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_iempty + 8 * (k & 1));
      if (slot.x < 0) break;
      const int n = slot.y;
      if (n == 0) continue;
      const int x = k & 1;
      const int uq = x ? qu1++ : qu0++;
      const int uo = x ? ou1++ : ou0++;
      const uint64_t dQx = desc_add(dQ, (uint32_t)(x * TILE));
      // S of the item's step i (global step g0 + i) into score buffer (g0 + i) & 1
      const int g0 = g;
      auto issue_scores = [&](int i) -> bool {
        const int gg = g0 + i, s = gg % KST;
        if (!mbar_wait_warp(bar_kfull + 8 * s, (gg / KST) & 1, p.status, &abort_flag)) return false;
        tc_fence_after();
        if (leader) {
          issue_s<HD>(tmem + 128u * (uint32_t)(gg & 1), dQx, desc_add(dK, (uint32_t)(s * TILE)));
          mma_commit(bar_sfull + 8 * (gg & 1));
          mma_commit(bar_kempty + 8 * s);
        }
        __syncwarp();
        return true;
      };
      bool ok = mbar_wait_warp(bar_qfull + 8 * x, uq & 1, p.status, &abort_flag) && issue_scores(0);
      if (ok && n > 1) ok = issue_scores(1);
      // the item's O accumulator: read out by the epilogue of the item before
      // the previous one in it
      if (ok && uo > 0) ok = mbar_wait_warp(bar_oempty + 8 * x, (uo - 1) & 1, p.status, &abort_flag);
      for (int i = 0; ok && i < n; ++i) {
        const int gg = g0 + i, xb = gg & 1, s = gg % VST;
        if (!mbar_wait_warp(bar_pfull + 8 * xb, (gg >> 1) & 1, p.status, &abort_flag) ||
            !mbar_wait_warp(bar_vfull + 8 * s, (gg / VST) & 1, p.status, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
          issue_pv4<HD>(tmem + 256u + 128u * (uint32_t)x, tmem + 128u * (uint32_t)xb,
                        desc_add(dVmn, (uint32_t)(s * TILE)), i > 0 ? 1u : 0u);
          mma_commit(bar_vempty + 8 * s);
        }
        __syncwarp();
        // S of step i + 2 overwrites P_i's buffer after PV_i (in-order MMAs)
        if (i + 2 < n && !issue_scores(i + 2)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      g = g0 + n;
      if (leader) {
        mma_commit(bar_ofull + 8 * x);   // the item's O is complete
        mma_commit(bar_qempty + 8 * x);  // and its Q no longer read
      }
      __syncwarp();
    }
    // The MMA thread does not wait for its own commit here: warp 1 re-checks
    // it before freeing TMEM.
    if (leader) mma_commit(bar_final);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax and epilogue
    const int sw = warp - 2;                     // 0..15
    const int cq = sw >> 2;                      // key columns [32 cq, 32 cq + 32) of each step
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_quarter = tmem + lane_off + 32u * (uint32_t)cq;   // + 128 x: score buffer x
    const Xf xf = make_xf<METHOD>(p.cap, p.sm_scale);
    float rmul, radd;
    row_consts<METHOD>(p.cap, p.sm_scale, 1.f, &rmul, &radd);
    float x_hi = 0.f, span = 0.f;
    if constexpr (METHOD == CAPATTN_CAP_TANH || METHOD == CAPATTN_CAP_SOFT_SIGN) {
      x_hi = fabsf(rmul);
      span = 2.f * fabsf(rmul);
    } else {
      x_hi = fmaxf(radd, rmul + radd);
      span = fabsf(rmul);
    }
    const float m_use = fixed_reference(x_hi, span);
    const float addm = radd - m_use;
    TanhFold tf{};
    if constexpr (METHOD == CAPATTN_CAP_TANH) tf = tanh_fold(xf.in, rmul);
    __nv_bfloat16* const out = static_cast<__nv_bfloat16*>(p.o);
    int g = 0;                 // steps consumed so far
    int ou0 = 0, ou1 = 0;      // items read from each O accumulator so far
    int ex = 0;                // l exchanges so far
    // The O of an item leaves after the next item's first step (its last P V
    // completes meanwhile): pend = accumulator | (use parity) << 1, or -1.
    int pend = -1, pend_b = 0, pend_h = 0, pend_i = 0;
    float pend_l = 0.f;
    // writes row pend_i's OQ columns of the pending item's O, 16 at a time,
    // straight to global memory (O [B, L, Hq, HD] bf16; rows past L are not
    // written), frees the accumulator and writes the row's LSE
    auto drain = [&]() -> bool {
      const int xx = pend & 1;
      if (!mbar_wait_warp(bar_ofull + 8 * xx, (pend >> 1) & 1, p.status, &abort_flag)) return false;
      tc_fence_after();
      const bool pvalid = pend_i < p.L;
      const bool live = pend_l > 0.f;
      const float inv = live ? 1.f / pend_l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(out + (((size_t)pend_b * p.L + (pvalid ? pend_i : 0)) * p.Hq + pend_h) * HD +
                                            OQ * cq);
      const uint32_t ob = tmem + lane_off + 256u + 128u * (uint32_t)xx + (uint32_t)(OQ * cq);
#pragma unroll
      for (int hh = 0; hh < OQ / 16; ++hh) {
        uint32_t o[16], pk[8];
        tmem_ld16(ob + 16u * (uint32_t)hh, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e)
          pk[e] = pack_bf16x2(live ? __uint_as_float(o[2 * e]) * inv : 0.f,
                              live ? __uint_as_float(o[2 * e + 1]) * inv : 0.f);
        if (pvalid) {
          dst[2 * hh] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[2 * hh + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      // every read of the accumulator is done: it is free again
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_oempty + 8 * xx);
      if (pvalid && cq == 0)
        p.lse[((size_t)pend_b * p.Hq + pend_h) * p.L + pend_i] = live ? (m_use + log2f(pend_l)) * kLn2 : -INFINITY;
      return true;
    };
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!mbar_wait_warp(bar_ifull + 8 * (k & 1), (k >> 1) & 1, p.status, &abort_flag)) break;
      const int4 slot = items[k & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_iempty + 8 * (k & 1));
      if (slot.x < 0) break;
      const Item w = decode_item(p, slot.x);
      const uint32_t* map = p.qmap + ((size_t)w.b * p.nq + w.qt) * p.wk;
      const int n = slot.y;
      const int i = w.qt * BM + r;
      const bool valid = i < p.L;
      // the row's live keys: the pre-pass's span, or in closed form without a
      // window, segment ids or ranker bounds ([0, i + 1) causal, [0, Lk) otherwise)
      int4 ri = make_int4(0, 0, -1, 0);
      if (valid) {
        if constexpr (SPANS)
          ri = p.rowinfo[(size_t)w.b * p.L + i];
        else
          ri = make_int4(0, p.causal ? imin32(i + 1, p.Lk) : p.Lk, -1, 0);
      }
      float lsum = 0.f;
      TileIter ti(map, p.wk, (uint32_t)slot.z);
      int t;
      // one step: the quarter-row's P over its score buffer, handed to the issuer
      auto step = [&](int st, int t) -> bool {
        const int gg = g + st;
        const int k0 = t * BN;
        const int c0 = k0 + 32 * cq;
        const uint32_t sb = s_quarter + 128u * (uint32_t)(gg & 1);
        if (!mbar_wait_warp(bar_sfull + 8 * (gg & 1), (gg >> 1) & 1, p.status, &abort_flag)) return false;
        tc_fence_after();
        const bool full = (ri.x <= k0) && (ri.y >= k0 + BN);
        const bool warp_partial = __any_sync(0xFFFFFFFFu, !full);
        uint32_t v[32], pk[16];
        tmem_ld32(sb, v);
        tmem_wait_ld();
        if (warp_partial && quarter_dead(ri, c0)) {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = 0u;
        } else if (METHOD == CAPATTN_CAP_ALSC && quarter_alsc_poly(v, p.cap.alsc_xmax)) {
          // the sigmoid on the FMA pipe: mul (f - sigma(alpha beta)) - m
          lsum += full ? p_chunk_alsc<false, 16>(v, pk, p.cap, rmul, -m_use, 0xFFFFFFFFu)
                       : p_chunk_alsc<true, 16>(v, pk, p.cap, rmul, -m_use, live_bits32(ri, c0));
        } else {
          const bool poly = quarter_poly<METHOD>(v, tf, xf);
          lsum += p_dispatch32<METHOD>(full, poly, v, pk, xf, tf, rmul, addm, c0, ri, true);
        }
        __syncwarp();
        tmem_st16(sb, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pfull + 8 * (gg & 1));
        return true;
      };
      int st = 0;
      if (n > 0 && ti.next(t)) {
        ok = step(0, t);
        st = 1;
      }
      // the previous item's O, once this item's first P is handed over (its
      // last P V has completed meanwhile)
      if (ok && n > 0 && pend >= 0) {
        ok = drain();
        pend = -1;
      }
      for (; ok && st < n && ti.next(t); ++st) ok = step(st, t);
      if (!ok) break;
      g += n;
      // ---- the item's l, and its O / LSE (now or after the next item's first step)
      const int x = k & 1;
      if (n > 0) {
        // l of the whole row: the four quarters add their parts
        float* xs = xch + (ex & 1) * 4 * BM;
        xs[cq * BM + r] = lsum;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_xch);
        if (!mbar_wait_warp(bar_xch, ex & 1, p.status, &abort_flag)) break;
        float l_row = 0.f;
#pragma unroll
        for (int o4 = 0; o4 < 4; ++o4) l_row += xs[o4 * BM + r];
        ++ex;
        const int uo = x ? ou1++ : ou0++;
        pend = x | ((uo & 1) << 1);
        pend_b = w.b;
        pend_h = w.h;
        pend_i = i;
        pend_l = l_row;
      } else {
        // no live key tile: the previous item's O first, then zero rows
        if (pend >= 0) {
          if (!drain()) break;
          pend = -1;
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + (((size_t)w.b * p.L + i) * p.Hq + w.h) * HD + OQ * cq);
#pragma unroll
          for (int e = 0; e < OQ / 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
          if (cq == 0) p.lse[((size_t)w.b * p.Hq + w.h) * p.L + i] = -INFINITY;
        }
      }
    }
    if (pend >= 0 && __all_sync(0xFFFFFFFFu, abort_flag == 0)) drain();
  }
  __syncwarp();  // every warp reaches the CTA barrier converged
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // Every MMA has completed before TMEM is released (bounded non-suspending poll).
    if (lane == 0) mbar_poll(bar_final, 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int METHOD, int HD>
cudaError_t launch_fwd_hd(const Params& p, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  cudaError_t e = make_bhld_map(&mq, p.q, p.B, p.L, p.Hq, HD, BM);
  if (e == cudaSuccess) e = make_bhld_map(&mk, p.k, p.B, p.Lk, p.Hkv, HD, BN);
  if (e == cudaSuccess) e = make_bhld_map(&mv, p.v, p.B, p.Lk, p.Hkv, HD, BN);
  if (e != cudaSuccess) return e;
  const bool spans = p.window_len > 0 || p.seg != nullptr || p.bounds != nullptr;
  auto kern = spans ? fwd3_tc_kernel<METHOD, HD, true> : fwd3_tc_kernel<METHOD, HD, false>;
  constexpr int SMEM_BYTES = smem_bytes<HD>();
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long nitems = (long long)p.B * p.Hq * p.nq;
  const unsigned grid = (unsigned)(nitems < sms ? nitems : sms);
  prof_begin(CAPATTN_KERNEL_FWD, s);
  prof_count(CAPATTN_KERNEL_FWD, 1);
  e = launch_pdl(kern, dim3(grid), dim3(NTHREADS), SMEM_BYTES, s, mq, mk, mv, p);
  if (e != cudaSuccess) return e;
  prof_end(CAPATTN_KERNEL_FWD, s);
  return cudaGetLastError();
}

template <int METHOD>
struct Fwd3TcLaunch {
  static cudaError_t run(const Params& p, cudaStream_t s) {
    if constexpr (METHOD == CAPATTN_CAP_NONE) {
      return cudaErrorInvalidValue;  // never chosen: the fixed reference needs a cap
    } else {
      return p.D == 64 ? launch_fwd_hd<METHOD, 64>(p, s) : launch_fwd_hd<METHOD, 128>(p, s);
    }
  }
};

}  // namespace

cudaError_t launch_fwd3_bf16(const Params& p, cudaStream_t s) {
  return dispatch_cap<Fwd3TcLaunch>(p.cap.method, p, s);
}

}  // namespace capattn
