// bf16 forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: triton_kernels.py make_triton_forward_kernel (scores, cap,
// temperature, masks, online softmax with the l / m residuals), with the cap
// forms of mosaic_backward.py _apply_cap_mosaic, the ranker mask of
// ranker_mask_mosaic_kv_q (transposed) and an exp2-domain softmax as in the
// Mosaic kernels.
//
// One CTA owns 128 query rows of one (batch, head) and walks the KV tiles of
// its visit map.  Warp roles:
//   warp 0      TMA producer: Q once, then K_j / V_j into a ring of stages;
//   warp 1      TMEM allocator and MMA issuer (one thread):
//                 S_j = Q K_j^T      (SS MMA, M=N=128, into a double-buffered
//                                     128-column TMEM region, so S_{j+1} runs
//                                     on the tensor pipe while the softmax
//                                     works on S_j)
//                 O  += P_j V_j      (TS MMA: P_j read from TMEM as bf16)
//   warps 2..5  softmax: one thread per query row (TMEM lane).  Loads S_j,
//               applies sm_scale, cap, temperature and the row's live span,
//               keeps a running max in the log2 domain, writes P_j = 2^(x - m)
//               as packed bf16 back over the first 64 columns of S_j, and
//               rescales O in TMEM when the max grows by more than 2^8
//               (otherwise the stale max is kept; P stays <= 256).
// TMEM: S0 [0,128), S1 [128,256), O [256,384) -> 512 columns allocated.
#include <math.h>

#include "cap_math.cuh"
#include "capattn_internal.h"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int HD = 128;
constexpr int NSTAGE = 2;
constexpr int SLAB = 128 * 64 * 2;          // one [128][64] bf16 box
constexpr int TILE = 2 * SLAB;               // 128 x 128 bf16
constexpr int SMEM_DATA = TILE + NSTAGE * 2 * TILE;
constexpr int SMEM_BYTES = SMEM_DATA + 1024;  // + alignment slack
constexpr int NTHREADS = 192;
constexpr float kRescaleThreshold = 8.0f;     // log2 units

template <int METHOD>
__global__ void __launch_bounds__(NTHREADS, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[16];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int hb = blockIdx.x;
  const int h = hb % p.Hq, b = hb / p.Hq;
  const int qt = p.nq - 1 - (int)blockIdx.y;  // heaviest (latest) query tiles first
  const int g = h / p.G;
  const int q0 = qt * BM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sKV = base + TILE;  // stage s: K at sKV + s*2*TILE, V at + TILE

  const uint32_t bar_q = smem_u32(&bars[0]);
  const uint32_t bar_kfull = smem_u32(&bars[1]);    // + s*8
  const uint32_t bar_vfull = smem_u32(&bars[3]);    // + s*8
  const uint32_t bar_empty = smem_u32(&bars[5]);    // + s*8
  const uint32_t bar_sfull = smem_u32(&bars[7]);    // + buf*8
  const uint32_t bar_pfull = smem_u32(&bars[9]);    // + buf*8
  const uint32_t bar_odone = smem_u32(&bars[11]);
  const uint32_t bar_final = smem_u32(&bars[12]);

  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_sfull + 8 * s, 1);
      mbar_init(bar_pfull + 8 * s, 4);
    }
    mbar_init(bar_odone, 1);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      mbar_expect_tx(bar_q, TILE);
      tma_load_4d(sQ, &mq, bar_q, 0, h, q0, b);
      tma_load_4d(sQ + SLAB, &mq, bar_q, 64, h, q0, b);
      TileIter it(map, p.wk);
      int t, j = 0;
      while (it.next(t)) {
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (u > 0 && !mbar_wait(bar_empty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) break;
        const uint32_t sK = sKV + s * 2 * TILE, sV = sK + TILE;
        mbar_expect_tx(bar_kfull + 8 * s, TILE);
        tma_load_4d(sK, &mk, bar_kfull + 8 * s, 0, g, t * BN, b);
        tma_load_4d(sK + SLAB, &mk, bar_kfull + 8 * s, 64, g, t * BN, b);
        mbar_expect_tx(bar_vfull + 8 * s, TILE);
        tma_load_4d(sV, &mv, bar_vfull + 8 * s, 0, g, t * BN, b);
        tma_load_4d(sV + SLAB, &mv, bar_vfull + 8 * s, 64, g, t * BN, b);
        ++j;
      }
      // Let every issued copy land before the CTA can exit.
      drain_wait(bar_q, 0);
      for (int jj = (j > NSTAGE ? j - NSTAGE : 0); jj < j; ++jj) {
        drain_wait(bar_kfull + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
        drain_wait(bar_vfull + 8 * (jj % NSTAGE), (jj / NSTAGE) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16(BM, HD, 0, 1);
      bool ok = mbar_wait(bar_q, 0, p.status, &abort_flag);
      auto issue_s = [&](int j) -> bool {
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (!mbar_wait(bar_kfull + 8 * s, u & 1, p.status, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t sK = sKV + s * 2 * TILE;
        const uint32_t d = tmem + (uint32_t)(j & 1) * 128u;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * SLAB + (ks & 3) * 32;
          mma_ss(d, smem_desc(sQ + off, 16, 1024), smem_desc(sK + off, 16, 1024), idesc_s, ks > 0);
        }
        mma_commit(bar_sfull + 8 * (j & 1));
        return true;
      };
      if (ok) {
        tc_fence_after();
        ok = issue_s(0);
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) break;
        if (!mbar_wait(bar_pfull + 8 * (j & 1), (j >> 1) & 1, p.status, &abort_flag)) break;
        const int s = j % NSTAGE, u = j / NSTAGE;
        if (!mbar_wait(bar_vfull + 8 * s, u & 1, p.status, &abort_flag)) break;
        tc_fence_after();
        const uint32_t sV = sKV + s * 2 * TILE + TILE;
        const uint32_t pt = tmem + (uint32_t)(j & 1) * 128u;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          mma_ts(tmem + 256u, pt + ks * 8, smem_desc(sV + ks * 2048, SLAB, 1024), idesc_o,
                 (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(bar_odone);
        mma_commit(bar_empty + 8 * s);
      }
      // All issued MMAs complete before TMEM is released.
      mma_commit(bar_final);
      drain_wait(bar_final, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int i = q0 + r;
    const bool valid = i < p.L;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int4 ri = valid ? p.rowinfo[(size_t)b * p.L + i] : make_int4(0, 0, -1, 0);
    const float tl = ((p.temp && valid) ? p.temp[(size_t)b * p.L + i] : 1.f) * kLog2e;
    const float sc = p.sm_scale;
    float m_use = -INFINITY, m_true = -INFINITY, lsum = 0.f;
    bool aborted = false;
    TileIter it(map, p.wk);
    for (int j = 0; j < n; ++j) {
      int t;
      it.next(t);
      const int k0 = t * BN;
      const uint32_t buf = (uint32_t)(j & 1);
      if (!mbar_wait(bar_sfull + 8 * buf, (j >> 1) & 1, p.status, &abort_flag)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      uint32_t x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld32(lane_base + buf * 128u + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]));
      tmem_wait_ld();
      const bool full = (ri.x <= k0) && (ri.y >= k0 + BN);
      float mx = -INFINITY;
      if (full) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float v = cap_value<METHOD>(__uint_as_float(x[c]) * sc, p.cap) * tl;
          x[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int jj = k0 + c;
          const bool lv = (jj >= ri.x && jj < ri.y) || jj == ri.z;
          const float v = lv ? cap_value<METHOD>(__uint_as_float(x[c]) * sc, p.cap) * tl : -INFINITY;
          x[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      }
      m_true = fmaxf(m_true, mx);
      const float m_new = fmaxf(m_use, mx);
      const bool resc = m_new > m_use + kRescaleThreshold;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_use - m_new);
        m_use = m_new;
      }
      float psum = 0.f;
      const bool any = m_use != -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = any ? ex2_approx(__uint_as_float(x[c * 32 + 2 * e]) - m_use) : 0.f;
          const float p1 = any ? ex2_approx(__uint_as_float(x[c * 32 + 2 * e + 1]) - m_use) : 0.f;
          psum += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(lane_base + buf * 128u + c * 16, pk);
      }
      lsum = lsum * alpha + psum;
      if (j > 0) {
        if (!mbar_wait(bar_odone, (j - 1) & 1, p.status, &abort_flag)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xFFFFFFFFu, resc)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + 256u + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_base + 256u + c * 32, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfull + 8 * buf);
    }
    // ---------------------------------------------------------- epilogue
    bool have_o = false;
    if (n > 0 && !aborted) {
      have_o = mbar_wait(bar_odone, (n - 1) & 1, p.status, &abort_flag);
      tc_fence_after();
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.o) + ((size_t)(b * p.L + i) * p.Hq + h) * HD;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(lane_base + 256u + c * 32, o);
        tmem_wait_ld();
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float a = have_o ? __uint_as_float(o[2 * e]) * inv : 0.f;
        const float bb = have_o ? __uint_as_float(o[2 * e + 1]) * inv : 0.f;
        pk[e] = pack_bf16x2(lsum > 0.f ? a : 0.f, lsum > 0.f ? bb : 0.f);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(og + c * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
    }
    if (valid) {
      const size_t rr = ((size_t)b * p.Hq + h) * p.L + i;
      const bool live = lsum > 0.f;
      p.lse[rr] = live ? (m_use + log2f(lsum)) * kLn2 : -INFINITY;
      if (p.m) p.m[rr] = live ? m_true * kLn2 : -INFINITY;
      if (p.l) p.l[rr] = live ? lsum * ex2_approx(m_use - m_true) : 0.f;
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
struct FwdTcLaunch {
  static cudaError_t run(const Params& p, cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    cudaError_t e = make_bhld_map(&mq, p.q, p.B, p.L, p.Hq, HD, BM);
    if (e == cudaSuccess) e = make_bhld_map(&mk, p.k, p.B, p.L, p.Hkv, HD, BN);
    if (e == cudaSuccess) e = make_bhld_map(&mv, p.v, p.B, p.L, p.Hkv, HD, BN);
    if (e != cudaSuccess) return e;
    auto kern = fwd_tc_kernel<METHOD>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    prof_begin(CAPATTN_KERNEL_FWD, s);
    prof_count(CAPATTN_KERNEL_FWD, 1);
    kern<<<dim3(p.Hq * p.B, p.nq), NTHREADS, SMEM_BYTES, s>>>(mq, mk, mv, p);
    prof_end(CAPATTN_KERNEL_FWD, s);
    return cudaGetLastError();
  }
};

}  // namespace

cudaError_t launch_fwd_bf16(const Params& p, cudaStream_t s) {
  return dispatch_cap<FwdTcLaunch>(p.cap.method, p, s);
}

}  // namespace capattn
