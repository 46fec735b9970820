// dQ of the stored-dX backward on the 5th-generation tensor cores.
//
// mosaic_backward.py make_mosaic_backward_dq_kernel accumulates, per query
// tile, dQ = sum over the visited key tiles t of dX_t K_t, recomputing the
// scores, P and dX of every tile.  Here the dK/dV kernel, which computes the
// same dX for its own dK = dX^T Q, has already written each tile's dX^T (bf16,
// 128 key rows of 128 query values) to a pool in the workspace, so dQ is a
// plain GEMM over those tiles:
//   dQ[128 queries x HD] = sum_t dX_t [128 x 128 keys] K_t [128 keys x HD]
// with both operands read from shared memory MN-major: the dX^T tile is dX
// with the query index contiguous, stored by the dK/dV kernel in the 32-byte
// swizzled operand layout (eight blocks of 16 queries x 128 key rows of 32
// bytes) and copied in with one contiguous bulk copy; the K tile is K with the
// head dim contiguous, loaded by TMA in the 128-byte swizzled layout.
//
// One CTA per (batch, query head, 128-query tile), heaviest tiles first.
// Warps: 0 TMA producer (a ring of NST stages, each a dX^T tile and a K tile),
// 1 TMEM allocator and MMA issuer, 2..5 the epilogue (TMEM -> bf16 -> shared
// memory -> TMA store), one TMEM lane quarter each.
#include "capattn_internal.h"
#include "row_span.h"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace capattn {

namespace {

constexpr int BT = 128;
constexpr int SLAB = 128 * 64 * 2;  // a [128][64] bf16 slab, 128-byte swizzled
constexpr int XTILE = 2 * SLAB;     // a dX^T tile: 128 key rows x 128 queries
constexpr int NST = 3;
constexpr int NTHREADS = 192;
template <int HD>
constexpr int ktile_bytes() { return (HD / 64) * SLAB; }
template <int HD>
constexpr int stage_bytes() { return XTILE + ktile_bytes<HD>(); }
template <int HD>
constexpr int smem_bytes() { return NST * stage_bytes<HD>() + 1024; }

template <int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
dq_gemm_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mdq,
               const Params p) {
  constexpr int STAGE = stage_bytes<HD>();
  constexpr int NSLAB = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * NST + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int hb = blockIdx.x;
  const int h = hb % p.Hq, b = hb / p.Hq;
  const int qt = p.nq - 1 - (int)blockIdx.y;
  const int g = h / p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;  // stage s at base + s * STAGE
  const uint32_t bar_full = smem_u32(&bars[0]);       // + s*8: stage s landed
  const uint32_t bar_empty = smem_u32(&bars[NST]);    // + s*8: stage s read by its MMAs
  const uint32_t bar_final = smem_u32(&bars[2 * NST]);

  const uint32_t* map = p.qmap + ((size_t)b * p.nq + qt) * p.wk;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), HD);
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
  // slot of key tile t in this query tile's band: slot0 + t - kt_lo
  const int kt_lo = p.dx_c >= 0 ? imax32(0, qt - p.dx_c) : 0;
  const size_t slot0 = ((size_t)(b * p.Hq + h) * p.nq + qt) * p.dx_wmax;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (n > 0) {
      const bool leader = elect_one_sync();
      if (leader) {
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mdq);
      }
      __syncwarp();
      TileIter it(map, p.wk);
      int t, j = 0;
      while (!__any_sync(0xFFFFFFFFu, abort_flag != 0) && it.next(t)) {
        const int s = j % NST, u = j / NST;
        if (u > 0 && !mbar_wait_warp(bar_empty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) break;
        const int d = t - kt_lo;
        if (d < 0 || d >= p.dx_wmax) {
          // no slot (never expected): report it and let every role give up
          if (lane == 0) {
            atomicOr(p.status, kStatusBandBit);
            *static_cast<volatile int*>(&abort_flag) = 1;
          }
          break;
        }
        if (leader) {
          const uint32_t sx = base + s * STAGE, sk = sx + XTILE;
          const char* tile = static_cast<const char*>(p.dx_pool) + (slot0 + (size_t)d) * kDxTileBytes;
          mbar_expect_tx(bar_full + 8 * s, STAGE);
          bulk_load(sx, tile, XTILE, bar_full + 8 * s);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sk + sl * SLAB, &mk, bar_full + 8 * s, 64 * sl, g, t * BT, b);
        }
        __syncwarp();
        ++j;
      }
      if (leader) {
        for (int jj = (j > NST ? j - NST : 0); jj < j; ++jj)
          drain_wait(bar_full + 8 * (jj % NST), (jj / NST) & 1);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      const bool leader = elect_one_sync();
      // A = dX (M = queries, K = keys) from the dX^T tile: MN-major, 32-byte
      // swizzle, 16-query blocks 4 KB apart, 8-row groups 256 bytes apart, 16
      // keys = 512 bytes per MMA.  B = K (N = head dim, K = keys) from the key
      // tile: MN-major, 128-byte swizzle, 64-wide slabs 16 KB apart, 8-row
      // groups 1024 bytes apart, 16 keys = 2048 bytes per MMA.
      constexpr uint32_t idesc = idesc_bf16(BT, HD, 1, 1);
      const uint64_t dA = smem_desc(base, 4096, 256, kSwizzle32B);
      const uint64_t dB = smem_desc(base + XTILE, SLAB, 1024);
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const int s = j % NST;
        if (!mbar_wait_warp(bar_full + 8 * s, (j / NST) & 1, p.status, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
          const uint32_t so = (uint32_t)(s * STAGE);
#pragma unroll
          for (int ks = 0; ks < BT / 16; ++ks)
            mma_ss(tmem, desc_add(dA, so + ks * 512), desc_add(dB, so + ks * 2048), idesc,
                   (j > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar_empty + 8 * s);
        }
        __syncwarp();
      }
      (void)ok;
      // No wait for this commit here: the epilogue warps wait for it, and
      // warp 1 re-checks it before freeing TMEM.
      if (leader) mma_commit(bar_final);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row within the tile (TMEM lane)
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    bool have = false;
    if (n > 0) {
      have = mbar_wait_warp(bar_final, 0, p.status, &abort_flag);
      tc_fence_after();
    }
    // dQ leaves through stage 0's dX^T slabs (every MMA has completed): rows in
    // the swizzled layout, then one TMA store per 64-column slab (rows past L
    // are clipped by the tensor map).  Without a visited tile dQ is zero.
#pragma unroll 1
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(lane_base + 32 * c, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
      const uint32_t slab = base + (uint32_t)(c >> 1) * SLAB;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        st_swz_chunk(slab, r, 4 * (c & 1) + e, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
    }
    fence_async_smem();
    named_bar_sync(1, 128);  // every row is in shared memory
    if (warp == 2 && lane == 0) {
      for (int sl = 0; sl < NSLAB; ++sl) tma_store_4d(&mdq, base + sl * SLAB, 64 * sl, h, qt * BT, b);
      bulk_commit();
      bulk_wait_read0();
    }
  }
  __syncwarp();  // warps 0 and 1 reach the CTA barrier converged
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // Every MMA has completed before TMEM is released (normally already
    // observed by the epilogue warps; bounded non-suspending poll).
    if (lane == 0 && n > 0) mbar_poll(bar_final, 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, HD);
  }
}

template <int HD>
cudaError_t launch_hd(const Params& p, cudaStream_t s) {
  CUtensorMap mk, mdq;
  cudaError_t e = make_bhld_map(&mk, p.k, p.B, p.Lk, p.Hkv, HD, BT);
  if (e == cudaSuccess) e = make_bhld_map(&mdq, p.dq, p.B, p.L, p.Hq, HD, BT);
  if (e != cudaSuccess) return e;
  constexpr int SMEM = smem_bytes<HD>();
  auto kern = dq_gemm_kernel<HD>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  prof_begin(CAPATTN_KERNEL_DQ, s);
  prof_count(CAPATTN_KERNEL_DQ, 1);
  e = launch_pdl(kern, dim3(p.Hq * p.B, p.nq), dim3(NTHREADS), SMEM, s, mk, mdq, p);
  if (e != cudaSuccess) return e;
  prof_end(CAPATTN_KERNEL_DQ, s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq_gemm(const Params& p, cudaStream_t s) {
  return p.D == 64 ? launch_hd<64>(p, s) : launch_hd<128>(p, s);
}

}  // namespace capattn
