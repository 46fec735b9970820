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
// Persistent: one CTA per SM takes work items (batch, query head, query tile)
// from a counter in heavy-first order (latest query tiles first).  Warps: 0
// TMA producer (fetches the items, a ring of NST stages each holding a dX^T
// tile and a K tile), 1 TMEM allocator and MMA issuer (two accumulators, so an
// item's MMAs run while the previous item's epilogue drains the other), 2..5
// the epilogue (TMEM -> bf16 -> this warp's shared-memory rows -> TMA store of
// its 32 rows), one TMEM lane quarter each.  Items reach the issuer and the
// epilogue through a two-slot ring in shared memory.  No role waits on a
// CTA-wide or warpgroup barrier inside its loop, so a role that gives up on a
// bounded wait cannot leave another one waiting without a limit.
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
constexpr int OUT_ROWS = 32;        // rows of dQ each epilogue warp stores
template <int HD>
constexpr int ktile_bytes() { return (HD / 64) * SLAB; }
template <int HD>
constexpr int stage_bytes() { return XTILE + ktile_bytes<HD>(); }
// an epilogue warp's output rows: HD / 64 slabs of [32][64] bf16
template <int HD>
constexpr int out_bytes() { return (HD / 64) * OUT_ROWS * 128; }
template <int HD>
constexpr int smem_bytes() { return NST * stage_bytes<HD>() + 4 * out_bytes<HD>() + 1024; }

struct Item {
  int b, h, qt;
};

__device__ __forceinline__ Item decode_item(const Params& p, int it) {
  const int planes = p.B * p.Hq;
  Item r;
  r.qt = p.nq - 1 - it / planes;  // heaviest (latest) query tiles first
  const int hb = it % planes;
  r.h = hb % p.Hq;
  r.b = hb / p.Hq;
  return r;
}

template <int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
dq_gemm_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mdq,
               const Params p) {
  constexpr int STAGE = stage_bytes<HD>();
  constexpr int NSLAB = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * NST + 9];
  __shared__ int items[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nitems = p.B * p.Hq * p.nq;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;  // stage s at base + s * STAGE
  const uint32_t out_base = base + NST * STAGE;                // epilogue warp w at + (w - 2) * out_bytes
  const uint32_t bar_full = smem_u32(&bars[0]);         // + s*8: stage s landed
  const uint32_t bar_empty = smem_u32(&bars[NST]);      // + s*8: stage s read by its MMAs
  const uint32_t bar_ifull = smem_u32(&bars[2 * NST]);  // + x*8: item slot x written
  const uint32_t bar_iempty = bar_ifull + 16;           // + x*8: item slot x read (issuer + 4 epilogue warps)
  const uint32_t bar_afull = bar_ifull + 32;            // + x*8: accumulator x complete
  const uint32_t bar_aempty = bar_ifull + 48;           // + x*8: accumulator x read (4 epilogue warps)
  const uint32_t bar_final = bar_ifull + 64;            // every MMA of the CTA complete

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar_ifull + 8 * x, 1);
      mbar_init(bar_iempty + 8 * x, 5);
      mbar_init(bar_afull + 8 * x, 1);
      mbar_init(bar_aempty + 8 * x, 4);
    }
    mbar_init(bar_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 2 * HD);
    tmem_relinquish();
  }
  // the setup above overlaps the previous kernel's tail; global memory only after it
  pdl_trigger();
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const bool leader = elect_one_sync();
    if (leader) {
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mdq);
    }
    int j = 0;  // steps loaded so far (stage ring position)
    for (int k = 0;; ++k) {
      int it = 0;
      if (lane == 0) it = (int)atomicAdd(p.dq_work, 1u);
      it = __shfl_sync(0xFFFFFFFFu, it, 0);
      if (it >= nitems) it = -1;
      if (k >= 2 && !mbar_wait_warp(bar_iempty + 8 * (k & 1), ((k >> 1) - 1) & 1, p.status, &abort_flag))
        break;
      if (lane == 0) {
        items[k & 1] = it;
        mbar_arrive(bar_ifull + 8 * (k & 1));
      }
      __syncwarp();
      if (it < 0) break;
      const Item w = decode_item(p, it);
      const uint32_t* map = p.qmap + ((size_t)w.b * p.nq + w.qt) * p.wk;
      const int kt_lo = p.dx_c >= 0 ? imax32(0, w.qt - p.dx_c) : 0;
      const size_t slot0 = ((size_t)(w.b * p.Hq + w.h) * p.nq + w.qt) * p.dx_wmax;
      const int g = w.h / p.G;
      TileIter ti(map, p.wk);
      int t;
      bool ok = true;
      while (ti.next(t)) {
        const int s = j % NST, u = j / NST;
        if (u > 0 && !mbar_wait_warp(bar_empty + 8 * s, (u - 1) & 1, p.status, &abort_flag)) {
          ok = false;
          break;
        }
        const int d = t - kt_lo;
        if (d < 0 || d >= p.dx_wmax) {
          // no slot (never expected): report it and let every role give up
          if (lane == 0) {
            atomicOr(p.status, kStatusBandBit);
            *static_cast<volatile int*>(&abort_flag) = 1;
          }
          ok = false;
          break;
        }
        if (leader) {
          const uint32_t sx = base + s * STAGE, sk = sx + XTILE;
          const char* tile = static_cast<const char*>(p.dx_pool) + (slot0 + (size_t)d) * kDxTileBytes;
          mbar_expect_tx(bar_full + 8 * s, STAGE);
          bulk_load(sx, tile, XTILE, bar_full + 8 * s);
          for (int sl = 0; sl < NSLAB; ++sl)
            tma_load_4d(sk + sl * SLAB, &mk, bar_full + 8 * s, 64 * sl, g, t * BT, w.b);
        }
        __syncwarp();
        ++j;
      }
      if (!ok) break;
    }
    if (leader) {
      for (int jj = (j > NST ? j - NST : 0); jj < j; ++jj)
        drain_wait(bar_full + 8 * (jj % NST), (jj / NST) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one_sync();
    // A = dX (M = queries, K = keys) from the dX^T tile: MN-major, 32-byte
    // swizzle, 16-query blocks 4 KB apart, 8-row groups 256 bytes apart, 16
    // keys = 512 bytes per MMA.  B = K (N = head dim, K = keys) from the key
    // tile: MN-major, 128-byte swizzle, 64-wide slabs 16 KB apart, 8-row
    // groups 1024 bytes apart, 16 keys = 2048 bytes per MMA.
    constexpr uint32_t idesc = idesc_bf16(BT, HD, 1, 1);
    const uint64_t dA = smem_desc(base, 4096, 256, kSwizzle32B);
    const uint64_t dB = smem_desc(base + XTILE, SLAB, 1024);
    int j = 0;                 // steps consumed (stage ring position)
    int uses0 = 0, uses1 = 0;  // items accumulated in each accumulator so far
    for (int k = 0;; ++k) {
      if (!mbar_wait_warp(bar_ifull + 8 * (k & 1), (k >> 1) & 1, p.status, &abort_flag)) break;
      const int it = *static_cast<volatile int*>(&items[k & 1]);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_iempty + 8 * (k & 1));
      if (it < 0) break;
      const Item w = decode_item(p, it);
      const int n = count_tiles(p.qmap + ((size_t)w.b * p.nq + w.qt) * p.wk, p.wk);
      if (n == 0) continue;  // the epilogue writes zeros without the accumulator
      const int x = k & 1;
      const int use = x ? uses1++ : uses0++;
      if (use > 0 && !mbar_wait_warp(bar_aempty + 8 * x, (use - 1) & 1, p.status, &abort_flag)) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(x * HD);
      bool ok = true;
      for (int i = 0; i < n; ++i, ++j) {
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
            mma_ss(acc, desc_add(dA, so + ks * 512), desc_add(dB, so + ks * 2048), idesc,
                   (i > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar_empty + 8 * s);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) mma_commit(bar_afull + 8 * x);
      __syncwarp();
    }
    // No wait for this commit here: warp 1 checks it before freeing TMEM.
    if (leader) mma_commit(bar_final);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t out = out_base + (uint32_t)(warp - 2) * out_bytes<HD>();
    int uses0 = 0, uses1 = 0;  // items read from each accumulator so far
    for (int k = 0;; ++k) {
      if (!mbar_wait_warp(bar_ifull + 8 * (k & 1), (k >> 1) & 1, p.status, &abort_flag)) break;
      const int it = *static_cast<volatile int*>(&items[k & 1]);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_iempty + 8 * (k & 1));
      if (it < 0) break;
      const Item w = decode_item(p, it);
      const int n = count_tiles(p.qmap + ((size_t)w.b * p.nq + w.qt) * p.wk, p.wk);
      const int x = k & 1;
      bool have = false;
      if (n > 0) {
        const int use = x ? uses1++ : uses0++;
        if (!mbar_wait_warp(bar_afull + 8 * x, use & 1, p.status, &abort_flag)) break;
        tc_fence_after();
        have = true;
      }
      // this warp's previous store has finished reading its rows
      if (lane == 0) bulk_wait_read0();
      __syncwarp();
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t v[32];
        if (have) {
          tmem_ld32(lane_base + (uint32_t)(x * HD + 32 * c), v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
        const uint32_t slab = out + (uint32_t)(c >> 1) * (OUT_ROWS * 128);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          st_swz_chunk(slab, lane, 4 * (c & 1) + e, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
      if (have) {
        // accumulator x is free for the item after next
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_aempty + 8 * x);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        // rows past L are clipped by the tensor map
        for (int sl = 0; sl < NSLAB; ++sl)
          tma_store_4d(&mdq, out + sl * (OUT_ROWS * 128), 64 * sl, w.h, w.qt * BT + quarter * 32, w.b);
        bulk_commit();
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
  }
  __syncwarp();  // every warp reaches the CTA barrier converged
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // Every MMA has completed before TMEM is released (bounded non-suspending poll).
    if (lane == 0) mbar_poll(bar_final, 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 2 * HD);
  }
}

template <int HD>
cudaError_t launch_hd(const Params& p, cudaStream_t s) {
  CUtensorMap mk, mdq;
  cudaError_t e = make_bhld_map(&mk, p.k, p.B, p.Lk, p.Hkv, HD, BT);
  if (e == cudaSuccess) e = make_bhld_map(&mdq, p.dq, p.B, p.L, p.Hq, HD, OUT_ROWS);
  if (e != cudaSuccess) return e;
  constexpr int SMEM = smem_bytes<HD>();
  auto kern = dq_gemm_kernel<HD>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long nitems = (long long)p.B * p.Hq * p.nq;
  const unsigned grid = (unsigned)(nitems < sms ? nitems : sms);
  prof_begin(CAPATTN_KERNEL_DQ, s);
  prof_count(CAPATTN_KERNEL_DQ, 1);
  e = launch_pdl(kern, dim3(grid), dim3(NTHREADS), SMEM, s, mk, mdq, p);
  if (e != cudaSuccess) return e;
  prof_end(CAPATTN_KERNEL_DQ, s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq_gemm(const Params& p, cudaStream_t s) {
  return p.D == 64 ? launch_hd<64>(p, s) : launch_hd<128>(p, s);
}

}  // namespace capattn
