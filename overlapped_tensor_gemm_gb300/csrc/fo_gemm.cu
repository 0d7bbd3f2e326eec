// Persistent tcgen05 GEMM with ring-aware tile schedule and epilogues.
//
// One launch computes every (rank, step) unit of a decomposed collective:
// Flash-AG (FlashOverlap technical summary, section 2 "Flash-All-Gather") and
// Flash-RS (section 2 "Flash-Reduce-Scatter").  The host lays the units out in
// the method's step order; the kernel walks the tiles in that order, so the
// slices that need no transfer (AG: local slice; RS: first hop) are computed
// while the ring moves the others, and the RS kept slice comes last.
//
// CTA layout (192 threads, one CTA per SM, persistent):
//   warp 0      TMA producer: waits for a slice's arrival flag (AG), then streams
//               128x64 A and 256x64 B bf16 tiles (128-byte swizzle) into a
//               4-stage shared-memory ring; K-major operands as one box each,
//               MN-major ones (transposed operands of the backward) as 64x64
//               boxes, one per 64-wide block.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//               issues tcgen05.mma (M=128, N=256, K=16) from one thread: the
//               kernel's critical path, so its loop is instantiated per operand
//               orientation and its waits test the barrier phase inline.
//   warps 2-5   epilogue: tcgen05.ld of its 32-lane quadrant; plain bf16 results
//               are stored from registers, fp32 partial sums (RS, after acquiring
//               the per-tile flag) go through a per-warp staging buffer so the
//               partial-sum loads and the stores move whole row segments; then
//               release of the per-tile flag read by the next rank.
// Accumulators are double-buffered so the epilogue of tile i overlaps the
// main loop of tile i+1.
#include <cuda_bf16.h>

#include "fo_gemm_common.cuh"
#include "fo_internal.h"
#include "fo_ptx.cuh"

namespace fo {
namespace {

constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 2 * kBN;      // two accumulators
constexpr uint32_t kIdesc = umma_idesc_bf16(kBM, kBN);
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;  // 200 ms for in-flight async work on abort

struct alignas(8) SmemCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t pad;
};

// operand stages, then the four epilogue warps' staging buffers, then the barriers
constexpr int kSmemBytes = kStages * kStageBytes + 4 * kEpiStageBytes + 1024 + static_cast<int>(sizeof(SmemCtl));
// The ring's device-to-device copies may run as a small copy kernel next to this
// persistent grid: leave shared memory free on every SM.
static_assert(kSmemBytes <= 232448 - 16 * 1024, "the persistent GEMM must leave 16 KiB of shared memory free");

// ---------------------------------------------------------------------------
// warp roles
// ---------------------------------------------------------------------------

template <bool TN>
__device__ void producer_loop(const GemmParams& p, uint8_t* tiles, SmemCtl* ctl) {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t armed = 0;        // bit s: stage s has been armed at least once
  uint32_t armed_phase = 0;  // bit s: phase parity of the last arming of stage s
  int waited_flag = -1;  // the last flag this thread has waited for
  bool ok = true;
  bool rows_all_done = false;
  const int mn = p.mn_major & 3;
  constexpr bool tn = TN;
  for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x) {
    const TileCoord tc = tile_coord<TN>(p, tile);
    if (!tile_ok(p, tc, tile, 1)) {
      ok = false;
      break;
    }
    const GemmUnit& u = p.units[tc.unit];
    // a step-pair unit's second 128-row block is the second step's slice
    const int wf = (tc.mb > 0 && u.wait_flag2 >= 0) ? u.wait_flag2 : u.wait_flag;
    if (wf >= 0 && wf != waited_flag) {
      ok = flag_wait(p.flags + wf, p.epoch, p.ctrl, p.timeout_ns, kSiteAgFlag, static_cast<uint32_t>(wf));
      if (!ok) break;
      // the slice was written by a ring copy; order the TMA reads after the acquire
      fence_proxy_async_global();
      waited_flag = wf;
    }
    if (!wait_rows_ready(p, u, tc.mb, &rows_all_done)) {  // A rows written by an earlier tile
      ok = false;
      break;
    }
    const int nk = (u.k + kBK - 1) / kBK;
    const bool lo = tc.mb == 0 && u.a_map_lo >= 0;  // a step-pair unit's first 128 rows, read in place
    const int a_row = lo ? u.a_row_lo : u.a_row0 + tc.mb * kBM;
    const bool gated = u.gated != 0;
    const int b_row = u.b_row0 + tc.nb * (gated ? kBN / 2 : kBN);
    const int b_row_up = u.b_row1 + tc.nb * (kBN / 2);
    // per-tile values in registers: the k loop below re-reads nothing from the parameters
    const bool chunked = u.kchunk > 0;
    const CUtensorMap* amap0 = &p.maps[lo ? u.a_map_lo : u.a_map];
    const CUtensorMap* bmap = &p.maps[u.b_map];
    for (int kb = 0; kb < nk; ++kb) {
      if (!mbar_wait_fast(&ctl->empty[stage], phase ^ 1u, p.ctrl, p.timeout_ns, kSiteEmpty,
                          static_cast<uint32_t>(tile))) {
        ok = false;
        break;
      }
      const CUtensorMap* amap = amap0;
      int arow = a_row, ax = kb * kBK, bx = kb * kBK;
      if (chunked) {
        int am, wait_src;
        kblock_coords(u, kb, a_row, &am, &arow, &ax, &bx, &wait_src);
        amap = &p.maps[am];
        if (wait_src >= 0) {  // a received K chunk: its copy must have landed
          const int f = u.chunk_flag_base + wait_src;
          if (!flag_wait(p.flags + f, p.epoch, p.ctrl, p.timeout_ns, kSiteAgFlag, static_cast<uint32_t>(f))) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
      }
      uint8_t* a = tiles + stage * kStageBytes;
      uint8_t* b = a + kABytes;
      uint64_t* bar = &ctl->full[stage];
      mbar_arrive_expect_tx(bar, kStageBytes);
      if (tn) {  // A: 128 features of the weight; B: the token rows of the tile's tn_S steps
        tma_load_2d(amap0, a, bar, kb * kBK, tc.nb * kBM);
        for (int su = 0; su < p.tn_S; ++su) {
          const GemmUnit& us = p.units[tc.unit + su];
          tma_load_2d(&p.maps[us.b_map], b + su * p.tn_rows * 128, bar, kb * kBK, us.b_row0);
        }
      } else {
        if (mn & 1) {  // A stored [K][M]: x runs along M
          tma_load_2d(amap, a, bar, arow, ax);
          tma_load_2d(amap, a + kMnBox, bar, arow + 64, ax);
        } else {
          tma_load_2d(amap, a, bar, ax, arow);
        }
        if (mn & 2) {  // B stored [K][N]
#pragma unroll
          for (int h = 0; h < kBN / 64; ++h) tma_load_2d(bmap, b + h * kMnBox, bar, b_row + h * 64, bx);
        } else if (gated) {  // gate rows -> B rows [0,128), up rows -> B rows [128,256) (128-row boxes)
          tma_load_2d(bmap, b, bar, bx, b_row);
          tma_load_2d(bmap, b + kBBytes / 2, bar, bx, b_row_up);
        } else {
          tma_load_2d(bmap, b, bar, bx, b_row);
        }
      }
      armed |= 1u << stage;
      armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok) {
    // leave no TMA write in flight into this CTA's shared memory
    for (int s = 0; s < kStages; ++s)
      if ((armed >> s) & 1u) mbar_wait_drain(&ctl->full[s], (armed_phase >> s) & 1u, kDrainNs);
  }
}

// The operand orientation is a template argument: the instruction descriptor stays a
// compile-time constant and the K loop carries no per-block dispatch.
template <bool AMN, bool BMN, bool TN>
__device__ void mma_loop(const GemmParams& p, uint8_t* tiles, SmemCtl* ctl, uint32_t tmem_base) {
  constexpr uint32_t idesc = kIdesc | (AMN ? kIdescAMn : 0u) | (BMN ? kIdescBMn : 0u);
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool issued = false;
  bool ok = true;
  const uint32_t tiles_addr = smem_u32(tiles);
  for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x) {
    const TileCoord tc = tile_coord<TN>(p, tile);
    if (!tile_ok(p, tc, tile, 1)) {
      ok = false;
      break;
    }
    const GemmUnit& u = p.units[tc.unit];
    if (!mbar_wait_fast(&ctl->tmem_empty[acc], acc_phase ^ 1u, p.ctrl, p.timeout_ns, kSiteTmemEmpty,
                   static_cast<uint32_t>(tile))) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
    const int nk = (u.k + kBK - 1) / kBK;
    for (int kb = 0; kb < nk; ++kb) {
      if (!mbar_wait_fast(&ctl->full[stage], phase, p.ctrl, p.timeout_ns, kSiteFull, static_cast<uint32_t>(tile))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_addr = tiles_addr + stage * kStageBytes;
      const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
      for (int k = 0; k < kBK / 16; ++k) {
        // K advance inside the swizzle atom: +32 bytes (K-major) or two 8-row groups (MN-major)
        umma_bf16_ss(d_tmem, operand_desc(a_addr, k, AMN), operand_desc(b_addr, k, BMN), idesc,
                     (kb | k) != 0 ? 1u : 0u);
      }
      issued = true;
      umma_commit(&ctl->empty[stage]);  // frees the stage once these MMAs have read it
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    umma_commit(&ctl->tmem_full[acc]);  // accumulator complete
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
  if (!ok && issued) {
    // wait for every issued MMA before TMEM is released
    umma_commit(&ctl->drain);
    mbar_wait_drain(&ctl->drain, 0, kDrainNs);
  }
}

template <bool TN>
__device__ void epilogue_loop(const GemmParams& p, SmemCtl* ctl, uint32_t tmem_base, int warp, int lane,
                              float* stage) {
  const int q = warp & 3;  // TMEM lanes [32q, 32q+32) are the only ones this warp may access
  int acc = 0;
  uint32_t acc_phase = 0;
  for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
    const TileCoord tc = tile_coord<TN>(p, tile);
    if (!tile_ok(p, tc, tile, 1)) return;
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
    if (!epilogue_tile<TN>(p, tc, tile, &ctl->tmem_full[acc], acc_phase, tbase, 0, 1, q, lane, stage,
                       [&] { mbar_arrive(&ctl->tmem_empty[acc]); }))
      return;
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
}

template <bool TN>
__global__ void __maxnreg__(kGemmMaxRegs) gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* tiles = smem_raw + ((1024u - (base & 1023u)) & 1023u);
  float* epi_stage = reinterpret_cast<float*>(tiles + kStages * kStageBytes);
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(tiles + kStages * kStageBytes + 4 * kEpiStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->tmem_full[b], 1);
      mbar_init(&ctl->tmem_empty[b], 4);
    }
    mbar_init(&ctl->drain, 1);
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.num_maps; ++i) tma_prefetch_desc(&p.maps[i]);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) producer_loop<TN>(p, tiles, ctl);
  } else if (warp == 1) {
    if (lane == 0) {
      if (TN) {  // transposed tiles: K-major operands only
        mma_loop<false, false, true>(p, tiles, ctl, tmem_base);
      } else {
        switch (p.mn_major & 3) {
          case 0: mma_loop<false, false, false>(p, tiles, ctl, tmem_base); break;
          case 2: mma_loop<false, true, false>(p, tiles, ctl, tmem_base); break;
          case 3: mma_loop<true, true, false>(p, tiles, ctl, tmem_base); break;
          default: mma_loop<true, false, false>(p, tiles, ctl, tmem_base); break;
        }
      }
    }
    __syncwarp();
  } else {
    epilogue_loop<TN>(p, ctl, tmem_base, warp, lane, epi_stage + (warp - 2) * (kEpiStageBytes / 4));
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

int gemm_smem_bytes() { return kSmemBytes; }

// Called once at context creation, before any persistent kernel runs: also loads the
// helper kernels (see preload_helper_kernels).
cudaError_t gemm_configure() {
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return e != cudaSuccess ? e : preload_helper_kernels();
}

cudaError_t gemm_launch(const GemmParams& p, int grid, cudaStream_t s) {
  if (p.tn_S > 0) {
    gemm_kernel<true><<<grid, kGemmThreads, kSmemBytes, s>>>(p);
  } else {
    gemm_kernel<false><<<grid, kGemmThreads, kSmemBytes, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fo
