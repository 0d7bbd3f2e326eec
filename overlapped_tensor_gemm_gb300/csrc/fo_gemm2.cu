// Persistent GEMM on SM pairs (tcgen05 cta_group::2): the same ring schedules
// and epilogues as fo_gemm.cu, with 256x256 tiles computed by a cluster of two
// CTAs.  Each CTA stages its own 128 rows of A and one half (128 rows) of B per
// 64-wide K step, so an SM receives 32 KiB per step instead of 48 KiB for the
// same work per SM, and six stages fit in shared memory instead of four.
//
// Pair roles: the CTA of rank 0 in the cluster (the leader) owns the "full"
// barriers of the operand ring (its producer posts the expected bytes of both
// CTAs; both CTAs' TMA loads complete on it) and issues the pair MMAs; every
// MMA commit is multicast to the "empty" barriers of both CTAs.  Each CTA's
// TMEM holds its 128 rows of the 256x256 fp32 accumulator (two buffers), its
// epilogue warps read them and report to the leader's "tmem empty" barrier.
//
// Tile order.  Short launches stride: pair c runs tiles c, c + pairs, c + 2 pairs, ...  Long
// launches (p.claim_tiles) claim tiles in order from one launch-wide counter: the leader's
// producer takes the next index with an atomic add and hands it to every role of both CTAs
// through a small ring in shared memory.  Then the tiles in progress at any moment are a
// window of about one tile per SM pair around the claim point, whatever the spread of the
// pairs' tile durations: tiles that read the same operand panels run at the same time and
// find them in L2, and the pairs finish together.  Either way every tile starts after all
// lower ones have been taken by running pairs, so a tile that waits on an earlier tile's
// flag waits on a tile in progress.
#include <cuda_bf16.h>

#include "fo_gemm_common.cuh"
#include "fo_internal.h"
#include "fo_ptx.cuh"

namespace fo {
namespace {

constexpr int kPairStages = 6;
constexpr uint32_t kPA = 128 * kBK * 2;      // 16 KiB: this CTA's 128 rows of A
constexpr uint32_t kPB = 128 * kBK * 2;      // 16 KiB: this CTA's half of B
constexpr uint32_t kPStage = kPA + kPB;
constexpr uint32_t kPTmemCols = 2 * kBN;     // two 128x256 accumulators per CTA
constexpr uint32_t kPIdesc = umma_idesc_bf16(2 * kBM, kBN);  // M = 256 over the pair, N = 256
constexpr uint64_t kPDrainNs = 200ull * 1000 * 1000;
constexpr int kSchedSlots = 8;  // claimed tile indices in flight per pair
// The leader claims the pair's next tile this many K blocks before the end of the current
// tile's loads: the atomic's round trip is hidden, and the claim comes as late as that allows
// (the later the claim, the narrower the window of tiles in progress).
constexpr int kClaimAheadBlocks = 12;
// Arrivals that free a slot of the ring: the peer's producer once it has read the index, and
// the leader's MMA thread once it has waited for the accumulator of two tiles later to be
// empty, which shows that every epilogue warp of both CTAs has read the index and the tile.
// (An arrive by the epilogue warps themselves would release their stores of the previous
// tile at cluster scope: measured 2.5% slower on short launches.)
constexpr uint32_t kSchedReaders = 2;

struct alignas(8) PairCtl {
  uint64_t full[kPairStages];   // leader: both CTAs' operands of the stage have landed
  uint64_t empty[kPairStages];  // each CTA: the pair MMAs reading the stage are done
  uint64_t tmem_full[2];        // each CTA: accumulator complete
  uint64_t tmem_empty[2];       // leader: both CTAs' epilogues have read the accumulator
  uint64_t drain;
  uint64_t sched_full[kSchedSlots];   // each CTA: the slot holds the pair's next tile index
  uint64_t sched_empty[kSchedSlots];  // leader: every reader has taken the slot's index
  int32_t sched_tile[kSchedSlots];
  uint32_t tmem_base;
  uint32_t pad;
};

// The pair's i-th claimed tile index (total_tiles or more: no tile left), or -1 when the
// wait gave up.  Called by one thread, or (kWarp) by a whole warp whose lane 0 waits and
// passes the index to the other lanes; `release`: the caller frees the slot once read.
template <bool kWarp>
__device__ __forceinline__ int sched_take(const GemmParams& p, PairCtl* ctl, int i, int lane, bool release) {
  int tile = -1;
  if (!kWarp || lane == 0) {
    const int slot = i & (kSchedSlots - 1);
    const uint32_t par = static_cast<uint32_t>(i / kSchedSlots) & 1u;
    if (mbar_try_wait_cluster(&ctl->sched_full[slot], par) ||
        mbar_wait_cluster(&ctl->sched_full[slot], par, p.ctrl, p.timeout_ns, kSiteSched, static_cast<uint32_t>(i))) {
      tile = *static_cast<volatile int32_t*>(&ctl->sched_tile[slot]);
      if (release) mbar_arrive_cluster(map_to_cta(smem_u32(&ctl->sched_empty[slot]), 0));
    }
  }
  if (kWarp) tile = __shfl_sync(0xffffffffu, tile, 0);
  return tile;
}

// operand stages, then the four epilogue warps' staging buffers, then the barriers
constexpr int kPairSmem = kPairStages * kPStage + 4 * kEpiStageBytes + 1024 + static_cast<int>(sizeof(PairCtl));
// The ring's device-to-device copies may run as a small copy kernel next to this
// persistent grid: leave shared memory free on every SM.
static_assert(kPairSmem <= 232448 - 16 * 1024, "the persistent GEMM must leave 16 KiB of shared memory free");

template <bool TN>
__device__ void pair_producer(const GemmParams& p, uint8_t* tiles, PairCtl* ctl, uint32_t cta) {
  const uint32_t leader_full = map_to_cta(smem_u32(&ctl->full[0]), 0);
  const int nclusters = gridDim.x >> 1;
  uint32_t* const counter = p.ctrl + kCtrlTiles;
  const bool claim = p.claim_tiles != 0;
  int next = cta == 0 && claim ? static_cast<int>(atomicAdd(counter, 1u)) : 0;
  int stage = 0;
  uint32_t phase = 0, armed = 0, armed_phase = 0;
  int waited_flag = -1;  // the last flag this thread has waited for
  bool ok = true;
  bool rows_all_done = false;
  const int mn = p.mn_major & 3;
  constexpr bool tn = TN;
  for (int i = 0; ok; ++i) {
    int tile = (blockIdx.x >> 1) + i * nclusters;
    if (claim && cta == 0) {  // publish the claimed index to both CTAs
      const int slot = i & (kSchedSlots - 1);
      const uint32_t par = (static_cast<uint32_t>(i / kSchedSlots) & 1u) ^ 1u;
      if (!mbar_try_wait_cluster(&ctl->sched_empty[slot], par) &&
          !mbar_wait_cluster(&ctl->sched_empty[slot], par, p.ctrl, p.timeout_ns, kSiteSched,
                             static_cast<uint32_t>(i))) {
        ok = false;
        break;
      }
      tile = next;
      ctl->sched_tile[slot] = tile;
      st_shared_cluster_u32(map_to_cta(smem_u32(&ctl->sched_tile[slot]), 1), static_cast<uint32_t>(tile));
      mbar_arrive(&ctl->sched_full[slot]);
      mbar_arrive_cluster(map_to_cta(smem_u32(&ctl->sched_full[slot]), 1));
      // every pair's last claim is past the end; the last of them all resets the counter
      // for the next launch on the stream
      if (tile == p.total_tiles + nclusters - 1) atomicExch(counter, 0u);
    } else if (claim) {
      tile = sched_take<false>(p, ctl, i, 0, true);
      if (tile < 0) {
        ok = false;
        break;
      }
    }
    if (tile >= p.total_tiles) break;
    const TileCoord tc = tile_coord<TN>(p, tile);
    if (!tile_ok(p, tc, tile, 2)) {
      ok = false;
      break;
    }
    const GemmUnit& u = p.units[tc.unit];
    // a step-pair unit's second 128 rows (this CTA's, when cta == 1) are the second step's slice
    const int wf = (cta == 1 && u.wait_flag2 >= 0) ? u.wait_flag2 : u.wait_flag;
    if (wf >= 0 && wf != waited_flag) {
      ok = flag_wait(p.flags + wf, p.epoch, p.ctrl, p.timeout_ns, kSiteAgFlag, static_cast<uint32_t>(wf));
      if (!ok) break;
      fence_proxy_async_global();
      waited_flag = wf;
    }
    if (!wait_rows_ready(p, u, tc.mb, &rows_all_done)) {  // A rows written by an earlier tile
      ok = false;
      break;
    }
    const int nk = (u.k + kBK - 1) / kBK;
    const int claim_kb = cta == 0 && claim ? (nk > kClaimAheadBlocks ? nk - kClaimAheadBlocks : 0) : -1;
    // a step-pair unit may read its first 128 rows (this CTA's, when cta == 0) in place
    const bool lo = cta == 0 && u.a_map_lo >= 0;
    const int a_row = lo ? u.a_row_lo + tc.mb * 2 * kBM : u.a_row0 + tc.mb * 2 * kBM + static_cast<int>(cta) * kBM;
    // B rows of this CTA: gated tiles put the gate rows in the leader and the up rows in the peer
    const int b_row = u.gated ? (cta == 0 ? u.b_row0 : u.b_row1) + tc.nb * (kBN / 2)
                              : u.b_row0 + tc.nb * kBN + static_cast<int>(cta) * (kBN / 2);
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
      if (kb == claim_kb) next = static_cast<int>(atomicAdd(counter, 1u));
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
      uint8_t* a = tiles + stage * kPStage;
      uint8_t* b = a + kPA;
      if (cta == 0) mbar_arrive_expect_tx(&ctl->full[stage], 2 * kPStage);
      const uint32_t bar = leader_full + stage * static_cast<uint32_t>(sizeof(uint64_t));
      if (tn) {
        // A: this CTA's 128 of the tile's 256 features; B: this CTA's half of the token
        // rows, the tile's steps cta * tn_S/2 .. (cta + 1) * tn_S/2 - 1
        tma_load_2d_pair(amap0, a, bar, kb * kBK, tc.nb * 2 * kBM + static_cast<int>(cta) * kBM);
        const int half = p.tn_S / 2;
        for (int su = 0; su < half; ++su) {
          const GemmUnit& us = p.units[tc.unit + static_cast<int>(cta) * half + su];
          tma_load_2d_pair(&p.maps[us.b_map], b + su * p.tn_rows * 128, bar, kb * kBK, us.b_row0);
        }
      } else if (mn == 0) {
        tma_load_2d_pair(amap, a, bar, ax, arow);
        tma_load_2d_pair(bmap, b, bar, bx, b_row);
      } else {
        if (mn & 1) {  // A stored [K][M]: x runs along M
          tma_load_2d_pair(amap, a, bar, arow, ax);
          tma_load_2d_pair(amap, a + kMnBox, bar, arow + 64, ax);
        } else {
          tma_load_2d_pair(amap, a, bar, ax, arow);
        }
        if (mn & 2) {  // B stored [K][N]: this CTA's 128 columns
          tma_load_2d_pair(bmap, b, bar, b_row, bx);
          tma_load_2d_pair(bmap, b + kMnBox, bar, b_row + 64, bx);
        } else {
          tma_load_2d_pair(bmap, b, bar, bx, b_row);
        }
      }
      armed |= 1u << stage;
      armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok) {
    if (cta == 0) {
      for (int s = 0; s < kPairStages; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&ctl->full[s], (armed_phase >> s) & 1u, kPDrainNs);
    } else {
      // this CTA's loads complete on the leader's barriers: give them time to land
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 50000ull) __nanosleep(1000);
    }
  }
}

// The operand orientation is a template argument: the instruction descriptor stays a
// compile-time constant and the K loop carries no per-block dispatch.
template <bool AMN, bool BMN, bool TN>
__device__ void pair_mma(const GemmParams& p, uint8_t* tiles, PairCtl* ctl, uint32_t tmem_base) {
  constexpr uint32_t idesc = kPIdesc | (AMN ? kIdescAMn : 0u) | (BMN ? kIdescBMn : 0u);
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool issued = false, ok = true;
  const uint32_t tiles_addr = smem_u32(tiles);
  const bool claim = p.claim_tiles != 0;
  for (int i = 0; ok; ++i) {
    const int tile = claim ? sched_take<false>(p, ctl, i, 0, false) : (blockIdx.x >> 1) + i * (gridDim.x >> 1);
    if (tile < 0) {
      ok = false;
      break;
    }
    if (tile >= p.total_tiles) break;
    const TileCoord tc = tile_coord<TN>(p, tile);
    if (!tile_ok(p, tc, tile, 2)) {
      ok = false;
      break;
    }
    const GemmUnit& u = p.units[tc.unit];
    if (!mbar_wait_fast(&ctl->tmem_empty[acc], acc_phase ^ 1u, p.ctrl, p.timeout_ns, kSiteTmemEmpty,
                   static_cast<uint32_t>(tile))) {
      ok = false;
      break;
    }
    // the accumulator's previous tile (i - 2) is read out: its index is free
    if (claim && i >= 2) mbar_arrive(&ctl->sched_empty[(i - 2) & (kSchedSlots - 1)]);
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
    const int nk = (u.k + kBK - 1) / kBK;
    for (int kb = 0; kb < nk; ++kb) {
      if (!mbar_wait_fast(&ctl->full[stage], phase, p.ctrl, p.timeout_ns, kSiteFull, static_cast<uint32_t>(tile))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_addr = tiles_addr + stage * kPStage;
      const uint32_t b_addr = a_addr + kPA;
#pragma unroll
      for (int k = 0; k < kBK / 16; ++k) {
        umma_bf16_pair(d_tmem, operand_desc(a_addr, k, AMN), operand_desc(b_addr, k, BMN), idesc,
                       (kb | k) != 0 ? 1u : 0u);
      }
      issued = true;
      umma_commit_pair_mc(&ctl->empty[stage], 0x3);  // frees the stage in both CTAs
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    umma_commit_pair_mc(&ctl->tmem_full[acc], 0x3);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
  if (!ok && issued) {
    umma_commit_pair(&ctl->drain);
    mbar_wait_drain(&ctl->drain, 0, kPDrainNs);
  }
}

template <bool TN>
__device__ void pair_epilogue(const GemmParams& p, PairCtl* ctl, uint32_t tmem_base, uint32_t cta, int warp,
                              int lane, float* stage) {
  const int q = warp & 3;
  const uint32_t leader_tmem_empty = map_to_cta(smem_u32(&ctl->tmem_empty[0]), 0);
  int acc = 0;
  uint32_t acc_phase = 0;
  const bool claim = p.claim_tiles != 0;
  for (int i = 0;; ++i) {
    const int tile = claim ? sched_take<true>(p, ctl, i, lane, false) : (blockIdx.x >> 1) + i * (gridDim.x >> 1);
    if (tile < 0 || tile >= p.total_tiles) return;
    const TileCoord tc = tile_coord<TN>(p, tile);
    if (!tile_ok(p, tc, tile, 2)) return;
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
    auto arrive_empty = [&] {
      if (cta == 0) {
        mbar_arrive(&ctl->tmem_empty[acc]);
      } else {
        mbar_arrive_cluster(leader_tmem_empty + acc * static_cast<uint32_t>(sizeof(uint64_t)));
      }
    };
    if (!epilogue_tile<TN>(p, tc, tile, &ctl->tmem_full[acc], acc_phase, tbase, static_cast<int>(cta), 2, q, lane, stage,
                       arrive_empty))
      return;
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
}

// TN: transposed reduce-scatter tiles (each tile kind is its own instantiation, with its
// own register count).
template <bool TN>
__global__ void __maxnreg__(kGemmMaxRegs) gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* tiles = smem_raw + ((1024u - (base & 1023u)) & 1023u);
  float* epi_stage = reinterpret_cast<float*>(tiles + kPairStages * kPStage);
  PairCtl* ctl = reinterpret_cast<PairCtl*>(tiles + kPairStages * kPStage + 4 * kEpiStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->tmem_full[b], 1);
      mbar_init(&ctl->tmem_empty[b], 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(&ctl->drain, 1);
    for (int s = 0; s < kSchedSlots; ++s) {
      mbar_init(&ctl->sched_full[s], 1);
      mbar_init(&ctl->sched_empty[s], kSchedReaders);
    }
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.num_maps; ++i) tma_prefetch_desc(&p.maps[i]);
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl->tmem_base, kPTmemCols);  // one warp of each CTA, collectively
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) pair_producer<TN>(p, tiles, ctl, cta);
  } else if (warp == 1) {
    if (lane == 0 && cta == 0) {
      if (TN) {  // transposed tiles: K-major operands only
        pair_mma<false, false, true>(p, tiles, ctl, tmem_base);
      } else {
        switch (p.mn_major & 3) {
          case 0: pair_mma<false, false, false>(p, tiles, ctl, tmem_base); break;
          case 2: pair_mma<false, true, false>(p, tiles, ctl, tmem_base); break;
          case 3: pair_mma<true, true, false>(p, tiles, ctl, tmem_base); break;
          default: pair_mma<true, false, false>(p, tiles, ctl, tmem_base); break;
        }
      }
    }
    __syncwarp();
  } else {
    pair_epilogue<TN>(p, ctl, tmem_base, cta, warp, lane, epi_stage + (warp - 2) * (kEpiStageBytes / 4));
  }

  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPTmemCols);
  }
}

}  // namespace

cudaError_t gemm_pair_configure() {
  cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
  return e;
}

// Number of SM pairs that can be resident at once (the persistent grid must not exceed it).
int gemm_pair_max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t gemm_pair_launch(const GemmParams& p, int clusters, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.tn_S > 0) return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<true>, p);
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<false>, p);
}

}  // namespace fo
