// Device helpers shared by the single-SM and the SM-pair GEMM kernels: tile
// decoding of the ring schedule, the epilogue stores (plain, fp32 partial-sum
// add, fused SiLU(gate)*up) and warp-uniform bounded waits.
#pragma once

#include <cuda_bf16.h>

#include "fo_internal.h"
#include "fo_ptx.cuh"

namespace fo {
namespace {

// Operand coordinates of K block kb of unit u.  `a_row` is the unit's A row for this
// tile (own rows); for K-chunked units the A map, A row and K offsets follow the chunk's
// source rank.  *wait_src >= 0: the first block of a received chunk (wait for its flag).
__device__ __forceinline__ void kblock_coords(const GemmUnit& u, int kb, int a_row, int* amap, int* arow, int* ax,
                                              int* bx, int* wait_src) {
  *wait_src = -1;
  if (u.kchunk <= 0) {
    *amap = u.a_map;
    *arow = a_row;
    *ax = *bx = kb * kBK;
    return;
  }
  const int cpk = u.kchunk / kBK;
  const int ci = kb / cpk;
  const int kk = (kb - ci * cpk) * kBK;
  const int s = u.chunk_order == 1 ? ci : (u.chunk_self - ci + u.chunk_nsrc) % u.chunk_nsrc;
  *ax = kk;
  *bx = s * u.kchunk + kk;
  if (s == u.chunk_self) {
    *amap = u.a_map;
    *arow = a_row;
  } else {
    *amap = u.a_map2;
    *arow = a_row - u.a_row0 + s * u.a2_row_stride;
    if (kk == 0 && u.chunk_flag_base >= 0) *wait_src = s;
  }
}

// An MN-major operand block in shared memory: `nblk` boxes of 64 MN elements (one
// 128-byte swizzled row per K index) x 64 K rows, kMnBox bytes apart.
constexpr uint32_t kMnBox = 64 * kBK * 2;
constexpr uint32_t kIdescAMn = 1u << 15;  // instruction descriptor: A is MN-major
constexpr uint32_t kIdescBMn = 1u << 16;  // B is MN-major

// Shared-memory descriptor of the K=16 slice k of a staged operand: K-major atoms
// advance 32 bytes inside the 128-byte row, MN-major ones by two 8-row groups.
__device__ __forceinline__ uint64_t operand_desc(uint32_t addr, int k, bool mn) {
  return mn ? umma_sdesc_sw128_mn(addr + k * 2048, kMnBox) : umma_sdesc_sw128(addr + k * 32);
}

__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, int tile) {
  int g = 0;
  while (g + 1 < p.num_groups && tile >= p.group_tile_begin[g + 1]) ++g;
  const int j = tile - p.group_tile_begin[g];
  const int u0 = p.group_unit_begin[g];
  const int nu = p.group_unit_begin[g + 1] - u0;
  const int tm = p.units[u0].tiles_m;
  const int tn = p.units[u0].tiles_n;
  TileCoord c;
  if ((p.group_nb_major >> g) & 1) {
    c.nb = j / (nu * tm);
    const int rem = j - c.nb * nu * tm;
    c.unit = u0 + rem / tm;
    c.mb = rem % tm;
  } else if (p.mblock_major) {
    c.mb = j / (nu * tn);
    const int rem = j - c.mb * nu * tn;
    c.unit = u0 + rem / tn;
    c.nb = rem % tn;
  } else {
    const int u = j / (tm * tn);
    const int rem = j - u * tm * tn;
    c.unit = u0 + u;
    c.nb = rem / tm;
    c.mb = rem % tm;
  }
  return c;
}

// ---------------------------------------------------------------------------
// Partial-sum and fp32 epilogues through a per-warp staging buffer.
//
// tcgen05.ld (32x32b) hands each lane one accumulator row, so a lane-per-row global access
// touches 32 rows per instruction.  Instead each epilogue warp writes its 32x32 fp32
// chunk to shared memory row by row, reads it back so that 8 lanes cover one row's 32
// columns (4 rows per instruction), and loads partial sums / stores results in that
// row-contiguous layout.  Rows are 128 bytes; 16-byte granule g of row r sits at
// g ^ (r & 7), which keeps both passes free of bank conflicts.
// ---------------------------------------------------------------------------
constexpr int kEpiStageBytes = 32 * 32 * 4;  // one warp's chunk

__device__ __forceinline__ int stage_index(int row, int g) { return row * 32 + ((g ^ (row & 7)) << 2); }

// Partial sums of one chunk in the coalesced layout: pf[i] = row 4i + lane/8 of the warp's
// rows (first row `row0`), columns col + 4*(lane%8) .. +3; zero outside the unit.
// The staged path's helpers copy the unit fields they use into locals first: read through
// the reference into the kernel's parameter space, they were read again after every global
// store (the stores' inline assembly may write memory), which measured 5-12% slower
// reduce-scatter launches at K = 1024-3584 per rank.
__device__ __forceinline__ void load_partial(const GemmUnit& u, int row0, int col, int lane, float4 (&pf)[8],
                                             bool stream = false) {
  const int c = col + 4 * (lane & 7);
  const int m_rows = u.m_rows, n_cols = u.n_cols;
  const float* acc_in = u.acc_in;
  const int64_t ld_acc = u.ld_acc;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = row0 + 4 * i + (lane >> 3);
    float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (r < m_rows && c < n_cols) {
      const float* src = acc_in + static_cast<int64_t>(r) * ld_acc + c;
      if (c + 4 <= n_cols) {
        x = stream ? ld_cs_f4(src) : ld_cg_f4(src);
      } else {
        x.x = __ldcg(src);
        if (c + 1 < n_cols) x.y = __ldcg(src + 1);
        if (c + 2 < n_cols) x.z = __ldcg(src + 2);
      }
    }
    pf[i] = x;
  }
}

// Stores one staged chunk (+ the partial sums when `add`) in the coalesced layout.  The
// chunk's eight stage reads are issued before its stores, which would otherwise order each
// read after the previous store (measured: short-K reduce-scatter launches 5-15% faster).
__device__ __forceinline__ void store_staged(const GemmUnit& u, void* out, int row0, int col, int lane,
                                             const float* stage, bool add, const float4 (&pf)[8],
                                             bool stream = false) {
  const int c = col + 4 * (lane & 7);
  const bool bf16_out = u.epi == kEpiBF16 || u.epi == kEpiAddBF16;
  const int m_rows = u.m_rows;
  const int ncol = u.n_cols - c;
  const int64_t ldc = u.ldc;
  float4 xs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) xs[i] = *reinterpret_cast<const float4*>(stage + stage_index(4 * i + (lane >> 3), lane & 7));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = row0 + 4 * i + (lane >> 3);
    float4 x = xs[i];
    if (add) {
      x.x += pf[i].x;
      x.y += pf[i].y;
      x.z += pf[i].z;
      x.w += pf[i].w;
    }
    if (r >= m_rows || ncol <= 0) continue;
    if (bf16_out) {
      uint16_t* dst = static_cast<uint16_t*>(out) + static_cast<int64_t>(r) * ldc + c;
      if (ncol >= 4) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
      } else {
        dst[0] = __bfloat16_as_ushort(__float2bfloat16_rn(x.x));
        if (ncol > 1) dst[1] = __bfloat16_as_ushort(__float2bfloat16_rn(x.y));
        if (ncol > 2) dst[2] = __bfloat16_as_ushort(__float2bfloat16_rn(x.z));
      }
    } else {
      float* dst = static_cast<float*>(out) + static_cast<int64_t>(r) * ldc + c;
      if (ncol >= 4) {
        if (stream) {
          st_cs_v4_u32(dst, __float_as_uint(x.x), __float_as_uint(x.y), __float_as_uint(x.z), __float_as_uint(x.w));
        } else {
          st_v4_u32(dst, __float_as_uint(x.x), __float_as_uint(x.y), __float_as_uint(x.z), __float_as_uint(x.w));
        }
      } else {
        dst[0] = x.x;
        if (ncol > 1) dst[1] = x.y;
        if (ncol > 2) dst[2] = x.z;
      }
    }
  }
}

// A plain bf16 chunk of one row (lane = row), stored straight from registers: without
// partial sums to load this was measured faster than the staged path.
__device__ __forceinline__ void store_bf16_row_chunk(const GemmUnit& u, void* out, int row, int col,
                                                     const uint32_t (&v)[32]) {
  uint16_t* dst = static_cast<uint16_t*>(out) + static_cast<int64_t>(row) * u.ldc + col;
  if (col + 32 <= u.n_cols) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st_v4_u32(dst + 8 * i,
                pack_bf16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1])),
                pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
    }
  } else {
    const int ncol = u.n_cols - col;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncol) dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[i])));
  }
}

// The kBN columns of the warp's 32 accumulator rows (first row `row0`), chunk by chunk.
// With a partial-sum add, `pf` holds chunk 0's partials on entry (loaded before the
// accumulator was complete) and the loads of chunk c+1 are in flight while chunk c is
// stored, through the warp's shared-memory stage in row-contiguous 128-byte segments
// (measured faster than storing lane per row straight from registers, which touches 32
// rows per instruction: Flash-RS launches 3-12% faster at 13-400 tiles per SM pair).
// tn_rows > 0: a unit of a transposed tile.  The warp's 32 TMEM lanes are then the output
// columns [col0, col0 + 32) and TMEM columns tbase .. tbase + tn_rows the unit's rows
// 0 .. tn_rows-1; each 32x32 chunk is staged transposed (row-major: every write
// instruction fills one 128-byte row of the stage) and stored by the same row-contiguous
// path.
template <bool kTn>
__device__ __forceinline__ void store_rows(const GemmUnit& u, void* out, uint32_t tbase, int row0, int col0, int lane,
                                           bool add, float4 (&pf)[8], float* stage, int tn_rows, bool stream) {
  constexpr bool tn = kTn;
  if (!tn && u.epi == kEpiBF16) {
    const int row = row0 + lane;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
      const int col = col0 + c * 32;
      if (col >= u.n_cols) break;
      uint32_t v[32];
      tmem_ld32(tbase + c * 32, v);
      tmem_wait_ld();
      if (row < u.m_rows) store_bf16_row_chunk(u, out, row, col, v);
    }
    return;
  }
  const int nchunks = tn ? tn_rows / 32 : kBN / 32;
  // Chunk c: its accumulator columns through the stage plus the partial sums `cur` (loaded
  // while the previous chunk was stored), while the next chunk's partial sums load into
  // `nxt`.  Two chunks per iteration, the buffers swapping roles: a copy of the loaded
  // registers at the end of a chunk would wait for its loads there (measured: the K = 1024
  // reduce-scatter launch 12% faster without that copy).
  float4 alt[8];
  auto chunk = [&](int c, float4 (&cur)[8], float4 (&nxt)[8]) -> bool {
    const int r0 = tn ? c * 32 : row0;    // first row of the chunk
    const int col = tn ? col0 : col0 + c * 32;
    if (col >= u.n_cols) return false;
    uint32_t v[32];
    tmem_ld32(tbase + c * 32, v);
    if (add && c + 1 < nchunks) load_partial(u, tn ? r0 + 32 : row0, tn ? col0 : col + 32, lane, nxt, stream);
    tmem_wait_ld();
    if (tn) {
#pragma unroll
      for (int j = 0; j < 32; ++j) stage[stage_index(j, lane >> 2) + (lane & 3)] = __uint_as_float(v[j]);
    } else {
#pragma unroll
      for (int g = 0; g < 8; ++g)
        *reinterpret_cast<float4*>(stage + stage_index(lane, g)) =
            make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]), __uint_as_float(v[4 * g + 2]),
                        __uint_as_float(v[4 * g + 3]));
    }
    __syncwarp();
    store_staged(u, out, r0, col, lane, stage, add, cur, stream);
    __syncwarp();  // the stage is rewritten by the next chunk
    return true;
  };
#pragma unroll 1
  for (int c = 0; c < nchunks; c += 2) {
    if (!chunk(c, pf, alt)) break;
    if (c + 1 < nchunks && !chunk(c + 1, alt, pf)) break;
  }
}

__device__ __forceinline__ float round_bf16(float x) {
  return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x))) << 16);
}

// MLP glue fused into the gate/up epilogue: the gate and up accumulators are
// rounded to bf16 first (as the unfused layer stores them), then
// SiLU(g) * u = g / (1 + exp(-g)) * u in fp32, rounded once to bf16.
__device__ __forceinline__ void store_silu_chunk(const GemmUnit& u, void* out, int row, int col,
                                                 const uint32_t (&g)[32], const uint32_t (&v)[32]) {
  float h[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float gi = round_bf16(__uint_as_float(g[i]));
    const float ui = round_bf16(__uint_as_float(v[i]));
    h[i] = gi / (1.0f + expf(-gi)) * ui;
  }
  uint16_t* dst = static_cast<uint16_t*>(out) + static_cast<int64_t>(row) * u.ldc + col;
  if (col + 32 <= u.n_cols) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st_v4_u32(dst + 8 * i, pack_bf16x2(h[8 * i + 0], h[8 * i + 1]), pack_bf16x2(h[8 * i + 2], h[8 * i + 3]),
                pack_bf16x2(h[8 * i + 4], h[8 * i + 5]), pack_bf16x2(h[8 * i + 6], h[8 * i + 7]));
    }
  } else {
    const int ncol = u.n_cols - col;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncol) dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(h[i]));
  }
}

// Lane 0 waits; the outcome is broadcast so the whole warp takes one path.
__device__ __forceinline__ bool warp_mbar_wait(uint64_t* bar, uint32_t parity, const GemmParams& p,
                                               uint32_t site, uint32_t detail, int lane) {
  uint32_t ok = 0;
  if (lane == 0) ok = mbar_wait_fast(bar, parity, p.ctrl, p.timeout_ns, site, detail) ? 1u : 0u;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ bool warp_flag_wait(const uint32_t* flag, const GemmParams& p, uint32_t site,
                                               uint32_t detail, int lane) {
  uint32_t ok = 0;
  if (lane == 0) ok = flag_wait(flag, p.epoch, p.ctrl, p.timeout_ns, site, detail) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)ld_acquire_gpu(flag);  // every lane orders its own partial-sum reads after the flag
  return ok != 0;
}

// ---------------------------------------------------------------------------
// Transposed reduce-scatter tiles (GemmParams::tn_S > 0)
// ---------------------------------------------------------------------------

// Tile -> (first unit of the tile, feature block in nb).  Order: feature-block group,
// pass, feature block inside the group, rank.
__device__ __forceinline__ TileCoord decode_tile_tn(const GemmParams& p, int tile) {
  const int per_pass = p.tn_fb_group * p.tn_ranks;
  const int per_group = per_pass * p.tn_passes;
  const int g = tile / per_group;
  int rem = tile - g * per_group;
  const int pass = rem / per_pass;
  rem -= pass * per_pass;
  const int fbi = rem / p.tn_ranks;
  const int r = rem - fbi * p.tn_ranks;
  TileCoord c;
  c.unit = (r * p.tn_passes + pass) * p.tn_S;
  c.mb = 0;
  c.nb = g * p.tn_fb_group + fbi;
  return c;
}

// TN: the launch runs transposed reduce-scatter tiles (the kernels are instantiated per
// tile kind, so the step-ordered instantiation carries none of the transposed code).
template <bool TN>
__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, int tile) {
  return TN ? decode_tile_tn(p, tile) : decode_tile(p, tile);
}

// Flag release and completion counters after a unit's rows of a tile are stored.
__device__ __forceinline__ void publish_unit(const GemmParams& p, const GemmUnit& u, int slot, int mb, int lane) {
  if (u.out_flag_base >= 0) {
    // rows of this quadrant are stored: publish them to the next rank
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_gpu(p.flags + u.out_flag_base + slot, p.epoch);
  }
  if (u.done_counter >= 0) {
    // this warp's rows of the tile are final: count them for a copy engine that waits
    __threadfence_system();
    __syncwarp();
    if (lane == 0) red_release_sys_add(p.flags + u.done_counter, 1u);
  }
  if (u.rows_done_base >= 0) {
    // this warp's rows of the tile are stored: count them for the tiles that read them
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      red_release_gpu_add(p.flags + u.rows_done_base + mb, 1u);
      if (p.rows_all_index >= 0) red_release_gpu_add(p.flags + p.rows_all_index, 1u);
    }
  }
}

// Producer side of the row counters: before loading A rows of m-block mb that earlier tiles
// of this launch write, wait for their count -- unless every producing tile of the launch
// is known to be done (*all_done), after which nothing is checked or fenced again.
__device__ __forceinline__ bool wait_rows_ready(const GemmParams& p, const GemmUnit& u, int mb, bool* all_done) {
  if (u.a_ready_base < 0 || *all_done) return true;
  if (p.rows_all_index >= 0 && ld_acquire_gpu(p.flags + p.rows_all_index) >= static_cast<uint32_t>(p.rows_all_count)) {
    *all_done = true;
  } else {
    const int f = u.a_ready_base + mb;
    if (!count_wait(p.flags + f, static_cast<uint32_t>(u.a_ready_count), p.ctrl, p.timeout_ns, kSiteRowsReady,
                    static_cast<uint32_t>(f)))
      return false;
  }
  fence_proxy_async_global();  // the rows were written through the generic proxy; TMA reads them
  return true;
}

// One tile's epilogue for one epilogue warp (TMEM lane quadrant q of CTA `cta` of `ncta`).
// A step-ordered tile has one unit: its partial sum's flag and first chunk are taken while
// the accumulator is still computed, and its flag is released after the accumulator is
// freed.  A transposed tile has tn_S units (ring steps of one rank), handled in step order:
// each after its incoming partial sum's flag, each released before the next.  This is the
// only call site of store_rows, so a kernel inlines one copy of it.  `arrive_empty()`
// frees the accumulator.  False if a wait gave up.
template <bool TN, class ArriveEmpty>
__device__ __forceinline__ bool epilogue_tile(const GemmParams& p, const TileCoord& tc, int tile, uint64_t* tmem_full,
                                              uint32_t acc_phase, uint32_t tbase, int cta, int ncta, int q, int lane,
                                              float* stage, ArriveEmpty arrive_empty) {
  constexpr bool tn = TN;
  const GemmUnit& u0 = p.units[tc.unit];
  const int blk = tn ? tc.nb : tc.mb * u0.tiles_n + tc.nb;
  const int slot = (blk * ncta + cta) * 4 + q;           // flags per (tile, CTA half, quadrant)
  int row0 = tn ? 0 : (tc.mb * ncta + cta) * kBM + q * 32;  // the warp's first row
  const int col0 = tn ? (tc.nb * ncta + cta) * kBM + q * 32 : tc.nb * kBN;
  void* out = u0.c;
  if (!tn && u0.c2 != nullptr && row0 >= kBM) {  // a step-pair unit: rows [kBM, 2 kBM) are the second step's
    out = u0.c2;
    row0 -= kBM;
  }
  float4 pf[8];
  if (!tn) {
    if (u0.in_flag_base >= 0) {
      const int f = u0.in_flag_base + slot;
      if (!warp_flag_wait(p.flags + f, p, kSiteAccInFlag, static_cast<uint32_t>(f), lane)) return false;
    }
    if (u0.epi == kEpiAddF32 || u0.epi == kEpiAddBF16) {
      load_partial(u0, row0, col0, lane, pf, p.stream_partials != 0);
    }
  }
  if (!warp_mbar_wait(tmem_full, acc_phase, p, kSiteTmemFull, static_cast<uint32_t>(tile), lane)) return false;
  tc_fence_after();
  const int nparts = tn ? p.tn_S : 1;
  for (int s = 0; s < nparts; ++s) {
    const GemmUnit& u = p.units[tc.unit + s];
    const bool add = u.epi == kEpiAddF32 || u.epi == kEpiAddBF16;
    if (tn) {
      if (u.in_flag_base >= 0) {
        const int f = u.in_flag_base + slot;
        if (!warp_flag_wait(p.flags + f, p, kSiteAccInFlag, static_cast<uint32_t>(f), lane)) return false;
      }
      if (add) load_partial(u, 0, col0, lane, pf, p.stream_partials != 0);
    }
    if (u.epi == kEpiSiluMul) {
      const int row = row0 + lane;
#pragma unroll 1
      for (int c = 0; c < kBN / 64; ++c) {
        uint32_t g[32], v[32];
        tmem_ld32(tbase + c * 32, g);
        tmem_ld32(tbase + kBN / 2 + c * 32, v);
        tmem_wait_ld();
        const int col = tc.nb * (kBN / 2) + c * 32;
        if (row < u.m_rows && col < u.n_cols) store_silu_chunk(u, out, row, col, g, v);
      }
    } else {
      // transposed: the unit's token rows are TMEM columns [s * tn_rows, +tn_rows)
      store_rows<TN>(u, tn ? u.c : out, tbase + (tn ? s * p.tn_rows : 0), row0, col0, lane, add, pf, stage,
                            tn ? p.tn_rows : 0, p.stream_partials != 0);
    }
    if (tn) publish_unit(p, u, slot, tc.mb, lane);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) arrive_empty();
  if (!tn) publish_unit(p, u0, slot, tc.mb, lane);
  return true;
}

// ---------------------------------------------------------------------------
// Debug build (FO_DEBUG_BOUNDS): index checks
// ---------------------------------------------------------------------------
// The tile's decoded coordinates, the operand maps of its units and every flag word the
// tile reads or writes are checked against the launch's extents.  A failure records
// FO_ERR_INTERNAL (site kSiteBounds, detail: the tile) and raises the abort word, and the
// role leaves its loop as after a wait that ran out.  The release build compiles the
// checks away.
__device__ __forceinline__ bool tile_ok(const GemmParams& p, const TileCoord& tc, int tile, int ncta) {
#ifdef FO_DEBUG_BOUNDS
  auto flag_ok = [&](int64_t i) { return i >= 0 && i < p.flag_words; };
  const int nunits = p.group_unit_begin[p.num_groups];
  const int nsub = p.tn_S > 0 ? p.tn_S : 1;
  bool ok = tc.unit >= 0 && tc.unit + nsub <= nunits && nunits <= kMaxUnits && tc.nb >= 0 && tc.mb >= 0;
  if (ok) ok = p.tn_S > 0 ? tc.nb < p.tn_fblocks
                          : tc.mb < p.units[tc.unit].tiles_m && tc.nb < p.units[tc.unit].tiles_n;
  if (p.rows_all_index >= 0) ok = ok && flag_ok(p.rows_all_index);
  for (int s = 0; ok && s < nsub; ++s) {
    const GemmUnit& u = p.units[tc.unit + s];
    // the largest flag slot of the tile: per (tile or feature block, CTA half, quadrant)
    const int64_t blk = p.tn_S > 0 ? tc.nb : static_cast<int64_t>(tc.mb) * u.tiles_n + tc.nb;
    const int64_t slot_max = (blk * ncta + ncta - 1) * 4 + 3;
    if (u.wait_flag >= 0) ok = ok && flag_ok(u.wait_flag);
    if (u.wait_flag2 >= 0) ok = ok && flag_ok(u.wait_flag2) && u.m_rows == 2 * kBM;
    if (u.a_map_lo >= 0) ok = ok && u.a_map_lo < p.num_maps && u.wait_flag2 >= 0;
    if (u.in_flag_base >= 0) ok = ok && flag_ok(u.in_flag_base + slot_max);
    if (u.out_flag_base >= 0) ok = ok && flag_ok(u.out_flag_base + slot_max);
    if (u.done_counter >= 0) ok = ok && flag_ok(u.done_counter);
    if (u.rows_done_base >= 0) ok = ok && flag_ok(static_cast<int64_t>(u.rows_done_base) + tc.mb);
    if (u.a_ready_base >= 0) ok = ok && flag_ok(static_cast<int64_t>(u.a_ready_base) + tc.mb);
    if (u.kchunk > 0 && u.chunk_flag_base >= 0) ok = ok && flag_ok(u.chunk_flag_base + u.chunk_nsrc - 1);
    ok = ok && u.a_map >= 0 && u.a_map < p.num_maps && u.b_map >= 0 && u.b_map < p.num_maps;
    if (u.kchunk > 0) ok = ok && u.a_map2 >= 0 && u.a_map2 < p.num_maps;
  }
  if (!ok) raise_error(p.ctrl, FO_ERR_INTERNAL, kSiteBounds, static_cast<uint32_t>(tile));
  return ok;
#else
  (void)p;
  (void)tc;
  (void)tile;
  (void)ncta;
  return true;
#endif
}

}  // namespace
}  // namespace fo
