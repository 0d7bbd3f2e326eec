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

// One 32-column chunk of one row: optional fp32 partial add, then store.
__device__ __forceinline__ void store_chunk(const GemmUnit& u, int row, int col, const uint32_t (&v)[32]) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  const bool full = col + 32 <= u.n_cols;
  const int ncol = full ? 32 : u.n_cols - col;
  if (u.epi == kEpiAddF32 || u.epi == kEpiAddBF16) {
    const float* src = u.acc_in + static_cast<int64_t>(row) * u.ld_acc + col;
    if (full) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 a = ld_cg_f4(src + 4 * i);
        f[4 * i + 0] += a.x;
        f[4 * i + 1] += a.y;
        f[4 * i + 2] += a.z;
        f[4 * i + 3] += a.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < ncol) f[i] += __ldcg(src + i);
    }
  }
  if (u.epi == kEpiBF16 || u.epi == kEpiAddBF16) {
    uint16_t* dst = static_cast<uint16_t*>(u.c) + static_cast<int64_t>(row) * u.ldc + col;
    if (full) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        st_v4_u32(dst + 8 * i, pack_bf16x2(f[8 * i + 0], f[8 * i + 1]), pack_bf16x2(f[8 * i + 2], f[8 * i + 3]),
                  pack_bf16x2(f[8 * i + 4], f[8 * i + 5]), pack_bf16x2(f[8 * i + 6], f[8 * i + 7]));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < ncol) dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(f[i]));
    }
  } else {
    float* dst = static_cast<float*>(u.c) + static_cast<int64_t>(row) * u.ldc + col;
    if (full) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        st_v4_u32(dst + 4 * i, __float_as_uint(f[4 * i + 0]), __float_as_uint(f[4 * i + 1]),
                  __float_as_uint(f[4 * i + 2]), __float_as_uint(f[4 * i + 3]));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < ncol) dst[i] = f[i];
    }
  }
}

__device__ __forceinline__ float round_bf16(float x) {
  return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x))) << 16);
}

// MLP glue fused into the gate/up epilogue: the gate and up accumulators are
// rounded to bf16 first (as the unfused layer stores them), then
// SiLU(g) * u = g / (1 + exp(-g)) * u in fp32, rounded once to bf16.
__device__ __forceinline__ void store_silu_chunk(const GemmUnit& u, int row, int col, const uint32_t (&g)[32],
                                                 const uint32_t (&v)[32]) {
  float h[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float gi = round_bf16(__uint_as_float(g[i]));
    const float ui = round_bf16(__uint_as_float(v[i]));
    h[i] = gi / (1.0f + expf(-gi)) * ui;
  }
  uint16_t* dst = static_cast<uint16_t*>(u.c) + static_cast<int64_t>(row) * u.ldc + col;
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

}  // namespace
}  // namespace fo
