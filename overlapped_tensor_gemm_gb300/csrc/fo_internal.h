// Internal definitions shared by the host side and the kernels of the
// Flash-Overlap library (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstring>

#include "../../include/fo.h"

namespace fo {

constexpr int kMaxP = 8;

// ---------------------------------------------------------------------------
// Persistent tcgen05 GEMM: problem description
// ---------------------------------------------------------------------------
//
// A launch computes a list of "units".  A unit is one rank's GEMM on one ring
// step: rows [a_row0, a_row0 + m_rows) of its A operand (via a TMA map)
// times the rows [b_row0, b_row0 + n_cols) of its B operand (nn.Linear
// layout, K contiguous; or both transposed, see GemmParams::mn_major), written
// through a per-unit epilogue.  Units are
// grouped (one group per ring step); the tiles of a launch are enumerated group
// by group, and inside a group either unit by unit (n-block outer, m-block
// inner: consecutive CTAs share the B tile, the whole A slice stays in L2) or
// m-block-major across units.  Every CTA
// walks the global tile sequence with stride gridDim.x, so a tile only ever
// waits on tiles with a smaller index (deadlock freedom of the in-kernel ring).

constexpr int kBM = 128;            // UMMA M
constexpr int kBN = 256;            // UMMA N
constexpr int kBK = 64;             // one 128-byte swizzle atom of bf16
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;   // warp 0: TMA, warp 1: MMA, warps 2-5: epilogue
// Registers per thread of the GEMM kernels.  Two of the six warps share an SM sub-partition
// (16K registers): at 200 they hold 12,800 of them, which leaves room for the ring's
// device-to-device copies when those run as a small copy kernel beside the persistent grid.
constexpr int kGemmMaxRegs = 200;
constexpr int kMaxMaps = 40;    // one launch of a whole MLP layer: 3P maps for Flash-AG + 2P for Flash-RS
constexpr int kMaxUnits = 128;  // P*P units per decomposed collective, two collectives per layer
constexpr int kMaxGroups = 24;

enum EpiMode : int32_t {
  kEpiBF16 = 0,        // C (bf16) = acc
  kEpiF32 = 1,         // C (fp32) = acc
  kEpiAddF32 = 2,      // C (fp32) = acc + acc_in
  kEpiAddBF16 = 3,     // C (bf16) = acc + acc_in
  kEpiSiluMul = 4,     // gated tile: C (bf16) = SiLU(bf16(acc[:, :128])) * bf16(acc[:, 128:])
};

struct GemmUnit {
  int32_t a_map, b_map;        // indices into GemmParams::maps
  int32_t a_row0, b_row0;      // row offsets into the A / B tensors
  int32_t m_rows, n_cols, k;   // valid extent of this unit
  int32_t tiles_m, tiles_n;
  int32_t wait_flag;           // AG: flag index that must reach `epoch` before A is read (-1: none)
  // A step-pair unit (AG with 128-row slices): its 256 rows are two ring steps' slices,
  // stored next to each other in step order; rows [128, 256) wait on wait_flag2 (not
  // wait_flag) and are stored at c2 (not c) from its row 0.  wait_flag2 = -1, c2 = null:
  // an ordinary unit.  a_map_lo >= 0: rows [0, 128) are read from that map at row a_row_lo
  // instead (the rank's own slice, read in place).
  int32_t wait_flag2;
  int32_t a_map_lo, a_row_lo;
  int32_t in_flag_base;        // RS: per-tile flags guarding acc_in (-1: none)
  int32_t out_flag_base;       // RS: per-tile flags released after C is written (-1: none)
  int32_t epi;                 // EpiMode
  int32_t gated;               // 1: B tile = 128 gate rows at b_row0 + 128 up rows at b_row1 (kEpiSiluMul)
  int32_t b_row1;              // gated: row offset of the up half of B
  // K-chunked A (all-to-all consumer): K is split into chunks of `kchunk` columns, one per
  // source rank.  Chunk 0 is the own block (a_map at a_row0); chunk ci > 0 comes from
  // source s = (chunk_self - ci) mod chunk_nsrc (ascending s = ci when chunk_order == 1)
  // at rows s * a2_row_stride of a_map2, after flag chunk_flag_base + s reaches `epoch`
  // (chunk_flag_base < 0: no wait).  B's K offset of chunk ci is s * kchunk.
  int32_t kchunk;              // 0: plain K
  int32_t chunk_self, chunk_nsrc, chunk_order;
  int32_t a_map2, a2_row_stride, chunk_flag_base;
  int32_t done_counter;        // >= 0: every epilogue warp adds 1 to flags[done_counter] after its
                               // part of a tile is stored (system-scope release)
  // One launch for a whole layer: a producing unit counts, per m-block of its tiles, the
  // epilogue warps that have stored their rows (flags[rows_done_base + m-block], gpu-scope
  // release); a consuming unit's producer waits before loading A rows of m-block mb until
  // flags[a_ready_base + mb] >= a_ready_count (the counters start at zero every launch).
  int32_t rows_done_base;      // -1: none
  int32_t a_ready_base;        // -1: none
  int32_t a_ready_count;
  void* c;                     // output
  void* c2;                    // step-pair unit: output of rows [128, 256)
  const float* acc_in;         // fp32 partial sum to add (kEpiAdd*)
  int64_t ldc, ld_acc;         // leading dimensions in elements
};

struct GemmParams {
  CUtensorMap maps[kMaxMaps];
  GemmUnit units[kMaxUnits];
  int32_t group_unit_begin[kMaxGroups + 1];
  int32_t group_tile_begin[kMaxGroups + 1];
  int32_t num_groups;
  int32_t num_maps;            // maps[0, num_maps) are valid
  int32_t mblock_major;        // 1: tiles of a group ordered (m-block, unit, n-block);
                               // 0: unit by unit, n-block outer, m-block inner
  int32_t group_nb_major;      // bit g: group g ordered (n-block, unit, m-block) instead
  // Operand orientation of every unit of the launch: bit 0 set: A is stored [K][M] (M
  // contiguous), bit 1 set: B is stored [K][N] (a transposed weight).  Such operands are
  // staged as 64 (M or N) x 64 (K) boxes, one per 64-wide block, and read by the MMA as
  // MN-major (no K chunks, no gating).  The kernels instantiate their MMA loop per value.
  int32_t mn_major;
  // Transposed reduce-scatter tiles (tn_S > 0).  For slices of 32-128 token rows the MMA's
  // M side is 128 output features (A = the rank's weight, K-major, one 128-row box) and its
  // N side the token rows of tn_S consecutive ring steps of one rank (B = the activations,
  // one box of tn_rows rows per step; tn_S * tn_rows = 256).  Units are laid out rank-major
  // in step order (unit of rank r, step t at index r * tn_S * tn_passes + t); a tile is
  // (rank r, pass, feature block fb) and covers the steps pass*tn_S .. +tn_S-1 of rank r.
  // Tiles are ordered (fb group, pass, fb in group, rank), so the tn_passes tiles that read
  // one weight block are close together (it is fetched from HBM about once), and the
  // epilogue adds each step's partial sums in step order, one ring hop per step.
  int32_t tn_S;
  int32_t tn_rows;      // token rows per unit (256 / tn_S)
  int32_t tn_ranks;
  int32_t tn_passes;    // tiles per rank and feature block
  int32_t tn_fblocks;   // feature blocks of 128 (single SM) or 256 (SM pair) features
  int32_t tn_fb_group;  // feature blocks per ordering group (divides tn_fblocks)
  // One launch for a whole layer: every epilogue warp that counts rows into a
  // rows_done_base counter also adds 1 to flags[rows_all_index]; once that word reaches
  // rows_all_count every producing tile has stored its rows, and a producer stops checking
  // per-block counters (-1: no such word).
  int32_t rows_all_index;
  int32_t rows_all_count;
  // 1: the fp32 partial sums are loaded and stored as streaming (evict-first) data: one ring
  // step's partial sums are larger than L2, so they come back from DRAM anyway, and should
  // not evict the operands the GEMM reuses.
  int32_t stream_partials;
  // SM-pair kernel: 1: pairs claim tiles in order from a launch-wide counter; 0: pair c runs
  // tiles c, c + pairs, c + 2 * pairs, ...
  int32_t claim_tiles;
  int32_t total_tiles;
  uint32_t epoch;
  uint64_t timeout_ns;
  uint32_t* flags;             // ring flags (epoch-valued)
  int32_t flag_words;          // words at `flags` (the debug build checks every flag index)
  uint32_t* ctrl;              // device control block (error word, abort flag)
};
static_assert(sizeof(GemmParams) <= 32764, "GemmParams must fit the kernel parameter space");

// A unit with every optional feature off (-1 indices, null pointers, zero counts): every
// builder starts from this, so a field added later has its neutral value everywhere.
inline GemmUnit blank_unit() {
  GemmUnit u;
  std::memset(&u, 0, sizeof(u));
  u.wait_flag = -1;
  u.wait_flag2 = -1;
  u.a_map_lo = -1;
  u.in_flag_base = -1;
  u.out_flag_base = -1;
  u.done_counter = -1;
  u.rows_done_base = -1;
  u.a_ready_base = -1;
  return u;
}

// A tile's position: unit index, m-block and n-block inside the unit.
struct TileCoord {
  int unit, mb, nb;
};

// Device control block layout (uint32 words).
enum CtrlWord : int {
  kCtrlError = 0,     // first error code (FO_ERR_*), 0 = none
  kCtrlAbort = 1,     // non-zero: every CTA leaves its loops
  kCtrlWhere = 2,     // where the first timeout happened (see WaitSite)
  kCtrlDetail = 3,    // flag index / tile index of the first timeout
  kCtrlTiles = 4,     // SM-pair GEMM: the next unclaimed tile of the running launch (zero
                      // between launches: the launch's last claim resets it)
  kCtrlItems = 5,     // attention: the next unclaimed item of the running launch (likewise)
  kCtrlWords = 8
};

enum WaitSite : uint32_t {
  kSiteAgFlag = 1, kSiteFull = 2, kSiteEmpty = 3, kSiteTmemFull = 4,
  kSiteTmemEmpty = 5, kSiteAccInFlag = 6, kSiteDrain = 7, kSiteAttnFlag = 8,
  kSiteAttnBar = 9, kSiteVRange = 10, kSiteRowsReady = 11, kSiteBounds = 12,
  kSiteSched = 13
};

// host launchers (fo_gemm.cu: single-SM 128x256 tiles; fo_gemm2.cu: SM-pair 256x256 tiles)
cudaError_t gemm_configure();
cudaError_t gemm_launch(const GemmParams& p, int grid, cudaStream_t s);
int gemm_smem_bytes();
cudaError_t gemm_pair_configure();
int gemm_pair_max_clusters();
cudaError_t gemm_pair_launch(const GemmParams& p, int clusters, cudaStream_t s);

// elementwise kernels (fo_elem.cu); bf16 data is passed as raw uint16_t
struct SiluMulArgs {
  const uint16_t* gu[kMaxP];
  uint16_t* h[kMaxP];
  int64_t ld_gu[kMaxP], ld_h[kMaxP];
  int64_t rows, f;
  int32_t P;
};
cudaError_t launch_silu_mul(const SiluMulArgs& a, cudaStream_t s);
// loads the helper kernels (glue, reduce adds) before any persistent kernel runs
cudaError_t preload_helper_kernels();
// flags[0, n) = value
cudaError_t launch_fill_u32(uint32_t* flags, int64_t n, uint32_t value, cudaStream_t s);
// c = a + b (fp32 inputs); c is fp32 (c_f32) or bf16 (c_bf16), exactly one non-null
cudaError_t launch_add_f32(const float* a, int64_t lda, const float* b, int64_t ldb, float* c_f32,
                           uint16_t* c_bf16, int64_t ldc, int64_t rows, int64_t cols, cudaStream_t s);

}  // namespace fo
