// Host side of the Flash-Overlap library: context and workspace, argument
// validation, the ring step engine (per-rank link streams, device-to-device copies,
// stream memory operations that publish per-slice flags), the step schedules
// of Flash-AG / Flash-RS and of the two baselines, and the C ABI of fo.h.
//
// Method: FlashOverlap (technical summary, section 2): collectives decomposed
// into ring P2P steps; Flash-AG computes the local slice first, Flash-RS
// defers the kept slice to the last step; section 1: data slicing leaves the
// last chunk's communication exposed (reproduced here as a baseline).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "fo_internal.h"

namespace fo {
fo_status attn_run(fo_ctx* ctx, const fo_mat* Q, const fo_mat* K, const fo_mat* V, int P, int heads,
                   int head_dim, int causal, const fo_mat* O, const fo_opts* opts, cudaStream_t stream, bool ring);
}

using namespace fo;

namespace {

thread_local std::string g_last_error;

fo_status fail(fo_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define FO_CUDA(expr)                                                                      \
  do {                                                                                     \
    cudaError_t e_ = (expr);                                                               \
    if (e_ != cudaSuccess) return fail(FO_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

// Driver entry points, resolved through the runtime so that the library has no
// link-time dependency on libcuda (it loads on hosts without a GPU driver).
typedef CUresult (*PfnEncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*PfnWriteValue32)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
typedef CUresult (*PfnWaitValue32)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
typedef CUresult (*PfnGetErrorString)(CUresult, const char**);

struct DriverFns {
  PfnEncodeTiled encode_tiled = nullptr;
  PfnWriteValue32 write_value32 = nullptr;
  PfnWaitValue32 wait_value32 = nullptr;
  PfnGetErrorString get_error_string = nullptr;
};

const DriverFns* driver() {
  static DriverFns fns;
  static bool loaded = false;
  if (!loaded) {
    cudaDriverEntryPointQueryResult q;
    cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&fns.encode_tiled), 12000,
                                     cudaEnableDefault, &q);
    cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", reinterpret_cast<void**>(&fns.write_value32), 12000,
                                     cudaEnableDefault, &q);
    cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", reinterpret_cast<void**>(&fns.wait_value32), 12000,
                                     cudaEnableDefault, &q);
    cudaGetDriverEntryPointByVersion("cuGetErrorString", reinterpret_cast<void**>(&fns.get_error_string), 12000,
                                     cudaEnableDefault, &q);
    loaded = fns.encode_tiled && fns.write_value32 && fns.wait_value32 && fns.get_error_string;
  }
  return loaded ? &fns : nullptr;
}

#define FO_CU(expr)                                                       \
  do {                                                                    \
    CUresult r_ = (expr);                                                 \
    if (r_ != CUDA_SUCCESS) {                                             \
      const char* s_ = nullptr;                                           \
      driver()->get_error_string(r_, &s_);                                \
      return fail(FO_ERR_CUDA, "%s: %s", #expr, s_ ? s_ : "unknown");     \
    }                                                                     \
  } while (0)

#define FO_TRY(expr)                \
  do {                              \
    fo_status st_ = (expr);         \
    if (st_ != FO_OK) return st_;   \
  } while (0)

enum BufId : int {
  kBufFlags = 0,
  kBufAgRecv,
  kBufRsRecv,
  kBufPart,
  kBufMlpY,
  kBufMlpH,
  kBufHostX,
  kBufHostZ,
  kBufLayerQkv,
  kBufLayerO,
  kBufA2aRecv,
  kBufA2aLocal,
  kBufBwdStack,
  kBufAttnRecv,
};

// Flag layout (uint32 words, epoch-valued):
//   [0, kMaxP*kMaxP)                AG / attention arrival: rank r holds slice s
//   [kDoneBase, kDoneBase + kMaxP)  RS: per-rank completion counters of the kept chunk's
//                                   tiles (running totals, not epochs)
//   [kRsFlagBase, ...)             RS per-(rank, hop, tile, quadrant) partial-sum flags
constexpr int64_t kAgFlagBase = 0;
constexpr int64_t kDoneBase = 64;
constexpr int64_t kRsFlagBase = 256;
// [kRowsBase, ...): one launch for a whole layer: per-(rank, slice, m-block) counts of the
// stored rows of the intermediate activations (reset to zero before each such launch)
constexpr int64_t kRowsBase = 1 << 18;
constexpr size_t kFlagBytes = 2u << 20;

constexpr int kMaxSlices = 16;

struct Buffer {
  void* ptr = nullptr;
  size_t bytes = 0;
};

}  // namespace

struct fo_ctx {
  int device = 0;
  int num_sms = 0;
  cudaStream_t link[kMaxP] = {};
  cudaStream_t aux = nullptr;
  cudaEvent_t ev_fork = nullptr;
  cudaEvent_t ev_join[kMaxP] = {};
  cudaEvent_t ev_hop[kMaxP][kMaxP] = {};
  cudaEvent_t ev_slice[kMaxSlices][kMaxP] = {};
  cudaEvent_t ev_aux = nullptr;
  cudaEvent_t ev_phase[3] = {};
  bool phase_valid = false;
  bool phase_gemm_first = false;  // RS serial: GEMM phase precedes the collective
  uint32_t* ctrl = nullptr;
  uint32_t epoch = 0;
  int pair_clusters = 0;  // resident SM pairs for the 256x256-tile kernel (0: unavailable)
  uint32_t done_total[kMaxP] = {};  // running targets of the per-rank completion counters
  std::map<int, Buffer> bufs;
};

namespace {

size_t elem_size(int32_t dtype) { return dtype == FO_F32 ? 4 : 2; }

fo_status ensure_buf(fo_ctx* ctx, int id, size_t bytes, void** out) {
  Buffer& b = ctx->bufs[id];
  if (b.bytes < bytes) {
    if (b.ptr) {
      FO_CUDA(cudaDeviceSynchronize());  // in-flight work may still use the old buffer
      FO_CUDA(cudaFree(b.ptr));
      b.ptr = nullptr;
      b.bytes = 0;
    }
    const size_t rounded = (bytes + (2u << 20) - 1) & ~static_cast<size_t>((2u << 20) - 1);
    if (cudaMalloc(&b.ptr, rounded) != cudaSuccess) {
      cudaGetLastError();
      b.ptr = nullptr;
      return fail(FO_ERR_OOM, "workspace growth to %zu bytes failed", rounded);
    }
    b.bytes = rounded;
    if (id == kBufFlags) FO_CUDA(cudaMemset(b.ptr, 0, rounded));  // epochs start at 1
  }
  *out = b.ptr;
  return FO_OK;
}

// --------------------------------------------------------------------------
// validation
// --------------------------------------------------------------------------

fo_status check_mat(const fo_mat& a, int32_t dtype, const char* what, int r) {
  if (!a.ptr && a.rows > 0 && a.cols > 0) return fail(FO_ERR_INVALID_ARG, "%s[%d]: null pointer", what, r);
  if (a.dtype != dtype)
    return fail(FO_ERR_INVALID_ARG, "%s[%d]: dtype %d, expected %d", what, r, a.dtype, dtype);
  if (a.rows < 0 || a.cols < 0 || a.ld < a.cols)
    return fail(FO_ERR_SHAPE, "%s[%d]: bad shape rows=%lld cols=%lld ld=%lld", what, r, (long long)a.rows,
                (long long)a.cols, (long long)a.ld);
  if (a.rows == 0 || a.cols == 0) return FO_OK;  // empty: no element is ever addressed
  if (reinterpret_cast<uintptr_t>(a.ptr) % 16 != 0)
    return fail(FO_ERR_UNSUPPORTED, "%s[%d]: pointer not 16-byte aligned", what, r);
  if ((a.ld * static_cast<int64_t>(elem_size(dtype))) % 16 != 0)
    return fail(FO_ERR_UNSUPPORTED, "%s[%d]: row pitch ld*size=%lld not a multiple of 16 bytes", what, r,
                (long long)(a.ld * elem_size(dtype)));
  if (a.rows > (1ll << 30) || a.cols > (1ll << 30))
    return fail(FO_ERR_UNSUPPORTED, "%s[%d]: dimension above 2^30", what, r);
  return FO_OK;
}

fo_status check_common(fo_ctx* ctx, int P, const fo_opts* opts) {
  if (!ctx) return fail(FO_ERR_INVALID_ARG, "null context");
  if (P < 1 || P > kMaxP) return fail(FO_ERR_INVALID_ARG, "P=%d outside [1, %d]", P, kMaxP);
  if (opts) {
    if (opts->order < FO_ORDER_FLASH || opts->order > FO_ORDER_SERIAL)
      return fail(FO_ERR_INVALID_ARG, "unknown order %d", opts->order);
    if (opts->link < FO_LINK_DEFAULT || opts->link > FO_LINK_PUSH)
      return fail(FO_ERR_INVALID_ARG, "unknown link %d", opts->link);
    if (opts->n_slices < 0 || opts->n_slices > kMaxSlices)
      return fail(FO_ERR_INVALID_ARG, "n_slices=%d outside [0, %d]", opts->n_slices, kMaxSlices);
    if (opts->fault < FO_FAULT_NONE || opts->fault > FO_FAULT_SKIP_HOP)
      return fail(FO_ERR_INVALID_ARG, "unknown fault %d", opts->fault);
    if (opts->num_sms < 0) return fail(FO_ERR_INVALID_ARG, "num_sms < 0");
    if (opts->epilogue < FO_EPI_PLAIN || opts->epilogue > FO_EPI_SILU_GATE)
      return fail(FO_ERR_INVALID_ARG, "unknown epilogue %d", opts->epilogue);
    if (opts->sm_pairs < 0 || opts->sm_pairs > 2) return fail(FO_ERR_INVALID_ARG, "sm_pairs must be 0, 1 or 2");
    if (opts->compute_only < 0 || opts->compute_only > 1)
      return fail(FO_ERR_INVALID_ARG, "compute_only must be 0 or 1");
    if (opts->split_layer < 0 || opts->split_layer > 1) return fail(FO_ERR_INVALID_ARG, "split_layer must be 0 or 1");
  }
  return FO_OK;
}

fo_opts default_opts() {
  fo_opts o;
  std::memset(&o, 0, sizeof(o));
  o.order = FO_ORDER_FLASH;
  o.link = FO_LINK_DEFAULT;
  return o;
}

uint64_t timeout_ns(const fo_opts& o) {
  return (o.timeout_us ? static_cast<uint64_t>(o.timeout_us) : 1000000ull) * 1000ull;
}

int grid_size(const fo_ctx* ctx, const fo_opts& o, int tiles) {
  int g = ctx->num_sms;
  if (o.num_sms > 0 && o.num_sms < g) g = o.num_sms;
  if (tiles < g) g = tiles;
  return g < 1 ? 1 : g;
}

// --------------------------------------------------------------------------
// TMA maps
// --------------------------------------------------------------------------

fo_status encode_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows,
                     CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  FO_CU(driver()->encode_tiled(map, dtype, 2, const_cast<void*>(ptr), dims, strides,
                               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
  return FO_OK;
}

// An MN-major operand stored [k_rows][mn_cols] (MN contiguous): boxes of 64 MN elements
// (one 128-byte swizzled row) x 64 K rows.
fo_status encode_map_mn(CUtensorMap* map, const void* ptr, int64_t k_rows, int64_t mn_cols, int64_t ld) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(mn_cols), static_cast<cuuint64_t>(k_rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(kBK)};
  cuuint32_t estr[2] = {1, 1};
  FO_CU(driver()->encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
  return FO_OK;
}

struct MapSpec {
  const void* ptr;
  int64_t rows, cols, ld;
  int box_rows;  // 0: MN-major map (fixed 64 x 64 boxes)
};

struct Launch {
  GemmParams p;
  MapSpec spec[kMaxMaps];
  int arrivals_per_tile = 4;  // epilogue warps that finish each tile (8 on SM pairs)
  bool tn_pair = false;       // transposed reduce-scatter tiles on SM pairs (p.tn_S > 0)
  int num_units = 0;
  int num_groups = 0;
  int num_maps = 0;
  Launch() { std::memset(&p, 0, sizeof(p)); }

  int add_map(fo_status* st, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    if (num_maps >= kMaxMaps) {
      *st = fail(FO_ERR_UNSUPPORTED, "too many operand maps");
      return -1;
    }
    *st = encode_map(&p.maps[num_maps], ptr, rows, cols, ld, box_rows);
    spec[num_maps] = MapSpec{ptr, rows, cols, ld, box_rows};
    return num_maps++;
  }
  // An operand stored transposed, [K][M or N]; the launch reading it sets p.mn_major.
  int add_map_mn(fo_status* st, const void* ptr, int64_t k_rows, int64_t mn_cols, int64_t ld) {
    if (num_maps >= kMaxMaps) {
      *st = fail(FO_ERR_UNSUPPORTED, "too many operand maps");
      return -1;
    }
    *st = encode_map_mn(&p.maps[num_maps], ptr, k_rows, mn_cols, ld);
    spec[num_maps] = MapSpec{ptr, k_rows, mn_cols, ld, 0};
    return num_maps++;
  }

  // SM-pair tiles: each CTA stages 128 rows of B (its half of the 256-wide tile), so
  // every B operand map is re-encoded with 128-row boxes.
  fo_status pair_boxes() {
    bool is_b[kMaxMaps] = {};
    for (int u = 0; u < num_units; ++u) is_b[p.units[u].b_map] = true;
    for (int m = 0; m < num_maps; ++m) {
      if (!is_b[m] || spec[m].box_rows == kBN / 2 || spec[m].box_rows == 0) continue;
      FO_TRY(encode_map(&p.maps[m], spec[m].ptr, spec[m].rows, spec[m].cols, spec[m].ld, kBN / 2));
      spec[m].box_rows = kBN / 2;
    }
    return FO_OK;
  }
  void begin_group(bool nb_major = false) {
    p.group_unit_begin[num_groups] = num_units;
    if (nb_major) p.group_nb_major |= 1 << num_groups;
    ++num_groups;
  }
  GemmUnit& add_unit() { return p.units[num_units++]; }

  // Tile grids for tiles of `bm` rows (128: single SM, 256: SM pair).  All units of a
  // group share one tile grid.
  fo_status retile(int bm) {
    int64_t tiles = 0;
    for (int g = 0; g < num_groups; ++g) {
      p.group_tile_begin[g] = static_cast<int32_t>(tiles);
      const int u0 = p.group_unit_begin[g], u1 = p.group_unit_begin[g + 1];
      for (int u = u0; u < u1; ++u) {
        GemmUnit& x = p.units[u];
        const int bn = x.gated ? kBN / 2 : kBN;  // output columns per tile
        x.tiles_m = (x.m_rows + bm - 1) / bm;
        x.tiles_n = (x.n_cols + bn - 1) / bn;
        if (x.tiles_m != p.units[u0].tiles_m || x.tiles_n != p.units[u0].tiles_n)
          return fail(FO_ERR_SHAPE, "units of one step must share a tile grid");
        tiles += static_cast<int64_t>(x.tiles_m) * x.tiles_n;
      }
    }
    if (tiles > (1ll << 30)) return fail(FO_ERR_UNSUPPORTED, "too many tiles");
    p.group_tile_begin[num_groups] = static_cast<int32_t>(tiles);
    p.total_tiles = static_cast<int32_t>(tiles);
    return FO_OK;
  }

  // Every unit's rows are a multiple of 256: the SM-pair kernel wastes no rows.
  bool pair_friendly() const {
    for (int u = 0; u < num_units; ++u)
      if (p.units[u].m_rows % (2 * kBM) != 0) return false;
    return num_units > 0;
  }

  // Finalises group boundaries and tile counts (single-SM tiles).
  fo_status finish(uint32_t epoch, uint64_t tmo, uint32_t* flags, uint32_t* ctrl, int mblock_major) {
    if (num_units > kMaxUnits || num_groups > kMaxGroups)
      return fail(FO_ERR_UNSUPPORTED, "too many units (%d) or groups (%d)", num_units, num_groups);
    p.group_unit_begin[num_groups] = num_units;
    FO_TRY(retile(kBM));
    p.num_groups = num_groups;
    p.num_maps = num_maps;
    p.mblock_major = mblock_major;
    p.epoch = epoch;
    p.timeout_ns = tmo;
    p.flags = flags;
    p.flag_words = static_cast<int32_t>(kFlagBytes / 4);
    p.ctrl = ctrl;
    p.rows_all_index = -1;
    return FO_OK;
  }
};

// SM-pair launches with at least this many tiles per pair claim their tiles from a counter
// (measured: 8K and 16K layers, 200-400 tiles per pair, 7-8% faster; the 4K layer, ~100,
// equal; the 2K and Llama-3-8B layers, 37-50, 1-2% slower than striding)
constexpr int kClaimTilesPerPair = 128;

// Resident SM pairs for a launch (the persistent grid never exceeds them).
int pair_grid(const fo_ctx* ctx, const fo_opts& o) {
  int clusters = ctx->pair_clusters;
  if (o.num_sms > 0 && o.num_sms / 2 < clusters) clusters = o.num_sms / 2 > 0 ? o.num_sms / 2 : 1;
  return clusters;
}

fo_status launch_gemm(fo_ctx* ctx, Launch& L, const fo_opts& o, cudaStream_t stream) {
  if (L.p.total_tiles == 0) return FO_OK;
  if (L.p.tn_S > 0) {  // transposed reduce-scatter tiles: the shape was chosen by the builder
    if (L.tn_pair) {
      int clusters = pair_grid(ctx, o);
      if (L.p.total_tiles < clusters) clusters = L.p.total_tiles;
      L.p.claim_tiles = L.p.total_tiles >= kClaimTilesPerPair * clusters;
      FO_CUDA(gemm_pair_launch(L.p, clusters, stream));
    } else {
      FO_CUDA(gemm_launch(L.p, grid_size(ctx, o, L.p.total_tiles), stream));
    }
    return FO_OK;
  }
  if (o.sm_pairs != 1 && ctx->pair_clusters > 0 && L.pair_friendly()) {
    // 256x256 tiles on SM pairs; the persistent grid never exceeds the resident clusters
    FO_TRY(L.retile(2 * kBM));
    FO_TRY(L.pair_boxes());
    int clusters = pair_grid(ctx, o);
    if (L.p.total_tiles < clusters) clusters = L.p.total_tiles;
    L.arrivals_per_tile = 8;
    L.p.claim_tiles = L.p.total_tiles >= kClaimTilesPerPair * clusters;
    FO_CUDA(gemm_pair_launch(L.p, clusters, stream));
    return FO_OK;
  }
  FO_CUDA(gemm_launch(L.p, grid_size(ctx, o, L.p.total_tiles), stream));
  return FO_OK;
}

int mod(int a, int P) { return ((a % P) + P) % P; }

// Step schedules (FlashOverlap technical summary, section 2).  Pure functions:
// the launch builders below and fo_step_order use exactly these.
//   Flash-AG: unit i of step t is rank i, computing slice (i - t) mod P (its own at t = 0).
//   Flash-RS: unit i of step t is rank (t + i) mod P, computing chunk (r - t - 1) mod P,
//             so the kept chunk r comes at t = P-1; the rotation places every unit at the
//             position of the unit of step t-1 whose partial sum it consumes.  (The fused
//             step-ordered launch computes the same units, grouped two steps at a time in
//             its tile order: build_rs_flash.)
//   naive RS: step c is chunk c on every rank, units in chain order r = c+1, c+2, ..., c.
void ag_unit(int P, int t, int i, int* rank, int* slice) {
  *rank = i;
  *slice = mod(i - t, P);
}

void rs_unit(int P, int order, int t, int i, int* rank, int* chunk) {
  if (order == FO_ORDER_NAIVE) {
    *rank = mod(t + 1 + i, P);
    *chunk = t;
  } else {
    *rank = mod(t + i, P);
    *chunk = mod(*rank - t - 1, P);
  }
}

//   Flash all-to-all, producer side (GEMM -> A2A): at step t rank r computes the output
//             block of destination (r + t + 1) mod P, so its own block comes last
//             (kept-last, as Flash-RS); naive: block t at step t.
//   Flash all-to-all, consumer side (A2A -> GEMM): at step t rank r folds in the K chunk
//             received from source (r - t) mod P, its own chunk first (local-first, as
//             Flash-AG); naive: chunk t at step t.
void a2a_block_unit(int P, int order, int t, int i, int* rank, int* block) {
  *rank = i;
  *block = order == FO_ORDER_NAIVE ? t : mod(i + t + 1, P);
}
void a2a_source_unit(int P, int order, int t, int i, int* rank, int* source) {
  *rank = i;
  *source = order == FO_ORDER_NAIVE ? t : mod(i - t, P);
}

char* bptr(const fo_mat& a, int64_t row) {
  return static_cast<char*>(a.ptr) + row * a.ld * static_cast<int64_t>(elem_size(a.dtype));
}

// Copy `rows` rows of `cols` bf16 elements (a rank's slice) on a link stream.
fo_status copy_rows(void* dst, int64_t dld, const void* src, int64_t sld, int64_t rows, int64_t cols,
                    size_t esz, cudaStream_t s) {
  if (rows == 0 || cols == 0) return FO_OK;
  if (dld == cols && sld == cols) {
    FO_CUDA(cudaMemcpyAsync(dst, src, rows * cols * esz, cudaMemcpyDeviceToDevice, s));
  } else {
    FO_CUDA(cudaMemcpy2DAsync(dst, dld * esz, src, sld * esz, cols * esz, rows, cudaMemcpyDeviceToDevice, s));
  }
  return FO_OK;
}

fo_status write_flag(cudaStream_t s, uint32_t* flag, uint32_t value) {
  // default flags: the write is ordered after (and made visible after) the prior copy on the stream
  FO_CU(driver()->write_value32(reinterpret_cast<CUstream>(s), reinterpret_cast<CUdeviceptr>(flag), value,
                             CU_STREAM_WRITE_VALUE_DEFAULT));
  return FO_OK;
}

// Host order of a ring's copies and the persistent kernel that waits on them.  The copies
// always depend only on work before the call, so the two run concurrently either way; the
// order decides who gets the SMs first.  Kernel first (default): the persistent grid takes
// every SM before the copies start; measured on GB300, enqueuing the 16K MLP layer's
// all-gather copies first made its launch 4% slower (no change at 4K tokens).  A tool that
// serialises the work it intercepts (a kernel profiler) would then run the kernel alone,
// waiting for copies queued behind it until its waits give up, so under such a tool the
// copies are enqueued first.  Such a tool is recognised by the environment it gives the
// process it runs: Nsight Compute's injection settings (NV_NSIGHT_INJECTION_TRANSPORT_TYPE,
// NV_COMPUTE_PROFILER_PERFWORKS_DIR) or an injection library (CUDA_INJECTION64_PATH).
// FO_COPIES_FIRST=1 / 0 forces the order.
bool copies_first() {
  static const bool v = [] {
    const char* force = std::getenv("FO_COPIES_FIRST");
    if (force && force[0]) return force[0] == '1';
    for (const char* name : {"NV_NSIGHT_INJECTION_TRANSPORT_TYPE", "NV_COMPUTE_PROFILER_PERFWORKS_DIR",
                             "CUDA_INJECTION64_PATH"}) {
      const char* v = std::getenv(name);
      if (v && v[0]) return true;
    }
    return false;
  }();
  return v;
}

fo_status fork_links(fo_ctx* ctx, int P, cudaStream_t stream) {
  FO_CUDA(cudaEventRecord(ctx->ev_fork, stream));
  for (int r = 0; r < P; ++r) FO_CUDA(cudaStreamWaitEvent(ctx->link[r], ctx->ev_fork, 0));
  return FO_OK;
}

fo_status join_links(fo_ctx* ctx, int P, cudaStream_t stream) {
  for (int r = 0; r < P; ++r) {
    FO_CUDA(cudaEventRecord(ctx->ev_join[r], ctx->link[r]));
    FO_CUDA(cudaStreamWaitEvent(stream, ctx->ev_join[r], 0));
  }
  return FO_OK;
}

// --------------------------------------------------------------------------
// Flash-AG and its baselines
// --------------------------------------------------------------------------

struct AgArgs {
  const fo_mat* X;
  const fo_mat* W;
  const fo_mat* Y;
  int P;
  int64_t m, K, N;
  char* recv;  // rank r's gathered copy: recv + r*M*K*2, slice s at row s*m
  bool w_kn;   // W[r] given as [K, N] (the transposed weight of a backward pass)
  const fo_mat* Xh;  // non-null: X[r] is first uploaded from these host shards (flash order:
                     // in rank order on the link streams, each slice's step-0 GEMM behind
                     // the upload's flag)
};

// Rank r's receive buffer holds the slices in ring-step order: slice s at position
// (r - s) mod P, the position of the step that computes it (position 0, the rank's own
// slice, stays empty: step-pair units read that slice in place), so two consecutive
// received steps are 2m contiguous rows.
int ag_position(const AgArgs& a, int r, int s) { return ((r - s) % a.P + a.P) % a.P; }
char* ag_rank_buffer(const AgArgs& a, int r) { return a.recv + static_cast<int64_t>(r) * a.P * a.m * a.K * 2; }
char* ag_slot(const AgArgs& a, int r, int s, int64_t row_in_slice) {
  return a.recv + ((static_cast<int64_t>(r) * a.P + ag_position(a, r, s)) * a.m + row_in_slice) * a.K * 2;
}

// The ring all-gather of rows [row0, row0 + rows) of every slice, on the link
// streams.  Hop t: rank r forwards slice (r - t + 1) mod P (its own at t = 1)
// to rank r+1 and, with `flags`, publishes arrival of that slice at r+1.
// Uploads of the host shards a.Xh into X (flash order): one at a time in rank order on the
// link streams, each publishing the (rank r, slice r) flag, which no ring hop uses, so the
// GEMM of rank 0's own slice starts after one slice has crossed the host link instead of
// all of them; each rank's first ring hop follows its upload on the same stream.
// Step pairs wait on the (r, r) flag too (a stream write, or the upload's completion).
fo_status enqueue_uploads(fo_ctx* ctx, const AgArgs& a, uint32_t epoch, uint32_t* flag_base) {
  for (int r = 0; r < a.P; ++r) {
    cudaStream_t ls = ctx->link[r];
    if (a.Xh) {
      if (r > 0) FO_CUDA(cudaStreamWaitEvent(ls, ctx->ev_hop[r - 1][0], 0));
      FO_CUDA(cudaMemcpy2DAsync(a.X[r].ptr, a.X[r].ld * 2, a.Xh[r].ptr, a.Xh[r].ld * 2, a.K * 2, a.m,
                                cudaMemcpyHostToDevice, ls));
      FO_CUDA(cudaEventRecord(ctx->ev_hop[r][0], ls));
    }
    FO_TRY(write_flag(ls, flag_base + kAgFlagBase + r * a.P + r, epoch));
  }
  return FO_OK;
}

fo_status enqueue_ag_ring(fo_ctx* ctx, const AgArgs& a, int64_t row0, int64_t rows, bool flags, uint32_t epoch,
                          int fault, uint32_t* flag_base) {
  const int P = a.P;
  for (int t = 1; t < P; ++t) {
    for (int r = 0; r < P; ++r) {
      const int d = mod(r + 1, P);
      const int s = mod(r - t + 1, P);
      if (fault == FO_FAULT_SKIP_HOP && t == P - 1 && r == 0) continue;
      cudaStream_t ls = ctx->link[r];
      if (t >= 2) FO_CUDA(cudaStreamWaitEvent(ls, ctx->ev_hop[mod(r - 1, P)][t - 1], 0));
      if (t == 1) {
        FO_TRY(copy_rows(ag_slot(a, d, s, row0), a.K, bptr(a.X[r], row0), a.X[r].ld, rows, a.K, 2, ls));
      } else {
        FO_TRY(copy_rows(ag_slot(a, d, s, row0), a.K, ag_slot(a, r, s, row0), a.K, rows, a.K, 2, ls));
      }
      if (flags) FO_TRY(write_flag(ls, flag_base + kAgFlagBase + d * P + s, epoch));
      FO_CUDA(cudaEventRecord(ctx->ev_hop[r][t], ls));
    }
  }
  return FO_OK;
}

// Adds the P*P (rank, slice) GEMM units over rows [row0, row0 + rows) of every slice.
// gated_f > 0: W_col[r] is [2F, K] (gate rows then up rows) and Y[r] receives
// H = SiLU(gate) * up, [M, F] (the MLP glue fused into the epilogue).
// Tile order of a whole-slice launch (weight_major): step 0 (every rank's own slice,
// no wait) first; then, rank by rank, the received slices of steps 1..P-1 with the
// weight's n-block outermost, so that one weight tile serves all of a rank's received
// slices while it is in L2 (the ring delivers them while step 0 computes).  Otherwise
// (sub-slice launches of the data-slicing baseline): step by step, one group per step
// when flash.
constexpr double kWeightMajorMaxBytes = 80.0 * (1 << 20);  // measured: 56 MiB better, 112 MiB equal

// rows_base >= 0 (one launch for a whole layer): rank r's unit for slice s counts its stored
// rows per m-block into counter rows_base + (r * P + s) * mblocks + mb.
// step_pairs (whole-slice flash launches with 128-row slices, P even): one unit per two
// consecutive steps (t, t+1) of a rank, 256 rows of its step-ordered receive buffer (for
// steps 0 and 1 the first 128 rows are the rank's own shard, read in place), so the launch
// runs 256-row tiles on SM pairs: the first 128 rows (slice of step t) wait on that slice's
// flag and are stored at its output rows, the next 128 likewise for step t+1.
fo_status add_ag_step_pairs(Launch& L, const AgArgs& a, const int* xmap, const int* rmap, const int* wmap,
                            int64_t gated_f, bool weight_major) {
  const int P = a.P, npairs = P / 2;
  auto add = [&](int r, int j) {
    int r0, s0, r1, s1;
    ag_unit(P, 2 * j, r, &r0, &s0);
    ag_unit(P, 2 * j + 1, r, &r1, &s1);
    GemmUnit& u = L.add_unit();
    u = blank_unit();
    u.a_map = rmap[r];
    u.a_row0 = static_cast<int32_t>(2 * j * a.m);  // positions 2j and 2j+1
    if (j == 0) {  // step 0 is the rank's own slice: read in place, no copy into position 0
      u.a_map_lo = xmap[r];
      u.a_row_lo = 0;
    }
    u.wait_flag = static_cast<int32_t>(kAgFlagBase + r * P + s0);
    u.wait_flag2 = static_cast<int32_t>(kAgFlagBase + r * P + s1);
    u.b_map = wmap[r];
    u.m_rows = static_cast<int32_t>(2 * a.m);
    u.k = static_cast<int32_t>(a.K);
    if (gated_f > 0) {
      u.gated = 1;
      u.b_row1 = static_cast<int32_t>(gated_f);
      u.n_cols = static_cast<int32_t>(gated_f);
      u.epi = kEpiSiluMul;
    } else {
      u.n_cols = static_cast<int32_t>(a.N);
      u.epi = kEpiBF16;
    }
    u.c = bptr(a.Y[r], s0 * a.m);
    u.c2 = bptr(a.Y[r], s1 * a.m);
    u.ldc = a.Y[r].ld;
  };
  if (weight_major) {  // steps (0, 1) of every rank, then rank by rank its other pairs, weight-major
    L.begin_group();
    for (int r = 0; r < P; ++r) add(r, 0);
    for (int r = 0; r < P && npairs > 1; ++r) {
      L.begin_group(true);
      for (int j = 1; j < npairs; ++j) add(r, j);
    }
  } else {
    for (int j = 0; j < npairs; ++j) {
      L.begin_group();
      for (int r = 0; r < P; ++r) add(r, j);
    }
  }
  return FO_OK;
}

fo_status add_ag_units(Launch& L, const AgArgs& a, const int* xmap, const int* rmap, const int* wmap, int64_t row0,
                       int64_t rows, bool flash, int64_t gated_f, bool weight_major = false, int64_t rows_base = -1,
                       int64_t mblocks = 0) {
  const int P = a.P;
  const int ngroups = weight_major ? 1 + (P > 1 ? P : 0) : P;
  for (int gi = 0; gi < ngroups; ++gi) {
    const bool step0 = gi == 0;
    if (weight_major || flash || gi == 0) L.begin_group(weight_major && !step0);
    const int nunits = weight_major && !step0 ? P - 1 : P;
    for (int k = 0; k < nunits; ++k) {
      int r, s, t;
      if (weight_major && !step0) {
        t = k + 1;
        ag_unit(P, t, gi - 1, &r, &s);  // rank gi - 1, received slice of step t
      } else {
        t = weight_major ? 0 : gi;
        ag_unit(P, t, k, &r, &s);  // local slice first
      }
      GemmUnit& u = L.add_unit();
      u = blank_unit();
      if (t == 0) {
        u.a_map = xmap[r];
        u.a_row0 = static_cast<int32_t>(row0);
        if (flash && a.Xh) u.wait_flag = static_cast<int32_t>(kAgFlagBase + r * P + r);  // uploaded slice
      } else {
        u.a_map = rmap[r];
        u.a_row0 = static_cast<int32_t>(ag_position(a, r, s) * a.m + row0);
        if (flash) u.wait_flag = static_cast<int32_t>(kAgFlagBase + r * P + s);
      }
      u.b_map = wmap[r];
      u.m_rows = static_cast<int32_t>(rows);
      u.k = static_cast<int32_t>(a.K);
      if (gated_f > 0) {
        u.gated = 1;
        u.b_row1 = static_cast<int32_t>(gated_f);
        u.n_cols = static_cast<int32_t>(gated_f);
        u.epi = kEpiSiluMul;
      } else {
        u.n_cols = static_cast<int32_t>(a.N);
        u.epi = kEpiBF16;
      }
      u.c = bptr(a.Y[r], s * a.m + row0);
      u.ldc = a.Y[r].ld;
      if (rows_base >= 0) u.rows_done_base = static_cast<int32_t>(rows_base + (static_cast<int64_t>(r) * P + s) * mblocks);
    }
  }
  return FO_OK;
}

// w_kn: W[r] is given as [K, N] (read MN-major by the MMA; not with `gated`).
fo_status ag_run(fo_ctx* ctx, const fo_mat* X, const fo_mat* W, int P, const fo_mat* Y, const fo_opts& o,
                 cudaStream_t stream, bool gated = false, bool w_kn = false, const fo_mat* Xh = nullptr) {
  const int64_t m = X[0].rows, K = X[0].cols, N = w_kn ? W[0].cols : W[0].rows, M = m * P;
  const int64_t gated_f = gated ? N / 2 : 0;
  if (gated && N % 2 != 0) return fail(FO_ERR_SHAPE, "gated weight must have 2F rows");
  if (gated && w_kn) return fail(FO_ERR_UNSUPPORTED, "gated projection with a transposed weight");
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(X[r], FO_BF16, "X_shards", r));
    FO_TRY(check_mat(W[r], FO_BF16, "W_col", r));
    FO_TRY(check_mat(Y[r], FO_BF16, "Y", r));
    if (X[r].rows != m || X[r].cols != K) return fail(FO_ERR_SHAPE, "X_shards[%d] shape differs from rank 0", r);
    if ((w_kn ? W[r].cols : W[r].rows) != N || (w_kn ? W[r].rows : W[r].cols) != K)
      return fail(FO_ERR_SHAPE, "W_col[%d] must be %s like rank 0", r, w_kn ? "[K, N]" : "[N, K]");
    if (Y[r].rows != M || Y[r].cols != (gated ? gated_f : N))
      return fail(FO_ERR_SHAPE, "Y[%d] must be [P*m, %s]", r, gated ? "F" : "N");
  }
  if (K % 8 != 0) return fail(FO_ERR_UNSUPPORTED, "K=%lld must be a multiple of 8", (long long)K);
  if (m == 0 || N == 0) return FO_OK;
  if (K == 0) return fail(FO_ERR_UNSUPPORTED, "K == 0");
  void* flags_v = nullptr;
  void* recv_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &flags_v));
  FO_TRY(ensure_buf(ctx, kBufAgRecv, static_cast<size_t>(P) * M * K * 2, &recv_v));
  uint32_t* flags = static_cast<uint32_t*>(flags_v);
  AgArgs a{X, W, Y, P, m, K, N, static_cast<char*>(recv_v), w_kn, nullptr};
  const bool flash = o.order == FO_ORDER_FLASH || o.order == FO_ORDER_NAIVE;
  if (Xh) {
    if (flash) {
      a.Xh = Xh;
    } else {  // the baselines upload everything first
      for (int r = 0; r < P; ++r)
        FO_CUDA(cudaMemcpy2DAsync(X[r].ptr, X[r].ld * 2, Xh[r].ptr, Xh[r].ld * 2, K * 2, m, cudaMemcpyHostToDevice,
                                  stream));
    }
  }
  const uint32_t epoch = ++ctx->epoch;
  const uint64_t tmo = timeout_ns(o);

  fo_status st = FO_OK;
  // 128-row slices in a whole-slice fused launch: two steps per 256-row tile on SM pairs
  const bool step_pairs = (o.order == FO_ORDER_FLASH || o.order == FO_ORDER_NAIVE) && m == kBM && P % 2 == 0 &&
                          o.sm_pairs != 1 && ctx->pair_clusters > 0;
  auto build = [&](Launch& L, int64_t row0, int64_t rows, bool flash, int* xmap, int* rmap, int* wmap,
                   bool weight_major) -> fo_status {
    for (int r = 0; r < P; ++r) {
      xmap[r] = L.add_map(&st, X[r].ptr, m, K, X[r].ld, kBM);
      if (st != FO_OK) return st;
      rmap[r] = L.add_map(&st, ag_rank_buffer(a, r), M, K, K, kBM);
      if (st != FO_OK) return st;
      wmap[r] = w_kn ? L.add_map_mn(&st, W[r].ptr, K, N, W[r].ld)
                     : L.add_map(&st, W[r].ptr, N, K, W[r].ld, gated ? kBN / 2 : kBN);
      if (st != FO_OK) return st;
    }
    if (flash && step_pairs && row0 == 0 && rows == m) {
      FO_TRY(add_ag_step_pairs(L, a, xmap, rmap, wmap, gated_f, weight_major));
    } else {
      FO_TRY(add_ag_units(L, a, xmap, rmap, wmap, row0, rows, flash, gated_f, weight_major));
    }
    L.p.mn_major = w_kn ? 2 : 0;
    return L.finish(epoch, tmo, flags, ctx->ctrl, 0);
  };
  int xmap[kMaxP], rmap[kMaxP], wmap[kMaxP];
  // The weight-major order pays off while one rank's received slices stay in L2
  // across its weight tiles; with larger slices the step order (each step's
  // slices reused across all weight tiles) moves fewer bytes.
  const bool weight_major = static_cast<double>(P - 1) * m * K * 2 <= kWeightMajorMaxBytes;

  const bool compute_only = o.compute_only != 0;
  if (compute_only && a.Xh) return fail(FO_ERR_UNSUPPORTED, "compute_only is a device-buffer timing mode");
  if (o.order == FO_ORDER_FLASH || o.order == FO_ORDER_NAIVE) {
    Launch L;
    FO_TRY(build(L, 0, m, true, xmap, rmap, wmap, weight_major));
    if (compute_only) {  // the same launch with every arrival flag already published
      FO_CUDA(launch_fill_u32(flags + kAgFlagBase, static_cast<int64_t>(P) * P, epoch, stream));
      return launch_gemm(ctx, L, o, stream);
    }
    // the ring's copies run concurrently with the persistent GEMM that waits on them (host
    // order: copies_first)
    FO_TRY(fork_links(ctx, P, stream));
    if (!copies_first()) FO_TRY(launch_gemm(ctx, L, o, stream));
    if (a.Xh || step_pairs) FO_TRY(enqueue_uploads(ctx, a, epoch, flags));
    FO_TRY(enqueue_ag_ring(ctx, a, 0, m, true, epoch, o.fault, flags));
    if (copies_first()) FO_TRY(launch_gemm(ctx, L, o, stream));
    return join_links(ctx, P, stream);
  }
  if (o.order == FO_ORDER_SERIAL) {
    Launch L;
    FO_TRY(build(L, 0, m, false, xmap, rmap, wmap, weight_major));
    if (compute_only) return launch_gemm(ctx, L, o, stream);
    FO_CUDA(cudaEventRecord(ctx->ev_phase[0], stream));
    FO_TRY(fork_links(ctx, P, stream));
    FO_TRY(enqueue_ag_ring(ctx, a, 0, m, false, epoch, FO_FAULT_NONE, flags));
    FO_TRY(join_links(ctx, P, stream));
    FO_CUDA(cudaEventRecord(ctx->ev_phase[1], stream));
    FO_TRY(launch_gemm(ctx, L, o, stream));
    FO_CUDA(cudaEventRecord(ctx->ev_phase[2], stream));
    ctx->phase_valid = true;
    ctx->phase_gemm_first = false;
    return FO_OK;
  }
  // FO_ORDER_SLICING: all-gather of sub-slice i, then one GEMM launch over sub-slice i
  const int n = o.n_slices ? o.n_slices : P;
  if (m % n != 0) return fail(FO_ERR_SHAPE, "slice rows m=%lld not divisible by n_slices=%d", (long long)m, n);
  const int64_t sub = m / n;
  if (compute_only) {  // the per-slice launches alone
    for (int i = 0; i < n; ++i) {
      Launch L;
      FO_TRY(build(L, i * sub, sub, false, xmap, rmap, wmap, false));
      FO_TRY(launch_gemm(ctx, L, o, stream));
    }
    return FO_OK;
  }
  FO_TRY(fork_links(ctx, P, stream));
  for (int i = 0; i < n; ++i) {
    FO_TRY(enqueue_ag_ring(ctx, a, i * sub, sub, false, epoch, FO_FAULT_NONE, flags));
    for (int r = 0; r < P; ++r) FO_CUDA(cudaEventRecord(ctx->ev_slice[i][r], ctx->link[r]));
  }
  for (int i = 0; i < n; ++i) {
    Launch L;
    FO_TRY(build(L, i * sub, sub, false, xmap, rmap, wmap, false));
    for (int r = 0; r < P; ++r) FO_CUDA(cudaStreamWaitEvent(stream, ctx->ev_slice[i][r], 0));
    FO_TRY(launch_gemm(ctx, L, o, stream));
  }
  return join_links(ctx, P, stream);
}

// --------------------------------------------------------------------------
// Flash-RS and its baselines
// --------------------------------------------------------------------------

struct RsArgs {
  const fo_mat* X;
  const fo_mat* W;
  const fo_mat* Y;
  int P;
  int64_t M, m, Kr, N;
  float* recv;  // rank r's receive slot for hop h: recv + ((r*P + h)*m)*N
  float* part;  // baselines: partial of rank r for chunk c: part + ((r*P + c)*m)*N
  bool w_kn;    // W[r] given as [Kr, N] (the transposed weight of a backward pass)
};

int add_rs_weight(Launch& L, fo_status* st, const RsArgs& a, int r) {
  return a.w_kn ? L.add_map_mn(st, a.W[r].ptr, a.Kr, a.N, a.W[r].ld)
                : L.add_map(st, a.W[r].ptr, a.N, a.Kr, a.W[r].ld, kBN);
}

// Completion of each rank's kept chunk in the fused reduce-scatter, for copies that wait
// on it (the host-buffer layer's copies back): the kept chunk's tiles count into
// flags[kDoneBase + r], and after the launch the stream writes every target, so a
// waiter is released even if the kernel gave up early.
struct DoneSignal {
  bool set = false;            // filled in by the flash launch
  uint32_t target[kMaxP] = {};
};

float* rs_slot(const RsArgs& a, float* base, int r, int h) {
  return base + (static_cast<int64_t>(r) * a.P + h) * a.m * a.N;
}

constexpr double kStreamPartialsBytes = 96.0 * (1 << 20);  // L2 is 126 MB
constexpr int kTnFbGroup = 32;  // feature blocks per ordering group of the transposed tiles (measured: 2..32)
// Ring steps per tile-order group of the step-ordered Flash-RS (measured 1, 2, 4, 8: every
// grouping beat one step per group; 2: 16K layer 2.2-2.4% and 4K layer ~3% faster than 1)
constexpr int kRsStepGroup = 2;

// Transposed reduce-scatter tiles (GemmParams::tn_S) for a slice of m rows: 0 if they do
// not apply, else the number of ring steps per tile, with *pair set when the tiles run on
// SM pairs (only on request, fo_opts.sm_pairs == 2: the single-SM form was measured faster,
// tail GEMM-RS 0.263-0.269 vs 0.274-0.281 ms, 1K sweep point 0.446-0.449 vs 0.455-0.457
// ms).  A tile waits on the tile of the previous rank in its pass group, which may
// come later in the tile order (the ring closes from the last rank to the first), so every
// rank's tile of a pass group must run at once: the grid must hold at least P tiles.
int rs_tn_steps(const fo_ctx* ctx, const RsArgs& a, const fo_opts& o, bool* pair) {
  const int P = a.P;
  if (a.w_kn || a.m <= 0 || a.m > kBM || a.m % 32 != 0 || 256 % a.m != 0) return 0;
  const int S = static_cast<int>(256 / a.m);
  if (S > P || P % S != 0) return 0;
  *pair = o.sm_pairs == 2 && ctx->pair_clusters > 0 && pair_grid(ctx, o) >= P;
  if (*pair) return S;
  return grid_size(ctx, o, 1 << 30) >= P ? S : 0;
}

// Appends the maps and units of a fused reduce-scatter (order FO_ORDER_FLASH or
// FO_ORDER_NAIVE) to L.  S > 0: transposed tiles (rs_tn_steps), which take the whole launch;
// otherwise step-ordered tiles, in groups of kRsStepGroup ring steps (Flash order) or one
// group per ring step (naive order).  `done`: the kept chunk's tiles count into the per-rank
// completion counters.  ready_base >= 0 (one launch for a whole layer): rank r's unit for
// chunk c waits, per m-block, until counter ready_base + (r * P + c) * mblocks + mb reaches
// ready_count (the epilogue warps of the tiles that wrote those rows of X[r]).
// *flag_end receives the end of the flag range the units use.
fo_status build_rs_flash(fo_ctx* ctx, Launch& L, const RsArgs& a, const fo_opts& o, uint32_t* flags, uint32_t epoch,
                         bool done, int S, bool tn_pair, int64_t* flag_end, int64_t ready_base = -1,
                         int64_t mblocks = 0, int ready_count = 0) {
  const int P = a.P;
  fo_status st = FO_OK;
  int xmap[kMaxP], wmap[kMaxP];
  for (int r = 0; r < P; ++r) {
    // transposed tiles: the tokens are the MMA's N side (one box of m rows per step) and
    // the weight its M side (128-row boxes)
    xmap[r] = L.add_map(&st, a.X[r].ptr, a.M, a.Kr, a.X[r].ld, S ? static_cast<int>(a.m) : kBM);
    if (st != FO_OK) return st;
    wmap[r] = S ? L.add_map(&st, a.W[r].ptr, a.N, a.Kr, a.W[r].ld, kBM) : add_rs_weight(L, &st, a, r);
    if (st != FO_OK) return st;
  }
  // one ring step's partial sums beyond kStreamPartialsBytes: stream them past L2
  L.p.stream_partials = static_cast<double>(P) * a.m * a.N * 4 > kStreamPartialsBytes ? 1 : 0;
  const int64_t tm = (a.m + kBM - 1) / kBM, tn = (a.N + kBN - 1) / kBN;
  // flags per (rank, hop): one per (tile, quadrant), or per (256-feature block, CTA half,
  // quadrant) for transposed tiles
  const int64_t per_hop = tm * tn * 4 > ((a.N + 255) / 256) * 8 ? tm * tn * 4 : ((a.N + 255) / 256) * 8;
  auto fbase = [&](int r, int h) { return kRsFlagBase + (static_cast<int64_t>(r) * P + h) * per_hop; };
  if (fbase(P - 1, P) > (1 << 18)) return fail(FO_ERR_UNSUPPORTED, "too many reduce-scatter tiles for the flag area");
  *flag_end = fbase(P - 1, P);
  auto add = [&](int r, int c) {
    const int h = mod(r - c - 1, P);  // position of rank r on chunk c's reduction chain
    GemmUnit& u = L.add_unit();
    u = blank_unit();
    if (S) {  // A = the weight's features, B = the chunk's token rows
      u.a_map = wmap[r];
      u.b_map = xmap[r];
      u.b_row0 = static_cast<int32_t>(c * a.m);
    } else {
      u.a_map = xmap[r];
      u.a_row0 = static_cast<int32_t>(c * a.m);
      u.b_map = wmap[r];
    }
    u.m_rows = static_cast<int32_t>(a.m);
    u.n_cols = static_cast<int32_t>(a.N);
    u.k = static_cast<int32_t>(a.Kr);
    if (ready_base >= 0) {
      u.a_ready_base = static_cast<int32_t>(ready_base + (static_cast<int64_t>(r) * P + c) * mblocks);
      u.a_ready_count = ready_count;
    }
    if (h > 0) {
      u.acc_in = rs_slot(a, a.recv, r, h);
      u.ld_acc = a.N;
      u.in_flag_base = static_cast<int32_t>(fbase(r, h));
    }
    if (h < P - 1) {
      const int d = mod(r + 1, P);
      u.c = rs_slot(a, a.recv, d, h + 1);
      u.ldc = a.N;
      u.out_flag_base = static_cast<int32_t>(fbase(d, h + 1));
      u.epi = h == 0 ? kEpiF32 : kEpiAddF32;
    } else {
      u.c = a.Y[r].ptr;
      u.ldc = a.Y[r].ld;
      u.epi = h == 0 ? kEpiBF16 : kEpiAddBF16;
      if (done) u.done_counter = static_cast<int32_t>(kDoneBase + r);
    }
  };
  if (S) {
    // units rank-major in step order: rank r computes at step t the chunk of rs_unit's order
    for (int r = 0; r < P; ++r)
      for (int t = 0; t < P; ++t) add(r, o.order == FO_ORDER_NAIVE ? t : mod(r - t - 1, P));
    const int ncta = tn_pair ? 2 : 1;
    GemmParams& q = L.p;
    q.num_groups = 1;
    q.group_unit_begin[0] = 0;
    q.group_unit_begin[1] = L.num_units;
    q.num_maps = L.num_maps;
    q.tn_S = S;
    q.tn_rows = static_cast<int32_t>(a.m);
    q.tn_ranks = P;
    q.tn_passes = P / S;
    q.tn_fblocks = static_cast<int32_t>((a.N + ncta * kBM - 1) / (ncta * kBM));
    // passes of one feature block kTnFbGroup blocks apart (a divisor of the block count)
    int fbg = kTnFbGroup < q.tn_fblocks ? kTnFbGroup : q.tn_fblocks;
    while (q.tn_fblocks % fbg != 0) --fbg;
    q.tn_fb_group = fbg;
    q.total_tiles = q.tn_fblocks * q.tn_passes * P;
    q.epoch = epoch;
    q.timeout_ns = timeout_ns(o);
    q.flags = flags;
    q.flag_words = static_cast<int32_t>(kFlagBytes / 4);
    q.ctrl = ctx->ctrl;
    q.rows_all_index = -1;
    L.tn_pair = tn_pair;
    L.arrivals_per_tile = 4 * ncta;
    for (int i = 0; i < L.num_units; ++i) {  // per unit: one feature block of tiles
      q.units[i].tiles_m = 1;
      q.units[i].tiles_n = q.tn_fblocks;
    }
  } else {
    if (o.order == FO_ORDER_FLASH) {
      // Groups of kRsStepGroup ring steps.  Inside a group each rank's units follow one
      // another (the weight it streams is read for the group's steps in close succession,
      // and a step's partial sums are read about one unit after they are written instead
      // of a whole step later); a unit whose producer (rank r-1, previous step) is not yet
      // placed is preceded by that producer's chain, so every unit waits only on units
      // earlier in the tile order.  The ranks' computations and the order of additions on
      // each chunk are those of the step schedule (rs_unit): only the tile order changes.
      for (int t0 = 0; t0 < P; t0 += kRsStepGroup) {
        const int gs = kRsStepGroup < P - t0 ? kRsStepGroup : P - t0;
        L.begin_group();
        bool placed[kMaxP][kRsStepGroup] = {};
        auto emit = [&](auto&& self, int r, int k) -> void {
          if (placed[r][k]) return;
          if (k > 0) self(self, mod(r - 1, P), k - 1);
          add(r, mod(r - (t0 + k) - 1, P));  // rank r at step t0 + k: chunk (r - t - 1) mod P
          placed[r][k] = true;
        };
        for (int r = 0; r < P; ++r)
          for (int k = 0; k < gs; ++k) emit(emit, r, k);
      }
    } else {
      for (int t = 0; t < P; ++t) {
        L.begin_group();
        for (int i = 0; i < P; ++i) {
          int r, c;
          rs_unit(P, o.order, t, i, &r, &c);
          add(r, c);
        }
      }
    }
    L.p.mn_major = a.w_kn ? 2 : 0;
  }
  return FO_OK;
}

// After the launch: the stream writes every kept-chunk completion counter's final value, so
// copies that wait on them are released even if the kernel gave up early.
fo_status publish_done(fo_ctx* ctx, const Launch& L, uint32_t* flags, cudaStream_t stream, DoneSignal* done) {
  for (int i = 0; i < L.num_units; ++i) {
    const GemmUnit& u = L.p.units[i];
    if (u.done_counter < 0) continue;
    const int r = static_cast<int>(u.done_counter - kDoneBase);
    const uint32_t n = static_cast<uint32_t>(u.tiles_m * u.tiles_n * L.arrivals_per_tile);
    ctx->done_total[r] += n;
    done->target[r] = ctx->done_total[r];
    FO_TRY(write_flag(stream, flags + kDoneBase + r, done->target[r]));
  }
  done->set = true;
  return FO_OK;
}

fo_status rs_flash(fo_ctx* ctx, const RsArgs& a, const fo_opts& o, cudaStream_t stream, uint32_t* flags,
                   uint32_t epoch, DoneSignal* done = nullptr) {
  Launch L;
  bool tn_pair = false;
  const int S = rs_tn_steps(ctx, a, o, &tn_pair);
  int64_t flag_end = 0;
  FO_TRY(build_rs_flash(ctx, L, a, o, flags, epoch, done != nullptr, S, tn_pair, &flag_end));
  if (!S) FO_TRY(L.finish(epoch, timeout_ns(o), flags, ctx->ctrl, 0));
  if (o.compute_only)  // every partial-sum flag published: no tile waits on another
    FO_CUDA(launch_fill_u32(flags + kRsFlagBase, flag_end - kRsFlagBase, epoch, stream));
  FO_TRY(launch_gemm(ctx, L, o, stream));
  if (done) FO_TRY(publish_done(ctx, L, flags, stream, done));
  return FO_OK;
}

// Baselines: partial GEMMs into `part`, then a ring reduce with device-to-device hops
// and fp32 add kernels.  Rows [row0, row0 + rows) of every chunk.
fo_status rs_partials(fo_ctx* ctx, const RsArgs& a, const fo_opts& o, cudaStream_t stream, int64_t row0,
                      int64_t rows, uint32_t* flags, uint32_t epoch) {
  const int P = a.P;
  Launch L;
  fo_status st = FO_OK;
  int xmap[kMaxP], wmap[kMaxP];
  for (int r = 0; r < P; ++r) {
    xmap[r] = L.add_map(&st, a.X[r].ptr, a.M, a.Kr, a.X[r].ld, kBM);
    if (st != FO_OK) return st;
    wmap[r] = add_rs_weight(L, &st, a, r);
    if (st != FO_OK) return st;
  }
  L.begin_group();
  for (int r = 0; r < P; ++r) {
    for (int c = 0; c < P; ++c) {
      GemmUnit& u = L.add_unit();
      u = blank_unit();
      u.a_map = xmap[r];
      u.a_row0 = static_cast<int32_t>(c * a.m + row0);
      u.b_map = wmap[r];
      u.m_rows = static_cast<int32_t>(rows);
      u.n_cols = static_cast<int32_t>(a.N);
      u.k = static_cast<int32_t>(a.Kr);
      u.epi = kEpiF32;
      u.c = rs_slot(a, a.part, r, c) + row0 * a.N;
      u.ldc = a.N;
    }
  }
  L.p.mn_major = a.w_kn ? 2 : 0;
  FO_TRY(L.finish(epoch, timeout_ns(o), flags, ctx->ctrl, 0));
  return launch_gemm(ctx, L, o, stream);
}

// Ring reduce of rows [row0, row0 + rows) of every chunk, issued on `rs` (adds)
// and the link streams (hops).  Hop h: rank c+h sends its running sum of chunk c
// to rank c+h+1, which adds its own partial (in place) or, at the owner, rounds
// the final sum into Y[c].  copies == false: the adds alone (compute-only timing).
fo_status rs_ring_reduce(fo_ctx* ctx, const RsArgs& a, cudaStream_t rs, int64_t row0, int64_t rows,
                         bool copies = true) {
  const int P = a.P;  // P >= 2 (a single rank takes the fused path)
  for (int h = 1; h < P; ++h) {
    if (copies) {
      FO_TRY(fork_links(ctx, P, rs));
      for (int c = 0; c < P; ++c) {
        const int s = mod(c + h, P), d = mod(c + h + 1, P);
        FO_TRY(copy_rows(rs_slot(a, a.recv, d, h) + row0 * a.N, a.N, rs_slot(a, a.part, s, c) + row0 * a.N, a.N,
                         rows, a.N, 4, ctx->link[s]));
      }
      FO_TRY(join_links(ctx, P, rs));
    }
    for (int c = 0; c < P; ++c) {
      const int d = mod(c + h + 1, P);
      float* mine = rs_slot(a, a.part, d, c) + row0 * a.N;
      const float* in = rs_slot(a, a.recv, d, h) + row0 * a.N;
      if (h < P - 1) {
        FO_CUDA(launch_add_f32(mine, a.N, in, a.N, mine, nullptr, a.N, rows, a.N, rs));
      } else {
        FO_CUDA(launch_add_f32(mine, a.N, in, a.N, nullptr, reinterpret_cast<uint16_t*>(bptr(a.Y[d], row0)),
                               a.Y[d].ld, rows, a.N, rs));
      }
    }
  }
  return FO_OK;
}

// w_kn: W[r] is given as [Kr, N] (read MN-major by the MMA).  done: see DoneSignal (fused
// order only; left unset otherwise).
fo_status rs_run(fo_ctx* ctx, const fo_mat* X, const fo_mat* W, int P, const fo_mat* Y, const fo_opts& o,
                 cudaStream_t stream, bool w_kn = false, DoneSignal* done = nullptr) {
  const int64_t M = X[0].rows, Kr = X[0].cols, N = w_kn ? W[0].cols : W[0].rows;
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(X[r], FO_BF16, "X", r));
    FO_TRY(check_mat(W[r], FO_BF16, "W_row", r));
    FO_TRY(check_mat(Y[r], FO_BF16, "Y", r));
    if (X[r].rows != M || X[r].cols != Kr) return fail(FO_ERR_SHAPE, "X[%d] shape differs from rank 0", r);
    if ((w_kn ? W[r].cols : W[r].rows) != N || (w_kn ? W[r].rows : W[r].cols) != Kr)
      return fail(FO_ERR_SHAPE, "W_row[%d] must be %s like rank 0", r, w_kn ? "[Kr, N]" : "[N, Kr]");
  }
  if (M % P != 0) return fail(FO_ERR_SHAPE, "M=%lld not divisible by P=%d", (long long)M, P);
  const int64_t m = M / P;
  for (int r = 0; r < P; ++r)
    if (Y[r].rows != m || Y[r].cols != N) return fail(FO_ERR_SHAPE, "Y[%d] must be [M/P, N]", r);
  if (Kr % 8 != 0) return fail(FO_ERR_UNSUPPORTED, "Kr=%lld must be a multiple of 8", (long long)Kr);
  if (N % 4 != 0) return fail(FO_ERR_UNSUPPORTED, "N=%lld must be a multiple of 4", (long long)N);
  if (m == 0 || N == 0) return FO_OK;
  if (Kr == 0) return fail(FO_ERR_UNSUPPORTED, "Kr == 0");
  void *flags_v = nullptr, *recv_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &flags_v));
  FO_TRY(ensure_buf(ctx, kBufRsRecv, static_cast<size_t>(P) * P * m * N * 4, &recv_v));
  RsArgs a{X, W, Y, P, M, m, Kr, N, static_cast<float*>(recv_v), nullptr, w_kn};
  uint32_t* flags = static_cast<uint32_t*>(flags_v);
  const uint32_t epoch = ++ctx->epoch;
  if (o.order == FO_ORDER_FLASH || o.order == FO_ORDER_NAIVE || P == 1) {
    if (o.link == FO_LINK_CE)
      return fail(FO_ERR_UNSUPPORTED, "fused reduce-scatter hops are epilogue pushes (FO_LINK_PUSH)");
    return rs_flash(ctx, a, o, stream, flags, epoch, done);
  }
  void* part_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufPart, static_cast<size_t>(P) * P * m * N * 4, &part_v));
  a.part = static_cast<float*>(part_v);
  if (o.compute_only) {  // the baselines' partial GEMMs and adds, no copies
    const int n = o.order == FO_ORDER_SLICING ? (o.n_slices ? o.n_slices : P) : 1;
    if (m % n != 0) return fail(FO_ERR_SHAPE, "slice rows m=%lld not divisible by n_slices=%d", (long long)m, n);
    for (int i = 0; i < n; ++i) {
      FO_TRY(rs_partials(ctx, a, o, stream, i * (m / n), m / n, flags, epoch));
      FO_TRY(rs_ring_reduce(ctx, a, stream, i * (m / n), m / n, false));
    }
    return FO_OK;
  }
  if (o.order == FO_ORDER_SERIAL) {
    FO_CUDA(cudaEventRecord(ctx->ev_phase[0], stream));
    FO_TRY(rs_partials(ctx, a, o, stream, 0, m, flags, epoch));
    FO_CUDA(cudaEventRecord(ctx->ev_phase[1], stream));
    FO_TRY(rs_ring_reduce(ctx, a, stream, 0, m));
    FO_CUDA(cudaEventRecord(ctx->ev_phase[2], stream));
    ctx->phase_valid = true;
    ctx->phase_gemm_first = true;
    return FO_OK;
  }
  // FO_ORDER_SLICING: partial GEMM of sub-slice i (main stream), its ring reduce on the aux stream
  const int n = o.n_slices ? o.n_slices : P;
  if (m % n != 0) return fail(FO_ERR_SHAPE, "slice rows m=%lld not divisible by n_slices=%d", (long long)m, n);
  const int64_t sub = m / n;
  for (int i = 0; i < n; ++i) {
    FO_TRY(rs_partials(ctx, a, o, stream, i * sub, sub, flags, epoch));
    FO_CUDA(cudaEventRecord(ctx->ev_aux, stream));
    FO_CUDA(cudaStreamWaitEvent(ctx->aux, ctx->ev_aux, 0));
    FO_TRY(rs_ring_reduce(ctx, a, ctx->aux, i * sub, sub));
  }
  FO_CUDA(cudaEventRecord(ctx->ev_aux, ctx->aux));
  FO_CUDA(cudaStreamWaitEvent(stream, ctx->ev_aux, 0));
  return FO_OK;
}

// --------------------------------------------------------------------------
// Flash all-to-all (Ulysses parallelism): GEMM -> A2A and A2A -> GEMM
// --------------------------------------------------------------------------

// Y_d[rows r*m..] = X_r W_r[rows d*Nb..]^T: rank r's output block d belongs to rank d.
// Flash / naive: one persistent launch; each unit's epilogue stores its tiles straight
// into the destination's buffer (the hop of this all-to-all is the epilogue store), in
// the step order of a2a_block_unit.  Serial baseline: the GEMM into a local buffer, then
// the all-to-all as P*P copies.
fo_status gemm_a2a_run(fo_ctx* ctx, const fo_mat* X, const fo_mat* W, int P, const fo_mat* Y, const fo_opts& o,
                       cudaStream_t stream) {
  const int64_t m = X[0].rows, K = X[0].cols, N = W[0].rows, M = m * P;
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(X[r], FO_BF16, "X_shards", r));
    FO_TRY(check_mat(W[r], FO_BF16, "W", r));
    FO_TRY(check_mat(Y[r], FO_BF16, "Y", r));
    if (X[r].rows != m || X[r].cols != K) return fail(FO_ERR_SHAPE, "X_shards[%d] shape differs from rank 0", r);
    if (W[r].rows != N || W[r].cols != K) return fail(FO_ERR_SHAPE, "W[%d] must be [N, K] like rank 0", r);
  }
  if (N % P != 0) return fail(FO_ERR_SHAPE, "N=%lld not divisible by P=%d", (long long)N, P);
  const int64_t Nb = N / P;
  for (int d = 0; d < P; ++d)
    if (Y[d].rows != M || Y[d].cols != Nb) return fail(FO_ERR_SHAPE, "Y[%d] must be [P*m, N/P]", d);
  if (K % 8 != 0) return fail(FO_ERR_UNSUPPORTED, "K=%lld must be a multiple of 8", (long long)K);
  if (o.order == FO_ORDER_SLICING) return fail(FO_ERR_UNSUPPORTED, "no data-slicing baseline for the all-to-all");
  if (m == 0 || Nb == 0) return FO_OK;
  if (K == 0) return fail(FO_ERR_UNSUPPORTED, "K == 0");
  void* flags_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &flags_v));
  const uint32_t epoch = ++ctx->epoch;
  const bool serial = o.order == FO_ORDER_SERIAL;
  char* local = nullptr;
  if (serial) {
    void* v = nullptr;
    FO_TRY(ensure_buf(ctx, kBufA2aLocal, static_cast<size_t>(P) * m * N * 2, &v));
    local = static_cast<char*>(v);
  }
  auto local_rank = [&](int r) { return local + static_cast<int64_t>(r) * m * N * 2; };
  fo_status st = FO_OK;
  Launch L;
  int xmap[kMaxP], wmap[kMaxP];
  for (int r = 0; r < P; ++r) {
    xmap[r] = L.add_map(&st, X[r].ptr, m, K, X[r].ld, kBM);
    if (st != FO_OK) return st;
    wmap[r] = L.add_map(&st, W[r].ptr, N, K, W[r].ld, kBN);
    if (st != FO_OK) return st;
  }
  for (int t = 0; t < (serial ? 1 : P); ++t) {
    L.begin_group();
    for (int i = 0; i < P; ++i) {
      int r, d;
      a2a_block_unit(P, o.order, t, i, &r, &d);
      GemmUnit& u = L.add_unit();
      u = blank_unit();
      u.a_map = xmap[r];
      u.b_map = wmap[r];
      u.m_rows = static_cast<int32_t>(m);
      u.k = static_cast<int32_t>(K);
      u.epi = kEpiBF16;
      if (serial) {  // the whole local output, all blocks
        u.b_row0 = 0;
        u.n_cols = static_cast<int32_t>(N);
        u.c = local_rank(r);
        u.ldc = N;
      } else {
        u.b_row0 = static_cast<int32_t>(d * Nb);
        u.n_cols = static_cast<int32_t>(Nb);
        u.c = bptr(Y[d], r * m);
        u.ldc = Y[d].ld;
      }
    }
  }
  FO_TRY(L.finish(epoch, timeout_ns(o), static_cast<uint32_t*>(flags_v), ctx->ctrl, 0));
  if (!serial) return launch_gemm(ctx, L, o, stream);
  FO_CUDA(cudaEventRecord(ctx->ev_phase[0], stream));
  FO_TRY(launch_gemm(ctx, L, o, stream));
  FO_CUDA(cudaEventRecord(ctx->ev_phase[1], stream));
  FO_TRY(fork_links(ctx, P, stream));
  for (int t = 0; t < P; ++t) {
    for (int r = 0; r < P; ++r) {
      const int d = mod(r + t, P);  // t = 0: the own block, a local move
      FO_TRY(copy_rows(bptr(Y[d], r * m), Y[d].ld, local_rank(r) + d * Nb * 2, N, m, Nb, 2, ctx->link[r]));
    }
  }
  FO_TRY(join_links(ctx, P, stream));
  FO_CUDA(cudaEventRecord(ctx->ev_phase[2], stream));
  ctx->phase_valid = true;
  ctx->phase_gemm_first = true;
  return FO_OK;
}

// Y_d = [C_0 rows d*m.. | C_1 rows d*m.. | ... ] W_d^T: every source s holds, in rows
// d*m.. of C_s, a K chunk of destination d's operand.  Hops: at step t source s copies its
// block for destination (s + t) mod P into that rank's receive slot and publishes a
// flag; the K-chunked GEMM folds in the own chunk first and each received chunk after its
// flag (a2a_source_unit order).  Serial baseline: every copy first, then the GEMM.
fo_status a2a_gemm_run(fo_ctx* ctx, const fo_mat* C, const fo_mat* W, int P, const fo_mat* Y, const fo_opts& o,
                       cudaStream_t stream) {
  const int64_t Mr = C[0].rows, Kc = C[0].cols, N = W[0].rows;
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(C[r], FO_BF16, "C", r));
    FO_TRY(check_mat(W[r], FO_BF16, "W", r));
    FO_TRY(check_mat(Y[r], FO_BF16, "Y", r));
    if (C[r].rows != Mr || C[r].cols != Kc) return fail(FO_ERR_SHAPE, "C[%d] shape differs from rank 0", r);
    if (W[r].rows != N || W[r].cols != P * Kc) return fail(FO_ERR_SHAPE, "W[%d] must be [N, P*Kc]", r);
  }
  if (Mr % P != 0) return fail(FO_ERR_SHAPE, "C rows=%lld not divisible by P=%d", (long long)Mr, P);
  const int64_t m = Mr / P;
  for (int d = 0; d < P; ++d)
    if (Y[d].rows != m || Y[d].cols != N) return fail(FO_ERR_SHAPE, "Y[%d] must be [rows/P, N]", d);
  if (Kc % kBK != 0) return fail(FO_ERR_UNSUPPORTED, "Kc=%lld must be a multiple of %d", (long long)Kc, kBK);
  if (o.order == FO_ORDER_SLICING) return fail(FO_ERR_UNSUPPORTED, "no data-slicing baseline for the all-to-all");
  if (m == 0 || N == 0) return FO_OK;
  if (Kc == 0) return fail(FO_ERR_UNSUPPORTED, "Kc == 0");
  void *flags_v = nullptr, *recv_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &flags_v));
  FO_TRY(ensure_buf(ctx, kBufA2aRecv, static_cast<size_t>(P) * Mr * Kc * 2, &recv_v));
  uint32_t* flags = static_cast<uint32_t*>(flags_v);
  auto recv = [&](int d) { return static_cast<char*>(recv_v) + static_cast<int64_t>(d) * Mr * Kc * 2; };
  const uint32_t epoch = ++ctx->epoch;
  const bool serial = o.order == FO_ORDER_SERIAL;
  fo_status st = FO_OK;
  Launch L;
  L.begin_group();
  for (int d = 0; d < P; ++d) {
    const int cmap = L.add_map(&st, C[d].ptr, Mr, Kc, C[d].ld, kBM);
    if (st != FO_OK) return st;
    const int rmap = L.add_map(&st, recv(d), Mr, Kc, Kc, kBM);
    if (st != FO_OK) return st;
    const int wmap = L.add_map(&st, W[d].ptr, N, P * Kc, W[d].ld, kBN);
    if (st != FO_OK) return st;
    GemmUnit& u = L.add_unit();
    u = blank_unit();
    u.a_map = cmap;
    u.a_row0 = static_cast<int32_t>(d * m);
    u.a_map2 = rmap;
    u.a2_row_stride = static_cast<int32_t>(m);
    u.kchunk = static_cast<int32_t>(Kc);
    u.chunk_self = d;
    u.chunk_nsrc = P;
    u.chunk_order = o.order == FO_ORDER_NAIVE ? 1 : 0;
    u.chunk_flag_base = serial ? -1 : static_cast<int32_t>(kAgFlagBase + d * P);
    u.b_map = wmap;
    u.m_rows = static_cast<int32_t>(m);
    u.n_cols = static_cast<int32_t>(N);
    u.k = static_cast<int32_t>(P * Kc);
    u.epi = kEpiBF16;
    u.c = Y[d].ptr;
    u.ldc = Y[d].ld;
  }
  FO_TRY(L.finish(epoch, timeout_ns(o), flags, ctx->ctrl, 0));
  auto hops = [&](bool with_flags) -> fo_status {
    for (int t = 1; t < P; ++t) {
      for (int s = 0; s < P; ++s) {
        const int d = mod(s + t, P);
        if (o.fault == FO_FAULT_SKIP_HOP && with_flags && t == 1 && s == 0) continue;
        FO_TRY(copy_rows(recv(d) + s * m * Kc * 2, Kc, bptr(C[s], d * m), C[s].ld, m, Kc, 2, ctx->link[s]));
        if (with_flags) FO_TRY(write_flag(ctx->link[s], flags + kAgFlagBase + d * P + s, epoch));
      }
    }
    return FO_OK;
  };
  if (serial) {
    FO_CUDA(cudaEventRecord(ctx->ev_phase[0], stream));
    FO_TRY(fork_links(ctx, P, stream));
    FO_TRY(hops(false));
    FO_TRY(join_links(ctx, P, stream));
    FO_CUDA(cudaEventRecord(ctx->ev_phase[1], stream));
    FO_TRY(launch_gemm(ctx, L, o, stream));
    FO_CUDA(cudaEventRecord(ctx->ev_phase[2], stream));
    ctx->phase_valid = true;
    ctx->phase_gemm_first = false;
    return FO_OK;
  }
  // the hops run concurrently with the GEMM that waits on them (host order: copies_first)
  FO_TRY(fork_links(ctx, P, stream));  // the links start after the caller's prior work
  if (!copies_first()) FO_TRY(launch_gemm(ctx, L, o, stream));
  FO_TRY(hops(true));
  if (copies_first()) FO_TRY(launch_gemm(ctx, L, o, stream));
  return join_links(ctx, P, stream);
}

// --------------------------------------------------------------------------
// Training backward of the two projections: the same collectives with the roles swapped
// --------------------------------------------------------------------------

// C[i] = A[i] B[i]^T (bf16) for i < n in one persistent launch.  a_mn: A[i] is given as
// its transpose, [K, M]; b_mn: B[i] as [K, N] (both read MN-major by the MMA, no copy).
// stream_a: tiles ordered m-block-major across the units, so each A panel is read once
// while B (shared by the units) cycles in L2; otherwise unit by unit, n-block outer, so
// each B panel is read once while A cycles.
fo_status gemm_batch(fo_ctx* ctx, int n, const fo_mat* A, bool a_mn, const fo_mat* B, bool b_mn, const fo_mat* C,
                     bool stream_a, const fo_opts& o, cudaStream_t stream) {
  Launch L;
  fo_status st = FO_OK;
  L.begin_group();
  for (int i = 0; i < n; ++i) {
    const int64_t M = a_mn ? A[i].cols : A[i].rows, K = a_mn ? A[i].rows : A[i].cols;
    const int64_t N = b_mn ? B[i].cols : B[i].rows;
    const int am = a_mn ? L.add_map_mn(&st, A[i].ptr, K, M, A[i].ld) : L.add_map(&st, A[i].ptr, M, K, A[i].ld, kBM);
    FO_TRY(st);
    const int bm = b_mn ? L.add_map_mn(&st, B[i].ptr, K, N, B[i].ld) : L.add_map(&st, B[i].ptr, N, K, B[i].ld, kBN);
    FO_TRY(st);
    GemmUnit& u = L.add_unit();
    u = blank_unit();
    u.a_map = am;
    u.b_map = bm;
    u.m_rows = static_cast<int32_t>(M);
    u.n_cols = static_cast<int32_t>(N);
    u.k = static_cast<int32_t>(K);
    u.epi = kEpiBF16;
    u.c = C[i].ptr;
    u.ldc = C[i].ld;
  }
  void* flags_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &flags_v));
  L.p.mn_major = (a_mn ? 1 : 0) | (b_mn ? 2 : 0);
  FO_TRY(L.finish(++ctx->epoch, timeout_ns(o), static_cast<uint32_t*>(flags_v), ctx->ctrl, stream_a ? 1 : 0));
  return launch_gemm(ctx, L, o, stream);
}

// The P token slices stacked into one [P*m, cols] buffer (the operand that the weight
// gradient contracts over all tokens).
fo_status stack_slices(const fo_mat* S, int P, void** buf, fo_ctx* ctx, int id, cudaStream_t s) {
  const int64_t m = S[0].rows, cols = S[0].cols;
  FO_TRY(ensure_buf(ctx, id, static_cast<size_t>(P) * m * cols * 2, buf));
  for (int r = 0; r < P; ++r)
    FO_TRY(copy_rows(static_cast<char*>(*buf) + r * m * cols * 2, cols, S[r].ptr, S[r].ld, m, cols, 2, s));
  return FO_OK;
}

// Column-parallel projection Y_r = AG(X) W_r^T, backward:
//   dX (token slices) = reduce-scatter of dY_r W_r  -> Flash-RS, W_r read as the [Nr, K]
//                                                     B^T it already is
//   dW_r = dY_r^T AG(X)                             -> local GEMM, dY_r and the stacked X
//                                                     read MN-major
fo_status col_backward_run(fo_ctx* ctx, const fo_mat* X, const fo_mat* W, const fo_mat* dY, int P, const fo_mat* dX,
                           const fo_mat* dW, const fo_opts& o, cudaStream_t s) {
  const int64_t m = X[0].rows, K = X[0].cols, Nr = W[0].rows, M = m * P;
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(X[r], FO_BF16, "X_shards", r));
    FO_TRY(check_mat(W[r], FO_BF16, "W_col", r));
    FO_TRY(check_mat(dY[r], FO_BF16, "dY", r));
    FO_TRY(check_mat(dX[r], FO_BF16, "dX", r));
    FO_TRY(check_mat(dW[r], FO_BF16, "dW", r));
    if (X[r].rows != m || X[r].cols != K || W[r].rows != Nr || W[r].cols != K || dY[r].rows != M ||
        dY[r].cols != Nr || dX[r].rows != m || dX[r].cols != K || dW[r].rows != Nr || dW[r].cols != K)
      return fail(FO_ERR_SHAPE, "rank %d: need X [m, K], W_col [Nr, K], dY [P*m, Nr], dX [m, K], dW [Nr, K]", r);
  }
  if (Nr % 8 != 0 || M % 8 != 0) return fail(FO_ERR_UNSUPPORTED, "Nr and P*m must be multiples of 8");
  if (m == 0 || K == 0 || Nr == 0) return FO_OK;
  void* xs = nullptr;
  FO_TRY(stack_slices(X, P, &xs, ctx, kBufBwdStack, s));
  fo_mat Xs[kMaxP];
  for (int r = 0; r < P; ++r) Xs[r] = fo_mat{xs, FO_BF16, 0, M, K, K};
  FO_TRY(rs_run(ctx, dY, W, P, dX, o, s, /*w_kn=*/true));
  // dY_r (58.7 MB per rank at 4096 tokens x 7168) is streamed; the stacked X is shared
  return gemm_batch(ctx, P, dY, /*a_mn=*/true, Xs, /*b_mn=*/true, dW, /*stream_a=*/true, o, s);
}

// Row-parallel projection Z = RS(H_r W_r^T), backward:
//   dH_r = AG(dZ) W_r                 -> Flash-AG, W_r read MN-major
//   dW_r = AG(dZ)^T H_r               -> local GEMM, the stacked dZ and H_r read MN-major
fo_status row_backward_run(fo_ctx* ctx, const fo_mat* H, const fo_mat* W, const fo_mat* dZ, int P, const fo_mat* dH,
                           const fo_mat* dW, const fo_opts& o, cudaStream_t s) {
  const int64_t M = H[0].rows, Fr = H[0].cols, N = W[0].rows;
  if (M % P != 0) return fail(FO_ERR_SHAPE, "H rows=%lld not divisible by P=%d", (long long)M, P);
  const int64_t m = M / P;
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(H[r], FO_BF16, "H", r));
    FO_TRY(check_mat(W[r], FO_BF16, "W_row", r));
    FO_TRY(check_mat(dZ[r], FO_BF16, "dZ", r));
    FO_TRY(check_mat(dH[r], FO_BF16, "dH", r));
    FO_TRY(check_mat(dW[r], FO_BF16, "dW", r));
    if (H[r].rows != M || H[r].cols != Fr || W[r].rows != N || W[r].cols != Fr || dZ[r].rows != m ||
        dZ[r].cols != N || dH[r].rows != M || dH[r].cols != Fr || dW[r].rows != N || dW[r].cols != Fr)
      return fail(FO_ERR_SHAPE, "rank %d: need H [P*m, Fr], W_row [N, Fr], dZ [m, N], dH [P*m, Fr], dW [N, Fr]", r);
  }
  if (N % 8 != 0 || M % 8 != 0) return fail(FO_ERR_UNSUPPORTED, "N and P*m must be multiples of 8");
  if (m == 0 || Fr == 0 || N == 0) return FO_OK;
  void* zs = nullptr;
  FO_TRY(stack_slices(dZ, P, &zs, ctx, kBufBwdStack, s));
  fo_mat Zs[kMaxP];
  for (int r = 0; r < P; ++r) Zs[r] = fo_mat{zs, FO_BF16, 0, M, N, N};
  fo_opts oa = o;
  if (oa.order == FO_ORDER_NAIVE) oa.order = FO_ORDER_FLASH;  // the naive order concerns the RS step
  FO_TRY(ag_run(ctx, dZ, W, P, dH, oa, s, /*gated=*/false, /*w_kn=*/true));
  // H_r is streamed; the stacked dZ is shared by the ranks' units
  return gemm_batch(ctx, P, Zs, /*a_mn=*/true, H, /*b_mn=*/true, dW, /*stream_a=*/false, o, s);
}

// --------------------------------------------------------------------------
// MLP layer
// --------------------------------------------------------------------------

// One persistent launch for a whole MLP layer (fused orders): the Flash-AG tiles (SiLU(gate)
// * up epilogue when gated) come first in the tile order, then the Flash-RS tiles.  Each RS
// tile's producer waits until every AG tile that writes its rows of H has stored them
// (per-(rank, slice, m-block) counters of the storing epilogue warps), so the RS tiles of
// the first ring steps -- which read slices the AG computed in its first steps -- fill the
// AG's last wave instead of waiting for a second launch.  Every tile waits only on tiles of
// smaller index.  *used = false (nothing enqueued) when the layer does not fit one launch.
fo_status mlp_fused_run(fo_ctx* ctx, const fo_mat* X, const fo_mat* Wc, const fo_mat* Wr, int P, bool gated,
                        const fo_mat* Z, const fo_opts& o, cudaStream_t stream, const fo_mat* Xh, DoneSignal* done,
                        bool* used) {
  *used = false;
  const int64_t m = X[0].rows, K = X[0].cols, Nc = Wc[0].rows, M = m * P;
  const int64_t F = gated ? Nc / 2 : Nc;
  if (o.split_layer || o.compute_only || (o.order != FO_ORDER_FLASH && o.order != FO_ORDER_NAIVE)) return FO_OK;
  if (m == 0 || K == 0 || F == 0 || K % 8 != 0 || F % 8 != 0 || K % 4 != 0) return FO_OK;
  if (5 * P > kMaxMaps || 2 * P * P > kMaxUnits) return FO_OK;
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(X[r], FO_BF16, "X_shards", r));
    FO_TRY(check_mat(Wc[r], FO_BF16, "W_col", r));
    FO_TRY(check_mat(Wr[r], FO_BF16, "W_row", r));
    FO_TRY(check_mat(Z[r], FO_BF16, "Z", r));
    if (X[r].rows != m || X[r].cols != K || Wc[r].rows != Nc || Wc[r].cols != K || Wr[r].rows != K ||
        Wr[r].cols != F || Z[r].rows != m || Z[r].cols != K)
      return fail(FO_ERR_SHAPE, "rank %d: need X [m, H], W_col [Nc, H], W_row [H, F], Z [m, H]", r);
  }
  fo_mat H[kMaxP];
  void* h_v = nullptr;
  FO_TRY(ensure_buf(ctx, gated ? kBufMlpH : kBufMlpY, static_cast<size_t>(P) * M * F * 2 + 16, &h_v));
  for (int r = 0; r < P; ++r)
    H[r] = fo_mat{static_cast<char*>(h_v) + static_cast<int64_t>(r) * M * F * 2, FO_BF16, 0, M, F, F};
  RsArgs b{H, Wr, Z, P, M, m, F, K, nullptr, nullptr, false};
  bool tn_pair = false;
  if (rs_tn_steps(ctx, b, o, &tn_pair) != 0) return FO_OK;  // its own tile shape: two launches
  const bool pairs = o.sm_pairs != 1 && ctx->pair_clusters > 0 && m % (2 * kBM) == 0;
  const int64_t block_rows = pairs ? 2 * kBM : kBM, mblocks = (m + block_rows - 1) / block_rows;
  if (kRowsBase + static_cast<int64_t>(P) * P * mblocks + 1 > static_cast<int64_t>(kFlagBytes / 4)) return FO_OK;

  void *flags_v = nullptr, *recv_v = nullptr, *rs_recv_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &flags_v));
  FO_TRY(ensure_buf(ctx, kBufAgRecv, static_cast<size_t>(P) * M * K * 2, &recv_v));
  FO_TRY(ensure_buf(ctx, kBufRsRecv, static_cast<size_t>(P) * P * m * K * 4, &rs_recv_v));
  uint32_t* flags = static_cast<uint32_t*>(flags_v);
  b.recv = static_cast<float*>(rs_recv_v);
  AgArgs a{X, Wc, H, P, m, K, Nc, static_cast<char*>(recv_v), false, Xh};
  const uint32_t epoch = ++ctx->epoch;
  Launch L;
  fo_status st = FO_OK;
  int xmap[kMaxP], rmap[kMaxP], wmap[kMaxP];
  for (int r = 0; r < P; ++r) {
    xmap[r] = L.add_map(&st, X[r].ptr, m, K, X[r].ld, kBM);
    FO_TRY(st);
    rmap[r] = L.add_map(&st, ag_rank_buffer(a, r), M, K, K, kBM);
    FO_TRY(st);
    wmap[r] = L.add_map(&st, Wc[r].ptr, Nc, K, Wc[r].ld, gated ? kBN / 2 : kBN);
    FO_TRY(st);
  }
  const bool weight_major = static_cast<double>(P - 1) * m * K * 2 <= kWeightMajorMaxBytes;
  FO_TRY(add_ag_units(L, a, xmap, rmap, wmap, 0, m, true, gated ? F : 0, weight_major, kRowsBase, mblocks));
  // the RS tiles of rows [mb * block_rows, +block_rows) of chunk c wait for every AG tile
  // (output columns per tile: 128 gated, 256 plain) of those rows of slice c to be stored
  const int64_t ag_tiles_n = (F + (gated ? kBN / 2 : kBN) - 1) / (gated ? kBN / 2 : kBN);
  const int ready = static_cast<int>(ag_tiles_n * (pairs ? 8 : 4));
  int64_t flag_end = 0;
  FO_TRY(build_rs_flash(ctx, L, b, o, flags, epoch, done != nullptr, 0, false, &flag_end, kRowsBase, mblocks, ready));
  FO_TRY(L.finish(epoch, timeout_ns(o), flags, ctx->ctrl, 0));
  if (pairs != (o.sm_pairs != 1 && ctx->pair_clusters > 0 && L.pair_friendly()))
    return fail(FO_ERR_UNSUPPORTED, "layer launch: inconsistent tile shape");
  // the word after the per-block counters counts every AG epilogue warp of the launch
  int64_t ag_arrivals = 0;
  for (int i = 0; i < L.num_units; ++i)
    if (L.p.units[i].rows_done_base >= 0)
      ag_arrivals += static_cast<int64_t>((m + block_rows - 1) / block_rows) * ag_tiles_n * (pairs ? 8 : 4);
  L.p.rows_all_index = static_cast<int32_t>(kRowsBase + static_cast<int64_t>(P) * P * mblocks);
  L.p.rows_all_count = static_cast<int32_t>(ag_arrivals);
  *used = true;
  FO_CUDA(cudaMemsetAsync(flags + kRowsBase, 0, (static_cast<size_t>(P) * P * mblocks + 1) * 4, stream));
  // the ring's copies run concurrently with the launch (host order: copies_first)
  FO_TRY(fork_links(ctx, P, stream));
  if (!copies_first()) FO_TRY(launch_gemm(ctx, L, o, stream));
  if (a.Xh) FO_TRY(enqueue_uploads(ctx, a, epoch, flags));
  FO_TRY(enqueue_ag_ring(ctx, a, 0, m, true, epoch, o.fault, flags));
  if (copies_first()) FO_TRY(launch_gemm(ctx, L, o, stream));
  FO_TRY(join_links(ctx, P, stream));
  if (done) FO_TRY(publish_done(ctx, L, flags, stream, done));
  return FO_OK;
}

// Xh non-null: X are device buffers that the Flash-AG first fills from the host shards Xh.
fo_status mlp_run(fo_ctx* ctx, const fo_mat* X, const fo_mat* Wc, const fo_mat* Wr, int P, int gated,
                  const fo_mat* Z, const fo_opts& o, cudaStream_t stream, const fo_mat* Xh = nullptr,
                  DoneSignal* done = nullptr) {
  const int64_t m = X[0].rows, M = m * P, Nc = Wc[0].rows;
  if (gated && Nc % 16 != 0) return fail(FO_ERR_UNSUPPORTED, "gated layer needs 2F with F % 8 == 0");
  const int64_t F = gated ? Nc / 2 : Nc;
  bool fused = false;
  FO_TRY(mlp_fused_run(ctx, X, Wc, Wr, P, gated != 0, Z, o, stream, Xh, done, &fused));
  if (fused) return FO_OK;
  fo_mat Y[kMaxP], H[kMaxP];
  if (!gated) {
    void* y_v = nullptr;
    FO_TRY(ensure_buf(ctx, kBufMlpY, static_cast<size_t>(P) * M * Nc * 2 + 16, &y_v));
    for (int r = 0; r < P; ++r)
      Y[r] = fo_mat{static_cast<char*>(y_v) + static_cast<int64_t>(r) * M * Nc * 2, FO_BF16, 0, M, Nc, Nc};
  }
  fo_opts oa = o;
  if (oa.order == FO_ORDER_NAIVE) oa.order = FO_ORDER_FLASH;  // the naive order concerns the RS step
  if (gated) {
    // SiLU(gate) * up is fused into the Flash-AG epilogue: H is written directly
    void* h_v = nullptr;
    FO_TRY(ensure_buf(ctx, kBufMlpH, static_cast<size_t>(P) * M * F * 2 + 16, &h_v));
    for (int r = 0; r < P; ++r)
      H[r] = fo_mat{static_cast<char*>(h_v) + static_cast<int64_t>(r) * M * F * 2, FO_BF16, 0, M, F, F};
    FO_TRY(ag_run(ctx, X, Wc, P, H, oa, stream, true, false, Xh));
  } else {
    FO_TRY(ag_run(ctx, X, Wc, P, Y, oa, stream, false, false, Xh));
    for (int r = 0; r < P; ++r) H[r] = Y[r];
  }
  return rs_run(ctx, H, Wr, P, Z, o, stream, false, done);
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================

extern "C" {

int fo_version(void) { return 100; }

const char* fo_last_error_string(void) { return g_last_error.c_str(); }

fo_status fo_ctx_create(int device, fo_ctx** out) {
  if (!out) return fail(FO_ERR_INVALID_ARG, "null out pointer");
  *out = nullptr;
  int ndev = 0;
  FO_CUDA(cudaGetDeviceCount(&ndev));
  if (device < 0 || device >= ndev) return fail(FO_ERR_INVALID_ARG, "device %d of %d", device, ndev);
  FO_CUDA(cudaSetDevice(device));
  cudaDeviceProp prop;
  FO_CUDA(cudaGetDeviceProperties(&prop, device));
  if (prop.major != 10 || prop.minor != 3)
    return fail(FO_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", device, prop.major,
                prop.minor);
  if (!driver()) return fail(FO_ERR_CUDA, "driver entry points (tensor maps, stream memory operations) unavailable");
  fo_ctx* c = new fo_ctx();
  c->device = device;
  c->num_sms = prop.multiProcessorCount;
  auto cleanup = [&](fo_status st) {
    fo_ctx_destroy(c);
    return st;
  };
  if (gemm_configure() != cudaSuccess) return cleanup(fail(FO_ERR_CUDA, "gemm kernel configuration failed"));
  if (gemm_pair_configure() == cudaSuccess) {
    c->pair_clusters = gemm_pair_max_clusters();
  } else {
    cudaGetLastError();
    c->pair_clusters = 0;
  }
  for (int r = 0; r < kMaxP; ++r) {
    if (cudaStreamCreateWithFlags(&c->link[r], cudaStreamNonBlocking) != cudaSuccess)
      return cleanup(fail(FO_ERR_CUDA, "stream creation failed"));
    if (cudaEventCreateWithFlags(&c->ev_join[r], cudaEventDisableTiming) != cudaSuccess)
      return cleanup(fail(FO_ERR_CUDA, "event creation failed"));
    for (int t = 0; t < kMaxP; ++t)
      if (cudaEventCreateWithFlags(&c->ev_hop[r][t], cudaEventDisableTiming) != cudaSuccess)
        return cleanup(fail(FO_ERR_CUDA, "event creation failed"));
    for (int i = 0; i < kMaxSlices; ++i)
      if (cudaEventCreateWithFlags(&c->ev_slice[i][r], cudaEventDisableTiming) != cudaSuccess)
        return cleanup(fail(FO_ERR_CUDA, "event creation failed"));
  }
  if (cudaStreamCreateWithFlags(&c->aux, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_aux, cudaEventDisableTiming) != cudaSuccess)
    return cleanup(fail(FO_ERR_CUDA, "stream/event creation failed"));
  for (int i = 0; i < 3; ++i)
    if (cudaEventCreate(&c->ev_phase[i]) != cudaSuccess) return cleanup(fail(FO_ERR_CUDA, "event creation failed"));
  if (cudaMalloc(&c->ctrl, kCtrlWords * sizeof(uint32_t)) != cudaSuccess)
    return cleanup(fail(FO_ERR_OOM, "control block allocation failed"));
  if (cudaMemset(c->ctrl, 0, kCtrlWords * sizeof(uint32_t)) != cudaSuccess)
    return cleanup(fail(FO_ERR_CUDA, "control block init failed"));
  *out = c;
  return FO_OK;
}

fo_status fo_ctx_destroy(fo_ctx* ctx) {
  if (!ctx) return FO_OK;
  cudaSetDevice(ctx->device);
  cudaDeviceSynchronize();
  for (auto& kv : ctx->bufs)
    if (kv.second.ptr) cudaFree(kv.second.ptr);
  if (ctx->ctrl) cudaFree(ctx->ctrl);
  for (int r = 0; r < kMaxP; ++r) {
    if (ctx->link[r]) cudaStreamDestroy(ctx->link[r]);
    if (ctx->ev_join[r]) cudaEventDestroy(ctx->ev_join[r]);
    for (int t = 0; t < kMaxP; ++t)
      if (ctx->ev_hop[r][t]) cudaEventDestroy(ctx->ev_hop[r][t]);
    for (int i = 0; i < kMaxSlices; ++i)
      if (ctx->ev_slice[i][r]) cudaEventDestroy(ctx->ev_slice[i][r]);
  }
  if (ctx->aux) cudaStreamDestroy(ctx->aux);
  if (ctx->ev_fork) cudaEventDestroy(ctx->ev_fork);
  if (ctx->ev_aux) cudaEventDestroy(ctx->ev_aux);
  for (int i = 0; i < 3; ++i)
    if (ctx->ev_phase[i]) cudaEventDestroy(ctx->ev_phase[i]);
  delete ctx;
  return FO_OK;
}

fo_status fo_ctx_poll(fo_ctx* ctx) {
  if (!ctx) return fail(FO_ERR_INVALID_ARG, "null context");
  uint32_t w[kCtrlWords];
  FO_CUDA(cudaMemcpy(w, ctx->ctrl, sizeof(w), cudaMemcpyDeviceToHost));
  if (w[kCtrlError] == 0) return FO_OK;
  FO_CUDA(cudaMemset(ctx->ctrl, 0, sizeof(w)));
  if (w[kCtrlError] == FO_ERR_RANGE)
    return fail(FO_ERR_RANGE, "input value out of the kernels' range (site %u, row %u): |V| above 65504, "
                "the largest finite fp16 value", w[kCtrlWhere], w[kCtrlDetail]);
  return fail(static_cast<fo_status>(w[kCtrlError]), "device wait gave up (site %u, index %u)", w[kCtrlWhere],
              w[kCtrlDetail]);
}

int fo_step_order(int op, int P, int order, int32_t* rank, int32_t* item, int capacity) {
  if (P < 1 || P > kMaxP || op < 0 || op > 3 || !rank || !item) return -1;
  if (order != FO_ORDER_FLASH && order != FO_ORDER_NAIVE) return -1;
  if (op == 0 && order != FO_ORDER_FLASH) return -1;
  if (capacity < P * P) return -1;
  for (int t = 0; t < P; ++t) {
    for (int i = 0; i < P; ++i) {
      int r, x;
      if (op == 0) {
        ag_unit(P, t, i, &r, &x);
      } else if (op == 1) {
        rs_unit(P, order, t, i, &r, &x);
      } else if (op == 2) {
        a2a_block_unit(P, order, t, i, &r, &x);
      } else {
        a2a_source_unit(P, order, t, i, &r, &x);
      }
      rank[t * P + i] = r;
      item[t * P + i] = x;
    }
  }
  return P * P;
}

fo_status fo_ctx_phase_ms(fo_ctx* ctx, float* collective_ms, float* gemm_ms) {
  if (!ctx || !collective_ms || !gemm_ms) return fail(FO_ERR_INVALID_ARG, "null argument");
  if (!ctx->phase_valid) return fail(FO_ERR_INVALID_ARG, "no FO_ORDER_SERIAL call on this context yet");
  float a = 0.f, b = 0.f;
  FO_CUDA(cudaEventElapsedTime(&a, ctx->ev_phase[0], ctx->ev_phase[1]));
  FO_CUDA(cudaEventElapsedTime(&b, ctx->ev_phase[1], ctx->ev_phase[2]));
  // AG: phase 0->1 is the ring, 1->2 the GEMM; RS: 0->1 the GEMM, 1->2 the ring
  *collective_ms = ctx->phase_gemm_first ? b : a;
  *gemm_ms = ctx->phase_gemm_first ? a : b;
  return FO_OK;
}

fo_status fo_gemm(fo_ctx* ctx, const fo_mat* A, const fo_mat* B, const fo_mat* C, const fo_opts* opts,
                  void* stream) {
  FO_TRY(check_common(ctx, 1, opts));
  if (!A || !B || !C) return fail(FO_ERR_INVALID_ARG, "null matrix");
  FO_TRY(check_mat(*A, FO_BF16, "A", 0));
  FO_TRY(check_mat(*B, FO_BF16, "B", 0));
  FO_TRY(check_mat(*C, C->dtype == FO_F32 ? FO_F32 : FO_BF16, "C", 0));
  if (A->cols != B->cols) return fail(FO_ERR_SHAPE, "A and B must share K");
  if (C->rows != A->rows || C->cols != B->rows) return fail(FO_ERR_SHAPE, "C must be [M, N]");
  if (A->cols % 8 != 0) return fail(FO_ERR_UNSUPPORTED, "K must be a multiple of 8");
  if (A->rows == 0 || B->rows == 0) return FO_OK;
  if (A->cols == 0) return fail(FO_ERR_UNSUPPORTED, "K == 0");
  FO_CUDA(cudaSetDevice(ctx->device));
  fo_opts o = opts ? *opts : default_opts();
  Launch L;
  fo_status st = FO_OK;
  const int am = L.add_map(&st, A->ptr, A->rows, A->cols, A->ld, kBM);
  FO_TRY(st);
  const int bm = L.add_map(&st, B->ptr, B->rows, B->cols, B->ld, kBN);
  FO_TRY(st);
  L.begin_group();
  GemmUnit& u = L.add_unit();
  u = blank_unit();
  u.a_map = am;
  u.b_map = bm;
  u.m_rows = static_cast<int32_t>(A->rows);
  u.n_cols = static_cast<int32_t>(B->rows);
  u.k = static_cast<int32_t>(A->cols);
  u.epi = C->dtype == FO_F32 ? kEpiF32 : kEpiBF16;
  u.c = C->ptr;
  u.ldc = C->ld;
  if (A->rows > (1 << 30)) return fail(FO_ERR_UNSUPPORTED, "M too large");
  void* flags_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &flags_v));
  FO_TRY(L.finish(++ctx->epoch, timeout_ns(o), static_cast<uint32_t*>(flags_v), ctx->ctrl, 0));
  return launch_gemm(ctx, L, o, static_cast<cudaStream_t>(stream));
}

fo_status fo_ag_gemm(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_col, int P, const fo_mat* Y,
                     const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!X_shards || !W_col || !Y) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  const fo_opts o = opts ? *opts : default_opts();
  if (o.order == FO_ORDER_NAIVE) return fail(FO_ERR_INVALID_ARG, "FO_ORDER_NAIVE applies to reduce-scatter only");
  return ag_run(ctx, X_shards, W_col, P, Y, o, static_cast<cudaStream_t>(stream), o.epilogue == FO_EPI_SILU_GATE);
}

fo_status fo_gemm_rs(fo_ctx* ctx, const fo_mat* X, const fo_mat* W_row, int P, const fo_mat* Y,
                     const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!X || !W_row || !Y) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  const fo_opts o = opts ? *opts : default_opts();
  return rs_run(ctx, X, W_row, P, Y, o, static_cast<cudaStream_t>(stream));
}

fo_status fo_silu_mul(fo_ctx* ctx, const fo_mat* GU, int P, const fo_mat* H, void* stream) {
  FO_TRY(check_common(ctx, P, nullptr));
  if (!GU || !H) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  SiluMulArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  const int64_t rows = GU[0].rows, F = GU[0].cols / 2;
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(GU[r], FO_BF16, "GU", r));
    FO_TRY(check_mat(H[r], FO_BF16, "H", r));
    if (GU[r].rows != rows || GU[r].cols != 2 * F || H[r].rows != rows || H[r].cols != F)
      return fail(FO_ERR_SHAPE, "GU[%d] must be [rows, 2F] and H[%d] [rows, F]", r, r);
    sa.gu[r] = static_cast<const uint16_t*>(GU[r].ptr);
    sa.h[r] = static_cast<uint16_t*>(H[r].ptr);
    sa.ld_gu[r] = GU[r].ld;
    sa.ld_h[r] = H[r].ld;
  }
  if (F % 8 != 0) return fail(FO_ERR_UNSUPPORTED, "F must be a multiple of 8");
  sa.rows = rows;
  sa.f = F;
  sa.P = P;
  FO_CUDA(launch_silu_mul(sa, static_cast<cudaStream_t>(stream)));
  return FO_OK;
}

fo_status fo_mlp_layer(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_col, const fo_mat* W_row, int P,
                       int gated, const fo_mat* Z, const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!X_shards || !W_col || !W_row || !Z) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  const fo_opts o = opts ? *opts : default_opts();
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(W_col[r], FO_BF16, "W_col", r));
    FO_TRY(check_mat(W_row[r], FO_BF16, "W_row", r));
    const int64_t F = gated ? W_col[r].rows / 2 : W_col[r].rows;
    if (W_row[r].cols != F) return fail(FO_ERR_SHAPE, "W_row[%d] must have F=%lld columns", r, (long long)F);
  }
  return mlp_run(ctx, X_shards, W_col, W_row, P, gated, Z, o, static_cast<cudaStream_t>(stream));
}

fo_status fo_mlp_layer_host(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_col, const fo_mat* W_row, int P,
                            int gated, const fo_mat* Z, const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (opts && opts->compute_only) return fail(FO_ERR_UNSUPPORTED, "compute_only is a device-buffer timing mode");
  if (!X_shards || !W_col || !W_row || !Z) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t m = X_shards[0].rows, Hd = X_shards[0].cols;
  for (int r = 0; r < P; ++r) {
    if (!X_shards[r].ptr || !Z[r].ptr) return fail(FO_ERR_INVALID_ARG, "null host pointer");
    if (X_shards[r].dtype != FO_BF16 || Z[r].dtype != FO_BF16) return fail(FO_ERR_INVALID_ARG, "bf16 expected");
    if (X_shards[r].rows != m || X_shards[r].cols != Hd || Z[r].rows != m || Z[r].cols != Hd ||
        X_shards[r].ld < Hd || Z[r].ld < Hd)
      return fail(FO_ERR_SHAPE, "host X_shards[%d] / Z[%d] must be [m, hidden]", r, r);
  }
  void *xv = nullptr, *zv = nullptr;
  const size_t bytes = static_cast<size_t>(P) * m * Hd * 2 + 16;
  FO_TRY(ensure_buf(ctx, kBufHostX, bytes, &xv));
  FO_TRY(ensure_buf(ctx, kBufHostZ, bytes, &zv));
  fo_mat Xd[kMaxP], Zd[kMaxP];
  for (int r = 0; r < P; ++r) {
    Xd[r] = fo_mat{static_cast<char*>(xv) + static_cast<int64_t>(r) * m * Hd * 2, FO_BF16, 0, m, Hd, Hd};
    Zd[r] = fo_mat{static_cast<char*>(zv) + static_cast<int64_t>(r) * m * Hd * 2, FO_BF16, 0, m, Hd, Hd};
    FO_TRY(check_mat(W_col[r], FO_BF16, "W_col", r));
    FO_TRY(check_mat(W_row[r], FO_BF16, "W_row", r));
    const int64_t F = gated ? W_col[r].rows / 2 : W_col[r].rows;
    if (W_row[r].cols != F) return fail(FO_ERR_SHAPE, "W_row[%d] must have F=%lld columns", r, (long long)F);
  }
  // the Flash-AG uploads the host shards itself, slice by slice, ahead of their GEMMs; in
  // the fused order each rank's output goes back as soon as its kept chunk is complete
  DoneSignal done;
  FO_TRY(mlp_run(ctx, Xd, W_col, W_row, P, gated, Zd, opts ? *opts : default_opts(), s, X_shards, &done));
  if (!done.set) {
    for (int r = 0; r < P; ++r)
      FO_CUDA(cudaMemcpy2DAsync(Z[r].ptr, Z[r].ld * 2, Zd[r].ptr, Hd * 2, Hd * 2, m, cudaMemcpyDeviceToHost, s));
    return FO_OK;
  }
  void* flags_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &flags_v));
  uint32_t* flags = static_cast<uint32_t*>(flags_v);
  for (int r = 0; r < P; ++r) {
    cudaStream_t ls = ctx->link[r];
    FO_CU(driver()->wait_value32(reinterpret_cast<CUstream>(ls), reinterpret_cast<CUdeviceptr>(flags + kDoneBase + r),
                                 done.target[r], CU_STREAM_WAIT_VALUE_GEQ));
    FO_CUDA(cudaMemcpy2DAsync(Z[r].ptr, Z[r].ld * 2, Zd[r].ptr, Hd * 2, Hd * 2, m, cudaMemcpyDeviceToHost, ls));
  }
  return join_links(ctx, P, s);
}

fo_status fo_qsplit_attn(fo_ctx* ctx, const fo_mat* Q, const fo_mat* K_shards, const fo_mat* V_shards, int P,
                         int heads, int head_dim, int causal, const fo_mat* O, const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!Q || !K_shards || !V_shards || !O) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  return attn_run(ctx, Q, K_shards, V_shards, P, heads, head_dim, causal, O, opts,
                  static_cast<cudaStream_t>(stream), true);
}

fo_status fo_col_linear_backward(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_col, const fo_mat* dY, int P,
                                 const fo_mat* dX, const fo_mat* dW, const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!X_shards || !W_col || !dY || !dX || !dW) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  return col_backward_run(ctx, X_shards, W_col, dY, P, dX, dW, opts ? *opts : default_opts(),
                          static_cast<cudaStream_t>(stream));
}

fo_status fo_row_linear_backward(fo_ctx* ctx, const fo_mat* H, const fo_mat* W_row, const fo_mat* dZ_shards, int P,
                                 const fo_mat* dH, const fo_mat* dW, const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!H || !W_row || !dZ_shards || !dH || !dW) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  return row_backward_run(ctx, H, W_row, dZ_shards, P, dH, dW, opts ? *opts : default_opts(),
                          static_cast<cudaStream_t>(stream));
}

fo_status fo_gemm_a2a(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W, int P, const fo_mat* Y,
                      const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!X_shards || !W || !Y) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  return gemm_a2a_run(ctx, X_shards, W, P, Y, opts ? *opts : default_opts(), static_cast<cudaStream_t>(stream));
}

fo_status fo_a2a_gemm(fo_ctx* ctx, const fo_mat* C, const fo_mat* W, int P, const fo_mat* Y, const fo_opts* opts,
                      void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!C || !W || !Y) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  FO_CUDA(cudaSetDevice(ctx->device));
  return a2a_gemm_run(ctx, C, W, P, Y, opts ? *opts : default_opts(), static_cast<cudaStream_t>(stream));
}

fo_status fo_attn_layer(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_qkv, const fo_mat* W_o, int P,
                        int heads, int head_dim, int causal, const fo_mat* Z, const fo_opts* opts, void* stream) {
  FO_TRY(check_common(ctx, P, opts));
  if (!X_shards || !W_qkv || !W_o || !Z) return fail(FO_ERR_INVALID_ARG, "null matrix array");
  if (heads < 1) return fail(FO_ERR_INVALID_ARG, "heads must be positive");
  if (head_dim != 128) return fail(FO_ERR_UNSUPPORTED, "head_dim must be 128");
  FO_CUDA(cudaSetDevice(ctx->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const fo_opts o = opts ? *opts : default_opts();
  const int64_t m = X_shards[0].rows, M = m * P, HD = static_cast<int64_t>(heads) * head_dim;
  for (int r = 0; r < P; ++r) {
    FO_TRY(check_mat(W_qkv[r], FO_BF16, "W_qkv", r));
    FO_TRY(check_mat(W_o[r], FO_BF16, "W_o", r));
    if (W_qkv[r].rows != 3 * HD) return fail(FO_ERR_SHAPE, "W_qkv[%d] must have 3*heads*head_dim rows", r);
    if (W_o[r].cols != HD) return fail(FO_ERR_SHAPE, "W_o[%d] must have heads*head_dim columns", r);
  }
  if (M % 128 != 0) return fail(FO_ERR_UNSUPPORTED, "P*m must be a multiple of 128");
  void *qkv_v = nullptr, *o_v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufLayerQkv, static_cast<size_t>(P) * M * 3 * HD * 2 + 16, &qkv_v));
  FO_TRY(ensure_buf(ctx, kBufLayerO, static_cast<size_t>(P) * M * HD * 2 + 16, &o_v));
  fo_mat QKV[kMaxP], Qm[kMaxP], Km[kMaxP], Vm[kMaxP], Om[kMaxP];
  for (int r = 0; r < P; ++r) {
    char* base = static_cast<char*>(qkv_v) + static_cast<int64_t>(r) * M * 3 * HD * 2;
    QKV[r] = fo_mat{base, FO_BF16, 0, M, 3 * HD, 3 * HD};
    Qm[r] = fo_mat{base, FO_BF16, 0, M, HD, 3 * HD};
    Km[r] = fo_mat{base + HD * 2, FO_BF16, 0, M, HD, 3 * HD};
    Vm[r] = fo_mat{base + 2 * HD * 2, FO_BF16, 0, M, HD, 3 * HD};
    Om[r] = fo_mat{static_cast<char*>(o_v) + static_cast<int64_t>(r) * M * HD * 2, FO_BF16, 0, M, HD, HD};
  }
  fo_opts oa = o;
  if (oa.order == FO_ORDER_NAIVE) oa.order = FO_ORDER_FLASH;  // the naive order concerns the RS step
  FO_TRY(ag_run(ctx, X_shards, W_qkv, P, QKV, oa, s));
  FO_TRY(attn_run(ctx, Qm, Km, Vm, P, heads, head_dim, causal, Om, &oa, s, false));
  return rs_run(ctx, Om, W_o, P, Z, o, s);
}

}  // extern "C"

// Host services for the attention module (fo_attn.cu), declared in fo_host.h.
namespace fo {
fo_status host_buffer(fo_ctx* ctx, int slot, size_t bytes, void** out) {
  return ensure_buf(ctx, kBufAttnRecv + slot, bytes, out);
}
fo_status host_flags(fo_ctx* ctx, uint32_t** out) {
  void* v = nullptr;
  FO_TRY(ensure_buf(ctx, kBufFlags, kFlagBytes, &v));
  *out = static_cast<uint32_t*>(v) + kAgFlagBase;
  return FO_OK;
}
uint32_t host_next_epoch(fo_ctx* ctx) { return ++ctx->epoch; }
uint32_t* host_ctrl(fo_ctx* ctx) { return ctx->ctrl; }
int host_num_sms(fo_ctx* ctx) { return ctx->num_sms; }
cudaStream_t host_link(fo_ctx* ctx, int r) { return ctx->link[r]; }
cudaEvent_t host_ev_hop(fo_ctx* ctx, int r, int t) { return ctx->ev_hop[r][t]; }
fo_status host_fork(fo_ctx* ctx, int P, cudaStream_t s) { return fork_links(ctx, P, s); }
fo_status host_join(fo_ctx* ctx, int P, cudaStream_t s) { return join_links(ctx, P, s); }
fo_status host_copy_rows(void* dst, int64_t dld, const void* src, int64_t sld, int64_t rows, int64_t cols,
                         size_t esz, cudaStream_t s) {
  return copy_rows(dst, dld, src, sld, rows, cols, esz, s);
}
fo_status host_write_flag(cudaStream_t s, uint32_t* flag, uint32_t value) { return write_flag(s, flag, value); }
fo_status host_encode_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows,
                          CUtensorMapDataType dtype) {
  return encode_map(map, ptr, rows, cols, ld, box_rows, dtype);
}
fo_status host_check_mat(const fo_mat& a, int32_t dtype, const char* what, int r) {
  return check_mat(a, dtype, what, r);
}
fo_status host_fail(fo_status st, const char* msg) { return fail(st, "%s", msg); }
bool host_copies_first() { return copies_first(); }
uint64_t host_timeout_ns(const fo_opts& o) { return timeout_ns(o); }
int host_grid(fo_ctx* ctx, const fo_opts& o, int work) { return grid_size(ctx, o, work); }
void host_phase_record(fo_ctx* ctx, int i, cudaStream_t s) { cudaEventRecord(ctx->ev_phase[i], s); }
void host_phase_done(fo_ctx* ctx, bool gemm_first) {
  ctx->phase_valid = true;
  ctx->phase_gemm_first = gemm_first;
}
}  // namespace fo
