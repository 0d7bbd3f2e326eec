// Flash-RS for callers that cannot allocate device memory.
//
// fo_gemm_rs needs scratch memory (the fp32 receive slots of the ring and the
// per-tile flags), which its context allocates with cudaMalloc.  Some callers
// cannot allocate: a host application whose device memory is owned entirely
// by its own allocator (nothing may be taken behind its back), or a
// latency-critical path that must not pay the device-wide synchronisation of
// cudaMalloc/cudaFree.  fo_gemm_rs_noalloc runs the same fused kernel with its
// scratch in a fixed file-scope device array instead.  The caller still passes
// the inputs and outputs.
//
// The array below is part of the library image: every GPU that loads the
// library holds kStaticScratchBytes of it until the process exits.  All calls
// share it, and it keeps the previous call's contents, so every call starts by
// clearing, on its own stream, the control words and the flag words its shape
// uses; its flags are then released with the fixed value 1.  Nothing a call
// reads depends on what an earlier call left behind.  Calls whose kernels
// overlap on the GPU race on the array.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "fo_host.h"
#include "fo_internal.h"

namespace fo {
namespace {

constexpr size_t kStaticScratchBytes = 64ull << 20;  // 64 MiB
constexpr size_t kCtrlBytes = 256;                     // device control block (kCtrlWords words used)
constexpr size_t kFlagBytes = 1ull << 20;              // 262144 epoch-valued flags
constexpr size_t kSlotBytes = kStaticScratchBytes - kCtrlBytes - kFlagBytes;

static __device__ __align__(256) unsigned char g_rs_scratch[kStaticScratchBytes];

struct DeviceState {
  bool ready = false;  // the GEMM kernel is configured for this device
  int num_sms = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_state[kMaxDevices];

// Once per device, with that device current: configure the kernel (its shared-memory
// size attribute) and read the SM count.
fo_status device_setup(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return host_fail(FO_ERR_UNSUPPORTED, "device index above 63");
  DeviceState& s = g_state[dev];
  if (!s.ready) {
    if (gemm_configure() != cudaSuccess) return host_fail(FO_ERR_CUDA, "gemm kernel configuration failed");
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return host_fail(FO_ERR_CUDA, "cannot read the SM count");
    s.num_sms = sms;
    s.ready = true;
  }
  *out = &s;
  return FO_OK;
}

// The array's address on the current device.  In host code the symbol is only a
// stand-in, so the address is asked for on every call (cheap); it is never cached.
fo_status scratch_address(unsigned char** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_rs_scratch);
  if (e != cudaSuccess) return host_fail(FO_ERR_CUDA, cudaGetErrorString(e));
  *out = static_cast<unsigned char*>(ptr);
  return FO_OK;
}

}  // namespace
}  // namespace fo

using namespace fo;

extern "C" FO_API fo_status fo_gemm_rs_noalloc(const fo_mat* X, const fo_mat* W_row, int P, const fo_mat* Y,
                                               uint32_t timeout_us, uint32_t* status, void* stream) {
  if (!X || !W_row || !Y) return host_fail(FO_ERR_INVALID_ARG, "null matrix array");
  if (P < 1 || P > kMaxP) return host_fail(FO_ERR_INVALID_ARG, "P outside [1, 8]");
  const int64_t M = X[0].rows, Kr = X[0].cols, N = W_row[0].rows;
  for (int r = 0; r < P; ++r) {
    fo_status st;
    if ((st = host_check_mat(X[r], FO_BF16, "X", r)) != FO_OK) return st;
    if ((st = host_check_mat(W_row[r], FO_BF16, "W_row", r)) != FO_OK) return st;
    if ((st = host_check_mat(Y[r], FO_BF16, "Y", r)) != FO_OK) return st;
    if (X[r].rows != M || X[r].cols != Kr) return host_fail(FO_ERR_SHAPE, "X shards must share one shape");
    if (W_row[r].rows != N || W_row[r].cols != Kr) return host_fail(FO_ERR_SHAPE, "W_row shards must be [N, Kr]");
  }
  if (M % P != 0) return host_fail(FO_ERR_SHAPE, "M not divisible by P");
  const int64_t m = M / P;
  for (int r = 0; r < P; ++r)
    if (Y[r].rows != m || Y[r].cols != N) return host_fail(FO_ERR_SHAPE, "Y shards must be [M/P, N]");
  if (Kr % 8 != 0 || Kr == 0) return host_fail(FO_ERR_UNSUPPORTED, "Kr must be a positive multiple of 8");
  if (N % 4 != 0) return host_fail(FO_ERR_UNSUPPORTED, "N must be a multiple of 4");
  if (m == 0 || N == 0) return FO_OK;
  const int64_t tm = (m + kBM - 1) / kBM, tn = (N + kBN - 1) / kBN;
  const size_t slot_bytes = static_cast<size_t>(P) * (P - 1) * m * N * 4;
  const size_t flag_bytes = static_cast<size_t>(P) * P * tm * tn * 4 * 4;
  if (slot_bytes > kSlotBytes || flag_bytes > kFlagBytes) {
    static thread_local char msg[256];
    snprintf(msg, sizeof(msg),
             "shape needs %zu bytes of receive slots and %zu of flags; the static scratch holds %zu and %zu",
             slot_bytes, flag_bytes, kSlotBytes, kFlagBytes);
    return host_fail(FO_ERR_UNSUPPORTED, msg);
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return host_fail(FO_ERR_CUDA, "no current device");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* ds = nullptr;
  unsigned char* scratch = nullptr;
  {
    fo_status st = device_setup(dev, &ds);
    if (st == FO_OK) st = scratch_address(&scratch);
    if (st != FO_OK) return st;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(scratch);
  uint32_t* flags = reinterpret_cast<uint32_t*>(scratch + kCtrlBytes);
  float* slots = reinterpret_cast<float*>(scratch + kCtrlBytes + kFlagBytes);
  // this call's control words and flags start at zero, whatever an earlier call left
  if (cudaMemsetAsync(ctrl, 0, kCtrlWords * sizeof(uint32_t), s) != cudaSuccess ||
      cudaMemsetAsync(flags, 0, flag_bytes, s) != cudaSuccess)
    return host_fail(FO_ERR_CUDA, "scratch reset failed");
  const uint32_t epoch = 1;  // every flag of this call is released with the value 1

  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < P; ++r) {
    fo_status st;
    if ((st = host_encode_map(&p.maps[r], X[r].ptr, M, Kr, X[r].ld, kBM)) != FO_OK) return st;
    if ((st = host_encode_map(&p.maps[P + r], W_row[r].ptr, N, Kr, W_row[r].ld, kBN)) != FO_OK) return st;
  }
  // receive slot of rank r for ring position h (1..P-1), and its per-(tile, quadrant) flags
  auto slot = [&](int r, int h) { return slots + (static_cast<int64_t>(r) * (P - 1) + (h - 1)) * m * N; };
  auto fbase = [&](int r, int h) { return static_cast<int32_t>((static_cast<int64_t>(r) * P + h) * tm * tn * 4); };
  int nu = 0;
  for (int t = 0; t < P; ++t) {
    p.group_unit_begin[t] = nu;
    p.group_tile_begin[t] = static_cast<int32_t>(static_cast<int64_t>(nu) * tm * tn);
    for (int i = 0; i < P; ++i) {
      const int r = (t + i) % P;
      const int c = ((r - t - 1) % P + P) % P;  // rank-adaptive: the kept chunk r comes at t = P-1
      const int h = t;
      GemmUnit& u = p.units[nu++];
      u = blank_unit();
      u.a_map = r;
      u.b_map = P + r;
      u.a_row0 = static_cast<int32_t>(c * m);
      u.m_rows = static_cast<int32_t>(m);
      u.n_cols = static_cast<int32_t>(N);
      u.k = static_cast<int32_t>(Kr);
      u.tiles_m = static_cast<int32_t>(tm);
      u.tiles_n = static_cast<int32_t>(tn);
      if (h > 0) {
        u.acc_in = slot(r, h);
        u.ld_acc = N;
        u.in_flag_base = fbase(r, h);
      }
      if (h < P - 1) {
        const int d = (r + 1) % P;
        u.c = slot(d, h + 1);
        u.ldc = N;
        u.out_flag_base = fbase(d, h + 1);
        u.epi = h == 0 ? kEpiF32 : kEpiAddF32;
      } else {
        u.c = Y[r].ptr;
        u.ldc = Y[r].ld;
        u.epi = h == 0 ? kEpiBF16 : kEpiAddBF16;
      }
    }
  }
  p.group_unit_begin[P] = nu;
  p.group_tile_begin[P] = static_cast<int32_t>(static_cast<int64_t>(nu) * tm * tn);
  p.num_groups = P;
  p.num_maps = 2 * P;
  p.mblock_major = 0;
  p.total_tiles = p.group_tile_begin[P];
  p.epoch = epoch;
  p.timeout_ns = (timeout_us ? static_cast<uint64_t>(timeout_us) : 1000000ull) * 1000ull;
  p.flags = flags;
  p.flag_words = static_cast<int32_t>(kFlagBytes / 4);
  p.rows_all_index = -1;
  p.ctrl = ctrl;
  // Tiles wait on tiles of smaller index owned by other CTAs, so every CTA of this grid must
  // be resident at once: the call needs the whole GPU while it runs.
  const int grid = p.total_tiles < ds->num_sms ? p.total_tiles : ds->num_sms;
  if (gemm_launch(p, grid, s) != cudaSuccess) return host_fail(FO_ERR_CUDA, "gemm kernel launch failed");
  if (status && cudaMemcpyAsync(status, ctrl + kCtrlError, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) !=
                    cudaSuccess)
    return host_fail(FO_ERR_CUDA, "status copy failed");
  return FO_OK;
}
