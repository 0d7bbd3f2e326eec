// Query-split causal attention with a K/V ring (FlashOverlap technical
// summary, section 2 "Query Split Attention"; section 4 on its benefit growing
// with sequence length).
//
// Rank r keeps its query slice; K and V slices travel the ring local-first,
// like Flash-AG slices, as copy-engine hops that publish a per-(rank, slice)
// arrival flag.  One persistent kernel processes work items (rank r, 128-query
// block qb, head h).  An item walks the ring steps t = 0, 1, ... (slice
// s = (r - t) mod P: its own slice first), skips slices that lie wholly above
// the causal diagonal, and folds every 128-key block into a running
// online-softmax state: row max and sum in registers, the output accumulator
// in TMEM.
//
// CTA layout (192 threads, one CTA per SM):
//   warp 0      TMA: Q block once per item, then K and V^T blocks (2 stages);
//               waits for the slice's arrival flag before reading it.
//   warp 1      tcgen05.mma: S = Q K^T into one of two TMEM score buffers
//               (the next block's scores overlap this block's softmax), then
//               O += P V into the TMEM accumulator.
//   warps 2-5   softmax: thread i owns query row i; loads its score row,
//               masks the diagonal block, updates max/sum, rescales its O row
//               only when the max grew by more than 2^8 (the final division
//               by the sum uses the same reference max, so this is exact), and
//               writes P into shared memory in the MMA's operand layout.
// V is transposed once per rank (V^T [heads*128, tokens]) before the ring so
// that both MMAs read K-major operands.  The P.V product runs in fp16: the
// transpose converts V's bf16 values to fp16 (exact for |v| within fp16's
// normal range, as for the N(0,1) workloads), and the softmax weights
// P in [0, 2^8] keep 11 significant bits instead of bf16's 8, which keeps the
// weight rounding well below the output's own bf16 rounding.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstring>

#include "fo_host.h"
#include "fo_internal.h"
#include "fo_ptx.cuh"

namespace fo {
namespace {

constexpr int kHd = 128;                 // head_dim
constexpr int kQB = 128;                 // queries per block
constexpr int kKB = 128;                 // keys per block
constexpr int kAttnThreads = 192;
constexpr uint32_t kTileBytes = 128 * 128 * 2;   // one 128x128 bf16 operand (two 64-column swizzle halves)
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr int kKvStages = 2;
constexpr uint32_t kTmemCols = 512;      // S0 [0,128), S1 [128,256), O [256,384)
constexpr uint32_t kOCol = 256;
constexpr uint32_t kIdescS = umma_idesc_bf16(128, 128);   // S = Q K^T, bf16 operands
constexpr uint32_t kIdescO = umma_idesc_f16(128, 128);    // O += P V, fp16 operands
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct AttnParams {
  CUtensorMap maps[4 * kMaxP];  // per rank r: Q = r, K local = P+r, K received = 2P+r, V^T = 3P+r
  uint16_t* out[kMaxP];
  int64_t ld_out[kMaxP];
  int32_t P, heads, nkb, causal;
  int32_t m;                    // tokens per slice
  int32_t total_items;
  uint32_t epoch;
  float scale_log2;             // log2(e) / sqrt(head_dim)
  uint64_t timeout_ns;
  uint32_t* flags;              // arrival flags, index rank*P + slice
  uint32_t* ctrl;
};

struct alignas(8) AttnCtl {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kKvStages], kv_empty[kKvStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, o_done, drain;
  uint32_t tmem_base;
  uint32_t pad;
};

// Shared memory: Q | K stage 0 | V^T stage 0 | K stage 1 | V^T stage 1 | P | control
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKv = kTileBytes;
constexpr uint32_t kOffP = kOffKv + kKvStages * 2 * kTileBytes;
constexpr uint32_t kOffCtl = kOffP + kTileBytes;
constexpr int kAttnSmem = static_cast<int>(kOffCtl + sizeof(AttnCtl) + 1024);

struct Item {
  int r, qb, h;
};

// Items in decreasing cost order: ranks with more visible slices first, then
// later query blocks (longer causal rows), then heads.
__device__ __forceinline__ Item decode_item(const AttnParams& p, int i) {
  const int per_rank = p.nkb * p.heads;
  Item it;
  it.r = p.P - 1 - i / per_rank;
  const int rem = i % per_rank;
  it.qb = p.nkb - 1 - rem / p.heads;
  it.h = rem % p.heads;
  return it;
}

__device__ __forceinline__ int steps_of(const AttnParams& p, int r) { return p.causal ? r + 1 : p.P; }
__device__ __forceinline__ int slice_of(const AttnParams& p, int r, int t) { return (r - t + p.P) % p.P; }
__device__ __forceinline__ int blocks_of(const AttnParams& p, const Item& it, int t) {
  return (p.causal && t == 0) ? it.qb + 1 : p.nkb;
}
__device__ __forceinline__ int item_blocks(const AttnParams& p, const Item& it) {
  return p.causal ? it.r * p.nkb + it.qb + 1 : p.P * p.nkb;
}

// ---------------------------------------------------------------------------

__device__ void attn_producer(const AttnParams& p, uint8_t* smem, AttnCtl* ctl) {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t q_uses = 0;
  uint64_t seen = 0;  // bit r*P+s: arrival of slice s at rank r already observed
  uint32_t armed = 0, armed_phase = 0;
  bool q_armed = false;
  uint32_t q_armed_phase = 0;
  bool ok = true;
  for (int i = blockIdx.x; ok && i < p.total_items; i += gridDim.x) {
    const Item it = decode_item(p, i);
    if (!mbar_wait(&ctl->q_empty, (q_uses & 1u) ^ 1u, p.ctrl, p.timeout_ns, kSiteEmpty, i)) break;
    mbar_arrive_expect_tx(&ctl->q_full, kTileBytes);
    for (int c = 0; c < 2; ++c)
      tma_load_2d(&p.maps[it.r], smem + kOffQ + c * kHalfBytes, &ctl->q_full, it.h * kHd + c * 64, it.qb * kQB);
    q_armed = true;
    q_armed_phase = q_uses & 1u;
    ++q_uses;
    const int nsteps = steps_of(p, it.r);
    for (int t = 0; ok && t < nsteps; ++t) {
      const int s = slice_of(p, it.r, t);
      const int fidx = it.r * p.P + s;
      if (t > 0 && !((seen >> fidx) & 1ull)) {
        if (!flag_wait(p.flags + fidx, p.epoch, p.ctrl, p.timeout_ns, kSiteAttnFlag, fidx)) {
          ok = false;
          break;
        }
        fence_proxy_async_global();
        seen |= 1ull << fidx;
      }
      const CUtensorMap* kmap = t == 0 ? &p.maps[p.P + it.r] : &p.maps[2 * p.P + it.r];
      const int krow0 = t == 0 ? 0 : s * p.m;
      const CUtensorMap* vmap = &p.maps[3 * p.P + it.r];
      const int vrow0 = (s * p.heads + it.h) * kHd;
      const int nb = blocks_of(p, it, t);
      for (int kb = 0; kb < nb; ++kb) {
        if (!mbar_wait(&ctl->kv_empty[stage], phase ^ 1u, p.ctrl, p.timeout_ns, kSiteEmpty, i)) {
          ok = false;
          break;
        }
        uint8_t* kt = smem + kOffKv + stage * 2 * kTileBytes;
        uint8_t* vt = kt + kTileBytes;
        mbar_arrive_expect_tx(&ctl->kv_full[stage], 2 * kTileBytes);
        for (int c = 0; c < 2; ++c) {
          tma_load_2d(kmap, kt + c * kHalfBytes, &ctl->kv_full[stage], it.h * kHd + c * 64, krow0 + kb * kKB);
          tma_load_2d(vmap, vt + c * kHalfBytes, &ctl->kv_full[stage], kb * kKB + c * 64, vrow0);
        }
        armed |= 1u << stage;
        armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kKvStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
  if (!ok) {
    if (q_armed) mbar_wait_drain(&ctl->q_full, q_armed_phase, kDrainNs);
    for (int s = 0; s < kKvStages; ++s)
      if ((armed >> s) & 1u) mbar_wait_drain(&ctl->kv_full[s], (armed_phase >> s) & 1u, kDrainNs);
  }
}

__device__ __forceinline__ void issue_s(uint32_t tmem_s, uint32_t q_addr, uint32_t k_addr) {
#pragma unroll
  for (int k = 0; k < kHd / 16; ++k) {
    const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
    umma_bf16_ss(tmem_s, umma_sdesc_sw128(q_addr + off), umma_sdesc_sw128(k_addr + off), kIdescS, k > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t p_addr, uint32_t v_addr, bool first) {
#pragma unroll
  for (int k = 0; k < kKB / 16; ++k) {
    const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
    umma_bf16_ss(tmem_o, umma_sdesc_sw128(p_addr + off), umma_sdesc_sw128(v_addr + off), kIdescO,
                 (first && k == 0) ? 0u : 1u);
  }
}

__device__ void attn_mma(const AttnParams& p, uint8_t* smem, AttnCtl* ctl, uint32_t tmem_base) {
  const uint32_t sbase = smem_u32(smem);
  uint32_t q_uses = 0, p_uses = 0;
  uint32_t g = 0;  // global key-block counter of this CTA
  bool issued = false, ok = true;
  for (int i = blockIdx.x; ok && i < p.total_items; i += gridDim.x) {
    const Item it = decode_item(p, i);
    const int n = item_blocks(p, it);
    if (!mbar_wait(&ctl->q_full, q_uses & 1u, p.ctrl, p.timeout_ns, kSiteFull, i)) break;
    ++q_uses;
    tc_fence_after();
    // S for block j: K of kv stage (g+j) % 2, score buffer (g+j) % 2
    auto issue_scores = [&](uint32_t gj) -> bool {
      const uint32_t st = gj % kKvStages, sb = gj & 1u;
      if (!mbar_wait(&ctl->kv_full[st], (gj / kKvStages) & 1u, p.ctrl, p.timeout_ns, kSiteFull, i)) return false;
      if (!mbar_wait(&ctl->s_empty[sb], ((gj >> 1) & 1u) ^ 1u, p.ctrl, p.timeout_ns, kSiteTmemEmpty, i))
        return false;
      tc_fence_after();
      issue_s(tmem_base + sb * 128, sbase + kOffQ, sbase + kOffKv + st * 2 * kTileBytes);
      issued = true;
      umma_commit(&ctl->s_full[sb]);
      return true;
    };
    if (!issue_scores(g)) {
      ok = false;
      break;
    }
    for (int j = 0; j < n; ++j) {
      const uint32_t gj = g + j;
      if (j + 1 < n) {
        if (!issue_scores(gj + 1)) {
          ok = false;
          break;
        }
      } else {
        umma_commit(&ctl->q_empty);  // Q is free once every score MMA of this item completes
      }
      if (!mbar_wait(&ctl->p_full, p_uses & 1u, p.ctrl, p.timeout_ns, kSiteFull, i)) {
        ok = false;
        break;
      }
      ++p_uses;
      tc_fence_after();
      const uint32_t st = gj % kKvStages;
      issue_pv(tmem_base + kOCol, sbase + kOffP, sbase + kOffKv + st * 2 * kTileBytes + kTileBytes, j == 0);
      umma_commit(&ctl->kv_empty[st]);
      umma_commit(&ctl->o_done);
    }
    g += n;
  }
  if (!ok && issued) {
    umma_commit(&ctl->drain);
    mbar_wait_drain(&ctl->drain, 0, kDrainNs);
  }
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const AttnParams& p, uint32_t site,
                                          uint32_t detail, int lane) {
  uint32_t ok = 0;
  if (lane == 0) ok = mbar_wait(bar, parity, p.ctrl, p.timeout_ns, site, detail) ? 1u : 0u;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ void attn_softmax(const AttnParams& p, uint8_t* smem, AttnCtl* ctl, uint32_t tmem_base, int warp,
                             int lane) {
  const int q = warp & 3;
  const int row = q * 32 + lane;  // query row inside the block == TMEM lane
  const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  uint8_t* prow = smem + kOffP + row * 128;
  uint32_t g = 0;
  for (int i = blockIdx.x; i < p.total_items; i += gridDim.x) {
    const Item it = decode_item(p, i);
    float m_ref = -INFINITY, l = 0.f;
    int j = 0;
    const int nsteps = steps_of(p, it.r);
    for (int t = 0; t < nsteps; ++t) {
      const int nb = blocks_of(p, it, t);
      for (int kb = 0; kb < nb; ++kb, ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj & 1u;
        if (!warp_wait(&ctl->s_full[sb], (gj >> 1) & 1u, p, kSiteTmemFull, i, lane)) return;
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_base + sb * 128 + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) s[c * 32 + k] = __uint_as_float(v[k]) * p.scale_log2;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->s_empty[sb]);
        const bool diag = p.causal && t == 0 && kb == it.qb;
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < 128; ++k) {
          if (diag && k > row) s[k] = -INFINITY;
          mx = fmaxf(mx, s[k]);
        }
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_ref = mx;
        } else if (mx > m_ref + kRescaleThreshold) {
          alpha = fast_exp2(m_ref - mx);
          m_ref = mx;
          l *= alpha;
          rescale = true;
        }
        // the row sum uses the fp16-rounded weights that the P.V product sees
        float sum = 0.f;
        uint32_t packed[64];
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          packed[k] = pack_f16x2(fast_exp2(s[2 * k] - m_ref), fast_exp2(s[2 * k + 1] - m_ref));
          const __half2 h = *reinterpret_cast<const __half2*>(&packed[k]);
          const float2 f = __half22float2(h);
          sum += f.x + f.y;
        }
        l += sum;
        if (j > 0) {
          // the previous P.V must be complete before P is overwritten or O rescaled
          if (!warp_wait(&ctl->o_done, (gj - 1) & 1u, p, kSiteDrain, i, lane)) return;
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(lane_base + kOCol + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(lane_base + kOCol + c * 32, v);
          }
          tmem_wait_st();
        }
        // P row -> two 128-byte-swizzled halves (keys 0-63, 64-127), 16-byte chunks
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int half = c >> 3, chunk = c & 7;
          uint4* dst = reinterpret_cast<uint4*>(prow + half * kHalfBytes + ((chunk ^ (row & 7)) << 4));
          *dst = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        }
        fence_proxy_async_shared();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full);
      }
    }
    // epilogue: O row / l -> bf16
    const uint32_t glast = g + j - 1;
    if (!warp_wait(&ctl->o_done, glast & 1u, p, kSiteDrain, i, lane)) return;
    tc_fence_after();
    const float inv = 1.f / l;
    uint16_t* orow = p.out[it.r] + static_cast<int64_t>(it.qb * kQB + row) * p.ld_out[it.r] + it.h * kHd;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t v[32];
      tmem_ld32(lane_base + kOCol + c * 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        st_v4_u32(orow + c * 32 + 8 * k,
                  pack_bf16x2(__uint_as_float(v[8 * k + 0]) * inv, __uint_as_float(v[8 * k + 1]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv));
      }
    }
    tc_fence_before();
    g += j;
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (base & 1023u)) & 1023u);
  AttnCtl* ctl = reinterpret_cast<AttnCtl*>(smem + kOffCtl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_empty, 1);
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&ctl->kv_full[s], 1);
      mbar_init(&ctl->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->s_full[b], 1);
      mbar_init(&ctl->s_empty[b], 4);
    }
    mbar_init(&ctl->p_full, 4);
    mbar_init(&ctl->o_done, 1);
    mbar_init(&ctl->drain, 1);
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < 4 * p.P; ++i) tma_prefetch_desc(&p.maps[i]);
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  if (warp == 0) {
    if (lane == 0) attn_producer(p, smem, ctl);
  } else if (warp == 1) {
    if (lane == 0) attn_mma(p, smem, ctl, tmem_base);
    __syncwarp();
  } else {
    attn_softmax(p, smem, ctl, tmem_base, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// V [m, heads*128] bf16 (row pitch ld) -> V^T [heads*128, m] fp16, 64x64 tiles
// through shared memory.  bf16 -> fp16 is exact inside fp16's normal range.
__global__ void transpose_kernel(const uint16_t* __restrict__ v, int64_t ld, uint16_t* __restrict__ vt, int64_t m,
                                 int64_t hd) {
  __shared__ uint16_t tile[64][66];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64;  // token
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 64;  // feature
  for (int i = threadIdx.y; i < 64; i += blockDim.y) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < m && c < hd) {
      const float f = __uint_as_float(static_cast<uint32_t>(v[r * ld + c]) << 16);
      tile[i][threadIdx.x] = __half_as_ushort(__float2half_rn(f));
    }
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 64; i += blockDim.y) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (r < m && c < hd) vt[c * m + r] = tile[threadIdx.x][i];
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

fo_status attn_run(fo_ctx* ctx, const fo_mat* Q, const fo_mat* K, const fo_mat* V, int P, int heads, int head_dim,
                   int causal, const fo_mat* O, const fo_opts* opts_in, cudaStream_t stream) {
  fo_opts o;
  if (opts_in) {
    o = *opts_in;
  } else {
    std::memset(&o, 0, sizeof(o));
  }
  if (o.order != FO_ORDER_FLASH) return host_fail(FO_ERR_UNSUPPORTED, "attention runs the ring order only");
  if (head_dim != kHd) return host_fail(FO_ERR_UNSUPPORTED, "head_dim must be 128");
  if (heads < 1) return host_fail(FO_ERR_INVALID_ARG, "heads must be positive");
  const int64_t m = Q[0].rows, HD = static_cast<int64_t>(heads) * kHd;
  for (int r = 0; r < P; ++r) {
    fo_status st;
    if ((st = host_check_mat(Q[r], FO_BF16, "Q", r)) != FO_OK) return st;
    if ((st = host_check_mat(K[r], FO_BF16, "K_shards", r)) != FO_OK) return st;
    if ((st = host_check_mat(V[r], FO_BF16, "V_shards", r)) != FO_OK) return st;
    if ((st = host_check_mat(O[r], FO_BF16, "O", r)) != FO_OK) return st;
    if (Q[r].rows != m || K[r].rows != m || V[r].rows != m || O[r].rows != m || Q[r].cols != HD ||
        K[r].cols != HD || V[r].cols != HD || O[r].cols != HD)
      return host_fail(FO_ERR_SHAPE, "Q/K/V/O shards must all be [m, heads*head_dim]");
  }
  if (m == 0) return FO_OK;
  if (m % kQB != 0) return host_fail(FO_ERR_UNSUPPORTED, "tokens per rank must be a multiple of 128");
  const int64_t M = m * P;
  void *kv = nullptr, *vt = nullptr;
  fo_status st;
  if ((st = host_buffer(ctx, 0, static_cast<size_t>(P) * M * HD * 2, &kv)) != FO_OK) return st;  // K received
  if ((st = host_buffer(ctx, 1, static_cast<size_t>(P) * P * HD * m * 2, &vt)) != FO_OK) return st;  // V^T slots
  uint32_t* flags = nullptr;
  if ((st = host_flags(ctx, &flags)) != FO_OK) return st;
  char* krecv = static_cast<char*>(kv);
  char* vtb = static_cast<char*>(vt);
  auto k_slot = [&](int r, int s) { return krecv + (static_cast<int64_t>(r) * M + s * m) * HD * 2; };
  auto vt_slot = [&](int r, int s) { return vtb + (static_cast<int64_t>(r) * P + s) * HD * m * 2; };

  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem) != cudaSuccess)
      return host_fail(FO_ERR_CUDA, "attention kernel configuration failed");
    configured = true;
  }
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < P; ++r) {
    if ((st = host_encode_map(&p.maps[r], Q[r].ptr, m, HD, Q[r].ld, kQB)) != FO_OK) return st;
    if ((st = host_encode_map(&p.maps[P + r], K[r].ptr, m, HD, K[r].ld, kKB)) != FO_OK) return st;
    if ((st = host_encode_map(&p.maps[2 * P + r], k_slot(r, 0), M, HD, HD, kKB)) != FO_OK) return st;
    if ((st = host_encode_map(&p.maps[3 * P + r], vt_slot(r, 0), static_cast<int64_t>(P) * HD, m, m, kHd,
                              CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != FO_OK)
      return st;
    p.out[r] = static_cast<uint16_t*>(O[r].ptr);
    p.ld_out[r] = O[r].ld;
  }
  const uint32_t epoch = host_next_epoch(ctx);
  p.P = P;
  p.heads = heads;
  p.nkb = static_cast<int32_t>(m / kKB);
  p.causal = causal ? 1 : 0;
  p.m = static_cast<int32_t>(m);
  p.total_items = P * p.nkb * heads;
  p.epoch = epoch;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHd)));
  p.timeout_ns = host_timeout_ns(o);
  p.flags = flags;
  p.ctrl = host_ctrl(ctx);

  // 1) every rank lays out its own V slice transposed (slot r of its V^T buffer)
  for (int r = 0; r < P; ++r) {
    dim3 grid(static_cast<unsigned>((HD + 63) / 64), static_cast<unsigned>((m + 63) / 64));
    transpose_kernel<<<grid, dim3(64, 8), 0, stream>>>(static_cast<const uint16_t*>(V[r].ptr), V[r].ld,
                                                       reinterpret_cast<uint16_t*>(vt_slot(r, r)), m, HD);
    if (cudaGetLastError() != cudaSuccess) return host_fail(FO_ERR_CUDA, "transpose launch failed");
  }
  // 2) the attention kernel, then 3) the K/V ring on the link streams, concurrently
  if ((st = host_fork(ctx, P, stream)) != FO_OK) return st;
  attn_kernel<<<host_grid(ctx, o, p.total_items), kAttnThreads, kAttnSmem, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return host_fail(FO_ERR_CUDA, "attention kernel launch failed");
  const bool prune = o.causal_prune && causal;
  for (int t = 1; t < P; ++t) {
    for (int r = 0; r < P; ++r) {
      const int d = (r + 1) % P;
      const int s = ((r - t + 1) % P + P) % P;
      if (prune && (d == 0 || d - t < 0)) continue;  // slice s is only needed by ranks above it
      // fault injection: the first hop into rank 1 (slice 0, which rank 1 always uses) is dropped
      if (o.fault == FO_FAULT_SKIP_HOP && t == 1 && r == 0) continue;
      cudaStream_t ls = host_link(ctx, r);
      if (t >= 2 && cudaStreamWaitEvent(ls, host_ev_hop(ctx, (r - 1 + P) % P, t - 1), 0) != cudaSuccess)
        return host_fail(FO_ERR_CUDA, "event wait failed");
      const void* ksrc = t == 1 ? K[r].ptr : k_slot(r, s);
      const int64_t kld = t == 1 ? K[r].ld : HD;
      if ((st = host_copy_rows(k_slot(d, s), HD, ksrc, kld, m, HD, 2, ls)) != FO_OK) return st;
      if ((st = host_copy_rows(vt_slot(d, s), m, vt_slot(r, s), m, HD, m, 2, ls)) != FO_OK) return st;
      if ((st = host_write_flag(ls, flags + d * P + s, epoch)) != FO_OK) return st;
      if (cudaEventRecord(host_ev_hop(ctx, r, t), ls) != cudaSuccess) return host_fail(FO_ERR_CUDA, "event failed");
    }
  }
  return host_join(ctx, P, stream);
}

}  // namespace fo
