/*
 * fo.h -- C ABI of the GB300 Flash-Overlap library.
 *
 * The method (FlashOverlap: Minimizing Tail Latency in Communication Overlap
 * for Distributed LLM Training, technical summary section 2 "Methodology")
 * replaces a tensor-parallel collective by ring point-to-point steps and
 * schedules the compute around them:
 *   - Flash-AG   all-gather -> column-parallel GEMM, local slice computed first;
 *   - Flash-RS   row-parallel GEMM -> reduce-scatter, the slice the rank keeps
 *                computed last (rank-adaptive scheduling);
 *   - query-split attention, whose K/V slices travel the ring like Flash-AG.
 *
 * Here all P "ranks" live on ONE GPU: rank r is a set of caller buffers plus a
 * disjoint arena of the context's workspace, and a ring hop is a device-local
 * copy (cudaMemcpyAsync on a link stream) or an epilogue store into the
 * successor's arena, signalled
 * through per-slice / per-tile flags in device memory.
 *
 * Conventions for every entry point
 *   - Matrices are row-major fo_mat views: element (i, j) at ptr + (i*ld + j)*size.
 *     Pointers are DEVICE pointers unless an entry point says otherwise, must be
 *     16-byte aligned, and ld*element_size must be a multiple of 16 bytes.
 *   - The caller owns every input and output buffer.  The context owns its
 *     workspace (ring receive slots, flags, intermediates) and grows it on demand.
 *   - Calls enqueue work on `stream` (a cudaStream_t, 0 = legacy default) and
 *     return without synchronising.  Argument errors are reported synchronously
 *     and nothing is enqueued.  Device-side failures (a wait that ran past its
 *     time limit) are reported by fo_ctx_poll after the stream has completed.
 *   - A context is not thread-safe; use one per host thread.  Calls on one
 *     context must be ordered (same stream, or streams the caller orders).
 *   - Weights use the nn.Linear layout [out_features, in_features].
 *   - Arithmetic: bf16 operands, fp32 accumulation (tensor cores), fp32 ring
 *     partials for reduce-scatter, outputs rounded once to bf16
 *     (round-to-nearest-even).
 */
#ifndef FO_H_
#define FO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FO_API __attribute__((visibility("default")))
#else
#define FO_API
#endif

typedef struct fo_ctx fo_ctx;

typedef enum {
  FO_OK = 0,
  FO_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, P out of range           */
  FO_ERR_SHAPE = 2,         /* shapes inconsistent across ranks or operands     */
  FO_ERR_UNSUPPORTED = 3,   /* valid but outside what the kernels handle        */
  FO_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed                */
  FO_ERR_TIMEOUT = 5,       /* a device wait ran past opts.timeout_us           */
  FO_ERR_OOM = 6,           /* workspace growth failed                          */
  FO_ERR_RANGE = 7,         /* an input value outside what a kernel represents  */
  FO_ERR_INTERNAL = 8       /* an index check of the debug build failed (a bug)  */
} fo_status;

typedef enum { FO_BF16 = 0, FO_F32 = 1 } fo_dtype;

typedef struct {
  void* ptr;       /* first element                                   */
  int32_t dtype;   /* fo_dtype                                        */
  int32_t reserved;
  int64_t rows;
  int64_t cols;
  int64_t ld;      /* elements between consecutive rows, >= cols      */
} fo_mat;

typedef enum {
  FO_ORDER_FLASH = 0,    /* the method: local-first AG, kept-slice-last RS, one fused launch    */
  FO_ORDER_NAIVE = 1,    /* RS only: every rank computes chunks in ascending index order         */
  FO_ORDER_SLICING = 2,  /* baseline: equal data slices, collective per slice, launch per slice  */
  FO_ORDER_SERIAL = 3    /* baseline: whole collective, then whole GEMM (or GEMM then collective) */
} fo_order;

typedef enum {
  FO_LINK_DEFAULT = 0, /* all-gather: FO_LINK_CE; fused reduce-scatter: FO_LINK_PUSH      */
  FO_LINK_CE = 1,      /* hop = device-to-device cudaMemcpyAsync on a per-rank link stream */
  FO_LINK_PUSH = 2     /* RS only: the epilogue stores the partial sum straight into the
                          successor's receive slot and releases a per-tile flag          */
} fo_link;

typedef enum {
  FO_FAULT_NONE = 0,
  FO_FAULT_SKIP_HOP = 1  /* fault injection (host side): one ring hop into rank 1 is not
                            enqueued (all-gather: the last hop from rank 0; attention: the
                            first), so a device wait runs out; the call must end with
                            FO_ERR_TIMEOUT from fo_ctx_poll and the context stays usable */
} fo_fault;

typedef enum {
  FO_EPI_PLAIN = 0,      /* Y = X W^T (bf16)                                                */
  FO_EPI_SILU_GATE = 1   /* W_col[r] = [gate rows; up rows] ([2F, K]); Y[r] = SiLU(gate) * up,
                            [M, F], each of gate/up rounded to bf16 first (MLP glue fused)  */
} fo_epilogue;

typedef struct {
  int32_t order;        /* fo_order                                                   */
  int32_t link;         /* fo_link; all-gather hops are always cudaMemcpyAsync copies   */
  int32_t n_slices;     /* FO_ORDER_SLICING: number of slices (0 = P)                 */
  uint32_t timeout_us;  /* limit of every device-side wait (0 = 1 second)             */
  int32_t causal_prune; /* attention: forward a K/V slice only to ranks that use it   */
  int32_t num_sms;      /* persistent grid size cap (0 = every SM)                    */
  int32_t fault;        /* fo_fault                                                   */
  int32_t epilogue;     /* fo_epilogue (fo_ag_gemm only)                              */
  int32_t sm_pairs;     /* GEMM tiles: 0 = automatic (256x256 tiles on SM pairs when every
                           unit's rows are a multiple of 256; the transposed reduce-scatter
                           tiles of 32-128-row slices on single SMs, measured faster there),
                           1 = single-SM 128x256 tiles everywhere, 2 = SM pairs wherever a
                           tile kind has that form (transposed tiles included) */
  int32_t compute_only; /* timing diagnostic (fo_ag_gemm, fo_gemm_rs, fo_qsplit_attn): every
                           kernel of the chosen order runs, every ring flag is published
                           before the launch and no ring copy is enqueued, so the call takes
                           the compute time of that order with the transfers removed.  The
                           receive buffers keep whatever an earlier call left in them: the
                           results are meaningless.  Not accepted with host buffers. */
  int32_t split_layer;  /* fo_mlp_layer / fo_mlp_layer_host: 0 = one persistent launch for
                           Flash-AG -> activation -> Flash-RS when the layer fits one launch
                           (the reduce-scatter's tiles wait per 256-row block for the rows
                           of the intermediate they read), 1 = two launches */
  int32_t reserved;
} fo_opts;

/* Version of this ABI (major*100 + minor). */
FO_API int fo_version(void);

/* Text of the last error raised on this host thread ("" if none).  Valid until
 * the next call on this thread. */
FO_API const char* fo_last_error_string(void);

/* Creates a context on CUDA device `device` (made current for the call).
 * Allocates the link streams, events and a small device control block; the
 * ring workspace is allocated on first use.  *out receives the context. */
FO_API fo_status fo_ctx_create(int device, fo_ctx** out);

/* Synchronises the context's streams, frees its workspace.  NULL is a no-op. */
FO_API fo_status fo_ctx_destroy(fo_ctx* ctx);

/* Reads the device error word after the caller has synchronised the stream of
 * the previous calls, and clears it.  FO_OK; FO_ERR_TIMEOUT when a device wait
 * gave up (the work of that call is then incomplete); FO_ERR_RANGE when an input
 * held a value the kernels cannot represent (see fo_qsplit_attn).  After a
 * FO_ERR_TIMEOUT, call this before the next call on the context: until then the
 * device keeps the failure's abort word set (later kernels leave their loops at
 * once) and the launch-wide work counters of the failed launch uncleared; this
 * call clears the whole control block. */
FO_API fo_status fo_ctx_poll(fo_ctx* ctx);

/* Device milliseconds of the two phases of the last FO_ORDER_SERIAL call on
 * this context: the ring collective alone and the GEMM alone (valid once that
 * call's stream has completed). */
FO_API fo_status fo_ctx_phase_ms(fo_ctx* ctx, float* collective_ms, float* gemm_ms);

/* Launch order of the fused ring launches, for inspection (host only, no GPU):
 * op 0 = Flash-AG (order FO_ORDER_FLASH), op 1 = Flash-RS, op 2 = the all-to-all's
 * producer GEMM (fo_gemm_a2a), op 3 = its consumer GEMM (fo_a2a_gemm); ops 1-3 take
 * FO_ORDER_FLASH or FO_ORDER_NAIVE.  Unit i of step t is written at index t*P + i:
 * rank[] gets the rank, item[] the slice (AG), chunk (RS), destination block (op 2) or
 * source chunk (op 3) it computes.  Returns P*P, or -1 on a bad argument (capacity <
 * P*P included).  Follows the technical summary's section 2: AG step 0 is the rank's
 * own slice; RS step P-1 is the rank's kept chunk; the all-to-all's producer computes
 * its own block last and its consumer its own chunk first. */
FO_API int fo_step_order(int op, int P, int order, int32_t* rank, int32_t* item, int capacity);

/* Plain GEMM on the tensor cores, C = A * B^T (no ring):
 * A [M, K] bf16, B [N, K] bf16, C [M, N] bf16 or fp32.  K % 8 == 0. */
FO_API fo_status fo_gemm(fo_ctx* ctx, const fo_mat* A, const fo_mat* B, const fo_mat* C,
                  const fo_opts* opts, void* stream);

/* Flash-AG (technical summary section 2, "Flash-All-Gather"): all-gather of the
 * sequence-sharded activations followed by the column-parallel GEMM.
 *   X_shards[r]  [m, K]  bf16   rank r's token slice (m = M/P rows)
 *   W_col[r]     [N, K]  bf16   rank r's column block of the weight
 *   Y[r]         [M, N]  bf16   rank r's output over all M = P*m tokens
 * Ring: at hop t (1..P-1) rank r forwards slice (r-t+1) mod P to rank r+1.
 * Rank r computes slice (r-t) mod P at step t, so step 0 is its own slice. */
FO_API fo_status fo_ag_gemm(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_col, int P,
                     const fo_mat* Y, const fo_opts* opts, void* stream);

/* Flash-RS (technical summary section 2, "Flash-Reduce-Scatter"): row-parallel
 * GEMM followed by the reduce-scatter of the partial sums.
 *   X[r]      [M, Kr] bf16   rank r's in-feature shard of the activations
 *   W_row[r]  [N, Kr] bf16   rank r's in-feature shard of the weight
 *   Y[r]      [m, N]  bf16   rank r's token slice of sum_r X[r] W_row[r]^T
 * At step t rank r computes chunk c = (r-t-1) mod P, adds the fp32 partial sum
 * received from rank r-1 and passes it to rank r+1; at t = P-1, c = r (the kept
 * slice) and the sum is rounded into Y[r].  FO_ORDER_NAIVE keeps the ring but
 * makes every rank compute chunk t at step t. */
FO_API fo_status fo_gemm_rs(fo_ctx* ctx, const fo_mat* X, const fo_mat* W_row, int P,
                     const fo_mat* Y, const fo_opts* opts, void* stream);

/* MLP activation glue: H = SiLU(G) * U elementwise, with G = columns [0, F) and
 * U = columns [F, 2F) of GU[r] ([M, 2F] bf16); H[r] [M, F] bf16.  Computed in
 * fp32 from the bf16 inputs, rounded once. */
FO_API fo_status fo_silu_mul(fo_ctx* ctx, const fo_mat* GU, int P, const fo_mat* H, void* stream);

/* One MLP layer (technical summary section 2, "Row/Column Parallel Projection"):
 * Flash-AG with W_col (gate rows then up rows when gated), SiLU(gate)*up when
 * gated (identity otherwise), then Flash-RS with W_row.
 *   X_shards[r] [m, Hd] bf16; W_col[r] [Nc, Hd]; W_row[r] [Hd, F_r] bf16 with
 *   F_r = Nc/2 (gated) or Nc; Z[r] [m, Hd] bf16 (rank r's token slice).
 * Intermediates live in the context's workspace. */
FO_API fo_status fo_mlp_layer(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_col,
                       const fo_mat* W_row, int P, int gated, const fo_mat* Z,
                       const fo_opts* opts, void* stream);

/* fo_mlp_layer with HOST activations: X_shards[r].ptr and Z[r].ptr point to host
 * memory (page-locked for asynchronous copies); weights are device pointers.
 * The call enqueues the host->device copies of X, the layer and the
 * device->host copies of Z on `stream`. */
FO_API fo_status fo_mlp_layer_host(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_col,
                            const fo_mat* W_row, int P, int gated, const fo_mat* Z,
                            const fo_opts* opts, void* stream);

/* Query-split attention (technical summary section 2, "Query Split Attention"):
 * rank r keeps its query slice; K/V slices travel the ring local-first.
 *   Q[r], K_shards[r], V_shards[r], O[r]: [m, heads*head_dim] bf16, token-major,
 *   head_dim contiguous.  head_dim == 128.  Scale 1/sqrt(head_dim).
 *   causal != 0: key j attends query i only if j <= i (global token indices);
 *   slices wholly above the diagonal are skipped.
 * Softmax statistics and the output accumulator are fp32 (online softmax).
 * The P.V product runs on fp16 tensor cores: V is converted from bf16 to fp16,
 * which is exact for |v| in [2^-14, 65504] and for 0.  A finite |v| above 65504
 * would become infinite: the conversion counts such values and the call then
 * ends with FO_ERR_RANGE from fo_ctx_poll (the outputs of that call are not
 * valid).  Nonzero |v| below 2^-14 keep fp16's subnormal precision (absolute
 * error at most 2^-25 in V, hence in O). 
 * opts->order: FO_ORDER_FLASH (the ring runs while the kernel computes) or
 * FO_ORDER_SERIAL (baseline: the whole K/V ring first, then the kernel). */
FO_API fo_status fo_qsplit_attn(fo_ctx* ctx, const fo_mat* Q, const fo_mat* K_shards,
                         const fo_mat* V_shards, int P, int heads, int head_dim, int causal,
                         const fo_mat* O, const fo_opts* opts, void* stream);

/* Flash all-to-all, producer side (technical summary section 2: Flash All-to-All,
 * the extension of the decomposition to the all-to-all of Ulysses parallelism): a
 * GEMM whose output blocks belong to other ranks.
 *   X_shards[r] [m, K] bf16; W[r] [N, K] bf16, N = P*Nb; Y[d] [P*m, Nb] bf16.
 *   Y[d][rows r*m..] = X_shards[r] W[r][rows d*Nb..]^T (rank r's block d goes to rank d).
 * FO_ORDER_FLASH: at step t rank r computes the block of rank (r + t + 1) mod P, its
 * own block last; each tile is stored straight into the destination's buffer (the hop
 * is the epilogue store).  FO_ORDER_NAIVE: block t at step t.  FO_ORDER_SERIAL
 * (baseline): the GEMM into a workspace buffer, then the all-to-all as copies. */
FO_API fo_status fo_gemm_a2a(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W, int P,
                      const fo_mat* Y, const fo_opts* opts, void* stream);

/* Flash all-to-all, consumer side: the all-to-all in front of a GEMM whose K
 * dimension is split over the source ranks.
 *   C[s] [P*m, Kc] bf16: rows d*m.. hold source s's K chunk for rank d (Kc % 64 == 0);
 *   W[d] [N, P*Kc] bf16 (K chunk s at columns s*Kc..); Y[d] [m, N] bf16.
 *   Y[d] = [C[0] rows d*m.. | ... | C[P-1] rows d*m..] W[d]^T.
 * Hops: at step t (1..P-1) rank s copies its chunk for rank (s + t) mod P into that
 * rank's receive slot and publishes an arrival flag.  FO_ORDER_FLASH: rank d folds in
 * its own chunk first, then each received chunk as it arrives (source d-1, d-2, ...),
 * inside one K loop.  FO_ORDER_NAIVE: chunks in ascending source order.
 * FO_ORDER_SERIAL (baseline): every copy first, then the GEMM. */
FO_API fo_status fo_a2a_gemm(fo_ctx* ctx, const fo_mat* C, const fo_mat* W, int P, const fo_mat* Y,
                      const fo_opts* opts, void* stream);

/* Training backward of a column-parallel projection (forward: Y[r] = AG(X) W_col[r]^T,
 * as fo_ag_gemm).  The all-gather's adjoint is a reduce-scatter, so the input gradient is
 * Flash-RS with the transposed weight (technical summary section 2: the same
 * decomposed collectives; the title's training setting).
 *   X_shards[r] [m, K]; W_col[r] [Nr, K]; dY[r] [P*m, Nr]            (inputs, bf16)
 *   dX[d] [m, K] = sum_r dY[r][rows d*m..] W_col[r]                  (Flash-RS)
 *   dW[r] [Nr, K] = dY[r]^T AG(X)                                     (local GEMM)
 * Nr and P*m multiples of 8.  W_col^T, dY^T and AG(X)^T are not materialised: the
 * tensor cores read W_col, dY and the token slices in place as MN-major operands (only
 * the P token slices are stacked into one workspace buffer for the weight gradient);
 * opts->order applies to the reduce-scatter. */
FO_API fo_status fo_col_linear_backward(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_col,
                                 const fo_mat* dY, int P, const fo_mat* dX, const fo_mat* dW,
                                 const fo_opts* opts, void* stream);

/* Training backward of a row-parallel projection (forward: Z = RS(H[r] W_row[r]^T), as
 * fo_gemm_rs).  The reduce-scatter's adjoint is an all-gather: the input gradient is
 * Flash-AG with the transposed weight.
 *   H[r] [P*m, Fr]; W_row[r] [N, Fr]; dZ_shards[d] [m, N]            (inputs, bf16)
 *   dH[r] [P*m, Fr] = AG(dZ) W_row[r]                                 (Flash-AG)
 *   dW[r] [N, Fr] = AG(dZ)^T H[r]                                     (local GEMM)
 * N and P*m multiples of 8; opts->order applies to the all-gather. */
FO_API fo_status fo_row_linear_backward(fo_ctx* ctx, const fo_mat* H, const fo_mat* W_row,
                                 const fo_mat* dZ_shards, int P, const fo_mat* dH, const fo_mat* dW,
                                 const fo_opts* opts, void* stream);

/* One attention block in the layout of the MLP layer (technical summary section 2:
 * the QKV projection is a column-parallel GEMM after an all-gather, the output
 * projection a row-parallel GEMM before a reduce-scatter): Flash-AG with W_qkv,
 * causal multi-head attention of every rank's own heads over all M = P*m tokens
 * (independent per rank, no ring: a rank holds the whole sequence of its heads),
 * then Flash-RS with W_o.
 *   X_shards[r] [m, Hd] bf16 (rank r's token slice of the block input)
 *   W_qkv[r]    [3*heads*head_dim, Hd] bf16: rank r's heads, Q rows, then K rows,
 *               then V rows (head h at rows h*head_dim.. of each part)
 *   W_o[r]      [Hd, heads*head_dim] bf16: the output projection's columns of
 *               rank r's heads
 *   Z[r]        [m, Hd] bf16 (rank r's token slice of the block output)
 * heads = heads per rank, head_dim == 128, M % 128 == 0.  QKV (bf16) and the
 * attention output (bf16) live in the context's workspace.  opts->order applies to
 * the two GEMMs as in fo_mlp_layer. */
FO_API fo_status fo_attn_layer(fo_ctx* ctx, const fo_mat* X_shards, const fo_mat* W_qkv,
                        const fo_mat* W_o, int P, int heads, int head_dim, int causal,
                        const fo_mat* Z, const fo_opts* opts, void* stream);

/* Flash-RS (as fo_gemm_rs, FO_ORDER_FLASH) for callers that cannot allocate
 * device memory.  (No counterpart on the pages: this is a deployment variant.)
 * fo_gemm_rs keeps its ring scratch -- fp32 receive slots and per-tile flags --
 * in a context that allocates it with cudaMalloc.  Callers whose device memory
 * is owned entirely by their own allocator, or that must not pay the
 * device-wide synchronisation of cudaMalloc/cudaFree on a latency-critical
 * path, cannot do that.  This entry point allocates nothing and needs no
 * context: its scratch is a fixed 64 MiB device array inside the library,
 * which every GPU that loads the library holds until the process exits.
 *   X, W_row, Y, P  as fo_gemm_rs (device pointers, caller-owned).
 *   timeout_us      limit of every device-side wait (0 = 1 second).
 *   status          optional device uint32: receives 0 or FO_ERR_TIMEOUT when
 *                   the call's work has completed on `stream` (NULL: none).
 * Shapes whose receive slots (P*(P-1)*m*N*4 bytes) or flags exceed the static
 * area are rejected with FO_ERR_UNSUPPORTED.  The first call on a device does a
 * one-time set-up (it configures the kernel with that device current).  Every
 * call asks for the array's device
 * address with the caller's device current (in host code the array's name is
 * only a stand-in).  Every call shares the array, which keeps the previous
 * call's contents: each call first clears, on `stream`, the control words and
 * the flag words it uses, so no call depends on what an earlier one left.  Calls
 * whose work overlaps on the GPU race on the array, so order them on one stream;
 * host threads that use one device at once must order their calls too.
 * The persistent kernel's CTAs wait on one another (a tile waits for the partial
 * sum of a tile of smaller index), so all of them must be resident at once: the
 * call needs the whole GPU while it runs.  Kernels running beside it can leave
 * some CTAs unscheduled; the waiting ones then give up after timeout_us and the
 * status reads FO_ERR_TIMEOUT. */
FO_API fo_status fo_gemm_rs_noalloc(const fo_mat* X, const fo_mat* W_row, int P, const fo_mat* Y,
                                    uint32_t timeout_us, uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FO_H_ */
