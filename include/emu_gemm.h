/*
 * emu_gemm.h -- FP32 GEMM emulated on GB300 (sm_103a) tensor cores.
 *
 * C ABI of libemu_gemm.so.  Two emulation modes, from the NVIDIA blog post
 * "Unlocking Tensor Core performance for machine-learning interatomic
 * potentials", section "How Tensor Core FP32 bridges the hardware gap":
 *
 *   EMU_MODE_BF16X9 (Fig. 1): every FP32 operand is split into three scaled
 *     BF16 components; the nine pairwise component products are evaluated on
 *     the tensor cores and accumulated in FP32 along the five anti-diagonal
 *     bands, smallest band first.
 *   EMU_MODE_TF32X3 (Fig. 2, Eq. 1): every operand is split into a leading
 *     and a residual TF32 component; a*b ~= a_hi b_hi + a_hi b_lo + a_lo b_hi
 *     (the residual*residual product is dropped), accumulated in FP32.
 *
 * FP32 in, FP32 out: the linear-layer entry points behave like nn.Linear, and
 * only the inner matrix product changes (section "TF32x3 on Ampere GPUs":
 * the layer keeps its weights, bias and shapes; the input gradient also runs
 * emulated, because forces are derivatives of the energy).
 *
 * Conventions (the blog leaves these open):
 *   - Layout: ROW-MAJOR, as in PyTorch (BLAS is column-major).  Element (i, j)
 *     of an R x C matrix X with leading dimension ldx is X[i * ldx + j].
 *   - op(X) = X when the op is EMU_OP_N, X^T when it is EMU_OP_T.
 *   - Pointers: caller-owned DEVICE memory of the current CUDA device.  The
 *     library keeps no caller pointer after the call returns and never frees
 *     caller memory.  Its only device allocations are a split-K workspace
 *     (partial tiles and arrival counters for problems with few tiles) and,
 *     for the TF32 modes, a buffer for op(B) split ahead of the product (when
 *     op(A) spans four or more 256-row tiles; EMU_AUTOPACK=0 turns that off),
 *     made with cudaMallocAsync on first need per (device, stream) and kept
 *     until emu_shutdown() or the end of the process; emu_sgemm_noalloc never
 *     allocates.  The library tracks at most 64 (device, stream) pairs with
 *     such buffers at once: a call that would need a 65th returns
 *     EMU_STATUS_ALLOC_FAILED (emu_shutdown() releases all of them).
 *   - Alignment (TMA): A and B must start on a 16-byte boundary and lda, ldb
 *     must be multiples of 4 elements; C the same (ldc multiple of 4).
 *     Violations return EMU_STATUS_NOT_SUPPORTED.
 *   - Execution: asynchronous on `stream` (NULL = the legacy default stream).
 *     All argument checks happen on the host before anything is enqueued;
 *     a call that returns an error has enqueued nothing.
 *   - Degenerate sizes: M == 0 or N == 0 is a no-op; K == 0 or alpha == 0
 *     gives C = beta * C (+ bias).  beta == 0 never reads C, so C may hold NaN.
 *   - Accuracy: BF16x9 results lie within 2*K*2^-24 * (|alpha| |op(A)||op(B)|
 *     + |beta||C| + |bias|) of the exact result, elementwise; TF32x3 within
 *     4*K*2^-24 times the same; EMU_MODE_FP32 within the usual bound of a
 *     sequential FP32 sum and its epilogue, (K+3)*2^-24 / (1 - (K+3)*2^-24)
 *     times the same.  Inputs must be finite: the split of an Inf
 *     produces NaN components (Inf - Inf), so Inf is not propagated as IEEE
 *     arithmetic would.  BF16 components below 2^-133 are lost, so inputs
 *     with |x| < 2^-110 are represented with reduced relative precision.
 *   - Errors: no exception crosses the ABI.  A kernel whose internal waits
 *     time out records a device-side flag instead of hanging and returns; it
 *     is reported as EMU_STATUS_DEVICE_TIMEOUT by the next emu_stream_check()
 *     on the device (the GEMM calls themselves do not read it).  A timed-out
 *     launch's output is incomplete; later launches are unaffected (the
 *     split-K arrival counters are tagged per launch).
 *   - Thread safety: all entry points may be called concurrently from
 *     several host threads.
 */
#ifndef EMU_GEMM_H
#define EMU_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (struct CUstream_st *); declared here so the
 * header does not need the CUDA headers. */
typedef struct CUstream_st *emu_stream_t;

typedef enum {
    EMU_MODE_BF16X9 = 0, /* three BF16 components, nine products, five bands (Fig. 1) */
    EMU_MODE_TF32X3 = 1, /* two TF32 components, three products (Fig. 2, Eq. 1) */
    /* Comparators, faster and less accurate: */
    EMU_MODE_TF32X1 = 2, /* one-pass TF32: hi(a) hi(b) only ("TF32x3 on Ampere GPUs": the one-pass
                            mode whose force jitter and drift the blog reports); error up to
                            2^-10 |a||b| per product */
    EMU_MODE_BF16X6 = 3, /* BF16x9 without bands 3 and 4 (six products); error up to 2^-20 |a||b| */
    /* Native FP32, the performant strategy's choice for small products: */
    EMU_MODE_FP32 = 4    /* CUDA cores, no tensor cores: each output is one chain of fmaf over
                            k = 0, 1, ..., K-1 from +0, then the epilogue.  No packed form;
                            N above 4,194,240 is NOT_SUPPORTED. */
} emu_mode_t;

typedef enum { EMU_OP_N = 0, EMU_OP_T = 1 } emu_op_t;

typedef enum {
    EMU_STATUS_SUCCESS = 0,
    EMU_STATUS_INVALID_VALUE = 1,   /* negative size, ld too small, NULL with non-zero size, bad enum */
    EMU_STATUS_NOT_SUPPORTED = 2,   /* pointer or leading dimension not aligned for TMA; size too large */
    EMU_STATUS_ARCH_MISMATCH = 3,   /* current device is not compute capability 10.3 (the library holds
                                       sm_103a code only) */
    EMU_STATUS_ALLOC_FAILED = 4,    /* a library buffer (split-K workspace, pre-split op(B)) could not be
                                       allocated, or the 64 (device, stream) slots are taken */
    EMU_STATUS_LAUNCH_FAILED = 5,   /* a CUDA call failed (no device, launch error, TMA encode error) */
    EMU_STATUS_DEVICE_TIMEOUT = 6   /* a kernel gave up on an internal wait and returned early */
} emu_status_t;

/*
 * emu_sgemm -- C = alpha * op(A) * op(B) + beta * C.
 *   op(A) is M x K, op(B) is K x N, C is M x N, all FP32, row-major.
 *   A: M x K (lda >= K) when transA == EMU_OP_N, K x M (lda >= M) when EMU_OP_T.
 *   B: K x N (ldb >= N) when transB == EMU_OP_N, N x K (ldb >= K) when EMU_OP_T.
 *   C: read only when beta != 0 (ldc >= N).  C must not overlap A or B.
 * Blog: "How Tensor Core FP32 bridges the hardware gap" (Fig. 1, Fig. 2, Eq. 1);
 * the SGEMM form is how the blog applies BF16x9 to unchanged models ("BF16x9
 * on Blackwell GPUs").
 */
emu_status_t emu_sgemm(emu_mode_t mode, emu_op_t transA, emu_op_t transB,
                       int64_t M, int64_t N, int64_t K,
                       float alpha, const float *A, int64_t lda,
                       const float *B, int64_t ldb,
                       float beta, float *C, int64_t ldc, emu_stream_t stream);

/*
 * emu_linear_fwd -- Y[M,N] = X[M,K] * W[N,K]^T + bias[N]   (bias may be NULL).
 *   X, W, Y dense row-major (leading dimensions K, K, N).  The forward pass
 *   of a linear layer with the layer's own weight layout (nn.Linear keeps W
 *   as out_features x in_features).  Blog: "TF32x3 on Ampere GPUs" (the
 *   layer keeps FP32 weights, bias and shapes; only the matmul changes).
 */
emu_status_t emu_linear_fwd(emu_mode_t mode, int64_t M, int64_t N, int64_t K,
                            const float *X, const float *W, const float *bias,
                            float *Y, emu_stream_t stream);

/*
 * emu_linear_bwd_input -- dX[M,K] = dY[M,N] * W[N,K].
 *   The input-gradient pass of the same layer, emulated as well (blog,
 *   "TF32x3 on Ampere GPUs": forces are derivatives of the energy, so the
 *   gradient to the layer input uses the emulated arithmetic too).  All
 *   operands dense row-major.  The weight gradient has its own call,
 *   emu_linear_bwd_weight.
 */
emu_status_t emu_linear_bwd_input(emu_mode_t mode, int64_t M, int64_t N, int64_t K,
                                  const float *dY, const float *W, float *dX,
                                  emu_stream_t stream);

/*
 * emu_linear_bwd_weight -- dW[N,K] = dY[M,N]^T * X[M,K] + beta * dW.
 *   The weight-gradient pass of the same layer, emulated: the contraction
 *   runs over the M tokens.  The blog computes this pass with standard FP32
 *   ("TF32x3 on Ampere GPUs": not needed for fixed-weight inference); it is
 *   offered here for training with the same arithmetic.  beta = 1
 *   accumulates into an existing gradient; beta = 0 never reads dW.
 */
emu_status_t emu_linear_bwd_weight(emu_mode_t mode, int64_t M, int64_t N, int64_t K,
                                   const float *dY, const float *X, float beta, float *dW,
                                   emu_stream_t stream);

/*
 * Weight pre-split ("packing") for fixed operands -- inference and
 * molecular dynamics, where a layer's weights do not change between calls:
 * the operand is split into the mode's components once, and later products
 * load the components directly (no per-call split of that operand, fewer
 * shared-memory bytes per k-stage).  Results are the same bits as the
 * unpacked calls.  Splitting a fixed weight once saves per-call work
 * where the blog's performant strategy ("BF16x9 on Blackwell GPUs") saves
 * it by choosing native FP32 (see emu_set_strategy).
 *
 * emu_pack_bytes -- device bytes a packed op(B) of N x K (output width N,
 *   contraction K) takes in `mode`: ncomp * N * Kp * elem, Kp = K rounded up
 *   to 32, elem 2 (BF16 modes) or 4 (TF32 modes), ncomp 3 / 2 / 1.  -1 for an
 *   invalid mode, EMU_MODE_FP32 or a negative size.  The packing calls return
 *   INVALID_VALUE for EMU_MODE_FP32.
 * emu_pack_b -- write the packed form of op(B) (K x N; transB as in
 *   emu_sgemm, B row-major with leading dimension ldb, device memory) to
 *   `packed` (device memory, emu_pack_bytes bytes, 16-byte aligned,
 *   caller-owned).  Layout: component planes of op(B)^T, N rows of Kp
 *   elements each (zero past K).  Asynchronous on `stream`.
 * emu_sgemm_packed_b -- C = alpha * op(A) * packed(op(B)) + beta * C; the
 *   other arguments as emu_sgemm; `packed_b` made by emu_pack_b with the
 *   same mode, N and K.
 * emu_linear_fwd_packed -- Y = X W^T + bias with W packed by
 *   emu_pack_b(mode, EMU_OP_T, N, K, W, K, ...).
 * emu_linear_bwd_input_packed -- dX = dY W with W packed by
 *   emu_pack_b(mode, EMU_OP_N, K, N, W, K, ...) (output width K,
 *   contraction N).
 * A packed buffer carries no header: passing one made for another mode, N or
 * K gives wrong results (or reads past it), not an error.
 */
int64_t emu_pack_bytes(emu_mode_t mode, int64_t N, int64_t K);
emu_status_t emu_pack_b(emu_mode_t mode, emu_op_t transB, int64_t N, int64_t K, const float *B,
                        int64_t ldb, void *packed, emu_stream_t stream);
emu_status_t emu_sgemm_packed_b(emu_mode_t mode, emu_op_t transA, int64_t M, int64_t N, int64_t K,
                                float alpha, const float *A, int64_t lda, const void *packed_b,
                                float beta, float *C, int64_t ldc, emu_stream_t stream);
emu_status_t emu_linear_fwd_packed(emu_mode_t mode, int64_t M, int64_t N, int64_t K, const float *X,
                                   const void *W_packed, const float *bias, float *Y,
                                   emu_stream_t stream);
emu_status_t emu_linear_bwd_input_packed(emu_mode_t mode, int64_t M, int64_t N, int64_t K,
                                         const float *dY, const void *Wt_packed, float *dX,
                                         emu_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *emu_status_string(emu_status_t s);

/*
 * emu_stream_check -- synchronise `stream`, then report and clear the
 * device-side timeout flag of the current device: EMU_STATUS_DEVICE_TIMEOUT
 * if a kernel gave up on a wait since the last check, EMU_STATUS_LAUNCH_FAILED
 * on a CUDA error, EMU_STATUS_SUCCESS otherwise.
 */
emu_status_t emu_stream_check(emu_stream_t stream);

/*
 * emu_split_dump -- diagnostic: run the kernels' own operand split on an
 * R x Kc FP32 matrix X (row-major, ldx, device memory; Kc <= 32 columns of
 * one k-block) and write the components the MMA would read, as raw bit
 * patterns, to `out` (device memory):
 *   BF16X9: 3 planes of R x Kc uint16 (BF16 words, band scale applied:
 *           component i equals the scaled component times 2^-8i);
 *   TF32X3: 2 planes of R x Kc uint32 (hi, lo as FP32 words).
 * mn_major != 0 feeds X through the transposing (MN-major) split path as
 * the K x R matrix X^T stored row-major with ldx >= R.
 * R <= 128.  Same alignment rules as emu_sgemm.
 */
emu_status_t emu_split_dump(emu_mode_t mode, int64_t R, int64_t Kc, const float *X, int64_t ldx,
                            int mn_major, void *out, emu_stream_t stream);

/*
 * emu_sgemm_noalloc -- emu_sgemm for callers that cannot allocate device
 * memory: applications that hand all device memory to their own pre-sized
 * pool or allocator and forbid driver allocations behind its back,
 * latency-critical loops that must not enter the driver's allocator (which
 * can block or synchronise), and callers that must never fail with an
 * out-of-memory error in the middle of a run.  The blog has no counterpart;
 * this is an engineering entry point of this library.
 *
 * Same arguments, same plan and same kernel as emu_sgemm (results are the
 * same bits).  The only device memory emu_sgemm may allocate is the split-K
 * scratch (partial tiles and counters for problems with few tiles, running
 * sums and counters for chained plans); here it lives in a fixed 64 MiB
 * device array inside the library instead.  The array is reserved on every
 * GPU that loads the library and kept until the process exits.
 *   - Size limit: a plan that splits some tiles into S pieces needs
 *     (split tiles) * S * 256 KiB, a chained plan that cuts tiles
 *     (pairs - 1) * 256 KiB (19 MiB with 76 pairs), each + 16 bytes per
 *     tile (tiles = ceil(M/256) * ceil(N/256)); if that exceeds 64 MiB the
 *     call returns EMU_STATUS_NOT_SUPPORTED and enqueues nothing.  Plans
 *     without a split or a cut use no scratch and are never rejected for
 *     size.
 *   - Allocation: none (no cudaMalloc/cudaFree, no allocating library
 *     routine).  The call enqueues one cudaMemsetAsync of the counters (the
 *     array keeps the previous call's contents, and the counters are cleared
 *     on every call) and the kernel.
 *   - First call per device: looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make this first call
 *     before any stream capture.
 *   - Concurrency: every call on a device shares the one array, so calls
 *     whose executions overlap on the GPU (different streams, or concurrent
 *     graph branches) race and corrupt each other's split-K partials;
 *     serialise them (one stream, or events).
 * Errors as for emu_sgemm.
 */
emu_status_t emu_sgemm_noalloc(emu_mode_t mode, emu_op_t transA, emu_op_t transB,
                               int64_t M, int64_t N, int64_t K,
                               float alpha, const float *A, int64_t lda,
                               const float *B, int64_t ldb,
                               float beta, float *C, int64_t ldc, emu_stream_t stream);

/*
 * emu_selftest_wait_timeout -- diagnostic for the device-side failure path:
 * launches one warp that waits, through the same bounded-wait routine as the
 * GEMM kernels, on a barrier that nothing ever completes.  After budget_ns
 * nanoseconds (0 < budget_ns <= 10 s) the wait gives up and the kernel
 * returns; the next emu_stream_check() on this stream reports
 * EMU_STATUS_DEVICE_TIMEOUT and clears the flag.  No fault, trap or hang.
 */
emu_status_t emu_selftest_wait_timeout(uint64_t budget_ns, emu_stream_t stream);

/*
 * emu_selftest_split_timeout -- diagnostic for the split-K counters after a
 * device timeout: takes the split-K workspace of (current device, `stream`)
 * (allocating counters for `tiles` tiles if it has fewer) and a launch epoch,
 * as a split launch would, and launches one block that arrives once on every
 * counter, as if one piece of every split tile had published, and then waits,
 * through the kernels' bounded wait, for a second arrival that never comes.
 * After budget_ns nanoseconds (0 < budget_ns <= 10 s) the wait gives up; the
 * next emu_stream_check() on this stream reports EMU_STATUS_DEVICE_TIMEOUT.
 * The arrivals it leaves behind belong to its own epoch, so a later split
 * launch on the stream is unaffected.  1 <= tiles <= 2^24, else
 * INVALID_VALUE.  No fault, trap or hang.
 */
emu_status_t emu_selftest_split_timeout(uint64_t budget_ns, int64_t tiles, emu_stream_t stream);

/*
 * emu_shutdown -- release the library's cached device buffers (split-K
 * workspaces, pre-split op(B) buffers) on every device that has them: each
 * such device is synchronised (cudaDeviceSynchronize) first, then the buffers
 * are freed and the (device, stream) slots cleared.  Later calls allocate
 * again on first need.  The current device is left as it was.  Returns
 * EMU_STATUS_LAUNCH_FAILED if a synchronisation or free failed (the slots
 * are cleared anyway).  Not to be called while another host thread is
 * inside a library call.  emu_sgemm_noalloc's fixed array is not freed (it
 * lives as long as the library is loaded).
 */
emu_status_t emu_shutdown(void);

/*
 * emu_debug_fail_allocations -- test hook: the next n device allocations the
 * library attempts (cudaMallocAsync of its workspace or pre-split buffers)
 * fail as if the device were out of memory, so that the calls needing them
 * return EMU_STATUS_ALLOC_FAILED having enqueued nothing.  n = 0 ends it.
 * INVALID_VALUE for n < 0.  Process-wide.
 */
emu_status_t emu_debug_fail_allocations(int n);

/*
 * emu_plan_query -- diagnostic, host only (no GPU, no CUDA call): the launch
 * plan emu_sgemm would use for an M x N x K product on a device with `pairs`
 * co-resident CTA pairs (76 on a GB300), honouring the EMU_SPLIT_K,
 * EMU_SPLIT_TAIL, EMU_CHAIN and EMU_PIPE overrides.  Writes EMU_PLAN_FIELDS values to out[0..]:
 *   0 pipeline shape (0 short-k, 1 long-k)   1 tile width (256)
 *   2 tiles along M (256 rows each)          3 tiles along N
 *   4 k-stages (32 each)                     5 tiles processed first (tiles_a)
 *   6 pieces per tile of those (split_a)     7 pieces per remaining tile (split_b)
 *   8 work units                             9 CTA pairs launched
 *  10 workspace partial tiles (256 x 256 FP32 each; 0 = no split tile)
 *  11 predicted time in hundredths of a pipeline stage (waves of work
 *     units, each its k-stages plus the output stores, plus the split-K
 *     reduction), the figure the plan minimises
 *  12 chained plan (1) or not (0)
 * Work unit u of the first group is piece u % split_a of tile u / split_a;
 * the remaining tiles follow, split_b units each; pair c runs units c,
 * c + pairs launched, ...  A chained plan (at least as many tiles as pairs;
 * fields 5-7 then read all tiles, 1, 1) instead gives pair c the stages
 * [b_c, b_c+1) of the U = tiles x k-stages stages taken tile by tile, each
 * tile's in decreasing k order (emu_plan_bounds gives b_0 = 0 < b_1 < ... <
 * b_P = U, P = pairs launched; each b_c lies within 2 stages of c U / P).
 * A tile that a run boundary cuts is split in two: the pair whose run starts
 * in it runs its low k-stages first and publishes the running FP32 sum (in
 * the workspace, one 256 x 256 slot per boundary); the pair whose run ends in
 * it runs the high k-stages last, starting from that sum, and stores the
 * tile.  The result is bit for bit that of the uncut tile.  INVALID_VALUE for
 * non-positive sizes, pairs < 1, a NULL `out` or n < EMU_PLAN_FIELDS.
 */
#define EMU_PLAN_FIELDS 13
emu_status_t emu_plan_query(int64_t M, int64_t N, int64_t K, int pairs, int64_t *out, int n);

/*
 * emu_plan_bounds -- diagnostic, host only: the run bounds b_0..b_P of the
 * chained plan emu_plan_query describes (P + 1 values to out[0..]).
 * NOT_SUPPORTED when that plan is not chained; INVALID_VALUE as for
 * emu_plan_query, or when n < P + 1.
 */
emu_status_t emu_plan_bounds(int64_t M, int64_t N, int64_t K, int pairs, int64_t *out, int n);

/*
 * Strategy.  Blog: "BF16x9 on Blackwell GPUs" (Fig. 4) compares two: the
 * eager one emulates whenever the operation allows it, the performant one
 * only where emulation is expected to beat native FP32.
 *   EMU_STRATEGY_EAGER (default): every product runs in the requested mode.
 *   EMU_STRATEGY_PERFORMANT: emu_sgemm, the unpacked emu_linear_* calls and
 *     emu_sgemm_noalloc
 *     run a product whose emulated form is predicted slower in
 *     EMU_MODE_FP32 instead (on GB300: small products, below about
 *     0.5 GFLOP).  Packed-operand calls always emulate.
 * Process-wide; emu_set_strategy returns INVALID_VALUE for an unknown value.
 */
typedef enum { EMU_STRATEGY_EAGER = 0, EMU_STRATEGY_PERFORMANT = 1 } emu_strategy_t;
emu_status_t emu_set_strategy(emu_strategy_t strategy);
emu_strategy_t emu_get_strategy(void);

/*
 * emu_dispatch_query -- host only (no GPU, no CUDA call): the mode in which
 * emu_sgemm would run an M x N x K product requested in `mode` under the
 * current strategy, on a device with `pairs` co-resident CTA pairs and
 * 2 * pairs SMs (76 pairs on a GB300).  INVALID_VALUE for an unknown mode,
 * non-positive sizes, pairs < 1 or a NULL `out`.
 */
emu_status_t emu_dispatch_query(emu_mode_t mode, int64_t M, int64_t N, int64_t K, int pairs, emu_mode_t *out);

/* Library version as an integer (major * 10000 + minor * 100 + patch). */
int emu_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EMU_GEMM_H */
