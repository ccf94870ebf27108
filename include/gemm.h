/*
 * gemm.h - C ABI of the GB300 (sm_103a) fused-epilogue dense GEMM.
 *
 * Operation (one call, all batches l < batch):
 *
 *   D(l) = act( alpha * scale_a * scale_b * op(A(l)) * op(B(l))
 *               + beta * C(l) + bias(l) )
 *
 * with fp32 accumulation, op in {N, T}, and D rounded to its type with
 * round-to-nearest-even.  This is the BLAS-style operation
 * "C = alpha * op(A) * op(B) + beta * C" of the page "CUTLASS" (knowledge
 * base, opening section) with a separate output D that may alias C
 * ("Technical Documentation: NVIDIA/cutlass", "Launching a GEMM kernel in
 * CUDA"), and the fused epilogue of the same page's "Epilogues" section and of
 * "Utilities for SM100", "Background - SM100 epilogue flow": accumulator, then
 * source C, then bias and activation, then the store.  scale_a / scale_b are
 * per-tensor dequantisation factors for 8-bit operands (the block-scaled form
 * of "Blackwell SM100 GEMMs", "Block Scaled GEMMs", with one factor per
 * tensor); pass 1.0 otherwise.
 *
 * Storage follows the BLAS convention: op(A) is M x K, stored as M x K (op N)
 * or K x M (op T) in row- or column-major order with leading dimension lda;
 * likewise op(B) is K x N; C and D are M x N.  All counts are in elements.
 * Batch l starts at base + l * stride_x.  bias is fp32: bias[n] (per column,
 * broadcast down M) or bias[m] (per row), batch stride stride_bias (0 shares
 * one vector across batches).
 *
 * Supported (anything else returns GEMM_ERR_UNSUPPORTED; there is no
 * fallback path):
 *   A, B: both F16, both BF16, or both E4M3 (a single tensor-core operand
 *         type per MMA); any op/order combination.
 *   C, D: F32, F16 or BF16, same type for C and D, same order for C and D.
 * Alignment (the tensor-alignment tables of "Technical Documentation:
 * NVIDIA/cutlass", "Layouts, Tensor Alignment Requirements to Target
 * tcgen05.mma Instructions": 8 elements for 16-bit, 16 for 8-bit operands):
 * every leading dimension and batch stride must be a multiple of 16 bytes and
 * every base pointer 16-byte aligned; otherwise GEMM_ERR_MISALIGNED.
 *
 * Ownership: the caller owns every device buffer.  A handle owns host state,
 * one 4-byte device status word and, when its schedule splits tiles between
 * workers (stream-K, see gemm_set_schedule), a workspace of fp32 partial sums
 * (one output tile per worker: 256 KiB per CTA pair, 128 KiB per CTA) plus one
 * flag word per worker epilogue warp; gemm_create / gemm_set_schedule
 * allocate them and gemm_destroy frees them.  gemm_run never allocates or
 * frees memory.  Launches through one handle share its status word and
 * workspace: issue them on one stream, or wait between them.
 *
 * Errors: argument errors are returned synchronously.  gemm_run is
 * asynchronous on the given stream; a failed launch returns GEMM_ERR_CUDA.
 * Every wait inside the kernel is bounded: if one runs out (default 2 s, see
 * gemm_set_debug) the kernel stops, records the fact in the status word and
 * returns without faulting, and the next gemm_check reports
 * GEMM_ERR_TIMEOUT.  The CUDA context stays usable.
 */
#ifndef GEMM_SM103_H
#define GEMM_SM103_H

#include <stddef.h>
#include <stdint.h>

#ifndef GEMM_API
#define GEMM_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,
    GEMM_ERR_UNSUPPORTED = 2,
    GEMM_ERR_MISALIGNED = 3,
    GEMM_ERR_CUDA = 4,
    GEMM_ERR_TIMEOUT = 5,
    GEMM_ERR_NO_DEVICE = 6,
    GEMM_ERR_BOUNDS = 7            /* diagnostic build (GEMM_DEBUG) only: an index check failed */
} gemm_status_t;

/* GEMM_E2M1: 4-bit float (sign, 2 exponent bits with bias 1, 1 mantissa bit;
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; "Blackwell Narrow Precision Data
 * Types"), two per byte along K, the element of lower K index in the low
 * nibble.  Operand type of GEMM_BLOCK_SCALE_NV only; leading dimensions and
 * batch strides still count elements. */
typedef enum { GEMM_F32 = 0, GEMM_F16 = 1, GEMM_BF16 = 2, GEMM_E4M3 = 3, GEMM_E2M1 = 4 } gemm_dtype_t;
typedef enum { GEMM_COL_MAJOR = 0, GEMM_ROW_MAJOR = 1 } gemm_order_t;
typedef enum { GEMM_OP_N = 0, GEMM_OP_T = 1 } gemm_op_t;
typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1, GEMM_ACT_GELU = 2 } gemm_act_t;
/* Reductions of the epilogue value t = act(alpha*scale_a*scale_b*acc + beta*C + bias), fp32, taken before
 * t is rounded to D's type; flags, combinable.  See gemm_run_ex. */
typedef enum {
    GEMM_REDUCE_NONE = 0,
    GEMM_REDUCE_ROW_SUM = 1,      /* row_sum[l*M + m] = sum over n of t(l, m, n) */
    GEMM_REDUCE_COL_SUM = 2,      /* col_sum[l*N + n] = sum over m of t(l, m, n) */
    GEMM_REDUCE_ABS_MAX = 4       /* abs_max[l] = max over m, n of |t(l, m, n)| (NaN if any t is NaN) */
} gemm_reduce_t;
typedef enum { GEMM_BIAS_NONE = 0, GEMM_BIAS_COL = 1, GEMM_BIAS_ROW = 2 } gemm_bias_t;
/* Block-scaled operands ("Technical Documentation: NVIDIA/cutlass", "Block
 * Scaled GEMMs"): D = act(alpha * sum_k (A(m,k) SFA(m,k/SV)) (B(k,n) SFB(n,k/SV))
 * + beta*C + bias), SV the scale-factor vector size.
 *   GEMM_BLOCK_SCALE_MX: A and B e4m3 (mx_float8), scale factors ue8m0
 *     (value 2^(code-127), code 255 = NaN), SV = 32.
 *   GEMM_BLOCK_SCALE_NV: A and B GEMM_E2M1 (nv_float4), scale factors ue4m3
 *     (e4m3 without its sign bit: code 0x7F = NaN, bit 7 must be 0), SV = 16.
 *     Both operands K-contiguous (the pages' TN layout), K even, leading
 *     dimensions and batch strides multiples of 32 elements (16 bytes);
 *     otherwise GEMM_ERR_UNSUPPORTED / GEMM_ERR_MISALIGNED.  A per-tensor
 *     fp32 global scale goes in scale_a / scale_b.
 * Scale factors are passed to gemm_run_args as byte tensors in the pages'
 * 512-byte basic-block layout ("Scale Factor Layouts"): for a matrix of R
 * rows (M for A, N for B; rows of op(A) / columns of op(B)) and
 * SFK = ceil(K/SV) factors per row, factor (r, f) of batch l is at byte
 *   l*ceil(R/128)*ceil(SFK/4)*512 + ((r/128)*ceil(SFK/4) + f/4)*512
 *   + (r%32)*16 + ((r%128)/32)*4 + f%4
 * Bytes of the padded tensor that name no real (r, f) are read by the
 * kernel and must not be NaN codes.  A batch whose A (B) is shared
 * (stride 0) shares SFA (SFB) too. */
typedef enum { GEMM_BLOCK_SCALE_NONE = 0, GEMM_BLOCK_SCALE_MX = 1, GEMM_BLOCK_SCALE_NV = 2 } gemm_block_scale_t;

/* Block-scaled output ("Technical Documentation: NVIDIA/cutlass", "Blackwell
 * SM100 GEMMs": an epilogue that writes elements plus a block scale factor
 * per SFDVectorSize elements).  GEMM_OUT_SCALE_MX: D is e4m3 (dtype_d =
 * GEMM_E4M3, row-major) and every 32 consecutive elements of a D row share
 * one ue8m0 factor, written to gemm_args_t.sfd in the same basic-block
 * layout as the input factors (rows = M, factors per row = ceil(N/32)).
 * Factor: the OCP MX rule on the fp32 epilogue value t of the block (shared
 * exponent floor(log2 max|t|) - 8, code clamped to [0, 254]; 255 and NaN
 * elements for a block holding NaN or inf); elements e4m3(t / 2^(code-127))
 * rounded to nearest even, saturated at +-448.  Needs beta = 0 and no
 * reductions (else GEMM_ERR_UNSUPPORTED).  Only the factors of real
 * (row, block) pairs are written.
 * GEMM_OUT_SCALE_NV (the page's example, SFDVectorSize = 16): D is e2m1
 * (dtype_d = GEMM_E2M1, row-major, two elements per byte, the lower column
 * in the low nibble; N even and ldd / stride_d multiples of 32 elements,
 * else GEMM_ERR_UNSUPPORTED / GEMM_ERR_MISALIGNED) and every 16 consecutive
 * elements of a D row share one ue4m3 factor, written to gemm_args_t.sfd in
 * the basic-block layout (rows = M, factors per row = ceil(N/16)).  With the
 * output's fp32 global scale g = desc.scale_d (a normal, finite fp32 > 0,
 * else GEMM_ERR_INVALID_ARG): factor = e4m3(amax / (6 g)) (nearest even,
 * saturating at 448; amax = the block's max |t|), elements
 * e2m1(t / (factor * g)) (nearest even, saturating at +-6), each the
 * rounding of the exact quotient of the fp32 values; 0 where the factor is
 * 0; a block holding NaN or inf gets factor 0x7F and zero elements.  So D * factor * g ~ t, and D with its
 * factors and g is an NVFP4 operand (GEMM_BLOCK_SCALE_NV) for the next GEMM.
 * Same restrictions as GEMM_OUT_SCALE_MX. */
typedef enum { GEMM_OUT_SCALE_NONE = 0, GEMM_OUT_SCALE_MX = 1, GEMM_OUT_SCALE_NV = 2 } gemm_out_scale_t;

typedef enum {
    GEMM_SCHED_AUTO = 0,
    GEMM_SCHED_DATA_PARALLEL = 1,
    GEMM_SCHED_STREAM_K = 2,
    GEMM_SCHED_SPLIT_TAIL = 3,
    GEMM_SCHED_DYNAMIC = 4
} gemm_sched_t;

/* Problem descriptor.  Enumerations are carried as int32_t. */
typedef struct {
    int64_t M, N, K, batch;                        /* batch >= 1; M, N, K >= 0 */
    int32_t op_a, op_b;                            /* gemm_op_t */
    int32_t order_a, order_b, order_c, order_d;    /* gemm_order_t */
    int64_t lda, ldb, ldc, ldd;                    /* leading dimensions, elements */
    int64_t stride_a, stride_b, stride_c, stride_d, stride_bias; /* batch strides, elements */
    int32_t dtype_a, dtype_b, dtype_c, dtype_d;    /* gemm_dtype_t */
    float alpha, beta;
    float scale_a, scale_b;                        /* 1.0 unless 8-bit operands */
    int32_t act;                                   /* gemm_act_t */
    int32_t bias;                                  /* gemm_bias_t; bias is fp32 */
    int32_t reduce;                                /* gemm_reduce_t flags; 0 = none */
    int32_t block_scale;                           /* gemm_block_scale_t; 0 = none */
    int32_t out_scale;                             /* gemm_out_scale_t; 0 = none */
    float scale_d;                                 /* output global scale of GEMM_OUT_SCALE_NV; else unused */
} gemm_desc_t;

/* How a descriptor is executed; filled by gemm_plan (host only, no GPU). */
typedef struct {
    int32_t swapped;          /* 1: computed as D^T = op(B)^T op(A)^T because D is column-major */
    int32_t a_k_major;        /* kernel operand A (after any swap) is K-contiguous */
    int32_t b_k_major;        /* kernel operand B (after any swap) is K-contiguous */
    int32_t tile_m, tile_n;   /* output tile per CTA (per CTA pair when cta_group == 2) */
    int32_t tile_k;           /* K elements per pipeline stage */
    int32_t cta_group;        /* SMs sharing one MMA: 1 or 2 */
    int32_t stages;           /* shared-memory pipeline depth */
    int32_t raster_group;     /* M tiles walked together by the persistent scheduler */
    int32_t epi_cols;         /* epilogue subtile width, columns */
    int64_t tiles_m, tiles_n, tiles;   /* tiles along M and N (kernel orientation), total incl. batch */
    int64_t kernel_m, kernel_n;        /* problem extents in kernel orientation */
} gemm_plan_info_t;

typedef struct gemm_handle_s* gemm_handle_t;

/* Validates `desc` and reports how it would run.  Host only: makes no CUDA
 * call and works without a GPU.  Returns GEMM_OK, GEMM_ERR_INVALID_ARG,
 * GEMM_ERR_UNSUPPORTED or GEMM_ERR_MISALIGNED (strides). */
GEMM_API gemm_status_t gemm_plan(const gemm_desc_t* desc, gemm_plan_info_t* info);

/* Validates `desc`, plans it and allocates the handle (host state plus a
 * 4-byte device status word on the current device).  Returns
 * GEMM_ERR_NO_DEVICE when no usable GPU is present.  *out is NULL on error. */
GEMM_API gemm_status_t gemm_create(gemm_handle_t* out, const gemm_desc_t* desc);

/* Launches the GEMM on `stream` (a cudaStream_t; NULL = legacy default
 * stream) with device pointers.  C may be NULL iff beta == 0; bias may be
 * NULL iff the descriptor has no bias.  D may equal C (same layout).
 * Asynchronous; never allocates.  M == 0 or N == 0 launches nothing. */
GEMM_API gemm_status_t gemm_run(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
                       const float* bias, void* stream);

/* gemm_run plus the reductions the descriptor asks for (desc.reduce), into
 * caller-owned fp32 device arrays: row_sum [batch*M], col_sum [batch*N],
 * abs_max [batch]; an array the descriptor does not ask for may be NULL, one
 * it asks for may not (GEMM_ERR_INVALID_ARG).  gemm_run on a descriptor with
 * reductions returns GEMM_ERR_INVALID_ARG.
 *
 * The pages list per-row and per-column reductions among the epilogue
 * fusions ("Technical Documentation: NVIDIA/cutlass", "What's New in CUTLASS
 * 4.8"); what is reduced is this library's reading: t, the fp32 epilogue
 * value after the activation and before rounding to D's type.  The GEMM
 * kernel writes one partial per (row, 256- or 128-column tile) and per
 * (32-row slab, column) into the handle's workspace (allocated by
 * gemm_create) and a second, small kernel on the same stream adds them in
 * index order, so the sums are the same on every run; the abs-max is an
 * atomic maximum, also order-independent.  M == 0 or N == 0 launches nothing
 * and leaves the outputs untouched. */
GEMM_API gemm_status_t gemm_run_ex(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
                                   const float* bias, float* row_sum, float* col_sum, float* abs_max, void* stream);

/* Waits for the handle's last launch and reads its device status word:
 * GEMM_ERR_TIMEOUT if any bounded wait ran out (the word is then cleared),
 * GEMM_ERR_CUDA on a CUDA error, else GEMM_OK. */
GEMM_API gemm_status_t gemm_check(gemm_handle_t h);

/* Frees the handle (synchronises with its last launch first). NULL is a no-op. */
GEMM_API gemm_status_t gemm_destroy(gemm_handle_t h);

/* Test hooks.  inject_fault = 1 makes the load warp skip the very first
 * tile load of the next launches (the consumer then waits until its bound
 * runs out); 0 restores normal operation.  timeout_ms bounds every
 * in-kernel wait (0 keeps the current bound; default 2000 ms). */
GEMM_API gemm_status_t gemm_set_debug(gemm_handle_t h, int32_t inject_fault, uint32_t timeout_ms);

/* Diagnostic builds.  The library can be built with -DGEMM_DEBUG (every
 * plain store and TMA store of the kernel checks its index against the
 * buffer's extents first; a failed check skips the access and gemm_check
 * returns GEMM_ERR_BOUNDS) and with -DGEMM_STAMPS (the kernel records
 * %globaltimer at 8 points of each CTA; see gemm_set_stamps).  The default
 * build has neither.  gemm_build_flags returns bit 0 for GEMM_DEBUG and
 * bit 1 for GEMM_STAMPS. */
GEMM_API int32_t gemm_build_flags(void);

/* GEMM_STAMPS builds: `stamps` is a device buffer of 8 uint64 per CTA of the
 * launch (workers x CTA group of gemm_get_schedule; the dynamic schedule
 * launches one CTA or pair per tile), in which the next
 * launches write %globaltimer (ns) at: 0 CTA entry, 1 set-up done, 2 first
 * operand loads issued, 3 first stage's data arrived at the MMA thread (the
 * pair's leader), 4 first accumulator committed, 5 the epilogue sees it,
 * 6 the epilogue's last store complete, 7 before TMEM is freed.  NULL stops
 * recording.  Other builds: GEMM_ERR_UNSUPPORTED. */
GEMM_API gemm_status_t gemm_set_stamps(gemm_handle_t h, void* stamps);

/* Work split of the persistent kernel.  The pages name split-K only as a
 * profiler option ("Technical Documentation: NVIDIA/cutlass", "Performance
 * Profiling": --split_k_mode=serial --split_k_slices=N); this library splits K
 * to even out the last, ragged wave of tiles, in two forms:
 *
 *   GEMM_SCHED_DATA_PARALLEL  every tile is computed whole by one worker (a
 *                             CTA, or a CTA pair), tile w, w + workers, ...
 *   GEMM_SCHED_SPLIT_TAIL     the full waves are computed whole; each of the
 *                             R tiles of the ragged last wave is cut into
 *                             floor(S / R) equal K ranges (at most one per K
 *                             block), one range per worker, where S is the
 *                             number of workers the GPU holds at once (SMs
 *                             per CTA group, or fewer if clusters do not all
 *                             fit).  A problem of fewer than S tiles is one
 *                             ragged wave: its launch then has one worker per
 *                             range.
 *   GEMM_SCHED_STREAM_K       all full waves but the last are computed whole;
 *                             the K blocks of the remaining tiles are cut
 *                             into one equal contiguous range per worker, S
 *                             workers.
 *   GEMM_SCHED_DYNAMIC        whole tiles, scheduled by the hardware
 *                             ("Technical Documentation: NVIDIA/cutlass",
 *                             "Blackwell Cluster Launch Control"): the
 *                             launch holds one cluster per tile and a running
 *                             cluster that finishes a tile cancels the launch
 *                             of one that has not started and computes its
 *                             tile instead.  SMs held by other work on the
 *                             GPU then delay no tile; with the GPU to itself
 *                             it matches DATA_PARALLEL.  Needs no workspace.
 *   GEMM_SCHED_AUTO (default) SPLIT_TAIL when there is at least one full
 *                             wave, a ragged last wave, and it cuts each of
 *                             its tiles into two or more ranges of at least
 *                             4 K blocks; else data parallel.
 *
 * A tile cut between workers is finished by the worker that ran its first K
 * block, after adding the other workers' fp32 partial sums, which they leave
 * in the handle's workspace.  Under SPLIT_TAIL the workers of one cut index
 * walk K together, as whole tiles of a wave do; under STREAM_K the ranges
 * start at unrelated K offsets.
 *
 * Results of the two schedules can differ in the last bits of non-integer
 * sums (fp32 summation order); each is deterministic from run to run.
 * Allocates or frees the workspace as needed (synchronising with the
 * handle's last launch first), so call it at set-up time, not between
 * launches that are being captured.  Returns GEMM_ERR_INVALID_ARG for an
 * unknown mode, GEMM_ERR_CUDA if the workspace cannot be allocated. */
GEMM_API gemm_status_t gemm_set_schedule(gemm_handle_t h, int32_t mode);

/* The handle's work split: workers (persistent CTAs, or CTA pairs), tiles
 * computed whole, K-block iterations of the cut tiles (0: data parallel) and
 * the number of ranges they are cut into.  Any output pointer may be NULL. */
GEMM_API gemm_status_t gemm_get_schedule(gemm_handle_t h, int32_t* workers, int64_t* dp_tiles, int64_t* sk_iters,
                                         int32_t* sk_ranges);

/* Kernel launches issued through this handle so far. */
GEMM_API uint64_t gemm_launch_count(gemm_handle_t h);

/* Allocation-free variant of gemm_run.  The pages have no counterpart; this
 * entry point exists for callers that must not call cudaMalloc: code running
 * inside a framework whose memory pool owns the whole device (a raw
 * allocation there can fail or fragment the pool) and latency-critical paths
 * where cudaMalloc/cudaFree may synchronise the device.
 *
 * It plans `desc` and launches the same kernel as gemm_run on `stream`, with
 * all host state on the stack and no handle.  The kernel's only scratch
 * memory, its 4-byte status word, lives in a fixed file-scope device array of
 * 64 words (256 bytes) that every GPU loading this library keeps until the
 * process exits; a call needs 1 word, and a call needing more than the array
 * holds is refused with GEMM_ERR_UNSUPPORTED.  No cudaMalloc, cudaFree or
 * other allocating routine is called.
 *
 * The first call on a device looks up that array's device address
 * (cudaGetSymbolAddress, with the device current) and sets the kernel up;
 * make that first call before any stream capture.  A set-up that fails
 * returns its error and is tried again on the next call.  Each call that
 * passes its checks clears the status word on `stream` right before its
 * launch (a rejected call queues nothing).  All calls on a device share the
 * array, so calls whose kernels overlap on the GPU race on the status word:
 * issue them on one stream, or wait between them.
 *
 * wait = 0: asynchronous; argument and launch errors are returned, an
 * in-kernel timeout is not reported.  wait = 1: the call synchronises
 * `stream` and returns GEMM_ERR_TIMEOUT if a bounded wait ran out; it
 * cannot be used while `stream` is being captured into a graph (the
 * synchronisation and the read-back would end the capture): only wait = 0
 * may be used there.
 * Pointers, alignment and errors are as for gemm_run; a descriptor with
 * reductions (which need a handle's workspace) or block scaling (no
 * scale-factor arguments here) returns GEMM_ERR_UNSUPPORTED. */
GEMM_API gemm_status_t gemm_run_noalloc(const gemm_desc_t* desc, const void* A, const void* B, const void* C,
                                        void* D, const float* bias, void* stream, int32_t wait);

/* Every buffer of one launch.  Pointers as for gemm_run / gemm_run_ex;
 * sfa / sfb: the scale-factor tensors of a block-scaled descriptor (16-byte
 * aligned; NULL otherwise). */
typedef struct {
    const void* A;
    const void* B;
    const void* C;
    void* D;
    const float* bias;
    const void* sfa;
    const void* sfb;
    float* row_sum;
    float* col_sum;
    float* abs_max;
    void* sfd;                     /* output factors of a GEMM_OUT_SCALE_MX / _NV descriptor */
} gemm_args_t;

/* gemm_run with every buffer in one struct: the entry point for
 * block-scaled descriptors (gemm_run / gemm_run_ex return
 * GEMM_ERR_INVALID_ARG for them, having no scale-factor arguments). */
GEMM_API gemm_status_t gemm_run_args(gemm_handle_t h, const gemm_args_t* args, void* stream);

/* Grouped GEMM ("Technical Documentation: NVIDIA/cutlass", "What's New in
 * CUTLASS 4.8": grouped GEMM with contiguous offsets).  `groups` problems in
 * one launch that share N, K, types, layouts and epilogue: group g owns rows
 * [group_rows[g], group_rows[g+1]) of one A, one C and one D (desc.M rows
 * each, the rows of all groups one after another) and uses batch g of B
 * (desc.stride_b elements apart; 0 = one B for all) and of the bias
 * (desc.stride_bias apart; 0 = shared):
 *   D[r, :] = act(alpha * A[r, :] op(B_g) + beta * C[r, :] + bias_g)   for r in group g.
 * Descriptor rules: desc.batch = 1 and stride_a = stride_c = stride_d = 0
 * (else GEMM_ERR_INVALID_ARG); A K-contiguous, D (and C) row-major; no
 * block-scaled output, reductions or per-row bias (else
 * GEMM_ERR_UNSUPPORTED); groups in [1, 65535].
 * Block-scaled operands (desc.block_scale) run through
 * gemm_grouped_run_args: SFB holds one basic-block tensor per group (as for a
 * batch); SFA keeps each group's rows in whole 128-row blocks, the groups'
 * blocks one after another: row r of group g (r counted from the group's
 * first row) has its factors in row block B_g + r/128, B_g = the sum over
 * earlier groups of ceil(rows/128), laid out as one batch of the
 * basic-block format with R = 128 * (ceil(M/128) + groups) rows; allocate
 * that many.  The handle runs whole tiles (gemm_set_schedule accepts
 * GEMM_SCHED_AUTO and GEMM_SCHED_DATA_PARALLEL only) and sizes its grid to the
 * GPU, since the tile count is known only on the device.
 * gemm_grouped_run: group_rows is a DEVICE array of groups + 1 int64 row
 * offsets, 8-byte aligned, read by the kernel (so it may be written by an
 * earlier kernel on the same stream).  Offsets are clamped to [0, desc.M]
 * and group g covers [e(g-1), e(g)), e(g) the running maximum of the
 * clamped offsets 0..g+1 (e(-1) = the first), so groups never overlap and
 * no row outside D is ever written; rows of D that no group covers are left
 * untouched.  gemm_run / gemm_run_ex /
 * gemm_run_args on a grouped handle, and gemm_grouped_run on another one,
 * return GEMM_ERR_INVALID_ARG.  Other arguments as for gemm_run. */
GEMM_API gemm_status_t gemm_grouped_create(gemm_handle_t* out, const gemm_desc_t* desc, int32_t groups);
GEMM_API gemm_status_t gemm_grouped_run(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
                                        const float* bias, const int64_t* group_rows, void* stream);
/* gemm_grouped_run with every buffer in one struct (the call for
 * block-scaled grouped descriptors: sfa / sfb as described above). */
GEMM_API gemm_status_t gemm_grouped_run_args(gemm_handle_t h, const gemm_args_t* args, const int64_t* group_rows,
                                             void* stream);

/* Static string for a status code. */
GEMM_API const char* gemm_status_str(gemm_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_SM103_H */
