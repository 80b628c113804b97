/*
 * tg_gemm.h -- C ABI of a tiled dense matrix multiply for NVIDIA GB300 (sm_103a).
 *
 * Operation.  Every GEMM entry point computes
 *
 *     C[m,n] = sum_{k=0}^{K-1} A[m,k] * B[k,n]      0 <= m < M, 0 <= n < N
 *
 * with A of shape [M,K], B of shape [K,N] and C of shape [M,N]: "Matrix
 * multiplication: reuse the inputs" (triton-cuda-lab lesson 6), section "The
 * three dimensions have different jobs".  The work is split into output tiles,
 * each accumulated over K in chunks with the accumulator kept on chip until it
 * is written once ("Matrix Multiplication", teenygrad docs, section "Tiles";
 * "Triton tiled matmul", llm-systems-cookbook, section "What").  Products are
 * accumulated in FP32 whatever the input type, the choice all of those pages
 * make, and the FP32 sum is rounded to nearest-even once into the output type.
 *
 * Layout.  All matrices are row-major with unit column stride and an explicit
 * leading dimension counted in ELEMENTS: A[m,k] is at a[m*lda + k], B[k,n] at
 * b[k*ldb + n], C[m,n] at c[m*ldc + n].  Requires lda >= K, ldb >= N, ldc >= N.
 * Elements outside the logical [rows, cols] block (the padding up to the
 * leading dimension) are never read and never written.
 *
 * Types (dtype_in, dtype_out):
 *     (TG_F16,  TG_F16)  (TG_F16,  TG_F32)
 *     (TG_BF16, TG_BF16) (TG_BF16, TG_F32)
 *     (TG_F32,  TG_F32)  -- FP32 operands contracted at TF32 precision (10
 *                           fraction bits), FP32 accumulate; the "TF32" input
 *                           precision of the teenygrad page, section "T::dot".
 *     (TG_E4M3 or TG_E5M2, TG_F16 / TG_BF16 / TG_F32)
 *                        -- 8-bit floating-point operands, FP32 accumulate: the
 *                           FP8 input path of "Triton tiled matmul"
 *                           (llm-systems-cookbook), section "Exercises", item 2.
 *                           Row pitches (lda, ldb) and bases of A and B that are
 *                           not multiples of 16 bytes are packed first.  Per-tensor
 *                           scale factors of FP8 data go in as the product
 *                           scale_a * scale_b in tg_gemm_fused's alpha.
 * Any other pair returns TG_ERR_UNSUPPORTED.
 *
 * Ownership.  a, b and c are DEVICE pointers owned by the caller and must stay
 * valid until the work enqueued on `stream` has finished.  The library owns only
 * temporary device workspace (stream-ordered, taken from and returned to a
 * memory pool of its own on the same stream; the pool keeps the memory for
 * later calls) and internal caches.  `stream` is a cudaStream_t passed as void*; NULL is the
 * legacy default stream.
 *
 * Asynchrony and errors.  The GEMM calls validate their arguments on the host,
 * enqueue kernels on `stream` and return without synchronising.  Argument
 * errors are returned before anything is enqueued and leave C untouched.  A CUDA
 * error while enqueueing returns TG_ERR_CUDA.  Every wait inside the kernels is
 * bounded (default 2 s); a kernel whose wait runs out records TG_ERR_TIMEOUT in
 * a per-device status word, releases what it holds and exits, which
 * tg_last_device_error() reports.
 *
 * Special sizes.  M == 0 or N == 0: nothing to do, TG_OK.  K == 0: C is set to
 * zero (the empty sum).
 *
 * Threading.  Calls may be made from several host threads; a device's lazily
 * built state is created under a lock.
 */
#ifndef TG_GEMM_H
#define TG_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TG_ABI_VERSION 10

typedef enum tg_dtype {
    TG_F16 = 0,   /* IEEE 754 binary16 */
    TG_BF16 = 1,  /* bfloat16 */
    TG_F32 = 2,   /* IEEE 754 binary32 */
    TG_E4M3 = 3,  /* OCP FP8 E4M3 (bias 7, 3 fraction bits, no Inf; max 448) */
    TG_E5M2 = 4   /* OCP FP8 E5M2 (bias 15, 2 fraction bits, IEEE-like) */
} tg_dtype;

typedef enum tg_status {
    TG_OK = 0,
    TG_ERR_INVALID_VALUE = 1,    /* bad size, leading dimension, pointer or overlap */
    TG_ERR_UNSUPPORTED = 2,      /* dtype pair or option not supported */
    TG_ERR_OUT_OF_MEMORY = 3,    /* workspace allocation failed */
    TG_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed */
    TG_ERR_ARCH = 5,             /* current device is not an sm_103 GPU */
    TG_ERR_TIMEOUT = 6,          /* a kernel's bounded wait ran out */
    TG_ERR_NOT_IMPLEMENTED = 7,
    TG_ERR_BOUNDS = 8            /* checked builds: a device-side bounds or
                                    alignment check failed (access skipped) */
} tg_status;

/* Execution paths the planner chooses between. */
typedef enum tg_path {
    TG_PATH_AUTO = 0,
    TG_PATH_TC = 1,        /* tcgen05 tensor-core kernel, one CTA per 128-row tile */
    TG_PATH_TC_PAIR = 2,   /* tcgen05 kernel with CTA pairs (cta_group::2), 256-row tiles */
    TG_PATH_SKINNY = 3     /* memory-streaming kernel for small M */
} tg_path;

/* Optional overrides for tg_gemm_ex.  Zero in any field means "let the planner
 * choose".  Values the compiled kernels cannot honour return
 * TG_ERR_UNSUPPORTED. */
typedef struct tg_options {
    int32_t path;         /* tg_path */
    int32_t splits;       /* number of K splits (>= 1); the small-M kernel splits K
                             over a cluster of 1, 2, 4 or 8 CTAs */
    int32_t block_n;      /* output tile width: 128, 192, 224 or 256 for the tile
                             kernels, also 512 for CTA pairs; 128, 256 or 512
                             for the small-M kernel */
    int32_t group_m;      /* grouped raster height in tiles (default 8) */
    int32_t max_ctas;     /* cap on the persistent grid (default: one per SM) */
    int32_t timeout_ms;   /* bound on every device-side wait (default 2000) */
    int32_t multicast;    /* 2 = two neighbouring tiles share their A tile by TMA
                             multicast inside a cluster of two CTA pairs (192-,
                             224- or 256-wide tiles; the pair path); 1 = no
                             sharing; 0 = planner */
    int32_t f32_mode;     /* FP32 operands only (tg_f32_mode): TG_F32_TF32 (0) or
                             TG_F32_3XTF32 (1) */
    int32_t reserved;     /* must be 0 */
} tg_options;

/*
 * How FP32 operands are contracted on the tensor cores.
 *   TG_F32_TF32    one pass at TF32 precision (10 fraction bits per operand).
 *   TG_F32_3XTF32  each operand x is split into TF32 parts x = hi + lo + r
 *                  (hi = x rounded to TF32, lo = the rest rounded to TF32,
 *                  |r| <= about 2^-22 |x|) and C = A_hi B_hi + A_lo B_hi +
 *                  A_hi B_lo is accumulated in FP32: near-FP32 accuracy at three
 *                  times the TF32 work.  The "TF32x3" alternative to IEEE mode
 *                  that "Matrix Multiplication" (teenygrad docs, section
 *                  "T::dot") lists among the input precisions.  The parts are
 *                  written to workspace as A' = [A_hi | A_lo | A_hi] ([M, 3K])
 *                  and B'^T = [B_hi | B_hi | B_lo]^T ([N, 3K]) and multiplied by
 *                  the TF32 kernel over K' = 3K.  Operands with an infinite or
 *                  NaN element, or of magnitude within 2^-11 of the largest
 *                  FP32 value, may give NaN or Inf where a one-pass product is
 *                  finite or +-Inf.  Other values of f32_mode, or a non-zero
 *                  reserved field, return TG_ERR_INVALID_VALUE; TG_F32_3XTF32
 *                  with other operand types, TG_ERR_UNSUPPORTED.
 */
typedef enum tg_f32_mode { TG_F32_TF32 = 0, TG_F32_3XTF32 = 1 } tg_f32_mode;

/* What a call would launch (see tg_plan_gemm). */
typedef struct tg_plan {
    int32_t path;          /* tg_path actually used */
    int32_t block_m, block_n, block_k;
    int32_t stages;        /* shared-memory ring depth */
    int32_t splits;        /* K splits (1 = none) */
    int32_t group_m;
    int32_t ctas;          /* grid size (persistent for the tile kernels) */
    int32_t pack_a;        /* 1 if A is first copied to an aligned workspace */
    int32_t pack_b;        /* 1 if B is first copied to an aligned workspace,
                              3 if B is split into TF32 parts (TG_F32_3XTF32;
                              pack_a is then 3 as well) */
    int32_t c_vector;      /* 1 if C's base and row pitch are 16-byte multiples:
                              the tile kernels then write C with TMA stores
                              when N x the output size is one too, else with
                              16-byte vector stores */
    int32_t kernels;       /* kernel launches per call */
    int64_t tiles;         /* work units: output tiles, or groups of `multicast`
                              neighbouring tiles; over all products of a batch */
    int64_t workspace_bytes;
    int32_t multicast;     /* tiles sharing one A tile (1 or 2) */
    int32_t per_batch;     /* strided batches only: 1 if each product of the batch
                              is run as its own call (kernels counts them all), 0
                              if one launch covers every product */
} tg_plan;

/*
 * tg_gemm -- C = A * B, the product of "Matrix multiplication: reuse the
 * inputs" (triton-cuda-lab lesson 6), section "The three dimensions have
 * different jobs" (see the top of this file for layout, types and errors).
 *   M, N, K   sizes (>= 0)
 *   a, lda    device pointer to A and its leading dimension (elements, >= K)
 *   b, ldb    device pointer to B and its leading dimension (elements, >= N)
 *   c, ldc    device pointer to C and its leading dimension (elements, >= N);
 *             C must not overlap A or B
 *   dtype_in  type of A and B; dtype_out type of C
 *   stream    cudaStream_t (as void*) the work is enqueued on
 */
tg_status tg_gemm(int64_t M, int64_t N, int64_t K,
                  const void *a, int64_t lda,
                  const void *b, int64_t ldb,
                  void *c, int64_t ldc,
                  tg_dtype dtype_in, tg_dtype dtype_out,
                  void *stream);

/*
 * tg_gemm_ex -- tg_gemm (the same operation, arguments, layout, ownership and
 * errors) with planner overrides; `opt` may be NULL.  The overrides pick among
 * the compiled variants of the tiled multiply -- tile width, CTA pair or single
 * CTA, K split, grouped-raster height -- which the pages fix per kernel as
 * constants ("Matrix Multiplication", teenygrad docs, section "Tiles"; "Triton
 * tiled matmul", llm-systems-cookbook, section "The kernel"); values the
 * compiled kernels cannot honour return TG_ERR_UNSUPPORTED.
 */
tg_status tg_gemm_ex(int64_t M, int64_t N, int64_t K,
                     const void *a, int64_t lda,
                     const void *b, int64_t ldb,
                     void *c, int64_t ldc,
                     tg_dtype dtype_in, tg_dtype dtype_out,
                     void *stream, const tg_options *opt);

/*
 * tg_plan_gemm -- host only, touches no device: validates the arguments exactly
 * as tg_gemm_ex does (pointers are inspected for alignment and overlap only,
 * never dereferenced) and fills *plan with what tg_gemm_ex would launch on a
 * device with `num_sms` SMs.  Returns the status tg_gemm_ex would return for
 * an argument error, else TG_OK.  No counterpart in the pages: it reports the
 * library's own choice of kernel variant.  `plan` is owned by the caller.
 */
tg_status tg_plan_gemm(int64_t M, int64_t N, int64_t K,
                       const void *a, int64_t lda,
                       const void *b, int64_t ldb,
                       const void *c, int64_t ldc,
                       tg_dtype dtype_in, tg_dtype dtype_out,
                       int32_t num_sms, const tg_options *opt, tg_plan *plan);

/* Activation of the fused epilogue (see tg_gemm_fused). */
typedef enum tg_activation {
    TG_ACT_NONE = 0,       /* x */
    TG_ACT_RELU = 1,       /* x if x > 0, else 0 */
    TG_ACT_SILU = 2,       /* x / (1 + exp(-x)) */
    TG_ACT_GELU_TANH = 3   /* x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))) */
} tg_activation;

/* Fused epilogue of tg_gemm_fused. */
typedef struct tg_epilogue {
    float alpha;            /* multiplies the product */
    float beta;             /* multiplies the residual */
    const float *scale;     /* N per-column FP32 factors on the device, or NULL (1) */
    const float *bias;      /* N per-column FP32 offsets on the device, or NULL (0) */
    const void *residual;   /* R: [M, ldr] of dtype_out on the device, or NULL */
    int64_t ldr;            /* leading dimension of R in elements (>= N) */
    int32_t activation;     /* tg_activation */
    int32_t reserved;       /* must be 0 */
} tg_epilogue;

/*
 * tg_gemm_fused -- the product with a fused epilogue, applied to each FP32
 * accumulator value where the kernel writes C, before its one rounding to
 * dtype_out:
 *
 *     C[m,n] = act(alpha * scale[n] * sum_k A[m,k] B[k,n] + bias[n]) + beta * R[m,n]
 *
 * "Matrix Multiplication" (teenygrad docs) closes by handing on to its next
 * chapter, "Fusing an Epilogue": extra work on the output tile while it is
 * still on chip.  The same book's fused kernel applies a per-channel scale and
 * shift (batch norm) and a SiLU to a GEMM this way.
 *
 *   M .. dtype_out, stream, opt   as for tg_gemm_ex
 *   epilogue   NULL: exactly tg_gemm_ex.  Otherwise: activation out of range
 *              or reserved != 0 -> TG_ERR_INVALID_VALUE; a residual needs
 *              ldr >= N and dtype_out alignment, and may be C itself (same
 *              pointer and ldr == ldc: C = act(...) + beta * C) but must not
 *              otherwise overlap C; scale / bias must be 4-byte aligned and
 *              not overlap C -> else TG_ERR_INVALID_VALUE.
 *
 * K == 0 writes act(bias[n]) + beta * R[m,n] (the epilogue of the empty sum).
 * With a K split the epilogue runs in the kernel that sums the partials.
 */
tg_status tg_gemm_fused(int64_t M, int64_t N, int64_t K,
                        const void *a, int64_t lda,
                        const void *b, int64_t ldb,
                        void *c, int64_t ldc,
                        tg_dtype dtype_in, tg_dtype dtype_out,
                        const tg_epilogue *epilogue,
                        void *stream, const tg_options *opt);

/*
 * tg_gemm_host -- C = A * B with A, B and C in HOST memory (the operation of
 * tg_gemm, "Matrix multiplication: reuse the inputs", triton-cuda-lab lesson 6,
 * section "The three dimensions have different jobs"): the library stages
 * them through device memory of its own and overlaps the transfers with the
 * multiply.  B is copied first, then A in row panels (at least 1024 rows, at
 * most 16 panels) on one copy stream; the panel products run on `stream` as
 * each panel of A arrives, and each panel of C is copied back on a second copy
 * stream while later panels are still being copied in or multiplied.
 *
 *   M .. dtype_out, opt   as for tg_gemm_ex, with a, b, c HOST pointers
 *                         (page-locked memory, e.g. cudaHostAlloc, lets the
 *                         copies run asynchronously and overlap; pageable
 *                         memory works but the copies serialise)
 *   stream                the multiply runs on it; the call returns at once and
 *                         C is complete when the work enqueued on `stream` so
 *                         far has finished (synchronise it before reading C)
 *
 * The staging buffers (M*K + K*N elements of dtype_in, M*N of dtype_out, row
 * pitches rounded up to 16 bytes) come from the library's memory pool and go
 * back to it in stream order.  The panels are separate products, so the
 * result is the one tg_gemm_ex gives for each row panel.  Argument errors as
 * for tg_gemm (the overlap rules apply to the host addresses).  One call per
 * device runs its enqueueing at a time (a lock); the copies of successive
 * calls may overlap on the GPU.
 */
tg_status tg_gemm_host(int64_t M, int64_t N, int64_t K,
                       const void *a, int64_t lda,
                       const void *b, int64_t ldb,
                       void *c, int64_t ldc,
                       tg_dtype dtype_in, tg_dtype dtype_out,
                       void *stream, const tg_options *opt);

/*
 * tg_gemm_strided_batched -- `batch` independent products
 *
 *     C_z = A_z * B_z,   A_z = a + z*stride_a,  B_z = b + z*stride_b,
 *                        C_z = c + z*stride_c,  0 <= z < batch
 *
 * each of them exactly the operation of tg_gemm (same sizes M, N, K, leading
 * dimensions, types and rounding).  This is the batched extension of the tiled
 * multiply with a third grid axis over the batch ("Triton tiled matmul",
 * llm-systems-cookbook, section "Exercises", item 3): the kernels treat the
 * batch index as the slowest dimension of their work list, and A / B are read
 * through rank-3 TMA tensor maps.
 *
 *   batch              number of products (>= 0; 0 does nothing)
 *   stride_a/b/c       distance in ELEMENTS between consecutive products' A, B,
 *                      C (>= 0).  stride_a == 0 (or stride_b == 0) uses one A
 *                      (one B) for every product.  C of different products
 *                      must not overlap: stride_c >= (M-1)*ldc + N (stacked
 *                      products), or stride_c >= N with
 *                      (batch-1)*stride_c + N <= ldc (products interleaved
 *                      along a row, C stored [M][batch][N]); else
 *                      TG_ERR_INVALID_VALUE.  The whole of C (all products)
 *                      must not overlap the whole of A or of B.
 *   opt                as for tg_gemm_ex; with batch > 1, opt->splits > 1 is
 *                      only accepted with opt->path == TG_PATH_SKINNY (the
 *                      on-chip K split).
 *
 * One launch covers every product when the operands are 16-bit, A and B are
 * 16-byte aligned with 16-byte row pitches and 16-byte batch strides.
 * Otherwise (TF32 operands, misaligned A or B) each product is run as its own
 * tg_gemm_ex call on `stream`, in order of z.  Ownership, asynchrony and error
 * behaviour as for tg_gemm; batch > 2^31-1 or more than 2^30 output tiles in
 * all return TG_ERR_UNSUPPORTED.
 */
tg_status tg_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                                  const void *a, int64_t lda, int64_t stride_a,
                                  const void *b, int64_t ldb, int64_t stride_b,
                                  void *c, int64_t ldc, int64_t stride_c,
                                  tg_dtype dtype_in, tg_dtype dtype_out,
                                  void *stream, const tg_options *opt);

/*
 * tg_gemm_strided_batched_fused -- tg_gemm_strided_batched with the epilogue
 * of tg_gemm_fused applied to every product:
 *
 *     C_z[m,n] = act(alpha * scale[n] * (A_z B_z)[m,n] + bias[n]) + beta * R_z[m,n]
 *     R_z = residual + z*stride_r
 *
 * The batched product and the fused epilogue together: the batch axis of the
 * tiled multiply ("Triton tiled matmul", llm-systems-cookbook, "Exercises")
 * with the output-tile work that "Matrix Multiplication" (teenygrad docs)
 * hands on to its chapter "Fusing an Epilogue".
 *
 *   batch .. stride_c, dtype_in, dtype_out, stream, opt
 *              as for tg_gemm_strided_batched
 *   epilogue   NULL: exactly tg_gemm_strided_batched (stride_r must be 0).
 *              alpha, beta, activation and the per-column scale / bias are
 *              shared by every product; rules as for tg_gemm_fused.
 *   stride_r   elements between consecutive products' residual blocks (>= 0;
 *              0 reads one residual block for every product; must be 0
 *              without a residual).  The residuals of all products may be C
 *              itself (residual == c, ldr == ldc, stride_r == stride_c: each
 *              product's C is its own residual) but must not otherwise
 *              overlap the whole of C -> else TG_ERR_INVALID_VALUE.
 *
 * One launch covers every product under the conditions of
 * tg_gemm_strided_batched; otherwise each product is one tg_gemm_fused call
 * on `stream`, in order of z.  K == 0 writes each product's epilogue of the
 * empty sum.
 */
tg_status tg_gemm_strided_batched_fused(int64_t batch, int64_t M, int64_t N, int64_t K,
                                        const void *a, int64_t lda, int64_t stride_a,
                                        const void *b, int64_t ldb, int64_t stride_b,
                                        void *c, int64_t ldc, int64_t stride_c,
                                        tg_dtype dtype_in, tg_dtype dtype_out,
                                        const tg_epilogue *epilogue, int64_t stride_r,
                                        void *stream, const tg_options *opt);

/*
 * tg_plan_gemm_strided_batched -- host only, like tg_plan_gemm: validates as
 * tg_gemm_strided_batched does and fills *plan with what it would launch on a
 * device with `num_sms` SMs (tiles counts the tiles of all products).  No
 * counterpart in the pages.
 */
tg_status tg_plan_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                                       const void *a, int64_t lda, int64_t stride_a,
                                       const void *b, int64_t ldb, int64_t stride_b,
                                       const void *c, int64_t ldc, int64_t stride_c,
                                       tg_dtype dtype_in, tg_dtype dtype_out,
                                       int32_t num_sms, const tg_options *opt, tg_plan *plan);

/* Static, human-readable name of a status code (library plumbing, no
 * counterpart in the pages; the string is owned by the library). */
const char *tg_status_string(tg_status status);

/*
 * tg_last_device_error -- synchronises `stream`, then reads and clears the
 * current device's status word.  Returns TG_OK if no kernel recorded a
 * failure since the last call, TG_ERR_TIMEOUT if a bounded wait ran out, or
 * TG_ERR_CUDA if the synchronisation itself failed or a kernel found its
 * shared memory not aligned as it requires (it then returns without writing
 * C), or, in a checked build, TG_ERR_BOUNDS if a device-side check failed.  No counterpart in the pages, which report no device-side failures.
 */
tg_status tg_last_device_error(void *stream);

/*
 * Checked builds.  `python -m tiled_matrix_multiplication_gb300.build --checked`
 * builds libtg_gemm_checked.so: the same library compiled with device-side
 * checks in front of the tensor-core kernels' shared-memory, tensor-memory,
 * TMA and cluster-remote accesses (each box of a TMA load or store inside its
 * ring or staging area with a 16-byte aligned innermost coordinate and no
 * negative store coordinate, each MMA's operands inside the ring, each
 * tensor-memory load inside its accumulator, each remote store and received
 * cell inside the receive area).  A failed check records TG_ERR_BOUNDS and the
 * check site in the status word and the access is skipped -- nothing traps;
 * the kernel ends through its bounded waits and tg_last_device_error()
 * returns TG_ERR_BOUNDS.  Python loads it instead of libtg_gemm.so when
 * TG_CHECKED=1 is set.  No counterpart in the pages.
 *
 * tg_checked_build -- 1 in a checked build, 0 otherwise.
 */
int32_t tg_checked_build(void);

/*
 * tg_selftest_bounds -- check of the checked-build mechanism: enqueues on
 * `stream` a one-warp kernel that makes one checked store to element `index`
 * of a 32-element device array; an index outside 0 .. 31 fails the check, so
 * the store is skipped and TG_ERR_BOUNDS is recorded (tg_last_device_error
 * then returns it and clears it).  TG_ERR_INVALID_VALUE for index < 0 or
 * index > 1024; TG_ERR_NOT_IMPLEMENTED in a normal build (no checks compiled
 * in).  No counterpart in the pages.
 */
tg_status tg_selftest_bounds(int32_t index, void *stream);

/*
 * tg_selftest_timeout -- failure-detection check: enqueues on `stream` a
 * one-thread kernel that waits on a shared-memory barrier nothing ever
 * arrives on, with the same bounded wait (global-time limit) the GEMM kernels
 * use, and records TG_ERR_TIMEOUT in the device status word when the limit
 * (timeout_ms, 1 .. 10000) runs out; the kernel then exits normally and the
 * context stays usable.  tg_last_device_error(stream) afterwards returns
 * TG_ERR_TIMEOUT (and clears it).  No GEMM counterpart in the pages: this
 * exercises the library's own bounded-wait failure path.
 */
tg_status tg_selftest_timeout(int32_t timeout_ms, void *stream);

/* TG_ABI_VERSION of the loaded library (no counterpart in the pages). */
int32_t tg_abi_version(void);

/* Size of the library-owned device array used by tg_gemm_splitk_noalloc. */
#define TG_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * tg_gemm_splitk_noalloc -- C = A * B split over `splits` ranges of K, with the
 * FP32 partial tiles kept in a fixed device array of TG_NOALLOC_SCRATCH_BYTES
 * that the library owns, so that the call allocates no device memory.  The
 * pages have no counterpart: this serves callers that cannot let a library
 * allocate -- an application whose device memory is all held by its own
 * allocator, or a code path that must not enter the allocator at all.
 *
 *   M, N, K, a, lda, b, ldb, c, ldc, dtype_out, stream  as for tg_gemm
 *   dtype_in   TG_F16 or TG_BF16
 *   splits     1 .. 128 K ranges; the planner may use fewer when K is short
 *
 * Returns TG_ERR_UNSUPPORTED when splits x M x N x 4 bytes exceeds
 * TG_NOALLOC_SCRATCH_BYTES, when A or B is not 16-byte aligned in base and row
 * pitch (they are read in place), or for other operand types; argument errors as for
 * tg_gemm.  The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress); make that first call outside
 * any stream capture.  Every call on a device shares the one array: calls
 * whose work may overlap on the GPU (unordered streams) race on it.
 */
tg_status tg_gemm_splitk_noalloc(int64_t M, int64_t N, int64_t K,
                                 const void *a, int64_t lda,
                                 const void *b, int64_t ldb,
                                 void *c, int64_t ldc,
                                 tg_dtype dtype_in, tg_dtype dtype_out,
                                 int32_t splits, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TG_GEMM_H */
