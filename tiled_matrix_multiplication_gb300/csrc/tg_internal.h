// tg_internal.h -- interface between the host side of the library (tg_api.cu)
// and its kernels.  Not installed; the public ABI is include/tg_gemm.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tg {

enum InKind : int { IN_F16 = 0, IN_BF16 = 1, IN_TF32 = 2, IN_E4M3 = 3, IN_E5M2 = 4 };

// Bytes of one operand element.
__host__ __device__ constexpr int in_esize(int in_kind) {
    return in_kind == IN_TF32 ? 4 : (in_kind == IN_E4M3 || in_kind == IN_E5M2 ? 1 : 2);
}
enum OutKind : int { OUT_F16 = 0, OUT_BF16 = 1, OUT_F32 = 2 };

// Device status word layout: [0] first tg_status code recorded, [1] where it
// was recorded (role << 16 | detail).
enum FailRole : int { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3, ROLE_DRAIN = 4,
                      ROLE_SELFTEST = 5, ROLE_LAYOUT = 6 };

enum Act : int { ACT_NONE = 0, ACT_RELU = 1, ACT_SILU = 2, ACT_GELU_TANH = 3 };

// Fused epilogue, applied to each FP32 accumulator value before its single
// rounding to the output type:  D = act(alpha * scale[n] * acc + bias[n]) +
// beta * R[m, n].  With on == 0 no other field is read.
struct EpiParams {
    int32_t on, act;
    float alpha, beta;
    const float *scale;         // [N] or null (1)
    const float *bias;          // [N] or null (0)
    const void *res;            // [M][ldr] in the output type, or null
    int64_t ldr;                // elements
    int64_t stride_r;           // elements between the residuals of batch products
    int32_t res_vector;         // res base and pitch allow 16-byte loads
    int32_t sb_vector;          // scale and bias allow 16-byte loads
};

// Parameters of the tensor-core GEMM kernel (one persistent launch).
struct TcParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n;
    int32_t k_tiles;            // ceil(K / BK)
    int32_t k_tiles_per_split;  // K tiles per split
    int32_t splits;             // 1: write C; > 1: write FP32 partials
    int32_t group_m;            // grouped raster height (tiles)
    int32_t out_kind;           // OutKind of C
    int32_t c_vector;           // C base and row pitch allow 16-byte stores
    int32_t mc;                 // tiles per work unit (2: two pairs share A by multicast)
    int64_t ldc;                // elements
    void *c;
    float *partial;             // [splits][M][N] when splits > 1
    int *status;                // device status word (2 ints)
    uint64_t timeout_ns;
    // 1: C is written by TMA stores through the tensor map tmC ([N, M] or, for
    // a batch, [N, M, batch]; boxes of 64 bytes x 32 rows, 64-byte swizzle);
    // 0: by the epilogue warps' own stores (split-K partials, or C whose base,
    // row pitch, row length or batch stride is not a multiple of 16 bytes)
    int32_t c_tma, pad1_;
    // Strided batch: `batch` independent products; A / B use rank-3 tensor maps
    // (z = batch index) when a_batched / b_batched, else one 2-D map shared by
    // every batch (stride 0); C of batch z starts at c + z * stride_c.
    int32_t batch, a_batched, b_batched, pad2_;
    int64_t stride_c;           // elements
    EpiParams epi;              // applied where C is written (splits == 1)
};

// Parameters of the small-M kernel (gemm_skinny.cu): C^T = B^T A^T with NT
// output columns per tile and all M <= 128 rows in one tile; one CTA per
// (tile, K range), the K ranges of a tile forming one cluster.
struct SkParams {
    int32_t M, N, K;
    int32_t tiles_n;            // ceil(N / NT)
    int32_t k_tiles;            // ceil(K / 64)
    int32_t k_tiles_per_split;
    int32_t splits;             // cluster size: 1, 2, 4 or 8
    int32_t out_kind;
    int32_t two_per_sm;         // half-size ring, two CTAs per SM
    int32_t batch;              // gridDim.y; A / B rank-3 when a_batched / b_batched
    int32_t a_batched, b_batched;
    int32_t c_vector;           // C base, row pitch and batch stride are 16-byte multiples
    int64_t stride_c;           // elements between the C of consecutive batches
    int64_t ldc;
    void *c;
    int *status;
    uint64_t timeout_ns;
    EpiParams epi;
};

// gemm_skinny.cu -- mp: MMA N used for the M rows (16, 32, 64, 128); nt: output
// columns per CTA (128, 256, 512)
int skinny_rows(int64_t M);
bool skinny_supported(int mp, int nt);
int skinny_stages(int mp, int nt, bool two);
cudaError_t launch_gemm_skinny(int in_kind, int mp, int nt, const CUtensorMap &tmA,
                               const CUtensorMap &tmB, const SkParams &p, cudaStream_t stream);
// gemm_skinny_fp8.cu: the E4M3 / E5M2 instantiations behind launch_gemm_skinny
cudaError_t launch_gemm_skinny_fp8(int in_kind, int mp, int nt, const CUtensorMap &tmA,
                                   const CUtensorMap &tmB, const SkParams &p,
                                   cudaStream_t stream);

// gemm_tc.cu
// `pair`: the CTA-pair (cta_group::2, 256-row tile) variant; `mc` = 2: clusters
// of two pairs sharing A by multicast; `ctas` counts CTAs.
int tc_stages(int in_kind, int block_n, bool pair);
// Tile widths: 128, 192, 224, 256 for single CTAs and pairs; 512 for pairs.
bool tc_supported_block_n(int in_kind, int block_n, bool pair);
// A-multicast clusters (mc = 2): pairs with 192-, 224- or 256-wide tiles.
bool tc_supported_mc(int block_n, int mc, bool pair);
// Swizzle (row bytes of a TMA box) of the N-major B tile of a variant.
int tc_b_swizzle_bytes(int in_kind, int block_n, bool pair);
// Clusters of `cluster_size` (2 or 4) CTAs of the pair kernel resident at
// once on the current device (0 if the query fails).
int tc_max_clusters(int cluster_size);
cudaError_t launch_gemm_tc(int in_kind, int block_n, bool pair, int mc, const CUtensorMap &tmA,
                           const CUtensorMap &tmB, const CUtensorMap &tmC, const TcParams &p,
                           int ctas, cudaStream_t stream);
// The instantiations behind launch_gemm_tc, one translation unit per operand
// type (gemm_tc_f16.cu, gemm_tc_tf32.cu, gemm_tc_fp8.cu).
cudaError_t launch_gemm_tc_16bit(int in_kind, int block_n, bool pair, int mc,
                                 const CUtensorMap &tmA, const CUtensorMap &tmB,
                                 const CUtensorMap &tmC, const TcParams &p, int ctas,
                                 cudaStream_t stream);
cudaError_t launch_gemm_tc_tf32(int block_n, bool pair, int mc, const CUtensorMap &tmA,
                                const CUtensorMap &tmB, const CUtensorMap &tmC,
                                const TcParams &p, int ctas, cudaStream_t stream);
cudaError_t launch_gemm_tc_fp8(int in_kind, int block_n, bool pair, int mc,
                               const CUtensorMap &tmA, const CUtensorMap &tmB,
                               const CUtensorMap &tmC, const TcParams &p, int ctas,
                               cudaStream_t stream);
cudaError_t status_word_address(int **out);
cudaError_t set_smem_once(const void *kernel, int bytes);

// aux_kernels.cu
cudaError_t launch_pack_rows(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                             int64_t rows, int64_t cols, int esize, cudaStream_t stream);
// One CTA waits, bounded by timeout_ns, on an mbarrier that nothing arrives
// on, and records TG_ERR_TIMEOUT in `status` the way the GEMM kernels do.
cudaError_t launch_selftest_timeout(int *status, uint64_t timeout_ns, cudaStream_t stream);
#ifdef TG_CHECKED
cudaError_t launch_selftest_bounds(int *status, int index, cudaStream_t stream);
#endif
// C = the sum of the `splits` partial planes, through the epilogue `epi`
// (splits == 0: the empty sum, i.e. the epilogue of zero).
// 3xTF32 operand splitting (x = hi + lo with both parts TF32 values):
// dst[m, 0:K) = hi(A), [K, 2K) = lo(A), [2K, 3K) = hi(A)   (A' rows, [M, 3K])
// dst rows [0, K) = hi(B), [K, 2K) = hi(B), [2K, 3K) = lo(B)  (B', [3K, N])
cudaError_t launch_split3_rows(const void *a, int64_t lda, void *dst, int64_t ld_dst, int64_t M,
                               int64_t K, cudaStream_t stream);
cudaError_t launch_split3_stack(const void *b, int64_t ldb, void *dst, int64_t ld_dst,
                                int64_t K, int64_t N, cudaStream_t stream);
cudaError_t launch_splitk_reduce(const float *partial, int splits, int64_t M, int64_t N,
                                 void *c, int64_t ldc, int out_kind, int c_vector,
                                 cudaStream_t stream, const EpiParams *epi = nullptr);

}  // namespace tg
