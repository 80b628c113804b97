// aux_kernels.cu -- the two memory-bound helper kernels of the GEMM path.
//
// pack_rows: copies a row-major block whose base or row pitch is not
//   16-byte aligned into a workspace with an aligned pitch.  The tensor-memory
//   copy engine (TMA) behind the "tensor descriptors" of the teenygrad page
//   ("Matrix Multiplication", section "The real tiled loop") imposes exactly
//   this alignment on its source; the padded columns are never read because
//   the descriptor's logical width stays the original one.
// pack_transpose: writes B^T ([N, K], K contiguous) into the workspace for
//   operand types whose MMA wants B K-major.
// splitk_reduce: C[m,n] = round(epilogue(sum_{s=0}^{S-1} P[s,m,n])) in increasing s --
//   the K-chunk sum of the lesson-6 walk-through ("the accumulator must survive
//   both steps"), finished across work units instead of inside one.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tg_epilogue.cuh"
#include "tg_internal.h"
#include "tg_kernel_common.cuh"
#include "tg_ptx.cuh"

namespace tg {
namespace {

template <typename T>
__global__ void pack_rows_kernel(const T *__restrict__ src, int64_t ld_src, T *__restrict__ dst,
                                 int64_t ld_dst, int64_t rows, int64_t cols) {
    const int64_t total = rows * cols;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / cols;
        const int64_t c = i - r * cols;
        dst[r * ld_dst + c] = src[r * ld_src + c];
    }
}

// dst[c * ld_dst + r] = src[r * ld_src + c] for a rows x cols block, through
// 32 x 32 shared-memory tiles so both the reads and the writes are coalesced.
template <typename T>
__global__ void pack_transpose_kernel(const T *__restrict__ src, int64_t ld_src,
                                      T *__restrict__ dst, int64_t ld_dst, int64_t rows,
                                      int64_t cols) {
    __shared__ T tile[32][33];
    const int64_t tiles_c = (cols + 31) / 32;
    const int64_t tiles_r = (rows + 31) / 32;
    for (int64_t t = blockIdx.x; t < tiles_r * tiles_c; t += gridDim.x) {
        const int64_t r0 = (t / tiles_c) * 32;
        const int64_t c0 = (t % tiles_c) * 32;
        for (int i = threadIdx.y; i < 32; i += blockDim.y) {
            const int64_t r = r0 + i, c = c0 + threadIdx.x;
            if (r < rows && c < cols) tile[i][threadIdx.x] = src[r * ld_src + c];
        }
        __syncthreads();
        for (int i = threadIdx.y; i < 32; i += blockDim.y) {
            const int64_t c = c0 + i, r = r0 + threadIdx.x;
            if (r < rows && c < cols) dst[c * ld_dst + r] = tile[threadIdx.x][i];
        }
        __syncthreads();
    }
}

// x = hi + lo + r with hi and lo TF32 values (10 fraction bits; the
// cvt.rna.tf32.f32 instruction: round to nearest, ties away from zero) and
// |r| <= 2^-11 |lo| <= about 2^-22 |x|; x - hi is exact in FP32.  A non-finite
// hi keeps lo = 0.
__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo) {
    uint32_t h, l;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
    hi = __uint_as_float(h);
    if (!isfinite(hi)) {
        lo = 0.f;
        return;
    }
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(x - hi));
    lo = __uint_as_float(l);
}

// A' = [hi(A) | lo(A) | hi(A)], [M, 3K] with pitch ld_dst.
__global__ void split3_rows_kernel(const float *__restrict__ a, int64_t lda, float *__restrict__ dst,
                                   int64_t ld_dst, int64_t M, int64_t K) {
    const int64_t total = M * K;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / K;
        const int64_t k = i - m * K;
        float hi, lo;
        split_tf32(a[m * lda + k], hi, lo);
        float *row = dst + m * ld_dst;
        row[k] = hi;
        row[K + k] = lo;
        row[2 * K + k] = hi;
    }
}

// B'^T = [hi(B)^T | hi(B)^T | lo(B)^T], [N, 3K] with pitch ld_dst, through
// 32 x 32 shared-memory tiles so reads of B and writes of B'^T are coalesced.
__global__ void split3_transpose_kernel(const float *__restrict__ b, int64_t ldb,
                                        float *__restrict__ dst, int64_t ld_dst, int64_t K,
                                        int64_t N) {
    __shared__ float hi_t[32][33], lo_t[32][33];
    const int64_t tiles_n = (N + 31) / 32;
    const int64_t tiles_k = (K + 31) / 32;
    for (int64_t t = blockIdx.x; t < tiles_k * tiles_n; t += gridDim.x) {
        const int64_t k0 = (t / tiles_n) * 32;
        const int64_t n0 = (t % tiles_n) * 32;
        for (int i = threadIdx.y; i < 32; i += blockDim.y) {
            const int64_t k = k0 + i, n = n0 + threadIdx.x;
            if (k < K && n < N) split_tf32(b[k * ldb + n], hi_t[i][threadIdx.x], lo_t[i][threadIdx.x]);
        }
        __syncthreads();
        for (int i = threadIdx.y; i < 32; i += blockDim.y) {
            const int64_t n = n0 + i, k = k0 + threadIdx.x;
            if (k < K && n < N) {
                float *row = dst + n * ld_dst;
                row[k] = hi_t[threadIdx.x][i];
                row[K + k] = hi_t[threadIdx.x][i];
                row[2 * K + k] = lo_t[threadIdx.x][i];
            }
        }
        __syncthreads();
    }
}

__device__ __forceinline__ void store_out(void *c, int64_t off, int out_kind, float v) {
    if (out_kind == OUT_F32)
        static_cast<float *>(c)[off] = v;
    else if (out_kind == OUT_F16)
        static_cast<__half *>(c)[off] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16 *>(c)[off] = __float2bfloat16_rn(v);
}

// One thread per 4 consecutive columns of one row.
__global__ void splitk_reduce_kernel(const float *__restrict__ partial, int splits, int64_t M,
                                     int64_t N, void *c, int64_t ldc, int out_kind,
                                     int vec_ok, const EpiParams epi) {
    const int64_t groups_per_row = (N + 3) / 4;
    const int64_t total = M * groups_per_row;
    const int64_t plane = M * N;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = g / groups_per_row;
        const int64_t n0 = (g - m * groups_per_row) * 4;
        const int64_t src = m * N + n0;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (vec_ok && n0 + 4 <= N) {
            for (int s = 0; s < splits; ++s) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(partial + s * plane + src));
                acc[0] += v.x;
                acc[1] += v.y;
                acc[2] += v.z;
                acc[3] += v.w;
            }
        } else {
            const int nv = static_cast<int>(N - n0 < 4 ? N - n0 : 4);
            for (int s = 0; s < splits; ++s)
                for (int j = 0; j < nv; ++j) acc[j] += partial[s * plane + src + j];
        }
        const int nv = static_cast<int>(N - n0 < 4 ? N - n0 : 4);
        if (epi.on)
            for (int j = 0; j < nv; ++j) acc[j] = epi_one(epi, out_kind, m, n0 + j, acc[j]);
        for (int j = 0; j < nv; ++j) store_out(c, m * ldc + n0 + j, out_kind, acc[j]);
    }
}

// Failure-detection check: the wait of the GEMM kernels (mbar_wait, bounded
// by global time) on a barrier whose phase never completes, then the same
// failure record.  One thread; no memory other than the status word.
__global__ void selftest_timeout_kernel(int *status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int never_abort;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        never_abort = 0;
        mbar_init(b, 1);
        fence_mbar_init();
        if (!mbar_wait(b, 0, timeout_ns, &never_abort))
            record_failure(status, 6, (ROLE_SELFTEST << 16) | 1);
    }
}

int grid_for(int64_t work, int threads) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    return static_cast<int>(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

}  // namespace

cudaError_t launch_pack_rows(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                             int64_t rows, int64_t cols, int esize, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = grid_for(rows * cols, threads);
    if (esize == 1)
        pack_rows_kernel<uint8_t><<<blocks, threads, 0, stream>>>(
            static_cast<const uint8_t *>(src), ld_src, static_cast<uint8_t *>(dst), ld_dst, rows,
            cols);
    else if (esize == 2)
        pack_rows_kernel<uint16_t><<<blocks, threads, 0, stream>>>(
            static_cast<const uint16_t *>(src), ld_src, static_cast<uint16_t *>(dst), ld_dst, rows,
            cols);
    else if (esize == 4)
        pack_rows_kernel<uint32_t><<<blocks, threads, 0, stream>>>(
            static_cast<const uint32_t *>(src), ld_src, static_cast<uint32_t *>(dst), ld_dst, rows,
            cols);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_pack_transpose(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                                  int64_t rows, int64_t cols, int esize, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int64_t tiles = ((rows + 31) / 32) * ((cols + 31) / 32);
    const dim3 block(32, 8);
    const int blocks = grid_for(tiles * 256, 256);
    if (esize == 2)
        pack_transpose_kernel<uint16_t><<<blocks, block, 0, stream>>>(
            static_cast<const uint16_t *>(src), ld_src, static_cast<uint16_t *>(dst), ld_dst,
            rows, cols);
    else if (esize == 4)
        pack_transpose_kernel<uint32_t><<<blocks, block, 0, stream>>>(
            static_cast<const uint32_t *>(src), ld_src, static_cast<uint32_t *>(dst), ld_dst,
            rows, cols);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(int *status, uint64_t timeout_ns, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

cudaError_t launch_split3_rows(const void *a, int64_t lda, void *dst, int64_t ld_dst, int64_t M,
                               int64_t K, cudaStream_t stream) {
    if (M <= 0 || K <= 0) return cudaSuccess;
    const int threads = 256;
    split3_rows_kernel<<<grid_for(M * K, threads), threads, 0, stream>>>(
        static_cast<const float *>(a), lda, static_cast<float *>(dst), ld_dst, M, K);
    return cudaGetLastError();
}

cudaError_t launch_split3_transpose(const void *b, int64_t ldb, void *dst, int64_t ld_dst,
                                    int64_t K, int64_t N, cudaStream_t stream) {
    if (K <= 0 || N <= 0) return cudaSuccess;
    const int64_t tiles = ((K + 31) / 32) * ((N + 31) / 32);
    split3_transpose_kernel<<<grid_for(tiles * 256, 256), dim3(32, 8), 0, stream>>>(
        static_cast<const float *>(b), ldb, static_cast<float *>(dst), ld_dst, K, N);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float *partial, int splits, int64_t M, int64_t N, void *c,
                                 int64_t ldc, int out_kind, int c_vector, cudaStream_t stream,
                                 const EpiParams *epi) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    (void)c_vector;
    const int threads = 256;
    const int64_t work = M * ((N + 3) / 4);
    const int vec_ok = (N % 4) == 0;
    EpiParams e{};
    if (epi) e = *epi;
    splitk_reduce_kernel<<<grid_for(work, threads), threads, 0, stream>>>(partial, splits, M, N, c,
                                                                          ldc, out_kind, vec_ok, e);
    return cudaGetLastError();
}

}  // namespace tg
