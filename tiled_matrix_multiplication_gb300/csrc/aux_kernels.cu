// aux_kernels.cu -- the memory-bound helper kernels of the GEMM path.
//
// pack_rows: copies a row-major block whose base or row pitch is not
//   16-byte aligned into a workspace with an aligned pitch.  The tensor-memory
//   copy engine (TMA) behind the "tensor descriptors" of the teenygrad page
//   ("Matrix Multiplication", section "The real tiled loop") imposes exactly
//   this alignment on its source; the padded columns are never read because
//   the descriptor's logical width stays the original one.
// split3_rows / split3_stack: the TF32 hi / lo parts of FP32 operands for the
//   3xTF32 mode.
// splitk_reduce: C[m,n] = round(epilogue(sum_{s=0}^{S-1} P[s,m,n])) in increasing s --
//   the K-chunk sum of the lesson-6 walk-through ("the accumulator must survive
//   both steps"), finished across work units instead of inside one.
//
// All of them are launched with programmatic dependent launch, like the GEMM
// kernels: a launch may be scheduled while the previous kernel of the stream
// drains, waits for that kernel's writes before its first global-memory
// access (griddepcontrol.wait), and at once lets the kernel after it be
// scheduled.  A call made of a pack and a GEMM then pays one launch latency
// instead of two (127 x 255 x 65 with both operands packed: 18.5 us a call
// with plain launches).
#include <algorithm>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tg_epilogue.cuh"
#include "tg_internal.h"
#include "tg_kernel_common.cuh"
#include "tg_ptx.cuh"

namespace tg {
namespace {

// grid.x over groups of V = 16 / sizeof(T) columns (one group per thread),
// grid.y over rows (each block loops over rows gridDim.y apart).  The
// destination's base and pitch are 16-byte aligned, so a thread gathers its V
// elements with plain loads (the source is the unaligned one) and writes them
// with one 16-byte store.
template <typename T>
__global__ void __launch_bounds__(256) pack_rows_kernel(const T *__restrict__ src, int64_t ld_src,
                                                        T *__restrict__ dst, int64_t ld_dst,
                                                        int64_t rows, int64_t cols) {
    grid_dependency_wait();
    grid_launch_dependents();
    constexpr int V = 16 / static_cast<int>(sizeof(T));
    const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * V;
    if (c >= cols) return;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const T *s = src + r * ld_src + c;
        T *d = dst + r * ld_dst + c;
        if (c + V <= cols) {
            union {
                T e[V];
                uint4 u;
            } w;
#pragma unroll
            for (int e = 0; e < V; ++e) w.e[e] = s[e];
            *reinterpret_cast<uint4 *>(d) = w.u;
        } else {
            for (int e = 0; c + e < cols; ++e) d[e] = s[e];
        }
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

// Both split kernels take a rows x cols source 4 columns per thread: grid.x
// over column groups (256 threads x 4 columns per block), grid.y over rows
// (each block loops over rows gridDim.y apart).  `vec`: the source base and
// pitch and every destination column block are 16-byte aligned, so a thread
// moves its 4 columns with one 16-byte load and 16-byte stores.

// A' = [hi(A) | lo(A) | hi(A)], [M, 3K] with pitch ld_dst.
__global__ void __launch_bounds__(256) split3_rows_kernel(const float *__restrict__ a, int64_t lda,
                                                          float *__restrict__ dst, int64_t ld_dst,
                                                          int64_t M, int64_t K, int vec) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t k = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (k >= K) return;
    for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
        const float *src = a + m * lda + k;
        float *row = dst + m * ld_dst;
        if (vec) {
            const float4 x = *reinterpret_cast<const float4 *>(src);
            float4 hi, lo;
            split_tf32(x.x, hi.x, lo.x);
            split_tf32(x.y, hi.y, lo.y);
            split_tf32(x.z, hi.z, lo.z);
            split_tf32(x.w, hi.w, lo.w);
            *reinterpret_cast<float4 *>(row + k) = hi;
            *reinterpret_cast<float4 *>(row + K + k) = lo;
            *reinterpret_cast<float4 *>(row + 2 * K + k) = hi;
        } else {
            for (int64_t c = k; c < K && c < k + 4; ++c) {
                float hi, lo;
                split_tf32(a[m * lda + c], hi, lo);
                row[c] = hi;
                row[K + c] = lo;
                row[2 * K + c] = hi;
            }
        }
    }
}

// B' = [hi(B); hi(B); lo(B)] stacked along K: [3K, N] with pitch ld_dst,
// read by the TF32 kernel N-major like B itself.
__global__ void __launch_bounds__(256) split3_stack_kernel(const float *__restrict__ b, int64_t ldb,
                                                           float *__restrict__ dst, int64_t ld_dst,
                                                           int64_t K, int64_t N, int vec) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t n = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (n >= N) return;
    for (int64_t k = blockIdx.y; k < K; k += gridDim.y) {
        float *d0 = dst + k * ld_dst + n;
        float *d1 = d0 + K * ld_dst;
        float *d2 = d1 + K * ld_dst;
        if (vec) {
            const float4 x = *reinterpret_cast<const float4 *>(b + k * ldb + n);
            float4 hi, lo;
            split_tf32(x.x, hi.x, lo.x);
            split_tf32(x.y, hi.y, lo.y);
            split_tf32(x.z, hi.z, lo.z);
            split_tf32(x.w, hi.w, lo.w);
            *reinterpret_cast<float4 *>(d0) = hi;
            *reinterpret_cast<float4 *>(d1) = hi;
            *reinterpret_cast<float4 *>(d2) = lo;
        } else {
            for (int64_t c = 0; c < 4 && n + c < N; ++c) {
                float hi, lo;
                split_tf32(b[k * ldb + n + c], hi, lo);
                d0[c] = hi;
                d1[c] = hi;
                d2[c] = lo;
            }
        }
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
    grid_dependency_wait();      // the partials of the GEMM kernel before it
    grid_launch_dependents();
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

#ifdef TG_CHECKED
// Checked builds: lane 0 makes one checked store to element `index` of a
// 32-element shared array; outside 0 .. 31 the check fails, the store is
// skipped and TG_ERR_BOUNDS is recorded.
__global__ void selftest_bounds_kernel(int *status, int index) {
    volatile __shared__ int cells[32];
    cells[threadIdx.x] = 0;
    __syncwarp();
    if (threadIdx.x == 0 && tg_check(status, index >= 0 && index < 32, CHK_SELFTEST, index))
        cells[index] = 1;
}
#endif

int grid_for(int64_t work, int threads) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    return static_cast<int>(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

// Launches `kern` with programmatic stream serialisation allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_rows(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                             int64_t rows, int64_t cols, int esize, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (esize != 1 && esize != 2 && esize != 4) return cudaErrorInvalidValue;
    const int threads = 256;
    const int64_t per_block = static_cast<int64_t>(threads) * (16 / esize);   // columns
    const int bx = static_cast<int>((cols + per_block - 1) / per_block);
    const int total = grid_for(static_cast<int64_t>(bx) * rows * threads, threads);
    const int by = static_cast<int>(std::min<int64_t>(std::min<int64_t>(rows, 65535),
                                                       std::max<int64_t>(1, total / bx)));
    const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(by));
    if (esize == 1)
        return launch_pdl(pack_rows_kernel<uint8_t>, grid, dim3(threads), stream,
                          static_cast<const uint8_t *>(src), ld_src, static_cast<uint8_t *>(dst),
                          ld_dst, rows, cols);
    if (esize == 2)
        return launch_pdl(pack_rows_kernel<uint16_t>, grid, dim3(threads), stream,
                          static_cast<const uint16_t *>(src), ld_src,
                          static_cast<uint16_t *>(dst), ld_dst, rows, cols);
    if (esize == 4)
        return launch_pdl(pack_rows_kernel<uint32_t>, grid, dim3(threads), stream,
                          static_cast<const uint32_t *>(src), ld_src,
                          static_cast<uint32_t *>(dst), ld_dst, rows, cols);
    return cudaErrorInvalidValue;
}

cudaError_t launch_selftest_timeout(int *status, uint64_t timeout_ns, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

#ifdef TG_CHECKED
cudaError_t launch_selftest_bounds(int *status, int index, cudaStream_t stream) {
    selftest_bounds_kernel<<<1, 32, 0, stream>>>(status, index);
    return cudaGetLastError();
}
#endif

// 2-D grid of the split kernels: column groups of 1024 (256 threads x 4) on
// x, rows on y (at most 65535 blocks; the kernels loop over the rest).
static dim3 split_grid(int64_t rows, int64_t cols) {
    const int64_t gx = (cols + 1023) / 1024;
    const int64_t gy = std::min<int64_t>(rows, std::max<int64_t>(1, 4096 / std::max<int64_t>(gx, 1)));
    return dim3(static_cast<unsigned>(gx), static_cast<unsigned>(std::min<int64_t>(std::max<int64_t>(gy, 1), 65535)));
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_split3_rows(const void *a, int64_t lda, void *dst, int64_t ld_dst, int64_t M,
                               int64_t K, cudaStream_t stream) {
    if (M <= 0 || K <= 0) return cudaSuccess;
    if ((K + 1023) / 1024 > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const int vec = aligned16(a) && aligned16(dst) && lda % 4 == 0 && ld_dst % 4 == 0 && K % 4 == 0;
    return launch_pdl(split3_rows_kernel, split_grid(M, K), dim3(256), stream,
                      static_cast<const float *>(a), lda, static_cast<float *>(dst), ld_dst, M,
                      K, vec);
}

cudaError_t launch_split3_stack(const void *b, int64_t ldb, void *dst, int64_t ld_dst,
                                int64_t K, int64_t N, cudaStream_t stream) {
    if (K <= 0 || N <= 0) return cudaSuccess;
    if ((N + 1023) / 1024 > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const int vec = aligned16(b) && aligned16(dst) && ldb % 4 == 0 && ld_dst % 4 == 0 && N % 4 == 0;
    return launch_pdl(split3_stack_kernel, split_grid(K, N), dim3(256), stream,
                      static_cast<const float *>(b), ldb, static_cast<float *>(dst), ld_dst, K,
                      N, vec);
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
    return launch_pdl(splitk_reduce_kernel, dim3(grid_for(work, threads)), dim3(threads), stream,
                      partial, splits, M, N, c, ldc, out_kind, vec_ok, e);
}

}  // namespace tg
