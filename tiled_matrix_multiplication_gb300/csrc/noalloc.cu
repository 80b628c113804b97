// noalloc.cu -- tg_gemm_splitk_noalloc: the split-K GEMM with its FP32 partial
// tiles kept in a fixed device array owned by the library, so a call allocates
// no device memory at all.
//
// Why: tg_gemm_ex takes its split-K workspace from cudaMallocAsync on the
// caller's stream.  Some callers cannot have the library allocate: an
// application whose device memory is entirely managed by its own allocator (a
// framework that reserved nearly all of HBM up front, where an extra
// allocation fails or fragments its pool), or a code path that must not touch
// the allocator at all (a latency-critical decode loop with a fixed memory
// plan).  This entry point gives them the same split-K GEMM with the partials
// in `g_splitk_scratch`, a file-scope array of TG_NOALLOC_SCRATCH_BYTES that
// every device which loads the library holds until the process exits.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it; a host-side
// use of the symbol itself would not be a device address.  Make that first
// call outside any stream capture.
//
// Sharing: every call on a device uses the same array.  Each call overwrites
// every partial element it later reads, so nothing needs clearing between
// calls, but two calls whose kernels overlap on the GPU (different streams
// without ordering between them) race on the array.
#include "tg_host_api.h"

namespace {

constexpr int64_t kScratchFloats = static_cast<int64_t>(TG_NOALLOC_SCRATCH_BYTES) / 4;

static __device__ __align__(256) float g_splitk_scratch[kScratchFloats];

using tgh::kMaxDevices;

struct NoAllocDevice {
    bool init = false;
    tg_status arch = TG_OK;
    int sms = 0;
    float *scratch = nullptr;
    int *status = nullptr;
};

std::mutex g_mu;
NoAllocDevice g_devs[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device set-up, done once with the device current.
tg_status setup_current_device(NoAllocDevice **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocDevice &d = g_devs[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TG_ERR_CUDA;
        d.sms = sms;
        d.arch = (major == 10 && minor == 3) ? TG_OK : TG_ERR_ARCH;
        if (d.arch == TG_OK) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_splitk_scratch) != cudaSuccess || p == nullptr)
                return TG_ERR_CUDA;
            d.scratch = static_cast<float *>(p);
            if (tg::status_word_address(&d.status) != cudaSuccess) return TG_ERR_CUDA;
            if (g_encode == nullptr) {
                void *fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q) != cudaSuccess ||
                    q != cudaDriverEntryPointSuccess || fn == nullptr)
                    return TG_ERR_CUDA;
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
            }
        }
        d.init = true;
    }
    *out = &d;
    return d.arch;
}

tg_status encode(CUtensorMap *map, tg_dtype t, const void *ptr, int64_t rows, int64_t cols,
                 int64_t ld, int box_cols, int box_rows) {
    const int es = tgh::esize_of(t);
    const int row_bytes = box_cols * es;
    const CUtensorMapSwizzle sw = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : row_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_32B;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * es)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = t == TG_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                   : t == TG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = g_encode(map, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TG_OK : TG_ERR_CUDA;
}

}  // namespace

extern "C" tg_status tg_gemm_splitk_noalloc(int64_t M, int64_t N, int64_t K, const void *a,
                                            int64_t lda, const void *b, int64_t ldb, void *c,
                                            int64_t ldc, tg_dtype dtype_in, tg_dtype dtype_out,
                                            int32_t splits, void *stream) {
    if (splits < 1 || splits > 128) return TG_ERR_INVALID_VALUE;
    if (dtype_in != TG_F16 && dtype_in != TG_BF16) return TG_ERR_UNSUPPORTED;
    tg_options opt;
    std::memset(&opt, 0, sizeof(opt));
    opt.path = TG_PATH_TC;
    opt.splits = splits;
    // Host-only validation (the rules of tg_gemm_ex).
    tg_status st = tgh::validate(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, &opt);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    NoAllocDevice *dev = nullptr;
    st = setup_current_device(&dev);
    if (st != TG_OK) return st;
    st = tgh::operands_local({c, K > 0 ? a : nullptr, K > 0 ? b : nullptr});
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int eo = tgh::esize_of(dtype_out);
    if (K == 0)
        return cudaMemset2DAsync(c, ldc * eo, 0, N * eo, M, s) == cudaSuccess ? TG_OK : TG_ERR_CUDA;
    // The planner's choice for this device; K tiles per split, tile width and
    // the wait bound are all taken from it.
    tgh::Plan pl;
    tgh::make_plan(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, dev->sms, &opt, &pl);
    if (!pl.valid) return TG_ERR_UNSUPPORTED;
    const tg_plan &plan = pl.pub;
    // A and B are read in place: no packed copies (that would need more memory).
    if (plan.pack_a || plan.pack_b) return TG_ERR_UNSUPPORTED;
    if (plan.splits > 1 && static_cast<int64_t>(plan.splits) * M * N > kScratchFloats)
        return TG_ERR_UNSUPPORTED;   // partials exceed TG_NOALLOC_SCRATCH_BYTES

    const int in_kind = tgh::in_kind_of(dtype_in);
    const int mc = 1;   // single CTAs (TG_PATH_TC) never share A
    CUtensorMap tmA, tmB;
    if (encode(&tmA, dtype_in, a, M, K, lda, plan.block_k, tgh::kBlockM) != TG_OK ||
        encode(&tmB, dtype_in, b, K, N, ldb,
               tg::tc_b_swizzle_bytes(in_kind, plan.block_n, false) / 2, plan.block_k) != TG_OK)
        return TG_ERR_CUDA;
    // without a split (K too short to split) the kernel writes C itself, by
    // TMA stores when C allows them
    CUtensorMap tmC;
    std::memset(&tmC, 0, sizeof(tmC));
    const bool c_tma = plan.splits == 1 && plan.c_vector && (N * eo) % 16 == 0 &&
                       encode(&tmC, dtype_out, c, M, N, ldc, 64 / eo, 32) == TG_OK;
    tg::TcParams tp;
    std::memset(&tp, 0, sizeof(tp));
    tp.M = static_cast<int32_t>(M);
    tp.N = static_cast<int32_t>(N);
    tp.K = static_cast<int32_t>(K);
    tp.tiles_m = static_cast<int32_t>(pl.tiles_m);
    tp.tiles_n = static_cast<int32_t>(pl.tiles_n);
    tp.k_tiles = static_cast<int32_t>(pl.k_tiles);
    tp.k_tiles_per_split = static_cast<int32_t>(pl.k_per_split);
    tp.splits = plan.splits;
    tp.group_m = plan.group_m;
    tp.out_kind = dtype_out == TG_F16 ? tg::OUT_F16 : (dtype_out == TG_BF16 ? tg::OUT_BF16 : tg::OUT_F32);
    tp.c_vector = plan.c_vector;
    tp.mc = mc;
    tp.ldc = ldc;
    tp.c = c;
    tp.partial = plan.splits > 1 ? dev->scratch : nullptr;
    tp.status = dev->status;
    tp.timeout_ns = pl.timeout_ns;
    tp.batch = 1;
    tp.c_tma = c_tma ? 1 : 0;
    if (tg::launch_gemm_tc(in_kind, plan.block_n, false, mc, tmA, tmB, tmC, tp, plan.ctas, s) !=
        cudaSuccess)
        return TG_ERR_CUDA;
    if (plan.splits > 1 &&
        tg::launch_splitk_reduce(dev->scratch, plan.splits, M, N, c, ldc, tp.out_kind,
                                 plan.c_vector, s) != cudaSuccess)
        return TG_ERR_CUDA;
    return TG_OK;
}
