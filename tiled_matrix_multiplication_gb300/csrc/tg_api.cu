// tg_api.cu -- host side of the C ABI declared in include/tg_gemm.h: per-device
// state, TMA tensor maps, workspace and the launches of the GEMM entry points
// (argument rules and planning are in tg_plan.cu, the host-operand pipeline in
// tg_host.cu).
#include "tg_host_api.h"

namespace tgh {
namespace {

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

}  // namespace

static tg_status init_encoder() {
    if (g_encode) return TG_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return TG_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return TG_OK;
}

tg_status device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TG_ERR_CUDA;
        d.sms = sms;
        d.arch = (major == 10 && minor == 3) ? TG_OK : TG_ERR_ARCH;
        if (d.arch == TG_OK) {
            if (tg::status_word_address(&d.status) != cudaSuccess) return TG_ERR_CUDA;
            if (init_encoder() != TG_OK) return TG_ERR_CUDA;
            cudaMemPoolProps props;
            std::memset(&props, 0, sizeof(props));
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) return TG_ERR_CUDA;
            uint64_t keep = ~0ull;
            if (cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess)
                return TG_ERR_CUDA;
            d.pair_slots = tg::tc_max_clusters(2);
            d.quad_slots = tg::tc_max_clusters(4);
        }
        d.init = true;
    }
    *out = &d;
    return d.arch;
}

static CUtensorMapDataType tma_type(tg_dtype t) {
    if (is_fp8(t)) return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // bytes moved as they are
    return t == TG_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                       : (t == TG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

// Row-major [rows, cols] with pitch `ld` elements; boxes of box_cols x box_rows
// whose rows (box_cols * esize bytes = 128, 64 or 32) are swizzled at that
// size -- in 32-byte atoms for `atom32` (4-byte elements read N-major by the
// TF32 MMA); zero fill out of range.  With nb > 1 the map has a third
// dimension of nb matrices `stride` elements apart (boxes one matrix deep).
static tg_status encode_2d(CUtensorMap *map, tg_dtype t, const void *ptr, int64_t rows, int64_t cols,
                    int64_t ld, int box_cols, int box_rows, int64_t nb = 1, int64_t stride = 0,
                    bool atom32 = false) {
    const int row_bytes = box_cols * esize_of(t);
    const CUtensorMapSwizzle sw = atom32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B
                                : row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : row_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_32B;
    const cuuint32_t rank = nb > 1 ? 3 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(nb)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * esize_of(t)),
                                   static_cast<cuuint64_t>(stride * esize_of(t))};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows),
                               1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, tma_type(t), rank, const_cast<void *>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TG_OK : TG_ERR_CUDA;
}

// Operands must be device memory of the current device: the tile kernels read
// A through TMA loads multicast to the CTAs of a cluster of this GPU, and no
// kernel of the library is meant to read host memory or a peer GPU's memory
// over the interconnect.  Memory from cudaMalloc, a stream-ordered pool or a
// mapping backed by this device qualifies; host, managed and peer memory do
// not.  Null pointers (absent epilogue vectors) are skipped.
tg_status operands_local(std::initializer_list<const void *> ptrs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    for (const void *p : ptrs) {
        if (p == nullptr) continue;
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            (void)cudaGetLastError();   // not a pointer the runtime knows
            return TG_ERR_INVALID_VALUE;
        }
        if (at.type != cudaMemoryTypeDevice || at.device != dev) return TG_ERR_INVALID_VALUE;
    }
    return TG_OK;
}

static tg_status epilogue_local(const tg_epilogue *ep) {
    return ep ? operands_local({ep->residual, ep->scale, ep->bias}) : TG_OK;
}

tg_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return TG_OK;
    if (e == cudaErrorMemoryAllocation) return TG_ERR_OUT_OF_MEMORY;
    return TG_ERR_CUDA;
}

// Enqueues one validated product with M, N, K > 0 -- or, with bt.count > 1,
// that many products in one launch (16-bit operands that need no packing).
// A tensor map the driver rejects for a batch sets *map_failed before
// anything is enqueued, so the caller can run the products one by one.
tg_status enqueue(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                  int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in, tg_dtype dtype_out,
                  cudaStream_t s, const tg_options *opt, DeviceState *dev, const Batch &bt,
                  bool *map_failed, const tg::EpiParams *epi) {
    tg_status st = TG_OK;
    Plan pl;
    pl.stride_c = bt.sc;
    make_plan(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, dev->sms, opt, &pl,
              dev->pair_slots, dev->quad_slots, bt.count);
    if (!pl.valid) return TG_ERR_UNSUPPORTED;
    const tg_plan &p = pl.pub;
    const int ei = esize_of(dtype_in);
    const bool batched = bt.count > 1;
    // operands that differ per product get a rank-3 map; a shared one (stride 0) stays 2-D
    const int64_t nb_a = batched && bt.sa ? bt.count : 1;
    const int64_t nb_b = batched && bt.sb ? bt.count : 1;
    auto map_error = [&]() {
        if (batched && map_failed) *map_failed = true;
        return TG_ERR_CUDA;
    };

    uint8_t *ws = nullptr;
    if (p.workspace_bytes > 0) {
        cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), p.workspace_bytes,
                                                dev->pool, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    auto fail = [&](tg_status code) {
        if (ws) cudaFreeAsync(ws, s);
        return code;
    };
    const void *A = a;
    const void *B = b;
    if (p.pack_a) {
        A = ws + pl.off_a;
        st = cuda_status(p.pack_a == 3
                             ? tg::launch_split3_rows(a, lda, ws + pl.off_a, pl.lda_p, M, K, s)
                             : tg::launch_pack_rows(a, lda, ws + pl.off_a, pl.lda_p, M, K, ei, s));
        if (st != TG_OK) return fail(st);
    }
    if (p.pack_b) {
        B = ws + pl.off_b;
        st = cuda_status(
            p.pack_b == 3 ? tg::launch_split3_stack(b, ldb, ws + pl.off_b, pl.ldb_p, K, N, s)
                          : tg::launch_pack_rows(b, ldb, ws + pl.off_b, pl.ldb_p, K, N, ei, s));
        if (st != TG_OK) return fail(st);
    }
    const int64_t Ke = pl.k_eff;   // K of the kernel's operands
    CUtensorMap tmA, tmB;
    const int chunk = 128 / ei;
    if (p.path == TG_PATH_SKINNY) {
        if (encode_2d(&tmA, dtype_in, A, M, K, pl.lda_p, p.block_k, p.block_m, nb_a, bt.sa) != TG_OK ||
            encode_2d(&tmB, dtype_in, B, K, N, pl.ldb_p, chunk, p.block_k, nb_b, bt.sb) != TG_OK)
            return fail(map_error());
        tg::SkParams sp;
        std::memset(&sp, 0, sizeof(sp));
        sp.M = static_cast<int32_t>(M);
        sp.N = static_cast<int32_t>(N);
        sp.K = static_cast<int32_t>(K);
        sp.tiles_n = static_cast<int32_t>(pl.tiles_n);
        sp.k_tiles = static_cast<int32_t>(pl.k_tiles);
        sp.k_tiles_per_split = static_cast<int32_t>(pl.k_per_split);
        sp.splits = p.splits;
        sp.out_kind = out_kind_of(dtype_out);
        sp.ldc = ldc;
        sp.c = c;
        sp.status = dev->status;
        sp.timeout_ns = pl.timeout_ns;
        sp.two_per_sm = pl.skinny_two ? 1 : 0;
        sp.batch = static_cast<int32_t>(bt.count);
        sp.a_batched = nb_a > 1;
        sp.b_batched = nb_b > 1;
        sp.stride_c = bt.sc;
        sp.c_vector = p.c_vector;
        if (epi) sp.epi = *epi;
        st = cuda_status(
            tg::launch_gemm_skinny(in_kind_of(dtype_in), p.block_m, p.block_n, tmA, tmB, sp, s));
        if (st != TG_OK) return fail(st);
        if (ws && cudaFreeAsync(ws, s) != cudaSuccess) return TG_ERR_CUDA;
        return TG_OK;
    }
    const bool pair = p.path == TG_PATH_TC_PAIR;
    // B N-major in boxes of b_chunk columns x block_k rows (B' [3K, N] for 3xTF32)
    const int b_chunk = tg::tc_b_swizzle_bytes(in_kind_of(dtype_in), p.block_n, pair) / ei;
    const tg_status sb = encode_2d(&tmB, dtype_in, B, Ke, N, pl.ldb_p, b_chunk, p.block_k, nb_b,
                                   bt.sb, dtype_in == TG_F32);
    // with A multicast each CTA loads half of its 128 rows of A
    const int a_rows = p.multicast == 2 ? kBlockM / 2 : kBlockM;
    if (encode_2d(&tmA, dtype_in, A, M, Ke, pl.lda_p, p.block_k, a_rows, nb_a, bt.sa) != TG_OK ||
        sb != TG_OK)
        return fail(map_error());
    // C through TMA stores: [N, M] (x batch) in boxes of 64 bytes x 32 rows,
    // when C's base, pitch and batch stride are 16-byte multiples, the kernel
    // writes C itself (no split-K partials) and each row of C ends on a
    // 16-byte boundary: a TMA store leaves out what lies beyond the tensor's
    // last column only in whole 16-byte pieces (measured on GB300: with N = 300
    // BF16 columns it wrote columns 300..303 of a padded C)
    CUtensorMap tmC;
    std::memset(&tmC, 0, sizeof(tmC));
    const int eo = esize_of(dtype_out);
    bool c_tma = p.c_vector && p.splits == 1 && (N * eo) % 16 == 0;
    if (c_tma) {
        const int64_t nb_c = batched ? bt.count : 1;
        c_tma = encode_2d(&tmC, dtype_out, c, M, N, ldc, 64 / eo, 32, nb_c, bt.sc) == TG_OK;
    }

    tg::TcParams tp;
    std::memset(&tp, 0, sizeof(tp));
    tp.M = static_cast<int32_t>(M);
    tp.N = static_cast<int32_t>(N);
    tp.K = static_cast<int32_t>(Ke);
    tp.tiles_m = static_cast<int32_t>(pl.tiles_m);
    tp.tiles_n = static_cast<int32_t>(pl.tiles_n);
    tp.k_tiles = static_cast<int32_t>(pl.k_tiles);
    tp.k_tiles_per_split = static_cast<int32_t>(pl.k_per_split);
    tp.splits = p.splits;
    tp.group_m = p.group_m;
    tp.out_kind = out_kind_of(dtype_out);
    tp.c_vector = p.c_vector;
    tp.mc = std::max(p.multicast, 1);
    tp.ldc = ldc;
    tp.c = c;
    tp.partial = p.splits > 1 ? reinterpret_cast<float *>(ws + pl.off_p) : nullptr;
    tp.status = dev->status;
    tp.timeout_ns = pl.timeout_ns;
    tp.batch = static_cast<int32_t>(bt.count);
    tp.a_batched = nb_a > 1;
    tp.b_batched = nb_b > 1;
    tp.stride_c = bt.sc;
    tp.c_tma = c_tma ? 1 : 0;
    // with a K split the epilogue runs where the partials are summed
    if (epi && p.splits == 1) tp.epi = *epi;
    st = cuda_status(tg::launch_gemm_tc(in_kind_of(dtype_in), p.block_n, pair,
                                        std::max(p.multicast, 1), tmA, tmB, tmC, tp, p.ctas, s));
    if (st != TG_OK) return fail(st);
    if (p.splits > 1) {
        st = cuda_status(tg::launch_splitk_reduce(tp.partial, p.splits, M, N, c, ldc,
                                                  tp.out_kind, p.c_vector, s, epi));
        if (st != TG_OK) return fail(st);
    }
    if (ws) {
        if (cudaFreeAsync(ws, s) != cudaSuccess) return TG_ERR_CUDA;
    }
    return TG_OK;
}

}  // namespace tgh

using namespace tgh;

extern "C" {

int32_t tg_abi_version(void) { return TG_ABI_VERSION; }

const char *tg_status_string(tg_status s) {
    switch (s) {
    case TG_OK: return "TG_OK";
    case TG_ERR_INVALID_VALUE: return "TG_ERR_INVALID_VALUE";
    case TG_ERR_UNSUPPORTED: return "TG_ERR_UNSUPPORTED";
    case TG_ERR_OUT_OF_MEMORY: return "TG_ERR_OUT_OF_MEMORY";
    case TG_ERR_CUDA: return "TG_ERR_CUDA";
    case TG_ERR_ARCH: return "TG_ERR_ARCH";
    case TG_ERR_TIMEOUT: return "TG_ERR_TIMEOUT";
    case TG_ERR_NOT_IMPLEMENTED: return "TG_ERR_NOT_IMPLEMENTED";
    case TG_ERR_BOUNDS: return "TG_ERR_BOUNDS";
    default: return "TG_ERR_UNKNOWN";
    }
}

tg_status tg_gemm_ex(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                     int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in, tg_dtype dtype_out,
                     void *stream, const tg_options *opt) {
    tg_status st = validate(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TG_OK) return st;
    st = operands_local({c, K > 0 ? a : nullptr, K > 0 ? b : nullptr});
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int eo = esize_of(dtype_out);
    if (K == 0)
        return cuda_status(cudaMemset2DAsync(c, ldc * eo, 0, N * eo, M, s));
    return enqueue(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, s, opt, dev, Batch{},
                   nullptr);
}

tg_status tg_gemm_fused(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda,
                        const void *b, int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in,
                        tg_dtype dtype_out, const tg_epilogue *epilogue, void *stream,
                        const tg_options *opt) {
    tg_status st = validate(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    tg::EpiParams e;
    st = validate_epilogue(M, N, c, ldc, dtype_out, epilogue, &e);
    if (st != TG_OK) return st;
    if (epilogue == nullptr)
        return tg_gemm_ex(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream, opt);
    if (M == 0 || N == 0) return TG_OK;
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TG_OK) return st;
    st = operands_local({c, K > 0 ? a : nullptr, K > 0 ? b : nullptr});
    if (st == TG_OK) st = epilogue_local(epilogue);
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)   // the epilogue of the empty sum
        return cuda_status(tg::launch_splitk_reduce(nullptr, 0, M, N, c, ldc,
                                                    out_kind_of(dtype_out), 0, s, &e));
    return enqueue(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, s, opt, dev, Batch{},
                   nullptr, &e);
}

tg_status tg_gemm(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                  int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in, tg_dtype dtype_out,
                  void *stream) {
    return tg_gemm_ex(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream, nullptr);
}

tg_status tg_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void *a,
                                  int64_t lda, int64_t stride_a, const void *b, int64_t ldb,
                                  int64_t stride_b, void *c, int64_t ldc, int64_t stride_c,
                                  tg_dtype dtype_in, tg_dtype dtype_out, void *stream,
                                  const tg_options *opt) {
    tg_status st = validate_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, c, ldc,
                                    stride_c, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    if (batch == 0 || M == 0 || N == 0) return TG_OK;
    if (batch == 1)
        return tg_gemm_ex(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream, opt);
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TG_OK) return st;
    st = operands_local({c, K > 0 ? a : nullptr, K > 0 ? b : nullptr});
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int ei = esize_of(dtype_in), eo = esize_of(dtype_out);
    auto c_of = [&](int64_t z) { return static_cast<uint8_t *>(c) + z * stride_c * eo; };
    if (K == 0) {
        for (int64_t z = 0; z < batch; ++z) {
            st = cuda_status(cudaMemset2DAsync(c_of(z), ldc * eo, 0, N * eo, M, s));
            if (st != TG_OK) return st;
        }
        return TG_OK;
    }
    if (batch_in_one_launch(dtype_in, a, lda, stride_a, b, ldb, stride_b)) {
        bool map_failed = false;
        st = enqueue(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, s, opt, dev,
                     Batch{batch, stride_a, stride_b, stride_c}, &map_failed);
        if (!map_failed) return st;
    }
    // one call per product, in order of z
    for (int64_t z = 0; z < batch; ++z) {
        st = tg_gemm_ex(M, N, K, static_cast<const uint8_t *>(a) + z * stride_a * ei, lda,
                        static_cast<const uint8_t *>(b) + z * stride_b * ei, ldb, c_of(z), ldc,
                        dtype_in, dtype_out, stream, opt);
        if (st != TG_OK) return st;
    }
    return TG_OK;
}

tg_status tg_gemm_strided_batched_fused(int64_t batch, int64_t M, int64_t N, int64_t K,
                                        const void *a, int64_t lda, int64_t stride_a,
                                        const void *b, int64_t ldb, int64_t stride_b, void *c,
                                        int64_t ldc, int64_t stride_c, tg_dtype dtype_in,
                                        tg_dtype dtype_out, const tg_epilogue *epilogue,
                                        int64_t stride_r, void *stream, const tg_options *opt) {
    tg_status st = validate_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, c, ldc,
                                    stride_c, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    if (epilogue == nullptr && stride_r != 0) return TG_ERR_INVALID_VALUE;
    tg::EpiParams e;
    st = validate_epilogue(M, N, c, ldc, dtype_out, epilogue, &e, batch, stride_c, stride_r);
    if (st != TG_OK) return st;
    if (epilogue == nullptr)
        return tg_gemm_strided_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, c, ldc,
                                       stride_c, dtype_in, dtype_out, stream, opt);
    if (batch == 0 || M == 0 || N == 0) return TG_OK;
    const int ei = esize_of(dtype_in), eo = esize_of(dtype_out);
    {
        DeviceState *dev = nullptr;
        st = device_state(&dev);
        if (st != TG_OK) return st;
        st = operands_local({c, K > 0 ? a : nullptr, K > 0 ? b : nullptr});
        if (st == TG_OK) st = epilogue_local(epilogue);
        if (st != TG_OK) return st;
    }
    if (K > 0 && batch > 1 && batch_in_one_launch(dtype_in, a, lda, stride_a, b, ldb, stride_b)) {
        DeviceState *dev = nullptr;
        st = device_state(&dev);
        if (st != TG_OK) return st;
        bool map_failed = false;
        st = enqueue(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out,
                     static_cast<cudaStream_t>(stream), opt, dev,
                     Batch{batch, stride_a, stride_b, stride_c}, &map_failed, &e);
        if (!map_failed) return st;
    }
    // one fused call per product, in order of z, each with its own residual
    tg_epilogue one = *epilogue;
    for (int64_t z = 0; z < batch; ++z) {
        if (epilogue->residual)
            one.residual = static_cast<const uint8_t *>(epilogue->residual) + z * stride_r * eo;
        st = tg_gemm_fused(M, N, K, static_cast<const uint8_t *>(a) + z * stride_a * ei, lda,
                           static_cast<const uint8_t *>(b) + z * stride_b * ei, ldb,
                           static_cast<uint8_t *>(c) + z * stride_c * eo, ldc, dtype_in,
                           dtype_out, &one, stream, opt);
        if (st != TG_OK) return st;
    }
    return TG_OK;
}

tg_status tg_selftest_timeout(int32_t timeout_ms, void *stream) {
    if (timeout_ms < 1 || timeout_ms > 10000) return TG_ERR_INVALID_VALUE;
    DeviceState *dev = nullptr;
    const tg_status st = device_state(&dev);
    if (st != TG_OK) return st;
    return cuda_status(tg::launch_selftest_timeout(
        dev->status, static_cast<uint64_t>(timeout_ms) * 1000000ull, static_cast<cudaStream_t>(stream)));
}

int32_t tg_checked_build(void) {
#ifdef TG_CHECKED
    return 1;
#else
    return 0;
#endif
}

tg_status tg_selftest_bounds(int32_t index, void *stream) {
    if (index < 0 || index > 1024) return TG_ERR_INVALID_VALUE;
#ifdef TG_CHECKED
    DeviceState *dev = nullptr;
    const tg_status st = device_state(&dev);
    if (st != TG_OK) return st;
    return cuda_status(tg::launch_selftest_bounds(dev->status, index,
                                                  static_cast<cudaStream_t>(stream)));
#else
    (void)stream;
    return TG_ERR_NOT_IMPLEMENTED;
#endif
}

tg_status tg_last_device_error(void *stream) {
    DeviceState *dev = nullptr;
    const tg_status st = device_state(&dev);
    if (st != TG_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TG_ERR_CUDA;
    int words[2] = {0, 0};
    if (cudaMemcpy(words, dev->status, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TG_ERR_CUDA;
    if (words[0] != 0) {
        const int zero[2] = {0, 0};
        if (cudaMemcpy(dev->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return TG_ERR_CUDA;
        return static_cast<tg_status>(words[0]);
    }
    return TG_OK;
}

}  // extern "C"
