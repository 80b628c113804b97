// tg_host.cu -- tg_gemm_host: a product whose operands and result live in
// host memory, staged through the library's pool with the copies pipelined
// against the multiply.
#include "tg_host_api.h"

namespace tgh {
namespace {

// Copy streams and events of the host-operand pipeline (tg_gemm_host), made
// once per device.  One call at a time uses them (the mutex), so an event is
// never re-recorded before the waits on it have been enqueued.
constexpr int kHostPanels = 16;
struct HostPipe {
    std::mutex mu;
    bool init = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, h2d_done = nullptr, done = nullptr;
    cudaEvent_t a_done[kHostPanels] = {}, c_done[kHostPanels] = {};
};
HostPipe g_pipe[kMaxDevices];

// Rows per panel of the host-operand pipeline: at least 1024 (four rows of
// pair tiles, so a panel still fills the GPU without a K split), at most
// kHostPanels panels.  Measured on GB300 at 4096^3 (host link about 200 GB/s
// each way): 4 panels of 1024 rows beat 1, 2, 8 and 16 panels; at 8192^3, 8
// panels of 1024 rows.
int64_t host_panel_rows(int64_t M) {
    return std::max<int64_t>(1024, round_up(cdiv(M, kHostPanels), 256));
}

tg_status host_pipe(int dev, HostPipe **out) {
    HostPipe &hp = g_pipe[dev];
    if (!hp.init) {
        if (cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) != cudaSuccess)
            return TG_ERR_CUDA;
        cudaEvent_t *evs[] = {&hp.start, &hp.h2d_done, &hp.done};
        for (cudaEvent_t *e : evs)
            if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return TG_ERR_CUDA;
        for (int i = 0; i < kHostPanels; ++i)
            if (cudaEventCreateWithFlags(&hp.a_done[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.c_done[i], cudaEventDisableTiming) != cudaSuccess)
                return TG_ERR_CUDA;
        hp.init = true;
    }
    *out = &hp;
    return TG_OK;
}

}  // namespace
}  // namespace tgh

using namespace tgh;

extern "C" {

tg_status tg_gemm_host(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda,
                       const void *b, int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in,
                       tg_dtype dtype_out, void *stream, const tg_options *opt) {
    tg_status st = validate(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TG_OK) return st;
    int dev_id = 0;
    if (cudaGetDevice(&dev_id) != cudaSuccess) return TG_ERR_CUDA;
    HostPipe *hp = nullptr;
    std::lock_guard<std::mutex> lk(g_pipe[dev_id].mu);
    if ((st = host_pipe(dev_id, &hp)) != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int ei = esize_of(dtype_in), eo = esize_of(dtype_out);
    // device copies with 16-byte row pitches (read in place by the kernels)
    const int64_t lda_d = round_up(std::max<int64_t>(K, 1), 16 / ei);
    const int64_t ldb_d = round_up(N, 16 / ei);
    const int64_t ldc_d = round_up(N, 16 / eo);
    const int64_t off_b = round_up(M * lda_d * ei, 256);
    const int64_t off_c = off_b + round_up(K * ldb_d * ei, 256);
    const int64_t bytes = off_c + round_up(M * ldc_d * eo, 256);
    uint8_t *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), bytes, dev->pool, s);
    if (e != cudaSuccess) return cuda_status(e);
    uint8_t *A_d = ws, *B_d = ws + off_b, *C_d = ws + off_c;
    const uint8_t *ah = static_cast<const uint8_t *>(a);
    const uint8_t *bh = static_cast<const uint8_t *>(b);
    uint8_t *ch = static_cast<uint8_t *>(c);
    auto ok = [](cudaError_t r) { return r == cudaSuccess; };
    bool good = ok(cudaEventRecord(hp->start, s));
    const int64_t rows = host_panel_rows(M);
    const int panels = static_cast<int>(cdiv(M, rows));
    if (K > 0) {
        // one copy stream in order: all of B, then the panels of A (several
        // copy streams measured no faster: the host link is the limit)
        good = ok(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) &&
               ok(cudaMemcpy2DAsync(B_d, ldb_d * ei, bh, ldb * ei, N * ei, K,
                                    cudaMemcpyHostToDevice, hp->h2d));
        for (int p = 0; p < panels && good; ++p) {
            const int64_t r0 = p * rows, rn = std::min(M, r0 + rows) - r0;
            good = ok(cudaMemcpy2DAsync(A_d + r0 * lda_d * ei, lda_d * ei, ah + r0 * lda * ei,
                                        lda * ei, K * ei, rn, cudaMemcpyHostToDevice, hp->h2d)) &&
                   ok(cudaEventRecord(hp->a_done[p], hp->h2d));
        }
    }
    if (good) good = ok(cudaStreamWaitEvent(hp->d2h, hp->start, 0));
    for (int p = 0; p < panels && good; ++p) {
        const int64_t r0 = p * rows, rn = std::min(M, r0 + rows) - r0;
        uint8_t *cp = C_d + r0 * ldc_d * eo;
        if (K == 0) {
            good = ok(cudaMemset2DAsync(cp, ldc_d * eo, 0, N * eo, rn, s));
        } else {
            good = ok(cudaStreamWaitEvent(s, hp->a_done[p], 0));
            if (good) {
                st = enqueue(rn, N, K, A_d + r0 * lda_d * ei, lda_d, B_d, ldb_d, cp, ldc_d,
                             dtype_in, dtype_out, s, opt, dev, Batch{}, nullptr);
                good = st == TG_OK;
            }
        }
        if (good)
            good = ok(cudaEventRecord(hp->c_done[p], s)) &&
                   ok(cudaStreamWaitEvent(hp->d2h, hp->c_done[p], 0)) &&
                   ok(cudaMemcpy2DAsync(ch + r0 * ldc * eo, ldc * eo, cp, ldc_d * eo, N * eo, rn,
                                        cudaMemcpyDeviceToHost, hp->d2h));
    }
    // the caller's stream resumes after every copy of the call (also after a
    // failure part way); then the staging memory goes back to the pool
    const bool joined = ok(cudaEventRecord(hp->done, hp->d2h)) &&
                        ok(cudaStreamWaitEvent(s, hp->done, 0)) &&
                        ok(cudaEventRecord(hp->h2d_done, hp->h2d)) &&
                        ok(cudaStreamWaitEvent(s, hp->h2d_done, 0));
    if (!joined) return TG_ERR_CUDA;   // never free what copies may still use
    if (!ok(cudaFreeAsync(ws, s))) return TG_ERR_CUDA;
    if (!good) return st != TG_OK ? st : TG_ERR_CUDA;
    return TG_OK;
}

}  // extern "C"
