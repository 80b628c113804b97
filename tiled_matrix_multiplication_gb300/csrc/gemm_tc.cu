// gemm_tc.cu -- host side of the tensor-core GEMM kernel: the device status
// word, shared-memory opt-in, variant queries and the dispatch to the
// per-operand-type instantiations (gemm_tc_f16.cu, gemm_tc_tf32.cu,
// gemm_tc_fp8.cu).  The kernel itself is in gemm_tc_kernel.cuh.
#include "gemm_tc_kernel.cuh"

namespace tg {

__device__ int g_status_word[2];

cudaError_t status_word_address(int **out) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(out), g_status_word);
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel and device.
cudaError_t set_smem_once(const void *kern, int bytes) {
    static std::mutex mu;
    static const void *done[256][2];
    static int count = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < count; ++i)
        if (done[i][0] == kern && done[i][1] == reinterpret_cast<const void *>(static_cast<intptr_t>(dev)))
            return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && count < 256) {
        done[count][0] = kern;
        done[count][1] = reinterpret_cast<const void *>(static_cast<intptr_t>(dev));
        ++count;
    }
    return e;
}

bool tc_supported_block_n(int in_kind, int block_n, bool pair) {
    (void)in_kind;
    if (block_n == 512) return pair;
    return block_n == 128 || block_n == 192 || block_n == 224 || block_n == 256;
}

int tc_stages(int in_kind, int block_n, bool pair) {
    switch (in_kind) {
    case IN_F16:
        return pair ? stages_kind<IN_F16, true>(block_n) : stages_kind<IN_F16, false>(block_n);
    case IN_BF16:
        return pair ? stages_kind<IN_BF16, true>(block_n) : stages_kind<IN_BF16, false>(block_n);
    case IN_TF32:
        return pair ? stages_kind<IN_TF32, true>(block_n) : stages_kind<IN_TF32, false>(block_n);
    case IN_E4M3:
        return pair ? stages_kind<IN_E4M3, true>(block_n) : stages_kind<IN_E4M3, false>(block_n);
    case IN_E5M2:
        return pair ? stages_kind<IN_E5M2, true>(block_n) : stages_kind<IN_E5M2, false>(block_n);
    default: return 0;
    }
}

int tc_b_swizzle_bytes(int in_kind, int block_n, bool pair) {
    const int es = in_esize(in_kind);
    if (in_kind == IN_TF32) return 128;                       // 32-byte-atom swizzle
    const int mma_n = block_n > 256 ? 256 : block_n;          // N of one MMA
    const int cols = pair ? mma_n / 2 : mma_n;                // its B columns per CTA
    return ((cols * es) % 128 != 0 && (cols * es) % 64 == 0) ? 64 : 128;
}

bool tc_supported_mc(int block_n, int mc, bool pair) {
    if (mc == 1) return true;
    if (mc != 2) return false;
    return pair && (block_n == 192 || block_n == 224 || block_n == 256);
}

cudaError_t launch_gemm_tc(int in_kind, int block_n, bool pair, int mc, const CUtensorMap &tmA,
                           const CUtensorMap &tmB, const CUtensorMap &tmC, const TcParams &p,
                           int ctas, cudaStream_t stream) {
    if (!tc_supported_mc(block_n, mc, pair) || !tc_supported_block_n(in_kind, block_n, pair))
        return cudaErrorInvalidValue;
    switch (in_kind) {
    case IN_F16:
    case IN_BF16:
        return launch_gemm_tc_16bit(in_kind, block_n, pair, mc, tmA, tmB, tmC, p, ctas, stream);
    case IN_TF32:
        return launch_gemm_tc_tf32(block_n, pair, mc, tmA, tmB, tmC, p, ctas, stream);
    case IN_E4M3:
    case IN_E5M2:
        return launch_gemm_tc_fp8(in_kind, block_n, pair, mc, tmA, tmB, tmC, p, ctas, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tg
