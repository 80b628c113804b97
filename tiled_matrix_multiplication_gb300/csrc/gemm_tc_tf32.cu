// gemm_tc_tf32.cu -- the tensor-core GEMM kernel instantiated for FP32
// operands contracted at TF32 (kind::tf32, B given K-major).
#include "gemm_tc_kernel.cuh"

namespace tg {

cudaError_t launch_gemm_tc_tf32(int block_n, bool pair, int mc, const CUtensorMap &tmA,
                                const CUtensorMap &tmB, const CUtensorMap &tmC,
                                const TcParams &p, int ctas, cudaStream_t stream) {
    return launch_variant<IN_TF32>(block_n, pair, mc, tmA, tmB, tmC, p, ctas, stream);
}

}  // namespace tg
