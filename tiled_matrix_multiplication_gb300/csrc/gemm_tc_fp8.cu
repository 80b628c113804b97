// gemm_tc_fp8.cu -- the tensor-core GEMM kernel instantiated for 8-bit
// floating-point operands, E4M3 or E5M2 (kind::f8f6f4, FP32 accumulate).
#include "gemm_tc_kernel.cuh"

namespace tg {

cudaError_t launch_gemm_tc_fp8(int in_kind, int block_n, bool pair, int mc,
                               const CUtensorMap &tmA, const CUtensorMap &tmB,
                               const CUtensorMap &tmC, const TcParams &p, int ctas,
                               cudaStream_t stream) {
    if (in_kind == IN_E4M3)
        return launch_variant<IN_E4M3>(block_n, pair, mc, tmA, tmB, tmC, p, ctas, stream);
    if (in_kind == IN_E5M2)
        return launch_variant<IN_E5M2>(block_n, pair, mc, tmA, tmB, tmC, p, ctas, stream);
    return cudaErrorInvalidValue;
}

}  // namespace tg
