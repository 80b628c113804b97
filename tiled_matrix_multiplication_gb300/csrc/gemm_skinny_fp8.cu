// gemm_skinny_fp8.cu -- the small-M kernel (gemm_skinny_kernel.cuh) for 8-bit
// floating-point operands, E4M3 or E5M2 (kind::f8f6f4): 128 K elements per
// 128-byte row, one 128-column box of B^T per MMA.
#include "gemm_skinny_kernel.cuh"

namespace tg {

cudaError_t launch_gemm_skinny_fp8(int in_kind, int mp, int nt, const CUtensorMap &tmA,
                                   const CUtensorMap &tmB, const SkParams &p,
                                   cudaStream_t stream) {
    if (in_kind == IN_E4M3) return sk_launch_kind<IN_E4M3>(mp, nt, tmA, tmB, p, stream);
    if (in_kind == IN_E5M2) return sk_launch_kind<IN_E5M2>(mp, nt, tmA, tmB, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace tg
