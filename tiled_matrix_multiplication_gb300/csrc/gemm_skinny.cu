// gemm_skinny.cu -- the small-M kernel (gemm_skinny_kernel.cuh) for FP16 and
// BF16 operands, its planning queries, and the dispatch by operand type.
#include "gemm_skinny_kernel.cuh"

namespace tg {

int skinny_rows(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128)); }

bool skinny_supported(int mp, int nt) {
    return (nt == 128 || nt == 256 || nt == 512) && !(mp == 128 && nt == 512);
}

int skinny_stages(int mp, int nt, bool two) {
    switch (nt) {
    case 128: return two ? stages_nt<128, true>(mp) : stages_nt<128, false>(mp);
    case 256: return two ? 0 : stages_nt<256, false>(mp);
    case 512: return two ? 0 : stages_nt<512, false>(mp);
    default: return 0;
    }
}

cudaError_t launch_gemm_skinny(int in_kind, int mp, int nt, const CUtensorMap &tmA,
                               const CUtensorMap &tmB, const SkParams &p, cudaStream_t stream) {
    if (p.splits != 1 && p.splits != 2 && p.splits != 4 && p.splits != 8)
        return cudaErrorInvalidValue;
    switch (in_kind) {
    case IN_F16: return sk_launch_kind<IN_F16>(mp, nt, tmA, tmB, p, stream);
    case IN_BF16: return sk_launch_kind<IN_BF16>(mp, nt, tmA, tmB, p, stream);
    case IN_E4M3:
    case IN_E5M2: return launch_gemm_skinny_fp8(in_kind, mp, nt, tmA, tmB, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tg
