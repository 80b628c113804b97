// gemm_tc_f16.cu -- the tensor-core GEMM kernel instantiated for FP16 and
// BF16 operands (kind::f16), and the resident-cluster query, which measures
// the FP16 pair kernel (every variant takes one CTA per SM).
#include "gemm_tc_kernel.cuh"

namespace tg {

cudaError_t launch_gemm_tc_16bit(int in_kind, int block_n, bool pair, int mc,
                                 const CUtensorMap &tmA, const CUtensorMap &tmB,
                                 const CUtensorMap &tmC, const TcParams &p, int ctas,
                                 cudaStream_t stream) {
    if (in_kind == IN_F16)
        return launch_variant<IN_F16>(block_n, pair, mc, tmA, tmB, tmC, p, ctas, stream);
    if (in_kind == IN_BF16)
        return launch_variant<IN_BF16>(block_n, pair, mc, tmA, tmB, tmC, p, ctas, stream);
    return cudaErrorInvalidValue;
}

int tc_max_clusters(int cluster_size) {
    // Clusters of 2 or 4 CTAs of the widest-stage kernel that fit at once
    // (every variant of the kernel takes one CTA per SM, so the count is the
    // same for all of them).
    static std::mutex mu;
    static int cache[64][2];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int slot = cluster_size == 4 ? 1 : 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev][slot] == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(cluster_size, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        int n = 0;
        if (cluster_size == 4) {
            using Cfg = TcCfg<IN_F16, 256, true, 2>;
            auto kern = gemm_tc_kernel<IN_F16, 256, true, 2>;
            cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
            if (set_smem_once(reinterpret_cast<const void *>(kern), Cfg::SMEM_BYTES) != cudaSuccess ||
                cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess)
                return 0;
        } else {
            using Cfg = TcCfg<IN_F16, 256, true, 1>;
            auto kern = gemm_tc_kernel<IN_F16, 256, true, 1>;
            cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
            if (set_smem_once(reinterpret_cast<const void *>(kern), Cfg::SMEM_BYTES) != cudaSuccess ||
                cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess)
                return 0;
        }
        cache[dev][slot] = n;
    }
    return cache[dev][slot];
}

}  // namespace tg
