// gemm_skinny_kernel.cuh -- tcgen05 GEMM for small M (decode-like shapes),
// HBM-bound: the kernel template and its launchers, instantiated per operand
// type by gemm_skinny.cu (FP16, BF16) and gemm_skinny_fp8.cu (E4M3, E5M2).
//
// "Fast matrix multiplication" (ch. 12), section "Decode is a different
// problem: GEMV": with a handful of rows there is almost nothing to reuse, so
// the kernel's job is to stream B -- the large operand -- at full bandwidth,
// with coalesced wide reads and enough parallelism.
//
// The product is computed transposed, C^T = B^T A^T, so that the MMA's
// 128-row dimension runs over 128 output COLUMNS n and its N dimension over
// the few output rows m (M rounded up to MP = 16, 32, 64 or 128):
//   * MMA operand A = a B^T tile [128 n x BK k] (BK = 128 bytes of K: 64
//     16-bit or 128 FP8 elements), read N-major straight from row-major B
//     (two 64-column TMA boxes, or one 128-column box for FP8);
//   * MMA operand B = an A^T tile [BK k x MP m], read K-major from row-major A
//     (one TMA box of MP rows);
//   * the FP32 accumulator is 128 TMEM lanes (n) x MP columns (m).
// A CTA owns NT = 128, 256 or 512 consecutive columns (NT/128 MMAs per k step,
// each into its own accumulator), so each row of B is read in contiguous runs
// of NT elements and A is re-read once per NT columns.  Almost all of each
// shared-memory stage is B.
//
// Work split: one CTA per (NT-column tile, K range).  The S CTAs that share a
// column tile form a thread-block cluster (S = 1, 2, 4 or 8, cluster rank =
// K range).  After its main loop each CTA parks its FP32 partial tile in its
// own shared memory; after a cluster barrier, CTA r sums columns
// [r*NT/S, (r+1)*NT/S) of the tile over all S partials, read in rank order
// from the peers' shared memory (distributed shared memory), rounds once and
// writes C.  No partials go to global memory and no second kernel runs; the
// sum order is fixed, so results do not depend on timing.
//
// Roles: warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2..5 = TMEM -> shared epilogue; all six warps then do the cluster
// reduction.  Every mbarrier wait is bounded (status word + abort flag, as in
// gemm_tc.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tg_epilogue.cuh"
#include "tg_internal.h"
#include "tg_kernel_common.cuh"
#include "tg_ptx.cuh"

namespace tg {
namespace {

constexpr int kThreads = 192;
constexpr int kSmemBudget = 232448 - 1024 - 256;
constexpr int kSubN = 128;    // output columns per MMA (the MMA's M)

// TWO: a half-size ring so that two CTAs share an SM (twice the CTAs, and
// twice the independent TMA streams, for the same shared memory).
template <int IN_KIND, int MP, int NT, bool TWO>
struct SkCfg {
    static constexpr int ESIZE = in_esize(IN_KIND);   // 2 (FP16, BF16) or 1 (FP8)
    static constexpr int BK = 128 / ESIZE;        // 128 bytes of K per row
    static constexpr int UMMA_K = 32 / ESIZE;     // K of one MMA (32 bytes)
    static constexpr int CHUNK_N = 128 / ESIZE;   // n per 128-byte B row
    static constexpr int BOXES_PER_MMA = kSubN / CHUNK_N;     // B^T boxes per 128 columns
    static constexpr int KIND = ESIZE == 1 ? 2 : 0;           // kind::f8f6f4 / kind::f16
    static constexpr uint32_t FMT = (IN_KIND == IN_BF16 || IN_KIND == IN_E5M2) ? 1u : 0u;
    static constexpr int SUB = NT / kSubN;        // MMAs (accumulators) per k step
    static constexpr int BT_BOX = BK * 128;       // one CHUNK_N-column box: BK rows of 128 B
    static constexpr int BT_STAGE = (NT / CHUNK_N) * BT_BOX;   // NT columns of B
    static constexpr int AT_STAGE = MP * 128;     // MP rows of A
    static constexpr int STAGE_BYTES = BT_STAGE + AT_STAGE;
    static constexpr int BUDGET = TWO ? 112 * 1024 : kSmemBudget;
    static constexpr int STAGES = BUDGET / STAGE_BYTES > 12 ? 12 : BUDGET / STAGE_BYTES;
    static constexpr int PARTIAL_BYTES = NT * MP * 4;   // FP32 partial tile, [m][n]
    static constexpr int ACC_COLS = MP < 32 ? 32 : MP;  // TMEM columns per accumulator
    static constexpr int TMEM_COLS = SUB * ACC_COLS;
    static constexpr int NUM_BARS = 2 * STAGES + 1;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;
    // A operand (B^T) N-major, B operand (A^T) K-major; M = 128, N = MP.
    static constexpr uint32_t IDESC =
        make_idesc(FMT, 1u, 0u, kSubN, MP);
    static_assert(STAGE_BYTES % 1024 == 0, "stages keep 1024-byte swizzle alignment");
    static_assert(PARTIAL_BYTES <= STAGES * STAGE_BYTES, "partial tile reuses the ring");
    static_assert(MP % 16 == 0 && MP >= 16 && MP <= 128, "MMA N");
    static_assert(NT % kSubN == 0 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "accumulators fit one power-of-two TMEM allocation");
    static_assert(STAGES >= 2, "at least a double-buffered ring");
};

__device__ __forceinline__ void sk_store(const SkParams &p, int m, int n, float v) {
    const int64_t off = static_cast<int64_t>(blockIdx.y) * p.stride_c +   // batch
                        static_cast<int64_t>(m) * p.ldc + n;
    if (p.epi.on) v = epi_one(p.epi, p.out_kind, m, n, v, static_cast<int>(blockIdx.y));
    if (p.out_kind == OUT_F32)
        static_cast<float *>(p.c)[off] = v;
    else if (p.out_kind == OUT_F16)
        static_cast<__half *>(p.c)[off] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16 *>(p.c)[off] = __float2bfloat16_rn(v);
}

template <int IN_KIND, int MP, int NT, bool TWO>
__global__ void __launch_bounds__(kThreads, TWO ? 2 : 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const SkParams p) {
    using Cfg = SkCfg<IN_KIND, MP, NT, TWO>;
    constexpr int S = Cfg::STAGES;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sBt = base;                           // S x BT_STAGE
    const uint32_t sAt = base + S * Cfg::BT_STAGE;       // S x AT_STAGE
    const uint32_t bars = sAt + S * Cfg::AT_STAGE;
    uint8_t *gbars = gbase + (bars - base);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    const uint32_t tfull_bar = bars + 8u * (2 * S);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbars + 8 * Cfg::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *partial = reinterpret_cast<float *>(gbase);  // after the main loop: [MP][NT]
    __shared__ int never_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Cluster = `share` adjacent column tiles x `splits` K ranges; cluster rank
    // jn * splits + split.  With share = 2 the two CTAs of a K range (one per
    // column tile) each load half of the A^T rows and multicast them to both.
    const int share = p.a_share > 1 ? 2 : 1;
    const int csize = static_cast<int>(cluster_num_ctas());     // splits * share
    const int splits = csize / share;                            // == p.splits
    const int crank = static_cast<int>(cluster_cta_rank());
    const int split = crank % splits;
    const int jn = crank / splits;
    const int tn = (static_cast<int>(blockIdx.x) / csize) * share + jn;
    const uint16_t share_mask =
        static_cast<uint16_t>((1u << split) | (1u << (splits + split)));   // share == 2
    const int kt0 = split * p.k_tiles_per_split;
    const int kt1 = min(kt0 + p.k_tiles_per_split, p.k_tiles);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), share);   // one MMA commit per CTA reading the stage's A^T
        }
        mbar_init(tfull_bar, 1);
        *abort_flag = 0;
        never_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_addr(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (share > 1) cluster_sync_all();   // the partner's barriers exist before any multicast
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Prologue done: let the next kernel's prologue start, then wait for the
    // previous kernel's writes before the first global-memory access.
    if (threadIdx.x == 0) grid_launch_dependents();
    grid_dependency_wait();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int kt = kt0; kt < kt1; ++kt) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full_bar(stage), Cfg::STAGE_BYTES);
                const uint32_t fb = full_bar(stage);
                const int z = static_cast<int>(blockIdx.y);   // batch
                if (share > 1) {
                    // rows [jn*MP/2, (jn+1)*MP/2) of A^T, to this CTA and its partner
                    const uint32_t dst = sAt + stage * Cfg::AT_STAGE + jn * (Cfg::AT_STAGE / 2);
                    if (p.a_batched)
                        tma_load_3d_mc(dst, &tmA, fb, kt * Cfg::BK, jn * (MP / 2), z, share_mask);
                    else
                        tma_load_2d_mc(dst, &tmA, fb, kt * Cfg::BK, jn * (MP / 2), share_mask);
                } else if (p.a_batched) {
                    tma_load_3d(sAt + stage * Cfg::AT_STAGE, &tmA, fb, kt * Cfg::BK, 0, z);
                } else {
                    tma_load_2d(sAt + stage * Cfg::AT_STAGE, &tmA, fb, kt * Cfg::BK, 0);
                }
#pragma unroll
                for (int j = 0; j < NT / Cfg::CHUNK_N; ++j) {
                    const uint32_t dst = sBt + stage * Cfg::BT_STAGE + j * Cfg::BT_BOX;
                    if (p.b_batched)
                        tma_load_3d(dst, &tmB, fb, tn * NT + j * Cfg::CHUNK_N, kt * Cfg::BK, z);
                    else
                        tma_load_2d(dst, &tmB, fb, tn * NT + j * Cfg::CHUNK_N, kt * Cfg::BK);
                }
                ++issued;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                record_failure(p.status, 6, (ROLE_PRODUCER << 16) | stage);
                *abort_flag = 1;
            }
            const int64_t first = issued > S ? issued - S : 0;
            for (int64_t i = first; i < issued; ++i) {
                if (!mbar_wait(full_bar(static_cast<int>(i % S)),
                               static_cast<uint32_t>((i / S) & 1), p.timeout_ns, &never_abort)) {
                    record_failure(p.status, 6, (ROLE_DRAIN << 16) | 1);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kt = kt0; kt < kt1; ++kt) {
                if (!mbar_wait(full_bar(stage), phase, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t bt0 = sBt + stage * Cfg::BT_STAGE;
                const uint32_t at0 = sAt + stage * Cfg::AT_STAGE;
#pragma unroll
                for (int kk = 0; kk < Cfg::BK / Cfg::UMMA_K; ++kk) {
                    const uint64_t bd = smem_desc_sw128(at0 + kk * 32, 16, 1024);
#pragma unroll
                    for (int j = 0; j < Cfg::SUB; ++j) {
                        // columns [j*128, j*128+128): boxes BOXES_PER_MMA*j .. of the stage
                        const uint64_t ad = smem_desc_sw128(
                            bt0 + j * Cfg::BOXES_PER_MMA * Cfg::BT_BOX + kk * Cfg::UMMA_K * 128,
                            Cfg::BT_BOX, 1024);
                        umma_ss<Cfg::KIND, 1>(tmem_base + j * Cfg::ACC_COLS, ad, bd, Cfg::IDESC,
                                              (kt > kt0 || kk > 0) ? 1u : 0u);
                    }
                }
                if (share > 1)
                    umma_commit_mc(empty_bar(stage), share_mask);   // both CTAs filled the A^T
                else
                    umma_commit(empty_bar(stage));
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                record_failure(p.status, 6, (ROLE_MMA << 16) | stage);
                *abort_flag = 1;
            }
            // Accumulator complete; waiting for it also drains every issued MMA
            // before tensor memory is released.
            umma_commit(tfull_bar);
            if (!mbar_wait(tfull_bar, 0, p.timeout_ns, &never_abort))
                record_failure(p.status, 6, (ROLE_DRAIN << 16) | 2);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------- epilogue: TMEM -> smem
        // Thread (quad, lane) owns column n = quad*32 + lane of the tile.
        const int quad = warp & 3;
        const bool got = mbar_wait(tfull_bar, 0, p.timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) record_failure(p.status, 6, (ROLE_EPILOGUE << 16) | quad);
            *abort_flag = 1;
        } else {
            tc_fence_after_sync();
#pragma unroll 1
            for (int j = 0; j < Cfg::SUB; ++j) {
                const int nl = j * kSubN + quad * 32 + lane;   // column within the tile
                const int n = tn * NT + nl;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                       j * Cfg::ACC_COLS;
                if constexpr (MP == 16) {
                    uint32_t r[16];
                    tmem_load_16cols_sync(taddr, r);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        if (splits > 1)
                            partial[q * NT + nl] = __uint_as_float(r[q]);
                        else if (q < p.M && n < p.N)
                            sk_store(p, q, n, __uint_as_float(r[q]));
                    }
                } else {
#pragma unroll 1
                    for (int c0 = 0; c0 < MP; c0 += 32) {
                        uint32_t r[32];
                        tmem_load_32cols_sync(taddr + c0, r);
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            if (splits > 1)
                                partial[(c0 + q) * NT + nl] = __uint_as_float(r[q]);
                            else if (c0 + q < p.M && n < p.N)
                                sk_store(p, c0 + q, n, __uint_as_float(r[q]));
                        }
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (splits > 1) {
        // --------------------------- cluster reduction over distributed smem
        cluster_sync_all();                       // every CTA's partial is in place
        const int cols = NT / splits;             // columns reduced by this CTA
        const int rows = min(p.M, MP);
        const uint32_t part_addr = smem_addr(partial);
        for (int i = threadIdx.x; i < rows * cols; i += kThreads) {
            const int m = i / cols;
            const int nl = split * cols + (i - m * cols);
            const int n = tn * NT + nl;
            const uint32_t off = part_addr + static_cast<uint32_t>((m * NT + nl) * 4);
            float acc = 0.f;
            for (int s = 0; s < splits; ++s)
                acc += ld_shared_cluster_f32(map_to_cta(off, jn * splits + s));
            if (n < p.N) sk_store(p, m, n, acc);
        }
        cluster_sync_all();                       // peers are done reading this CTA's smem
    } else if (share > 1) {
        cluster_sync_all();   // the partner's last commits to this CTA's barriers have landed
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int IN_KIND, int MP, int NT, bool TWO>
cudaError_t sk_launch_cfg(const CUtensorMap &tmA, const CUtensorMap &tmB, const SkParams &p,
                          cudaStream_t stream) {
    using Cfg = SkCfg<IN_KIND, MP, NT, TWO>;
    auto kern = gemm_skinny_kernel<IN_KIND, MP, NT, TWO>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    const int share = p.a_share > 1 ? 2 : 1;
    const int tiles = (p.tiles_n + share - 1) / share * share;   // whole sharing groups
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * p.splits),
                       static_cast<unsigned>(p.batch > 0 ? p.batch : 1), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.splits * share);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int IN_KIND, int MP, int NT>
cudaError_t sk_launch(const CUtensorMap &tmA, const CUtensorMap &tmB, const SkParams &p,
                      cudaStream_t stream) {
    if (p.two_per_sm) {
        // the half-size ring exists for 128-column tiles only
        if constexpr (NT == 128) return sk_launch_cfg<IN_KIND, MP, NT, true>(tmA, tmB, p, stream);
        return cudaErrorInvalidValue;
    }
    return sk_launch_cfg<IN_KIND, MP, NT, false>(tmA, tmB, p, stream);
}
template <int IN_KIND, int NT>
cudaError_t sk_launch_mp(int mp, const CUtensorMap &tmA, const CUtensorMap &tmB,
                         const SkParams &p, cudaStream_t stream) {
    switch (mp) {
    case 16: return sk_launch<IN_KIND, 16, NT>(tmA, tmB, p, stream);
    case 32: return sk_launch<IN_KIND, 32, NT>(tmA, tmB, p, stream);
    case 64: return sk_launch<IN_KIND, 64, NT>(tmA, tmB, p, stream);
    case 128:
        if constexpr (NT <= 256) return sk_launch<IN_KIND, 128, NT>(tmA, tmB, p, stream);
        return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

template <int IN_KIND>
cudaError_t sk_launch_kind(int mp, int nt, const CUtensorMap &tmA, const CUtensorMap &tmB,
                           const SkParams &p, cudaStream_t stream) {
    switch (nt) {
    case 128: return sk_launch_mp<IN_KIND, 128>(mp, tmA, tmB, p, stream);
    case 256: return sk_launch_mp<IN_KIND, 256>(mp, tmA, tmB, p, stream);
    case 512: return sk_launch_mp<IN_KIND, 512>(mp, tmA, tmB, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <int NT, bool TWO>
int stages_nt(int mp) {
    switch (mp) {
    case 16: return SkCfg<IN_F16, 16, NT, TWO>::STAGES;
    case 32: return SkCfg<IN_F16, 32, NT, TWO>::STAGES;
    case 64: return SkCfg<IN_F16, 64, NT, TWO>::STAGES;
    case 128: if constexpr (NT <= 256) return SkCfg<IN_F16, 128, NT, TWO>::STAGES; return 0;
    default: return 0;
    }
}

}  // namespace
}  // namespace tg
