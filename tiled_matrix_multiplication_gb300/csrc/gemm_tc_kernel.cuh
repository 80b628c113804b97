// gemm_tc_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a
// (the kernel template and its launcher; instantiated per operand type by
// gemm_tc_f16.cu, gemm_tc_tf32.cu and gemm_tc_fp8.cu, dispatched by gemm_tc.cu).
//
// C[m,n] = sum_k A[m,k] * B[k,n], A [M,K] row-major (K-major), B [K,N]
// row-major (N-major), FP32 accumulation in tensor memory.
//
// What the pages' tile kernels do ("Matrix Multiplication", teenygrad docs,
// sections "Tiles" and "The real tiled loop"; "Triton tiled matmul",
// llm-systems-cookbook, section "The kernel"; "Fast matrix multiplication",
// ch. 12, section "The CUDA kernel") and how it maps here:
//   * one output tile per program, grouped raster over tiles
//       -> a persistent grid (one CTA, or one CTA pair, per SM / SM pair)
//          walks tile indices unit0, unit0 + units_per_step, ...; each index
//          goes through the grouped ordering (GROUP_M tile rows down, then one
//          tile right);
//   * K walked in BLOCK_K chunks, tiles loaded through zero-padding tensor
//     descriptors
//       -> one producer thread issues TMA loads of the A tile and the B tile
//          into a ring of shared-memory stages, each guarded by a "full" and an
//          "empty" mbarrier; out-of-range rows/columns/K come back as zeros,
//          which leave the dot products unchanged;
//   * acc = dot(a, b, acc) on the tensor cores, accumulator on chip for the
//     whole K loop
//       -> one thread issues tcgen05.mma into an FP32 accumulator in tensor
//          memory (128 lanes x BN columns per CTA), double buffered so the
//          epilogue of tile i overlaps the main loop of tile i+1;
//   * cast and masked store of the tile, written once
//       -> four epilogue warps read the accumulator with tcgen05.ld, round to
//          the output type and store only in-range rows and columns.
//   * Split-K (several work units per tile, each over a K range) writes FP32
//     partial tiles that a separate kernel sums in a fixed order.
//
// Two variants:
//   PAIR = false: one CTA owns a 128 x BN tile (tcgen05 cta_group::1).
//   PAIR = true : a cluster of two CTAs owns a 256 x BN tile (cta_group::2).
//     Each CTA loads its own 128 rows of A and half (BN/2 columns) of B; the
//     leader CTA (rank 0) issues the MMAs, which read A and B from both CTAs'
//     shared memory and leave rows 0..127 of the accumulator in the leader's
//     tensor memory and rows 128..255 in the peer's.  Per SM this halves the
//     B bytes that have to be staged per FLOP.
//     Synchronisation of the pair:
//       full[s]   leader's only: one arrive (leader, expect_tx of both CTAs'
//                 bytes) + the TMA completions of both CTAs;
//       empty[s]  in both CTAs: the leader's MMA commit, multicast to both;
//       tfull[b]  in both CTAs: the leader's commit after a tile's last MMA;
//       tempty[b] leader's only: one arrive per epilogue warp of both CTAs.
//   MC = 2 (with PAIR): a cluster of two pairs works on two horizontally
//     adjacent tiles, which read the same A rows.  Each CTA loads half of its
//     128 rows of A and multicasts them to the CTA in the same position of the
//     other pair, so A is read from L2 once per two pairs.  A stage may then
//     be refilled only after both pairs' MMAs are done with it: empty[s]
//     counts one commit from each pair leader.
//
// Roles: warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2..5 = epilogue (warp w may read TMEM lanes 32*(w%4) .. +31).
//
// Every mbarrier wait is bounded; on expiry the CTA records TG_ERR_TIMEOUT in
// the status word, raises a shared abort flag so the other roles stop early,
// lets its in-flight copies and MMAs finish (bounded), frees its tensor memory
// and exits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "tg_epilogue.cuh"
#include "tg_internal.h"
#include "tg_kernel_common.cuh"
#include "tg_ptx.cuh"

namespace tg {

namespace {

constexpr int kThreads = 192;
// Dynamic shared memory for the stage ring: the 227 KB a CTA may use, less
// the alignment slack and the barriers.
constexpr int kSmemBudget = 232448 - 1024 - 256;

template <int IN_KIND, int BN, bool PAIR, int MC = 1>
struct TcCfg {
    static constexpr int ESIZE = in_esize(IN_KIND);
    static constexpr int BK = 128 / ESIZE;        // one 128-byte swizzle row of K
    static constexpr int UMMA_K = 32 / ESIZE;     // K of one tcgen05.mma
    // N-major B: 128-byte swizzled rows, or 64-byte ones when those tile the
    // CTA's columns exactly and 128-byte ones do not (96 columns per CTA); 32-byte
    // rows measured much slower than loading a partly unused 128-byte box.
    static constexpr int BN_CTA_ = PAIR ? BN / 2 : BN;
    static constexpr int B_SW = ((BN_CTA_ * ESIZE) % 128 != 0 && (BN_CTA_ * ESIZE) % 64 == 0) ? 64 : 128;
    static constexpr int CHUNK_N = B_SW / ESIZE;  // N elements in one B row of a box
    // 0: kind::f16, 1: kind::tf32, 2: kind::f8f6f4
    static constexpr int KIND = IN_KIND == IN_TF32 ? 1 : (ESIZE == 1 ? 2 : 0);
    // operand format code of the instruction descriptor: f16 0 / bf16 1 under
    // kind::f16, tf32 2, and e4m3 0 / e5m2 1 under kind::f8f6f4
    static constexpr uint32_t FMT = IN_KIND == IN_TF32 ? 2u
                                    : (IN_KIND == IN_BF16 || IN_KIND == IN_E5M2) ? 1u : 0u;
    static constexpr int CTA_GROUP = PAIR ? 2 : 1;
    static constexpr int CLUSTER = CTA_GROUP * MC;      // CTAs per cluster
    static constexpr int CTA_M = 128;             // accumulator rows held by one CTA
    static constexpr int TILE_M = PAIR ? 256 : 128;
    static constexpr int BN_CTA = PAIR ? BN / 2 : BN;   // B columns staged by one CTA
    // B operand layout in shared memory.  16-bit and 8-bit operands are
    // consumed N-major, straight from row-major B.  kind::tf32 is given a
    // K-major B (the host transposes B into the workspace first): N-major B
    // tiles gave wrong products with kind::tf32 on this hardware (all zeros
    // with one descriptor variant; with the N-major descriptors that are exact
    // for FP16 and FP8, errors of 10-20 % of sum |a b|).
    static constexpr bool B_KMAJOR = IN_KIND == IN_TF32;
    static constexpr int A_STAGE = CTA_M * 128;   // bytes
    static constexpr int B_BOX = BK * B_SW;       // one CHUNK_N-wide N-major TMA box
    static constexpr int B_CHUNKS = (BN_CTA + CHUNK_N - 1) / CHUNK_N;   // last may run past
    // N-major: B_CHUNKS boxes; K-major (TF32): BN_CTA rows of 128 bytes.
    static constexpr int B_STAGE = B_KMAJOR ? BN_CTA * 128 : B_CHUNKS * B_BOX;
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
    static constexpr int TX_BYTES = STAGE_BYTES * CTA_GROUP;   // per full-barrier phase
    static constexpr int STAGES = kSmemBudget / STAGE_BYTES > 8 ? 8 : kSmemBudget / STAGE_BYTES;
    static constexpr int ACC_STRIDE = BN <= 128 ? 128 : 256;   // TMEM columns per buffer
    static constexpr int TMEM_COLS = 2 * ACC_STRIDE;           // two accumulator buffers
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;
    static constexpr uint32_t IDESC =
        make_idesc(FMT, 0u, B_KMAJOR ? 0u : 1u, TILE_M, BN);
    static_assert(BN % 32 == 0, "the epilogue reads 32 accumulator columns at a time");
    static_assert(BN_CTA % 16 == 0, "each CTA stages whole 16-column groups of B");
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
    static_assert(TMEM_COLS >= 32 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM alloc size");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(MC == 1 || MC == 2, "A is shared by at most two tiles");
};

struct Work {
    int tm, tn, split, kt0, kt1;
    int tail;   // index among the tail-split tiles, or -1
    int z;      // batch index
};

// Columns of work units: with A multicast one unit is two adjacent tiles.
__device__ __forceinline__ int unit_cols(const TcParams &p) {
    return (p.tiles_n + p.mc - 1) / p.mc;
}

__device__ __forceinline__ int units_per_batch(const TcParams &p) {
    return p.tiles_m * unit_cols(p) * p.splits;
}

__device__ __forceinline__ int total_units(const TcParams &p) {
    return p.tail_tiles > 0 ? p.tail_start + p.tail_tiles * p.tail_splits
                            : units_per_batch(p) * p.batch;
}

// `q`: which tile of a multicast unit this CTA's pair works on.
__device__ __forceinline__ Work decode_work(const TcParams &p, int w, int q = 0) {
    Work r;
    int t;
    r.z = 0;
    if (p.batch > 1) {   // batches are the slowest dimension (no tail split)
        const int per = units_per_batch(p);
        r.z = w / per;
        w -= r.z * per;
    }
    if (p.tail_tiles > 0 && w >= p.tail_start) {
        const int u = w - p.tail_start;
        r.tail = u / p.tail_splits;
        r.split = u - r.tail * p.tail_splits;
        t = p.tail_start + r.tail;
    } else {
        t = w / p.splits;
        r.split = w - t * p.splits;
        r.tail = -1;
    }
    const int per_group = p.group_m * unit_cols(p);
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int size_m = min(p.tiles_m - first_m, p.group_m);
    const int pos = t - g * per_group;
    r.tm = first_m + pos % size_m;
    r.tn = (pos / size_m) * p.mc + q;
    const int kps = r.tail >= 0 ? p.tail_kps : p.k_tiles_per_split;
    r.kt0 = r.split * kps;
    r.kt1 = min(r.kt0 + kps, p.k_tiles);
    return r;
}

__device__ __forceinline__ void epilogue_bar_sync() {
    asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
}

// Store 32 consecutive accumulator values (columns col .. col+31 of `row`).
__device__ __forceinline__ void store_chunk(const TcParams &p, int split, int row, int col,
                                            uint32_t (&r)[32], int z = 0) {
    const int ncols = min(32, p.N - col);
    if (p.splits > 1) {
        float *dst = p.partial + (static_cast<int64_t>(split) * p.M + row) * p.N + col;
        if (ncols == 32 && (p.N & 3) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<uint4 *>(dst + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < ncols) dst[j] = __uint_as_float(r[j]);
        }
        return;
    }
    if (p.epi.on) epi_chunk32(p.epi, p.out_kind, row, col, ncols, r, z);
    const int64_t off = static_cast<int64_t>(z) * p.stride_c + static_cast<int64_t>(row) * p.ldc + col;
    if (p.out_kind == OUT_F32) {
        float *dst = static_cast<float *>(p.c) + off;
        if (ncols == 32 && p.c_vector) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<uint4 *>(dst + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < ncols) dst[j] = __uint_as_float(r[j]);
        }
    } else if (p.out_kind == OUT_F16) {
        __half *dst = static_cast<__half *>(p.c) + off;
        if (ncols == 32 && p.c_vector) {
#pragma unroll
            for (int j = 0; j < 32; j += 8)
                *reinterpret_cast<uint4 *>(dst + j) =
                    make_uint4(pack_half2(r[j], r[j + 1]), pack_half2(r[j + 2], r[j + 3]),
                               pack_half2(r[j + 4], r[j + 5]), pack_half2(r[j + 6], r[j + 7]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < ncols) dst[j] = __float2half_rn(__uint_as_float(r[j]));
        }
    } else {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.c) + off;
        if (ncols == 32 && p.c_vector) {
#pragma unroll
            for (int j = 0; j < 32; j += 8)
                *reinterpret_cast<uint4 *>(dst + j) =
                    make_uint4(pack_bf162(r[j], r[j + 1]), pack_bf162(r[j + 2], r[j + 3]),
                               pack_bf162(r[j + 4], r[j + 5]), pack_bf162(r[j + 6], r[j + 7]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < ncols) dst[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
        }
    }
}

template <int IN_KIND, int BN, bool PAIR, int MC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams p) {
    using Cfg = TcCfg<IN_KIND, BN, PAIR, MC>;
    constexpr int S = Cfg::STAGES;
    constexpr int CG = Cfg::CTA_GROUP;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;       // 1024-B aligned (swizzle atoms)
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base;                            // S x A_STAGE
    const uint32_t sB = base + S * Cfg::A_STAGE;         // S x B_STAGE
    const uint32_t bars = sB + S * Cfg::B_STAGE;
    uint8_t *gbars = gbase + (bars - base);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto tfull_bar = [&](int b) { return bars + 8u * (2 * S + b); };
    auto tempty_bar = [&](int b) { return bars + 8u * (2 * S + 2 + b); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbars + 8 * Cfg::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int never_abort;
    __shared__ int tail_last;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool CLUSTERED = PAIR || MC > 1;
    const uint32_t crank = CLUSTERED ? cluster_cta_rank() : 0u;  // rank in the cluster
    const uint32_t rank = crank % CG;                             // position in the pair
    const int q = static_cast<int>(crank / CG);                   // pair within the cluster
    const uint32_t pair_leader = static_cast<uint32_t>(q * CG);   // cluster rank of my leader
    const bool leader = rank == 0;
    const int unit0 = static_cast<int>(blockIdx.x) / Cfg::CLUSTER;
    const int unit_step = static_cast<int>(gridDim.x) / Cfg::CLUSTER;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), MC);   // one MMA commit per pair sharing the stage
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4 * CG);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        never_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_addr(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CLUSTERED) cluster_sync_all();   // peer barriers initialised before any remote signal
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Prologue done: let the next kernel's prologue start, then wait for the
    // previous kernel's writes before the first global-memory access.
    if (threadIdx.x == 0) grid_launch_dependents();
    grid_dependency_wait();

    const int total = total_units(p);

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int w = unit0; w < total && ok; w += unit_step) {
                const Work wk = decode_work(p, w, q);
                const int row0 = wk.tm * Cfg::TILE_M + static_cast<int>(rank) * Cfg::CTA_M;
                const int col0 = wk.tn * BN + static_cast<int>(rank) * Cfg::BN_CTA;
                for (int kt = wk.kt0; kt < wk.kt1; ++kt) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full_bar(stage), Cfg::TX_BYTES);
                    const uint32_t fb =
                        PAIR ? map_to_cta(full_bar(stage), pair_leader) : full_bar(stage);
                    // rank-3 maps for batched operands (z = batch), 2-D otherwise
                    auto load = [&](uint32_t dst, const CUtensorMap *map, bool batched, int x,
                                    int y) {
                        if constexpr (PAIR) {
                            if (batched)
                                tma_load_3d_pair(dst, map, fb, x, y, wk.z);
                            else
                                tma_load_2d_pair(dst, map, fb, x, y);
                        } else {
                            if (batched)
                                tma_load_3d(dst, map, fb, x, y, wk.z);
                            else
                                tma_load_2d(dst, map, fb, x, y);
                        }
                    };
                    if constexpr (MC == 2) {
                        // my half (q) of this CTA's A rows, to me and my counterpart
                        const uint16_t mask =
                            static_cast<uint16_t>((1u << rank) | (1u << (CG + rank)));
                        const uint32_t dst = sA + stage * Cfg::A_STAGE + q * (Cfg::A_STAGE / 2);
                        const int ya = row0 + q * (Cfg::CTA_M / 2);
                        if constexpr (PAIR) {
                            if (p.a_batched)
                                tma_load_3d_pair_mc(dst, &tmA, fb, kt * Cfg::BK, ya, wk.z, mask);
                            else
                                tma_load_2d_pair_mc(dst, &tmA, fb, kt * Cfg::BK, ya, mask);
                        } else {
                            if (p.a_batched)
                                tma_load_3d_mc(dst, &tmA, fb, kt * Cfg::BK, ya, wk.z, mask);
                            else
                                tma_load_2d_mc(dst, &tmA, fb, kt * Cfg::BK, ya, mask);
                        }
                    } else {
                        load(sA + stage * Cfg::A_STAGE, &tmA, p.a_batched, kt * Cfg::BK, row0);
                    }
                    if constexpr (Cfg::B_KMAJOR) {
                        // B^T tile [BN_CTA rows of N] x [BK of K], one box
                        load(sB + stage * Cfg::B_STAGE, &tmB, p.b_batched, kt * Cfg::BK, col0);
                    } else {
#pragma unroll
                        for (int j = 0; j < Cfg::B_CHUNKS; ++j)
                            load(sB + stage * Cfg::B_STAGE + j * Cfg::B_BOX, &tmB, p.b_batched,
                                 col0 + j * Cfg::CHUNK_N, kt * Cfg::BK);
                    }
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                record_failure(p.status, 6, (ROLE_PRODUCER << 16) | stage);
                *abort_flag = 1;
            }
            // Every issued copy must land before the CTA may exit.  The full
            // barriers live in the leader, which waits for both CTAs' copies.
            if (leader) {
                const int64_t first = issued > S ? issued - S : 0;
                for (int64_t i = first; i < issued; ++i) {
                    if (!mbar_wait(full_bar(static_cast<int>(i % S)),
                                   static_cast<uint32_t>((i / S) & 1), p.timeout_ns,
                                   &never_abort)) {
                        record_failure(p.status, 6, (ROLE_DRAIN << 16) | 1);
                        break;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_count = 0;
            bool ok = true;
            for (int w = unit0; w < total && ok; w += unit_step) {
                const Work wk = decode_work(p, w, q);
                const uint32_t buf = acc_count & 1u;
                const uint32_t acc_phase = (acc_count >> 1) & 1u;
                if (!mbar_wait<PAIR>(tempty_bar(buf), acc_phase ^ 1u, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * Cfg::ACC_STRIDE;
                for (int kt = wk.kt0; kt < wk.kt1; ++kt) {
                    if (!mbar_wait(full_bar(stage), phase, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a0 = sA + stage * Cfg::A_STAGE;
                    const uint32_t b0 = sB + stage * Cfg::B_STAGE;
#pragma unroll
                    for (int kk = 0; kk < Cfg::BK / Cfg::UMMA_K; ++kk) {
                        const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd =
                            Cfg::B_KMAJOR
                                ? smem_desc_sw128(b0 + kk * 32, 16, 1024)
                                : smem_desc_mn<Cfg::B_SW>(b0 + kk * Cfg::UMMA_K * Cfg::B_SW,
                                                          Cfg::B_BOX);
                        umma_ss<Cfg::KIND, CG>(d_tmem, ad, bd, Cfg::IDESC,
                                               (kt > wk.kt0 || kk > 0) ? 1u : 0u);
                    }
                    if constexpr (PAIR)   // every CTA whose stage this pair read from
                        umma_commit_pair(empty_bar(stage), MC == 2 ? 0xF : 0x3);
                    else if constexpr (MC == 2)   // both CTAs filled this stage's A
                        umma_commit_mc(empty_bar(stage), 0x3);
                    else
                        umma_commit(empty_bar(stage));
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    umma_commit_pair(tfull_bar(buf), static_cast<uint16_t>(0x3u << pair_leader));
                else
                    umma_commit(tfull_bar(buf));
                ++acc_count;
            }
            if (!ok) {
                record_failure(p.status, 6, (ROLE_MMA << 16) | stage);
                *abort_flag = 1;
            }
            // All issued MMAs complete before tensor memory is released.
            if constexpr (PAIR)
                umma_commit_pair(drain_bar, static_cast<uint16_t>(1u << crank));
            else
                umma_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, p.timeout_ns, &never_abort))
                record_failure(p.status, 6, (ROLE_DRAIN << 16) | 2);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- epilogue
        const int quad = warp & 3;
        uint32_t acc_count = 0;
        for (int w = unit0; w < total; w += unit_step) {
            const Work wk = decode_work(p, w, q);
            const uint32_t buf = acc_count & 1u;
            const uint32_t acc_phase = (acc_count >> 1) & 1u;
            const bool got = mbar_wait<PAIR>(tfull_bar(buf), acc_phase, p.timeout_ns, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) record_failure(p.status, 6, (ROLE_EPILOGUE << 16) | quad);
                *abort_flag = 1;
                break;
            }
            tc_fence_after_sync();
            const int trow = static_cast<int>(rank) * Cfg::CTA_M + quad * 32 + lane;  // in tile
            const int row = wk.tm * Cfg::TILE_M + trow;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * Cfg::ACC_STRIDE;
            // tail-split unit: this range's FP32 partial tile, laid out as
            // [BN/4 column quads][TILE_M rows][4] so that one store or load of
            // a warp (32 consecutive rows, one column quad) covers 512
            // contiguous bytes
            float *ptile = nullptr;
            if (wk.tail >= 0)
                ptile = p.tail_partial +
                        (static_cast<int64_t>(wk.tail) * p.tail_splits + wk.split) * Cfg::TILE_M * BN;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r[32];
                tmem_load_32cols_sync(taddr + c0, r);
                const int col = wk.tn * BN + c0;
                if (ptile != nullptr) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<uint4 *>(
                            ptile + ((static_cast<int64_t>(c0 + j) >> 2) * Cfg::TILE_M + trow) * 4) =
                            make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
                } else if (row < p.M && col < p.N) {
                    store_chunk(p, wk.split, row, col, r, wk.z);
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_cluster(tempty_bar(buf), pair_leader);
                else
                    mbar_arrive(tempty_bar(buf));
            }
            if (wk.tail >= 0) {
                // The range that completes the tile last sums all ranges'
                // partials, in range order, and writes C.  No range waits for
                // another, so the order in which ranges run does not matter.
                epilogue_bar_sync();                 // this CTA's partial rows written
                if (threadIdx.x == 64) {
                    __threadfence();
                    const unsigned int old =
                        atomicAdd(p.tail_count + wk.tail * Cfg::CTA_GROUP + rank, 1u);
                    tail_last = (old == static_cast<unsigned int>(p.tail_splits - 1)) ? 1 : 0;
                    __threadfence();
                }
                epilogue_bar_sync();
                if (tail_last && row < p.M) {
                    const float *base = p.tail_partial +
                                        static_cast<int64_t>(wk.tail) * p.tail_splits * Cfg::TILE_M * BN;
                    const int64_t split_stride = static_cast<int64_t>(Cfg::TILE_M) * BN;
#pragma unroll 1
                    for (int c0 = 0; c0 < BN; c0 += 32) {
                        const int col = wk.tn * BN + c0;
                        if (col >= p.N) break;
                        float acc[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
                        for (int sidx = 0; sidx < p.tail_splits; ++sidx) {
                            const float *src = base + sidx * split_stride;
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                    src + ((static_cast<int64_t>(c0 + j) >> 2) * Cfg::TILE_M + trow) * 4));
                                acc[j] += v.x;
                                acc[j + 1] += v.y;
                                acc[j + 2] += v.z;
                                acc[j + 3] += v.w;
                            }
                        }
                        uint32_t r[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(acc[j]);
                        store_chunk(p, 0, row, col, r);
                    }
                }
                epilogue_bar_sync();                 // tail_last is reused by the next unit
            }
            ++acc_count;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // the peers are done with this CTA's smem, barriers and TMEM
    if constexpr (CLUSTERED) cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, Cfg::TMEM_COLS);
    }
}


struct ClusterCache {
    std::mutex mu;
    int max_clusters[64] = {0};
};

template <int IN_KIND, int BN, bool PAIR, int MC>
cudaError_t launch_impl(const CUtensorMap &tmA, const CUtensorMap &tmB, const TcParams &p,
                        int ctas, cudaStream_t stream) {
    using Cfg = TcCfg<IN_KIND, BN, PAIR, MC>;
    auto kern = gemm_tc_kernel<IN_KIND, BN, PAIR, MC>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (PAIR || MC > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = Cfg::CLUSTER;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        // Cap the persistent grid at the clusters that fit at once.
        static ClusterCache cache;
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        int maxc = 0;
        {
            std::lock_guard<std::mutex> lk(cache.mu);
            maxc = (dev >= 0 && dev < 64) ? cache.max_clusters[dev] : 0;
        }
        if (maxc == 0) {
            cfg.gridDim = dim3(Cfg::CLUSTER, 1, 1);
            if ((e = cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg)) != cudaSuccess) return e;
            if (maxc < 1) return cudaErrorInvalidConfiguration;
            std::lock_guard<std::mutex> lk(cache.mu);
            if (dev >= 0 && dev < 64) cache.max_clusters[dev] = maxc;
        }
        int clusters = (ctas + Cfg::CLUSTER - 1) / Cfg::CLUSTER;
        if (clusters > maxc) clusters = maxc;
        cfg.gridDim = dim3(Cfg::CLUSTER * clusters, 1, 1);
    } else {
        cfg.gridDim = dim3(ctas, 1, 1);
    }
    e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int IN_KIND, bool PAIR, int MC>
cudaError_t launch_kind(int block_n, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const TcParams &p, int ctas, cudaStream_t stream) {
    if constexpr (MC == 2 && PAIR) {
        switch (block_n) {
        case 192: return launch_impl<IN_KIND, 192, true, 2>(tmA, tmB, p, ctas, stream);
        case 224: return launch_impl<IN_KIND, 224, true, 2>(tmA, tmB, p, ctas, stream);
        case 256: return launch_impl<IN_KIND, 256, true, 2>(tmA, tmB, p, ctas, stream);
        default: return cudaErrorInvalidValue;
        }
    } else if constexpr (MC == 2) {
        switch (block_n) {
        case 128: return launch_impl<IN_KIND, 128, false, 2>(tmA, tmB, p, ctas, stream);
        case 256: return launch_impl<IN_KIND, 256, false, 2>(tmA, tmB, p, ctas, stream);
        default: return cudaErrorInvalidValue;
        }
    } else if constexpr (PAIR) {
        switch (block_n) {
        case 128: return launch_impl<IN_KIND, 128, true, 1>(tmA, tmB, p, ctas, stream);
        case 192: return launch_impl<IN_KIND, 192, true, 1>(tmA, tmB, p, ctas, stream);
        case 224: return launch_impl<IN_KIND, 224, true, 1>(tmA, tmB, p, ctas, stream);
        case 256: return launch_impl<IN_KIND, 256, true, 1>(tmA, tmB, p, ctas, stream);
        default: return cudaErrorInvalidValue;
        }
    } else {
        switch (block_n) {
        case 128: return launch_impl<IN_KIND, 128, false, 1>(tmA, tmB, p, ctas, stream);
        case 192: return launch_impl<IN_KIND, 192, false, 1>(tmA, tmB, p, ctas, stream);
        case 224: return launch_impl<IN_KIND, 224, false, 1>(tmA, tmB, p, ctas, stream);
        case 256: return launch_impl<IN_KIND, 256, false, 1>(tmA, tmB, p, ctas, stream);
        default: return cudaErrorInvalidValue;
        }
    }
}

template <int IN_KIND, bool PAIR>
int stages_kind(int block_n) {
    switch (block_n) {
    case 128: return TcCfg<IN_KIND, 128, PAIR>::STAGES;
    case 192: return TcCfg<IN_KIND, 192, PAIR>::STAGES;
    case 224: return TcCfg<IN_KIND, 224, PAIR>::STAGES;
    case 256: return TcCfg<IN_KIND, 256, PAIR>::STAGES;
    default: return 0;
    }
}


// Kernel variants of one operand type: A-multicast pairs, pairs, single CTAs.
template <int IN_KIND>
cudaError_t launch_variant(int block_n, bool pair, int mc, const CUtensorMap &tmA,
                           const CUtensorMap &tmB, const TcParams &p, int ctas,
                           cudaStream_t stream) {
    if (mc == 2)
        return pair ? launch_kind<IN_KIND, true, 2>(block_n, tmA, tmB, p, ctas, stream)
                    : launch_kind<IN_KIND, false, 2>(block_n, tmA, tmB, p, ctas, stream);
    return pair ? launch_kind<IN_KIND, true, 1>(block_n, tmA, tmB, p, ctas, stream)
                : launch_kind<IN_KIND, false, 1>(block_n, tmA, tmB, p, ctas, stream);
}

}  // namespace
}  // namespace tg
