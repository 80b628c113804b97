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
//          memory (128 lanes x BN columns per CTA), double buffered up to 256
//          columns so the epilogue of tile i overlaps the main loop of tile i+1;
//   * cast and store of the tile through its output descriptor, written once
//       -> four epilogue warps read the accumulator with tcgen05.ld, round to
//          the output type, stage 32-row boxes in shared memory and write them
//          with TMA stores, which leave out everything outside C ("The real
//          tiled loop": the result leaves through the output descriptor).
//          Where C's base or row pitch is not 16-byte aligned, or for split-K
//          partials, the warps store their rows directly instead.
//   * Split-K (several work units per tile, each over a K range) writes FP32
//     partial tiles that a separate kernel sums in a fixed order.
//
// Variants:
//   PAIR = false: one CTA owns a 128 x BN tile (tcgen05 cta_group::1).
//   PAIR = true : a cluster of two CTAs owns a 256 x BN tile (cta_group::2).
//     Each CTA loads its own 128 rows of A and half of the B columns of every
//     MMA; the leader CTA (rank 0) issues the MMAs, which read A and B from
//     both CTAs' shared memory and leave rows 0..127 of the accumulator in the
//     leader's tensor memory and rows 128..255 in the peer's.  Per SM this
//     halves the B bytes that have to be staged per FLOP.
//     Synchronisation of the pair:
//       full[s]   leader's only: one arrive (leader, expect_tx of both CTAs'
//                 bytes) + the TMA completions of both CTAs;
//       empty[s]  in both CTAs: the leader's MMA commit, multicast to both;
//       tfull[b]  in both CTAs: the leader's commit after a tile's last MMA;
//       tempty[b] leader's only: one arrive per epilogue warp of both CTAs.
//   BN = 512 (pairs only): two N = 256 MMAs per K step on one A tile, into
//     the two halves of a 512-column accumulator that fills the tensor memory
//     (one accumulator buffer); a stage then holds 48 bytes per SM-clock of MMA
//     work instead of the 64 of a 256-wide pair tile.
//   MC = 2 (pairs, BN <= 256): a cluster of two pairs works on two
//     horizontally adjacent tiles, which read the same A rows.  Each CTA loads
//     half of its 128 rows of A and multicasts them to the CTA in the same
//     position of the other pair, so A is read from L2 once per two pairs.  A
//     stage may then be refilled only after both pairs' MMAs are done with it:
//     empty[s] counts one commit from each pair leader.
//
// Roles: warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2..9 = epilogue.  Warp w may read TMEM lanes 32*(w%4) .. +31, so two
// warps serve each lane quarter; warps 2..5 drain the first half of the
// accumulator's 32-column chunks and warps 6..9 the rest.  Per chunk a warp's
// work is a chain of short dependent steps (TMEM load, convert, stage, fence,
// TMA store, buffer wait), so two warps per quarter halve the time from a
// tile's last MMA to its last store.
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

constexpr int kEpiWarps = 8;                 // two per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;
// Dynamic shared memory for the stage ring and the output staging: the
// 227 KB a CTA may use, less the alignment slack and the barriers.
constexpr int kSmemBudget = 232448 - 1024 - 256;
// Output staging: per epilogue warp, kOutBufs boxes of 32 rows x 64 bytes
// (32 columns of a 16-bit type or 16 of FP32), 64-byte swizzled.
constexpr int kOutBox = 32 * 64;
constexpr int kOutBufs = 2;
constexpr int kOutStaging = kEpiWarps * kOutBufs * kOutBox;

template <int IN_KIND, int BN, bool PAIR, int MC = 1>
struct TcCfg {
    static constexpr int ESIZE = in_esize(IN_KIND);
    static constexpr int BK = 128 / ESIZE;        // one 128-byte swizzle row of K
    static constexpr int UMMA_K = 32 / ESIZE;     // K of one tcgen05.mma
    static constexpr int CTA_GROUP = PAIR ? 2 : 1;
    static constexpr int CLUSTER = CTA_GROUP * MC;      // CTAs per cluster
    static constexpr int CTA_M = 128;             // accumulator rows held by one CTA
    static constexpr int TILE_M = PAIR ? 256 : 128;
    // N of one MMA; a 512-wide tile issues two per K step
    static constexpr int MMA_N = BN > 256 ? 256 : BN;
    static constexpr int N_MMAS = BN / MMA_N;
    static constexpr int MMA_N_CTA = PAIR ? MMA_N / 2 : MMA_N;   // B columns of one MMA per CTA
    static constexpr int BN_CTA = N_MMAS * MMA_N_CTA;            // B columns staged by one CTA
    // B is read N-major, straight from row-major memory, for every operand
    // type.  TF32 (4-byte elements) takes 128-byte rows swizzled in 32-byte
    // atoms (smem_desc_mn_tf32).  16-bit and 8-bit operands take 128-byte
    // swizzled rows, or 64-byte ones when those tile the CTA's columns of one
    // MMA exactly and 128-byte ones do not (96 columns per CTA); 32-byte rows
    // measured much slower than loading a partly unused 128-byte box.
    static constexpr bool B_TF32 = IN_KIND == IN_TF32;
    static constexpr int B_SW =
        (!B_TF32 && (MMA_N_CTA * ESIZE) % 128 != 0 && (MMA_N_CTA * ESIZE) % 64 == 0) ? 64 : 128;
    static constexpr int CHUNK_N = B_SW / ESIZE;  // N elements in one B row of a box
    // 0: kind::f16, 1: kind::tf32, 2: kind::f8f6f4
    static constexpr int KIND = IN_KIND == IN_TF32 ? 1 : (ESIZE == 1 ? 2 : 0);
    // operand format code of the instruction descriptor: f16 0 / bf16 1 under
    // kind::f16, tf32 2, and e4m3 0 / e5m2 1 under kind::f8f6f4
    static constexpr uint32_t FMT = IN_KIND == IN_TF32 ? 2u
                                    : (IN_KIND == IN_BF16 || IN_KIND == IN_E5M2) ? 1u : 0u;
    static constexpr int A_STAGE = CTA_M * 128;   // bytes
    static constexpr int B_BOX = BK * B_SW;       // one CHUNK_N-wide N-major TMA box
    // boxes per MMA (the last may run past the MMA's columns)
    static constexpr int CHUNKS_PER_MMA = (MMA_N_CTA + CHUNK_N - 1) / CHUNK_N;
    static constexpr int B_CHUNKS = N_MMAS * CHUNKS_PER_MMA;
    static constexpr int B_MMA_STRIDE = CHUNKS_PER_MMA * B_BOX;  // bytes between MMAs' B
    static constexpr int B_STAGE = B_CHUNKS * B_BOX;
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
    static constexpr int TX_BYTES = STAGE_BYTES * CTA_GROUP;   // per full-barrier phase
    static constexpr int STAGES_FIT = (kSmemBudget - kOutStaging) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int ACC_STRIDE = BN <= 128 ? 128 : (BN <= 256 ? 256 : 512);  // TMEM columns
    static constexpr int NUM_ACC = ACC_STRIDE == 512 ? 1 : 2;  // accumulator buffers
    static constexpr int TMEM_COLS = NUM_ACC * ACC_STRIDE;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * NUM_ACC + 1;
    static constexpr int SMEM_BYTES =
        1024 + STAGES * STAGE_BYTES + kOutStaging + NUM_BARS * 8 + 16;
    static constexpr uint32_t IDESC =
        make_idesc(FMT, 0u, 1u, TILE_M, MMA_N);
    static_assert(BN % 32 == 0, "the epilogue reads 32 accumulator columns at a time");
    static_assert(MMA_N_CTA % 16 == 0, "each CTA stages whole 16-column groups of B");
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
    static_assert(STAGES >= 2, "a ring needs two stages");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM alloc size");
    static_assert(MMA_N % 16 == 0 && MMA_N >= 16 && MMA_N <= 256, "MMA N");
    static_assert(BN <= 256 || (PAIR && BN == 512 && MC == 1),
                  "512-wide tiles: CTA pairs without multicast");
    // one MMA reads K rows kk*UMMA_K .. +UMMA_K-1 of each of its boxes: in bounds
    static_assert((BK / UMMA_K) * UMMA_K * B_SW <= B_BOX, "MMA reads stay inside the box");
    static_assert(MC == 1 || (MC == 2 && PAIR), "A is shared by two CTA pairs at most");
};

struct Work {
    int tm, tn, split, kt0, kt1;
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
    return units_per_batch(p) * p.batch;
}

// `q`: which tile of a multicast unit this CTA's pair works on.
__device__ __forceinline__ Work decode_work(const TcParams &p, int w, int q = 0) {
    Work r;
    r.z = 0;
    if (p.batch > 1) {   // batches are the slowest dimension
        const int per = units_per_batch(p);
        r.z = w / per;
        w -= r.z * per;
    }
    const int t = w / p.splits;
    r.split = w - t * p.splits;
    const int per_group = p.group_m * unit_cols(p);
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int size_m = min(p.tiles_m - first_m, p.group_m);
    const int pos = t - g * per_group;
    r.tm = first_m + pos % size_m;
    r.tn = (pos / size_m) * p.mc + q;
    r.kt0 = r.split * p.k_tiles_per_split;
    r.kt1 = min(r.kt0 + p.k_tiles_per_split, p.k_tiles);
    return r;
}

// Store 32 consecutive accumulator values (columns col .. col+31 of `row`)
// straight from registers: the split-K partials, and C where its base or row
// pitch rules out TMA stores.
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

// Store a warp's 32 rows x 32 columns chunk (this lane's row `row` in r[])
// through the warp's staging area `stg` (32 x 32 words, 16-byte aligned): each
// lane writes its row with 16-byte stores, then the warp writes one row at a
// time with lanes on consecutive columns, so a store instruction covers 32
// consecutive columns of one row instead of one column of 32 rows.  Row i of
// the chunk takes 128 bytes with its 16-byte pieces swizzled (piece p at
// p ^ (i & 7)), so neither pass has bank conflicts.  For C whose base or row
// pitch rules out wide stores, and split-K partials whose row length is not a
// multiple of 4.  Called by all 32 lanes with the same wrow0 (the warp's
// first row) and col < N.
__device__ __forceinline__ void store_chunk_rows(const TcParams &p, int split, int wrow0, int col,
                                                 int lane, uint32_t (&r)[32], float *stg,
                                                 int z = 0) {
    const int ncols = min(32, p.N - col);
    const int row = wrow0 + lane;
    if (p.splits == 1 && p.epi.on && row < p.M) epi_chunk32(p.epi, p.out_kind, row, col, ncols, r, z);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4 *>(stg + lane * 32 + ((k ^ (lane & 7)) << 2)) =
            make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
    __syncwarp();
    const int rows = min(32, p.M - wrow0);
    const int piece = lane >> 2, word = lane & 3;
#pragma unroll 1
    for (int i = 0; i < rows; ++i) {
        const float v = stg[i * 32 + ((piece ^ (i & 7)) << 2) + word];
        if (lane >= ncols) continue;
        if (p.splits > 1) {
            p.partial[(static_cast<int64_t>(split) * p.M + wrow0 + i) * p.N + col + lane] = v;
            continue;
        }
        const int64_t off = static_cast<int64_t>(z) * p.stride_c +
                            static_cast<int64_t>(wrow0 + i) * p.ldc + col + lane;
        if (p.out_kind == OUT_F32)
            static_cast<float *>(p.c)[off] = v;
        else if (p.out_kind == OUT_F16)
            static_cast<__half *>(p.c)[off] = __float2half_rn(v);
        else
            static_cast<__nv_bfloat16 *>(p.c)[off] = __float2bfloat16_rn(v);
    }
    __syncwarp();   // the staging area is free for the next chunk
}

// Writes 16 bytes (four 32-bit words) as chunk `chunk` (0..3) of this lane's
// 64-byte row of an output staging box, with the 64-byte swizzle a TMA store
// of that box expects (16-byte chunk index XOR address bits 7..8).  Eight
// consecutive lanes hit eight different 16-byte bank groups.
__device__ __forceinline__ void stage_chunk(uint32_t box, int lane, int chunk, uint32_t a,
                                            uint32_t b, uint32_t c, uint32_t d) {
    const uint32_t addr = box + static_cast<uint32_t>(lane) * 64u +
                          (static_cast<uint32_t>(chunk ^ ((lane >> 1) & 3)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

template <int IN_KIND, int BN, bool PAIR, int MC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
    using Cfg = TcCfg<IN_KIND, BN, PAIR, MC>;
    constexpr int S = Cfg::STAGES;
    constexpr int CG = Cfg::CTA_GROUP;
    constexpr int NACC = Cfg::NUM_ACC;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;       // 1024-B aligned (swizzle atoms)
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base;                            // S x A_STAGE
    const uint32_t sB = base + S * Cfg::A_STAGE;         // S x B_STAGE
    const uint32_t sOut = sB + S * Cfg::B_STAGE;         // output staging boxes
    const uint32_t bars = sOut + kOutStaging;
    uint8_t *gbars = gbase + (bars - base);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto tfull_bar = [&](int b) { return bars + 8u * (2 * S + b); };
    auto tempty_bar = [&](int b) { return bars + 8u * (2 * S + NACC + b); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 2 * NACC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbars + 8 * Cfg::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int never_abort;

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
        for (int b = 0; b < NACC; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), kEpiWarps * CG);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        never_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        if (p.c_tma) tma_prefetch_map(&tmC);
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
                // this CTA's B columns of MMA 0; MMA h adds h * MMA_N
                const int colb = wk.tn * BN + static_cast<int>(rank) * Cfg::MMA_N_CTA;
                for (int kt = wk.kt0; kt < wk.kt1; ++kt) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full_bar(stage), Cfg::TX_BYTES);
                    const uint32_t fb =
                        PAIR ? map_to_cta(full_bar(stage), pair_leader) : full_bar(stage);
                    // rank-3 maps for batched operands (z = batch), 2-D otherwise
                    // (checked builds: the box lies in the ring, x is 16-byte aligned)
                    auto load = [&](uint32_t dst, const CUtensorMap *map, bool batched, int x,
                                    int y, uint32_t bytes, int site) {
                        if (!tg_check(p.status,
                                      dst >= sA && dst + bytes <= sOut &&
                                          tma_x_aligned(x, Cfg::ESIZE),
                                      site, stage))
                            return;
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
                        if (tg_check(p.status,
                                     dst >= sA && dst + Cfg::A_STAGE / 2 <= sB &&
                                         tma_x_aligned(kt * Cfg::BK, Cfg::ESIZE),
                                     CHK_TC_LOAD_A, stage)) {
                            if (p.a_batched)
                                tma_load_3d_pair_mc(dst, &tmA, fb, kt * Cfg::BK, ya, wk.z, mask);
                            else
                                tma_load_2d_pair_mc(dst, &tmA, fb, kt * Cfg::BK, ya, mask);
                        }
                    } else {
                        load(sA + stage * Cfg::A_STAGE, &tmA, p.a_batched, kt * Cfg::BK, row0,
                             Cfg::A_STAGE, CHK_TC_LOAD_A);
                    }
#pragma unroll
                    for (int j = 0; j < Cfg::B_CHUNKS; ++j)
                        load(sB + stage * Cfg::B_STAGE + j * Cfg::B_BOX, &tmB, p.b_batched,
                             colb + (j / Cfg::CHUNKS_PER_MMA) * Cfg::MMA_N +
                                 (j % Cfg::CHUNKS_PER_MMA) * Cfg::CHUNK_N,
                             kt * Cfg::BK, Cfg::B_BOX, CHK_TC_LOAD_B);
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
                const uint32_t buf = NACC == 2 ? (acc_count & 1u) : 0u;
                const uint32_t acc_phase = NACC == 2 ? ((acc_count >> 1) & 1u) : (acc_count & 1u);
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
                    // (checked builds: the stage's operands lie in the ring; if not,
                    // its MMAs are left out and the ring still advances)
                    const int kk_end = tg_check(p.status,
                                                a0 + Cfg::A_STAGE <= sB &&
                                                    b0 + Cfg::N_MMAS * Cfg::B_MMA_STRIDE <= sOut,
                                                CHK_TC_MMA, stage)
                                           ? Cfg::BK / Cfg::UMMA_K
                                           : 0;
#pragma unroll
                    for (int kk = 0; kk < Cfg::BK / Cfg::UMMA_K; ++kk) {
                        if (kk >= kk_end) break;
                        const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
#pragma unroll
                        for (int h = 0; h < Cfg::N_MMAS; ++h) {
                            const uint32_t bs =
                                b0 + h * Cfg::B_MMA_STRIDE + kk * Cfg::UMMA_K * Cfg::B_SW;
                            const uint64_t bd = Cfg::B_TF32
                                                    ? smem_desc_mn_tf32(bs, Cfg::B_BOX)
                                                    : smem_desc_mn<Cfg::B_SW>(bs, Cfg::B_BOX);
                            umma_ss<Cfg::KIND, CG>(d_tmem + h * Cfg::MMA_N, ad, bd, Cfg::IDESC,
                                                   (kt > wk.kt0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    if constexpr (PAIR)   // every CTA whose stage this pair read from
                        umma_commit_pair(empty_bar(stage), MC == 2 ? 0xF : 0x3);
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
        const int ew = warp - 2;                       // epilogue warp 0..7
        const int quad = warp & 3;                     // its TMEM lane quarter
        // its 32-column chunks of the accumulator: the first or second half
        constexpr int kChunks = BN / 32;
        constexpr int kHalf = (kChunks + 1) / 2;
        const int cbeg = (ew / 4) * kHalf * 32;
        const int cend = min(BN, cbeg + kHalf * 32);
        const bool f32_out = p.out_kind == OUT_F32;
        // this warp's staging boxes; boxes are used round-robin, and a box is
        // rewritten only after the TMA store issued kOutBufs boxes earlier has
        // finished reading it
        const uint32_t my_boxes = sOut + static_cast<uint32_t>(ew * kOutBufs * kOutBox);
        // the same 4 KB as 32 x 32 words, for C written without TMA stores
        float *my_stg = reinterpret_cast<float *>(gbase + (my_boxes - base));
        static_assert(kOutBufs * kOutBox >= 32 * 32 * 4, "a warp's staging holds a 32 x 32 chunk");
        uint32_t nbox = 0;
        auto next_box = [&]() {
            if (nbox >= kOutBufs) {
                if (lane == 0) bulk_wait_group_read<kOutBufs - 1>();
                __syncwarp();
            }
            const uint32_t box = my_boxes + (nbox % kOutBufs) * kOutBox;
            // (checked builds: the box lies in the staging area; after a failed
            // check the warp stages into the first box instead -- in bounds, the
            // result is invalid and the status word says so)
            if (!tg_check(p.status, box >= sOut && box + kOutBox <= sOut + kOutStaging,
                          CHK_TC_STAGE, ew))
                return sOut;
            return box;
        };
        auto store_box = [&](uint32_t box, int x, int y, int z, bool in_range) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // (checked builds: x 16-byte aligned, no negative coordinate)
                if (in_range && tg_check(p.status,
                                         tma_x_aligned(x, f32_out ? 4 : 2) && x >= 0 && y >= 0,
                                         CHK_TC_STORE, quad)) {
                    if (p.batch > 1)
                        tma_store_3d(&tmC, box, x, y, z);
                    else
                        tma_store_2d(&tmC, box, x, y);
                }
                bulk_commit_group();
            }
            ++nbox;
        };
        uint32_t acc_count = 0;
        for (int w = unit0; w < total; w += unit_step) {
            const Work wk = decode_work(p, w, q);
            const uint32_t buf = NACC == 2 ? (acc_count & 1u) : 0u;
            const uint32_t acc_phase = NACC == 2 ? ((acc_count >> 1) & 1u) : (acc_count & 1u);
            const bool got = mbar_wait<PAIR>(tfull_bar(buf), acc_phase, p.timeout_ns, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) record_failure(p.status, 6, (ROLE_EPILOGUE << 16) | ew);
                *abort_flag = 1;
                break;
            }
            tc_fence_after_sync();
            const int wrow0 = wk.tm * Cfg::TILE_M + static_cast<int>(rank) * Cfg::CTA_M + quad * 32;
            const int row = wrow0 + lane;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * Cfg::ACC_STRIDE;
            const bool tma = p.c_tma != 0;
#pragma unroll 1
            for (int c0 = cbeg; c0 < cend; c0 += 32) {
                uint32_t r[32];
                // (checked builds: the columns lie in this accumulator buffer)
                if (!tg_check(p.status, c0 + 32 <= Cfg::ACC_STRIDE && buf < NACC, CHK_TC_TMEM, c0))
                    break;
                tmem_load_32cols_sync(taddr + c0, r);
                const int col = wk.tn * BN + c0;
                if (!tma) {
                    if (col < p.N) {
                        // wide per-row stores where C (or the partials) allow
                        // them, else one row at a time through the staging area
                        const bool wide = (p.splits > 1 ? (p.N & 3) == 0 : p.c_vector != 0) &&
                                          col + 32 <= p.N;
                        if (wide) {
                            if (row < p.M) store_chunk(p, wk.split, row, col, r, wk.z);
                        } else if (wrow0 < p.M) {
                            store_chunk_rows(p, wk.split, wrow0, col, lane, r, my_stg, wk.z);
                        }
                    }
                    continue;
                }
                const bool in_range = wrow0 < p.M && col < p.N;   // the box holds valid C
                if (p.epi.on && row < p.M && col < p.N)
                    epi_chunk32(p.epi, p.out_kind, row, col, min(32, p.N - col), r, wk.z);
                if (f32_out) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t box = next_box();
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            stage_chunk(box, lane, j, r[16 * half + 4 * j], r[16 * half + 4 * j + 1],
                                        r[16 * half + 4 * j + 2], r[16 * half + 4 * j + 3]);
                        store_box(box, col + 16 * half, wrow0, wk.z,
                                  in_range && col + 16 * half < p.N);
                    }
                } else {
                    const uint32_t box = next_box();
                    const bool bf = p.out_kind == OUT_BF16;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t h[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            h[t] = bf ? pack_bf162(r[8 * j + 2 * t], r[8 * j + 2 * t + 1])
                                      : pack_half2(r[8 * j + 2 * t], r[8 * j + 2 * t + 1]);
                        stage_chunk(box, lane, j, h[0], h[1], h[2], h[3]);
                    }
                    store_box(box, col, wrow0, wk.z, in_range);
                }
            }
            // every tcgen05.ld of this accumulator has completed (each waited):
            // hand the buffer back to the MMA issuer; the TMA stores still in
            // flight read shared memory only
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_cluster(tempty_bar(buf), pair_leader);
                else
                    mbar_arrive(tempty_bar(buf));
            }
            ++acc_count;
        }
        // the stores of this warp are complete (global writes done, staging
        // no longer read) before the CTA exits
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
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
cudaError_t launch_impl(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const TcParams &p, int ctas, cudaStream_t stream) {
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
    e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// 512-wide tiles exist for CTA pairs (every operand type).
template <int IN_KIND>
constexpr bool has_wide_tile() {
    return true;
}

template <int IN_KIND, bool PAIR, int MC>
cudaError_t launch_kind(int block_n, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const CUtensorMap &tmC, const TcParams &p, int ctas, cudaStream_t stream) {
    if constexpr (MC == 2 && PAIR) {
        switch (block_n) {
        case 192: return launch_impl<IN_KIND, 192, true, 2>(tmA, tmB, tmC, p, ctas, stream);
        case 224: return launch_impl<IN_KIND, 224, true, 2>(tmA, tmB, tmC, p, ctas, stream);
        case 256: return launch_impl<IN_KIND, 256, true, 2>(tmA, tmB, tmC, p, ctas, stream);
        default: return cudaErrorInvalidValue;
        }
    } else if constexpr (PAIR) {
        switch (block_n) {
        case 128: return launch_impl<IN_KIND, 128, true, 1>(tmA, tmB, tmC, p, ctas, stream);
        case 192: return launch_impl<IN_KIND, 192, true, 1>(tmA, tmB, tmC, p, ctas, stream);
        case 224: return launch_impl<IN_KIND, 224, true, 1>(tmA, tmB, tmC, p, ctas, stream);
        case 256: return launch_impl<IN_KIND, 256, true, 1>(tmA, tmB, tmC, p, ctas, stream);
        case 512:
            if constexpr (has_wide_tile<IN_KIND>())
                return launch_impl<IN_KIND, 512, true, 1>(tmA, tmB, tmC, p, ctas, stream);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
        }
    } else if constexpr (MC == 1) {
        switch (block_n) {
        case 128: return launch_impl<IN_KIND, 128, false, 1>(tmA, tmB, tmC, p, ctas, stream);
        case 192: return launch_impl<IN_KIND, 192, false, 1>(tmA, tmB, tmC, p, ctas, stream);
        case 224: return launch_impl<IN_KIND, 224, false, 1>(tmA, tmB, tmC, p, ctas, stream);
        case 256: return launch_impl<IN_KIND, 256, false, 1>(tmA, tmB, tmC, p, ctas, stream);
        default: return cudaErrorInvalidValue;
        }
    } else {
        return cudaErrorInvalidValue;
    }
}

template <int IN_KIND, bool PAIR>
int stages_kind(int block_n) {
    switch (block_n) {
    case 128: return TcCfg<IN_KIND, 128, PAIR>::STAGES;
    case 192: return TcCfg<IN_KIND, 192, PAIR>::STAGES;
    case 224: return TcCfg<IN_KIND, 224, PAIR>::STAGES;
    case 256: return TcCfg<IN_KIND, 256, PAIR>::STAGES;
    case 512:
        if constexpr (PAIR && has_wide_tile<IN_KIND>()) return TcCfg<IN_KIND, 512, true>::STAGES;
        return 0;
    default: return 0;
    }
}


// Kernel variants of one operand type: A-multicast pairs, pairs, single CTAs.
template <int IN_KIND>
cudaError_t launch_variant(int block_n, bool pair, int mc, const CUtensorMap &tmA,
                           const CUtensorMap &tmB, const CUtensorMap &tmC, const TcParams &p,
                           int ctas, cudaStream_t stream) {
    if (mc == 2)
        return pair ? launch_kind<IN_KIND, true, 2>(block_n, tmA, tmB, tmC, p, ctas, stream)
                    : cudaErrorInvalidValue;
    return pair ? launch_kind<IN_KIND, true, 1>(block_n, tmA, tmB, tmC, p, ctas, stream)
                : launch_kind<IN_KIND, false, 1>(block_n, tmA, tmB, tmC, p, ctas, stream);
}

}  // namespace
}  // namespace tg
