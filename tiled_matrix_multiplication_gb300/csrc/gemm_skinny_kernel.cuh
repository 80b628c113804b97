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
// K range).  After its main loop, and a cluster barrier, each CTA pushes the
// FP32 partial of every column straight from tensor memory to the CTA that
// owns the column -- CTA r owns columns [r*NT/S, (r+1)*NT/S) -- with
// asynchronous remote stores (st.async) into the owner's idle ring, and its
// own columns into its own ring with plain shared-memory stores (the remote
// stores run at about 40 GB/s per SM, so this saves 1/S of their time); the
// owner waits on one mbarrier for the peers' bytes, sums the S partials in
// K-range order, rounds once, stages the tile and writes C in 16-byte
// pieces.  No partials go to global memory and no second kernel runs; the sum
// order is fixed, so results do not depend on timing.  (Pulling the partials with remote loads instead cost one cluster
// round trip per few outputs: 5 to 10 us per call at 64 to 128 rows.)
//
// Roles: warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2..5 = TMEM epilogue (direct stores, or the pushes), and at 128 rows
// with two CTAs per SM warp 6 = a second TMA producer for a separate A^T
// ring; with one CTA per SM warps 6..15 wait for the K-split sum.  All warps
// then sum the received partials.  Every mbarrier wait is bounded
// (status word + abort flag, as in gemm_tc.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "tg_epilogue.cuh"
#include "tg_internal.h"
#include "tg_kernel_common.cuh"
#include "tg_ptx.cuh"

namespace tg {
namespace {

constexpr int kSmemBudget = 232448 - 1024 - 256;   // one CTA per SM (227 KB per CTA)
constexpr int kTwoSmemPerCta = 233472 / 2 - 1024;  // two per SM (228 KB, 1 KB each reserved)
constexpr int kSubN = 128;    // output columns per MMA (the MMA's M)

// TWO: a half-size ring so that two CTAs share an SM (twice the CTAs, and
// twice the independent TMA streams, for the same shared memory).
// SPLIT (128 rows, two per SM): A^T tiles are as large as B^T tiles there and
// only three (B^T, A^T) stage pairs would fit; separate rings -- 4 B^T stages
// from HBM, 3 A^T stages (L2 hits) with a producer warp of their own -- keep
// more of B in flight (measured 1 us faster per call at N = K = 8192).  The
// ring then starts at the 1024-byte aligned base of the dynamic area (no
// alignment pad; checked at run time).
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
    static constexpr bool SPLIT = TWO && MP == 128;
    // + the A^T producer warp when SPLIT; one CTA per SM: ten more warps,
    // idle until the K-split sum, where they add warps to that latency-bound
    // pass (2048 cells of 4 rows per CTA at 128 rows, S = 2)
    static constexpr int THREADS = SPLIT ? 224 : (TWO ? 192 : 512);
    static constexpr int PAD = SPLIT ? 0 : 1024;        // room to align the ring
    static constexpr int BUDGET =
        TWO ? (SPLIT ? kTwoSmemPerCta - 512 : 112 * 1024) : kSmemBudget;
    static constexpr int A_SPLIT = 3;                   // A^T stages when SPLIT
    static constexpr int FIT = SPLIT ? (BUDGET - A_SPLIT * AT_STAGE) / BT_STAGE
                                     : BUDGET / STAGE_BYTES;
    static constexpr int STAGES = FIT > 12 ? 12 : FIT;  // B^T stages (pairs unless SPLIT)
    static constexpr int A_STAGES = SPLIT ? A_SPLIT : STAGES;
    static constexpr int RING_BYTES = STAGES * BT_STAGE + A_STAGES * AT_STAGE;
    // received K-split partials: [K range][row group of 4][column][4 rows] FP32,
    // then the finished tile [row group][column][4 rows] in the output type
    static constexpr int G4 = MP / 4;
    static constexpr int RECV_BYTES = NT * MP * 4;
    static constexpr int OUT_STAGE_MAX = MP * (NT / 2) * 4;   // K split >= 2, FP32 out
    static constexpr int ACC_COLS = MP < 32 ? 32 : MP;  // TMEM columns per accumulator
    static constexpr int TMEM_COLS = SUB * ACC_COLS;
    // ring(s), TMEM full, partials received
    static constexpr int NUM_BARS = 2 * STAGES + (SPLIT ? 2 * A_STAGES : 0) + 2;
    static constexpr int SMEM_BYTES = PAD + RING_BYTES + NUM_BARS * 8 + 16;
    // A operand (B^T) N-major, B operand (A^T) K-major; M = 128, N = MP.
    static constexpr uint32_t IDESC =
        make_idesc(FMT, 1u, 0u, kSubN, MP);
    static_assert(BT_STAGE % 1024 == 0 && AT_STAGE % 1024 == 0,
                  "stages keep 1024-byte swizzle alignment");
    static_assert(RECV_BYTES + OUT_STAGE_MAX <= RING_BYTES,
                  "received partials and the output tile reuse the ring");
    static_assert(!TWO || SMEM_BYTES <= kTwoSmemPerCta, "two CTAs per SM");
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
__global__ void __launch_bounds__(SkCfg<IN_KIND, MP, NT, TWO>::THREADS, TWO ? 2 : 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const SkParams p) {
    using Cfg = SkCfg<IN_KIND, MP, NT, TWO>;
    constexpr int S = Cfg::STAGES;      // B^T stages
    constexpr int SA = Cfg::A_STAGES;   // A^T stages (== S unless SPLIT)
    constexpr bool SPLIT = Cfg::SPLIT;
    constexpr int kThreads = Cfg::THREADS;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    if (SPLIT && base != raw) {
        // no pad was reserved: the declared alignment must hold.  Every CTA of
        // the launch sees the same layout, so all of them (whole clusters)
        // return here and the call reports the failure.
        if (threadIdx.x == 0) record_failure(p.status, 4, ROLE_LAYOUT << 16);
        return;
    }
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sBt = base;                           // S x BT_STAGE
    const uint32_t sAt = base + S * Cfg::BT_STAGE;       // SA x AT_STAGE
    const uint32_t bars = sAt + SA * Cfg::AT_STAGE;
    uint8_t *gbars = gbase + (bars - base);
    // full / empty: the (B^T, A^T) stage pairs, or the B^T ring when SPLIT
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    // afull / aempty: the A^T ring when SPLIT
    constexpr int kABars = SPLIT ? 2 * SA : 0;
    auto afull_bar = [&](int s) { return bars + 8u * (2 * S + s); };
    auto aempty_bar = [&](int s) { return bars + 8u * (2 * S + SA + s); };
    const uint32_t tfull_bar = bars + 8u * (2 * S + kABars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbars + 8 * Cfg::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int &never_abort = *reinterpret_cast<int *>(tmem_slot + 2);
    // after the main loop the ring receives the K-split partials
    const uint32_t recv_base = base;
    const uint32_t recv_bar = bars + 8u * (2 * S + kABars + 1);
    bool epi_ok = true;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Cluster = the `splits` K ranges of one column tile; cluster rank = K range.
    const int splits = static_cast<int>(cluster_num_ctas());     // == p.splits
    const int split = static_cast<int>(cluster_cta_rank());
    const int tn = static_cast<int>(blockIdx.x) / splits;
    const int kt0 = split * p.k_tiles_per_split;
    const int kt1 = min(kt0 + p.k_tiles_per_split, p.k_tiles);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        if constexpr (SPLIT) {
            for (int s = 0; s < SA; ++s) {
                mbar_init(afull_bar(s), 1);
                mbar_init(aempty_bar(s), 1);
            }
        }
        mbar_init(tfull_bar, 1);
        mbar_init(recv_bar, 1);
        *abort_flag = 0;
        never_abort = 0;
        fence_mbar_init();
        // one phase: the peers' partials of this CTA's columns, rows rounded
        // up to 4 (pushed after the cluster barrier that follows the main loop)
        if (splits > 1)
            mbar_arrive_expect_tx(recv_bar, (NT - NT / splits) * 16 * ((min(p.M, MP) + 3) / 4));
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
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Prologue done: let the next kernel's prologue start, then wait for the
    // previous kernel's writes before the first global-memory access.
    if (threadIdx.x == 0) grid_launch_dependents();
    grid_dependency_wait();

    // A TMA producer thread fills its ring: waits for a free slot, announces
    // the slot's bytes, issues the loads; then waits for the loads it still
    // has in flight (the CTA may leave only after they have landed).  One
    // producer loads (B^T, A^T) stage pairs, or with SPLIT one per ring.
    auto produce = [&](bool with_a, bool with_b, int slots, uint32_t full0, uint32_t empty0,
                       uint32_t bytes, int tag) {
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        const int z = static_cast<int>(blockIdx.y);   // batch
        for (int kt = kt0; kt < kt1; ++kt) {
            if (!mbar_wait(empty0 + 8u * stage, phase ^ 1u, p.timeout_ns, abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t fb = full0 + 8u * stage;
            mbar_arrive_expect_tx(fb, bytes);
            // (checked builds: every box lies in its ring, x 16-byte aligned)
            const bool a_ok = tg_check(p.status,
                                       sAt + (stage + 1) * Cfg::AT_STAGE <= bars &&
                                           tma_x_aligned(kt * Cfg::BK, Cfg::ESIZE),
                                       CHK_SK_LOAD, stage);
            const bool b_ok = tg_check(p.status,
                                       sBt + (stage + 1) * Cfg::BT_STAGE <= sAt &&
                                           tma_x_aligned(tn * NT, Cfg::ESIZE),
                                       CHK_SK_LOAD, 0x100 | stage);
            if (with_a && a_ok) {
                if (p.a_batched) {
                    tma_load_3d(sAt + stage * Cfg::AT_STAGE, &tmA, fb, kt * Cfg::BK, 0, z);
                } else {
                    tma_load_2d(sAt + stage * Cfg::AT_STAGE, &tmA, fb, kt * Cfg::BK, 0);
                }
            }
            if (with_b && b_ok) {
#pragma unroll
                for (int j = 0; j < NT / Cfg::CHUNK_N; ++j) {
                    const uint32_t dst = sBt + stage * Cfg::BT_STAGE + j * Cfg::BT_BOX;
                    if (p.b_batched)
                        tma_load_3d(dst, &tmB, fb, tn * NT + j * Cfg::CHUNK_N, kt * Cfg::BK, z);
                    else
                        tma_load_2d(dst, &tmB, fb, tn * NT + j * Cfg::CHUNK_N, kt * Cfg::BK);
                }
            }
            ++issued;
            if (++stage == slots) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) {
            record_failure(p.status, 6, (ROLE_PRODUCER << 16) | tag | stage);
            *abort_flag = 1;
        }
        const int64_t first = issued > slots ? issued - slots : 0;
        for (int64_t i = first; i < issued; ++i) {
            if (!mbar_wait(full0 + 8u * static_cast<uint32_t>(i % slots),
                           static_cast<uint32_t>((i / slots) & 1), p.timeout_ns, &never_abort)) {
                record_failure(p.status, 6, (ROLE_DRAIN << 16) | tag | 1);
                break;
            }
        }
    };

    if (warp == 0) {
        // ------------------------------------- TMA producer: B^T (and A^T)
        if (lane == 0)
            produce(!SPLIT, true, S, full_bar(0), empty_bar(0),
                    SPLIT ? Cfg::BT_STAGE : Cfg::STAGE_BYTES, 0);
        __syncwarp();
    } else if (SPLIT && warp == 6) {
        // ----------------------------------- TMA producer: the A^T ring (L2)
        if (lane == 0) produce(true, false, SA, afull_bar(0), aempty_bar(0), Cfg::AT_STAGE, 0x100);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0, astage = 0;   // astage == stage unless SPLIT
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            for (int kt = kt0; kt < kt1; ++kt) {
                if (!mbar_wait(full_bar(stage), phase, p.timeout_ns, abort_flag) ||
                    (SPLIT && !mbar_wait(afull_bar(astage), aphase, p.timeout_ns, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t bt0 = sBt + stage * Cfg::BT_STAGE;
                const uint32_t at0 = sAt + astage * Cfg::AT_STAGE;
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
                // release the stage (and, with separate rings, the A^T slot)
                umma_commit(empty_bar(stage));
                if (SPLIT) umma_commit(aempty_bar(astage));
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++astage == SA) {
                    astage = 0;
                    aphase ^= 1u;
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
    } else if (warp < 6) {
        // ------------------------------------------- epilogue: wait for TMEM
        // Thread (quad, lane) owns column n = quad*32 + lane of each 128-column
        // accumulator.  Without a K split it writes C here; with one it pushes
        // its column to the owning CTA after the cluster barrier below.
        const int quad = warp & 3;
        const bool got = mbar_wait(tfull_bar, 0, p.timeout_ns, abort_flag);
        epi_ok = __all_sync(0xffffffffu, got);
        if (!epi_ok) {
            if (lane == 0) record_failure(p.status, 6, (ROLE_EPILOGUE << 16) | quad);
            *abort_flag = 1;
        } else if (splits == 1) {
            tc_fence_after_sync();
#pragma unroll 1
            for (int j = 0; j < Cfg::SUB; ++j) {
                const int n = tn * NT + j * kSubN + quad * 32 + lane;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                       j * Cfg::ACC_COLS;
                if constexpr (MP == 16) {
                    uint32_t r[16];
                    tmem_load_16cols_sync(taddr, r);
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (q < p.M && n < p.N) sk_store(p, q, n, __uint_as_float(r[q]));
                } else {
#pragma unroll 1
                    for (int c0 = 0; c0 < MP; c0 += 32) {
                        uint32_t r[32];
                        if (!tg_check(p.status, c0 + 32 <= Cfg::ACC_COLS, CHK_SK_TMEM, c0)) break;
                        tmem_load_32cols_sync(taddr + c0, r);
#pragma unroll
                        for (int q = 0; q < 32; ++q)
                            if (c0 + q < p.M && n < p.N)
                                sk_store(p, c0 + q, n, __uint_as_float(r[q]));
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (splits > 1) {
        // ------------------------ K-split reduction through distributed smem
        // CTA r of the K ranges owns columns [r*cols, (r+1)*cols) of the tile.
        // Each CTA pushes every other CTA's columns of its FP32 partial to
        // their owner with asynchronous remote stores into the owner's (now
        // idle) ring, and stores its own columns into its own ring; the owner
        // waits on one barrier for the peers' bytes, sums the S partials in
        // K-range order and writes C.
        cluster_sync_all();   // every ring of the cluster is idle from here on
        const int cols = NT / splits;
        const int push_groups = (min(p.M, MP) + 3) / 4;   // groups of 4 rows
        if (warp >= 2 && warp < 6 && epi_ok) {
            const int quad = warp & 3;
            tc_fence_after_sync();
#pragma unroll 1
            for (int j = 0; j < Cfg::SUB; ++j) {
                const int nl = j * kSubN + quad * 32 + lane;   // column within the tile
                const int owner = nl / cols;
                const int c = nl - owner * cols;
                const uint32_t rank = static_cast<uint32_t>(owner);
                const bool self = owner == split;   // this CTA's own columns
                // lanes hold consecutive columns: each push of a warp fills one
                // contiguous run of 16-byte (4-row) cells at the owner
                const uint32_t off =
                    recv_base + static_cast<uint32_t>((split * Cfg::G4 * cols + c) * 16);
                const uint32_t dst = self ? off : map_to_cta(off, rank);
                const uint32_t gstep = static_cast<uint32_t>(cols * 16);   // next row group
                const uint32_t rbar = map_to_cta(recv_bar, rank);
                // (checked builds: the column's cells lie in the receive area)
                if (!tg_check(p.status,
                              off >= recv_base &&
                                  off + gstep * (push_groups - 1) + 16 <= recv_base + Cfg::RECV_BYTES &&
                                  owner < splits,
                              CHK_SK_PUSH, nl))
                    continue;
                auto put = [&](uint32_t a, uint32_t x, uint32_t y, uint32_t zz, uint32_t w) {
                    if (self)
                        st_shared_v4(a, x, y, zz, w);
                    else
                        st_async_v4(a, x, y, zz, w, rbar);
                };
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                       j * Cfg::ACC_COLS;
                // only the groups of 4 rows that hold rows < M are sent
                if constexpr (MP == 16) {
                    uint32_t r[16];
                    tmem_load_16cols_sync(taddr, r);
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (g < push_groups)
                            put(dst + gstep * g, r[4 * g], r[4 * g + 1], r[4 * g + 2], r[4 * g + 3]);
                } else {
#pragma unroll 1
                    for (int c0 = 0; c0 < 4 * push_groups; c0 += 32) {
                        uint32_t r[32];
                        if (!tg_check(p.status, c0 + 32 <= Cfg::ACC_COLS, CHK_SK_TMEM, c0)) break;
                        tmem_load_32cols_sync(taddr + c0, r);
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            if (c0 / 4 + g < push_groups)
                                put(dst + gstep * (c0 / 4 + g), r[4 * g], r[4 * g + 1],
                                    r[4 * g + 2], r[4 * g + 3]);
                    }
                }
            }
        }
        const bool got = mbar_wait<true>(recv_bar, 0, p.timeout_ns, abort_flag);
        if (!got && !*abort_flag) {
            record_failure(p.status, 6, (ROLE_DRAIN << 16) | 4);
            *abort_flag = 1;
        }
        // Every push to this CTA has landed and its own pushes are issued: tell
        // the cluster, and wait for the others only before leaving (no CTA may
        // leave while a peer can still push to it).  Nothing is published
        // through this barrier -- the pushes are ordered by the receivers'
        // mbarriers -- so the arrive is relaxed and need not wait for them.
        tc_fence_before_sync();
        cluster_arrive_relaxed();
        __syncthreads();   // this CTA's own partial (plain stores) is visible
        // Sum the S partials of each (row group, column) cell in K-range order,
        // apply the epilogue, round, and write the cell's 4 rows to C.  Lanes
        // take consecutive cells (columns), so each load of a warp reads 512
        // contiguous bytes and each store writes 32 consecutive columns of one
        // row.
        const bool all_got = __syncthreads_and(got);
        const int n_base = tn * NT + split * cols;
        const int z = static_cast<int>(blockIdx.y);
        const int rows = min(p.M, MP);
        // (S a compile-time constant: a cell's S loads issue back to back)
        auto sum_write = [&](auto s_const) {
            constexpr int SS = decltype(s_const)::value;
            constexpr int COLS = NT / SS;
            for (int i = threadIdx.x; i < push_groups * COLS; i += kThreads) {
                const int g = i / COLS;
                const int c = i - g * COLS;
                const int n = n_base + c;
                // (checked builds: the cell's last partial lies in the receive area)
                if (!tg_check(p.status, ((SS - 1) * Cfg::G4 + g) * COLS + c < Cfg::RECV_BYTES / 16,
                              CHK_SK_SUM, i))
                    continue;
                float4 v[SS];
#pragma unroll
                for (int s = 0; s < SS; ++s)
                    v[s] = *reinterpret_cast<const float4 *>(gbase + ((s * Cfg::G4 + g) * COLS + c) * 16);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < SS; ++s) {
                    acc[0] += v[s].x;
                    acc[1] += v[s].y;
                    acc[2] += v[s].z;
                    acc[3] += v[s].w;
                }
                if (n >= p.N) continue;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int m = 4 * g + u;
                    if (m >= rows) break;
                    float x = acc[u];
                    if (p.epi.on) x = epi_one(p.epi, p.out_kind, m, n, x, z);
                    const int64_t off = static_cast<int64_t>(z) * p.stride_c +
                                        static_cast<int64_t>(m) * p.ldc + n;
                    if (p.out_kind == OUT_F32)
                        static_cast<float *>(p.c)[off] = x;
                    else if (p.out_kind == OUT_F16)
                        static_cast<__half *>(p.c)[off] = __float2half_rn(x);
                    else
                        static_cast<__nv_bfloat16 *>(p.c)[off] = __float2bfloat16_rn(x);
                }
            }
        };
        if (all_got) {
            switch (splits) {
            case 2: sum_write(std::integral_constant<int, 2>{}); break;
            case 4: sum_write(std::integral_constant<int, 4>{}); break;
            default: sum_write(std::integral_constant<int, 8>{}); break;
            }
        }
        cluster_wait();
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
    cfg.gridDim = dim3(static_cast<unsigned>(p.tiles_n * p.splits),
                       static_cast<unsigned>(p.batch > 0 ? p.batch : 1), 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.splits);
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
