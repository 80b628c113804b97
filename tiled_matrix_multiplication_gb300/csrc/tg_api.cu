// tg_api.cu -- host side of the C ABI declared in include/tg_gemm.h:
// argument validation, planning, TMA tensor maps, workspace and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "tg_gemm.h"
#include "tg_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kBlockM = 128;
constexpr int kDefaultGroupM = 8;
constexpr int kDefaultTimeoutMs = 2000;

struct DeviceState {
    bool init = false;
    tg_status arch = TG_OK;
    int sms = 0;
    int *status = nullptr;
    // The library's own stream-ordered memory pool for workspace.  Its release
    // threshold is unlimited, so memory freed at the end of a call is kept for
    // the next one instead of being unmapped and mapped again; the process's
    // default pool is left untouched.
    cudaMemPool_t pool = nullptr;
    int pair_slots = 0, quad_slots = 0;   // resident clusters of 2 / 4 CTAs
};

// Copy streams and events of the host-operand pipeline (tg_gemm_host), made
// once per device.  One call at a time uses them (the mutex), so an event is
// never re-recorded before the waits on it have been enqueued.
constexpr int kHostPanels = 16;
struct HostPipe {
    std::mutex mu;
    bool init = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, h2d_done = nullptr, done = nullptr;
    cudaEvent_t a_done[kHostPanels] = {}, c_done[kHostPanels] = {};
};
HostPipe g_pipe[64];

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int esize_of(tg_dtype t) { return t == TG_F32 ? 4 : (t == TG_E4M3 || t == TG_E5M2 ? 1 : 2); }

bool is_fp8(int t) { return t == TG_E4M3 || t == TG_E5M2; }

bool valid_dtype(int t) { return t == TG_F16 || t == TG_BF16 || t == TG_F32 || is_fp8(t); }

bool supported_pair(tg_dtype in, tg_dtype out) {
    if (in == TG_F16) return out == TG_F16 || out == TG_F32;
    if (in == TG_BF16) return out == TG_BF16 || out == TG_F32;
    if (in == TG_F32) return out == TG_F32;
    if (is_fp8(in)) return out == TG_F16 || out == TG_BF16 || out == TG_F32;
    return false;
}

int in_kind_of(tg_dtype t) {
    switch (t) {
    case TG_F16: return tg::IN_F16;
    case TG_BF16: return tg::IN_BF16;
    case TG_E4M3: return tg::IN_E4M3;
    case TG_E5M2: return tg::IN_E5M2;
    default: return tg::IN_TF32;
    }
}

int out_kind_of(tg_dtype t) {
    return t == TG_F16 ? tg::OUT_F16 : (t == TG_BF16 ? tg::OUT_BF16 : tg::OUT_F32);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// Byte span [lo, hi) touched by a rows x cols block with pitch ld.
void span(const void *p, int64_t rows, int64_t cols, int64_t ld, int esize, uintptr_t *lo,
          uintptr_t *hi) {
    *lo = reinterpret_cast<uintptr_t>(p);
    *hi = *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * esize);
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

struct Plan {
    tg_plan pub;
    int64_t k_tiles = 0, k_per_split = 0, tiles_m = 0, tiles_n = 0;
    int64_t lda_p = 0, ldb_p = 0;              // pitches after packing
    int64_t off_a = 0, off_b = 0, off_p = 0;   // workspace offsets
    int64_t off_tail = 0, off_cnt = 0;         // tail-split partials and counters
    int64_t tail_start = 0, tail_kps = 0;
    bool skinny_two = false;                   // small-M kernel: two CTAs per SM
    uint64_t timeout_ns = 0;
    int64_t stride_c = 0;                      // C batch stride (set before make_plan)
    int64_t k_eff = 0;                         // K of the kernel (3K for 3xTF32)
    bool valid = true;                         // false: no kernel variant fits the options
};

constexpr int64_t kMaxGridY = 65535;           // gridDim.y: one row per product (small M)

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

tg_status validate(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                   int64_t ldb, const void *c, int64_t ldc, int din, int dout,
                   const tg_options *opt) {
    if (!valid_dtype(din) || !valid_dtype(dout)) return TG_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return TG_ERR_INVALID_VALUE;
    if (lda < K || ldb < N || ldc < N) return TG_ERR_INVALID_VALUE;
    if (!supported_pair(static_cast<tg_dtype>(din), static_cast<tg_dtype>(dout)))
        return TG_ERR_UNSUPPORTED;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TG_ERR_UNSUPPORTED;
    if (lda > (int64_t(1) << 36) || ldb > (int64_t(1) << 36) || ldc > (int64_t(1) << 36))
        return TG_ERR_UNSUPPORTED;
    if (opt) {
        if (opt->multicast < 0 || opt->multicast > 2) return TG_ERR_INVALID_VALUE;
        if (opt->f32_mode < TG_F32_TF32 || opt->f32_mode > TG_F32_3XTF32 || opt->reserved != 0)
            return TG_ERR_INVALID_VALUE;
        if (opt->f32_mode == TG_F32_3XTF32 && (din != TG_F32 || 3 * K > kMaxDim))
            return TG_ERR_UNSUPPORTED;
        if (opt->multicast == 2) {
            const bool pair_ok = opt->path != TG_PATH_TC &&
                                 (!opt->block_n || tg::tc_supported_mc(opt->block_n, 2, true));
            const bool single_ok = opt->path != TG_PATH_TC_PAIR &&
                                   (!opt->block_n || tg::tc_supported_mc(opt->block_n, 2, false));
            if (opt->path == TG_PATH_SKINNY || opt->tail_splits || (!pair_ok && !single_ok))
                return TG_ERR_UNSUPPORTED;
        }
        if (opt->tail_splits < 0 || opt->tail_splits == 1 || opt->tail_splits > 8)
            return TG_ERR_INVALID_VALUE;
        if (opt->path < TG_PATH_AUTO || opt->path > TG_PATH_SKINNY) return TG_ERR_INVALID_VALUE;
        if (opt->splits < 0 || opt->block_n < 0 || opt->group_m < 0 || opt->max_ctas < 0 ||
            opt->timeout_ms < 0)
            return TG_ERR_INVALID_VALUE;
        if (opt->path == TG_PATH_SKINNY) {
            // C^T = B^T A^T with all rows in one tile: 16-bit or 8-bit operands,
            // M <= 128, K split over a cluster of 1, 2, 4 or 8 CTAs (none of
            // them empty), 128, 256 or 512 columns per CTA
            if (din == TG_F32 || M > 128) return TG_ERR_UNSUPPORTED;
            if (opt->block_n && !tg::skinny_supported(tg::skinny_rows(M), opt->block_n))
                return TG_ERR_UNSUPPORTED;
            const int64_t s = opt->splits;
            if (s != 0 && s != 1 && s != 2 && s != 4 && s != 8) return TG_ERR_UNSUPPORTED;
            const int64_t kt = std::max<int64_t>(cdiv(K, 128 / esize_of(static_cast<tg_dtype>(din))), 1);
            if (s > 1 && (s - 1) * cdiv(kt, s) >= kt) return TG_ERR_UNSUPPORTED;
        }
        if (opt->block_n && opt->path != TG_PATH_SKINNY) {
            const bool one = tg::tc_supported_block_n(opt->block_n, false);
            const bool two = tg::tc_supported_block_n(opt->block_n, true);
            if ((opt->path == TG_PATH_TC && !one) || (opt->path == TG_PATH_TC_PAIR && !two) ||
                (!one && !two))
                return TG_ERR_UNSUPPORTED;
        }
    }
    const int ei = esize_of(static_cast<tg_dtype>(din));
    const int eo = esize_of(static_cast<tg_dtype>(dout));
    if (M == 0 || N == 0) return TG_OK;
    if (c == nullptr) return TG_ERR_INVALID_VALUE;
    if (K > 0 && (a == nullptr || b == nullptr)) return TG_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(c) % eo) != 0) return TG_ERR_INVALID_VALUE;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(a) % ei) || (reinterpret_cast<uintptr_t>(b) % ei)))
        return TG_ERR_INVALID_VALUE;
    uintptr_t c0, c1;
    span(c, M, N, ldc, eo, &c0, &c1);
    if (K > 0) {
        uintptr_t a0, a1, b0, b1;
        span(a, M, K, lda, ei, &a0, &a1);
        span(b, K, N, ldb, ei, &b0, &b1);
        if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return TG_ERR_INVALID_VALUE;
    }
    return TG_OK;
}

// K ranges for each tile of a short last wave (1 = no tail split): at most
// `want`, no more than fill the idle slots, and at least 8 K tiles per range.
// (On GB300 the in-kernel sum of the partials currently costs more than the
// balanced wave saves, so the planner only splits a tail when asked to.)
int64_t tail_split_for(int64_t tiles, int64_t slots, int64_t k_tiles, int64_t want) {
    if (slots < 2 || want < 2) return 1;
    const int64_t tail = tiles % slots;
    if (tail == 0 || tail * 2 > slots) return 1;
    int64_t ts = std::min<int64_t>(want, slots / tail);
    ts = std::min<int64_t>(ts, k_tiles / 8);
    return std::max<int64_t>(ts, 1);
}

// `pair_slots` / `quad_slots`: clusters of 2 / 4 CTAs resident at once
// (0: estimate from the SM count).
// `batch` > 1: that many products with 16-byte aligned operands (no packing,
// no K split across kernels, no tail split) in one launch; the batch index is
// the slowest dimension of the work list.
void make_plan(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
               int64_t ldb, const void *c, int64_t ldc, tg_dtype din, tg_dtype dout, int num_sms,
               const tg_options *opt, Plan *pl, int pair_slots = 0, int quad_slots = 0,
               int64_t batch = 1) {
    tg_plan &p = pl->pub;
    std::memset(&p, 0, sizeof(p));
    const int ei = esize_of(din), eo = esize_of(dout);
    const int align_elems = 16 / ei;
    num_sms = std::max(num_sms, 1);
    p.block_k = 128 / ei;
    p.group_m = (opt && opt->group_m) ? opt->group_m : kDefaultGroupM;
    // 3xTF32: the kernel contracts the split operands over K' = 3K
    const bool x3 = din == TG_F32 && opt && opt->f32_mode == TG_F32_3XTF32;
    pl->k_eff = x3 ? 3 * K : K;
    pl->k_tiles = std::max<int64_t>(cdiv(pl->k_eff, p.block_k), 1);
    const int64_t cap = (opt && opt->max_ctas) ? opt->max_ctas : num_sms;

    // Choose the kernel variant (single CTA with a 128-row tile, or CTA pair
    // with a 256-row tile), the tile width and the K split by a simple time
    // model.  Every CTA (pair) runs about units / slots work units one after
    // the other; a unit costs (tile width x K tiles) divided by the measured
    // relative efficiency of the variant; under a split each unit also writes
    // an FP32 partial tile that a second kernel sums (about 24 K tiles' worth
    // for 128 rows, less for fewer rows).  Ties go to the earlier candidate.
    // Relative efficiencies (percent of the best variant) measured on GB300 at
    // 8192^3 and on the prefill shapes; single-CTA clusters sharing A measured
    // about 5 % slower than unshared single CTAs at 128 to 2048 rows.
    // mc = 2: clusters of two pairs (or two single CTAs) sharing A by multicast
    // (two tiles per unit).
    struct Cand { bool pair; int mc; int bn; int eff; };
    static const Cand kCands[] = {
        {true, 2, 256, 105}, {true, 1, 256, 100}, {true, 2, 224, 90}, {true, 2, 192, 86},
        {true, 1, 224, 92}, {true, 1, 192, 84}, {false, 1, 256, 90}, {false, 2, 256, 85},
        {false, 1, 192, 82}, {false, 1, 224, 80}, {false, 1, 128, 62}, {true, 1, 128, 62},
        {false, 2, 128, 58}};
    // At most 128 rows the product streams B (memory-bound): single-CTA tiles
    // 128 wide, with the K split below, measured fastest (pair tiles would be
    // half empty; wider tiles give fewer concurrent streams).
    const bool few_rows = M <= kBlockM && !(opt && (opt->block_n || opt->multicast ||
                                                     opt->path == TG_PATH_TC_PAIR));
    double best_cost = -1.0;
    for (const Cand &cd : kCands) {
        if (few_rows && (cd.pair || cd.mc != 1 || cd.bn != 128)) continue;
        if (opt && opt->path == TG_PATH_TC && cd.pair) continue;
        if (opt && opt->path == TG_PATH_TC_PAIR && !cd.pair) continue;
        if (opt && opt->block_n && opt->block_n != cd.bn) continue;
        const int64_t cl = (cd.pair ? 2 : 1) * cd.mc;   // CTAs per cluster
        if (cap < cl) continue;
        if (opt && opt->multicast && opt->multicast != cd.mc) continue;
        if (cd.mc == 2 && opt && opt->tail_splits) continue;
        const int64_t tile_m = cd.pair ? 2 * kBlockM : kBlockM;
        // resident clusters: 4-CTA clusters can leave SMs of a GPC unused
        int64_t resident = cap;
        if (cl > 1) {
            // without a device: 4-CTA clusters measured at 36 on 152 SMs
            const int64_t est = cl == 4 ? (quad_slots ? quad_slots : num_sms * 19 / 80)
                                        : (pair_slots ? pair_slots : num_sms / 2);
            resident = std::min<int64_t>(cap / cl, est);
        }
        const int64_t slots = std::max<int64_t>(1, resident);
        // work units: tiles, or pairs of horizontally adjacent tiles
        const int64_t tiles = cdiv(M, tile_m) * cdiv(cdiv(N, cd.bn), cd.mc) * batch;
        int64_t s_lo = 1, s_hi = 1;
        if (opt && opt->splits && batch == 1) {
            s_lo = s_hi = opt->splits;
        } else if (tiles < slots / 2 && batch == 1) {
            s_hi = std::min<int64_t>(pl->k_tiles, 16);   // too few tiles: consider split K
        }
        for (int64_t s = s_lo; s <= s_hi; ++s) {
            const int64_t sc = std::max<int64_t>(1, std::min<int64_t>(s, pl->k_tiles));
            const int64_t kps = cdiv(pl->k_tiles, sc);
            const int64_t se = cdiv(pl->k_tiles, kps);   // no empty split
            const int64_t units = tiles * se;
            // Fractional waves, with the idle part of a partial last wave charged
            // at a quarter: fewer busy CTAs run faster (less contention for L2
            // bandwidth and power), so an idle slot costs less than a busy one.
            const double used = static_cast<double>(units) / static_cast<double>(std::max<int64_t>(1, std::min(units, slots)));
            double waves = units > 0 ? used + 0.25 * (static_cast<double>(cdiv(units, std::min(units, slots))) - used) : 0.0;
            // A requested tail split (below) turns a short last wave into 1/ts
            // of a wave plus the partials' round trip.
            if (se == 1 && opt && opt->tail_splits && !opt->splits && batch == 1) {
                const int64_t ts = tail_split_for(tiles, slots, pl->k_tiles, opt->tail_splits);
                if (ts > 1) waves = static_cast<double>(tiles / slots) + 1.15 / static_cast<double>(ts);
            }
            const int64_t rows = std::min<int64_t>(M, kBlockM);
            const int64_t partial = se > 1 ? std::max<int64_t>(1, 24 * rows / kBlockM) : 0;
            const double cost =
                waves * static_cast<double>(cd.bn * (kps + partial)) * 100.0 / cd.eff;
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                p.path = cd.pair ? TG_PATH_TC_PAIR : TG_PATH_TC;
                p.block_m = static_cast<int32_t>(tile_m);
                p.block_n = cd.bn;
                p.multicast = cd.mc;
                pl->k_per_split = kps;
                p.splits = static_cast<int32_t>(se);
                p.tiles = tiles;
            }
        }
    }
    // Small M with 16-bit operands: the transposed streaming kernel (one tile
    // holds all rows; work is spread over 128-column tiles and K splits).
    const bool forced_skinny = opt && opt->path == TG_PATH_SKINNY;
    // The transposed streaming kernel wins for up to 64 rows of 16-bit operands
    // and up to 32 of FP8 ones; beyond that (to 128 rows, where it can still
    // be forced) the tile kernel with a K split measured faster on GB300
    // (M = 128, N = K = 8192: FP16 35.0 vs 39.0 us, E4M3 23.7 vs 29.6 us).
    const int64_t skinny_rows_max = forced_skinny ? 128 : (is_fp8(din) ? 32 : 64);
    const bool skinny_ok = din != TG_F32 && M <= skinny_rows_max &&
                           (forced_skinny || !(opt && opt->block_n)) &&
                           !(opt && (opt->path == TG_PATH_TC || opt->path == TG_PATH_TC_PAIR)) &&
                           batch <= kMaxGridY;
    if (skinny_ok) {
        // One CTA per (128-column tile, K range); the K ranges of a tile form a
        // cluster of 1, 2, 4 or 8 CTAs that sums its partials on chip.  Take the
        // largest cluster that keeps every CTA resident at once (and every K
        // range non-empty): the kernel streams B, so more CTAs means more bytes
        // in flight.
        const int64_t ktiles = std::max<int64_t>(cdiv(K, 128 / ei), 1);   // 128-byte K rows
        const int mp = tg::skinny_rows(M);
        // 128 columns per CTA by default: on GB300 wider tiles (256, 512: longer
        // contiguous runs of B, fewer re-reads of A) measured no faster at
        // M <= 64 and slower at M = 128; they remain selectable.
        const int nt = (opt && opt->block_n) ? opt->block_n : 128;
        // (with a batch, one grid row of tiles x K ranges per product)
        const int64_t tiles = cdiv(N, nt) * batch;
        int64_t best_s = 1;
        // a batch with more CTAs than SMs even unsplit: two CTAs per SM
        bool two = batch > 1 && nt == 128 && tiles > cap;
        for (int64_t sc : {2, 4, 8}) {
            const int64_t kps = cdiv(ktiles, sc);
            if ((sc - 1) * kps >= ktiles) continue;          // a K range would be empty
            if (opt && opt->splits && opt->splits != sc) continue;
            if (tiles * sc <= cap) {
                best_s = sc;
                two = false;
            } else if (nt == 128 && tiles * sc <= 2 * cap) {
                // more CTAs than SMs: two half-size CTAs per SM keep them all
                // resident (measured faster than one full-size CTA per SM for
                // every M from 1 to 128 at N = K = 8192)
                best_s = sc;
                two = true;
                break;
            }
        }
        if (opt && opt->splits) {
            best_s = opt->splits;                            // validated in validate()
            two = nt == 128 && tiles * best_s > cap;
        }
        pl->skinny_two = two;
        p.path = TG_PATH_SKINNY;
        p.block_m = mp;
        p.block_n = nt;
        p.block_k = 128 / ei;
        p.splits = static_cast<int32_t>(best_s);
        p.tiles = tiles;
        pl->k_tiles = ktiles;
        pl->k_per_split = cdiv(ktiles, best_s);
    }
    if (best_cost < 0 && p.path != TG_PATH_SKINNY) {
        // the options exclude every variant (e.g. a CTA budget below one
        // cluster of the forced variant): nothing to launch
        pl->valid = false;
        return;
    }
    const bool pair = p.path == TG_PATH_TC_PAIR;
    p.stages = p.path == TG_PATH_SKINNY ? tg::skinny_stages(p.block_m, p.block_n, pl->skinny_two)
                                         : tg::tc_stages(in_kind_of(din), p.block_n, pair);
    pl->tiles_m = cdiv(M, p.block_m);
    pl->tiles_n = cdiv(N, p.block_n);
    const int64_t splits = p.splits;
    const int64_t units = p.tiles * splits;   // (tiles = work units: tile pairs when mc = 2)
    if (p.path == TG_PATH_SKINNY) {
        p.ctas = static_cast<int32_t>(units);   // not persistent: one CTA per unit
        p.multicast = 1;
    } else if (pair || p.multicast == 2) {
        const int64_t cl = (pair ? 2 : 1) * std::max(p.multicast, 1);
        int64_t resident = cap / cl;
        if (cl == 4) resident = std::min<int64_t>(resident, quad_slots ? quad_slots : num_sms * 19 / 80);
        else resident = std::min<int64_t>(resident, pair_slots ? pair_slots : num_sms / 2);
        const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(units, resident));
        p.ctas = static_cast<int32_t>(cl * clusters);
    } else {
        p.ctas = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(units, cap)));
    }
    p.pack_a = !(aligned16(a) && (lda * ei) % 16 == 0);
    p.pack_b = !(aligned16(b) && (ldb * ei) % 16 == 0);
    if (din == TG_F32) p.pack_b = 2;   // kind::tf32 reads B K-major: B^T into the workspace
    if (x3) p.pack_a = p.pack_b = 3;   // hi / lo TF32 parts of A and of B^T
    p.c_vector = aligned16(c) && (ldc * eo) % 16 == 0 && (batch == 1 || (pl->stride_c * eo) % 16 == 0);
    pl->lda_p = p.pack_a ? round_up(pl->k_eff, align_elems) : lda;
    pl->ldb_p = p.pack_b >= 2 ? round_up(pl->k_eff, align_elems)
                              : (p.pack_b ? round_up(N, align_elems) : ldb);
    int64_t ws = 0;
    if (p.pack_a) {
        pl->off_a = ws;
        ws = round_up(ws + M * pl->lda_p * ei, 256);
    }
    if (p.pack_b) {
        pl->off_b = ws;
        ws = round_up(ws + (p.pack_b >= 2 ? N : K) * pl->ldb_p * ei, 256);
    }
    const bool global_partials = splits > 1 && p.path != TG_PATH_SKINNY;
    if (global_partials) {
        pl->off_p = ws;
        ws = round_up(ws + splits * M * N * 4, 256);
    }
    // Tail split of the tensor-core paths (auto plans without a K split).
    if (p.path != TG_PATH_SKINNY && splits == 1 && opt && opt->tail_splits && !opt->splits &&
        batch == 1) {
        const int64_t slots = pair ? std::max<int64_t>(1, cap / 2) : std::max<int64_t>(1, cap);
        const int64_t ts = tail_split_for(p.tiles, slots, pl->k_tiles, opt->tail_splits);
        if (ts > 1) {
            p.tail_tiles = static_cast<int32_t>(p.tiles % slots);
            pl->tail_start = p.tiles - p.tail_tiles;
            pl->tail_kps = cdiv(pl->k_tiles, ts);
            p.tail_splits = static_cast<int32_t>(cdiv(pl->k_tiles, pl->tail_kps));
            const int64_t cta_group = pair ? 2 : 1;
            pl->off_tail = ws;
            ws = round_up(ws + static_cast<int64_t>(p.tail_tiles) * p.tail_splits * p.block_m *
                                   p.block_n * 4, 256);
            pl->off_cnt = ws;
            ws = round_up(ws + static_cast<int64_t>(p.tail_tiles) * cta_group * 4, 256);
            if (pair) {
                const int64_t pairs = std::max<int64_t>(
                    1, std::min<int64_t>(pl->tail_start + p.tail_tiles * p.tail_splits, cap / 2));
                p.ctas = static_cast<int32_t>(2 * pairs);
            } else {
                p.ctas = static_cast<int32_t>(std::max<int64_t>(
                    1, std::min<int64_t>(pl->tail_start + p.tail_tiles * p.tail_splits, cap)));
            }
        }
    }
    p.workspace_bytes = ws;
    p.kernels = (p.pack_a ? 1 : 0) + (p.pack_b ? 1 : 0) + 1 + (global_partials ? 1 : 0);
    const int tmo = (opt && opt->timeout_ms) ? opt->timeout_ms : kDefaultTimeoutMs;
    pl->timeout_ns = static_cast<uint64_t>(tmo) * 1000000ull;
}

tg_status init_encoder() {
    if (g_encode) return TG_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return TG_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return TG_OK;
}

tg_status device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TG_ERR_CUDA;
        d.sms = sms;
        d.arch = (major == 10 && minor == 3) ? TG_OK : TG_ERR_ARCH;
        if (d.arch == TG_OK) {
            if (tg::status_word_address(&d.status) != cudaSuccess) return TG_ERR_CUDA;
            if (init_encoder() != TG_OK) return TG_ERR_CUDA;
            cudaMemPoolProps props;
            std::memset(&props, 0, sizeof(props));
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) return TG_ERR_CUDA;
            uint64_t keep = ~0ull;
            if (cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess)
                return TG_ERR_CUDA;
            d.pair_slots = tg::tc_max_clusters(2);
            d.quad_slots = tg::tc_max_clusters(4);
        }
        d.init = true;
    }
    *out = &d;
    return d.arch;
}

CUtensorMapDataType tma_type(tg_dtype t) {
    if (is_fp8(t)) return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // bytes moved as they are
    return t == TG_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                       : (t == TG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

// Row-major [rows, cols] with pitch `ld` elements; boxes of box_cols x box_rows
// whose rows (box_cols * esize bytes = 128, 64 or 32) are swizzled at that
// size; zero fill out of range.  With nb > 1 the map has a third dimension of
// nb matrices `stride` elements apart (boxes one matrix deep).
tg_status encode_2d(CUtensorMap *map, tg_dtype t, const void *ptr, int64_t rows, int64_t cols,
                    int64_t ld, int box_cols, int box_rows, int64_t nb = 1, int64_t stride = 0) {
    const int row_bytes = box_cols * esize_of(t);
    const CUtensorMapSwizzle sw = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : row_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_32B;
    const cuuint32_t rank = nb > 1 ? 3 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(nb)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * esize_of(t)),
                                   static_cast<cuuint64_t>(stride * esize_of(t))};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows),
                               1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, tma_type(t), rank, const_cast<void *>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TG_OK : TG_ERR_CUDA;
}

tg_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return TG_OK;
    if (e == cudaErrorMemoryAllocation) return TG_ERR_OUT_OF_MEMORY;
    return TG_ERR_CUDA;
}

// Products of one launch: `count` of them, whose A / B / C start sa / sb / sc
// elements apart (sa or sb == 0: one operand shared by every product).
struct Batch {
    int64_t count = 1, sa = 0, sb = 0, sc = 0;
};

// Enqueues one validated product with M, N, K > 0 -- or, with bt.count > 1,
// that many products in one launch (16-bit operands that need no packing).
// A tensor map the driver rejects for a batch sets *map_failed before
// anything is enqueued, so the caller can run the products one by one.
tg_status enqueue(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                  int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in, tg_dtype dtype_out,
                  cudaStream_t s, const tg_options *opt, DeviceState *dev, const Batch &bt,
                  bool *map_failed, const tg::EpiParams *epi = nullptr) {
    tg_status st = TG_OK;
    Plan pl;
    pl.stride_c = bt.sc;
    make_plan(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, dev->sms, opt, &pl,
              dev->pair_slots, dev->quad_slots, bt.count);
    if (!pl.valid) return TG_ERR_UNSUPPORTED;
    const tg_plan &p = pl.pub;
    const int ei = esize_of(dtype_in);
    const bool batched = bt.count > 1;
    // operands that differ per product get a rank-3 map; a shared one (stride 0) stays 2-D
    const int64_t nb_a = batched && bt.sa ? bt.count : 1;
    const int64_t nb_b = batched && bt.sb ? bt.count : 1;
    auto map_error = [&]() {
        if (batched && map_failed) *map_failed = true;
        return TG_ERR_CUDA;
    };

    uint8_t *ws = nullptr;
    if (p.workspace_bytes > 0) {
        cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), p.workspace_bytes,
                                                dev->pool, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    auto fail = [&](tg_status code) {
        if (ws) cudaFreeAsync(ws, s);
        return code;
    };
    const void *A = a;
    const void *B = b;
    if (p.pack_a) {
        A = ws + pl.off_a;
        st = cuda_status(p.pack_a == 3
                             ? tg::launch_split3_rows(a, lda, ws + pl.off_a, pl.lda_p, M, K, s)
                             : tg::launch_pack_rows(a, lda, ws + pl.off_a, pl.lda_p, M, K, ei, s));
        if (st != TG_OK) return fail(st);
    }
    if (p.pack_b) {
        B = ws + pl.off_b;
        st = cuda_status(
            p.pack_b == 3 ? tg::launch_split3_transpose(b, ldb, ws + pl.off_b, pl.ldb_p, K, N, s)
            : p.pack_b == 2
                ? tg::launch_pack_transpose(b, ldb, ws + pl.off_b, pl.ldb_p, K, N, ei, s)
                : tg::launch_pack_rows(b, ldb, ws + pl.off_b, pl.ldb_p, K, N, ei, s));
        if (st != TG_OK) return fail(st);
    }
    const int64_t Ke = pl.k_eff;   // K of the kernel's operands
    CUtensorMap tmA, tmB;
    const int chunk = 128 / ei;
    if (p.path == TG_PATH_SKINNY) {
        if (encode_2d(&tmA, dtype_in, A, M, K, pl.lda_p, p.block_k, p.block_m, nb_a, bt.sa) != TG_OK ||
            encode_2d(&tmB, dtype_in, B, K, N, pl.ldb_p, chunk, p.block_k, nb_b, bt.sb) != TG_OK)
            return fail(map_error());
        tg::SkParams sp;
        std::memset(&sp, 0, sizeof(sp));
        sp.M = static_cast<int32_t>(M);
        sp.N = static_cast<int32_t>(N);
        sp.K = static_cast<int32_t>(K);
        sp.tiles_n = static_cast<int32_t>(pl.tiles_n);
        sp.k_tiles = static_cast<int32_t>(pl.k_tiles);
        sp.k_tiles_per_split = static_cast<int32_t>(pl.k_per_split);
        sp.splits = p.splits;
        sp.out_kind = out_kind_of(dtype_out);
        sp.ldc = ldc;
        sp.c = c;
        sp.status = dev->status;
        sp.timeout_ns = pl.timeout_ns;
        sp.two_per_sm = pl.skinny_two ? 1 : 0;
        sp.batch = static_cast<int32_t>(bt.count);
        sp.a_batched = nb_a > 1;
        sp.b_batched = nb_b > 1;
        sp.stride_c = bt.sc;
        if (epi) sp.epi = *epi;
        st = cuda_status(
            tg::launch_gemm_skinny(in_kind_of(dtype_in), p.block_m, p.block_n, tmA, tmB, sp, s));
        if (st != TG_OK) return fail(st);
        if (ws && cudaFreeAsync(ws, s) != cudaSuccess) return TG_ERR_CUDA;
        return TG_OK;
    }
    const bool pair = p.path == TG_PATH_TC_PAIR;
    const int bn_cta = pair ? p.block_n / 2 : p.block_n;   // B columns staged per CTA
    const int b_chunk = tg::tc_b_swizzle_bytes(in_kind_of(dtype_in), p.block_n, pair) / ei;
    const tg_status sb = p.pack_b >= 2
                             ? encode_2d(&tmB, dtype_in, B, N, Ke, pl.ldb_p, p.block_k, bn_cta)
                             : encode_2d(&tmB, dtype_in, B, K, N, pl.ldb_p, b_chunk, p.block_k,
                                         nb_b, bt.sb);
    // with A multicast each CTA loads half of its 128 rows of A
    const int a_rows = p.multicast == 2 ? kBlockM / 2 : kBlockM;
    if (encode_2d(&tmA, dtype_in, A, M, Ke, pl.lda_p, p.block_k, a_rows, nb_a, bt.sa) != TG_OK ||
        sb != TG_OK)
        return fail(map_error());

    tg::TcParams tp;
    std::memset(&tp, 0, sizeof(tp));
    tp.M = static_cast<int32_t>(M);
    tp.N = static_cast<int32_t>(N);
    tp.K = static_cast<int32_t>(Ke);
    tp.tiles_m = static_cast<int32_t>(pl.tiles_m);
    tp.tiles_n = static_cast<int32_t>(pl.tiles_n);
    tp.k_tiles = static_cast<int32_t>(pl.k_tiles);
    tp.k_tiles_per_split = static_cast<int32_t>(pl.k_per_split);
    tp.splits = p.splits;
    tp.group_m = p.group_m;
    tp.out_kind = out_kind_of(dtype_out);
    tp.c_vector = p.c_vector;
    tp.mc = std::max(p.multicast, 1);
    tp.ldc = ldc;
    tp.c = c;
    tp.partial = p.splits > 1 ? reinterpret_cast<float *>(ws + pl.off_p) : nullptr;
    tp.status = dev->status;
    tp.timeout_ns = pl.timeout_ns;
    tp.batch = static_cast<int32_t>(bt.count);
    tp.a_batched = nb_a > 1;
    tp.b_batched = nb_b > 1;
    tp.stride_c = bt.sc;
    // with a K split the epilogue runs where the partials are summed
    if (epi && p.splits == 1) tp.epi = *epi;
    if (p.tail_tiles > 0) {
        tp.tail_start = static_cast<int32_t>(pl.tail_start);
        tp.tail_tiles = p.tail_tiles;
        tp.tail_splits = p.tail_splits;
        tp.tail_kps = static_cast<int32_t>(pl.tail_kps);
        tp.tail_partial = reinterpret_cast<float *>(ws + pl.off_tail);
        tp.tail_count = reinterpret_cast<unsigned int *>(ws + pl.off_cnt);
        const size_t cnt_bytes = static_cast<size_t>(p.tail_tiles) * (pair ? 2 : 1) * 4;
        st = cuda_status(cudaMemsetAsync(tp.tail_count, 0, cnt_bytes, s));
        if (st != TG_OK) return fail(st);
    }
    st = cuda_status(tg::launch_gemm_tc(in_kind_of(dtype_in), p.block_n, pair,
                                        std::max(p.multicast, 1), tmA, tmB, tp, p.ctas, s));
    if (st != TG_OK) return fail(st);
    if (p.splits > 1) {
        st = cuda_status(tg::launch_splitk_reduce(tp.partial, p.splits, M, N, c, ldc,
                                                  tp.out_kind, p.c_vector, s, epi));
        if (st != TG_OK) return fail(st);
    }
    if (ws) {
        if (cudaFreeAsync(ws, s) != cudaSuccess) return TG_ERR_CUDA;
    }
    return TG_OK;
}

// Argument rules of tg_gemm_strided_batched on top of those of one product.
tg_status validate_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void *a,
                           int64_t lda, int64_t sa, const void *b, int64_t ldb, int64_t sb,
                           const void *c, int64_t ldc, int64_t sc, int din, int dout,
                           const tg_options *opt) {
    if (batch < 0 || sa < 0 || sb < 0 || sc < 0) return TG_ERR_INVALID_VALUE;
    const tg_status v = validate(M, N, K, a, lda, b, ldb, c, ldc, din, dout, opt);
    if (v != TG_OK) return v;
    if (batch > kMaxDim) return TG_ERR_UNSUPPORTED;
    if (batch > 1 && opt) {
        if (opt->tail_splits) return TG_ERR_UNSUPPORTED;
        if (opt->splits > 1 && opt->path != TG_PATH_SKINNY) return TG_ERR_UNSUPPORTED;
    }
    if (batch <= 1 || M == 0 || N == 0) return TG_OK;
    const int64_t lim = int64_t(1) << 46;   // elements spanned by the batch strides
    for (const int64_t st : {sa, sb, sc})
        if (st > 0 && batch - 1 > lim / st) return TG_ERR_UNSUPPORTED;
    if (cdiv(M, 128) * cdiv(N, 128) > (int64_t(1) << 30) / batch) return TG_ERR_UNSUPPORTED;
    // the products' C blocks must be disjoint: stacked, or interleaved along rows
    const int64_t span_c = (M - 1) * ldc + N;
    const bool stacked = sc >= span_c;
    const bool interleaved = sc >= N && (batch - 1) * sc + N <= ldc;
    if (!stacked && !interleaved) return TG_ERR_INVALID_VALUE;
    if (K > 0) {
        const int ei = esize_of(static_cast<tg_dtype>(din));
        const int eo = esize_of(static_cast<tg_dtype>(dout));
        auto range = [](const void *p, int64_t elems, int es, uintptr_t *lo, uintptr_t *hi) {
            *lo = reinterpret_cast<uintptr_t>(p);
            *hi = *lo + static_cast<uintptr_t>(elems * es);
        };
        uintptr_t a0, a1, b0, b1, c0, c1;
        range(a, (batch - 1) * sa + (M - 1) * lda + K, ei, &a0, &a1);
        range(b, (batch - 1) * sb + (K - 1) * ldb + N, ei, &b0, &b1);
        range(c, (batch - 1) * sc + span_c, eo, &c0, &c1);
        if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return TG_ERR_INVALID_VALUE;
    }
    return TG_OK;
}

// One launch for the whole batch: 16-bit operands read in place (16-byte
// aligned base, row pitch and batch stride; strides within the TMA limit).
bool batch_in_one_launch(tg_dtype din, const void *a, int64_t lda, int64_t sa, const void *b,
                         int64_t ldb, int64_t sb) {
    if (din == TG_F32) return false;
    const int ei = esize_of(din);
    auto ok = [&](const void *p, int64_t ld, int64_t st) {
        return aligned16(p) && (ld * ei) % 16 == 0 && (st * ei) % 16 == 0 &&
               st * ei < (int64_t(1) << 40);
    };
    return ok(a, lda, sa) && ok(b, ldb, sb);
}

// Argument rules of the fused epilogue (on top of those of the product);
// fills *e for the kernels.
tg_status validate_epilogue(int64_t M, int64_t N, const void *c, int64_t ldc, tg_dtype dout,
                            const tg_epilogue *ep, tg::EpiParams *e) {
    std::memset(e, 0, sizeof(*e));
    if (ep == nullptr) return TG_OK;
    if (ep->activation < TG_ACT_NONE || ep->activation > TG_ACT_GELU_TANH || ep->reserved != 0)
        return TG_ERR_INVALID_VALUE;
    const int eo = esize_of(dout);
    e->on = 1;
    e->act = ep->activation;
    e->alpha = ep->alpha;
    e->beta = ep->beta;
    e->scale = ep->scale;
    e->bias = ep->bias;
    e->res = ep->residual;
    e->ldr = ep->residual ? ep->ldr : 0;
    if (M == 0 || N == 0) return TG_OK;
    uintptr_t c0, c1;
    span(c, M, N, ldc, eo, &c0, &c1);
    for (const float *v : {ep->scale, ep->bias}) {
        if (v == nullptr) continue;
        if (reinterpret_cast<uintptr_t>(v) % 4) return TG_ERR_INVALID_VALUE;
        const uintptr_t v0 = reinterpret_cast<uintptr_t>(v);
        if (overlaps(c0, c1, v0, v0 + static_cast<uintptr_t>(N) * 4)) return TG_ERR_INVALID_VALUE;
    }
    if (ep->residual) {
        if (ep->ldr < N || ep->ldr > (int64_t(1) << 36)) return TG_ERR_INVALID_VALUE;
        if (reinterpret_cast<uintptr_t>(ep->residual) % eo) return TG_ERR_INVALID_VALUE;
        const bool in_place = ep->residual == c && ep->ldr == ldc;
        uintptr_t r0, r1;
        span(ep->residual, M, N, ep->ldr, eo, &r0, &r1);
        if (!in_place && overlaps(c0, c1, r0, r1)) return TG_ERR_INVALID_VALUE;
        e->res_vector = aligned16(ep->residual) && (ep->ldr * eo) % 16 == 0;
    }
    e->sb_vector = (!ep->scale || aligned16(ep->scale)) && (!ep->bias || aligned16(ep->bias));
    return TG_OK;
}

// Rows per panel of the host-operand pipeline: at least 1024 (four rows of
// pair tiles, so a panel still fills the GPU without a K split), at most
// kHostPanels panels.  Measured on GB300 at 4096^3 (host link about 200 GB/s
// each way): 4 panels of 1024 rows beat 1, 2, 8 and 16 panels; at 8192^3, 8
// panels of 1024 rows.
int64_t host_panel_rows(int64_t M) {
    return std::max<int64_t>(1024, round_up(cdiv(M, kHostPanels), 256));
}

tg_status host_pipe(int dev, HostPipe **out) {
    HostPipe &hp = g_pipe[dev];
    if (!hp.init) {
        if (cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) != cudaSuccess)
            return TG_ERR_CUDA;
        cudaEvent_t *evs[] = {&hp.start, &hp.h2d_done, &hp.done};
        for (cudaEvent_t *e : evs)
            if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return TG_ERR_CUDA;
        for (int i = 0; i < kHostPanels; ++i)
            if (cudaEventCreateWithFlags(&hp.a_done[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.c_done[i], cudaEventDisableTiming) != cudaSuccess)
                return TG_ERR_CUDA;
        hp.init = true;
    }
    *out = &hp;
    return TG_OK;
}

}  // namespace

extern "C" {

int32_t tg_abi_version(void) { return TG_ABI_VERSION; }

const char *tg_status_string(tg_status s) {
    switch (s) {
    case TG_OK: return "TG_OK";
    case TG_ERR_INVALID_VALUE: return "TG_ERR_INVALID_VALUE";
    case TG_ERR_UNSUPPORTED: return "TG_ERR_UNSUPPORTED";
    case TG_ERR_OUT_OF_MEMORY: return "TG_ERR_OUT_OF_MEMORY";
    case TG_ERR_CUDA: return "TG_ERR_CUDA";
    case TG_ERR_ARCH: return "TG_ERR_ARCH";
    case TG_ERR_TIMEOUT: return "TG_ERR_TIMEOUT";
    case TG_ERR_NOT_IMPLEMENTED: return "TG_ERR_NOT_IMPLEMENTED";
    default: return "TG_ERR_UNKNOWN";
    }
}

tg_status tg_plan_gemm(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda,
                       const void *b, int64_t ldb, const void *c, int64_t ldc, tg_dtype dtype_in,
                       tg_dtype dtype_out, int32_t num_sms, const tg_options *opt,
                       tg_plan *plan) {
    if (plan == nullptr) return TG_ERR_INVALID_VALUE;
    const tg_status v = validate(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, opt);
    if (v != TG_OK) return v;
    Plan pl;
    make_plan(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, num_sms, opt, &pl);
    if (!pl.valid) return TG_ERR_UNSUPPORTED;
    if (M == 0 || N == 0 || K == 0) {   // nothing, or a memset of C: no kernel of the library
        pl.pub.kernels = 0;
        pl.pub.workspace_bytes = 0;
        pl.pub.tail_tiles = 0;
        pl.pub.tail_splits = 0;
    }
    *plan = pl.pub;
    return TG_OK;
}

tg_status tg_gemm_ex(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                     int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in, tg_dtype dtype_out,
                     void *stream, const tg_options *opt) {
    tg_status st = validate(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int eo = esize_of(dtype_out);
    if (K == 0)
        return cuda_status(cudaMemset2DAsync(c, ldc * eo, 0, N * eo, M, s));
    return enqueue(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, s, opt, dev, Batch{},
                   nullptr);
}

tg_status tg_gemm_fused(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda,
                        const void *b, int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in,
                        tg_dtype dtype_out, const tg_epilogue *epilogue, void *stream,
                        const tg_options *opt) {
    tg_status st = validate(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    tg::EpiParams e;
    st = validate_epilogue(M, N, c, ldc, dtype_out, epilogue, &e);
    if (st != TG_OK) return st;
    if (epilogue == nullptr)
        return tg_gemm_ex(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream, opt);
    if (M == 0 || N == 0) return TG_OK;
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)   // the epilogue of the empty sum
        return cuda_status(tg::launch_splitk_reduce(nullptr, 0, M, N, c, ldc,
                                                    out_kind_of(dtype_out), 0, s, &e));
    return enqueue(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, s, opt, dev, Batch{},
                   nullptr, &e);
}

tg_status tg_gemm_host(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda,
                       const void *b, int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in,
                       tg_dtype dtype_out, void *stream, const tg_options *opt) {
    tg_status st = validate(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TG_OK) return st;
    int dev_id = 0;
    if (cudaGetDevice(&dev_id) != cudaSuccess) return TG_ERR_CUDA;
    HostPipe *hp = nullptr;
    std::lock_guard<std::mutex> lk(g_pipe[dev_id].mu);
    if ((st = host_pipe(dev_id, &hp)) != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int ei = esize_of(dtype_in), eo = esize_of(dtype_out);
    // device copies with 16-byte row pitches (read in place by the kernels)
    const int64_t lda_d = round_up(std::max<int64_t>(K, 1), 16 / ei);
    const int64_t ldb_d = round_up(N, 16 / ei);
    const int64_t ldc_d = round_up(N, 16 / eo);
    const int64_t off_b = round_up(M * lda_d * ei, 256);
    const int64_t off_c = off_b + round_up(K * ldb_d * ei, 256);
    const int64_t bytes = off_c + round_up(M * ldc_d * eo, 256);
    uint8_t *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), bytes, dev->pool, s);
    if (e != cudaSuccess) return cuda_status(e);
    uint8_t *A_d = ws, *B_d = ws + off_b, *C_d = ws + off_c;
    const uint8_t *ah = static_cast<const uint8_t *>(a);
    const uint8_t *bh = static_cast<const uint8_t *>(b);
    uint8_t *ch = static_cast<uint8_t *>(c);
    auto ok = [](cudaError_t r) { return r == cudaSuccess; };
    bool good = ok(cudaEventRecord(hp->start, s));
    const int64_t rows = host_panel_rows(M);
    const int panels = static_cast<int>(cdiv(M, rows));
    if (K > 0) {
        // one copy stream in order: all of B, then the panels of A (several
        // copy streams measured no faster: the host link is the limit)
        good = ok(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) &&
               ok(cudaMemcpy2DAsync(B_d, ldb_d * ei, bh, ldb * ei, N * ei, K,
                                    cudaMemcpyHostToDevice, hp->h2d));
        for (int p = 0; p < panels && good; ++p) {
            const int64_t r0 = p * rows, rn = std::min(M, r0 + rows) - r0;
            good = ok(cudaMemcpy2DAsync(A_d + r0 * lda_d * ei, lda_d * ei, ah + r0 * lda * ei,
                                        lda * ei, K * ei, rn, cudaMemcpyHostToDevice, hp->h2d)) &&
                   ok(cudaEventRecord(hp->a_done[p], hp->h2d));
        }
    }
    if (good) good = ok(cudaStreamWaitEvent(hp->d2h, hp->start, 0));
    for (int p = 0; p < panels && good; ++p) {
        const int64_t r0 = p * rows, rn = std::min(M, r0 + rows) - r0;
        uint8_t *cp = C_d + r0 * ldc_d * eo;
        if (K == 0) {
            good = ok(cudaMemset2DAsync(cp, ldc_d * eo, 0, N * eo, rn, s));
        } else {
            good = ok(cudaStreamWaitEvent(s, hp->a_done[p], 0));
            if (good) {
                st = enqueue(rn, N, K, A_d + r0 * lda_d * ei, lda_d, B_d, ldb_d, cp, ldc_d,
                             dtype_in, dtype_out, s, opt, dev, Batch{}, nullptr);
                good = st == TG_OK;
            }
        }
        if (good)
            good = ok(cudaEventRecord(hp->c_done[p], s)) &&
                   ok(cudaStreamWaitEvent(hp->d2h, hp->c_done[p], 0)) &&
                   ok(cudaMemcpy2DAsync(ch + r0 * ldc * eo, ldc * eo, cp, ldc_d * eo, N * eo, rn,
                                        cudaMemcpyDeviceToHost, hp->d2h));
    }
    // the caller's stream resumes after every copy of the call (also after a
    // failure part way); then the staging memory goes back to the pool
    const bool joined = ok(cudaEventRecord(hp->done, hp->d2h)) &&
                        ok(cudaStreamWaitEvent(s, hp->done, 0)) &&
                        ok(cudaEventRecord(hp->h2d_done, hp->h2d)) &&
                        ok(cudaStreamWaitEvent(s, hp->h2d_done, 0));
    if (!joined) return TG_ERR_CUDA;   // never free what copies may still use
    if (!ok(cudaFreeAsync(ws, s))) return TG_ERR_CUDA;
    if (!good) return st != TG_OK ? st : TG_ERR_CUDA;
    return TG_OK;
}

tg_status tg_gemm(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                  int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in, tg_dtype dtype_out,
                  void *stream) {
    return tg_gemm_ex(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream, nullptr);
}

tg_status tg_plan_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                                       const void *a, int64_t lda, int64_t stride_a,
                                       const void *b, int64_t ldb, int64_t stride_b,
                                       const void *c, int64_t ldc, int64_t stride_c,
                                       tg_dtype dtype_in, tg_dtype dtype_out, int32_t num_sms,
                                       const tg_options *opt, tg_plan *plan) {
    if (plan == nullptr) return TG_ERR_INVALID_VALUE;
    const tg_status v = validate_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, c,
                                         ldc, stride_c, dtype_in, dtype_out, opt);
    if (v != TG_OK) return v;
    Plan pl;
    const bool one = batch > 1 &&
                     batch_in_one_launch(dtype_in, a, lda, stride_a, b, ldb, stride_b);
    pl.stride_c = stride_c;
    make_plan(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, num_sms, opt, &pl, 0, 0,
              one ? batch : 1);
    if (!pl.valid) return TG_ERR_UNSUPPORTED;
    if (batch > 1 && !one) {   // one call per product
        pl.pub.per_batch = 1;
        pl.pub.kernels *= static_cast<int32_t>(std::min<int64_t>(batch, 1 << 24));
        pl.pub.tiles *= batch;
    }
    if (batch == 0 || M == 0 || N == 0 || K == 0) {
        pl.pub.kernels = 0;
        pl.pub.workspace_bytes = 0;
        pl.pub.tail_tiles = 0;
        pl.pub.tail_splits = 0;
    }
    *plan = pl.pub;
    return TG_OK;
}

tg_status tg_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void *a,
                                  int64_t lda, int64_t stride_a, const void *b, int64_t ldb,
                                  int64_t stride_b, void *c, int64_t ldc, int64_t stride_c,
                                  tg_dtype dtype_in, tg_dtype dtype_out, void *stream,
                                  const tg_options *opt) {
    tg_status st = validate_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, c, ldc,
                                    stride_c, dtype_in, dtype_out, opt);
    if (st != TG_OK) return st;
    if (batch == 0 || M == 0 || N == 0) return TG_OK;
    if (batch == 1)
        return tg_gemm_ex(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream, opt);
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TG_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int ei = esize_of(dtype_in), eo = esize_of(dtype_out);
    auto c_of = [&](int64_t z) { return static_cast<uint8_t *>(c) + z * stride_c * eo; };
    if (K == 0) {
        for (int64_t z = 0; z < batch; ++z) {
            st = cuda_status(cudaMemset2DAsync(c_of(z), ldc * eo, 0, N * eo, M, s));
            if (st != TG_OK) return st;
        }
        return TG_OK;
    }
    if (batch_in_one_launch(dtype_in, a, lda, stride_a, b, ldb, stride_b)) {
        bool map_failed = false;
        st = enqueue(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, s, opt, dev,
                     Batch{batch, stride_a, stride_b, stride_c}, &map_failed);
        if (!map_failed) return st;
    }
    // one call per product, in order of z
    for (int64_t z = 0; z < batch; ++z) {
        st = tg_gemm_ex(M, N, K, static_cast<const uint8_t *>(a) + z * stride_a * ei, lda,
                        static_cast<const uint8_t *>(b) + z * stride_b * ei, ldb, c_of(z), ldc,
                        dtype_in, dtype_out, stream, opt);
        if (st != TG_OK) return st;
    }
    return TG_OK;
}

tg_status tg_selftest_timeout(int32_t timeout_ms, void *stream) {
    if (timeout_ms < 1 || timeout_ms > 10000) return TG_ERR_INVALID_VALUE;
    DeviceState *dev = nullptr;
    const tg_status st = device_state(&dev);
    if (st != TG_OK) return st;
    return cuda_status(tg::launch_selftest_timeout(
        dev->status, static_cast<uint64_t>(timeout_ms) * 1000000ull, static_cast<cudaStream_t>(stream)));
}

tg_status tg_last_device_error(void *stream) {
    DeviceState *dev = nullptr;
    const tg_status st = device_state(&dev);
    if (st != TG_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TG_ERR_CUDA;
    int words[2] = {0, 0};
    if (cudaMemcpy(words, dev->status, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TG_ERR_CUDA;
    if (words[0] != 0) {
        const int zero[2] = {0, 0};
        if (cudaMemcpy(dev->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return TG_ERR_CUDA;
        return static_cast<tg_status>(words[0]);
    }
    return TG_OK;
}

}  // extern "C"
