// tg_plan.cu -- argument rules and the planner of the C ABI (host only, no
// device access): which kernel variant, tile width, K split and grid a call
// uses, and the entry points that report a plan.
#include "tg_host_api.h"

namespace tgh {

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
        // A multicast: clusters of two CTA pairs (192-, 224- or 256-wide tiles)
        if (opt->multicast == 2 &&
            (opt->path == TG_PATH_TC || opt->path == TG_PATH_SKINNY ||
             (opt->block_n && !tg::tc_supported_mc(opt->block_n, 2, true))))
            return TG_ERR_UNSUPPORTED;
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
            const int ik = in_kind_of(static_cast<tg_dtype>(din));
            const bool one = tg::tc_supported_block_n(ik, opt->block_n, false);
            const bool two = tg::tc_supported_block_n(ik, opt->block_n, true);
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

// `pair_slots` / `quad_slots`: clusters of 2 / 4 CTAs resident at once
// (0: estimate from the SM count).
// `batch` > 1: that many products with 16-byte aligned operands (no packing,
// no K split across kernels) in one launch; the batch index is the slowest
// dimension of the work list.
static void make_plan_uncached(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda,
                               const void *b, int64_t ldb, const void *c, int64_t ldc,
                               tg_dtype din, tg_dtype dout, int num_sms, const tg_options *opt,
                               Plan *pl, int pair_slots, int quad_slots, int64_t batch) {
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
    // 8192^3 and on the prefill shapes.  mc = 2: clusters of two pairs sharing
    // A by multicast (two tiles per unit).
    struct Cand { bool pair; int mc; int bn; int eff; };
    static const Cand kCands[] = {
        {true, 1, 512, 98}, {true, 2, 256, 105}, {true, 1, 256, 100}, {true, 2, 224, 90},
        {true, 2, 192, 86}, {true, 1, 224, 92}, {true, 1, 192, 84}, {false, 1, 256, 90},
        {false, 1, 192, 82}, {false, 1, 224, 80}, {false, 1, 128, 62}, {true, 1, 128, 62}};
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
            const double waves = units > 0 ? used + 0.25 * (static_cast<double>(cdiv(units, std::min(units, slots))) - used) : 0.0;
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
    // The transposed streaming kernel wins up to 128 rows for 16-bit and FP8
    // operands alike (GB300, N = K = 8192, M = 128: FP16 30.5 vs 35.0 us for
    // the tile kernel with a K split, E4M3 20.8 vs 24.7 us).
    const int64_t skinny_rows_max = 128;
    const bool skinny_ok = din != TG_F32 && M <= skinny_rows_max &&
                           (forced_skinny || !(opt && (opt->block_n || opt->multicast == 2))) &&
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
            // K ranges of fewer than 4 k-tiles (512 bytes of K) stream too little
            // to pay for the reduction (127 x 255 x 65: 10.3 us unsplit, 13.7 us
            // with two ranges of one k-tile each)
            if (kps < 4) continue;
            if (opt && opt->splits && opt->splits != sc) continue;
            if (tiles * sc <= cap) {
                best_s = sc;
                two = false;
            } else if (nt == 128 && tiles * sc <= 2 * cap) {
                // more CTAs than SMs: two half-size CTAs per SM keep them all
                // resident (measured faster than one full-size CTA per SM for
                // every M from 1 to 64 at N = K = 8192).  At 128 rows a K split
                // already spread over the SMs one CTA each is kept instead: the
                // doubled split sends twice the partial bytes over the cluster
                // network (N = K = 8192: FP16 27.6 vs 28.1 us, E4M3 17.7 vs
                // 18.6 us for 2 against 4 ranges)
                if (mp == 128 && best_s > 1) break;
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
        p.multicast = 1;
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
        // not persistent: one CTA per (column tile, K range)
        p.ctas = static_cast<int32_t>(p.tiles * splits);
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
    if (x3) p.pack_a = p.pack_b = 3;   // hi / lo TF32 parts of A and of B
    p.c_vector = aligned16(c) && (ldc * eo) % 16 == 0 && (batch == 1 || (pl->stride_c * eo) % 16 == 0);
    pl->lda_p = p.pack_a ? round_up(pl->k_eff, align_elems) : lda;
    pl->ldb_p = p.pack_b ? round_up(N, align_elems) : ldb;
    int64_t ws = 0;
    if (p.pack_a) {
        pl->off_a = ws;
        ws = round_up(ws + M * pl->lda_p * ei, 256);
    }
    if (p.pack_b) {   // B [K, N], or B' [3K, N] of the 3xTF32 parts
        pl->off_b = ws;
        ws = round_up(ws + pl->k_eff * pl->ldb_p * ei, 256);
    }
    const bool global_partials = splits > 1 && p.path != TG_PATH_SKINNY;
    if (global_partials) {
        pl->off_p = ws;
        ws = round_up(ws + splits * M * N * 4, 256);
    }
    p.workspace_bytes = ws;
    p.kernels = (p.pack_a ? 1 : 0) + (p.pack_b ? 1 : 0) + 1 + (global_partials ? 1 : 0);
    const int tmo = (opt && opt->timeout_ms) ? opt->timeout_ms : kDefaultTimeoutMs;
    pl->timeout_ns = static_cast<uint64_t>(tmo) * 1000000ull;
}

// The plans of recent calls.  make_plan_uncached is a pure function of its
// arguments -- of the operand pointers only whether each is 16-byte aligned --
// and tries every kernel variant and split count (about 1 us of host time for
// a small product, a fifth of a call's), so a repeated shape takes its plan
// from here.  16 entries, replaced round-robin, under a lock.
namespace {
struct PlanKey {
    int64_t M, N, K, lda, ldb, ldc, stride_c, batch;
    int32_t din, dout, num_sms, pair_slots, quad_slots, align, has_opt, pad;
    tg_options opt;
};
struct PlanCache {
    std::mutex mu;
    PlanKey key[16];
    Plan plan[16];
    int used = 0, next = 0;
};
PlanCache &plan_cache() {
    static PlanCache cache;
    return cache;
}
}  // namespace

void make_plan(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
               int64_t ldb, const void *c, int64_t ldc, tg_dtype din, tg_dtype dout, int num_sms,
               const tg_options *opt, Plan *pl, int pair_slots, int quad_slots,
               int64_t batch) {
    PlanKey k;
    std::memset(&k, 0, sizeof(k));   // padding included: keys compare bytewise
    k.M = M, k.N = N, k.K = K, k.lda = lda, k.ldb = ldb, k.ldc = ldc;
    k.stride_c = pl->stride_c, k.batch = batch;
    k.din = din, k.dout = dout, k.num_sms = num_sms;
    k.pair_slots = pair_slots, k.quad_slots = quad_slots;
    k.align = (aligned16(a) ? 1 : 0) | (aligned16(b) ? 2 : 0) | (aligned16(c) ? 4 : 0);
    k.has_opt = opt != nullptr;
    if (opt) k.opt = *opt;
    PlanCache &cache = plan_cache();
    {
        std::lock_guard<std::mutex> lock(cache.mu);
        for (int i = 0; i < cache.used; ++i) {
            if (std::memcmp(&cache.key[i], &k, sizeof(k)) == 0) {
                *pl = cache.plan[i];
                return;
            }
        }
    }
    make_plan_uncached(M, N, K, a, lda, b, ldb, c, ldc, din, dout, num_sms, opt, pl, pair_slots,
                       quad_slots, batch);
    std::lock_guard<std::mutex> lock(cache.mu);
    const int i = cache.used < 16 ? cache.used++ : (cache.next++ & 15);
    cache.key[i] = k;
    cache.plan[i] = *pl;
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
    if (batch > 1 && opt && opt->splits > 1 && opt->path != TG_PATH_SKINNY)
        return TG_ERR_UNSUPPORTED;
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
// fills *e for the kernels.  With `batch` > 1 the products' C blocks start
// `sc` elements apart and their residuals `sr` apart (0: one residual block
// read by every product); scale and bias are shared.
tg_status validate_epilogue(int64_t M, int64_t N, const void *c, int64_t ldc, tg_dtype dout,
                            const tg_epilogue *ep, tg::EpiParams *e, int64_t batch, int64_t sc,
                            int64_t sr) {
    std::memset(e, 0, sizeof(*e));
    if (ep == nullptr) return TG_OK;
    if (ep->activation < TG_ACT_NONE || ep->activation > TG_ACT_GELU_TANH || ep->reserved != 0)
        return TG_ERR_INVALID_VALUE;
    if (sr < 0 || (sr != 0 && ep->residual == nullptr)) return TG_ERR_INVALID_VALUE;
    const int eo = esize_of(dout);
    e->on = 1;
    e->act = ep->activation;
    e->alpha = ep->alpha;
    e->beta = ep->beta;
    e->scale = ep->scale;
    e->bias = ep->bias;
    e->res = ep->residual;
    e->ldr = ep->residual ? ep->ldr : 0;
    e->stride_r = batch > 1 ? sr : 0;
    if (M == 0 || N == 0 || batch == 0) return TG_OK;
    const int64_t last = batch > 1 ? batch - 1 : 0;   // index of the last product
    if (sr > 0 && last > (int64_t(1) << 46) / sr) return TG_ERR_UNSUPPORTED;
    // bytes spanned by every product's C block
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(c);
    const uintptr_t c1 = c0 + static_cast<uintptr_t>((last * sc + (M - 1) * ldc + N) * eo);
    for (const float *v : {ep->scale, ep->bias}) {
        if (v == nullptr) continue;
        if (reinterpret_cast<uintptr_t>(v) % 4) return TG_ERR_INVALID_VALUE;
        const uintptr_t v0 = reinterpret_cast<uintptr_t>(v);
        if (overlaps(c0, c1, v0, v0 + static_cast<uintptr_t>(N) * 4)) return TG_ERR_INVALID_VALUE;
    }
    if (ep->residual) {
        if (ep->ldr < N || ep->ldr > (int64_t(1) << 36)) return TG_ERR_INVALID_VALUE;
        if (reinterpret_cast<uintptr_t>(ep->residual) % eo) return TG_ERR_INVALID_VALUE;
        // in place: every product reads its own C block as the residual
        const bool in_place = ep->residual == c && ep->ldr == ldc && (last == 0 || sr == sc);
        const uintptr_t r0 = reinterpret_cast<uintptr_t>(ep->residual);
        const uintptr_t r1 =
            r0 + static_cast<uintptr_t>((last * sr + (M - 1) * ep->ldr + N) * eo);
        if (!in_place && overlaps(c0, c1, r0, r1)) return TG_ERR_INVALID_VALUE;
        e->res_vector = aligned16(ep->residual) && (ep->ldr * eo) % 16 == 0 &&
                        (last == 0 || (sr * eo) % 16 == 0);
    }
    e->sb_vector = (!ep->scale || aligned16(ep->scale)) && (!ep->bias || aligned16(ep->bias));
    return TG_OK;
}

}  // namespace tgh

using namespace tgh;

extern "C" {

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
    }
    *plan = pl.pub;
    return TG_OK;
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
    }
    *plan = pl.pub;
    return TG_OK;
}

}  // extern "C"
