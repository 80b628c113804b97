// tg_host_api.h -- what the host-side files of the C ABI share: argument
// rules, the plan, per-device state and the launch of one planned product.
// tg_plan.cu validates and plans, tg_api.cu owns device state, tensor maps and
// launches, tg_host.cu the host-operand pipeline.  Private to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <initializer_list>
#include <cstring>
#include <mutex>

#include "tg_gemm.h"
#include "tg_internal.h"

namespace tgh {

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

inline int esize_of(tg_dtype t) {
    return t == TG_F32 ? 4 : (t == TG_E4M3 || t == TG_E5M2 ? 1 : 2);
}

inline bool is_fp8(int t) { return t == TG_E4M3 || t == TG_E5M2; }

inline bool valid_dtype(int t) {
    return t == TG_F16 || t == TG_BF16 || t == TG_F32 || is_fp8(t);
}

inline bool supported_pair(tg_dtype in, tg_dtype out) {
    if (in == TG_F16) return out == TG_F16 || out == TG_F32;
    if (in == TG_BF16) return out == TG_BF16 || out == TG_F32;
    if (in == TG_F32) return out == TG_F32;
    if (is_fp8(in)) return out == TG_F16 || out == TG_BF16 || out == TG_F32;
    return false;
}

inline int in_kind_of(tg_dtype t) {
    switch (t) {
    case TG_F16: return tg::IN_F16;
    case TG_BF16: return tg::IN_BF16;
    case TG_E4M3: return tg::IN_E4M3;
    case TG_E5M2: return tg::IN_E5M2;
    default: return tg::IN_TF32;
    }
}

inline int out_kind_of(tg_dtype t) {
    return t == TG_F16 ? tg::OUT_F16 : (t == TG_BF16 ? tg::OUT_BF16 : tg::OUT_F32);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// Byte span [lo, hi) touched by a rows x cols block with pitch ld.
inline void span(const void *p, int64_t rows, int64_t cols, int64_t ld, int esize,
                 uintptr_t *lo, uintptr_t *hi) {
    *lo = reinterpret_cast<uintptr_t>(p);
    *hi = *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * esize);
}

inline bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
    return a0 < b1 && b0 < a1;
}

struct Plan {
    tg_plan pub;
    int64_t k_tiles = 0, k_per_split = 0, tiles_m = 0, tiles_n = 0;
    int64_t lda_p = 0, ldb_p = 0;              // pitches after packing
    int64_t off_a = 0, off_b = 0, off_p = 0;   // workspace offsets
    bool skinny_two = false;                   // small-M kernel: two CTAs per SM
    uint64_t timeout_ns = 0;
    int64_t stride_c = 0;                      // C batch stride (set before make_plan)
    int64_t k_eff = 0;                         // K of the kernel (3K for 3xTF32)
    bool valid = true;                         // false: no kernel variant fits the options
};

constexpr int64_t kMaxGridY = 65535;           // gridDim.y: one row per product (small M)

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// Products of one launch: `count` of them, whose A / B / C start sa / sb / sc
// elements apart (sa or sb == 0: one operand shared by every product).
struct Batch {
    int64_t count = 1, sa = 0, sb = 0, sc = 0;
};

// tg_plan.cu
tg_status validate(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                   int64_t ldb, const void *c, int64_t ldc, int din, int dout,
                   const tg_options *opt);
void make_plan(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
               int64_t ldb, const void *c, int64_t ldc, tg_dtype din, tg_dtype dout, int num_sms,
               const tg_options *opt, Plan *pl, int pair_slots = 0, int quad_slots = 0,
               int64_t batch = 1);
tg_status validate_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void *a,
                           int64_t lda, int64_t sa, const void *b, int64_t ldb, int64_t sb,
                           const void *c, int64_t ldc, int64_t sc, int din, int dout,
                           const tg_options *opt);
bool batch_in_one_launch(tg_dtype din, const void *a, int64_t lda, int64_t sa, const void *b,
                         int64_t ldb, int64_t sb);
tg_status validate_epilogue(int64_t M, int64_t N, const void *c, int64_t ldc, tg_dtype dout,
                            const tg_epilogue *ep, tg::EpiParams *e, int64_t batch = 1,
                            int64_t sc = 0, int64_t sr = 0);

// tg_api.cu
tg_status device_state(DeviceState **out);
// TG_OK if every non-null pointer is device memory of the current device,
// else TG_ERR_INVALID_VALUE (TG_ERR_CUDA if there is no current device).
tg_status operands_local(std::initializer_list<const void *> ptrs);
tg_status cuda_status(cudaError_t e);
tg_status enqueue(int64_t M, int64_t N, int64_t K, const void *a, int64_t lda, const void *b,
                  int64_t ldb, void *c, int64_t ldc, tg_dtype dtype_in, tg_dtype dtype_out,
                  cudaStream_t s, const tg_options *opt, DeviceState *dev, const Batch &bt,
                  bool *map_failed, const tg::EpiParams *epi = nullptr);

}  // namespace tgh
