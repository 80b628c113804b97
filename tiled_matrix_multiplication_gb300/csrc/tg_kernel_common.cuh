// tg_kernel_common.cuh -- device helpers shared by the tensor-core kernels:
// failure recording, tensor-memory loads that wait in the same statement, and
// FP32 -> FP16/BF16 packing with round-to-nearest-even.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tg {

__device__ __forceinline__ void record_failure(int *status, int code, int where) {
    if (atomicCAS(status, 0, code) == 0) atomicExch(status + 1, where);
}

// Checked builds (compiled with -DTG_CHECKED, libtg_gemm_checked.so): device-side
// bounds and alignment checks in front of the kernels' shared-memory, tensor-
// memory, TMA and remote accesses.  A failed check records TG_ERR_BOUNDS (8)
// and the site in the status word and the caller skips the access (the kernel
// then ends through its bounded waits); nothing traps.  In the normal build
// tg_check is `true` and its condition is never evaluated at run time.
#ifdef TG_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
constexpr int kErrBounds = 8;
// check sites (high half of the recorded `where`; the low half is a detail)
enum CheckSite : int {
    CHK_TC_LOAD_A = 1, CHK_TC_LOAD_B = 2, CHK_TC_MMA = 3, CHK_TC_TMEM = 4, CHK_TC_STAGE = 5,
    CHK_TC_STORE = 6, CHK_SK_LOAD = 7, CHK_SK_TMEM = 8, CHK_SK_PUSH = 9, CHK_SK_SUM = 10,
    CHK_SELFTEST = 15
};
__device__ __forceinline__ bool tg_check(int *status, bool ok, int site, int detail) {
    if constexpr (kChecked) {
        if (!ok) {
            record_failure(status, kErrBounds, (site << 16) | (detail & 0xffff));
            return false;
        }
    }
    return true;
}
// a TMA tile coordinate along the innermost dimension starts on a 16-byte boundary
__device__ __forceinline__ bool tma_x_aligned(int x, int esize) { return ((x * esize) & 15) == 0; }

// Load 32 accumulator columns of this thread's row and wait for them in one
// statement, so no use of r[] can be scheduled ahead of the wait.
__device__ __forceinline__ void tmem_load_32cols_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
        " [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo, uint32_t hi) {
    __half2 h = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(uint32_t lo, uint32_t hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t *>(&h);
}

// Same with 16 columns (x16).
__device__ __forceinline__ void tmem_load_16cols_sync(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15},"
        " [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

}  // namespace tg
