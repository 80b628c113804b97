// tg_epilogue.cuh -- the fused epilogue D = act(alpha * scale[n] * acc +
// bias[n]) + beta * R[m, n], applied to FP32 accumulator values where the
// kernels write C (before the one rounding to the output type).
//
// Activations: relu (x if x > 0, else 0), silu (x / (1 + e^-x)) and the tanh
// form of the Gaussian error linear unit (x/2 * (1 + tanh(u)), u = sqrt(2/pi)
// * (x + 0.044715 x^3), Hendrycks and Gimpel 2016).  Since (1 + tanh(u)) / 2 =
// 1 / (1 + e^(-2u)), both smooth activations are x / (1 + e^(-z)) with z = x
// or z = 2u, evaluated in FP32 with CUDA's __expf and __fdividef intrinsics
// (a few ulp each; for z below about -87 the quotient is 0, the limit).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tg_internal.h"

namespace tg {

__device__ __forceinline__ float epi_sigmoid_gate(float x, float z) {
    return __fdividef(x, 1.f + __expf(-z));
}

// z of the smooth activations: x (silu) or 2u (tanh-form GELU).
__device__ __forceinline__ float epi_gate_arg(bool gelu, float x) {
    return gelu ? 1.5957691216057308f * fmaf(0.044715f * x, x * x, x) : x;   // 2 sqrt(2/pi)
}

__device__ __forceinline__ float epi_act(int act, float x) {
    if (act == ACT_RELU) return x > 0.f ? x : 0.f;
    if (act == ACT_SILU || act == ACT_GELU_TANH)
        return epi_sigmoid_gate(x, epi_gate_arg(act == ACT_GELU_TANH, x));
    return x;
}

__device__ __forceinline__ float epi_load_res(const EpiParams &e, int out_kind, int64_t off) {
    if (out_kind == OUT_F32) return static_cast<const float *>(e.res)[off];
    if (out_kind == OUT_F16) return __half2float(static_cast<const __half *>(e.res)[off]);
    return __bfloat162float(static_cast<const __nv_bfloat16 *>(e.res)[off]);
}

// One element (m, n) of batch product z; acc is the FP32 accumulator value.
__device__ __forceinline__ float epi_one(const EpiParams &e, int out_kind, int64_t m, int64_t n,
                                         float acc, int z = 0) {
    const float s = e.scale ? e.scale[n] : 1.f;
    const float b = e.bias ? e.bias[n] : 0.f;
    float v = epi_act(e.act, fmaf(acc * e.alpha, s, b));
    if (e.res) v = fmaf(e.beta, epi_load_res(e, out_kind, z * e.stride_r + m * e.ldr + n), v);
    return v;
}

// Columns col .. col + ncols - 1 (ncols <= 32) of row `row`, in place on the
// FP32 bit patterns r[].  The residual is read before C is written, by the
// thread that writes it, so R may be C itself.
__device__ __forceinline__ void epi_chunk32(const EpiParams &e, int out_kind, int row, int col,
                                            int ncols, uint32_t (&r)[32], int z = 0) {
    float sc[32], bi[32], res[32];
    const bool full = ncols == 32;
    if (full && e.sb_vector) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 s4 = e.scale ? *reinterpret_cast<const float4 *>(e.scale + col + j)
                                      : make_float4(1.f, 1.f, 1.f, 1.f);
            const float4 b4 = e.bias ? *reinterpret_cast<const float4 *>(e.bias + col + j)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            sc[j] = s4.x, sc[j + 1] = s4.y, sc[j + 2] = s4.z, sc[j + 3] = s4.w;
            bi[j] = b4.x, bi[j + 1] = b4.y, bi[j + 2] = b4.z, bi[j + 3] = b4.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            sc[j] = (e.scale && j < ncols) ? e.scale[col + j] : 1.f;
            bi[j] = (e.bias && j < ncols) ? e.bias[col + j] : 0.f;
        }
    }
    if (e.res) {
        const int64_t off = z * e.stride_r + static_cast<int64_t>(row) * e.ldr + col;
        if (full && e.res_vector && out_kind != OUT_F32) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const uint16_t *>(e.res) + off);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 w = src[q];
                const uint32_t h[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    float lo, hi;
                    if (out_kind == OUT_F16) {
                        const __half2 v = *reinterpret_cast<const __half2 *>(&h[t]);
                        lo = __low2float(v), hi = __high2float(v);
                    } else {
                        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&h[t]);
                        lo = __low2float(v), hi = __high2float(v);
                    }
                    res[q * 8 + 2 * t] = lo;
                    res[q * 8 + 2 * t + 1] = hi;
                }
            }
        } else if (full && e.res_vector) {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(e.res) + off);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = src[q];
                res[4 * q] = v.x, res[4 * q + 1] = v.y, res[4 * q + 2] = v.z, res[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) res[j] = j < ncols ? epi_load_res(e, out_kind, off + j) : 0.f;
        }
    }
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = fmaf(__uint_as_float(r[j]) * e.alpha, sc[j], bi[j]);
    // one loop per activation (the choice is uniform), not a branch per element
    if (e.act == ACT_RELU) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = v[j] > 0.f ? v[j] : 0.f;
    } else if (e.act == ACT_SILU || e.act == ACT_GELU_TANH) {
        const bool gelu = e.act == ACT_GELU_TANH;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = epi_sigmoid_gate(v[j], epi_gate_arg(gelu, v[j]));
    }
    if (e.res) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaf(e.beta, res[j], v[j]);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
}

}  // namespace tg
