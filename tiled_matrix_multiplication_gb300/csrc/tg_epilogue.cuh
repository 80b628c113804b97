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
    const bool full = ncols == 32;
    const bool vec_sb = full && e.sb_vector;
    const bool vec_res = full && e.res_vector;
    const int64_t roff = e.res ? z * e.stride_r + static_cast<int64_t>(row) * e.ldr + col : 0;
    const bool gelu = e.act == ACT_GELU_TANH;
    const bool gate = e.act == ACT_SILU || gelu;
    // eight columns at a time, so that scale, bias and residual values of the
    // whole chunk are never live at once
#pragma unroll
    for (int g = 0; g < 32; g += 8) {
        float sc[8], bi[8], res[8];
        if (vec_sb) {
#pragma unroll
            for (int h = 0; h < 8; h += 4) {
                const float4 s4 = e.scale ? *reinterpret_cast<const float4 *>(e.scale + col + g + h)
                                          : make_float4(1.f, 1.f, 1.f, 1.f);
                const float4 b4 = e.bias ? *reinterpret_cast<const float4 *>(e.bias + col + g + h)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                sc[h] = s4.x, sc[h + 1] = s4.y, sc[h + 2] = s4.z, sc[h + 3] = s4.w;
                bi[h] = b4.x, bi[h + 1] = b4.y, bi[h + 2] = b4.z, bi[h + 3] = b4.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                sc[j] = (e.scale && g + j < ncols) ? e.scale[col + g + j] : 1.f;
                bi[j] = (e.bias && g + j < ncols) ? e.bias[col + g + j] : 0.f;
            }
        }
        if (e.res) {
            if (vec_res && out_kind != OUT_F32) {
                const uint4 w = reinterpret_cast<const uint4 *>(
                    static_cast<const uint16_t *>(e.res) + roff)[g / 8];
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
                    res[2 * t] = lo;
                    res[2 * t + 1] = hi;
                }
            } else if (vec_res) {
                const float4 *src =
                    reinterpret_cast<const float4 *>(static_cast<const float *>(e.res) + roff + g);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float4 v = src[q];
                    res[4 * q] = v.x, res[4 * q + 1] = v.y, res[4 * q + 2] = v.z, res[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    res[j] = g + j < ncols ? epi_load_res(e, out_kind, roff + g + j) : 0.f;
            }
        }
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = fmaf(__uint_as_float(r[g + j]) * e.alpha, sc[j], bi[j]);
        // one loop per activation (the choice is uniform), not a branch per element
        if (e.act == ACT_RELU) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = v[j] > 0.f ? v[j] : 0.f;
        } else if (gate) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = epi_sigmoid_gate(v[j], epi_gate_arg(gelu, v[j]));
        }
        if (e.res) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = fmaf(e.beta, res[j], v[j]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) r[g + j] = __float_as_uint(v[j]);
    }
}

}  // namespace tg
