// Fused epilogue applied to a few consecutive output columns of one row, after
// v = alpha*acc + beta*C and before the single rounding to the output type:
//     v += bias[n];  v = act(v);  v *= aux[m, n]
// ("TorchInductor ganha suporte a GEMMs de alta performance com CuteDSL",
// epilogue-fusion roadmap paragraph: auxiliary tensor loads, element-wise add
// and mul, ReLU, sigmoid, tanh). sigmoid is 1 / (1 + e^-v) and tanh is
// 1 - 2 / (1 + e^2v), both with CUDA's fast exponential (__expf) and fast
// division (__fdividef): a few instructions each, with a relative error near
// 1e-6 (tanh: an absolute error near 2e-7 around 0), well inside the output
// tolerances, and exact limits (0 and 1, -1 and 1) when the exponential
// overflows. In the fused tiled kernel the epilogue runs beside the next
// tile's MMAs, and the accurate tanhf made it the slower of the two.
#pragma once

#include <stdint.h>

namespace tpg {

struct EpiParams {
    const void *bias; // null or N values (bias_f32 ? fp32 : bf16), 16-byte aligned
    int32_t bias_f32;
    int32_t act;      // 0 none, 1 relu, 2 sigmoid, 3 tanh
    const void *aux;  // null or [M, N] of the output type, row stride ldaux
    int64_t ldaux;
};

__device__ __forceinline__ float sigmoid_fast(float v) { return __fdividef(1.0f, 1.0f + __expf(-v)); }
__device__ __forceinline__ float tanh_fast(float v) { return 1.0f - __fdividef(2.0f, 1.0f + __expf(2.0f * v)); }

__device__ __forceinline__ float apply_act(int32_t act, float v) {
    switch (act) {
    case 1: return v > 0.0f ? v : 0.0f;
    case 2: return sigmoid_fast(v);
    case 3: return tanh_fast(v);
    default: return v;
    }
}

// The activation as a compile-time choice (the fused tiled epilogue).
template <int kAct>
__device__ __forceinline__ float apply_act_t(float v) {
    if constexpr (kAct == 1) return v > 0.0f ? v : 0.0f;
    else if constexpr (kAct == 2) return sigmoid_fast(v);
    else if constexpr (kAct == 3) return tanh_fast(v);
    else return v;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// The 16-byte aux cell at columns col0 .. of row grow, read through the
// read-only path; issued for a whole chunk before any of it is used, so the
// loads overlap instead of each waiting for the previous cell's shared-memory
// store. Only whole cells of rows inside D are loaded (the others return 0 and
// take the element-wise path of epilogue_cell).
template <bool kOutF32>
__device__ __forceinline__ uint4 load_aux_cell(const EpiParams &e, int32_t N, int64_t grow, bool row_ok,
                                               int32_t col0) {
    constexpr int W = kOutF32 ? 4 : 8;
    if (!e.aux || !row_ok || col0 + W > N) return make_uint4(0u, 0u, 0u, 0u);
    const char *base = static_cast<const char *>(e.aux) + (grow * e.ldaux + col0) * (kOutF32 ? 4 : 2);
    return __ldg(reinterpret_cast<const uint4 *>(base));
}

// W consecutive columns col0 .. col0+W-1 of global row `grow`. Whole cells
// (col0 + W <= N) use 16-byte (or 8-byte) vector loads, which the host's
// alignment checks make legal, and take aux from `auxq` (see load_aux_cell);
// cells at the ragged edge load element by element and never past N. Rows
// outside D skip the aux load (their values are never stored).
template <int W, bool kOutF32, int kAct>
__device__ __forceinline__ void epilogue_cell(const EpiParams &e, int32_t N, int64_t grow, bool row_ok,
                                              int32_t col0, float (&v)[W], uint4 auxq) {
    static_assert(W == 4 || W == 8, "cells of 4 fp32 or 8 bf16 values");
    const bool full = col0 + W <= N;
    if (e.bias) {
        if (e.bias_f32) {
            const float *b = static_cast<const float *>(e.bias) + col0;
            if (full) {
#pragma unroll
                for (int q = 0; q < W / 4; ++q) {
                    const float4 t = __ldg(reinterpret_cast<const float4 *>(b) + q);
                    v[4 * q] += t.x;
                    v[4 * q + 1] += t.y;
                    v[4 * q + 2] += t.z;
                    v[4 * q + 3] += t.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if (col0 + i < N) v[i] += b[i];
            }
        } else {
            const uint16_t *b = static_cast<const uint16_t *>(e.bias) + col0;
            if (full) {
                uint32_t w[W / 2];
                if constexpr (W == 8) {
                    const uint4 t = __ldg(reinterpret_cast<const uint4 *>(b));
                    w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
                } else {
                    const uint2 t = __ldg(reinterpret_cast<const uint2 *>(b));
                    w[0] = t.x; w[1] = t.y;
                }
#pragma unroll
                for (int q = 0; q < W / 2; ++q) {
                    v[2 * q] += __uint_as_float(w[q] << 16);
                    v[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
                }
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if (col0 + i < N) v[i] += bf16_bits_to_f32(b[i]);
            }
        }
    }
    if constexpr (kAct != 0) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] = apply_act_t<kAct>(v[i]);
    }
    if (e.aux && row_ok) {
        if constexpr (kOutF32) {
            const float *x = static_cast<const float *>(e.aux) + grow * e.ldaux + col0;
            if (full) {
                v[0] *= __uint_as_float(auxq.x);
                v[1] *= __uint_as_float(auxq.y);
                v[2] *= __uint_as_float(auxq.z);
                v[3] *= __uint_as_float(auxq.w);
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if (col0 + i < N) v[i] *= x[i];
            }
        } else {
            const uint16_t *x = static_cast<const uint16_t *>(e.aux) + grow * e.ldaux + col0;
            if (full) {
                const uint32_t w[4] = {auxq.x, auxq.y, auxq.z, auxq.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[2 * q] *= __uint_as_float(w[q] << 16);
                    v[2 * q + 1] *= __uint_as_float(w[q] & 0xFFFF0000u);
                }
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if (col0 + i < N) v[i] *= bf16_bits_to_f32(x[i]);
            }
        }
    }
}

// One value (the streaming and K == 0 kernels, which work element by element).
template <bool kOutF32>
__device__ __forceinline__ float epilogue_one(const EpiParams &e, int64_t m, int32_t n, float v) {
    if (e.bias)
        v += e.bias_f32 ? static_cast<const float *>(e.bias)[n]
                        : bf16_bits_to_f32(static_cast<const uint16_t *>(e.bias)[n]);
    v = apply_act(e.act, v);
    if (e.aux) {
        const int64_t idx = m * e.ldaux + n;
        v *= kOutF32 ? static_cast<const float *>(e.aux)[idx]
                     : bf16_bits_to_f32(static_cast<const uint16_t *>(e.aux)[idx]);
    }
    return v;
}

} // namespace tpg
