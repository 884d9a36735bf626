// epilogue.cuh -- element-wise epilogue operations shared by the kernels:
// bias, activation and BF16 conversion ("GEMM on NVIDIA GPUs", section 4
// "Epilogue": alpha/beta, bias, activation and dtype conversion applied where
// the accumulator is written out).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace gemm {

enum : int { kActNone = 0, kActRelu = 1, kActGelu = 2 };

// ReLU: max(x, 0).  GELU, tanh form (Hendrycks & Gimpel):
// 0.5 x (1 + tanh(sqrt(2 / pi) (x + 0.044715 x^3))), with CUDA's tanhf.
__device__ __forceinline__ float apply_activation(float x, int act) {
    if (act == kActRelu) return fmaxf(x, 0.f);
    if (act == kActGelu) {
        const float kSqrt2OverPi = 0.7978845608028654f;
        const float u = kSqrt2OverPi * fmaf(0.044715f * x, x * x, x);
        return 0.5f * x * (1.f + tanhf(u));
    }
    return x;
}

// FP32 -> BF16 bit pattern, round to nearest even.
__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Two BF16 values packed low-first into 32 bits.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(to_bf16_bits(lo)) | (static_cast<uint32_t>(to_bf16_bits(hi)) << 16);
}

}  // namespace gemm
