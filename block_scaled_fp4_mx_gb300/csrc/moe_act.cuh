// moe_act.cuh -- the MoE layer's activation, shared by the two gate/up GEMM kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace fp4mx {

// silu(g) * u of two fp32 accumulator words: g / (1 + e^-g) * u in fp32 with the
// fast exponential and division intrinsics (relative error well below 2^-15 of the
// result, far under the bf16 rounding that follows; a gate below about -87 gives
// e^-g = inf and a signed zero).
__device__ __forceinline__ float silu_mul(uint32_t gate_bits, uint32_t up_bits) {
    const float g = __uint_as_float(gate_bits);
    return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), __uint_as_float(up_bits));
}

}  // namespace fp4mx
