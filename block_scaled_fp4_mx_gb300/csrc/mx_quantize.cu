// mx_quantize.cu -- bf16 to MXFP4 (E2M1 codes + one E8M0 scale per 32) on sm_103a.
//
// The step before the unpack: "vllm-project/vllm pull 51583", "Key source
// snippets" quantises bf16 weights with MXFP4QuantizeUtil.quantize (packed
// codes, per-32 scales) without printing its rule. The rule used is the OCP
// Microscaling (MX) v1.0 conversion: shared exponent s = floor(log2 amax) - 2
// (clamped at -127; E8M0 = s + 127), each element x / 2^s rounded to nearest
// even on the E2M1 grid with saturation at 6, the sign kept; a block holding
// Inf or NaN gets the E8M0 NaN byte 0xFF and zero codes.
//
// Per 32 elements: 64 bytes in, 16 + 1 bytes out (2.53 bytes per element, 79%
// reads): HBM-bound like the unpack. Four threads share a block, each loading
// one 16-byte quarter (a warp instruction reads 512 contiguous bytes and writes
// 128 contiguous bytes of codes); the block's amax is reduced with two quad
// shuffles. floor(log2 amax) is read off the bf16 exponent field, x / 2^s is an
// exact fp32 multiply by 2^(127 - E) (2^(127 - E) is 2^(127 - E) in fp32 for
// every E in 0..252), and the rounding onto the E2M1 grid is the hardware
// cvt.rn.satfinite.e2m1x2.f32 (two elements per instruction, four per word).
#include "fp4_decode.cuh"
#include "launch.h"

namespace fp4mx {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// E8M0 byte of a block from max(|bits|) over its bf16 patterns (NaN and Inf
// compare above every finite magnitude).
__device__ __forceinline__ uint32_t e8m0_of_amax(uint32_t amax_bits) {
    if (amax_bits >= 0x7F80u) return 0xFFu;
    const int field = (int)(amax_bits >> 7);
    return (uint32_t)(field > 2 ? field - 2 : 0);
}

// Eight bf16 (four 32-bit words, element 2i in the low half of word i) scaled
// by `pow2` -> eight E2M1 codes in one word, element j in nibble j. The hardware
// conversion rounds to nearest even, saturates at +-6 and keeps the sign of a
// result that rounds to zero (-0.0 -> code 8), as the parity tests check.
__device__ __forceinline__ uint32_t e2m1x8_of(const uint4 &v, float pow2) {
    const float f0 = __fmul_rn(__uint_as_float(v.x << 16), pow2);
    const float f1 = __fmul_rn(__uint_as_float(v.x & 0xFFFF0000u), pow2);
    const float f2 = __fmul_rn(__uint_as_float(v.y << 16), pow2);
    const float f3 = __fmul_rn(__uint_as_float(v.y & 0xFFFF0000u), pow2);
    const float f4 = __fmul_rn(__uint_as_float(v.z << 16), pow2);
    const float f5 = __fmul_rn(__uint_as_float(v.z & 0xFFFF0000u), pow2);
    const float f6 = __fmul_rn(__uint_as_float(v.w << 16), pow2);
    const float f7 = __fmul_rn(__uint_as_float(v.w & 0xFFFF0000u), pow2);
    uint32_t d;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(d)
        : "f"(f0), "f"(f1), "f"(f2), "f"(f3), "f"(f4), "f"(f5), "f"(f6), "f"(f7));
    return d;
}

__global__ void __launch_bounds__(kThreads)
mx_quantize_words_kernel(const uint4 *__restrict__ in, uint32_t *__restrict__ packed,
                         uint8_t *__restrict__ scales, int64_t n_quarters) {
    const int64_t base = (int64_t)blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t q = base + u * kThreads;
        v[u] = (q < n_quarters) ? __ldcs(in + q) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t q = base + u * kThreads;
        // max |bits| of this quarter, then of the block (lanes 4j..4j+3)
        const uint32_t m01 = __vmaxu2(v[u].x & 0x7FFF7FFFu, v[u].y & 0x7FFF7FFFu);
        const uint32_t m23 = __vmaxu2(v[u].z & 0x7FFF7FFFu, v[u].w & 0x7FFF7FFFu);
        const uint32_t m = __vmaxu2(m01, m23);
        uint32_t amax = max(m & 0xFFFFu, m >> 16);
        amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        const uint32_t e8m0 = e8m0_of_amax(amax);
        uint32_t codes = 0;
        if (e8m0 != 0xFFu) codes = e2m1x8_of(v[u], __uint_as_float((254u - e8m0) << 23));
        if (q < n_quarters) {
            __stcs(packed + q, codes);
            if ((q & 3) == 0) scales[q >> 2] = (uint8_t)e8m0;
        }
    }
}

// Any alignment (2-byte aligned input): one thread per block, written without
// the hardware conversion -- the E2M1 code is the number of rounding thresholds
// the scaled magnitude passes (a tie rounds to the even code).
__device__ __forceinline__ uint32_t e2m1_code_by_thresholds(uint32_t bits, float pow2) {
    const float a = __fmul_rn(__uint_as_float((bits & 0x7FFFu) << 16), pow2);
    const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                       (a >= 3.5f) + (a > 5.0f);
    return m | ((bits >> 12) & 8u);
}

__global__ void __launch_bounds__(kThreads)
mx_quantize_blocks_kernel(const uint16_t *__restrict__ in, uint8_t *__restrict__ packed,
                          uint8_t *__restrict__ scales, int64_t n_blocks) {
    for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < n_blocks;
         b += (int64_t)gridDim.x * kThreads) {
        const uint16_t *x = in + b * 32;
        uint32_t amax = 0;
        for (int i = 0; i < 32; ++i) amax = max(amax, (uint32_t)(x[i] & 0x7FFFu));
        const uint32_t e8m0 = e8m0_of_amax(amax);
        scales[b] = (uint8_t)e8m0;
        const float pow2 = __uint_as_float((254u - (e8m0 == 0xFFu ? 127u : e8m0)) << 23);
        for (int i = 0; i < 32; i += 2) {
            uint32_t byte = 0;
            if (e8m0 != 0xFFu)
                byte = e2m1_code_by_thresholds(x[i], pow2) |
                       (e2m1_code_by_thresholds(x[i + 1], pow2) << 4);
            packed[b * 16 + i / 2] = (uint8_t)byte;
        }
    }
}

}  // namespace

cudaError_t launch_mx_quantize(const uint16_t *in, uint8_t *packed, uint8_t *scales,
                               int64_t n_elems, cudaStream_t stream) {
    const bool vector_ok = (reinterpret_cast<uintptr_t>(in) % 16 == 0) &&
                           (reinterpret_cast<uintptr_t>(packed) % 4 == 0);
    if (vector_ok) {
        constexpr int64_t kChunk = (int64_t)kThreads * kUnroll;
        constexpr int64_t kMaxGrid = 1ll << 30;
        const int64_t n_quarters = n_elems / 8;
        for (int64_t q0 = 0; q0 < n_quarters; q0 += kMaxGrid * kChunk) {
            const int64_t n = (n_quarters - q0 < kMaxGrid * kChunk) ? n_quarters - q0 : kMaxGrid * kChunk;
            const int grid = (int)((n + kChunk - 1) / kChunk);
            mx_quantize_words_kernel<<<grid, kThreads, 0, stream>>>(
                reinterpret_cast<const uint4 *>(in) + q0,
                reinterpret_cast<uint32_t *>(packed) + q0, scales + q0 / 4, n);
        }
    } else {
        const int64_t n_blocks = n_elems / 32;
        const int64_t blocks = (n_blocks + kThreads - 1) / kThreads;
        const int cap = max_resident_ctas((const void *)mx_quantize_blocks_kernel, kThreads, 5);
        const int grid = (int)(blocks < cap ? blocks : cap);
        mx_quantize_blocks_kernel<<<grid, kThreads, 0, stream>>>(in, packed, scales, n_blocks);
    }
    return cudaGetLastError();
}

}  // namespace fp4mx
