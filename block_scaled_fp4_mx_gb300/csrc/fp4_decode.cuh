// fp4_decode.cuh -- register-level decode of packed E2M1 codes (sm_103a).
//
// A "word" is 4 packed bytes = 8 codes = 8 bf16 outputs = 16 output bytes.
// Codes go from nibbles to bf16 bit patterns with byte permutes (PRMT) against
// 8-entry byte tables held in registers, so no table lives in local or shared
// memory and nothing is indexed dynamically.
//
// E2M1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} (low 3 bits of a code; bit 3 is
// the sign) have the bf16 patterns
//     0x0000 0x3F00 0x3F80 0x3FC0 0x4000 0x4040 0x4080 0x40C0
// ("sgl-project/sglang pull 34222", "Key source snippets", _E2M1_LUT). The low
// bytes of the eight patterns are the table LO, the high bytes the table HI;
// each table is two 32-bit registers (entries 0-3, entries 4-7).
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

namespace fp4mx {

// Byte tables of the unscaled magnitudes.
constexpr uint32_t kLoA = 0xC0800000u;  // low bytes of entries 0..3: 00 00 80 C0
constexpr uint32_t kLoB = 0xC0804000u;  // low bytes of entries 4..7: 00 40 80 C0
constexpr uint32_t kHiA = 0x3F3F3F00u;  // high bytes of entries 0..3: 00 3F 3F 3F
constexpr uint32_t kHiB = 0x40404040u;  // high bytes of entries 4..7: 40 40 40 40

// PRMT in its default mode: output byte n is byte sel.nibble[n] & 7 of the
// 8-byte value {b:a}; when bit 3 of the nibble is set the selected byte's top
// bit is replicated instead. Every selector used here has bit 3 clear.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

struct ByteTable {
    uint32_t lo_a, lo_b, hi_a, hi_b;
};

// MXFP4: the table of one 32-element block with its E8M0 exponent folded in.
// Entry m (m = 1..7) is (magnitude bits + ((E - 127) << 7)) mod 2^16 and entry
// 0 is +0.0, so both zero codes come out as 0x0000 (the sign of a zero code is
// dropped below) and no per-lane zero test is needed.
// The 16-bit adds are done two at a time in 32-bit words: the magnitudes are
// below 0x8000, so adding the offset's low 15 bits cannot carry across the
// halves, and adding its bit 15 modulo 2^16 is an XOR.
__device__ __forceinline__ ByteTable mx_scaled_table(uint32_t e8m0) {
    const uint32_t offset = ((e8m0 - 127u) << 7) & 0xFFFFu;
    const uint32_t offset2 = offset | (offset << 16);
    const uint32_t low15 = offset2 & 0x7FFF7FFFu;
    const uint32_t top = offset2 & 0x80008000u;
    // pairs of entries: (0,1) (2,3) (4,5) (6,7); the even entry in the low half
    const uint32_t t01 = ((0x3F000000u + low15) ^ top) & 0xFFFF0000u;
    const uint32_t t23 = (0x3FC03F80u + low15) ^ top;
    const uint32_t t45 = (0x40404000u + low15) ^ top;
    const uint32_t t67 = (0x40C04080u + low15) ^ top;
    ByteTable t;
    t.lo_a = prmt(t01, t23, 0x6420u);
    t.hi_a = prmt(t01, t23, 0x7531u);
    t.lo_b = prmt(t45, t67, 0x6420u);
    t.hi_b = prmt(t45, t67, 0x7531u);
    return t;
}

// Look up the 8 codes of `w` in table `t`, flip the sign bit of every code in
// `sign_nibbles` (bit 3 of a nibble set = flip that element) and interleave the
// low and high bytes into four words of two bf16 each (element 2i in the low
// half of word i, matching little-endian memory order).
__device__ __forceinline__ uint4 lookup_word(uint32_t w, const ByteTable &t,
                                             uint32_t sign_nibbles) {
    const uint32_t m = w & 0x77777777u;  // magnitude indices; selector bit 3 clear
    const uint32_t m_hi = m >> 16;
    uint32_t l0 = prmt(t.lo_a, t.lo_b, m);
    uint32_t h0 = prmt(t.hi_a, t.hi_b, m);
    uint32_t l1 = prmt(t.lo_a, t.lo_b, m_hi);
    uint32_t h1 = prmt(t.hi_a, t.hi_b, m_hi);
    // nibble k's bit 3 sits at bit 4k+3; move it to bit 7 of high byte k.
    const uint32_t s4 = sign_nibbles << 4;
    h0 ^= prmt(sign_nibbles, s4, 0x1504u) & 0x80808080u;
    h1 ^= prmt(sign_nibbles, s4, 0x3726u) & 0x80808080u;
    uint4 o;
    o.x = prmt(l0, h0, 0x5140u);
    o.y = prmt(l0, h0, 0x7362u);
    o.z = prmt(l1, h1, 0x5140u);
    o.w = prmt(l1, h1, 0x7362u);
    return o;
}

// MXFP4 decode of one word whose block table is `t`. Only nonzero codes take
// their sign: a nibble's low 3 bits plus 7 sets its bit 3 exactly when they are
// nonzero (no carry leaves the nibble).
__device__ __forceinline__ uint4 mx_decode_word(uint32_t w, const ByteTable &t) {
    const uint32_t m = w & 0x77777777u;
    const uint32_t negative_nonzero = w & (m + 0x77777777u) & 0x88888888u;
    return lookup_word(w, t, negative_nonzero);
}

// MXFP4 decode of one code, written independently of the table path (used by
// the kernel for unaligned buffers).
__device__ __forceinline__ uint16_t mx_decode_code(uint32_t code, uint32_t e8m0) {
    const uint32_t m = code & 7u;
    if (m == 0) return 0;
    const uint32_t magnitude = (m == 1) ? 0x3F00u : 0x3F00u + (m << 6);
    const uint32_t bits = magnitude | ((code & 8u) << 12);
    return (uint16_t)((bits + ((e8m0 - 127u) << 7)) & 0xFFFFu);
}

// e4m3fn byte -> fp32 (exact; through the hardware fp8 -> f16 conversion).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)byte, __NV_E4M3);
    return __half2float(__half(h));
}

// Two fp32 -> one bf16x2 word, round to nearest even: `lo` to the low half.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// NVFP4 decode of one word: every code (including 0x8 = -0.0) takes its sign;
// each value is multiplied by `eff` in fp32 and rounded to bf16.
__device__ __forceinline__ uint4 nv_decode_word(uint32_t w, float eff) {
    const ByteTable t{kLoA, kLoB, kHiA, kHiB};
    const uint4 v = lookup_word(w, t, w & 0x88888888u);
    uint4 o;
    o.x = pack_bf16x2_rn(__fmul_rn(__uint_as_float(v.x << 16), eff),
                         __fmul_rn(__uint_as_float(v.x & 0xFFFF0000u), eff));
    o.y = pack_bf16x2_rn(__fmul_rn(__uint_as_float(v.y << 16), eff),
                         __fmul_rn(__uint_as_float(v.y & 0xFFFF0000u), eff));
    o.z = pack_bf16x2_rn(__fmul_rn(__uint_as_float(v.z << 16), eff),
                         __fmul_rn(__uint_as_float(v.z & 0xFFFF0000u), eff));
    o.w = pack_bf16x2_rn(__fmul_rn(__uint_as_float(v.w << 16), eff),
                         __fmul_rn(__uint_as_float(v.w & 0xFFFF0000u), eff));
    return o;
}

// NVFP4 value of one code as fp32, written independently of the table path.
__device__ __forceinline__ float nv_code_value(uint32_t code) {
    const uint32_t m = code & 7u;
    uint32_t bits = 0;
    if (m == 1) bits = 0x3F000000u;                                   // 0.5
    else if (m >= 2) bits = ((126u + (m >> 1)) << 23) | ((m & 1u) << 22);  // 2^(e-1) * 1.m
    return __uint_as_float(bits | ((code & 8u) << 28));
}

// Streaming (read-once / write-once) global accesses.
__device__ __forceinline__ uint32_t ld_stream(const uint32_t *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) { __stcs(p, v); }

}  // namespace fp4mx
