/*
 * fp4_oracle.c -- CPU oracle for decoding block-scaled FP4 (E2M1) to bf16.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm load this file's library. The GPU library never
 * links, includes or calls it, and it shares no code, header or table with the
 * CUDA kernels.
 *
 * It is deliberately plain: one element at a time, in the order the method is
 * described, with no vectorisation and no reordering of arithmetic. Build with
 * -O2 -ffp-contract=off and without -ffast-math so that every float statement
 * is one IEEE-754 binary32 operation rounded to nearest-even. OpenMP (when the
 * compiler has it) splits only the outermost loop, for the timed CPU baseline.
 *
 * Sources (web pages, cited by title and section):
 *  [MX]  "vllm-project/vllm pull 51583" (prhub digest): CPU MXFP4 unpack,
 *        zero-code special case folded from 4 instructions to 2.
 *        Sections "Motivation" (功能与动机), "Implementation breakdown" (实现拆解),
 *        "Key source snippets" (关键源码片段: vec.h and the pytest file).
 *  [NV]  "sgl-project/sglang pull 34222" (prhub digest): NVFP4 token embedding,
 *        dequantised at gather time. Sections "Implementation breakdown" and
 *        "Key source snippets" (modelopt_quant.py, test_nvfp4_embedding.py).
 *
 * Readings of points the pages leave open are stated next to the code that
 * takes them. Every function here is pinned by the CPU tests
 * (tests/test_oracle_pins.py) to facts the pages or mathematics fix.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* E2M1 codes                                                                */
/* ------------------------------------------------------------------------ */

/* [NV] "Key source snippets", _E2M1_LUT: the low three bits of a code index
 * the magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; bit 3 is the sign. [MX] uses
 * the same 16-code E2M1 codebook (its MXFP4_VALUES table is not printed; the
 * reading taken is this standard codebook). */
static const float kMagnitude[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

/* Value of one 4-bit code as a float (exact: every E2M1 value is a float). */
static float e2m1_value(unsigned code) {
    float magnitude = kMagnitude[code & 7u];
    return (code & 8u) ? -magnitude : magnitude;
}

/* Code of element j of a packed stream. Two codes per byte: the even element
 * in the low nibble, the odd element in the high nibble ([NV] "Key source
 * snippets": codes[:, 0::2] = low 4 bits, codes[:, 1::2] = high 4 bits; the
 * same order is taken for MX, whose CPU register order is a prepacked layout
 * and not a logical order). */
static unsigned code_of(const uint8_t *packed, int64_t j) {
    unsigned byte = packed[j >> 1];
    return (j & 1) ? (byte >> 4) : (byte & 0x0Fu);
}

/* bf16 bit pattern of a float that bf16 represents exactly: bf16 is the upper
 * half of binary32, so for an exactly representable value the low half is 0. */
static uint16_t bf16_bits_of_exact(float v) {
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return (uint16_t)(u >> 16);
}

/* The code -> bf16 table of [MX] "Key source snippets" (LUT built from the 16
 * E2M1 values), one entry at a time. */
uint16_t oracle_e2m1_bf16_bits(unsigned code) {
    return bf16_bits_of_exact(e2m1_value(code & 0x0Fu));
}

/* ------------------------------------------------------------------------ */
/* MXFP4: E8M0 per-32 scale as an integer add into the bf16 exponent field   */
/* ------------------------------------------------------------------------ */

/* [MX] "Motivation": the E8M0 block scale is applied as an integer addition
 * into the bf16 exponent field. The offset added is (E - 127) << 7 (bf16 has 7
 * mantissa bits), taken modulo 2^16: the pages' add is the wrapping 16-bit add
 * (maskz_add_epi16), not the saturating one, so E = 0..255 are all plain
 * exponents (E = 255 is not treated as NaN). */
static uint16_t e8m0_offset(unsigned e8m0) {
    int32_t offset = ((int32_t)e8m0 - 127) * 128;
    return (uint16_t)offset; /* conversion to unsigned: value modulo 2^16 */
}

/* One output element, in the order of the current sequence ([MX]
 * "Implementation breakdown" item 2): a lane whose table bits are non-zero
 * once the sign is cleared (bits & 0x7FFF) gets bits + offset; every other
 * lane -- the two zero codes, +0.0 and -0.0 -- is written as 0x0000. */
static uint16_t mx_element(const uint8_t *packed, const uint8_t *scales, int64_t j) {
    unsigned code = code_of(packed, j);
    uint16_t bits = oracle_e2m1_bf16_bits(code);
    uint16_t offset = e8m0_offset(scales[j >> 5]); /* one E8M0 byte per 32 elements */
    int nonzero = (bits & 0x7FFFu) != 0;
    return nonzero ? (uint16_t)(bits + offset) : (uint16_t)0;
}

/* The same element by the older four-step sequence ([MX] "Implementation
 * breakdown" item 1): find the zero lanes ((bits & 0x7FFF) == 0), add the
 * offset to every lane, then blend 0 back into the zero lanes. The pages
 * report that the two sequences agree on every lane; the tests check it. */
static uint16_t mx_element_old_sequence(const uint8_t *packed, const uint8_t *scales,
                                        int64_t j) {
    unsigned code = code_of(packed, j);
    uint16_t bits = oracle_e2m1_bf16_bits(code);
    uint16_t masked = (uint16_t)(bits & 0x7FFFu);
    int zero_lane = (masked == 0);
    uint16_t sum = (uint16_t)(bits + e8m0_offset(scales[j >> 5]));
    return zero_lane ? (uint16_t)0 : sum;
}

/* Decode n_elems elements of a contiguous stream: packed[n_elems / 2],
 * scales[n_elems / 32], out[n_elems]. n_elems must be a multiple of 32. */
void oracle_mx_unpack(const uint8_t *packed, const uint8_t *scales, int64_t n_elems,
                      uint16_t *out, int threads) {
    int64_t n_blocks = n_elems / 32;
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t b = 0; b < n_blocks; ++b)
        for (int64_t j = b * 32; j < b * 32 + 32; ++j)
            out[j] = mx_element(packed, scales, j);
}

void oracle_mx_unpack_old_sequence(const uint8_t *packed, const uint8_t *scales,
                                   int64_t n_elems, uint16_t *out, int threads) {
    int64_t n_blocks = n_elems / 32;
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t b = 0; b < n_blocks; ++b)
        for (int64_t j = b * 32; j < b * 32 + 32; ++j)
            out[j] = mx_element_old_sequence(packed, scales, j);
}

/* Selected elements only (for full-size workloads): out[i] = element idx[i]. */
void oracle_mx_unpack_at(const uint8_t *packed, const uint8_t *scales, const int64_t *idx,
                         int64_t n_idx, uint16_t *out) {
    for (int64_t i = 0; i < n_idx; ++i)
        out[i] = mx_element(packed, scales, idx[i]);
}

/* ------------------------------------------------------------------------ */
/* NVFP4: e4m3 per-16 block scale x fp32 global scale, rounded to bf16       */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN; there
 * are no infinities. The value is built from its definition. */
float oracle_e4m3_to_f32(uint8_t byte) {
    unsigned sign = byte >> 7;
    unsigned exponent = (byte >> 3) & 0x0Fu;
    unsigned mantissa = byte & 0x07u;
    float magnitude;
    if (exponent == 15 && mantissa == 7)
        magnitude = NAN;
    else if (exponent == 0)
        magnitude = ldexpf((float)mantissa, -9);
    else
        magnitude = ldexpf(1.0f + (float)mantissa / 8.0f, (int)exponent - 7);
    return sign ? -magnitude : magnitude;
}

/* binary32 -> bf16, round to nearest, ties to even: add 0x7FFF plus the lowest
 * kept bit, then truncate. NaN keeps its sign and becomes quiet. */
uint16_t oracle_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lowest_kept = (u >> 16) & 1u;
    u += 0x7FFFu + lowest_kept;
    return (uint16_t)(u >> 16);
}

/* One output element of the NVFP4 gather-dequant ([NV] "Implementation
 * breakdown" item 2, and the reference_dequant loop of the test file): the
 * code's value, times (block scale * global scale), rounded to bf16. The
 * order of the two multiplies is the one the pages' implementation uses,
 * eff = scale.float() * weight_scale_2.float() and then vals * eff, each a
 * separate fp32 operation. */
static uint16_t nv_element(const uint8_t *weight_row, const uint8_t *scale_row,
                           float global_scale, int64_t c, int64_t group_size) {
    unsigned code = code_of(weight_row, c);
    float value = e2m1_value(code);
    float block_scale = oracle_e4m3_to_f32(scale_row[c / group_size]);
    float effective = block_scale * global_scale;
    float scaled = value * effective;
    return oracle_f32_to_bf16_rne(scaled);
}

/* Gather-dequant of num_ids rows: out[t, :] = decode(weight[ids[t]], scale[ids[t]]).
 * weight is [vocab, hidden/2] bytes, scales is [vocab, hidden/group_size] e4m3
 * bytes, out is [num_ids, hidden] bf16 bits. An id outside [0, vocab) gives a
 * row of +0.0 (0x0000); the return value counts such ids. */
int64_t oracle_nv_embedding_gather(const int64_t *ids, int64_t num_ids, const uint8_t *weight,
                                   const uint8_t *scales, float global_scale, int64_t vocab,
                                   int64_t hidden, int64_t group_size, uint16_t *out,
                                   int threads) {
    int64_t bad = 0;
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) reduction(+ : bad) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t t = 0; t < num_ids; ++t) {
        int64_t id = ids[t];
        uint16_t *out_row = out + t * hidden;
        if (id < 0 || id >= vocab) {
            for (int64_t c = 0; c < hidden; ++c)
                out_row[c] = 0;
            bad += 1;
            continue;
        }
        const uint8_t *weight_row = weight + id * (hidden / 2);
        const uint8_t *scale_row = scales + id * (hidden / group_size);
        for (int64_t c = 0; c < hidden; ++c)
            out_row[c] = nv_element(weight_row, scale_row, global_scale, c, group_size);
    }
    return bad;
}

/* Selected elements only: out[i] = element (rows[i], cols[i]) of the gathered
 * output, i.e. column cols[i] of the row for ids[rows[i]]. */
void oracle_nv_embedding_gather_at(const int64_t *ids, const uint8_t *weight,
                                   const uint8_t *scales, float global_scale, int64_t vocab,
                                   int64_t hidden, int64_t group_size, const int64_t *rows,
                                   const int64_t *cols, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) {
        int64_t id = ids[rows[i]];
        if (id < 0 || id >= vocab) {
            out[i] = 0;
            continue;
        }
        out[i] = nv_element(weight + id * (hidden / 2), scales + id * (hidden / group_size),
                            global_scale, cols[i], group_size);
    }
}

/* Dense dequant of a whole NVFP4 table: out[r, :] = decode(weight[r], scale[r])
 * for r = 0..rows-1 -- the same element rule as the gather, for every row in
 * order ("sgl-project/sglang pull 34222", "Comments" and "Risks": a tied lm_head
 * needs the table itself, which the gather-only method cannot serve). */
void oracle_nv_dequant(const uint8_t *weight, const uint8_t *scales, float global_scale,
                       int64_t rows, int64_t hidden, int64_t group_size, uint16_t *out,
                       int threads) {
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t *weight_row = weight + r * (hidden / 2);
        const uint8_t *scale_row = scales + r * (hidden / group_size);
        for (int64_t c = 0; c < hidden; ++c)
            out[r * hidden + c] = nv_element(weight_row, scale_row, global_scale, c, group_size);
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP4 quantise: bf16 -> E2M1 codes + one E8M0 scale per 32 elements       */
/* ------------------------------------------------------------------------ */

/* The pages name the step that produces MXFP4 weights
 * ("vllm-project/vllm pull 51583", "Key source snippets": MXFP4QuantizeUtil
 * .quantize returns packed codes and per-32 scales) but do not print its rule.
 * Reading: the OCP Microscaling (MX) v1.0 conversion.
 *   - shared exponent s = floor(log2(max_i |x_i|)) - 2 (2 = the exponent of
 *     E2M1's largest value 6 = 1.5 * 2^2), clamped below at -127; the E8M0 byte
 *     is s + 127. An all-zero block takes the smallest scale, E8M0 = 0.
 *   - each element is x_i / 2^s rounded to the nearest E2M1 magnitude
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}; on a tie the magnitude with an even code
 *     (mantissa bit 0) wins; magnitudes above 6 saturate to 6. The sign bit of
 *     x_i is kept (so -0.0 and small negatives that round to zero give code 8).
 *   - a block holding Inf or NaN gets the E8M0 NaN byte 0xFF and zero codes. */
static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static unsigned nearest_e2m1_magnitude(double a) {
    unsigned best = 0;
    double best_err = fabs(a - (double)kMagnitude[0]);
    for (unsigned m = 1; m < 8; ++m) {
        double err = fabs(a - (double)kMagnitude[m]);
        if (err < best_err || (err == best_err && (m % 2) == 0 && (best % 2) == 1)) {
            best = m;
            best_err = err;
        }
    }
    return best; /* a > 6 is nearest to 6: saturation */
}

static void mx_quantize_block(const uint16_t *x, uint8_t *packed16, uint8_t *scale) {
    double amax = 0.0;
    int finite = 1;
    for (int i = 0; i < 32; ++i) {
        double v = bf16_value(x[i]);
        if (isnan(v) || isinf(v))
            finite = 0;
        else if (fabs(v) > amax)
            amax = fabs(v);
    }
    if (!finite) {
        *scale = 0xFF;
        memset(packed16, 0, 16);
        return;
    }
    int shared = -127;
    if (amax > 0.0) {
        int e;
        frexp(amax, &e); /* amax = f * 2^e with f in [0.5, 1): floor(log2 amax) = e - 1 */
        shared = (e - 1) - 2;
        if (shared < -127)
            shared = -127;
    }
    *scale = (uint8_t)(shared + 127);
    for (int i = 0; i < 32; i += 2) {
        unsigned codes[2];
        for (int h = 0; h < 2; ++h) {
            double v = bf16_value(x[i + h]);
            double scaled = ldexp(fabs(v), -shared); /* exact: a power-of-two scaling */
            unsigned code = nearest_e2m1_magnitude(scaled);
            if (signbit(v))
                code |= 8u;
            codes[h] = code;
        }
        packed16[i / 2] = (uint8_t)(codes[0] | (codes[1] << 4));
    }
}

/* Quantise n_elems (a multiple of 32) bf16 values: packed[n/2], scales[n/32]. */
void oracle_mx_quantize(const uint16_t *in_bf16, int64_t n_elems, uint8_t *packed,
                        uint8_t *scales, int threads) {
    int64_t n_blocks = n_elems / 32;
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t b = 0; b < n_blocks; ++b)
        mx_quantize_block(in_bf16 + b * 32, packed + b * 16, scales + b);
}

/* Batched (paged) MXFP4 dequant of a KV cache: out[i, :] = the MXFP4 unpack of
 * pool page page_ids[i] ([pool_pages, page_elems/2] codes, [pool_pages,
 * page_elems/32] E8M0). "sgl-project/sglang pull 34222", "Risks" item 3: the KV
 * path scales FP4 by E8M0 powers of two (batched_dequantize), unlike the NVFP4
 * embedding; the element rule taken is the MXFP4 unpack above. A page id outside
 * [0, pool_pages) gives a +0.0 row; the return value counts them. */
int64_t oracle_mx_unpack_pages(const int64_t *page_ids, int64_t num_pages, const uint8_t *packed,
                               const uint8_t *scales, int64_t pool_pages, int64_t page_elems,
                               uint16_t *out, int threads) {
    int64_t bad = 0;
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) reduction(+ : bad) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t i = 0; i < num_pages; ++i) {
        int64_t id = page_ids[i];
        uint16_t *out_row = out + i * page_elems;
        if (id < 0 || id >= pool_pages) {
            for (int64_t j = 0; j < page_elems; ++j)
                out_row[j] = 0;
            bad += 1;
            continue;
        }
        const uint8_t *page = packed + id * (page_elems / 2);
        const uint8_t *page_scales = scales + id * (page_elems / 32);
        for (int64_t j = 0; j < page_elems; ++j)
            out_row[j] = mx_element(page, page_scales, j);
    }
    return bad;
}

/* Threads OpenMP would use (1 when built without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
