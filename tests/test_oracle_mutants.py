"""Plant plausible mistakes in a COPY of the oracle's C source and check that the
pins catch each one (CPU only; the real oracle source is never modified).

Each mutation is (original snippet, mistaken snippet, what it models). The copy
is compiled into a temporary library and every pin is run against it; at least
one pin must fail.
"""
import os

import pytest

import oracle
import oracle_pins

MUTATIONS = [
    ("(j & 1) ? (byte >> 4) : (byte & 0x0Fu)", "(j & 1) ? (byte & 0x0Fu) : (byte >> 4)",
     "nibble order swapped"),
    ("1.5f, 2.0f, 3.0f, 4.0f", "1.5f, 2.0f, 2.5f, 4.0f", "codebook entry wrong"),
    ("return (code & 8u) ? -magnitude : magnitude;", "return magnitude;", "sign dropped"),
    ("return (code & 8u) ? -magnitude : magnitude;", "return (code & 4u) ? -magnitude : magnitude;",
     "sign taken from the wrong bit"),
    ("((int32_t)e8m0 - 127) * 128", "(127 - (int32_t)e8m0) * 128", "scale offset negated"),
    ("((int32_t)e8m0 - 127) * 128", "((int32_t)e8m0 - 128) * 128", "E8M0 bias off by one"),
    ("((int32_t)e8m0 - 127) * 128", "((int32_t)e8m0 - 127) * 64", "exponent field misplaced"),
    ("uint16_t offset = e8m0_offset(scales[j >> 5]);", "uint16_t offset = e8m0_offset(scales[j >> 4]);",
     "one scale per 16 elements instead of 32"),
    ("int nonzero = (bits & 0x7FFFu) != 0;", "int nonzero = bits != 0;",
     "-0.0 not recognised as a zero code"),
    ("return nonzero ? (uint16_t)(bits + offset) : (uint16_t)0;",
     "return nonzero ? (uint16_t)(bits + offset) : bits;", "zero codes not forced to +0.0"),
    ("return nonzero ? (uint16_t)(bits + offset) : (uint16_t)0;",
     "return nonzero ? (uint16_t)((uint32_t)bits + offset > 0xFFFFu ? 0xFFFFu : bits + offset)"
     " : (uint16_t)0;", "saturating add instead of the wrapping add"),
    ("return nonzero ? (uint16_t)(bits + offset) : (uint16_t)0;",
     "return scales[j >> 5] == 255 ? (uint16_t)0x7FC0 : nonzero ? (uint16_t)(bits + offset)"
     " : (uint16_t)0;", "E8M0 255 read as NaN"),
    ("return zero_lane ? (uint16_t)0 : sum;", "return zero_lane ? bits : sum;",
     "old sequence blends the wrong value"),
    ("(int)exponent - 7)", "(int)exponent - 8)", "e4m3 bias wrong"),
    ("ldexpf((float)mantissa, -9)", "ldexpf((float)mantissa, -10)", "e4m3 subnormal scale wrong"),
    ("1.0f + (float)mantissa / 8.0f", "1.0f + (float)mantissa / 16.0f", "e4m3 mantissa width wrong"),
    ("if (exponent == 15 && mantissa == 7)", "if (exponent == 15)", "e4m3 NaN set too wide"),
    ("u += 0x7FFFu + lowest_kept;", "u += 0x8000u;", "bf16 rounding ties away from zero"),
    ("u += 0x7FFFu + lowest_kept;", "u += 0u;", "bf16 truncation instead of rounding"),
    ("float effective = block_scale * global_scale;", "float effective = block_scale;",
     "global scale dropped"),
    ("float effective = block_scale * global_scale;",
     "float effective = block_scale / global_scale;", "global scale inverted"),
    ("scale_row[c / group_size]", "scale_row[c / 8]", "NVFP4 group of 8 instead of 16"),
    ("const uint8_t *weight_row = weight + id * (hidden / 2);",
     "const uint8_t *weight_row = weight + t * (hidden / 2);", "row gathered by position not id"),
    ("const uint8_t *scale_row = scales + id * (hidden / group_size);",
     "const uint8_t *scale_row = scales + t * (hidden / group_size);",
     "scale row gathered by position not id"),
    ("const uint8_t *scale_row = scales + r * (hidden / group_size);",
     "const uint8_t *scale_row = scales + r * (hidden / 16 / group_size);",
     "dense dequant scale row pitch wrong"),
    ("out[r * hidden + c] = nv_element(", "out[r * (hidden / 2) + c] = nv_element(",
     "dense dequant output row pitch wrong"),
    ("const uint8_t *page_scales = scales + id * (page_elems / 32);",
     "const uint8_t *page_scales = scales + i * (page_elems / 32);",
     "paged dequant: scales of the wrong page"),
    ("if (id < 0 || id >= pool_pages) {", "if (id < 0 || id > pool_pages) {",
     "paged dequant: last valid page id off by one"),
    ("shared = (e - 1) - 2;", "shared = (e - 1) - 1;", "quantise: E2M1 emax taken as 1"),
    ("shared = (e - 1) - 2;", "shared = e - 2;", "quantise: floor(log2) off by one"),
    ("if (err < best_err || (err == best_err && (m % 2) == 0 && (best % 2) == 1)) {",
     "if (err <= best_err) {", "quantise: ties go up instead of to even"),
    ("if (err < best_err || (err == best_err && (m % 2) == 0 && (best % 2) == 1)) {",
     "if (err < best_err) {", "quantise: ties go down instead of to even"),
    ("            if (signbit(v))\n                code |= 8u;", "",
     "quantise: sign dropped"),
    ("        *scale = 0xFF;", "        *scale = 0x00;", "quantise: NaN block scale wrong"),
    ("packed16[i / 2] = (uint8_t)(codes[0] | (codes[1] << 4));",
     "packed16[i / 2] = (uint8_t)(codes[1] | (codes[0] << 4));", "quantise: nibble order swapped"),
    ("        if (shared < -127)\n            shared = -127;", "",
     "quantise: scale not clamped at the smallest E8M0"),
    ("else if (fabs(v) > amax)", "else if (v > amax)", "quantise: amax ignores negatives"),
    ("if (id < 0 || id >= vocab) {\n            for", "if (id < 0 || id > vocab) {\n            for",
     "last valid id off by one"),
]


def _source():
    with open(oracle.SOURCE) as fh:
        return fh.read()


def test_mutations_apply_once():
    src = _source()
    for before, _, what in MUTATIONS:
        assert src.count(before) >= 1, what


@pytest.mark.parametrize("before,after,what", MUTATIONS, ids=[m[2] for m in MUTATIONS])
def test_pins_catch_mutant(before, after, what, tmp_path):
    src = _source().replace(before, after, 1)
    c_path = tmp_path / "mutant.c"
    c_path.write_text(src)
    lib_path = oracle.compile_source(str(c_path), str(tmp_path / "libmutant.so"), openmp=False)
    mutant = oracle.Oracle(oracle.bind(lib_path))
    failed = []
    import warnings
    warnings.simplefilter("ignore", RuntimeWarning)  # a broken mutant may decode NaNs
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the mutant: {what}"
