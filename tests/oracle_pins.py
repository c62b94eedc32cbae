"""Pins that tie the CPU oracle to facts fixed outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError when
the oracle disagrees with what the pages print, a closed form, an invariant, or a
library routine (torch's float8 / bfloat16 conversions, a bf16 value table). The
pins are shared by ``test_oracle_pins.py`` (the real oracle must pass all) and
``test_oracle_mutants.py`` (every planted mistake must fail at least one).
"""
from __future__ import annotations

import os

import numpy as np
import torch

from block_scaled_fp4_mx_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict[str, list[str]]:
    """Parse a ``key: v1 v2 ...`` fixture (``#`` lines are citations)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            out[key.strip()] = rest.split()
    return out


# ---------------------------------------------------------------------------
# independent references (library routines, definitions)
# ---------------------------------------------------------------------------

def torch_bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns of float64 values that bf16 represents EXACTLY, via torch."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float64))
    return t.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


_BF16_TABLE = None


def _bf16_finite_table():
    """All finite non-negative bf16 values (float64, ascending) and their bit
    patterns, enumerated from torch's bfloat16 type."""
    global _BF16_TABLE
    if _BF16_TABLE is None:
        bits = np.arange(0, 0x7F80, dtype=np.int64)  # +0 .. largest finite
        vals = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
        _BF16_TABLE = (vals, bits.astype(np.uint16))
    return _BF16_TABLE


def bf16_nearest_even(x: float) -> int:
    """Definition of round-to-nearest-even into bf16 for a finite float64 x inside
    the finite bf16 range: the nearest bf16 value, and on a tie the one whose bit
    pattern is even. Works on the value set, not on bit tricks."""
    vals, bits = _bf16_finite_table()
    mag = abs(x)
    sign = 0x8000 if np.signbit(x) else 0
    i = int(np.searchsorted(vals, mag, side="left"))
    if i < len(vals) and vals[i] == mag:
        return sign | int(bits[i])
    lo, hi = i - 1, i
    if hi >= len(vals):
        raise ValueError("outside finite bf16 range")
    dlo, dhi = mag - vals[lo], vals[hi] - mag
    pick = lo if dlo < dhi else hi if dhi < dlo else (lo if bits[lo] % 2 == 0 else hi)
    return sign | int(bits[pick])


def codebook():
    g = golden("e2m1_codebook.txt")
    mags = [float(v) for v in g["magnitudes"]]
    values = [(-mags[c & 7] if c & 8 else mags[c & 7]) for c in range(16)]
    # -0.0 for code 8, written explicitly (``-0.0`` of a Python float).
    values[8] = -0.0
    return values


def nibble_codes(packed: np.ndarray) -> np.ndarray:
    """Codes of a packed stream in element order: even element = low nibble."""
    p = packed.reshape(-1)
    codes = np.empty(p.size * 2, dtype=np.uint8)
    codes[0::2] = p & 0x0F
    codes[1::2] = p >> 4
    return codes


def mx_closed_form(packed, scales) -> np.ndarray:
    """For E8M0 exponents in [2, 252]: bf16(value * 2^(E-127)) for nonzero codes
    and +0.0 for the zero codes. Every such product is exactly representable."""
    codes = nibble_codes(packed)
    e = np.repeat(scales.reshape(-1).astype(np.int64), 32)
    assert e.min() >= 2 and e.max() <= 252
    vals = np.asarray(codebook(), dtype=np.float64)[codes]
    exact = vals * np.exp2((e - 127).astype(np.float64))
    out = torch_bf16_bits(exact)
    out[(codes & 7) == 0] = 0
    return out


# ---------------------------------------------------------------------------
# pins: element conversions
# ---------------------------------------------------------------------------

def pin_e2m1_codebook(o):
    """The code -> bf16 table is the pages' codebook, zero codes 0x0000 / 0x8000."""
    g = golden("e2m1_codebook.txt")
    expect = torch_bf16_bits(codebook())
    got = np.array([o.e2m1_bf16_bits(c) for c in range(16)], dtype=np.uint16)
    assert np.array_equal(got, expect), (got, expect)
    for pair in g["zero_code_bf16"]:
        code, bits = pair.split("=")
        assert o.e2m1_bf16_bits(int(code, 16)) == int(bits, 16)


def pin_e4m3_decoder_matches_torch(o):
    """All 256 e4m3fn codes decode as torch.float8_e4m3fn -> float32 does."""
    ref = torch.arange(256, dtype=torch.int16).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.float().numpy()
    got = np.array([o.e4m3_to_f32(b) for b in range(256)], dtype=np.float32)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))


def _rne_probe_values() -> np.ndarray:
    rng = np.random.default_rng(1234)
    rand_bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # exact ties and near-ties around several exponents, both signs, both parities
    heads = np.array([0x3F80, 0x3F81, 0x4000, 0x4001, 0x0000, 0x0001, 0x007F, 0x0080, 0x7F7F,
                      0x7F7E, 0x3400, 0x3401], dtype=np.uint32)
    tails = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    ties = ((heads[:, None] << 16) | tails[None, :]).reshape(-1)
    ties = np.concatenate([ties, ties | 0x80000000])
    special = np.array([0x7F800000, 0xFF800000, 0x7F7FFFFF, 0xFF7FFFFF, 0x00000001,
                        0x80000001, 0x00800000], dtype=np.uint32)
    return np.concatenate([rand_bits, ties, special]).view(np.float32)


def pin_bf16_rne_matches_torch(o):
    """float32 -> bf16 equals torch's round-to-nearest-even conversion on random bit
    patterns, exact ties, subnormals, the overflow edge and the infinities."""
    vals = _rne_probe_values()
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([o.f32_to_bf16_rne(v) for v in vals], dtype=np.uint16)
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], ref[~nan])
    # NaN stays NaN (bit pattern outside the contract)
    g = got[nan]
    assert np.all(((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0))


# ---------------------------------------------------------------------------
# pins: MXFP4
# ---------------------------------------------------------------------------

def pin_mx_zero_codes_stay_zero(o):
    """The pages' zero bytes x exponents (0..255 ends included) give exactly 0x0000."""
    g = golden("mx_zero_codes.txt")
    expect = int(g["expected_bf16"][0], 16)
    for zb in (int(b, 16) for b in g["zero_bytes"]):
        for e in (int(v) for v in g["e8m0"]):
            packed = np.full(64, zb, dtype=np.uint8)  # 128 lanes, 4 blocks
            scales = np.full(4, e, dtype=np.uint8)
            out = o.mx_unpack(packed, scales)
            assert np.all(out == expect), (hex(zb), e, out[:4])


def pin_mx_negative_zero_all_exponents(o):
    """The -0.0 code against every exponent: 16,384 lanes, all +0.0."""
    g = golden("mx_verification_counts.txt")
    packed = np.full(256 * 32, 0x88, dtype=np.uint8)  # 64 lanes per exponent
    scales = np.repeat(np.arange(256, dtype=np.int64), 2).astype(np.uint8)
    out = o.mx_unpack(packed, scales)
    assert out.size == int(g["negative_zero_lanes"][0])
    assert np.all(out == 0)


def pin_mx_identity_at_127(o):
    """E = 127 is the identity scale: the output is the raw codebook, zero codes +0.0."""
    packed = np.arange(256, dtype=np.int64).astype(np.uint8).repeat(16)  # 16 bytes per block
    scales = np.full(256, 127, dtype=np.uint8)
    out = o.mx_unpack(packed, scales)
    codes = nibble_codes(packed)
    expect = torch_bf16_bits(np.asarray(codebook())[codes])
    expect[(codes & 7) == 0] = 0
    assert np.array_equal(out, expect)


def pin_mx_closed_form_interval(o):
    """Every (byte, E) with E in [2, 252]: the exponent add equals bf16(value * 2^(E-127))
    exactly (the result stays a normal number, so no carry reaches the sign)."""
    x = inputs.mx_exhaustive()
    flat_scales = x.scales.reshape(-1)
    keep = (flat_scales >= 2) & (flat_scales <= 252)
    blocks = np.nonzero(keep)[0]
    packed = x.packed.reshape(-1, 16)[blocks].reshape(-1)
    scales = flat_scales[blocks]
    assert np.array_equal(o.mx_unpack(packed, scales), mx_closed_form(packed, scales))


def pin_mx_exponent_step(o):
    """For a nonzero code, raising E by one adds exactly 0x0080 modulo 2^16 -- the
    scale is an integer add into the exponent field -- at every E from 0 to 254.
    With the closed form at E in [2, 252] this fixes the outputs at E = 0, 1, 253,
    254 and 255 as well."""
    codes = np.arange(16, dtype=np.uint8)
    packed = np.tile(codes | (codes << 4), 2)  # 32 bytes = two blocks per exponent
    outs = []
    for e in range(256):
        outs.append(o.mx_unpack(packed, np.full(2, e, dtype=np.uint8))[:32:2][:16])
    outs = np.stack(outs).astype(np.int64)  # [E, code]
    nonzero = (codes & 7) != 0
    step = (outs[1:, nonzero] - outs[:-1, nonzero]) % 65536
    assert np.all(step == 0x80), np.unique(step)
    assert np.all(outs[:, ~nonzero] == 0)


def pin_mx_mixed_lanes(o):
    """Zero and nonzero codes alternating inside one block, at the pages' exponents:
    zero lanes are +0.0, nonzero lanes follow the closed form (lane semantics)."""
    g = golden("mx_mixed_exponents.txt")
    rng = np.random.default_rng(7)
    for e in (int(v) for v in g["e8m0"]):
        nz = rng.choice([1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15], size=(64, 16))
        zc = rng.choice([0, 8], size=(64, 16))
        lo, hi = nz, zc  # element 2i nonzero, 2i+1 zero
        packed = (lo | (hi << 4)).astype(np.uint8).reshape(-1)
        packed2 = (zc | (nz << 4)).astype(np.uint8).reshape(-1)
        for p in (packed, packed2):
            scales = np.full(p.size // 16, e, dtype=np.uint8)
            out = o.mx_unpack(p, scales)
            assert np.array_equal(out, mx_closed_form(p, scales))
            codes = nibble_codes(p)
            assert np.all(out[(codes & 7) == 0] == 0)
            assert np.all(out[(codes & 7) != 0] != 0)


def pin_mx_two_sequences_agree(o):
    """The current sequence and the older and/cmpeq/add/blend sequence agree on the
    pages' 4,194,304 exhaustive lanes and 1,280,000 random lanes."""
    g = golden("mx_verification_counts.txt")
    # every (byte, E) pair run as one 64-lane vector: 32 copies of the byte, two blocks of E
    byte = np.arange(256, dtype=np.int64)
    e = np.arange(256, dtype=np.int64)
    packed = np.repeat(byte[None, :], 256, axis=0).reshape(-1).astype(np.uint8).repeat(32)
    scales = np.repeat(e, 256).astype(np.uint8).repeat(2)
    a = o.mx_unpack(packed, scales)
    assert a.size == int(g["exhaustive_lanes"][0])
    assert np.array_equal(a, o.mx_unpack_old_sequence(packed, scales))
    x = inputs.mx_random(1, int(g["random_lanes"][0]), seed=11)
    a = o.mx_unpack(x.packed, x.scales)
    assert a.size == int(g["random_lanes"][0])
    assert np.array_equal(a, o.mx_unpack_old_sequence(x.packed, x.scales))


def pin_mx_element_order(o):
    """Even elements come from low nibbles and odd ones from high nibbles; element j
    uses scale byte j // 32 (one E8M0 per 32 consecutive elements)."""
    packed = np.zeros(32, dtype=np.uint8)
    packed[0] = 0x42  # element 0: code 2 (1.0), element 1: code 4 (2.0)
    packed[16] = 0x42  # first byte of the second block
    scales = np.array([127, 128], dtype=np.uint8)
    out = o.mx_unpack(packed, scales)
    assert out[0] == torch_bf16_bits([1.0])[0] and out[1] == torch_bf16_bits([2.0])[0]
    assert out[32] == torch_bf16_bits([2.0])[0] and out[33] == torch_bf16_bits([4.0])[0]
    assert np.all(out[2:32] == 0) and np.all(out[34:] == 0)


def pin_mx_pages_are_unpacked_pool_pages(o):
    """Each output row of the paged dequant is the MXFP4 unpack of the pool page its
    id names (repeats allowed, id shape kept); ids outside the pool give +0.0 rows
    and are counted."""
    pool = inputs.mx_random(9, 256, seed=91, zero_fraction=True)
    dense = o.mx_unpack(pool.packed, pool.scales).reshape(9, 256)
    ids = np.array([[4, 0], [8, 4], [-1, 9]], dtype=np.int64)
    out, bad = o.mx_unpack_pages(ids, pool.packed, pool.scales)
    assert out.shape == (3, 2, 256) and bad == 2
    flat = out.reshape(6, 256)
    for i, pid in enumerate(ids.reshape(-1)):
        if 0 <= pid < 9:
            assert np.array_equal(flat[i], dense[pid])
        else:
            assert np.all(flat[i] == 0)


def pin_mx_sampled_equals_full(o):
    x = inputs.mx_random(8, 256, seed=5)
    full = o.mx_unpack(x.packed, x.scales)
    idx = np.random.default_rng(0).integers(0, full.size, size=500)
    assert np.array_equal(o.mx_unpack_at(x.packed, x.scales, idx), full[idx])


# ---------------------------------------------------------------------------
# pins: MXFP4 quantise (bf16 -> codes + E8M0)
# ---------------------------------------------------------------------------

def _bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns of float64 values (rounded by torch)."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def _quantize_test_blocks(seed=61, n_blocks=4000):
    return inputs.bf16_blocks_wide_range(n_blocks, seed)


def pin_mx_quantize_scale_closed_form(o):
    """The E8M0 byte of a finite block is max(exponent field of its bf16 amax - 2, 0):
    floor(log2 amax) - 2 biased by 127, read straight off the bit pattern (an
    all-zero or subnormal block takes byte 0)."""
    x = _quantize_test_blocks()
    _, scales = o.mx_quantize(x)
    amax_field = ((x & 0x7FFF).max(axis=1) >> 7).astype(np.int64)
    assert np.array_equal(scales.reshape(-1), np.maximum(amax_field - 2, 0).astype(np.uint8))


def pin_mx_quantize_roundtrip_of_decoded_blocks(o):
    """Decoding then quantising then decoding returns the same bf16 values for every
    block the unpack represents exactly (E in [2, 252]): quantise is a right inverse
    of the unpack on its own outputs."""
    x = inputs.mx_random(64, 1024, seed=62, e_lo=2, e_hi=252, zero_fraction=True)
    decoded = o.mx_unpack(x.packed, x.scales).reshape(64, 1024)
    p2, s2 = o.mx_quantize(decoded)
    assert np.array_equal(o.mx_unpack(p2, s2).reshape(64, 1024), decoded)


def pin_mx_quantize_ties_and_saturation(o):
    """Hand-worked rounding cases (nearest, ties to the even code, saturation at 6)."""
    g = golden("mx_quantize_ties.txt")
    for key in ("cases", "saturate"):
        for pair in g[key]:
            val, code = pair.split("=")
            blk = np.zeros(32)
            blk[0] = 6.0 if key == "cases" else 0.0
            blk[1] = float(val)
            p, s = o.mx_quantize(_bf16_bits(blk)[None, :])
            assert s[0, 0] == 127, (val, s)
            got = (p[0, 0] >> 4) & 0xF
            assert got == int(code, 16), (val, hex(got), code)


def pin_mx_quantize_specials(o):
    """All-zero block: scale 0, codes 0 (-0.0 keeps its sign bit: code 8); a block
    holding Inf or NaN: the E8M0 NaN byte 0xFF and zero codes."""
    blk = np.zeros((4, 32))
    blk[1, 5] = -0.0
    blk[2, 9] = np.inf
    blk[3, 0] = np.nan
    bits = _bf16_bits(blk)
    bits[1, 5] = 0x8000
    p, s = o.mx_quantize(bits)
    assert list(s.reshape(-1)) == [0, 0, 0xFF, 0xFF]
    assert np.all(p[0] == 0) and np.all(p[2:] == 0)
    assert (p[1, 2] >> 4) == 8 and np.count_nonzero(p[1]) == 1


def pin_mx_quantize_sign_symmetry_and_order(o):
    """quantise(-x) flips exactly the sign bit of every code; within one block the
    decoded magnitude is non-decreasing in |x|."""
    x = _quantize_test_blocks(seed=63, n_blocks=500)
    p, s = o.mx_quantize(x)
    pn, sn = o.mx_quantize(x ^ 0x8000)
    assert np.array_equal(s, sn) and np.array_equal(pn, p ^ 0x88)
    mags = np.abs(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy())
    codes = nibble_codes(p).reshape(500, 32) & 7
    order = np.argsort(mags, axis=1, kind="stable")
    assert np.all(np.diff(np.take_along_axis(codes, order, axis=1).astype(int), axis=1) >= 0)


def pin_mx_quantize_error_bound(o):
    """Each decoded value is within half a grid step of the input (the grid step at
    magnitude m is 0.5 below 2, 1 below 4, 2 above, times 2^s), except saturated
    values, which decode to exactly +-6 * 2^s."""
    x = _quantize_test_blocks(seed=64, n_blocks=2000)
    x = x[(x & 0x7F80).max(axis=1) >> 7 >= 2]  # blocks whose scale is not clamped
    p, s = o.mx_quantize(x)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    step = np.exp2(s.astype(np.float64) - 127)  # 2^s per block
    mag = np.asarray([0, 0.5, 1, 1.5, 2, 3, 4, 6])[nibble_codes(p).reshape(x.shape) & 7]
    deq = mag * step
    a = np.abs(xv)
    spacing = np.where(a < 2 * step, 0.5, np.where(a < 4 * step, 1.0, 2.0)) * step
    sat = a > 6 * step
    assert np.all(np.abs(a - deq)[~sat] <= spacing[~sat] / 2)
    assert np.all(deq[sat] == (6 * step * np.ones_like(a))[sat])


# ---------------------------------------------------------------------------
# pins: grouped MoE GEMM (activations x unpacked weights)
# ---------------------------------------------------------------------------

def _diag_weights(experts, n, k, e8m0_of_expert):
    """Packed weights whose unpack is 2^(E_e - 127) on the diagonal (code 2 = 1.0)
    and 0 elsewhere."""
    codes = np.zeros((experts, n, k), dtype=np.uint8)
    for j in range(min(n, k)):
        codes[:, j, j] = 2
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    scales = np.zeros((experts, n, k // 32), dtype=np.uint8)
    for e in range(experts):
        scales[e] = e8m0_of_expert(e)
    return packed, scales


def pin_moe_gemm_routes_rows_to_their_expert(o):
    """With expert e's weights 2^e times the identity, each row comes out as its own
    first n values times 2^e of the expert that owns it (empty experts included)."""
    rng = np.random.default_rng(81)
    k, n = 64, 32
    offsets = np.array([0, 3, 3, 10, 11])
    a_bits = _bf16_bits(rng.standard_normal((11, k)))
    packed, scales = _diag_weights(4, n, k, lambda e: 127 + e)
    out, _ = o.mx_moe_gemm(a_bits, offsets, packed, scales)
    a = o.bf16_to_f64(a_bits)
    for e in range(4):
        r0, r1 = offsets[e], offsets[e + 1]
        assert np.array_equal(out[r0:r1], a[r0:r1, :n] * 2.0 ** e)


def pin_moe_gemm_brute_force(o):
    """Small grouped GEMM against a plain triple loop over the decoded values
    (values are dyadic with few bits, so every sum is exact in either order)."""
    rng = np.random.default_rng(82)
    k, n, experts = 64, 32, 2
    offsets = np.array([0, 2, 5])
    a_vals = rng.integers(-8, 9, size=(5, k)) / 4.0
    a_bits = _bf16_bits(a_vals)
    x = inputs.mx_random(experts * n, k, seed=83, e_lo=125, e_hi=129)
    packed = x.packed.reshape(experts, n, k // 2)
    scales = x.scales.reshape(experts, n, k // 32)
    out, absdot = o.mx_moe_gemm(a_bits, offsets, packed, scales)
    codes = nibble_codes(x.packed).reshape(experts, n, k)
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for e in range(experts):
        for r in range(offsets[e], offsets[e + 1]):
            for j in range(n):
                acc = 0.0
                acc_abs = 0.0
                for kk in range(k):
                    c = int(codes[e, j, kk])
                    wv = (-1.0 if c & 8 else 1.0) * mags[c & 7] * 2.0 ** (int(scales[e, j, kk // 32]) - 127)
                    acc += a_vals[r, kk] * wv
                    acc_abs += abs(a_vals[r, kk] * wv)
                assert out[r, j] == acc and absdot[r, j] == acc_abs, (e, r, j)


# ---------------------------------------------------------------------------
# pins: the MoE layer (gate/up GEMM, silu(gate) * up, down GEMM, top-k sum)
# ---------------------------------------------------------------------------

def pin_moe_forward_zero_codes_collapse(o):
    """The pages' zero-code MoE test ("vllm-project/vllm pull 51583", the test with
    N = K = 64, E = 2, M = 4): gate/up weights made only of one zero code at any
    E8M0 give silu(0) * 0 = 0 in every slot, so the whole layer must be exactly 0
    whatever the (nonzero) down weights are."""
    n, k, experts, m_tok = 64, 64, 2, 4
    rng = np.random.default_rng(91)
    a_bits = _bf16_bits(rng.standard_normal((m_tok, k)))
    w2 = inputs.mx_random(experts * k, n, seed=92, e_lo=118, e_hi=126)
    w2p, w2s = w2.packed.reshape(experts, k, n // 2), w2.scales.reshape(experts, k, n // 32)
    for zero_byte in (0x00, 0x88, 0x08, 0x80):
        for e8m0 in (0, 1, 127, 200, 254, 255):
            w1p = np.full((experts, 2 * n, k // 2), zero_byte, dtype=np.uint8)
            w1s = np.full((experts, 2 * n, k // 32), e8m0, dtype=np.uint8)
            r = o.mx_moe_forward(a_bits, np.zeros((m_tok, 1), np.int64),
                                 np.ones((m_tok, 1), np.float32), w1p, w1s, w2p, w2s)
            assert np.all(r["out"] == 0.0), (zero_byte, e8m0)


def _bf16_round_scalar(x: float) -> float:
    """Nearest bf16 value (ties to even) of a Python float, by frexp and round()."""
    import math
    if x == 0.0 or not math.isfinite(x):
        return x
    _, e = math.frexp(x)
    ulp = 2.0 ** (max(e, -125) - 8)
    return round(x / ulp) * ulp


def pin_bf16_round_matches_torch(o):
    """The oracle's float64 -> bf16 rounding equals torch's float32 -> bfloat16
    conversion (a library routine, ties to even) on values that are exact in
    float32, including ties, subnormals and both signs."""
    rng = np.random.default_rng(99)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        (rng.integers(-2 ** 15, 2 ** 15, 4000) * 2.0 + 1) * 2.0 ** -16,  # ties
                        rng.standard_normal(2000) * 2.0 ** -128]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o.bf16_round(x.astype(np.float64)), want)


def pin_moe_forward_brute_force(o):
    """A tiny layer against plain scalar loops over the decoded codes (gate rows
    first, silu(x) = x / (1 + e^-x), both GEMMs, bf16 roundings of act, y and out,
    the weighted top-k sum)."""
    import math
    rng = np.random.default_rng(93)
    m_tok, k, n, experts, topk = 3, 32, 32, 3, 2
    a_vals = rng.integers(-6, 7, size=(m_tok, k)) / 8.0
    a_bits = _bf16_bits(a_vals)
    ids = np.array([[0, 2], [1, 1], [2, 0]])
    wts = np.array([[0.25, 0.75], [0.5, 0.125], [1.0, -0.5]], dtype=np.float32)
    w1 = inputs.mx_random(experts * 2 * n, k, seed=94, e_lo=123, e_hi=127)
    w2 = inputs.mx_random(experts * k, n, seed=95, e_lo=123, e_hi=127)
    r = o.mx_moe_forward(a_bits, ids, wts, w1.packed.reshape(experts, 2 * n, k // 2),
                         w1.scales.reshape(experts, 2 * n, k // 32),
                         w2.packed.reshape(experts, k, n // 2), w2.scales.reshape(experts, k, n // 32))
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    c1 = nibble_codes(w1.packed).reshape(experts, 2 * n, k)
    c2 = nibble_codes(w2.packed).reshape(experts, k, n)
    s1 = w1.scales.reshape(experts, 2 * n, k // 32)
    s2 = w2.scales.reshape(experts, k, n // 32)

    def val(c, e8m0):
        c = int(c)
        return (-1.0 if c & 8 else 1.0) * mags[c & 7] * 2.0 ** (int(e8m0) - 127)

    for m in range(m_tok):
        total = [0.0] * k
        for j in range(topk):
            e = int(ids[m, j])
            hid = []
            for i in range(n):
                gate = sum(a_vals[m, kk] * val(c1[e, i, kk], s1[e, i, kk // 32]) for kk in range(k))
                up = sum(a_vals[m, kk] * val(c1[e, n + i, kk], s1[e, n + i, kk // 32]) for kk in range(k))
                hid.append(_bf16_round_scalar(gate / (1.0 + math.exp(-gate)) * up))
            for c in range(k):
                yc = _bf16_round_scalar(sum(hid[i] * val(c2[e, c, i], s2[e, c, i // 32]) for i in range(n)))
                total[c] += float(wts[m, j]) * yc
        expect = [_bf16_round_scalar(t) for t in total]
        assert np.array_equal(r["out"][m], expect), m


def pin_moe_forward_routing_invariants(o):
    """Permuting tokens permutes the output rows; a slot whose expert id is out of
    range adds nothing (and is counted); two slots on one expert add up like one
    slot with the summed weight."""
    rng = np.random.default_rng(96)
    m_tok, k, n, experts = 5, 64, 32, 3
    a_bits = _bf16_bits(rng.standard_normal((m_tok, k)))
    w1 = inputs.mx_random(experts * 2 * n, k, seed=97, e_lo=120, e_hi=126)
    w2 = inputs.mx_random(experts * k, n, seed=98, e_lo=120, e_hi=126)
    wp = (w1.packed.reshape(experts, 2 * n, k // 2), w1.scales.reshape(experts, 2 * n, k // 32),
          w2.packed.reshape(experts, k, n // 2), w2.scales.reshape(experts, k, n // 32))
    ids = np.array([[0, 1], [2, 2], [1, 0], [0, 2], [2, 1]])
    wts = np.array([[0.5, 0.5], [0.25, 0.5], [1.0, 0.0], [0.75, 0.125], [0.5, 0.25]], np.float32)
    base = o.mx_moe_forward(a_bits, ids, wts, *wp)
    perm = np.array([3, 0, 4, 1, 2])
    r = o.mx_moe_forward(a_bits[perm], ids[perm], wts[perm], *wp)
    assert np.array_equal(r["out"], base["out"][perm])
    bad_ids = ids.copy()
    bad_ids[1, 0] = experts
    bad_ids[4, 1] = -1
    r = o.mx_moe_forward(a_bits, bad_ids, wts, *wp)
    assert r["bad"] == 2
    ref = o.mx_moe_forward(a_bits, bad_ids.clip(0, experts - 1),
                           np.where((bad_ids < 0) | (bad_ids >= experts), 0.0, wts).astype(np.float32), *wp)
    assert np.array_equal(r["out"], ref["out"])
    one = o.mx_moe_forward(a_bits[1:2], np.array([[2]]), np.array([[0.75]], np.float32), *wp)
    assert np.allclose(base["out"][1], one["out"][0], rtol=1e-14, atol=0)


# ---------------------------------------------------------------------------
# pins: NVFP4
# ---------------------------------------------------------------------------

def _nv_single(o, code: int, scale_byte: int, gs) -> int:
    weight = np.full((1, 8), code | (code << 4), dtype=np.uint8)  # hidden 16
    scales = np.array([[scale_byte]], dtype=np.uint8)
    out, _ = o.nv_embedding_gather(np.array([0]), weight, scales, gs)
    assert np.all(out == out[0, 0])
    return int(out[0, 0])


def pin_nv_textbook_scales(o):
    """Block scale 1.0 (e4m3 0x38) with global scale 1.0, and block scale 448 (0x7E)
    with global scale fp32(1/448) (product exactly 1.0), give the codebook itself,
    including -0.0 for code 8."""
    expect = torch_bf16_bits(codebook())
    for sb, gs in ((0x38, np.float32(1.0)), (0x7E, inputs.GLOBAL_SCALE_1_OVER_448)):
        got = np.array([_nv_single(o, c, sb, gs) for c in range(16)], dtype=np.uint16)
        assert np.array_equal(got, expect), (hex(sb), got, expect)


def pin_nv_exact_product(o):
    """For every finite e4m3 block scale and every code, the fp32 order
    (block * global, then * value) rounds to the same bf16 as the exact product
    value * block * global rounded once (the pages' test oracle computes in double),
    for the global scales 1/448, 1, 1/3 and 0.1."""
    vals = codebook()
    bs_all = torch.arange(256, dtype=torch.int16).to(torch.uint8).view(torch.float8_e4m3fn)
    bs_all = bs_all.double().numpy()
    for gs in (inputs.GLOBAL_SCALE_1_OVER_448, np.float32(1.0), np.float32(1 / 3),
               np.float32(0.1)):
        # one row per scale byte: codes 0..15 twice -> hidden 32 (two groups, same scale)
        codes = np.arange(16, dtype=np.uint8)
        row = np.concatenate([codes, codes])
        w_row = (row[0::2] | (row[1::2] << 4)).astype(np.uint8)
        finite = [b for b in range(256) if (b & 0x7F) != 0x7F]
        weight = np.tile(w_row[None, :], (len(finite), 1))
        scales = np.array([[b, b] for b in finite], dtype=np.uint8)
        out, _ = o.nv_embedding_gather(np.arange(len(finite)), weight, scales, gs)
        for i, b in enumerate(finite):
            for c in range(16):
                exact = vals[c] * bs_all[b] * float(gs)  # at most 30 significant bits
                if exact == 0.0:
                    expect = 0x8000 if np.signbit(exact) else 0
                else:
                    expect = bf16_nearest_even(exact)
                assert out[i, c] == expect, (hex(b), c, float(gs), hex(out[i, c]), hex(expect))


def pages_torch_formulation(ids, weight, scales, global_scale, group_size=16):
    """The pages' gather-time dequant re-run with CPU torch tensor ops (flatten ids,
    gather packed rows and scale rows, split nibbles even=low / odd=high, table by
    the low 3 bits, sign by bit 3, times e4m3 scale * fp32 global scale, reshape,
    cast to bf16) -- written from the description of the steps."""
    ids_t = torch.as_tensor(np.asarray(ids, dtype=np.int64))
    flat = ids_t.reshape(-1)
    w = torch.from_numpy(np.ascontiguousarray(weight))[flat]
    s = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn)[flat]
    rows, half = w.shape
    hidden = 2 * half
    codes = torch.empty((rows, hidden), dtype=torch.uint8)
    codes[:, 0::2] = w & 0x0F
    codes[:, 1::2] = w >> 4
    table = torch.tensor([float(v) for v in golden("e2m1_codebook.txt")["magnitudes"]],
                         dtype=torch.float32)
    mag = table[(codes & 7).long()]
    vals = torch.where((codes & 8) != 0, -mag, mag)
    eff = s.float() * torch.tensor(np.float32(global_scale)).float()
    out = vals.view(rows, hidden // group_size, group_size) * eff.unsqueeze(-1)
    out = out.view(*ids_t.shape, hidden).to(torch.bfloat16)
    return out.view(torch.int16).numpy().astype(np.uint16)


def pin_nv_matches_pages_torch(o):
    """Bit-exact (including -0.0) against the pages' tensor formulation on CPU torch."""
    for seed, (vocab, hidden, shape), gs in (
            (21, (50, 64, (7,)), inputs.GLOBAL_SCALE_1_OVER_448),
            (22, (33, 48, (3, 5)), np.float32(0.37)),
            (23, (10, 2880, (4,)), np.float32(1.0))):
        x = inputs.nv_random(vocab, hidden, shape, seed, global_scale=gs)
        got, bad = o.nv_embedding_gather(x.ids, x.weight, x.scales, x.global_scale)
        assert bad == 0
        assert np.array_equal(got, pages_torch_formulation(x.ids, x.weight, x.scales,
                                                           x.global_scale))


def pin_nv_gather_invariants(o):
    """out[t] is the dequantised row ids[t]; repeated ids give identical rows; the id
    shape is kept; an id outside the vocabulary gives a +0.0 row and is counted."""
    x = inputs.nv_random(40, 96, (6,), seed=31)
    dense, bad = o.nv_embedding_gather(np.arange(40), x.weight, x.scales, x.global_scale)
    assert bad == 0
    ids = np.array([[3, 3, 39], [0, 17, 3]], dtype=np.int64)
    got, bad = o.nv_embedding_gather(ids, x.weight, x.scales, x.global_scale)
    assert bad == 0 and got.shape == (2, 3, 96)
    assert np.array_equal(got.reshape(6, 96), dense[ids.reshape(-1)])
    ids_bad = np.array([5, -1, 40, 7], dtype=np.int64)
    got, bad = o.nv_embedding_gather(ids_bad, x.weight, x.scales, x.global_scale)
    assert bad == 2
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    assert np.array_equal(got[0], dense[5]) and np.array_equal(got[3], dense[7])


def pin_nv_dense_is_gather_of_every_row(o):
    """The dense dequant of a table equals the gather of ids 0..vocab-1, row by row,
    and its row r does not depend on the other rows."""
    x = inputs.nv_random(23, 2880, (1,), seed=51)
    dense = o.nv_dequant(x.weight, x.scales, x.global_scale)
    gathered, bad = o.nv_embedding_gather(np.arange(23), x.weight, x.scales, x.global_scale)
    assert bad == 0 and np.array_equal(dense, gathered)
    one = o.nv_dequant(x.weight[7:8], x.scales[7:8], x.global_scale)
    assert np.array_equal(one[0], dense[7])


def pin_nv_sampled_equals_full(o):
    x = inputs.nv_random(30, 64, (9,), seed=41)
    full, _ = o.nv_embedding_gather(x.ids, x.weight, x.scales, x.global_scale)
    rng = np.random.default_rng(1)
    rows = rng.integers(0, 9, size=300)
    cols = rng.integers(0, 64, size=300)
    got = o.nv_embedding_gather_at(x.ids, x.weight, x.scales, x.global_scale, rows, cols)
    assert np.array_equal(got, full[rows, cols])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
