"""GPU parity of the grouped MoE GEMM (MXFP4 weights decoded into the tcgen05 operand).

The oracle is exact (float64 sums of exact bf16 x bf16 products). The GPU sums in
fp32 inside the tensor core, in an order it does not specify, then rounds to bf16,
so the comparison takes the bound of that arithmetic: with S = sum_k |a_k w_k|,
|fp32 sum - exact| <= K * 2^-23 * S (twice the textbook gamma_K = K * 2^-24, which
leaves room for adders that truncate), and the bf16 rounding adds at most 2^-8 of
the magnitude. A dropped K-slice, a swapped operand, a wrong scale or a wrong row
of weights is orders of magnitude outside it.
"""
import numpy as np
import pytest

import block_scaled_fp4_mx_gb300 as fp4
from block_scaled_fp4_mx_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def tolerance(exact, absdot, k):
    return 2.0 ** -8 * np.abs(exact) + (1 + 2.0 ** -8) * k * 2.0 ** -23 * absdot


def run_case(ref, rows, n, k, seed, e_lo=118, e_hi=132, max_rows=None, a_scale=1.0):
    experts = len(rows)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    total = int(offsets[-1])
    rng = np.random.default_rng(seed)
    a_bits = inputs.bf16_normal_bits(rng, max(total, 1) * k, scale=a_scale)[: total * k].reshape(total, k)
    w = inputs.mx_random(experts * n, k, seed + 1, e_lo=e_lo, e_hi=e_hi, zero_fraction=True)
    packed = w.packed.reshape(experts, n, k // 2)
    scales = w.scales.reshape(experts, n, k // 32)
    a_t = torch.from_numpy(a_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    out, status = fp4.fp4_mx_moe_gemm(
        a_t, torch.from_numpy(offsets).to(DEV), torch.from_numpy(packed).to(DEV),
        torch.from_numpy(scales).to(DEV), max(rows) if max_rows is None else max_rows)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    got = out.float().cpu().numpy().astype(np.float64)
    exact, absdot = ref.mx_moe_gemm(a_bits, offsets, packed, scales, threads=ref.max_threads())
    err = np.abs(got - exact)
    tol = tolerance(exact, absdot, k)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outside the bound; first {tuple(i)}: "
                             f"gpu {got[tuple(i)]} exact {exact[tuple(i)]} tol {tol[tuple(i)]}")
    return got, exact


@pytest.mark.parametrize("rows,n,k", [([8, 8, 3, 8], 256, 576), ([100, 70, 100], 256, 576),
                                      ([300, 40], 128, 320)])
def test_negative_zero_codes_equal_positive_zero(rows, n, k):
    """The GEMM's decode lets the zero code with the sign bit set (code 8) through as
    -0.0, where fp4_mx_unpack gives +0.0. As a factor it is the same value: with every
    code 0 of random weights turned into code 8, every output is the same value, and
    bit for bit the same wherever it is not zero (decode-time, 128-token and 256-token
    configurations). Weights of code 8 alone give zeros."""
    experts = len(rows)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    total = int(offsets[-1])
    rng = np.random.default_rng(4242)
    a_bits = inputs.bf16_normal_bits(rng, total * k).reshape(total, k)
    w = inputs.mx_random(experts * n, k, 4243, e_lo=118, e_hi=132, zero_fraction=True)
    packed = w.packed.reshape(experts, n, k // 2)
    lo, hi = packed & 0x0F, packed >> 4
    flipped = (np.where(lo == 0, 8, lo) | (np.where(hi == 0, 8, hi) << 4)).astype(np.uint8)
    assert (lo == 0).any() and (hi == 0).any()
    a_t = torch.from_numpy(a_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    off_t = torch.from_numpy(offsets).to(DEV)
    s_t = torch.from_numpy(w.scales.reshape(experts, n, k // 32)).to(DEV)
    outs = []
    for pk in (packed, flipped, np.full_like(packed, 0x88)):
        out, status = fp4.fp4_mx_moe_gemm(a_t, off_t, torch.from_numpy(pk).to(DEV), s_t, max(rows))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append(out)
    plus, minus, zero = (o.float().cpu().numpy() for o in outs)
    assert np.array_equal(plus, minus)  # as values (-0.0 == +0.0)
    nz = plus != 0
    bits = [o.view(torch.int16).cpu().numpy() for o in outs[:2]]
    assert np.array_equal(bits[0][nz], bits[1][nz])
    assert (zero == 0).all()


@pytest.mark.parametrize("rows,n,k", [([5, 0, 3], 160, 32), ([5, 9], 96, 96), ([100, 70], 256, 32),
                                      ([128, 1], 128, 96), ([300], 128, 32), ([257, 3], 96, 96)])
def test_single_partial_k_slice(oracle_impl, rows, n, k):
    """k of 32 or 96: one K slice of 128 (or of 64 with 256-token slabs), mostly past k
    (the tensor maps read zeros there), in each configuration: decode-time (up to 64
    tokens), 128-token and 256-token."""
    run_case(oracle_impl, rows, n, k, seed=sum(rows) + 7 * n + k)


def test_single_tile(oracle_impl):
    """One expert, one 128 x 128 tile, one 64-wide K slice (four MMAs)."""
    run_case(oracle_impl, [128], 128, 64, seed=1)


def test_k_loop_and_tiles(oracle_impl):
    """Several K slices, several row and column tiles."""
    run_case(oracle_impl, [256], 256, 512, seed=2)


@pytest.mark.parametrize("rows,n,k", [([1], 32, 32), ([77], 96, 2880), ([130, 5], 160, 96),
                                      ([0, 200, 3, 0, 128], 2880 // 2, 256)])
def test_ragged_shapes(oracle_impl, rows, n, k):
    """Ragged rows per expert (including empty experts), n and k that are not
    multiples of the 128 x 64 tile."""
    run_case(oracle_impl, rows, n, k, seed=sum(rows) + n + k)


def test_identity_weights_exact(oracle_impl):
    """Weights 2^e * identity for expert e: the product is exact, so the bf16 output
    must equal the activations times 2^e bit for bit."""
    import oracle_pins
    k, n = 128, 128
    rows = [64, 0, 70]
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    rng = np.random.default_rng(5)
    a_bits = oracle_pins._bf16_bits(rng.standard_normal((134, k)))
    packed, scales = oracle_pins._diag_weights(3, n, k, lambda e: 127 + e)
    out, status = fp4.fp4_mx_moe_gemm(
        torch.from_numpy(a_bits.view(np.int16)).to(DEV).view(torch.bfloat16),
        torch.from_numpy(offsets).to(DEV), torch.from_numpy(packed).to(DEV),
        torch.from_numpy(scales).to(DEV), 70)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    exact, _ = oracle_impl.mx_moe_gemm(a_bits, offsets, packed, scales)
    assert np.array_equal(got, oracle_pins._bf16_bits(exact))


@pytest.mark.parametrize("rows,n,k", [([8] * 4, 704, 2880), ([1, 2, 15, 16, 17], 224, 320),
                                      ([32, 0, 31, 33], 384, 704), ([64, 63, 48, 49], 160, 1088),
                                      ([40, 3], 128, 64), ([5, 32, 17], 256, 2912),
                                      ([70, 2, 33], 288, 1056)])
def test_decode_sized_batches(oracle_impl, rows, n, k):
    """Decode-time batches. Up to 64 tokens per expert: one 128-row weight tile per
    item, MMA N = the expert's tokens rounded up to 16, activation boxes of the
    capacity rounded up to 16 rows, four MMA issuers each summing a quarter of the K
    slices (of 128) into a partial accumulator, read out as the sum of the partials;
    70 tokens: the 128-token configuration. Ragged n (last tiles of 64, 96 and 32 rows)
    and an empty expert included; k = 2912 and 1056 end on a half-empty K slice (the
    tensor map reads zeros past k) after 45 and 16 full ones."""
    run_case(oracle_impl, rows, n, k, seed=sum(rows) + n + k)


@pytest.mark.parametrize("tokens", [8, 32])
def test_decode_sized_full_moe_shape(oracle_impl, tokens):
    """32 experts x 8 or 32 tokens against the gate+up weights [32, 5760, 2880] (the
    benchmark's decode-sized workloads): the whole output against the oracle."""
    run_case(oracle_impl, [tokens] * 32, 5760, 2880, seed=17 + tokens)


def test_moe_gate_up_shape(oracle_impl):
    """32 experts x 128 tokens against the gate+up weights [32, 5760, 2880]."""
    run_case(oracle_impl, [128] * 32, 5760, 2880, seed=7)


@pytest.mark.parametrize("rows,n,k", [([512, 300, 129, 0, 1], 512, 2880), ([256, 255, 257], 288, 704)])
def test_256_token_slabs(oracle_impl, rows, n, k):
    """More than 128 rows per expert: 256-token slabs against one decoded weight
    tile; slabs with at most 128 live tokens (N = 128 MMAs), a ragged last slab
    and an empty expert included."""
    run_case(oracle_impl, rows, n, k, seed=sum(rows) + k)


@pytest.mark.parametrize("rows,n,k", [([320, 321, 576, 577, 33, 260], 192, 320),
                                      ([289, 304, 316, 830], 96, 2880)])
def test_extended_last_slabs(oracle_impl, rows, n, k):
    """An expert's last slab takes up to 64 rows past 256 with a second MMA per K
    step: 320 rows in one item (N = 256 + 64), 321 in two (256, then 65 at
    N = 128), 576 in two (256, 256 + 64), 577 in three; extensions of 4 to 60
    rows (second MMA N = 16 to 64)."""
    run_case(oracle_impl, rows, n, k, seed=sum(rows) + k)


@pytest.mark.parametrize("big", [False, True])
def test_more_experts_than_the_compact_item_list(oracle_impl, big):
    """1030 experts, more than the kernel's per-expert slab prefix holds: the CTAs
    walk the dense item list (every expert gets max_rows' slabs, dead items are
    skipped, no slab extension). Up to 128 rows (two-tile items), then up to 300
    (256-token slabs: 300 rows are a 256-token slab and a 44-token one)."""
    rng = np.random.default_rng(61 + big)
    rows = rng.integers(0, 4, size=1030)
    rows[[5, 700]] = [130, 300] if big else [128, 77]
    run_case(oracle_impl, [int(r) for r in rows], 64, 64, seed=63 + big)


def test_full_size_512_tokens_sampled_rows(oracle_impl):
    """32 experts x 512 tokens against the gate+up weights [32, 5760, 2880] (the
    benchmark's 512-token workload) on the GPU; the oracle recomputes 8 rows of
    experts 0 and 31 (an output row depends on its own activation row only)."""
    experts, rows_e, n, k, sample = 32, 512, 5760, 2880, 8
    rows = [rows_e] * experts
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    total = int(offsets[-1])
    rng = np.random.default_rng(71)
    a_bits = inputs.bf16_normal_bits(rng, total * k).reshape(total, k)
    w = inputs.mx_random(experts * n, k, 72, e_lo=118, e_hi=132, zero_fraction=True)
    packed = w.packed.reshape(experts, n, k // 2)
    scales = w.scales.reshape(experts, n, k // 32)
    a_t = torch.from_numpy(a_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    out, status = fp4.fp4_mx_moe_gemm(a_t, torch.from_numpy(offsets).to(DEV), torch.from_numpy(packed).to(DEV),
                                      torch.from_numpy(scales).to(DEV), rows_e)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_all = out.float().cpu().numpy().astype(np.float64)
    pick = [0, experts - 1]
    sel = np.concatenate([np.arange(offsets[e], offsets[e] + sample) for e in pick])
    sub_off = np.arange(len(pick) + 1, dtype=np.int64) * sample
    exact, absdot = oracle_impl.mx_moe_gemm(a_bits[sel], sub_off, packed[pick], scales[pick],
                                            threads=oracle_impl.max_threads())
    err = np.abs(got_all[sel] - exact)
    tol = tolerance(exact, absdot, k)
    assert (err <= tol).all(), (int((err > tol).sum()), float(err.max()))


def test_256_token_slabs_rows_beyond_capacity_flagged(oracle_impl):
    """The capacity check holds with 256-token slabs as well."""
    k, n = 64, 64
    offsets = torch.tensor([0, 10, 400], dtype=torch.int64, device=DEV)
    a = torch.zeros(400, k, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(2, n, k // 2, dtype=torch.uint8, device=DEV)
    s = torch.full((2, n, k // 32), 127, dtype=torch.uint8, device=DEV)
    _, status = fp4.fp4_mx_moe_gemm(a, offsets, w, s, 256)
    torch.cuda.synchronize()
    assert int(status.item()) == fp4.Status.ERR_SHAPE


@pytest.mark.parametrize("experts", [3, 1030])
def test_inconsistent_offsets_flagged(oracle_impl, experts):
    """Offsets that run past total_rows (expert 1) or decrease (expert 2): those
    experts are not computed, their rows of the output keep what was there, the
    consistent expert 0 is computed, and the status word says FP4_ERR_SHAPE. Three
    experts walk the compact item list, 1,030 the dense one."""
    k, n, total = 64, 64, 60
    offsets = np.full(experts + 1, total, dtype=np.int64)
    offsets[:4] = [0, 20, 80, 60]  # expert 0: rows 0..19; 1: 20..79 (past 60); 2: 80..60
    rng = np.random.default_rng(71)
    a_bits = inputs.bf16_normal_bits(rng, total * k).reshape(total, k)
    w = inputs.mx_random(experts * n, k, seed=72, e_lo=118, e_hi=132)
    packed, scales = w.packed.reshape(experts, n, k // 2), w.scales.reshape(experts, n, k // 32)
    canary = 0x7FC1
    out = torch.full((total, n), canary, dtype=torch.int16, device=DEV)
    _, status = fp4.fp4_mx_moe_gemm(
        torch.from_numpy(a_bits.view(np.int16)).to(DEV).view(torch.bfloat16),
        torch.from_numpy(offsets).to(DEV), torch.from_numpy(packed).to(DEV),
        torch.from_numpy(scales).to(DEV), 64, out=out)
    torch.cuda.synchronize()
    assert int(status.item()) == fp4.Status.ERR_SHAPE
    got = out.cpu().numpy()
    assert (got[20:] == canary).all()
    exact, absdot = oracle_impl.mx_moe_gemm(a_bits[:20], np.array([0, 20], dtype=np.int64),
                                            packed[:1], scales[:1])
    first = out[:20].view(torch.bfloat16).float().cpu().numpy().astype(np.float64)
    assert (np.abs(first - exact) <= tolerance(exact, absdot, k)).all()


def test_large_k(oracle_impl):
    """A long reduction: k = 4160, 65 slices of 64."""
    run_case(oracle_impl, [40, 130], 160, 4096 + 64, seed=11)


def test_unaligned_scales(oracle_impl):
    """Scale buffers at an odd byte address give the same result as aligned ones
    (the E8M0 bytes are read with byte loads)."""
    rows, n, k = [96, 33], 320, 1024
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    rng = np.random.default_rng(12)
    a_bits = inputs.bf16_normal_bits(rng, 129 * k).reshape(129, k)
    w = inputs.mx_random(2 * n, k, 13, e_lo=118, e_hi=132)
    packed = torch.from_numpy(w.packed.reshape(2, n, k // 2)).to(DEV)
    scales_host = w.scales.reshape(2, n, k // 32)
    buf = torch.zeros(scales_host.size + 16, dtype=torch.uint8, device=DEV)
    buf[1:1 + scales_host.size] = torch.from_numpy(scales_host.reshape(-1)).to(DEV)
    scales_odd = buf[1:1 + scales_host.size].view(2, n, k // 32)
    scales_even = torch.from_numpy(scales_host).to(DEV)
    a_t = torch.from_numpy(a_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    off_t = torch.from_numpy(offsets).to(DEV)
    out_odd, st1 = fp4.fp4_mx_moe_gemm(a_t, off_t, packed, scales_odd, 96)
    out_even, st2 = fp4.fp4_mx_moe_gemm(a_t, off_t, packed, scales_even, 96)
    torch.cuda.synchronize()
    assert int(st1.item()) == 0 and int(st2.item()) == 0
    exact, absdot = oracle_impl.mx_moe_gemm(a_bits, offsets, w.packed.reshape(2, n, k // 2),
                                            scales_host)
    assert torch.equal(out_odd.view(torch.int16), out_even.view(torch.int16))
    for got in (out_odd, out_even):
        g = got.float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(g - exact) <= tolerance(exact, absdot, k))


def test_rows_beyond_capacity_flagged(oracle_impl):
    """An expert with more rows than max_rows_per_expert is not computed and the
    status word says FP4_ERR_SHAPE."""
    k, n = 64, 64
    offsets = torch.tensor([0, 10, 300], dtype=torch.int64, device=DEV)
    a = torch.zeros(300, k, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(2, n, k // 2, dtype=torch.uint8, device=DEV)
    s = torch.full((2, n, k // 32), 127, dtype=torch.uint8, device=DEV)
    _, status = fp4.fp4_mx_moe_gemm(a, offsets, w, s, 128)
    torch.cuda.synchronize()
    assert int(status.item()) == fp4.Status.ERR_SHAPE
