"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit for bit.

Tolerance is zero for both entry points (bf16 bit patterns compared as uint16):
MXFP4 is integer work, and NVFP4 fixes its fp32 op order and rounding, so both
sides take every rounding decision in the same precision. NaN (only from the e4m3
NaN scale byte, outside the workloads) is compared as "both NaN".
"""
import ctypes

import numpy as np
import pytest

import block_scaled_fp4_mx_gb300 as fp4
from block_scaled_fp4_mx_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
THREADS = 0  # oracle threads: 0 -> all host cores


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(scope="module")
def ref(oracle_impl):
    global THREADS
    THREADS = oracle_impl.max_threads()
    return oracle_impl


def bits(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_same(got: np.ndarray, want: np.ndarray, what: str):
    got, want = got.reshape(-1), want.reshape(-1)
    assert got.shape == want.shape, what
    if not np.array_equal(got, want):
        diff = np.nonzero(got != want)[0]
        i = int(diff[0])
        raise AssertionError(f"{what}: {diff.size} mismatches, first at {i}: "
                             f"gpu {got[i]:#06x} oracle {want[i]:#06x}")


def gpu_mx(x, out=None):
    p = torch.from_numpy(x.packed).to(DEV)
    s = torch.from_numpy(x.scales).to(DEV)
    return fp4.fp4_mx_unpack(p, s, out=out)


def gpu_nv(x, err=None, ids=None):
    ids = x.ids if ids is None else ids
    return fp4.fp4_nv_embedding_gather(
        torch.from_numpy(np.ascontiguousarray(ids)).to(DEV), torch.from_numpy(x.weight).to(DEV),
        torch.from_numpy(x.scales).to(DEV),
        torch.tensor([x.global_scale], dtype=torch.float32, device=DEV), err_flag=err)


# ---------------------------------------------------------------------------
# MXFP4
# ---------------------------------------------------------------------------

def test_mx_exhaustive(ref):
    """Every packed byte x every E8M0 exponent, once each."""
    x = inputs.mx_exhaustive()
    assert_same(bits(gpu_mx(x)), ref.mx_unpack(x.packed, x.scales), "mx exhaustive")


def test_mx_pages_zero_codes(ref):
    """The pages' zero bytes x exponents, as whole blocks: exactly +0.0."""
    for zb in (0x00, 0x88, 0x08, 0x80):
        for e in (0, 1, 127, 200, 254, 255):
            x = inputs.MxInput(np.full((4, 64), zb, np.uint8), np.full((4, 4), e, np.uint8))
            assert np.all(bits(gpu_mx(x)) == 0)


@pytest.mark.parametrize("rows,k,seed", [(1, 32, 1), (3, 64, 2), (7, 2880, 3), (33, 4096, 4),
                                         (1, 1024 * 32 + 32, 5), (129, 96, 6), (2048, 2880, 7)])
def test_mx_random_shapes(ref, rows, k, seed):
    """Several tiles, a ragged tail (word count not a multiple of the CTA chunk),
    random exponents over 0..255 and a 30% share of zero codes."""
    x = inputs.mx_random(rows, k, seed, zero_fraction=(seed % 2 == 0))
    assert_same(bits(gpu_mx(x)), ref.mx_unpack(x.packed, x.scales, THREADS), f"mx {rows}x{k}")


def test_mx_leading_dims_and_empty(ref):
    x = inputs.mx_random(6, 64, seed=9)
    p = torch.from_numpy(x.packed.reshape(2, 3, 32)).to(DEV)
    s = torch.from_numpy(x.scales.reshape(2, 3, 2)).to(DEV)
    out = fp4.fp4_mx_unpack(p, s)
    assert out.shape == (2, 3, 64)
    assert_same(bits(out), ref.mx_unpack(x.packed, x.scales), "mx 3-d")
    empty = fp4.fp4_mx_unpack(torch.empty(0, 16, dtype=torch.uint8, device=DEV),
                              torch.empty(0, 1, dtype=torch.uint8, device=DEV))
    assert empty.shape == (0, 32)


@pytest.mark.parametrize("p_off,o_off", [(1, 0), (0, 2), (3, 6), (2, 8)])
def test_mx_unaligned_buffers(ref, p_off, o_off):
    """Buffers that are not 4 / 16-byte aligned take the byte kernel: same bits."""
    x = inputs.mx_random(5, 352, seed=10 + p_off, zero_fraction=True)
    n = x.n_elems
    pbuf = torch.zeros(x.packed.size + 16, dtype=torch.uint8, device=DEV)
    pbuf[p_off:p_off + x.packed.size] = torch.from_numpy(x.packed.reshape(-1)).to(DEV)
    obuf = torch.zeros(2 * n + 32, dtype=torch.uint8, device=DEV)
    out = obuf[o_off:o_off + 2 * n].view(torch.uint8)
    lib = fp4.load()
    s = torch.from_numpy(x.scales).to(DEV)
    code = lib.fp4_mx_unpack(ctypes.c_void_p(pbuf.data_ptr() + p_off), ctypes.c_void_p(s.data_ptr()),
                             ctypes.c_void_p(obuf.data_ptr() + o_off), x.rows, x.k,
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    got = out.cpu().numpy().view(np.uint16)
    assert_same(got, ref.mx_unpack(x.packed, x.scales), "mx unaligned")


def test_mx_output_canaries(ref):
    """Nothing is written outside the output range."""
    x = inputs.mx_random(17, 320, seed=12)
    n = x.n_elems
    guard = 4096
    buf = torch.full((n + 2 * guard,), 0x5A5A, dtype=torch.int16, device=DEV)
    out = buf[guard:guard + n].view(torch.bfloat16).view(17, 320)
    gpu_mx(x, out=out)
    host = buf.cpu().numpy().view(np.uint16)
    assert np.all(host[:guard] == 0x5A5A) and np.all(host[guard + n:] == 0x5A5A)
    assert_same(host[guard:guard + n], ref.mx_unpack(x.packed, x.scales), "mx canary")


def test_mx_errors_through_binding():
    p = torch.zeros(4, 16, dtype=torch.uint8, device=DEV)
    s = torch.zeros(4, 1, dtype=torch.uint8, device=DEV)
    lib = fp4.load()
    host = (ctypes.c_uint8 * 64)()
    # a plain host pointer is refused before any launch
    code = lib.fp4_mx_unpack(ctypes.addressof(host), s.data_ptr(),
                             torch.empty(4, 32, dtype=torch.bfloat16, device=DEV).data_ptr(),
                             4, 32, None)
    assert code == fp4.Status.ERR_POINTER
    out = torch.empty(4, 32, dtype=torch.bfloat16, device=DEV)
    alias = lib.fp4_mx_unpack(out.data_ptr(), s.data_ptr(), out.data_ptr(), 4, 32, None)
    assert alias == fp4.Status.ERR_ALIAS
    with pytest.raises(ValueError):
        fp4.fp4_mx_unpack(p, torch.zeros(4, 2, dtype=torch.uint8, device=DEV))


# full-size workloads, compared in full (the oracle runs on all host cores)

def test_mx_moe_full(ref):
    for x in inputs.mx_moe():
        out = gpu_mx(x)
        assert_same(bits(out), ref.mx_unpack(x.packed, x.scales, THREADS), x.name)
        del out


def test_mx_stress_full(ref):
    x = inputs.mx_stress()
    out = gpu_mx(x)
    got = bits(out)
    del out
    torch.cuda.empty_cache()
    assert_same(got, ref.mx_unpack(x.packed, x.scales, THREADS), x.name)


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------

def nv_check(ref, x, what, ids=None):
    ids = x.ids if ids is None else ids
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gpu_nv(x, err, ids)
    want, bad = ref.nv_embedding_gather(ids, x.weight, x.scales, x.global_scale, threads=THREADS)
    assert tuple(out.shape) == want.shape
    assert_same(bits(out), want, what)
    assert int(err.item()) == (fp4.Status.ERR_INDEX if bad else 0)
    return bad


def test_nv_embedding_32k(ref):
    x = inputs.nv_embedding_32k()
    assert nv_check(ref, x, x.name) == 0


def test_nv_embedding_200k_full(ref):
    x = inputs.nv_embedding_200k()
    assert nv_check(ref, x, x.name) == 0


@pytest.mark.parametrize("vocab,hidden,shape,seed", [
    (1, 16, (1,), 1), (5, 32, (9,), 2), (64, 2880, (3, 5), 3), (100, 4096 + 16, (17,), 4),
    (300, 8192, (2, 2, 3), 5), (7, 48, (0,), 6)])
def test_nv_shapes(ref, vocab, hidden, shape, seed):
    """One-group rows, ragged segments (hidden 2880 -> 360 words), id shapes of
    several ranks, and no ids at all."""
    x = inputs.nv_random(vocab, hidden, shape, seed)
    nv_check(ref, x, f"nv {vocab}x{hidden}")


@pytest.mark.parametrize("gs", [1.0, 0.37, 1e-36, 3.0e4, -0.5])
def test_nv_global_scales(ref, gs):
    """Global scales other than 1/448, including a negative one (signs of zeros
    flip) and ones that take products to bf16 subnormals / large values."""
    x = inputs.nv_random(50, 256, (40,), seed=7, global_scale=np.float32(gs))
    nv_check(ref, x, f"nv gs={gs}")


def test_nv_every_scale_byte(ref):
    """Every e4m3 byte as a block scale (NaN bytes compared as NaN)."""
    codes = np.arange(16, dtype=np.uint8)
    w_row = np.tile(codes[0::2] | (codes[1::2] << 4), 2)  # hidden 32
    weight = np.tile(w_row[None, :], (256, 1))
    scales = np.stack([np.arange(256), np.arange(256)], axis=1).astype(np.uint8)
    x = inputs.NvInput(np.arange(256, dtype=np.int64), weight, scales, np.float32(1.0 / 3))
    out = bits(gpu_nv(x))
    want, _ = ref.nv_embedding_gather(x.ids, weight, scales, x.global_scale)
    nan_rows = np.array([b for b in range(256) if (b & 0x7F) == 0x7F])
    finite = np.setdiff1d(np.arange(256), nan_rows)
    assert_same(out[finite], want[finite], "nv all scale bytes")
    is_nan = lambda b: ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    assert np.all(is_nan(out[nan_rows][:, [1, 2, 3, 9]]) == is_nan(want[nan_rows][:, [1, 2, 3, 9]]))


@pytest.mark.parametrize("hidden", [2880, 64])
def test_nv_out_of_range_ids(ref, hidden):
    """Bad ids give +0.0 rows and set the error flag; good rows are untouched
    (row-segment kernel at hidden 2880, flat kernel at hidden 64)."""
    x = inputs.nv_random(20, hidden, (6,), seed=8)
    ids = np.array([3, -1, 20, 19, -(2 ** 40), 0], dtype=np.int64)
    assert nv_check(ref, x, "nv bad ids", ids=ids) == 3


def test_nv_repeated_ids_and_dense(ref):
    x = inputs.nv_random(12, 64, (1,), seed=9)
    dense = bits(gpu_nv(x, ids=np.arange(12)))
    rep = bits(gpu_nv(x, ids=np.array([[5, 5], [11, 5]])))
    assert rep.shape == (2, 2, 64)
    assert np.array_equal(rep[0, 0], dense[5]) and np.array_equal(rep[1, 0], dense[11])
    assert np.array_equal(rep[0, 1], rep[1, 1])


@pytest.mark.parametrize("w_off,o_off", [(1, 0), (0, 2), (2, 6)])
def test_nv_unaligned_buffers(ref, w_off, o_off):
    x = inputs.nv_random(30, 160, (11,), seed=20 + w_off)
    lib = fp4.load()
    wbuf = torch.zeros(x.weight.size + 16, dtype=torch.uint8, device=DEV)
    wbuf[w_off:w_off + x.weight.size] = torch.from_numpy(x.weight.reshape(-1)).to(DEV)
    obuf = torch.zeros(x.ids.size * x.hidden * 2 + 32, dtype=torch.uint8, device=DEV)
    ids = torch.from_numpy(x.ids).to(DEV)
    s = torch.from_numpy(x.scales).to(DEV)
    gs = torch.tensor([x.global_scale], dtype=torch.float32, device=DEV)
    code = lib.fp4_nv_embedding_gather(ids.data_ptr(), x.ids.size, wbuf.data_ptr() + w_off,
                                       s.data_ptr(), gs.data_ptr(), x.vocab, x.hidden, 16,
                                       obuf.data_ptr() + o_off, None,
                                       torch.cuda.current_stream().cuda_stream)
    assert code == 0
    got = obuf[o_off:o_off + x.ids.size * x.hidden * 2].cpu().numpy().view(np.uint16)
    want, _ = ref.nv_embedding_gather(x.ids, x.weight, x.scales, x.global_scale)
    assert_same(got, want, "nv unaligned")


def test_nv_output_canaries(ref):
    x = inputs.nv_random(40, 2880, (13,), seed=21)
    n = x.n_elems
    guard = 4096
    buf = torch.full((n + 2 * guard,), 0x5A5A, dtype=torch.int16, device=DEV)
    out = buf[guard:guard + n].view(torch.bfloat16).view(13, 2880)
    fp4.fp4_nv_embedding_gather(torch.from_numpy(x.ids).to(DEV), torch.from_numpy(x.weight).to(DEV),
                                torch.from_numpy(x.scales).to(DEV),
                                torch.tensor([x.global_scale], device=DEV), out=out)
    host = buf.cpu().numpy().view(np.uint16)
    assert np.all(host[:guard] == 0x5A5A) and np.all(host[guard + n:] == 0x5A5A)
    want, _ = ref.nv_embedding_gather(x.ids, x.weight, x.scales, x.global_scale)
    assert_same(host[guard:guard + n], want, "nv canary")


def test_nv_guards_through_binding():
    w = torch.zeros(4, 50, dtype=torch.uint8, device=DEV)  # hidden 100
    s = torch.zeros(4, 6, dtype=torch.uint8, device=DEV)
    ids = torch.zeros(2, dtype=torch.int64, device=DEV)
    gs = torch.ones(1, device=DEV)
    with pytest.raises(fp4.Fp4Error) as e:
        fp4.fp4_nv_embedding_gather(ids, w, s, gs)
    assert e.value.code == fp4.Status.ERR_GROUP
    w = torch.zeros(4, 48, dtype=torch.uint8, device=DEV)  # hidden 96
    with pytest.raises(fp4.Fp4Error) as e:
        fp4.fp4_nv_embedding_gather(ids, w, torch.zeros(4, 3, dtype=torch.uint8, device=DEV), gs,
                                    group_size=32)
    assert e.value.code == fp4.Status.ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# streams and graphs
# ---------------------------------------------------------------------------

def test_side_stream_and_graph_capture(ref):
    """Both calls enqueue on the given stream and can be captured in a CUDA graph."""
    xm = inputs.mx_random(64, 2880, seed=30)
    xn = inputs.nv_random(500, 4096, (64,), seed=31)
    p, s = torch.from_numpy(xm.packed).to(DEV), torch.from_numpy(xm.scales).to(DEV)
    ids, w = torch.from_numpy(xn.ids).to(DEV), torch.from_numpy(xn.weight).to(DEV)
    sc = torch.from_numpy(xn.scales).to(DEV)
    gs = torch.tensor([xn.global_scale], device=DEV)
    out_m = torch.empty(64, 2880, dtype=torch.bfloat16, device=DEV)
    out_n = torch.empty(64, 4096, dtype=torch.bfloat16, device=DEV)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        fp4.fp4_mx_unpack(p, s, out=out_m)
        fp4.fp4_nv_embedding_gather(ids, w, sc, gs, out=out_n)
    side.synchronize()
    want_m = ref.mx_unpack(xm.packed, xm.scales)
    want_n, _ = ref.nv_embedding_gather(xn.ids, xn.weight, xn.scales, xn.global_scale)
    assert_same(bits(out_m), want_m, "side stream mx")
    assert_same(bits(out_n), want_n, "side stream nv")
    out_m.zero_()
    out_n.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fp4.fp4_mx_unpack(p, s, out=out_m)
        fp4.fp4_nv_embedding_gather(ids, w, sc, gs, out=out_n)
    g.replay()
    torch.cuda.synchronize()
    assert_same(bits(out_m), want_m, "graph mx")
    assert_same(bits(out_n), want_n, "graph nv")


# ---------------------------------------------------------------------------
# NVFP4 dense dequant of a whole table
# ---------------------------------------------------------------------------

def gpu_dense(x, out=None):
    return fp4.fp4_nv_dequant(torch.from_numpy(x.weight).to(DEV), torch.from_numpy(x.scales).to(DEV),
                              torch.tensor([x.global_scale], dtype=torch.float32, device=DEV),
                              out=out)


@pytest.mark.parametrize("rows,hidden,seed", [(1, 16, 1), (5, 48, 2), (64, 2880, 3),
                                              (300, 8192, 4), (7, 4096 + 16, 5)])
def test_nv_dequant_shapes(ref, rows, hidden, seed):
    """Flat kernel (hidden < 256) and row-segment kernel with ragged segments."""
    x = inputs.nv_random(rows, hidden, (1,), seed)
    assert_same(bits(gpu_dense(x)), ref.nv_dequant(x.weight, x.scales, x.global_scale),
                f"dense {rows}x{hidden}")


def test_nv_dequant_table_32k(ref):
    x = inputs.nv_embedding_32k()
    assert_same(bits(gpu_dense(x)), ref.nv_dequant(x.weight, x.scales, x.global_scale, threads=THREADS),
                "dense 32000x4096")


def test_nv_dequant_table_200k_full(ref):
    x = inputs.nv_embedding_200k()
    out = gpu_dense(x)
    got = bits(out)
    del out
    torch.cuda.empty_cache()
    assert_same(got, ref.nv_dequant(x.weight, x.scales, x.global_scale, threads=THREADS),
                "dense 200000x8192")


def test_nv_dequant_matches_gather_of_every_id():
    x = inputs.nv_random(97, 2880, (1,), seed=6)
    dense = bits(gpu_dense(x))
    gathered = bits(gpu_nv(x, ids=np.arange(97)))
    assert np.array_equal(dense, gathered)


@pytest.mark.parametrize("w_off,o_off", [(1, 0), (0, 2)])
def test_nv_dequant_unaligned(ref, w_off, o_off):
    x = inputs.nv_random(19, 160, (1,), seed=7 + w_off)
    lib = fp4.load()
    wbuf = torch.zeros(x.weight.size + 16, dtype=torch.uint8, device=DEV)
    wbuf[w_off:w_off + x.weight.size] = torch.from_numpy(x.weight.reshape(-1)).to(DEV)
    obuf = torch.zeros(19 * 160 * 2 + 32, dtype=torch.uint8, device=DEV)
    s = torch.from_numpy(x.scales).to(DEV)
    gs = torch.tensor([x.global_scale], dtype=torch.float32, device=DEV)
    code = lib.fp4_nv_dequant(wbuf.data_ptr() + w_off, s.data_ptr(), gs.data_ptr(), 19, 160, 16,
                              obuf.data_ptr() + o_off, torch.cuda.current_stream().cuda_stream)
    assert code == 0
    got = obuf[o_off:o_off + 19 * 160 * 2].cpu().numpy().view(np.uint16)
    assert_same(got, ref.nv_dequant(x.weight, x.scales, x.global_scale), "dense unaligned")


def test_nv_dequant_canaries_and_guards(ref):
    x = inputs.nv_random(13, 2880, (1,), seed=8)
    n = x.vocab * x.hidden
    guard = 4096
    buf = torch.full((n + 2 * guard,), 0x5A5A, dtype=torch.int16, device=DEV)
    gpu_dense(x, out=buf[guard:guard + n].view(torch.bfloat16).view(13, 2880))
    host = buf.cpu().numpy().view(np.uint16)
    assert np.all(host[:guard] == 0x5A5A) and np.all(host[guard + n:] == 0x5A5A)
    assert_same(host[guard:guard + n], ref.nv_dequant(x.weight, x.scales, x.global_scale), "dense canary")
    with pytest.raises(fp4.Fp4Error) as e:
        fp4.fp4_nv_dequant(torch.zeros(4, 50, dtype=torch.uint8, device=DEV),
                           torch.zeros(4, 6, dtype=torch.uint8, device=DEV), torch.ones(1, device=DEV))
    assert e.value.code == fp4.Status.ERR_GROUP


# ---------------------------------------------------------------------------
# MXFP4 quantise (bf16 -> codes + E8M0)
# ---------------------------------------------------------------------------

def gpu_quantize(x_bits: np.ndarray):
    t = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(DEV).view(torch.bfloat16)
    p, s = fp4.fp4_mx_quantize(t)
    return p.cpu().numpy(), s.cpu().numpy()


def assert_same_bytes(got, want, what):
    got, want = got.reshape(-1), want.reshape(-1)
    if not np.array_equal(got, want):
        i = int(np.nonzero(got != want)[0][0])
        raise AssertionError(f"{what}: first mismatch at {i}: gpu {got[i]:#04x} oracle {want[i]:#04x}")


@pytest.mark.parametrize("n_blocks,seed", [(1, 1), (3, 2), (33, 3), (4000, 4), (1024 * 8 + 3, 5)])
def test_mx_quantize_wide_range(ref, n_blocks, seed):
    """Blocks over the whole bf16 exponent range (zeros, subnormals, the top of the
    range, negatives), ragged counts of blocks."""
    x = inputs.bf16_blocks_wide_range(n_blocks, seed)
    p, s = gpu_quantize(x)
    wp, ws = ref.mx_quantize(x)
    assert_same_bytes(s, ws, "quantise scales")
    assert_same_bytes(p, wp, "quantise codes")


def test_mx_quantize_ties_specials_and_signs(ref):
    """Hand-worked ties, saturation, +-0, Inf and NaN blocks, negatives rounding to 0."""
    import oracle_pins
    g = oracle_pins.golden("mx_quantize_ties.txt")
    rows = []
    for key in ("cases", "saturate"):
        for pair in g[key]:
            blk = np.zeros(32)
            blk[0] = 6.0 if key == "cases" else 0.0
            blk[1] = float(pair.split("=")[0])
            rows.append(blk)
    x = oracle_pins._bf16_bits(np.stack(rows))
    x[len(rows) - 1, 5] = 0x8000  # -0.0
    special = np.zeros((4, 32), np.uint16)
    special[1, 3] = 0x7F80   # +Inf
    special[2, 7] = 0xFFC1   # NaN
    special[3, :] = 0x8001   # negative subnormals
    x = np.concatenate([x, special])
    p, s = gpu_quantize(x)
    wp, ws = ref.mx_quantize(x)
    assert_same_bytes(s, ws, "special scales")
    assert_same_bytes(p, wp, "special codes")


def test_mx_quantize_roundtrip_through_unpack(ref):
    """GPU quantise of GPU-decoded blocks returns codes that decode to the same values."""
    x = inputs.mx_random(64, 2880, seed=70, e_lo=2, e_hi=252, zero_fraction=True)
    decoded = gpu_mx(x)
    p, s = fp4.fp4_mx_quantize(decoded)
    assert_same(bits(fp4.fp4_mx_unpack(p, s)), bits(decoded), "roundtrip")


def test_mx_quantize_moe_full(ref):
    """The bf16 MoE weights (normal / 10) quantised in full."""
    for w in inputs.bf16_moe():
        p, s = gpu_quantize(w.x)
        wp, ws = ref.mx_quantize(w.x, threads=THREADS)
        assert_same_bytes(s, ws, w.name + " scales")
        assert_same_bytes(p, wp, w.name + " codes")


@pytest.mark.parametrize("x_off,p_off", [(2, 0), (0, 1), (6, 3)])
def test_mx_quantize_unaligned(ref, x_off, p_off):
    """Buffers off the 16 / 4-byte boundaries take the per-block kernel: same bytes."""
    x = inputs.bf16_blocks_wide_range(37, seed=9)
    n = x.size
    xbuf = torch.zeros(2 * n + 32, dtype=torch.uint8, device=DEV)
    xbuf[x_off:x_off + 2 * n] = torch.from_numpy(x.reshape(-1).view(np.uint8)).to(DEV)
    pbuf = torch.zeros(n // 2 + 32, dtype=torch.uint8, device=DEV)
    sbuf = torch.zeros(n // 32 + 32, dtype=torch.uint8, device=DEV)
    lib = fp4.load()
    code = lib.fp4_mx_quantize(xbuf.data_ptr() + x_off, pbuf.data_ptr() + p_off, sbuf.data_ptr() + 5,
                               37, 32, torch.cuda.current_stream().cuda_stream)
    assert code == 0
    wp, ws = ref.mx_quantize(x)
    assert_same_bytes(pbuf[p_off:p_off + n // 2].cpu().numpy(), wp, "unaligned codes")
    assert_same_bytes(sbuf[5:5 + n // 32].cpu().numpy(), ws, "unaligned scales")
    assert int(pbuf[:p_off].sum()) == 0 and int(pbuf[p_off + n // 2:].sum()) == 0
    assert int(sbuf[:5].sum()) == 0 and int(sbuf[5 + n // 32:].sum()) == 0


def test_mx_quantize_errors():
    lib = fp4.load()
    x = torch.zeros(2, 64, dtype=torch.bfloat16, device=DEV)
    p = torch.zeros(2, 32, dtype=torch.uint8, device=DEV)
    s = torch.zeros(2, 2, dtype=torch.uint8, device=DEV)
    assert lib.fp4_mx_quantize(x.data_ptr() + 1, p.data_ptr(), s.data_ptr(), 2, 64, None) == fp4.Status.ERR_ALIGN
    assert lib.fp4_mx_quantize(x.data_ptr(), x.data_ptr() + 8, s.data_ptr(), 2, 64, None) == fp4.Status.ERR_ALIAS
    with pytest.raises(ValueError):
        fp4.fp4_mx_quantize(torch.zeros(2, 48, dtype=torch.bfloat16, device=DEV))


# ---------------------------------------------------------------------------
# paged MXFP4 dequant (KV cache)
# ---------------------------------------------------------------------------

def gpu_pages(ids, pool, err=None):
    return fp4.fp4_mx_unpack_pages(torch.from_numpy(np.ascontiguousarray(ids)).to(DEV),
                                   torch.from_numpy(pool.packed).to(DEV),
                                   torch.from_numpy(pool.scales).to(DEV), err_flag=err)


@pytest.mark.parametrize("pages,elems,ids_shape,seed", [(5, 32, (7,), 1), (9, 64, (3, 4), 2),
                                                        (40, 2880, (33,), 3), (64, 16384, (2, 16), 4)])
def test_mx_pages_shapes(ref, pages, elems, ids_shape, seed):
    """Flat kernel (pages under 256 codes), segment kernel with ragged segments."""
    pool = inputs.mx_random(pages, elems, seed, zero_fraction=True)
    ids = np.random.default_rng(seed).integers(0, pages, size=ids_shape).astype(np.int64)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = gpu_pages(ids, pool, err)
    want, bad = ref.mx_unpack_pages(ids, pool.packed, pool.scales)
    assert tuple(got.shape) == want.shape and bad == 0 and int(err.item()) == 0
    assert_same(bits(got), want, f"pages {pages}x{elems}")


@pytest.mark.parametrize("elems", [64, 2880])
def test_mx_pages_bad_ids(ref, elems):
    pool = inputs.mx_random(6, elems, 7)
    ids = np.array([2, -1, 6, 5, 2, 10 ** 12], dtype=np.int64)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = bits(gpu_pages(ids, pool, err))
    want, bad = ref.mx_unpack_pages(ids, pool.packed, pool.scales)
    assert bad == 3 and int(err.item()) == fp4.Status.ERR_INDEX
    assert_same(got, want, "pages bad ids")


def test_mx_pages_unaligned(ref):
    pool = inputs.mx_random(11, 96, 8, zero_fraction=True)
    ids = np.array([3, 0, 10, 3], dtype=np.int64)
    pbuf = torch.zeros(pool.packed.size + 16, dtype=torch.uint8, device=DEV)
    pbuf[1:1 + pool.packed.size] = torch.from_numpy(pool.packed.reshape(-1)).to(DEV)
    obuf = torch.zeros(4 * 96 * 2 + 32, dtype=torch.uint8, device=DEV)
    lib = fp4.load()
    t_ids = torch.from_numpy(ids).to(DEV)
    s = torch.from_numpy(pool.scales).to(DEV)
    code = lib.fp4_mx_unpack_pages(t_ids.data_ptr(), 4, pbuf.data_ptr() + 1, s.data_ptr(), 11, 96,
                                   obuf.data_ptr() + 2, None, torch.cuda.current_stream().cuda_stream)
    assert code == 0
    want, _ = ref.mx_unpack_pages(ids, pool.packed, pool.scales)
    assert_same(obuf[2:2 + 4 * 96 * 2].cpu().numpy().view(np.uint16), want, "pages unaligned")


def test_mx_pages_kv_workload(ref):
    """The KV workload: 8,192 pages of 16,384 codes from a 32,768-page pool."""
    kv = inputs.kv_pages()
    got = bits(gpu_pages(kv.page_ids, kv.pool))
    want, bad = ref.mx_unpack_pages(kv.page_ids, kv.pool.packed, kv.pool.scales, threads=THREADS)
    assert bad == 0
    assert_same(got, want, kv.name)
