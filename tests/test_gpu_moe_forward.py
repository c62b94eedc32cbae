"""GPU parity of the MoE layer (routing, gate/up GEMM with silu(gate) * up, down GEMM,
top-k weighted sum) against the float64 oracle, which rounds act, y and out to bf16
exactly where the layer stores bf16.

The bound follows the kernels' arithmetic stage by stage. Before each bf16 store
the GPU value differs from the oracle's exact value by at most `pre` (below);
rounding then gives the same bf16 value unless a rounding midpoint lies within
`pre` of the exact value, in which case the two can differ by `pre` plus one bf16
spacing:
  act  pre = 1.1 |u| dg + (|silu(g)| + 1.1 dg) du + 2^-15 |act| + 1e-30, with
       dg = (1 + 2^-8) k 2^-23 sum|a w1| the fp32 accumulation bound of the gate
       (du likewise), 2^-15 for fp32 silu with the fast exponential and division
       intrinsics, and 1e-30 for e^-g overflowing to inf below g = -87;
       dg = du = 0 when the inputs make the gate/up sums exact in fp32 (dyadic
       activations and weight scales: every partial sum fits in 24 bits)
  y    pre = dact @ |W2|^T + (1 + 2^-8) n 2^-23 (|act| + dact) @ |W2|^T
  out  pre = sum_j |w_j| dy_j + topk 2^-23 sum_j |w_j| (|y_j| + dy_j).
With dyadic inputs the bound is about the down GEMM's own accumulation bound, so
a swapped gate/up, a wrong activation, a dropped weight or a slot routed to the
wrong expert is far outside it. With normal activations the gate/up bound, taken
worst case through the down GEMM, is loose; those tests add a median-error check.
"""
import numpy as np
import pytest

import block_scaled_fp4_mx_gb300 as fp4
from block_scaled_fp4_mx_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"
EPS = 2.0 ** -23


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def bf16_spacing(x):
    """Spacing of bf16 values at |x| (2^-133 below the smallest normal)."""
    _, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, np.maximum(e, -125) - 8)


def after_rounding(exact, pre):
    """Bound on |bf16(gpu) - bf16(exact)| given |gpu - exact| <= pre: zero unless a
    rounding midpoint lies within pre of exact (checked with half the spacing, so
    the spacing change at a power of two is covered)."""
    sp = bf16_spacing(exact)
    t = np.abs(exact) / sp
    dist_mid = np.abs(t - np.floor(t) - 0.5) * sp * 0.5
    return np.where(pre < dist_mid, 0.0, pre + bf16_spacing(np.abs(exact) + pre))


def forward_bound(r, ids, wts, k, n, topk, exact_gemm1):
    g, u = r["g"], r["u"]
    if exact_gemm1:
        d1 = np.zeros_like(g)
    else:
        dg = (1 + 2.0 ** -8) * k * EPS * r["sg"]
        du = (1 + 2.0 ** -8) * k * EPS * r["su"]
        with np.errstate(over="ignore"):
            silu = g / (1.0 + np.exp(-g))
        d1 = 1.1 * np.abs(u) * dg + (np.abs(silu) + 1.1 * dg) * du
    act_pre = d1 + 2.0 ** -15 * (np.abs(r["act_exact"]) + d1) + 1e-30
    dact = after_rounding(r["act_exact"], act_pre)
    experts = r["w2"].shape[0]
    dy = np.zeros_like(r["y"])
    for e in range(experts):
        ms, js = np.nonzero(ids == e)
        if ms.size == 0:
            continue
        w2abs = np.abs(r["w2"][e]).T  # [n, k]
        pre = dact[ms, js] @ w2abs + (1 + 2.0 ** -8) * n * EPS * ((np.abs(r["act"][ms, js]) + dact[ms, js]) @ w2abs)
        dy[ms, js] = after_rounding(r["y_exact"][ms, js], pre)
    valid = ((ids >= 0) & (ids < experts)).astype(np.float64)
    wabs = np.abs(wts.astype(np.float64)) * valid
    pre = np.einsum("mj,mjc->mc", wabs, dy + topk * EPS * (np.abs(r["y"]) + dy))
    return after_rounding(r["out_exact"], pre)


def make_layer(tokens, k, n, experts, topk, seed, dyadic=True):
    """Random layer. dyadic: activations in {-1, -7/8, ..., 1} and gate/up scales
    2^-2..2^1, so that every gate/up partial sum is exact in fp32."""
    rng = np.random.default_rng(seed)
    if dyadic:
        a_vals = rng.integers(-8, 9, size=(tokens, k)) / 8.0
        a_bits = (a_vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        e1 = (125, 128)
    else:
        a_bits = inputs.bf16_normal_bits(rng, tokens * k).reshape(tokens, k)
        e1 = (119, 125)
    ids = np.stack([rng.permutation(experts)[:topk] for _ in range(tokens)]).astype(np.int32)
    wts = rng.random((tokens, topk)).astype(np.float32)
    wts /= wts.sum(axis=1, keepdims=True)
    w1 = inputs.mx_random(experts * 2 * n, k, seed + 1, e_lo=e1[0], e_hi=e1[1], zero_fraction=True)
    w2 = inputs.mx_random(experts * k, n, seed + 2, e_lo=119, e_hi=125, zero_fraction=True)
    return dict(a_bits=a_bits, ids=ids, wts=wts, dyadic=dyadic,
                w1p=w1.packed.reshape(experts, 2 * n, k // 2), w1s=w1.scales.reshape(experts, 2 * n, k // 32),
                w2p=w2.packed.reshape(experts, k, n // 2), w2s=w2.scales.reshape(experts, k, n // 32))


def run_gpu(L, max_rows=None):
    t = {key: torch.from_numpy(v).to(DEV) for key, v in L.items()
         if isinstance(v, np.ndarray) and key != "a_bits"}
    a = torch.from_numpy(L["a_bits"].view(np.int16)).to(DEV).view(torch.bfloat16)
    out, status = fp4.fp4_mx_moe_forward(a, t["ids"], t["wts"], t["w1p"], t["w1s"], t["w2p"], t["w2s"],
                                         max_rows_per_expert=max_rows)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), int(status.item())


def check(oracle_impl, L, max_rows=None, expect_status=0, oracle_ids=None):
    got, status = run_gpu(L, max_rows)
    assert status == expect_status, f"device status {status}"
    ids = L["ids"] if oracle_ids is None else oracle_ids
    k, n = L["a_bits"].shape[1], L["w2p"].shape[2] * 2
    r = oracle_impl.mx_moe_forward(L["a_bits"], ids, L["wts"], L["w1p"], L["w1s"], L["w2p"], L["w2s"],
                                   threads=oracle_impl.max_threads())
    tol = forward_bound(r, ids, L["wts"], k, n, ids.shape[1], exact_gemm1=L["dyadic"])
    err = np.abs(got - r["out"])
    bad = err > tol
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outside the bound; first {i}: gpu {got[i]} "
                             f"oracle {r['out'][i]} tol {tol[i]}")
    if not L["dyadic"]:  # the worst-case bound is loose here: typical error must still be small
        nz = np.abs(r["out"]) > 0
        assert np.median(err[nz] / np.abs(r["out"][nz])) <= 2.0 ** -6
    return got, r


def test_pages_zero_code_layer_is_exactly_zero():
    """The pages' zero-code MoE test (N = K = 64, E = 2, M = 4, every token on expert
    0): gate/up weights of one zero code at any E8M0 give exact zeros."""
    n, k, experts, tokens = 64, 64, 2, 4
    rng = np.random.default_rng(7)
    a = torch.from_numpy(inputs.bf16_normal_bits(rng, tokens * k).view(np.int16)).to(DEV)
    a = a.view(torch.bfloat16).reshape(tokens, k)
    w2 = inputs.mx_random(experts * k, n, seed=8, e_lo=118, e_hi=126)
    w2p = torch.from_numpy(w2.packed.reshape(experts, k, n // 2)).to(DEV)
    w2s = torch.from_numpy(w2.scales.reshape(experts, k, n // 32)).to(DEV)
    ids = torch.zeros((tokens, 1), dtype=torch.int32, device=DEV)
    wts = torch.ones((tokens, 1), dtype=torch.float32, device=DEV)
    for zero_byte in (0x00, 0x88, 0x08, 0x80):
        for e8m0 in (0, 1, 127, 200, 254, 255):
            w1p = torch.full((experts, 2 * n, k // 2), zero_byte, dtype=torch.uint8, device=DEV)
            w1s = torch.full((experts, 2 * n, k // 32), e8m0, dtype=torch.uint8, device=DEV)
            out, status = fp4.fp4_mx_moe_forward(a, ids, wts, w1p, w1s, w2p, w2s)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert bool((out.float() == 0).all()), (zero_byte, e8m0)


@pytest.mark.parametrize("tokens,k,n,experts,topk", [(1, 32, 32, 1, 1), (40, 128, 96, 5, 2),
                                                     (37, 64, 160, 3, 3), (130, 96, 64, 4, 1),
                                                     (300, 128, 96, 3, 2), (700, 64, 224, 2, 1),
                                                     (400, 32, 32, 2, 1), (100, 192, 96, 4, 2)])
def test_small_layers(oracle_impl, tokens, k, n, experts, topk):
    """Single token and expert; n and k that are not multiples of the tiles; more
    than 128 tokens (256-token slabs: gate and up halves in one tile, N = 128 MMAs
    for slabs with at most 128 live tokens, ragged 64-column tiles, and n = 32: half
    of one 64-column tile); a capacity of 100 (gate and up tiles of 128 rows, K slices
    of 128 ending half-empty); topk 1 to 3."""
    check(oracle_impl, make_layer(tokens, k, n, experts, topk, seed=tokens + k + n))


@pytest.mark.parametrize("topk", [6, 8, 9, 16])
def test_wide_topk(oracle_impl, topk):
    """Top-6 and top-8 take the combine's path that loads every slot's row vector
    before the sum (8 slots at most); top-9 and top-16 its slot-by-slot loop."""
    check(oracle_impl, make_layer(50, 64, 96, 24, topk, seed=71 + topk))


def test_wide_topk_skips_bad_and_dropped_slots(oracle_impl):
    """The slot-by-slot combine (top-12) skips a slot with a bad expert id, and the
    slots of an expert over capacity, as the 8-slot path does."""
    L = make_layer(30, 64, 64, 16, 12, seed=83)
    ids = L["ids"]
    for m in range(ids.shape[0]):  # expert 0 in every token, at slot 5
        hit = np.flatnonzero(ids[m] == 0)
        if hit.size:
            ids[m, hit[0]], ids[m, 5] = ids[m, 5], ids[m, hit[0]]
        else:
            ids[m, 5] = 0
    counts = np.bincount(ids.reshape(-1), minlength=16)
    assert counts[0] == 30 and counts[1:].max() <= 29
    ids[7, 2] = 16  # a bad id in a token that keeps its other slots
    oracle_ids = ids.copy()
    oracle_ids[oracle_ids == 0] = -1  # expert 0 holds 30 rows > capacity 29
    got, status = run_gpu(L, max_rows=29)
    assert status in (fp4.Status.ERR_SHAPE, fp4.Status.ERR_INDEX)
    k, n = L["a_bits"].shape[1], L["w2p"].shape[2] * 2
    r = oracle_impl.mx_moe_forward(L["a_bits"], oracle_ids, L["wts"], L["w1p"], L["w1s"], L["w2p"],
                                   L["w2s"], threads=oracle_impl.max_threads())
    tol = forward_bound(r, oracle_ids, L["wts"], k, n, 12, exact_gemm1=True)
    assert (np.abs(got - r["out"]) <= tol).all()


def test_extended_last_slabs(oracle_impl):
    """Experts holding 300, 320, 321, 577 and 40 rows (top-1 routing fixed per
    token): last slabs extended past 256 tokens by up to 64 in both GEMMs, the
    gate/up epilogue reading accumulator columns 256-319."""
    counts = [300, 320, 321, 577, 40]
    L = make_layer(sum(counts), 64, 96, len(counts), 1, seed=53)
    rng = np.random.default_rng(54)
    L["ids"] = rng.permutation(np.repeat(np.arange(len(counts)), counts)).astype(np.int32)[:, None]
    check(oracle_impl, L)


@pytest.mark.parametrize("tokens,experts", [(64, 5000), (64, 600), (128, 4096), (129, 300)])
def test_many_experts(oracle_impl, tokens, experts):
    """5000 experts: more than the route kernel's shared-memory histogram holds
    (global atomics) and more than the GEMMs' compact item list (dense list). 600 and
    4096 experts with at most 256 slots: one route block scans its own histogram,
    several experts per thread; 129 tokens: 258 slots, two route blocks."""
    check(oracle_impl, make_layer(tokens, 32, 32, experts, 2, seed=57 + experts))


def test_full_size_layer_sampled_tokens(oracle_impl):
    """The benchmark's layer at full size (4096 tokens, top-4 of 32 experts, hidden =
    intermediate = 2880: experts of about 512 +- 22 rows, so 256-token slabs and
    extended last slabs in both GEMMs) on the GPU; the oracle recomputes 8 tokens,
    whose outputs depend on nothing else. Those tokens are routed among experts 0-3
    so that the oracle decodes only four experts' weights."""
    tokens, k, n, experts, topk, sample = 4096, 2880, 2880, 32, 4, 8
    L = make_layer(tokens, k, n, experts, topk, seed=61)
    rng = np.random.default_rng(62)
    L["ids"][:sample] = np.stack([rng.permutation(4) for _ in range(sample)]).astype(np.int32)
    got, status = run_gpu(L)
    assert status == 0, status
    ids, wts = L["ids"][:sample], L["wts"][:sample]
    r = oracle_impl.mx_moe_forward(L["a_bits"][:sample], ids, wts, L["w1p"][:4], L["w1s"][:4],
                                   L["w2p"][:4], L["w2s"][:4], threads=oracle_impl.max_threads())
    tol = forward_bound(r, ids, wts, k, n, topk, exact_gemm1=True)
    err = np.abs(got[:sample] - r["out"])
    bad = err > tol
    assert not bad.any(), (int(bad.sum()), float(err.max()))


def test_decode_step_layer(oracle_impl):
    """A decode-time step: 8 tokens, top-4 of 8 experts, hidden = intermediate = 2880
    (four tokens or so per expert: both GEMMs take one 128-row weight tile per item,
    N = 16 MMAs from four issuers into partial accumulators)."""
    check(oracle_impl, make_layer(8, 2880, 2880, 8, 4, seed=35))


def test_gpt_oss_like_layer(oracle_impl):
    """Hidden 2880, intermediate 2880, 4 experts, top-4 of 64 tokens."""
    check(oracle_impl, make_layer(64, 2880, 2880, 4, 4, seed=31))


def test_gpt_oss_like_layer_128_tokens(oracle_impl):
    """Hidden 2880, intermediate 2880, 4 experts, top-4 of 128 tokens: the gate/up
    GEMM with gate and up tiles of 128 rows and the down GEMM's two-tile items."""
    check(oracle_impl, make_layer(128, 2880, 2880, 4, 4, seed=37))


def test_gpt_oss_like_layer_normal_activations(oracle_impl):
    """The same shapes with normal activations (loose worst-case bound plus the
    median-error check)."""
    check(oracle_impl, make_layer(64, 2880, 2880, 4, 4, seed=33, dyadic=False))


def test_bad_expert_ids_contribute_nothing(oracle_impl):
    L = make_layer(24, 64, 64, 3, 2, seed=41)
    L["ids"][3, 0] = 3
    L["ids"][9, 1] = -2
    check(oracle_impl, L, expect_status=fp4.Status.ERR_INDEX)


def test_repeated_expert_in_one_token(oracle_impl):
    """A token may pick the same expert twice: two rows in that expert's segment."""
    L = make_layer(16, 64, 64, 3, 2, seed=43)
    L["ids"][:, 1] = L["ids"][:, 0]
    check(oracle_impl, L, max_rows=32)


def test_expert_over_capacity_is_dropped_and_flagged(oracle_impl):
    """An expert holding more rows than max_rows_per_expert: its slots contribute
    nothing and the status word says FP4_ERR_SHAPE."""
    L = make_layer(20, 64, 64, 3, 1, seed=45)
    L["ids"][:, 0] = np.where(np.arange(20) < 12, 1, np.arange(20) % 2 * 2).astype(np.int32)
    oracle_ids = L["ids"].copy()
    oracle_ids[oracle_ids == 1] = -1  # expert 1 holds 12 rows > capacity 10
    check(oracle_impl, L, max_rows=10, expect_status=fp4.Status.ERR_SHAPE, oracle_ids=oracle_ids)


def test_zero_capacity_drops_every_slot():
    """max_rows_per_expert = 0: every expert with a slot is over capacity, so the
    layer launches no GEMM work, writes zeros and reports FP4_ERR_SHAPE."""
    L = make_layer(24, 64, 64, 3, 2, seed=111)
    got, status = run_gpu(L, max_rows=0)
    assert status == fp4.Status.ERR_SHAPE
    assert (got == 0).all()


def test_equals_gemm_composition():
    """With top-1 routing and weight 1 the layer is the gate/up GEMM, the activation
    and the down GEMM of the standalone entry point, bit for bit in the down GEMM's
    inputs: compare against fp4_mx_moe_gemm run on the layer's own activations."""
    tokens, k, n, experts = 48, 128, 64, 2
    L = make_layer(tokens, k, n, experts, 1, seed=47)
    order = np.argsort(L["ids"][:, 0], kind="stable")
    L["a_bits"], L["ids"] = L["a_bits"][order], L["ids"][order]
    L["wts"] = np.ones_like(L["wts"])
    got, status = run_gpu(L)
    assert status == 0
    counts = np.bincount(L["ids"][:, 0], minlength=experts)
    offsets = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)).to(DEV)
    a = torch.from_numpy(L["a_bits"].view(np.int16)).to(DEV).view(torch.bfloat16)
    h, st1 = fp4.fp4_mx_moe_gemm(a, offsets, torch.from_numpy(L["w1p"]).to(DEV),
                                 torch.from_numpy(L["w1s"]).to(DEV), int(counts.max()))
    torch.cuda.synchronize()
    assert int(st1.item()) == 0
    # the layer keeps gate/up in fp32; from the bf16 GEMM output the activation can
    # differ by one bf16 step, so compare the layer with a tolerance of a few steps
    hf = h.float()
    act = (torch.nn.functional.silu(hf[:, :n]) * hf[:, n:]).to(torch.bfloat16)
    y, st2 = fp4.fp4_mx_moe_gemm(act, offsets, torch.from_numpy(L["w2p"]).to(DEV),
                                 torch.from_numpy(L["w2s"]).to(DEV), int(counts.max()))
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = y.float().cpu().numpy().astype(np.float64)
    scale = np.abs(ref).max()
    assert np.abs(got - ref).max() <= 0.05 * scale


def test_graph_capture_and_replay(oracle_impl):
    """The layer (one memset and five launches on the caller's stream) can be captured
    in a CUDA graph once and replayed for new activations, routing and weights of the
    top-k written into the captured buffers; each replay matches the oracle for its
    own inputs. 150 rows per expert on average: 256-token slabs."""
    tokens, k, n, experts, topk = 300, 128, 96, 4, 2
    layers = [make_layer(tokens, k, n, experts, topk, seed=91)]
    for seed in (92, 93):  # new activations and routing, the same expert weights
        L = make_layer(tokens, k, n, experts, topk, seed=seed)
        L.update({key: layers[0][key] for key in ("w1p", "w1s", "w2p", "w2s")})
        layers.append(L)
    w = {key: torch.from_numpy(layers[0][key]).to(DEV) for key in ("w1p", "w1s", "w2p", "w2s")}
    a = torch.empty(tokens, k, dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(tokens, topk, dtype=torch.int32, device=DEV)
    wts = torch.empty(tokens, topk, dtype=torch.float32, device=DEV)
    ws = torch.empty(fp4.fp4_mx_moe_workspace_bytes(tokens, topk, experts, n, k), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty(tokens, k, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)

    def load(L):
        a.copy_(torch.from_numpy(L["a_bits"].view(np.int16)).view(torch.bfloat16))
        ids.copy_(torch.from_numpy(L["ids"]))
        wts.copy_(torch.from_numpy(L["wts"]))
        out.zero_()
        status.zero_()

    def call():
        fp4.fp4_mx_moe_forward(a, ids, wts, w["w1p"], w["w1s"], w["w2p"], w["w2s"], out=out,
                               workspace=ws, status=status)

    load(layers[0])
    call()  # eager warm-up: host-side lookups happen outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for L in layers[1:] + layers[:1]:
        load(L)
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.float().cpu().numpy().astype(np.float64)
        r = oracle_impl.mx_moe_forward(L["a_bits"], L["ids"], L["wts"], L["w1p"], L["w1s"], L["w2p"],
                                       L["w2s"], threads=oracle_impl.max_threads())
        tol = forward_bound(r, L["ids"], L["wts"], k, n, topk, exact_gemm1=True)
        assert (np.abs(got - r["out"]) <= tol).all()


@pytest.mark.parametrize("tokens,topk", [(40, 2), (300, 2)])
def test_back_to_back_calls_on_inputs_written_just_before(oracle_impl, tokens, topk):
    """Four layer calls in a row on one stream, with no host synchronisation between
    them: before each call, device copies on the same stream overwrite every input
    (activations, routing, top-k weights and all four weight tensors) in the same
    buffers, and the call reuses one workspace and one output, whose copy is taken
    right after it. The kernels after the routing kernel start while their
    predecessor finishes; each result must still match the oracle for its own
    inputs. 40 tokens: the decode-time GEMMs; 300: 256-token slabs."""
    k, n, experts = 128, 96, 4
    layers = [make_layer(tokens, k, n, experts, topk, seed=500 + i) for i in range(4)]
    keys = ("ids", "wts", "w1p", "w1s", "w2p", "w2s")
    src = [dict({key: torch.from_numpy(L[key]).to(DEV) for key in keys},
                a=torch.from_numpy(L["a_bits"].view(np.int16)).to(DEV).view(torch.bfloat16))
           for L in layers]
    buf = {key: torch.empty_like(src[0][key]) for key in keys + ("a",)}
    ws = torch.empty(fp4.fp4_mx_moe_workspace_bytes(tokens, topk, experts, n, k), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty(tokens, k, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    results = []
    for s in src:
        for key in buf:
            buf[key].copy_(s[key])
        fp4.fp4_mx_moe_forward(buf["a"], buf["ids"], buf["wts"], buf["w1p"], buf["w1s"], buf["w2p"],
                               buf["w2s"], out=out, workspace=ws, status=status)
        results.append(out.clone())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for L, res in zip(layers, results):
        got = res.float().cpu().numpy().astype(np.float64)
        r = oracle_impl.mx_moe_forward(L["a_bits"], L["ids"], L["wts"], L["w1p"], L["w1s"], L["w2p"],
                                       L["w2s"], threads=oracle_impl.max_threads())
        tol = forward_bound(r, L["ids"], L["wts"], k, n, topk, exact_gemm1=True)
        assert (np.abs(got - r["out"]) <= tol).all()


def test_concurrent_host_threads(oracle_impl):
    """Four host threads, each on its own CUDA stream, call the MXFP4 unpack, the
    NVFP4 gather and the layer ten times each into outputs of their own: every result
    equals the oracle's (unpack, gather) or the first single-threaded layer call's,
    bit for bit. The layer is deterministic: the order of rows inside an expert's
    segment changes no value."""
    import threading
    xm = inputs.mx_random(96, 2880, seed=101)
    xn = inputs.nv_random(700, 2048, (128,), seed=102)
    want_m = oracle_impl.mx_unpack(xm.packed, xm.scales).reshape(-1)
    want_n = oracle_impl.nv_embedding_gather(xn.ids, xn.weight, xn.scales, xn.global_scale)[0].reshape(-1)
    p, s = torch.from_numpy(xm.packed).to(DEV), torch.from_numpy(xm.scales).to(DEV)
    ids, w = torch.from_numpy(xn.ids).to(DEV), torch.from_numpy(xn.weight).to(DEV)
    sc = torch.from_numpy(xn.scales).to(DEV)
    gs = torch.tensor([xn.global_scale], dtype=torch.float32, device=DEV)
    L = make_layer(200, 128, 96, 6, 3, seed=103)
    t = {key: torch.from_numpy(L[key]).to(DEV) for key in ("ids", "wts", "w1p", "w1s", "w2p", "w2s")}
    a = torch.from_numpy(L["a_bits"].view(np.int16)).to(DEV).view(torch.bfloat16)

    def layer():
        return fp4.fp4_mx_moe_forward(a, t["ids"], t["wts"], t["w1p"], t["w1s"], t["w2p"], t["w2s"])

    first, st0 = layer()
    torch.cuda.synchronize()
    assert int(st0.item()) == 0
    want_l = first.view(torch.int16).cpu().numpy()
    errors = []

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for r in range(10):
                    om = fp4.fp4_mx_unpack(p, s)
                    on = fp4.fp4_nv_embedding_gather(ids, w, sc, gs)
                    ol, status = layer()
                    stream.synchronize()
                    if not np.array_equal(om.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1), want_m):
                        errors.append(f"thread {i} round {r}: unpack")
                    if not np.array_equal(on.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1), want_n):
                        errors.append(f"thread {i} round {r}: gather")
                    if int(status.item()) != 0 or not np.array_equal(ol.view(torch.int16).cpu().numpy(), want_l):
                        errors.append(f"thread {i} round {r}: layer")
        except Exception as exc:  # noqa: BLE001 -- reported below
            errors.append(f"thread {i}: {exc!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors[:5]
