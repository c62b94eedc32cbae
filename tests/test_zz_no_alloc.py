"""fp4_mx_moe_forward_noalloc: the MoE layer on the library's static device scratch.

This entry point serves callers that cannot allocate device memory themselves (a
host application that owns all of it, or a path where an allocation must not
happen); the file is named so that pytest collects it after the other test
files, but every test here also passes alone, first or last in a process.

Host side (no GPU): the entry points are exported, the scratch size is reported,
and a layer that needs more scratch than the static area is rejected before any
CUDA call. GPU: the result equals fp4_mx_moe_forward with a caller workspace bit
for bit on two calls in a row, also for a layer whose scratch reaches to within
3 KiB of the end of the area; once the area is loaded, repeated calls leave the
device's free memory unchanged (nothing is allocated); the area is reused across
layer sizes; an oversized layer launches nothing.
"""
import numpy as np
import pytest

import block_scaled_fp4_mx_gb300 as fp4
from block_scaled_fp4_mx_gb300 import inputs

torch = pytest.importorskip("torch")


def test_static_scratch_size_and_rejection():
    lib = fp4.load()
    cap = lib.fp4_mx_moe_static_scratch_bytes()
    assert cap == 288 << 20
    # 4096 tokens, top-4, hidden = intermediate = 2880 fits; twice the tokens does not
    assert lib.fp4_mx_moe_workspace_bytes(4096, 4, 32, 2880, 2880) <= cap
    assert lib.fp4_mx_moe_workspace_bytes(8192, 4, 32, 2880, 2880) > cap
    base = 1 << 40  # fake device addresses: the size check comes before any CUDA call
    code = lib.fp4_mx_moe_forward_noalloc(base, base + (1 << 20), base + (2 << 20), 8192, 4, 32,
                                          8192, base + (3 << 20), base + (4 << 20),
                                          base + (5 << 20), base + (6 << 20), 2880, 2880,
                                          base + (8 << 20), base + (9 << 20), None)
    assert code == fp4.Status.ERR_SHAPE
    assert "static area" in fp4.last_error()
    assert lib.fp4_mx_moe_forward_noalloc(None, None, None, 0, 4, 32, 0, None, None, None, None,
                                          2880, 2880, None, None, None) == fp4.Status.OK


def _layer(tokens, k, n, experts, topk, seed):
    rng = np.random.default_rng(seed)
    a = torch.from_numpy(inputs.bf16_normal_bits(rng, tokens * k).view(np.int16)).to("cuda:0")
    ids = np.stack([rng.permutation(experts)[:topk] for _ in range(tokens)]).astype(np.int32)
    wts = rng.random((tokens, topk)).astype(np.float32)
    w1 = inputs.mx_random(experts * 2 * n, k, seed + 1, e_lo=119, e_hi=125)
    w2 = inputs.mx_random(experts * k, n, seed + 2, e_lo=119, e_hi=125)
    dev = lambda x: torch.from_numpy(x).to("cuda:0")
    return (a.view(torch.bfloat16).reshape(tokens, k), dev(ids), dev(wts),
            dev(w1.packed.reshape(experts, 2 * n, k // 2)), dev(w1.scales.reshape(experts, 2 * n, k // 32)),
            dev(w2.packed.reshape(experts, k, n // 2)), dev(w2.scales.reshape(experts, k, n // 32)))


@pytest.mark.gpu
def test_noalloc_equals_workspace_forward_and_allocates_nothing():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    big = _layer(200, 256, 192, 6, 2, seed=3)
    small = _layer(17, 128, 64, 3, 3, seed=5)
    for args in (big, small, big):  # the area is reused across sizes
        ref, st0 = fp4.fp4_mx_moe_forward(*args)
        got, st1 = fp4.fp4_mx_moe_forward_noalloc(*args)
        torch.cuda.synchronize()
        assert int(st0.item()) == 0 and int(st1.item()) == 0
        assert torch.equal(ref.view(torch.int16), got.view(torch.int16))
    out = torch.empty_like(big[0])
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    # one call of exactly the measured form first: whatever loads on first use
    # (the scratch module, the binding's own state) is in place before the reading
    fp4.fp4_mx_moe_forward_noalloc(*big, out=out, status=status)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        fp4.fp4_mx_moe_forward_noalloc(*big, out=out, status=status)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert int(status.item()) == 0


@pytest.mark.gpu
def test_noalloc_layer_filling_the_area():
    """8,736 tokens, top-2 of 2 experts, 2880 x 2880: the scratch ends 3,072 bytes
    before the end of the static area, so its last bytes are written and read."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tokens, k, n, experts, topk = 8736, 2880, 2880, 2, 2
    need = fp4.fp4_mx_moe_workspace_bytes(tokens, topk, experts, n, k)
    cap = fp4.fp4_mx_moe_static_scratch_bytes()
    assert 0 <= cap - need <= 4096, (need, cap)
    args = _layer(tokens, k, n, experts, topk, seed=11)
    for _ in range(2):
        ref, st0 = fp4.fp4_mx_moe_forward(*args)
        got, st1 = fp4.fp4_mx_moe_forward_noalloc(*args)
        torch.cuda.synchronize()
        assert int(st0.item()) == 0 and int(st1.item()) == 0
        assert torch.equal(ref.view(torch.int16), got.view(torch.int16))


@pytest.mark.gpu
def test_noalloc_oversized_layer_launches_nothing():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tokens, k, n, experts, topk = 8192, 2880, 2880, 2, 4
    a = torch.zeros(tokens, k, dtype=torch.bfloat16, device="cuda:0")
    ids = torch.zeros(tokens, topk, dtype=torch.int32, device="cuda:0")
    wts = torch.zeros(tokens, topk, dtype=torch.float32, device="cuda:0")
    w1p = torch.zeros(experts, 2 * n, k // 2, dtype=torch.uint8, device="cuda:0")
    w1s = torch.zeros(experts, 2 * n, k // 32, dtype=torch.uint8, device="cuda:0")
    w2p = torch.zeros(experts, k, n // 2, dtype=torch.uint8, device="cuda:0")
    w2s = torch.zeros(experts, k, n // 32, dtype=torch.uint8, device="cuda:0")
    out = torch.full((tokens, k), 7.0, dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(fp4.Fp4Error):
        fp4.fp4_mx_moe_forward_noalloc(a, ids, wts, w1p, w1s, w2p, w2s, out=out)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
