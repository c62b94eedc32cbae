"""GPU parity of the grouped MoE GEMM and the MoE layer on seeded random shapes.

Each case draws the expert count, the rows per expert (ragged, some empty), n and
k (multiples of 32) from a fixed seed, so that over the cases every configuration
of the tensor-core GEMM is hit: capacities up to 64 (decode-time: four MMA issuers,
K slices of 128), up to 128 (two weight tiles, K slices of 128) and above (256-token
slabs with their extension), with k ending on full, half-empty and quarter-empty
K slices. The oracle is exact; the bound is the fp32-accumulation / bf16-rounding
bound of tests/test_gpu_tcgen05_gemm.py.
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


def _bound(exact, absdot, k):
    return 2.0 ** -8 * np.abs(exact) + (1 + 2.0 ** -8) * k * 2.0 ** -23 * absdot


def _shape(rng, cap):
    experts = int(rng.integers(1, 7))
    rows = [int(r) for r in rng.integers(0, cap + 1, size=experts)]
    rows[int(rng.integers(0, experts))] = cap  # one expert at the capacity
    n = 32 * int(rng.integers(1, 13))
    k = 32 * int(rng.integers(1, 33))
    return rows, n, k


@pytest.mark.parametrize("case", range(18))
def test_random_gemm_shapes(oracle_impl, case):
    rng = np.random.default_rng(1000 + case)
    cap = [5, 16, 31, 32, 33, 48, 64, 65, 100, 128, 129, 200, 256, 257, 300, 330, 511, 580][case]
    rows, n, k = _shape(rng, cap)
    experts = len(rows)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    total = int(offsets[-1])
    a_bits = inputs.bf16_normal_bits(rng, max(total, 1) * k)[: total * k].reshape(total, k)
    w = inputs.mx_random(experts * n, k, 2000 + case, e_lo=118, e_hi=132, zero_fraction=True)
    packed, scales = w.packed.reshape(experts, n, k // 2), w.scales.reshape(experts, n, k // 32)
    out, status = fp4.fp4_mx_moe_gemm(
        torch.from_numpy(a_bits.view(np.int16)).to(DEV).view(torch.bfloat16),
        torch.from_numpy(offsets).to(DEV), torch.from_numpy(packed).to(DEV),
        torch.from_numpy(scales).to(DEV), cap)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())} for rows {rows} n {n} k {k}"
    got = out.float().cpu().numpy().astype(np.float64)
    exact, absdot = oracle_impl.mx_moe_gemm(a_bits, offsets, packed, scales,
                                            threads=oracle_impl.max_threads())
    bad = np.abs(got - exact) > _bound(exact, absdot, k)
    assert not bad.any(), (f"rows {rows} n {n} k {k}: {int(bad.sum())} of {bad.size} outside the "
                           f"bound, first {tuple(np.argwhere(bad)[0])}")


@pytest.mark.parametrize("case", range(8))
def test_random_layers(oracle_impl, case):
    """Random MoE layers (tokens, top-k, experts, n, k) checked as in
    tests/test_gpu_moe_forward.py, with the default capacity (= tokens)."""
    from test_gpu_moe_forward import check, make_layer
    rng = np.random.default_rng(3000 + case)
    tokens = [3, 20, 47, 64, 90, 128, 150, 260][case]
    experts = int(rng.integers(2, 9))
    topk = int(rng.integers(1, min(experts, 4) + 1))
    n = 32 * int(rng.integers(1, 8))
    k = 32 * int(rng.integers(1, 12))
    check(oracle_impl, make_layer(tokens, k, n, experts, topk, seed=4000 + case))
