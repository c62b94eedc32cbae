"""The oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_impl):
    pin(oracle_impl)


def test_bf16_nearest_even_definition():
    """The value-set rounding used by the exact-product pin rounds ties to even."""
    # 1 + 2^-8 lies halfway between 1.0 (0x3F80, even) and 1 + 2^-7 (0x3F81, odd)
    assert oracle_pins.bf16_nearest_even(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle_pins.bf16_nearest_even(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle_pins.bf16_nearest_even(-(1.0 + 2.0 ** -9)) == 0xBF80
    assert oracle_pins.bf16_nearest_even(2.0 ** -133) == 0x0001  # bf16 subnormal


def test_workload_exhaustive_covers_every_pair():
    import numpy as np
    from block_scaled_fp4_mx_gb300 import inputs
    x = inputs.mx_exhaustive()
    blocks = x.packed.reshape(-1, 16)
    e = x.scales.reshape(-1)
    pairs = set()
    for b in range(blocks.shape[0]):
        for byte in blocks[b]:
            pairs.add((int(byte), int(e[b])))
    assert len(pairs) == 65536 and x.n_elems == 131072
