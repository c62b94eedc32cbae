"""Plant plausible mistakes in a copy of the oracle's MoE-layer and grouped-GEMM
functions (their Python source, rewritten and re-executed; the real oracle is
untouched) and check that the matching pins catch each one (CPU only)."""
import inspect
import textwrap
import warnings

import numpy as np
import pytest

import oracle
import oracle_pins

MUTATIONS = [
    ("act_e = h[:, :n] / (1.0 + np.exp(-h[:, :n])) * h[:, n:]",
     "act_e = h[:, n:] / (1.0 + np.exp(-h[:, n:])) * h[:, :n]", "gate and up rows swapped"),
    ("act_e = h[:, :n] / (1.0 + np.exp(-h[:, :n])) * h[:, n:]",
     "act_e = 1.0 / (1.0 + np.exp(-h[:, :n])) * h[:, n:]", "sigmoid instead of silu"),
    ("act_e = h[:, :n] / (1.0 + np.exp(-h[:, :n])) * h[:, n:]",
     "act_e = h[:, :n] / (1.0 + np.exp(h[:, :n])) * h[:, n:]", "silu with the wrong sign"),
    ("act_e = h[:, :n] / (1.0 + np.exp(-h[:, :n])) * h[:, n:]",
     "act_e = np.maximum(h[:, :n], 0.0) * h[:, n:]", "relu instead of silu"),
    ("np.add.at(out_exact, ms, wts[ms, js][:, None] * y_r)", "np.add.at(out_exact, ms, y_r)",
     "top-k weights dropped"),
    ("np.add.at(out_exact, ms, wts[ms, js][:, None] * y_r)",
     "out_exact[ms] = wts[ms, js][:, None] * y_r", "slots of one token overwrite instead of add"),
    ("act_r = self.bf16_round(act_e)", "act_r = act_e", "activation not rounded to bf16"),
    ("y_r = self.bf16_round(y_e)", "y_r = y_e", "down GEMM output not rounded to bf16"),
    ("h = rows @ w1[e].T", "h = rows @ w1[(e + 1) % experts].T", "another expert's gate/up weights"),
    ("y_e = act_r @ w2[e].T", "y_e = act_r @ w2[(e + 1) % experts].T", "another expert's down weights"),
    (".reshape(k, n) for e in range(experts)]", ".reshape(n, k).T for e in range(experts)]",
     "down weights read transposed"),
    ("bad = int(np.count_nonzero((ids < 0) | (ids >= experts)))",
     "bad = int(np.count_nonzero((ids < 0) | (ids > experts)))", "last valid id off by one"),
]

FORWARD_PINS = [p for p in oracle_pins.ALL_PINS if p.__name__.startswith("pin_moe_forward")]


def _source():
    return textwrap.dedent(inspect.getsource(oracle.Oracle.mx_moe_forward))


def test_mutations_apply():
    src = _source()
    for before, _, what in MUTATIONS:
        assert src.count(before) >= 1, what


@pytest.mark.parametrize("before,after,what", MUTATIONS, ids=[m[2] for m in MUTATIONS])
def test_forward_pins_catch_mutant(before, after, what):
    namespace = dict(vars(oracle))
    exec(compile(_source().replace(before, after, 1), "<mutant>", "exec"), namespace)
    mutant_cls = type("MutantOracle", (oracle.Oracle,), {"mx_moe_forward": namespace["mx_moe_forward"]})
    mutant = mutant_cls(oracle.lib())
    failed = []
    with warnings.catch_warnings():
        warnings.simplefilter("ignore", RuntimeWarning)
        for pin in FORWARD_PINS:
            try:
                pin(mutant)
            except (AssertionError, ValueError, IndexError):
                failed.append(pin.__name__)
    assert failed, f"no pin caught the mutant: {what}"


# The grouped GEMM oracle the MoE GEMM tests compare with: the same check against
# its own two pins (rows routed to their expert; a brute-force triple loop).
GEMM_MUTATIONS = [
    ("out[r0:r1] = a[r0:r1] @ w.T", "out[r0:r1] = a[r0:r1] @ w[::-1].T", "weight rows reversed"),
    (".reshape(n, 2 * half)", ".reshape(2 * half, n).T", "codes read column-major"),
    ("self.mx_unpack(w_packed[e], w_scales[e], threads)",
     "self.mx_unpack(w_packed[e], w_scales[(e + 1) % experts], threads)", "another expert's scales"),
    ("r0, r1 = int(offsets[e]), int(offsets[e + 1])",
     "r0, r1 = int(offsets[e]) + 1, int(offsets[e + 1])", "an expert's first row skipped"),
    ("if r1 <= r0:", "if r1 <= r0 + 1:", "single-row experts skipped"),
    ("absdot[r0:r1] = np.abs(a[r0:r1]) @ np.abs(w).T", "absdot[r0:r1] = np.abs(a[r0:r1] @ w.T)",
     "|sum| instead of the sum of |products|"),
]

GEMM_PINS = [p for p in oracle_pins.ALL_PINS if p.__name__.startswith("pin_moe_gemm")]


def _gemm_source():
    return textwrap.dedent(inspect.getsource(oracle.Oracle.mx_moe_gemm))


def test_gemm_mutations_apply():
    src = _gemm_source()
    assert len(GEMM_PINS) >= 2
    for before, _, what in GEMM_MUTATIONS:
        assert src.count(before) >= 1, what


@pytest.mark.parametrize("before,after,what", GEMM_MUTATIONS, ids=[m[2] for m in GEMM_MUTATIONS])
def test_gemm_pins_catch_mutant(before, after, what):
    namespace = dict(vars(oracle))
    exec(compile(_gemm_source().replace(before, after, 1), "<mutant>", "exec"), namespace)
    mutant_cls = type("MutantOracle", (oracle.Oracle,), {"mx_moe_gemm": namespace["mx_moe_gemm"]})
    mutant = mutant_cls(oracle.lib())
    failed = []
    with warnings.catch_warnings():
        warnings.simplefilter("ignore", RuntimeWarning)
        for pin in GEMM_PINS:
            try:
                pin(mutant)
            except (AssertionError, ValueError, IndexError):
                failed.append(pin.__name__)
    assert failed, f"no pin caught the mutant: {what}"
