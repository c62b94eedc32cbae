"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random bytes, ids and scales. It holds none of the decode
arithmetic, imports neither the GPU library nor the oracle, and is the one piece
that both sides of a parity check share. Every generator is deterministic in its
seed (numpy PCG64) and returns host arrays:

* MXFP4 inputs: ``packed`` uint8 ``[rows, k/2]`` (two E2M1 codes a byte, even
  element in the low nibble) and ``scales`` uint8 ``[rows, k/32]`` (E8M0 bytes).
* NVFP4 inputs: ``ids`` int64 of any shape, ``weight`` uint8 ``[vocab, hidden/2]``,
  ``scales`` uint8 ``[vocab, hidden/16]`` (float8 e4m3fn bit patterns) and an
  fp32 ``global_scale``.

The five named workloads follow the shapes and value distributions of the
decode workloads the pages describe (an MoE expert stack with hidden 2880, and a
200k-vocabulary token embedding), written out as:

==================  ==========================================================
mx_exhaustive       65,536 packed bytes, byte j = j mod 256, block b has E = b // 16:
                    every (byte, E8M0) pair once -> 131,072 outputs
nv_embedding_32k    vocab 32,000 x hidden 4,096; scales U[2^-6, 448] -> e4m3 (RNE);
                    global 1/448; 2,048 ids uniform in [0, vocab)
mx_moe              gate+up [32, 5760, 2880] and down [32, 2880, 2880] codes;
                    bytes uniform; E uniform in [118, 132]
nv_embedding_200k   vocab 200,000 x hidden 8,192; scales as above; 16,384 ids
                    from a Zipf(s=1.1) law truncated to the vocabulary, [64, 256]
mx_stress           2^30 packed bytes; each nibble a zero code with p = 0.3
                    (0x0 or 0x8, half each), else uniform over the 14 nonzero
                    codes; E per block uniform over {0, 107, 127, 137, 255}
bf16_moe            (input of the quantiser) gate+up and down MoE weights as bf16,
                    standard normal / 10 as the pages' MoE test draws them
kv_pages            (paged dequant) an MXFP4 KV pool of 32,768 pages of 16 tokens x
                    8 heads x 128 dims (16,384 codes each), bytes uniform, E uniform
                    in [118, 132]; a page table of 64 sequences x 128 pages drawn
                    without replacement
==================  ==========================================================
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GROUP_SIZE = 16
MX_BLOCK = 32
# fp32 nearest to 1/448: the global scale that maps the largest e4m3 value to 1.
GLOBAL_SCALE_1_OVER_448 = np.float32(1.0 / 448.0)


@dataclass
class MxInput:
    packed: np.ndarray  # uint8 [rows, k/2]
    scales: np.ndarray  # uint8 [rows, k/32]
    name: str = ""

    @property
    def rows(self) -> int:
        return self.packed.shape[0]

    @property
    def k(self) -> int:
        return self.packed.shape[1] * 2

    @property
    def n_elems(self) -> int:
        return self.packed.size * 2

    def algorithmic_bytes(self) -> int:
        """Bytes a decode must move at least: read packed + scales, write bf16."""
        return self.packed.size + self.scales.size + 2 * self.n_elems


@dataclass
class NvInput:
    ids: np.ndarray  # int64, any shape
    weight: np.ndarray  # uint8 [vocab, hidden/2]
    scales: np.ndarray  # uint8 [vocab, hidden/group] e4m3fn bits
    global_scale: np.float32
    group_size: int = GROUP_SIZE
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def vocab(self) -> int:
        return self.weight.shape[0]

    @property
    def hidden(self) -> int:
        return self.weight.shape[1] * 2

    @property
    def n_elems(self) -> int:
        return self.ids.size * self.hidden

    def algorithmic_bytes(self) -> int:
        """Logical bytes: ids, the gathered packed rows and scale rows, bf16 out."""
        row_in = self.hidden // 2 + self.hidden // self.group_size
        return self.ids.size * (8 + row_in + 2 * self.hidden)

    def distinct_row_bytes(self) -> int:
        """Minimum bytes when every distinct row is read once."""
        distinct = np.unique(self.ids[(self.ids >= 0) & (self.ids < self.vocab)]).size
        row_in = self.hidden // 2 + self.hidden // self.group_size
        return self.ids.size * (8 + 2 * self.hidden) + distinct * row_in


# ---------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------

_CHUNK = 1 << 26


def uniform_bytes(rng: np.random.Generator, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = rng.integers(0, 256, size=e - s, dtype=np.uint8)
    return out


def e8m0_uniform(rng: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    """E8M0 bytes uniform over the integers lo..hi (inclusive)."""
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.uint8)


def e8m0_choice(rng: np.random.Generator, n: int, values) -> np.ndarray:
    table = np.asarray(values, dtype=np.uint8)
    return table[rng.integers(0, table.size, size=n, dtype=np.int64)]


# Nibble draw for the stress stream: 200 equally likely outcomes, 30 -> code 0x0,
# 30 -> code 0x8, and 10 for each of the 14 nonzero codes (1..7, 9..15). A byte
# is one uniform draw over 200 x 200 outcomes (low nibble = draw % 200, high
# nibble = draw // 200), i.e. two independent nibble draws, looked up in a table.
_NONZERO_CODES = np.array([1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15], dtype=np.uint8)
_STRESS_NIBBLE = np.concatenate([
    np.zeros(30, dtype=np.uint8),
    np.full(30, 8, dtype=np.uint8),
    np.tile(_NONZERO_CODES, 10),
])
_STRESS_BYTE = (_STRESS_NIBBLE[np.arange(40000) % 200]
                | (_STRESS_NIBBLE[np.arange(40000) // 200] << 4)).astype(np.uint8)


def packed_with_zero_fraction(rng: np.random.Generator, n_bytes: int) -> np.ndarray:
    """Bytes whose nibbles are zero codes with p = 0.3 (0x0 / 0x8 half each), else
    uniform over the 14 nonzero codes; drawn independently per nibble."""
    out = np.empty(n_bytes, dtype=np.uint8)
    for s in range(0, n_bytes, _CHUNK):
        e = min(n_bytes, s + _CHUNK)
        draw = rng.integers(0, _STRESS_BYTE.size, size=e - s, dtype=np.uint16)
        out[s:e] = _STRESS_BYTE[draw]
    return out


def e4m3_scales_uniform(rng: np.random.Generator, n: int, lo: float = 2.0 ** -6,
                        hi: float = 448.0) -> np.ndarray:
    """Positive finite e4m3fn bytes: fp32 uniform in [lo, hi], cast with torch's
    round-to-nearest-even float8_e4m3fn conversion (both ends are representable)."""
    import torch

    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        u = rng.random(e - s, dtype=np.float32)
        vals = np.minimum(np.float32(lo) + u * np.float32(hi - lo), np.float32(hi))
        out[s:e] = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return out


def zipf_ids(rng: np.random.Generator, n: int, vocab: int, s: float) -> np.ndarray:
    """Ids by inverse CDF of a Zipf law truncated to the vocabulary:
    P(rank k) proportional to k^-s for k = 1..vocab, id = k - 1."""
    weights = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(weights)
    cdf /= cdf[-1]
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1).astype(np.int64)


def bf16_normal_bits(rng: np.random.Generator, n: int, scale: float = 0.1) -> np.ndarray:
    """bf16 bit patterns of standard-normal draws times ``scale`` (torch's
    round-to-nearest-even float32 -> bfloat16 cast)."""
    import torch

    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        v = rng.standard_normal(e - s, dtype=np.float32) * np.float32(scale)
        out[s:e] = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out


@dataclass
class Bf16Input:
    x: np.ndarray  # uint16 bf16 bit patterns [rows, k]
    name: str = ""

    @property
    def rows(self) -> int:
        return self.x.shape[0]

    @property
    def k(self) -> int:
        return self.x.shape[1]

    @property
    def n_elems(self) -> int:
        return self.x.size

    def algorithmic_bytes(self) -> int:
        """Quantise: read bf16, write packed codes + scales."""
        return 2 * self.n_elems + self.n_elems // 2 + self.n_elems // MX_BLOCK


def bf16_moe(seed: int = 5) -> list[Bf16Input]:
    """MoE expert weights in bf16 (gate+up 32 x 5760 rows, down 32 x 2880 rows, 2880
    columns), standard normal / 10: the input the pages' MoE test quantises."""
    rng = np.random.default_rng(seed)
    return [Bf16Input(bf16_normal_bits(rng, rows * 2880).reshape(rows, 2880), name=f"bf16_moe_{nm}")
            for nm, rows in (("gate_up", 32 * 5760), ("down", 32 * 2880))]


def bf16_blocks_wide_range(n_blocks: int, seed: int) -> np.ndarray:
    """uint16 [n_blocks, 32] bf16 blocks spanning the exponent range: normal draws
    times 2^k with k per block in [-140, 120] (so zeros, subnormals and values near
    the top of the range occur), a third of the entries of every 7th block zero,
    every 11th block negated."""
    import torch

    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n_blocks, 32)) * np.exp2(rng.integers(-140, 121, (n_blocks, 1)))
    x[::7, ::3] = 0.0
    x[::11] *= -1
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# generic small generators (tests)
# ---------------------------------------------------------------------------

def mx_random(rows: int, k: int, seed: int, e_lo: int = 0, e_hi: int = 255,
              e_values=None, zero_fraction: bool = False) -> MxInput:
    if k % MX_BLOCK:
        raise ValueError("k must be a multiple of 32")
    rng = np.random.default_rng(seed)
    n_bytes = rows * k // 2
    packed = (packed_with_zero_fraction(rng, n_bytes) if zero_fraction
              else uniform_bytes(rng, n_bytes))
    n_blocks = rows * k // MX_BLOCK
    scales = (e8m0_choice(rng, n_blocks, e_values) if e_values is not None
              else e8m0_uniform(rng, n_blocks, e_lo, e_hi))
    return MxInput(packed.reshape(rows, k // 2), scales.reshape(rows, k // MX_BLOCK),
                   name=f"mx_random_{rows}x{k}_s{seed}")


def nv_random(vocab: int, hidden: int, ids_shape, seed: int, zipf_s: float | None = None,
              global_scale=GLOBAL_SCALE_1_OVER_448, group_size: int = GROUP_SIZE,
              scale_lo: float = 2.0 ** -6, scale_hi: float = 448.0) -> NvInput:
    rng = np.random.default_rng(seed)
    weight = uniform_bytes(rng, vocab * hidden // 2).reshape(vocab, hidden // 2)
    scales = e4m3_scales_uniform(rng, vocab * (hidden // group_size), scale_lo, scale_hi)
    scales = scales.reshape(vocab, hidden // group_size)
    n_ids = int(np.prod(ids_shape)) if len(tuple(ids_shape)) else 1
    if zipf_s is None:
        ids = rng.integers(0, vocab, size=n_ids, dtype=np.int64)
    else:
        ids = zipf_ids(rng, n_ids, vocab, zipf_s)
    return NvInput(ids.reshape(ids_shape), weight, scales, np.float32(global_scale),
                   group_size, name=f"nv_random_{vocab}x{hidden}_s{seed}")


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

def mx_exhaustive() -> MxInput:
    """Every (packed byte, E8M0) pair once: byte j = j mod 256 and block b (16
    packed bytes) has E = b // 16, so the 16 blocks of one exponent cover the
    bytes 0..255."""
    j = np.arange(65536, dtype=np.int64)
    packed = (j & 0xFF).astype(np.uint8)
    scales = (np.arange(4096, dtype=np.int64) >> 4).astype(np.uint8)
    return MxInput(packed.reshape(64, 1024), scales.reshape(64, 64), name="mx_exhaustive")


def nv_embedding_32k(seed: int = 1) -> NvInput:
    x = nv_random(32000, 4096, (2048,), seed)
    x.name = "nv_embedding_32000x4096_ids2048"
    return x


def mx_moe(seed: int = 2) -> list[MxInput]:
    """MoE expert weights: gate+up [32, 2*2880, 2880] and down [32, 2880, 2880]
    codes (rows = experts x output channels), E uniform in [118, 132]."""
    rng = np.random.default_rng(seed)
    out = []
    for name, rows in (("gate_up", 32 * 5760), ("down", 32 * 2880)):
        k = 2880
        packed = uniform_bytes(rng, rows * k // 2).reshape(rows, k // 2)
        scales = e8m0_uniform(rng, rows * k // MX_BLOCK, 118, 132).reshape(rows, k // MX_BLOCK)
        out.append(MxInput(packed, scales, name=f"mx_moe_{name}"))
    return out


def nv_embedding_200k(seed: int = 3) -> NvInput:
    x = nv_random(200000, 8192, (64, 256), seed, zipf_s=1.1)
    x.name = "nv_embedding_200000x8192_zipf_ids64x256"
    return x


def mx_stress(seed: int = 4) -> MxInput:
    rng = np.random.default_rng(seed)
    rows, k = 65536, 32768  # 2^30 packed bytes, 2^31 codes
    packed = packed_with_zero_fraction(rng, rows * k // 2).reshape(rows, k // 2)
    scales = e8m0_choice(rng, rows * k // MX_BLOCK, (0, 107, 127, 137, 255))
    return MxInput(packed, scales.reshape(rows, k // MX_BLOCK), name="mx_stress")


@dataclass
class KvPagesInput:
    page_ids: np.ndarray  # int64, any shape
    pool: MxInput         # packed [pool_pages, page_elems/2], scales [pool_pages, page_elems/32]
    name: str = ""

    @property
    def page_elems(self) -> int:
        return self.pool.k

    @property
    def n_elems(self) -> int:
        return self.page_ids.size * self.page_elems

    def algorithmic_bytes(self) -> int:
        """ids + the gathered pages' codes and scales + bf16 out."""
        return self.page_ids.size * (8 + self.page_elems // 2 + self.page_elems // MX_BLOCK
                                     + 2 * self.page_elems)


def kv_pages(seed: int = 8, pool_pages: int = 32768, page_elems: int = 16 * 8 * 128,
             table_shape=(64, 128)) -> KvPagesInput:
    rng = np.random.default_rng(seed)
    packed = uniform_bytes(rng, pool_pages * page_elems // 2).reshape(pool_pages, page_elems // 2)
    scales = e8m0_uniform(rng, pool_pages * page_elems // MX_BLOCK, 118, 132)
    pool = MxInput(packed, scales.reshape(pool_pages, page_elems // MX_BLOCK), name="kv_pool")
    n = int(np.prod(table_shape))
    ids = rng.permutation(pool_pages)[:n].astype(np.int64).reshape(table_shape)
    return KvPagesInput(ids, pool, name=f"kv_pages_{pool_pages}x{page_elems}_table{n}")
