"""CPU oracle for the FP4 (E2M1) block-scaled decode path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package. The GPU library never calls it and shares
no code with it: the arithmetic lives in ``fp4_oracle.c`` (plain C, one element
at a time, fp32 where the pages fix fp32), and this module only compiles that
file with gcc and marshals numpy arrays through ctypes.

Functions and the passages they follow (web pages cited by title and section):

* ``mx_unpack`` / ``mx_unpack_old_sequence`` / ``mx_unpack_at`` -- MXFP4 unpack,
  "vllm-project/vllm pull 51583" (prhub digest), "Motivation" and
  "Implementation breakdown" items 1-2: E2M1 code -> bf16 bits, E8M0 scale as a
  wrapping int16 add of (E-127)<<7, zero codes forced to +0.0 lane by lane.
* ``mx_unpack_pages`` -- batched (paged) MXFP4 dequant of a KV cache: the unpack
  of the pool pages a page table names ("sgl-project/sglang pull 34222", "Risks"
  item 3: the KV path's E8M0 power-of-two scales).
* ``mx_quantize`` -- the step before the unpack (bf16 -> E2M1 codes + E8M0 per
  32), named but not printed by the same page; written from the OCP MX v1.0
  conversion (shared exponent floor(log2 amax) - 2, nearest-even rounding onto
  the E2M1 grid, saturation at 6).
* ``e4m3_to_f32``, ``f32_to_bf16_rne``, ``e2m1_bf16_bits`` -- the element
  conversions those steps use (OCP FP8 E4M3 definition; IEEE round to nearest
  even into bf16; the E2M1 codebook).
* ``mx_moe_gemm`` -- the grouped MoE GEMM the unpack feeds ("vllm-project/vllm
  pull 51583", the unpack_B loop of the CPU MoE GEMM): per expert, activations
  times the unpacked weights transposed, exact in float64 (numpy matmul as the
  step), with the sum of |a||w| that bounds fp32 accumulation error.
* ``mx_moe_forward`` -- the MoE layer around that GEMM (same page: the CPU test of
  ops.fused_experts_cpu with MXFP4 experts): gate/up GEMM, silu(gate) * up, down
  GEMM, top-k weighted sum, exact in float64 with its intermediates.
* ``nv_dequant`` -- the same NVFP4 element rule over every row of a table (the
  dense dequant a tied lm_head needs; same page, "Comments" and "Risks").
* ``nv_embedding_gather`` / ``nv_embedding_gather_at`` -- NVFP4 gather-dequant,
  "sgl-project/sglang pull 34222" (prhub digest), "Implementation breakdown"
  item 2 and the ``reference_dequant`` test oracle: value * (e4m3 block scale *
  fp32 global scale) in fp32, rounded to bf16.

Every function is pinned by ``tests/test_oracle_pins.py`` to values the pages
print, closed forms and library routines; ``tests/test_oracle_mutants.py`` checks
that plausible mistakes planted in a copy of the C source fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fp4_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libfp4oracle.so")

_BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
_lock = threading.Lock()
_lib = None


def compile_source(source: str, output: str, openmp: bool = True) -> str:
    """Compile an oracle C source into a shared library with gcc.

    Tries OpenMP first (for the timed multi-core baseline) and falls back to a
    single-threaded build when the compiler or runtime lacks it.
    """
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = f"{output}.{os.getpid()}.tmp"
    attempts = ([["-fopenmp"]] if openmp else []) + [[]]
    last = None
    for extra in attempts:
        cmd = ["gcc", *_BASE_FLAGS, *extra, source, "-o", tmp, "-lm"]
        proc = subprocess.run(cmd, capture_output=True, text=True)
        if proc.returncode == 0:
            os.replace(tmp, output)
            return output
        last = proc
    raise RuntimeError(f"oracle build failed:\n{last.stderr if last else ''}")


def build(force: bool = False) -> str:
    """Build ``_build/libfp4oracle.so`` if missing or older than its source."""
    with _lock:
        stale = (not os.path.exists(LIBRARY)
                 or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))
        if force or stale:
            compile_source(SOURCE, LIBRARY)
    return LIBRARY


_P8 = ctypes.POINTER(ctypes.c_uint8)
_P16 = ctypes.POINTER(ctypes.c_uint16)
_P64 = ctypes.POINTER(ctypes.c_int64)


def bind(path: str):
    """Load an oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    lib.oracle_e2m1_bf16_bits.argtypes = [ctypes.c_uint]
    lib.oracle_e2m1_bf16_bits.restype = ctypes.c_uint16
    lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
    for name in ("oracle_mx_unpack", "oracle_mx_unpack_old_sequence"):
        fn = getattr(lib, name)
        fn.argtypes = [_P8, _P8, ctypes.c_int64, _P16, ctypes.c_int]
        fn.restype = None
    lib.oracle_mx_unpack_at.argtypes = [_P8, _P8, _P64, ctypes.c_int64, _P16]
    lib.oracle_mx_unpack_at.restype = None
    lib.oracle_nv_embedding_gather.argtypes = [
        _P64, ctypes.c_int64, _P8, _P8, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, _P16, ctypes.c_int]
    lib.oracle_nv_embedding_gather.restype = ctypes.c_int64
    lib.oracle_nv_embedding_gather_at.argtypes = [
        _P64, _P8, _P8, ctypes.c_float, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        _P64, _P64, ctypes.c_int64, _P16]
    lib.oracle_nv_embedding_gather_at.restype = None
    lib.oracle_nv_dequant.argtypes = [_P8, _P8, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int64, _P16, ctypes.c_int]
    lib.oracle_nv_dequant.restype = None
    lib.oracle_mx_quantize.argtypes = [_P16, ctypes.c_int64, _P8, _P8, ctypes.c_int]
    lib.oracle_mx_quantize.restype = None
    lib.oracle_mx_unpack_pages.argtypes = [_P64, ctypes.c_int64, _P8, _P8, ctypes.c_int64,
                                           ctypes.c_int64, _P16, ctypes.c_int]
    lib.oracle_mx_unpack_pages.restype = ctypes.c_int64
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def lib():
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"expected uint8, got {a.dtype}")
    return a


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """numpy-facing wrapper over one loaded oracle library (the real one, or a
    test-built variant)."""

    def __init__(self, library):
        self.lib = library

    # -- element conversions ------------------------------------------------
    def e2m1_bf16_bits(self, code: int) -> int:
        return int(self.lib.oracle_e2m1_bf16_bits(code))

    def e4m3_to_f32(self, byte: int) -> float:
        return float(self.lib.oracle_e4m3_to_f32(byte))

    def f32_to_bf16_rne(self, value) -> int:
        return int(self.lib.oracle_f32_to_bf16_rne(float(np.float32(value))))

    # -- MXFP4 ----------------------------------------------------------------
    def _mx(self, fn, packed, scales, threads):
        packed, scales = _u8(packed).reshape(-1), _u8(scales).reshape(-1)
        n = packed.size * 2
        if n % 32 or scales.size != n // 32:
            raise ValueError("need packed[n/2] and scales[n/32] with n % 32 == 0")
        out = np.empty(n, dtype=np.uint16)
        fn(_ptr(packed, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8), n,
           _ptr(out, ctypes.c_uint16), int(threads))
        return out

    def mx_unpack(self, packed, scales, threads: int = 1) -> np.ndarray:
        """Flat bf16 bits (uint16[n]) of a packed stream."""
        return self._mx(self.lib.oracle_mx_unpack, packed, scales, threads)

    def mx_unpack_old_sequence(self, packed, scales, threads: int = 1) -> np.ndarray:
        return self._mx(self.lib.oracle_mx_unpack_old_sequence, packed, scales, threads)

    def mx_unpack_at(self, packed, scales, idx) -> np.ndarray:
        packed, scales, idx = _u8(packed).reshape(-1), _u8(scales).reshape(-1), _i64(idx)
        n = packed.size * 2
        if idx.size and (idx.min() < 0 or idx.max() >= n):
            raise IndexError("element index out of range")
        out = np.empty(idx.size, dtype=np.uint16)
        self.lib.oracle_mx_unpack_at(_ptr(packed, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                     _ptr(idx, ctypes.c_int64), idx.size,
                                     _ptr(out, ctypes.c_uint16))
        return out

    def mx_unpack_pages(self, page_ids, packed_pool, scales_pool, threads: int = 1):
        """Paged MXFP4 dequant: uint16[*page_ids.shape, page_elems] and the number of
        page ids outside the pool (their rows are +0.0)."""
        shape = np.shape(page_ids)
        ids = _i64(page_ids).reshape(-1)
        packed_pool, scales_pool = _u8(packed_pool), _u8(scales_pool)
        pool_pages, half = packed_pool.shape
        page_elems = 2 * half
        if page_elems % 32 or scales_pool.shape != (pool_pages, page_elems // 32):
            raise ValueError("pool must be [pages, page_elems/2] codes and [pages, page_elems/32] scales")
        out = np.empty((ids.size, page_elems), dtype=np.uint16)
        bad = self.lib.oracle_mx_unpack_pages(
            _ptr(ids, ctypes.c_int64), ids.size, _ptr(packed_pool, ctypes.c_uint8),
            _ptr(scales_pool, ctypes.c_uint8), pool_pages, page_elems,
            _ptr(out, ctypes.c_uint16), int(threads))
        return out.reshape(*shape, page_elems), int(bad)

    def mx_quantize(self, x_bf16_bits, threads: int = 1):
        """bf16 bit patterns (uint16[..., k], k % 32 == 0) -> (packed uint8[..., k/2],
        E8M0 scales uint8[..., k/32])."""
        x = np.ascontiguousarray(x_bf16_bits)
        if x.dtype != np.uint16:
            raise TypeError("expected uint16 bf16 bit patterns")
        shape = x.shape
        if shape[-1] % 32:
            raise ValueError("last dimension must be a multiple of 32")
        flat = x.reshape(-1)
        packed = np.empty(flat.size // 2, dtype=np.uint8)
        scales = np.empty(flat.size // 32, dtype=np.uint8)
        self.lib.oracle_mx_quantize(_ptr(flat, ctypes.c_uint16), flat.size,
                                    _ptr(packed, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                    int(threads))
        return (packed.reshape(*shape[:-1], shape[-1] // 2),
                scales.reshape(*shape[:-1], shape[-1] // 32))

    def bf16_to_f64(self, bits) -> np.ndarray:
        """Exact float64 values of bf16 bit patterns (bf16 is the top half of fp32)."""
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def mx_moe_gemm(self, a_bits, offsets, w_packed, w_scales, threads: int = 1):
        """Grouped MoE GEMM, exact in float64: for expert e and its rows
        [offsets[e], offsets[e+1]) of ``a`` (bf16 bits [T, k]),
        out = a_rows @ W_e^T with W_e the MXFP4 unpack of expert e's weights
        ([n, k/2] codes, [n, k/32] E8M0). The products of two bf16 values are exact in
        float64 and the float64 sums are far more precise than the fp32 accumulation
        they are compared with. Returns (out, sum of |a||w| per output element)."""
        a = self.bf16_to_f64(a_bits)
        offsets = np.asarray(offsets, dtype=np.int64)
        experts, n, half = w_packed.shape
        out = np.zeros((a.shape[0], n))
        absdot = np.zeros((a.shape[0], n))
        for e in range(experts):
            r0, r1 = int(offsets[e]), int(offsets[e + 1])
            if r1 <= r0:
                continue
            w = self.bf16_to_f64(self.mx_unpack(w_packed[e], w_scales[e], threads)).reshape(n, 2 * half)
            out[r0:r1] = a[r0:r1] @ w.T
            absdot[r0:r1] = np.abs(a[r0:r1]) @ np.abs(w).T
        return out, absdot

    @staticmethod
    def bf16_round(x) -> np.ndarray:
        """Round float64 values to the nearest bf16 value (ties to even), as float64:
        8 significant bits, spacing 2^-133 below the smallest normal 2^-126."""
        x = np.asarray(x, dtype=np.float64)
        out = x.copy()
        nz = (x != 0) & np.isfinite(x)
        _, e = np.frexp(x[nz])  # x = f * 2^e, 0.5 <= |f| < 1
        ulp = np.ldexp(1.0, np.maximum(e, -125) - 8)
        out[nz] = np.rint(x[nz] / ulp) * ulp
        return out

    def mx_moe_forward(self, a_bits, topk_ids, topk_weights, w1_packed, w1_scales, w2_packed,
                       w2_scales, threads: int = 1) -> dict:
        """The MoE layer the unpack feeds ("vllm-project/vllm pull 51583": the test that
        runs ops.fused_experts_cpu with MXFP4 experts, and the zero-code test whose
        comment says silu(0) * 0 = 0 collapses the whole layer). For token m and each
        of its top-k slots j, with expert e = topk_ids[m, j] and weight w =
        topk_weights[m, j]:
            h   = a[m] @ W1_e^T                  W1_e [2N, K] unpacked (gate rows, then up)
            act = bf16(silu(h[:N]) * h[N:])      silu(x) = x / (1 + exp(-x))
            y   = bf16(act @ W2_e^T)             W2_e [K, N] unpacked
            out[m] = bf16(sum_j w * y)
        where each bf16() rounds the exact value (nearest, ties to even) -- the places
        the layer stores bf16 -- and everything else is float64 (bf16 x bf16 products
        are exact, the sums far more precise than the fp32 work they are compared
        with). A slot whose expert id is outside [0, E) contributes nothing and is
        counted.

        Returns a dict: out [M, K] (rounded) and out_exact (before its rounding); per
        slot g, u, act_exact, act [M, topk, N] and y_exact, y [M, topk, K]; sg, su
        [M, topk, N] = sums of |a||w1| behind g and u; the unpacked weights w1 [E, 2N,
        K], w2 [E, K, N] (float64); bad (count)."""
        a = self.bf16_to_f64(a_bits)
        ids = np.asarray(topk_ids, dtype=np.int64)
        wts = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
        m_tok, k = a.shape
        topk = ids.shape[1]
        experts, two_n, half_k = w1_packed.shape
        n = two_n // 2
        if 2 * half_k != k or w2_packed.shape != (experts, k, n // 2):
            raise ValueError("inconsistent MoE shapes")
        w1 = np.stack([self.bf16_to_f64(self.mx_unpack(w1_packed[e], w1_scales[e], threads))
                       .reshape(two_n, k) for e in range(experts)]) if experts else np.zeros((0, two_n, k))
        w2 = np.stack([self.bf16_to_f64(self.mx_unpack(w2_packed[e], w2_scales[e], threads))
                       .reshape(k, n) for e in range(experts)]) if experts else np.zeros((0, k, n))
        g = np.zeros((m_tok, topk, n))
        u = np.zeros((m_tok, topk, n))
        sg = np.zeros((m_tok, topk, n))
        su = np.zeros((m_tok, topk, n))
        act_exact = np.zeros((m_tok, topk, n))
        act = np.zeros((m_tok, topk, n))
        y_exact = np.zeros((m_tok, topk, k))
        y = np.zeros((m_tok, topk, k))
        out_exact = np.zeros((m_tok, k))
        bad = int(np.count_nonzero((ids < 0) | (ids >= experts)))
        for e in range(experts):
            ms, js = np.nonzero(ids == e)
            if ms.size == 0:
                continue
            rows = a[ms]
            h = rows @ w1[e].T
            habs = np.abs(rows) @ np.abs(w1[e]).T
            g[ms, js], u[ms, js] = h[:, :n], h[:, n:]
            sg[ms, js], su[ms, js] = habs[:, :n], habs[:, n:]
            with np.errstate(over="ignore"):
                act_e = h[:, :n] / (1.0 + np.exp(-h[:, :n])) * h[:, n:]
            act_exact[ms, js] = act_e
            act_r = self.bf16_round(act_e)
            act[ms, js] = act_r
            y_e = act_r @ w2[e].T
            y_exact[ms, js] = y_e
            y_r = self.bf16_round(y_e)
            y[ms, js] = y_r
            np.add.at(out_exact, ms, wts[ms, js][:, None] * y_r)
        return {"out": self.bf16_round(out_exact), "out_exact": out_exact, "g": g, "u": u,
                "sg": sg, "su": su, "act_exact": act_exact, "act": act, "y_exact": y_exact,
                "y": y, "w1": w1, "w2": w2, "bad": bad}

    # -- NVFP4 ----------------------------------------------------------------
    def nv_embedding_gather(self, ids, weight, scales, global_scale, group_size: int = 16,
                            threads: int = 1):
        """Returns (uint16[*ids.shape, hidden], number of out-of-range ids)."""
        ids_shape = np.shape(ids)
        ids = _i64(ids).reshape(-1)
        weight, scales = _u8(weight), _u8(scales)
        vocab, half = weight.shape
        hidden = 2 * half
        if scales.shape != (vocab, hidden // group_size):
            raise ValueError("scales must be [vocab, hidden / group_size]")
        out = np.empty((ids.size, hidden), dtype=np.uint16)
        bad = self.lib.oracle_nv_embedding_gather(
            _ptr(ids, ctypes.c_int64), ids.size, _ptr(weight, ctypes.c_uint8),
            _ptr(scales, ctypes.c_uint8), float(np.float32(global_scale)), vocab, hidden,
            group_size, _ptr(out, ctypes.c_uint16), int(threads))
        return out.reshape(*ids_shape, hidden), int(bad)

    def nv_embedding_gather_at(self, ids, weight, scales, global_scale, rows, cols,
                               group_size: int = 16) -> np.ndarray:
        ids = _i64(ids).reshape(-1)
        weight, scales = _u8(weight), _u8(scales)
        rows, cols = _i64(rows), _i64(cols)
        vocab, half = weight.shape
        hidden = 2 * half
        if rows.size and (rows.min() < 0 or rows.max() >= ids.size
                          or cols.min() < 0 or cols.max() >= hidden):
            raise IndexError("sample index out of range")
        out = np.empty(rows.size, dtype=np.uint16)
        self.lib.oracle_nv_embedding_gather_at(
            _ptr(ids, ctypes.c_int64), _ptr(weight, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
            float(np.float32(global_scale)), vocab, hidden, group_size,
            _ptr(rows, ctypes.c_int64), _ptr(cols, ctypes.c_int64), rows.size,
            _ptr(out, ctypes.c_uint16))
        return out

    def nv_dequant(self, weight, scales, global_scale, group_size: int = 16,
                   threads: int = 1) -> np.ndarray:
        """Whole-table dequant: uint16[vocab, hidden]."""
        weight, scales = _u8(weight), _u8(scales)
        rows, half = weight.shape
        hidden = 2 * half
        if scales.shape != (rows, hidden // group_size):
            raise ValueError("scales must be [rows, hidden / group_size]")
        out = np.empty((rows, hidden), dtype=np.uint16)
        self.lib.oracle_nv_dequant(_ptr(weight, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                   float(np.float32(global_scale)), rows, hidden, group_size,
                                   _ptr(out, ctypes.c_uint16), int(threads))
        return out

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


_default = None


def get() -> Oracle:
    """The oracle built from ``fp4_oracle.c``."""
    global _default
    if _default is None:
        _default = Oracle(lib())
    return _default
