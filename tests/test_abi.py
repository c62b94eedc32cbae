"""The C-ABI library without a GPU: it loads, exports every declared symbol, and
rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import block_scaled_fp4_mx_gb300 as fp4
from block_scaled_fp4_mx_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as fh:
                text = fh.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(fp4_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return fp4.load()


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("fp4_mx_unpack", "fp4_nv_embedding_gather", "fp4_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks a signature for {name}"


def test_only_api_symbols_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fp4.library_path()],
                         capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    syms = [l.split()[-1] for l in out.stdout.splitlines() if l.strip()]
    public = [s for s in syms if not s.startswith("_")]
    assert sorted(p for p in public if p.startswith("fp4_")) == declared_functions()


def test_status_strings(lib):
    assert fp4.fp4_status_string(0) == "ok"
    for code in range(1, 11):
        assert fp4.fp4_status_string(code) not in ("", "unknown status")
    assert fp4.fp4_status_string(99) == "unknown status"
    assert lib.fp4_abi_version() == 108


def test_mx_host_validation(lib):
    f = lib.fp4_mx_unpack
    assert f(None, None, None, 1, 33, None) == fp4.Status.ERR_SHAPE      # k % 32
    assert f(None, None, None, -1, 32, None) == fp4.Status.ERR_SHAPE
    assert f(None, None, None, 1, -32, None) == fp4.Status.ERR_SHAPE
    assert f(None, None, None, 0, 64, None) == fp4.Status.OK             # empty: no launch
    assert f(None, None, None, 5, 0, None) == fp4.Status.OK
    assert f(None, None, None, 2, 64, None) == fp4.Status.ERR_NULL_PTR
    assert f(None, None, None, 2 ** 62, 2 ** 10, None) == fp4.Status.ERR_SHAPE  # overflow
    # output overlapping the input is refused before any CUDA call
    buf = ctypes.create_string_buffer(4096)
    base = ctypes.addressof(buf)
    assert f(base, base + 2048, base + 16, 1, 64, None) == fp4.Status.ERR_ALIAS


def test_nv_host_validation(lib):
    f = lib.fp4_nv_embedding_gather
    args = lambda n, v, h, g: (None, n, None, None, None, v, h, g, None, None, None)
    assert f(*args(4, 10, 100, 16)) == fp4.Status.ERR_GROUP       # hidden % group_size
    assert f(*args(4, 10, 96, 32)) == fp4.Status.ERR_UNSUPPORTED  # NVFP4 groups are 16
    assert f(*args(4, 10, 0, 16)) == fp4.Status.ERR_SHAPE
    assert f(*args(-1, 10, 64, 16)) == fp4.Status.ERR_SHAPE
    assert f(*args(4, 10, 64, 0)) == fp4.Status.ERR_SHAPE
    assert f(*args(0, 10, 64, 16)) == fp4.Status.OK               # no ids: no launch
    assert f(*args(4, 0, 64, 16)) == fp4.Status.ERR_SHAPE         # ids but empty table
    assert f(*args(4, 10, 64, 16)) == fp4.Status.ERR_NULL_PTR
    # rows longer than 2^31 codes are refused (32-bit word and segment counts), even
    # when there are no ids; 2^31 itself passes the size checks
    assert f(*args(4, 10, 2 ** 31 + 16, 16)) == fp4.Status.ERR_SHAPE
    assert f(*args(0, 10, 2 ** 31 + 16, 16)) == fp4.Status.ERR_SHAPE
    assert f(*args(1, 10, 2 ** 31, 16)) == fp4.Status.ERR_NULL_PTR


def test_nv_dequant_host_validation(lib):
    f = lib.fp4_nv_dequant
    args = lambda r, h, g: (None, None, None, r, h, g, None, None)
    assert f(*args(4, 100, 16)) == fp4.Status.ERR_GROUP
    assert f(*args(4, 96, 32)) == fp4.Status.ERR_UNSUPPORTED
    assert f(*args(-1, 64, 16)) == fp4.Status.ERR_SHAPE
    assert f(*args(4, 0, 16)) == fp4.Status.ERR_SHAPE
    assert f(*args(0, 64, 16)) == fp4.Status.OK
    assert f(*args(4, 64, 16)) == fp4.Status.ERR_NULL_PTR
    assert f(*args(4, 2 ** 31 + 16, 16)) == fp4.Status.ERR_SHAPE
    assert f(*args(1, 2 ** 31, 16)) == fp4.Status.ERR_NULL_PTR


def test_mx_quantize_host_validation(lib):
    f = lib.fp4_mx_quantize
    assert f(None, None, None, 1, 33, None) == fp4.Status.ERR_SHAPE
    assert f(None, None, None, -1, 32, None) == fp4.Status.ERR_SHAPE
    assert f(None, None, None, 0, 64, None) == fp4.Status.OK
    assert f(None, None, None, 2, 64, None) == fp4.Status.ERR_NULL_PTR
    buf = ctypes.create_string_buffer(8192)
    base = ctypes.addressof(buf)
    base += (-base) % 16
    assert f(base + 1, base + 4096, base + 6000, 1, 64, None) == fp4.Status.ERR_ALIGN
    assert f(base, base + 64, base + 6000, 1, 64, None) == fp4.Status.ERR_ALIAS
    assert f(base, base + 4096, base + 4100, 1, 256, None) == fp4.Status.ERR_ALIAS


def test_alignment_refused_before_cuda(lib):
    buf = ctypes.create_string_buffer(1 << 16)
    base = ctypes.addressof(buf)
    base += (-base) % 16
    # odd bf16 output of the unpack
    assert lib.fp4_mx_unpack(base, base + 1024, base + 4097, 1, 64, None) == fp4.Status.ERR_ALIGN
    # ids not 8-aligned, global scale not 4-aligned, output odd
    g = lambda ids, gs, out: lib.fp4_nv_embedding_gather(ids, 2, base + 8192, base + 12288, gs, 4,
                                                         64, 16, out, None, None)
    assert g(base + 4, base + 16000, base + 20000) == fp4.Status.ERR_ALIGN
    assert g(base, base + 16002, base + 20000) == fp4.Status.ERR_ALIGN
    assert g(base, base + 16000, base + 20001) == fp4.Status.ERR_ALIGN
    assert lib.fp4_nv_dequant(base + 8192, base + 12288, base + 16001, 4, 64, 16, base + 20000,
                              None) == fp4.Status.ERR_ALIGN


def test_moe_gemm_host_validation(lib):
    f = lib.fp4_mx_moe_gemm
    g = lambda e, mr, n, k, ptr=None: f(ptr, ptr, e, mr, ptr, ptr, n, k, 8, ptr, ptr, None)
    assert g(1, 8, 64, 48) == fp4.Status.ERR_SHAPE       # k % 32
    assert g(1, 8, 48, 64) == fp4.Status.ERR_SHAPE       # n % 32
    assert g(70000, 8, 64, 64) == fp4.Status.ERR_SHAPE   # experts > 65535
    assert f(None, None, 1, 8, None, None, 64, 64, 2 ** 31 - 1000, None, None, None) \
        == fp4.Status.ERR_SHAPE                           # rows past 32-bit TMA coordinates
    assert g(32768, 8, 65536, 64) == fp4.Status.ERR_SHAPE  # weight rows experts * n = 2^31
    assert g(32767, 8, 65536, 64) == fp4.Status.ERR_NULL_PTR  # 2^31 - 2^16: within the bound
    assert g(0, 8, 64, 64) == fp4.Status.OK
    assert g(1, 0, 64, 64) == fp4.Status.OK
    assert g(1, 8, 64, 64) == fp4.Status.ERR_NULL_PTR
    buf = ctypes.create_string_buffer(1 << 16)
    base = ctypes.addressof(buf)
    base += (-base) % 16
    assert f(base + 8, base, 1, 8, base, base, 64, 64, 8, base, base, None) == fp4.Status.ERR_ALIGN


def test_pages_host_validation(lib):
    f = lib.fp4_mx_unpack_pages
    g = lambda n, pool, elems: f(None, n, None, None, pool, elems, None, None, None)
    assert g(2, 4, 48) == fp4.Status.ERR_SHAPE    # page_elems % 32
    assert g(2, 4, 0) == fp4.Status.ERR_SHAPE
    assert g(-1, 4, 64) == fp4.Status.ERR_SHAPE
    assert g(0, 4, 64) == fp4.Status.OK
    assert g(2, 0, 64) == fp4.Status.ERR_SHAPE    # ids but no pool
    assert g(2, 4, 64) == fp4.Status.ERR_NULL_PTR
    # pages longer than 2^31 codes are refused (32-bit word and segment counts)
    assert g(2, 4, 2 ** 31 + 32) == fp4.Status.ERR_SHAPE
    assert g(0, 4, 2 ** 31 + 32) == fp4.Status.ERR_SHAPE
    assert g(1, 4, 2 ** 31) == fp4.Status.ERR_NULL_PTR


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError, match="CUDA"):
        fp4.fp4_mx_unpack(torch.zeros(2, 16, dtype=torch.uint8), torch.zeros(2, 1, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        fp4.fp4_nv_embedding_gather(torch.zeros(3, dtype=torch.int64),
                                    torch.zeros(4, 8, dtype=torch.uint8),
                                    torch.zeros(4, 1, dtype=torch.uint8),
                                    torch.ones(1, dtype=torch.float32))


def test_wait_selftest_host_validation(lib):
    """Mode, null and alignment are checked before any CUDA call."""
    f = lib.fp4_wait_selftest
    base = 1 << 40
    assert f(3, base, None) == fp4.Status.ERR_SHAPE
    assert f(-1, base, None) == fp4.Status.ERR_SHAPE
    assert f(0, None, None) == fp4.Status.ERR_NULL_PTR
    assert f(1, base + 2, None) == fp4.Status.ERR_ALIGN


def test_moe_forward_host_validation(lib):
    """Sizes, pointers, alignment, workspace size and aliasing are checked on the host
    before any CUDA call (fake device addresses: nothing is dereferenced)."""
    ws = lib.fp4_mx_moe_workspace_bytes
    assert ws(16, 2, 4, 64, 64) > 16 * 2 * (4 * 64 + 2 * 64)
    assert ws(16, 2, 4, 63, 64) == -1 and ws(16, 2, 4, 64, 48) == -1      # n, k % 32
    assert ws(16, 0, 4, 64, 64) == -1 and ws(16, 2, 0, 64, 64) == -1      # topk, experts
    assert ws(2 ** 30, 4, 4, 64, 64) == -1                                 # slots >= 2^31
    assert ws(2 ** 31 - 1000, 1, 4, 64, 64) == -1                          # TMA row coordinates
    assert ws(16, 2, 2048, 2 ** 19, 64) == -1                              # experts * 2n = 2^31
    assert ws(16, 2, 2048, 64, 2 ** 20) == -1                              # experts * k = 2^31
    assert ws(16, 2, 2047, 2 ** 19, 2 ** 20) > 0                           # both just within
    f = lib.fp4_mx_moe_forward
    base = 1 << 40
    tokens, topk, experts, n, k = 16, 2, 4, 64, 64
    need = ws(tokens, topk, experts, n, k)
    a, ids, wts = base, base + (1 << 20), base + (2 << 20)
    w1, s1, w2, s2 = base + (3 << 20), base + (4 << 20), base + (5 << 20), base + (6 << 20)
    work, out, st = base + (8 << 20), base + (16 << 20), base + (17 << 20)

    def call(**kw):
        args = dict(a=a, ids=ids, wts=wts, tokens=tokens, topk=topk, experts=experts, cap=tokens,
                    w1=w1, s1=s1, w2=w2, s2=s2, n=n, k=k, work=work, work_bytes=need, out=out, st=st)
        args.update(kw)
        return f(args["a"], args["ids"], args["wts"], args["tokens"], args["topk"], args["experts"],
                 args["cap"], args["w1"], args["s1"], args["w2"], args["s2"], args["n"], args["k"],
                 args["work"], args["work_bytes"], args["out"], args["st"], None)

    assert call(n=48) == fp4.Status.ERR_SHAPE
    assert call(cap=-1) == fp4.Status.ERR_SHAPE
    assert call(tokens=0, a=None, ids=None) == fp4.Status.OK               # nothing launched
    assert call(st=None) == fp4.Status.ERR_NULL_PTR
    assert call(work=None) == fp4.Status.ERR_NULL_PTR
    assert call(a=a + 2) == fp4.Status.ERR_ALIGN
    assert call(work=work + 16) == fp4.Status.ERR_ALIGN                    # 256-byte workspace
    assert call(work_bytes=need - 1) == fp4.Status.ERR_SHAPE
    assert call(out=a) == fp4.Status.ERR_ALIAS
    assert call(work=w1 - 256) == fp4.Status.ERR_ALIAS                     # workspace over w1
    assert call(out=work + 256) == fp4.Status.ERR_ALIAS
