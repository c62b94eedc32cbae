"""GB300 (sm_103a) decode of block-scaled FP4 (E2M1) into bf16.

Python binding of the C ABI in ``include/fp4mx.h``. The functions below carry the
C entry points' names and only marshal arguments: they check dtypes, devices and
shapes, allocate the output tensor when none is given, and pass raw device
pointers plus the current CUDA stream to the library, where every step of the
decode runs in hand-written CUDA kernels. PyTorch supplies device memory and
streams only. There is no CPU path: CPU tensors, a missing library or a non-OK
status raise.

* ``fp4_mx_unpack(packed, scales_e8m0)`` -- MXFP4: E8M0 scale per 32 codes,
  applied as a wrapping int16 add of (E-127)<<7 into the bf16 exponent field,
  zero codes forced to +0.0 ("vllm-project/vllm pull 51583", "Motivation",
  "Implementation breakdown").
* ``fp4_mx_unpack_pages(page_ids, packed_pool, scales_pool)`` -- the MXFP4 unpack
  of pool pages picked by id (a paged FP4 KV cache with E8M0 scales).
* ``fp4_mx_quantize(x_bf16)`` -- the inverse direction: bf16 -> (packed E2M1
  codes, E8M0 scales), by the OCP MX v1.0 conversion (the pages name the step,
  MXFP4QuantizeUtil.quantize, but not its rule).
* ``fp4_mx_moe_gemm(a, expert_offsets, w_packed, w_scales)`` -- grouped MoE GEMM,
  bf16 activations x MXFP4 expert weights decoded into the tcgen05 operand.
* ``fp4_nv_embedding_gather(ids, weight, block_scale, global_scale)`` -- NVFP4
  embedding lookup dequantised at gather time: value * (e4m3 block scale * fp32
  global scale) in fp32, rounded to bf16 ("sgl-project/sglang pull 34222",
  "Implementation breakdown", "Key source snippets").
* ``fp4_nv_dequant(weight, block_scale, global_scale)`` -- the same NVFP4 decode
  over every row of a table (e.g. a tied lm_head; same page, "Comments", "Risks").
"""
from __future__ import annotations

from ._lib import Status, last_error, library_path, load, status_string  # noqa: F401

__all__ = ["fp4_mx_unpack", "fp4_mx_unpack_pages", "fp4_mx_quantize", "fp4_mx_moe_gemm",
           "fp4_mx_moe_forward", "fp4_mx_moe_workspace_bytes", "fp4_mx_moe_forward_noalloc",
           "fp4_mx_moe_static_scratch_bytes", "fp4_wait_selftest",
           "fp4_nv_embedding_gather",
           "fp4_nv_dequant",
           "fp4_status_string",
           "Fp4Error",
           "Status", "load", "library_path"]


class Fp4Error(ValueError):
    """A non-OK status from the library."""

    def __init__(self, where: str, code: int):
        self.code = Status(code) if code in Status._value2member_map_ else code
        detail = last_error() if code == Status.ERR_CUDA or code == Status.ERR_POINTER else ""
        super().__init__(f"{where}: {status_string(code)}" + (f" ({detail})" if detail else ""))


def fp4_status_string(code: int) -> str:
    return status_string(code)


def _torch():
    import torch
    return torch


def _check_cuda(t, name: str, dtypes):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path), got {t.device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes_void(stream.cuda_stream)


def ctypes_void(v):
    import ctypes
    return ctypes.c_void_p(int(v) if v else None)


def _ptr(t):
    return ctypes_void(t.data_ptr()) if t is not None and t.numel() else ctypes_void(0)


def _call(device, name: str, *args):
    """Calls the C entry point ``name`` with ``device`` (the tensors' device) as the
    current CUDA device, which the library's pointer checks and launches use."""
    torch = _torch()
    with torch.cuda.device(device):
        return getattr(load(), name)(*args)


def fp4_mx_unpack(packed, scales_e8m0, out=None, stream=None):
    """MXFP4 -> bf16. ``packed`` uint8 [..., k/2], ``scales_e8m0`` uint8 [..., k/32]
    with the same leading dimensions; returns (or fills ``out``) bf16 [..., k].
    Enqueued on ``stream`` (default: the current stream of the tensors' device)."""
    torch = _torch()
    _check_cuda(packed, "packed", (torch.uint8,))
    _check_cuda(scales_e8m0, "scales_e8m0", (torch.uint8,))
    if packed.dim() < 1 or scales_e8m0.dim() != packed.dim():
        raise ValueError("packed and scales_e8m0 must have the same number of dimensions")
    if packed.shape[:-1] != scales_e8m0.shape[:-1]:
        raise ValueError("packed and scales_e8m0 leading dimensions differ")
    k = packed.shape[-1] * 2
    if scales_e8m0.shape[-1] * 32 != k:
        raise ValueError(f"scales_e8m0 last dim must be k/32 = {k // 32}")
    rows = packed.numel() // packed.shape[-1] if packed.shape[-1] else 0
    shape = (*packed.shape[:-1], k)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=packed.device)
    else:
        _check_cuda(out, "out", (torch.bfloat16, torch.int16, torch.uint16))
        if tuple(out.shape) != shape:
            raise ValueError(f"out must have shape {shape}")
    code = _call(packed.device, "fp4_mx_unpack", _ptr(packed), _ptr(scales_e8m0), _ptr(out),
                 rows, k, _stream_handle(stream, packed.device))
    if code != Status.OK:
        raise Fp4Error("fp4_mx_unpack", code)
    return out


def fp4_nv_embedding_gather(ids, weight, block_scale, global_scale, group_size: int = 16,
                            out=None, err_flag=None, stream=None):
    """NVFP4 embedding gather-dequant -> bf16 [*ids.shape, hidden].

    ``ids`` int64 (any shape), ``weight`` uint8 [vocab, hidden/2], ``block_scale``
    float8_e4m3fn (or its uint8 bits) [vocab, hidden/16], ``global_scale`` fp32
    CUDA tensor with one element. ``err_flag`` (optional int32 CUDA tensor with one
    element) is set to Status.ERR_INDEX when an id is outside [0, vocab); such a
    row is written as +0.0."""
    torch = _torch()
    _check_cuda(ids, "ids", (torch.int64,))
    _check_cuda(weight, "weight", (torch.uint8,))
    _check_cuda(block_scale, "block_scale", (torch.float8_e4m3fn, torch.uint8))
    _check_cuda(global_scale, "global_scale", (torch.float32,))
    if global_scale.numel() != 1:
        raise ValueError("global_scale must have exactly one element")
    if weight.dim() != 2 or block_scale.dim() != 2:
        raise ValueError("weight and block_scale must be 2-D [vocab, ...]")
    vocab, half = weight.shape
    hidden = 2 * half
    if block_scale.shape[0] != vocab:
        raise ValueError("weight and block_scale have different vocab sizes")
    if group_size > 0 and hidden % group_size == 0 and block_scale.shape[1] * group_size != hidden:
        raise ValueError(f"block_scale must be [vocab, hidden/{group_size}]")
    shape = (*ids.shape, hidden)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=weight.device)
    else:
        _check_cuda(out, "out", (torch.bfloat16, torch.int16, torch.uint16))
        if tuple(out.shape) != shape:
            raise ValueError(f"out must have shape {shape}")
    if err_flag is not None:
        _check_cuda(err_flag, "err_flag", (torch.int32,))
    code = _call(
        weight.device, "fp4_nv_embedding_gather",
        _ptr(ids), ids.numel(), _ptr(weight), _ptr(block_scale), _ptr(global_scale), vocab,
        hidden, int(group_size), _ptr(out), _ptr(err_flag),
        _stream_handle(stream, weight.device))
    if code != Status.OK:
        raise Fp4Error("fp4_nv_embedding_gather", code)
    return out


def fp4_nv_dequant(weight, block_scale, global_scale, group_size: int = 16, out=None,
                   stream=None):
    """Dequantise a whole NVFP4 table -> bf16 [rows, hidden]: row r is what
    fp4_nv_embedding_gather writes for id r. ``weight`` uint8 [rows, hidden/2],
    ``block_scale`` float8_e4m3fn (or uint8 bits) [rows, hidden/16], ``global_scale``
    fp32 CUDA tensor with one element."""
    torch = _torch()
    _check_cuda(weight, "weight", (torch.uint8,))
    _check_cuda(block_scale, "block_scale", (torch.float8_e4m3fn, torch.uint8))
    _check_cuda(global_scale, "global_scale", (torch.float32,))
    if global_scale.numel() != 1:
        raise ValueError("global_scale must have exactly one element")
    if weight.dim() != 2 or block_scale.dim() != 2:
        raise ValueError("weight and block_scale must be 2-D [rows, ...]")
    rows, half = weight.shape
    hidden = 2 * half
    if block_scale.shape[0] != rows:
        raise ValueError("weight and block_scale have different row counts")
    if group_size > 0 and hidden % group_size == 0 and block_scale.shape[1] * group_size != hidden:
        raise ValueError(f"block_scale must be [rows, hidden/{group_size}]")
    if out is None:
        out = torch.empty((rows, hidden), dtype=torch.bfloat16, device=weight.device)
    else:
        _check_cuda(out, "out", (torch.bfloat16, torch.int16, torch.uint16))
        if tuple(out.shape) != (rows, hidden):
            raise ValueError(f"out must have shape {(rows, hidden)}")
    code = _call(weight.device, "fp4_nv_dequant", _ptr(weight), _ptr(block_scale),
                 _ptr(global_scale), rows, hidden, int(group_size), _ptr(out),
                 _stream_handle(stream, weight.device))
    if code != Status.OK:
        raise Fp4Error("fp4_nv_dequant", code)
    return out


def fp4_mx_quantize(x, packed_out=None, scales_out=None, stream=None):
    """bf16 [..., k] (k % 32 == 0) -> (packed uint8 [..., k/2], E8M0 uint8 [..., k/32]):
    shared exponent floor(log2 amax) - 2 per 32 values, elements rounded to nearest
    even on the E2M1 grid with saturation at 6 (OCP MX v1.0)."""
    torch = _torch()
    _check_cuda(x, "x", (torch.bfloat16, torch.int16, torch.uint16))
    if x.dim() < 1 or x.shape[-1] % 32:
        raise ValueError("x must have a last dimension that is a multiple of 32")
    k = x.shape[-1]
    rows = x.numel() // k if k else 0
    p_shape, s_shape = (*x.shape[:-1], k // 2), (*x.shape[:-1], k // 32)
    if packed_out is None:
        packed_out = torch.empty(p_shape, dtype=torch.uint8, device=x.device)
    if scales_out is None:
        scales_out = torch.empty(s_shape, dtype=torch.uint8, device=x.device)
    _check_cuda(packed_out, "packed_out", (torch.uint8,))
    _check_cuda(scales_out, "scales_out", (torch.uint8,))
    if tuple(packed_out.shape) != p_shape or tuple(scales_out.shape) != s_shape:
        raise ValueError(f"outputs must have shapes {p_shape} and {s_shape}")
    code = _call(x.device, "fp4_mx_quantize", _ptr(x), _ptr(packed_out), _ptr(scales_out), rows,
                 k, _stream_handle(stream, x.device))
    if code != Status.OK:
        raise Fp4Error("fp4_mx_quantize", code)
    return packed_out, scales_out


def fp4_mx_moe_gemm(a, expert_offsets, w_packed, w_scales, max_rows_per_expert: int,
                    out=None, status=None, stream=None):
    """Grouped MoE GEMM: ``a`` bf16 [T, k] (rows grouped by expert), ``expert_offsets``
    int64 [E + 1] on the device, ``w_packed`` uint8 [E, n, k/2], ``w_scales`` uint8
    [E, n, k/32] -> bf16 [T, n] with out[r] = a[r] @ W_e^T for r in expert e's rows.
    ``status`` (int32 CUDA tensor, one element; allocated if None) receives
    Status.ERR_TIMEOUT or Status.ERR_SHAPE from the device; the caller reads it after
    synchronising. Returns (out, status)."""
    torch = _torch()
    _check_cuda(a, "a", (torch.bfloat16, torch.int16, torch.uint16))
    _check_cuda(expert_offsets, "expert_offsets", (torch.int64,))
    _check_cuda(w_packed, "w_packed", (torch.uint8,))
    _check_cuda(w_scales, "w_scales", (torch.uint8,))
    if a.dim() != 2 or w_packed.dim() != 3 or w_scales.dim() != 3:
        raise ValueError("a must be [T, k], w_packed [E, n, k/2], w_scales [E, n, k/32]")
    experts, n, half = w_packed.shape
    k = 2 * half
    if a.shape[1] != k or tuple(w_scales.shape) != (experts, n, k // 32):
        raise ValueError("inconsistent k / n / expert counts")
    if expert_offsets.numel() != experts + 1:
        raise ValueError("expert_offsets must have experts + 1 entries")
    if out is None:
        out = torch.empty((a.shape[0], n), dtype=torch.bfloat16, device=a.device)
    _check_cuda(out, "out", (torch.bfloat16, torch.int16, torch.uint16))
    if tuple(out.shape) != (a.shape[0], n):
        raise ValueError(f"out must have shape {(a.shape[0], n)}")
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=a.device)
    _check_cuda(status, "status", (torch.int32,))
    code = _call(a.device, "fp4_mx_moe_gemm", _ptr(a), _ptr(expert_offsets), experts,
                 int(max_rows_per_expert), _ptr(w_packed), _ptr(w_scales), n, k, a.shape[0],
                 _ptr(out), _ptr(status), _stream_handle(stream, a.device))
    if code != Status.OK:
        raise Fp4Error("fp4_mx_moe_gemm", code)
    return out, status


def fp4_mx_moe_workspace_bytes(tokens: int, topk: int, experts: int, n: int, k: int) -> int:
    """Bytes of device workspace fp4_mx_moe_forward needs (raises on invalid sizes)."""
    size = load().fp4_mx_moe_workspace_bytes(int(tokens), int(topk), int(experts), int(n), int(k))
    if size < 0:
        raise ValueError("invalid MoE layer sizes")
    return int(size)


def fp4_mx_moe_forward(a, topk_ids, topk_weights, w1_packed, w1_scales, w2_packed, w2_scales,
                       max_rows_per_expert=None, out=None, workspace=None, status=None,
                       stream=None):
    """The MoE layer with MXFP4 experts: ``a`` bf16 [M, k], ``topk_ids`` int32 [M, topk],
    ``topk_weights`` fp32 [M, topk], ``w1_*`` [E, 2n, k/2] / [E, 2n, k/32] (gate rows
    then up rows), ``w2_*`` [E, k, n/2] / [E, k, n/32] -> bf16 [M, k]:
    out[m] = sum_j w[m, j] * (silu(gate) * up) @ W2_e^T. ``max_rows_per_expert``
    defaults to M (enough whenever no token repeats an expert among its slots);
    ``workspace`` (uint8 CUDA tensor, allocated if None) must hold
    fp4_mx_moe_workspace_bytes(M, topk, E, n, k) bytes. Returns (out, status)."""
    torch = _torch()
    _check_cuda(a, "a", (torch.bfloat16, torch.int16, torch.uint16))
    _check_cuda(topk_ids, "topk_ids", (torch.int32,))
    _check_cuda(topk_weights, "topk_weights", (torch.float32,))
    for t, name in ((w1_packed, "w1_packed"), (w1_scales, "w1_scales"), (w2_packed, "w2_packed"),
                    (w2_scales, "w2_scales")):
        _check_cuda(t, name, (torch.uint8,))
    if a.dim() != 2 or topk_ids.dim() != 2 or w1_packed.dim() != 3 or w2_packed.dim() != 3:
        raise ValueError("a [M, k], topk_ids [M, topk], w1_packed [E, 2n, k/2], w2_packed [E, k, n/2]")
    tokens, k = a.shape
    topk = topk_ids.shape[1]
    experts, two_n, half_k = w1_packed.shape
    n = two_n // 2
    if (2 * half_k != k or two_n % 2 or topk_ids.shape[0] != tokens
            or tuple(topk_weights.shape) != tuple(topk_ids.shape)
            or tuple(w1_scales.shape) != (experts, two_n, k // 32)
            or tuple(w2_packed.shape) != (experts, k, n // 2)
            or tuple(w2_scales.shape) != (experts, k, n // 32)):
        raise ValueError("inconsistent MoE layer shapes")
    need = fp4_mx_moe_workspace_bytes(tokens, topk, experts, n, k)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=a.device)
    _check_cuda(workspace, "workspace", (torch.uint8,))
    if out is None:
        out = torch.empty((tokens, k), dtype=torch.bfloat16, device=a.device)
    _check_cuda(out, "out", (torch.bfloat16, torch.int16, torch.uint16))
    if tuple(out.shape) != (tokens, k):
        raise ValueError(f"out must have shape {(tokens, k)}")
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=a.device)
    _check_cuda(status, "status", (torch.int32,))
    max_rows = tokens if max_rows_per_expert is None else int(max_rows_per_expert)
    code = _call(
        a.device, "fp4_mx_moe_forward",
        _ptr(a), _ptr(topk_ids), _ptr(topk_weights), tokens, topk, experts, max_rows,
        _ptr(w1_packed), _ptr(w1_scales), _ptr(w2_packed), _ptr(w2_scales), n, k,
        _ptr(workspace), workspace.numel(), _ptr(out), _ptr(status),
        _stream_handle(stream, a.device))
    if code != Status.OK:
        raise Fp4Error("fp4_mx_moe_forward", code)
    return out, status


def fp4_mx_moe_static_scratch_bytes() -> int:
    """Bytes of the static device scratch fp4_mx_moe_forward_noalloc uses."""
    return int(load().fp4_mx_moe_static_scratch_bytes())


def fp4_mx_moe_forward_noalloc(a, topk_ids, topk_weights, w1_packed, w1_scales, w2_packed,
                               w2_scales, max_rows_per_expert=None, out=None, status=None,
                               stream=None):
    """fp4_mx_moe_forward on the library's static device scratch: no workspace and
    no allocation by the library (``out`` and ``status`` are allocated here when
    not given). Layers that need more scratch than fp4_mx_moe_static_scratch_bytes()
    raise Fp4Error (ERR_SHAPE). Calls must be ordered on one device. Returns
    (out, status)."""
    torch = _torch()
    _check_cuda(a, "a", (torch.bfloat16, torch.int16, torch.uint16))
    _check_cuda(topk_ids, "topk_ids", (torch.int32,))
    _check_cuda(topk_weights, "topk_weights", (torch.float32,))
    for t, name in ((w1_packed, "w1_packed"), (w1_scales, "w1_scales"), (w2_packed, "w2_packed"),
                    (w2_scales, "w2_scales")):
        _check_cuda(t, name, (torch.uint8,))
    if a.dim() != 2 or topk_ids.dim() != 2 or w1_packed.dim() != 3 or w2_packed.dim() != 3:
        raise ValueError("a [M, k], topk_ids [M, topk], w1_packed [E, 2n, k/2], w2_packed [E, k, n/2]")
    tokens, k = a.shape
    topk = topk_ids.shape[1]
    experts, two_n, half_k = w1_packed.shape
    n = two_n // 2
    if (2 * half_k != k or two_n % 2 or topk_ids.shape[0] != tokens
            or tuple(topk_weights.shape) != tuple(topk_ids.shape)
            or tuple(w1_scales.shape) != (experts, two_n, k // 32)
            or tuple(w2_packed.shape) != (experts, k, n // 2)
            or tuple(w2_scales.shape) != (experts, k, n // 32)):
        raise ValueError("inconsistent MoE layer shapes")
    if out is None:
        out = torch.empty((tokens, k), dtype=torch.bfloat16, device=a.device)
    _check_cuda(out, "out", (torch.bfloat16, torch.int16, torch.uint16))
    if tuple(out.shape) != (tokens, k):
        raise ValueError(f"out must have shape {(tokens, k)}")
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=a.device)
    _check_cuda(status, "status", (torch.int32,))
    max_rows = tokens if max_rows_per_expert is None else int(max_rows_per_expert)
    code = _call(
        a.device, "fp4_mx_moe_forward_noalloc",
        _ptr(a), _ptr(topk_ids), _ptr(topk_weights), tokens, topk, experts, max_rows,
        _ptr(w1_packed), _ptr(w1_scales), _ptr(w2_packed), _ptr(w2_scales), n, k, _ptr(out),
        _ptr(status), _stream_handle(stream, a.device))
    if code != Status.OK:
        raise Fp4Error("fp4_mx_moe_forward_noalloc", code)
    return out, status


def fp4_wait_selftest(mode, status=None, device="cuda", stream=None):
    """Run one bounded mbarrier wait of the kind that guards the tensor-core
    kernels on a barrier nothing arrives on (mode 0: spinning wait, 1: sleeping
    wait; mode 2: a control whose phase completes). The kernel ends when the wait
    gives up and sets ``status`` (an int32 CUDA tensor, allocated here as zero when
    not given) to Status.ERR_TIMEOUT. Returns ``status``."""
    torch = _torch()
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=device)
    _check_cuda(status, "status", (torch.int32,))
    code = _call(status.device, "fp4_wait_selftest", int(mode), _ptr(status),
                 _stream_handle(stream, status.device))
    if code != Status.OK:
        raise Fp4Error("fp4_wait_selftest", code)
    return status


def fp4_mx_unpack_pages(page_ids, packed_pool, scales_pool, out=None, err_flag=None,
                        stream=None):
    """Paged MXFP4 dequant: ``page_ids`` int64 (any shape), ``packed_pool`` uint8
    [pool_pages, page_elems/2], ``scales_pool`` uint8 [pool_pages, page_elems/32] ->
    bf16 [*page_ids.shape, page_elems], each row the fp4_mx_unpack of its page.
    ``err_flag`` (optional int32 CUDA tensor) is set to Status.ERR_INDEX for ids
    outside the pool; their rows are +0.0."""
    torch = _torch()
    _check_cuda(page_ids, "page_ids", (torch.int64,))
    _check_cuda(packed_pool, "packed_pool", (torch.uint8,))
    _check_cuda(scales_pool, "scales_pool", (torch.uint8,))
    if packed_pool.dim() != 2 or scales_pool.dim() != 2:
        raise ValueError("pools must be 2-D [pool_pages, ...]")
    pool_pages, half = packed_pool.shape
    page_elems = 2 * half
    if page_elems % 32 or tuple(scales_pool.shape) != (pool_pages, page_elems // 32):
        raise ValueError("scales_pool must be [pool_pages, page_elems/32], page_elems % 32 == 0")
    shape = (*page_ids.shape, page_elems)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=packed_pool.device)
    else:
        _check_cuda(out, "out", (torch.bfloat16, torch.int16, torch.uint16))
        if tuple(out.shape) != shape:
            raise ValueError(f"out must have shape {shape}")
    if err_flag is not None:
        _check_cuda(err_flag, "err_flag", (torch.int32,))
    code = _call(packed_pool.device, "fp4_mx_unpack_pages", _ptr(page_ids), page_ids.numel(),
                 _ptr(packed_pool), _ptr(scales_pool), pool_pages, page_elems, _ptr(out),
                 _ptr(err_flag), _stream_handle(stream, packed_pool.device))
    if code != Status.OK:
        raise Fp4Error("fp4_mx_unpack_pages", code)
    return out
