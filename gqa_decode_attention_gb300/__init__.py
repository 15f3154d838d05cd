"""GB300-native grouped-query decode attention: Python binding.

A thin ctypes layer over ``libgqa_decode.so`` (the C ABI declared in
``include/gqa_decode.h``).  Functions carry the C entry points' names and
only marshal arguments: torch tensors supply device memory and the current
CUDA stream; every step of the computation runs in the library's kernels.
There is no fallback: if the library is missing, importing a function that
needs it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_decode.so")

STATUS = {
    0: "GQA_OK",
    1: "GQA_ERR_INVALID_ARG",
    2: "GQA_ERR_UNSUPPORTED",
    3: "GQA_ERR_ALIGNMENT",
    4: "GQA_ERR_NO_MEMORY",
    5: "GQA_ERR_CUDA",
    6: "GQA_ERR_DEVICE_TIMEOUT",
    7: "GQA_ERR_DEVICE_INDEX",
}
GQA_OK = 0

# Every symbol the headers in include/ declare.
EXPORTS = [
    "gqa_status_string", "gqa_version", "gqa_decode", "gqa_decode_num_splits",
    "gqa_decode_workspace_bytes", "gqa_decode_ex", "gqa_decode_dv", "gqa_decode_dv_num_splits",
    "gqa_decode_dv_workspace_bytes", "gqa_decode_dense_engine",
    "gqa_decode_noalloc", "gqa_decode_noalloc_scratch_bytes",
    "gqa_decode_host", "gqa_decode_paged_fp8", "gqa_decode_paged_fp8_dev_scales", "gqa_decode_paged", "gqa_decode_paged_ex",
    "gqa_decode_paged_num_splits", "gqa_decode_paged_workspace_bytes", "gqa_decode_paged_dev_scales",
    "gqa_paged_gather_fp8", "gqa_fp8_e4m3fn_to_f32", "gqa_device_status", "gqa_set_wait_limit_ns",
    "gqa_debug_set_fault_mode", "gqa_debug_set_kernel_events", "gqa_debug_read_stream",
    "gqa_decode_paged_engine", "gqa_debug_set_paged_engine",
]


class GQAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(int(status), status)}")


_lib_handle = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libgqa_decode.so (built by ``gqa_decode_attention_gb300.build``)."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m gqa_decode_attention_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i, f, st, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
    lib.gqa_status_string.restype = ctypes.c_char_p
    lib.gqa_status_string.argtypes = [st]
    lib.gqa_version.restype = ctypes.c_char_p
    lib.gqa_version.argtypes = []
    lib.gqa_decode.restype = st
    lib.gqa_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.gqa_decode_num_splits.restype = i
    lib.gqa_decode_num_splits.argtypes = [i] * 6
    lib.gqa_decode_workspace_bytes.restype = sz
    lib.gqa_decode_workspace_bytes.argtypes = [i] * 7
    lib.gqa_decode_ex.restype = st
    lib.gqa_decode_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
    lib.gqa_decode_dv.restype = st
    lib.gqa_decode_dv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, sz, vp]
    lib.gqa_decode_dv_num_splits.restype = i
    lib.gqa_decode_dv_num_splits.argtypes = [i] * 7
    lib.gqa_decode_dense_engine.restype = i
    lib.gqa_decode_dense_engine.argtypes = [i] * 7
    lib.gqa_decode_dv_workspace_bytes.restype = sz
    lib.gqa_decode_dv_workspace_bytes.argtypes = [i] * 8
    lib.gqa_decode_noalloc.restype = st
    lib.gqa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.gqa_decode_noalloc_scratch_bytes.restype = sz
    lib.gqa_decode_noalloc_scratch_bytes.argtypes = []
    lib.gqa_decode_host.restype = st
    lib.gqa_decode_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.gqa_decode_paged_fp8.restype = st
    lib.gqa_decode_paged_fp8.argtypes = [vp, vp, vp, vp, vp, vp, f, f, vp, vp] + [i] * 8 + [f, vp]
    lib.gqa_decode_paged_fp8_dev_scales.restype = st
    lib.gqa_decode_paged_fp8_dev_scales.argtypes = [vp] * 8 + [i, vp, vp] + [i] * 8 + [f, vp]
    lib.gqa_decode_paged.restype = st
    lib.gqa_decode_paged.argtypes = [vp, vp, vp, i, f, f, vp, vp, vp, vp] + [i] * 8 + [f, vp]
    lib.gqa_decode_paged_ex.restype = st
    lib.gqa_decode_paged_ex.argtypes = [vp, vp, vp, i, f, f, vp, vp, vp, vp] + [i] * 8 + [f, i, vp, sz, vp]
    lib.gqa_decode_paged_dev_scales.restype = st
    lib.gqa_decode_paged_dev_scales.argtypes = [vp, vp, vp, i, vp, vp, i, vp, vp, vp, vp] + [i] * 8 + [f, i, vp, sz, vp]
    lib.gqa_decode_paged_num_splits.restype = i
    lib.gqa_decode_paged_num_splits.argtypes = [i] * 8
    lib.gqa_decode_paged_workspace_bytes.restype = sz
    lib.gqa_decode_paged_workspace_bytes.argtypes = [i] * 9
    lib.gqa_paged_gather_fp8.restype = st
    lib.gqa_paged_gather_fp8.argtypes = [vp, vp, vp, vp] + [i] * 7 + [vp]
    lib.gqa_fp8_e4m3fn_to_f32.restype = st
    lib.gqa_fp8_e4m3fn_to_f32.argtypes = [vp, vp, i, vp]
    lib.gqa_device_status.restype = st
    lib.gqa_device_status.argtypes = [vp]
    lib.gqa_set_wait_limit_ns.restype = None
    lib.gqa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.gqa_debug_set_fault_mode.restype = None
    lib.gqa_debug_set_fault_mode.argtypes = [i]
    lib.gqa_debug_set_kernel_events.restype = None
    lib.gqa_debug_set_kernel_events.argtypes = [vp, vp]
    lib.gqa_decode_paged_engine.restype = i
    lib.gqa_decode_paged_engine.argtypes = [i] * 7
    lib.gqa_debug_set_paged_engine.restype = None
    lib.gqa_debug_set_paged_engine.argtypes = [i]
    lib.gqa_debug_read_stream.restype = st
    lib.gqa_debug_read_stream.argtypes = [vp, sz, vp, vp]
    _lib_handle = lib
    return lib


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != GQA_OK:
        raise GQAError(status, where)


def _need(t: torch.Tensor, name: str, dtype, device_type: str):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device.type != device_type:
        raise ValueError(f"{name}: expected a {device_type} tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _need_shape(t, name: str, shape, dtype, like: torch.Tensor):
    """A caller-supplied tensor the library reads or writes through a raw
    pointer: it must have exactly the shape the call implies (a smaller one
    would be read or written out of bounds), the dtype, and lie contiguous on
    the device of `like`."""
    if t is None:
        return
    _need(t, name, dtype, like.device.type)
    if t.device != like.device:
        raise ValueError(f"{name}: expected a tensor on {like.device}, got {t.device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _dense_shapes(fn: str, q, k, v, out, lse, Dv=None):
    """Shape checks shared by the dense entry points: q [B,Sq,Hq,D],
    k [B,Skv,Hkv,D], v [B,Skv,Hkv,Dv], out [B,Sq,Hq,Dv], lse [B,Hq,Sq]."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError(f"{fn}: q, k and v must be 4-D")
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    Dv = D if Dv is None else Dv
    if tuple(k.shape) != (B, Skv, Hkv, D) or tuple(v.shape) != (B, Skv, Hkv, Dv):
        raise ValueError(f"{fn}: k must be [B,Skv,Hkv,{D}] and v [B,Skv,Hkv,{Dv}] with q's batch")
    for t, n in ((k, "k"), (v, "v")):
        if t.device != q.device:
            raise ValueError(f"{fn}: {n} is on {t.device}, q on {q.device}")
    _need_shape(out, "out", (B, Sq, Hq, Dv), torch.bfloat16, q)
    _need_shape(lse, "lse", (B, Hq, Sq), torch.float32, q)


def _scale_arg(scale):
    return 0.0 if scale is None else float(scale)


# ---------------------------------------------------------------------------
# dense
# ---------------------------------------------------------------------------
def gqa_decode(q, k, v, out=None, lse=None, scale=None, stream=None, with_lse=True):
    """Dense GQA decode.  q [B,Sq,Hq,D], k/v [B,Skv,Hkv,D] bf16 on CUDA.

    Returns (out [B,Sq,Hq,D] bf16, lse [B,Hq,Sq] fp32 or None).
    """
    return gqa_decode_ex(q, k, v, out=out, lse=lse, scale=scale, num_splits=0, workspace=None,
                         stream=stream, with_lse=with_lse)


def gqa_decode_ex(q, k, v, out=None, lse=None, scale=None, num_splits=0, workspace=None, stream=None,
                  with_lse=True):
    """gqa_decode with an explicit split count (0 = automatic) and an optional
    caller workspace (a CUDA uint8 tensor of at least gqa_decode_workspace_bytes)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, "cuda")
    _dense_shapes("gqa_decode_ex", q, k, v, out, lse)
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    st = lib.gqa_decode_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Sq, Skv, Hq, Hkv, D,
                           _scale_arg(scale), int(num_splits), ws_ptr, ws_bytes, _stream(stream))
    _check(st, "gqa_decode_ex")
    return out, lse


def gqa_decode_dv(q, k, v, out=None, lse=None, scale=None, num_splits=0, workspace=None, stream=None,
                  with_lse=True):
    """Dense decode with a score head size Dqk (q, k) different from the value
    head size Dv (v, out): q [B,Sq,Hq,Dqk], k [B,Skv,Hkv,Dqk], v [B,Skv,Hkv,Dv].

    Returns (out [B,Sq,Hq,Dv] bf16, lse [B,Hq,Sq] fp32 or None)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, "cuda")
    B, Sq, Hq, Dqk = q.shape
    _, Skv, Hkv, _ = k.shape
    Dv = v.shape[-1]
    _dense_shapes("gqa_decode_dv", q, k, v, out, lse, Dv=Dv)
    if out is None:
        out = torch.empty((B, Sq, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    st = lib.gqa_decode_dv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Sq, Skv, Hq, Hkv, Dqk, Dv,
                           _scale_arg(scale), int(num_splits), ws_ptr, ws_bytes, _stream(stream))
    _check(st, "gqa_decode_dv")
    return out, lse


def gqa_decode_dv_num_splits(B, Sq, Skv, Hq, Hkv, Dqk, Dv) -> int:
    n = load_library().gqa_decode_dv_num_splits(B, Sq, Skv, Hq, Hkv, Dqk, Dv)
    if n < 0:
        raise GQAError(-n, "gqa_decode_dv_num_splits")
    return n


ENGINES = {0: "mma.sync", 1: "tcgen05"}


def gqa_decode_dense_engine(B, Sq, Skv, Hq, Hkv, Dqk, Dv=None) -> str:
    """Kernel engine a dense call of this shape runs: "mma.sync" or "tcgen05"."""
    n = load_library().gqa_decode_dense_engine(B, Sq, Skv, Hq, Hkv, Dqk, Dqk if Dv is None else Dv)
    if n < 0:
        raise GQAError(-n, "gqa_decode_dense_engine")
    return ENGINES[n]


def gqa_decode_dv_workspace_bytes(B, Sq, Skv, Hq, Hkv, Dqk, Dv, num_splits=0) -> int:
    return int(load_library().gqa_decode_dv_workspace_bytes(B, Sq, Skv, Hq, Hkv, Dqk, Dv, int(num_splits)))


def gqa_decode_noalloc(q, k, v, out, lse=None, scale=None, num_splits=0, stream=None):
    """Allocation-free dense decode (fixed in-library scratch, caller-owned
    out / lse; see include/gqa_decode.h).  Allocates nothing, not even outputs."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, "cuda")
    _dense_shapes("gqa_decode_noalloc", q, k, v, out, lse)
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    st = lib.gqa_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Sq, Skv, Hq, Hkv, D,
                                _scale_arg(scale), int(num_splits), _stream(stream))
    _check(st, "gqa_decode_noalloc")
    return out, lse


def gqa_decode_noalloc_scratch_bytes() -> int:
    return int(load_library().gqa_decode_noalloc_scratch_bytes())


def gqa_decode_num_splits(B, Sq, Skv, Hq, Hkv, D) -> int:
    n = load_library().gqa_decode_num_splits(B, Sq, Skv, Hq, Hkv, D)
    if n < 0:
        raise GQAError(-n, "gqa_decode_num_splits")
    return n


def gqa_decode_workspace_bytes(B, Sq, Skv, Hq, Hkv, D, num_splits=0) -> int:
    return int(load_library().gqa_decode_workspace_bytes(B, Sq, Skv, Hq, Hkv, D, int(num_splits)))


def gqa_decode_host(q, k, v, out, lse=None, scale=None, stream=None):
    """End-to-end form on HOST (ideally pinned) tensors; returns when done."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, "cpu")
    _dense_shapes("gqa_decode_host", q, k, v, out, lse)
    B, Sq, Hq, D = q.shape
    _, Skv, Hkv, _ = k.shape
    st = lib.gqa_decode_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Sq, Skv, Hq, Hkv, D,
                             _scale_arg(scale), _stream(stream))
    _check(st, "gqa_decode_host")
    return out, lse


# ---------------------------------------------------------------------------
# sparse paged FP8
# ---------------------------------------------------------------------------
def gqa_decode_paged_fp8(q, gate, k_pool, v_pool, page_table, topk_idx, k_scale=1.0, v_scale=1.0, out=None,
                         lse=None, scale=None, stream=None, with_lse=True, k_scales=None, v_scales=None):
    """Sparse paged decode over an FP8 E4M3FN pool with a sigmoid gate.

    q, gate [B,Hq,D] bf16; pools uint8 [num_pages, page_size, Hkv, D];
    page_table int32 [B, pages_per_req]; topk_idx int32 [B, topk].
    k_scales / v_scales: optional CUDA fp32 tensors of 1 or Hkv device-side
    scales (replace k_scale / v_scale).
    Returns (out [B,Hq,D] bf16, lse [B,Hq] fp32 or None).
    """
    lib = load_library()
    _need(q, "q", torch.bfloat16, "cuda")
    _need(gate, "gate", torch.bfloat16, "cuda")
    for t, n in ((k_pool, "k_pool"), (v_pool, "v_pool")):
        _need(t, n, torch.uint8, "cuda")
    _need(page_table, "page_table", torch.int32, "cuda")
    _need(topk_idx, "topk_idx", torch.int32, "cuda")
    if q.dim() != 3 or k_pool.dim() != 4 or page_table.dim() != 2 or topk_idx.dim() != 2:
        raise ValueError("gqa_decode_paged_fp8: q [B,Hq,D], pools [pages,page_size,Hkv,D], page_table and "
                         "topk_idx 2-D")
    B, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_pool.shape
    if tuple(v_pool.shape) != tuple(k_pool.shape) or k_pool.shape[3] != D:
        raise ValueError("gqa_decode_paged_fp8: v_pool must have k_pool's shape, with q's head size")
    if page_table.shape[0] != B or topk_idx.shape[0] != B:
        raise ValueError("gqa_decode_paged_fp8: page_table and topk_idx need one row per request")
    for t, n in ((k_pool, "k_pool"), (v_pool, "v_pool"), (page_table, "page_table"), (topk_idx, "topk_idx")):
        if t.device != q.device:
            raise ValueError(f"gqa_decode_paged_fp8: {n} is on {t.device}, q on {q.device}")
    _need_shape(gate, "gate", (B, Hq, D), torch.bfloat16, q)
    _need_shape(out, "out", (B, Hq, D), torch.bfloat16, q)
    _need_shape(lse, "lse", (B, Hq), torch.float32, q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if k_scales is not None or v_scales is not None:
        _need(k_scales, "k_scales", torch.float32, "cuda")
        _need(v_scales, "v_scales", torch.float32, "cuda")
        st = lib.gqa_decode_paged_fp8_dev_scales(_ptr(q), _ptr(gate), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                                 _ptr(topk_idx), _ptr(k_scales), _ptr(v_scales), k_scales.numel(),
                                                 _ptr(out), _ptr(lse), B, Hq, Hkv, D, page_size,
                                                 page_table.shape[1], num_pages, topk_idx.shape[1],
                                                 _scale_arg(scale), _stream(stream))
        _check(st, "gqa_decode_paged_fp8_dev_scales")
        return out, lse
    st = lib.gqa_decode_paged_fp8(_ptr(q), _ptr(gate), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                  _ptr(topk_idx), float(k_scale), float(v_scale), _ptr(out), _ptr(lse),
                                  B, Hq, Hkv, D, page_size, page_table.shape[1], num_pages,
                                  topk_idx.shape[1], _scale_arg(scale), _stream(stream))
    _check(st, "gqa_decode_paged_fp8")
    return out, lse


GQA_KV_BF16 = 0
GQA_KV_FP8_E4M3FN = 1
GQA_KV_INT8 = 2


def _kv_dtype(k_pool) -> int:
    if k_pool.dtype == torch.bfloat16:
        return GQA_KV_BF16
    if k_pool.dtype == torch.uint8:
        return GQA_KV_FP8_E4M3FN
    if k_pool.dtype == torch.int8:
        return GQA_KV_INT8
    raise TypeError(f"k_pool: expected bfloat16, uint8 (E4M3FN codes) or int8, got {k_pool.dtype}")


def gqa_decode_paged(q, k_pool, v_pool, page_table, seq_lens, k_scale=1.0, v_scale=1.0, out=None, lse=None,
                     scale=None, num_splits=0, workspace=None, stream=None, with_lse=True, k_scales=None,
                     v_scales=None):
    """Paged decode over every token of each request (no top-K).

    q [B,Sq,Hq,D] bf16; pools [num_pages, page_size, Hkv, D] of bf16, of
    uint8 E4M3FN codes or of int8 codes (for 8-bit codes k_scale / v_scale
    apply); page_table int32
    [B, pages_per_req]; seq_lens int32 [B].  num_splits 0 = automatic;
    workspace: optional CUDA uint8 tensor of gqa_decode_paged_workspace_bytes.
    k_scales / v_scales: optional CUDA fp32 tensors of 1 or Hkv device-side
    scales (8-bit pools; replace k_scale / v_scale).
    Returns (out [B,Sq,Hq,D] bf16, lse [B,Hq,Sq] fp32 or None).
    """
    lib = load_library()
    _need(q, "q", torch.bfloat16, "cuda")
    kvd = _kv_dtype(k_pool)
    for t, n in ((k_pool, "k_pool"), (v_pool, "v_pool")):
        _need(t, n, k_pool.dtype, "cuda")
    _need(page_table, "page_table", torch.int32, "cuda")
    _need(seq_lens, "seq_lens", torch.int32, "cuda")
    if q.dim() != 4 or k_pool.dim() != 4 or page_table.dim() != 2:
        raise ValueError("gqa_decode_paged: q [B,Sq,Hq,D], pools [pages,page_size,Hkv,D], page_table 2-D")
    B, Sq, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_pool.shape
    if tuple(v_pool.shape) != tuple(k_pool.shape) or k_pool.shape[3] != D:
        raise ValueError("gqa_decode_paged: v_pool must have k_pool's shape, with q's head size")
    if page_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("gqa_decode_paged: page_table needs one row and seq_lens one entry per request")
    for t, n in ((k_pool, "k_pool"), (v_pool, "v_pool"), (page_table, "page_table"), (seq_lens, "seq_lens")):
        if t.device != q.device:
            raise ValueError(f"gqa_decode_paged: {n} is on {t.device}, q on {q.device}")
    _need_shape(out, "out", (B, Sq, Hq, D), torch.bfloat16, q)
    _need_shape(lse, "lse", (B, Hq, Sq), torch.float32, q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and with_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    if k_scales is not None or v_scales is not None:
        _need(k_scales, "k_scales", torch.float32, "cuda")
        _need(v_scales, "v_scales", torch.float32, "cuda")
        st = lib.gqa_decode_paged_dev_scales(_ptr(q), _ptr(k_pool), _ptr(v_pool), kvd, _ptr(k_scales),
                                             _ptr(v_scales), k_scales.numel(), _ptr(page_table), _ptr(seq_lens),
                                             _ptr(out), _ptr(lse), B, Sq, Hq, Hkv, D, page_size,
                                             page_table.shape[1], num_pages, _scale_arg(scale), int(num_splits),
                                             ws_ptr, ws_bytes, _stream(stream))
        _check(st, "gqa_decode_paged_dev_scales")
        return out, lse
    st = lib.gqa_decode_paged_ex(_ptr(q), _ptr(k_pool), _ptr(v_pool), kvd, float(k_scale), float(v_scale),
                                 _ptr(page_table), _ptr(seq_lens), _ptr(out), _ptr(lse), B, Sq, Hq, Hkv, D,
                                 page_size, page_table.shape[1], num_pages, _scale_arg(scale), int(num_splits),
                                 ws_ptr, ws_bytes, _stream(stream))
    _check(st, "gqa_decode_paged_ex")
    return out, lse


def gqa_decode_paged_engine(B, Sq, Hq, Hkv, D, kv_dtype=1, topk_form=False) -> str:
    """Kernel engine a paged call of this shape runs: "mma.sync" or "tcgen05"
    (topk_form: the sparse top-K form; else whole requests with kv_dtype 0
    bf16, 1 FP8, 2 int8)."""
    n = load_library().gqa_decode_paged_engine(B, Sq, Hq, Hkv, D, int(kv_dtype), 1 if topk_form else 0)
    if n < 0:
        raise GQAError(-n, "gqa_decode_paged_engine")
    return ENGINES[n]


def gqa_debug_set_paged_engine(mode: int):
    """mode 1: every later paged call runs on the mma.sync engine; 0: by shape."""
    load_library().gqa_debug_set_paged_engine(int(mode))


def gqa_decode_paged_num_splits(B, Sq, Hq, Hkv, D, kv_dtype, page_size, pages_per_req) -> int:
    return load_library().gqa_decode_paged_num_splits(B, Sq, Hq, Hkv, D, kv_dtype, page_size, pages_per_req)


def gqa_decode_paged_workspace_bytes(B, Sq, Hq, Hkv, D, kv_dtype, page_size, pages_per_req, num_splits=0) -> int:
    return load_library().gqa_decode_paged_workspace_bytes(B, Sq, Hq, Hkv, D, kv_dtype, page_size, pages_per_req,
                                                           num_splits)


def gqa_paged_gather_fp8(pool, page_table, topk_idx, out=None, stream=None):
    """Test hook: the paged kernel's index map as a byte copy -> uint8 [B, topk, Hkv, D]."""
    lib = load_library()
    _need(pool, "pool", torch.uint8, "cuda")
    _need(page_table, "page_table", torch.int32, "cuda")
    _need(topk_idx, "topk_idx", torch.int32, "cuda")
    num_pages, page_size, Hkv, D = pool.shape
    B, topk = topk_idx.shape
    if out is None:
        out = torch.empty((B, topk, Hkv, D), dtype=torch.uint8, device=pool.device)
    st = lib.gqa_paged_gather_fp8(_ptr(pool), _ptr(page_table), _ptr(topk_idx), _ptr(out), B, Hkv, D,
                                  page_size, page_table.shape[1], num_pages, topk, _stream(stream))
    _check(st, "gqa_paged_gather_fp8")
    return out


def gqa_fp8_e4m3fn_to_f32(codes, out=None, stream=None):
    """Test hook: the paged kernel's E4M3FN widening, as fp32."""
    lib = load_library()
    _need(codes, "codes", torch.uint8, "cuda")
    if out is None:
        out = torch.empty(codes.shape, dtype=torch.float32, device=codes.device)
    st = lib.gqa_fp8_e4m3fn_to_f32(_ptr(codes), _ptr(out), codes.numel(), _stream(stream))
    _check(st, "gqa_fp8_e4m3fn_to_f32")
    return out


# ---------------------------------------------------------------------------
# status and controls
# ---------------------------------------------------------------------------
def gqa_device_status(stream=None) -> int:
    """Waits for the stream; returns and clears the device error status code."""
    return int(load_library().gqa_device_status(_stream(stream)))


def gqa_set_wait_limit_ns(ns: int):
    load_library().gqa_set_wait_limit_ns(int(ns))


def gqa_debug_set_fault_mode(mode: int):
    load_library().gqa_debug_set_fault_mode(int(mode))


def gqa_debug_set_kernel_events(before=None, after=None):
    """Measurement hook: torch.cuda.Event pair recorded around the main kernel
    of later calls (None, None stops it)."""
    lib = load_library()
    if before is None or after is None:
        lib.gqa_debug_set_kernel_events(None, None)
    else:
        lib.gqa_debug_set_kernel_events(ctypes.c_void_p(before.cuda_event), ctypes.c_void_p(after.cuda_event))


def gqa_debug_read_stream(buf, sink, stream=None):
    """Measurement hook: reads every byte of the CUDA tensor `buf` once and
    XORs its words into `sink` (a CUDA int32 tensor of one element)."""
    lib = load_library()
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf: expected a contiguous CUDA tensor")
    _need(sink, "sink", torch.int32, "cuda")
    st = lib.gqa_debug_read_stream(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink), _stream(stream))
    _check(st, "gqa_debug_read_stream")


def gqa_status_string(status: int) -> str:
    return load_library().gqa_status_string(int(status)).decode()


def gqa_version() -> str:
    return load_library().gqa_version().decode()
