"""fp64 CPU oracle for grouped-query decode attention -- TEST INFRASTRUCTURE.

This package checks the product and is not part of it.  Only the test suite, the
package's ``smoke()`` check and the benchmark's CPU-baseline leg may import
it; the CUDA library never does, and the two share no code.  The arithmetic
lives in ``gqa_oracle.c`` (plain C, double precision, OpenMP over rows); this
module only compiles it with gcc and marshals arrays through ctypes.

Inputs are passed as the exact stored bytes: bf16 tensors as their 16-bit
patterns, FP8 E4M3FN pools as their byte codes, indices as int32.  Outputs
are float64 numpy arrays.

Functions and the passages they restate (web pages on grouped-query decode
attention):

* ``kv_head`` -- "When the K/V copy costs more than the attention", section
  "What I was looking at": kv_head_idx = head_idx // (H_q // H_kv).
* ``gqa_decode`` -- the dense decode: softmax(scale * q K^T) V per query head,
  K/V read in place from the mapped KV head, bottom-right causal mask for
  S_q > 1 (a reading: the pages print no mask rule), natural-log LSE.
* ``e4m3fn_value`` -- "Sparse paged GQA decode attention with FP8 KV cache on
  SM89", section "Workload": the FP8 E4M3FN cache format, decoded from the
  OCP definition.
* ``paged_gather`` -- same page, section "Workload": page size, page table,
  top-K token indices; byte-exact gather of the selected K/V rows.
* ``gqa_decode_paged_fp8`` -- same page, sections "Workload" and
  "Implementations": attention over the selected tokens with k_scale in the
  scores, v_scale on the values, then a sigmoid gate.
* ``gqa_decode_dv`` -- the dense decode with a score head size (q, K) that
  differs from the value head size (V, O): the kv-copies page's d192x128
  flavour ("Limits, and what I'd do next").
* ``gqa_decode_paged`` -- the same page-table addressing without a top-K list:
  every token of each request up to its own sequence length, bf16, FP8 or
  int8 pools, the dense path's bottom-right mask per request (the serving layout
  both pages leave as an open question).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()

_dbl_p = ctypes.POINTER(ctypes.c_double)
_u16_p = ctypes.POINTER(ctypes.c_uint16)
_u8_p = ctypes.POINTER(ctypes.c_uint8)
_i32_p = ctypes.POINTER(ctypes.c_int32)


def build(out: str = _LIB, plant_bug: int = 0, force: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp) into a shared library.

    ``plant_bug`` > 0 compiles a deliberately wrong variant for the test
    suite's mutation self-check.
    """
    with _lock:
        if (not force and os.path.exists(out)
                and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
            return out
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               f"-DORACLE_PLANT_BUG={int(plant_bug)}", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
        return out


def _as_u16(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 bit patterns."""
    if hasattr(x, "dtype") and "torch" in type(x).__module__:
        import torch
        assert x.dtype == torch.bfloat16, x.dtype
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.ascontiguousarray(x)
    assert a.dtype == np.uint16, a.dtype
    return a


def _as_u8(x) -> np.ndarray:
    if hasattr(x, "dtype") and "torch" in type(x).__module__:
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        return np.ascontiguousarray(t.numpy())
    a = np.ascontiguousarray(x)
    if a.dtype == np.int8:
        a = a.view(np.uint8)
    assert a.dtype == np.uint8, a.dtype
    return a


def _as_i32(x) -> np.ndarray:
    if hasattr(x, "dtype") and "torch" in type(x).__module__:
        x = x.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(x)
    assert a.dtype == np.int32, a.dtype
    return a


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_e4m3fn_value.restype = ctypes.c_double
        lib.oracle_e4m3fn_value.argtypes = [ctypes.c_uint8]
        lib.oracle_kv_head.restype = ctypes.c_int
        lib.oracle_kv_head.argtypes = [ctypes.c_int] * 3
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.restype = None
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_gqa_decode.restype = None
        lib.oracle_gqa_decode.argtypes = [
            _u16_p, _u16_p, _u16_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, _i32_p, ctypes.c_int, _dbl_p, _dbl_p]
        lib.oracle_gqa_decode_dv.restype = None
        lib.oracle_gqa_decode_dv.argtypes = [
            _u16_p, _u16_p, _u16_p] + [ctypes.c_int] * 7 + [ctypes.c_double, _i32_p, ctypes.c_int, _dbl_p, _dbl_p]
        lib.oracle_paged_gather.restype = None
        lib.oracle_paged_gather.argtypes = [
            _u8_p, _i32_p, _i32_p] + [ctypes.c_int] * 6 + [_u8_p]
        lib.oracle_gqa_decode_paged_fp8.restype = None
        lib.oracle_gqa_decode_paged_fp8.argtypes = [
            _u16_p, _u16_p, _u8_p, _u8_p, _i32_p, _i32_p,
            ctypes.c_double, ctypes.c_double] + [ctypes.c_int] * 8 + [
            ctypes.c_double, _i32_p, ctypes.c_int, _dbl_p, _dbl_p, _dbl_p]
        lib.oracle_gqa_decode_paged.restype = None
        lib.oracle_gqa_decode_paged.argtypes = [
            _u16_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_double,
            _i32_p, _i32_p] + [ctypes.c_int] * 7 + [
            ctypes.c_double, _i32_p, ctypes.c_int, _dbl_p, _dbl_p]
        self._lib = lib

    # -- formats and mapping -------------------------------------------
    def e4m3fn_value(self, code: int) -> float:
        return self._lib.oracle_e4m3fn_value(int(code) & 0xFF)

    def kv_head(self, h: int, Hq: int, Hkv: int) -> int:
        return self._lib.oracle_kv_head(int(h), int(Hq), int(Hkv))

    def num_threads(self) -> int:
        return self._lib.oracle_num_threads()

    def set_num_threads(self, n: int) -> None:
        """Threads of later calls (timing only; results are identical)."""
        self._lib.oracle_set_num_threads(int(n))

    # -- dense ---------------------------------------------------------
    def gqa_decode(self, q, k, v, scale: float, rows=None):
        """Dense decode.  q [B,Sq,Hq,D], k/v [B,Skv,Hkv,D] (bf16).

        Returns (O, LSE).  Without ``rows``: O [B,Sq,Hq,D] float64 and
        LSE [B,Hq,Sq].  With ``rows`` (flattened ids (b*Hq + h)*Sq + i):
        O [n,D] and LSE [n] in the order given.
        """
        qa, ka, va = _as_u16(q), _as_u16(k), _as_u16(v)
        B, Sq, Hq, D = qa.shape
        _, Skv, Hkv, _ = ka.shape
        assert ka.shape == (B, Skv, Hkv, D) and va.shape == ka.shape
        if rows is None:
            n = B * Hq * Sq
            rp = None
        else:
            ra = _as_i32(np.asarray(rows, dtype=np.int32))
            n = ra.size
            rp = _p(ra, _i32_p)
        out = np.zeros((n, D), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        self._lib.oracle_gqa_decode(
            _p(qa, _u16_p), _p(ka, _u16_p), _p(va, _u16_p),
            B, Sq, Skv, Hq, Hkv, D, float(scale), rp, n, _p(out, _dbl_p), _p(lse, _dbl_p))
        if rows is not None:
            return out, lse
        o = out.reshape(B, Hq, Sq, D).transpose(0, 2, 1, 3).copy()
        return o, lse.reshape(B, Hq, Sq)

    def gqa_decode_dv(self, q, k, v, scale: float, rows=None):
        """Dense decode with Dqk != Dv.  q [B,Sq,Hq,Dqk], k [B,Skv,Hkv,Dqk],
        v [B,Skv,Hkv,Dv] (bf16).  Returns (O [B,Sq,Hq,Dv], LSE [B,Hq,Sq]) or,
        with ``rows``, (O [n,Dv], LSE [n])."""
        qa, ka, va = _as_u16(q), _as_u16(k), _as_u16(v)
        B, Sq, Hq, Dqk = qa.shape
        _, Skv, Hkv, _ = ka.shape
        Dv = va.shape[3]
        assert ka.shape == (B, Skv, Hkv, Dqk) and va.shape == (B, Skv, Hkv, Dv)
        if rows is None:
            n = B * Hq * Sq
            rp = None
        else:
            ra = _as_i32(np.asarray(rows, dtype=np.int32))
            n = ra.size
            rp = _p(ra, _i32_p)
        out = np.zeros((n, Dv), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        self._lib.oracle_gqa_decode_dv(
            _p(qa, _u16_p), _p(ka, _u16_p), _p(va, _u16_p),
            B, Sq, Skv, Hq, Hkv, Dqk, Dv, float(scale), rp, n, _p(out, _dbl_p), _p(lse, _dbl_p))
        if rows is not None:
            return out, lse
        o = out.reshape(B, Hq, Sq, Dv).transpose(0, 2, 1, 3).copy()
        return o, lse.reshape(B, Hq, Sq)

    # -- paged FP8 -----------------------------------------------------
    def paged_gather(self, pool, page_table, topk, page_size: int):
        """Byte-exact gather: returns uint8 [B, topk, Hkv, D]."""
        pa, pt, tk = _as_u8(pool), _as_i32(page_table), _as_i32(topk)
        _, ps, Hkv, D = pa.shape
        assert ps == page_size
        B, ppr = pt.shape
        topk_n = tk.shape[1]
        out = np.zeros((B, topk_n, Hkv, D), dtype=np.uint8)
        self._lib.oracle_paged_gather(_p(pa, _u8_p), _p(pt, _i32_p), _p(tk, _i32_p),
                                      B, Hkv, D, ps, ppr, topk_n, _p(out, _u8_p))
        return out

    def gqa_decode_paged_fp8(self, q, gate, k_pool, v_pool, page_table, topk,
                             k_scale: float, v_scale: float, scale: float, rows=None):
        """Sparse paged FP8 decode with sigmoid gate.

        q, gate [B,Hq,D] bf16; pools [num_pages, ps, Hkv, D] E4M3FN codes;
        page_table [B, ppr] int32; topk [B, K] int32.
        Returns (out, lse, attn): out/attn [B,Hq,D] (or [n,D] with ``rows`` =
        flattened b*Hq + h ids), lse [B,Hq] (or [n]).
        """
        qa, ga = _as_u16(q), _as_u16(gate)
        ka, va = _as_u8(k_pool), _as_u8(v_pool)
        pt, tk = _as_i32(page_table), _as_i32(topk)
        B, Hq, D = qa.shape
        num_pages, ps, Hkv, D2 = ka.shape
        assert D2 == D and va.shape == ka.shape and ga.shape == qa.shape
        ppr = pt.shape[1]
        topk_n = tk.shape[1]
        if rows is None:
            n = B * Hq
            rp = None
        else:
            ra = _as_i32(np.asarray(rows, dtype=np.int32))
            n = ra.size
            rp = _p(ra, _i32_p)
        out = np.zeros((n, D), dtype=np.float64)
        attn = np.zeros((n, D), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        self._lib.oracle_gqa_decode_paged_fp8(
            _p(qa, _u16_p), _p(ga, _u16_p), _p(ka, _u8_p), _p(va, _u8_p),
            _p(pt, _i32_p), _p(tk, _i32_p), float(k_scale), float(v_scale),
            B, Hq, Hkv, D, ps, ppr, num_pages, topk_n, float(scale), rp, n,
            _p(out, _dbl_p), _p(lse, _dbl_p), _p(attn, _dbl_p))
        if rows is not None:
            return out, lse, attn
        return out.reshape(B, Hq, D), lse.reshape(B, Hq), attn.reshape(B, Hq, D)

    # -- paged, whole requests -------------------------------------------
    def gqa_decode_paged(self, q, k_pool, v_pool, page_table, seq_lens, scale: float,
                         k_scale: float = 1.0, v_scale: float = 1.0, rows=None, kv_type=None):
        """Paged decode over every token of each request (no top-K).

        q [B,Sq,Hq,D] bf16; pools [num_pages, ps, Hkv, D] of bf16, E4M3FN codes
        (uint8 / float8 tensors) or int8 codes (int8 tensors); kv_type 0/1/2
        overrides the inference from the pool dtype; page_table [B, ppr] int32;
        seq_lens [B] int32.  Returns (O, LSE): O [B,Sq,Hq,D] and LSE [B,Hq,Sq] float64, or
        with ``rows`` (flattened ids (b*Hq + h)*Sq + i) O [n,D] and LSE [n].
        """
        qa = _as_u16(q)
        dt = str(k_pool.dtype) if hasattr(k_pool, "dtype") else ""
        if kv_type is None:
            kv_type = 0 if dt in ("torch.bfloat16", "uint16") else 2 if dt in ("torch.int8", "int8") else 1
        if kv_type == 0:
            ka, va = _as_u16(k_pool), _as_u16(v_pool)
        else:
            ka, va = _as_u8(k_pool), _as_u8(v_pool)
        pt, sl = _as_i32(page_table), _as_i32(seq_lens)
        B, Sq, Hq, D = qa.shape
        _, ps, Hkv, D2 = ka.shape
        assert D2 == D and va.shape == ka.shape and sl.shape == (B,)
        ppr = pt.shape[1]
        assert int(sl.min(initial=0)) >= 0 and int(sl.max(initial=0)) <= ppr * ps
        if rows is None:
            n = B * Hq * Sq
            rp = None
        else:
            ra = _as_i32(np.asarray(rows, dtype=np.int32))
            n = ra.size
            rp = _p(ra, _i32_p)
        out = np.zeros((n, D), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        self._lib.oracle_gqa_decode_paged(
            _p(qa, _u16_p), ka.ctypes.data_as(ctypes.c_void_p), va.ctypes.data_as(ctypes.c_void_p),
            int(kv_type), float(k_scale), float(v_scale), _p(pt, _i32_p), _p(sl, _i32_p),
            B, Sq, Hq, Hkv, D, ps, ppr, float(scale), rp, n, _p(out, _dbl_p), _p(lse, _dbl_p))
        if rows is not None:
            return out, lse
        o = out.reshape(B, Hq, Sq, D).transpose(0, 2, 1, 3).copy()
        return o, lse.reshape(B, Hq, Sq)


_default: Oracle | None = None


def load(path: str | None = None) -> Oracle:
    """Load (building first if needed) the oracle library."""
    global _default
    if path is not None:
        return Oracle(path)
    if _default is None:
        _default = Oracle(build())
    return _default
