"""C ABI boundary checks that need no GPU: the library loads, exports every
symbol its headers declare, and rejects bad arguments with the documented
status before touching the device."""
import ctypes
import glob
import os
import re

import pytest

import gqa_decode_attention_gb300 as gq
from gqa_decode_attention_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gq.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(gqa_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_something():
    names = _declared_functions()
    assert "gqa_decode" in names and "gqa_decode_paged_fp8" in names


def test_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert sorted(gq.EXPORTS) == _declared_functions()


def test_status_strings(lib):
    for code, name in gq.STATUS.items():
        assert gq.gqa_status_string(code) == name
    assert "sm_103a" in gq.gqa_version()


# Fake, never-dereferenced device addresses: validation must reject the call
# before any CUDA work happens.
A = 0x7F0000000000  # 16-byte aligned
MIS = A + 2         # misaligned


def _device_visible() -> bool:
    """A call with valid arguments would launch a kernel on the fake addresses
    above; such calls are made only where no CUDA device is visible (they then
    fail in the runtime with GQA_ERR_CUDA and touch no device)."""
    import torch
    return torch.cuda.is_available()


def _dense(lib, q=A, k=A, v=A, out=A, lse=A, B=1, Sq=1, Skv=64, Hq=8, Hkv=2, D=128):
    return lib.gqa_decode(q, k, v, out, lse, B, Sq, Skv, Hq, Hkv, D, 0.0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), 1),          # Hq % Hkv != 0
    (dict(Sq=3, Skv=2), 1),          # Sq > Skv
    (dict(B=0), 1),
    (dict(Sq=0), 1),
    (dict(Skv=0), 1),
    (dict(Hkv=0), 1),
    (dict(D=96), 2),                 # unsupported head dim
    (dict(D=512), 2),
    (dict(Hq=4096 * 2, Hkv=1, Sq=1), 2),  # group rows beyond the limit
    (dict(q=0), 1),                  # null pointers
    (dict(k=0), 1),
    (dict(out=0), 1),
    (dict(q=MIS), 3),                # alignment
    (dict(k=MIS), 3),
    (dict(v=MIS), 3),
    (dict(out=MIS), 3),
    (dict(lse=A + 1), 3),
])
def test_dense_rejects(lib, kw, status):
    assert _dense(lib, **kw) == status


def test_dense_ex_rejects(lib):
    assert lib.gqa_decode_ex(A, A, A, A, A, 1, 1, 64, 8, 2, 128, 0.0, -1, None, 0, None) == 1
    assert lib.gqa_decode_workspace_bytes(1, 1, 64, 6, 4, 128, 0) == 0
    assert lib.gqa_decode_num_splits(1, 1, 64, 6, 4, 128) == -1
    assert lib.gqa_decode_num_splits(1, 1, 64, 8, 2, 96) == -2


def test_dense_engine_choice(lib):
    """Host-only: d256 always on tcgen05, d128 on tcgen05 from 8 decode rows
    per head, the rest on mma.sync; the group size never changes the engine."""
    eng = lib.gqa_decode_dense_engine
    for Hq, Hkv in [(8, 8), (64, 8), (64, 1)]:
        assert eng(1, 1, 100, Hq, Hkv, 256, 256) == 1
        assert eng(1, 7, 100, Hq, Hkv, 128, 128) == 0
        assert eng(1, 8, 100, Hq, Hkv, 128, 128) == 1
        assert eng(1, 64, 100, Hq, 1, 128, 128) == 1
        assert eng(1, 8, 100, Hq, Hkv, 64, 64) == 0
        assert eng(1, 8, 100, Hq, Hkv, 192, 128) == 0
    assert eng(1, 2, 1, 8, 2, 128, 128) == -1     # Sq > Skv
    assert eng(1, 8, 100, 8, 2, 96, 96) == -2     # unsupported head size
    assert eng(1, 8, 100, 8, 2, 128, 192) == -2


def test_paged_engine_choice(lib):
    """Host-only: FP8 pools of head dim 128 with KV heads in blocks of 8 and at
    most 4 query rows per KV head run on tcgen05 (both forms); every other
    paged shape on mma.sync; the measurement hook forces mma.sync."""
    eng = lib.gqa_decode_paged_engine
    # whole requests: (B, Sq, Hq, Hkv, D, kv_dtype, topk_form)
    assert eng(4, 1, 32, 8, 128, 1, 0) == 1         # FP8, 4 rows per KV head
    assert eng(4, 2, 16, 8, 128, 1, 0) == 1         # 2 x 2 rows
    assert eng(4, 1, 64, 16, 128, 1, 0) == 1        # two blocks of 8 KV heads
    assert eng(4, 1, 8, 8, 128, 1, 0) == 1          # one row per KV head
    assert eng(4, 1, 64, 8, 128, 1, 0) == 0         # 8 rows per KV head
    assert eng(4, 2, 64, 8, 128, 1, 0) == 0         # 16 rows per KV head
    assert eng(4, 1, 32, 4, 128, 1, 0) == 0         # 4 KV heads
    assert eng(4, 1, 96, 12, 128, 1, 0) == 0        # 12 KV heads
    assert eng(4, 1, 64, 8, 64, 1, 0) == 0          # head dim 64
    assert eng(4, 1, 64, 8, 128, 0, 0) == 0         # bf16 pool
    assert eng(4, 1, 64, 8, 128, 2, 0) == 0         # int8 pool
    # top-K form (FP8, Sq = 1; kv_dtype ignored)
    assert eng(256, 1, 32, 8, 128, 0, 1) == 1
    assert eng(256, 1, 32, 4, 128, 0, 1) == 0
    assert eng(256, 1, 64, 8, 128, 0, 1) == 0       # 8 rows per KV head
    assert eng(4, 1, 6, 4, 128, 1, 0) == -1         # Hq % Hkv != 0
    assert eng(4, 1, 64, 8, 96, 1, 0) == -2         # unsupported head size
    lib.gqa_debug_set_paged_engine(1)
    try:
        assert eng(4, 1, 32, 8, 128, 1, 0) == 0
        assert eng(256, 1, 32, 8, 128, 0, 1) == 0
    finally:
        lib.gqa_debug_set_paged_engine(0)
    assert eng(4, 1, 32, 8, 128, 1, 0) == 1


def test_engine_names_match_header():
    """The binding's engine names follow the header's GQA_ENGINE_* values."""
    text = open(os.path.join(ROOT, "include", "gqa_decode.h")).read()
    vals = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define GQA_ENGINE_(\w+) (\d+)", text)}
    assert vals == {"MMA_SYNC": 0, "TCGEN05": 1}
    assert gq.ENGINES == {vals["MMA_SYNC"]: "mma.sync", vals["TCGEN05"]: "tcgen05"}


def test_dense_dv_rejects(lib):
    def dv(Dqk=192, Dv=128, splits=0, B=1, Sq=1, Skv=64, Hq=8, Hkv=2, q=A, v=A, ws_bytes=0):
        return lib.gqa_decode_dv(q, A, v, A, A, B, Sq, Skv, Hq, Hkv, Dqk, Dv, 0.0, splits, None, ws_bytes, None)
    assert dv(Dqk=128, Dv=192) == 2      # only (192, 128) and equal sizes
    assert dv(Dqk=192, Dv=192) == 2
    assert dv(Dqk=192, Dv=64) == 2
    assert dv(Dqk=96, Dv=96) == 2
    assert dv(Hq=6, Hkv=4) == 1
    assert dv(Sq=3, Skv=2) == 1
    assert dv(splits=-1) == 1
    assert dv(q=0) == 1
    assert dv(v=MIS) == 3
    assert lib.gqa_decode_dv_workspace_bytes(1, 1, 64, 8, 2, 128, 192, 0) == 0
    # explicit split count needs no device: 2 splits of the 2 blocks of 64 keys,
    # rows = B * Hkv * splits * (G * Sq), fp32 partials of Dv dims plus one LSE each
    rows = 1 * 2 * 2 * 4
    want = ((rows * 128 * 4 + 255) // 256) * 256 + ((rows * 4 + 255) // 256) * 256
    assert lib.gqa_decode_dv_workspace_bytes(1, 1, 128, 8, 2, 192, 128, 2) == want
    assert lib.gqa_decode_dv_workspace_bytes(1, 1, 128, 8, 2, 192, 128, 1) == 0
    # equal sizes report what the dense entry point reports
    assert (lib.gqa_decode_dv_workspace_bytes(1, 1, 300, 8, 2, 128, 128, 3)
            == lib.gqa_decode_workspace_bytes(1, 1, 300, 8, 2, 128, 3))


def _paged(lib, q=A, gate=A, kp=A, vp=A, pt=A, tk=A, ks=1.0, vs=1.0, out=A, lse=A, B=2, Hq=8, Hkv=2, D=128,
           ps=16, ppr=4, num_pages=16, topk=32):
    return lib.gqa_decode_paged_fp8(q, gate, kp, vp, pt, tk, ks, vs, out, lse, B, Hq, Hkv, D, ps, ppr,
                                    num_pages, topk, 0.0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), 1),
    (dict(topk=65), 1),              # more entries than the request has tokens
    (dict(topk=-1), 1),
    (dict(ps=0), 1),
    (dict(num_pages=0), 1),
    (dict(D=96), 2),
    (dict(D=256), 2),                # not built for the paged path
    (dict(Hq=64, Hkv=2), 2),         # group of 32 > 16
    (dict(ks=float("inf")), 1),
    (dict(vs=float("nan")), 1),
    (dict(q=0), 1),
    (dict(gate=0), 1),
    (dict(tk=0), 1),
    (dict(kp=MIS), 3),
    (dict(gate=MIS), 3),
    (dict(pt=A + 2), 3),
])
def test_paged_rejects(lib, kw, status):
    assert _paged(lib, **kw) == status


def _paged_kv(lib, q=A, kp=A, vp=A, kvd=0, ks=1.0, vs=1.0, pt=A, sl=A, out=A, lse=A, B=2, Sq=1, Hq=8, Hkv=2,
              D=128, ps=16, ppr=4, num_pages=16, splits=0, ws=None, ws_bytes=0):
    return lib.gqa_decode_paged_ex(q, kp, vp, kvd, ks, vs, pt, sl, out, lse, B, Sq, Hq, Hkv, D, ps, ppr,
                                   num_pages, 0.0, splits, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), 1),
    (dict(Sq=0), 1),
    (dict(ps=0), 1),
    (dict(ppr=0), 1),
    (dict(num_pages=0), 1),
    (dict(kvd=3), 1),                # unknown pool type
    (dict(kvd=2, vs=float("inf")), 1),  # int8 pools need finite scales
    (dict(splits=-1), 1),
    (dict(D=96), 2),
    (dict(D=256), 2),
    (dict(Hq=64, Hkv=2), 2),         # group of 32 rows > 16
    (dict(Hq=16, Hkv=2, Sq=3), 2),   # 8 heads x 3 decode rows > 16
    (dict(kvd=1, ks=float("inf")), 1),
    (dict(kvd=1, vs=float("nan")), 1),
    (dict(kvd=0, ks=float("inf")), None),  # scales ignored for bf16 pools: not an argument error
    (dict(q=0), 1),
    (dict(sl=0), 1),
    (dict(pt=0), 1),
    (dict(kp=MIS), 3),
    (dict(out=MIS), 3),
    (dict(sl=A + 2), 3),
    (dict(lse=A + 2), 3),
])
def test_paged_kv_rejects(lib, kw, status):
    if status is None:
        if _device_visible():
            pytest.skip("valid arguments: would launch on fake device addresses")
        assert _paged_kv(lib, **kw) not in (1, 2, 3)
    else:
        assert _paged_kv(lib, **kw) == status


def test_paged_dev_scales_rejects(lib):
    def call(kvd=1, ks=A, vs=A, n=1, Hkv=2):
        return lib.gqa_decode_paged_dev_scales(A, A, A, kvd, ks, vs, n, A, A, A, A, 2, 1, 8, Hkv, 128, 16, 4, 16,
                                               0.0, 0, None, 0, None)
    assert call(kvd=0) == 1          # bf16 pools take no scales
    assert call(ks=None) == 1
    assert call(n=3) == 1            # neither per tensor nor per head
    assert call(ks=MIS) == 3
    if not _device_visible():
        assert call(n=2) not in (1, 2, 3)  # per head: valid arguments


def test_paged_kv_sizes(lib):
    # automatic split count and workspace reject bad shapes with a negative status / zero
    assert lib.gqa_decode_paged_num_splits(2, 1, 8, 2, 96, 0, 16, 4) == -2
    assert lib.gqa_decode_paged_num_splits(2, 1, 6, 4, 128, 0, 16, 4) == -1
    assert lib.gqa_decode_paged_workspace_bytes(2, 1, 8, 2, 96, 0, 16, 4, 3) == 0
    # explicit worker counts need no device: 1 head block of 2 heads x 3 workers x
    # 2 partial slots x 4 rows
    rows = 1 * 3 * 2 * 2 * 4
    want = ((rows * 128 * 4 + 255) // 256) * 256 + ((rows * 4 + 255) // 256) * 256 + 256  # + step prefix of 3 longs
    assert lib.gqa_decode_paged_workspace_bytes(2, 1, 8, 2, 128, 0, 16, 64, 3) == want
    assert lib.gqa_decode_paged_workspace_bytes(2, 1, 8, 2, 128, 0, 16, 64, 1) == 0


def test_paged_fp8_dev_scales_rejects(lib):
    def call(ks=A, vs=A, n=1, Hkv=2):
        return lib.gqa_decode_paged_fp8_dev_scales(A, A, A, A, A, A, ks, vs, n, A, A, 2, 8, Hkv, 128, 16, 4, 16, 32,
                                                   0.0, None)
    assert call(ks=None) == 1
    assert call(vs=None) == 1
    assert call(n=3) == 1            # neither per tensor nor per head
    assert call(n=0) == 1
    assert call(ks=MIS) == 3
    assert call(vs=A + 1) == 3


def test_gather_and_convert_reject(lib):
    assert lib.gqa_paged_gather_fp8(A, A, A, A, 2, 2, 128, 16, 4, 16, 65, None) == 1
    assert lib.gqa_paged_gather_fp8(MIS, A, A, A, 2, 2, 128, 16, 4, 16, 32, None) == 3
    assert lib.gqa_fp8_e4m3fn_to_f32(A, A, -1, None) == 1
    assert lib.gqa_fp8_e4m3fn_to_f32(A, A + 2, 4, None) == 3
    assert lib.gqa_fp8_e4m3fn_to_f32(None, None, 0, None) == 0  # nothing to do


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("gqa_decode_attention_gb300")
    saved = mod._lib_handle
    mod._lib_handle = None
    try:
        with pytest.raises(ImportError):
            mod.load_library(str(tmp_path / "missing.so"))
    finally:
        mod._lib_handle = saved
