"""The allocation-free dense decode entry point, through the C ABI.

gqa_decode_noalloc serves callers that cannot allocate device memory while
they decode (a memory budget fixed at start-up, real-time loops, hosts that
hand the library only its inputs and outputs): it keeps the split partials in
a fixed scratch array inside the library.  These checks compare it with the
allocating entry point, twice in a row on different shapes (the scratch keeps
the previous call's contents), and check that a shape needing more scratch
than exists is refused.  This file is collected last so that a stop at its
first failure has already run every other test; it also passes on its own in
a fresh process.
"""
import pytest
import torch

import gqa_inputs
from parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    from gqa_decode_attention_gb300 import build as gbuild
    gbuild.build()
    import gqa_decode_attention_gb300 as m
    m.load_library()
    assert torch.cuda.is_available()
    return m


def _pair(gq, shape, seed, num_splits):
    B, Sq, Skv, Hq, Hkv, D = shape
    q, k, v = (t.cuda() for t in gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=seed))
    ref_o, ref_l = gq.gqa_decode_ex(q, k, v, num_splits=num_splits)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    gq.gqa_decode_noalloc(q, k, v, out, lse, num_splits=num_splits)
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    return out, lse, ref_o, ref_l


def test_noalloc_matches_allocating_entry_point_twice(gq):
    assert gq.gqa_decode_noalloc_scratch_bytes() == 32 << 20
    cases = [((1, 2, 8192, 64, 8, 128), 31, 0),    # automatic split count (many splits)
             ((2, 3, 3001, 16, 4, 64), 32, 7)]     # second call, other shape, leftover scratch
    for shape, seed, splits in cases:
        B, Sq, Skv, Hq, Hkv, D = shape
        assert gq.gqa_decode_workspace_bytes(B, Sq, Skv, Hq, Hkv, D, splits) > 0  # the scratch is used
        out, lse, ref_o, ref_l = _pair(gq, shape, seed, splits)
        assert_o_close(out.cpu(), ref_o.cpu().double(), f"noalloc {shape}")
        assert_lse_close(lse.cpu(), ref_l.cpu().double(), f"noalloc {shape}")


def test_noalloc_refuses_oversized_problem(gq):
    # 32 batch rows x 8 KV heads x 128 rows x 64 splits of fp32 partials >> 32 MiB
    B, Sq, Skv, Hq, Hkv, D = 32, 8, 8192, 128, 8, 128
    need = gq.gqa_decode_workspace_bytes(B, Sq, Skv, Hq, Hkv, D, 64)
    assert need > gq.gqa_decode_noalloc_scratch_bytes()
    q = torch.zeros((B, Sq, Hq, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, Skv, Hkv, D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(gq.GQAError) as ei:
        gq.gqa_decode_noalloc(q, k, k, out, None, num_splits=64)
    assert ei.value.status == 4
    assert gq.gqa_device_status() == 0
