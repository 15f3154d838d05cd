"""The allocation-free dense decode entry point, through the C ABI.

gqa_decode_noalloc serves callers that cannot allocate device memory while
they decode (a memory budget fixed at start-up, real-time loops, hosts that
hand the library only its inputs and outputs): it keeps the split partials in
a fixed scratch array inside the library.  Each case below is checked against
the fp64 oracle at the method's tolerances, and bit for bit against the
allocating entry point given the same split argument (0 = the automatic plan;
the same kernels run, only the partials live elsewhere).  The cases run back to back on different
shapes, so every call after the first starts on the previous call's leftover
scratch; they cover both kernel engines (mma.sync and tcgen05).  A shape
needing more scratch than exists is refused.  This file is collected last so
that a stop at its first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import math

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


# (B, Sq, Skv, Hq, Hkv, D), seed, split count (0 = automatic)
CASES = [
    ((1, 2, 8192, 64, 8, 128), 31, 0),    # mma.sync engine, automatic split count (many splits)
    ((2, 3, 3001, 16, 4, 64), 32, 7),     # other shape on leftover scratch, ragged last split
    ((1, 8, 4096, 32, 4, 128), 33, 4),    # tcgen05 engine (d 128, 8 decode rows), 4 splits
    ((1, 2, 2500, 16, 2, 256), 34, 3),    # tcgen05 engine (d 256), 3 splits
]


def test_noalloc_matches_oracle_and_allocating_entry_point(gq, orc):
    assert gq.gqa_decode_noalloc_scratch_bytes() == 32 << 20
    engines = set()
    for shape, seed, splits in CASES:
        B, Sq, Skv, Hq, Hkv, D = shape
        assert gq.gqa_decode_workspace_bytes(B, Sq, Skv, Hq, Hkv, D, splits) > 0  # the scratch is used
        engines.add(gq.gqa_decode_dense_engine(B, Sq, Skv, Hq, Hkv, D))
        qc, kc, vc = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=seed)
        q, k, v = qc.cuda(), kc.cuda(), vc.cuda()
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
        gq.gqa_decode_noalloc(q, k, v, out, lse, num_splits=splits)
        torch.cuda.synchronize()
        assert gq.gqa_device_status() == 0
        ref_o, ref_l = orc.gqa_decode(qc, kc, vc, 1.0 / math.sqrt(D))
        assert_o_close(out.cpu(), ref_o, f"noalloc O {shape} vs oracle")
        assert_lse_close(lse.cpu(), ref_l, f"noalloc LSE {shape} vs oracle")
        ex_o, ex_l = gq.gqa_decode_ex(q, k, v, num_splits=splits)
        torch.cuda.synchronize()
        assert gq.gqa_device_status() == 0
        assert torch.equal(out, ex_o), f"noalloc O {shape} differs from gqa_decode_ex"
        assert torch.equal(lse, ex_l), f"noalloc LSE {shape} differs from gqa_decode_ex"
    assert engines == {"mma.sync", "tcgen05"}


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
