"""GPU parity of the paged decode's tcgen05 engine (FP8 pools, head dim 128,
KV heads in blocks of 8, up to 4 query rows per KV head), both forms, through
the C ABI, against the fp64 oracle on the same stored codes and scales; and
against the mma.sync engine on the same inputs."""
import math

import numpy as np
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


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _topk(gq, inp):
    d = _cuda(inp)
    out, lse = gq.gqa_decode_paged_fp8(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["page_table"], d["topk"],
                                       d["k_scale"], d["v_scale"])
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def _whole(gq, inp, **kw):
    d = _cuda(inp)
    out, lse = gq.gqa_decode_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"],
                                   d["k_scale"], d["v_scale"], **kw)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def _check_rows(out, lse, ref_o, ref_l, what):
    """Rows with no visible token: exactly zero output and -inf LSE; the rest
    within the tolerances.  out [B, Sq, Hq, D] (or [B, Hq, D]), lse [B, Hq, Sq]
    (or [B, Hq])."""
    if out.dim() == 3:
        out, lse = out.unsqueeze(1), lse.unsqueeze(-1)
        ref_o, ref_l = ref_o[:, None], ref_l[..., None]
    empty = np.isneginf(ref_l)
    if empty.any():
        e = torch.from_numpy(empty)
        assert torch.all(torch.isneginf(lse[e])), what
        assert torch.all(out.float().permute(0, 2, 1, 3)[e] == 0), what
    ok = ~empty
    o_ok = torch.from_numpy(ok).permute(0, 2, 1)
    assert_o_close(out[o_ok], ref_o[o_ok.numpy()], what)
    assert_lse_close(lse[torch.from_numpy(ok)], ref_l[ok], what)


# (B, Hq, Hkv, page_size, pages_per_req, topk, pad_tail)
TOPK = [
    (3, 32, 8, 16, 32, 512, 0),     # the benchmark's shape, 4 rows per KV head
    (2, 8, 8, 16, 8, 100, 5),       # one row per KV head, ragged list with padding
    (2, 16, 8, 1, 70, 67, 0),       # page size 1
    (4, 24, 8, 64, 3, 150, 9),      # 3 rows per KV head (one padding row of 4), page size 64
    (2, 32, 8, 16, 12, 190, 0),     # 4 rows per KV head, ragged last block
    (1, 24, 8, 16, 20, 300, 1),     # 3 rows per KV head, padding entry
    (2, 64, 16, 16, 8, 128, 0),     # two blocks of 8 KV heads
    (5, 32, 8, 16, 4, 1, 0),        # a single selected token
    (2, 32, 8, 16, 8, 128, 128),    # every entry padding: O = 0, LSE = -inf
    (1, 32, 8, 16, 200, 3000, 11),  # a long list (many blocks, lazy rescales)
]


@pytest.mark.parametrize("shape", TOPK, ids=lambda s: "b{}_h{}x{}_ps{}_ppr{}_k{}_pad{}".format(*s))
def test_topk_vs_oracle(gq, orc, shape):
    B, Hq, Hkv, ps, ppr, topk, pad = shape
    assert gq.gqa_decode_paged_engine(B, 1, Hq, Hkv, 128, 1, topk_form=True) == "tcgen05"
    inp = gqa_inputs.paged_inputs(B, Hq, Hkv, 128, ps, ppr, B * ppr + 3, topk, seed=sum(shape) + 7, pad_tail=pad)
    out, lse = _topk(gq, inp)
    assert gq.gqa_device_status() == 0
    ref_o, ref_l, _ = orc.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"],
                                               inp["page_table"], inp["topk"], inp["k_scale"], inp["v_scale"],
                                               1.0 / math.sqrt(128))
    _check_rows(out, lse, ref_o, ref_l, f"topk {shape}")


# (B, Sq, Hq, Hkv, page_size, pages_per_req, seq_lens)
WHOLE = [
    (3, 1, 32, 8, 16, 8, (128, 100, 17)),
    (2, 2, 16, 8, 1, 90, (90, 33)),          # 4 rows per KV head with the causal mask, page size 1
    (2, 4, 8, 8, 64, 3, (192, 5)),           # 4 decode rows, a request of 5 tokens
    (3, 3, 8, 8, 16, 6, (96, 2, 0)),         # 3 rows (instance of 4); shorter than Sq; empty
    (1, 1, 32, 8, 16, 300, (4800,)),         # long request, 4 rows per KV head
    (2, 1, 8, 8, 32, 4, (111, 64)),          # one row per KV head
    (1, 2, 32, 16, 16, 40, (600,)),          # two blocks of 8 KV heads, 4 rows each
]


@pytest.mark.parametrize("shape", WHOLE, ids=lambda s: "b{}_sq{}_h{}x{}_ps{}_ppr{}".format(*s[:6]))
@pytest.mark.parametrize("splits", [0, 1, 5, 37])
def test_whole_request_vs_oracle(gq, orc, shape, splits):
    B, Sq, Hq, Hkv, ps, ppr, lens = shape
    assert gq.gqa_decode_paged_engine(B, Sq, Hq, Hkv, 128, 1) == "tcgen05"
    inp = gqa_inputs.paged_kv_inputs(B, Sq, Hq, Hkv, 128, ps, ppr, B * ppr + 2, seed=sum(lens) + ps + Sq,
                                     kv_dtype="fp8", seq_lens=list(lens))
    out, lse = _whole(gq, inp, num_splits=splits)
    assert gq.gqa_device_status() == 0
    ref_o, ref_l = orc.gqa_decode_paged(inp["q"], inp["k_pool"], inp["v_pool"], inp["page_table"],
                                        inp["seq_lens"], 1.0 / math.sqrt(128), inp["k_scale"], inp["v_scale"])
    _check_rows(out, lse, ref_o, ref_l, f"whole {shape} splits={splits}")


def test_eight_rows_per_head_run_on_mma_sync(gq):
    """Shapes with 5-8 query rows per KV head stay on the mma.sync engine."""
    assert gq.gqa_decode_paged_engine(4, 1, 64, 8, 128, 1) == "mma.sync"
    assert gq.gqa_decode_paged_engine(4, 2, 32, 8, 128, 1) == "mma.sync"
    assert gq.gqa_decode_paged_engine(256, 1, 64, 8, 128, 1, topk_form=True) == "mma.sync"
    assert gq.gqa_decode_paged_engine(4, 1, 32, 8, 128, 1) == "tcgen05"


def test_engines_agree_and_repeat_bitwise(gq):
    """The tcgen05 and mma.sync engines give the same results within rounding
    on the same inputs; a tcgen05 call repeated is bit for bit the same."""
    inp = gqa_inputs.paged_inputs(4, 32, 8, 128, 16, 16, 70, 250, seed=91, pad_tail=3)
    a1, l1 = _topk(gq, inp)
    a2, l2 = _topk(gq, inp)
    assert torch.equal(a1, a2) and torch.equal(l1, l2)
    gq.gqa_debug_set_paged_engine(1)
    try:
        assert gq.gqa_decode_paged_engine(4, 1, 32, 8, 128, 1, topk_form=True) == "mma.sync"
        b1, m1 = _topk(gq, inp)
    finally:
        gq.gqa_debug_set_paged_engine(0)
    assert torch.allclose(a1.float(), b1.float(), atol=1e-2, rtol=1e-2)
    assert torch.allclose(l1, m1, atol=1e-3, rtol=0)
    w = gqa_inputs.paged_kv_inputs(3, 2, 16, 8, 128, 16, 20, 70, seed=92, kv_dtype="fp8", seq_lens=[300, 17, 2])
    c1, n1 = _whole(gq, w, num_splits=5)
    gq.gqa_debug_set_paged_engine(1)
    try:
        c2, n2 = _whole(gq, w, num_splits=5)
    finally:
        gq.gqa_debug_set_paged_engine(0)
    fin = torch.isfinite(n1)
    assert torch.equal(fin, torch.isfinite(n2))
    assert torch.allclose(c1.float(), c2.float(), atol=1e-2, rtol=1e-2)
    assert torch.allclose(n1[fin], n2[fin], atol=1e-3, rtol=0)
    assert gq.gqa_device_status() == 0


def test_device_scales_per_head_topk(gq, orc):
    """Per-KV-head device scales on the tcgen05 top-K path: the oracle runs once
    per KV head with that head's scalars."""
    B, Hq, Hkv = 2, 32, 8
    inp = gqa_inputs.paged_inputs(B, Hq, Hkv, 128, 16, 8, B * 8 + 1, 100, seed=93)
    ks = torch.tensor([0.5 + 0.1 * e for e in range(Hkv)], dtype=torch.float32)
    vs = torch.tensor([1.5 - 0.1 * e for e in range(Hkv)], dtype=torch.float32)
    d = _cuda(inp)
    out, lse = gq.gqa_decode_paged_fp8(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["page_table"], d["topk"],
                                       k_scales=ks.cuda(), v_scales=vs.cuda())
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    G = Hq // Hkv
    for g in range(Hkv):
        ref_o, ref_l, _ = orc.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"],
                                                   inp["page_table"], inp["topk"], float(ks[g]), float(vs[g]),
                                                   1.0 / math.sqrt(128))
        hs = slice(g * G, (g + 1) * G)
        assert_o_close(out[:, hs].cpu(), ref_o[:, hs], f"head {g}")
        assert_lse_close(lse[:, hs].cpu(), ref_l[:, hs], f"head {g}")


def test_wait_timeout_whole_request(gq):
    """Forced wait timeout on the tcgen05 whole-request path: flagged, not hung,
    and the next call works."""
    inp = gqa_inputs.paged_kv_inputs(2, 1, 32, 8, 128, 16, 8, 17, seed=94, kv_dtype="fp8")
    d = _cuda(inp)
    gq.gqa_set_wait_limit_ns(50_000_000)
    gq.gqa_debug_set_fault_mode(1)
    try:
        gq.gqa_decode_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"], d["k_scale"],
                            d["v_scale"], num_splits=3)
        assert gq.gqa_device_status() == 6
    finally:
        gq.gqa_debug_set_fault_mode(0)
        gq.gqa_set_wait_limit_ns(0)
    out, lse = _whole(gq, inp)
    assert gq.gqa_device_status() == 0
    assert torch.isfinite(lse).all()
