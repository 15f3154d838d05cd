"""GPU parity at the largest sizes the C ABI accepts: the biggest group of
query rows per KV head, the largest batch, a cache long enough to push the
split count to its cap, the longest top-K list and a very long paged request.
Each is checked against the fp64 oracle (all rows, or sampled rows where the
oracle would take long)."""
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


def _dense(gq, q, k, v, num_splits=0):
    out, lse = gq.gqa_decode_ex(q, k, v, num_splits=num_splits)
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("D", [64, 128, 256])
def test_largest_query_group(gq, orc, D):
    """d 64 (mma.sync engine) and d 128 (tcgen05 engine, Sq 8): 4096 query rows
    per KV head (512 heads over 1, 8 decode rows), 32 row groups of 128; d 256
    (tcgen05 engine): 512 rows, 4 row groups."""
    Hq = 64 if D == 256 else 512
    Sq = 8
    q, k, v = gqa_inputs.dense_inputs(1, Sq, 300, Hq, 1, D, seed=500 + D, device="cuda")
    out, lse = _dense(gq, q, k, v)
    ref_o, ref_l = orc.gqa_decode(q.cpu(), k.cpu(), v.cpu(), 1.0 / math.sqrt(D))
    assert_o_close(out, ref_o, f"{Hq * Sq} group rows, d{D}")
    assert_lse_close(lse, ref_l)


def test_largest_batch(gq, orc):
    """B = 65535 (the grid limit), each request a 3-key cache."""
    B = 65535
    q, k, v = gqa_inputs.dense_inputs(B, 1, 3, 2, 1, 64, seed=501, device="cuda")
    out, lse = _dense(gq, q, k, v)
    ref_o, ref_l = orc.gqa_decode(q.cpu(), k.cpu(), v.cpu(), 1.0 / 8.0)
    assert_o_close(out, ref_o, "B = 65535")
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("splits", [0, 4096])
def test_two_million_keys(gq, orc, splits):
    """A 2M-key cache (one KV head, 8 query heads): the automatic split count,
    and the maximum of 4096 splits, whose combine reads most partial rows past
    the part it stages in shared memory."""
    Skv = 1 << 21
    q, k, v = gqa_inputs.dense_inputs(1, 1, Skv, 8, 1, 64, seed=502, device="cuda")
    out, lse = _dense(gq, q, k, v, num_splits=splits)
    ref_o, ref_l = orc.gqa_decode(q.cpu(), k.cpu(), v.cpu(), 1.0 / 8.0)
    assert_o_close(out, ref_o, f"2M keys, splits {splits}")
    assert_lse_close(lse, ref_l)


def test_longest_topk_list(gq, orc):
    """A top-K list of 65536 entries (the limit) over a 4096-page request,
    spread over every resident CTA slot and merged."""
    inp = gqa_inputs.paged_inputs(B=1, Hq=32, Hkv=8, D=128, page_size=16, pages_per_req=4096, num_pages=4100,
                                  topk=65536, seed=503, device="cuda")
    out, lse = gq.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["page_table"],
                                       inp["topk"], inp["k_scale"], inp["v_scale"])
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    ref_o, ref_l, _ = orc.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"],
                                               inp["page_table"], inp["topk"], inp["k_scale"], inp["v_scale"],
                                               1.0 / math.sqrt(128))
    assert_o_close(out.cpu(), ref_o, "top-K 65536")
    assert_lse_close(lse.cpu(), ref_l)


def test_quarter_million_token_request(gq, orc):
    """One paged FP8 request of 262144 tokens (16384 pages of 16) and a short
    one beside it; sampled rows of both against the oracle."""
    lens = [262144, 700]
    inp = gqa_inputs.paged_kv_inputs(2, 1, 64, 8, 128, 16, 16384, 2 * 16384, seed=504, kv_dtype="fp8",
                                     seq_lens=lens, device="cuda")
    out, lse = gq.gqa_decode_paged(inp["q"], inp["k_pool"], inp["v_pool"], inp["page_table"], inp["seq_lens"],
                                   inp["k_scale"], inp["v_scale"])
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    rows = [0, 7, 8, 33, 63, 64, 100, 127]  # (b * Hq + h) * Sq + i with Sq = 1
    ref_o, ref_l = orc.gqa_decode_paged(inp["q"], inp["k_pool"], inp["v_pool"], inp["page_table"], inp["seq_lens"],
                                        1.0 / math.sqrt(128), inp["k_scale"], inp["v_scale"], rows=rows)
    got_o = out.cpu().view(-1, 128)[rows]
    got_l = lse.cpu().view(-1)[rows]
    assert_o_close(got_o, ref_o, "262144-token request")
    assert_lse_close(got_l, ref_l)
    assert np.all(np.isfinite(ref_l))
