"""GPU parity of the sparse paged FP8 decode path: the index map and the FP8
widening bit for bit, the attention output against the fp64 oracle run on the
same stored codes and scales."""
import math

import numpy as np
import pytest
import torch

import gqa_inputs
from parity import assert_lse_close, assert_o_close, diagnostics

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


def _paged_run(gq, inp, scale=None):
    d = _cuda(inp)
    out, lse = gq.gqa_decode_paged_fp8(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["page_table"], d["topk"],
                                       d["k_scale"], d["v_scale"], scale=scale)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def test_fp8_widening_all_codes(gq, orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).cuda()
    got = gq.gqa_fp8_e4m3fn_to_f32(codes).cpu().double().numpy()
    ref = np.array([orc.e4m3fn_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # odd length exercises the lone last code
    got3 = gq.gqa_fp8_e4m3fn_to_f32(codes[:3].contiguous()).cpu().double().numpy()
    assert np.array_equal(got3, ref[:3])


@pytest.mark.parametrize("ps,ppr,topk,pad", [(1, 40, 33, 0), (16, 32, 512, 0), (16, 8, 100, 7), (64, 3, 150, 1)])
def test_gather_bitexact(gq, orc, ps, ppr, topk, pad):
    inp = gqa_inputs.paged_inputs(B=5, Hq=16, Hkv=4, D=128, page_size=ps, pages_per_req=ppr,
                                  num_pages=5 * ppr + 3, topk=topk, seed=ps * 1000 + topk, pad_tail=pad)
    d = _cuda(inp)
    got = gq.gqa_paged_gather_fp8(d["k_pool"], d["page_table"], d["topk"]).cpu().numpy()
    ref = orc.paged_gather(inp["k_pool"], inp["page_table"], inp["topk"], ps)
    assert np.array_equal(got, ref)
    assert gq.gqa_device_status() == 0


def test_gather_bitexact_full_workload(gq, orc):
    cfg = gqa_inputs.CONFIGS["paged_fp8_b256_h32x8_d128_top512_ps16"]
    inp = gqa_inputs.paged_config_inputs(cfg, device="cuda")
    got = gq.gqa_paged_gather_fp8(inp["v_pool"], inp["page_table"], inp["topk"]).cpu().numpy()
    ref = orc.paged_gather(inp["v_pool"], inp["page_table"], inp["topk"], cfg.page_size)
    assert np.array_equal(got, ref)


def test_out_of_range_index_flagged(gq):
    inp = gqa_inputs.paged_inputs(B=2, Hq=8, Hkv=2, D=64, page_size=4, pages_per_req=4, num_pages=8, topk=16,
                                  seed=3)
    inp["page_table"][1, 2] = 999          # page id outside the pool
    d = _cuda(inp)
    gq.gqa_decode_paged_fp8(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["page_table"], d["topk"],
                            d["k_scale"], d["v_scale"])
    assert gq.gqa_device_status() == 7
    assert gq.gqa_device_status() == 0     # read-and-clear


# (B, Hq, Hkv, D, page_size, pages_per_req, topk, pad_tail)
SMALL = [
    (2, 8, 2, 64, 16, 4, 64, 0), (3, 32, 8, 128, 16, 32, 512, 0), (2, 16, 1, 128, 16, 8, 100, 0),
    (1, 4, 4, 128, 1, 70, 70, 5), (2, 12, 4, 64, 64, 2, 97, 3), (1, 16, 16, 128, 8, 200, 1300, 0),
    (2, 2, 2, 128, 16, 2, 1, 0), (2, 8, 8, 64, 16, 2, 17, 16),
    # CTAs serving part of a head block: 3 heads of 4, 12 heads as 8 + 4, two n-tiles with 3 heads of 4
    (2, 6, 3, 128, 16, 4, 50, 2), (2, 96, 12, 64, 16, 4, 60, 0), (2, 48, 3, 128, 16, 8, 120, 2),
    # more selected entries than one pass of the index map resolves (2048), ragged last pass
    (1, 8, 2, 64, 16, 170, 2600, 3), (1, 16, 8, 128, 32, 80, 2049, 0),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}_h{}x{}_d{}_ps{}_ppr{}_k{}_pad{}".format(*s))
def test_paged_small_vs_oracle(gq, orc, shape):
    B, Hq, Hkv, D, ps, ppr, topk, pad = shape
    inp = gqa_inputs.paged_inputs(B, Hq, Hkv, D, ps, ppr, B * ppr + 1, topk, seed=sum(shape), pad_tail=pad)
    scale = 1.0 / math.sqrt(D)
    out, lse = _paged_run(gq, inp)
    ref_o, ref_l, _ = orc.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"],
                                               inp["page_table"], inp["topk"], inp["k_scale"], inp["v_scale"],
                                               scale)
    assert_o_close(out, ref_o, f"paged {shape}")
    assert_lse_close(lse, ref_l, f"paged {shape}")
    assert gq.gqa_device_status() == 0


def test_wait_timeout_is_reported_not_hung(gq):
    """The producer withholds each CTA's first stage (test hook): the consumers'
    bounded waits run out, the kernel returns and flags a timeout, and the
    context stays usable for the next call."""
    inp = gqa_inputs.paged_inputs(2, 32, 8, 128, 16, 8, 17, 128, seed=31)
    d = _cuda(inp)
    gq.gqa_set_wait_limit_ns(50_000_000)
    gq.gqa_debug_set_fault_mode(1)
    try:
        gq.gqa_decode_paged_fp8(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["page_table"], d["topk"],
                                d["k_scale"], d["v_scale"])
        assert gq.gqa_device_status() == 6
    finally:
        gq.gqa_debug_set_fault_mode(0)
        gq.gqa_set_wait_limit_ns(0)
    out, lse = _paged_run(gq, inp)
    assert gq.gqa_device_status() == 0
    assert torch.isfinite(lse).all()


def test_all_padding_row(gq):
    inp = gqa_inputs.paged_inputs(2, 8, 2, 128, 16, 2, 32, 5, seed=21)
    inp["topk"][1, :] = -1
    out, lse = _paged_run(gq, inp)
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    assert torch.isfinite(lse[0]).all()


def test_gate_zero_halves_and_topk_order(gq):
    inp = gqa_inputs.paged_inputs(2, 16, 4, 128, 16, 8, 128, 17, seed=22)
    out, lse = _paged_run(gq, inp)
    inp0 = dict(inp, gate=torch.zeros_like(inp["gate"]))
    big = dict(inp, gate=torch.full_like(inp["gate"], 30.0))
    o0, _ = _paged_run(gq, inp0)
    ob, _ = _paged_run(gq, big)
    assert torch.equal(o0.float(), (0.5 * ob.float()).to(torch.bfloat16).float()) or \
        torch.allclose(o0.float(), 0.5 * ob.float(), atol=1e-2, rtol=1e-2)
    n = inp["topk"].shape[1]
    perm = torch.stack([torch.randperm(n, generator=torch.Generator().manual_seed(b)) for b in range(2)])
    inp_p = dict(inp, topk=torch.gather(inp["topk"], 1, perm).contiguous())
    op, lp = _paged_run(gq, inp_p)
    assert torch.allclose(op.float(), out.float(), atol=1e-2, rtol=1e-2)
    assert torch.allclose(lp, lse, atol=1e-4, rtol=0)


@pytest.mark.slow
def test_full_workload_sampled_rows(gq, orc):
    cfg = gqa_inputs.CONFIGS["paged_fp8_b256_h32x8_d128_top512_ps16"]
    inp = gqa_inputs.paged_config_inputs(cfg, device="cuda")
    out, lse = gq.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["page_table"],
                                       inp["topk"], inp["k_scale"], inp["v_scale"])
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    rng = np.random.default_rng(5)
    rows = sorted({0, cfg.B * cfg.Hq - 1} | set(int(x) for x in rng.integers(0, cfg.B * cfg.Hq, 60)))
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    ref_o, ref_l, _ = orc.gqa_decode_paged_fp8(cpu["q"], cpu["gate"], cpu["k_pool"], cpu["v_pool"],
                                               cpu["page_table"], cpu["topk"], cpu["k_scale"], cpu["v_scale"],
                                               cfg.scale, rows=rows)
    got_o = out.view(-1, cfg.D)[rows].cpu()
    got_l = lse.view(-1)[rows].cpu()
    assert_o_close(got_o, ref_o, "paged full")
    assert_lse_close(got_l, ref_l, "paged full")
    print(diagnostics(got_o, ref_o))


def test_topk_device_scales_per_head_and_per_tensor(gq, orc):
    """Top-K form with scales in device memory: per KV head against the oracle
    run once per KV head with that head's scales (rows are independent), and
    per tensor equal to the host scalars within rounding of the multiplier."""
    B, Hq, Hkv, D = 6, 32, 8, 128
    inp = gqa_inputs.paged_inputs(B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=16, pages_per_req=8, num_pages=B * 8 + 5,
                                  topk=100, seed=4242, pad_tail=3)
    ks = torch.tensor([inp["k_scale"] * (0.5 + 0.125 * e) for e in range(Hkv)], dtype=torch.float32)
    vs = torch.tensor([inp["v_scale"] * (1.5 - 0.0625 * e) for e in range(Hkv)], dtype=torch.float32)
    d = _cuda(inp)
    out, lse = gq.gqa_decode_paged_fp8(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["page_table"], d["topk"],
                                       k_scales=ks.cuda(), v_scales=vs.cuda())
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    for g in range(Hkv):
        rows = [b * Hq + h for b in range(B) for h in range(g * G, (g + 1) * G)]
        ref_o, ref_l, _ = orc.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"],
                                                   inp["page_table"], inp["topk"], float(ks[g]), float(vs[g]),
                                                   scale, rows=rows)
        got_o = out.cpu().view(B * Hq, D)[rows]
        got_l = lse.cpu().view(B * Hq)[rows]
        assert_o_close(got_o, ref_o, f"per-head device scales, KV head {g}")
        assert_lse_close(got_l, ref_l, f"per-head device scales, KV head {g}")
    o1, l1 = gq.gqa_decode_paged_fp8(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["page_table"], d["topk"],
                                     k_scales=torch.tensor([inp["k_scale"]], device="cuda"),
                                     v_scales=torch.tensor([inp["v_scale"]], device="cuda"))
    o2, l2 = _paged_run(gq, inp)
    torch.cuda.synchronize()
    assert torch.allclose(o1.cpu().float(), o2.float(), atol=1e-3, rtol=1e-2)
    assert torch.allclose(l1.cpu(), l2, atol=1e-5, rtol=0)
