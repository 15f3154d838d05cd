"""GPU parity of paged decode over whole requests (no top-K), bf16 and FP8
pools, through the C ABI, against the fp64 oracle on the same stored bytes."""
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


def _run(gq, inp, **kw):
    d = _cuda(inp)
    out, lse = gq.gqa_decode_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"],
                                   d["k_scale"], d["v_scale"], **kw)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def _ref(orc, inp, scale):
    return orc.gqa_decode_paged(inp["q"], inp["k_pool"], inp["v_pool"], inp["page_table"], inp["seq_lens"],
                                scale, inp["k_scale"], inp["v_scale"])


def _check(out, lse, ref_o, ref_l, what):
    # rows that see no token: exactly zero output, -inf LSE
    empty = np.isneginf(ref_l)                     # [B, Hq, Sq]
    if empty.any():
        e = torch.from_numpy(empty)
        assert torch.all(torch.isneginf(lse[e])), what
        oe = out.float().permute(0, 2, 1, 3)[e]    # [n, D]
        assert torch.all(oe == 0), what
    ok = ~empty
    o_ok = torch.from_numpy(ok).permute(0, 2, 1)   # [B, Sq, Hq]
    assert_o_close(out[o_ok], ref_o[o_ok.numpy()], what)
    assert_lse_close(lse[torch.from_numpy(ok)], ref_l[ok], what)


# (B, Sq, Hq, Hkv, D, page_size, pages_per_req, kv, seq_lens)
SMALL = [
    (3, 1, 32, 8, 128, 16, 8, "bf16", (128, 77, 1)),
    (3, 1, 32, 8, 128, 16, 8, "fp8", (128, 100, 17)),
    (2, 2, 16, 4, 128, 1, 90, "bf16", (90, 33)),          # page size 1, two decode rows
    (2, 4, 8, 2, 64, 64, 3, "fp8", (192, 5)),             # four decode rows, one request shorter than a page
    (2, 3, 12, 3, 128, 16, 6, "bf16", (96, 2)),           # request shorter than S_q: rows without tokens
    (2, 1, 16, 1, 64, 16, 10, "bf16", (160, 0)),          # an empty request
    (1, 1, 96, 12, 64, 32, 4, "fp8", (111,)),             # 12 heads: a full and a partial head block
    (2, 2, 64, 8, 128, 16, 12, "fp8", (190, 64)),         # 16 rows per KV head: two n-tiles
    (1, 1, 16, 1, 128, 16, 300, "bf16", (4800,)),         # more tokens than one index-map pass
    (3, 1, 32, 8, 128, 16, 8, "int8", (128, 100, 17)),    # int8 pools
    (2, 4, 8, 2, 64, 64, 3, "int8", (192, 5)),
    (2, 2, 64, 8, 128, 16, 12, "int8", (190, 64)),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}_sq{}_h{}x{}_d{}_ps{}_ppr{}_{}".format(*s[:8]))
@pytest.mark.parametrize("splits", [0, 1, 5])
def test_paged_kv_small_vs_oracle(gq, orc, shape, splits):
    B, Sq, Hq, Hkv, D, ps, ppr, kv, lens = shape
    inp = gqa_inputs.paged_kv_inputs(B, Sq, Hq, Hkv, D, ps, ppr, B * ppr + 2, seed=sum(lens) + D + ps, kv_dtype=kv,
                                     seq_lens=list(lens))
    out, lse = _run(gq, inp, num_splits=splits)
    ref_o, ref_l = _ref(orc, inp, 1.0 / math.sqrt(D))
    _check(out, lse, ref_o, ref_l, f"paged kv {shape} splits={splits}")
    assert gq.gqa_device_status() == 0


@pytest.mark.parametrize("lens,workers", [((0, 0, 32), 31), ((0, 0, 0), 4), ((1, 0, 5, 0), 9),
                                          ((700, 3, 0, 260), 200), ((64, 64), 3)])
def test_balanced_schedule_edges(gq, orc, lens, workers):
    """More workers than 16-token steps, empty requests between and after
    shared ones, an all-empty batch."""
    B = len(lens)
    inp = gqa_inputs.paged_kv_inputs(B, 1, 16, 4, 64, 16, 48, B * 48 + 1, seed=50 + sum(lens), kv_dtype="bf16",
                                     seq_lens=list(lens))
    out, lse = _run(gq, inp, num_splits=workers)
    ref_o, ref_l = _ref(orc, inp, 0.125)
    _check(out, lse, ref_o, ref_l, f"balanced {lens} W={workers}")
    assert gq.gqa_device_status() == 0


def test_int8_extreme_codes(gq, orc):
    """int8 pools holding every code, -128 and 127 included, against the oracle
    (the quantiser of the workloads never emits -128)."""
    inp = gqa_inputs.paged_kv_inputs(2, 1, 16, 4, 128, 16, 4, 9, seed=60, kv_dtype="int8", seq_lens=[64, 40])
    g = torch.Generator().manual_seed(61)
    for name in ("k_pool", "v_pool"):
        codes = torch.randint(-128, 128, tuple(inp[name].shape), generator=g, dtype=torch.int16).to(torch.int8)
        codes.view(-1)[:256] = torch.arange(-128, 128, dtype=torch.int16).to(torch.int8)
        inp[name] = codes.contiguous()
    inp["k_scale"], inp["v_scale"] = 0.01, 0.02
    out, lse = _run(gq, inp)
    ref_o, ref_l = _ref(orc, inp, 1.0 / math.sqrt(128))
    _check(out, lse, ref_o, ref_l, "int8 extreme codes")
    assert gq.gqa_device_status() == 0


@pytest.mark.parametrize("kv", ["fp8", "int8"])
def test_device_scales_per_head_and_per_tensor(gq, orc, kv):
    """Device-side scales: per KV head (power-of-two scales, so the
    dequantised pool is exact in bf16 and the oracle runs on that bf16 pool)
    and per tensor (the same as the host scalars)."""
    B, Hq, Hkv, D = 3, 32, 8, 128
    inp = gqa_inputs.paged_kv_inputs(B, 1, Hq, Hkv, D, 16, 8, B * 8 + 1, seed=70, kv_dtype=kv, seq_lens=[128, 77, 9])
    ks = torch.tensor([2.0 ** -(e % 4 + 5) for e in range(Hkv)], dtype=torch.float32)
    vs = torch.tensor([2.0 ** -((3 * e) % 5 + 4) for e in range(Hkv)], dtype=torch.float32)
    d = _cuda(inp)
    out, lse = gq.gqa_decode_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"],
                                   k_scales=ks.cuda(), v_scales=vs.cuda())
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    codes_k = inp["k_pool"].view(torch.float8_e4m3fn).double() if kv == "fp8" else inp["k_pool"].double()
    codes_v = inp["v_pool"].view(torch.float8_e4m3fn).double() if kv == "fp8" else inp["v_pool"].double()
    kb = (codes_k * ks.double().view(1, 1, Hkv, 1)).to(torch.bfloat16)
    vb = (codes_v * vs.double().view(1, 1, Hkv, 1)).to(torch.bfloat16)
    assert torch.equal(kb.double(), codes_k * ks.double().view(1, 1, Hkv, 1))
    ref_o, ref_l = orc.gqa_decode_paged(inp["q"], kb, vb, inp["page_table"], inp["seq_lens"], 1.0 / math.sqrt(D))
    _check(out.cpu(), lse.cpu(), ref_o, ref_l, f"{kv} per-head device scales")
    # per tensor on the device == the host scalars
    o1, l1 = gq.gqa_decode_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"],
                                 k_scales=torch.tensor([inp["k_scale"]], device="cuda"),
                                 v_scales=torch.tensor([inp["v_scale"]], device="cuda"))
    o2, l2 = gq.gqa_decode_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"],
                                 inp["k_scale"], inp["v_scale"])
    torch.cuda.synchronize()
    assert torch.allclose(o1.float(), o2.float(), atol=1e-3, rtol=1e-2)
    assert torch.allclose(l1, l2, atol=1e-5, rtol=0)


def test_split_counts_agree(gq):
    """Worker counts from one (every request whole in one CTA) to more workers
    than steps agree within rounding."""
    inp = gqa_inputs.paged_kv_inputs(4, 1, 32, 8, 128, 16, 64, 300, seed=41, kv_dtype="bf16")
    ref, ref_l = _run(gq, inp, num_splits=1)
    for s in (2, 3, 7, 64, 300):
        out, lse = _run(gq, inp, num_splits=s)
        assert torch.allclose(out.float(), ref.float(), atol=2e-2, rtol=2e-2), s
        assert torch.allclose(lse, ref_l, atol=1e-3, rtol=0), s


def test_page_permutation_and_caller_workspace(gq, orc):
    """Moving every page elsewhere in the pool (and the table with it) changes
    nothing; a caller workspace gives the same result as the library pool."""
    inp = gqa_inputs.paged_kv_inputs(3, 1, 32, 8, 128, 16, 16, 60, seed=42, kv_dtype="fp8")
    out, lse = _run(gq, inp, num_splits=4)
    perm = torch.randperm(60, generator=torch.Generator().manual_seed(43))
    inv = torch.argsort(perm)
    moved = dict(inp, k_pool=inp["k_pool"][perm].contiguous(), v_pool=inp["v_pool"][perm].contiguous(),
                 page_table=inv[inp["page_table"].long()].to(torch.int32).contiguous())
    out2, lse2 = _run(gq, moved, num_splits=4)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    nbytes = gq.gqa_decode_paged_workspace_bytes(3, 1, 32, 8, 128, 1, 16, 16, 4)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out3, lse3 = _run(gq, inp, num_splits=4, workspace=ws)
    assert torch.equal(out, out3) and torch.equal(lse, lse3)


def test_sequence_length_out_of_range_flagged(gq):
    inp = gqa_inputs.paged_kv_inputs(2, 1, 8, 2, 64, 16, 4, 9, seed=44, kv_dtype="bf16", seq_lens=[64, 10])
    inp["seq_lens"][1] = 65                       # capacity is 64
    _run(gq, inp)
    assert gq.gqa_device_status() == 7
    assert gq.gqa_device_status() == 0


def test_wait_timeout_is_reported_not_hung(gq):
    """The producer withholds the first stage of every CTA (test hook): the
    bounded waits run out, the kernel returns and flags a timeout, and the
    next call works."""
    inp = gqa_inputs.paged_kv_inputs(2, 1, 32, 8, 128, 16, 8, 17, seed=45, kv_dtype="bf16")
    d = _cuda(inp)
    gq.gqa_set_wait_limit_ns(50_000_000)
    gq.gqa_debug_set_fault_mode(1)
    try:
        gq.gqa_decode_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"], num_splits=1)
        assert gq.gqa_device_status() == 6
    finally:
        gq.gqa_debug_set_fault_mode(0)
        gq.gqa_set_wait_limit_ns(0)
    out, lse = _run(gq, inp)
    assert gq.gqa_device_status() == 0
    assert torch.isfinite(lse).all()


def test_automatic_splits_reported(gq):
    n = gq.gqa_decode_paged_num_splits(4, 1, 32, 8, 128, 0, 16, 256)
    assert n >= 1
    assert gq.gqa_decode_paged_workspace_bytes(4, 1, 32, 8, 128, 0, 16, 256) == (
        0 if n == 1 else gq.gqa_decode_paged_workspace_bytes(4, 1, 32, 8, 128, 0, 16, 256, n))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["paged_bf16_b32_h64x8_d128_kv32k_ps16", "paged_fp8_b32_h64x8_d128_kv32k_ps16",
                                  "paged_int8_b32_h64x8_d128_kv32k_ps16"])
def test_full_workload_sampled_rows(gq, orc, name):
    """The benchmark workloads at full size, in the launch configuration the
    benchmark times (automatic splits); sampled rows of three requests checked
    against the oracle on a compact copy of just those requests' pages."""
    cfg = gqa_inputs.CONFIGS[name]
    inp = gqa_inputs.paged_kv_config_inputs(cfg, device="cuda")
    out, lse = gq.gqa_decode_paged(inp["q"], inp["k_pool"], inp["v_pool"], inp["page_table"], inp["seq_lens"],
                                   inp["k_scale"], inp["v_scale"])
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    reqs = [0, 17, cfg.B - 1]
    pt = inp["page_table"][reqs].long()                       # [3, ppr] pool pages
    kc = inp["k_pool"][pt.flatten()].cpu()                    # compact pools: request j's pages at j*ppr ..
    vc = inp["v_pool"][pt.flatten()].cpu()
    ppr = cfg.pages_per_req
    ptc = torch.arange(len(reqs) * ppr, dtype=torch.int32).view(len(reqs), ppr)
    sl = inp["seq_lens"][reqs].cpu()
    qc = inp["q"][reqs].cpu()
    rng = np.random.default_rng(7)
    nrow = cfg.Hq * cfg.Sq
    rows = sorted({0, len(reqs) * nrow - 1} | set(int(x) for x in rng.integers(0, len(reqs) * nrow, 40)))
    ref_o, ref_l = orc.gqa_decode_paged(qc, kc, vc, ptc, sl, cfg.scale, inp["k_scale"], inp["v_scale"], rows=rows)
    og = out[reqs].cpu()                                      # [3, Sq, Hq, D]
    lg = lse[reqs].cpu()                                      # [3, Hq, Sq]
    got_o = torch.stack([og[r // nrow, r % cfg.Sq, (r // cfg.Sq) % cfg.Hq] for r in rows])
    got_l = torch.stack([lg[r // nrow, (r // cfg.Sq) % cfg.Hq, r % cfg.Sq] for r in rows])
    assert_o_close(got_o, ref_o, name)
    assert_lse_close(got_l, ref_l, name)


@pytest.mark.parametrize("kv", ["int8", "fp8", "bf16"])
def test_contiguous_cache_as_one_page_per_request(gq, orc, kv):
    """A contiguous (unpaged) 8-bit or bf16 cache is the paged form with one
    page of the whole capacity per request.  Against the oracle, and bit for bit
    equal to the same bytes addressed as pages of 16 tokens: the kernel's
    arithmetic follows 16-token steps, never the page size."""
    B, Sq, Hq, Hkv, D, cap = 2, 2, 64, 8, 128, 2048
    inp = gqa_inputs.paged_kv_inputs(B, Sq, Hq, Hkv, D, cap, 1, B, seed=80, kv_dtype=kv, seq_lens=[cap, 1500])
    out1, lse1 = _run(gq, inp, num_splits=7)
    ref_o, ref_l = _ref(orc, inp, 1.0 / math.sqrt(D))
    _check(out1, lse1, ref_o, ref_l, f"contiguous {kv}")
    per = cap // 16
    inp16 = dict(inp)
    inp16["k_pool"] = inp["k_pool"].reshape(B * per, 16, Hkv, D).contiguous()
    inp16["v_pool"] = inp["v_pool"].reshape(B * per, 16, Hkv, D).contiguous()
    inp16["page_table"] = (inp["page_table"].long() * per + torch.arange(per)).to(torch.int32).contiguous()
    out16, lse16 = _run(gq, inp16, num_splits=7)
    assert torch.equal(out1, out16) and torch.equal(lse1, lse16)
    assert gq.gqa_device_status() == 0
