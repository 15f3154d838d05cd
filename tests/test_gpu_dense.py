"""GPU parity of the dense GQA decode path against the fp64 oracle, through
the C ABI (ctypes binding)."""
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


def _run(gq, q, k, v, scale=None, num_splits=0):
    out, lse = gq.gqa_decode_ex(q.cuda(), k.cuda(), v.cuda(), scale=scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    return out.cpu(), lse.cpu()


# (B, Sq, Skv, Hq, Hkv, D): every head dim, head ratio, decode-row count and a
# spread of KV lengths around tile (64) and split boundaries, ragged tails.
SMALL = [
    (1, 1, 1, 8, 1, 64), (1, 1, 2, 4, 2, 128), (2, 1, 63, 16, 4, 128), (1, 1, 64, 8, 4, 256),
    (1, 1, 65, 8, 2, 64), (3, 1, 1000, 64, 8, 128), (1, 1, 4097, 32, 2, 256), (2, 2, 2, 8, 1, 128),
    (1, 2, 63, 4, 2, 64), (1, 2, 65, 8, 4, 128), (2, 2, 1000, 64, 8, 128), (1, 2, 4097, 16, 4, 256),
    (1, 3, 3, 8, 2, 128), (2, 3, 64, 16, 4, 64), (1, 3, 1000, 8, 1, 256), (1, 3, 4097, 8, 4, 128),
    (1, 8, 8, 32, 2, 256), (1, 8, 65, 8, 2, 128), (2, 8, 1000, 16, 4, 64), (1, 8, 4097, 32, 2, 128),
    (1, 1, 300, 1, 1, 128), (1, 4, 777, 64, 8, 64), (1, 2, 129, 128, 2, 64),  # 128 rows / group
    (1, 4, 200, 64, 1, 128),  # 256 rows: two row groups
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}_sq{}_kv{}_h{}x{}_d{}".format(*s))
def test_dense_small_vs_oracle(gq, orc, shape):
    B, Sq, Skv, Hq, Hkv, D = shape
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=hash(shape) % 100000)
    scale = 1.0 / math.sqrt(D)
    out, lse = _run(gq, q, k, v)
    ref_o, ref_l = orc.gqa_decode(q, k, v, scale)
    assert_o_close(out, ref_o, f"O {shape}")
    assert_lse_close(lse, ref_l, f"LSE {shape}")


# Head dim 128 with 8 or more decode rows per head runs on the tcgen05 engine:
# partial tiles (32, 36, 64 rows), one full 128-row tile, two and three row
# groups, ragged key tails, a cache shorter than one 64-key tile.
UMMA128 = [
    (1, 8, 8, 8, 1, 128), (2, 8, 65, 8, 2, 128), (1, 8, 1000, 64, 8, 128), (1, 9, 777, 16, 4, 128),
    (1, 16, 4097, 64, 8, 128), (2, 12, 3000, 32, 2, 128), (1, 33, 500, 8, 1, 128), (1, 64, 200, 4, 1, 128),
]


@pytest.mark.parametrize("shape", UMMA128, ids=lambda s: "b{}_sq{}_kv{}_h{}x{}_d{}".format(*s))
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_d128_tcgen05_vs_oracle(gq, orc, shape, splits):
    B, Sq, Skv, Hq, Hkv, D = shape
    assert gq.gqa_decode_dense_engine(B, Sq, Skv, Hq, Hkv, D) == "tcgen05"
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=hash(shape) % 100000 + splits)
    out, lse = _run(gq, q, k, v, num_splits=splits)
    ref_o, ref_l = orc.gqa_decode(q, k, v, 1.0 / math.sqrt(D))
    assert_o_close(out, ref_o, f"O {shape} splits {splits}")
    assert_lse_close(lse, ref_l, f"LSE {shape} splits {splits}")


# More than 128 rows per KV head: 256 (64 query heads on 8 KV heads, 32
# decode rows; two row groups per request, KV head and split) and 640 (five).
MANY_ROWS128 = [(2, 32, 3001, 64, 8, 128), (1, 40, 1500, 16, 1, 128)]


@pytest.mark.parametrize("shape", MANY_ROWS128, ids=lambda s: "b{}_sq{}_kv{}_h{}x{}_d{}".format(*s))
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_d128_many_row_groups_vs_oracle(gq, orc, shape, splits):
    B, Sq, Skv, Hq, Hkv, D = shape
    assert gq.gqa_decode_dense_engine(B, Sq, Skv, Hq, Hkv, D) == "tcgen05"
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=Sq * 1000 + Skv + splits)
    out, lse = _run(gq, q, k, v, num_splits=splits)
    assert gq.gqa_device_status() == 0
    ref_o, ref_l = orc.gqa_decode(q, k, v, 1.0 / math.sqrt(D))
    assert_o_close(out, ref_o, f"O {shape} splits {splits}")
    assert_lse_close(lse, ref_l, f"LSE {shape} splits {splits}")


# Small caches that the automatic choice would split run as one CTA per
# (b, g, row group) whose warps split the walk (key lanes) and merge in shared
# memory: 6 lanes of 16 rows or 4 lanes of 32; ragged tails, lanes with no
# tile (200 keys: 7 tiles of 32 for 6 lanes; 130 and 150 keys: 3 tiles of 64),
# causal rows, the 256 KiB bound.
LANES = [(1, 1, 1000, 8, 1, 64), (1, 1, 512, 8, 1, 128), (2, 2, 500, 32, 8, 128), (1, 4, 1024, 16, 2, 64),
         (1, 4, 400, 64, 4, 128), (2, 3, 300, 64, 4, 128),
         (1, 1, 200, 8, 1, 128), (1, 4, 150, 8, 1, 64), (1, 2, 480, 16, 1, 128), (1, 1, 130, 4, 1, 64)]


@pytest.mark.parametrize("shape", LANES, ids=lambda s: "b{}_sq{}_kv{}_h{}x{}_d{}".format(*s))
def test_key_lanes_vs_oracle(gq, orc, shape):
    B, Sq, Skv, Hq, Hkv, D = shape
    assert gq.gqa_decode_num_splits(B, Sq, Skv, Hq, Hkv, D) == 1
    assert gq.gqa_decode_workspace_bytes(B, Sq, Skv, Hq, Hkv, D, 0) == 0
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=Skv * 10 + Sq)
    out, lse = _run(gq, q, k, v)
    ref_o, ref_l = orc.gqa_decode(q, k, v, 1.0 / math.sqrt(D))
    assert_o_close(out, ref_o, f"O {shape}")
    assert_lse_close(lse, ref_l, f"LSE {shape}")
    # an explicit split count takes the split + combine path: same values within rounding
    o2, l2 = _run(gq, q, k, v, num_splits=2)
    assert_o_close(o2, out.double(), f"O {shape} vs 2 splits")
    assert torch.allclose(l2, lse, atol=1e-4, rtol=0)


# Longer caches over few (batch row, KV head) units: one wave of key-lane CTAs,
# SMs // units splits, then the combine -- at least 4 splits a unit; one (no
# combine) when that fills 80 % of the SMs, or 60 % with at most 2K keys; 2-3
# when the wave fills 80 % of the SMs with splits of 2K keys or more.  Tiles
# per lane from under one to past the ring depth, ragged last splits, both
# lane layouts.
LANE_SPLITS = [(1, 2, 5000, 16, 2, 128), (2, 1, 3001, 32, 8, 128), (1, 4, 4100, 16, 2, 64),
               (4, 1, 2500, 32, 8, 64), (1, 1, 20000, 8, 1, 64), (1, 2, 40000, 16, 2, 128),
               (1, 1, 60000, 8, 1, 128), (8, 1, 8200, 32, 8, 128), (9, 2, 5000, 16, 8, 64),
               (16, 1, 2100, 32, 8, 128), (19, 2, 2500, 16, 8, 64), (128, 1, 2048, 8, 1, 128),
               (16, 1, 600, 32, 8, 128), (12, 2, 1024, 16, 8, 128),
               (1, 4, 5000, 64, 4, 128), (2, 4, 3001, 128, 8, 128)]  # the last two: 64 rows a CTA


def _lane_plan_splits(B, Sq, Skv, Hq, Hkv, D):
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    units = B * Hkv  # Sq * G <= 32 rows: one row group
    n_blocks = -(-Skv // 64)
    ls = min(nsm // units, n_blocks)
    tps = -(-n_blocks // ls)
    return nsm // units, -(-n_blocks // tps)


@pytest.mark.parametrize("shape", LANE_SPLITS, ids=lambda s: "b{}_sq{}_kv{}_h{}x{}_d{}".format(*s))
def test_key_lane_splits_vs_oracle(gq, orc, shape):
    B, Sq, Skv, Hq, Hkv, D = shape
    per_sm, want = _lane_plan_splits(*shape)
    assert per_sm >= 1
    assert gq.gqa_decode_num_splits(B, Sq, Skv, Hq, Hkv, D) == want
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=Skv + Sq)
    out, lse = _run(gq, q, k, v)
    ref_o, ref_l = orc.gqa_decode(q, k, v, 1.0 / math.sqrt(D))
    assert_o_close(out, ref_o, f"O {shape}")
    assert_lse_close(lse, ref_l, f"LSE {shape}")


def test_key_lanes_bound(gq):
    """Past 256 KiB of K and V per (b, g) the automatic choice splits across CTAs."""
    assert gq.gqa_decode_num_splits(1, 1, 1024, 8, 1, 64) == 1       # exactly 256 KiB
    assert gq.gqa_decode_num_splits(1, 1, 1088, 8, 1, 64) > 1        # just above
    assert gq.gqa_decode_num_splits(1, 1, 1000, 8, 1, 256) > 1       # head dim 256: split kernel
    assert gq.gqa_decode_num_splits(1, 8, 1000, 64, 8, 128) > 1      # 64 rows per CTA
    # one wave of 3 key-lane splits a unit would fill only 120 of the SMs: general choice
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    if 5 * 40 * (nsm // 40) < 4 * nsm:
        assert gq.gqa_decode_num_splits(5, 1, 8192, 32, 8, 128) != nsm // 40
    # 96 units, one CTA each, would leave a third of the SMs idle: general
    # choice unless the caches are short; 80 units: general choice
    if nsm // 96 == 1 and 100 * 96 // nsm < 80:
        assert gq.gqa_decode_num_splits(12, 1, 8192, 32, 8, 128) > 1
        if 100 * 96 // nsm >= 60:
            assert gq.gqa_decode_num_splits(12, 1, 2048, 32, 8, 128) == 1
    if nsm // 80 == 1 and 100 * 80 // nsm < 60:
        assert gq.gqa_decode_num_splits(10, 1, 2048, 32, 8, 128) > 1
    # two-split waves need splits of 2K keys or more
    if nsm // 64 == 2 and 5 * 64 * 2 >= 4 * nsm:
        assert gq.gqa_decode_num_splits(8, 1, 2048, 32, 8, 128) != 2


def test_d128_engine_boundary(gq, orc):
    """Sq = 7 (mma.sync) and Sq = 8 (tcgen05) on the same cache agree with the
    oracle and with each other on the rows they share (the last 7 rows of the
    Sq = 8 call see the same keys as the Sq = 7 call)."""
    B, Skv, Hq, Hkv, D = 1, 2000, 16, 2, 128
    q8, k, v = gqa_inputs.dense_inputs(B, 8, Skv, Hq, Hkv, D, seed=77)
    q7 = q8[:, 1:].contiguous()
    assert gq.gqa_decode_dense_engine(B, 7, Skv, Hq, Hkv, D) == "mma.sync"
    o7, l7 = _run(gq, q7, k, v)
    o8, l8 = _run(gq, q8, k, v)
    for o, l, q in ((o7, l7, q7), (o8, l8, q8)):
        ref_o, ref_l = orc.gqa_decode(q, k, v, 1.0 / math.sqrt(D))
        assert_o_close(o, ref_o, f"Sq {q.shape[1]}")
        assert_lse_close(l, ref_l)
    assert_o_close(o8[:, 1:], o7.double(), "Sq 8 rows 1.. vs Sq 7")
    assert torch.allclose(l8[:, :, 1:], l7, atol=1e-4, rtol=0)


@pytest.mark.parametrize("splits", [1, 2, 7, 10**6])
def test_split_counts_agree(gq, orc, splits):
    B, Sq, Skv, Hq, Hkv, D = 1, 2, 1000, 16, 2, 128
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=77)
    out, lse = _run(gq, q, k, v, num_splits=splits)
    ref_o, ref_l = orc.gqa_decode(q, k, v, 1 / math.sqrt(D))
    assert_o_close(out, ref_o, f"splits={splits}")
    assert_lse_close(lse, ref_l, f"splits={splits}")


def test_split_invariance(gq):
    """Splitting the KV walk changes results only by rounding."""
    q, k, v = gqa_inputs.dense_inputs(2, 3, 3000, 32, 4, 64, seed=5)
    o1, l1 = _run(gq, q, k, v, num_splits=1)
    for s in (2, 7, 47):
        o2, l2 = _run(gq, q, k, v, num_splits=s)
        assert_o_close(o2, o1.double(), f"splits {s} vs 1")
        assert torch.allclose(l1, l2, atol=1e-4, rtol=0)


def test_same_splits_bitwise_repeatable(gq):
    q, k, v = gqa_inputs.dense_inputs(1, 2, 5000, 64, 8, 128, seed=6)
    a = _run(gq, q, k, v, num_splits=9)
    b = _run(gq, q, k, v, num_splits=9)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("shape", [(1, 2, 5000, 64, 8, 128), (1, 1, 1000, 8, 1, 64), (16, 1, 2100, 32, 8, 128)],
                         ids=["lane_splits", "lane_one_cta_small", "lane_one_cta_per_unit"])
def test_key_lanes_bitwise_repeatable(gq, shape):
    """The key-lane merge runs in lane order: repeated calls give the same bits."""
    q, k, v = gqa_inputs.dense_inputs(*shape, seed=8)
    a = _run(gq, q, k, v)
    for _ in range(3):
        b = _run(gq, q, k, v)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("Hq,Hkv", [(8, 4), (8, 2), (4, 2), (16, 4), (8, 1), (64, 8), (32, 2)])
@pytest.mark.parametrize("Sq", [1, 2, 8, 32])
@pytest.mark.parametrize("D", [128, 256])
def test_gqa_bitwise_equals_expanded_mha(gq, Hq, Hkv, Sq, D):
    """Native GQA == the same kernel on K/V pre-expanded to Hq heads, bit for bit
    (split count pinned: the automatic choice depends on B*Hkv)."""
    B, Skv = 2, 700
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=Hq * 100 + Hkv)
    G = Hq // Hkv
    o1, l1 = _run(gq, q, k, v, num_splits=5)
    o2, l2 = _run(gq, q, k.repeat_interleave(G, dim=2).contiguous(), v.repeat_interleave(G, dim=2).contiguous(),
                  num_splits=5)
    assert torch.equal(o1, o2), (Hq, Hkv)
    assert torch.equal(l1, l2), (Hq, Hkv)


def test_single_key_exact(gq):
    """Degenerate single-key softmax: O is V_0 exactly, LSE is the one score."""
    q, k, v = gqa_inputs.dense_inputs(3, 1, 1, 16, 4, 128, seed=9)
    out, lse = _run(gq, q, k, v)
    G = 4
    assert torch.equal(out, v.repeat_interleave(G, dim=2))
    s0 = (q.double() * k.double().repeat_interleave(G, dim=2)).sum(-1) / math.sqrt(128)  # [B,1,Hq]
    assert torch.allclose(lse.double(), s0.permute(0, 2, 1), atol=1e-4, rtol=0)


def test_causal_row0_sees_one_key(gq):
    """Sq == Skv: row 0 sees only key 0 (bottom-right alignment)."""
    q, k, v = gqa_inputs.dense_inputs(1, 4, 4, 8, 2, 64, seed=10)
    out, _ = _run(gq, q, k, v)
    assert torch.equal(out[:, 0], v[:, 0].repeat_interleave(4, dim=1))


@pytest.mark.parametrize("D", [128, 256])
def test_short_last_split_fully_masked(gq, orc, D):
    """The last split holds keys no earlier row may see: its partial LSE is -inf
    and its weight in the combine must be exactly zero (no NaN)."""
    for (Sq, Skv, splits) in [(2, 65, 2), (8, 70, 2), (8, 129, 3), (3, 130, 3)]:
        q, k, v = gqa_inputs.dense_inputs(1, Sq, Skv, 16, 2, D, seed=Skv)
        out, lse = _run(gq, q, k, v, num_splits=splits)
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        ref_o, ref_l = orc.gqa_decode(q, k, v, 1 / math.sqrt(D))
        assert_o_close(out, ref_o, f"short last split {Sq},{Skv},{splits}")
        assert_lse_close(lse, ref_l)


def test_closed_forms_on_gpu(gq):
    """K == 0: LSE = ln(#visible), O = mean of visible V.  Constant V: O = V row."""
    B, Sq, Skv, Hq, Hkv, D = 2, 3, 3001, 16, 4, 128
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=11)
    kz = torch.zeros_like(k)
    out, lse = _run(gq, q, kz, v)
    G = Hq // Hkv
    for i in range(Sq):
        nvis = Skv - Sq + 1 + i
        assert torch.allclose(lse[:, :, i].double(), torch.full((B, Hq), math.log(nvis), dtype=torch.float64),
                              atol=1e-3, rtol=0)
        mean = v[:, :nvis].double().mean(dim=1).repeat_interleave(G, dim=1)
        assert_o_close(out[:, i], mean, "zero-K mean")
    vc = v[:, :1].expand(B, Skv, Hkv, D).contiguous()
    out, _ = _run(gq, q, k, vc)
    for i in range(Sq):
        assert_o_close(out[:, i], vc[:, 0].double().repeat_interleave(G, dim=1), "constant V")


def test_scale_default_and_explicit(gq, orc):
    q, k, v = gqa_inputs.dense_inputs(1, 1, 500, 8, 2, 64, seed=12)
    o_def, l_def = _run(gq, q, k, v, scale=None)
    o_exp, l_exp = _run(gq, q, k, v, scale=1 / 8.0)
    assert torch.equal(o_def, o_exp) and torch.equal(l_def, l_exp)
    o3, l3 = _run(gq, q, k, v, scale=0.37)
    ref_o, ref_l = orc.gqa_decode(q, k, v, 0.37)
    assert_o_close(o3, ref_o)
    assert_lse_close(l3, ref_l)


def test_caller_workspace(gq, orc):
    B, Sq, Skv, Hq, Hkv, D = 1, 2, 2000, 64, 8, 128
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=13)
    need = gq.gqa_decode_workspace_bytes(B, Sq, Skv, Hq, Hkv, D, 6)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o1, l1 = gq.gqa_decode_ex(q.cuda(), k.cuda(), v.cuda(), num_splits=6, workspace=ws)
    o2, l2 = gq.gqa_decode_ex(q.cuda(), k.cuda(), v.cuda(), num_splits=6)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(gq.GQAError) as ei:
        gq.gqa_decode_ex(q.cuda(), k.cuda(), v.cuda(), num_splits=6, workspace=small)
    assert ei.value.status == 4


def test_without_lse(gq):
    q, k, v = gqa_inputs.dense_inputs(1, 1, 300, 8, 1, 128, seed=14)
    a, _ = gq.gqa_decode(q.cuda(), k.cuda(), v.cuda(), with_lse=False)
    b, _ = gq.gqa_decode(q.cuda(), k.cuda(), v.cuda())
    assert torch.equal(a, b)


def test_host_entry_point(gq):
    """The host-buffer entry point gives the device path's result."""
    q, k, v = gqa_inputs.dense_inputs(1, 2, 3000, 64, 8, 128, seed=15)
    out_h = torch.empty_like(q).pin_memory()
    lse_h = torch.empty((1, 64, 2), dtype=torch.float32).pin_memory()
    gq.gqa_decode_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), out_h, lse_h)
    o_d, l_d = gq.gqa_decode(q.cuda(), k.cuda(), v.cuda())
    assert torch.equal(out_h, o_d.cpu()) and torch.equal(lse_h, l_d.cpu())


def test_invalid_args_launch_nothing(gq):
    q, _, _ = (t.cuda() for t in gqa_inputs.dense_inputs(1, 1, 64, 8, 2, 128, seed=16))
    _, k, v = (t.cuda() for t in gqa_inputs.dense_inputs(1, 1, 64, 8, 8 // 3 + 1, 128, seed=16))  # 3 KV heads
    with pytest.raises(gq.GQAError) as ei:
        gq.gqa_decode(q, k, v)                # 8 query heads over 3 KV heads
    assert ei.value.status == 1
    assert gq.gqa_device_status() == 0


@pytest.mark.parametrize("D,Sq", [(128, 1), (128, 8), (256, 1)])
def test_wait_timeout_is_reported_not_hung(gq, D, Sq):
    """A load that never arrives makes the bounded pipeline wait run out: the
    kernel flags GQA_ERR_DEVICE_TIMEOUT and returns; the context stays usable.
    (d128 with Sq 1: mma.sync engine; d128 with Sq 8 and d256: tcgen05.)"""
    q, k, v = (t.cuda() for t in gqa_inputs.dense_inputs(1, Sq, 1000, 8, 2, D, seed=17))
    gq.gqa_set_wait_limit_ns(50_000_000)
    gq.gqa_debug_set_fault_mode(1)
    try:
        gq.gqa_decode_ex(q, k, v, num_splits=2)
        assert gq.gqa_device_status() == 6
    finally:
        gq.gqa_debug_set_fault_mode(0)
        gq.gqa_set_wait_limit_ns(0)
    out, lse = gq.gqa_decode_ex(q, k, v, num_splits=2)
    assert gq.gqa_device_status() == 0
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("shape", [(1, 1, 1000, 8, 1, 64), (1, 2, 5000, 64, 8, 128), (1, 4, 1024, 16, 2, 64)],
                         ids=["lanes_whole_cache", "lane_splits", "lanes_32_rows"])
def test_key_lanes_wait_timeout_is_reported_not_hung(gq, shape):
    """The key-lane instances under the same forced timeout (automatic plan): the
    lane whose tile never lands gives up, the others stop at the abort flag,
    every consumer warp still reaches the merge barriers, and the context stays
    usable."""
    q, k, v = (t.cuda() for t in gqa_inputs.dense_inputs(*shape, seed=19))
    gq.gqa_set_wait_limit_ns(50_000_000)
    gq.gqa_debug_set_fault_mode(1)
    try:
        gq.gqa_decode_ex(q, k, v, num_splits=0)
        assert gq.gqa_device_status() == 6
    finally:
        gq.gqa_debug_set_fault_mode(0)
        gq.gqa_set_wait_limit_ns(0)
    out, lse = gq.gqa_decode_ex(q, k, v, num_splits=0)
    assert gq.gqa_device_status() == 0
    assert torch.isfinite(out.float()).all()


FULL = [c for c in gqa_inputs.CONFIGS.values() if isinstance(c, gqa_inputs.DenseConfig) and c.dv == c.D]


@pytest.mark.slow
@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_full_size_sampled_rows(gq, orc, cfg):
    """Configurations at full size, automatic splits (the benchmark's launch):
    sampled (batch, KV head) groups checked row by row against the oracle run
    on that group's slice of the cache."""
    q, k, v = gqa_inputs.dense_config_inputs(cfg, device="cuda")
    out, lse = gq.gqa_decode(q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    G = cfg.Hq // cfg.Hkv
    rng = np.random.default_rng(cfg.seed)
    picks = {(0, 0), (cfg.B - 1, cfg.Hkv - 1)}
    while len(picks) < min(4, cfg.B * cfg.Hkv):
        picks.add((int(rng.integers(cfg.B)), int(rng.integers(cfg.Hkv))))
    for b, g in sorted(picks):
        qs = q[b:b + 1, :, g * G:(g + 1) * G].cpu()
        ks = k[b:b + 1, :, g:g + 1].cpu()
        vs = v[b:b + 1, :, g:g + 1].cpu()
        ref_o, ref_l = orc.gqa_decode(qs, ks, vs, cfg.scale)
        got_o = out[b:b + 1, :, g * G:(g + 1) * G].cpu()
        got_l = lse[b:b + 1, g * G:(g + 1) * G].cpu()
        assert_o_close(got_o, ref_o, f"{cfg.name} b={b} g={g}")
        assert_lse_close(got_l, ref_l, f"{cfg.name} b={b} g={g}")
        print(cfg.name, b, g, diagnostics(got_o, ref_o))


def test_cuda_graph_capture_and_replay(gq, orc):
    """The decode call (split kernel, programmatically dependent combine and
    the stream-ordered workspace from the library pool) can be captured in a
    CUDA graph; replays recompute from the current inputs."""
    B, Sq, Skv, Hq, Hkv, D = 2, 1, 3000, 32, 8, 128
    q, k, v = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=77, device="cuda")
    assert gq.gqa_decode_num_splits(B, Sq, Skv, Hq, Hkv, D) > 1
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gq.gqa_decode(q, k, v, out=out, lse=lse)  # first call outside capture (pool, attributes)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            gq.gqa_decode(q, k, v, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    for seed in (78, 79):
        q2, _, _ = gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed=seed, device="cuda")
        q.copy_(q2)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = orc.gqa_decode(q.cpu(), k.cpu(), v.cpu(), 1.0 / math.sqrt(D))
        assert_o_close(out.cpu(), ref_o, "graph replay")
        assert_lse_close(lse.cpu(), ref_l, "graph replay lse")
    assert gq.gqa_device_status() == 0
