"""GPU parity of dense decode with a score head size different from the value
head size (the d192x128 flavour: q and K of 192 dims, V and the output of
128) against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import gqa_inputs
from parity import assert_lse_close, assert_o_close, diagnostics

pytestmark = pytest.mark.gpu

DQK, DV = 192, 128


@pytest.fixture(scope="module")
def gq():
    from gqa_decode_attention_gb300 import build as gbuild
    gbuild.build()
    import gqa_decode_attention_gb300 as m
    m.load_library()
    assert torch.cuda.is_available()
    return m


def _inputs(B, Sq, Skv, Hq, Hkv, seed):
    return gqa_inputs.dense_inputs(B, Sq, Skv, Hq, Hkv, DQK, seed=seed, Dv=DV)


def _run(gq, q, k, v, scale=None, num_splits=0, workspace=None):
    out, lse = gq.gqa_decode_dv(q.cuda(), k.cuda(), v.cuda(), scale=scale, num_splits=num_splits,
                                workspace=workspace)
    torch.cuda.synchronize()
    assert gq.gqa_device_status() == 0
    return out.cpu(), lse.cpu()


# (B, Sq, Skv, Hq, Hkv): head ratios 1..32, decode rows 1..16, group rows up
# to 192 (two row groups), KV lengths around tile and split boundaries.
SMALL = [
    (1, 1, 1, 8, 1), (1, 1, 63, 8, 2), (2, 1, 65, 16, 4), (1, 1, 1000, 64, 8), (3, 1, 4097, 32, 4),
    (1, 2, 2, 8, 1), (1, 2, 129, 64, 8), (2, 4, 777, 16, 2), (1, 8, 1000, 32, 4), (1, 3, 300, 128, 2),
    (1, 16, 4097, 64, 8), (2, 1, 3000, 4, 4),
]


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}_sq{}_kv{}_h{}x{}".format(*s))
def test_dv_small_vs_oracle(gq, orc, shape, splits):
    B, Sq, Skv, Hq, Hkv = shape
    q, k, v = _inputs(B, Sq, Skv, Hq, Hkv, seed=hash(shape) % 100000)
    out, lse = _run(gq, q, k, v, num_splits=splits)
    assert out.shape == (B, Sq, Hq, DV)
    ref_o, ref_l = orc.gqa_decode_dv(q, k, v, 1.0 / math.sqrt(DQK))
    assert_o_close(out, ref_o, f"O {shape} splits={splits}")
    assert_lse_close(lse, ref_l, f"LSE {shape} splits={splits}")


# Key lanes: caches of at most 256 KiB of K and V per (b, g) (409 keys at
# 640 bytes a key) in one CTA, and longer caches over few units split across
# one wave of key-lane CTAs (SMs // units splits); both lane layouts (16 and
# 32 rows), ragged tails, causal rows.
DV_LANES_ONE = [(1, 1, 409, 8, 1), (1, 2, 300, 16, 2), (1, 4, 350, 16, 2), (2, 1, 200, 32, 8)]
DV_LANE_SPLITS = [(1, 2, 5000, 64, 8), (2, 1, 3001, 32, 8), (1, 1, 20000, 8, 1), (1, 4, 4100, 16, 2)]


@pytest.mark.parametrize("shape", DV_LANES_ONE, ids=lambda s: "b{}_sq{}_kv{}_h{}x{}".format(*s))
def test_dv_key_lanes_one_cta_vs_oracle(gq, orc, shape):
    B, Sq, Skv, Hq, Hkv = shape
    assert gq.gqa_decode_dv_num_splits(B, Sq, Skv, Hq, Hkv, DQK, DV) == 1
    assert gq.gqa_decode_dv_workspace_bytes(B, Sq, Skv, Hq, Hkv, DQK, DV, 0) == 0
    q, k, v = _inputs(B, Sq, Skv, Hq, Hkv, seed=Skv * 7 + Sq)
    out, lse = _run(gq, q, k, v)
    ref_o, ref_l = orc.gqa_decode_dv(q, k, v, 1.0 / math.sqrt(DQK))
    assert_o_close(out, ref_o, f"O {shape}")
    assert_lse_close(lse, ref_l, f"LSE {shape}")


@pytest.mark.parametrize("shape", DV_LANE_SPLITS, ids=lambda s: "b{}_sq{}_kv{}_h{}x{}".format(*s))
def test_dv_key_lane_splits_vs_oracle(gq, orc, shape):
    B, Sq, Skv, Hq, Hkv = shape
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    units = B * Hkv  # Sq * G <= 32 rows: one row group
    n_blocks = -(-Skv // 64)
    ls = min(nsm // units, n_blocks)
    tps = -(-n_blocks // ls)
    assert nsm // units >= 4
    assert gq.gqa_decode_dv_num_splits(B, Sq, Skv, Hq, Hkv, DQK, DV) == -(-n_blocks // tps)
    q, k, v = _inputs(B, Sq, Skv, Hq, Hkv, seed=Skv * 3 + Sq)
    out, lse = _run(gq, q, k, v)
    ref_o, ref_l = orc.gqa_decode_dv(q, k, v, 1.0 / math.sqrt(DQK))
    assert_o_close(out, ref_o, f"O {shape}")
    assert_lse_close(lse, ref_l, f"LSE {shape}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 4), (8, 2), (16, 4), (64, 8)])
def test_dv_gqa_bitwise_equals_expanded_mha(gq, Hq, Hkv):
    q, k, v = _inputs(2, 2, 700, Hq, Hkv, seed=Hq * 10 + Hkv)
    G = Hq // Hkv
    o1, l1 = _run(gq, q, k, v, num_splits=4)
    o2, l2 = _run(gq, q, k.repeat_interleave(G, dim=2).contiguous(), v.repeat_interleave(G, dim=2).contiguous(),
                  num_splits=4)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_equal_head_sizes_route_to_dense(gq):
    """Dqk == Dv runs exactly what gqa_decode_ex runs."""
    q, k, v = gqa_inputs.dense_inputs(1, 2, 2000, 32, 4, 128, seed=21)
    a = gq.gqa_decode_dv(q.cuda(), k.cuda(), v.cuda(), num_splits=5)
    b = gq.gqa_decode_ex(q.cuda(), k.cuda(), v.cuda(), num_splits=5)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_dv_closed_forms(gq):
    """K == 0: LSE = ln(#visible keys) and O = mean of the visible V rows."""
    B, Sq, Skv, Hq, Hkv = 2, 3, 2001, 16, 4
    q, k, v = _inputs(B, Sq, Skv, Hq, Hkv, seed=22)
    out, lse = _run(gq, q, torch.zeros_like(k), v)
    G = Hq // Hkv
    for i in range(Sq):
        nvis = Skv - Sq + 1 + i
        assert torch.allclose(lse[:, :, i].double(), torch.full((B, Hq), math.log(nvis), dtype=torch.float64),
                              atol=1e-3, rtol=0)
        assert_o_close(out[:, i], v[:, :nvis].double().mean(dim=1).repeat_interleave(G, dim=1), "zero-K mean")


def test_dv_single_key_exact(gq):
    q, k, v = _inputs(3, 1, 1, 16, 4, seed=23)
    out, lse = _run(gq, q, k, v)
    assert torch.equal(out, v.repeat_interleave(4, dim=2))
    s0 = (q.double() * k.double().repeat_interleave(4, dim=2)).sum(-1) / math.sqrt(DQK)
    assert torch.allclose(lse.double(), s0.permute(0, 2, 1), atol=1e-4, rtol=0)


def test_dv_short_last_split_fully_masked(gq, orc):
    for (Sq, Skv, splits) in [(2, 65, 2), (8, 70, 2), (8, 129, 3)]:
        q, k, v = _inputs(1, Sq, Skv, 16, 2, seed=Skv)
        out, lse = _run(gq, q, k, v, num_splits=splits)
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        ref_o, ref_l = orc.gqa_decode_dv(q, k, v, 1 / math.sqrt(DQK))
        assert_o_close(out, ref_o, f"short last split {Sq},{Skv},{splits}")
        assert_lse_close(lse, ref_l)


def test_dv_explicit_scale(gq, orc):
    q, k, v = _inputs(1, 1, 500, 8, 2, seed=24)
    o_def, l_def = _run(gq, q, k, v, scale=None)
    o_exp, l_exp = _run(gq, q, k, v, scale=1 / math.sqrt(DQK))
    assert torch.equal(o_def, o_exp) and torch.equal(l_def, l_exp)
    o3, l3 = _run(gq, q, k, v, scale=0.21)
    ref_o, ref_l = orc.gqa_decode_dv(q, k, v, 0.21)
    assert_o_close(o3, ref_o)
    assert_lse_close(l3, ref_l)


def test_dv_caller_workspace(gq):
    B, Sq, Skv, Hq, Hkv = 1, 2, 2000, 64, 8
    q, k, v = _inputs(B, Sq, Skv, Hq, Hkv, seed=25)
    need = gq.gqa_decode_dv_workspace_bytes(B, Sq, Skv, Hq, Hkv, DQK, DV, 6)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o1, l1 = _run(gq, q, k, v, num_splits=6, workspace=ws)
    o2, l2 = _run(gq, q, k, v, num_splits=6)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(gq.GQAError) as ei:
        gq.gqa_decode_dv(q.cuda(), k.cuda(), v.cuda(), num_splits=6, workspace=small)
    assert ei.value.status == 4


def test_dv_wait_timeout_is_reported_not_hung(gq):
    q, k, v = (t.cuda() for t in _inputs(1, 1, 1000, 8, 2, seed=26))
    gq.gqa_set_wait_limit_ns(50_000_000)
    gq.gqa_debug_set_fault_mode(1)
    try:
        gq.gqa_decode_dv(q, k, v, num_splits=2)
        assert gq.gqa_device_status() == 6
    finally:
        gq.gqa_debug_set_fault_mode(0)
        gq.gqa_set_wait_limit_ns(0)
    out, lse = gq.gqa_decode_dv(q, k, v, num_splits=2)
    assert gq.gqa_device_status() == 0
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("shape", [(1, 1, 409, 8, 1), (1, 2, 5000, 64, 8)], ids=["lanes_whole_cache", "lane_splits"])
def test_dv_key_lanes_wait_timeout_is_reported_not_hung(gq, shape):
    """Forced timeout on the d192x128 key-lane instances (automatic plan); the
    whole-cache one has 6 lanes over 8 stages, so its lanes also take the
    empty-barrier wait for a stage's previous tile."""
    q, k, v = (t.cuda() for t in _inputs(*shape, seed=27))
    gq.gqa_set_wait_limit_ns(50_000_000)
    gq.gqa_debug_set_fault_mode(1)
    try:
        gq.gqa_decode_dv(q, k, v, num_splits=0)
        assert gq.gqa_device_status() == 6
    finally:
        gq.gqa_debug_set_fault_mode(0)
        gq.gqa_set_wait_limit_ns(0)
    out, lse = gq.gqa_decode_dv(q, k, v, num_splits=0)
    assert gq.gqa_device_status() == 0
    assert torch.isfinite(out.float()).all()


FULL = [c for c in gqa_inputs.CONFIGS.values() if isinstance(c, gqa_inputs.DenseConfig) and c.dv != c.D]


@pytest.mark.slow
@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_dv_full_size_sampled_rows(gq, orc, cfg):
    """Full size, automatic splits (the benchmark's launch): sampled (batch,
    KV head) groups checked against the oracle on that group's slice."""
    q, k, v = gqa_inputs.dense_config_inputs(cfg, device="cuda")
    out, lse = gq.gqa_decode_dv(q, k, v)
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
        ref_o, ref_l = orc.gqa_decode_dv(qs, ks, vs, cfg.scale)
        got_o = out[b:b + 1, :, g * G:(g + 1) * G].cpu()
        got_l = lse[b:b + 1, g * G:(g + 1) * G].cpu()
        assert_o_close(got_o, ref_o, f"{cfg.name} b={b} g={g}")
        assert_lse_close(got_l, ref_l, f"{cfg.name} b={b} g={g}")
        print(cfg.name, b, g, diagnostics(got_o, ref_o))
