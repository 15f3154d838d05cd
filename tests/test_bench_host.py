"""Host-side logic of bench.py (CPU only): the byte / FLOP accounting against
figures the pages print, clock parsing, the max-over-ranks reduction on two
gloo ranks, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "byte_model.txt")


def _golden():
    for ln in open(GOLDEN):
        if ln.strip() and not ln.startswith("#"):
            kind, args, val, unit, tol, src = [c.strip() for c in ln.split("|")]
            yield kind, [float(a) for a in args.split()], float(val), float(tol), src


def test_byte_and_flop_model_matches_pages():
    n = 0
    for kind, a, val, tol, src in _golden():
        if kind == "kv_bytes":
            got = bench.kv_bytes(*map(int, a))
        elif kind == "kv_gbs":
            got = bench.gbs(bench.kv_bytes(*map(int, a[:5])), a[5] * 1e-3)
        elif kind == "flops_paged":
            B, Hq, K, D = map(int, a)
            got = bench.paged_flops(B, Hq, K, D)
        elif kind == "tflops_paged":
            B, Hq, K, D = map(int, a[:4])
            got = bench.paged_flops(B, Hq, K, D) / (a[4] * 1e-3) / 1e12
        else:
            raise AssertionError(kind)
        assert abs(got - val) <= tol * abs(val), (kind, a, got, val, src)
        n += 1
    assert n == 7


def test_workload_bytes():
    import gqa_inputs
    c = gqa_inputs.CONFIGS
    assert bench.workload_kv_bytes(c["dense_b1_h64x8_d128_sq2_kv128k"]) == 512 << 20
    assert bench.workload_kv_bytes(c["dense_b32_h64x8_d128_sq1_kv32k"]) == 4 << 30
    assert bench.workload_kv_bytes(c["dense_b8_h32x2_d256_sq8_kv128k"]) == 2 << 30
    assert bench.workload_kv_bytes(c["paged_fp8_b256_h32x8_d128_top512_ps16"]) == 256 << 20
    assert bench.workload_kv_bytes(c["dense_b1_h8x1_d64_sq1_kv1k"]) == 256 << 10
    # 131072 keys x 8 KV heads x (192 K dims + 128 V dims) x 2 bytes
    assert bench.workload_kv_bytes(c["dense_b1_h64x8_d192x128_sq2_kv128k"]) == 640 << 20
    # flops: 4 B Hq Sq Skv D for equal head sizes (8.59 G for the 128K headline)
    assert bench.workload_flops(c["dense_b1_h64x8_d128_sq2_kv128k"]) == 4 * 64 * 2 * 131072 * 128
    assert bench.workload_flops(c["dense_b1_h64x8_d192x128_sq2_kv128k"]) == 2 * 64 * 2 * 131072 * (192 + 128)
    assert bench.workload_flops(c["paged_fp8_b256_h32x8_d128_top512_ps16"]) == 4 * 256 * 512 * 32 * 128


CLOCKS = """index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], clocks_event_reasons.active, clocks_event_reasons.hw_slowdown, clocks_event_reasons.hw_thermal_slowdown, clocks_event_reasons.sw_thermal_slowdown, clocks_event_reasons.sw_power_cap
0, 345 MHz, 2070 MHz, 150.00 W, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active
0, 1965 MHz, 2070 MHz, 900.00 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
0, 1980 MHz, 2070 MHz, 950.00 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active
0, 1950 MHz, 2070 MHz, 940.00 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
"""


def test_workload_kernel_names_the_engine():
    """The roofline's kernel is the engine the library picks (host-only query)."""
    import gqa_inputs
    from gqa_decode_attention_gb300 import build as gbuild
    gbuild.build()
    c = gqa_inputs.CONFIGS
    assert bench.workload_kernel(c["dense_b1_h64x8_d128_sq2_kv128k"]) == "gqa_dense_split_kernel"
    assert bench.workload_kernel(c["dense_b1_h64x8_d128_sq8_kv128k"]) == "gqa_dense_umma_kernel"
    assert bench.workload_kernel(c["dense_b8_h32x2_d256_sq8_kv128k"]) == "gqa_dense_umma_kernel"
    assert bench.workload_kernel(c["dense_b1_h64x8_d192x128_sq2_kv128k"]) == "gqa_dense_split_kernel"
    assert bench.workload_kernel(c["paged_fp8_b256_h32x8_d128_top512_ps16"]) == "gqa_paged_umma_kernel"
    assert bench.workload_kernel(c["paged_fp8_b32_h64x8_d128_kv32k_ps16"]) == "gqa_paged_kernel"  # 8 rows per KV head
    assert bench.workload_kernel(c["paged_bf16_b32_h64x8_d128_kv32k_ps16"]) == "gqa_paged_kernel"
    assert bench.workload_kernel(c["paged_int8_b32_h64x8_d128_kv32k_ps16"]) == "gqa_paged_kernel"
    assert bench.workload_kv_bytes(c["dense_b1_h64x8_d128_sq8_kv128k"]) == 512 << 20


def test_parse_clocks():
    c = bench.parse_clocks(CLOCKS)
    assert c["sm_mhz"] == 1965 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    assert c["samples"] == 4 and c["samples_under_load"] == 3
    assert bench.parse_clocks("") is None


def test_percentile():
    assert bench.percentile([1, 2, 3, 4, 5], 50) == 3
    assert bench.percentile([1, 2], 10) == pytest.approx(1.1)


_RANK_SCRIPT = r"""
import os, sys, json
sys.path.insert(0, os.environ["REPO"])
import torch.distributed as dist
dist.init_process_group("gloo")
import bench
r = dist.get_rank()
out = bench.reduce_over_ranks([10.0 + r, 5.0 - r], "max")
s = bench.reduce_over_ranks([1.0], "sum")
with open(os.path.join(os.environ["OUTDIR"], f"rank{r}.json"), "w") as f:
    json.dump({"rank": r, "max": out, "sum": s}, f)
dist.destroy_process_group()
"""


def test_reduce_over_two_gloo_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(_RANK_SCRIPT)
    env = dict(os.environ, REPO=os.path.dirname(os.path.dirname(os.path.abspath(__file__))), OUTDIR=str(tmp_path))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29613", str(script)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    outs = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    assert len(outs) == 2
    for o in outs:
        assert o["max"] == [11.0, 5.0] and o["sum"] == [2.0]


def test_reference_arm_json(capsys):
    rc = bench.main(["--impl", "reference", "--config", "dense_b1_h8x1_d64_sq1_kv1k", "--steps", "3",
                     "--warmup", "3"])
    assert rc == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["steps"] == 3
    assert line["metric"] == bench.METRIC


def test_cpu_model_and_single_thread_baseline(orc):
    """The CPU baseline names the host CPU and times the oracle on one thread
    (restoring the thread count afterwards)."""
    import gqa_inputs
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
    cfg = gqa_inputs.CONFIGS["dense_b1_h8x1_d64_sq1_kv1k"]
    q, k, v = gqa_inputs.dense_config_inputs(cfg)
    threads = orc.num_threads()
    r = bench._single_thread_baseline(orc, cfg, {"q": q, "k": k, "v": v}, seconds=0.05)
    assert r["cores"] == 1 and r["value"] > 0 and r["unit"] == "GB/s"
    assert orc.num_threads() == threads


def test_size_overrides_reject_the_wrong_form():
    """--skv / --sq shrink dense workloads and --pages-per-req whole-request
    paged ones; each refuses the other form before any device work."""
    with pytest.raises(SystemExit):
        bench.main(["--config", "paged_fp8_b32_h64x8_d128_kv32k_ps16", "--skv", "4096"])
    with pytest.raises(SystemExit):
        bench.main(["--config", "dense_b1_h64x8_d128_sq2_kv128k", "--pages-per-req", "512"])
    with pytest.raises(SystemExit):
        bench.main(["--config", "paged_fp8_b256_h32x8_d128_top512_ps16", "--pages-per-req", "512"])
