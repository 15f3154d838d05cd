#!/usr/bin/env python3
"""Benchmark of the GB300 grouped-query decode attention library.

One step = one decode call over the configuration's whole synthetic KV cache
(the dense path: split kernel + LSE combine; or the sparse paged FP8 path),
with inputs resident in HBM and the L2 flushed (a memset larger than L2)
before every step.  Prints one JSON line on rank 0.

Metric: KV-cache HBM GB/s on K/V bytes read once, with the byte model of
"Attention Kernel Portability Across GPU Architectures", section "Decode"
(2 * B * Hkv * N * D * bytes per element), plus us per call.

  python bench.py [--gpus N --steps K --warmup W] [--config NAME] [--impl gqa|reference]

--impl reference times the fp64 CPU oracle (the only reference this project
has) on the host cores, on the same workload and metric.  Under torchrun
(N > 1) each rank runs an independent replica of the workload (the path needs
no collective); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gqa_inputs  # noqa: E402

METRIC = "GQA decode µs/call and KV-cache HBM GB/s (% of measured GB300 peak)"
FALLBACK_HBM_GBS = 6800.0
# Every source of the library: the kernels, and the host code that picks the
# kernel, its grid and its split count for a shape (all of which set the DRAM
# traffic a recorded capture stands for).
KERNEL_SOURCES = sorted(n for n in os.listdir(os.path.join(ROOT, "gqa_decode_attention_gb300", "csrc"))
                        if n.endswith((".cu", ".cuh", ".h")))


# ---------------------------------------------------------------------------
# host-side accounting (unit-tested on CPU)
# ---------------------------------------------------------------------------
def kv_bytes(B: int, Hkv: int, N: int, D: int, bytes_per_elem: int) -> int:
    """K and V bytes of one decode step, each byte counted once."""
    return 2 * B * Hkv * N * D * bytes_per_elem


def dense_flops(B, Hq, Sq, Skv, D, Dv=None) -> int:
    """Score and P.V products: 2 flops per multiply-add, D (score) + Dv
    (value) dims per key, every key counted for every query row."""
    return 2 * B * Hq * Sq * Skv * (D + (D if Dv is None else Dv))


def paged_flops(B, Hq, topk, D) -> int:
    return 4 * B * topk * Hq * D


def paged_kv_lens(cfg) -> list[int]:
    return [int(x) for x in gqa_inputs.paged_kv_seq_lens(cfg.B, cfg.Sq, cfg.pages_per_req * cfg.page_size, cfg.seed)]


def workload_kv_bytes(cfg) -> int:
    if isinstance(cfg, gqa_inputs.DenseConfig):
        # K rows of D dims and V rows of Dv dims (kv_bytes counts 2 x D per key)
        return cfg.B * cfg.Hkv * cfg.Skv * (cfg.D + cfg.dv) * 2
    if isinstance(cfg, gqa_inputs.PagedKVConfig):
        elem = 2 if cfg.kv_dtype == "bf16" else 1
        return sum(kv_bytes(1, cfg.Hkv, n, cfg.D, elem) for n in paged_kv_lens(cfg))
    return kv_bytes(cfg.B, cfg.Hkv, cfg.topk, cfg.D, 1)


def workload_flops(cfg) -> int:
    if isinstance(cfg, gqa_inputs.DenseConfig):
        return dense_flops(cfg.B, cfg.Hq, cfg.Sq, cfg.Skv, cfg.D, cfg.dv)
    if isinstance(cfg, gqa_inputs.PagedKVConfig):
        return sum(dense_flops(1, cfg.Hq, cfg.Sq, n, cfg.D) for n in paged_kv_lens(cfg))
    return paged_flops(cfg.B, cfg.Hq, cfg.topk, cfg.D)


def workload_config(cfg) -> dict:
    if isinstance(cfg, gqa_inputs.DenseConfig):
        c = {"workload": cfg.name, "B": cfg.B, "Sq": cfg.Sq, "Skv": cfg.Skv, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
             "D": cfg.D, "kv_dtype": "bf16", "mask": "bottom-right causal" if cfg.Sq > 1 else "none"}
        if cfg.dv != cfg.D:
            c["Dv"] = cfg.dv
        return c
    if isinstance(cfg, gqa_inputs.PagedKVConfig):
        lens = paged_kv_lens(cfg)
        cap = cfg.pages_per_req * cfg.page_size
        return {"workload": cfg.name, "B": cfg.B, "Sq": cfg.Sq, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "D": cfg.D,
                "page_size": cfg.page_size, "pages_per_req": cfg.pages_per_req, "num_pages": cfg.num_pages,
                "seq_lens": f"uniform in [{max(cfg.Sq, cap // 2)}, {cap}], total {sum(lens)} tokens",
                "kv_dtype": {"bf16": "bf16", "fp8": "fp8_e4m3fn", "int8": "int8"}[cfg.kv_dtype]}
    return {"workload": cfg.name, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "D": cfg.D,
            "page_size": cfg.page_size, "pages_per_req": cfg.pages_per_req, "num_pages": cfg.num_pages,
            "topk": cfg.topk, "kv_dtype": "fp8_e4m3fn"}


def workload_dtype(cfg) -> str:
    if isinstance(cfg, gqa_inputs.DenseConfig) or (isinstance(cfg, gqa_inputs.PagedKVConfig) and cfg.kv_dtype == "bf16"):
        return "bf16"
    if isinstance(cfg, gqa_inputs.PagedKVConfig) and cfg.kv_dtype == "int8":
        return "int8 kv, bf16 q/out, f16 mma"
    if workload_kernel(cfg) == "gqa_paged_umma_kernel":
        return "fp8_e4m3fn kv, bf16 q/out, e4m3 mma (q and p as two e4m3 terms)"
    return "fp8_e4m3fn kv, bf16 q/out, f16 mma"


def workload_kernel(cfg) -> str:
    if isinstance(cfg, gqa_inputs.DenseConfig):
        import gqa_decode_attention_gb300 as gq
        eng = gq.gqa_decode_dense_engine(cfg.B, cfg.Sq, cfg.Skv, cfg.Hq, cfg.Hkv, cfg.D, cfg.dv)
        return "gqa_dense_umma_kernel" if eng == "tcgen05" else "gqa_dense_split_kernel"
    import gqa_decode_attention_gb300 as gq
    if isinstance(cfg, gqa_inputs.PagedKVConfig):
        kvd = {"bf16": 0, "fp8": 1, "int8": 2}[cfg.kv_dtype]
        eng = gq.gqa_decode_paged_engine(cfg.B, cfg.Sq, cfg.Hq, cfg.Hkv, cfg.D, kvd)
    else:
        eng = gq.gqa_decode_paged_engine(cfg.B, 1, cfg.Hq, cfg.Hkv, cfg.D, 1, topk_form=True)
    return "gqa_paged_umma_kernel" if eng == "tcgen05" else "gqa_paged_kernel"


def gbs(nbytes: float, ms: float) -> float:
    return nbytes / (ms * 1e-3) / 1e9


def percentile(xs, p):
    xs = sorted(xs)
    if not xs:
        return float("nan")
    k = (len(xs) - 1) * p / 100.0
    lo, hi = math.floor(k), math.ceil(k)
    return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)


def parse_clocks(csv_text: str) -> dict | None:
    """Summary of `nvidia-smi --query-gpu=... --format=csv -lms` samples."""
    lines = [ln.strip() for ln in csv_text.strip().splitlines() if ln.strip()]
    if len(lines) < 2:
        return None
    hdr = [h.strip() for h in lines[0].split(",")]
    rows = [[c.strip() for c in ln.split(",")] for ln in lines[1:] if not ln.startswith("index")]
    rows = [r for r in rows if len(r) == len(hdr)]
    if not rows:
        return None

    def col(name):
        for i, h in enumerate(hdr):
            if h.startswith(name):
                return i
        return None

    ism, imax, ipow = col("clocks.current.sm") or col("clocks.sm"), col("clocks.max.sm"), col("power.draw")

    def num(s):
        try:
            return float(s.split()[0])
        except (ValueError, IndexError):
            return float("nan")

    sm = [num(r[ism]) for r in rows] if ism is not None else []
    mx = [num(r[imax]) for r in rows] if imax is not None else []
    pw = [num(r[ipow]) for r in rows] if ipow is not None else []
    # samples under load: power above the midpoint of the observed range
    if pw and max(pw) > min(pw):
        thr = 0.5 * (max(pw) + min(pw))
        loaded = [s for s, p in zip(sm, pw) if p >= thr]
    else:
        loaded = sm
    reasons = set()
    for i, h in enumerate(hdr):
        if h.startswith("clocks_event_reasons.") and h != "clocks_event_reasons.active":
            if any(r[i].lower().startswith("active") for r in rows):
                reasons.add(h.split(".", 1)[1].split(" ")[0])
    return {"sm_mhz": statistics.median(loaded) if loaded else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded)}


def measured_hbm_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gqa_decode_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str) -> float | None:
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash():
        return None
    return float(ent["dram_bytes_per_launch"])


def reduce_over_ranks(values: list[float], op: str = "max") -> list[float]:
    """Element-wise reduction across torch.distributed ranks (identity at N=1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return t.cpu().tolist()


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            # The sampler's start-up (its first query of the device) disturbs a
            # step that overlaps it: let it write its first sample before the
            # timed region begins.
            deadline = time.monotonic() + 5.0
            while time.monotonic() < deadline and self.proc.poll() is None:
                with open(self.path) as f:
                    if len(f.read().splitlines()) >= 2:
                        break
                time.sleep(0.05)
            time.sleep(0.1)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return None
        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)
        return parse_clocks(text)


# ---------------------------------------------------------------------------
# the library arm
# ---------------------------------------------------------------------------
def _dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def _barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def _make_call(gq, cfg, dev, seed_offset):
    import torch
    if isinstance(cfg, gqa_inputs.DenseConfig):
        q, k, v = gqa_inputs.dense_inputs(cfg.B, cfg.Sq, cfg.Skv, cfg.Hq, cfg.Hkv, cfg.D,
                                          cfg.seed + seed_offset, device=dev, Dv=cfg.dv)
        out = torch.empty((cfg.B, cfg.Sq, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((cfg.B, cfg.Hq, cfg.Sq), dtype=torch.float32, device=dev)
        if cfg.dv == cfg.D:
            def call():
                gq.gqa_decode(q, k, v, out=out, lse=lse)
        else:
            def call():
                gq.gqa_decode_dv(q, k, v, out=out, lse=lse)
        splits = gq.gqa_decode_dv_num_splits(cfg.B, cfg.Sq, cfg.Skv, cfg.Hq, cfg.Hkv, cfg.D, cfg.dv)
        return call, dict(q=q, k=k, v=v, out=out, lse=lse), (2 if splits > 1 else 1), splits
    if isinstance(cfg, gqa_inputs.PagedKVConfig):
        inp = gqa_inputs.paged_kv_inputs(cfg.B, cfg.Sq, cfg.Hq, cfg.Hkv, cfg.D, cfg.page_size, cfg.pages_per_req,
                                         cfg.num_pages, cfg.seed + seed_offset, cfg.kv_dtype,
                                         seq_lens=paged_kv_lens(cfg), device=dev)
        out = torch.empty_like(inp["q"])
        lse = torch.empty((cfg.B, cfg.Hq, cfg.Sq), dtype=torch.float32, device=dev)

        def call():
            gq.gqa_decode_paged(inp["q"], inp["k_pool"], inp["v_pool"], inp["page_table"], inp["seq_lens"],
                                inp["k_scale"], inp["v_scale"], out=out, lse=lse)
        splits = gq.gqa_decode_paged_num_splits(cfg.B, cfg.Sq, cfg.Hq, cfg.Hkv, cfg.D,
                                                {"bf16": 0, "fp8": 1, "int8": 2}[cfg.kv_dtype], cfg.page_size,
                                                cfg.pages_per_req)
        return call, dict(inp, out=out, lse=lse), (2 if splits > 1 else 1), splits
    inp = gqa_inputs.paged_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.page_size, cfg.pages_per_req,
                                  cfg.num_pages, cfg.topk, cfg.seed + seed_offset, device=dev)
    out = torch.empty_like(inp["q"])
    lse = torch.empty((cfg.B, cfg.Hq), dtype=torch.float32, device=dev)

    def call():
        gq.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["page_table"],
                                inp["topk"], inp["k_scale"], inp["v_scale"], out=out, lse=lse)
    return call, dict(inp, out=out, lse=lse), 1, 1


def _copy_peak_gbs(dev) -> float:
    """Device-to-device copy bandwidth (read + write bytes) of a 2 GiB copy,
    best of 5, measured in this run."""
    import torch
    n = 1 << 30
    a = torch.empty(n, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    best = 0.0
    for _ in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, gbs(2 * a.numel() * a.element_size(), e0.elapsed_time(e1)))
    del a, b
    torch.cuda.empty_cache()
    return best


def _read_peak_gbs(gq, dev) -> float:
    """Read-only stream bandwidth of this run: the library's read-stream hook
    over 4 GiB (bytes read / time), best of 5.  A decode kernel only reads its
    K/V, so this is the denominator that matches its traffic; the copy peak
    (read + write) is the one the benchmark configuration quotes, and a
    read-only stream can exceed it."""
    import torch
    a = torch.ones(1 << 30, dtype=torch.float32, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    best = 0.0
    for _ in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gq.gqa_debug_read_stream(a, sink)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, gbs(a.numel() * a.element_size(), e0.elapsed_time(e1)))
    del a, sink
    torch.cuda.empty_cache()
    return best


def _cpu_baseline(cfg, tensors, max_seconds=30.0, min_seconds=10.0) -> dict:
    """The fp64 oracle, as it stands, on this host's cores: the full workload
    repeated until min_seconds (or a row subset when one pass would exceed
    max_seconds)."""
    import oracle
    orc = oracle.load()
    if isinstance(cfg, gqa_inputs.DenseConfig):
        q, k, v = (tensors[n].cpu() for n in ("q", "k", "v"))
        nrows = cfg.B * cfg.Hq * cfg.Sq
        t0 = time.perf_counter()
        dense_oracle(orc, cfg, q, k, v, rows=list(range(min(nrows, 8))))
        per_row = (time.perf_counter() - t0) / min(nrows, 8)
        rows = None if per_row * nrows <= max_seconds else list(range(max(1, int(max_seconds / 3 / per_row))))
        frac = 1.0 if rows is None else len(rows) / nrows
        reps, elapsed = 0, 0.0
        while elapsed < min_seconds and reps < 1000:
            t0 = time.perf_counter()
            dense_oracle(orc, cfg, q, k, v, rows=rows)
            elapsed += time.perf_counter() - t0
            reps += 1
        sample = (f"{'all' if rows is None else len(rows)} of {nrows} query rows "
                  f"(the rows of whole KV-head groups), {reps} pass(es)")
    elif isinstance(cfg, gqa_inputs.PagedKVConfig):
        cpu = {n: (t.cpu() if hasattr(t, "cpu") else t) for n, t in tensors.items()}
        res = _paged_kv_oracle_timing(orc, cfg, cpu, max_seconds, min_seconds)
        return dict(res, nproc=os.cpu_count(), cpu_model=cpu_model(),
                    single_thread=_single_thread_baseline(orc, cfg, cpu))
    else:
        cpu = {n: (t.cpu() if hasattr(t, "cpu") else t) for n, t in tensors.items()}
        nrows = cfg.B * cfg.Hq
        t0 = time.perf_counter()
        orc.gqa_decode_paged_fp8(cpu["q"], cpu["gate"], cpu["k_pool"], cpu["v_pool"], cpu["page_table"],
                                 cpu["topk"], cpu["k_scale"], cpu["v_scale"], cfg.scale, rows=list(range(64)))
        per_row = (time.perf_counter() - t0) / 64
        rows = None if per_row * nrows <= max_seconds else list(range(int(max_seconds / 3 / per_row)))
        frac = 1.0 if rows is None else len(rows) / nrows
        reps, elapsed = 0, 0.0
        while elapsed < min_seconds and reps < 1000:
            t0 = time.perf_counter()
            orc.gqa_decode_paged_fp8(cpu["q"], cpu["gate"], cpu["k_pool"], cpu["v_pool"], cpu["page_table"],
                                     cpu["topk"], cpu["k_scale"], cpu["v_scale"], cfg.scale, rows=rows)
            elapsed += time.perf_counter() - t0
            reps += 1
        sample = f"{'all' if rows is None else len(rows)} of {nrows} (request, head) rows, {reps} pass(es)"
    per_pass = elapsed / reps
    cpu = {"q": q, "k": k, "v": v} if isinstance(cfg, gqa_inputs.DenseConfig) else cpu
    # KV bytes in proportion to the rows covered (every row reads its group's K/V)
    return {"value": gbs(workload_kv_bytes(cfg) * frac, per_pass * 1e3), "unit": "GB/s",
            "cores": orc.num_threads(), "kind": "oracle", "sample": sample,
            "us_per_call_equiv": per_pass / frac * 1e6, "nproc": os.cpu_count(), "cpu_model": cpu_model(),
            "single_thread": _single_thread_baseline(orc, cfg, cpu)}


def dense_oracle(orc, cfg, q, k, v, rows=None):
    """The oracle's dense decode for a dense workload (Dqk != Dv included)."""
    if cfg.dv == cfg.D:
        return orc.gqa_decode(q, k, v, cfg.scale, rows=rows)
    return orc.gqa_decode_dv(q, k, v, cfg.scale, rows=rows)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _single_thread_baseline(orc, cfg, cpu, seconds=1.5) -> dict:
    """The oracle on one host thread over the first rows of the workload,
    repeated for about `seconds`; bytes credited as in the multi-thread leg."""
    threads = orc.num_threads()
    orc.set_num_threads(1)
    try:
        if isinstance(cfg, gqa_inputs.DenseConfig):
            nrows = cfg.B * cfg.Hq * cfg.Sq
            rows = list(range(min(nrows, 4)))
            run = lambda: dense_oracle(orc, cfg, cpu["q"], cpu["k"], cpu["v"], rows=rows)  # noqa: E731
            credit = workload_kv_bytes(cfg) * len(rows) / nrows
        elif isinstance(cfg, gqa_inputs.PagedKVConfig):
            lens = [int(x) for x in cpu["seq_lens"]]
            elem = 2 if cfg.kv_dtype == "bf16" else 1
            G = cfg.Hq // cfg.Hkv
            rows = [0, 1]
            run = lambda: orc.gqa_decode_paged(cpu["q"], cpu["k_pool"], cpu["v_pool"], cpu["page_table"],  # noqa: E731
                                               cpu["seq_lens"], cfg.scale, cpu["k_scale"], cpu["v_scale"], rows=rows)
            credit = sum(2 * lens[r // (cfg.Hq * cfg.Sq)] * cfg.D * elem / (G * cfg.Sq) for r in rows)
        else:
            nrows = cfg.B * cfg.Hq
            rows = list(range(16))
            run = lambda: orc.gqa_decode_paged_fp8(cpu["q"], cpu["gate"], cpu["k_pool"], cpu["v_pool"],  # noqa: E731
                                                   cpu["page_table"], cpu["topk"], cpu["k_scale"], cpu["v_scale"],
                                                   cfg.scale, rows=rows)
            credit = workload_kv_bytes(cfg) * len(rows) / nrows
        reps, elapsed = 0, 0.0
        while elapsed < seconds and reps < 1000:
            t0 = time.perf_counter()
            run()
            elapsed += time.perf_counter() - t0
            reps += 1
    finally:
        orc.set_num_threads(threads)
    return {"value": gbs(credit, elapsed / reps * 1e3), "unit": "GB/s", "cores": 1,
            "sample": f"{len(rows)} query rows, {reps} pass(es)"}


def _paged_kv_oracle_timing(orc, cfg, cpu, max_seconds, min_seconds) -> dict:
    """The oracle on whole-request paged inputs: rows of request 0 first (a
    row sample when a pass would exceed max_seconds); bytes credited per row
    as its share of its request's K/V."""
    lens = [int(x) for x in cpu["seq_lens"]]
    elem = 2 if cfg.kv_dtype == "bf16" else 1
    nrows = cfg.B * cfg.Hq * cfg.Sq
    G = cfg.Hq // cfg.Hkv

    def row_bytes(r):  # row r = (b*Hq + h)*Sq + i reads 1/(G*Sq) of its KV head's bytes
        b = r // (cfg.Hq * cfg.Sq)
        return 2 * lens[b] * cfg.D * elem / (G * cfg.Sq)

    def run(rows):
        orc.gqa_decode_paged(cpu["q"], cpu["k_pool"], cpu["v_pool"], cpu["page_table"], cpu["seq_lens"],
                             cfg.scale, cpu["k_scale"], cpu["v_scale"], rows=rows)

    t0 = time.perf_counter()
    run(list(range(8)))
    per_row = (time.perf_counter() - t0) / 8
    rows = None if per_row * nrows <= max_seconds else list(range(max(1, int(max_seconds / 3 / per_row))))
    covered = sum(row_bytes(r) for r in (range(nrows) if rows is None else rows))
    reps, elapsed = 0, 0.0
    while elapsed < min_seconds and reps < 1000:
        t0 = time.perf_counter()
        run(rows)
        elapsed += time.perf_counter() - t0
        reps += 1
    per_pass = elapsed / reps
    sample = f"{'all' if rows is None else len(rows)} of {nrows} query rows, {reps} pass(es)"
    return {"value": gbs(covered, per_pass * 1e3), "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
            "sample": sample, "seconds_per_pass": per_pass, "bytes_covered": covered}


def run_gqa(args) -> int:
    import torch
    world, rank, local = _dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from gqa_decode_attention_gb300 import build as gbuild
    if rank == 0:
        gbuild.build()
    _barrier()
    import gqa_decode_attention_gb300 as gq
    gq.load_library()
    cfg = gqa_inputs.CONFIGS[args.config]
    nbytes = workload_kv_bytes(cfg)
    peak, peak_kind = measured_hbm_peak()

    copy_peak = _copy_peak_gbs(dev)
    read_peak = _read_peak_gbs(gq, dev)
    call, tensors, launches_per_call, splits = _make_call(gq, cfg, dev, seed_offset=rank)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_bytes = max(512 << 20, 4 * l2)
    flush_w = torch.empty(flush_bytes, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(flush_bytes // 8, dtype=torch.int64, device=dev)

    def flush_l2():
        # Write a buffer larger than L2, then read another one: L2 is left
        # holding clean lines only, so the timed step neither hits in L2 nor
        # pays for write-backs of the flush's own dirty lines.
        flush_w.zero_()
        flush_r.sum()

    def step_events(n, hook=False):
        times, ktimes = [], []
        for _ in range(n):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if hook:
                k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                # record once from torch so it treats them as recorded; the
                # library re-records both around its kernel (latest record wins)
                k0.record()
                k1.record()
                gq.gqa_debug_set_kernel_events(k0, k1)
            e0.record()
            call()
            e1.record()
            if hook:
                gq.gqa_debug_set_kernel_events(None, None)
                ktimes.append((k0, k1))
            times.append((e0, e1))
        torch.cuda.synchronize()
        return ([a.elapsed_time(b) for a, b in times], [a.elapsed_time(b) for a, b in ktimes])

    for _ in range(args.warmup):
        flush_l2()
        call()
    torch.cuda.synchronize()
    if gq.gqa_device_status() != 0:
        raise RuntimeError("device error during warm-up")

    # ---- timed region: exactly K steps.  The clock sampler starts first (the
    # GPU idles while it comes up), then two more untimed steps bring the
    # clocks back before the barrier + synchronize that open the region.
    with ClockSampler(local) as clk:
        for _ in range(2):
            flush_l2()
            call()
        _barrier()
        torch.cuda.synchronize()
        step_ms, _ = step_events(args.steps)
        torch.cuda.synchronize()
        _barrier()
    clocks = clk.summary()
    total_ms = sum(step_ms)
    (max_total_ms,) = reduce_over_ranks([total_ms], "max")
    if gq.gqa_device_status() != 0:
        raise RuntimeError("device error in the timed region")

    # ---- dominant kernel alone (split kernel / paged kernel), same workload
    _, kern_ms = step_events(args.steps, hook=True)
    kern_avg = statistics.mean(kern_ms)

    # ---- end to end through the host-buffer entry point (dense path)
    e2e = None
    if not args.no_e2e and isinstance(cfg, gqa_inputs.DenseConfig) and cfg.dv != cfg.D:
        # no host-buffer entry point for this flavour: pinned host -> device
        # copies, the device call and the device -> host copies of out / lse,
        # all inside the timed call
        qh, kh, vh = (tensors[n].cpu().pin_memory() for n in ("q", "k", "v"))
        oh = torch.empty(tuple(tensors["out"].shape), dtype=torch.bfloat16).pin_memory()
        lh = torch.empty(tuple(tensors["lse"].shape), dtype=torch.float32).pin_memory()
        qd, kd, vd = (torch.empty_like(t, device=dev) for t in (qh, kh, vh))
        od, ld = torch.empty_like(oh, device=dev), torch.empty_like(lh, device=dev)

        def e2e_call():
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            gq.gqa_decode_dv(qd, kd, vd, out=od, lse=ld)
            oh.copy_(od, non_blocking=True)
            lh.copy_(ld, non_blocking=True)
            torch.cuda.current_stream().synchronize()
        e2e_call()  # warm-up
        ts = []
        for _ in range(max(1, args.e2e_steps)):
            t0 = time.perf_counter()
            e2e_call()
            ts.append((time.perf_counter() - t0) * 1e3)
        (e2e_ms,) = reduce_over_ranks([statistics.mean(ts)], "max")
        e2e = {"value": gbs(world * nbytes, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": (qh.numel() + kh.numel() + vh.numel()) * 2,
               "d2h_bytes_per_step": oh.numel() * 2 + lh.numel() * 4,
               "api": "gqa_decode_dv with pinned host copies in the timed call"}
        del qh, kh, vh, oh, lh, qd, kd, vd, od, ld
    elif not args.no_e2e and isinstance(cfg, gqa_inputs.DenseConfig):
        qh = tensors["q"].cpu().pin_memory()
        kh = tensors["k"].cpu().pin_memory()
        vh = tensors["v"].cpu().pin_memory()
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty(tuple(tensors["lse"].shape), dtype=torch.float32).pin_memory()
        gq.gqa_decode_host(qh, kh, vh, oh, lh)  # warm-up
        ts = []
        for _ in range(max(1, args.e2e_steps)):
            t0 = time.perf_counter()
            gq.gqa_decode_host(qh, kh, vh, oh, lh)
            ts.append((time.perf_counter() - t0) * 1e3)
        (e2e_ms,) = reduce_over_ranks([statistics.mean(ts)], "max")
        e2e = {"value": gbs(world * nbytes, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": qh.numel() * 2 + kh.numel() * 2 + vh.numel() * 2,
               "d2h_bytes_per_step": oh.numel() * 2 + lh.numel() * 4,
               "api": "gqa_decode_host (pinned host buffers, copies inside the timed call)"}
        del qh, kh, vh, oh, lh

    cpu_base = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        cpu_base = _cpu_baseline(cfg, tensors)

    if rank == 0:
        us = [t * 1e3 for t in step_ms]
        value = gbs(world * args.steps * nbytes, max_total_ms)
        achieved = gbs(nbytes, kern_avg)
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(max_total_ms / args.steps, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": workload_dtype(cfg),
            "data": "synthetic (seeded N(0,1), generated on the device)",
            "config": dict(workload_config(cfg),
                           l2=f"flushed before every step: {flush_bytes >> 20} MiB written, then {flush_bytes >> 20} MiB read",
                           splits=splits, parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
            "us_per_call": {"median": round(statistics.median(us), 2), "p10": round(percentile(us, 10), 2),
                            "p90": round(percentile(us, 90), 2)},
            "kv_bytes_per_call": nbytes,
            "flops_per_call": workload_flops(cfg),
            "tflops": round(world * workload_flops(cfg) / (max_total_ms / args.steps * 1e-3) / 1e12, 2),
            "frac_of_peak": round(value / world / peak, 4),
            "peak_gbs": peak, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback",
            "copy_peak_gbs_this_run": round(copy_peak, 1),
            "frac_of_copy_peak_this_run": round(value / world / copy_peak, 4),
            "read_peak_gbs_this_run": round(read_peak, 1),
            "frac_of_read_peak_this_run": round(value / world / read_peak, 4),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": recorded_traffic(cfg.name),
                         "kernel": workload_kernel(cfg),
                         "kernel_us": round(kern_avg * 1e3, 2),
                         "algorithmic_bytes_per_launch": nbytes,
                         "read_peak_this_run": round(read_peak, 1),
                         "frac_of_read_peak_this_run": round(achieved / read_peak, 4)},
            "cpu_baseline": cpu_base,
            "e2e": e2e,
            "gpu_launches": args.steps * launches_per_call,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args) -> int:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    import oracle
    orc = oracle.load()
    cfg = gqa_inputs.CONFIGS[args.config]
    nbytes = workload_kv_bytes(cfg)
    if isinstance(cfg, gqa_inputs.DenseConfig):
        q, k, v = gqa_inputs.dense_config_inputs(cfg, device="cpu")
        nrows = cfg.B * cfg.Hq * cfg.Sq
        t0 = time.perf_counter()
        dense_oracle(orc, cfg, q, k, v, rows=list(range(min(8, nrows))))
        per_row = (time.perf_counter() - t0) / min(8, nrows)
        budget_s = 150.0 / max(1, args.steps + args.warmup)   # whole run within a few minutes
        rows = None if per_row * nrows <= budget_s else list(range(max(1, int(budget_s / per_row))))

        def step():
            dense_oracle(orc, cfg, q, k, v, rows=rows)
    elif isinstance(cfg, gqa_inputs.PagedKVConfig):
        inp = gqa_inputs.paged_kv_config_inputs(cfg, device="cpu")
        budget_s = 150.0 / max(1, args.steps + args.warmup)
        probe = _paged_kv_oracle_timing(orc, cfg, inp, max_seconds=budget_s, min_seconds=0.0)
        ts = []
        for _ in range(args.steps):
            r = _paged_kv_oracle_timing(orc, cfg, inp, max_seconds=budget_s, min_seconds=0.0)
            ts.append(r["seconds_per_pass"] * 1e3)
        total = sum(ts)
        value = gbs(args.steps * probe["bytes_covered"], total)
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), CPU)",
            "config": workload_config(cfg), "impl": "reference",
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
                             "nproc": os.cpu_count(), "cpu_model": cpu_model(),
                             "sample": probe["sample"] + " per step"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return 0
    else:
        inp = gqa_inputs.paged_config_inputs(cfg, device="cpu")
        nrows = cfg.B * cfg.Hq
        t0 = time.perf_counter()
        orc.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["page_table"],
                                 inp["topk"], inp["k_scale"], inp["v_scale"], cfg.scale, rows=list(range(64)))
        per_row = (time.perf_counter() - t0) / 64
        budget_s = 150.0 / max(1, args.steps + args.warmup)
        rows = None if per_row * nrows <= budget_s else list(range(max(1, int(budget_s / per_row))))

        def step():
            orc.gqa_decode_paged_fp8(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["page_table"],
                                     inp["topk"], inp["k_scale"], inp["v_scale"], cfg.scale, rows=rows)
    frac = 1.0 if rows is None else len(rows) / nrows
    for _ in range(args.warmup):
        step()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        ts.append((time.perf_counter() - t0) * 1e3)
    total = sum(ts)
    value = gbs(args.steps * nbytes * frac, total)
    sample = f"{'all' if rows is None else len(rows)} of {nrows} rows of the workload per step"
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), CPU)",
        "config": workload_config(cfg), "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
                             "nproc": os.cpu_count(), "cpu_model": cpu_model(),
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_latency_grid(args) -> int:
    """Small-cache decode latency over the grid the portability study measured
    (32/8 heads, d 128, bf16, Sq 1; batch 1 .. 64 x KV length 512 .. 16384):
    per cell the automatic split count, device time per call (CUDA events,
    L2 flushed, median of 20), and host time per call back to back, eager
    and replayed from a captured CUDA graph.  One JSON line per cell."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from gqa_decode_attention_gb300 import build as gbuild
    gbuild.build()
    import gqa_decode_attention_gb300 as gq
    gq.load_library()
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones((512 << 20) // 8, dtype=torch.int64, device=dev)

    def device_us(fn, n=20):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(n):
            flush_w.zero_()
            flush_r.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    def host_us(fn, n=200):
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n * 1e6

    Hq, Hkv, D = 32, 8, 128
    for B in (1, 4, 8, 16, 32, 64):
        for N in (512, 2048, 8192, 16384):
            q, k, v = gqa_inputs.dense_inputs(B, 1, N, Hq, Hkv, D, 7, device=dev)
            out = torch.empty_like(q)
            lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=dev)

            def call():
                gq.gqa_decode(q, k, v, out=out, lse=lse)
            d_us = device_us(call)
            h_eager = host_us(call)
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                call()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    call()
            torch.cuda.current_stream().wait_stream(side)
            h_graph = host_us(g.replay)
            nbytes = kv_bytes(B, Hkv, N, D, 2)
            print(json.dumps({"B": B, "N": N, "Hq": Hq, "Hkv": Hkv, "D": D,
                              "splits": gq.gqa_decode_num_splits(B, 1, N, Hq, Hkv, D),
                              "device_us": round(d_us, 2), "gbs": round(gbs(nbytes, d_us * 1e-3), 1),
                              "host_us_eager": round(h_eager, 2), "host_us_graph": round(h_graph, 2)}), flush=True)
            del q, k, v, out, lse, g
    return 0


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["gqa", "reference"], default="gqa")
    p.add_argument("--config", default=gqa_inputs.HEADLINE, choices=sorted(gqa_inputs.CONFIGS))
    p.add_argument("--skv", type=int, default=0,
                   help="override the KV length of a dense configuration (smaller cases for profiling)")
    p.add_argument("--sq", type=int, default=0,
                   help="override the decode rows per query head of a dense configuration (row-count sweeps)")
    p.add_argument("--pages-per-req", type=int, default=0,
                   help="override the page-table length of a whole-request paged configuration (smaller pools "
                        "for profiling)")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--latency-grid", action="store_true",
                   help="small-cache latency sweep (eager and CUDA graph) instead of the benchmark line")
    args = p.parse_args(argv)
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 untimed warm-up steps
    if args.skv or args.sq:
        import dataclasses
        cfg = gqa_inputs.CONFIGS[args.config]
        if not isinstance(cfg, gqa_inputs.DenseConfig):
            p.error("--skv and --sq apply to dense configurations only")
        name = cfg.name + (f"@skv{args.skv}" if args.skv else "") + (f"@sq{args.sq}" if args.sq else "")
        gqa_inputs.CONFIGS[name] = dataclasses.replace(cfg, name=name, Skv=args.skv or cfg.Skv, Sq=args.sq or cfg.Sq)
        args.config = name
    if args.pages_per_req:
        import dataclasses
        cfg = gqa_inputs.CONFIGS[args.config]
        if not isinstance(cfg, gqa_inputs.PagedKVConfig):
            p.error("--pages-per-req applies to whole-request paged configurations only")
        name = f"{cfg.name}@ppr{args.pages_per_req}"
        gqa_inputs.CONFIGS[name] = dataclasses.replace(cfg, name=name, pages_per_req=args.pages_per_req)
        args.config = name
    if args.impl == "reference":
        return run_reference(args)
    if args.latency_grid:
        return run_latency_grid(args)
    try:
        return run_gqa(args)
    finally:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
