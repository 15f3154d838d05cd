"""Seeded synthetic inputs for grouped-query decode attention.

This module only draws random tensors and index tables; it holds none of the
attention arithmetic.  Both the CUDA path (tests, benchmark) and the fp64
oracle consume what it produces, so the two sides always see identical bytes.

Workloads (the shapes the pages measure, scaled to the configurations this
library is benchmarked on):

* dense decode: q [B, Sq, Hq, D], K/V [B, Skv, Hkv, D], all bf16 drawn as
  N(0, 1) in fp32 and rounded to bf16 (round-to-nearest-even);
* sparse paged FP8 decode ("Sparse paged GQA decode attention with FP8 KV
  cache on SM89", section "Workload"): 256 requests, 32/8 heads, d 128, page
  size 16, 32 pages per request drawn as a random permutation of a shared
  pool, top-K = 512 token indices per request (a random permutation of its
  tokens), q and gate bf16 N(0, 1), K/V pools FP8 E4M3FN quantised from
  N(0, 1) with a per-tensor scale amax / 448;
* paged decode over whole requests (the serving layout: no top-K, every
  token of each request up to its own length): q [B, Sq, Hq, D] bf16, K/V
  pools [num_pages, page_size, Hkv, D] in bf16 (N(0, 1) rounded), FP8
  E4M3FN (quantised as above) or int8 (symmetric per-tensor, scale amax/127), each request's pages a random permutation of
  the pool, sequence lengths drawn uniformly from [capacity / 2, capacity]
  (a length mix), or given.
"""
from __future__ import annotations

import dataclasses
import math

import torch

E4M3FN_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class DenseConfig:
    name: str
    B: int
    Sq: int
    Skv: int
    Hq: int
    Hkv: int
    D: int
    seed: int
    Dv: int = 0  # value head size; 0 = D

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def dv(self) -> int:
        return self.Dv or self.D


@dataclasses.dataclass(frozen=True)
class PagedConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    pages_per_req: int
    num_pages: int
    topk: int
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclasses.dataclass(frozen=True)
class PagedKVConfig:
    name: str
    B: int
    Sq: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    pages_per_req: int
    kv_dtype: str  # "bf16", "fp8" or "int8"
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def num_pages(self) -> int:
        return self.B * self.pages_per_req


CONFIGS = {
    "dense_b1_h8x1_d64_sq1_kv1k": DenseConfig(
        "dense_b1_h8x1_d64_sq1_kv1k", B=1, Sq=1, Skv=1024, Hq=8, Hkv=1, D=64, seed=1001),
    "dense_b1_h64x8_d128_sq2_kv128k": DenseConfig(
        "dense_b1_h64x8_d128_sq2_kv128k", B=1, Sq=2, Skv=131072, Hq=64, Hkv=8, D=128, seed=1002),
    "dense_b32_h64x8_d128_sq1_kv32k": DenseConfig(
        "dense_b32_h64x8_d128_sq1_kv32k", B=32, Sq=1, Skv=32768, Hq=64, Hkv=8, D=128, seed=1003),
    "dense_b8_h32x2_d256_sq8_kv128k": DenseConfig(
        "dense_b8_h32x2_d256_sq8_kv128k", B=8, Sq=8, Skv=131072, Hq=32, Hkv=2, D=256, seed=1004),
    # eight decode rows per head (draft tokens verified in one call) on the
    # headline's long-cache shape: 64 query rows per KV head
    "dense_b1_h64x8_d128_sq8_kv128k": DenseConfig(
        "dense_b1_h64x8_d128_sq8_kv128k", B=1, Sq=8, Skv=131072, Hq=64, Hkv=8, D=128, seed=1010),
    # the d192x128 head flavour (scores over 192 dims, values of 128) on the
    # headline's long-cache shape
    "dense_b1_h64x8_d192x128_sq2_kv128k": DenseConfig(
        "dense_b1_h64x8_d192x128_sq2_kv128k", B=1, Sq=2, Skv=131072, Hq=64, Hkv=8, D=192, Dv=128, seed=1009),
    "paged_fp8_b256_h32x8_d128_top512_ps16": PagedConfig(
        "paged_fp8_b256_h32x8_d128_top512_ps16", B=256, Hq=32, Hkv=8, D=128, page_size=16,
        pages_per_req=32, num_pages=8192, topk=512, seed=1005),
    # whole requests through page tables (the serving layout): the batched
    # 32 x 32K shape, page size 16, lengths uniform in [16K, 32K]
    "paged_bf16_b32_h64x8_d128_kv32k_ps16": PagedKVConfig(
        "paged_bf16_b32_h64x8_d128_kv32k_ps16", B=32, Sq=1, Hq=64, Hkv=8, D=128, page_size=16,
        pages_per_req=2048, kv_dtype="bf16", seed=1006),
    "paged_fp8_b32_h64x8_d128_kv32k_ps16": PagedKVConfig(
        "paged_fp8_b32_h64x8_d128_kv32k_ps16", B=32, Sq=1, Hq=64, Hkv=8, D=128, page_size=16,
        pages_per_req=2048, kv_dtype="fp8", seed=1007),
    "paged_int8_b32_h64x8_d128_kv32k_ps16": PagedKVConfig(
        "paged_int8_b32_h64x8_d128_kv32k_ps16", B=32, Sq=1, Hq=64, Hkv=8, D=128, page_size=16,
        pages_per_req=2048, kv_dtype="int8", seed=1008),
}

# The configuration the headline throughput is quoted on: the largest
# single-GPU one, 32 requests x 32K keys, 64 query heads over 8 KV heads,
# d 128, one decode row (4 GiB of K/V).
HEADLINE = "dense_b32_h64x8_d128_sq1_kv32k"


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, g: torch.Generator, device, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """N(0,1) drawn in fp32 then rounded to bf16, in chunks to bound memory."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for off in range(0, n, chunk_elems):
        m = min(chunk_elems, n - off)
        out[off:off + m] = torch.randn(m, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def dense_inputs(B, Sq, Skv, Hq, Hkv, D, seed, device="cpu", Dv=None):
    """q [B,Sq,Hq,D], k [B,Skv,Hkv,D], v [B,Skv,Hkv,Dv] (Dv defaults to D),
    all bf16 ~ N(0,1)."""
    g = _gen(seed, device)
    q = _randn_bf16((B, Sq, Hq, D), g, device)
    k = _randn_bf16((B, Skv, Hkv, D), g, device)
    v = _randn_bf16((B, Skv, Hkv, D if Dv is None else Dv), g, device)
    return q, k, v


def dense_config_inputs(cfg: DenseConfig, device="cpu"):
    return dense_inputs(cfg.B, cfg.Sq, cfg.Skv, cfg.Hq, cfg.Hkv, cfg.D, cfg.seed, device, Dv=cfg.dv)


def quantize_e4m3fn(x: torch.Tensor):
    """Per-tensor FP8 E4M3FN codes of x with scale amax/448 (test data only).

    Returns (codes uint8, scale float).  The cast is torch's own round-to-
    nearest-even conversion after clamping to the format's range.
    """
    amax = float(x.abs().max())
    scale = amax / E4M3FN_MAX if amax > 0 else 1.0
    y = (x / scale).clamp_(-E4M3FN_MAX, E4M3FN_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8), scale


def quantize_int8(x: torch.Tensor):
    """Per-tensor symmetric int8 codes of x with scale amax/127 (test data only).

    Returns (codes int8, scale float); codes = round-to-nearest-even(x / scale)
    clamped to [-127, 127].
    """
    amax = float(x.abs().max())
    scale = amax / 127.0 if amax > 0 else 1.0
    y = torch.round(x / scale).clamp_(-127, 127)
    return y.to(torch.int8), scale


def paged_inputs(B, Hq, Hkv, D, page_size, pages_per_req, num_pages, topk, seed,
                 device="cpu", pad_tail: int = 0):
    """Sparse paged FP8 inputs.

    Returns dict with q, gate [B,Hq,D] bf16; k_pool, v_pool uint8
    [num_pages, page_size, Hkv, D]; k_scale, v_scale floats; page_table int32
    [B, pages_per_req] (distinct pages drawn from a random permutation of the
    pool); topk int32 [B, topk] (a random selection of each request's logical
    tokens, in random order).  ``pad_tail`` > 0 replaces the last entries of
    every topk row by -1 (padding).
    """
    assert B * pages_per_req <= num_pages
    assert topk <= pages_per_req * page_size
    g = _gen(seed, device)
    q = _randn_bf16((B, Hq, D), g, device)
    gate = _randn_bf16((B, Hq, D), g, device)
    kx = torch.randn((num_pages, page_size, Hkv, D), generator=g, device=device, dtype=torch.float32)
    k_pool, k_scale = quantize_e4m3fn(kx)
    del kx
    vx = torch.randn((num_pages, page_size, Hkv, D), generator=g, device=device, dtype=torch.float32)
    v_pool, v_scale = quantize_e4m3fn(vx)
    del vx
    perm = torch.randperm(num_pages, generator=g, device=device)[: B * pages_per_req]
    page_table = perm.view(B, pages_per_req).to(torch.int32).contiguous()
    ntok = pages_per_req * page_size
    rows = [torch.randperm(ntok, generator=g, device=device)[:topk] for _ in range(B)]
    topk_idx = torch.stack(rows).to(torch.int32).contiguous()
    if pad_tail:
        topk_idx[:, topk - pad_tail:] = -1
    return dict(q=q, gate=gate, k_pool=k_pool.contiguous(), v_pool=v_pool.contiguous(),
                k_scale=k_scale, v_scale=v_scale, page_table=page_table, topk=topk_idx,
                page_size=page_size)


def paged_config_inputs(cfg: PagedConfig, device="cpu"):
    return paged_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.page_size, cfg.pages_per_req,
                        cfg.num_pages, cfg.topk, cfg.seed, device)


def paged_kv_inputs(B, Sq, Hq, Hkv, D, page_size, pages_per_req, num_pages, seed, kv_dtype="bf16",
                    seq_lens=None, device="cpu"):
    """Paged inputs over whole requests.

    Returns dict with q [B,Sq,Hq,D] bf16; k_pool, v_pool [num_pages,
    page_size, Hkv, D] (bf16, uint8 E4M3FN codes for kv_dtype "fp8", or int8
    codes for "int8");
    k_scale, v_scale floats (1.0 for bf16); page_table int32 [B, pages_per_req]
    (distinct pages from a random permutation of the pool); seq_lens int32 [B]
    (given, or uniform in [capacity / 2, capacity]).
    """
    assert B * pages_per_req <= num_pages and kv_dtype in ("bf16", "fp8", "int8")
    cap = pages_per_req * page_size
    g = _gen(seed, device)
    q = _randn_bf16((B, Sq, Hq, D), g, device)
    shape = (num_pages, page_size, Hkv, D)
    if kv_dtype == "bf16":
        k_pool = _randn_bf16(shape, g, device)
        v_pool = _randn_bf16(shape, g, device)
        k_scale = v_scale = 1.0
    else:
        quant = quantize_e4m3fn if kv_dtype == "fp8" else quantize_int8
        kx = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        k_pool, k_scale = quant(kx)
        del kx
        vx = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        v_pool, v_scale = quant(vx)
        del vx
    perm = torch.randperm(num_pages, generator=g, device=device)[: B * pages_per_req]
    page_table = perm.view(B, pages_per_req).to(torch.int32).contiguous()
    if seq_lens is None:
        seq_lens = paged_kv_seq_lens(B, Sq, cap, seed)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).to(device).contiguous()
    return dict(q=q, k_pool=k_pool.contiguous(), v_pool=v_pool.contiguous(), k_scale=float(k_scale),
                v_scale=float(v_scale), page_table=page_table, seq_lens=seq_lens, page_size=page_size)


def paged_kv_seq_lens(B, Sq, cap, seed) -> torch.Tensor:
    """Request lengths uniform in [max(Sq, cap / 2), cap], drawn on the CPU from
    their own seed, so a configuration has the same lengths (and KV bytes) on
    every device."""
    g = torch.Generator().manual_seed(seed + 7919)
    lo = max(Sq, cap // 2)
    return torch.randint(lo, cap + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def paged_kv_config_inputs(cfg: PagedKVConfig, device="cpu"):
    return paged_kv_inputs(cfg.B, cfg.Sq, cfg.Hq, cfg.Hkv, cfg.D, cfg.page_size, cfg.pages_per_req,
                           cfg.num_pages, cfg.seed, cfg.kv_dtype, device=device)
