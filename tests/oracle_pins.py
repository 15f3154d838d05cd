"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes a loaded oracle and raises AssertionError when
the oracle disagrees with a fact fixed by the pages or by mathematics:

* brute force at 50 significant digits on tiny inputs (no max subtraction,
  K/V expanded to every query head with numpy),
* a special case that reduces to library routines (torch float64 softmax,
  logsumexp and matmul over explicitly expanded heads with a ``tril`` mask),
* closed forms (all-zero K, constant V, a single key, zero scale, hard max),
* invariants (native GQA == pre-expanded MHA bit for bit, top-K order),
* the head-map table printed on the page (tests/golden),
* every FP8 E4M3FN code against torch's float8 -> float32 conversion,
* the byte-exact paged gather against numpy fancy indexing.

The same pins run against deliberately broken builds of the oracle (see
test_oracle_mutants.py), which proves each plausible mistake is caught.
"""
from __future__ import annotations

import math
import os

import mpmath
import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------
# helpers (data only; no attention arithmetic)
# ----------------------------------------------------------------------
def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _visible_mask(Sq, Skv):
    """Bottom-right aligned causal mask as a library ``tril`` with offset."""
    return torch.ones(Sq, Skv, dtype=torch.bool).tril(diagonal=Skv - Sq).numpy()


def _assert_close(a, b, rtol, atol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    bad = ~(np.abs(a - b) <= atol + rtol * np.abs(b))
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    bad &= ~both_inf
    assert not bad.any(), f"{what}: max err {np.nanmax(np.abs(a - b))}"


# ----------------------------------------------------------------------
# dense pins
# ----------------------------------------------------------------------
def pin_bruteforce_dense(orc):
    """Tiny inputs at 50 digits: softmax = exp(s) / sum exp(s), no shifting."""
    mpmath.mp.dps = 50
    cases = [(1, 1, 1, 2, 1, 4), (2, 1, 5, 4, 2, 3), (1, 3, 6, 4, 2, 4), (2, 2, 4, 6, 3, 2),
             (1, 2, 2, 2, 1, 4), (1, 3, 3, 4, 4, 2)]
    for ci, (B, Sq, Skv, Hq, Hkv, D) in enumerate(cases):
        q = _bf16((B, Sq, Hq, D), 11 + ci)
        k = _bf16((B, Skv, Hkv, D), 21 + ci)
        v = _bf16((B, Skv, Hkv, D), 31 + ci)
        scale = 0.7 / math.sqrt(D)
        O, L = orc.gqa_decode(q, k, v, scale)
        G = Hq // Hkv
        ke = np.repeat(_f64(k), G, axis=2)  # expand to every query head
        ve = np.repeat(_f64(v), G, axis=2)
        qn = _f64(q)
        vis = _visible_mask(Sq, Skv)
        for b in range(B):
            for h in range(Hq):
                for i in range(Sq):
                    ws, ls = [], []
                    for j in range(Skv):
                        if not vis[i, j]:
                            continue
                        s = mpmath.mpf(0)
                        for d in range(D):
                            s += mpmath.mpf(qn[b, i, h, d]) * mpmath.mpf(ke[b, j, h, d])
                        s *= mpmath.mpf(scale)
                        ws.append(mpmath.e ** s)
                        ls.append(j)
                    Z = mpmath.fsum(ws)
                    lse = float(mpmath.log(Z))
                    assert abs(L[b, h, i] - lse) <= 1e-12 * max(1.0, abs(lse)), (ci, b, h, i, L[b, h, i], lse)
                    for d in range(D):
                        o = float(mpmath.fsum(w * mpmath.mpf(ve[b, j, h, d]) for w, j in zip(ws, ls)) / Z)
                        assert abs(O[b, i, h, d] - o) <= 1e-12 * max(1.0, abs(o)), (ci, b, h, i, d)


def pin_library_dense(orc):
    """torch float64: expanded heads, tril mask, softmax / logsumexp / matmul."""
    for ci, (B, Sq, Skv, Hq, Hkv, D) in enumerate(
            [(2, 1, 300, 8, 2, 64), (1, 4, 257, 8, 4, 32), (1, 8, 40, 32, 2, 16), (3, 2, 65, 4, 1, 8)]):
        q = _bf16((B, Sq, Hq, D), 101 + ci)
        k = _bf16((B, Skv, Hkv, D), 201 + ci)
        v = _bf16((B, Skv, Hkv, D), 301 + ci)
        scale = 1.0 / math.sqrt(D)
        O, L = orc.gqa_decode(q, k, v, scale)
        G = Hq // Hkv
        qt = q.double().permute(0, 2, 1, 3)                        # [B,Hq,Sq,D]
        kt = k.double().repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
        vt = v.double().repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
        s = torch.matmul(qt, kt.transpose(-1, -2)) * scale          # [B,Hq,Sq,Skv]
        mask = torch.from_numpy(_visible_mask(Sq, Skv))
        s = s.masked_fill(~mask, float("-inf"))
        ref_L = torch.logsumexp(s, dim=-1)                          # [B,Hq,Sq]
        ref_O = torch.matmul(torch.softmax(s, dim=-1), vt).permute(0, 2, 1, 3)
        _assert_close(L, ref_L.numpy(), 1e-12, 1e-12, f"library lse case {ci}")
        _assert_close(O, ref_O.numpy(), 1e-12, 1e-12, f"library O case {ci}")


def pin_gqa_equals_expanded_mha(orc):
    """Native GQA == the same inputs pre-expanded to Hq KV heads, bit for bit.

    K differs per KV head, so a kernel that confuses query heads per KV head
    with the KV-head count reads the wrong rows at 8/4 and 8/2.
    """
    for ci, (Hq, Hkv) in enumerate([(8, 4), (8, 2), (4, 2), (16, 4), (8, 1), (64, 8), (32, 2)]):
        B, Sq, Skv, D = 2, 2, 23, 8
        q = _bf16((B, Sq, Hq, D), 401 + ci)
        k = _bf16((B, Skv, Hkv, D), 501 + ci)
        v = _bf16((B, Skv, Hkv, D), 601 + ci)
        G = Hq // Hkv
        O, L = orc.gqa_decode(q, k, v, 0.3)
        Oe, Le = orc.gqa_decode(q, k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2), 0.3)
        assert np.array_equal(O, Oe) and np.array_equal(L, Le), (Hq, Hkv)


def pin_head_map_table(orc):
    """The right map reproduces the table printed on the kv-copies-gqa page."""
    path = os.path.join(GOLDEN, "head_map_kv_copies_gqa.txt")
    rows = [ln for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 4
    for ln in rows:
        hk, right, wrong, same = [c.strip() for c in ln.split("|")]
        Hq, Hkv = map(int, hk.split())
        right = list(map(int, right.split()))
        wrong = list(map(int, wrong.split()))
        got = [orc.kv_head(h, Hq, Hkv) for h in range(Hq)]
        assert got == right, (Hq, Hkv, got, right)
        # the printed wrong map coincides with the right one exactly where the page says so
        assert (right == wrong) == (same == "yes"), ln


def pin_zero_keys(orc):
    """K == 0: every visible score is 0, so LSE = ln(#visible) and O = mean of visible V."""
    for (B, Sq, Skv, Hq, Hkv, D) in [(1, 1, 37, 4, 2, 8), (2, 3, 9, 8, 2, 4), (1, 8, 8, 4, 1, 4)]:
        q = _bf16((B, Sq, Hq, D), 701)
        k = torch.zeros((B, Skv, Hkv, D), dtype=torch.bfloat16)
        v = _bf16((B, Skv, Hkv, D), 702)
        O, L = orc.gqa_decode(q, k, v, 0.125)
        G = Hq // Hkv
        vn = _f64(v)
        for i in range(Sq):
            nvis = Skv - Sq + 1 + i
            _assert_close(L[:, :, i], np.full((B, Hq), math.log(nvis)), 1e-14, 1e-14, "zero-K lse")
            mean = vn[:, :nvis].mean(axis=1)                  # [B,Hkv,D]
            _assert_close(O[:, i], np.repeat(mean, G, axis=1), 1e-13, 1e-13, "zero-K O")


def pin_constant_v(orc):
    """Every V row equal to c (per KV head) gives O = c whatever the scores."""
    B, Sq, Skv, Hq, Hkv, D = 2, 2, 50, 8, 2, 16
    q = _bf16((B, Sq, Hq, D), 801, scale=3.0)
    k = _bf16((B, Skv, Hkv, D), 802)
    c = _bf16((B, 1, Hkv, D), 803)
    v = c.expand(B, Skv, Hkv, D).contiguous()
    O, _ = orc.gqa_decode(q, k, v, 0.25)
    G = Hq // Hkv
    want = np.repeat(_f64(c)[:, 0], G, axis=1)                # [B,Hq,D]
    for i in range(Sq):
        _assert_close(O[:, i], want, 1e-13, 1e-13, "constant V")


def pin_single_key(orc):
    """Degenerate single-key softmax: O = V_0 exactly and LSE = scale * q.k_0.

    Covers Skv = 1 and, with Sq = Skv, row 0, which sees only key 0.
    """
    for (B, Sq, Skv, Hq, Hkv, D) in [(2, 1, 1, 4, 2, 8), (1, 3, 3, 4, 2, 8)]:
        q = _bf16((B, Sq, Hq, D), 901)
        k = _bf16((B, Skv, Hkv, D), 902)
        v = _bf16((B, Skv, Hkv, D), 903)
        scale = 0.5
        O, L = orc.gqa_decode(q, k, v, scale)
        G = Hq // Hkv
        qn, kn, vn = _f64(q), _f64(k), _f64(v)
        for b in range(B):
            for h in range(Hq):
                assert np.array_equal(O[b, 0, h], vn[b, 0, h // G]), (b, h)
                s0 = scale * math.fsum(qn[b, 0, h] * kn[b, 0, h // G])
                assert abs(L[b, h, 0] - s0) <= 1e-14 * max(1.0, abs(s0)), (b, h)


def pin_zero_scale(orc):
    """scale = 0 makes every visible key equally likely."""
    B, Sq, Skv, Hq, Hkv, D = 1, 2, 30, 4, 2, 8
    q = _bf16((B, Sq, Hq, D), 1001)
    k = _bf16((B, Skv, Hkv, D), 1002)
    v = _bf16((B, Skv, Hkv, D), 1003)
    O, L = orc.gqa_decode(q, k, v, 0.0)
    vn = _f64(v)
    for i in range(Sq):
        nvis = Skv - Sq + 1 + i
        _assert_close(L[:, :, i], np.full((B, Hq), math.log(nvis)), 1e-14, 1e-14, "zero-scale lse")
        _assert_close(O[:, i], np.repeat(vn[:, :nvis].mean(axis=1), Hq // Hkv, axis=1), 1e-13, 1e-13,
                      "zero-scale O")


def pin_hardmax(orc):
    """q = lambda * k_{j*} with large lambda: O -> V_{j*}, LSE -> scale * lambda * |k_{j*}|^2."""
    B, Sq, Skv, Hq, Hkv, D = 1, 1, 16, 2, 1, 8
    k = torch.zeros((B, Skv, Hkv, D), dtype=torch.bfloat16)
    for j in range(Skv):
        k[0, j, 0, j % D] = 1.0 if j < D else -1.0          # orthogonal rows
    v = _bf16((B, Skv, Hkv, D), 1101)
    jstar = 5
    q = (64.0 * k[:, jstar:jstar + 1, 0:1, :]).expand(B, Sq, Hq, D).contiguous()
    O, L = orc.gqa_decode(q, k, v, 1.0)
    _assert_close(O[0, 0], np.repeat(_f64(v)[0, jstar], Hq, axis=0).reshape(Hq, D), 1e-20, 1e-20, "hardmax O")
    _assert_close(L[0, :, 0], np.full(Hq, 64.0), 1e-15, 1e-15, "hardmax lse")


# ----------------------------------------------------------------------
# FP8 / paged pins
# ----------------------------------------------------------------------
def pin_e4m3fn_table(orc):
    """All 256 codes against torch's float8_e4m3fn -> float32 conversion."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    mine = np.array([orc.e4m3fn_value(c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(mine))
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(mine[~nan], lib[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def _paged_small(seed, B=3, Hq=8, Hkv=2, D=16, ps=4, ppr=5, num_pages=20, topk=13, kscale=0.37, vscale=1.9):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, D), generator=g).to(torch.bfloat16)
    gate = torch.randn((B, Hq, D), generator=g).to(torch.bfloat16)
    kp = (torch.randn((num_pages, ps, Hkv, D), generator=g) * 40).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    vp = (torch.randn((num_pages, ps, Hkv, D), generator=g) * 40).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    pt = torch.randperm(num_pages, generator=g)[: B * ppr].view(B, ppr).to(torch.int32)
    tk = torch.stack([torch.randperm(ppr * ps, generator=g)[:topk] for _ in range(B)]).to(torch.int32)
    return q, gate, kp, vp, pt, tk, kscale, vscale


def _gather_numpy(pool, pt, tk):
    """Fancy-index route: the request's logical cache is its pages in order."""
    pool = pool.numpy()
    pt = pt.numpy()
    tk = tk.numpy()
    num_pages, ps, Hkv, D = pool.shape
    B, ppr = pt.shape
    out = np.zeros((B, tk.shape[1], Hkv, D), dtype=np.uint8)
    for b in range(B):
        logical = pool[pt[b]].reshape(ppr * ps, Hkv, D)
        sel = tk[b]
        ok = sel >= 0
        out[b, ok] = logical[sel[ok]]
    return out


def pin_paged_gather(orc):
    """Byte-exact gather against numpy fancy indexing, page sizes 1, 16, 64."""
    for ci, (ps, ppr, topk) in enumerate([(1, 37, 20), (16, 6, 96), (64, 2, 100)]):
        _, _, kp, _, pt, tk, _, _ = _paged_small(1200 + ci, ps=ps, ppr=ppr, num_pages=4 * ppr, topk=topk)
        tk[1, 3] = -1                                            # one padding entry
        got = orc.paged_gather(kp, pt, tk, ps)
        assert np.array_equal(got, _gather_numpy(kp, pt, tk)), ps


def pin_bruteforce_paged(orc):
    """Tiny paged case at 50 digits, decoded through torch's FP8 table."""
    mpmath.mp.dps = 50
    q, gate, kp, vp, pt, tk, ks, vs = _paged_small(1300, B=2, Hq=4, Hkv=2, D=4, ps=2, ppr=3,
                                                   num_pages=7, topk=5)
    tk[1, 4] = -1
    scale = 0.5
    out, lse, attn = orc.gqa_decode_paged_fp8(q, gate, kp, vp, pt, tk, ks, vs, scale)
    kg = torch.from_numpy(_gather_numpy(kp, pt, tk)).view(torch.float8_e4m3fn).double().numpy()
    vg = torch.from_numpy(_gather_numpy(vp, pt, tk)).view(torch.float8_e4m3fn).double().numpy()
    qn, gn, tkn = _f64(q), _f64(gate), tk.numpy()
    B, Hq, D = qn.shape
    Hkv = kp.shape[2]
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ws, ks_ = [], []
            for kk in range(tkn.shape[1]):
                if tkn[b, kk] < 0:
                    continue
                s = mpmath.mpf(scale) * mpmath.fsum(
                    mpmath.mpf(qn[b, h, d]) * mpmath.mpf(kg[b, kk, g, d]) * mpmath.mpf(ks) for d in range(D))
                ws.append(mpmath.e ** s)
                ks_.append(kk)
            Z = mpmath.fsum(ws)
            assert abs(lse[b, h] - float(mpmath.log(Z))) <= 1e-12
            for d in range(D):
                a = mpmath.fsum(w * mpmath.mpf(vg[b, kk, g, d]) * mpmath.mpf(vs) for w, kk in zip(ws, ks_)) / Z
                sig = 1 / (1 + mpmath.e ** (-mpmath.mpf(gn[b, h, d])))
                assert abs(attn[b, h, d] - float(a)) <= 1e-12 * max(1.0, abs(float(a)))
                assert abs(out[b, h, d] - float(sig * a)) <= 1e-12 * max(1.0, abs(float(a)))


def pin_paged_equals_dense(orc):
    """Identity page table and top-K over a cache whose dequantised values are
    bf16-exact equal the dense oracle at Sq = 1; gate = 0 halves the output."""
    B, Hq, Hkv, D, ps, ppr = 2, 8, 2, 16, 4, 3
    ntok = ps * ppr
    g = torch.Generator().manual_seed(1400)
    q = torch.randn((B, Hq, D), generator=g).to(torch.bfloat16)
    kp = (torch.randn((B * ppr, ps, Hkv, D), generator=g) * 30).to(torch.float8_e4m3fn).view(torch.uint8)
    vp = (torch.randn((B * ppr, ps, Hkv, D), generator=g) * 30).to(torch.float8_e4m3fn).view(torch.uint8)
    pt = torch.arange(B * ppr, dtype=torch.int32).view(B, ppr)
    tk = torch.arange(ntok, dtype=torch.int32).expand(B, ntok).contiguous()
    ks, vs = 0.25, 2.0                                            # powers of two keep bf16 exactness
    gate = torch.zeros((B, Hq, D), dtype=torch.bfloat16)
    out, lse, attn = orc.gqa_decode_paged_fp8(q, gate, kp, vp, pt, tk, ks, vs, 0.2)
    kd = (kp.view(torch.float8_e4m3fn).double() * ks).view(B, ntok, Hkv, D).to(torch.bfloat16)
    vd = (vp.view(torch.float8_e4m3fn).double() * vs).view(B, ntok, Hkv, D).to(torch.bfloat16)
    assert torch.equal(kd.double(), kp.view(torch.float8_e4m3fn).double().view(B, ntok, Hkv, D) * ks)
    O, L = orc.gqa_decode(q.view(B, 1, Hq, D), kd, vd, 0.2)
    _assert_close(attn, O[:, 0], 1e-13, 1e-13, "paged vs dense O")
    _assert_close(lse, L[:, :, 0], 1e-13, 1e-13, "paged vs dense lse")
    assert np.array_equal(out, 0.5 * attn)


def pin_topk_order_and_padding(orc):
    """Permuting a request's top-K list changes nothing beyond rounding; padding
    entries (-1) count as absent; an all-padding row gives O = 0, LSE = -inf."""
    q, gate, kp, vp, pt, tk, ks, vs = _paged_small(1500)
    out, lse, _ = orc.gqa_decode_paged_fp8(q, gate, kp, vp, pt, tk, ks, vs, 0.3)
    g = torch.Generator().manual_seed(1501)
    perm = torch.stack([torch.randperm(tk.shape[1], generator=g) for _ in range(tk.shape[0])])
    tk2 = torch.gather(tk, 1, perm).contiguous()
    out2, lse2, _ = orc.gqa_decode_paged_fp8(q, gate, kp, vp, pt, tk2, ks, vs, 0.3)
    _assert_close(out2, out, 1e-13, 1e-13, "topk permutation")
    _assert_close(lse2, lse, 1e-13, 1e-13, "topk permutation lse")
    # padding entries appended == the shorter list
    tk3 = torch.cat([tk, torch.full((tk.shape[0], 3), -1, dtype=torch.int32)], dim=1).contiguous()
    out3, lse3, _ = orc.gqa_decode_paged_fp8(q, gate, kp, vp, pt, tk3, ks, vs, 0.3)
    assert np.array_equal(out3, out) and np.array_equal(lse3, lse)
    tk4 = torch.full_like(tk, -1)
    out4, lse4, _ = orc.gqa_decode_paged_fp8(q, gate, kp, vp, pt, tk4, ks, vs, 0.3)
    assert np.all(out4 == 0.0) and np.all(np.isneginf(lse4))


def pin_gate_and_scales(orc):
    """sigmoid(0) = 1/2, a saturated gate passes O through, v_scale is linear,
    and k_scale multiplies the scores exactly like the softmax scale does."""
    q, gate, kp, vp, pt, tk, ks, vs = _paged_small(1600)
    zero = torch.zeros_like(gate)
    big = torch.full_like(gate, 100.0)
    out0, lse0, attn0 = orc.gqa_decode_paged_fp8(q, zero, kp, vp, pt, tk, ks, vs, 0.3)
    assert np.array_equal(out0, 0.5 * attn0)
    outb, _, attnb = orc.gqa_decode_paged_fp8(q, big, kp, vp, pt, tk, ks, vs, 0.3)
    assert np.array_equal(outb, attnb)
    _, _, attn2 = orc.gqa_decode_paged_fp8(q, zero, kp, vp, pt, tk, ks, 2 * vs, 0.3)
    _assert_close(attn2, 2 * attn0, 1e-14, 1e-14, "v_scale linear")
    _, lse3, attn3 = orc.gqa_decode_paged_fp8(q, zero, kp, vp, pt, tk, 1.0, vs, 0.3 * ks)
    _assert_close(attn3, attn0, 1e-13, 1e-13, "k_scale folds into scale")
    _assert_close(lse3, lse0, 1e-13, 1e-13, "k_scale folds into scale (lse)")
    # the gate is sigmoid: compare against scipy's logistic function
    from scipy.special import expit
    out4, _, attn4 = orc.gqa_decode_paged_fp8(q, gate, kp, vp, pt, tk, ks, vs, 0.3)
    _assert_close(out4, expit(_f64(gate)) * attn4, 1e-15, 1e-15, "sigmoid gate")


# ----------------------------------------------------------------------
# paged decode over whole requests (no top-K)
# ----------------------------------------------------------------------
def _logical_cache(pool, pt, lens):
    """Fancy-index route: request b's cache is its pages in order, cut at its
    own length.  Returns a list of [len_b, Hkv, D] tensors."""
    num_pages, ps, Hkv, D = pool.shape
    B, ppr = pt.shape
    return [pool[pt[b].long()].reshape(ppr * ps, Hkv, D)[: int(lens[b])] for b in range(B)]


def _paged_kv_small(seed, B=3, Sq=2, Hq=8, Hkv=2, D=16, ps=4, ppr=5, lens=(20, 7, 13)):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Sq, Hq, D), generator=g).to(torch.bfloat16)
    num_pages = B * ppr + 3
    kp = torch.randn((num_pages, ps, Hkv, D), generator=g).to(torch.bfloat16)
    vp = torch.randn((num_pages, ps, Hkv, D), generator=g).to(torch.bfloat16)
    pt = torch.randperm(num_pages, generator=g)[: B * ppr].view(B, ppr).to(torch.int32).contiguous()
    sl = torch.tensor(lens, dtype=torch.int32)
    return q, kp, vp, pt, sl


def pin_paged_requests_equal_dense(orc):
    """Each request of a bf16 paged cache equals the dense oracle run on that
    request's own logical cache (its pages in table order, cut at its own
    length), bit for bit, for S_q = 1 and 2 and page sizes 1, 4, 16."""
    for ci, (Sq, ps, ppr, lens) in enumerate([(2, 4, 5, (20, 7, 13)), (1, 1, 9, (9, 1, 4)), (2, 16, 2, (32, 17, 2))]):
        q, kp, vp, pt, sl = _paged_kv_small(1700 + ci, Sq=Sq, ps=ps, ppr=ppr, lens=lens)
        O, L = orc.gqa_decode_paged(q, kp, vp, pt, sl, 0.3)
        ks, vs = _logical_cache(kp, pt, sl), _logical_cache(vp, pt, sl)
        for b in range(q.shape[0]):
            Od, Ld = orc.gqa_decode(q[b:b + 1], ks[b][None], vs[b][None], 0.3)
            assert np.array_equal(O[b:b + 1], Od), (ci, b)
            assert np.array_equal(L[b:b + 1], Ld), (ci, b)


def pin_paged_fp8_equals_bf16(orc):
    """An FP8 pool with power-of-two k_scale != v_scale equals a bf16 pool that
    holds the dequantised values (bf16-exact), bit for bit."""
    q, _, _, pt, sl = _paged_kv_small(1800)
    g = torch.Generator().manual_seed(1801)
    shape = (pt.numel() + 3, 4, 2, 16)
    k8 = (torch.randn(shape, generator=g) * 40).to(torch.float8_e4m3fn)
    v8 = (torch.randn(shape, generator=g) * 40).to(torch.float8_e4m3fn)
    ks, vs = 0.125, 4.0
    kb = (k8.double() * ks).to(torch.bfloat16)
    vb = (v8.double() * vs).to(torch.bfloat16)
    assert torch.equal(kb.double(), k8.double() * ks) and torch.equal(vb.double(), v8.double() * vs)
    O8, L8 = orc.gqa_decode_paged(q, k8.view(torch.uint8), v8.view(torch.uint8), pt, sl, 0.3, ks, vs)
    Ob, Lb = orc.gqa_decode_paged(q, kb, vb, pt, sl, 0.3)
    assert np.array_equal(O8, Ob) and np.array_equal(L8, Lb)


def pin_paged_int8_equals_bf16(orc):
    """An int8 pool with power-of-two k_scale != v_scale equals a bf16 pool that
    holds the dequantised values (code * scale, exact in bf16 for |code| <= 128),
    bit for bit; codes at both ends of the range (-128, 127) included."""
    q, _, _, pt, sl = _paged_kv_small(2000)
    g = torch.Generator().manual_seed(2001)
    shape = (pt.numel() + 3, 4, 2, 16)
    k8 = torch.randint(-128, 128, shape, generator=g, dtype=torch.int16).to(torch.int8)
    v8 = torch.randint(-128, 128, shape, generator=g, dtype=torch.int16).to(torch.int8)
    k8.view(-1)[:2] = torch.tensor([-128, 127], dtype=torch.int8)
    v8.view(-1)[:2] = torch.tensor([127, -128], dtype=torch.int8)
    ks, vs = 0.0078125, 0.25
    kb = (k8.double() * ks).to(torch.bfloat16)
    vb = (v8.double() * vs).to(torch.bfloat16)
    assert torch.equal(kb.double(), k8.double() * ks) and torch.equal(vb.double(), v8.double() * vs)
    O8, L8 = orc.gqa_decode_paged(q, k8, v8, pt, sl, 0.3, ks, vs)
    Ob, Lb = orc.gqa_decode_paged(q, kb, vb, pt, sl, 0.3)
    assert np.array_equal(O8, Ob) and np.array_equal(L8, Lb)


def pin_paged_zero_keys_and_short_requests(orc):
    """K = 0: LSE = ln(#visible tokens) and O = the mean of the visible V rows
    (numpy over the fancy-indexed cache); a request shorter than S_q leaves its
    first rows with no visible token: O = 0, LSE = -inf."""
    q, kp, vp, pt, sl = _paged_kv_small(1900, Sq=3, lens=(20, 2, 0))
    kz = torch.zeros_like(kp)
    O, L = orc.gqa_decode_paged(q, kz, vp, pt, sl, 0.3)
    vs = _logical_cache(vp, pt, sl)
    B, Sq, Hq, D = q.shape
    Hkv = kp.shape[2]
    for b in range(B):
        for i in range(Sq):
            n_vis = int(sl[b]) - Sq + i + 1
            for h in range(Hq):
                g = h // (Hq // Hkv)
                if n_vis <= 0:
                    assert np.all(O[b, i, h] == 0.0) and np.isneginf(L[b, h, i]), (b, i, h)
                    continue
                assert abs(L[b, h, i] - math.log(n_vis)) <= 1e-13
                mean = _f64(vs[b][:n_vis, g]).mean(axis=0)
                _assert_close(O[b, i, h], mean, 1e-13, 1e-13, "paged mean of visible V")


# ----------------------------------------------------------------------
# Dqk != Dv
# ----------------------------------------------------------------------
def pin_dv_equals_padded_v(orc):
    """Dqk = 192, Dv = 128 equals the dense oracle run with V zero-padded to
    192 columns: the first 128 output columns and the LSE bit for bit (the
    padded columns come out exactly 0); Sq = 1 and 3 (causal)."""
    for ci, (B, Sq, Skv, Hq, Hkv) in enumerate([(2, 1, 37, 8, 2), (1, 3, 20, 4, 4)]):
        q = _bf16((B, Sq, Hq, 192), 2100 + ci)
        k = _bf16((B, Skv, Hkv, 192), 2110 + ci)
        v = _bf16((B, Skv, Hkv, 128), 2120 + ci)
        vp = torch.cat([v, torch.zeros((B, Skv, Hkv, 64), dtype=torch.bfloat16)], dim=3).contiguous()
        O, L = orc.gqa_decode_dv(q, k, v, 0.07)
        Op, Lp = orc.gqa_decode(q, k, vp, 0.07)
        assert np.array_equal(O, Op[..., :128]) and np.all(Op[..., 128:] == 0.0)
        assert np.array_equal(L, Lp)


def pin_bruteforce_dv(orc):
    """Tiny Dqk != Dv case at 50 digits, no max subtraction."""
    mpmath.mp.dps = 50
    B, Sq, Skv, Hq, Hkv, Dqk, Dv = 1, 2, 5, 4, 2, 6, 3
    q, k, v = _bf16((B, Sq, Hq, Dqk), 2200), _bf16((B, Skv, Hkv, Dqk), 2201), _bf16((B, Skv, Hkv, Dv), 2202)
    O, L = orc.gqa_decode_dv(q, k, v, 0.4)
    qn, kn, vn = _f64(q), _f64(k), _f64(v)
    vis = _visible_mask(Sq, Skv)
    for i in range(Sq):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ws = [mpmath.e ** (mpmath.mpf(0.4) * mpmath.fsum(mpmath.mpf(qn[0, i, h, d]) * mpmath.mpf(kn[0, j, g, d])
                                                          for d in range(Dqk))) if vis[i, j] else mpmath.mpf(0)
                  for j in range(Skv)]
            Z = mpmath.fsum(ws)
            assert abs(L[0, h, i] - float(mpmath.log(Z))) <= 1e-12
            for d in range(Dv):
                ref = float(mpmath.fsum(w * mpmath.mpf(vn[0, j, g, d]) for j, w in enumerate(ws)) / Z)
                assert abs(O[0, i, h, d] - ref) <= 1e-12 * max(1.0, abs(ref))


DENSE_PINS = [pin_bruteforce_dense, pin_library_dense, pin_gqa_equals_expanded_mha, pin_head_map_table,
              pin_zero_keys, pin_constant_v, pin_single_key, pin_zero_scale, pin_hardmax]
PAGED_PINS = [pin_e4m3fn_table, pin_paged_gather, pin_bruteforce_paged, pin_paged_equals_dense,
              pin_topk_order_and_padding, pin_gate_and_scales]
PAGED_KV_PINS = [pin_paged_requests_equal_dense, pin_paged_fp8_equals_bf16, pin_paged_int8_equals_bf16,
                 pin_paged_zero_keys_and_short_requests]
DV_PINS = [pin_dv_equals_padded_v, pin_bruteforce_dv]
ALL_PINS = DENSE_PINS + PAGED_PINS + PAGED_KV_PINS + DV_PINS
