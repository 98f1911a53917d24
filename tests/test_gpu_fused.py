"""The fused decode step (dattn_append_decode), the selector's pool-page output and the
decode that reads it, and the head-aligned split of block-sparse launches.

dattn_append_decode must leave exactly what dattn_kv_append (one token) followed by
dattn_decode leaves: the same outputs bit for bit (the new token's K/V enters the attention
with the same bf16 values, or with a quantized pool the same codes and scales), the same
pool, scales, statistics, lengths and error bits. The two-call
path is itself checked against the oracle elsewhere; the fused path is also checked against
the oracle here, on every (request, query head), so that its parity does not rest on the
other path alone.
"""
import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_distattention_gb300 import workloads as W

from _util import (assert_e_close, assert_m_close, assert_out_close, check_dense, check_selection,
                   host_kv)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _lib():
    import split_kv_decode_distattention_gb300 as dattn
    dattn.load_library()
    return dattn


def _pair(case, **kw):
    """Two caches filled identically (zeroed first, so that the unwritten slots agree too):
    one stepped by two calls, one by the fused call."""
    from split_kv_decode_distattention_gb300.harness import PagedCache
    kw["zero_pool"] = True
    return PagedCache(case, DEV, **kw), PagedCache(case, DEV, **kw)


def _outs(case):
    out = torch.full((case.B, case.Hq, case.d), float("nan"), device=DEV)
    m = torch.full((case.B, case.Hq), float("nan"), device=DEV)
    e = torch.full((case.B, case.Hq), float("nan"), device=DEV)
    return out, m, e


def _assert_same_state(a, b, what):
    torch.cuda.synchronize()
    assert a.seq_lens.tolist() == b.seq_lens.tolist(), what
    assert int(a.dev_err.item()) == int(b.dev_err.item()), what
    for name in ("k_pool", "v_pool", "stats", "kv_scale"):
        x, y = getattr(a, name), getattr(b, name)
        if x is None:
            continue
        diff = (x.view(torch.int32) != y.view(torch.int32)).nonzero() if name == "kv_scale" \
            else (x.view(torch.uint8) != y.view(torch.uint8)).nonzero()
        assert diff.shape[0] == 0, f"{what}: {name} differs at {diff[:4].tolist()}"


def _steps(case, sep, fus, nsteps, splits, sel=None, sel_phys=None, check_oracle=True):
    """Runs nsteps of append + decode both ways and compares them after every step."""
    sp_sep = sep.sparse_config(sel) if sel is not None else None
    sp_fus = fus.sparse_config(sel, sel_phys) if sel is not None else None
    ws_sep, ws_fus = sep.workspace(num_splits=splits), fus.workspace(num_splits=splits)
    for step in range(nsteps):
        kn, vn = sep.new_tokens(1)
        q = case.q(step, DEV)
        o1, m1, e1 = _outs(case)
        o2, m2, e2 = _outs(case)
        sep.append(kn, vn)
        sep.decode(q, o1, ws_sep, m_g=m1, e_g=e1, sparse=sp_sep, num_splits=splits)
        fus.append_decode(kn, vn, q, o2, ws_fus, m_g=m2, e_g=e2, sparse=sp_fus,
                          num_splits=splits)
        _assert_same_state(sep, fus, f"step {step}")
        assert torch.equal(o1, o2), f"step {step}: outputs differ"
        assert torch.equal(m1, m2) and torch.equal(e1, e2), f"step {step}: m/e differ"
        if check_oracle and sel is None:
            check_dense(case, q, fus.lens, o2, m2, e2, DEV, what=f"fused step {step}")
    return q, o2, m2, e2


@pytest.mark.parametrize("d,P,lens,Hq,Hkv,splits", [
    (128, 16, [1000, 31, 16, 0, 511], 16, 4, 0),     # page and logical-page boundaries, L = 0
    (64, 64, [300, 64, 127, 5000], 8, 2, 7),         # 64-token pages, few CTAs
    (128, 16, [4097, 2000], 32, 32, 5000),           # MHA, more CTAs than tiles
    (128, 32, [15, 1, 33], 8, 8, 0),                 # one-token and one-tile requests
])
def test_append_decode_equals_append_then_decode_dense(d, P, lens, Hq, Hkv, splits):
    _lib()
    case = W.Case("fused", B=len(lens), Hq=Hq, Hkv=Hkv, d=d, P=P, lens=lens, seed=31 + d + P)
    sep, fus = _pair(case, with_stats=True)
    _steps(case, sep, fus, 3, splits)


@pytest.mark.parametrize("kinds,splits", [
    ([1, 2, 1, 2], 0),   # the head-aligned split
    ([1, 2, 1, 2], 9),   # one CTA per retrieval segment, all streaming segments in one CTA
    ([1, 2, 1, 2], 5),   # too few CTAs for the head-aligned split: the balanced split
    ([1, 0, 2, 1], 0),   # a dense head: the balanced split
    ([2, 2, 2, 2], 0),   # streaming heads only
    ([1, 1, 1, 1], 3),   # retrieval heads only, fewer CTAs than retrieval segments
])
def test_append_decode_equals_append_then_decode_sparse(kinds, splits):
    """Block-sparse steps with a reused selection, with and without the selector's pool
    pages, against the two-call path, then against the oracle's token sets."""
    _lib()
    case = W.Case("fused-sparse", B=4, Hq=16, Hkv=4, d=128, P=64,
                  lens=[64 * 60 + 63, 64 * 8, 1000, 12], seed=41, head_kind=kinds, top_k=8,
                  sinks=4, local=8, n_highsim=4)
    sep, fus = _pair(case, with_stats=True)
    q0 = case.q(0, DEV)
    sel = torch.empty(case.B, case.Hkv, case.top_k, dtype=torch.int32, device=DEV)
    phys = torch.full_like(sel, 12345)
    sep.select(q0, sel, sep.workspace(top_k=case.top_k), selected_phys=phys)
    torch.cuda.synchronize()
    # the pool pages are the block table's entries of the selected pages
    bt = sep.block_table.cpu().numpy()
    s, ph = sel.cpu().numpy(), phys.cpu().numpy()
    for b in range(case.B):
        for h in range(case.Hkv):
            for i in range(case.top_k):
                assert ph[b, h, i] == (bt[b, s[b, h, i]] if s[b, h, i] >= 0 else -1)
    _steps(case, sep, fus, 3, splits, sel=sel, sel_phys=phys)
    # the last step against the oracle: every query head over its token set
    q = case.q(3, DEV)
    kn, vn = fus.new_tokens(1)
    out, m_g, e_g = _outs(case)
    fus.append_decode(kn, vn, q, out, fus.workspace(num_splits=splits), m_g=m_g, e_g=e_g,
                      sparse=fus.sparse_config(sel, phys), num_splits=splits)
    torch.cuda.synchronize()
    assert int(fus.dev_err.item()) == 0
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    for b in range(case.B):
        L = fus.lens[b]
        K, V = host_kv(case, b, L, DEV)
        for h in range(case.Hq):
            kvh = h // case.g
            rows = oracle.sparse_rows(kinds[kvh], L, case.P, s[b, kvh], case.sinks, case.local)
            r, rm, re = oracle.attention(qb[b, h], K[:, kvh].copy(), V[:, kvh].copy(),
                                         case.scale, rows=rows)
            assert_out_close(o[b, h], r, f"b={b} h={h}")
            assert abs(mg[b, h] - rm) <= 1e-4 * max(1.0, abs(rm)) or rm == mg[b, h]
            assert abs(eg[b, h] - re) <= 1e-4 * max(abs(re), 1e-30)


def test_decode_with_pool_pages_equals_table_lookup():
    """dattn_decode with dattn_sparse.selected_phys gives the same bits as the block-table
    lookup, and the selection itself is a valid top-K of the fp64 scores."""
    _lib()
    case = W.Case("phys", B=3, Hq=32, Hkv=8, d=128, P=64, lens=[64 * 100 + 17, 3000, 64],
                  seed=43, head_kind=[1, 1, 1, 1, 2, 2, 2, 2], top_k=16, sinks=4, local=8,
                  n_highsim=8)
    from split_kv_decode_distattention_gb300.harness import PagedCache
    cache = PagedCache(case, DEV, with_stats=True)
    q = case.q(0, DEV)
    sel = torch.empty(case.B, case.Hkv, case.top_k, dtype=torch.int32, device=DEV)
    phys = torch.empty_like(sel)
    cache.select(q, sel, cache.workspace(top_k=case.top_k), selected_phys=phys)
    outs = []
    for sp in (cache.sparse_config(sel), cache.sparse_config(sel, phys)):
        out, m_g, e_g = _outs(case)
        cache.decode(q, out, cache.workspace(), m_g=m_g, e_g=e_g, sparse=sp)
        outs.append((out, m_g, e_g))
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    qb = oracle.bf16_bits(q)
    got = sel.cpu().numpy()
    for b in range(case.B):
        K, _ = host_kv(case, b, cache.lens[b], DEV)
        for h in range(4):
            score, bound = oracle.page_scores(qb[b, h * case.g:(h + 1) * case.g],
                                              K[:, h].copy(), cache.lens[b], case.P,
                                              with_bounds=True)
            check_selection(got[b, h], score, bound, case.top_k, f"b={b} h={h}")


def test_append_decode_flags_unmapped_new_page_like_append():
    """A new token whose page is unmapped is not written, and flagged, exactly as by
    dattn_kv_append; the decode skips that tile in both paths."""
    dattn = _lib()
    case = W.Case("unm-new", B=2, Hq=4, Hkv=2, d=128, P=16, lens=[32, 40], seed=5)
    sep, fus = _pair(case)
    for c in (sep, fus):
        c.block_table[0, 2] = -1  # request 0's next token (position 32) has no page
    _steps(case, sep, fus, 1, 0, check_oracle=False)
    assert int(fus.dev_err.item()) & dattn.DEVERR["UNMAPPED_PAGE"]


def _fmt_kw(dattn, fmt, kinds):
    """PagedCache arguments of a pool format ("mixed": streaming heads 4-bit, others 8-bit)."""
    if fmt == "fp8":
        return dict(kv_format=dattn.KV_FP8_E4M3)
    if fmt == "int4":
        return dict(kv_format=dattn.KV_INT4)
    return dict(kv_format=dattn.KV_MIXED,
                head_format=[dattn.KV_INT4 if k == W.HEAD_STREAMING else dattn.KV_FP8_E4M3
                             for k in kinds])


@pytest.mark.parametrize("fmt", ["fp8", "int4", "mixed"])
@pytest.mark.parametrize("d,P,lens,Hq,Hkv,splits", [
    (128, 16, [1000, 31, 16, 0, 511], 16, 4, 0),   # page and logical-page boundaries, L = 0
    (64, 64, [300, 64, 127, 5000], 8, 2, 7),       # 64-token pages, few CTAs
])
def test_append_decode_equals_append_then_decode_quantized(fmt, d, P, lens, Hq, Hkv, splits):
    """A quantized pool: the fused launch stores the new rows quantized exactly as
    dattn_kv_append does (codes, scales and statistics bit for bit) and attends the same
    codes (outputs bit for bit). The two-call path is checked against the oracle elsewhere."""
    dattn = _lib()
    kinds = [W.HEAD_RETRIEVAL if h % 2 == 0 else W.HEAD_STREAMING for h in range(Hkv)]
    case = W.Case("fused-q", B=len(lens), Hq=Hq, Hkv=Hkv, d=d, P=P, lens=lens, seed=37 + d + P)
    kw = _fmt_kw(dattn, fmt, kinds)
    sep, fus = _pair(case, with_stats=True, **kw)
    q, out, m_g, e_g = _steps(case, sep, fus, 3, splits, check_oracle=False)
    # the last step against the oracle's fp64 attention over its own dequantized rows, each
    # head in its format
    four = [fmt == "int4" or (fmt == "mixed" and k == W.HEAD_STREAMING) for k in kinds]
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    for b in range(case.B):
        K, V = host_kv(case, b, fus.lens[b], DEV)
        for h in range(case.Hq):
            kvh = h // case.g
            quant, deq = ((oracle.quantize_rows_int4, oracle.dequantize_rows_int4) if four[kvh]
                          else (oracle.quantize_rows_fp8, oracle.dequantize_rows_fp8))
            Kd = deq(*quant(K[:, kvh].copy()))
            Vd = deq(*quant(V[:, kvh].copy()))
            r, rm, re = oracle.attention_f64(qb[b, h], Kd, Vd, case.scale)
            assert_out_close(o[b, h], r, f"{fmt} b={b} h={h}")
            assert_m_close(mg[b, h], rm, f"{fmt} b={b} h={h}")
            assert_e_close(eg[b, h], re, f"{fmt} b={b} h={h}")


@pytest.mark.parametrize("fmt", ["fp8", "int4", "mixed"])
def test_append_decode_equals_append_then_decode_sparse_quantized(fmt):
    """Block-sparse steps over a quantized pool (retrieval heads 8-bit and streaming heads
    4-bit in the mixed one), with the selector's pool pages, against the two-call path."""
    dattn = _lib()
    kinds = [1, 2, 1, 2]
    case = W.Case("fused-sq", B=4, Hq=16, Hkv=4, d=128, P=64,
                  lens=[64 * 60 + 63, 64 * 8, 1000, 12], seed=47, head_kind=kinds, top_k=8,
                  sinks=4, local=8, n_highsim=4)
    sep, fus = _pair(case, with_stats=True, **_fmt_kw(dattn, fmt, kinds))
    sel = torch.empty(case.B, case.Hkv, case.top_k, dtype=torch.int32, device=DEV)
    phys = torch.empty_like(sel)
    sep.select(case.q(0, DEV), sel, sep.workspace(top_k=case.top_k), selected_phys=phys)
    torch.cuda.synchronize()
    _steps(case, sep, fus, 3, 0, sel=sel, sel_phys=phys, check_oracle=False)
