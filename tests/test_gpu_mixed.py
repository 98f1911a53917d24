"""GPU parity of the mixed-precision pool: every KV head in its own format, FP8 E4M3 or 4-bit
("LLM长序列服务优化：LServe的块稀疏注意力技术" §3.2.1: 4-bit streaming heads, 2-8-bit retrieval
heads in one cache), decoded in one launch.

The pool is the 8-bit heads' region [num_pages][H8][P][d] followed by the 4-bit heads'
region [num_pages][H4][P][d/2]; the row scales keep the [num_pages][Hkv][P/16][2][16] layout.
The append is compared bit for bit with the oracle's per-format writes placed in that layout;
every attention result with the oracle's float64 attention over the oracle's own
dequantized values, each head in its own format.
"""
import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_distattention_gb300 import workloads as W

from _util import assert_e_close, assert_m_close, assert_out_close, host_kv

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _lib():
    import split_kv_decode_distattention_gb300 as dattn
    dattn.load_library()
    return dattn


def _formats(dattn, spec):
    """'84' -> [KV_FP8_E4M3, KV_INT4]."""
    return [dattn.KV_INT4 if c == "4" else dattn.KV_FP8_E4M3 for c in spec]


def _cache(case, spec, **kw):
    dattn = _lib()
    from split_kv_decode_distattention_gb300.harness import PagedCache
    return PagedCache(case, DEV, kv_format=dattn.KV_MIXED, head_format=_formats(dattn, spec),
                      **kw)


def _deq(K, V, spec):
    """The oracle's round trip of token-ordered bf16 rows [L][Hkv][d], head h in format
    spec[h] (float64)."""
    out = {}
    for name, quant, deq in (("8", oracle.quantize_rows_fp8, oracle.dequantize_rows_fp8),
                             ("4", oracle.quantize_rows_int4, oracle.dequantize_rows_int4)):
        kc, ks = quant(K)
        vc, vs = quant(V)
        out[name] = (deq(kc, ks), deq(vc, vs))
    Kd = np.stack([out[spec[h]][0][:, h] for h in range(len(spec))], axis=1)
    Vd = np.stack([out[spec[h]][1][:, h] for h in range(len(spec))], axis=1)
    return Kd, Vd


def _oracle_pool(case, lens, spec):
    """The mixed pool's bytes (K, V), scales (K, V [num_pages][Hkv][P]) and statistics as
    the oracle's per-format writes leave them, placed in the mixed layout."""
    P, d = case.P, case.d
    full = {}
    for name, write, row in (("8", oracle.kv_write_fp8, d), ("4", oracle.kv_write_int4, d // 2)):
        kp = np.zeros((case.num_pages, case.Hkv, P, row), np.uint8)
        vp = np.zeros_like(kp)
        ks = np.zeros((case.num_pages, case.Hkv, P), np.float32)
        vs = np.zeros_like(ks)
        for b in range(case.B):
            K, V = host_kv(case, b, lens[b], DEV)
            assert write(kp, vp, ks, vs, P, case.block_table[b], case.num_pages, K, V, 0) == 0
        full[name] = (kp, vp, ks, vs)
    h8 = [h for h in range(case.Hkv) if spec[h] == "8"]
    h4 = [h for h in range(case.Hkv) if spec[h] == "4"]
    kbytes = np.concatenate([full["8"][0][:, h8].reshape(-1), full["4"][0][:, h4].reshape(-1)])
    vbytes = np.concatenate([full["8"][1][:, h8].reshape(-1), full["4"][1][:, h4].reshape(-1)])
    ks = np.stack([full[spec[h]][2][:, h] for h in range(case.Hkv)], axis=1)
    vs = np.stack([full[spec[h]][3][:, h] for h in range(case.Hkv)], axis=1)
    return kbytes, vbytes, ks, vs


def _assert_pool(cache, want):
    kb, vb, ks, vs = want
    np.testing.assert_array_equal(cache.k_pool.cpu().numpy(), kb)
    np.testing.assert_array_equal(cache.v_pool.cpu().numpy(), vb)
    sc = cache.kv_scale.cpu().numpy()
    n, h, P = ks.shape
    np.testing.assert_array_equal(sc[:, :, :, 0, :].reshape(n, h, P).view(np.uint32),
                                  ks.view(np.uint32))
    np.testing.assert_array_equal(sc[:, :, :, 1, :].reshape(n, h, P).view(np.uint32),
                                  vs.view(np.uint32))


def _outs(case):
    out = torch.full((case.B, case.Hq, case.d), float("nan"), device=DEV)
    m = torch.full((case.B, case.Hq), float("nan"), device=DEV)
    e = torch.full((case.B, case.Hq), float("nan"), device=DEV)
    return out, m, e


def _check_dense(case, q, lens, spec, out, m_g, e_g, what, rows_of=None):
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    for b in range(case.B):
        Kd, Vd = _deq(*host_kv(case, b, lens[b], DEV), spec)
        for h in range(case.Hq):
            kvh = h // case.g
            rows = rows_of(b, kvh, lens[b]) if rows_of is not None else None
            r, rm, re = oracle.attention_f64(qb[b, h], Kd[:, kvh], Vd[:, kvh], case.scale,
                                             rows=rows)
            assert_out_close(o[b, h], r, f"{what} b={b} h={h} ({spec[kvh]}-bit head)")
            assert_m_close(mg[b, h], rm, f"{what} b={b} h={h}")
            assert_e_close(eg[b, h], re, f"{what} b={b} h={h}")


# ---------------------------------------------------------------- append

@pytest.mark.parametrize("spec,d,P,chunk", [
    ("84", 128, 16, 37),
    ("4884", 64, 64, 200),
    ("48", 128, 64, 5),
    ("8", 128, 16, 64),       # one 8-bit head: no 4-bit region
    ("44", 64, 16, 64),       # no 8-bit region
])
def test_mixed_append_codes_and_scales_bit_exact(spec, d, P, chunk):
    _lib()
    Hkv = len(spec)
    case = W.Case("append-mixed", B=3, Hq=2 * Hkv, Hkv=Hkv, d=d, P=P, lens=[0, 131, 290],
                  seed=13)
    cache = _cache(case, spec, with_stats=True, fill=False, zero_pool=True, chunk_tokens=chunk)
    cache.fill()
    for _ in range(3):
        kn, vn = cache.new_tokens(1)
        cache.append(kn, vn)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    assert cache.seq_lens.tolist() == cache.lens
    _assert_pool(cache, _oracle_pool(case, cache.lens, spec))


def test_mixed_pool_of_one_format_is_that_format():
    """A mixed pool whose heads are all 8-bit holds the 8-bit pool's bytes and decodes to the
    8-bit pool's results bit for bit (same stages, same order); all-4-bit holds the 4-bit
    pool's bytes."""
    dattn = _lib()
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.Case("one-format", B=3, Hq=16, Hkv=4, d=128, P=16, lens=[1000, 31, 4097], seed=7)
    for spec, fmt in (("8888", dattn.KV_FP8_E4M3), ("4444", dattn.KV_INT4)):
        mixed = _cache(case, spec, zero_pool=True)
        plain = PagedCache(case, DEV, kv_format=fmt, zero_pool=True)
        torch.cuda.synchronize()
        assert torch.equal(mixed.k_pool, plain.k_pool.view(-1))
        assert torch.equal(mixed.v_pool, plain.v_pool.view(-1))
        assert torch.equal(mixed.kv_scale, plain.kv_scale)
        if fmt != dattn.KV_FP8_E4M3:
            continue
        q = case.q(0, DEV)
        res = []
        for c in (mixed, plain):
            out, m_g, e_g = _outs(case)
            c.decode(q, out, c.workspace(num_splits=37), m_g=m_g, e_g=e_g, num_splits=37)
            res.append((out, m_g, e_g))
        torch.cuda.synchronize()
        for a, b in zip(*res):
            assert torch.equal(a, b)


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("spec,d,Hq,P,lens,splits", [
    ("84", 128, 8, 16, [1000, 31, 16, 0, 511], 0),
    ("4884", 128, 16, 64, [64 * 40 + 7, 3000], 0),
    ("48", 64, 16, 64, [999, 1, 2048], 5),
    ("8448", 128, 8, 16, [5000], 0),
    ("84", 128, 4, 16, [1, 15, 16, 17], 500),   # more CTAs than tiles
    ("48", 128, 2, 16, [700, 33, 4000], 0),      # one query head per KV head (MHA)
    ("4", 64, 1, 64, [129, 3000], 3),            # MHA, d = 64
])
def test_mixed_decode_dense_matches_oracle(spec, d, Hq, P, lens, splits):
    _lib()
    case = W.Case("dense-mixed", B=len(lens), Hq=Hq, Hkv=len(spec), d=d, P=P, lens=lens,
                  seed=(sum(map(ord, spec)) + d + P + sum(lens)) % 1000 + 3)
    cache = _cache(case, spec)
    q = case.q(0, DEV)
    out, m_g, e_g = _outs(case)
    ws = cache.workspace(num_splits=splits)
    cache.decode(q, out, ws, m_g=m_g, e_g=e_g, num_splits=splits)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    _check_dense(case, q, cache.lens, spec, out, m_g, e_g, "mixed decode")
    out2 = torch.empty_like(out)
    cache.decode(q, out2, ws, num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


@pytest.mark.parametrize("spec,Hq,lens,T,splits", [
    ("48", 4, [700, 2, 1500], 2, 0),       # group 2, 2 query tokens: 4 columns per KV head
    ("4884", 4, [517, 3, 64], 4, 5),       # MHA, 4 query tokens: 4 columns
    ("84", 2, [300, 1000], 2, 0),          # MHA, 2 query tokens: 2 columns
    ("48", 4, [900, 5], 3, 0),             # group 2, 3 query tokens: 6 columns
])
def test_mixed_decode_multi_matches_oracle(spec, Hq, lens, T, splits):
    """Multi-query decode over the mixed pool: query token t of request b attends tokens
    0 .. L_b - T + t of each head in that head's own format."""
    dattn = _lib()
    case = W.Case("multi-mixed", B=len(lens), Hq=Hq, Hkv=len(spec), d=128, P=16, lens=lens,
                  seed=(sum(map(ord, spec)) + Hq + T + sum(lens)) % 1000 + 11)
    cache = _cache(case, spec)
    q = torch.stack([case.q(200 + t, DEV) for t in range(T)], dim=1).contiguous()
    out = torch.full((case.B, T, Hq, case.d), float("nan"), device=DEV)
    m_g = torch.full((case.B, T, Hq), float("nan"), device=DEV)
    e_g = torch.full((case.B, T, Hq), float("nan"), device=DEV)
    ws = dattn.Workspace(case.B, T * Hq, case.Hkv, case.d, num_splits=splits)
    dattn.dattn_decode_multi(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                             cache.seq_lens, out, ws, m_g=m_g, e_g=e_g, num_splits=splits,
                             dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    for b in range(case.B):
        L = cache.lens[b]
        Kd, Vd = _deq(*host_kv(case, b, L, DEV), spec)
        for t in range(T):
            rows = np.arange(max(0, L - T + t + 1), dtype=np.int64)
            for h in range(Hq):
                kvh = h // case.g
                r, rm, re = oracle.attention_f64(qb[b, t, h], Kd[:, kvh], Vd[:, kvh],
                                                 case.scale, rows=rows)
                tag = f"mixed multi b={b} t={t} h={h} ({spec[kvh]}-bit head)"
                assert_out_close(o[b, t, h], r, tag)
                assert_m_close(mg[b, t, h], rm, tag)
                assert_e_close(eg[b, t, h], re, tag)


def test_mixed_partial_then_merge():
    """Partials over 4 chunks of 1024 tokens of a mixed pool, then the merge."""
    dattn = _lib()
    spec = "48"
    case = W.Case("partial-mixed", B=1, Hq=8, Hkv=2, d=64, P=16, lens=[4096], seed=5)
    cache = _cache(case, spec)
    q = case.q(0, DEV)
    C, per = 4, 1024 // case.P
    chunk_req = torch.zeros(C, dtype=torch.int32, device=DEV)
    indptr = torch.arange(0, (C + 1) * per, per, dtype=torch.int32, device=DEV)
    pages = torch.arange(C * per, dtype=torch.int32, device=DEV)  # request-relative pages
    m = torch.empty(C, case.Hq, device=DEV)
    e = torch.empty_like(m)
    MA = torch.empty(C, case.Hq, case.d, device=DEV)
    dattn.dattn_partial(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                        chunk_req, indptr, pages, m, e, MA, dattn.Workspace(C, case.Hq, case.Hkv,
                                                                            case.d),
                        num_splits=9, dev_err=cache.dev_err)
    out, m_g, e_g = _outs(case)
    dattn.dattn_merge(torch.tensor([0, C], dtype=torch.int32, device=DEV), m, e, MA, out=out,
                      m_g=m_g, e_g=e_g)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    Kd, Vd = _deq(*host_kv(case, 0, 4096, DEV), spec)
    qb = oracle.bf16_bits(q)
    for h in range(case.Hq):
        kvh = h // case.g
        for c in range(C):
            rows = np.arange(c * 1024, (c + 1) * 1024)
            rm, re, rMA = oracle.partial_f64(qb[0, h], Kd[:, kvh], Vd[:, kvh], case.scale,
                                             rows=rows)
            assert_m_close(m[c, h].item(), rm, f"chunk {c} head {h}")
            assert_e_close(e[c, h].item(), re, f"chunk {c} head {h}")
            assert_out_close(MA[c, h].cpu().numpy() / e[c, h].item(), rMA / re,
                             f"chunk {c} head {h}")
    _check_dense(case, q, [4096], spec, out, m_g, e_g, "mixed merged")


@pytest.mark.parametrize("kinds,splits,phys", [
    ([1, 2, 1, 2], 0, True),    # the head-aligned split
    ([1, 2, 1, 2], 5, False),   # the balanced split
    ([2, 1, 0, 1], 0, True),    # a dense (8-bit) head among them
])
def test_mixed_sparse_decode_retrieval_8bit_streaming_4bit(kinds, splits, phys):
    """Block-sparse decode of a mixed pool in the layout §3.2.1 describes: retrieval and dense
    heads 8-bit, streaming heads 4-bit, with a reused selection while tokens are appended."""
    _lib()
    spec = "".join("4" if k == W.HEAD_STREAMING else "8" for k in kinds)
    case = W.Case("sparse-mixed", B=4, Hq=16, Hkv=4, d=128, P=64,
                  lens=[64 * 120 + 5, 3000, 12, 700], seed=23, head_kind=kinds, top_k=16,
                  sinks=4, local=8, n_highsim=6)
    cache = _cache(case, spec, with_stats=True)
    q0 = case.q(0, DEV)
    sel = torch.empty(case.B, case.Hkv, case.top_k, dtype=torch.int32, device=DEV)
    sel_phys = torch.empty_like(sel) if phys else None
    cache.select(q0, sel, cache.workspace(top_k=case.top_k), selected_phys=sel_phys)
    torch.cuda.synchronize()
    want_sel = sel.cpu().numpy()
    sp = cache.sparse_config(sel, sel_phys)
    ws = cache.workspace(num_splits=splits)
    for step in range(2):
        kn, vn = cache.new_tokens(1)
        cache.append(kn, vn)
        q = case.q(step + 1, DEV)
        out, m_g, e_g = _outs(case)
        cache.decode(q, out, ws, m_g=m_g, e_g=e_g, sparse=sp, num_splits=splits)
        torch.cuda.synchronize()
        assert int(cache.dev_err.item()) == 0

        def rows_of(b, kvh, L):
            return oracle.sparse_rows(kinds[kvh], L, case.P, want_sel[b, kvh], case.sinks,
                                      case.local)

        _check_dense(case, q, cache.lens, spec, out, m_g, e_g, f"step {step}", rows_of=rows_of)


def test_mixed_decode_flags_bad_pages_without_fault():
    """An unmapped page and a page outside the pool, in a mixed pool: both flagged, their
    tiles skipped in both formats' heads, the other tokens attended as the oracle does."""
    dattn = _lib()
    spec = "8448"
    case = W.Case("unm-mixed", B=1, Hq=4, Hkv=4, d=128, P=16, lens=[100], seed=4)
    cache = _cache(case, spec)
    cache.block_table[0, 2] = -1
    cache.block_table[0, 3] = case.num_pages + 5
    q = case.q(0, DEV)
    out, m_g, e_g = _outs(case)
    cache.decode(q, out, cache.workspace(), m_g=m_g, e_g=e_g)
    torch.cuda.synchronize()
    err = int(cache.dev_err.item())
    assert err & dattn.DEVERR["UNMAPPED_PAGE"] and err & dattn.DEVERR["PAGE_OOB"]
    rows = np.array([t for t in range(100) if t // 16 not in (2, 3)], np.int64)
    _check_dense(case, q, [100], spec, out, m_g, e_g, "bad pages",
                 rows_of=lambda b, kvh, L: rows)


@pytest.mark.parametrize("spec", ["4444", "8448"])
def test_mixed_and_4bit_pools_across_simulated_ranks(spec):
    """The cross-GPU merge over a quantized pool: each simulated rank's dattn_partial over the
    pages it holds, then dattn_merge_gathered, against the oracle over each head's
    dequantized rows."""
    _lib()
    import split_kv_decode_distattention_gb300 as dattn
    from split_kv_decode_distattention_gb300 import distributed as D
    case = W.Case("dist-q", B=3, Hq=8, Hkv=4, d=128, P=16, lens=[2000, 37, 700], seed=29)
    cache = _cache(case, spec)
    q = case.q(0, DEV)
    world = 3
    m, e, MA = D.stacked_partials(world, case.B, case.Hq, case.d, DEV)
    for r in range(world):
        pages = [D.rank_pages(-(-L // case.P), r, world, "strided") for L in case.lens]
        D.local_partials(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                         cache.seq_lens, pages, m[r], e[r], MA[r], dev_err=cache.dev_err)
    out, m_g, e_g = _outs(case)
    dattn.dattn_merge_gathered(m, e, MA, out=out, m_g=m_g, e_g=e_g, dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    _check_dense(case, q, case.lens, spec, out, m_g, e_g, f"{world} ranks")
