"""GPU parity of every entry point against the oracle, at sizes the oracle finishes in
seconds. The sizes span several tiles, CTAs and pages, with ragged tails and the
degenerate cases (empty requests, one token, page and tile boundaries)."""
import math

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_distattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _lib():
    import split_kv_decode_distattention_gb300 as dattn
    dattn.load_library()
    return dattn


def _cache(case, **kw):
    from split_kv_decode_distattention_gb300.harness import PagedCache
    return PagedCache(case, DEV, **kw)


from _util import (assert_e_close, assert_m_close, assert_out_close, check_dense,  # noqa: E402
                   check_selection, host_kv)


# ---------------------------------------------------------------- paged append + statistics

@pytest.mark.parametrize("d,P,chunk", [(128, 16, 37), (64, 64, 200), (128, 64, 5), (64, 16, 64)])
def test_append_layout_and_stats_bit_exact(d, P, chunk):
    _lib()
    case = W.Case("append", B=3, Hq=4, Hkv=2, d=d, P=P, lens=[0, 131, 290], seed=3)
    cache = _cache(case, with_stats=True, fill=False, zero_pool=True, chunk_tokens=chunk)
    cache.fill()
    for _ in range(3):  # decode-style single-token appends for every request
        kn, vn = cache.new_tokens(1)
        cache.append(kn, vn)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    lens = cache.lens
    assert cache.seq_lens.tolist() == lens
    kp = np.zeros((case.num_pages, case.Hkv, P, d), np.uint16)
    vp = np.zeros_like(kp)
    st = np.zeros((case.num_pages, case.Hkv, P // 16, 2, d), np.uint16)
    for b in range(case.B):
        K, V = host_kv(case, b, lens[b], DEV)
        assert oracle.kv_write(kp, vp, case.block_table[b], case.num_pages, K, V, 0) == 0
        for h in range(case.Hkv):
            for t0 in range(0, lens[b], 16):
                kmax, kmin = oracle.logical_page_stats(K[:, h].copy(), t0, min(t0 + 16, lens[b]))
                page = case.block_table[b][t0 // P]
                st[page, h, (t0 % P) // 16, 0] = kmax
                st[page, h, (t0 % P) // 16, 1] = kmin
    np.testing.assert_array_equal(oracle.bf16_bits(cache.k_pool), kp)
    np.testing.assert_array_equal(oracle.bf16_bits(cache.v_pool), vp)
    np.testing.assert_array_equal(oracle.bf16_bits(cache.stats), st)


def test_append_flags_unmapped_pages_and_skips_them():
    dattn = _lib()
    case = W.Case("bad", B=1, Hq=2, Hkv=1, d=64, P=16, lens=[40], seed=1)
    case.block_table[0, 1] = -1  # tokens 16..31 have no page
    cache = _cache(case, fill=False, zero_pool=True)
    cache.fill()
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) & dattn.DEVERR["UNMAPPED_PAGE"]
    assert cache.seq_lens.tolist() == [40]


# ---------------------------------------------------------------- fused dense decode

DENSE_CASES = [
    # (d, Hq, Hkv, P, lens, num_splits)
    (128, 4, 4, 16, [1, 15, 16, 17], 0),
    (128, 8, 2, 16, [1000, 33, 0, 2500], 7),
    (64, 8, 2, 16, [4096], 0),
    (128, 32, 8, 16, [700, 1300, 31], 64),
    (128, 8, 1, 64, [257, 64, 1], 3),
    (64, 16, 2, 64, [999, 1, 2048], 1),
    (128, 2, 2, 32, [480, 500], 2),
    (128, 6, 3, 16, [5000], 0),
    # more CTAs than tiles: only the first W CTAs take work
    (128, 4, 4, 16, [1, 15, 16, 17], 500),
    (64, 8, 2, 64, [100, 3], 1000),
]


@pytest.mark.parametrize("d,Hq,Hkv,P,lens,splits", DENSE_CASES)
def test_decode_dense_matches_oracle(d, Hq, Hkv, P, lens, splits):
    _lib()
    case = W.Case("dense", B=len(lens), Hq=Hq, Hkv=Hkv, d=d, P=P, lens=lens,
                  seed=hash((d, Hq, P, tuple(lens))) % 1000)
    cache = _cache(case)
    q = case.q(0, DEV)
    out = torch.full((case.B, Hq, d), float("nan"), device=DEV)
    m_g = torch.full((case.B, Hq), float("nan"), device=DEV)
    e_g = torch.full((case.B, Hq), float("nan"), device=DEV)
    ws = cache.workspace(num_splits=splits)
    cache.decode(q, out, ws, m_g=m_g, e_g=e_g, num_splits=splits)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    check_dense(case, q, cache.lens, out, m_g, e_g, DEV)
    # the workspace counters are back to zero: a second call gives the same bits
    out2 = torch.empty_like(out)
    cache.decode(q, out2, ws, num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_decode_split_count_does_not_change_result_beyond_tolerance():
    _lib()
    case = W.Case("splits", B=2, Hq=8, Hkv=2, d=128, P=16, lens=[3000, 1777], seed=9)
    cache = _cache(case)
    q = case.q(0, DEV)
    outs = []
    for splits in (1, 2, 5, 16, 100, 0):
        out = torch.empty(case.B, case.Hq, case.d, device=DEV)
        cache.decode(q, out, cache.workspace(num_splits=splits), num_splits=splits)
        outs.append(out.cpu().numpy())
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert_out_close(o, outs[0], "split count")
    check_dense(case, q, cache.lens, torch.as_tensor(outs[-1]), None, None, DEV)


def test_decode_after_append_step_includes_new_token():
    _lib()
    case = W.Case("step", B=3, Hq=8, Hkv=2, d=128, P=16, lens=[64, 100, 15], seed=4)
    cache = _cache(case)
    ws = cache.workspace()
    for step in range(3):
        kn, vn = cache.new_tokens(1)
        cache.append(kn, vn)
        q = case.q(step, DEV)
        out = torch.empty(case.B, case.Hq, case.d, device=DEV)
        cache.decode(q, out, ws)
        torch.cuda.synchronize()
        check_dense(case, q, cache.lens, out, None, None, DEV, what=f"step {step}")


# ---------------------------------------------------------------- partial + merge

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dense_tiny_partial_then_merge(seed):
    """Batch 1, 8 q / 2 KV heads, d 64, 4096 tokens, 4 chunks of 1024 (identity table)."""
    dattn = _lib()
    case = W.dense_tiny(seed=seed)
    cache = _cache(case)
    q = case.q(0, DEV)
    pages_per_chunk = case.chunk_tokens // case.P
    C = 4
    chunk_req = torch.zeros(C, dtype=torch.int32, device=DEV)
    indptr = torch.arange(0, (C + 1) * pages_per_chunk, pages_per_chunk, dtype=torch.int32,
                          device=DEV)
    pages = torch.arange(C * pages_per_chunk, dtype=torch.int32, device=DEV)
    m = torch.empty(C, case.Hq, device=DEV)
    e = torch.empty_like(m)
    MA = torch.empty(C, case.Hq, case.d, device=DEV)
    ws = dattn.Workspace(C, case.Hq, case.Hkv, case.d)
    dattn.dattn_partial(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                        chunk_req, indptr, pages, m, e, MA, ws, dev_err=cache.dev_err)
    out = torch.empty(1, case.Hq, case.d, device=DEV)
    m_g = torch.empty(1, case.Hq, device=DEV)
    e_g = torch.empty_like(m_g)
    ci = torch.tensor([0, C], dtype=torch.int32, device=DEV)
    dattn.dattn_merge(ci, m, e, MA, out=out, m_g=m_g, e_g=e_g)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    K, V = host_kv(case, 0, 4096, DEV)
    qb = oracle.bf16_bits(q)
    for h in range(case.Hq):
        kvh = h // case.g
        for c in range(C):
            rows = np.arange(c * 1024, (c + 1) * 1024)
            rm, re, rMA = oracle.partial(qb[0, h], K[:, kvh].copy(), V[:, kvh].copy(),
                                         case.scale, rows=rows)
            assert_m_close(m[c, h].item(), rm, f"chunk {c} head {h}")
            assert_e_close(e[c, h].item(), re, f"chunk {c} head {h}")
            # MA_j = e_j * (normalised chunk output): compare normalised values
            assert_out_close(MA[c, h].cpu().numpy() / e[c, h].item(), rMA / re,
                             f"chunk {c} head {h}")
    check_dense(case, q, [4096], out, m_g, e_g, DEV, what="merged")


def test_partial_flags_chunk_page_ranges_outside_the_list():
    """A chunk whose page range starts below 0, or ends past chunk_page_indptr[C], is flagged
    with CHUNK_OOB and left empty (m = -inf, e = 0, MA = 0); its pages are never read. The
    valid chunk beside it is computed as usual."""
    dattn = _lib()
    case = W.Case("badchunk", B=1, Hq=4, Hkv=2, d=64, P=16, lens=[160], seed=4)
    cache = _cache(case)
    q = case.q(0, DEV)
    # list ranges: chunk 0 [0, 3) is valid; chunk 1 [3, -2) has a negative count; chunk 2
    # [-2, 7) starts before the list and ends past indptr[C] = 5; chunk 3 [7, 5) lies past the
    # end. Only chunk 0 is computed.
    C = 4
    chunk_req = torch.zeros(C, dtype=torch.int32, device=DEV)
    indptr = torch.tensor([0, 3, -2, 7, 5], dtype=torch.int32, device=DEV)
    pages = torch.tensor([0, 1, 2, 5, 6], dtype=torch.int32, device=DEV)
    m = torch.empty(C, case.Hq, device=DEV)
    e = torch.empty_like(m)
    MA = torch.empty(C, case.Hq, case.d, device=DEV)
    ws = dattn.Workspace(C, case.Hq, case.Hkv, case.d)
    dattn.dattn_partial(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                        chunk_req, indptr, pages, m, e, MA, ws, dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) & dattn.DEVERR["CHUNK_OOB"]
    for c in (1, 2, 3):
        assert (m[c] == -math.inf).all() and (e[c] == 0).all() and (MA[c] == 0).all(), c
    K, V = host_kv(case, 0, 160, DEV)
    qb = oracle.bf16_bits(q)
    for h in range(case.Hq):
        rm, re, rMA = oracle.partial(qb[0, h], K[:, h // case.g].copy(),
                                     V[:, h // case.g].copy(), case.scale, rows=np.arange(48))
        assert_m_close(m[0, h].item(), rm, f"chunk 0 head {h}")
        assert_e_close(e[0, h].item(), re, f"chunk 0 head {h}")
        assert_out_close(MA[0, h].cpu().numpy() / e[0, h].item(), rMA / re, f"chunk 0 head {h}")


def test_page_sets_partials_merge_to_fused_decode():
    """Ragged GQA batch; each request's pages split into 2-8 disjoint non-contiguous sets."""
    dattn = _lib()
    case = W.gqa_ragged(seed=1, B=5, lo=40, hi=3000)
    cache = _cache(case)
    q = case.q(0, DEV)
    reqs, indptr, pages = [], [0], []
    ranges = [0]
    for b in range(case.B):
        for s in case.page_sets_of(b):
            reqs.append(b)
            pages.extend(s.tolist())
            indptr.append(len(pages))
        ranges.append(len(reqs))
    C = len(reqs)
    chunk_req = torch.tensor(reqs, dtype=torch.int32, device=DEV)
    indptr_t = torch.tensor(indptr, dtype=torch.int32, device=DEV)
    pages_t = torch.tensor(pages, dtype=torch.int32, device=DEV)
    m = torch.empty(C, case.Hq, device=DEV)
    e = torch.empty_like(m)
    MA = torch.empty(C, case.Hq, case.d, device=DEV)
    ws = dattn.Workspace(C, case.Hq, case.Hkv, case.d)
    dattn.dattn_partial(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                        chunk_req, indptr_t, pages_t, m, e, MA, ws, num_splits=11,
                        dev_err=cache.dev_err)
    out = torch.empty(case.B, case.Hq, case.d, device=DEV)
    m_g = torch.empty(case.B, case.Hq, device=DEV)
    e_g = torch.empty_like(m_g)
    dattn.dattn_merge(torch.tensor(ranges, dtype=torch.int32, device=DEV), m, e, MA, out=out,
                      m_g=m_g, e_g=e_g)
    fused = torch.empty_like(out)
    fm = torch.empty_like(m_g)
    fe = torch.empty_like(e_g)
    cache.decode(q, fused, cache.workspace(), m_g=fm, e_g=fe)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    check_dense(case, q, cache.lens, out, m_g, e_g, DEV, what="page-set merge")
    assert_out_close(out.cpu().numpy(), fused.cpu().numpy(), "merge vs fused")
    np.testing.assert_allclose(m_g.cpu().numpy(), fm.cpu().numpy(), rtol=1e-5)
    np.testing.assert_allclose(e_g.cpu().numpy(), fe.cpu().numpy(), rtol=1e-4)


def test_nested_merge_of_merged_partials():
    dattn = _lib()
    case = W.Case("nest", B=1, Hq=4, Hkv=4, d=128, P=16, lens=[1600], seed=6, shuffle=False)
    cache = _cache(case)
    q = case.q(0, DEV)
    C = 10  # chunks of 10 pages
    chunk_req = torch.zeros(C, dtype=torch.int32, device=DEV)
    indptr = torch.arange(0, 101, 10, dtype=torch.int32, device=DEV)
    pages = torch.arange(100, dtype=torch.int32, device=DEV)
    m = torch.empty(C, 4, device=DEV)
    e = torch.empty_like(m)
    MA = torch.empty(C, 4, 128, device=DEV)
    dattn.dattn_partial(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                        chunk_req, indptr, pages, m, e, MA, dattn.Workspace(C, 4, 4, 128))
    # level 1: chunks {0..3}, {4}, {5..9} -> 3 merged partials; level 2: one merge
    m1 = torch.empty(3, 4, device=DEV)
    e1 = torch.empty_like(m1)
    MA1 = torch.empty(3, 4, 128, device=DEV)
    dattn.dattn_merge(torch.tensor([0, 4, 5, 10], dtype=torch.int32, device=DEV), m, e, MA,
                      m_g=m1, e_g=e1, MA_g=MA1)
    out = torch.empty(1, 4, 128, device=DEV)
    m2 = torch.empty(1, 4, device=DEV)
    e2 = torch.empty_like(m2)
    dattn.dattn_merge(torch.tensor([0, 3], dtype=torch.int32, device=DEV), m1, e1, MA1, out=out,
                      m_g=m2, e_g=e2)
    torch.cuda.synchronize()
    check_dense(case, q, [1600], out, m2, e2, DEV, what="nested merge")


def test_merge_of_empty_chunks():
    dattn = _lib()
    m = torch.full((3, 2), -math.inf, device=DEV)
    e = torch.zeros(3, 2, device=DEV)
    MA = torch.zeros(3, 2, 64, device=DEV)
    m[1, 0], e[1, 0] = 0.5, 2.0
    MA[1, 0] = 3.0
    out = torch.full((2, 2, 64), 7.0, device=DEV)
    m_g = torch.empty(2, 2, device=DEV)
    e_g = torch.empty(2, 2, device=DEV)
    dattn.dattn_merge(torch.tensor([0, 2, 3], dtype=torch.int32, device=DEV), m, e, MA, out=out,
                      m_g=m_g, e_g=e_g)
    torch.cuda.synchronize()
    assert torch.allclose(out[0, 0], torch.full((64,), 1.5, device=DEV))
    assert m_g[0, 0].item() == 0.5 and e_g[0, 0].item() == 2.0
    assert (out[0, 1] == 0).all() and m_g[0, 1].item() == -math.inf and e_g[0, 1].item() == 0
    assert (out[1] == 0).all()


# ---------------------------------------------------------------- page selection

def _check_selection(case, cache, q, sel):
    """Checks every row of a GPU selection against the oracle's fp64 page scores and their
    fp32 error bounds (check_selection); rows of other head kinds must be all -1. Prints how
    many retrieval rows were ambiguous (margin within the bounds) and checked for validity
    only."""
    qb = oracle.bf16_bits(q)
    got = sel.cpu().numpy()
    rows = ambiguous = 0
    for b in range(case.B):
        K, _ = host_kv(case, b, cache.lens[b], DEV)
        for h in range(case.Hkv):
            if case.head_kind[h] != W.HEAD_RETRIEVAL:
                assert (got[b, h] == -1).all(), f"b={b} h={h}: row of a non-retrieval head"
                continue
            score, bound = oracle.page_scores(qb[b, h * case.g:(h + 1) * case.g],
                                              K[:, h].copy(), cache.lens[b], case.P,
                                              with_bounds=True)
            rows += 1
            ambiguous += not check_selection(got[b, h], score, bound, case.top_k,
                                             f"selection b={b} h={h}")
    print(f"page selection: {rows} retrieval rows, {ambiguous} ambiguous within the fp32 bound")
    return got


@pytest.mark.parametrize("P,d,lens,top_k,splits", [
    (64, 128, [64 * 300 + 17, 64 * 90], 16, 0),
    (64, 128, [5000, 20], 64, 7),
    (16, 64, [3000, 1, 777], 32, 0),
    (64, 64, [64 * 40], 64, 3),  # top_k covers every page
    (64, 128, [64 * 50 + 3, 64 * 7], 8, 4000),  # more CTAs than pages
    (256, 128, [256 * 30 + 100, 256 * 3], 5, 0),  # 16 logical pages per page, odd top_k
    (32, 128, [32 * 500 + 7], 100, 5),  # 2 logical pages per page, top_k not a power of two
    (64, 128, [64 * 600, 64 * 300 + 1], 256, 0),  # the largest top_k
    (128, 64, [128 * 40 + 77, 129], 1, 2),  # top-1
])
def test_page_select_matches_fp64_scores(P, d, lens, top_k, splits):
    _lib()
    case = W.Case("sel", B=len(lens), Hq=16, Hkv=4, d=d, P=P, lens=lens, seed=P + d + top_k,
                  head_kind=[1, 2, 1, 0], top_k=top_k, n_highsim=8)
    cache = _cache(case, with_stats=True)
    q = case.q(0, DEV)
    sel = torch.full((case.B, case.Hkv, top_k), 12345, dtype=torch.int32, device=DEV)
    cache.select(q, sel, cache.workspace(top_k=top_k, num_splits=splits), num_splits=splits)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    _check_selection(case, cache, q, sel)


# ---------------------------------------------------------------- block-sparse decode

@pytest.mark.parametrize("P,lens,splits", [(64, [64 * 200 + 5, 3000, 12, 5], 0),
                                           (16, [2000, 700], 9)])
def test_sparse_decode_matches_oracle_token_sets(P, lens, splits):
    _lib()
    case = W.Case("sparse", B=len(lens), Hq=16, Hkv=4, d=128, P=P, lens=lens, seed=21,
                  head_kind=[1, 2, 1, 2], top_k=16, sinks=4, local=8, n_highsim=6)
    cache = _cache(case, with_stats=True)
    q0 = case.q(0, DEV)
    sel = torch.empty(case.B, case.Hkv, case.top_k, dtype=torch.int32, device=DEV)
    cache.select(q0, sel, cache.workspace(top_k=case.top_k))
    torch.cuda.synchronize()
    want_sel = _check_selection(case, cache, q0, sel)  # the validated GPU rows
    sp = cache.sparse_config(sel)
    ws = cache.workspace(num_splits=splits)
    for step in range(3):  # the selection is reused while tokens are appended
        kn, vn = cache.new_tokens(1)
        cache.append(kn, vn)
        q = case.q(step, DEV)
        out = torch.empty(case.B, case.Hq, case.d, device=DEV)
        m_g = torch.empty(case.B, case.Hq, device=DEV)
        e_g = torch.empty_like(m_g)
        cache.decode(q, out, ws, m_g=m_g, e_g=e_g, sparse=sp, num_splits=splits)
        torch.cuda.synchronize()
        assert int(cache.dev_err.item()) == 0
        qb = oracle.bf16_bits(q)
        o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
        for b in range(case.B):
            L = cache.lens[b]
            K, V = host_kv(case, b, L, DEV)
            for h in range(case.Hq):
                kvh = h // case.g
                rows = oracle.sparse_rows(case.head_kind[kvh], L, P, want_sel[b, kvh],
                                          case.sinks, case.local)
                r, rm, re = oracle.attention(qb[b, h], K[:, kvh].copy(), V[:, kvh].copy(),
                                             case.scale, rows=rows)
                assert_out_close(o[b, h], r, f"step {step} b={b} h={h}")
                assert_m_close(mg[b, h], rm, f"step {step} b={b} h={h}")
                assert_e_close(eg[b, h], re, f"step {step} b={b} h={h}")


def test_sparse_with_all_pages_selected_equals_dense():
    dattn = _lib()
    case = W.Case("alltop", B=2, Hq=8, Hkv=2, d=128, P=64, lens=[900, 1000], seed=5,
                  head_kind=[1, 1], top_k=32)
    cache = _cache(case, with_stats=True)
    q = case.q(0, DEV)
    sel = torch.empty(case.B, case.Hkv, 32, dtype=torch.int32, device=DEV)
    cache.select(q, sel, cache.workspace(top_k=32))
    dense = torch.empty(case.B, case.Hq, case.d, device=DEV)
    sparse = torch.empty_like(dense)
    cache.decode(q, dense, cache.workspace())
    cache.decode(q, sparse, cache.workspace(), sparse=cache.sparse_config(sel))
    torch.cuda.synchronize()
    assert_out_close(sparse.cpu().numpy(), dense.cpu().numpy(), "all pages selected")


# ---------------------------------------------------------------- device error handling

def test_decode_flags_unmapped_page_without_fault():
    dattn = _lib()
    case = W.Case("unm", B=1, Hq=4, Hkv=4, d=128, P=16, lens=[100], seed=2)
    cache = _cache(case)
    cache.block_table[0, 2] = -1
    cache.block_table[0, 3] = case.num_pages + 5
    q = case.q(0, DEV)
    out = torch.empty(1, 4, 128, device=DEV)
    cache.decode(q, out, cache.workspace())
    torch.cuda.synchronize()
    err = int(cache.dev_err.item())
    assert err & dattn.DEVERR["UNMAPPED_PAGE"] and err & dattn.DEVERR["PAGE_OOB"]
    assert torch.isfinite(out).all()
    # the result is attention over the tokens whose pages stayed mapped
    K, V = host_kv(case, 0, 100, DEV)
    rows = [t for t in range(100) if t // 16 not in (2, 3)]
    qb = oracle.bf16_bits(q)
    for h in range(4):
        r, _, _ = oracle.attention(qb[0, h], K[:, h].copy(), V[:, h].copy(), case.scale,
                                   rows=rows)
        assert_out_close(out[0, h].cpu().numpy(), r, f"head {h}")


def test_decode_length_beyond_table_is_flagged_and_clamped():
    dattn = _lib()
    case = W.Case("long", B=1, Hq=2, Hkv=2, d=64, P=16, lens=[50], seed=2, reserve_tokens=0)
    cache = _cache(case)
    cache.seq_lens.fill_(10 ** 6)
    out = torch.empty(1, 2, 64, device=DEV)
    cache.decode(case.q(0, DEV), out, cache.workspace())
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) & dattn.DEVERR["LEN_OOB"]


@pytest.mark.parametrize("Hq,Hkv,d,P", [(16, 2, 128, 64), (8, 8, 128, 16), (24, 3, 64, 64),
                                       (8, 1, 64, 128)])
def test_page_select_matches_fp64_scores_group_sizes(Hq, Hkv, d, P):
    """GQA groups of 8 (8-channel chunks), 1 and 3, and 128-token pages (8 logical pages)."""
    _lib()
    kinds = [1] * Hkv
    case = W.Case("selg", B=2, Hq=Hq, Hkv=Hkv, d=d, P=P, lens=[P * 70 + 9, P * 33], seed=Hq + P,
                  head_kind=kinds, top_k=16, n_highsim=4)
    cache = _cache(case, with_stats=True)
    q = case.q(0, DEV)
    sel = torch.full((case.B, case.Hkv, 16), 7777, dtype=torch.int32, device=DEV)
    cache.select(q, sel, cache.workspace(top_k=16))
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    _check_selection(case, cache, q, sel)
