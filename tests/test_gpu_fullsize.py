"""Full-size parity of the five workloads, of mha-32k over the 8-bit and 4-bit pools and of
the 32K prefill, run in the launch configuration the benchmark times (automatic split
count). Outputs are checked against the oracle on sampled (request, head) pairs or query
rows, which the oracle computes one at a time. Properties that hold at any size are checked
on everything: the page-set merge equals the fused decode, and no device error is flagged.
The page selection is checked against the oracle's fp64 page scores: bit for bit where the
margin exceeds the fp32 error bound, else for validity."""
import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_distattention_gb300 import workloads as W

from _util import assert_e_close, assert_m_close, assert_out_close, check_selection

pytestmark = pytest.mark.gpu
# every workload is also run with seeds 1 and 2
SEEDS = [0, 1, 2]
DEV = "cuda"


def _lib():
    import split_kv_decode_distattention_gb300 as dattn
    dattn.load_library()
    return dattn


def _cache(case, **kw):
    from split_kv_decode_distattention_gb300.harness import PagedCache
    kw.setdefault("chunk_tokens", 32768)
    return PagedCache(case, DEV, **kw)


def _host_heads(case, b, L, heads, chunk=65536):
    """Token-ordered K, V of request b for the given KV heads: uint16 [len(heads)][L][d]."""
    Ks = np.empty((len(heads), L, case.d), np.uint16)
    Vs = np.empty_like(Ks)
    for t0 in range(0, L, chunk):
        t1 = min(L, t0 + chunk)
        K, V = case.kv(b, t0, t1, DEV)
        for i, h in enumerate(heads):
            Ks[i, t0:t1] = oracle.bf16_bits(K[:, h])
            Vs[i, t0:t1] = oracle.bf16_bits(V[:, h])
    return Ks, Vs


def _check_pairs(case, q, lens, out, m_g, e_g, pairs, what, rows_of=None):
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    by_b = {}
    for b, h in pairs:
        by_b.setdefault(b, set()).add(h // case.g)
    for b, kvhs in by_b.items():
        kvhs = sorted(kvhs)
        Ks, Vs = _host_heads(case, b, lens[b], kvhs)
        for bb, h in pairs:
            if bb != b:
                continue
            i = kvhs.index(h // case.g)
            rows = rows_of(b, h // case.g) if rows_of else None
            r, rm, re = oracle.attention(qb[b, h], Ks[i], Vs[i], case.scale, rows=rows)
            assert_out_close(o[b, h], r, f"{what} b={b} h={h}")
            assert_m_close(mg[b, h], rm, f"{what} b={b} h={h}")
            assert_e_close(eg[b, h], re, f"{what} b={b} h={h}")


def _step(cache, case, sparse=None):
    kn, vn = cache.new_tokens(1)
    cache.append(kn, vn)
    q = case.q(1, DEV)
    out = torch.empty(case.B, case.Hq, case.d, device=DEV)
    m_g = torch.empty(case.B, case.Hq, device=DEV)
    e_g = torch.empty_like(m_g)
    cache.decode(q, out, cache.workspace(), m_g=m_g, e_g=e_g, sparse=sparse)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    return q, out, m_g, e_g


@pytest.mark.parametrize("seed", SEEDS)
def test_mha_32k_batch8_full_size(seed):
    """Llama-2-7B MHA: batch 8, 32 heads, d 128, 32K tokens, shuffled 16-token pages."""
    _lib()
    case = W.mha_32k(seed=seed)
    cache = _cache(case)
    q, out, m_g, e_g = _step(cache, case)
    assert torch.isfinite(out).all()
    pairs = [(b, (7 * b + 3) % 32) for b in range(8)] + [(0, 0), (7, 31)]
    _check_pairs(case, q, cache.lens, out, m_g, e_g, pairs, "mha-32k")
    # the paged append wrote the new token where the block table says, bit for bit
    K1, V1 = case.kv(5, cache.lens[5] - 1, cache.lens[5], DEV)
    pos = cache.lens[5] - 1
    page = case.block_table[5][pos // case.P]
    assert torch.equal(cache.k_pool[page, :, pos % case.P], K1[0])
    assert torch.equal(cache.v_pool[page, :, pos % case.P], V1[0])


@pytest.mark.parametrize("seed", SEEDS)
def test_mha_1m_single_request_full_size(seed):
    """One request of 2^20 tokens, 32 heads MHA, 64 needle keys; split across all SMs."""
    _lib()
    case = W.mha_1m(seed=seed)
    cache = _cache(case)
    q, out, m_g, e_g = _step(cache, case)
    _check_pairs(case, q, cache.lens, out, m_g, e_g, [(0, 0), (0, 13), (0, 31)], "mha-1m")


@pytest.mark.parametrize("seed", SEEDS)
def test_gqa_ragged_full_size_and_page_set_merge(seed):
    """64 requests, 32 q / 8 KV heads, lengths 1K-256K; page-set partials merge to fused."""
    dattn = _lib()
    case = W.gqa_ragged(seed=seed)
    cache = _cache(case)
    q, out, m_g, e_g = _step(cache, case)
    order = np.argsort(case.lens)
    sample_b = [int(order[0]), int(order[31]), int(order[-1])]
    pairs = [(b, h) for b in sample_b for h in (0, 13, 31)]
    _check_pairs(case, q, cache.lens, out, m_g, e_g, pairs, "gqa-ragged")
    # every request split into 2-8 disjoint page sets: partials + merge == fused decode
    reqs, indptr, pages, ranges = [], [0], [], [0]
    for b in range(case.B):
        for s in case.page_sets_of(b, cache.lens[b]):
            reqs.append(b)
            pages.extend(s.tolist())
            indptr.append(len(pages))
        ranges.append(len(reqs))
    C = len(reqs)
    m = torch.empty(C, case.Hq, device=DEV)
    e = torch.empty_like(m)
    MA = torch.empty(C, case.Hq, case.d, device=DEV)
    dattn.dattn_partial(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                        torch.tensor(reqs, dtype=torch.int32, device=DEV),
                        torch.tensor(indptr, dtype=torch.int32, device=DEV),
                        torch.tensor(pages, dtype=torch.int32, device=DEV), m, e, MA,
                        dattn.Workspace(C, case.Hq, case.Hkv, case.d), dev_err=cache.dev_err)
    merged = torch.empty_like(out)
    mm = torch.empty_like(m_g)
    me = torch.empty_like(e_g)
    dattn.dattn_merge(torch.tensor(ranges, dtype=torch.int32, device=DEV), m, e, MA, out=merged,
                      m_g=mm, e_g=me)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    assert_out_close(merged.cpu().numpy(), out.cpu().numpy(), "page-set merge vs fused")
    np.testing.assert_allclose(mm.cpu().numpy(), m_g.cpu().numpy(), rtol=1e-5)
    np.testing.assert_allclose(me.cpu().numpy(), e_g.cpu().numpy(), rtol=1e-4)


@pytest.mark.parametrize("seed", SEEDS)
def test_sparse_512k_full_size(seed):
    """LServe block-sparse: batch 8, 32 q / 8 KV heads, 512K, 64-token pages, top-64."""
    _lib()
    case = W.sparse_512k(seed=seed)
    cache = _cache(case, with_stats=True)
    kn, vn = cache.new_tokens(1)
    cache.append(kn, vn)  # the first step of the window appends, then selects
    q0 = case.q(0, DEV)
    sel = torch.empty(case.B, case.Hkv, case.top_k, dtype=torch.int32, device=DEV)
    cache.select(q0, sel, cache.workspace(top_k=case.top_k))
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    got = sel.cpu().numpy()
    # non-retrieval rows are all -1; retrieval rows are sorted, distinct and in range
    for h in range(case.Hkv):
        if case.head_kind[h] != W.HEAD_RETRIEVAL:
            assert (got[:, h] == -1).all()
    qb = oracle.bf16_bits(q0)
    ret = [h for h in range(case.Hkv) if case.head_kind[h] == W.HEAD_RETRIEVAL]
    ambiguous = 0
    for b in (0, 3, 7):
        Ks, _ = _host_heads(case, b, cache.lens[b], ret)
        for i, h in enumerate(ret):
            score, bound = oracle.page_scores(qb[b, h * case.g:(h + 1) * case.g], Ks[i],
                                              cache.lens[b], case.P, with_bounds=True)
            ambiguous += not check_selection(got[b, h], score, bound, case.top_k,
                                             f"selection b={b} h={h}")
            # the seeded high-similarity pages are all selected
            assert set(case.highsim_pages(b, h).tolist()) <= set(got[b, h].tolist())
    print(f"sparse-512k selection: {3 * len(ret)} rows, {ambiguous} ambiguous within the "
          f"fp32 bound")
    # decode with the selection reused for the rest of the window
    sp = cache.sparse_config(sel)
    q, out, m_g, e_g = _step(cache, case, sparse=sp)

    def rows_of(b, kvh):
        return oracle.sparse_rows(case.head_kind[kvh], cache.lens[b], case.P, got[b, kvh],
                                  case.sinks, case.local)
    pairs = [(0, 0), (0, 17), (3, 8), (7, 15), (7, 31), (5, 20)]
    _check_pairs(case, q, cache.lens, out, m_g, e_g, pairs, "sparse-512k", rows_of=rows_of)


def _fused_step(cache, case, sparse=None):
    """The benchmark's step: the one-token append and the decode in one launch."""
    kn, vn = cache.new_tokens(1)
    q = case.q(1, DEV)
    out = torch.empty(case.B, case.Hq, case.d, device=DEV)
    m_g = torch.empty(case.B, case.Hq, device=DEV)
    e_g = torch.empty_like(m_g)
    cache.append_decode(kn, vn, q, out, cache.workspace(), m_g=m_g, e_g=e_g, sparse=sparse)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    assert cache.seq_lens.tolist() == cache.lens
    return q, out, m_g, e_g


def _select_full(case, cache):
    """The window's first step: append one token, then select (with the pool pages)."""
    kn, vn = cache.new_tokens(1)
    cache.append(kn, vn)
    sel = torch.empty(case.B, case.Hkv, case.top_k, dtype=torch.int32, device=DEV)
    phys = torch.empty_like(sel)
    cache.select(case.q(0, DEV), sel, cache.workspace(top_k=case.top_k), selected_phys=phys)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    return sel, phys


def test_sparse_512k_fused_step_full_size():
    """The benchmark's step: dattn_append_decode with the selector's pool pages, two steps
    of the window, sampled pairs against the oracle over the token sets of the selection."""
    _lib()
    case = W.sparse_512k(seed=0)
    cache = _cache(case, with_stats=True)
    sel, phys = _select_full(case, cache)
    got = sel.cpu().numpy()
    sp = cache.sparse_config(sel, phys)
    ws = cache.workspace()
    for step in (1, 2):
        kn, vn = cache.new_tokens(1)
        q = case.q(step, DEV)
        out = torch.empty(case.B, case.Hq, case.d, device=DEV)
        m_g = torch.empty(case.B, case.Hq, device=DEV)
        e_g = torch.empty_like(m_g)
        cache.append_decode(kn, vn, q, out, ws, m_g=m_g, e_g=e_g, sparse=sp)
        torch.cuda.synchronize()
        assert int(cache.dev_err.item()) == 0
        assert cache.seq_lens.tolist() == cache.lens

    def rows_of(b, kvh):
        return oracle.sparse_rows(case.head_kind[kvh], cache.lens[b], case.P, got[b, kvh],
                                  case.sinks, case.local)
    pairs = [(0, 1), (2, 9), (4, 18), (6, 27), (7, 30)]
    _check_pairs(case, q, cache.lens, out, m_g, e_g, pairs, "sparse-512k fused",
                 rows_of=rows_of)


def test_sparse_512k_mixed_pool_full_size():
    """sparse-512k over the mixed pool (retrieval and dense heads 8-bit, streaming heads
    4-bit), stepped as the benchmark steps it (the fused append and decode with the
    selector's pool pages): sampled pairs of both kinds against the oracle's float64
    attention over its own dequantized rows of each head's format."""
    dattn = _lib()
    case = W.sparse_512k(seed=1)
    formats = [dattn.KV_INT4 if k == W.HEAD_STREAMING else dattn.KV_FP8_E4M3
               for k in case.head_kind]
    cache = _cache(case, with_stats=True, kv_format=dattn.KV_MIXED, head_format=formats)
    sel, phys = _select_full(case, cache)
    got = sel.cpu().numpy()
    q, out, m_g, e_g = _fused_step(cache, case, sparse=cache.sparse_config(sel, phys))
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    kinds_seen = set()
    for b, h in [(0, 0), (1, 5), (3, 13), (6, 22), (7, 31)]:
        kvh = h // case.g
        kind = case.head_kind[kvh]
        kinds_seen.add(kind)
        if kind == W.HEAD_STREAMING:
            quant, deq = oracle.quantize_rows_int4, oracle.dequantize_rows_int4
        else:
            quant, deq = oracle.quantize_rows_fp8, oracle.dequantize_rows_fp8
        Ks, Vs = _host_heads(case, b, cache.lens[b], [kvh])
        Kd, Vd = deq(*quant(Ks[0])), deq(*quant(Vs[0]))
        rows = oracle.sparse_rows(kind, cache.lens[b], case.P, got[b, kvh], case.sinks,
                                  case.local)
        r, rm, re = oracle.attention_f64(qb[b, h], Kd, Vd, case.scale, rows=rows)
        assert_out_close(o[b, h], r, f"sparse-512k mixed b={b} h={h}")
        assert_m_close(mg[b, h], rm, f"sparse-512k mixed b={b} h={h}")
        assert_e_close(eg[b, h], re, f"sparse-512k mixed b={b} h={h}")
    assert {W.HEAD_RETRIEVAL, W.HEAD_STREAMING} <= kinds_seen


@pytest.mark.parametrize("fmt", ["fp8", "int4"])
def test_mha_32k_quantized_pools_full_size(fmt):
    """mha-32k over the 8-bit and the 4-bit pool: the append quantizes the seeded rows, and the
    benchmark's step (the fused append and decode) attends them; sampled pairs against the
    oracle's float64 attention over its own dequantized rows."""
    dattn = _lib()
    case = W.mha_32k(seed=0)
    kv_format = dattn.KV_FP8_E4M3 if fmt == "fp8" else dattn.KV_INT4
    quant, deq = ((oracle.quantize_rows_fp8, oracle.dequantize_rows_fp8) if fmt == "fp8" else
                  (oracle.quantize_rows_int4, oracle.dequantize_rows_int4))
    cache = _cache(case, kv_format=kv_format)
    q, out, m_g, e_g = _fused_step(cache, case)
    assert torch.isfinite(out).all()
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    for b, h in [(0, 0), (3, 17), (7, 31)]:
        Ks, Vs = _host_heads(case, b, cache.lens[b], [h])
        Kd, Vd = deq(*quant(Ks[0])), deq(*quant(Vs[0]))
        r, rm, re = oracle.attention_f64(qb[b, h], Kd, Vd, case.scale)
        assert_out_close(o[b, h], r, f"mha-32k {fmt} b={b} h={h}")
        assert_m_close(mg[b, h], rm, f"mha-32k {fmt} b={b} h={h}")
        assert_e_close(eg[b, h], re, f"mha-32k {fmt} b={b} h={h}")


@pytest.mark.parametrize("dense", [False, True])
def test_prefill_32k_full_size(dense):
    """The 32K prefill exactly as the benchmark runs it: one 32K-token chunk, 32 q / 8 KV
    heads, retrieval heads keeping a seeded 65% of the earlier blocks, streaming heads one
    sink and 16 local blocks (or every head causal). Sampled query rows across the chunk
    against the oracle's attention over their prefill rows."""
    dattn = _lib()
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.prefill_32k(seed=0)
    L = case.lens[0]
    cache = PagedCache(case, DEV, fill=False)
    q = case.prefill_queries(L, DEV)
    K, V = case.kv(0, 0, L, DEV)
    cache.append(K.unsqueeze(0).contiguous(), V.unsqueeze(0).contiguous())
    del K, V
    kinds = [0] * case.Hkv if dense else list(case.head_kind)
    lists = case.prefill_block_lists(W.PREFILL_KEEP)
    sinks, local = W.PREFILL_SINK_BLOCKS, W.PREFILL_LOCAL_BLOCKS
    sp = None
    if not dense:
        sp = dattn.PrefillSparseConfig(torch.tensor(kinds, dtype=torch.int8, device=DEV), sinks,
                                       local, torch.from_numpy(lists).to(DEV))
    out = torch.empty(1, L, case.Hq, case.d, device=DEV)
    m = torch.empty(1, L, case.Hq, device=DEV)
    e = torch.empty_like(m)
    dattn.dattn_prefill(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                        out, m, e, sparse=sp, dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    qb = oracle.bf16_bits(q[0, [0, 64, 5000, 20000, L - 1]])
    ts = [0, 64, 5000, 20000, L - 1]
    heads = [0, 5, 13, 18, 27, 31]  # KV heads 0, 1, 3 (retrieval) and 4, 6, 7 (streaming)
    kvhs = sorted({h // case.g for h in heads})
    Ks, Vs = _host_heads(case, 0, L, kvhs)
    o, mm, ee = out[0, ts].cpu().numpy(), m[0, ts].cpu().numpy(), e[0, ts].cpu().numpy()
    for i, t in enumerate(ts):
        for h in heads:
            kvh = h // case.g
            blocks = lists[0, kvh, t // 64] if kinds[kvh] == W.HEAD_RETRIEVAL else None
            rows = oracle.prefill_rows(kinds[kvh], L, L, t, sinks, local, blocks=blocks)
            j = kvhs.index(kvh)
            r, rm, re = oracle.attention(qb[i, h], Ks[j], Vs[j], case.scale, rows=rows)
            tag = f"prefill-32k{' dense' if dense else ''} t={t} h={h}"
            assert_out_close(o[i, h], r, tag)
            assert_m_close(mm[i, h], rm, tag)
            assert_e_close(ee[i, h], re, tag)
