"""GPU parity of the quantized KV paths: the 8-bit pool (FP8 E4M3 codes) and the 4-bit pool
(symmetric integer codes, two per byte), each with one fp32 scale per row.

The append is compared bit for bit with the oracle's write of the same bf16 inputs in the
same format: codes, scales and the logical-page statistics. Every attention result is
compared with the oracle's float64 attention over the oracle's own dequantized values
(code * scale), never over anything read back from the GPU pool. The tolerance is the bf16
path's.
"""
import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_distattention_gb300 import workloads as W

from _util import assert_e_close, assert_m_close, assert_out_close, check_selection, host_kv

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _lib():
    import split_kv_decode_distattention_gb300 as dattn
    dattn.load_library()
    return dattn


FORMATS = ["fp8", "int4"]


def _cache(case, fmt, **kw):
    from split_kv_decode_distattention_gb300 import KV_FP8_E4M3, KV_INT4
    from split_kv_decode_distattention_gb300.harness import PagedCache
    return PagedCache(case, DEV, kv_format=KV_INT4 if fmt == "int4" else KV_FP8_E4M3, **kw)


def _quant(fmt):
    """The oracle's row quantizer, dequantizer and paged write of a format."""
    if fmt == "int4":
        return oracle.quantize_rows_int4, oracle.dequantize_rows_int4, oracle.kv_write_int4
    return oracle.quantize_rows_fp8, oracle.dequantize_rows_fp8, oracle.kv_write_fp8


def _deq(K, V, fmt):
    """The oracle's round trip of token-ordered bf16 rows [L][Hkv][d] (float64)."""
    quant, deq, _ = _quant(fmt)
    kc, ks = quant(K)
    vc, vs = quant(V)
    return deq(kc, ks), deq(vc, vs)


def _ref_dense(case, q, lens, fmt, kv=None):
    """Oracle attention of every (b, h) over the dequantized tokens 0..L-1."""
    qb = oracle.bf16_bits(q)
    res = {}
    for b in range(case.B):
        K, V = kv[b] if kv is not None else host_kv(case, b, lens[b], DEV)
        Kd, Vd = _deq(K, V, fmt)
        for h in range(case.Hq):
            kvh = h // case.g
            res[(b, h)] = oracle.attention_f64(qb[b, h], Kd[:, kvh], Vd[:, kvh], case.scale)
    return res


def _check(res, out, m_g, e_g, lens, what):
    o = out.cpu().numpy()
    mg = m_g.cpu().numpy() if m_g is not None else None
    eg = e_g.cpu().numpy() if e_g is not None else None
    for (b, h), (r, rm, re) in res.items():
        assert_out_close(o[b, h], r, f"{what} b={b} h={h} L={lens[b]}")
        if mg is not None:
            assert_m_close(mg[b, h], rm, f"{what} b={b} h={h}")
            assert_e_close(eg[b, h], re, f"{what} b={b} h={h}")


def _oracle_pool(case, lens, fmt, kv=None):
    """Codes, scales and statistics the oracle writes for every request's tokens."""
    P, d = case.P, case.d
    write = _quant(fmt)[2]
    kp = np.zeros((case.num_pages, case.Hkv, P, d // 2 if fmt == "int4" else d), np.uint8)
    vp = np.zeros_like(kp)
    ks = np.zeros((case.num_pages, case.Hkv, P), np.float32)
    vs = np.zeros_like(ks)
    st = np.zeros((case.num_pages, case.Hkv, P // 16, 2, d), np.uint16)
    for b in range(case.B):
        K, V = kv[b] if kv is not None else host_kv(case, b, lens[b], DEV)
        assert write(kp, vp, ks, vs, P, case.block_table[b], case.num_pages, K, V, 0) == 0
        for h in range(case.Hkv):
            for t0 in range(0, lens[b], 16):
                kmax, kmin = oracle.logical_page_stats(K[:, h].copy(), t0, min(t0 + 16, lens[b]))
                page = case.block_table[b][t0 // P]
                st[page, h, (t0 % P) // 16, 0] = kmax
                st[page, h, (t0 % P) // 16, 1] = kmin
    return kp, vp, ks, vs, st


def _assert_pool(cache, want):
    kp, vp, ks, vs, st = want
    np.testing.assert_array_equal(cache.k_pool.cpu().numpy(), kp)
    np.testing.assert_array_equal(cache.v_pool.cpu().numpy(), vp)
    # scales bit for bit; the pool keeps them as [page][head][P/16][K, V][16]
    sc = cache.kv_scale.cpu().numpy()
    n, h, P = ks.shape
    gk = sc[:, :, :, 0, :].reshape(n, h, P)
    gv = sc[:, :, :, 1, :].reshape(n, h, P)
    np.testing.assert_array_equal(gk.view(np.uint32), ks.view(np.uint32))
    np.testing.assert_array_equal(gv.view(np.uint32), vs.view(np.uint32))
    if cache.stats is not None:
        np.testing.assert_array_equal(oracle.bf16_bits(cache.stats), st)


# ---------------------------------------------------------------- quantized append

@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("d,P,chunk", [(128, 16, 37), (64, 64, 200), (128, 64, 5), (64, 16, 64)])
def test_quant_append_codes_scales_and_stats_bit_exact(fmt, d, P, chunk):
    _lib()
    case = W.Case("append8", B=3, Hq=4, Hkv=2, d=d, P=P, lens=[0, 131, 290], seed=3)
    cache = _cache(case, fmt, with_stats=True, fill=False, zero_pool=True, chunk_tokens=chunk)
    cache.fill()
    for _ in range(3):  # decode-style single-token appends for every request
        kn, vn = cache.new_tokens(1)
        cache.append(kn, vn)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    assert cache.seq_lens.tolist() == cache.lens
    _assert_pool(cache, _oracle_pool(case, cache.lens, fmt))


def _special_rows(Hkv, d, T, seed):
    """bf16 rows that reach the corners of the formats: zero rows, -0, rows whose small
    elements fall to E4M3 subnormals or to zero, exact ties of both formats, and a wide range
    of row scales."""
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, Hkv, d)).astype(np.float32)
    x *= np.exp2(rng.integers(-30, 30, size=(T, Hkv, 1))).astype(np.float32)  # row scales
    x[0] = 0.0                               # all-zero rows: scale 0, +0 codes
    x[1, :, 0] = -0.0
    x[1, :, 1:] = 0.0                        # a row of zeros with one -0
    x[2, :, :] = 1e-3
    x[2, :, 0] = 448.0                       # small elements: subnormal codes
    x[3, :, :] = 1e-6
    x[3, :, 0] = -1000.0                     # elements far below the smallest subnormal
    x[4, :, :] = np.float32(1.0 + 1.0 / 16)  # halfway between two codes after scaling...
    x[4, :, 0] = 448.0                       # ...by 1: ties go to the even code
    x[5, :, :] = rng.choice([-3.0, 3.0], size=(Hkv, d))
    x[6, :, :] = rng.choice([0.5, 1.5, 2.5, -0.5, -1.5, -6.5], size=(Hkv, d))
    x[6, :, 0] = 7.0                         # 4-bit scale 1: every element is a tie
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("fmt", FORMATS)
def test_quant_append_corner_rows_bit_exact(fmt):
    dattn = _lib()
    case = W.Case("corner8", B=1, Hq=2, Hkv=2, d=128, P=16, lens=[0], seed=1, shuffle=True,
                  reserve_tokens=64)
    cache = _cache(case, fmt, fill=False, zero_pool=True)
    K = _special_rows(2, 128, 40, 7)
    V = _special_rows(2, 128, 40, 8)
    dattn.dattn_kv_append(cache.layout, cache.k_pool, cache.v_pool, None,
                          K.unsqueeze(0).to(DEV), V.unsqueeze(0).to(DEV), cache.seq_lens,
                          cache.dev_err)
    cache.lens = [40]
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    kv = [(oracle.bf16_bits(K), oracle.bf16_bits(V))]
    _assert_pool(cache, _oracle_pool(case, [40], fmt, kv=kv))


# ---------------------------------------------------------------- quantized fused dense decode

FP8_DENSE_CASES = [
    # (d, Hq, Hkv, P, lens, num_splits)
    (128, 4, 4, 16, [1, 15, 16, 17], 0),
    (128, 8, 2, 16, [1000, 33, 0, 2500], 7),
    (64, 8, 2, 16, [4096], 0),
    (128, 32, 8, 16, [700, 1300, 31], 64),
    (128, 8, 1, 64, [257, 64, 1], 3),
    (64, 16, 2, 64, [999, 1, 2048], 1),
    (128, 6, 3, 16, [5000], 0),
    (128, 4, 4, 16, [1, 15, 16, 17], 500),  # more CTAs than tiles
]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("d,Hq,Hkv,P,lens,splits", FP8_DENSE_CASES)
def test_quant_decode_dense_matches_oracle(fmt, d, Hq, Hkv, P, lens, splits):
    _lib()
    case = W.Case("dense8", B=len(lens), Hq=Hq, Hkv=Hkv, d=d, P=P, lens=lens,
                  seed=hash((d, Hq, P, tuple(lens))) % 1000 + 1)
    cache = _cache(case, fmt)
    q = case.q(0, DEV)
    out = torch.full((case.B, Hq, d), float("nan"), device=DEV)
    m_g = torch.full((case.B, Hq), float("nan"), device=DEV)
    e_g = torch.full((case.B, Hq), float("nan"), device=DEV)
    ws = cache.workspace(num_splits=splits)
    cache.decode(q, out, ws, m_g=m_g, e_g=e_g, num_splits=splits)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    _check(_ref_dense(case, q, cache.lens, fmt), out, m_g, e_g, cache.lens, f"{fmt} decode")
    out2 = torch.empty_like(out)
    cache.decode(q, out2, ws, num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("q_exp", [-40, 0, 40])
def test_quant_decode_wide_value_ranges(fmt, q_exp):
    """Row scales spread over 2^-30..2^30 (the V-scale bound r is raised many times inside a
    piece), rows that quantize to subnormals and zeros, and queries far outside the fp16
    range (the per-piece power-of-two query scaling)."""
    dattn = _lib()
    case = W.Case("wide8", B=2, Hq=8, Hkv=2, d=128, P=16, lens=[0, 0], seed=2,
                  reserve_tokens=700)
    cache = _cache(case, fmt, fill=False)
    lens = [600, 77]
    kv = []
    for b, L in enumerate(lens):
        K = _special_rows(case.Hkv, case.d, L, 100 + b)
        V = _special_rows(case.Hkv, case.d, L, 200 + b)
        dattn.dattn_kv_append(cache._row_layout(b), cache.k_pool, cache.v_pool, None,
                              K.unsqueeze(0).to(DEV), V.unsqueeze(0).to(DEV),
                              cache.seq_lens[b:b + 1], cache.dev_err)
        kv.append((oracle.bf16_bits(K), oracle.bf16_bits(V)))
    cache.lens = lens
    # K rows reach 2^30 in magnitude: the softmax scale 2^(-q_exp - 34) keeps the largest
    # logits of order one
    q = (case.q(0, DEV).float() * 2.0 ** q_exp).to(torch.bfloat16)
    scale = 2.0 ** (-q_exp - 34)
    out = torch.empty(case.B, case.Hq, case.d, device=DEV)
    m_g = torch.empty(case.B, case.Hq, device=DEV)
    e_g = torch.empty_like(m_g)
    dattn.dattn_decode(cache.layout, cache.k_pool, cache.v_pool, q, scale, cache.seq_lens, out,
                       cache.workspace(num_splits=5), m_g=m_g, e_g=e_g, num_splits=5,
                       dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    for b in range(case.B):
        Kd, Vd = _deq(*kv[b], fmt)
        for h in range(case.Hq):
            kvh = h // case.g
            r, rm, re = oracle.attention_f64(qb[b, h], Kd[:, kvh], Vd[:, kvh], scale)
            # outputs live on the scale of the largest V rows: compare relative to it
            vmax = np.abs(Vd[:, kvh]).max()
            assert_out_close(o[b, h] / vmax, r / vmax, f"b={b} h={h}")
            assert_m_close(mg[b, h], rm, f"b={b} h={h}")
            assert_e_close(eg[b, h], re, f"b={b} h={h}")


# ---------------------------------------------------------------- quantized partials and merge

@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("seed", [0, 1])
def test_quant_partial_then_merge(fmt, seed):
    """Batch 1, 8 q / 2 KV heads, d 64, 4096 tokens, 4 chunks of 1024 (identity table)."""
    dattn = _lib()
    case = W.dense_tiny(seed=seed)
    cache = _cache(case, fmt)
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
                        chunk_req, indptr, pages, m, e, MA, ws, num_splits=9,
                        dev_err=cache.dev_err)
    out = torch.empty(1, case.Hq, case.d, device=DEV)
    m_g = torch.empty(1, case.Hq, device=DEV)
    e_g = torch.empty_like(m_g)
    dattn.dattn_merge(torch.tensor([0, C], dtype=torch.int32, device=DEV), m, e, MA, out=out,
                      m_g=m_g, e_g=e_g)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    K, V = host_kv(case, 0, 4096, DEV)
    Kd, Vd = _deq(K, V, fmt)
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
    _check(_ref_dense(case, q, [4096], fmt), out, m_g, e_g, [4096], f"{fmt} merged")


# ---------------------------------------------------------------- quantized block-sparse decode

@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("P,lens,splits", [(64, [64 * 200 + 5, 3000, 12, 5], 0),
                                           (16, [2000, 700], 9)])
def test_quant_sparse_decode_matches_oracle_token_sets(fmt, P, lens, splits):
    _lib()
    case = W.Case("sparse8", B=len(lens), Hq=16, Hkv=4, d=128, P=P, lens=lens, seed=21,
                  head_kind=[1, 2, 1, 2], top_k=16, sinks=4, local=8, n_highsim=6)
    cache = _cache(case, fmt, with_stats=True)
    q0 = case.q(0, DEV)
    sel = torch.empty(case.B, case.Hkv, case.top_k, dtype=torch.int32, device=DEV)
    cache.select(q0, sel, cache.workspace(top_k=case.top_k))
    torch.cuda.synchronize()
    # the statistics come from the bf16 keys, so the selection is checked as the bf16 path's:
    # against the fp64 page scores within their fp32 error bounds
    qb0 = oracle.bf16_bits(q0)
    want_sel = sel.cpu().numpy()
    for b in range(case.B):
        K, _ = host_kv(case, b, cache.lens[b], DEV)
        for h in range(case.Hkv):
            if case.head_kind[h] != W.HEAD_RETRIEVAL:
                assert (want_sel[b, h] == -1).all()
                continue
            score, bound = oracle.page_scores(qb0[b, h * case.g:(h + 1) * case.g],
                                              K[:, h].copy(), cache.lens[b], P,
                                              with_bounds=True)
            check_selection(want_sel[b, h], score, bound, case.top_k, f"b={b} h={h}")
    sp = cache.sparse_config(sel)
    ws = cache.workspace(num_splits=splits)
    for step in range(2):  # the selection is reused while tokens are appended
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
            Kd, Vd = _deq(*host_kv(case, b, L, DEV), fmt)
            for h in range(case.Hq):
                kvh = h // case.g
                rows = oracle.sparse_rows(case.head_kind[kvh], L, P, want_sel[b, kvh],
                                          case.sinks, case.local)
                r, rm, re = oracle.attention_f64(qb[b, h], Kd[:, kvh], Vd[:, kvh], case.scale,
                                                 rows=rows)
                assert_out_close(o[b, h], r, f"step {step} b={b} h={h}")
                assert_m_close(mg[b, h], rm, f"step {step} b={b} h={h}")
                assert_e_close(eg[b, h], re, f"step {step} b={b} h={h}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_quant_decode_flags_unmapped_page_without_fault(fmt):
    dattn = _lib()
    case = W.Case("unm8", B=1, Hq=4, Hkv=4, d=128, P=16, lens=[100], seed=2)
    cache = _cache(case, fmt)
    cache.block_table[0, 2] = -1
    cache.block_table[0, 3] = case.num_pages + 5
    q = case.q(0, DEV)
    out = torch.empty(1, 4, 128, device=DEV)
    cache.decode(q, out, cache.workspace())
    torch.cuda.synchronize()
    err = int(cache.dev_err.item())
    assert err & dattn.DEVERR["UNMAPPED_PAGE"] and err & dattn.DEVERR["PAGE_OOB"]
    K, V = host_kv(case, 0, 100, DEV)
    Kd, Vd = _deq(K, V, fmt)
    rows = [t for t in range(100) if t // 16 not in (2, 3)]
    qb = oracle.bf16_bits(q)
    for h in range(4):
        r, _, _ = oracle.attention_f64(qb[0, h], Kd[:, h], Vd[:, h], case.scale, rows=rows)
        assert_out_close(out[0, h].cpu().numpy(), r, f"head {h}")
