"""GPU parity of the multi-query decode (dattn_decode_multi): T new query tokens per request,
causal over the T newest tokens of the cache. Query token t of request b attends tokens
0 .. L_b - T + t; the oracle computes each (request, query token, head) as plain attention
over exactly those rows (an empty set when L_b - T + t < 0)."""
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


def _cache(case, fmt, **kw):
    from split_kv_decode_distattention_gb300 import KV_BF16, KV_FP8_E4M3, KV_INT4
    from split_kv_decode_distattention_gb300.harness import PagedCache
    kv_format = {"bf16": KV_BF16, "fp8": KV_FP8_E4M3, "int4": KV_INT4}[fmt]
    return PagedCache(case, DEV, kv_format=kv_format, **kw)


def _queries(case, T):
    """[B][T][Hq][d] bf16: query token t is the case's seeded query of step 100 + t."""
    return torch.stack([case.q(100 + t, DEV) for t in range(T)], dim=1).contiguous()


def _check(case, q, lens, T, out, m_g, e_g, fmt, what):
    qb = oracle.bf16_bits(q)
    o, mg, eg = out.cpu().numpy(), m_g.cpu().numpy(), e_g.cpu().numpy()
    for b in range(case.B):
        L = lens[b]
        K, V = host_kv(case, b, L, DEV)
        if fmt == "fp8":
            K = oracle.dequantize_rows_fp8(*oracle.quantize_rows_fp8(K))
            V = oracle.dequantize_rows_fp8(*oracle.quantize_rows_fp8(V))
        elif fmt == "int4":
            K = oracle.dequantize_rows_int4(*oracle.quantize_rows_int4(K))
            V = oracle.dequantize_rows_int4(*oracle.quantize_rows_int4(V))
        for t in range(T):
            rows = np.arange(max(0, L - T + t + 1), dtype=np.int64)
            for h in range(case.Hq):
                kvh = h // case.g
                if fmt != "bf16":
                    r, rm, re = oracle.attention_f64(qb[b, t, h], K[:, kvh], V[:, kvh],
                                                     case.scale, rows=rows)
                else:
                    r, rm, re = oracle.attention(qb[b, t, h], K[:, kvh].copy(), V[:, kvh].copy(),
                                                 case.scale, rows=rows)
                tag = f"{what} b={b} t={t} h={h} L={L}"
                assert_out_close(o[b, t, h], r, tag)
                assert_m_close(mg[b, t, h], rm, tag)
                assert_e_close(eg[b, t, h], re, tag)


MULTI_CASES = [
    # (d, Hq, Hkv, P, lens, T, num_splits, pool format)
    (128, 4, 4, 16, [1, 5, 16, 17, 40], 8, 0, "bf16"),    # MHA, T = 8, lengths below T
    (128, 8, 2, 16, [1000, 33, 2500], 2, 7, "bf16"),      # GQA group 4, T = 2
    (64, 8, 4, 64, [999, 3, 2048], 4, 1, "bf16"),         # group 2, T = 4, d = 64
    (128, 6, 3, 16, [260, 1], 4, 0, "bf16"),              # group 2 of 3 KV heads
    (128, 8, 8, 16, [517, 2000], 3, 5, "fp8"),            # 8-bit pool, odd T
    (128, 4, 4, 16, [1, 5, 16, 17, 40], 8, 300, "fp8"),   # 8-bit pool, more CTAs than tiles
    (64, 16, 2, 64, [700], 1, 0, "fp8"),                  # T = 1, group 8
    (128, 8, 8, 16, [517, 2000], 3, 5, "int4"),           # 4-bit pool, odd T
    (64, 8, 4, 64, [999, 3, 2048], 2, 0, "int4"),         # 4-bit pool, d = 64, group 2
    (128, 4, 4, 16, [300, 1, 40, 17], 2, 0, "int4"),      # 4-bit pool, MHA, T = 2: 2 columns
    (128, 8, 8, 16, [517, 2, 100], 4, 3, "int4"),         # 4-bit pool, MHA, T = 4: 4 columns
]


@pytest.mark.parametrize("d,Hq,Hkv,P,lens,T,splits,fmt", MULTI_CASES)
def test_decode_multi_matches_oracle(d, Hq, Hkv, P, lens, T, splits, fmt):
    dattn = _lib()
    case = W.Case("multi", B=len(lens), Hq=Hq, Hkv=Hkv, d=d, P=P, lens=lens,
                  seed=hash((d, Hq, Hkv, T, tuple(lens))) % 1000 + 7)
    cache = _cache(case, fmt)
    q = _queries(case, T)
    out = torch.full((case.B, T, Hq, d), float("nan"), device=DEV)
    m_g = torch.full((case.B, T, Hq), float("nan"), device=DEV)
    e_g = torch.full((case.B, T, Hq), float("nan"), device=DEV)
    ws = dattn.Workspace(case.B, T * Hq, Hkv, d, num_splits=splits)
    dattn.dattn_decode_multi(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                             cache.seq_lens, out, ws, m_g=m_g, e_g=e_g, num_splits=splits,
                             dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    _check(case, q, cache.lens, T, out, m_g, e_g, fmt, "multi")
    # the workspace counters are back to zero: a second call gives the same bits
    out2 = torch.empty_like(out)
    dattn.dattn_decode_multi(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                             cache.seq_lens, out2, ws, num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "int4"])
def test_chunk_append_then_multi_decode(fmt):
    """The chunked step: append T new tokens per request in one call, then attend them."""
    dattn = _lib()
    T = 4
    case = W.Case("chunk", B=3, Hq=8, Hkv=4, d=128, P=16, lens=[300, 17, 1024], seed=12)
    cache = _cache(case, fmt)
    ws = dattn.Workspace(case.B, T * case.Hq, case.Hkv, case.d)
    for step in range(2):
        kn, vn = cache.new_tokens(T)
        cache.append(kn, vn)
        q = torch.stack([case.q(10 * step + t, DEV) for t in range(T)], dim=1).contiguous()
        out = torch.empty(case.B, T, case.Hq, case.d, device=DEV)
        m_g = torch.empty(case.B, T, case.Hq, device=DEV)
        e_g = torch.empty_like(m_g)
        dattn.dattn_decode_multi(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                                 cache.seq_lens, out, ws, m_g=m_g, e_g=e_g,
                                 dev_err=cache.dev_err)
        torch.cuda.synchronize()
        assert int(cache.dev_err.item()) == 0
        assert cache.seq_lens.tolist() == cache.lens
        _check(case, q, cache.lens, T, out, m_g, e_g, fmt, f"step {step}")


def test_multi_with_one_token_equals_decode_bits():
    dattn = _lib()
    case = W.Case("one", B=3, Hq=16, Hkv=4, d=128, P=16, lens=[3000, 77, 1500], seed=3)
    cache = _cache(case, "bf16")
    q = case.q(0, DEV)
    out1 = torch.empty(case.B, case.Hq, case.d, device=DEV)
    cache.decode(q, out1, cache.workspace(num_splits=9), num_splits=9)
    outm = torch.empty(case.B, 1, case.Hq, case.d, device=DEV)
    dattn.dattn_decode_multi(cache.layout, cache.k_pool, cache.v_pool, q.unsqueeze(1).contiguous(),
                             case.scale, cache.seq_lens, outm,
                             dattn.Workspace(case.B, case.Hq, case.Hkv, case.d, num_splits=9),
                             num_splits=9)
    torch.cuda.synchronize()
    assert torch.equal(outm[:, 0], out1)


def test_multi_rejects_groups_wider_than_the_tile():
    dattn = _lib()
    case = W.Case("wide", B=1, Hq=8, Hkv=2, d=64, P=16, lens=[64], seed=1)
    cache = _cache(case, "bf16")
    q = torch.zeros(1, 3, 8, 64, dtype=torch.bfloat16, device=DEV)  # g = 4, T = 3
    out = torch.empty(1, 3, 8, 64, device=DEV)
    with pytest.raises(dattn.DattnError, match="UNSUPPORTED"):
        dattn.dattn_decode_multi(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                                 cache.seq_lens, out, dattn.Workspace(1, 24, 2, 64))
