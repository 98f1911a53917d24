"""GPU parity of the block-sparse prefill (dattn_prefill) against the oracle.

Each (request, query token, query head) is compared with the oracle's attention over the
rows orc_prefill_rows gives: causal for dense heads, the Lambda blocks for streaming heads,
the listed blocks for retrieval heads (key blocks of 64 tokens). Chunks start on and off
block boundaries, lengths are ragged, and lists hold blocks after the query and -1 padding.
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


def _queries(case, Tq, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(case.B, Tq, case.Hq, case.d, generator=g, device=DEV).to(torch.bfloat16)


def _lists(case, stride, max_sel, seed):
    """Seeded key-block lists [B][Hkv][stride][max_sel]: distinct blocks up to two past the
    query block, padded with -1; the query's own block is usually, not always, listed."""
    rng = np.random.default_rng(seed)
    out = np.full((case.B, case.Hkv, stride, max_sel), -1, np.int32)
    for b in range(case.B):
        for h in range(case.Hkv):
            for qb in range(stride):
                n = int(rng.integers(0, max_sel + 1))
                cand = rng.permutation(qb + 3)[:n]
                out[b, h, qb, :len(cand)] = cand
    return out


def _check(case, q, Tq, out, m, e, kinds=None, sinks=0, local=0, lists=None, what="prefill"):
    qb_ = oracle.bf16_bits(q)
    o, mm, ee = out.cpu().numpy(), m.cpu().numpy(), e.cpu().numpy()
    for b in range(case.B):
        L = case.lens[b]
        K, V = host_kv(case, b, L, DEV)
        for t in range(Tq):
            qblk = (L - Tq + t) // 64
            for h in range(case.Hq):
                kvh = h // case.g
                kind = 0 if kinds is None else kinds[kvh]
                blocks = lists[b, kvh, qblk] if (lists is not None and kind == 1) else None
                rows = oracle.prefill_rows(kind, L, Tq, t, sinks, local, blocks=blocks)
                r, rm, re = oracle.attention(qb_[b, t, h], K[:, kvh].copy(), V[:, kvh].copy(),
                                             case.scale, rows=rows)
                tag = f"{what} b={b} t={t} h={h} L={L}"
                assert_out_close(o[b, t, h], r, tag)
                assert_m_close(mm[b, t, h], rm, tag)
                assert_e_close(ee[b, t, h], re, tag)


def _run(dattn, cache, q, sparse=None):
    B, Tq, Hq, d = q.shape
    out = torch.full((B, Tq, Hq, d), float("nan"), device=DEV)
    m = torch.full((B, Tq, Hq), float("nan"), device=DEV)
    e = torch.full((B, Tq, Hq), float("nan"), device=DEV)
    dattn.dattn_prefill(cache.layout, cache.k_pool, cache.v_pool, q, cache.case.scale,
                        cache.seq_lens, out, m, e, sparse=sparse, dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    return out, m, e


CAUSAL_CASES = [
    # (d, Hq, Hkv, P, lens, Tq)
    (128, 8, 2, 16, [300, 130], 130),     # a chunk starting mid-block, and a whole request
    (64, 4, 4, 64, [1000], 200),          # MHA, d = 64, 64-token pages
    (128, 16, 2, 16, [64, 129, 65], 64),  # group 8, block-aligned and ragged chunks
    (128, 4, 1, 32, [777, 20], 1),        # one-token chunks
]


@pytest.mark.parametrize("d,Hq,Hkv,P,lens,Tq", CAUSAL_CASES)
def test_causal_prefill_matches_oracle(d, Hq, Hkv, P, lens, Tq):
    dattn = _lib()
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.Case("prefill", B=len(lens), Hq=Hq, Hkv=Hkv, d=d, P=P, lens=lens, seed=Tq + d)
    cache = PagedCache(case, DEV)
    q = _queries(case, Tq, 5)
    out, m, e = _run(dattn, cache, q)
    _check(case, q, Tq, out, m, e, what="causal")
    out2, _, _ = _run(dattn, cache, q)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("P,lens,Tq,sinks,local,Hq", [(16, [700, 333], 300, 1, 2, 8),
                                                      (64, [1024], 1024, 2, 3, 8),
                                                      (16, [200, 64], 64, 0, 1, 8),
                                                      (16, [700, 333], 300, 1, 2, 12),
                                                      (64, [1024], 1000, 2, 3, 4)])
def test_block_sparse_prefill_matches_oracle(P, lens, Tq, sinks, local, Hq):
    """Group 2 (a CTA takes one query block of two heads) and groups 3 and 1 (a CTA takes two
    query blocks of one head)."""
    dattn = _lib()
    from split_kv_decode_distattention_gb300.harness import PagedCache
    kinds = [0, 1, 2, 1]
    case = W.Case("bsprefill", B=len(lens), Hq=Hq, Hkv=4, d=128, P=P, lens=lens, seed=Tq + P)
    cache = PagedCache(case, DEV)
    q = _queries(case, Tq, 6)
    stride = max(lens) // 64 + 1
    lists = _lists(case, stride, 6, Tq)
    hk = torch.tensor(kinds, dtype=torch.int8, device=DEV)
    bl = torch.from_numpy(lists).to(DEV)
    sp = dattn.PrefillSparseConfig(hk, sinks, local, bl)
    out, m, e = _run(dattn, cache, q, sparse=sp)
    _check(case, q, Tq, out, m, e, kinds, sinks, local, lists, what="block-sparse")


def test_full_block_masks_equal_causal():
    dattn = _lib()
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.Case("fullmask", B=1, Hq=8, Hkv=2, d=128, P=16, lens=[500], seed=3)
    cache = PagedCache(case, DEV)
    q = _queries(case, 500, 7)
    causal, _, _ = _run(dattn, cache, q)
    stride = 8
    lists = np.full((1, 2, stride, stride), -1, np.int32)
    for qb in range(stride):
        lists[0, :, qb, :qb + 1] = np.arange(qb + 1)
    hk = torch.tensor([1, 2], dtype=torch.int8, device=DEV)  # retrieval, streaming
    sp = dattn.PrefillSparseConfig(hk, 0, stride, torch.from_numpy(lists).to(DEV))
    full, _, _ = _run(dattn, cache, q, sparse=sp)
    torch.testing.assert_close(full, causal, rtol=0, atol=0)


def test_prefill_flags_short_lengths_without_fault():
    dattn = _lib()
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.Case("short", B=2, Hq=4, Hkv=2, d=64, P=16, lens=[10, 100], seed=1)
    cache = PagedCache(case, DEV)
    q = _queries(case, 50, 8)
    out = torch.zeros(2, 50, 4, 64, device=DEV)
    dattn.dattn_prefill(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                        out, dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) & dattn.DEVERR["LEN_OOB"]
    assert (out[0] == 0).all()            # request 0 (10 < 50 tokens) is skipped
    assert torch.isfinite(out[1]).all()   # request 1 is computed


@pytest.mark.parametrize("scale", [-0.07, 0.0, 0.5])
def test_prefill_scale_sign_and_zero(scale):
    """The logit is scale * (q . k) for any real scale: a negative one flips the order of the
    scores, zero gives the plain average of the visible V rows, a large one a peaked row."""
    dattn = _lib()
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.Case("scale", B=2, Hq=4, Hkv=2, d=128, P=16, lens=[333, 140], seed=21)
    case.scale = scale
    cache = PagedCache(case, DEV)
    q = _queries(case, 140, 9)
    out, m, e = _run(dattn, cache, q)
    _check(case, q, 140, out, m, e, what=f"scale {scale}")
