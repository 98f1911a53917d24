"""Pins of the oracle's block-sparse prefill row sets (reading R11 of the oracle).

Key blocks are 64 tokens. Query token t of a Tq-token chunk sits at position p = L - Tq + t
and attends the keys i <= p of the blocks its head keeps for the query block qb = p // 64.
The expected sets below are written out by hand from that definition, and the dense case is
also checked against a causally masked softmax computed with scipy.
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle


def _r(*ranges):
    return np.concatenate([np.arange(a, b) for a, b in ranges]).astype(np.int64)


@pytest.mark.parametrize("L,Tq,t", [(1, 1, 0), (64, 64, 63), (300, 300, 250), (200, 10, 0),
                                    (200, 10, 9), (1000, 1, 0)])
def test_dense_rows_are_the_causal_prefix(orc, L, Tq, t):
    np.testing.assert_array_equal(orc.prefill_rows(0, L, Tq, t), np.arange(L - Tq + t + 1))


def test_streaming_rows_golden(orc):
    # p = 250, qb = 3: sink block 0, local blocks 2..3 (two blocks ending at qb)
    np.testing.assert_array_equal(orc.prefill_rows(2, 300, 300, 250, 1, 2), _r((0, 64), (128, 251)))
    # p = 190, qb = 2: sink block 0, local block 2 only
    np.testing.assert_array_equal(orc.prefill_rows(2, 200, 10, 0, 1, 1), _r((0, 64), (128, 191)))
    # p = 195, qb = 3; no sinks, one local block: the query's own block up to itself
    np.testing.assert_array_equal(orc.prefill_rows(2, 200, 10, 5, 0, 1), _r((192, 196)))
    # sinks and band overlap inside block 0: every key up to p
    np.testing.assert_array_equal(orc.prefill_rows(2, 40, 40, 39, 2, 1), np.arange(40))
    # p = 700, qb = 10: sinks 0..1, band 8..10
    np.testing.assert_array_equal(orc.prefill_rows(2, 701, 1, 0, 2, 3), _r((0, 128), (512, 701)))


def test_retrieval_rows_golden(orc):
    # p = 250 (qb = 3): listed blocks 0 and 2
    np.testing.assert_array_equal(orc.prefill_rows(1, 300, 300, 250, blocks=[2, 0]),
                                  _r((0, 64), (128, 192)))
    # the query's own block, cut at the query
    np.testing.assert_array_equal(orc.prefill_rows(1, 300, 300, 250, blocks=[3]), _r((192, 251)))
    # blocks past the query, -1 entries and repeats add nothing
    np.testing.assert_array_equal(orc.prefill_rows(1, 300, 300, 250, blocks=[5, -1, 1, 1]),
                                  _r((64, 128)))
    assert orc.prefill_rows(1, 300, 300, 250, blocks=[4]).size == 0
    assert orc.prefill_rows(1, 300, 300, 250, blocks=None).size == 0


def test_full_masks_reduce_to_dense(orc):
    for L, Tq, t in [(300, 300, 250), (1000, 37, 20), (64, 64, 0)]:
        dense = orc.prefill_rows(0, L, Tq, t)
        qb = (L - Tq + t) // 64
        np.testing.assert_array_equal(orc.prefill_rows(1, L, Tq, t, blocks=list(range(qb + 1))),
                                      dense)
        np.testing.assert_array_equal(orc.prefill_rows(2, L, Tq, t, 1, qb), dense)
        np.testing.assert_array_equal(orc.prefill_rows(2, L, Tq, t, 0, qb + 1), dense)


def test_causal_prefill_equals_masked_softmax(orc):
    rng = np.random.default_rng(11)
    L, d, scale = 150, 16, 0.25
    Q = torch.from_numpy(rng.normal(size=(L, d)).astype(np.float32)).to(torch.bfloat16)
    K = torch.from_numpy(rng.normal(size=(L, d)).astype(np.float32)).to(torch.bfloat16)
    V = torch.from_numpy(rng.normal(size=(L, d)).astype(np.float32)).to(torch.bfloat16)
    Qd, Kd, Vd = (x.double().numpy() for x in (Q, K, V))
    logits = scale * Qd @ Kd.T
    logits[np.triu_indices(L, 1)] = -np.inf
    want = softmax(logits, axis=1) @ Vd
    for t in (0, 1, 63, 64, 149):
        out, _, _ = orc.attention(Q[t], K, V, scale, rows=orc.prefill_rows(0, L, L, t))
        np.testing.assert_allclose(out, want[t], rtol=1e-12, atol=1e-12)
