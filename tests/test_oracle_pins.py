"""Pins for the oracle. They check it against facts that come from outside the oracle itself.

Each pin is tied to the pages, to mathematics or to a library routine:
  * hand-derived worked examples (tests/golden/worked_examples.json, each with its citation);
  * closed forms: a single key, equal logits, and one-hot values that reduce to scipy's
    softmax;
  * DistAttention's equivalence claim (the Infinite-LLM notes call MicroAttention plus
    aggregation mathematically equivalent to attention): every partition of the keys,
    merged in any order, equals full attention, checked by brute force over all set
    partitions of tiny key sets;
  * LServe's statistics and selection: numpy max/min, the upper-bound property of the page
    score, and a brute-force sort for top-K.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))


def bf(x):
    """bf16 bit patterns of a float array (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def f64(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def rand_bf(rng, *shape, scale=1.0):
    return bf(rng.standard_normal(shape).astype(np.float32) * scale)


# ---------------------------------------------------------------- worked examples (golden)

@pytest.mark.parametrize("name", ["two_token", "three_token", "three_token_half_scale"])
def test_worked_example_full_attention(orc, name):
    g = GOLD[name]
    out, m, e = orc.attention(bf(g["q"]), bf(g["K"]), bf(g["V"]), g["scale"])
    np.testing.assert_allclose(out, g["out"], rtol=0, atol=1e-15)
    assert m == pytest.approx(g["m"], abs=1e-15)
    assert e == pytest.approx(g["e"], abs=1e-15)


def test_worked_example_two_token_partials(orc):
    g = GOLD["two_token"]
    q, K, V = bf(g["q"]), bf(g["K"]), bf(g["V"])
    parts = [orc.partial(q, K, V, g["scale"], rows=[i]) for i in range(2)]
    for (m, e, MA), (gm, ge, gMA) in zip(parts, g["partials"]):
        assert m == gm and e == ge
        np.testing.assert_array_equal(MA, gMA)
    for order in ([0, 1], [1, 0]):
        mg, eg, out, _ = orc.merge([parts[i][0] for i in order], [parts[i][1] for i in order],
                                   [parts[i][2] for i in order])
        np.testing.assert_allclose(out, g["out"], rtol=0, atol=1e-15)
        assert mg == g["m"] and eg == pytest.approx(g["e"], abs=1e-15)


# ---------------------------------------------------------------- closed forms

def test_single_key_returns_its_value(orc):
    rng = np.random.default_rng(1)
    for d in (1, 3, 64, 128):
        q, K, V = rand_bf(rng, d), rand_bf(rng, 1, d), rand_bf(rng, 1, d)
        out, m, e = orc.attention(q, K, V, 0.37)
        np.testing.assert_array_equal(out, f64(V[0]))
        assert e == 1.0
        assert m == pytest.approx(0.37 * float(f64(q) @ f64(K[0])), rel=1e-15, abs=1e-300)


def test_equal_logits_give_mean_of_values(orc):
    rng = np.random.default_rng(2)
    n, d = 37, 16
    V = rand_bf(rng, n, d)
    # q = 0: every logit is 0
    out, m, e = orc.attention(bf(np.zeros(d)), rand_bf(rng, n, d), V, 0.25)
    np.testing.assert_allclose(out, f64(V).mean(0), rtol=0, atol=1e-14)
    assert m == 0.0 and e == float(n)
    # identical keys, q != 0: every logit equals s
    q = rand_bf(rng, d)
    k = rand_bf(rng, d)
    out, m, e = orc.attention(q, np.tile(k, (n, 1)), V, 0.5)
    np.testing.assert_allclose(out, f64(V).mean(0), rtol=0, atol=1e-14)
    assert e == float(n)
    assert m == pytest.approx(0.5 * float(f64(q) @ f64(k)), rel=1e-15)


def test_one_hot_values_reduce_to_scipy_softmax(orc):
    """With V = identity rows, out is the softmax weight vector (scipy.special.softmax)."""
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    d = 24
    q, K = rand_bf(rng, d), rand_bf(rng, d, d)
    V = bf(np.eye(d))
    scale = 1 / math.sqrt(d)
    out, m, e = orc.attention(q, K, V, scale)
    logits = scale * (f64(K) @ f64(q))
    np.testing.assert_allclose(out, softmax(logits), rtol=1e-13, atol=1e-16)
    assert m == pytest.approx(logits.max(), rel=1e-15)
    assert e == pytest.approx(np.exp(logits - logits.max()).sum(), rel=1e-14)


def test_empty_key_set(orc):
    d = 8
    z = np.zeros((0, d), np.uint16)
    out, m, e = orc.attention(bf(np.ones(d)), z, z, 1.0)
    assert m == -math.inf and e == 0.0 and not out.any()
    m, e, MA = orc.partial(bf(np.ones(d)), z, z, 1.0)
    assert m == -math.inf and e == 0.0 and not MA.any()
    mg, eg, out, MAg = orc.merge([-math.inf, -math.inf], [0, 0], np.zeros((2, d)))
    assert mg == -math.inf and eg == 0.0 and not out.any() and not MAg.any()


# ---------------------------------------------------------------- DistAttention equivalence

def _set_partitions(items):
    if not items:
        yield []
        return
    first, rest = items[0], items[1:]
    for p in _set_partitions(rest):
        for i in range(len(p)):
            yield p[:i] + [[first] + p[i]] + p[i + 1:]
        yield [[first]] + p


def test_bell_numbers_of_partition_enumerator():
    assert [sum(1 for _ in _set_partitions(list(range(n)))) for n in range(7)] == \
        [1, 1, 2, 5, 15, 52, 203]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_every_partition_and_order_merges_to_full_attention(orc, n):
    rng = np.random.default_rng(10 + n)
    d = 5
    q, K, V = rand_bf(rng, d), rand_bf(rng, n, d, scale=2.0), rand_bf(rng, n, d)
    ref, mref, eref = orc.attention(q, K, V, 0.7)
    perm_rng = np.random.default_rng(99)
    for part in _set_partitions(list(range(n))):
        parts = [orc.partial(q, K, V, 0.7, rows=blk) for blk in part]
        orders = list(itertools.permutations(range(len(part)))) if len(part) <= 4 else \
            [perm_rng.permutation(len(part)) for _ in range(24)]
        for order in orders:
            mg, eg, out, _ = orc.merge([parts[i][0] for i in order],
                                       [parts[i][1] for i in order],
                                       [parts[i][2] for i in order])
            np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)
            assert mg == mref
            assert eg == pytest.approx(eref, rel=1e-13)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_partitions_long_context(orc, seed):
    """b = 1, single-token chunks, random non-contiguous partitions, permuted order."""
    rng = np.random.default_rng(seed)
    n, d = 4096 if seed == 0 else 1500, 64
    q, K, V = rand_bf(rng, d), rand_bf(rng, n, d), rand_bf(rng, n, d)
    scale = 1 / math.sqrt(d)
    ref, mref, eref = orc.attention(q, K, V, scale)
    cases = [np.zeros(n, int),                    # b = 1
             rng.integers(0, 7, size=n),           # 7 random non-contiguous chunks
             np.arange(n) // 1024]                 # contiguous chunks of 1024
    if seed != 0:
        cases.append(np.arange(n))                # single-token chunks
    for assign in cases:
        blocks = [np.nonzero(assign == j)[0] for j in np.unique(assign)]
        parts = [orc.partial(q, K, V, scale, rows=blk) for blk in blocks]
        order = rng.permutation(len(parts))
        mg, eg, out, _ = orc.merge([parts[i][0] for i in order], [parts[i][1] for i in order],
                                   [parts[i][2] for i in order])
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        assert mg == mref and eg == pytest.approx(eref, rel=1e-12)


def test_nested_merge_equals_flat_merge(orc):
    rng = np.random.default_rng(5)
    n, d = 900, 32
    q, K, V = rand_bf(rng, d), rand_bf(rng, n, d), rand_bf(rng, n, d)
    ref, mref, eref = orc.attention(q, K, V, 0.2)
    blocks = np.array_split(rng.permutation(n), 12)
    parts = [orc.partial(q, K, V, 0.2, rows=b) for b in blocks]
    level1 = []
    for grp in (parts[0:5], parts[5:6], parts[6:12]):
        mg, eg, _, MAg = orc.merge([p[0] for p in grp], [p[1] for p in grp], [p[2] for p in grp])
        level1.append((mg, eg, MAg))
    mg, eg, out, _ = orc.merge([p[0] for p in level1], [p[1] for p in level1],
                               [p[2] for p in level1])
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    assert mg == mref and eg == pytest.approx(eref, rel=1e-12)


def test_strided_rows_match_contiguous(orc):
    """Multi-head token-ordered storage ([n][Hkv][d]) reads the right head."""
    rng = np.random.default_rng(6)
    n, Hkv, Hq, d = 300, 3, 6, 16
    q = rand_bf(rng, 1, Hq, d)
    K, V = rand_bf(rng, n, Hkv, d), rand_bf(rng, n, Hkv, d)
    pairs = [(0, h) for h in range(Hq)]
    out, m, e, _ = orc.attention_pairs(q, K, V, [0, n], pairs, 0.25, nthreads=3)
    for i, (_, h) in enumerate(pairs):
        kvh = h // (Hq // Hkv)
        r, mr, er = orc.attention(q[0, h], K[:, kvh].copy(), V[:, kvh].copy(), 0.25)
        np.testing.assert_array_equal(out[i], r)
        assert m[i] == mr and e[i] == er


# ---------------------------------------------------------------- paged layout (append)

def test_identity_table_single_head_pool_is_token_order(orc):
    rng = np.random.default_rng(7)
    P, d, L = 16, 8, 100
    npages = -(-L // P)
    K, V = rand_bf(rng, L, 1, d), rand_bf(rng, L, 1, d)
    kp = np.zeros((npages, 1, P, d), np.uint16)
    vp = np.zeros_like(kp)
    assert orc.kv_write(kp, vp, np.arange(npages), npages, K, V, 0) == 0
    np.testing.assert_array_equal(kp.reshape(-1, d)[:L], K.reshape(L, d))
    np.testing.assert_array_equal(vp.reshape(-1, d)[:L], V.reshape(L, d))


def test_pool_positions_hand_checked(orc):
    """Token 17 of head 1 with P=16, Hkv=2, block table [5, 2]: page 2, slot 1."""
    P, d, Hkv = 16, 4, 2
    kp = np.zeros((6, Hkv, P, d), np.uint16)
    vp = np.zeros_like(kp)
    T = 20
    K = (np.arange(T * Hkv * d, dtype=np.uint16) + 1).reshape(T, Hkv, d)
    V = K + 1000
    assert orc.kv_write(kp, vp, [5, 2], 6, K, V, 0) == 0
    flat = kp.reshape(-1)
    # element (page 2, head 1, slot 1, channel 3) at ((2*Hkv + 1)*P + 1)*d + 3
    assert flat[((2 * Hkv + 1) * P + 1) * d + 3] == K[17, 1, 3]
    assert kp[5, 0, 0, 0] == K[0, 0, 0] and kp[5, 1, 15, 2] == K[15, 1, 2]
    assert vp[2, 0, 3, 1] == V[19, 0, 1]
    # appending in two calls equals one call
    kp2, vp2 = np.zeros_like(kp), np.zeros_like(vp)
    orc.kv_write(kp2, vp2, [5, 2], 6, K[:9], V[:9], 0)
    orc.kv_write(kp2, vp2, [5, 2], 6, K[9:], V[9:], 9)
    np.testing.assert_array_equal(kp2, kp)
    np.testing.assert_array_equal(vp2, vp)


def test_unmapped_pages_are_skipped(orc):
    P, d = 16, 4
    kp = np.zeros((3, 1, P, d), np.uint16)
    vp = np.zeros_like(kp)
    K = np.ones((40, 1, d), np.uint16)
    # page 1 unmapped (-1), page 2 beyond the pool (7 >= 3); 40 tokens span 3 table entries
    assert orc.kv_write(kp, vp, [0, -1, 7], 3, K, K, 0) == 16 + 8
    assert kp[0].all() and not kp[1:].any()
    # positions beyond the table width are skipped too
    assert orc.kv_write(kp, vp, [0], 3, K[:20], K[:20], 0) == 4


# ---------------------------------------------------------------- page statistics and scores

def test_page_stats_match_numpy_max_min(orc):
    rng = np.random.default_rng(8)
    n, d = 16, 128
    K = rand_bf(rng, n, d)
    for t0, t1 in [(0, 16), (0, 1), (3, 11), (15, 16)]:
        kmax, kmin = orc.logical_page_stats(K, t0, t1)
        np.testing.assert_array_equal(f64(kmax), f64(K[t0:t1]).max(0))
        np.testing.assert_array_equal(f64(kmin), f64(K[t0:t1]).min(0))


def test_page_stats_tie_keeps_first_seen_zero(orc):
    K = np.array([[0x8000], [0x0000]], np.uint16)  # -0 then +0
    kmax, kmin = orc.logical_page_stats(K, 0, 2)
    assert kmax[0] == 0x8000 and kmin[0] == 0x8000


def test_page_score_worked_example(orc):
    g = GOLD["page_score"]
    keys = bf(g["keys"])
    kmax, kmin = orc.logical_page_stats(keys, 0, len(g["keys"]))
    np.testing.assert_array_equal(f64(kmax), g["kmax"])
    np.testing.assert_array_equal(f64(kmin), g["kmin"])
    assert orc.logical_score(bf(g["q"]), kmax, kmin) == g["score"]
    np.testing.assert_array_equal(f64(keys) @ f64(bf(g["q"])), g["qk"])


def test_page_score_bounds_every_key_and_is_tight_for_one_key(orc):
    rng = np.random.default_rng(9)
    d = 128
    for trial in range(20):
        n = 1 + trial % 16
        K = rand_bf(rng, n, d)
        q = rand_bf(rng, d)
        kmax, kmin = orc.logical_page_stats(K, 0, n)
        s = orc.logical_score(q, kmax, kmin)
        qk = f64(K) @ f64(q)
        assert np.all(qk <= s + 1e-12)
        if n == 1:
            assert s == pytest.approx(qk[0], rel=1e-15, abs=1e-15)


def _fp32_sums(terms, rng):
    """fp32 sums of exact fp32 terms in several orders: ascending, descending, a pairwise
    tree, random permutations, and the 2d-term sum of a k_max half and a k_min half."""
    t = np.asarray(terms, np.float32)

    def seq(v):
        acc = np.float32(0.0)
        for x in v:
            acc = np.float32(acc + x)
        return acc

    def tree(v):
        v = list(v)
        while len(v) > 1:
            v = [np.float32(v[i] + v[i + 1]) if i + 1 < len(v) else v[i]
                 for i in range(0, len(v), 2)]
        return v[0]

    sums = [seq(t), seq(t[::-1]), tree(t), tree(t[::-1])]
    sums += [seq(rng.permutation(t)) for _ in range(4)]
    sums += [tree(rng.permutation(t)) for _ in range(4)]
    halves = np.concatenate([np.where(t >= 0, t, 0), np.where(t >= 0, 0, t)]).astype(np.float32)
    sums += [tree(halves), seq(halves)]
    return [float(x) for x in sums]


def test_fp32_bound_covers_fp32_sums_in_any_order(orc):
    """The error bound of reading R9 holds for fp32 evaluations of the score in any order."""
    rng = np.random.default_rng(10)
    for trial in range(60):
        d = (64, 128)[trial % 2]
        n = 1 + trial % 16
        K = rand_bf(rng, n, d, scale=(1.0, 8.0, 1e-3)[trial % 3])
        q = rand_bf(rng, d)
        kmax, kmin = orc.logical_page_stats(K, 0, n)
        s64 = orc.logical_score(q, kmax, kmin)
        bound = orc.logical_score_bound(q, kmax, kmin)
        # products of two bf16 values are exact in fp32, so the terms are
        qd = f64(q)
        terms = np.where(qd >= 0, qd * f64(kmax), qd * f64(kmin))
        assert np.all(np.float32(terms) == terms)
        for s32 in _fp32_sums(terms, rng):
            assert abs(s32 - s64) <= bound, (trial, s32, s64, bound)


def test_fp32_bound_is_reached_by_adversarial_sums(orc):
    """Sums whose fp32 evaluation loses what the bound must cover: the factor d (127 terms
    of 2^-24 absorbed by a leading 1) and the absolute values (1 + 2^-25 - 1 evaluates to 0)."""
    d = 128
    q = bf(np.ones(d))
    k = np.full(d, 2.0 ** -24)
    k[0] = 1.0
    kb = bf(k)
    s64 = orc.logical_score(q, kb, kb)
    assert s64 == 1.0 + 127 * 2.0 ** -24
    acc = np.float32(0.0)  # sequential fp32 sum: every 2^-24 is lost against the leading 1
    for x in f64(kb):
        acc = np.float32(acc + np.float32(x))
    assert float(acc) == 1.0
    assert orc.logical_score_bound(q, kb, kb) >= s64 - 1.0
    q2 = np.zeros(d)
    q2[:3] = 1.0
    k2 = np.zeros(d)
    k2[:3] = [1.0, 2.0 ** -25, -1.0]
    q2b, k2b = bf(q2), bf(k2)
    s64 = orc.logical_score(q2b, k2b, k2b)
    assert s64 == 2.0 ** -25
    acc = np.float32(0.0)
    for x in f64(k2b)[:3]:
        acc = np.float32(acc + np.float32(x))
    assert float(acc) == 0.0
    assert orc.logical_score_bound(q2b, k2b, k2b) >= s64


def test_physical_score_is_max_over_logical_pages_and_heads(orc):
    rng = np.random.default_rng(11)
    d, P, L, g = 32, 64, 150, 3
    K = rand_bf(rng, L, d)
    Q = rand_bf(rng, g, d)
    sc, bd = orc.page_scores(Q, K, L, P, with_bounds=True)
    assert sc.shape == (3,) and bd.shape == (3,)
    for p in range(3):
        best, err = -math.inf, 0.0
        for t0 in range(p * P, min((p + 1) * P, L), 16):
            kmax, kmin = orc.logical_page_stats(K, t0, min(t0 + 16, L))
            for j in range(g):
                best = max(best, orc.logical_score(Q[j], kmax, kmin))
                err = max(err, orc.logical_score_bound(Q[j], kmax, kmin))
        assert sc[p] == best and bd[p] == err
    # the max over logical pages bounds every key of the physical page, for every head
    qk = f64(K) @ f64(Q).T
    for t in range(L):
        assert qk[t].max() <= sc[t // P] + 1e-12


# ---------------------------------------------------------------- top-K

def test_topk_worked_example(orc):
    g = GOLD["topk"]
    for k, want in g["cases"]:
        np.testing.assert_array_equal(orc.topk(g["scores"], k), want)


def test_topk_matches_bruteforce_sort_with_ties(orc):
    rng = np.random.default_rng(12)
    for trial in range(40):
        n = int(rng.integers(1, 300))
        scores = rng.integers(-5, 6, size=n).astype(np.float64)  # many ties
        k = int(rng.integers(1, 80))
        want = sorted(sorted(range(n), key=lambda i: (-scores[i], i))[:k])
        want = want + [-1] * (k - len(want))
        np.testing.assert_array_equal(orc.topk(scores, k), want)


# ---------------------------------------------------------------- sparse token sets

def test_streaming_rows_worked_examples(orc):
    g = GOLD["streaming_rows"]
    for L, want in g["cases"]:
        np.testing.assert_array_equal(orc.sparse_rows(2, L, 64, None, g["sinks"], g["local"]),
                                      want)


def test_retrieval_rows_are_the_selected_pages_tokens(orc):
    P, L = 16, 100
    sel = np.array([0, 3, 6, -1], np.int32)
    rows = orc.sparse_rows(1, L, P, sel, 4, 8)
    want = [t for t in range(L) if t // P in (0, 3, 6)]
    np.testing.assert_array_equal(rows, want)
    # all pages selected: the retrieval head is dense
    allp = np.arange(-(-L // P), dtype=np.int32)
    np.testing.assert_array_equal(orc.sparse_rows(1, L, P, allp, 4, 8), np.arange(L))
    np.testing.assert_array_equal(orc.sparse_rows(0, L, P, None, 4, 8), np.arange(L))


def test_topk_covering_all_pages_makes_sparse_equal_dense(orc):
    rng = np.random.default_rng(13)
    d, P, L, g = 64, 64, 333, 4
    K, V = rand_bf(rng, L, d), rand_bf(rng, L, d)
    Q = rand_bf(rng, g, d)
    sel = orc.select_pages(Q, K, L, P, top_k=16)
    assert (sel[:6] == np.arange(6)).all() and (sel[6:] == -1).all()
    rows = orc.sparse_rows(1, L, P, sel, 4, 8)
    for j in range(g):
        a = orc.attention(Q[j], K, V, 0.125, rows=rows)
        b = orc.attention(Q[j], K, V, 0.125)
        np.testing.assert_array_equal(a[0], b[0])
