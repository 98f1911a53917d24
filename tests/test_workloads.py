"""Host-side checks of the seeded input generators (no GPU, no method arithmetic)."""
import numpy as np
import torch

from split_kv_decode_distattention_gb300 import workloads as W


def test_kv_stream_is_regenerable_in_pieces():
    c = W.Case("t", B=2, Hq=4, Hkv=2, d=16, P=16, lens=[5000, 300], seed=3)
    K, V = c.kv(0, 0, 5000)
    K1, V1 = c.kv(0, 0, 123)
    K2, V2 = c.kv(0, 123, 5000)
    assert torch.equal(torch.cat([K1, K2]), K) and torch.equal(torch.cat([V1, V2]), V)
    K3, _ = c.kv(0, 4095, 4097)  # crosses a generation chunk boundary
    assert torch.equal(K3, K[4095:4097])
    assert not torch.equal(c.kv(1, 0, 300)[0], K[:300])  # requests differ
    c2 = W.Case("t", B=2, Hq=4, Hkv=2, d=16, P=16, lens=[5000, 300], seed=3)
    assert torch.equal(c2.kv(0, 0, 5000)[0], K)  # same seed, same values


def test_block_table_is_a_permutation_with_reserve():
    c = W.mha_32k(seed=1, B=3, L=1000)
    bt = c.block_table
    caps = [-(-(L + c.reserve_tokens) // c.P) for L in c.lens]
    used = np.concatenate([bt[b, :caps[b]] for b in range(c.B)])
    assert sorted(used.tolist()) == list(range(c.num_pages))
    assert (bt[:, max(caps):] == -1).all() if bt.shape[1] > max(caps) else True
    ident = W.dense_tiny()
    assert (ident.block_table[0, :ident.max_pages] == np.arange(ident.max_pages)).all()


def test_page_sets_are_disjoint_and_cover():
    c = W.gqa_ragged(seed=0, B=6, lo=100, hi=3000)
    for b in range(c.B):
        sets = c.page_sets_of(b)
        assert 2 <= len(sets) <= 8 or len(sets) == -(-c.lens[b] // c.P)
        allp = np.sort(np.concatenate(sets))
        assert (allp == np.arange(-(-c.lens[b] // c.P))).all()
        assert all(s.size > 0 for s in sets)


def test_needles_align_with_query():
    c = W.Case("n", B=1, Hq=4, Hkv=4, d=32, P=16, lens=[3000], seed=5, n_needles=8)
    pos = c._needles(0)
    assert len(set(pos.tolist())) == 8 and pos.max() < 3000
    K, _ = c.kv(0, 0, 3000)
    q = c.q(0)[0].float()
    for h in range(4):
        want = (4.0 * q[h] / q[h].norm()).to(torch.bfloat16)
        for p in pos:
            assert torch.equal(K[p, h], want)


def test_highsim_pages_only_on_retrieval_heads():
    c = W.sparse_512k(seed=0, B=1, L=64 * 100)
    for h in range(c.Hkv):
        pages = c.highsim_pages(0, h)
        if c.head_kind[h] == W.HEAD_RETRIEVAL:
            assert pages.size == 32 and pages.max() < 100
        else:
            assert pages.size == 0
    # keys of a high-similarity page lean toward the group's mean query
    p = int(c.highsim_pages(0, 0)[0])
    K, _ = c.kv(0, p * 64, (p + 1) * 64)
    u = c._direction(0, 0, "cpu")
    assert (K[:, 0].float() @ u).mean() > 1.5


def test_ragged_lengths_log_uniform_range():
    c = W.gqa_ragged(seed=0)
    lens = np.array(c.lens)
    assert lens.min() >= 1024 and lens.max() <= 262144 and c.B == 64
    assert W.gqa_ragged(seed=0).lens == c.lens
