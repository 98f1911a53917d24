"""The cross-GPU DistAttention exchange on the CPU: world-size-2 (and 3) gloo process groups.

Each rank holds a share of every request's pages ([IL] DistAttention's sub-blocks on
different instances), computes its partials, and one all-gather stacks them; the merge then
gives full attention on every rank. On the CPU the oracle's MicroAttention partials and
aggregation stand in for the kernels, so this checks the host logic of the exchange: the page
shares cover every page once, rank r's partials land in row r on every rank, and a rank that
holds none of a short request's pages contributes an empty partial.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    from split_kv_decode_distattention_gb300 import workloads as W
    return W.Case("dist", B=3, Hq=4, Hkv=2, d=64, P=16, lens=[100, 37, 5], seed=8)


def _worker(rank, world, port, out_dir, scheme):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch
    import torch.distributed as dist
    import oracle
    from split_kv_decode_distattention_gb300 import distributed as D
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = _case()
        q = case.q(0, "cpu")
        qb = oracle.bf16_bits(q)
        kv = [case.kv(b, 0, L, "cpu") for b, L in enumerate(case.lens)]
        pages = [D.rank_pages(-(-L // case.P), rank, world, scheme) for L in case.lens]

        def partial_fn(m_row, e_row, MA_row):
            for b, L in enumerate(case.lens):
                K, V = (oracle.bf16_bits(x) for x in kv[b])
                rows = [t for p in pages[b] for t in range(p * case.P, min((p + 1) * case.P, L))]
                for h in range(case.Hq):
                    kvh = h // case.g
                    mm, ee, ma = oracle.partial(qb[b, h], K[:, kvh].copy(), V[:, kvh].copy(),
                                                case.scale, rows=rows)
                    m_row[b, h], e_row[b, h] = mm, ee
                    MA_row[b, h] = torch.from_numpy(ma)

        def merge_fn(m, e, MA, out, m_g, e_g):
            for b in range(case.B):
                for h in range(case.Hq):
                    mg, eg, o, _ = oracle.merge(m[:, b, h].double().numpy(),
                                                e[:, b, h].double().numpy(),
                                                MA[:, b, h].double().numpy())
                    out[b, h] = torch.from_numpy(o)
                    m_g[b, h], e_g[b, h] = mg, eg

        import torch as T
        out = T.zeros(case.B, case.Hq, case.d, dtype=T.float64)
        m_g = T.zeros(case.B, case.Hq, dtype=T.float64)
        e_g = T.zeros_like(m_g)
        # fp64 buffers on the CPU so that the oracle's values travel unrounded
        orig = D.stacked_partials
        D.stacked_partials = lambda w, B, Hq, d, dev: tuple(
            t.double() for t in orig(w, B, Hq, d, dev))
        m, e, MA = D.dist_decode(None, None, None, q, case.scale, None, pages, out, rank, world,
                                 m_g=m_g, e_g=e_g, partial_fn=partial_fn, merge_fn=merge_fn)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), out=out.numpy(), m_g=m_g.numpy(),
                 e_g=e_g.numpy(), m=m.numpy(), e=e.numpy(), MA=MA.numpy(),
                 pages=np.array([p.tolist() for p in pages], dtype=object), allow_pickle=True)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(tmp_path, world, scheme):
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path), scheme), nprocs=world,
                       join=True, start_method="spawn")
    return [np.load(tmp_path / f"rank{r}.npz", allow_pickle=True) for r in range(world)]


@pytest.mark.parametrize("world,scheme", [(2, "blocked"), (3, "strided"), (2, "strided")])
def test_exchange_merges_to_full_attention_on_every_rank(tmp_path, world, scheme):
    import oracle
    res = _run(tmp_path, world, scheme)
    case = _case()
    qb = oracle.bf16_bits(case.q(0, "cpu"))
    # the shares cover every page exactly once
    for b, L in enumerate(case.lens):
        got = sorted(p for r in res for p in r["pages"][b])
        assert got == list(range(-(-L // case.P)))
    for b, L in enumerate(case.lens):
        K, V = (oracle.bf16_bits(x) for x in case.kv(b, 0, L, "cpu"))
        for h in range(case.Hq):
            ref, rm, re = oracle.attention(qb[b, h], K[:, h // case.g].copy(),
                                           V[:, h // case.g].copy(), case.scale)
            for r in res:  # every rank holds the full result
                np.testing.assert_allclose(r["out"][b, h], ref, rtol=0, atol=1e-12)
                assert abs(r["m_g"][b, h] - rm) <= 1e-12 and abs(r["e_g"][b, h] - re) <= 1e-9
    # every rank sees the same stacked partials, row r being rank r's
    for r in res[1:]:
        np.testing.assert_array_equal(r["m"], res[0]["m"])
        np.testing.assert_array_equal(r["MA"], res[0]["MA"])


def test_short_request_leaves_empty_partials_on_ranks_without_its_pages(tmp_path):
    res = _run(tmp_path, 3, "blocked")
    # request 2 has 5 tokens: one page, held by rank 2 (blocked: ranks 0, 1 get none)
    m = res[0]["m"]
    assert np.isneginf(m[0, 2]).all() and np.isneginf(m[1, 2]).all()
    assert (res[0]["e"][0, 2] == 0).all() and np.isfinite(m[2, 2]).all()


def test_page_schemes_partition_the_pages():
    from split_kv_decode_distattention_gb300.distributed import rank_pages
    for npages in (0, 1, 5, 64, 1001):
        for world in (1, 2, 3, 8):
            for scheme in ("blocked", "strided"):
                parts = [rank_pages(npages, r, world, scheme) for r in range(world)]
                allp = np.sort(np.concatenate(parts))
                np.testing.assert_array_equal(allp, np.arange(npages))
    with pytest.raises(ValueError):
        rank_pages(4, 2, 2)
