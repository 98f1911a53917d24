"""The kernels of the cross-GPU DistAttention decode on one GPU: the ranks' shares of every
request's pages run through dattn_partial one after another, each into its row of the stacked
partials, and dattn_merge_gathered merges them. Only the all-gather between GPUs is left out
(every box here has one GPU); its host logic is tested over gloo in test_distributed.py."""
import math

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_distattention_gb300 import workloads as W

from _util import assert_out_close, check_dense

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _lib():
    import split_kv_decode_distattention_gb300 as dattn
    dattn.load_library()
    return dattn


@pytest.mark.parametrize("world,scheme", [(2, "blocked"), (3, "strided"), (4, "blocked"),
                                          (1, "blocked")])
def test_simulated_ranks_merge_to_full_attention(world, scheme):
    dattn = _lib()
    from split_kv_decode_distattention_gb300 import distributed as D
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.Case("dist", B=4, Hq=16, Hkv=4, d=128, P=16, lens=[3000, 16, 1, 777], seed=19)
    cache = PagedCache(case, DEV)
    q = case.q(0, DEV)
    m, e, MA = D.stacked_partials(world, case.B, case.Hq, case.d, DEV)
    for r in range(world):
        pages = [D.rank_pages(-(-L // case.P), r, world, scheme) for L in case.lens]
        D.local_partials(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                         cache.seq_lens, pages, m[r], e[r], MA[r], dev_err=cache.dev_err)
    out = torch.empty(case.B, case.Hq, case.d, device=DEV)
    m_g = torch.empty(case.B, case.Hq, device=DEV)
    e_g = torch.empty_like(m_g)
    dattn.dattn_merge_gathered(m, e, MA, out=out, m_g=m_g, e_g=e_g, dev_err=cache.dev_err)
    ref = torch.empty_like(out)
    ref_m, ref_e = torch.empty_like(m_g), torch.empty_like(e_g)
    cache.decode(q, ref, cache.workspace(), m_g=ref_m, e_g=ref_e)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    check_dense(case, q, case.lens, out, m_g, e_g, DEV, what=f"{world} ranks {scheme}")
    assert_out_close(out.cpu().numpy(), ref.cpu().numpy(), "vs the fused decode")
    # request 2 (one token) lives on one rank: the other ranks' partials are empty
    owners = [r for r in range(world) if math.isfinite(m[r, 2, 0].item())]
    assert len(owners) == 1 and all((e[r, 2] == 0).all() for r in range(world) if r not in owners)


def test_dist_decode_single_rank_is_the_product_path():
    dattn = _lib()
    from split_kv_decode_distattention_gb300 import distributed as D
    from split_kv_decode_distattention_gb300.harness import PagedCache
    case = W.Case("dist1", B=2, Hq=8, Hkv=2, d=64, P=16, lens=[500, 64], seed=20)
    cache = PagedCache(case, DEV)
    q = case.q(0, DEV)
    pages = [D.rank_pages(-(-L // case.P), 0, 1) for L in case.lens]
    out = torch.empty(case.B, case.Hq, case.d, device=DEV)
    m_g = torch.empty(case.B, case.Hq, device=DEV)
    e_g = torch.empty_like(m_g)
    D.dist_decode(cache.layout, cache.k_pool, cache.v_pool, q, case.scale, cache.seq_lens,
                  pages, out, 0, 1, m_g=m_g, e_g=e_g, dev_err=cache.dev_err)
    torch.cuda.synchronize()
    assert int(cache.dev_err.item()) == 0
    check_dense(case, q, case.lens, out, m_g, e_g, DEV, what="one rank")


def test_merge_gathered_of_no_ranks_and_of_empty_partials():
    dattn = _lib()
    B, Hq, d = 2, 4, 64
    m = torch.full((3, B, Hq), -math.inf, device=DEV)
    e = torch.zeros(3, B, Hq, device=DEV)
    MA = torch.zeros(3, B, Hq, d, device=DEV)
    m[1, 0], e[1, 0], MA[1, 0] = 0.5, 2.0, 3.0  # one non-empty partial for request 0
    out = torch.full((B, Hq, d), float("nan"), device=DEV)
    m_g = torch.full((B, Hq), float("nan"), device=DEV)
    e_g = torch.full_like(m_g, float("nan"))
    dattn.dattn_merge_gathered(m, e, MA, out=out, m_g=m_g, e_g=e_g)
    torch.cuda.synchronize()
    assert torch.allclose(out[0], torch.full((Hq, d), 1.5, device=DEV))
    assert (m_g[0] == 0.5).all() and (e_g[0] == 2.0).all()
    assert (out[1] == 0).all() and (m_g[1] == -math.inf).all() and (e_g[1] == 0).all()
