"""Cross-GPU DistAttention decode: partials on every rank, one all-gather, one merge.

"Infinite-LLM: Efficient LLM Service for Long Context with DistAttention and Distributed
KVCache" ("结果聚合与通信开销降低", Fig. 4b) spreads the KV cache of one request over
instances. Each instance computes MicroAttention partials (m_j, e_j, MA_j) over the KV it
holds, and the partials are sent back and aggregated. "LoongServe" §4.2 (multi-master
distributed decoding) does the same with every instance as a master of its own requests.

Here a rank is one GPU with its own paged pool. It holds a share of every request's pages,
mapped by its own block table (pages it does not hold are unmapped). One decode step is:

1. ``dattn_partial`` over the rank's pages, one chunk per request, writing its rows of the
   stacked buffers m, e [R][B][Hq] and MA [R][B][Hq][d] in place (row r is rank r's);
2. one all-gather of those rows (``torch.distributed.all_gather_into_tensor``), which moves
   B * Hq * (d + 2) floats per rank;
3. ``dattn_merge_gathered`` on every rank, which leaves the full attention of every request.

The page assignment and the gather are host logic. They are tested on the CPU over gloo, with
the oracle's partials and merge standing in for the kernels (the ``partial_fn`` and
``merge_fn`` arguments). The kernels themselves are tested on one GPU with the ranks' shares
computed one after another into the stacked buffers.
"""
from __future__ import annotations

import numpy as np
import torch

from . import Workspace, dattn_merge_gathered, dattn_partial


def rank_pages(npages: int, rank: int, world: int, scheme: str = "blocked") -> np.ndarray:
    """Request-relative pages rank `rank` of `world` holds.

    "blocked": contiguous runs of about npages / world pages (DistAttention's sub-blocks);
    "strided": page p on rank p mod world (round robin). Every page is held by exactly one
    rank, and a rank may hold none of a short request's pages.
    """
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if scheme == "blocked":
        lo, hi = npages * rank // world, npages * (rank + 1) // world
        return np.arange(lo, hi, dtype=np.int32)
    if scheme == "strided":
        return np.arange(rank, npages, world, dtype=np.int32)
    raise ValueError(f"unknown page scheme {scheme!r}")


def chunk_lists(page_lists):
    """chunk_req, chunk_page_indptr and chunk_pages (int32 numpy) for one chunk per request,
    chunk b over the pages in page_lists[b]."""
    B = len(page_lists)
    indptr = np.zeros(B + 1, np.int32)
    for b, pages in enumerate(page_lists):
        indptr[b + 1] = indptr[b] + len(pages)
    pages = (np.concatenate([np.asarray(p, np.int32) for p in page_lists])
             if indptr[-1] > 0 else np.zeros(1, np.int32))
    return np.arange(B, dtype=np.int32), indptr, pages


def stacked_partials(world: int, B: int, Hq: int, d: int, device):
    """The stacked buffers m, e [world][B][Hq] and MA [world][B][Hq][d] (fp32)."""
    m = torch.empty(world, B, Hq, dtype=torch.float32, device=device)
    e = torch.empty_like(m)
    MA = torch.empty(world, B, Hq, d, dtype=torch.float32, device=device)
    return m, e, MA


def gather_partials(m, e, MA, rank: int, group=None):
    """Fills every rank's rows of the stacked buffers from the rank that computed them (each
    rank has written row `rank`)."""
    import torch.distributed as dist
    for t in (m, e, MA):
        # NCCL gathers in place when the input is the output's own row; other backends get a
        # separate input
        mine = t[rank] if t.is_cuda else t[rank].clone()
        # the output as the concatenation of the ranks' rows along dim 0 (every backend)
        dist.all_gather_into_tensor(t.view(-1, *t.shape[2:]), mine, group=group)


def local_partials(layout, k_pool, v_pool, q, scale: float, seq_lens, page_lists, m_row,
                   e_row, MA_row, ws: Workspace | None = None, dev_err=None, stream=None):
    """dattn_partial of this rank's pages of every request into its rows of the stacked
    buffers (m_row, e_row [B][Hq], MA_row [B][Hq][d]: views of row `rank`)."""
    dev = q.device
    req, indptr, pages = chunk_lists(page_lists)
    chunk_req = torch.as_tensor(req, device=dev)
    chunk_indptr = torch.as_tensor(indptr, device=dev)
    chunk_pages = torch.as_tensor(pages, device=dev)
    B, Hq, d = q.shape[0], q.shape[1], layout.head_dim
    if ws is None:
        ws = Workspace(B, Hq, layout.num_kv_heads, d, device=dev)
    dattn_partial(layout, k_pool, v_pool, q, scale, seq_lens, chunk_req, chunk_indptr,
                  chunk_pages, m_row, e_row, MA_row, ws, dev_err=dev_err, stream=stream)


def dist_decode(layout, k_pool, v_pool, q, scale: float, seq_lens, page_lists, out,
                rank: int, world: int, group=None, m_g=None, e_g=None, ws=None, dev_err=None,
                partial_fn=None, merge_fn=None):
    """One cross-GPU decode step on this rank (see the module notes). page_lists[b] holds
    the request-relative pages of request b that this rank's pool maps. Returns the stacked
    partials (m, e, MA) after the gather.

    partial_fn(m_row, e_row, MA_row) and merge_fn(m, e, MA, out, m_g, e_g) replace the
    kernels (tests on the CPU); by default they are dattn_partial and dattn_merge_gathered.
    """
    B, Hq = q.shape[0], q.shape[1]
    d = layout.head_dim if layout is not None else out.shape[-1]
    m, e, MA = stacked_partials(world, B, Hq, d, q.device)
    if partial_fn is None:
        local_partials(layout, k_pool, v_pool, q, scale, seq_lens, page_lists, m[rank],
                       e[rank], MA[rank], ws=ws, dev_err=dev_err)
    else:
        partial_fn(m[rank], e[rank], MA[rank])
    if world > 1:
        gather_partials(m, e, MA, rank, group)
    if merge_fn is None:
        dattn_merge_gathered(m, e, MA, out=out, m_g=m_g, e_g=e_g, dev_err=dev_err)
    else:
        merge_fn(m, e, MA, out, m_g, e_g)
    return m, e, MA
