"""Device-side driver for a seeded workload: allocate the paged pool, fill it through
dattn_kv_append, and run decode steps. Used by the smoke check, the GPU tests and the
benchmark. It calls only the library's entry points; the workload values come from
``workloads``.
"""
from __future__ import annotations

import torch

from . import (KV_BF16, KV_FP8_E4M3, KV_INT4, KV_MIXED, KVLayout, SparseConfig, Workspace,
               mixed_pool_bytes,
               dattn_append_decode, dattn_decode, dattn_decode_multi, dattn_kv_append,
               dattn_page_select)
from .workloads import Case


class PagedCache:
    """Pool [num_pages][Hkv][P][d] (K and V) plus statistics, block table and lengths.

    kv_format KV_BF16 keeps bf16 values; KV_FP8_E4M3 keeps uint8 E4M3 codes plus one float32
    scale per (token, KV head) row in kv_scale [num_pages][Hkv][P/16][2][16] (per logical
    page: 16 K scales, then 16 V scales); KV_INT4 keeps [num_pages][Hkv][P][d/2] bytes of two
    4-bit codes each, with kv_scale as for KV_FP8_E4M3. KV_MIXED keeps each KV head in the
    format head_format[h] names (flat uint8 pools: the 8-bit heads' region, then the 4-bit
    heads' region).
    """

    def __init__(self, case: Case, device="cuda", with_stats: bool = False, fill: bool = True,
                 chunk_tokens: int = 8192, zero_pool: bool = False, kv_format: int = KV_BF16,
                 head_format=None):
        self.case = case
        self.device = torch.device(device)
        c = case
        alloc = torch.zeros if zero_pool else torch.empty
        self.kv_format = kv_format
        self.head_format = list(head_format) if head_format is not None else None
        quant = kv_format in (KV_FP8_E4M3, KV_INT4, KV_MIXED)
        elem = torch.uint8 if quant else torch.bfloat16
        if kv_format == KV_MIXED:
            nbytes = mixed_pool_bytes(c.num_pages, self.head_format, c.d, c.P)
            self.k_pool = alloc(nbytes, dtype=elem, device=device)
            self.v_pool = alloc(nbytes, dtype=elem, device=device)
        else:
            row = c.d // 2 if kv_format == KV_INT4 else c.d
            self.k_pool = alloc(c.num_pages, c.Hkv, c.P, row, dtype=elem, device=device)
            self.v_pool = alloc(c.num_pages, c.Hkv, c.P, row, dtype=elem, device=device)
        self.kv_scale = None
        if quant:
            self.kv_scale = alloc(c.num_pages, c.Hkv, c.P // 16, 2, 16, dtype=torch.float32,
                                  device=device)
        self.stats = None
        if with_stats:
            self.stats = alloc(c.num_pages, c.Hkv, c.P // 16, 2, c.d, dtype=torch.bfloat16,
                               device=device)
        self.block_table = torch.as_tensor(c.block_table, dtype=torch.int32, device=device)
        self.layout = self._layout(self.block_table)
        self.seq_lens = torch.zeros(c.B, dtype=torch.int32, device=device)
        self.lens = [0] * c.B  # host mirror of seq_lens
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)
        self.chunk_tokens = chunk_tokens
        self._head_kind = None
        if fill:
            self.fill()

    def _layout(self, block_table) -> KVLayout:
        c = self.case
        return KVLayout(c.num_pages, c.Hkv, c.d, c.P, block_table, self.kv_format,
                        self.kv_scale, head_format=self.head_format)

    def _row_layout(self, b: int) -> KVLayout:
        return self._layout(self.block_table[b:b + 1])

    def fill(self, lens=None):
        """Append each request's tokens up to lens (default: the case's step-0 lengths)."""
        lens = self.case.lens if lens is None else lens
        for b, L in enumerate(lens):
            lay = self._row_layout(b)
            while self.lens[b] < L:
                t0 = self.lens[b]
                t1 = min(L, t0 + self.chunk_tokens)
                K, V = self.case.kv(b, t0, t1, self.device)
                dattn_kv_append(lay, self.k_pool, self.v_pool, self.stats,
                                K.unsqueeze(0).contiguous(), V.unsqueeze(0).contiguous(),
                                self.seq_lens[b:b + 1], self.dev_err)
                self.lens[b] = t1

    def new_tokens(self, T: int = 1):
        """The next T tokens of every request (continuing each seeded stream): [B][T][Hkv][d]."""
        ks, vs = [], []
        for b in range(self.case.B):
            K, V = self.case.kv(b, self.lens[b], self.lens[b] + T, self.device)
            ks.append(K)
            vs.append(V)
        return torch.stack(ks).contiguous(), torch.stack(vs).contiguous()

    def append(self, k_new, v_new):
        """One batched append of k_new/v_new ([B][T][Hkv][d]) at the current lengths."""
        T = k_new.shape[1]
        dattn_kv_append(self.layout, self.k_pool, self.v_pool, self.stats, k_new, v_new,
                        self.seq_lens, self.dev_err)
        self.lens = [L + T for L in self.lens]

    def workspace(self, top_k: int = 0, num_splits: int = 0, queries: int = 1) -> Workspace:
        """A workspace for decode (T query tokens per request: queries = T) or selection."""
        c = self.case
        return Workspace(c.B, c.Hq * queries, c.Hkv, c.d, top_k=top_k, num_splits=num_splits,
                         device=self.device)

    def head_kind(self) -> torch.Tensor:
        """The per-KV-head kinds on the device, copied once: a copy from pageable host memory
        would make every later call wait for the GPU to drain."""
        if self._head_kind is None:
            self._head_kind = torch.as_tensor(self.case.head_kind_array(), dtype=torch.int8,
                                              device=self.device)
        return self._head_kind

    def sparse_config(self, selected, selected_phys=None) -> SparseConfig:
        c = self.case
        return SparseConfig(self.head_kind(), c.sinks, c.local, c.top_k, selected, selected_phys)

    def decode(self, q, out, ws, m_g=None, e_g=None, sparse=None, num_splits=0):
        """q [B][Hq][d]: dattn_decode; q [B][T][Hq][d]: dattn_decode_multi (dense only)."""
        if q.dim() == 4:
            if sparse is not None:
                raise ValueError("the multi-query decode is dense only")
            dattn_decode_multi(self.layout, self.k_pool, self.v_pool, q, self.case.scale,
                               self.seq_lens, out, ws, m_g=m_g, e_g=e_g, num_splits=num_splits,
                               dev_err=self.dev_err)
            return
        dattn_decode(self.layout, self.k_pool, self.v_pool, q, self.case.scale, self.seq_lens,
                     out, ws, m_g=m_g, e_g=e_g, sparse=sparse, num_splits=num_splits,
                     dev_err=self.dev_err)

    def append_decode(self, k_new, v_new, q, out, ws, m_g=None, e_g=None, sparse=None,
                      num_splits=0):
        """One-token append and decode in one launch (dattn_append_decode)."""
        dattn_append_decode(self.layout, self.k_pool, self.v_pool, self.stats, k_new, v_new, q,
                            self.case.scale, self.seq_lens, out, ws, m_g=m_g, e_g=e_g,
                            sparse=sparse, num_splits=num_splits, dev_err=self.dev_err)
        self.lens = [L + 1 for L in self.lens]

    def select(self, q, selected, ws, num_splits=0, selected_phys=None):
        c = self.case
        dattn_page_select(self.layout, self.stats, q, self.seq_lens, self.head_kind(), c.top_k,
                          selected, ws, num_splits=num_splits, dev_err=self.dev_err,
                          selected_phys=selected_phys)
