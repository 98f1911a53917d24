"""Seeded synthetic inputs for the split-KV decode path.

This module produces inputs only: query vectors, token-ordered K/V streams, block tables,
lengths, page-set partitions and head kinds. It holds none of the method's arithmetic, so the
oracle and the CUDA path can both consume what it produces without sharing any computation.

Every value is a deterministic function of (seed, what, indices). K/V of a request are
generated in fixed chunks of ``GEN_CHUNK`` tokens, so any token range can be regenerated on
its own: a test can rebuild the keys of one (request, head) long after the pool was filled.

The workload shapes follow the pages' settings:
  * "dense-tiny": a small GQA case (8 query heads over 2 KV heads, head_dim 64, 4096 tokens,
    16-token pages, identity block table). It is split into 4 chunks of 1024 tokens.
  * "mha-32k": Llama-2-7B-shaped MHA decode (32 heads, head_dim 128, batch 8, 32K tokens),
    with 16-token pages scattered through a shuffled pool. The LoongServe notes evaluate on
    the Llama-2-7B-based LWM-1M model.
  * "mha-1m": one request of 2^20 tokens with 64 "needle" keys aligned to the query.
  * "gqa-ragged": 64 requests of Llama-3-8B GQA shape (32 q / 8 KV heads) with
    log-uniform lengths from 1K to 256K, plus page-set partitions (2-8 sets per request).
    This matches DistAttention sub-blocks and LoongServe multi-master decoding.
  * "sparse-512k": the LServe block-sparse decode. It uses 64-token physical pages of four
    16-token logical pages, retrieval heads (top-64 pages) and streaming heads (4 sinks plus
    8 local tokens), with 32 high-similarity pages per retrieval head.
  * "prefill-32k": the LServe block-sparse prefill of one 32K-token request of Llama-3-8B
    GQA shape, as one chunk: half the KV heads streaming (one sink block and 16 local blocks
    of 64 tokens), half retrieval, whose key-block lists keep a seeded 65% of the earlier
    blocks plus the query's own block (the pages report that block sparsity skips about 35%
    of the retrieval heads' prefill work).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

GEN_CHUNK = 2048  # tokens per independently seeded K/V block

HEAD_DENSE, HEAD_RETRIEVAL, HEAD_STREAMING = 0, 1, 2


def _mix(*vals: int) -> int:
    """splitmix64 over a tuple of integers; a stable seed for torch/numpy generators."""
    x = 0x9E3779B97F4A7C15
    for v in vals:
        x = (x ^ (int(v) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x = z ^ (z >> 31)
    return x & 0x7FFFFFFFFFFFFFFF


_TAG = {"q": 1, "kv": 2, "table": 3, "lens": 4, "needle": 5, "highsim": 6, "sets": 7,
        "new": 8, "blocks": 9, "qchunk": 10}


def _gen(device, *key) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(*key))
    return g


def _np_rng(*key) -> np.random.Generator:
    return np.random.default_rng(_mix(*key))


@dataclass
class Case:
    """A paged decode workload: shapes, lengths, block table and sparse settings."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    P: int
    lens: list            # context length of each request at step 0
    seed: int = 0
    scale: float = 0.0
    shuffle: bool = True  # False: identity block table (request b owns a contiguous range)
    reserve_tokens: int = 64  # spare capacity per request for appended tokens
    n_needles: int = 0
    head_kind: list | None = None   # per KV head: 0 dense, 1 retrieval, 2 streaming
    top_k: int = 0
    sinks: int = 4
    local: int = 8
    reuse: int = 16
    n_highsim: int = 0
    chunk_tokens: int = 0  # > 0: dattn_partial chunks of this many tokens (dense-tiny)
    page_sets: bool = False
    block_table: np.ndarray = field(default=None, repr=False)
    num_pages: int = 0
    max_pages: int = 0

    def __post_init__(self):
        self._memo = {}
        if self.scale == 0.0:
            self.scale = 1.0 / math.sqrt(self.d)
        self.lens = [int(x) for x in self.lens]
        if self.block_table is None:
            self._make_block_table()

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    def _make_block_table(self):
        caps = [-(-(L + self.reserve_tokens) // self.P) for L in self.lens]
        self.max_pages = max(caps) if caps else 0
        self.num_pages = int(sum(caps))
        perm = np.arange(self.num_pages, dtype=np.int64)
        if self.shuffle:
            perm = _np_rng(self.seed, _TAG["table"]).permutation(self.num_pages)
        bt = np.full((self.B, max(self.max_pages, 1)), -1, np.int32)
        off = 0
        for b, c in enumerate(caps):
            bt[b, :c] = perm[off:off + c]
            off += c
        self.block_table = bt

    # -------------------------------------------------------------------- queries
    def q(self, step: int = 0, device="cpu") -> torch.Tensor:
        """Query vectors [B][Hq][d] (bf16) of decode step ``step``."""
        g = _gen(device, self.seed, _TAG["q"], step)
        x = torch.randn(self.B, self.Hq, self.d, generator=g, device=device)
        return x.to(torch.bfloat16)

    # -------------------------------------------------------------------- K / V
    def _needles(self, b: int) -> np.ndarray:
        L = self.lens[b]
        n = min(self.n_needles, L)
        if n <= 0:
            return np.zeros(0, np.int64)
        key = ("needle", b)
        if key not in self._memo:
            self._memo[key] = np.sort(_np_rng(self.seed, _TAG["needle"], b)
                                      .choice(L, size=n, replace=False))
        return self._memo[key]

    def highsim_pages(self, b: int, kvh: int) -> np.ndarray:
        """Request-relative physical pages whose keys lean toward the group's query."""
        if self.n_highsim <= 0 or self.head_kind is None or \
                self.head_kind[kvh] != HEAD_RETRIEVAL:
            return np.zeros(0, np.int64)
        key = ("hs", b, kvh)
        if key not in self._memo:
            npages = -(-self.lens[b] // self.P)
            n = min(self.n_highsim, npages)
            self._memo[key] = np.sort(_np_rng(self.seed, _TAG["highsim"], b, kvh)
                                      .choice(npages, size=n, replace=False))
        return self._memo[key]

    def _direction(self, b: int, kvh: int, device) -> torch.Tensor:
        """Unit vector of the mean query of KV head kvh's group at step 0 (fp32, [d])."""
        key = ("dir", str(device), b, kvh)
        if key not in self._memo:
            q = self.q(0, device)[b, kvh * self.g:(kvh + 1) * self.g].float().mean(0)
            self._memo[key] = q / q.norm()
        return self._memo[key]

    def kv(self, b: int, t0: int, t1: int, device="cpu"):
        """Token-ordered K and V of request b, tokens [t0, t1): bf16 [t1-t0][Hkv][d] each.

        Tokens past the step-0 length continue the same seeded stream. They are the tokens
        that decode steps append.
        """
        t0, t1 = int(t0), int(t1)
        n = max(t1 - t0, 0)
        K = torch.empty(n, self.Hkv, self.d, dtype=torch.bfloat16, device=device)
        V = torch.empty_like(K)
        c0, c1 = t0 // GEN_CHUNK, (t1 - 1) // GEN_CHUNK if n else -1
        for c in range(c0, c1 + 1):
            g = _gen(device, self.seed, _TAG["kv"], b, c)
            Kc = torch.randn(GEN_CHUNK, self.Hkv, self.d, generator=g, device=device)
            Vc = torch.randn(GEN_CHUNK, self.Hkv, self.d, generator=g, device=device)
            base = c * GEN_CHUNK
            # input structure: high-similarity pages (sparse workload)
            if self.n_highsim > 0:
                for kvh in range(self.Hkv):
                    pages = self.highsim_pages(b, kvh)
                    if pages.size == 0:
                        continue
                    lo_p, hi_p = base // self.P, (base + GEN_CHUNK - 1) // self.P
                    inside = pages[(pages >= lo_p) & (pages <= hi_p)]
                    if inside.size == 0:
                        continue
                    u = self._direction(b, kvh, device)
                    for p in inside:
                        a = max(int(p) * self.P, base)
                        z = min((int(p) + 1) * self.P, base + GEN_CHUNK)
                        if a < z:
                            Kc[a - base:z - base, kvh] += 8.0 * u
            lo, hi = max(t0, base), min(t1, base + GEN_CHUNK)
            K[lo - t0:hi - t0] = Kc[lo - base:hi - base].to(torch.bfloat16)
            V[lo - t0:hi - t0] = Vc[lo - base:hi - base].to(torch.bfloat16)
        # input structure: needle keys aligned with each head's query (1M-token workload)
        if self.n_needles > 0 and n:
            pos = self._needles(b)
            sel = pos[(pos >= t0) & (pos < t1)]
            if sel.size:
                q = self.q(0, device)[b].float()  # [Hq][d]
                for kvh in range(self.Hkv):
                    qg = q[kvh * self.g:(kvh + 1) * self.g].mean(0)
                    key = (4.0 * qg / qg.norm()).to(torch.bfloat16)
                    idx = torch.as_tensor(sel - t0, device=device)
                    K[idx, kvh] = key
        return K, V

    # -------------------------------------------------------------------- structure
    def page_sets_of(self, b: int, L: int | None = None) -> list:
        """Disjoint, non-contiguous sets of request-relative pages covering request b."""
        L = self.lens[b] if L is None else L
        npages = -(-L // self.P)
        rng = _np_rng(self.seed, _TAG["sets"], b)
        n = int(rng.integers(2, 9))
        n = min(n, max(npages, 1))
        while True:
            assign = rng.integers(0, n, size=npages)
            sets = [np.nonzero(assign == j)[0].astype(np.int32) for j in range(n)]
            if all(s.size for s in sets) or npages == 0:
                return sets

    def prefill_queries(self, Tq: int, device="cpu", step: int = 0) -> torch.Tensor:
        """Query vectors [B][Tq][Hq][d] (bf16) of a prefill chunk of Tq tokens."""
        g = _gen(device, self.seed, _TAG["qchunk"], step)
        x = torch.randn(self.B, Tq, self.Hq, self.d, generator=g, device=device)
        return x.to(torch.bfloat16)

    def prefill_block_lists(self, keep: float = 0.65, stride: int | None = None) -> np.ndarray:
        """Key-block lists [B][Hkv][stride][stride] (int32, -1 padded) for retrieval heads:
        row qb holds a seeded fraction `keep` of the blocks 0 .. qb-1, then qb itself."""
        stride = stride or max(-(-L // 64) for L in self.lens)
        out = np.full((self.B, self.Hkv, stride, stride), -1, np.int32)
        for b in range(self.B):
            for h in range(self.Hkv):
                rng = _np_rng(self.seed, _TAG["blocks"], b, h)
                for qb in range(stride):
                    kept = np.nonzero(rng.random(qb) < keep)[0]
                    row = np.concatenate([kept, [qb]]).astype(np.int32)
                    out[b, h, qb, :row.size] = row
        return out

    def head_kind_array(self) -> np.ndarray:
        hk = self.head_kind if self.head_kind is not None else [HEAD_DENSE] * self.Hkv
        return np.asarray(hk, np.int8)

    def kv_bytes(self, lens=None) -> int:
        """K+V bytes of the valid tokens (bf16)."""
        lens = self.lens if lens is None else lens
        return int(sum(lens)) * self.Hkv * self.d * 2 * 2


# --------------------------------------------------------------------------- named cases

def dense_tiny(seed: int = 0) -> Case:
    """Batch 1, 8 q heads / 2 KV heads, head_dim 64, 4096 tokens, identity table, 4 chunks."""
    return Case("dense-tiny", B=1, Hq=8, Hkv=2, d=64, P=16, lens=[4096], seed=seed,
                shuffle=False, chunk_tokens=1024)


def mha_32k(seed: int = 0, B: int = 8, L: int = 32768) -> Case:
    """Llama-2-7B-shaped MHA: batch 8, 32 heads, head_dim 128, 32K tokens, shuffled pool."""
    return Case("mha-32k", B=B, Hq=32, Hkv=32, d=128, P=16, lens=[L] * B, seed=seed)


def mha_1m(seed: int = 0, L: int = 1 << 20) -> Case:
    """One request of 2^20 tokens, 32 heads MHA, head_dim 128, 64 needle keys."""
    return Case("mha-1m", B=1, Hq=32, Hkv=32, d=128, P=16, lens=[L], seed=seed, n_needles=64)


def gqa_ragged(seed: int = 0, B: int = 64, lo: int = 1024, hi: int = 262144) -> Case:
    """64 requests, 32 q / 8 KV heads, head_dim 128, lengths log-uniform in [1K, 256K]."""
    rng = _np_rng(seed, _TAG["lens"])
    lens = np.round(np.exp(rng.uniform(math.log(lo), math.log(hi), size=B))).astype(np.int64)
    return Case("gqa-ragged", B=B, Hq=32, Hkv=8, d=128, P=16, lens=lens.tolist(), seed=seed,
                page_sets=True)


def sparse_512k(seed: int = 0, B: int = 8, L: int = 524288) -> Case:
    """LServe block-sparse: 32 q / 8 KV heads, 64-token pages, top-64, reuse 16, 4+8 window."""
    kinds = [HEAD_RETRIEVAL] * 4 + [HEAD_STREAMING] * 4
    return Case("sparse-512k", B=B, Hq=32, Hkv=8, d=128, P=64, lens=[L] * B, seed=seed,
                head_kind=kinds, top_k=64, sinks=4, local=8, reuse=16, n_highsim=32)


def prefill_32k(seed: int = 0, L: int = 32768) -> Case:
    """LServe block-sparse prefill: one 32K request, 32 q / 8 KV heads, head_dim 128, as one
    chunk; KV heads 0-3 retrieval (65% of earlier blocks), 4-7 streaming (1 + 16 blocks)."""
    kinds = [HEAD_RETRIEVAL] * 4 + [HEAD_STREAMING] * 4
    return Case("prefill-32k", B=1, Hq=32, Hkv=8, d=128, P=16, lens=[L], seed=seed,
                head_kind=kinds, reserve_tokens=0)


PREFILL_SINK_BLOCKS, PREFILL_LOCAL_BLOCKS, PREFILL_KEEP = 1, 16, 0.65

CASES = {
    "dense-tiny": dense_tiny,
    "mha-32k": mha_32k,
    "mha-1m": mha_1m,
    "gqa-ragged": gqa_ragged,
    "sparse-512k": sparse_512k,
    "prefill-32k": prefill_32k,
}


def random_bf16(shape, seed: int, *key, device="cpu", scale: float = 1.0) -> torch.Tensor:
    """N(0, scale^2) values rounded to bf16, from a generator seeded by (seed, key)."""
    g = _gen(device, seed, 99, *key)
    return (torch.randn(*shape, generator=g, device=device) * scale).to(torch.bfloat16)
