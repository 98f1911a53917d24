"""split_kv_decode_distattention_gb300: split-KV decode attention over a paged KV cache.

This module is a thin Python binding of libdattn.so, the C-ABI library built from ``csrc/``.
It only marshals arguments: torch tensors become device pointers, and the current torch
stream becomes the launch stream. Every step of the computation runs in the library's
CUDA kernels. There is no CPU fallback: if the library is missing, the first call raises.

Entry points, with the same names as in include/dattn.h:
  dattn_kv_append    paged KV append (bf16, or 8-bit E4M3 or 4-bit codes with row scales),
                     plus logical-page k_max/k_min statistics
  dattn_partial      MicroAttention partials (m, e, MA) over explicit chunks of pages
  dattn_merge        log-sum-exp aggregation of partials
  dattn_decode       fused split-KV decode, dense or block-sparse
  dattn_append_decode one decode step with its one-token append, in one launch (bf16 pool)
  dattn_decode_multi fused decode of T new query tokens per request, causal over them
  dattn_page_select  page scoring and top-K selection for retrieval heads
  dattn_prefill      block-sparse prefill of a chunk of new tokens (64-token key blocks)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "KVLayout", "SparseConfig", "DattnError", "load_library", "library_path",
    "dattn_kv_append", "dattn_partial", "dattn_merge", "dattn_decode", "dattn_page_select",
    "dattn_append_decode", "dattn_merge_gathered",
    "dattn_decode_noalloc", "dattn_decode_multi", "dattn_prefill", "PrefillSparseConfig",
    "dattn_workspace_size", "dattn_workspace_init", "dattn_auto_splits", "dattn_split_range",
    "dattn_split_owner", "dattn_status_string", "dattn_version", "Workspace",
    "HEAD_DENSE", "HEAD_RETRIEVAL", "HEAD_STREAMING", "DEVERR", "KV_BF16", "KV_FP8_E4M3",
    "KV_INT4", "KV_MIXED", "mixed_pool_bytes",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libdattn.so")
_lib = None
_lock = threading.Lock()

HEAD_DENSE, HEAD_RETRIEVAL, HEAD_STREAMING = 0, 1, 2
KV_BF16, KV_FP8_E4M3, KV_INT4, KV_MIXED = 0, 1, 2, 3
_QUANT = (KV_FP8_E4M3, KV_INT4, KV_MIXED)
DEVERR = {"UNMAPPED_PAGE": 0x1, "PAGE_OOB": 0x2, "LEN_OOB": 0x4, "TIMEOUT": 0x8,
          "CHUNK_OOB": 0x10, "SELECT_OOB": 0x20, "SMEM_ALIGN": 0x40}


class DattnError(RuntimeError):
    """A dattn call returned a status other than DATTN_OK."""


class _Layout(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("block_table", ctypes.c_void_p), ("max_pages_per_req", ctypes.c_int32),
                ("kv_format", ctypes.c_int32), ("kv_scale", ctypes.c_void_p),
                ("head_format", ctypes.c_void_p)]


class _Sparse(ctypes.Structure):
    _fields_ = [("head_kind", ctypes.c_void_p), ("sinks", ctypes.c_int32),
                ("local", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("selected", ctypes.c_void_p), ("selected_phys", ctypes.c_void_p)]


class _PrefillSparse(ctypes.Structure):
    _fields_ = [("head_kind", ctypes.c_void_p), ("sink_blocks", ctypes.c_int32),
                ("local_blocks", ctypes.c_int32), ("max_sel", ctypes.c_int32),
                ("qblock_stride", ctypes.c_int32), ("block_lists", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_SIGS = {
    "dattn_kv_append": (_I, [ctypes.POINTER(_Layout), _P, _P, _P, _P, _P, _I, _I, _P, _P, _P]),
    "dattn_partial": (_I, [ctypes.POINTER(_Layout), _P, _P, _P, _I, _I, _F, _P, _I, _P, _P, _P,
                           _P, _P, _P, _P, _SZ, _I, _P, _P]),
    "dattn_merge": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dattn_merge_gathered": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dattn_decode": (_I, [ctypes.POINTER(_Layout), _P, _P, _P, _I, _I, _F, _P,
                          ctypes.POINTER(_Sparse), _I, _P, _SZ, _P, _P, _P, _P, _P]),
    "dattn_page_select": (_I, [ctypes.POINTER(_Layout), _P, _P, _I, _I, _P, _P, _I, _P, _P, _P,
                               _SZ, _I, _P, _P]),
    "dattn_append_decode": (_I, [ctypes.POINTER(_Layout), _P, _P, _P, _P, _P, _P, _I, _I, _F, _P,
                                 ctypes.POINTER(_Sparse), _I, _P, _SZ, _P, _P, _P, _P, _P]),
    "dattn_decode_noalloc": (_I, [ctypes.POINTER(_Layout), _P, _P, _P, _I, _I, _F, _P,
                                  ctypes.POINTER(_Sparse), _I, _P, _P, _P, _P, _P]),
    "dattn_decode_multi": (_I, [ctypes.POINTER(_Layout), _P, _P, _P, _I, _I, _I, _F, _P, _I, _P,
                                _SZ, _P, _P, _P, _P, _P]),
    "dattn_prefill": (_I, [ctypes.POINTER(_Layout), _P, _P, _P, _I, _I, _I, _F, _P,
                           ctypes.POINTER(_PrefillSparse), _P, _P, _P, _P, _P]),
    "dattn_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "dattn_workspace_init": (_I, [_P, _SZ, _P]),
    "dattn_auto_splits": (_I, [_I64]),
    "dattn_split_range": (None, [_I64, _I, _I, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "dattn_split_owner": (_I, [_I64, _I64, _I]),
    "dattn_status_string": (ctypes.c_char_p, [_I]),
    "dattn_version": (ctypes.c_char_p, []),
}


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load libdattn.so (built in-tree by ``_build.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise DattnError(
                f"{p} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _check(status: int, what: str):
    if status != 0:
        msg = load_library().dattn_status_string(status).decode()
        raise DattnError(f"{what} failed: {msg}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bf16(t, name):
    if t is not None and t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    return t


def _i32(t, name):
    if t is not None and t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return t


def _f32(t, name):
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    return t


def _size(t, n: int, name: str):
    """A tensor argument must hold at least the n elements the call will touch: the kernels
    see only a pointer, so a short tensor would be read or written past its end."""
    if t is not None and t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements; the call needs {n}")
    return t


def mixed_pool_bytes(num_pages: int, head_format, head_dim: int, page_size: int) -> int:
    """Bytes of one (K or V) mixed pool: the 8-bit region [num_pages][H8][P][d], then the 4-bit
    region [num_pages][H4][P][d/2]."""
    h4 = sum(1 for f in head_format if f == KV_INT4)
    h8 = len(head_format) - h4
    return num_pages * page_size * (h8 * head_dim + h4 * (head_dim // 2))


def _layout_sizes(layout, B: int, k_pool, v_pool, stats=None):
    """The pools, block table, scales and statistics must cover the layout for B requests."""
    c = layout.c
    n = c.num_pages * c.num_kv_heads * c.page_size
    if c.kv_format == KV_MIXED:
        pool = mixed_pool_bytes(c.num_pages, layout.head_format, c.head_dim, c.page_size)
    else:
        pool = n * (c.head_dim // 2 if c.kv_format == KV_INT4 else c.head_dim)
    _size(k_pool, pool, "k_pool")
    _size(v_pool, pool, "v_pool")
    _size(layout.block_table, B * c.max_pages_per_req, "block_table")
    if c.kv_format in _QUANT:
        _size(layout.kv_scale, 2 * n, "kv_scale")
    _size(stats, n // 16 * 2 * c.head_dim, "stats")


def _pool(layout, t, name):
    """A K or V pool must hold the layout's element type: bf16, uint8 E4M3 codes, or uint8
    bytes of two 4-bit codes (the mixed pool: both kinds of bytes)."""
    want = torch.uint8 if layout.kv_format in _QUANT else torch.bfloat16
    if t is not None and t.dtype != want and not (
            want == torch.uint8 and t.dtype == getattr(torch, "float8_e4m3fn", None)):
        raise TypeError(f"{name} must be {want} for this layout")
    return t


class KVLayout:
    """Shape of a paged pool [num_pages][Hkv][P][d] plus its int32 block table [B][max_pages].

    kv_format KV_BF16: the pools hold bf16 values. KV_FP8_E4M3: they hold uint8 E4M3 codes,
    and kv_scale (float32 [num_pages][Hkv][P/16][2][16]) holds one scale per row: for the 16
    tokens of each logical page, their K scales, then their V scales. KV_INT4: they hold
    [num_pages][Hkv][P][d/2] bytes of two 4-bit codes each (code + 8, even channel in the low
    nibble), with kv_scale as for KV_FP8_E4M3. KV_MIXED: head_format[h] (KV_FP8_E4M3 or
    KV_INT4) gives each KV head's format; the pools are that many bytes
    (mixed_pool_bytes): the 8-bit heads' region, then the 4-bit heads' region, each head at
    its index among the heads of its format.
    """

    def __init__(self, num_pages: int, num_kv_heads: int, head_dim: int, page_size: int,
                 block_table: torch.Tensor, kv_format: int = KV_BF16,
                 kv_scale: torch.Tensor | None = None, head_format=None):
        _i32(block_table, "block_table")
        if kv_format in _QUANT:
            if kv_scale is None:
                raise ValueError("the quantized formats need kv_scale")
            _f32(kv_scale, "kv_scale")
        self.head_format = None
        self._head_format_c = None
        if kv_format == KV_MIXED:
            if head_format is None or len(head_format) != num_kv_heads:
                raise ValueError("the mixed format needs one head_format entry per KV head")
            self.head_format = [int(f) for f in head_format]
            self._head_format_c = (ctypes.c_int8 * num_kv_heads)(*self.head_format)
        self.block_table = block_table  # keeps the tensors alive
        self.kv_scale = kv_scale
        self.c = _Layout(num_pages, num_kv_heads, head_dim, page_size,
                         block_table.data_ptr(), block_table.shape[-1], kv_format,
                         kv_scale.data_ptr() if kv_scale is not None else None,
                         ctypes.addressof(self._head_format_c)
                         if self._head_format_c is not None else None)

    @property
    def kv_format(self): return self.c.kv_format

    @property
    def num_pages(self): return self.c.num_pages

    @property
    def num_kv_heads(self): return self.c.num_kv_heads

    @property
    def head_dim(self): return self.c.head_dim

    @property
    def page_size(self): return self.c.page_size


class SparseConfig:
    """Block-sparse settings: per-KV-head kinds, streaming window and retrieval selection."""

    def __init__(self, head_kind: torch.Tensor, sinks: int, local: int, top_k: int,
                 selected: torch.Tensor | None, selected_phys: torch.Tensor | None = None):
        if head_kind.dtype != torch.int8:
            raise TypeError("head_kind must be int8")
        for t, n in ((selected, "selected"), (selected_phys, "selected_phys")):
            if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
                raise TypeError(f"{n} must be a contiguous int32 tensor")
        if selected is not None and selected_phys is not None and \
                selected_phys.numel() < selected.numel():
            raise ValueError("selected_phys must have the shape of selected")
        self.head_kind, self.selected, self.selected_phys = head_kind, selected, selected_phys
        self.c = _Sparse(head_kind.data_ptr(), sinks, local, top_k,
                         selected.data_ptr() if selected is not None else None,
                         selected_phys.data_ptr() if selected_phys is not None else None)


class PrefillSparseConfig:
    """Block-sparse prefill settings: per-KV-head kinds, the streaming heads' sink and local
    block counts, and the retrieval heads' key-block lists (int32 [B][Hkv][qblock_stride]
    [max_sel], row qb for query block qb, -1 padded)."""

    def __init__(self, head_kind: torch.Tensor, sink_blocks: int, local_blocks: int,
                 block_lists: torch.Tensor | None = None):
        if head_kind.dtype != torch.int8:
            raise TypeError("head_kind must be int8")
        _i32(block_lists, "block_lists")
        self.head_kind, self.block_lists = head_kind, block_lists
        qs, ms = (block_lists.shape[2], block_lists.shape[3]) if block_lists is not None else (0, 0)
        self.c = _PrefillSparse(head_kind.data_ptr(), sink_blocks, local_blocks, ms, qs,
                                block_lists.data_ptr() if block_lists is not None else None)


class Workspace:
    """A zeroed device workspace sized by dattn_workspace_size (allocated by torch)."""

    def __init__(self, items: int, Hq: int, Hkv: int, head_dim: int, top_k: int = 0,
                 num_splits: int = 0, device=None):
        self.nbytes = dattn_workspace_size(items, Hq, Hkv, head_dim, top_k, num_splits)
        n = max(self.nbytes, 256)
        self.buffer = torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def dattn_workspace_size(items, Hq, Hkv, head_dim, top_k=0, num_splits=0) -> int:
    return int(load_library().dattn_workspace_size(items, Hq, Hkv, head_dim, top_k, num_splits))


def dattn_workspace_init(ws: Workspace, stream=None):
    _check(load_library().dattn_workspace_init(_ptr(ws.buffer), ws.buffer.numel(),
                                               _stream(stream)), "dattn_workspace_init")


def dattn_auto_splits(total_tiles: int) -> int:
    return int(load_library().dattn_auto_splits(total_tiles))


def dattn_split_range(total_tiles: int, num_splits: int, cta: int):
    b, e = ctypes.c_int64(), ctypes.c_int64()
    load_library().dattn_split_range(total_tiles, num_splits, cta, ctypes.byref(b),
                                     ctypes.byref(e))
    return b.value, e.value


def dattn_split_owner(tile: int, total_tiles: int, num_splits: int) -> int:
    return int(load_library().dattn_split_owner(tile, total_tiles, num_splits))


def dattn_status_string(status: int) -> str:
    return load_library().dattn_status_string(status).decode()


def dattn_version() -> str:
    return load_library().dattn_version().decode()


def dattn_kv_append(layout: KVLayout, k_pool, v_pool, stats, k_new, v_new, seq_lens,
                    dev_err=None, stream=None):
    """Append k_new/v_new ([B][T][Hkv][d] bf16) at seq_lens (int32 [B], advanced by T)."""
    _pool(layout, k_pool, "k_pool"); _pool(layout, v_pool, "v_pool"); _bf16(stats, "stats")
    _bf16(k_new, "k_new"); _bf16(v_new, "v_new"); _i32(seq_lens, "seq_lens")
    B, T = k_new.shape[0], k_new.shape[1]
    Hkv, d = layout.num_kv_heads, layout.head_dim
    _layout_sizes(layout, B, k_pool, v_pool, stats)
    _size(k_new, B * T * Hkv * d, "k_new"); _size(v_new, B * T * Hkv * d, "v_new")
    _size(seq_lens, B, "seq_lens")
    _check(load_library().dattn_kv_append(
        ctypes.byref(layout.c), _ptr(k_pool), _ptr(v_pool), _ptr(stats), _ptr(k_new),
        _ptr(v_new), B, T, _ptr(seq_lens), _ptr(dev_err), _stream(stream)), "dattn_kv_append")


def dattn_partial(layout: KVLayout, k_pool, v_pool, q, scale: float, seq_lens, chunk_req,
                  chunk_page_indptr, chunk_pages, m, e, MA, ws: Workspace, num_splits=0,
                  dev_err=None, stream=None):
    """MicroAttention partials of C chunks: m, e fp32 [C][Hq], MA fp32 [C][Hq][d]."""
    _pool(layout, k_pool, "k_pool"); _pool(layout, v_pool, "v_pool"); _bf16(q, "q"); _i32(seq_lens, "seq_lens"); _i32(chunk_req, "chunk_req")
    _i32(chunk_page_indptr, "chunk_page_indptr"); _i32(chunk_pages, "chunk_pages")
    _f32(m, "m"); _f32(e, "e"); _f32(MA, "MA")
    B, Hq = q.shape[0], q.shape[1]
    C = chunk_req.shape[0]
    d = layout.head_dim
    _layout_sizes(layout, B, k_pool, v_pool)
    _size(q, B * Hq * d, "q"); _size(seq_lens, B, "seq_lens")
    _size(chunk_page_indptr, C + 1, "chunk_page_indptr")
    _size(m, C * Hq, "m"); _size(e, C * Hq, "e"); _size(MA, C * Hq * d, "MA")
    _check(load_library().dattn_partial(
        ctypes.byref(layout.c), _ptr(k_pool), _ptr(v_pool), _ptr(q), B, Hq, scale,
        _ptr(seq_lens), C, _ptr(chunk_req), _ptr(chunk_page_indptr), _ptr(chunk_pages),
        _ptr(m), _ptr(e), _ptr(MA), _ptr(ws.buffer), ws.buffer.numel(), num_splits,
        _ptr(dev_err), _stream(stream)), "dattn_partial")


def dattn_merge(chunk_indptr, m, e, MA, out=None, m_g=None, e_g=None, MA_g=None, dev_err=None,
                stream=None):
    """Aggregate partials per request (chunk ranges from chunk_indptr int32 [B+1])."""
    _i32(chunk_indptr, "chunk_indptr")
    for t, n in ((m, "m"), (e, "e"), (MA, "MA"), (out, "out"), (m_g, "m_g"), (e_g, "e_g"),
                 (MA_g, "MA_g")):
        _f32(t, n)
    B = chunk_indptr.shape[0] - 1
    C, Hq, d = MA.shape
    _size(m, C * Hq, "m"); _size(e, C * Hq, "e")
    _size(out, B * Hq * d, "out"); _size(m_g, B * Hq, "m_g"); _size(e_g, B * Hq, "e_g")
    _size(MA_g, B * Hq * d, "MA_g")
    _check(load_library().dattn_merge(
        B, C, Hq, d, _ptr(chunk_indptr), _ptr(m), _ptr(e), _ptr(MA), _ptr(out), _ptr(m_g),
        _ptr(e_g), _ptr(MA_g), _ptr(dev_err), _stream(stream)), "dattn_merge")


def dattn_merge_gathered(m, e, MA, out=None, m_g=None, e_g=None, MA_g=None, dev_err=None,
                         stream=None):
    """Aggregate partials gathered from R ranks: m, e fp32 [R][B][Hq], MA fp32 [R][B][Hq][d]
    (rank r's dattn_partial over its pages, one chunk per request) -> out fp32 [B][Hq][d]."""
    for t, n in ((m, "m"), (e, "e"), (MA, "MA"), (out, "out"), (m_g, "m_g"), (e_g, "e_g"),
                 (MA_g, "MA_g")):
        _f32(t, n)
    if MA.dim() != 4:
        raise ValueError("MA must be fp32 [R][B][Hq][d]")
    R, B, Hq, d = MA.shape
    _size(m, R * B * Hq, "m"); _size(e, R * B * Hq, "e")
    _size(out, B * Hq * d, "out"); _size(m_g, B * Hq, "m_g"); _size(e_g, B * Hq, "e_g")
    _size(MA_g, B * Hq * d, "MA_g")
    _check(load_library().dattn_merge_gathered(
        B, R, Hq, d, _ptr(m), _ptr(e), _ptr(MA), _ptr(out), _ptr(m_g), _ptr(e_g), _ptr(MA_g),
        _ptr(dev_err), _stream(stream)), "dattn_merge_gathered")


def _decode_sizes(layout, B, T, Hq, k_pool, v_pool, q, seq_lens, out, m_g, e_g, sparse):
    d, Hkv = layout.head_dim, layout.num_kv_heads
    _layout_sizes(layout, B, k_pool, v_pool)
    _size(q, B * T * Hq * d, "q"); _size(out, B * T * Hq * d, "out")
    _size(m_g, B * T * Hq, "m_g"); _size(e_g, B * T * Hq, "e_g"); _size(seq_lens, B, "seq_lens")
    if sparse is not None:
        _size(sparse.head_kind, Hkv, "head_kind")
        _size(sparse.selected, B * Hkv * sparse.c.top_k, "selected")


def dattn_decode(layout: KVLayout, k_pool, v_pool, q, scale: float, seq_lens, out,
                 ws: Workspace, m_g=None, e_g=None, sparse: SparseConfig | None = None,
                 num_splits=0, dev_err=None, stream=None):
    """Fused split-KV decode: out fp32 [B][Hq][d] (+ m_g, e_g fp32 [B][Hq])."""
    _pool(layout, k_pool, "k_pool"); _pool(layout, v_pool, "v_pool"); _bf16(q, "q"); _i32(seq_lens, "seq_lens"); _f32(out, "out")
    B, Hq = q.shape[0], q.shape[1]
    _decode_sizes(layout, B, 1, Hq, k_pool, v_pool, q, seq_lens, out, m_g, e_g, sparse)
    sp = ctypes.byref(sparse.c) if sparse is not None else None
    _check(load_library().dattn_decode(
        ctypes.byref(layout.c), _ptr(k_pool), _ptr(v_pool), _ptr(q), B, Hq, scale,
        _ptr(seq_lens), sp, num_splits, _ptr(ws.buffer), ws.buffer.numel(), _ptr(out),
        _ptr(m_g), _ptr(e_g), _ptr(dev_err), _stream(stream)), "dattn_decode")


def dattn_append_decode(layout: KVLayout, k_pool, v_pool, stats, k_new, v_new, q, scale: float,
                        seq_lens, out, ws: Workspace, m_g=None, e_g=None,
                        sparse: SparseConfig | None = None, num_splits=0, dev_err=None,
                        stream=None):
    """dattn_kv_append of one token per request (k_new/v_new bf16 [B][1][Hkv][d]) and
    dattn_decode over the advanced lengths, in one launch (any pool format; a quantized pool
    stores the new rows quantized as dattn_kv_append would): out fp32 [B][Hq][d]
    (+ m_g, e_g fp32 [B][Hq]); seq_lens advances by one."""
    _pool(layout, k_pool, "k_pool"); _pool(layout, v_pool, "v_pool"); _bf16(stats, "stats")
    _bf16(k_new, "k_new"); _bf16(v_new, "v_new"); _bf16(q, "q"); _i32(seq_lens, "seq_lens")
    _f32(out, "out")
    B, Hq = q.shape[0], q.shape[1]
    Hkv, d = layout.num_kv_heads, layout.head_dim
    if k_new.dim() != 4 or k_new.shape[1] != 1 or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be bf16 [B][1][Hkv][d]")
    _layout_sizes(layout, B, k_pool, v_pool, stats)
    _size(k_new, B * Hkv * d, "k_new"); _size(v_new, B * Hkv * d, "v_new")
    _decode_sizes(layout, B, 1, Hq, k_pool, v_pool, q, seq_lens, out, m_g, e_g, sparse)
    sp = ctypes.byref(sparse.c) if sparse is not None else None
    _check(load_library().dattn_append_decode(
        ctypes.byref(layout.c), _ptr(k_pool), _ptr(v_pool), _ptr(stats), _ptr(k_new),
        _ptr(v_new), _ptr(q), B, Hq, scale, _ptr(seq_lens), sp, num_splits, _ptr(ws.buffer),
        ws.buffer.numel(), _ptr(out), _ptr(m_g), _ptr(e_g), _ptr(dev_err), _stream(stream)),
        "dattn_append_decode")


def dattn_decode_multi(layout: KVLayout, k_pool, v_pool, q, scale: float, seq_lens, out,
                       ws: Workspace, m_g=None, e_g=None, num_splits=0, dev_err=None, stream=None):
    """T query tokens per request (q bf16 [B][T][Hq][d]), causal over the T newest tokens:
    out fp32 [B][T][Hq][d] (+ m_g, e_g fp32 [B][T][Hq]). The workspace is sized for T * Hq
    query heads."""
    _pool(layout, k_pool, "k_pool"); _pool(layout, v_pool, "v_pool"); _bf16(q, "q")
    _i32(seq_lens, "seq_lens"); _f32(out, "out")
    B, T, Hq = q.shape[0], q.shape[1], q.shape[2]
    _decode_sizes(layout, B, T, Hq, k_pool, v_pool, q, seq_lens, out, m_g, e_g, None)
    _check(load_library().dattn_decode_multi(
        ctypes.byref(layout.c), _ptr(k_pool), _ptr(v_pool), _ptr(q), B, T, Hq, scale,
        _ptr(seq_lens), num_splits, _ptr(ws.buffer), ws.buffer.numel(), _ptr(out), _ptr(m_g),
        _ptr(e_g), _ptr(dev_err), _stream(stream)), "dattn_decode_multi")


def dattn_prefill(layout: KVLayout, k_pool, v_pool, q, scale: float, seq_lens, out, m=None,
                  e=None, sparse: PrefillSparseConfig | None = None, dev_err=None, stream=None):
    """Block-sparse (sparse given) or causal prefill of q bf16 [B][Tq][Hq][d], the last Tq
    tokens of each request: out fp32 [B][Tq][Hq][d] (+ m, e fp32 [B][Tq][Hq])."""
    _pool(layout, k_pool, "k_pool"); _pool(layout, v_pool, "v_pool"); _bf16(q, "q")
    _i32(seq_lens, "seq_lens"); _f32(out, "out"); _f32(m, "m"); _f32(e, "e")
    B, Tq, Hq = q.shape[0], q.shape[1], q.shape[2]
    _decode_sizes(layout, B, Tq, Hq, k_pool, v_pool, q, seq_lens, out, m, e, None)
    if sparse is not None:
        _size(sparse.head_kind, layout.num_kv_heads, "head_kind")
        if sparse.block_lists is not None and (sparse.block_lists.dim() != 4 or
                                               sparse.block_lists.shape[0] < B or
                                               sparse.block_lists.shape[1] < layout.num_kv_heads):
            raise ValueError("block_lists must be int32 [B][Hkv][qblock_stride][max_sel]")
    sp = ctypes.byref(sparse.c) if sparse is not None else None
    _check(load_library().dattn_prefill(
        ctypes.byref(layout.c), _ptr(k_pool), _ptr(v_pool), _ptr(q), B, Tq, Hq, scale,
        _ptr(seq_lens), sp, _ptr(out), _ptr(m), _ptr(e), _ptr(dev_err), _stream(stream)),
        "dattn_prefill")


def dattn_decode_noalloc(layout: KVLayout, k_pool, v_pool, q, scale: float, seq_lens, out,
                         m_g=None, e_g=None, sparse: SparseConfig | None = None, num_splits=0,
                         dev_err=None, stream=None):
    """dattn_decode with the library's fixed 8 MiB scratch array instead of a workspace.

    For callers that cannot allocate device memory. Calls on one device share the array, so
    they must not overlap on the GPU. The first call on a device should come before any
    stream capture.
    """
    _pool(layout, k_pool, "k_pool"); _pool(layout, v_pool, "v_pool"); _bf16(q, "q"); _i32(seq_lens, "seq_lens"); _f32(out, "out")
    B, Hq = q.shape[0], q.shape[1]
    _decode_sizes(layout, B, 1, Hq, k_pool, v_pool, q, seq_lens, out, m_g, e_g, sparse)
    sp = ctypes.byref(sparse.c) if sparse is not None else None
    _check(load_library().dattn_decode_noalloc(
        ctypes.byref(layout.c), _ptr(k_pool), _ptr(v_pool), _ptr(q), B, Hq, scale,
        _ptr(seq_lens), sp, num_splits, _ptr(out), _ptr(m_g), _ptr(e_g), _ptr(dev_err),
        _stream(stream)), "dattn_decode_noalloc")


def dattn_page_select(layout: KVLayout, stats, q, seq_lens, head_kind, top_k: int, selected,
                      ws: Workspace, num_splits=0, dev_err=None, stream=None, selected_phys=None):
    """Top-K physical pages per retrieval head into selected int32 [B][Hkv][top_k] (and their
    pool pages into selected_phys, of the same shape, when given)."""
    _bf16(stats, "stats"); _bf16(q, "q"); _i32(seq_lens, "seq_lens"); _i32(selected, "selected")
    _i32(selected_phys, "selected_phys")
    B, Hq = q.shape[0], q.shape[1]
    c = layout.c
    _size(stats, c.num_pages * c.num_kv_heads * (c.page_size // 16) * 2 * c.head_dim, "stats")
    _size(layout.block_table, B * c.max_pages_per_req, "block_table")
    _size(q, B * Hq * c.head_dim, "q"); _size(seq_lens, B, "seq_lens")
    _size(head_kind, c.num_kv_heads, "head_kind")
    _size(selected, B * c.num_kv_heads * top_k, "selected")
    if selected_phys is not None:
        _size(selected_phys, B * c.num_kv_heads * top_k, "selected_phys")
    _check(load_library().dattn_page_select(
        ctypes.byref(layout.c), _ptr(stats), _ptr(q), B, Hq, _ptr(seq_lens), _ptr(head_kind),
        top_k, _ptr(selected), _ptr(selected_phys), _ptr(ws.buffer), ws.buffer.numel(),
        num_splits, _ptr(dev_err), _stream(stream)), "dattn_page_select")
