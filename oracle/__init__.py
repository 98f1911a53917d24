"""dattn oracle: TEST INFRASTRUCTURE ONLY.

This is a plain, slow, double-precision CPU implementation of what the split-KV decode path
computes. The arithmetic lives in ``dattn_oracle.c``, which is plain C compiled with gcc
without fast-math and without floating-point contraction. This module only marshals numpy
arrays into it.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this package. The CUDA library never calls it, and it never calls the CUDA library.

bf16 tensors travel as their raw 16-bit patterns (numpy ``uint16``). The C code widens them
exactly to double.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

# gcc flags: no fast-math and no contraction, so every rounding step is the one written in C.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-pthread", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build_oracle(out_path: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile dattn_oracle.c into a shared library with gcc and return its path."""
    cmd = ["gcc", *CFLAGS, *extra_flags, _SRC, "-o", out_path + ".tmp", "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(out_path + ".tmp", out_path)
    return out_path


def _needs_rebuild() -> bool:
    if not os.path.exists(_LIB_PATH):
        return True
    lib_t = os.path.getmtime(_LIB_PATH)
    return any(os.path.getmtime(os.path.join(_HERE, f)) > lib_t
               for f in ("dattn_oracle.c", "dattn_oracle.h"))


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_D = ctypes.c_double

_SIGS = {
    "orc_bf16_to_double": (_D, [ctypes.c_uint16]),
    "orc_attention": (None, [_P, _P, _P, _I64, _I, _P, _I64, _D, _P, _P, _P]),
    "orc_partial": (None, [_P, _P, _P, _I64, _I, _P, _I64, _D, _P, _P, _P]),
    "orc_merge": (None, [_I, _P, _P, _P, _I, _P, _P, _P, _P]),
    "orc_kv_write": (_I64, [_P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _I64, _I64]),
    "orc_logical_page_stats": (None, [_P, _I64, _I, _I64, _I64, _P, _P]),
    "orc_logical_score_f64": (_D, [_P, _P, _P, _I]),
    "orc_logical_score_bound": (_D, [_P, _P, _P, _I]),
    "orc_page_scores": (None, [_P, _I, _P, _I64, _I, _I64, _I, _P, _P]),
    "orc_topk": (None, [_P, _I64, _I, _P]),
    "orc_sparse_rows": (_I64, [_I, _I64, _I, _P, _I, _I, _I, _P]),
    "orc_prefill_rows": (_I64, [_I, _I64, _I64, _I64, _I, _I, _P, _I, _P]),
    "orc_attention_pairs_mt": (_I, [_P, _P, _P, _P, _I, _I, _I, _D, _P, _I64, _I, _P, _P, _P]),
    "orc_e4m3_value": (_D, [ctypes.c_uint8]),
    "orc_e4m3_code": (ctypes.c_uint8, [ctypes.c_float]),
    "orc_quantize_row_fp8": (None, [_P, _I, _P, _P]),
    "orc_dequantize_row_fp8": (None, [_P, ctypes.c_float, _I, _P]),
    "orc_quantize_rows_fp8": (None, [_P, _I64, _I, _P, _P]),
    "orc_dequantize_rows_fp8": (None, [_P, _P, _I64, _I, _P]),
    "orc_kv_write_fp8": (_I64, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _I64, _I64]),
    "orc_quantize_row_int4": (None, [_P, _I, _P, _P]),
    "orc_int4_code": (_I, [_P, _I]),
    "orc_dequantize_row_int4": (None, [_P, ctypes.c_float, _I, _P]),
    "orc_quantize_rows_int4": (None, [_P, _I64, _I, _P, _P]),
    "orc_dequantize_rows_int4": (None, [_P, _P, _I64, _I, _P]),
    "orc_kv_write_int4": (_I64, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _I64, _I64]),
    "orc_attention_f64": (None, [_P, _P, _P, _I64, _I, _P, _I64, _D, _P, _P, _P]),
    "orc_partial_f64": (None, [_P, _P, _P, _I64, _I, _P, _I64, _D, _P, _P, _P]),
}


def load(path: str | None = None):
    """Load the compiled oracle, building it first if it is missing or stale."""
    global _lib
    with _lock:
        if path is not None:
            lib = ctypes.CDLL(path)
        else:
            if _lib is not None:
                return _lib
            if _needs_rebuild():
                build_oracle()
            lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


# ----------------------------------------------------------------------------- marshalling

def bf16_bits(x) -> np.ndarray:
    """Raw 16-bit patterns of a bf16 tensor (torch) or of an existing uint16 array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("expected bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch  # only for torch inputs
    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected a bfloat16 tensor, got {x.dtype}")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows):
    if rows is None:
        return None
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


# ------------------------------------------------------------------------------ functions

def attention(q, K, V, scale: float, rows=None, lib=None):
    """Full softmax attention of one query (``q`` [d]) over rows of K, V ([n][d]).

    Returns (out [d] float64, m, e). Infinite-LLM notes, full-attention equations.
    """
    lib = lib or load()
    q, K, V = bf16_bits(q), bf16_bits(K), bf16_bits(V)
    d = q.shape[-1]
    K2 = K.reshape(-1, d)
    V2 = V.reshape(-1, d)
    r = _rows(rows)
    n = K2.shape[0] if r is None else r.shape[0]
    out = np.zeros(d, np.float64)
    m = ctypes.c_double()
    e = ctypes.c_double()
    lib.orc_attention(_ptr(q), _ptr(K2), _ptr(V2), d, d, _ptr(r), n, scale, _ptr(out),
                      ctypes.byref(m), ctypes.byref(e))
    return out, m.value, e.value


def partial(q, K, V, scale: float, rows=None, lib=None):
    """MicroAttention triple (m_j, e_j, MA_j) over rows of K, V. Infinite-LLM notes."""
    lib = lib or load()
    q, K, V = bf16_bits(q), bf16_bits(K), bf16_bits(V)
    d = q.shape[-1]
    K2 = K.reshape(-1, d)
    V2 = V.reshape(-1, d)
    r = _rows(rows)
    n = K2.shape[0] if r is None else r.shape[0]
    MA = np.zeros(d, np.float64)
    m = ctypes.c_double()
    e = ctypes.c_double()
    lib.orc_partial(_ptr(q), _ptr(K2), _ptr(V2), d, d, _ptr(r), n, scale, ctypes.byref(m),
                    ctypes.byref(e), _ptr(MA))
    return m.value, e.value, MA


def merge(m, e, MA, lib=None):
    """Aggregate b partials. Returns (m_g, e_g, out [d], MA_g [d]). Infinite-LLM notes."""
    lib = lib or load()
    m = np.ascontiguousarray(np.asarray(m, np.float64).reshape(-1))
    e = np.ascontiguousarray(np.asarray(e, np.float64).reshape(-1))
    MA = np.ascontiguousarray(np.asarray(MA, np.float64))
    b = m.shape[0]
    d = MA.shape[-1]
    MA = MA.reshape(b, d)
    out = np.zeros(d, np.float64)
    MA_g = np.zeros(d, np.float64)
    mg = ctypes.c_double()
    eg = ctypes.c_double()
    lib.orc_merge(b, _ptr(m), _ptr(e), _ptr(MA), d, ctypes.byref(mg), ctypes.byref(eg),
                  _ptr(out), _ptr(MA_g))
    return mg.value, eg.value, out, MA_g


def kv_write(k_pool: np.ndarray, v_pool: np.ndarray, block_table_row, num_pages: int,
             k_new, v_new, pos0: int, lib=None) -> int:
    """Write T tokens of one request into uint16 pools [num_pages][Hkv][P][d] in place.

    ``k_new``/``v_new`` are [T][Hkv][d]. Returns the number of tokens skipped because their
    page is unmapped or out of range. LoongServe notes §4.2 (the master saves new KV).
    """
    lib = lib or load()
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    _, Hkv, P, d = k_pool.shape
    kn, vn = bf16_bits(k_new), bf16_bits(v_new)
    T = kn.shape[0]
    bt = np.ascontiguousarray(np.asarray(block_table_row, np.int32))
    return lib.orc_kv_write(_ptr(k_pool), _ptr(v_pool), Hkv, P, d, _ptr(bt), bt.shape[0],
                            num_pages, _ptr(kn), _ptr(vn), pos0, T)


def logical_page_stats(K, t0: int, t1: int, lib=None):
    """(k_max, k_min) over token rows [t0, t1) of K ([n][d]). LServe notes §3.1.2."""
    lib = lib or load()
    K = bf16_bits(K)
    d = K.shape[-1]
    K2 = K.reshape(-1, d)
    kmax = np.zeros(d, np.uint16)
    kmin = np.zeros(d, np.uint16)
    lib.orc_logical_page_stats(_ptr(K2), d, d, t0, t1, _ptr(kmax), _ptr(kmin))
    return kmax, kmin


def logical_score(q, kmax, kmin, lib=None) -> float:
    """Logical-page score sum_d max(q_d kmax_d, q_d kmin_d) in fp64. LServe notes §3.1.2."""
    lib = lib or load()
    q, kmax, kmin = bf16_bits(q), bf16_bits(kmax), bf16_bits(kmin)
    return float(lib.orc_logical_score_f64(_ptr(q), _ptr(kmax), _ptr(kmin), q.shape[-1]))


def logical_score_bound(q, kmax, kmin, lib=None) -> float:
    """Bound on the error of any fp32 evaluation of logical_score (reading R9)."""
    lib = lib or load()
    q, kmax, kmin = bf16_bits(q), bf16_bits(kmax), bf16_bits(kmin)
    return float(lib.orc_logical_score_bound(_ptr(q), _ptr(kmax), _ptr(kmin), q.shape[-1]))


def page_scores(Q, K, L: int, P: int, with_bounds: bool = False, lib=None):
    """fp64 physical-page scores of one request/KV head (Q: [g][d], K: [>=L][d] in token
    order). With ``with_bounds`` also the fp32 error bound of each score: (score, bound)."""
    lib = lib or load()
    Q, K = bf16_bits(Q), bf16_bits(K)
    d = Q.shape[-1]
    Q2 = Q.reshape(-1, d)
    K2 = K.reshape(-1, d)
    n = (L + P - 1) // P
    score = np.zeros(max(n, 1), np.float64)
    bound = np.zeros(max(n, 1), np.float64)
    lib.orc_page_scores(_ptr(Q2), Q2.shape[0], _ptr(K2), d, d, L, P, _ptr(score), _ptr(bound))
    return (score[:n], bound[:n]) if with_bounds else score[:n]


def topk(score, top_k: int, lib=None) -> np.ndarray:
    """Top-K page indices (ties to the lower index), ascending, padded with -1."""
    lib = lib or load()
    s = np.ascontiguousarray(np.asarray(score, np.float64))
    sel = np.zeros(max(top_k, 1), np.int32)
    lib.orc_topk(_ptr(s), s.shape[0], top_k, _ptr(sel))
    return sel[:top_k]


def select_pages(Q, K, L: int, P: int, top_k: int, lib=None) -> np.ndarray:
    """Page selection of one request/KV head: the top-K of the fp64 page scores."""
    return topk(page_scores(Q, K, L, P, lib=lib), top_k, lib=lib)


def sparse_rows(kind: int, L: int, P: int, sel, sinks: int, local: int, lib=None) -> np.ndarray:
    """Token rows attended by one head: 0 dense, 1 retrieval (selected pages), 2 streaming."""
    lib = lib or load()
    s = np.ascontiguousarray(np.asarray(sel if sel is not None else [-1], np.int32))
    rows = np.zeros(max(L, 1), np.int64)
    n = lib.orc_sparse_rows(kind, L, P, _ptr(s), s.shape[0] if sel is not None else 0,
                            sinks, local, _ptr(rows))
    return rows[:n]


def prefill_rows(kind: int, L: int, Tq: int, t: int, sink_blocks: int = 0,
                 local_blocks: int = 0, blocks=None, lib=None) -> np.ndarray:
    """Key rows query token t of a Tq-token chunk attends in the block-sparse prefill:
    kind 0 dense, 1 retrieval (blocks: its query block's key-block list), 2 streaming."""
    lib = lib or load()
    b = np.ascontiguousarray(np.asarray(blocks if blocks is not None else [-1], np.int32))
    rows = np.zeros(max(L, 1), np.int64)
    n = lib.orc_prefill_rows(kind, L, Tq, t, sink_blocks, local_blocks, _ptr(b),
                             b.shape[0] if blocks is not None else 0, _ptr(rows))
    return rows[:n]


def attention_pairs(q, K_cat, V_cat, offs, pairs, scale: float, nthreads: int | None = None,
                    lib=None):
    """Dense decode attention for (request, query head) pairs on host threads.

    q: [B][Hq][d]; K_cat/V_cat: token-ordered [sum L][Hkv][d]; offs: [B+1] token offsets.
    Returns (out [n][d], m [n], e [n], threads used).
    """
    lib = lib or load()
    q, K, V = bf16_bits(q), bf16_bits(K_cat), bf16_bits(V_cat)
    B, Hq, d = q.shape
    Hkv = K.shape[-2]
    offs = np.ascontiguousarray(np.asarray(offs, np.int64))
    pairs = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    n = pairs.shape[0]
    out = np.zeros((n, d), np.float64)
    m = np.zeros(n, np.float64)
    e = np.zeros(n, np.float64)
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    used = lib.orc_attention_pairs_mt(_ptr(q), _ptr(K), _ptr(V), _ptr(offs), Hq, Hkv, d,
                                      scale, _ptr(pairs), n, nthreads, _ptr(out), _ptr(m),
                                      _ptr(e))
    return out, m, e, used


# ----------------------------------------------------------------- 8-bit KV (reading R10)

def e4m3_value(code: int, lib=None) -> float:
    """Value of an FP8 E4M3 code."""
    return float((lib or load()).orc_e4m3_value(int(code)))


def e4m3_code(f: float, lib=None) -> int:
    """E4M3 code of a float (rounded to fp32 first): nearest, ties to even, saturating."""
    return int((lib or load()).orc_e4m3_code(float(np.float32(f))))


def quantize_rows_fp8(X, lib=None):
    """Rows of bf16 values ([n][d] or [d]) -> (codes uint8 [n][d], scales float32 [n])."""
    lib = lib or load()
    X = bf16_bits(X)
    d = X.shape[-1]
    X2 = np.ascontiguousarray(X.reshape(-1, d))
    codes = np.zeros(X2.shape, np.uint8)
    scales = np.zeros(X2.shape[0], np.float32)
    lib.orc_quantize_rows_fp8(_ptr(X2), X2.shape[0], d, _ptr(codes), _ptr(scales))
    return codes.reshape(X.shape), scales.reshape(X.shape[:-1])


def dequantize_rows_fp8(codes, scales, lib=None) -> np.ndarray:
    """code * scale of every row, in float64."""
    lib = lib or load()
    codes = np.ascontiguousarray(codes, np.uint8)
    d = codes.shape[-1]
    c2 = codes.reshape(-1, d)
    s2 = np.ascontiguousarray(np.asarray(scales, np.float32).reshape(-1))
    out = np.zeros(c2.shape, np.float64)
    lib.orc_dequantize_rows_fp8(_ptr(c2), _ptr(s2), c2.shape[0], d, _ptr(out))
    return out.reshape(codes.shape)


def kv_write_fp8(k_pool, v_pool, k_scale, v_scale, P: int, block_table_row, num_pages: int,
                 k_new, v_new, pos0: int, lib=None) -> int:
    """Paged 8-bit write of k_new/v_new ([T][Hkv][d] bf16) into uint8 pools
    [num_pages][Hkv][P][d] and float32 scales [num_pages][Hkv][P]; returns skipped tokens."""
    lib = lib or load()
    k_new, v_new = bf16_bits(k_new), bf16_bits(v_new)
    T, Hkv, d = k_new.shape
    bt = np.ascontiguousarray(np.asarray(block_table_row, np.int32))
    return int(lib.orc_kv_write_fp8(_ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), Hkv,
                                    P, d, _ptr(bt), bt.shape[0], num_pages, _ptr(k_new),
                                    _ptr(v_new), pos0, T))


# ----------------------------------------------------------------- 4-bit KV (reading R12)

def quantize_rows_int4(X, lib=None):
    """Rows of bf16 values ([n][d] or [d], d even) -> (packed uint8 [n][d/2], scales float32
    [n]): byte i of a row holds code + 8 of channel 2i (low nibble) and 2i + 1 (high)."""
    lib = lib or load()
    X = bf16_bits(X)
    d = X.shape[-1]
    X2 = np.ascontiguousarray(X.reshape(-1, d))
    packed = np.zeros((X2.shape[0], d // 2), np.uint8)
    scales = np.zeros(X2.shape[0], np.float32)
    lib.orc_quantize_rows_int4(_ptr(X2), X2.shape[0], d, _ptr(packed), _ptr(scales))
    return packed.reshape(X.shape[:-1] + (d // 2,)), scales.reshape(X.shape[:-1])


def int4_codes(packed, lib=None) -> np.ndarray:
    """The signed codes (-8 .. 7) of packed 4-bit rows ([..][d/2] -> [..][d] int8)."""
    lib = lib or load()
    packed = np.ascontiguousarray(packed, np.uint8)
    h = packed.shape[-1]
    flat = packed.reshape(-1, h)
    out = np.zeros((flat.shape[0], 2 * h), np.int8)
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        for c in range(2 * h):
            out[r, c] = lib.orc_int4_code(_ptr(row), c)
    return out.reshape(packed.shape[:-1] + (2 * h,))


def dequantize_rows_int4(packed, scales, lib=None) -> np.ndarray:
    """code * scale of every packed 4-bit row, in float64 ([..][d/2] -> [..][d])."""
    lib = lib or load()
    packed = np.ascontiguousarray(packed, np.uint8)
    h = packed.shape[-1]
    p2 = packed.reshape(-1, h)
    s2 = np.ascontiguousarray(np.asarray(scales, np.float32).reshape(-1))
    out = np.zeros((p2.shape[0], 2 * h), np.float64)
    lib.orc_dequantize_rows_int4(_ptr(p2), _ptr(s2), p2.shape[0], 2 * h, _ptr(out))
    return out.reshape(packed.shape[:-1] + (2 * h,))


def kv_write_int4(k_pool, v_pool, k_scale, v_scale, P: int, block_table_row, num_pages: int,
                  k_new, v_new, pos0: int, lib=None) -> int:
    """Paged 4-bit write of k_new/v_new ([T][Hkv][d] bf16) into uint8 pools
    [num_pages][Hkv][P][d/2] and float32 scales [num_pages][Hkv][P]; returns skipped tokens."""
    lib = lib or load()
    k_new, v_new = bf16_bits(k_new), bf16_bits(v_new)
    T, Hkv, d = k_new.shape
    bt = np.ascontiguousarray(np.asarray(block_table_row, np.int32))
    return int(lib.orc_kv_write_int4(_ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
                                     Hkv, P, d, _ptr(bt), bt.shape[0], num_pages, _ptr(k_new),
                                     _ptr(v_new), pos0, T))


def attention_f64(q, K, V, scale: float, rows=None, lib=None):
    """orc_attention over float64 keys and values ([n][d]): (out [d], m, e)."""
    lib = lib or load()
    q = bf16_bits(q)
    K2 = np.ascontiguousarray(np.asarray(K, np.float64))
    V2 = np.ascontiguousarray(np.asarray(V, np.float64))
    d = q.shape[-1]
    r = _rows(rows)
    n = K2.shape[0] if r is None else r.shape[0]
    out = np.zeros(d, np.float64)
    m = ctypes.c_double()
    e = ctypes.c_double()
    lib.orc_attention_f64(_ptr(q), _ptr(K2), _ptr(V2), d, d, _ptr(r), n, scale, _ptr(out),
                          ctypes.byref(m), ctypes.byref(e))
    return out, m.value, e.value


def partial_f64(q, K, V, scale: float, rows=None, lib=None):
    """orc_partial over float64 keys and values: (m_j, e_j, MA_j [d])."""
    lib = lib or load()
    q = bf16_bits(q)
    K2 = np.ascontiguousarray(np.asarray(K, np.float64))
    V2 = np.ascontiguousarray(np.asarray(V, np.float64))
    d = q.shape[-1]
    r = _rows(rows)
    n = K2.shape[0] if r is None else r.shape[0]
    MA = np.zeros(d, np.float64)
    m = ctypes.c_double()
    e = ctypes.c_double()
    lib.orc_partial_f64(_ptr(q), _ptr(K2), _ptr(V2), d, d, _ptr(r), n, scale, ctypes.byref(m),
                        ctypes.byref(e), _ptr(MA))
    return m.value, e.value, MA
