"""Helpers shared by the GPU parity tests: tolerances and oracle references of a Case."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Output tolerance (bf16 inputs, fp32 accumulation): an element passes iff
#   |gpu - ref| <= 2e-3  and  |gpu - ref| / max(|ref|, 0.2) <= 1e-2.
ATOL, RTOL, RFLOOR = 2e-3, 1e-2, 0.2
M_RTOL, E_RTOL = 1e-4, 1e-4


def assert_out_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    rel = err / np.maximum(np.abs(ref), RFLOOR)
    bad = (err > ATOL) | (rel > RTOL) | ~np.isfinite(got)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err, -1)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: got {got[i]!r}, ref {ref[i]!r}")


def assert_m_close(got, ref, what=""):
    got, ref = float(got), float(ref)
    if ref == -np.inf:
        assert got == -np.inf, f"{what}: m {got} != -inf"
        return
    assert abs(got - ref) <= M_RTOL * max(1.0, abs(ref)), f"{what}: m {got} vs {ref}"


def assert_e_close(got, ref, what=""):
    got, ref = float(got), float(ref)
    assert abs(got - ref) <= E_RTOL * max(abs(ref), 1e-30), f"{what}: e {got} vs {ref}"


def host_kv(case, b: int, L: int, device):
    """Token-ordered K, V of request b (tokens 0..L-1) as uint16 numpy arrays [L][Hkv][d]."""
    K, V = case.kv(b, 0, L, device)
    return oracle.bf16_bits(K), oracle.bf16_bits(V)


def oracle_dense(case, q, lens, device, pairs=None, nthreads=None):
    """Oracle dense attention of (b, h) pairs: dict (b, h) -> (out, m, e)."""
    qb = oracle.bf16_bits(q)
    if pairs is None:
        pairs = [(b, h) for b in range(case.B) for h in range(case.Hq)]
    res = {}
    by_req = {}
    for b, h in pairs:
        by_req.setdefault(b, []).append(h)
    for b, hs in by_req.items():
        K, V = host_kv(case, b, lens[b], device)
        out, m, e, _ = oracle.attention_pairs(qb[b:b + 1], K, V, [0, lens[b]],
                                              [(0, h) for h in hs], case.scale,
                                              nthreads=nthreads)
        for i, h in enumerate(hs):
            res[(b, h)] = (out[i], m[i], e[i])
    return res


def check_dense(case, q, lens, out, m_g, e_g, device, pairs=None, what="decode"):
    ref = oracle_dense(case, q, lens, device, pairs=pairs)
    o = out.cpu().numpy()
    mg = m_g.cpu().numpy() if m_g is not None else None
    eg = e_g.cpu().numpy() if e_g is not None else None
    for (b, h), (r, rm, re) in ref.items():
        assert_out_close(o[b, h], r, f"{what} b={b} h={h} L={lens[b]}")
        if mg is not None:
            assert_m_close(mg[b, h], rm, f"{what} b={b} h={h}")
        if eg is not None:
            assert_e_close(eg[b, h], re, f"{what} b={b} h={h}")


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits(t)


def check_selection(got, score, bound, top_k, what=""):
    """Checks one row of a GPU page selection against the fp64 page scores.

    LServe article §3.1.2 keeps the top_k pages by score, ties to the lower page (reading
    R6 of the oracle). The GPU scores in fp32, and ``bound`` holds each fp64 score's fp32
    error bound. Where every page of the fp64 top-K stays above every other page by more
    than their bounds, the selection is unique and the row must equal the oracle's bit for
    bit. Otherwise the row must be a valid top-K under the bounds: no rejected page may be
    certainly above a chosen one. Returns True for a unique row, False for an ambiguous one.
    """
    got = np.asarray(got)
    score = np.asarray(score, np.float64)
    bound = np.asarray(bound, np.float64)
    n = score.shape[0]
    k = min(top_k, n)
    want = oracle.topk(score, top_k)
    assert got.shape == (top_k,), f"{what}: row shape {got.shape}"
    assert (got[k:] == -1).all(), f"{what}: padding {got[k:]}"
    sel = got[:k]
    assert ((sel >= 0) & (sel < n)).all(), f"{what}: pages out of range {sel}"
    assert (np.diff(sel) > 0).all(), f"{what}: not strictly ascending {sel}"
    if k == n:
        np.testing.assert_array_equal(got, want, err_msg=what)
        return True
    inset = np.zeros(n, bool)
    inset[want[:k]] = True
    if (score - bound)[inset].min() > (score + bound)[~inset].max():
        np.testing.assert_array_equal(got, want, err_msg=f"{what}: unique selection")
        return True
    chosen = np.zeros(n, bool)
    chosen[sel] = True
    lo = (score + bound)[chosen].min()
    hi = (score - bound)[~chosen].max()
    assert lo >= hi, (f"{what}: a rejected page (fp64 score - bound {hi!r}) is certainly above "
                      f"a chosen one (score + bound {lo!r})")
    return False
