"""Host-side checks of libdattn.so that need no GPU: it loads, it exports every symbol
include/dattn.h declares, it rejects bad arguments before launching anything, and its
balanced split plan partitions the tiles exactly."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dattn():
    from split_kv_decode_distattention_gb300 import _build
    _build.build()
    import split_kv_decode_distattention_gb300 as d
    d.load_library()
    return d


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "dattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dattn_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(dattn):
    names = _declared_symbols()
    assert {"dattn_kv_append", "dattn_partial", "dattn_merge", "dattn_decode",
            "dattn_page_select"} <= set(names)
    lib = ctypes.CDLL(dattn.library_path())
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_version_and_status_strings(dattn):
    assert "sm_103a" in dattn.dattn_version()
    assert dattn.dattn_status_string(0) == "DATTN_OK"
    assert dattn.dattn_status_string(3) == "DATTN_ERR_WORKSPACE"
    assert dattn.dattn_status_string(99) == "DATTN_UNKNOWN_STATUS"


def test_split_plan_partitions_tiles_exactly(dattn):
    rng = np.random.default_rng(0)
    for _ in range(200):
        W = int(rng.integers(0, 5000))
        G = int(rng.integers(1, 700))
        ranges = [dattn.dattn_split_range(W, G, c) for c in range(G)]
        assert ranges[0][0] == 0 and ranges[-1][1] == W
        sizes = [e - b for b, e in ranges]
        assert all(ranges[c][1] == ranges[c + 1][0] for c in range(G - 1))
        assert max(sizes) - min(sizes) <= 1
        if W:
            for t in rng.integers(0, W, size=20):
                c = dattn.dattn_split_owner(int(t), W, G)
                b, e = ranges[c]
                assert b <= t < e
    assert dattn.dattn_split_owner(5, 5, 3) == -1


def test_split_slots_are_distinct_per_cta_and_segment(dattn):
    """A piece of segment s in CTA c uses workspace slot c + s; slots never collide."""
    rng = np.random.default_rng(1)
    for _ in range(50):
        lens = rng.integers(0, 40, size=int(rng.integers(1, 30)))
        W = int(lens.sum())
        G = int(rng.integers(1, 50))
        if W == 0:
            continue
        starts = np.concatenate([[0], np.cumsum(lens)])
        used = set()
        for s, n in enumerate(lens):
            if n == 0:
                continue
            c0 = dattn.dattn_split_owner(int(starts[s]), W, G)
            c1 = dattn.dattn_split_owner(int(starts[s] + n - 1), W, G)
            if c0 == c1:
                continue  # finished inside one CTA, no slot
            for c in range(c0, c1 + 1):
                assert (c + s) not in used
                used.add(c + s)
                assert c + s < G + len(lens)


def _lay(dattn, **kw):
    import torch
    bt = torch.zeros(1, 4, dtype=torch.int32)
    args = dict(num_pages=8, num_kv_heads=2, head_dim=128, page_size=16)
    args.update(kw)
    return dattn.KVLayout(args["num_pages"], args["num_kv_heads"], args["head_dim"],
                          args["page_size"], bt)


def _decode_status(dattn, layout, B=1, Hq=4, sparse=None):
    lib = dattn.load_library()
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    return lib.dattn_decode(ctypes.byref(layout.c) if layout else None, p, p, p, B, Hq, 0.1, p,
                            sparse, 0, p, 1 << 20, p, None, None, None, None)


def test_decode_rejects_bad_shapes_before_launch(dattn):
    INVALID, UNSUPPORTED = 1, 2
    assert _decode_status(dattn, None) == INVALID
    assert _decode_status(dattn, _lay(dattn, head_dim=96)) == UNSUPPORTED
    assert _decode_status(dattn, _lay(dattn, page_size=24)) == UNSUPPORTED
    assert _decode_status(dattn, _lay(dattn, page_size=512)) == UNSUPPORTED
    assert _decode_status(dattn, _lay(dattn), Hq=3) == INVALID          # Hq % Hkv != 0
    assert _decode_status(dattn, _lay(dattn), Hq=18 * 2) == UNSUPPORTED  # group of 18
    assert _decode_status(dattn, _lay(dattn), B=5000) == UNSUPPORTED
    assert _decode_status(dattn, _lay(dattn), B=-1) == INVALID
    assert _decode_status(dattn, _lay(dattn, num_pages=0)) == INVALID
    # a block table too large for 32-bit TMA coordinates
    assert _decode_status(dattn, _lay(dattn, num_pages=1 << 26, page_size=64)) == UNSUPPORTED


def test_kv_format_is_validated(dattn):
    INVALID, UNSUPPORTED = 1, 2

    def lay(fmt, kv_scale):
        out = _lay(dattn)
        out.c.kv_format, out.c.kv_scale = fmt, kv_scale
        return out

    assert _decode_status(dattn, lay(4, 128)) == INVALID     # unknown format
    assert _decode_status(dattn, lay(-1, None)) == INVALID
    for fmt in (dattn.KV_FP8_E4M3, dattn.KV_INT4):
        assert _decode_status(dattn, lay(fmt, None)) == INVALID  # the scale pool missing
        assert _decode_status(dattn, lay(fmt, 72)) == INVALID    # not 16-byte aligned
        # well-formed layouts pass the layout checks: the group-size check answers next
        assert _decode_status(dattn, lay(fmt, 128), Hq=36) == UNSUPPORTED
    assert _decode_status(dattn, lay(0, None), Hq=36) == UNSUPPORTED
    import torch
    for fmt in (dattn.KV_FP8_E4M3, dattn.KV_INT4):
        with pytest.raises(ValueError):
            dattn.KVLayout(8, 2, 128, 16, torch.zeros(1, 4, dtype=torch.int32), kv_format=fmt)


def test_mixed_format_is_validated(dattn):
    """A mixed layout needs one FP8 or 4-bit entry per KV head in its host head_format."""
    INVALID, UNSUPPORTED = 1, 2
    import torch

    def lay(formats):
        out = _lay(dattn)
        out.c.kv_format, out.c.kv_scale = dattn.KV_MIXED, 128
        arr = None
        if formats is not None:
            arr = (ctypes.c_int8 * len(formats))(*formats)
            out.c.head_format = ctypes.addressof(arr)
        return out, arr

    for formats, want in [(None, INVALID),                                      # no table
                          ([dattn.KV_FP8_E4M3, dattn.KV_BF16], INVALID),        # bf16 head
                          ([dattn.KV_INT4, 7], INVALID),                        # unknown
                          ([dattn.KV_FP8_E4M3, dattn.KV_INT4], UNSUPPORTED),    # well formed:
                          ([dattn.KV_INT4, dattn.KV_INT4], UNSUPPORTED)]:       # the group size
        layout, keep = lay(formats)                                             # answers next
        assert _decode_status(dattn, layout, Hq=36) == want, formats
    bt = torch.zeros(1, 4, dtype=torch.int32)
    sc = torch.zeros(8 * 2 * 16 * 2, dtype=torch.float32)
    with pytest.raises(ValueError):
        dattn.KVLayout(8, 2, 128, 16, bt, kv_format=dattn.KV_MIXED, kv_scale=sc)
    with pytest.raises(ValueError):
        dattn.KVLayout(8, 2, 128, 16, bt, kv_format=dattn.KV_MIXED, kv_scale=sc,
                       head_format=[dattn.KV_INT4])
    ok = dattn.KVLayout(8, 2, 128, 16, bt, kv_format=dattn.KV_MIXED, kv_scale=sc,
                        head_format=[dattn.KV_INT4, dattn.KV_FP8_E4M3])
    # 8 pages x 16 tokens: one 8-bit head of 128 bytes per row, one 4-bit head of 64
    assert dattn.mixed_pool_bytes(8, ok.head_format, 128, 16) == 8 * 16 * (128 + 64)


def test_decode_multi_is_validated(dattn):
    INVALID, UNSUPPORTED = 1, 2
    lib = dattn.load_library()
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first

    def status(T, Hq, lay=None):
        lay = lay or _lay(dattn)  # Hkv = 2
        return lib.dattn_decode_multi(ctypes.byref(lay.c), p, p, p, 1, T, Hq, 0.1, p, 0, p,
                                      1 << 20, p, None, None, None, None)

    assert status(0, 4) == INVALID             # no query token
    assert status(-2, 4) == INVALID
    assert status(3, 8) == UNSUPPORTED         # group 4 x 3 tokens > 8 columns
    assert status(9, 2) == UNSUPPORTED         # group 1 x 9 tokens
    assert status(2, 3) == INVALID             # Hq % Hkv != 0
    assert status(2, 4, _lay(dattn, head_dim=96)) == UNSUPPORTED


def test_page_select_needs_power_of_two_logical_pages(dattn):
    lib = dattn.load_library()
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    lay = _lay(dattn, page_size=48)  # three logical pages per physical page
    assert lib.dattn_page_select(ctypes.byref(lay.c), p, p, 1, 4, p, p, 8, p, None, p, 1 << 20,
                                 0, None, None) == 2  # DATTN_ERR_UNSUPPORTED
    lay = _lay(dattn, page_size=64)
    assert lib.dattn_page_select(ctypes.byref(lay.c), p, p, 1, 4, p, p, 300, p, None, p,
                                 1 << 20, 0, None, None) == 2  # top_k above 256


def test_sparse_settings_are_validated(dattn):
    import torch
    hk = torch.zeros(2, dtype=torch.int8)
    lay = _lay(dattn)
    bad = dattn.SparseConfig(hk, -1, 8, 4, torch.zeros(1, 2, 4, dtype=torch.int32))
    assert _decode_status(dattn, lay, sparse=ctypes.byref(bad.c)) == 1
    big = dattn.SparseConfig(hk, 4, 8, 1000, torch.zeros(1, 2, 4, dtype=torch.int32))
    assert _decode_status(dattn, lay, sparse=ctypes.byref(big.c)) == 2
    nosel = dattn.SparseConfig(hk, 4, 8, 4, None)
    assert _decode_status(dattn, lay, sparse=ctypes.byref(nosel.c)) == 1


def test_other_entry_points_validate(dattn):
    lib = dattn.load_library()
    p = ctypes.c_void_p(16)
    lay = _lay(dattn)
    # append: negative sizes, misaligned pointers
    assert lib.dattn_kv_append(ctypes.byref(lay.c), p, p, None, p, p, -1, 1, p, None, None) == 1
    assert lib.dattn_kv_append(ctypes.byref(lay.c), ctypes.c_void_p(18), p, None, p, p, 1, 1, p,
                               None, None) == 1
    assert lib.dattn_kv_append(ctypes.byref(lay.c), p, p, None, p, p, 0, 5, p, None, None) == 0
    # merge: unsupported head_dim, null indptr
    assert lib.dattn_merge(1, 1, 4, 256, p, p, p, p, p, None, None, None, None, None) == 2
    assert lib.dattn_merge(1, 1, 4, 64, None, p, p, p, p, None, None, None, None, None) == 1
    assert lib.dattn_merge(0, 0, 4, 64, None, None, None, None, None, None, None, None, None,
                           None) == 0
    # partial: C too large, nulls
    assert lib.dattn_partial(ctypes.byref(lay.c), p, p, p, 1, 4, 0.1, p, 5000, p, p, p, p, p, p,
                             p, 1 << 20, 0, None, None) == 2
    assert lib.dattn_partial(ctypes.byref(lay.c), p, p, p, 1, 4, 0.1, p, 2, None, p, p, p, p, p,
                             p, 1 << 20, 0, None, None) == 1
    # page select: top_k too large
    assert lib.dattn_page_select(ctypes.byref(lay.c), p, p, 1, 4, p, p, 300, p, None, p,
                                 1 << 20, 0, None, None) == 2
    # fused append and decode: null or misaligned new rows are invalid, for every pool format
    lay8 = _lay(dattn)
    lay8.c.kv_format = dattn.KV_FP8_E4M3
    lay8.c.kv_scale = p
    assert lib.dattn_append_decode(ctypes.byref(lay8.c), p, p, None, None, p, p, 1, 4, 0.1, p,
                                   None, 0, p, 1 << 20, p, None, None, None, None) == 1
    assert lib.dattn_append_decode(ctypes.byref(lay.c), p, p, None, None, p, p, 1, 4, 0.1, p,
                                   None, 0, p, 1 << 20, p, None, None, None, None) == 1
    assert lib.dattn_append_decode(ctypes.byref(lay.c), p, p, None, p, ctypes.c_void_p(18), p, 1,
                                   4, 0.1, p, None, 0, p, 1 << 20, p, None, None, None, None) == 1


def test_workspace_size(dattn):
    assert dattn.dattn_workspace_size(8, 32, 32, 128, 0, 304) > 0
    assert dattn.dattn_workspace_size(8, 32, 32, 96, 0, 0) == 0
    assert dattn.dattn_workspace_size(8, 30, 8, 128, 0, 0) == 0
    a = dattn.dattn_workspace_size(8, 32, 8, 128, 0, 100)
    b = dattn.dattn_workspace_size(8, 32, 8, 128, 64, 100)
    assert b >= a
    # counters (8*8 per segment plus the fused append's one: 65 ints, padded to 256 B) +
    # (G + segments) slots of g*d + 2g floats, rounded up to a multiple of 4 floats
    assert a == 512 + (100 + 64) * (4 * 128 + 8) * 4
    c = dattn.dattn_workspace_size(8, 24, 8, 128, 0, 100)  # g = 3: 6 -> 8 trailing floats
    assert c == 512 + (100 + 64) * (3 * 128 + 8) * 4


def test_binding_rejects_short_tensors_before_any_call(dattn):
    """The C entry points see only pointers, so the binding checks every tensor holds the
    elements the call touches (these tensors live on the CPU: the check comes first)."""
    import torch
    lay = _lay(dattn)  # 8 pages x 2 KV heads x 16 tokens x d 128, block table [1][4]
    pool = torch.zeros(8 * 2 * 16 * 128, dtype=torch.bfloat16)
    short = torch.zeros(10, dtype=torch.bfloat16)
    q = torch.zeros(1, 4, 128, dtype=torch.bfloat16)
    seq = torch.zeros(1, dtype=torch.int32)
    out = torch.zeros(1, 4, 128)
    ws = type("W", (), {"buffer": torch.zeros(256, dtype=torch.uint8)})()
    with pytest.raises(ValueError, match="k_pool"):
        dattn.dattn_decode(lay, short, pool, q, 0.1, seq, out, ws)
    with pytest.raises(ValueError, match="out"):
        dattn.dattn_decode(lay, pool, pool, q, 0.1, seq, torch.zeros(3), ws)
    q_half = torch.zeros(1, 5, 4, 64, dtype=torch.bfloat16)  # d = 64 rows for a d = 128 layout
    with pytest.raises(ValueError, match="q"):
        dattn.dattn_prefill(lay, pool, pool, q_half, 0.1, seq, torch.zeros(1, 5, 4, 128))
    k_half = torch.zeros(1, 2, 2, 64, dtype=torch.bfloat16)
    v_full = torch.zeros(1, 2, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="k_new"):
        dattn.dattn_kv_append(lay, pool, pool, None, k_half, v_full, seq)
    with pytest.raises(ValueError, match="block_table"):
        dattn.dattn_decode(lay, pool, pool, torch.zeros(2, 4, 128, dtype=torch.bfloat16), 0.1,
                           torch.zeros(2, dtype=torch.int32), torch.zeros(2, 4, 128), ws)
