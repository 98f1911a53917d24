"""The benchmark's algorithmic bytes and flops, checked on the CPU.

The byte counts are pinned to the workload definitions: K+V of every valid token (in the
pool's format), the queries, the outputs with their (m, e), the block-table entries and the
lengths, and for the block-sparse step the selected pages, the streaming window and the
statistics scan of each selection. The prefill's attended pairs are counted against the
oracle's own row sets.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from split_kv_decode_distattention_gb300 import workloads as W  # noqa: E402


def test_row_bytes_of_each_pool_format():
    # bf16 values; E4M3 codes plus an fp32 scale; two 4-bit codes per byte plus the scale
    assert bench.row_bytes(128, "bf16") == 256
    assert bench.row_bytes(128, "fp8") == 132
    assert bench.row_bytes(128, "int4") == 68
    assert bench.row_bytes(64, "int4") == 36


def _side_bytes(B, Hq, d, T=1):
    q = T * B * Hq * d * 2
    out = T * (B * Hq * d * 4 + 2 * B * Hq * 4)
    return q, out


def test_mha_32k_decode_bytes():
    case = W.mha_32k(seed=0)
    lens = [32768] * 8
    sb = bench.step_bytes(case, lens, False)
    q, out = _side_bytes(8, 32, 128)
    kv = 4_294_967_296  # 8 requests x 32 heads x 32768 tokens x (K + V) x 256 bytes
    bt = 8 * (32768 // 16) * 4
    assert sb["decode"] == kv + q + out + bt + 8 * 4
    assert sb["append"] == 8 * 32 * (128 * 2 + 256) * 2
    fp8 = bench.step_bytes(case, lens, False, "fp8")
    int4 = bench.step_bytes(case, lens, False, "int4")
    assert fp8["decode"] - sb["decode"] == 8 * 32 * 32768 * 2 * (132 - 256)
    assert int4["decode"] - sb["decode"] == 8 * 32 * 32768 * 2 * (68 - 256)


def test_multi_query_counts_queries_and_outputs_per_token():
    case = W.mha_32k(seed=0)
    lens = [32768] * 8
    one = bench.step_bytes(case, lens, False, T=1)
    eight = bench.step_bytes(case, lens, False, T=8)
    q1, out1 = _side_bytes(8, 32, 128, 1)
    q8, out8 = _side_bytes(8, 32, 128, 8)
    assert eight["decode"] - one["decode"] == (q8 - q1) + (out8 - out1)  # K/V read once


def test_sparse_512k_step_and_selection_bytes():
    case = W.sparse_512k(seed=0)
    lens = [524288] * 8
    plain = bench.step_bytes(case, lens, False)
    sel = bench.step_bytes(case, lens, True)
    q, out = _side_bytes(8, 32, 128)
    sel_rows = 8 * 4 * 64 * 4
    retrieval = 67_108_864  # 8 x 4 heads x 64 pages x 64 tokens x (K + V) x 256 bytes
    streaming = 196_608     # 8 x 4 heads x (4 sinks + 8 local) x (K + V) x 256 bytes
    # the selection rows are read with their pool pages (dattn_sparse.selected_phys)
    assert plain["decode"] == retrieval + streaming + q + out + 2 * sel_rows + 8 * 4
    stats = 536_870_912     # 8 x 4 heads x 32768 logical pages x 512 bytes
    bt = 8 * (524288 // 64) * 4
    assert sel["select"] == stats + q + 2 * sel_rows + bt
    assert plain["select"] == 0


def test_prefill_pairs_equal_the_oracle_row_sets():
    case = W.Case("pairs", B=2, Hq=4, Hkv=4, d=64, P=16, lens=[700, 333], seed=3)
    Tq, sinks, local = 300, 1, 2
    kinds = [0, 1, 2, 1]
    lists = case.prefill_block_lists(0.65, stride=12)
    want = 0
    for b, L in enumerate(case.lens):
        for t in range(Tq):
            qb = (L - Tq + t) // 64
            for kvh in range(case.Hkv):
                blocks = lists[b, kvh, qb] if kinds[kvh] == 1 else None
                rows = oracle.prefill_rows(kinds[kvh], L, Tq, t, sinks, local, blocks=blocks)
                want += case.g * rows.size
    assert bench.prefill_pairs(case, Tq, kinds, lists, sinks, local) == want
    dense = bench.prefill_pairs(case, Tq, [0] * 4, lists, sinks, local)
    assert dense == case.Hq * sum(sum(L - Tq + t + 1 for t in range(Tq)) for L in case.lens)
    assert np.all(lists[:, :, :, 0] >= 0)  # every row lists at least its own block


def test_prefill_32k_least_bytes():
    case = W.prefill_32k(seed=0)
    q = 32768 * 32 * 128 * 2      # bf16 queries of the chunk
    kv = 32768 * 8 * 128 * 2 * 2  # K and V of every token, bf16, read once
    out = 32768 * 32 * 128 * 4    # fp32 outputs
    assert bench.prefill_bytes(case, 32768) == q + kv + out + 2048 * 4 == 939_532_288


def test_traffic_records_apply_to_full_size_runs_of_their_own_kernel():
    class A:
        config, kv_format, queries, batch, ctx, prefill_dense = "mha-32k", "bf16", 1, 0, 0, False
    a = A()
    assert bench.traffic_key(a) == "mha-32k"
    a.kv_format, a.queries = "int4", 8
    assert bench.traffic_key(a) == "mha-32k/int4/T8"
    a.ctx = 4096  # a reduced run: no full-size record describes it
    assert bench.traffic_key(a) is None and bench.traffic_record(None) is None
    a.config, a.ctx, a.prefill_dense = "prefill-32k", 0, True
    assert bench.traffic_key(a) == "prefill-32k/dense"
    # a record is taken on one kernel's sources: the prefill's hash never matches a decode one
    assert bench.kernel_source_hash(bench.PREFILL_SOURCES) != bench.kernel_source_hash()
    assert bench.traffic_record("mha-32k", bench.PREFILL_SOURCES) is None


def test_traffic_records_scale_to_the_run_by_their_ratio():
    """A record's DRAM/algorithmic ratio (taken on a reduced case) scales to a run's launch
    by that run's algorithmic bytes."""
    import json
    recs = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for key, rec in recs.items():
        if key.startswith("_"):
            continue
        assert 0.8 < rec["ratio_to_algorithmic"] < 1.1, key
        want = round(rec["captured_dram_bytes_per_launch"] /
                     rec["captured_algorithmic_bytes_per_launch"], 4)
        assert rec["ratio_to_algorithmic"] == want, key
    rec = recs["mha-32k"]
    if rec["source_hash"] == bench.kernel_source_hash():  # else the record is stale: null
        assert bench.traffic_record("mha-32k", alg_bytes=10**9) == round(
            rec["ratio_to_algorithmic"] * 10**9)


def test_prefill_cpu_sample_is_bounded_and_covers_rows_once():
    oracle.build_oracle()
    case = W.prefill_32k(seed=0, L=640)
    kinds = list(case.head_kind)
    lists = case.prefill_block_lists(W.PREFILL_KEEP)
    args = (case, "cpu", kinds, lists, W.PREFILL_SINK_BLOCKS, W.PREFILL_LOCAL_BLOCKS, 640)
    heads = sorted({kinds.index(k) for k in set(kinds)})
    want = sum(oracle.prefill_rows(kinds[h], 640, 640, t, W.PREFILL_SINK_BLOCKS,
                                   W.PREFILL_LOCAL_BLOCKS,
                                   blocks=lists[0, h, t // 64] if kinds[h] == 1 else None).size
               for h in heads for t in range(640))
    full = bench.prefill_cpu_baseline(*args, target_s=1e9)
    assert full["sample"].startswith(f"{640 * len(heads)} query rows")
    assert f" {want} query-key pairs" in full["sample"]
    one = bench.prefill_cpu_baseline(*args, target_s=0.0)  # stops after its first batch
    nrows = int(one["sample"].split()[0])
    assert 0 < nrows <= 16 * os.cpu_count() * len(heads) and nrows % len(heads) == 0
