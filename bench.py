"""Benchmark of the split-KV decode path on GB300.

One step is one decode layer-step of the whole batch through the library's C ABI:
  dense workloads:  dattn_kv_append (one new token per request), then dattn_decode
                    (split-KV MicroAttention partials plus the in-launch merge), the second
                    launch overlapping the first's tail (programmatic dependent launch);
                    --fused times dattn_append_decode instead (the two in one launch),
                    which measures slower on GB300; --queries T: dattn_decode_multi;
  sparse-512k:      the same, plus dattn_page_select at the start of every reuse window.
The metric is achieved HBM bandwidth in GB/s: the algorithmic bytes of the step (valid K/V
read, statistics scanned, new tokens written, queries, outputs, block table) divided by
the device time of the step. The time per layer-step and the fraction of the 8 TB/s
roofline are reported beside it. L2 is flushed before every timed step whose K/V is under
four times the L2; larger steps evict it themselves and run back to back.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl dattn|reference]
                  [--kv-format bf16|fp8|int4|mixed] [--queries T]

--kv-format fp8 runs the same workload over the 8-bit pool (FP8 E4M3 codes with one fp32
scale per (token, KV head) row): a K or V row then moves d + 4 bytes instead of 2 d.
--kv-format int4 runs it over the 4-bit pool (symmetric 4-bit codes, two per byte, with the
same scales): d / 2 + 4 bytes per row.
--kv-format mixed (block-sparse workloads) keeps every KV head in the format of its kind in
one pool: streaming heads 4-bit, retrieval and dense heads 8-bit, decoded in one launch.

--queries T (dense workloads) makes each step a chunked one: T new tokens per request are
appended, then dattn_decode_multi attends all T query tokens, causal over the new tokens.
The K/V is read once per step, as for T = 1; queries, outputs and appends scale with T.

The default run (mha-1m, bf16) also times sparse-512k afterwards and reports it under
"also" in the same line (--also none skips it, --also NAME picks another workload).

--impl reference times the CPU oracle (test infrastructure) on the host cores over a
bounded sample of the same workload and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "split-KV decode attention: achieved HBM GB/s vs 8 TB/s; μs per layer-step"
ROOFLINE_8TBS = 8000.0  # GB/s, the roofline the metric is quoted against
FALLBACK_HBM_GBS = 6800.0

WORKLOAD_TEXT = {
    "dense-tiny": "dense GQA decode, batch 1, 8 q / 2 KV heads, head_dim 64, 4096 tokens, "
                  "16-token pages, identity block table",
    "mha-32k": "Llama-2-7B-shaped MHA decode, one layer: batch 8, 32 heads, head_dim 128, "
               "32K tokens per sequence, bf16 paged KV (16-token pages, shuffled pool)",
    "mha-1m": "single 1M-token request, 32 heads MHA, head_dim 128, 16-token pages, "
              "64 needle keys",
    "gqa-ragged": "ragged Llama-3-8B GQA batch: 64 requests, 32 q / 8 KV heads, head_dim 128, "
                  "lengths log-uniform 1K-256K, 16-token pages",
    "sparse-512k": "LServe-style block-sparse decode: batch 8, 32 q / 8 KV heads, head_dim "
                   "128, 512K context, 64-token pages of four 16-token logical pages, "
                   "4 retrieval + 4 streaming KV heads, top-64 pages reused 16 steps, "
                   "4 sinks + 8 local",
    "prefill-32k": "LServe-style block-sparse prefill, Llama-3-8B GQA (32 q / 8 KV heads, head_dim "
                   "128): one 32K-token request prefilled as one chunk, 64-token key blocks; 4 "
                   "retrieval KV heads keep a seeded 65% of the earlier blocks plus their own, 4 "
                   "streaming KV heads keep 1 sink block and 16 local blocks",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="mha-1m", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="dattn", choices=["dattn", "reference"])
    ap.add_argument("--kv-format", default="bf16", choices=["bf16", "fp8", "int4", "mixed"],
                    help="element format of the paged KV pool")
    ap.add_argument("--prefill-dense", action="store_true",
                    help="prefill-32k: every head dense (causal) instead of the LServe mix")
    ap.add_argument("--queries", type=int, default=1,
                    help="query tokens per request and step (dense workloads; 1 = decode)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override the batch (profiling only)")
    ap.add_argument("--ctx", type=int, default=0, help="override the context (profiling only)")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--fused", action="store_true",
                    help="step = dattn_append_decode (the append and the decode in one launch) "
                         "instead of dattn_kv_append then dattn_decode")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--also", default="auto",
                    help="a second workload timed after the first and summarised in the same "
                         "line under 'also' (auto: sparse-512k after the default mha-1m bf16 "
                         "run; none: no second workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="replay one CUDA graph per timed step instead of eager library calls")
    ap.add_argument("--no-info", action="store_true",
                    help="skip the informational warm-L2 / CUDA-graph / append timings")
    ap.add_argument("--flush", action="store_true", help="flush L2 before every step")
    ap.add_argument("--profile", action="store_true",
                    help="short run for ncu: no e2e, no CPU baseline, no clock sampling")
    return ap.parse_args()


def info_steps(args) -> int:
    """Steps of each informational pass after the timed region (warm L2, CUDA graphs)."""
    return 0 if (args.profile or args.no_info) else min(64, args.steps)


def fused_step(args) -> bool:
    """A step is dattn_kv_append then dattn_decode (two launches), unless --fused asks for
    one dattn_append_decode launch (one query token per request, any pool format). On GB300
    the two launches measure faster: the append kernel's tail overlaps the decode's prologue,
    while the fused launch's heavier kernel (its append work and the new tokens' patches)
    costs more than the launch it saves."""
    return args.fused and args.queries == 1


def make_case(args):
    from split_kv_decode_distattention_gb300 import workloads as W
    name = args.config
    kw = {}
    if name in ("mha-32k", "sparse-512k"):
        if args.batch:
            kw["B"] = args.batch
        if args.ctx:
            kw["L"] = args.ctx
    elif name == "mha-1m" and args.ctx:
        kw["L"] = args.ctx
    elif name == "gqa-ragged" and args.batch:
        kw["B"] = args.batch
    elif name == "prefill-32k" and args.ctx:
        kw["L"] = args.ctx
    case = W.CASES[name](seed=args.seed, **kw)
    if args.queries < 1 or (args.queries > 1 and case.head_kind is not None):
        raise SystemExit("--queries T needs T >= 1 and a dense workload")
    # room for the tokens the timed and warm-up steps append
    case.reserve_tokens = max(case.reserve_tokens, 2 * args.queries *
                              (args.steps + args.warmup + 3 * info_steps(args)) + 64)
    case._make_block_table()
    return case


KV_FORMAT_NOTE = {
    "bf16": "bf16",
    "fp8": "fp8_e4m3 codes + one fp32 scale per (token, KV head) row",
    "int4": "symmetric 4-bit codes (two per byte) + one fp32 scale per (token, KV head) row",
    "mixed": "per KV head kind: fp8_e4m3 codes (retrieval, dense) or symmetric 4-bit codes "
             "(streaming), one fp32 scale per (token, KV head) row, one pool",
}
QUANT_NOTE = {"fp8": " over the dequantized 8-bit rows", "int4": " over the dequantized 4-bit rows",
              "mixed": " over the dequantized rows (8-bit retrieval, 4-bit streaming heads)"}


def row_bytes(d: int, fmt: str) -> int:
    """Bytes of one K (or V) row of one token and KV head in the pool (format bf16, fp8 or
    int4; the quantized formats count their fp32 row scale)."""
    return {"bf16": 2 * d, "fp8": d + 4, "int4": d // 2 + 4}[fmt]


def head_format(fmt: str, kind: int) -> str:
    """The format of a KV head of kind `kind` in a pool of format fmt: the mixed pool keeps
    streaming heads at 4 bits and the other heads at 8 bits."""
    if fmt != "mixed":
        return fmt
    return "int4" if kind == 2 else "fp8"


def step_bytes(case, lens_after, sparse_sel_step: bool, fmt: str = "bf16", T: int = 1) -> dict:
    """Algorithmic bytes of one layer-step, given the lengths after the append (T query
    tokens per request: T appended tokens, T queries and outputs, the K/V read once)."""
    B, Hq, Hkv, d, P = case.B, case.Hq, case.Hkv, case.d, case.P
    q_bytes = T * B * Hq * d * 2
    out_bytes = T * (B * Hq * d * 4 + 2 * B * Hq * 4)
    bt = sum(-(-L // P) for L in lens_after) * 4
    if case.head_kind is None:
        if fmt == "mixed":
            raise ValueError("the mixed pool takes its formats from the head kinds")
        rb = row_bytes(d, fmt)
        new_kv = T * B * Hkv * (d * 2 + rb) * 2  # read k_new/v_new (bf16), write the pool
        kv = sum(lens_after) * Hkv * rb * 2
        decode = kv + q_bytes + out_bytes + bt + B * 4
        return {"decode": decode, "append": new_kv, "select": 0,
                "step": decode + new_kv}
    kinds = case.head_kind
    nret = sum(1 for k in kinds if k == 1)
    nstr = sum(1 for k in kinds if k == 2)
    nden = sum(1 for k in kinds if k == 0)
    rb_of = [row_bytes(d, head_format(fmt, k)) for k in (0, 1, 2)]  # by head kind
    # read k_new/v_new (bf16), write into the pool in each head's format
    new_kv = T * B * sum(d * 2 + rb_of[k] for k in kinds) * 2
    kv = 0
    for L in lens_after:
        kv += nden * L * rb_of[0] * 2
        kv += nret * min(case.top_k * P, L) * rb_of[1] * 2
        s_end = min(case.sinks, L)
        l0 = max(case.sinks, L - case.local)
        kv += nstr * (s_end + max(0, L - l0)) * rb_of[2] * 2
    sel_rows = B * nret * case.top_k * 4
    # the decode reads the selection rows and their pool pages (dattn_sparse.selected_phys)
    decode = kv + q_bytes + out_bytes + 2 * sel_rows + B * 4
    stats = sum(L // 16 + (1 if L % 16 else 0) for L in lens_after) * nret * 2 * d * 2
    select = (stats + q_bytes + 2 * sel_rows + bt) if sparse_sel_step else 0
    # the stats update inside the append (read + write one logical page per request/head)
    new_kv += B * Hkv * 2 * d * 2 * 2
    return {"decode": decode, "append": new_kv, "select": select,
            "step": decode + new_kv + select}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources that build the decode (prefill) kernel and choose its launch configuration
DECODE_SOURCES = ("abi.cu", "attention.cu", "common.cuh", "internal.h")
PREFILL_SOURCES = ("abi.cu", "prefill.cu", "common.cuh", "internal.h")


def kernel_source_hash(sources=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "split_kv_decode_distattention_gb300", "csrc")
    for f in sources:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_key(args):
    """Key of the full-size workload's record in profiles/traffic.json; None for a run
    reduced by --batch or --ctx, which no full-size record describes."""
    if args.batch or args.ctx:
        return None
    if args.config == "prefill-32k":
        return args.config + ("/dense" if args.prefill_dense else "")
    return (args.config + (f"/{args.kv_format}" if args.kv_format != "bf16" else "") +
            (f"/T{args.queries}" if args.queries > 1 else ""))


def traffic_record(config, sources=DECODE_SOURCES, alg_bytes=None):
    """DRAM bytes per launch of the workload's dominant kernel from the committed ncu
    summary, if it was taken on the current sources of that kernel. The records were
    captured on reduced cases; their ratio of DRAM to algorithmic bytes scales to this run's
    launch by its algorithmic bytes (alg_bytes), both growing with the attended tokens."""
    if config is None:
        return None
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(p)).get(config)
    except Exception:
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(sources):
        return None
    if alg_bytes is not None and "ratio_to_algorithmic" in rec:
        return int(round(rec["ratio_to_algorithmic"] * alg_bytes))
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------ GPU arm

def reduce_over_ranks(ms_total: float, units: float, world: int, device) -> tuple:
    """Whole-job figures of a run on `world` ranks, each timing its own replica of the
    workload (weak scaling): the slowest rank's time and the units (bytes or flops) of all
    ranks. Collective over the default process group when world > 1."""
    if world <= 1:
        return ms_total, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_total, float(units)], dtype=torch.float64, device=device)
    tmax = t.clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(tmax[0]), float(t[1])


KERNEL_EVERY = 8  # at most this many steps between the ones whose decode kernel is timed


def kernel_every(steps: int) -> int:
    """Steps between the ones whose decode kernel is timed on its own: every 8th, but often
    enough that at least 10 launches are timed whenever there are 10 steps or more."""
    return max(1, min(KERNEL_EVERY, steps // 10))


L2_FALLBACK_BYTES = 129 * 10 ** 6  # GB300's L2, when no device can be asked


def device_l2_bytes() -> int:
    try:
        import torch
        if torch.cuda.is_available():
            return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        pass
    return L2_FALLBACK_BYTES


def l2_policy(case, args) -> tuple:
    """(flush?, text) for the timed steps: a step whose K/V is more than 4x the L2 evicts what
    the previous step left there and runs back to back; smaller steps are preceded by an L2
    flush (L2Flush). Both arms state the same text in their config."""
    sparse = case.head_kind is not None
    sb0 = step_bytes(case, list(case.lens), sparse, args.kv_format, args.queries)
    l2 = device_l2_bytes()
    flush = sb0["decode"] < 4 * l2 or args.flush
    text = (f"flushed before every timed step ({L2Flush.TEXT})" if flush else
            f"inputs larger than L2: {sb0['decode'] / 1e9:.2f} GB of K/V per step vs "
            f"{l2 / 1e6:.0f} MB L2, timed back to back without a flush")
    return flush, text


def measure_read_peak(dev, gib: int = 4, reps: int = 10) -> float:
    """A read-only HBM stream for context beside the copy peak: torch.sum over `gib` GiB of
    fp32, best of `reps`, timed with CUDA events (GB/s of bytes read)."""
    import torch
    x = torch.ones(gib * (1 << 30) // 4, dtype=torch.float32, device=dev)
    acc = torch.empty((), dtype=torch.float32, device=dev)
    torch.sum(x, dim=0, out=acc)
    best = float("inf")
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        torch.sum(x, dim=0, out=acc)
        b.record()
        b.synchronize()
        best = min(best, a.elapsed_time(b))
    del x
    torch.cuda.empty_cache()
    return gib * (1 << 30) / (best * 1e-3) / 1e9


READ_PEAK_HOW = "torch.sum over 4 GiB of fp32, best of 10, CUDA events (bytes read)"


class L2Flush:
    """Evicts every line of L2 without leaving dirty ones behind: a 512 MiB write pushes
    everything out, then a 512 MiB read replaces the written (dirty) lines with clean ones.
    Their write-back therefore lands before the timed region instead of inside it."""
    TEXT = "512 MiB write, then 512 MiB read, so L2 holds only clean unrelated lines"

    def __init__(self, dev):
        import torch
        n = 512 * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.acc)


def run_dattn(args, rank: int, world: int):
    import torch
    import torch.distributed as dist

    import split_kv_decode_distattention_gb300 as dattn
    from split_kv_decode_distattention_gb300.harness import PagedCache

    dattn.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    case = make_case(args)
    sparse = case.head_kind is not None
    fmt = args.kv_format
    if fmt == "mixed" and not sparse:
        raise SystemExit("--kv-format mixed needs a block-sparse workload (its head kinds)")
    hfmt = None
    if fmt == "mixed":
        hfmt = [dattn.KV_INT4 if head_format(fmt, k) == "int4" else dattn.KV_FP8_E4M3
                for k in case.head_kind]
    cache = PagedCache(case, dev, with_stats=sparse, chunk_tokens=16384,
                       kv_format={"bf16": dattn.KV_BF16, "fp8": dattn.KV_FP8_E4M3,
                                  "int4": dattn.KV_INT4, "mixed": dattn.KV_MIXED}[fmt],
                       head_format=hfmt)
    B, Hq, d = case.B, case.Hq, case.d
    T = args.queries
    ws = cache.workspace(top_k=case.top_k, num_splits=args.num_splits, queries=T)
    qshape = (B, Hq) if T == 1 else (B, T, Hq)  # one query token, or T of them
    out = torch.empty(*qshape, d, dtype=torch.float32, device=dev)
    m_g = torch.empty(*qshape, dtype=torch.float32, device=dev)
    e_g = torch.empty(*qshape, dtype=torch.float32, device=dev)
    sel = torch.full((B, case.Hkv, max(case.top_k, 1)), -1, dtype=torch.int32, device=dev)
    sel_phys = torch.full_like(sel, -1)
    spc = cache.sparse_config(sel, sel_phys) if sparse else None
    fused = fused_step(args)
    stream = torch.cuda.current_stream()
    n_info = info_steps(args)
    total = args.warmup + args.steps + 3 * n_info + 1
    # per-step inputs prepared up front (device-resident for the kernel timing)
    if T == 1:
        qs = [case.q(s, dev) for s in range(total)]
    else:
        qs = [torch.stack([case.q(s * T + t, dev) for t in range(T)], dim=1).contiguous()
              for s in range(total)]
    per_req = [case.kv(b, case.lens[b], case.lens[b] + total * T, dev) for b in range(B)]
    k_all = torch.stack([k for k, _ in per_req])  # [B][total * T][Hkv][d]
    v_all = torch.stack([v for _, v in per_req])
    del per_req
    news = [(k_all[:, s * T:(s + 1) * T].contiguous(), v_all[:, s * T:(s + 1) * T].contiguous())
            for s in range(total)]
    del k_all, v_all
    # L2 hygiene (l2_policy): steps whose K/V is over 4x the L2 run back to back, smaller
    # ones after an L2 flush
    do_flush, l2_text = l2_policy(case, args)
    every = kernel_every(args.steps)
    flush = L2Flush(dev)
    torch.cuda.synchronize()

    def pre_step(s):  # the append (unless fused), and at a reuse window's start the selection
        n = 0
        if not fused:
            kn, vn = news[s]
            cache.append(kn, vn)
            n += 1
        if sparse and s % case.reuse == 0:
            cache.select(qs[s], sel, ws, num_splits=args.num_splits, selected_phys=sel_phys)
            n += 1
        return n

    def dec_step(s):
        if fused:
            kn, vn = news[s]
            cache.append_decode(kn, vn, qs[s], out, ws, m_g=m_g, e_g=e_g, sparse=spc,
                                num_splits=args.num_splits)
        else:
            cache.decode(qs[s], out, ws, m_g=m_g, e_g=e_g, sparse=spc,
                         num_splits=args.num_splits)
        return 1

    def one_step(s, ev=None):
        launches = pre_step(s)
        if ev is not None:
            ev[0].record(stream)
        launches += dec_step(s)
        if ev is not None:
            ev[1].record(stream)
        return launches

    for s in range(args.warmup):
        one_step(s)
    torch.cuda.synchronize()
    lens0 = list(cache.lens)
    # With --graph each timed step is replayed from a CUDA graph captured beforehand (one per
    # step, as the steps' inputs differ). A step whose decode kernel is timed on its own is
    # captured as two graphs with the events between them.
    graphs = {}
    if args.graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)

        def capture(fn, s):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
                n = fn(s)
            return g, n
        for i in range(args.steps):
            s = args.warmup + i
            if i % every == 0:
                graphs[s] = (capture(pre_step, s), capture(dec_step, s))
            else:
                graphs[s] = (capture(one_step, s),)
        stream.wait_stream(side)
        torch.cuda.synchronize()
    clocks = ClockSampler(dev.index) if (rank == 0 and not args.no_clocks and
                                         not args.profile) else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    step_ms, dec_ms, launches = [], [], 0
    bytes_total, dec_bytes_total = 0, 0
    for i in range(args.steps):
        s = args.warmup + i
        if do_flush:
            flush()  # outside the timed region
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        # Every `every`-th step also brackets the decode kernel with events. An event
        # between two launches keeps the second from starting early (programmatic dependent
        # launch), so the other steps run without it.
        kev = None
        if i % every == 0:
            kev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        e0.record(stream)
        if not args.graph:
            launches += one_step(s, kev)
        elif kev is None:
            (g, n), = graphs[s]
            g.replay()
            launches += n
        else:
            (g1, n1), (g2, n2) = graphs[s]
            g1.replay()
            kev[0].record(stream)
            g2.replay()
            kev[1].record(stream)
            launches += n1 + n2
        e1.record(stream)
        lens_after = [L + (i + 1) * T for L in lens0]
        sb = step_bytes(case, lens_after, sparse and s % case.reuse == 0, fmt, T)
        bytes_total += sb["step"]
        step_ms.append((e0, e1))
        if kev is not None:
            # the timed kernel is the decode launch (with the fused step, also the append)
            dec_bytes_total += sb["decode"] + (sb["append"] if fused else 0)
            dec_ms.append(kev)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    step_t = [a.elapsed_time(b) for a, b in step_ms]
    dec_t = [a.elapsed_time(b) for a, b in dec_ms]
    err = int(cache.dev_err.item())
    if err:
        raise RuntimeError(f"device error word {err:#x}")
    ms_max, bytes_all = reduce_over_ranks(sum(step_t), float(bytes_total), world, dev)
    res = {
        "l2_policy": l2_text, "kernel_every": every,
        "ms_total": ms_max, "bytes_all": bytes_all, "step_ms": step_t, "dec_ms": dec_t,
        "dec_bytes": dec_bytes_total / len(dec_ms), "launches": launches, "clocks": clk,
        "case": case, "lens0": lens0,
    }

    # ---- information only (outside the timed region): warm L2, CUDA graphs, the append ---
    if n_info:
        res["info"] = run_info(args, case, cache, one_step, news, qs, ws, out, m_g, e_g, spc, sel,
                               flush if do_flush else None, args.warmup + args.steps, n_info,
                               fused=fused, sel_phys=sel_phys)

    # ---- end to end through the public API with host buffers (pinned) ----------------
    if not args.no_e2e and not args.profile:
        res["e2e"] = run_e2e(args, case, cache, ws, spc, sel, flush if do_flush else None, dev,
                             fused=fused, sel_phys=sel_phys)
    if rank == 0 and not args.profile:
        res["read_peak"] = measure_read_peak(dev)
    return res


def run_info(args, case, cache, one_step, news, qs, ws, out, m_g, e_g, spc, sel, flush, s0, n,
             fused=False, sel_phys=None):
    """Informational timings after the timed region, microseconds per step as mean (the
    headline's averaging: it includes the steps that run the selection) and median:
    - eager: eager library calls, flushed like the timed steps;
    - graph: each step captured once in a CUDA graph and replayed, flushed likewise;
    - warm_l2: the captured steps replayed back to back without an L2 flush;
    - append: the kv append kernel of an eager step timed on its own (two-launch steps)."""
    import torch
    stream = torch.cuda.current_stream()
    sparse = case.head_kind is not None

    def stat(pairs):
        t = sorted(a.elapsed_time(b) * 1e3 for a, b in pairs)
        return {"mean": round(sum(t) / len(t), 2), "median": round(t[len(t) // 2], 2)}

    info = {"steps": n}
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    steps, apps = [], []
    for i in range(n):
        s = s0 + i
        if flush is not None:
            flush()
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(stream)
        kn, vn = news[s]
        if fused:
            if sparse and s % case.reuse == 0:
                cache.select(qs[s], sel, ws, num_splits=args.num_splits, selected_phys=sel_phys)
            cache.append_decode(kn, vn, qs[s], out, ws, m_g=m_g, e_g=e_g, sparse=spc,
                                num_splits=args.num_splits)
        else:
            cache.append(kn, vn)
            e1.record(stream)
            apps.append((e0, e1))
            if sparse and s % case.reuse == 0:
                cache.select(qs[s], sel, ws, num_splits=args.num_splits, selected_phys=sel_phys)
            cache.decode(qs[s], out, ws, m_g=m_g, e_g=e_g, sparse=spc,
                         num_splits=args.num_splits)
        e2.record(stream)
        steps.append((e0, e2))
    torch.cuda.synchronize()
    info["eager_us_per_step"] = stat(steps)
    if apps:
        info["append_us"] = stat(apps)
    # CUDA graphs: one graph per step (its inputs differ), replayed in order
    graphs = []
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    for i in range(2 * n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
            one_step(s0 + n + i)
        graphs.append(g)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    steps = []
    for g in graphs[:n]:
        if flush is not None:
            flush()
        e0, e1 = ev(), ev()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        steps.append((e0, e1))
    torch.cuda.synchronize()
    info["graph_us_per_step"] = stat(steps)
    events = [ev() for _ in range(n + 1)]
    events[0].record(stream)
    for i, g in enumerate(graphs[n:]):
        g.replay()
        events[i + 1].record(stream)
    torch.cuda.synchronize()
    info["warm_l2_graph_us_per_step"] = stat(list(zip(events[:-1], events[1:])))
    info["l2"] = ("eager and graph steps flushed like the timed steps; warm_l2 back to back"
                  if flush is not None else "every pass back to back (steps larger than L2)")
    return info


def run_e2e(args, case, cache, ws, spc, sel, flush, dev, fused=False, sel_phys=None):
    """The same steps through the public API with host buffers: every step copies its q and
    new K/V from pinned host memory and reads its output back into pinned host memory."""
    import torch
    B, Hq, Hkv, d = case.B, case.Hq, case.Hkv, case.d
    steps = max(3, min(args.steps, 50))
    T = args.queries
    qsh = (B, Hq, d) if T == 1 else (B, T, Hq, d)
    hq = [(case.q(100 + s, "cpu") if T == 1 else
           torch.stack([case.q(100 + s * T + t, "cpu") for t in range(T)], dim=1)).pin_memory()
          for s in range(steps)]
    hk = [torch.randn(B, T, Hkv, d).to(torch.bfloat16).pin_memory() for _ in range(steps)]
    hv = [torch.randn(B, T, Hkv, d).to(torch.bfloat16).pin_memory() for _ in range(steps)]
    houts = [torch.empty(*qsh, dtype=torch.float32).pin_memory() for _ in range(steps)]
    dq = torch.empty(*qsh, dtype=torch.bfloat16, device=dev)
    dk = torch.empty(B, T, Hkv, d, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    out = torch.empty(*qsh, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    lens0 = list(cache.lens)
    tot_ms, tot_bytes = 0.0, 0
    pairs = []
    e_all0 = torch.cuda.Event(enable_timing=True)
    e_all1 = torch.cuda.Event(enable_timing=True)
    if flush is None:
        e_all0.record(stream)
    for i in range(steps):
        if flush is not None:
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        dq.copy_(hq[i], non_blocking=True)
        dk.copy_(hk[i], non_blocking=True)
        dv.copy_(hv[i], non_blocking=True)
        if not fused:
            cache.append(dk, dv)
        if spc is not None and i % case.reuse == 0:
            cache.select(dq, sel, ws, selected_phys=sel_phys)
        if fused:
            cache.append_decode(dk, dv, dq, out, ws, sparse=spc)
        else:
            cache.decode(dq, out, ws, sparse=spc)
        houts[i].copy_(out, non_blocking=True)
        if flush is not None:
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(stream)
            pairs.append((e0, e1))
        lens_after = [L + (i + 1) * T for L in lens0]
        tot_bytes += step_bytes(case, lens_after, spc is not None and i % case.reuse == 0,
                                args.kv_format, T)["step"]
    if flush is None:
        e_all1.record(stream)
    torch.cuda.synchronize()
    tot_ms = (sum(a.elapsed_time(b) for a, b in pairs) if flush is not None
              else e_all0.elapsed_time(e_all1))
    h2d = hq[0].numel() * 2 + hk[0].numel() * 2 + hv[0].numel() * 2
    d2h = houts[0].numel() * 4
    return {"value": round(tot_bytes / (tot_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "us_per_layer_step": round(tot_ms / steps * 1e3, 2), "steps": steps}


# ------------------------------------------------------------------------------ CPU oracle

def oracle_sample(case, device, max_pairs: int, seed_step: int = 0, fmt: str = "bf16"):
    """Host copies of a bounded sample of the workload: evenly spaced (request, query head)
    pairs over their full contexts. Only the KV heads the sample reads are copied. With a
    quantized format the rows are the oracle's dequantized values (float64), made before
    any timing."""
    import oracle
    allp = [(b, h) for b in range(case.B) for h in range(case.Hq)]
    stride = max(1, len(allp) // max_pairs)
    pairs = allp[::stride][:max_pairs]
    q = oracle.bf16_bits(case.q(seed_step, device))
    need = {}
    for b, h in pairs:
        need.setdefault(b, set()).add(h // case.g)
    kv = {}
    for b, kvhs in need.items():
        L = case.lens[b]
        kvhs = sorted(kvhs)
        arrs = {h: (np.empty((L, case.d), np.uint16), np.empty((L, case.d), np.uint16))
                for h in kvhs}
        for t0 in range(0, L, 65536):
            t1 = min(L, t0 + 65536)
            K, V = case.kv(b, t0, t1, device)
            for h in kvhs:
                arrs[h][0][t0:t1] = oracle.bf16_bits(K[:, h])
                arrs[h][1][t0:t1] = oracle.bf16_bits(V[:, h])
        for h in kvhs:
            kv[(b, h)] = dequantized(arrs[h], fmt) if fmt != "bf16" else arrs[h]
    return q, pairs, kv


def dequantized(kv, fmt: str):
    """The oracle's round trip of (K, V) rows through a quantized format: float64
    code * scale."""
    import oracle
    if fmt == "int4":
        return tuple(oracle.dequantize_rows_int4(*oracle.quantize_rows_int4(x)) for x in kv)
    return tuple(oracle.dequantize_rows_fp8(*oracle.quantize_rows_fp8(x)) for x in kv)


def time_oracle(case, q, pairs, kv, nthreads, fmt: str = "bf16", qs=None):
    """Wall time of the oracle's dense attention over the sampled pairs, run on nthreads
    host threads (each call is one plain C routine that releases the GIL). With qs (T query
    arrays) each pair attends T query tokens, token t over the rows 0 .. L - T + t."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    attend = oracle.attention_f64 if fmt != "bf16" else oracle.attention

    def one(pair):
        b, h = pair
        K, V = kv[(b, h // case.g)]
        if qs is None:
            attend(q[b, h], K, V, case.scale)
        else:
            L, T = K.shape[0], len(qs)
            for t in range(T):
                attend(qs[t][b, h], K, V, case.scale,
                       rows=np.arange(max(0, L - T + t + 1), dtype=np.int64))
        return K.shape[0] * row_bytes(case.d, fmt) * 2

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        nbytes = sum(ex.map(one, pairs))
    return time.perf_counter() - t0, nbytes, min(nthreads, len(pairs))


def sparse_oracle_sample(case, device, n_ret: int = 2, n_str: int = 2):
    """Host copies for the oracle's block-sparse step: full K/V of n_ret retrieval KV heads
    and the sink and local-window tokens of n_str streaming KV heads of request 0 (bf16)."""
    import oracle
    b, L = 0, case.lens[0]
    kinds = list(case.head_kind)
    ret = [h for h in range(case.Hkv) if kinds[h] == 1][:n_ret]
    strm = [h for h in range(case.Hkv) if kinds[h] == 2][:n_str]
    q = oracle.bf16_bits(case.q(0, device))
    kv = {h: (np.empty((L, case.d), np.uint16), np.empty((L, case.d), np.uint16)) for h in ret}
    for t0 in range(0, L, 65536):
        t1 = min(L, t0 + 65536)
        K, V = case.kv(b, t0, t1, device)
        for h in ret:
            kv[h][0][t0:t1] = oracle.bf16_bits(K[:, h])
            kv[h][1][t0:t1] = oracle.bf16_bits(V[:, h])
    rows = oracle.sparse_rows(2, L, case.P, None, case.sinks, case.local)
    for h in strm:
        parts = [case.kv(b, int(r), int(r) + 1, device) for r in rows]
        K = np.stack([oracle.bf16_bits(k[0, h]) for k, _ in parts])
        V = np.stack([oracle.bf16_bits(v[0, h]) for _, v in parts])
        kv[h] = (K, V)
    return q, b, ret, strm, kv


class SparseOracleStep:
    """The oracle's block-sparse layer-step on the sampled KV heads, on host threads. A
    retrieval head selects its pages from its keys (statistics, fp32 scores, top-K) at the
    start of each reuse window and attends the selected tokens; a streaming head attends its
    sinks and local window. Bytes are counted as the GPU metric counts them."""

    def __init__(self, case, q, b, ret, strm, kv, nthreads, fmt: str = "bf16"):
        from concurrent.futures import ThreadPoolExecutor
        self.case, self.q, self.b, self.ret, self.strm, self.kv = case, q, b, ret, strm, kv
        # with a quantized format the attention runs over the dequantized rows (the
        # selection still reads the bf16 keys, as the statistics do)
        self.fmt = fmt
        self.hfmt = {h: head_format(fmt, case.head_kind[h]) for h in kv}
        self.att = ({h: dequantized(kv[h], self.hfmt[h]) for h in kv} if fmt != "bf16"
                    else kv)
        self.used = min(nthreads, len(ret) + len(strm))
        self.ex = ThreadPoolExecutor(max_workers=self.used)
        self.sels = {}

    def select(self):
        """Returns (seconds, statistics bytes scanned)."""
        import oracle
        c, b = self.case, self.b
        L, g = c.lens[b], c.g

        def one(h):
            self.sels[h] = oracle.select_pages(self.q[b, h * g:(h + 1) * g], self.kv[h][0], L,
                                               c.P, c.top_k)
        t0 = time.perf_counter()
        list(self.ex.map(one, self.ret))
        return time.perf_counter() - t0, len(self.ret) * ((L + 15) // 16) * 2 * c.d * 2

    def attend(self):
        """Returns (seconds, K/V bytes of the attended tokens)."""
        import oracle
        c, b = self.case, self.b
        L, g = c.lens[b], c.g

        attend = oracle.attention_f64 if self.fmt != "bf16" else oracle.attention

        def one(h):
            K, V = self.att[h]
            if h in self.ret:
                rows = oracle.sparse_rows(1, L, c.P, self.sels[h], c.sinks, c.local)
            else:
                rows = np.arange(K.shape[0], dtype=np.int64)
            for j in range(g):
                attend(self.q[b, h * g + j], K, V, c.scale, rows=rows)
            return rows.shape[0] * row_bytes(c.d, self.hfmt[h]) * 2
        t0 = time.perf_counter()
        nbytes = sum(self.ex.map(one, self.ret + self.strm))
        return time.perf_counter() - t0, nbytes

    def window(self):
        """One reuse window: a selection, then reuse steps. Returns (seconds, bytes)."""
        secs, nbytes = self.select()
        for _ in range(self.case.reuse):
            s1, n1 = self.attend()
            secs, nbytes = secs + s1, nbytes + n1
        return secs, nbytes


def cpu_baseline_sparse(case, device, fmt: str = "bf16"):
    import oracle
    oracle.load()
    nthreads = len(os.sched_getaffinity(0))
    q, b, ret, strm, kv = sparse_oracle_sample(case, device)
    st = SparseOracleStep(case, q, b, ret, strm, kv, nthreads, fmt)
    secs, nbytes = st.window()
    windows = 1
    while secs * st.used < 10.0 and windows < 8:
        s2, n2 = st.window()
        secs, nbytes, windows = secs + s2, nbytes + n2, windows + 1
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": st.used,
            "kind": "oracle",
            "sample": f"request 0, retrieval KV heads {ret} (selection from the keys, then "
                      f"attention over the selected pages) and streaming KV heads {strm} "
                      f"(sinks and local window), {case.g} query heads each; {windows} reuse "
                      f"window(s) of 1 selection + {case.reuse} steps"
                      f"{QUANT_NOTE.get(fmt, '')}, {secs:.1f} s wall"}


def cpu_baseline(case, device, fmt: str = "bf16", T: int = 1):
    import oracle
    if case.head_kind is not None:
        return cpu_baseline_sparse(case, device, fmt)
    oracle.load()
    nthreads = len(os.sched_getaffinity(0))
    per_pair = max(1, sum(case.lens) // case.B) * case.d * (16 if fmt != "bf16" else 4)
    budget = max(nthreads, min(case.B * case.Hq, int(4e9 // per_pair) // T))
    q, pairs, kv = oracle_sample(case, device, budget, fmt=fmt)
    qs = None if T == 1 else [oracle.bf16_bits(case.q(t, device)) for t in range(T)]
    # repeat the sample until about 10 s of CPU work has been timed
    secs, nbytes, used = time_oracle(case, q, pairs, kv, nthreads, fmt, qs)
    reps = 1
    while secs * used < 10.0 and reps < 64:
        s2, n2, _ = time_oracle(case, q, pairs, kv, nthreads, fmt, qs)
        secs, nbytes, reps = secs + s2, nbytes + n2, reps + 1
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": used,
            "kind": "oracle",
            "sample": f"{len(pairs)} of {case.B * case.Hq} (request, query head) pairs of the "
                      f"{case.name} workload over their full contexts (fp64 dense attention"
                      f"{QUANT_NOTE.get(fmt, '')}"
                      f"{f', {T} causal query tokens each' if T > 1 else ''}), "
                      f"repeated {reps}x: {secs:.1f} s wall on {used} threads"}


def run_reference_sparse(args, world, case, device, nthreads):
    q, b, ret, strm, kv = sparse_oracle_sample(case, device)
    st = SparseOracleStep(case, q, b, ret, strm, kv, nthreads, args.kv_format)
    st.select()
    for _ in range(min(args.warmup, 1)):
        st.attend()
    secs, nbytes = 0.0, 0.0
    for i in range(args.steps):  # a selection at the start of every reuse window
        if i % case.reuse == 0:
            s1, n1 = st.select()
            secs, nbytes = secs + s1, nbytes + n1 / case.reuse * min(case.reuse, args.steps - i)
        s1, n1 = st.attend()
        secs, nbytes = secs + s1, nbytes + n1
    value = nbytes / secs / 1e9
    # a layer-step is the whole batch: scale the sampled heads to every (request, KV head)
    us_step = secs / args.steps * (case.B * case.Hkv / (len(ret) + len(strm))) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "us_per_layer_step": round(us_step, 1),
        "config": config_obj(case, args),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": st.used,
                         "kind": "oracle",
                         "sample": f"request 0, retrieval KV heads {ret} and streaming KV heads "
                                   f"{strm} per step, a selection every {case.reuse} steps"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The CPU oracle timed on the host cores, on a bounded sample of the same workload."""
    import oracle
    if rank != 0:
        return
    if args.config == "prefill-32k":
        from split_kv_decode_distattention_gb300 import workloads as W
        import torch
        case = make_case(args)
        kinds = [0] * case.Hkv if args.prefill_dense else list(case.head_kind)
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        cpu = prefill_cpu_baseline(case, dev, kinds, case.prefill_block_lists(W.PREFILL_KEEP),
                                   W.PREFILL_SINK_BLOCKS, W.PREFILL_LOCAL_BLOCKS, case.lens[0])
        print(json.dumps({"impl": "reference", "metric": PREFILL_METRIC, "value": cpu["value"],
                          "unit": "TFLOP/s", "n_gpus": world, "steps": 1, "warmup": 0,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f64", "data": "synthetic", "cpu_baseline": cpu,
                          "config": prefill_config(case, args, case.lens[0]),
                          "e2e": {"value": cpu["value"], "unit": "TFLOP/s",
                                  "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    import torch
    oracle.load()
    case = make_case(args)
    device = "cuda" if torch.cuda.is_available() else "cpu"
    nthreads = len(os.sched_getaffinity(0))
    if case.head_kind is not None:
        run_reference_sparse(args, world, case, device, nthreads)
        return
    fmt = args.kv_format
    per_pair = max(1, sum(case.lens) // case.B) * case.d * (16 if fmt != "bf16" else 4)
    budget = max(nthreads, min(case.B * case.Hq, int(1e9 // per_pair)))
    q, pairs, kv = oracle_sample(case, device, budget, fmt=fmt)
    T = args.queries
    qs = None if T == 1 else [oracle.bf16_bits(case.q(t, device)) for t in range(T)]
    for _ in range(min(args.warmup, 1)):
        time_oracle(case, q, pairs[:nthreads], kv, nthreads, fmt, qs)
    times, used, nbytes = [], nthreads, 0
    for _ in range(args.steps):
        secs, nb, used = time_oracle(case, q, pairs, kv, nthreads, fmt, qs)
        times.append(secs)
        nbytes += nb
    total = sum(times)
    value = nbytes / total / 1e9
    # a layer-step is the whole batch: scale the sample time to every (request, head) pair
    us_step = total / args.steps * (case.B * case.Hq / len(pairs)) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "us_per_layer_step": round(us_step, 1),
        "config": config_obj(case, args),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used,
                         "kind": "oracle",
                         "sample": f"{len(pairs)} of {case.B * case.Hq} (request, query head) "
                                   f"pairs per step, full contexts, fp64 dense attention"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ prefill leg

PREFILL_METRIC = ("block-sparse prefill: achieved TFLOP/s (4*d flops per attended query-key "
                  "pair) vs the measured bf16 tensor peak; ms per layer-step")


def prefill_pairs(case, Tq: int, kinds, lists, sinks: int, local: int) -> int:
    """Attended (query, key) pairs of one prefill chunk, summed over query heads, from the
    block rules: a query at position p sees 64 keys of every kept block before its own block
    qb, and p - 64*qb + 1 keys of block qb when it is kept."""
    total = 0
    for b, L in enumerate(case.lens):
        for qb in range((L - Tq) // 64, (L - 1) // 64 + 1):
            p0, p1 = max(L - Tq, 64 * qb), min(L, 64 * qb + 64)
            nq = p1 - p0
            diag = sum(p - 64 * qb + 1 for p in range(p0, p1))
            for kvh in range(case.Hkv):
                kind = kinds[kvh]
                if kind == 0:
                    before, own = qb, True
                elif kind == 2:
                    s_end = min(sinks, qb + 1)
                    l0 = max(s_end, qb - local + 1)
                    blocks = set(range(s_end)) | set(range(l0, qb + 1))
                    before, own = len([k for k in blocks if k < qb]), qb in blocks
                else:
                    row = set(int(x) for x in lists[b, kvh, qb] if 0 <= x <= qb)
                    before, own = len([k for k in row if k < qb]), qb in row
                total += case.g * (nq * 64 * before + (diag if own else 0))
    return total


def prefill_bytes(case, Tq: int) -> int:
    """Least DRAM bytes of one prefill launch: the chunk's bf16 queries read, the K/V of
    every valid token read once (bf16), the fp32 outputs written, and the block table."""
    L = case.lens[0]
    q = case.B * Tq * case.Hq * case.d * 2
    kv = case.B * L * case.Hkv * case.d * 2 * 2
    out = case.B * Tq * case.Hq * case.d * 4
    bt = case.B * (-(-L // case.P)) * 4
    return q + kv + out + bt


def run_prefill(args, rank: int, world: int):
    """One layer-step of block-sparse prefill: the chunk's K/V appended through
    dattn_kv_append, then dattn_prefill over the whole chunk (the lengths are reset outside the
    timed region, so every step prefills the same chunk)."""
    import torch

    import split_kv_decode_distattention_gb300 as dattn
    from split_kv_decode_distattention_gb300 import workloads as W
    from split_kv_decode_distattention_gb300.harness import PagedCache

    dattn.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    case = make_case(args)
    L = case.lens[0]
    Tq = L
    dense = args.prefill_dense
    kinds = [0] * case.Hkv if dense else list(case.head_kind)
    sinks, local = W.PREFILL_SINK_BLOCKS, W.PREFILL_LOCAL_BLOCKS
    cache = PagedCache(case, dev, fill=False)
    q = case.prefill_queries(Tq, dev)
    K, V = case.kv(0, 0, L, dev)
    kn, vn = K.unsqueeze(0).contiguous(), V.unsqueeze(0).contiguous()
    del K, V
    lists = case.prefill_block_lists(W.PREFILL_KEEP)
    sp = None
    if not dense:
        sp = dattn.PrefillSparseConfig(torch.tensor(kinds, dtype=torch.int8, device=dev), sinks,
                                       local, torch.from_numpy(lists).to(dev))
    out = torch.empty(1, Tq, case.Hq, case.d, dtype=torch.float32, device=dev)
    flops = 4 * case.d * prefill_pairs(case, Tq, kinds, lists, sinks, local)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def step(ev=None):
        cache.append(kn, vn)
        if ev is not None:
            ev[0].record(stream)
        dattn.dattn_prefill(cache.layout, cache.k_pool, cache.v_pool, q, case.scale,
                            cache.seq_lens, out, sparse=sp, dev_err=cache.dev_err)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        cache.seq_lens.zero_()
        step()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index) if (rank == 0 and not args.no_clocks) else None
    if clocks:
        clocks.start()
    times, kern = [], []
    for _ in range(args.steps):
        cache.seq_lens.zero_()
        flush()  # outside the timed region
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        kev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        e0.record(stream)
        step(kev)
        e1.record(stream)
        times.append((e0, e1))
        kern.append(kev)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    err = int(cache.dev_err.item())
    if err:
        raise RuntimeError(f"device error word {err:#x}")
    step_ms = [a.elapsed_time(b) for a, b in times]
    kern_ms = [a.elapsed_time(b) for a, b in kern]
    # whole job: the slowest rank's time, every rank's flops
    ms_all, flops_all = reduce_over_ranks(sum(step_ms), flops * len(step_ms), world, dev)
    ms = ms_all / len(step_ms)
    kms = sum(kern_ms) / len(kern_ms)
    res = {"flops": flops_all / len(step_ms), "flops_rank": flops, "ms": ms, "kms": kms,
           "kern_ms": kern_ms, "clocks": clk, "case": case, "Tq": Tq}
    # end to end: the chunk's q and K/V from pinned host memory, out back to pinned memory
    if not args.no_e2e:
        hq, hk, hv = q.cpu().pin_memory(), kn.cpu().pin_memory(), vn.cpu().pin_memory()
        hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(kn), torch.empty_like(vn)
        n = max(2, min(args.steps, 5))
        tot = 0.0
        for _ in range(n):
            cache.seq_lens.zero_()
            flush()
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            cache.append(dk, dv)
            dattn.dattn_prefill(cache.layout, cache.k_pool, cache.v_pool, dq, case.scale,
                                cache.seq_lens, out, sparse=sp, dev_err=cache.dev_err)
            hout.copy_(out, non_blocking=True)
            b2.record(stream)
            torch.cuda.synchronize()
            tot += a.elapsed_time(b2)
        res["e2e"] = {"value": round(flops / (tot / n * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                      "h2d_bytes_per_step": hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2,
                      "d2h_bytes_per_step": hout.numel() * 4,
                      "ms_per_layer_step": round(tot / n, 3), "steps": n}
    return res


def prefill_cpu_baseline(case, device, kinds, lists, sinks, local, Tq, target_s: float = 10.0):
    """The oracle's prefill attention on the host cores over a sample of query rows of two
    heads (the first of each kind present), as TFLOP/s. Rows are taken in a seeded random
    order of the chunk, a batch at a time, until about target_s seconds have passed."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.load()
    nthreads = len(os.sched_getaffinity(0))
    L = case.lens[0]
    q = oracle.bf16_bits(case.prefill_queries(Tq, device))
    heads = sorted({kinds.index(k) for k in set(kinds)})
    kv = {}
    for h in heads:
        K, V = case.kv(0, 0, L, device)
        kv[h] = (oracle.bf16_bits(K[:, h]), oracle.bf16_bits(V[:, h]))
    order = np.random.default_rng(case.seed).permutation(Tq)
    per_batch = 16 * nthreads

    def one(ht):
        h, t = ht
        qblk = (L - Tq + t) // 64
        rows = oracle.prefill_rows(kinds[h], L, Tq, t, sinks, local,
                                   blocks=lists[0, h, qblk] if kinds[h] == 1 else None)
        oracle.attention(q[0, t, h * case.g], kv[h][0], kv[h][1], case.scale, rows=rows)
        return rows.shape[0]

    pairs, nrows, i = 0, 0, 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        while i < Tq and (i == 0 or time.perf_counter() - t0 < target_s):
            work = [(h, int(t)) for t in order[i:i + per_batch] for h in heads]
            pairs += sum(ex.map(one, work))
            nrows += len(work)
            i += per_batch
    secs = time.perf_counter() - t0
    return {"value": round(4 * case.d * pairs / secs / 1e12, 6), "unit": "TFLOP/s",
            "cores": min(nthreads, nrows), "kind": "oracle",
            "sample": f"{nrows} query rows (a seeded random order of the chunk's rows) of KV "
                      f"heads {heads}, one query head each, fp64 attention over their prefill "
                      f"rows: {pairs} query-key pairs in {secs:.1f} s wall"}


def prefill_config(case, args, Tq: int) -> dict:
    """The config object of the prefill leg, the same in both arms."""
    return {"workload": f"{case.name}: {WORKLOAD_TEXT[case.name]}" +
                        (" (every head dense: causal attention)" if args.prefill_dense else ""),
            "batch": case.B, "q_heads": case.Hq, "kv_heads": case.Hkv, "head_dim": case.d,
            "page_size": case.P, "context_tokens": case.lens[0], "chunk_tokens": Tq,
            "seed": args.seed, "parallelism": "replicas" if args.gpus > 1 else "single GPU",
            "step": "dattn_kv_append (the chunk's K/V) + dattn_prefill",
            "l2": f"flushed before every timed step ({L2Flush.TEXT})",
            "launch": "eager library calls"}


def prefill_main(args, rank: int, world: int):
    from split_kv_decode_distattention_gb300 import workloads as W
    res = run_prefill(args, rank, world)
    case = res["case"]
    dense = args.prefill_dense
    kinds = [0] * case.Hkv if dense else list(case.head_kind)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = prefill_cpu_baseline(case, "cuda", kinds, case.prefill_block_lists(W.PREFILL_KEEP),
                                   W.PREFILL_SINK_BLOCKS, W.PREFILL_LOCAL_BLOCKS, res["Tq"])
    if rank != 0:
        return
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = float(peaks.get("bf16_tflops", 1900.0))
    tflops = res["flops"] / (res["ms"] * 1e-3) / 1e12
    ktf = res["flops_rank"] / (res["kms"] * 1e-3) / 1e12
    cfg = prefill_config(case, args, res["Tq"])
    line = {
        "metric": PREFILL_METRIC, "value": round(tflops, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(res["ms"], 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q)", "config": cfg,
        "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel (dattn_prefill)",
                     "achieved": round(ktf, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(ktf / peak, 4),
                     "peak_source": "measured" if "bf16_tflops" in peaks else "fallback",
                     "traffic": traffic_record(traffic_key(args), PREFILL_SOURCES,
                                               alg_bytes=prefill_bytes(case, res["Tq"])),
                     "algorithmic_flops_per_launch": int(res["flops_rank"]),
                     "algorithmic_bytes_per_launch": prefill_bytes(case, res["Tq"]),
                     "avg_launch_ms": round(res["kms"], 4),
                     "kernel_timing": "CUDA events around the prefill kernel in every step"},
        # the chunk's append is two launches (the kernel, then the length update), then one
        "gpu_launches": 3 * args.steps,
        "clocks": res["clocks"], "cpu_baseline": cpu,
    }
    if "e2e" in res:
        line["e2e"] = res["e2e"]
    print(json.dumps(line), flush=True)


def config_obj(case, args):
    c = {"workload": f"{case.name}: {WORKLOAD_TEXT[case.name]}", "batch": case.B,
         "q_heads": case.Hq, "kv_heads": case.Hkv, "head_dim": case.d, "page_size": case.P,
         "context_tokens": (case.lens[0] if len(set(case.lens)) == 1 else
                            f"{min(case.lens)}-{max(case.lens)} (sum {sum(case.lens)})"),
         "seed": args.seed,
         "kv_format": KV_FORMAT_NOTE[args.kv_format],
         "parallelism": "replicas" if args.gpus > 1 else "single GPU",
         "step": (("dattn_append_decode (1 token/request appended and attended in one launch)"
                   if fused_step(args) else
                   "dattn_kv_append (1 token/request) + dattn_decode") +
                  (" + dattn_page_select every 16 steps (block-sparse)"
                   if case.head_kind is not None else "")
                  if args.queries == 1 else
                  f"dattn_kv_append ({args.queries} tokens/request) + dattn_decode_multi "
                  f"({args.queries} query tokens/request, causal over the new tokens)"),
         "launch": ("one CUDA graph per step, captured from the library calls"
                    if getattr(args, "graph", False) else "eager library calls"),
         "l2": l2_policy(case, args)[1]}
    if args.queries > 1:
        c["queries_per_request"] = args.queries
    if args.batch or args.ctx:
        c["reduced_for_profiling"] = True
    return c


def main():
    args = parse_args()
    if args.profile:
        args.no_e2e = args.no_cpu_baseline = args.no_clocks = True
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    import torch.distributed as dist
    if world > 1:
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.config == "prefill-32k":
        prefill_main(args, rank, world)
        if world > 1:
            dist.destroy_process_group()
        return
    res = run_dattn(args, rank, world)
    also_args = also_config(args)
    res_also = run_dattn(also_args, rank, world) if also_args is not None else None
    case = res["case"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, "cuda", args.kv_format, args.queries)
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    steps = args.steps
    ms_step = res["ms_total"] / steps
    value = res["bytes_all"] / (res["ms_total"] * 1e-3) / 1e9
    dec_avg_ms = sum(res["dec_ms"]) / len(res["dec_ms"])
    dec_med_ms = statistics.median(res["dec_ms"])
    achieved = res["dec_bytes"] / (dec_avg_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    traffic = traffic_record(traffic_key(args), alg_bytes=res["dec_bytes"])
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16",
                  "fp8": "fp8_e4m3 KV (fp16 tensor-core products, fp32 accumulate)",
                  "int4": "int4 KV (fp16 tensor-core products, fp32 accumulate)",
                  "mixed": "fp8_e4m3 retrieval/dense heads + int4 streaming heads KV (fp16 "
                           "tensor-core products, fp32 accumulate)"}[args.kv_format],
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q" +
                {"bf16": ")", "fp8": "; K/V quantized to 8 bits by the append)",
                 "int4": "; K/V quantized to 4 bits by the append)",
                 "mixed": "; K/V quantized by the append: 8 bits for retrieval and dense "
                          "heads, 4 bits for streaming heads)"}[args.kv_format],
        "us_per_layer_step": round(ms_step * 1e3, 2),
        "frac_of_8tbs": round(value / ROOFLINE_8TBS, 4),
        "config": config_obj(case, args),
        "roofline": {"bound": "hbm",
                     "kernel": ("attention_kernel (dattn_append_decode)" if fused_step(args)
                                else "attention_kernel (dattn_decode)"),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "peak_source": (f"{peak_kind}: HBM copy bandwidth (read + write bytes of a "
                                     f"copy); the decode kernel only reads, see read_peak"),
                     "traffic": traffic, "algorithmic_bytes_per_launch": int(res["dec_bytes"]),
                     "avg_launch_us": round(dec_avg_ms * 1e3, 2),
                     "median_launch_us": round(dec_med_ms * 1e3, 2),
                     "achieved_at_median": round(res["dec_bytes"] / (dec_med_ms * 1e-3) / 1e9, 1),
                     "frac_of_8tbs": round(achieved / ROOFLINE_8TBS, 4),
                     "timed_launches": len(res["dec_ms"]),
                     "kernel_timing": f"CUDA events around the decode kernel in every "
                                      f"{res['kernel_every']}th timed step",
                     "launch_us_min_med_max": [round(min(res["dec_ms"]) * 1e3, 1),
                                               round(statistics.median(res["dec_ms"]) * 1e3, 1),
                                               round(max(res["dec_ms"]) * 1e3, 1)]},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "cpu_baseline": cpu,
    }
    if "read_peak" in res:
        line["roofline"]["read_peak"] = {"gbs": round(res["read_peak"], 1), "how": READ_PEAK_HOW,
                                         "frac": round(achieved / res["read_peak"], 4)}
    if "info" in res:
        line["info"] = res["info"]
    if "e2e" in res:
        line["e2e"] = res["e2e"]
    if res_also is not None:
        line["also"] = also_summary(res_also, also_args, peak)
    print(json.dumps(line), flush=True)


def also_config(args):
    """The arguments of the second workload (None: no second workload). The default run adds
    the block-sparse workload, so that one line carries both decode paths."""
    name = args.also
    if name == "auto":
        plain = (args.config == "mha-1m" and args.kv_format == "bf16" and args.queries == 1
                 and not (args.batch or args.ctx or args.profile))
        name = "sparse-512k" if plain else "none"
    if name in ("none", args.config):
        return None
    if name not in WORKLOAD_TEXT or name == "prefill-32k":
        raise SystemExit(f"--also {name}: not a decode workload")
    a = argparse.Namespace(**vars(args))
    a.config, a.also, a.no_cpu_baseline = name, "none", True
    return a


def also_summary(res, args, peak) -> dict:
    """The second workload's figures: its steps' value and time and its decode kernel's
    roofline, timed as the main line's."""
    case = res["case"]
    ms_step = res["ms_total"] / args.steps
    value = res["bytes_all"] / (res["ms_total"] * 1e-3) / 1e9
    dec_avg_ms = sum(res["dec_ms"]) / len(res["dec_ms"])
    achieved = res["dec_bytes"] / (dec_avg_ms * 1e-3) / 1e9
    out = {"config": config_obj(case, args), "value": round(value, 2), "unit": "GB/s",
           "steps": args.steps, "us_per_layer_step": round(ms_step * 1e3, 2),
           "frac_of_8tbs": round(value / ROOFLINE_8TBS, 4),
           "roofline": {"bound": "hbm",
                        "kernel": ("attention_kernel (dattn_append_decode)" if fused_step(args)
                                   else "attention_kernel (dattn_decode)"),
                        "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(achieved / peak, 4),
                        "traffic": traffic_record(traffic_key(args),
                                                  alg_bytes=res["dec_bytes"]),
                        "algorithmic_bytes_per_launch": int(res["dec_bytes"]),
                        "avg_launch_us": round(dec_avg_ms * 1e3, 2),
                        "median_launch_us": round(statistics.median(res["dec_ms"]) * 1e3, 2),
                        "timed_launches": len(res["dec_ms"])},
           "gpu_launches": res["launches"], "clocks": res["clocks"]}
    if "e2e" in res:
        out["e2e"] = res["e2e"]
    return out


if __name__ == "__main__":
    main()
