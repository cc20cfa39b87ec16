#!/usr/bin/env python3
"""Benchmark of the QSA-indexer hot path: paged MQA-logits scoring + top-k.

One step = qsa_paged_mqa_logits + qsa_select_topk_bounded (the batch's
longest visible count as the host bound) over one batch of the workload (two
kernel launches; with --step fused one qsa_paged_mqa_topk call).  Prints one
JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Timing: K steps back to back on one stream between a barrier and a device
synchronize on both sides, enqueued as CUDA graph replays (one graph of the K
steps up to 256) so host launch overhead is not on the device timeline; CUDA events
around the K steps give the step time, and graphs of scoring-only and
top-k-only launches give each kernel's average launch time.  Inputs and
outputs rotate over enough copies that their footprint exceeds twice the L2,
so no step reads another step's data from L2.  `value` is key-cache bytes processed
per second over the whole step (each request's visible keys counted once),
summed over ranks with the max time over ranks.  Under torchrun each rank runs
its own replica of the workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import qsa_inputs as qi  # noqa: E402

METRIC = "paged index-scoring µs/call and key-cache GB/s vs HBM peak; top-k µs/row"
DEFAULT_WORKLOAD = "single_row_decode"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# Host-side helpers (unit-tested on CPU, including the multi-rank reduction)
# ---------------------------------------------------------------------------


def rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def algorithmic_bytes(spec: qi.Spec):
    """Bytes each kernel must move at least once per launch.  Scorer: each
    request's visible key columns once (fp8 scales included), q, the weights,
    the block-table entries of the pages read, the visible counts and the
    logits written.  Top-k: the visible logits read, the counts and the
    indices written."""
    R, H = spec.num_rows, spec.num_heads
    pages = int(spec.pages_needed().sum())
    score = {
        "keys": spec.key_bytes_touched(),
        "q": R * H * spec.head_dim * 2,
        "weights": R * H * 4,
        "block_table": pages * 4,
        "visible": R * 4,
        "logits_out": R * spec.out_cols * 4,
    }
    vis = spec.live_visible().astype(np.int64)
    topk = {"logits_in": int(np.minimum(vis, spec.out_cols).sum()) * 4, "visible": R * 4,
            "indices_out": R * spec.k * 4}
    return score, topk


def strip_comments(src: str) -> str:
    """C/C++ source without // and /* */ comments (string and character
    literals kept) and without blank lines or trailing spaces: what the
    compiler sees, so a comment edit leaves a kernel's recorded counters valid."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def source_sha(paths):
    """Hash of the kernel sources as compiled (comments and blank lines aside)."""
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


_CS = "sparse_attention_indexer_02_gb300/csrc/"
_COMMON = [_CS + "device_common.cuh", _CS + "sm100_ptx.cuh"]  # headers every kernel below includes
KERNEL_SOURCES = {
    "rowcore": [_CS + "rowcore.cu", _CS + "device_common.cuh"],
    "umma_lean": [_CS + "umma_kernel.cuh", _CS + "umma.cu", _CS + "topk_select.cuh"] + _COMMON,
    "umma": [_CS + "umma_kernel.cuh", _CS + "umma.cu", _CS + "topk_select.cuh"] + _COMMON,
    "topk": [_CS + "topk.cu", _CS + "topk_select.cuh"] + _COMMON,
    "umma+topk": [_CS + "umma_kernel.cuh", _CS + "umma.cu", _CS + "topk_select.cuh"] + _COMMON,
}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since it was captured; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel, {}).get(workload)
    except Exception:
        return None
    if not rec or rec.get("source_sha") != source_sha(KERNEL_SOURCES[kernel]):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons over a window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index
        try:
            import tempfile

            fd, self.path = tempfile.mkstemp(prefix="qsa_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        import datetime

        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append((ts, parts))
        os.unlink(self.path)
        inside = [p for ts, p in rows if t0 - 0.06 <= ts <= t1 + 0.06] or [p for _, p in rows[-3:]]
        if not inside:
            return None
        sm = [float(p[2]) for p in inside if p[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in inside:
            for name, v in zip(names, p[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(inside[0][3]) if inside[0][3].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------------------
# CPU oracle arm (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------


def oracle_sample_run(inp, requests, threads):
    """Oracle scoring + top-k for whole requests; returns (seconds, key bytes)."""
    import oracle

    spec = inp.spec
    rows = [r for b in requests for r in range(b * spec.rows_per_req, (b + 1) * spec.rows_per_req)]
    t0 = time.perf_counter()
    lg = oracle.paged_mqa_logits(inp, rows=rows, threads=threads)
    oracle.select_topk(lg, spec.live_visible()[rows], spec.k, threads=threads)
    dt = time.perf_counter() - t0
    vis = spec.live_visible().reshape(spec.num_requests, spec.rows_per_req).max(axis=1)
    key_bytes = int(sum(int(vis[b]) for b in requests)) * spec.key_bytes_per_col
    return dt, key_bytes, len(rows)


def cpu_baseline(inp, budget_s: float = 10.0, threads=None):
    """The oracle on the host cores (all of them, or `threads`): whole requests
    (scoring + top-k), repeated until about budget_s seconds of work;
    prefill-sized requests are sampled by rows instead.  Returns key-cache GB/s
    over the sample."""
    import oracle

    oracle.build()
    threads = threads or oracle.default_threads()
    spec = inp.spec
    rng = np.random.default_rng(0)
    order = rng.permutation(spec.num_requests).tolist()
    if spec.rows_per_req > 64:
        t_rows = time.perf_counter()
        sub_rows = [order[0] * spec.rows_per_req + i for i in range(min(64, spec.rows_per_req))]
        oracle.paged_mqa_logits(inp, rows=sub_rows, threads=threads)
        per_row = (time.perf_counter() - t_rows) / len(sub_rows)
        n_rows = max(1, min(spec.num_rows, int(budget_s / max(per_row, 1e-9) * 0.8)))
        rows = sorted(rng.choice(spec.num_rows, n_rows, replace=False).tolist())
        t0 = time.perf_counter()
        lg = oracle.paged_mqa_logits(inp, rows=rows, threads=threads)
        oracle.select_topk(lg, spec.live_visible()[rows], spec.k, threads=threads)
        dt = time.perf_counter() - t0
        # keys of a request are shared by its rows: credit each sampled row with
        # its share of the request's key bytes
        key_bytes = spec.key_bytes_touched() * len(rows) / spec.num_rows
        sample = f"{len(rows)} of {spec.num_rows} rows (scoring + top-k), key bytes credited pro rata"
        return {"value": key_bytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": sample, "seconds": round(dt, 3)}
    dt1, _, _ = oracle_sample_run(inp, order[:1], threads)  # one request, to size the sample
    if dt1 * spec.num_requests / threads >= budget_s:
        n_req = max(1, min(spec.num_requests, int(budget_s * threads / max(dt1, 1e-9))))
        dt, kb, nrows = oracle_sample_run(inp, order[:n_req], threads)
        sample = f"{n_req} of {spec.num_requests} requests ({nrows} rows, scoring + top-k)"
    else:
        passes = dt = kb = 0
        while dt < budget_s:  # whole steps until the budget is spent
            d, b, nrows = oracle_sample_run(inp, order, threads)
            dt += d
            kb += b
            passes += 1
        sample = f"the whole step (all {spec.num_requests} requests, {spec.num_rows} rows), {passes} times"
    return {"value": kb / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
            "seconds": round(dt, 3)}


def run_reference(args):
    rank, world, _ = rank_env()
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    threads = oracle.default_threads()
    spec = qi.WORKLOADS[args.workload]()
    inp = qi.build_inputs(spec)
    rng = np.random.default_rng(0)
    # size each step's sample so the whole run stays within a few minutes
    dt1, _, _ = oracle_sample_run(inp, [0], threads)
    budget_step = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    n_req = max(1, min(spec.num_requests, int(budget_step / max(dt1, 1e-6))))
    steps = []
    kbytes = 0
    for i in range(args.warmup + args.steps):
        reqs = rng.choice(spec.num_requests, n_req, replace=False).tolist()
        dt, kb, nrows = oracle_sample_run(inp, reqs, threads)
        if i >= args.warmup:
            steps.append(dt)
            kbytes += kb
    total = sum(steps)
    value = kbytes / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(spec, None),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_req} of {spec.num_requests} requests per step (scoring + top-k)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def workload_config(spec: qi.Spec, l2_note):
    cfg = {"workload": spec.name, "requests": spec.num_requests, "rows_per_req": spec.rows_per_req,
           "heads": spec.num_heads, "head_dim": spec.head_dim, "page_cols": spec.page_cols,
           "out_cols": spec.out_cols, "k": spec.k, "kv": "bf16" if spec.kv_dtype == qi.KV_BF16 else "fp8_e4m3",
           "q": "bf16" if spec.q_dtype == qi.Q_BF16 else "fp8_e4m3",
           "visible_cols_total": int(spec.live_visible().astype(np.int64).sum()),
           "key_bytes_per_step": spec.key_bytes_touched()}
    if spec.next_n_lens is not None:
        cfg["live_rows"] = int(spec.live_rows().sum())
    if l2_note:
        cfg["l2"] = l2_note
    return cfg


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


def stats(samples):
    """median / min / max of per-launch times (µs), and how many launches."""
    v = sorted(x for x, _ in samples)
    return {"median": round(statistics.median(v), 3), "min": round(v[0], 3), "max": round(v[-1], 3),
            "launches": int(sum(n for _, n in samples))}


def build_record():
    """Units build.py had to compile without ptxas optimisation (its fallback
    when the compiler crashes); empty for a normal build."""
    from sparse_attention_indexer_02_gb300 import build as qbuild

    return {"ptxas_O0_units": qbuild.o0_units()}


FORCED = {"variant": -1}  # the scorer variant --variant forces (-1: the dispatch's)

SWEEP = ["tiny_mtp", "single_row_decode", "mtp3_verify_p16", "mtp3_verify_p64", "mtp3_large_p16",
         "mtp3_large_p64", "fp8_h64", "prefill_chunk", "fp8q_h64", "ragged_nn8"]


class Workload:
    """One workload on the device: rotating input/output copies (their
    footprint over twice the L2), the three call forms, and graphs of them."""

    def __init__(self, name, dev, rank=0, rotate=True):
        import torch
        from sparse_attention_indexer_02_gb300 import torch_api

        base = qi.WORKLOADS[name]()
        self.spec = spec = dataclasses.replace(base, seed=base.seed + 7919 * rank)  # per-rank data, same shape
        self.inp = inp = qi.build_inputs(spec)
        self.host = qi.device_tensors(inp, pin=True)
        self.dev = dev
        R, k = spec.num_rows, spec.k
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        per_copy = inp.kv.nbytes + R * spec.out_cols * 4 + inp.q.nbytes + R * k * 4
        self.copies = copies = 1 if not rotate else int(min(16, max(1, math.ceil(2.0 * l2 / per_copy))))
        self.sets = []
        for _ in range(copies):
            d = {n: t.to(dev, non_blocking=False) for n, t in self.host.items()}
            d["out"] = torch.empty((R, spec.out_cols), dtype=torch.float32, device=dev)
            d["idx"] = torch.empty((R, k), dtype=torch.int32, device=dev)
            self.sets.append(d)
        self.l2_note = (f"rotating {copies} input/output copies ({copies * per_copy / 1e6:.0f} MB, > 2x the "
                        f"{l2 / 1e6:.0f} MB L2)" if copies > 1 else
                        f"single copy ({per_copy / 1e6:.0f} MB of inputs+outputs, larger than 2x L2)"
                        if per_copy > 2 * l2 else f"single copy ({per_copy / 1e6:.0f} MB), L2 not defeated")
        self.max_visible = int(spec.live_visible().max()) if R else 0
        self.api = torch_api
        # the pages the scorer reads (each request's pages holding a visible
        # column of a live row), for the page-stream reference
        need = spec.pages_needed()
        self.page_list = np.concatenate([inp.block_table[b, :need[b]] for b in range(spec.num_requests)]
                                        ).astype(np.int32) if spec.num_requests else np.zeros(0, np.int32)
        self.page_bytes = inp.key_page_stride  # a whole page: bf16 keys, or fp8 keys and their scales
        pages_dev = torch.from_numpy(self.page_list).to(dev)
        for d in self.sets:
            d["pages"] = pages_dev
            d["pcheck"] = torch.zeros(1, dtype=torch.int32, device=dev)
        self.per_graph = copies * max(1, -(-16 // copies))

    def score(self, d):
        s = self.spec
        self.api.paged_mqa_logits(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"],
                                  page_cols=s.page_cols, out_cols=s.out_cols, kv_dtype=s.kv_dtype,
                                  scale_offset=self.inp.scale_offset, out=d["out"], next_n_lens=d.get("next_n_lens"))

    def stream(self, d):
        """The page-stream reference: the scorer's pages, read and discarded."""
        self.api.page_stream(d["kv"], self.inp.key_page_stride, self.page_bytes, d["pages"], checksum=d["pcheck"])

    def topk(self, d):
        # the ragged call's top-k reads the live rows' visible counts; the
        # batch's longest one is the host bound (qsa_select_topk_bounded)
        self.api.select_topk(d["out"], d.get("visible_live", d["visible"]), self.spec.k, out=d["idx"],
                             max_visible=self.max_visible)

    def one_call(self, d):
        # qsa_paged_mqa_topk; the host bound of the visible counts steers its
        # dispatch (the selection inside the scoring kernel for decode-sized calls)
        s = self.spec
        self.api.paged_mqa_topk(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"], s.k,
                                page_cols=s.page_cols, out_cols=s.out_cols, kv_dtype=s.kv_dtype,
                                scale_offset=self.inp.scale_offset, max_visible=self.max_visible,
                                out_logits=d["out"], out_idx=d["idx"], next_n_lens=d.get("next_n_lens"))

    def step(self, d, form):
        if form == "one-call":
            self.one_call(d)
        else:
            self.score(d)
            self.topk(d)

    def capture(self, n, what):
        import torch

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                d = self.sets[i % self.copies]
                if what == "score":
                    self.score(d)
                elif what == "stream":
                    self.stream(d)
                elif what == "topk":
                    self.topk(d)
                else:
                    self.step(d, what)
        return g

    def time_graph(self, g, n_launch, reps):
        """Per-launch mean of each of `reps` replays of a graph of n_launch calls."""
        import torch

        stream = torch.cuda.current_stream(self.dev)
        for _ in range(2):
            g.replay()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        torch.cuda.synchronize(self.dev)
        ev[0].record(stream)
        for i in range(reps):
            g.replay()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(self.dev)
        return [(1e3 * ev[i].elapsed_time(ev[i + 1]) / n_launch, n_launch) for i in range(reps)]

    def kernel_stats(self, min_launches=64):
        """scoring, top-k, two-call step and one-call step: per-launch median/min/max."""
        import sparse_attention_indexer_02_gb300 as qsa
        import torch

        for i in range(3):  # eager first calls (kernel attributes; the one-call workspace)
            d = self.sets[i % self.copies]
            self.score(d)
            self.topk(d)
        variant = qsa.VARIANT_NAMES.get(qsa.last_variant(), "none")
        for i in range(3):
            self.one_call(self.sets[i % self.copies])
        one_variant = qsa.VARIANT_NAMES.get(qsa.last_variant(), "none")
        torch.cuda.synchronize(self.dev)
        n = self.per_graph
        reps = max(4, -(-min_launches // n))
        out = {"variant": variant, "one_call_variant": one_variant}
        for key, what in (("scoring_us", "score"), ("topk_us", "topk"), ("step_us", "two-call"),
                          ("one_call_us", "one-call")):
            g = self.capture(n, what)
            out[key] = stats(self.time_graph(g, n, reps))
            del g
        if self.page_list.size:  # the same pages, streamed with no arithmetic
            self.stream(self.sets[0])
            torch.cuda.synchronize(self.dev)
            g = self.capture(n, "stream")
            out["page_stream_us"] = stats(self.time_graph(g, n, reps))
            del g
        # the one call with the selection inside the scoring kernel (forced;
        # the dispatch takes the two launches), where that kernel serves the shape
        qsa.force_variant(qsa.VARIANT_UMMA_TOPK)
        try:
            for i in range(3):
                self.one_call(self.sets[i % self.copies])
            if qsa.last_variant() == qsa.VARIANT_UMMA_TOPK:
                torch.cuda.synchronize(self.dev)
                g = self.capture(n, "one-call")
                out["fused_kernel_us"] = stats(self.time_graph(g, n, reps))
                del g
        finally:
            qsa.force_variant(FORCED["variant"])
        return out

    def summary(self, ks, peaks):
        """The per-workload entry of the bench line."""
        spec = self.spec
        sb, tb = algorithmic_bytes(spec)
        key_bytes = spec.key_bytes_touched()
        t_score = ks["scoring_us"]["median"] * 1e-6
        t_topk = ks["topk_us"]["median"] * 1e-6
        e = {"config": workload_config(spec, self.l2_note), **ks,
             "key_gbs_scoring": round(key_bytes / t_score / 1e9, 1),
             "frac_key_bytes": round(key_bytes / t_score / 1e9 / peaks["hbm_gbs"], 4),
             "frac_all_bytes": round(sum(sb.values()) / t_score / 1e9 / peaks["hbm_gbs"], 4),
             "topk_gbs": round(sum(tb.values()) / t_topk / 1e9, 1),
             "topk_frac": round(sum(tb.values()) / t_topk / 1e9 / peaks["hbm_gbs"], 4),
             "topk_us_per_row": round(ks["topk_us"]["median"] / spec.num_rows, 4)}
        if "page_stream_us" in ks:
            t_stream = ks["page_stream_us"]["median"] * 1e-6
            sbytes = self.page_list.size * self.page_bytes
            e["page_stream_gbs"] = round(sbytes / t_stream / 1e9, 1)
            e["page_stream_frac"] = round(sbytes / t_stream / 1e9 / peaks["hbm_gbs"], 4)
            e["scoring_vs_page_stream"] = round(t_stream / t_score, 4)
        flops = 2 * spec.head_dim * spec.num_heads * int(spec.live_visible().astype(np.int64).sum())
        if spec.rows_per_req > 64:  # the contraction-heavy case: tensor-core rate too
            e["mma_tflops"] = round(flops / t_score / 1e12, 1)
            e["frac_bf16_peak"] = round(flops / t_score / 1e12 / peaks["bf16_tflops"], 4)
        return e

    def free(self):
        import torch

        self.sets = []
        self.host = None
        torch.cuda.empty_cache()


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import sparse_attention_indexer_02_gb300 as qsa
    from sparse_attention_indexer_02_gb300 import build as qbuild

    rank, world, local = rank_env()
    if world > 1:
        dist.init_process_group(backend="nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qbuild.build()
    qsa.load_library()
    FORCED["variant"] = {"auto": qsa.VARIANT_AUTO, "rowcore": qsa.VARIANT_ROWCORE, "umma": qsa.VARIANT_UMMA,
                         "lean": qsa.VARIANT_UMMA_LEAN}[args.variant]
    qsa.force_variant(FORCED["variant"])
    peaks = measured_peaks()

    W = Workload(args.workload, dev, rank, rotate=not args.no_rotate)
    spec, inp, host, sets, copies = W.spec, W.inp, W.host, W.sets, W.copies
    R, k = spec.num_rows, spec.k
    form = "one-call" if args.step == "fused" else "two-call"
    for i in range(args.warmup):  # eager warm-up (first calls set kernel attributes)
        d = sets[i % copies]
        W.score(d)
        W.topk(d)
        W.one_call(d)
    torch.cuda.synchronize(dev)

    # the timed region: K steps as graph replays - one graph of exactly K steps
    # up to 256, else graphs of 256 and one of the rest - so host launch
    # overhead is not on the device timeline
    K = args.steps
    per_graph = K if K <= 256 else 256
    full_graphs, rem = divmod(K, per_graph)
    g_step = W.capture(per_graph, form)
    g_rem = W.capture(rem, form) if rem else None

    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local) if rank == 0 and not args.no_clocks else None
    time.sleep(0.3 if sampler else 0.0)  # the sampler is up before the last warm-up
    # warm-up replays of the graph right before the timed region (after the
    # sampler's start-up, so the GPU has not idled since)
    for _ in range(max(1, -(-args.warmup // per_graph))):
        g_step.replay()
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(full_graphs):
        g_step.replay()
    if g_rem is not None:
        g_rem.replay()
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier()
    clocks = sampler.stop(t0, t1) if sampler else None
    total_ms = e_start.elapsed_time(e_end)
    del g_step, g_rem

    # per-kernel launch times on the same workload (median/min/max over replays)
    ks = W.kernel_stats()
    head = W.summary(ks, peaks)

    max_ms = max_over_ranks(total_ms)
    ms_step = max_ms / K
    key_bytes = spec.key_bytes_touched()
    value = sum_over_ranks(key_bytes * K) / (max_ms / 1e3) / 1e9

    # roofline of the dominant kernel of the step
    sb, tb = algorithmic_bytes(spec)
    variant = ks["variant"]
    score_us, topk_us = ks["scoring_us"]["median"], ks["topk_us"]["median"]
    if form == "one-call":  # one kernel: its bytes are the scoring's and the selection's
        kname, kbytes, kus = ks["one_call_variant"], sum(sb.values()) + sum(tb.values()), ks["one_call_us"]["median"]
    elif score_us >= topk_us:
        kname, kbytes, kus = variant, sum(sb.values()), score_us
    else:
        kname, kbytes, kus = "topk", sum(tb.values()), topk_us
    achieved = kbytes / (kus * 1e-6) / 1e9
    traffic = recorded_traffic(kname, spec.name) if kname in KERNEL_SOURCES else None
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "algorithmic_bytes": int(kbytes), "peak_source": f"{peaks['source']} (copy bandwidth)",
                "key_bytes_frac": head["frac_key_bytes"] if kname != "topk" else None}
    if kname != "topk" and "page_stream_gbs" in head:
        # the achievable side: the scorer's pages streamed with no arithmetic
        # (qsa_page_stream), and the scoring call's time against it
        roofline["page_stream"] = {"achieved": head["page_stream_gbs"], "unit": "GB/s",
                                   "frac_of_peak": head["page_stream_frac"],
                                   "scoring_frac_of_stream": head["scoring_vs_page_stream"]}

    # end to end through the public API with host buffers: H2D of every input
    # from pinned memory, both calls, D2H of the top-k indices, every step
    e2e = None
    if not args.no_e2e:
        # two input buffers let step i+1's copies run on a copy stream while
        # step i's kernels run
        bufs = [sets[0], sets[1 % copies] if copies > 1 else
                {name: torch.empty_like(t) for name, t in sets[0].items()}]
        out_host = [torch.empty((R, k), dtype=torch.int32).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host[0].numel() * 4
        Ke = max(5, min(K, 200))
        comp = torch.cuda.current_stream(dev)
        cstream = torch.cuda.Stream(dev)
        ready = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        for f in free:
            f.record(comp)

        def e2e_step(i):
            b = bufs[i % 2]
            with torch.cuda.stream(cstream):
                cstream.wait_event(free[i % 2])  # the buffer's previous step is done with it
                for name, t in host.items():
                    b[name].copy_(t, non_blocking=True)
                ready[i % 2].record(cstream)
            comp.wait_event(ready[i % 2])
            W.step(b, form)
            out_host[i % 2].copy_(b["idx"], non_blocking=True)
            free[i % 2].record(comp)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        cstream.wait_stream(comp)  # no copy of the timed steps starts before e0
        for i in range(Ke):
            e2e_step(i)
        comp.wait_stream(cstream)
        e1.record(comp)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1))
        e2e = {"value": sum_over_ranks(key_bytes * Ke) / (e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms / Ke, "steps": Ke,
               "pipeline": "step i+1's host-to-device copies overlap step i's kernels (two input buffers)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp)
        one = cpu_baseline(inp, budget_s=5.0, threads=1)
        cpu["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": 1, "sample": one["sample"],
                                "seconds": one["seconds"]}
    W.free()
    del W, sets, host

    # every configuration of the workload statement (and the ragged and fp8-q
    # calls), timed the same way, one after another
    workloads = {spec.name: head}
    if rank == 0 and not args.no_workloads:
        for name in SWEEP:
            if name == args.workload:
                continue
            Wn = Workload(name, dev, rank, rotate=not args.no_rotate)
            workloads[Wn.spec.name] = Wn.summary(Wn.kernel_stats(), peaks)
            Wn.free()
            del Wn

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ("bf16" if spec.kv_dtype == qi.KV_BF16 else
                                           "fp8e4m3-keys/bf16-q" if spec.q_dtype == qi.Q_BF16 else "fp8e4m3"),
            "data": "synthetic (seeded; shapes of the pages' workloads)",
            "config": head["config"],
            "variant": variant,
            "us_per_call": score_us, "key_gbs_scoring": head["key_gbs_scoring"],
            "topk_us_per_row": head["topk_us_per_row"], "topk_us_per_call": topk_us,
            "step_us": round(1e3 * ms_step, 3),
            "one_call_us": ks["one_call_us"]["median"], "one_call_variant": ks["one_call_variant"],
            "fused_kernel_us": ks.get("fused_kernel_us", {}).get("median"),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": (1 if form == "one-call" else 2) * K, "clocks": clocks,
            "build": build_record(), "workloads": workloads,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(qi.WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--variant", choices=["auto", "rowcore", "umma", "lean"], default="auto")
    ap.add_argument("--step", choices=["two-call", "fused"], default="two-call",
                    help="time the step as qsa_paged_mqa_logits + qsa_select_topk_bounded, or as one qsa_paged_mqa_topk")
    ap.add_argument("--no-rotate", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload timings of the other configurations")
    args = ap.parse_args(argv)
    if args.warmup < 3:  # at least 3 warm-up steps; the JSON line reports the count used
        print(f"bench: --warmup {args.warmup} raised to 3", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
