"""Benchmark of the MSA decode step on GB300.

One step = one decode pass over a batch: insert the step's new K/V/index-key
tokens (with quantisation), score every candidate block, select the top
blocks, run split-K sparse GQA and its combine. The headline workload is the
largest configuration: batch 64 with contexts drawn from 8K to 128K tokens,
1 query token, 64/4/4 heads, FP8 index keys, bf16 KV, top-16 blocks. The line
then carries, under ``configs``, the same measurements for batch 32 x 32K,
batch 32 x 64K with 8 speculative positions, and batch 16 x 256K with NVFP4
K/V (``--configs``).

Prints one JSON line (rank 0). ``value`` is query-tokens/s over all ranks with
the inputs already resident in HBM; ``e2e`` is the same metric through the
public API with the per-step inputs copied from pinned host memory and the
output copied back inside the timed region. By default the L2 is not flushed:
each step reads several hundred MB (every index key of every request plus the
selected KV pages), far more than the 129 MB L2; ``--flush read|write`` adds a
512 MB read or write before every step. ``--impl reference`` times the fp64
CPU oracle instead, on a bounded sample of the same workload.

Multi-GPU (torchrun): every rank runs its own full copy of the workload (the
requests are independent; no data-path collective), so scaling is weak and
``value`` sums the query tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MSA decode query-tokens/s at 1 GB300; achieved HBM GB/s vs peak per kernel"
FALLBACK_HBM_GBS = 6800.0

# ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, keyed by kernel,
# workload and the hash of the kernel's sources (comments and blank space left
# out) when it was measured: a changed kernel reports null until it is measured
# again. Summaries: profiles/.
NCU_TRAFFIC = {
    ("index_score", "ragged", "2752585a1a31559d"): 2316357120 + 973312,
    ("sparse_gqa", "ragged", "9279da445860967d"): 270273024 + 555008,
    ("index_score", "b32_32k", "2752585a1a31559d"): 551655680 + 210688,
    ("sparse_gqa", "b32_32k", "9279da445860967d"): 134991104 + 344320,
    ("index_score", "spec8", "2752585a1a31559d"): 1105795328 + 1702144,
    ("sparse_gqa", "spec8", "9279da445860967d"): 886477312 + 436736,
    ("index_score", "nvfp4_256k", "2752585a1a31559d"): 2213771520 + 564480,
    ("sparse_gqa", "nvfp4_256k", "9279da445860967d"): 19318272 + 0,
}

# The headline workload (the largest configuration on one GPU: batch 64, ragged
# 8K-128K contexts) and the further configurations measured after it.
DEFAULT_WORKLOAD = "ragged"
DEFAULT_CONFIGS = "b32_32k,spec8,nvfp4_256k"


def _code_only(text):
    """The source without its comments and blank space, so that a comment edit
    leaves a measured kernel's key unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def _src_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_sparse_attention_07_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def workload_desc(w):
    ctx = f"context {w.ctx}" if w.ctx else f"context U[{w.ctx_range[0]},{w.ctx_range[1]}]"
    return (f"msa_decode_{w.name}: batch {w.batch}, {ctx}, q_len {w.q_len}, {w.n_heads} q / {w.n_kv_heads} kv / "
            f"{w.n_idx_heads} index heads, head_dim {w.head_dim}, block {w.block_size}, top-{w.topk} incl. local, "
            f"{ {'fp8': 'FP8 E4M3', 'nvfp4': 'NVFP4', 'f32': 'fp32'}[w.idx_dtype]} index keys, {w.kv_dtype} KV")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------- rank logic --
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_seconds: float, local_units: int, world: int, device=None):
    """Max time and summed units over ranks (identity for one rank)."""
    if world == 1:
        return local_seconds, local_units
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), int(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        """Starts sampling and returns once the first sample has arrived, so that
        the sampler's start-up does not overlap the timed region."""
        self.first = ""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        import select
        ready, _, _ = select.select([self.proc.stdout], [], [], 5.0)
        if ready:
            self.first = self.proc.stdout.readline()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        out = self.first + out
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), hw=parts[5], hwt=parts[6], swt=parts[7],
                                 pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = sorted({name for r in rows for name, key in (("hw_slowdown", "hw"),
                                                              ("hw_thermal_slowdown", "hwt"),
                                                              ("sw_thermal_slowdown", "swt"),
                                                              ("sw_power_cap", "pcap"))
                          if r[key].lower() == "active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- byte models --
def index_bytes(dw):
    """Algorithmic bytes of one index-score launch: every scored block's FP8 keys and
    per-token scales for all index heads, the index queries, the score rows."""
    w = dw.w
    units = sum(max(0, (int(L) - 1) // w.block_size) for L in dw.lens)
    per_token_head = {"fp8": w.head_dim + 4, "nvfp4": w.head_dim // 2 + w.head_dim // 16,
                      "f32": 4 * w.head_dim}[w.idx_dtype]
    per_unit = w.n_idx_heads * w.block_size * per_token_head
    q = dw.q_idx.numel() * dw.q_idx.element_size()
    scores = dw.scores.numel() * 4
    return units * per_unit + q + scores


def attention_bytes(dw, sel):
    """Algorithmic bytes of one sparse-GQA launch: the union over positions of the
    selected blocks' K and V for each (request, KV head), plus q and out."""
    w = dw.w
    per_tok = {"bf16": 2 * w.head_dim * 2, "fp8": 2 * w.head_dim,
               "nvfp4": 2 * (w.head_dim // 2 + w.head_dim // 16)}[w.kv_dtype]
    total = 0
    for bi in range(sel.shape[0]):
        L = int(dw.lens[bi])
        for g in range(sel.shape[2]):
            blocks = np.unique(sel[bi, :, g][sel[bi, :, g] >= 0])
            toks = sum(min(w.block_size, L - int(b) * w.block_size) for b in blocks)
            total += toks * per_tok
    return total + 2 * dw.q.numel() * 2


# ------------------------------------------------------------------ our arm --
class StepTimer:
    """Timed passes of one workload's decode step on one device (CUDA events on
    the launching stream)."""

    NAMES = ("insert", "index_score", "select", "sparse_gqa")

    def __init__(self, dw, stream, flush):
        self.dw, self.stream, self.flush = dw, stream, flush

    def steps(self, n, events):
        """n steps. events "step": records only at step boundaries, so the
        kernels launch back to back and overlap through programmatic dependent
        launch (the insert inside the index launch and the selection inside the
        attention launch where the workload's step does that,
        ``dw.merges_insert`` / ``dw.fuses_selection``); "index": the insert as
        its own launch, with events around the index-score kernel (its duration
        for the roofline; the events cut the overlap on both sides of it);
        "other": step boundaries only, the other selection composition;
        "unmerged": step boundaries only, the insert as its own launch; "all":
        four separate launches with events between every kernel (no overlap;
        the per-kernel breakdown)."""
        import torch
        dw, stream = self.dw, self.stream
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
        for s in range(n):
            self.flush(s)
            e = ev[s]
            e[0].record(stream)
            if dw.merges_insert and events in ("step", "other"):
                dw.insert_index_score()
            else:
                dw.insert_step_tokens()
                if events in ("index", "all"):
                    e[1].record(stream)
                dw.index_score()
                if events in ("index", "all"):
                    e[2].record(stream)
            fused = dw.fuses_selection if events in ("step", "index", "unmerged") else (
                not dw.fuses_selection if events == "other" else False)
            if fused:
                dw.select_attend()
            else:
                dw.select()
                if events == "all":
                    e[3].record(stream)
                dw.attend()
            e[4].record(stream)
        torch.cuda.synchronize(dw.device)
        step = [ev[s][0].elapsed_time(ev[s][4]) for s in range(n)]
        idx = [ev[s][1].elapsed_time(ev[s][2]) for s in range(n)] if events in ("index", "all") else None
        per = None
        if events == "all":
            per = {nm: [ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(n)] for i, nm in enumerate(self.NAMES)}
        return step, idx, per

    def launches_per_step(self):
        """[insert,] index, [select,] attention (the split-K combine is fused)."""
        return (1 if self.dw.merges_insert else 2) + (1 if self.dw.fuses_selection else 2)


def kernel_rooflines(args, dw, idx_ms, att_ms, peak, peak_kind, idx_step_ms):
    """The index kernel's and the attention kernel's achieved HBM GB/s: algorithmic
    bytes per launch over the mean launch duration timed live on this machine."""
    ib = index_bytes(dw)
    ab = attention_bytes(dw, dw.selected.cpu().numpy())
    name = dw.w.name if not args.batch else None
    traffic = NCU_TRAFFIC.get(("index_score", name, _src_hash("index_score.cu", "insert_rows.cuh", "msa_device.cuh")))
    att_traffic = NCU_TRAFFIC.get(("sparse_gqa", name, _src_hash("sparse_gqa.cu", "select_row.cuh", "msa_device.cuh")))
    idx = {"bound": "hbm", "kernel": "index_score", "achieved": ib / (idx_ms / 1e3) / 1e9, "peak": peak,
           "unit": "GB/s", "frac": ib / (idx_ms / 1e3) / 1e9 / peak, "peak_source": peak_kind, "traffic": traffic,
           "algorithmic_bytes_per_launch": ib, "avg_launch_ms": idx_ms,
           "timed_in": f"{args.steps} further steps (insert as its own launch) with events around the kernel "
                       f"({idx_step_ms:.4f} ms per step there)"}
    att = {"bound": "hbm", "kernel": "sparse_gqa", "achieved": ab / (att_ms / 1e3) / 1e9, "peak": peak,
           "unit": "GB/s", "frac": ab / (att_ms / 1e3) / 1e9 / peak, "peak_source": peak_kind,
           "algorithmic_bytes_per_launch": ab, "avg_launch_ms": att_ms, "traffic": att_traffic,
           "timed_in": "per-kernel breakdown pass (events between every kernel, selection as its own launch)"}
    return idx, att


def measure_config(args, name, dev, stream, flush, world, peak, peak_kind):
    """One further workload, measured like the headline's step (outside its timed
    region): value, ms per step, both kernels' roofline fractions, bytes."""
    import torch
    from block_sparse_attention_07_gb300 import synth
    from block_sparse_attention_07_gb300.workload import DeviceWorkload
    w = synth.WORKLOADS[name]
    t0 = time.perf_counter()
    dw = DeviceWorkload(w, dev)
    build_s = time.perf_counter() - t0
    tm = StepTimer(dw, stream, flush)
    for s in range(args.warmup):
        flush(s)
        dw.step()
    torch.cuda.synchronize(dev)
    assert dw.check_flags() == 0, f"device flags raised during warm-up ({name})"
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.15)
    barrier(world)
    step_ms, _, _ = tm.steps(args.steps, "step")
    barrier(world)
    idx_step_ms, idx_launch_ms, _ = tm.steps(args.steps, "index")
    clk = clocks.stop()
    _, _, per = tm.steps(min(args.steps, 50), "all")
    assert dw.check_flags() == 0, f"device flags raised ({name})"
    B, Q = len(dw.which), w.q_len
    tot_s, tot_units = aggregate(sum(step_ms) / 1e3, B * Q * args.steps, world, dev)
    idx, att = kernel_rooflines(args, dw, statistics.mean(idx_launch_ms), statistics.mean(per["sparse_gqa"]),
                                peak, peak_kind, statistics.mean(idx_step_ms))
    out = {"workload": workload_desc(w), "value": tot_units / tot_s, "unit": "query-tokens/s",
           "ms_per_step": statistics.mean(step_ms), "global_batch": B * world, "q_len": Q,
           "index_frac": idx["frac"], "sparse_gqa_frac": att["frac"],
           "index_bytes_per_launch": idx["algorithmic_bytes_per_launch"],
           "sparse_gqa_bytes_per_launch": att["algorithmic_bytes_per_launch"],
           "index_ms": idx["avg_launch_ms"], "sparse_gqa_ms": att["avg_launch_ms"],
           "index_traffic": idx["traffic"], "sparse_gqa_traffic": att["traffic"],
           "kernels_ms": {n: statistics.mean(v) for n, v in per.items()},
           "gpu_launches_per_step": tm.launches_per_step(), "clocks": clk,
           "setup_s": build_s}
    del tm, dw
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    import torch
    from block_sparse_attention_07_gb300 import synth
    from block_sparse_attention_07_gb300.workload import DeviceWorkload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = synth.scaled(w, batch=args.batch)
    dw = DeviceWorkload(w, dev)
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    B, Q = len(dw.which), w.q_len

    def flush(s):
        if args.flush == "write":
            flush_buf.fill_(float(s))
        elif args.flush == "read":
            torch.sum(flush_buf, dim=0, out=sink)

    tm = StepTimer(dw, stream, flush)
    for s in range(args.warmup):
        flush(s)
        dw.step()
    torch.cuda.synchronize(dev)
    assert dw.check_flags() == 0, "device flags raised during warm-up"

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.15)
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    step_ms, _, _ = tm.steps(args.steps, "step")
    barrier(world)
    wall = time.perf_counter() - wall0
    # the index-score kernel's launch duration (roofline), timed live over K more steps
    idx_step_ms, idx_launch_ms, _ = tm.steps(args.steps, "index")
    clk = clocks.stop()
    launches = args.steps * tm.launches_per_step()
    # the same steps in the other composition (selection fused or separate)
    other_step_ms, _, _ = tm.steps(args.steps, "other")
    # the same steps with the insert as its own launch
    unmerged_step_ms = tm.steps(args.steps, "unmerged")[0] if dw.merges_insert else None
    # per-kernel breakdown, outside the timed region, with an event between every kernel
    _, _, per = tm.steps(min(args.steps, 50), "all")
    local_s = sum(step_ms) / 1e3
    tot_s, tot_units = aggregate(local_s, B * Q * args.steps, world, dev)
    value = tot_units / tot_s

    # end to end through the public API: per-step inputs from pinned host memory,
    # output back to pinned host memory, inside the timed region.
    # (the per-step inputs — queries, new K/V/index keys, slots, block table,
    # lengths — sit in one device buffer, so they arrive in one copy)
    host_in = dw.step_inputs.cpu().pin_memory()
    host_out = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
    h2d = host_in.numel()
    d2h = host_out.numel() * host_out.element_size()

    def copies_and_step(st=None):
        dw.step_inputs.copy_(host_in, non_blocking=True)
        dw.step(st)
        host_out.copy_(dw.out, non_blocking=True)

    def e2e_eager():
        copies_and_step()
        torch.cuda.current_stream(dev).synchronize()

    # The library's calls (and the copies around them) captured once into a
    # CUDA graph, as a serving loop would run them: one replay per step.
    e2e_graph = dw.capture(copies_and_step)

    def e2e_replay():
        e2e_graph.replay()
        torch.cuda.current_stream(dev).synchronize()

    def e2e_timed(fn):
        for _ in range(args.warmup):
            fn()
        ms = []
        barrier(world)
        for s in range(args.steps):
            flush(s)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            ms.append((time.perf_counter() - t0) * 1e3)
        tot, _ = aggregate(sum(ms) / 1e3, 0, world, dev)
        return tot

    e2e_tot = e2e_timed(e2e_replay)
    e2e_eager_tot = e2e_timed(e2e_eager)
    del e2e_graph
    assert dw.check_flags() == 0, "device flags raised"

    def event_timed(fn, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for s in range(n):
            flush(s)
            ev[s][0].record(stream)
            fn()
            ev[s][1].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ev]

    # The same step replayed from one CUDA graph per step.
    graph = dw.capture(dw.step)
    for _ in range(args.warmup):
        graph.replay()
    graph_ms = event_timed(graph.replay, args.steps)
    del graph
    assert dw.check_flags() == 0, "device flags raised (graph replay)"
    # The fused QK-norm + RoPE + K/V/index insert of the step's tokens, alone and
    # as the first kernel of a step (in place of the plain insert).
    prologue_ms = pro_step_ms = None
    if w.idx_dtype != "f32":
        # per launch: 20 launches back to back from one captured graph (a launch
        # marshalled from Python takes longer on the host than the kernel on the GPU)
        dw.qk_norm_rope_insert()          # allocates its buffers outside the capture
        burst = dw.capture(lambda st: [dw.qk_norm_rope_insert(st) for _ in range(20)])
        for _ in range(args.warmup):
            burst.replay()
        prologue_ms = [t / 20 for t in event_timed(burst.replay, args.steps)]
        del burst

        def pro_step():
            dw.qk_norm_rope_insert()
            dw.index_score()
            if dw.fuses_selection:
                dw.select_attend()
            else:
                dw.select()
                dw.attend()
        pro_step_ms = event_timed(pro_step, args.steps)
        assert dw.check_flags() == 0, "device flags raised (fused norm/RoPE/insert)"
        dw.insert_step_tokens()           # restore the plain-insert cache contents
    # A layer that reuses this step's selection: K/V insert + sparse GQA only.
    reuse_ms = None
    if not args.no_layer_reuse:
        layer = DeviceWorkload.layer_like(dw, 1)
        for _ in range(args.warmup):
            layer.reuse_step(dw.selected)
        reuse_ms = event_timed(lambda: layer.reuse_step(dw.selected), args.steps)
        assert layer.check_flags() == 0, "device flags raised (reusing layer)"
        del layer

    peak, peak_kind = measured_peaks()
    ib = index_bytes(dw)
    per_step_mb = (ib + attention_bytes(dw, dw.selected.cpu().numpy())) / 1e6
    l2_note = {"none": f"not flushed: each step reads {per_step_mb:.0f} MB of inputs, more than the 129 MB L2",
               "read": "flushed by reading a 512 MB buffer before every step",
               "write": "flushed by writing a 512 MB buffer before every step"}[args.flush]
    roof, att_roof = kernel_rooflines(args, dw, statistics.mean(idx_launch_ms), statistics.mean(per["sparse_gqa"]),
                                      peak, peak_kind, statistics.mean(idx_step_ms))
    line = {
        "metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(step_ms), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8/bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": B * world, "q_len": Q, "l2": l2_note,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "kernels_ms": {n: statistics.mean(v) for n, v in per.items()},
        "selection_in_attention_launch": dw.fuses_selection,
        "insert_in_index_launch": dw.merges_insert,
        "insert_as_own_launch": (None if unmerged_step_ms is None else
                                 {"value": B * Q / (statistics.mean(unmerged_step_ms) / 1e3),
                                  "unit": "query-tokens/s", "ms_per_step": statistics.mean(unmerged_step_ms),
                                  "what": "the same step with the insert as its own launch"}),
        "other_composition": {"value": B * Q / (statistics.mean(other_step_ms) / 1e3), "unit": "query-tokens/s",
                              "ms_per_step": statistics.mean(other_step_ms),
                              "what": ("selection as its own launch" if dw.fuses_selection
                                       else "selection inside the attention launch")},
        "sparse_gqa_roofline": att_roof,
        "e2e": {"value": B * Q * args.steps * world / e2e_tot, "unit": "query-tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "what": "host wall clock per step: the step's inputs copied from pinned host memory, the library "
                        "calls, the output copied back, synchronised; copies and calls replayed from one "
                        "captured CUDA graph",
                "eager_value": B * Q * args.steps * world / e2e_eager_tot},
        "graph": {"value": B * Q / (statistics.mean(graph_ms) / 1e3), "unit": "query-tokens/s",
                  "ms_per_step": statistics.mean(graph_ms),
                  "what": "the same step replayed from one captured CUDA graph per step"},
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if prologue_ms is not None:
        line["qk_norm_rope_insert"] = {
            "ms_per_launch": statistics.mean(prologue_ms),
            "step_value": B * Q / (statistics.mean(pro_step_ms) / 1e3), "unit": "query-tokens/s",
            "step_ms": statistics.mean(pro_step_ms),
            "what": "fused RMSNorm + RoPE of the step's query/key/index projections and K/V/index-key insert "
                    "(ms_per_launch: 20 launches replayed from one graph); step_value: that kernel in place of "
                    "the plain insert, then score, select, attend"}
    if reuse_ms is not None:
        line["selection_reuse_layer"] = {
            "value": B * Q / (statistics.mean(reuse_ms) / 1e3), "unit": "query-tokens/s",
            "ms_per_step": statistics.mean(reuse_ms),
            "what": "a second layer (own q/K/V) reusing this step's block selection: K/V insert + sparse GQA, "
                    "no index keys, scoring or selection"}
    cfg_w = w
    del tm, dw
    torch.cuda.empty_cache()
    # The other workloads, each measured like the headline (after its timed region).
    names = [n for n in (args.configs.split(",") if args.configs not in ("", "none") else []) if n != args.workload]
    if names and not args.batch:
        line["configs"] = {n: measure_config(args, n, dev, stream, flush, world, peak, peak_kind) for n in names}
    if rank != 0:
        return None
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg_w, args.cpu_requests)
    return line


# ---------------------------------------------------------- oracle / CPU --
def cpu_baseline(w, n_requests, budget_s=20.0):
    """The fp64 oracle as it stands, single-threaded, on a bounded sample of requests."""
    from block_sparse_attention_07_gb300 import synth
    from oracle import run as orun
    lens = synth.seq_lens(w)
    kg = kv = synth.kv_scale(w)
    idx_g = float(np.float32(synth.NVFP4_IDX_SYNTH_GLOBAL)) if w.idx_dtype == "nvfp4" else 1.0
    spent, done = 0.0, 0
    for b in range(min(n_requests, w.batch)):
        req = synth.request(w, b, int(lens[b]))
        t0 = time.perf_counter()
        orun.run_request(req, int(lens[b]), w.topk, w.softmax_scale, w.block_size, w.idx_dtype, w.kv_dtype, kg, kv,
                         idx_global=idx_g)
        spent += time.perf_counter() - t0
        done += 1
        if spent > budget_s:
            break
    line = {"value": done * w.q_len / spent, "unit": "query-tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {w.batch} requests of the same workload, all stages, fp64 numpy, 1 thread",
            "seconds": spent}
    try:
        line["all_cores"] = cpu_all_cores(w)
    except Exception as e:                     # reported, never fatal to the GPU figures
        line["all_cores"] = {"error": f"{type(e).__name__}: {e}"}
    return line


def _oracle_worker(w, bs, barrier, out_q):
    """One spawned process: builds its requests, waits for the others, then
    runs them through the oracle (numpy with one BLAS thread)."""
    from block_sparse_attention_07_gb300 import synth
    from oracle import run as orun
    lens = synth.seq_lens(w)
    kg = synth.kv_scale(w)
    idx_g = float(np.float32(synth.NVFP4_IDX_SYNTH_GLOBAL)) if w.idx_dtype == "nvfp4" else 1.0
    reqs = [(b, synth.request(w, b, int(lens[b]))) for b in bs]
    barrier.wait(timeout=900)
    t0 = time.monotonic()
    for b, req in reqs:
        orun.run_request(req, int(lens[b]), w.topk, w.softmax_scale, w.block_size, w.idx_dtype, w.kv_dtype, kg, kg,
                         idx_global=idx_g)
    out_q.put((t0, time.monotonic(), len(reqs)))


def cpu_all_cores(w, mem_budget=32 << 30):
    """The same oracle on every host core: one spawned process per request (at
    most one per core, and few enough that their fp64 working sets, about 32 KB
    per context token, fit in mem_budget); wall clock from the first start to
    the last finish, request generation excluded."""
    import multiprocessing as mp
    from block_sparse_attention_07_gb300 import synth
    ctx = mp.get_context("spawn")
    max_ctx = int(synth.seq_lens(w).max())
    C = max(1, min(os.cpu_count() or 1, w.batch, mem_budget // max(1, max_ctx * 32 * 1024)))
    barrier = ctx.Barrier(C)
    q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(w, [k], barrier, q), daemon=True) for k in range(C)]
    for pr in procs:
        pr.start()
    import queue as _queue
    res = []
    deadline = time.monotonic() + 1800
    try:
        while len(res) < C:
            try:
                res.append(q.get(timeout=2))
            except _queue.Empty:
                if any(pr.exitcode not in (None, 0) for pr in procs) or time.monotonic() > deadline:
                    raise RuntimeError("an oracle process failed or ran out of time")
    finally:
        for pr in procs:
            pr.join(timeout=60)
            if pr.is_alive():
                pr.terminate()
    wall = max(r[1] for r in res) - min(r[0] for r in res)
    n = sum(r[2] for r in res)
    return {"value": n * w.q_len / wall, "unit": "query-tokens/s", "cores": C, "kind": "oracle",
            "sample": f"{n} of {w.batch} requests, one spawned process each (fp64 numpy, 1 BLAS thread per "
                      f"process) on {os.cpu_count()} host cores",
            "wall_s": wall}


def run_reference(args, world, rank):
    from block_sparse_attention_07_gb300 import synth
    from oracle import run as orun
    if rank != 0:
        return None
    w = synth.WORKLOADS[args.workload]
    lens = synth.seq_lens(w)
    kg = kv = synth.kv_scale(w)
    idx_g = float(np.float32(synth.NVFP4_IDX_SYNTH_GLOBAL)) if w.idx_dtype == "nvfp4" else 1.0
    reqs = {}

    def one(s):
        b = s % w.batch
        if b not in reqs:
            reqs[b] = synth.request(w, b, int(lens[b]))
        t0 = time.perf_counter()
        orun.run_request(reqs[b], int(lens[b]), w.topk, w.softmax_scale, w.block_size, w.idx_dtype, w.kv_dtype,
                         kg, kv, idx_global=idx_g)
        return time.perf_counter() - t0

    for s in range(args.warmup):
        one(s)
    times = [one(s) for s in range(args.steps)]
    value = len(times) * w.q_len / sum(times)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": w.batch, "q_len": w.q_len,
                   "step": "one request of the batch per step (bounded sample), all stages"},
        "cpu_baseline": {"value": value, "unit": "query-tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "one request of the workload per step, fp64 numpy, 1 thread"},
        "e2e": {"value": value, "unit": "query-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--configs", default=DEFAULT_CONFIGS,
                    help="further workloads measured after the headline, comma-separated ('none' for none)")
    ap.add_argument("--batch", type=int, default=0, help="override the batch size (smaller profiling cases)")
    ap.add_argument("--flush", default="none", choices=("none", "read", "write"),
                    help="L2 treatment before each timed step: none (per-step inputs exceed L2), "
                         "read a 512 MB buffer, or write one")
    ap.add_argument("--cpu-requests", type=int, default=6)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-layer-reuse", action="store_true",
                    help="skip building a second layer for the selection-reuse timing")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return 0
            world = 1
        else:
            import torch
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
    line = run_reference(args, world, rank) if args.impl == "reference" else run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
