#!/usr/bin/env python
"""Benchmark of the sparse-MLA decode hot path on GB300.

One step = one pass of the whole path over one decode batch: the
deterministic top-k over the indexer scores, then sparse MLA attention
(split kernel + fixed-order combine) over the selected entries of the paged
latent KV cache. Workload: the TP2-shaped decode batch (32 requests, 64
heads, contexts uniform in [4096, 32768], top-k 2048, bf16 latent KV in
64-entry pages, d_qk 576, d_v 512), seeded synthetic data.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0. `value` is decode tokens/s of the whole job
(one token = one request row per step, all heads), measured with CUDA events
around exactly K steps (after exactly W warm-up steps) replayed from CUDA
graphs (a run of up to 512 steps is one graph), inputs resident in HBM; a
spin kernel queued ahead of the start event keeps the host's launch latency
out of the timed region. Four independent input sets rotate so the
gathered KV (4 x 75.5 MB) exceeds the 129 MB L2 between reuses. The same step
keeps running for a second after the timed region so that the nvidia-smi
clock record holds samples under this load. `e2e` repeats the step through
the public API with pinned host buffers: the step's inputs are copied
host->device, and out, lse and idx are read back, inside the timed region,
with four steps in flight on four streams (copies run at about 200 GB/s, so
one step's 9 MB of transfers take about as long as its kernels); it runs at
least 200 steps and 0.5 s. Independent steps' kernels then overlap too, so
`e2e` can exceed the single-stream `value`. The default run also measures
the TP1 FP8 decode batch and the chunked-prefill chunk (`other_configs`, each
with its own roofline blocks). Under torchrun every rank runs its own batch
(rows are independent: weak scaling, no collective on the data path).

`--impl reference` times the CPU oracle (test infrastructure, the
reference arm of this comparison) on bounded samples of the same workload.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "tp2_decode"
WORKLOAD_DESCS = {
    "tp2_decode": ("TP2-shaped sparse MLA decode: batch 32, 64 heads, contexts uniform int in "
                   "[4096, 32768], topk 2048, bf16 paged latent KV (page 64, random block-table "
                   "permutation), d_qk 576 (512+64), d_v 512, fp32 N(0,1) scores, scale 1/sqrt(576)"),
    "tp1_fp8_decode": ("TP1 sparse MLA decode at scale: batch 128, 128 heads, contexts uniform int in "
                       "[8192, 131072], topk 2048, FP8 e4m3 latent KV (fp32 scale per 128 dims) + "
                       "bf16 rope, page 64, fp32 N(0,1) scores"),
    "chunked_prefill": ("chunked sparse MLA prefill: 1 request, 4096 query tokens at positions "
                        "61440..65535 of a 65536 context, causal, topk 2048, 128 heads, bf16 KV, "
                        "fp32 N(0,1) scores"),
    "tp2_decode_swa": ("TP2-shaped sparse MLA decode over [top-k 2048 compressed entries || a "
                       "128-entry sliding window of a second pool] with per-head attention sinks: "
                       "batch 32, 64 heads, contexts uniform int in [4096, 32768], bf16 KV, fp32 "
                       "N(0,1) scores"),
    "fp8_cache_write": ("FP8 KV cache write: 65536 new bf16 latent rows (576 dims) quantised to the "
                        "656-byte E4M3 layout (fp32 scale per 128 dims, bf16 rope) at randomly "
                        "permuted slots of a 1024-page pool"),
    "tp2_mtp4_decode": ("MTP4 sparse MLA decode: 32 requests x 5 query tokens (1 target + 4 draft), "
                        "64 heads, request lengths uniform int in [4096, 32768], token j of a "
                        "request sees seq_len - 4 + j positions, topk 2048, bf16 KV, fp32 N(0,1) "
                        "scores"),
}
METRIC = "sparse-MLA decode tokens/s and top-k rows/s on 1 GB300; % of roofline"
N_SETS = 4
E2E_SLOTS = 4   # steps in flight end to end: 2 -> 500 K, 3 -> 708 K, 4 -> 816 K, 6 -> 786 K tokens/s measured
E2E_MIN_STEPS = 200
E2E_MIN_SECS = 0.5
CLOCK_WINDOW_S = 1.0
SPIN_CYCLES = 200_000   # about 0.1 ms at 2 GHz, before the start event
CPU_BASELINE_S = 10.0
REFERENCE_CAP_S = 120.0
EXTRA_STEPS = {"tp1_fp8_decode": 100, "chunked_prefill": 20}
HBM_CONTRACT_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=400)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the TP1 FP8 decode and chunked-prefill lines of the default run")
    ap.add_argument("--e2e-slots", type=int, default=E2E_SLOTS,
                    help="steps in flight in the end-to-end loop (each its own stream and buffers)")
    ap.add_argument("--sets", type=int, default=N_SETS,
                    help="rotating input sets (profiling runs use 1 to stay small)")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_DESCS) + ["tp2_indexer"],
                    default=WORKLOAD,
                    help="the TP2 decode batch is the headline; the others are for the record")
    ap.add_argument("--rows", type=int, default=None,
                    help="keep only the first N rows of a decode or prefill workload (profiling "
                         "captures of a reduced case)")
    args = ap.parse_args()
    if args.e2e_slots < 1:
        ap.error("--e2e-slots must be at least 1")
    if args.steps < 1 or args.warmup < 0 or args.sets < 1:
        ap.error("--steps must be at least 1, --warmup at least 0, --sets at least 1")
    return args


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def max_over_ranks(x, world):
    """Max of a float over ranks (the job finishes when the slowest does)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def kernel_source_sha():
    """Hash of the kernel sources' code: comments and blank lines are dropped
    first, so editing a comment does not orphan the committed ncu counters."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "invariant_sparse_mla_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"(?m)^\s*//.*$", "", text)        # whole-line comments
        text = re.sub(r"(?m)\s+//[^\"\n]*$", "", text)    # trailing comments (no quote after //)
        code = "\n".join(l.rstrip() for l in text.splitlines() if l.strip())
        h.update(name.encode())
        h.update(code.encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` ("attention" or "topk") on
    `workload` from the committed ncu summary, if it was taken on the current
    kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("source_sha") != kernel_source_sha():
            return None
        rec = t["records"].get(f"{workload}:{kernel}")
        return int(rec["bytes_per_launch"]) if rec else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id is not None:
            cmd += ["-i", str(self.gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.5)   # nvidia-smi start-up

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, smax, reasons = [], None, set()
        for ts, line in self.lines:
            if not (t0 <= ts <= t1 + 0.06):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for_smi(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids):
            return ids[local]
    return local


def algorithmic_bytes(case, idx):
    """Bytes the path must move at minimum (no re-reads, no workspaces).

    top-k: every in-range score read once (4 B) + idx written (4 B each).
    attention: every distinct selected KV row read once (1152 B bf16 or
    656 B FP8; prefill tokens of one request share rows) + q read + out
    (bf16) and lse written + idx read. FLOPs: 2 * H * (576 + 512) per valid
    selected entry.
    """
    import torch
    L = (case.row_ends - case.row_starts).clamp(min=0).to(torch.int64)
    topk = 4 * int(L.sum()) + 4 * idx.numel()
    valid_mask = idx >= 0
    valid = int(valid_mask.sum())
    key = case.row_req.to(torch.int64)[:, None] * (1 << 32) + idx.to(torch.int64)
    distinct = int(torch.unique(key[valid_mask]).numel())
    row_bytes = 1152 if case.kv_dtype == "bf16" else 656
    R, H = case.q.shape[0], case.q.shape[1]
    attn = distinct * row_bytes + case.q.numel() * 2 + R * H * 512 * 2 + R * H * 4 + idx.numel() * 4
    if getattr(case, "win", None) is not None:   # window entries: distinct per row
        wvalid = int(((case.win[2] >= 0) & (case.win[2] < case.win[3][:, None])).sum())
        attn += wvalid * row_bytes + case.win[2].numel() * 4
        valid += wvalid
    flops = 2 * valid * H * (576 + 512)
    return topk, attn, flops


def job_value(world, rows_per_rank, steps, secs):
    """Whole-job throughput: the rows all ranks processed in `steps` steps,
    over the slowest rank's time (`secs`, already the max over ranks)."""
    return world * rows_per_rank * steps / secs


def build_sets(wl, n_sets, rank, device, rows=None):
    """`n_sets` independent input sets of workload `wl` (shifted seeds per
    set and rank; set 0 of rank 0 is the workload's own seed), each with its
    idx, out, lse and workspace buffers."""
    import torch
    import invariant_sparse_mla_gb300 as ds
    from synthetic import WORKLOADS, decode_case, prefill_case, mtp_case, window_case, _uniform_ints
    w = WORKLOADS[wl]
    sets = []
    for s in range(n_sets):
        seed = w["seed"] + 1000 * rank + 17 * s
        own = s == 0 and rank == 0
        if w["kind"] in ("decode", "decode_swa"):
            ctx = _uniform_ints(w["ctx"][0], w["ctx"][1], w["B"], w["seed"] if own else seed)
            ctx = ctx[:rows] if rows else ctx
            c = decode_case(wl, ctx, w["H"], w["k"], w["kv"], w["seed"] if own else seed,
                            w["scores"], stride=w["stride"], device=device)
            if w["kind"] == "decode_swa":
                # The window cache holds each request's last swa_width tokens.
                c.win = window_case([min(n, w["swa_width"]) for n in ctx], w["swa_width"], w["kv"],
                                    seed + 7, device=device)
                c.sink = torch.randn(w["H"], generator=torch.Generator().manual_seed(seed)).to(device)
        elif w["kind"] == "mtp":
            lens = _uniform_ints(w["ctx"][0], w["ctx"][1], w["B"], w["seed"] if own else seed)
            c = mtp_case(wl, lens, w["next_n"], w["H"], w["k"], w["kv"], w["seed"] if own else seed,
                         w["scores"], stride=w["stride"], device=device)
        else:
            T = min(rows, w["T"]) if rows else w["T"]
            c = prefill_case(wl, w["ctx"], w["first_pos"], T, w["H"], w["k"], w["kv"],
                             w["seed"] if own else seed, device=device)
        R, H, k = c.q.shape[0], c.H, c.k
        c.idx = torch.empty((R, k), dtype=torch.int32, device=device)
        c.out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=device)
        c.lse = torch.empty((R, H), dtype=torch.float32, device=device)
        c.ws = torch.empty(ds.swa_workspace_size(R, H, k, w.get("swa_width", 0)),
                           dtype=torch.uint8, device=device)
        sets.append(c)
    return sets


def make_calls(ds, kind, stream):
    """The public calls of one step: top-k, then the attention call."""
    import torch
    tk_ws = {}   # one top-k workspace per shape: the calls run in order on one stream

    def topk(c):
        shape = (c.scores.shape[0], c.scores.shape[1], c.k)
        if shape not in tk_ws:
            tk_ws[shape] = torch.empty(max(ds.topk_workspace_size(*shape), 1), dtype=torch.uint8,
                                       device=c.scores.device)
        ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k, idx_out=c.idx, stream=stream,
                        workspace=tk_ws[shape])

    def decode(c):
        if kind == "decode":
            ds.sparse_mla_decode(c.q, c.kv_pages, c.kv_dtype, c.block_table, c.idx, c.lens,
                                 c.scale, out=c.out, lse=c.lse, workspace=c.ws, stream=stream)
        elif kind == "decode_swa":
            ds.sparse_mla_decode_swa(c.q, c.kv_pages, c.kv_dtype, c.block_table, c.idx, c.lens,
                                     c.scale, swa_pages=c.win[0], swa_block_table=c.win[1],
                                     swa_idx=c.win[2], swa_lens=c.win[3], attn_sink=c.sink,
                                     out=c.out, lse=c.lse, workspace=c.ws, stream=stream)
        else:
            ds.sparse_mla_prefill(c.q, c.kv_pages, c.kv_dtype, c.block_table, c.row_req, c.idx,
                                  c.lens, c.scale, out=c.out, lse=c.lse, workspace=c.ws,
                                  stream=stream)

    def step(c):
        topk(c)
        decode(c)

    return topk, decode, step


class Replayer:
    """Runs any number of steps exactly, cycling through the input sets in
    order. A whole pass over the sets replays one CUDA graph of all of them,
    captured once per starting set (so consecutive steps keep their
    programmatic-launch overlap wherever a run starts); the rest replay one
    graph per set."""

    MAX_RUN_GRAPH = 512   # a timed run of at most this many steps is one graph

    def __init__(self, stream, fn, sets):
        import torch
        self.stream = stream
        self.sets = sets

        def capture(cases):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in cases:
                    fn(c)
            return g

        self.capture = capture
        n = len(sets)
        self.cycles = [capture(sets[k:] + sets[:k]) for k in range(n)]
        self.single = [capture([c]) for c in sets]
        self.n = n
        self.pos = 0

    def run(self, steps):
        import torch
        with torch.cuda.stream(self.stream):   # replay() launches on the current stream
            while steps >= self.n:
                self.cycles[self.pos].replay()
                steps -= self.n
            for _ in range(steps):
                self.single[self.pos].replay()
                self.pos = (self.pos + 1) % self.n

    def timed(self, steps):
        """Seconds for `steps` steps, by CUDA events on the launching stream.
        Up to MAX_RUN_GRAPH steps are captured (before the timed region) as
        one graph of exactly those steps, so the region holds one launch."""
        import torch
        run_graph = None
        if steps <= self.MAX_RUN_GRAPH:
            order = [self.sets[(self.pos + i) % self.n] for i in range(steps)]
            run_graph = self.capture(order)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        # A short spin kernel ahead of the start event keeps the GPU busy
        # while the host queues the event and the graph, so the timed region
        # holds the steps and not the host's launch latency.
        with torch.cuda.stream(self.stream):
            torch.cuda._sleep(SPIN_CYCLES)
        e0.record(self.stream)
        if run_graph is not None:
            with torch.cuda.stream(self.stream):
                run_graph.replay()
            self.pos = (self.pos + steps) % self.n
        else:
            self.run(steps)
        e1.record(self.stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3


def per_call_seconds(rep, calls):
    """Mean seconds per call over `calls` calls (at least one whole pass)."""
    n = max(rep.n, calls // rep.n * rep.n)
    rep.run(rep.n)   # warm
    return rep.timed(n) / n


def roofline_block(kind, bytes_or_flops, secs, hbm, tflops, peak_kind, kernel, traffic=None):
    if kind == "hbm":
        gbs = bytes_or_flops / secs / 1e9
        return {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(gbs / hbm, 4), "peak_kind": f"{peak_kind} HBM copy",
                "traffic": traffic, "algorithmic_bytes": round(bytes_or_flops)}
    tf = bytes_or_flops / secs / 1e12
    return {"bound": "tensor", "kernel": kernel, "achieved": round(tf, 1), "peak": tflops,
            "unit": "TFLOP/s", "frac": round(tf / tflops, 4),
            "peak_kind": f"{peak_kind} bf16 dense (burst)", "traffic": traffic,
            "algorithmic_flops": round(bytes_or_flops)}


def contract_fraction(attn_bytes, attn_flops, secs, tflops):
    """Fraction of the contract roofline max(bytes / 8 TB/s, flops / bf16 peak)."""
    roof_s = max(attn_bytes / (HBM_CONTRACT_GBS * 1e9), attn_flops / (tflops * 1e12))
    return round(roof_s / secs, 4)


def measure_extra(ds, wl, dev, stream, steps, warmup):
    """Another workload on this GPU, for the record: one input set (its
    per-step traffic alone exceeds L2), `warmup` then `steps` steps replayed
    from CUDA graphs, and the two calls timed alone. Returns a dict for the
    JSON line."""
    import torch
    from synthetic import WORKLOADS
    w = WORKLOADS[wl]
    sets = build_sets(wl, 1, 0, dev)
    topk, decode, step = make_calls(ds, w["kind"], stream)
    with torch.cuda.stream(stream):
        for _ in range(2):
            step(sets[0])
    stream.synchronize()
    rs, rt, rd = (Replayer(stream, f, sets) for f in (step, topk, decode))
    rs.run(warmup)
    secs = rs.timed(steps)
    topk_s = per_call_seconds(rt, steps)
    dec_s = per_call_seconds(rd, steps)
    c = sets[0]
    tb, ab, fl = algorithmic_bytes(c, c.idx)
    hbm, tflops, peak_kind = load_peaks()
    R = c.q.shape[0]
    res = {"workload": WORKLOAD_DESCS[wl], "rows": R, "heads": c.H, "topk": c.k,
           "kv_dtype": c.kv_dtype, "steps": steps, "warmup": warmup,
           "step_us": round(secs / steps * 1e6, 3), "tokens_per_s": round(R * steps / secs, 1),
           "topk_us": round(topk_s * 1e6, 3), "attention_us": round(dec_s * 1e6, 3),
           "roofline_topk": roofline_block("hbm", tb, topk_s, hbm, tflops, peak_kind,
                                           "ds_topk_per_row", ncu_traffic(wl, "topk")),
           "roofline": roofline_block("tensor", fl, dec_s, hbm, tflops, peak_kind,
                                      "sparse_mla attention (split + combine)",
                                      ncu_traffic(wl, "attention")),
           "attention_algorithmic_bytes": round(ab),
           "frac_of_contract_roofline": contract_fraction(ab, fl, dec_s, tflops),
           "l2": "1 input set; its per-step traffic exceeds the 129 MB L2"}
    del rs, rt, rd, sets, c
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def measure_indexer(ds, dev, stream, steps, warmup):
    """The indexer in front of the TP2 decode batch: its logits (MQA scores
    over the paged bf16 key cache, 64 heads x 128 dims) and the top-k 2048
    over them, replayed from CUDA graphs. Roofline of the logits kernel
    against HBM: every key row read once, q and w read, logits written."""
    import torch
    from synthetic import indexer_workload, INDEXER_WORKLOADS
    w = INDEXER_WORKLOADS["tp2_indexer"]
    c = indexer_workload("tp2_indexer", device=dev)
    R, H = c.q.shape[0], c.q.shape[1]
    logits = torch.empty((R, 64 * c.block_table.shape[1]), dtype=torch.float32, device=dev)
    idx = torch.empty((R, w["k"]), dtype=torch.int32, device=dev)
    starts = torch.zeros_like(c.lens)

    def lg(_):
        ds.indexer_logits(c.q, c.w, c.k_pages, c.block_table, c.lens, logits=logits, stream=stream)

    def tk(_):
        ds.topk_per_row(logits, starts, c.lens, w["k"], idx_out=idx, stream=stream)

    def step(x):
        lg(x)
        tk(x)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step(None)
    stream.synchronize()
    rs, rl, rt = (Replayer(stream, f, [None]) for f in (step, lg, tk))
    rs.run(warmup)
    secs = rs.timed(steps)
    lg_s = per_call_seconds(rl, steps)
    tk_s = per_call_seconds(rt, steps)
    positions = int(c.lens.clamp(min=0).sum())
    key_bytes = positions * 128 * 2
    lg_bytes = key_bytes + c.q.numel() * 2 + c.w.numel() * 4 + positions * 4
    lg_flops = 2 * H * 128 * positions
    tk_bytes = positions * 4 + idx.numel() * 4
    hbm, tflops, peak_kind = load_peaks()
    res = {"workload": ("indexer logits (64 heads x 128 dims, bf16 paged keys, fp32 head weights) "
                        "then top-k 2048, over the TP2 decode batch's 32 rows of contexts "
                        "uniform in [4096, 32768]"),
           "rows": R, "heads": H, "positions": positions, "steps": steps, "warmup": warmup,
           "step_us": round(secs / steps * 1e6, 3), "rows_per_s": round(R * steps / secs, 1),
           "logits_us": round(lg_s * 1e6, 3), "topk_us": round(tk_s * 1e6, 3),
           "roofline": roofline_block("hbm", lg_bytes, lg_s, hbm, tflops, peak_kind,
                                      "indexer_kernel", ncu_traffic("tp2_indexer", "logits")),
           "logits_tflops": round(lg_flops / lg_s / 1e12, 1),
           "roofline_topk": roofline_block("hbm", tk_bytes, tk_s, hbm, tflops, peak_kind,
                                           "ds_topk_per_row", None),
           "l2": f"one input set; {key_bytes / 1e6:.0f} MB of keys per step vs 129 MB L2"}
    del rs, rl, rt, c, logits, idx
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


EXTRA_WORKLOADS = ("tp1_fp8_decode", "chunked_prefill")


def run_ours(args, rank, world, local):
    import torch
    import invariant_sparse_mla_gb300 as ds
    from synthetic import WORKLOADS

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = args.workload
    w = WORKLOADS[wl]
    n_sets = args.sets
    sets = build_sets(wl, n_sets, rank, dev, rows=args.rows)
    R, H, k = sets[0].q.shape[0], sets[0].H, sets[0].k
    stream = torch.cuda.Stream(device=dev)
    topk, decode, step = make_calls(ds, w["kind"], stream)

    # Eager calls first (they also resolve lazy module loading), then graphs.
    with torch.cuda.stream(stream):
        for c in sets:
            step(c)
    stream.synchronize()
    rep_step = Replayer(stream, step, sets)
    rep_topk = Replayer(stream, topk, sets)
    rep_dec = Replayer(stream, decode, sets)

    steps, warmup = args.steps, args.warmup
    rep_step.run(warmup)
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_id_for_smi(local))
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    secs = rep_step.timed(steps)
    # The timed region of a short run is far below nvidia-smi's sampling
    # period: the same step keeps running for another second so the clock
    # record holds samples taken under this load.
    t_load = time.time()
    while time.time() - t_load < CLOCK_WINDOW_S:
        rep_step.run(max(n_sets, 256 // n_sets * n_sets))
        stream.synchronize()
    t1 = time.time()
    barrier(world)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    clocks["window"] = (f"the timed region plus {t1 - t_load:.2f} s of the same step "
                        "replayed right after it")
    secs = max_over_ranks(secs, world)

    # Per-call averages (graphs of one call per input set).
    n_k = max(8 * n_sets, min(500, steps))
    topk_s = per_call_seconds(rep_topk, n_k)
    dec_s = per_call_seconds(rep_dec, n_k)

    # Work per step (mean over the input sets).
    tb, ab, fl = zip(*[algorithmic_bytes(c, c.idx) for c in sets])
    topk_bytes, attn_bytes, attn_flops = (sum(tb) / n_sets, sum(ab) / n_sets, sum(fl) / n_sets)

    # End to end through the public API with pinned host buffers.
    e2e = None if (args.no_e2e or w["kind"] != "decode") else run_e2e(
        ds, sets, stream, dev, min_steps=E2E_MIN_STEPS, min_secs=E2E_MIN_SECS,
        n_slots=args.e2e_slots, world=world)

    hbm, tflops, peak_kind = load_peaks()
    value = job_value(world, R, steps, secs)
    ms_per_step = secs / steps * 1e3
    launches = steps * 3  # top-k + split + combine
    tensor_bound = attn_flops / (tflops * 1e12) > attn_bytes / (hbm * 1e9)
    frac_contract = contract_fraction(attn_bytes, attn_flops, dec_s, tflops)
    if tensor_bound:
        roof = roofline_block("tensor", attn_flops, dec_s, hbm, tflops, peak_kind,
                              "sparse_mla attention (split + combine)", ncu_traffic(wl, "attention"))
    else:
        roof = roofline_block("hbm", attn_bytes, dec_s, hbm, tflops, peak_kind,
                              "sparse_mla_decode (split + combine)", ncu_traffic(wl, "attention"))
    roof["frac_of_contract_roofline"] = frac_contract
    line = {
        "metric": METRIC if wl == WORKLOAD else METRIC + f" [{wl}]",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if sets[0].kv_dtype == "bf16" else "bf16 (FP8 e4m3 KV dequantised to bf16)",
        "data": "synthetic (seeded; random-init latent KV, N(0,1) scores)",
        "config": {"workload": WORKLOAD_DESCS[wl], "global_batch": R * world, "heads": H, "topk": k,
                   "parallelism": f"replicas x{world} (rows independent, no collective)",
                   "l2": f"{n_sets} rotating input sets, {n_sets * attn_bytes / 1e6:.0f} MB of "
                         f"gathered KV vs 129 MB L2", "cuda_graph": True},
        "topk_rows_per_s": round(world * R / topk_s, 1),
        "decode_tokens_per_s": round(world * R / dec_s, 1),
        "topk_us": round(topk_s * 1e6, 3),
        "decode_us": round(dec_s * 1e6, 3),
        "roofline": roof,
        "roofline_topk": roofline_block("hbm", topk_bytes, topk_s, hbm, tflops, peak_kind,
                                        "ds_topk_per_row", ncu_traffic(wl, "topk")),
        "e2e": e2e,
        "attention_tflops": round(attn_flops / dec_s / 1e12, 1),
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if args.rows:
        line["config"]["rows_kept"] = args.rows
    if rank == 0 and not args.no_cpu_baseline and world == 1 and wl == WORKLOAD:
        line["cpu_baseline"] = cpu_baseline(sets[0], budget_s=CPU_BASELINE_S)
    if wl == WORKLOAD and not args.no_extra and not args.rows:
        del rep_step, rep_topk, rep_dec, sets
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["other_configs"] = {x: measure_extra(ds, x, dev, stream, EXTRA_STEPS[x], 3)
                                 for x in EXTRA_WORKLOADS}
        line["other_configs"]["tp2_indexer_topk"] = measure_indexer(ds, dev, stream, 200, 3)
    return line


def run_e2e(ds, sets, stream, dev, min_steps, min_secs, world, n_slots=E2E_SLOTS):
    """Host -> device inputs, the two calls, device -> host results, every step.

    A serving loop: each step's inputs (scores, row bounds, q, block table,
    lengths) are packed in one pinned host buffer and copied with one H2D copy;
    idx, out and lse land in one device buffer read back with one D2H copy.
    `n_slots` steps are in flight (slots used in turn, each on its own stream),
    so one step's transfers overlap another's kernels. Before a slot is reused
    the host waits for that slot's previous download, so every step's result
    is on the host within the timed region. The loop runs at least
    `min_steps` steps and at least `min_secs` seconds (checked between steps).
    """
    import torch
    in_names = ("scores", "row_starts", "row_ends", "q", "block_table", "lens")
    out_names = ("idx", "out", "lse")

    def layout(c, names):
        off, spans = 0, {}
        for n in names:
            t = getattr(c, n)
            nb = t.numel() * t.element_size()
            spans[n] = (off, nb, t.dtype, tuple(t.shape))
            off += (nb + 255) // 256 * 256
        return off, spans

    def views(buf, spans):
        return {n: buf[o:o + nb].view(dt).view(shape) for n, (o, nb, dt, shape) in spans.items()}

    # The input sets differ in shape (block-table width): one layout per set,
    # slot buffers sized for the largest.
    lay_in = [layout(c, in_names) for c in sets]
    lay_out = [layout(c, out_names) for c in sets]
    host_in = []
    for c, (nbytes, spans) in zip(sets, lay_in):
        hb = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        hv = views(hb, spans)
        for n in in_names:
            hv[n].copy_(getattr(c, n).cpu())
        host_in.append(hb)
    tk_bytes = max(max(ds.topk_workspace_size(c.scores.shape[0], c.scores.shape[1], c.k)
                       for c in sets), 1)
    slots = []
    for _ in range(n_slots):
        din = torch.empty(max(b for b, _ in lay_in), dtype=torch.uint8, device=dev)
        dout = torch.empty(max(b for b, _ in lay_out), dtype=torch.uint8, device=dev)
        hout = torch.empty(dout.numel(), dtype=torch.uint8).pin_memory()
        slots.append({"din": din, "dinv": [views(din, sp) for _, sp in lay_in], "dout": dout,
                      "doutv": [views(dout, sp) for _, sp in lay_out], "hout": hout,
                      "ws": torch.empty_like(sets[0].ws),
                      "tkws": torch.empty(tk_bytes, dtype=torch.uint8, device=dev),
                      "out_done": torch.cuda.Event(), "used": False})
    h2d = round(sum(b for b, _ in lay_in) / len(lay_in))     # bytes copied per step (mean)
    d2h = round(sum(b for b, _ in lay_out) / len(lay_out))

    # Each (slot, input set) step is captured once as a CUDA graph of the
    # public calls: upload, top-k, decode, download (the calls allocate
    # nothing and never synchronise, so they capture as they are). Slot j
    # replays on its own stream, so the uploads and downloads of the steps in
    # flight overlap each other's kernels.
    streams = [torch.cuda.Stream(dev) for _ in range(n_slots)]

    def record(j, sl):
        c, hin = sets[j], host_in[j]
        nin, nout = lay_in[j][0], lay_out[j][0]
        d, o = sl["dinv"][j], sl["doutv"][j]
        st = torch.cuda.current_stream()
        sl["din"][:nin].copy_(hin, non_blocking=True)
        ds.topk_per_row(d["scores"], d["row_starts"], d["row_ends"], c.k, idx_out=o["idx"],
                        stream=st, workspace=sl["tkws"])
        ds.sparse_mla_decode(d["q"], c.kv_pages, c.kv_dtype, d["block_table"], o["idx"],
                             d["lens"], c.scale, out=o["out"], lse=o["lse"], workspace=sl["ws"],
                             stream=st)
        sl["hout"][:nout].copy_(sl["dout"][:nout], non_blocking=True)

    for si, sl in enumerate(slots):
        sl["graphs"] = []
        with torch.cuda.stream(streams[si]):
            for j in range(len(sets)):   # eager warm-up of every call before capture
                record(j, sl)
        streams[si].synchronize()
        for j in range(len(sets)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=streams[si]):
                record(j, sl)
            sl["graphs"].append(g)

    def one(i):
        si = i % n_slots
        sl = slots[si]
        if sl["used"]:
            sl["out_done"].synchronize()   # the host has step i - n_slots's result
        with torch.cuda.stream(streams[si]):
            sl["graphs"][i % len(sets)].replay()
            sl["out_done"].record(streams[si])
        sl["used"] = True

    def drain():
        for sl in slots:
            if sl["used"]:
                sl["out_done"].synchronize()

    for i in range(8):
        one(i)
    drain()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    n = 0
    while n < min_steps or time.perf_counter() - t0 < min_secs:
        one(n)
        n += 1
    drain()
    secs = max_over_ranks(time.perf_counter() - t0, world)
    R = sets[0].q.shape[0]
    return {"value": round(job_value(world, R, n, secs), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "seconds": round(secs, 3),
            "timing": "host wall clock from the first upload to the last result on the host",
            "pipelining": f"{n_slots} steps in flight; each step is one CUDA graph of the public "
                          "calls (upload, top-k, decode, download), each slot on its own stream",
            "kv_cache": "resident on the device (serving state, not a per-step input)"}


def oracle_sample_inputs(case, rows):
    """Host copies of what the oracle needs for `rows` of a decode batch."""
    import numpy as np
    import torch
    scores = case.scores[rows].cpu().numpy()
    starts = case.row_starts.cpu().numpy()[rows]
    ends = case.row_ends.cpu().numpy()[rows]
    bt = case.block_table.cpu().numpy()[case.row_req.cpu().numpy()[rows]]   # each row's table row
    q = case.q[rows].cpu().view(torch.int16).numpy().view(np.uint16)
    used = np.unique(bt[bt >= 0])
    remap = np.zeros(int(used.max()) + 1 if used.size else 1, dtype=np.int64)
    remap[used] = np.arange(used.size)
    kv = case.kv_pages.index_select(0, torch.as_tensor(used, device=case.kv_pages.device))
    kv = kv.cpu().view(torch.int16).numpy().view(np.uint16)
    bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1)
    lens = case.lens.cpu().numpy()[rows]
    return scores, starts, ends, q, kv, bt2, lens


def oracle_step(inputs, k, scale):
    import oracle
    scores, starts, ends, q, kv, bt, lens = inputs
    idx = oracle.topk_per_row(scores, starts, ends, k)
    return oracle.sparse_mla_decode(q, kv, "bf16", bt, idx, lens, scale)


class OracleBatch:
    """The oracle over one decode batch, row by row (top-k, then float64
    attention over all heads): the CPU side of both the `cpu_baseline` leg
    and the reference arm, so the two time the same work the same way."""

    def __init__(self, case):
        self.case = case
        self.R = case.q.shape[0]
        self.inputs = [oracle_sample_inputs(case, [r]) for r in range(self.R)]

    def run(self):
        """One step: every row of the batch once. Returns the seconds taken."""
        t0 = time.perf_counter()
        for inp in self.inputs:
            oracle_step(inp, self.case.k, self.case.scale)
        return time.perf_counter() - t0


def cpu_baseline(case, budget_s):
    """The oracle on the host cores over a bounded sample of the workload:
    whole passes over one input set's decode batch, one untimed pass first,
    then timed passes until `budget_s` seconds of oracle time."""
    cores = len(os.sched_getaffinity(0))
    ob = OracleBatch(case)
    ob.run()
    t_used, passes = 0.0, 0
    while t_used < budget_s:
        t_used += ob.run()
        passes += 1
    return {"value": round(passes * ob.R / t_used, 3), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{passes} passes over the {ob.R}-row batch of input set 0 (top-k + float64 "
                      f"attention over all heads, row by row) after one untimed pass, "
                      f"{t_used:.1f} s of oracle time; numpy BLAS may use all {cores} host cores"}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle; one step = one pass over the decode
    batch (every row: top-k + float64 attention over all heads)."""
    if rank != 0:
        return None
    from synthetic import workload_case
    case = workload_case(WORKLOAD, device="cpu")
    H = case.H
    cores = len(os.sched_getaffinity(0))
    ob = OracleBatch(case)
    for _ in range(args.warmup):
        ob.run()
    t_used, n = 0.0, 0
    for _ in range(args.steps):
        t_used += ob.run()
        n += 1
        if t_used > REFERENCE_CAP_S:   # bounds the run when --steps is large
            break
    value = n * ob.R / t_used
    sample = (f"{n} timed steps after {args.warmup} untimed, each one pass over the {ob.R}-row "
              f"decode batch: top-k + float64 attention over all {H} heads, {t_used:.1f} s")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": n, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_used / max(n, 1) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": WORKLOAD_DESCS[WORKLOAD], "global_batch": ob.R,
                       "parallelism": "CPU oracle, rank 0"},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_cache_write(args, rank, world, local):
    """The KV cache write alone: `value` in rows/s, roofline against HBM.

    Algorithmic bytes per row: 1152 read (bf16 latent) + 656 written (FP8
    row) + 8 read (the slot). Four rotating input sets (latent rows and
    slots), each writing a random permutation of a pool's slots; 4 x 75 MB of
    latent rows against 129 MB of L2.
    """
    import torch
    import invariant_sparse_mla_gb300 as ds
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    N, pages = 65536, 1024
    sets = []
    for s in range(args.sets):
        g = torch.Generator(device=dev).manual_seed(100 + 1000 * rank + s)
        lat = torch.randn((N, 576), generator=g, device=dev).to(torch.bfloat16)
        slots = torch.randperm(pages * 64, generator=g, device=dev)[:N].to(torch.int64)
        pool = torch.zeros((pages, 64, 656), dtype=torch.uint8, device=dev)
        sets.append((lat, slots, pool))
    stream = torch.cuda.Stream(device=dev)

    def step(c):
        ds.kv_cache_write(c[0], c[1], c[2], "fp8", stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            for c in sets:
                step(c)
    stream.synchronize()
    gph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gph, stream=stream):
        for c in sets:
            step(c)
    reps = max(1, math.ceil(args.steps / len(sets)))
    for _ in range(max(1, math.ceil(max(args.warmup, 3) / len(sets)))):
        with torch.cuda.stream(stream):
            gph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id_for_smi(local))
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            gph.replay()
        e1.record(stream)
    e1.synchronize()
    t1 = time.time()
    barrier(world)
    sampler.stop()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    steps = reps * len(sets)
    per_call = secs / steps
    hbm, _, peak_kind = load_peaks()
    row_bytes = 1152 + 656 + 8
    gbs = N * row_bytes / per_call / 1e9
    line = {"metric": METRIC + " [fp8_cache_write]", "value": round(world * N / per_call, 1),
            "unit": "rows/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(per_call * 1e3, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 -> e4m3", "data": "synthetic (seeded N(0,1) rows)",
            "config": {"workload": WORKLOAD_DESCS["fp8_cache_write"], "rows": N, "pages": pages,
                       "l2": f"{args.sets} rotating input sets, "
                             f"{args.sets * N * 1152 // 2**20} MB of latent rows vs 129 MB L2",
                       "cuda_graph": True},
            "roofline": {"bound": "hbm", "kernel": "kv_write_fp8_kernel", "achieved": round(gbs, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                         "peak_kind": f"{peak_kind} HBM copy", "traffic": None,
                         "algorithmic_bytes": N * row_bytes},
            "gpu_launches": steps, "clocks": sampler.summary(t0, t1)}
    if rank == 0 and not args.no_cpu_baseline:
        import numpy as np
        import oracle
        bits = sets[0][0][:4096].cpu().view(torch.int16).numpy().view(np.uint16)
        t = time.perf_counter()
        n_done = 0
        while time.perf_counter() - t < 5.0:
            oracle.quantize_latent_rows(bits)
            n_done += bits.shape[0]
        dt = time.perf_counter() - t
        line["cpu_baseline"] = {"value": round(n_done / dt, 1), "unit": "rows/s",
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": f"{n_done} rows of input set 0 quantised by the oracle "
                                          f"({dt:.1f} s)"}
    return line


def main():
    args = parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.workload == "fp8_cache_write":
        line = run_cache_write(args, rank, world, local)
    elif args.workload == "tp2_indexer":
        import torch
        import invariant_sparse_mla_gb300 as ds
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        res = measure_indexer(ds, dev, torch.cuda.Stream(device=dev), args.steps, args.warmup)
        line = {"metric": METRIC + " [tp2_indexer]", "value": res["rows_per_s"] * world,
                "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(res["step_us"] / 1e3, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded)", "config": {"workload": res["workload"]}, **res}
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
