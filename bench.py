#!/usr/bin/env python
"""Benchmark of the CSA2 decode step over an FP4 global KV cache on GB300.

One step = one decode token for every sequence of the batch through one
CSA2 group: Full-layer index scores + top-512 selection, then the sparse
attention of the Full layer and of each Reuse layer (which reuses the Full
layer's indices).  Default workload: batch 64, 131072 compressed entries per
sequence (128K context, ratio 1), 1 Full + 3 Reuse layers, FP4 main KV with
one power-of-two scale per 32 channels, 1% outlier channels scaled by 8.

value  : query-tokens/s with every input resident in HBM (device-timed).
e2e    : the same metric through the public API with host (pinned) inputs and
         outputs, host<->device copies inside the timed region.
roofline: the indexer-score kernel (the dominant one) against measured HBM
         bandwidth; its duration is taken with CUDA events on its stream.
--impl reference times the CPU oracle (test infrastructure) on the box's
host cores on a bounded sample of the same workload.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, one process per GPU, each running its own replica
(sequences are independent: weak scaling, no collective on the data path).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode query-tokens/s at 128K ctx, B=64; achieved HBM GB/s vs peak"
UNIT = "query-tokens/s"
INDEXER_SRC = os.path.join(ROOT, "fp4_kv_cache_index_gb300", "csrc", "k_index.cu")
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "k_index_decode_traffic.txt")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["csa2", "reference"], default="csa2")
    p.add_argument("--workload", type=int, default=2)
    p.add_argument("--layout", type=int, default=0, help="0 = L32_UE8M0, 1 = L16_E4M3")
    p.add_argument("--batch", type=int, default=None,
                   help="override the workload's batch (smaller profiling cases only)")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-bf16-scores", action="store_true",
                   help="skip the bf16-rounded index score measurement")
    p.add_argument("--no-epilogue", action="store_true",
                   help="skip the sink / output-RoPE readout measurement")
    p.add_argument("--no-paper-cache", action="store_true",
                   help="skip the step over the pages' exact cache formats")
    p.add_argument("--no-hsi", action="store_true",
                   help="skip the Hierarchical Sparse Indexer / Reindex measurement")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads (decode 0, 1, 3 and prefill 4) in the line")
    p.add_argument("--no-decoder", action="store_true",
                   help="skip the pages' 20-layer decoder (Full/Reindex groups) measurement")
    p.add_argument("--pages-formats-only", action="store_true",
                   help="measure only the steps over the pages' cache formats (the decode "
                        "group and the 20-layer decoder) and print their figures (a profiling "
                        "aid; not the benchmark line)")
    p.add_argument("--repeats", type=int, default=25,
                   help="timed regions of --steps steps each; value is the median")
    p.add_argument("--no-graph", action="store_true",
                   help="time eager API calls instead of the captured CUDA graph")
    p.add_argument("--micro-batches", type=int, default=2,
                   help="split the batch into this many micro-batches on their own streams "
                        "(1: one stream, the whole batch per kernel)")
    p.add_argument("--index-sms", type=int, default=112,
                   help="SMs for the indexer's grid when micro-batches > 1 (the rest run "
                        "the other micro-batch's top-k and readout concurrently)")
    p.add_argument("--attn-split", action="store_true",
                   help="with micro-batches, spread each query's readout over two CTAs")
    p.add_argument("--input-sets", type=int, default=4,
                   help="step i reads input set i mod this (distinct seeded queries, weights "
                        "and windows, hence distinct selections): no step finds the previous "
                        "step's readout inputs still in L2")
    return p.parse_args(argv)


# ---------------------------------------------------------------- micro-batches
def packed(specs, dev):
    """One device buffer holding tensors of the given (shape, dtype) at
    256-byte aligned offsets: (the uint8 buffer, the tensors as views)."""
    import torch
    offs, o = [], 0
    for shape, dt in specs:
        offs.append(o)
        nbytes = math.prod(shape) * torch.empty((), dtype=dt).element_size()
        o = (o + nbytes + 255) // 256 * 256
    buf = torch.empty(max(o, 16), dtype=torch.uint8, device=dev)
    views = []
    for (shape, dt), off in zip(specs, offs):
        nbytes = math.prod(shape) * torch.empty((), dtype=dt).element_size()
        views.append(buf[off:off + nbytes].view(dt).view(shape))
    return buf, views


def make_micro_batches(C, cache, wl, bufs0, ld, n_valid, M, split, dev):
    """Per micro-batch device buffers: its queries' inputs (the indexer's
    queries and weights, the layers' queries and windows) packed in one
    buffer, its outputs (selection, the layers' outputs and lse) in another,
    so that the end-to-end pipeline moves each with one copy, and its own
    score / histogram / top-k scratch."""
    import torch
    B, L = wl.batch, wl.layers
    mbs = []
    for m in range(M):
        lo, hi = B * m // M, B * (m + 1) // M
        n = hi - lo
        srcs = [bufs0["q_idx"][lo:hi], bufs0["w"][lo:hi]] + [x[lo:hi] for x in bufs0["qs"]] + \
               [x[lo:hi] for x in bufs0["swas"]]
        in_buf, ins = packed([(tuple(t.shape), t.dtype) for t in srcs], dev)
        for v, t in zip(ins, srcs):
            v.copy_(t)
        out_buf, outv = packed([((n, 512), torch.int32)] +
                               [((n, 64, 512), torch.bfloat16)] * L +
                               [((n, 64), torch.float32)] * L, dev)
        mbs.append(dict(
            seq=list(range(lo, hi)), nv=n_valid[lo:hi],
            in_buf=in_buf, out_buf=out_buf,
            q_idx=ins[0], w=ins[1], qs=ins[2:2 + L], swas=ins[2 + L:2 + 2 * L],
            scores=torch.empty(n, ld, dtype=torch.float32, device=dev),
            hist=torch.empty(n, 2048, dtype=torch.int32, device=dev),
            topk=outv[0],
            tws=torch.empty(max(16, C.csa2_topk_workspace_bytes(n, max(n_valid))),
                            dtype=torch.uint8, device=dev),
            aws=torch.empty(C.csa2_sparse_attn_workspace_bytes(cache, n) if split else 0,
                            dtype=torch.uint8, device=dev),
            outs=outv[1:1 + L], lses=outv[1 + L:1 + 2 * L]))
    return mbs


def mb_index(C, cache, d):
    """One micro-batch's indexer scores, on the current stream."""
    C.csa2_index_scores_decode(cache, d["q_idx"], d["w"], d["scores"], seq_ids=d["seq"],
                               key_hist=d["hist"])


def mb_rest(C, cache, d, L, scale):
    """One micro-batch's top-k and readout layers (one launch for the group's
    layers), on the current stream."""
    C.csa2_topk(d["scores"], d["nv"], 512, idx_out=d["topk"], key_hist=d["hist"],
                workspace=d["tws"])
    C.csa2_sparse_attn_decode_layers(cache, d["qs"], d["swas"], d["topk"], scale, d["outs"],
                                     d["lses"], seq_ids=d["seq"], workspace=d["aws"])


def mb_run(C, cache, d, L, scale, before_index=None, after_index=None):
    """One micro-batch through the whole path, on the current stream;
    before_index / after_index: called around the indexer launch (the
    schedule orders the micro-batches' indexers there)."""
    if before_index is not None:
        before_index()
    mb_index(C, cache, d)
    if after_index is not None:
        after_index()
    mb_rest(C, cache, d, L, scale)


# ---------------------------------------------------------------- distributed helpers
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- peaks and clocks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        if self.out is not None:
            self.out.flush()
            with open(self.out.name) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm.append(float(parts[1]))
                        mx.append(float(parts[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[5:9]):
                        if v.lower().startswith("active"):
                            reasons.add(n)
            os.unlink(self.out.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle sample
class OracleSample:
    """Host inputs of a few sequences of the workload, generated once, and the
    oracle's full decode step for one of them."""

    def __init__(self, wl, layout, n_seqs=4):
        self.wl, self.layout = wl, layout
        self.seqs = list(range(min(n_seqs, wl.batch)))
        self.inputs = {}

    def _inputs(self, b):
        if b not in self.inputs:
            wl = self.wl
            self.inputs[b] = (wl.idx_k(b), wl.q_idx(b, 1)[0], wl.w(b, 1)[0],
                              [wl.q(l, b, 1)[0] for l in range(wl.layers)],
                              [wl.swa(l, b, 1)[0] for l in range(wl.layers)])
        return self.inputs[b]

    def step(self, i, k=512):
        """Oracle time (s) of one query's decode step: fp64 index scores over
        every entry, top-k, then every layer's attention over the selected
        entries and the window.  Generating the selected entries is not timed."""
        import numpy as np
        import oracle as O
        b = self.seqs[i % len(self.seqs)]
        kk, qi, w, qs, sw = self._inputs(b)
        t0 = time.perf_counter()
        idx, _ = O.index_topk(kk, qi, w, k)
        t1 = time.perf_counter()
        sel = idx[idx >= 0]
        rows = self.wl.entry_rows(b, sel)
        t2 = time.perf_counter()
        codes, scales = O.quantise(rows, self.layout)
        local = np.arange(len(sel), dtype=np.int32)
        for l in range(self.wl.layers):
            O.sparse_attention(qs[l], codes, scales, self.layout, local, sw[l],
                               np.float32(512 ** -0.5))
        return (t1 - t0) + (time.perf_counter() - t2)


def cpu_baseline(wl, target_s, layout):
    import oracle as O
    smp = OracleSample(wl, layout)
    smp.step(0)                       # warm-up (also generates the inputs)
    done, spent = 0, 0.0
    while done == 0 or (spent < target_s and done < 64):
        spent += smp.step(done)
        done += 1
    return {"value": done / spent, "unit": UNIT, "cores": O.num_threads(), "kind": "oracle",
            "sample": f"{done} query decode steps of the workload over sequences "
                      f"{smp.seqs} (fp64 index over all entries, top-k, {wl.layers} "
                      f"attention layers each); input generation not timed; "
                      f"{spent:.1f} s of oracle time"}


# ---------------------------------------------------------------- reference arm
def run_reference(args, budget_s=150.0):
    """The oracle on the host cores, one query's decode step per step; the
    run stops early once `budget_s` of oracle time is spent so that any
    --steps finishes within minutes (the line reports the steps timed)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from csa2_synth.workloads import WORKLOADS
    import oracle as O
    wl = WORKLOADS[args.workload]
    smp = OracleSample(wl, args.layout)
    for i in range(max(1, min(args.warmup, 3))):
        smp.step(i)
    spent, n = 0.0, 0
    while n < args.steps and (n == 0 or spent < budget_s):
        spent += smp.step(n)
        n += 1
    value = n / spent
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": n, "warmup": args.warmup, "ms_per_step": 1000 * spent / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, args.layout),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": O.num_threads(),
                         "kind": "oracle",
                         "sample": f"{n} of {args.steps} requested steps (oracle-time budget "
                                   f"{budget_s:.0f} s); each step is one query's full decode "
                                   "step of the workload on the CPU oracle, input generation "
                                   "not timed"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, layout):
    n = wl.n_entries()
    return {"workload": wl.name, "batch": wl.batch, "ctx_tokens": int(wl.ctx),
            "entries_per_seq": int(n[0]) if len(set(n.tolist())) == 1 else n.tolist(),
            "ratio": wl.ratio, "layers": f"1 Full + {wl.layers - 1} Reuse",
            "heads": 64, "head_dim": 512, "idx_heads": 32, "idx_dim": 128, "topk": 512,
            "swa": 128, "layout": "L32_UE8M0" if layout == 0 else "L16_E4M3",
            "outliers": "1% channels x8" if wl.outliers else "none",
            "l2": "inputs larger than L2: every step streams all indexer keys "
                  f"({int(n.sum()) * 256 / 1e9:.2f} GB, L2 evict-first) through the 129 MB "
                  "L2, and step i reads input set i mod input_sets (queries, weights, "
                  "windows; hence selections), so no step finds its readout inputs left "
                  "in L2 by the step before",
            "parallelism": "replica per GPU (sequences are independent)"}


def kernel_traffic_record():
    """ncu DRAM bytes per indexer launch, if recorded for this exact source."""
    try:
        src = hashlib.sha256(open(INDEXER_SRC, "rb").read()).hexdigest()
        rec = {}
        with open(TRAFFIC_RECORD) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
        if rec.get("k_index.cu sha256") == src and rec.get("workload") is not None:
            return rec
    except OSError:
        pass
    return None


# ---------------------------------------------------------------- GPU arm
def run_csa2(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import fp4_kv_cache_index_gb300 as C
    from csa2_synth import workloads as W
    wl = W.WORKLOADS[args.workload]
    if args.batch is not None:
        import dataclasses
        wl = dataclasses.replace(wl, batch=args.batch, name=f"{wl.name}@batch{args.batch}")
    assert not wl.prefill, "the decode benchmark takes a decode workload"
    L = wl.layers
    B = wl.batch
    n_ent = wl.n_entries()
    cfg = C.config(ratio=wl.ratio, layout=args.layout)
    cache = C.Cache(cfg, [int(x) for x in n_ent], device=dev)
    W.fill_cache(wl, cache)
    S = max(2, args.input_sets)

    def make_inputs(s):
        # set 0 is the workload's own stream; set s > 0 draws the same
        # distributions from the streams of "layers" past the model's
        return dict(q_idx=W.dev_q_idx(wl, layer=s), w=W.dev_w(wl, layer=s),
                    qs=[W.dev_q(wl, L * s + l) for l in range(L)],
                    swas=[W.dev_swa(wl, L * s + l) for l in range(L)])

    def make_outputs():
        return dict(topk=torch.empty(B, 512, dtype=torch.int32, device=dev),
                    outs=[torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev)
                          for _ in range(L)],
                    lses=[torch.empty(B, 64, dtype=torch.float32, device=dev) for _ in range(L)])

    ld = max(4, (int(n_ent.max()) + 3) // 4 * 4)
    scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
    key_hist = torch.empty(B, 2048, dtype=torch.int32, device=dev)
    topk_ws = torch.empty(max(16, C.csa2_topk_workspace_bytes(B, int(n_ent.max()))),
                          dtype=torch.uint8, device=dev)
    n_valid = [int(x) for x in n_ent]
    attn_ws = torch.empty(max(16, C.csa2_sparse_attn_workspace_bytes(cache, B)),
                          dtype=torch.uint8, device=dev)
    scale = 512 ** -0.5
    stream = torch.cuda.current_stream()

    # S input sets, step i on set i mod S; outputs double-buffered (set s
    # writes output buffer s mod 2, the end-to-end leg's two buffer sets)
    out_sets = [make_outputs(), make_outputs()]
    bufs = [dict(**make_inputs(s), **out_sets[s % 2]) for s in range(S)]

    def step(ev=None, b=0):
        d = bufs[b]
        if ev is not None:
            ev[0].record(stream)
        C.csa2_index_scores_decode(cache, d["q_idx"], d["w"], scores, key_hist=key_hist)
        if ev is not None:
            ev[1].record(stream)
        C.csa2_topk(scores, n_valid, 512, idx_out=d["topk"], key_hist=key_hist, workspace=topk_ws)
        if ev is not None:
            ev[2].record(stream)
        C.csa2_sparse_attn_decode_layers(cache, d["qs"], d["swas"], d["topk"], scale, d["outs"],
                                         d["lses"], workspace=attn_ws)
        if ev is not None:
            ev[3].record(stream)

    torch.cuda.synchronize()
    sampler = ClockSampler(local).start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- the step captured once as a CUDA graph (every call is stream-ordered
    #      and allocation-free), replayed for the headline timing
    graphs = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for b in range(S):
                step(b=b)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graphs = [torch.cuda.CUDAGraph() for _ in range(S)]
        for b in range(S):
            with torch.cuda.graph(graphs[b]):
                step(b=b)
        for i in range(max(3, args.warmup)):
            graphs[i % S].replay()
        torch.cuda.synchronize()

    R = max(1, args.repeats)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)

    def timed_region(run_steps):
        # exactly --steps steps between a barrier + synchronize on both sides
        barrier(world)
        torch.cuda.synchronize()
        t_start.record(stream)
        run_steps()
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return t_start.elapsed_time(t_end) / 1000.0

    def single_steps():
        for i in range(args.steps):
            if graphs is not None:
                graphs[i % S].replay()
            else:
                step(b=i % S)

    singles = [timed_region(single_steps) for _ in range(R)]
    elapsed_single = statistics.median(singles)
    elapsed = elapsed_single
    repeats = singles

    # ---- the headline schedule: the batch split into micro-batches, each on
    #      its own stream and in order there, step after step; the indexer's
    #      grid is capped so that the other micro-batch's latency-bound top-k
    #      and readout run on the remaining SMs while it streams the keys.
    #      The indexers of the micro-batches run one after the other (each
    #      waits for the previous one's completion event): a persistent grid
    #      whose CTAs start while another indexer still holds SMs would
    #      finish late
    M = args.micro_batches
    mb_sets, mb_streams, graph_steps = None, None, 0
    if M > 1:
        mb_sets = [make_micro_batches(C, cache, wl, bufs[s], ld, n_valid, M, args.attn_split, dev)
                   for s in range(S)]
        mb_streams = [torch.cuda.Stream() for _ in range(M)]

        def mb_steps(n):
            main = torch.cuda.current_stream()
            for s_ in mb_streams:
                s_.wait_stream(main)
            prev = [None]

            def before():
                if prev[0] is not None:
                    torch.cuda.current_stream().wait_event(prev[0])

            def after():
                ev = torch.cuda.Event()
                ev.record(torch.cuda.current_stream())
                prev[0] = ev

            for i in range(n):
                for s_, d in zip(mb_streams, mb_sets[i % S]):
                    with torch.cuda.stream(s_):
                        mb_run(C, cache, d, L, scale, before, after)
            for s_ in mb_streams:
                main.wait_stream(s_)

        cache.set_index_sms(args.index_sms)
        for _ in range(max(3, args.warmup)):
            mb_steps(S)
        torch.cuda.synchronize()
        graph_steps = max(1, min(args.steps, 20 // S * S))
        g_main = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_main):
            mb_steps(graph_steps)
        g_rest = None
        if args.steps % graph_steps:
            g_rest = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_rest):
                mb_steps(args.steps % graph_steps)
        cache.set_index_sms(0)
        g_main.replay()
        torch.cuda.synchronize()

        def mb_timed_steps():
            for _ in range(args.steps // graph_steps):
                g_main.replay()
            if g_rest is not None:
                g_rest.replay()

        repeats = [timed_region(mb_timed_steps) for _ in range(R)]
        elapsed = statistics.median(repeats)
    clocks = sampler.stop()

    # ---- per-kernel split: eager calls with CUDA events around each launch
    n_split = max(3, min(args.steps, 500))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_split)]
    torch.cuda.synchronize()
    e_a = torch.cuda.Event(enable_timing=True)
    e_b = torch.cuda.Event(enable_timing=True)
    e_a.record(stream)
    for i in range(n_split):
        step(evs[i], b=i % S)
    e_b.record(stream)
    torch.cuda.synchronize()
    eager_ms = e_a.elapsed_time(e_b) / n_split
    t_idx = sum(e[0].elapsed_time(e[1]) for e in evs) / n_split / 1000.0
    t_topk = sum(e[1].elapsed_time(e[2]) for e in evs) / n_split / 1000.0
    t_attn = sum(e[2].elapsed_time(e[3]) for e in evs) / n_split / 1000.0
    if cache.device_error() != 0:
        raise RuntimeError("device error word set during the benchmark")
    elapsed_max = max_over_ranks(elapsed, world, dev)
    single_max = max_over_ranks(elapsed_single, world, dev)
    rep_ms = [1000 * max_over_ranks(x, world, dev) / args.steps for x in repeats]

    # the indexer alone on the schedule's capped grid, one micro-batch's
    # queries (the launch configuration of the headline schedule)
    sched_idx = None
    if M > 1:
        d0 = mb_sets[0][0]
        cache.set_index_sms(args.index_sms)
        for _ in range(3):
            C.csa2_index_scores_decode(cache, d0["q_idx"], d0["w"], d0["scores"], seq_ids=d0["seq"],
                                       key_hist=d0["hist"])
        n_si = max(3, min(args.steps, 100))
        e_si = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_si)]
        for e in e_si:
            e[0].record(stream)
            C.csa2_index_scores_decode(cache, d0["q_idx"], d0["w"], d0["scores"], seq_ids=d0["seq"],
                                       key_hist=d0["hist"])
            e[1].record(stream)
        torch.cuda.synchronize()
        cache.set_index_sms(0)
        t_si = statistics.median(e[0].elapsed_time(e[1]) for e in e_si) / 1000.0
        si_bytes = int(sum(d0["nv"])) * 256 + len(d0["seq"]) * (32 * 128 * 2 + 32 * 4)
        hbm_pk, _ = measured_peaks()
        sched_idx = {"sms": args.index_sms, "queries": len(d0["seq"]),
                     "ms": 1000 * t_si, "achieved": si_bytes / t_si / 1e9,
                     "frac": si_bytes / t_si / 1e9 / hbm_pk,
                     "timed_as": "one micro-batch's indexer alone on the schedule's capped "
                                 "grid (median of per-launch CUDA events)"}

    # ---- end to end: every step's inputs go host -> device and its outputs
    #      device -> host inside the timed region, double-buffered the way a
    #      serving loop would run it: the copies of step i+1's inputs and of
    #      step i-1's outputs run on a copy stream while step i computes
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 200))
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
    names_in = ["q_idx", "w", "qs", "swas"]
    names_out = ["topk", "outs", "lses"]
    flat = lambda d, names: [x for n in names for x in (d[n] if isinstance(d[n], list) else [d[n]])]
    # step i's inputs are input set i mod S, copied from the host
    h_in = [[pin(t) for t in flat(bufs[s], names_in)] for s in range(S)]
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in flat(bufs[0], names_out)]
             for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in[0])
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    copy_stream = torch.cuda.Stream()

    def run_e2e(n):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]
        with torch.cuda.stream(copy_stream):
            for h, d in zip(h_in[0], flat(bufs[0], names_in)):
                d.copy_(h, non_blocking=True)
            in_ready[0].record(copy_stream)
        for i in range(n):
            b = i % 2
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(out_free[b])
            if graphs:
                graphs[b].replay()
            else:
                step(b=b)
            done[b].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n:
                    if i >= 1:
                        copy_stream.wait_event(done[1 - b])
                    for h, d in zip(h_in[(i + 1) % S], flat(bufs[1 - b], names_in)):
                        d.copy_(h, non_blocking=True)
                    in_ready[1 - b].record(copy_stream)
                copy_stream.wait_event(done[b])
                for h, d in zip(h_out[b], flat(bufs[b], names_out)):
                    h.copy_(d, non_blocking=True)
                out_free[b].record(copy_stream)
        stream.wait_stream(copy_stream)

    e2e_note = ("inputs of step i+1 and outputs of step i-1 copied on a second stream "
                "while step i computes (pinned host buffers)")
    if M > 1:
        # the same double-buffered copy pipeline per micro-batch: each has a
        # compute stream and a copy stream; the micro-batches' pipelines
        # overlap one another, their indexers ordered one after the other by
        # events (as in the device-timed schedule).  With graphs (the
        # default) a run of steps -- copies, events and API calls -- is
        # captured as one CUDA graph, like the device-timed steps
        sets = [mb_sets[0], mb_sets[1]]
        copy_streams = [torch.cuda.Stream() for _ in range(M)]
        # one packed buffer of inputs and one of outputs per micro-batch: one
        # copy each way per micro-batch and step
        names_in, names_out = ["in_buf"], ["out_buf"]
        h_in_mb = [[[pin(t) for t in flat(mb_sets[s][m], names_in)] for m in range(M)]
                   for s in range(S)]
        h_out_mb = [[[torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                      for t in flat(mb_sets[0][m], names_out)] for _ in range(2)] for m in range(M)]
        h2d = sum(t.numel() * t.element_size() for h in h_in_mb[0] for t in h)
        d2h = sum(t.numel() * t.element_size() for h in h_out_mb for t in h[0])

        def e2e_pipeline(n):
            main = torch.cuda.current_stream()
            for s_ in mb_streams + copy_streams:
                s_.wait_stream(main)
            ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
            in_ready = [ev() for _ in range(M)]
            done = [ev() for _ in range(M)]
            out_free = [ev() for _ in range(M)]
            for m in range(M):
                with torch.cuda.stream(copy_streams[m]):
                    for h, t in zip(h_in_mb[0][m], flat(sets[0][m], names_in)):
                        t.copy_(h, non_blocking=True)
                    in_ready[m][0].record(copy_streams[m])
            prev_index = None
            for i in range(n):
                b = i % 2
                for m in range(M):
                    cs, ps = mb_streams[m], copy_streams[m]
                    cs.wait_event(in_ready[m][b])
                    if i >= 2:
                        cs.wait_event(out_free[m][b])
                    if prev_index is not None:
                        cs.wait_event(prev_index)
                    with torch.cuda.stream(cs):
                        mb_index(C, cache, sets[b][m])
                        prev_index = torch.cuda.Event()
                        prev_index.record(cs)
                        mb_rest(C, cache, sets[b][m], L, scale)
                    done[m][b].record(cs)
                    with torch.cuda.stream(ps):
                        if i + 1 < n:
                            if i >= 1:
                                ps.wait_event(done[m][1 - b])
                            for h, t in zip(h_in_mb[(i + 1) % S][m],
                                            flat(sets[1 - b][m], names_in)):
                                t.copy_(h, non_blocking=True)
                            in_ready[m][1 - b].record(ps)
                        ps.wait_event(done[m][b])
                        for h, t in zip(h_out_mb[m][b], flat(sets[b][m], names_out)):
                            h.copy_(t, non_blocking=True)
                        out_free[m][b].record(ps)
            for s_ in mb_streams + copy_streams:
                main.wait_stream(s_)

        cache.set_index_sms(args.index_sms)
        e2e_pipeline(3)
        torch.cuda.synchronize()
        e2e_graphs = {}
        if graphs is not None:
            # a graph of up to 20 steps replayed; a shorter one for the rest
            g_len = min(20, e2e_steps)
            try:
                for n_g in sorted({g_len, e2e_steps % g_len} - {0}):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        e2e_pipeline(n_g)
                    e2e_graphs[n_g] = g
            except RuntimeError as exc:   # host copies not capturable here: eager
                torch.cuda.synchronize()
                e2e_graphs = {}
                print(f"end-to-end steps run eagerly ({exc})", file=sys.stderr)
        cache.set_index_sms(0)

        def run_e2e(n):
            if not e2e_graphs:
                cache.set_index_sms(args.index_sms)
                e2e_pipeline(n)
                cache.set_index_sms(0)
                return
            g_len = max(e2e_graphs)
            for _ in range(n // g_len):
                e2e_graphs[g_len].replay()
            if n % g_len:
                e2e_graphs[n % g_len].replay()

        e2e_note = ("per micro-batch: inputs of step i+1 and outputs of step i-1 copied on "
                    "its copy stream while step i computes on its compute stream (pinned "
                    "host buffers); the micro-batches' pipelines overlap, their indexers "
                    "ordered one after the other as in the device-timed schedule; " +
                    ("runs of up to 20 steps (their copies, events and API calls) as one "
                     "CUDA graph" if e2e_graphs else "eager API calls"))
    run_e2e(e2e_steps if M > 1 else 3)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b_ = torch.cuda.Event(enable_timing=True)

    def e2e_region():
        barrier(world)
        torch.cuda.synchronize()
        a.record(stream)
        copy_stream.wait_stream(stream)
        run_e2e(e2e_steps)
        b_.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(a.elapsed_time(b_) / 1000.0, world, dev)

    e2e_reps = [e2e_region() for _ in range(R)]
    e2e_elapsed = statistics.median(e2e_reps)

    hbm_peak, peak_kind = measured_peaks()
    # the measurements below read input set 0 and its fp32 selection
    step(b=0)
    torch.cuda.synchronize()
    bf16 = None
    if not args.no_bf16_scores:
        bf16 = measure_bf16_scores(C, cache, wl, bufs[0]["q_idx"], bufs[0]["w"], n_valid,
                                   bufs[0]["topk"], key_hist, topk_ws, dev, stream,
                                   max(3, min(args.steps, 300)), t_idx, t_topk)
    epi = None
    if not args.no_epilogue:
        epi = measure_epilogue(C, cache, bufs[0], attn_ws, scale, wl, dev, stream,
                               max(3, min(args.steps, 300)))
    paper = None
    if not args.no_paper_cache:
        paper = measure_paper_cache(C, W, wl, dev, stream, max(3, min(args.steps, 300)), hbm_peak)
    hsi = None
    if not args.no_hsi:
        hsi = measure_hsi(C, W, wl, cache, scores, n_valid, dev, stream,
                          max(3, min(args.steps, 300)), hbm_peak)
    # the other workloads and the pages' decoder, each on its own cache
    configs, decoder = None, None
    iters = max(5, min(args.steps, 50))
    if not args.no_configs:
        configs = {}
        flush = make_l2_flush(dev)
        for wid in (0, 1, 3):
            r = measure_decode_config(C, W, wid, dev, stream, iters, hbm_peak, flush)
            configs[r["workload"]] = r
        r = measure_prefill(C, W, 4, args.layout, dev, stream, max(3, min(args.steps, 10)),
                            max(3, args.warmup))
        configs[r["workload"]] = r
        del flush
        torch.cuda.empty_cache()
    if not args.no_decoder:
        decoder = measure_decoder(C, W, dev, stream, iters, hbm_peak)
        torch.cuda.empty_cache()

    # ---- accounting
    tot_ent = int(n_ent.sum())
    idx_bytes = tot_ent * 256 + B * (32 * 128 * 2 + 32 * 4)
    entry_bytes = 256 + (16 if args.layout == 0 else 32)
    attn_bytes = L * B * (512 * entry_bytes + 128 * 512 * 2 + 2 * 64 * 512 * 2)
    step_bytes = idx_bytes + attn_bytes
    ms = 1000 * elapsed_max / args.steps
    achieved = idx_bytes / t_idx / 1e9
    rec = kernel_traffic_record()
    traffic = None
    if rec is not None and rec.get("workload") == wl.name:
        traffic = float(rec["dram_bytes_per_launch"])
    # this library's kernels per step: indexer, top-k segments, top-k, one
    # attention launch per layer (workspace memsets are not counted)
    launches_per_step = 4 * ((B + 1023) // 1024) * max(1, M)   # index, 2 x top-k, readout
    config = workload_config(wl, args.layout)
    config["input_sets"] = S
    nominal = 8000.0   # GB/s: the nominal HBM3e figure of the target
    line = {
        "metric": METRIC, "value": B * world * args.steps / elapsed_max, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config,
        "roofline": {"kernel": "k_index (indexer scores, tcgen05)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "frac_nominal": achieved / nominal,
                     "algorithmic_bytes_per_launch": idx_bytes,
                     "timed_as": "eager, the whole batch on every SM (median of per-launch "
                                 "CUDA events on the launching stream)",
                     "in_schedule": None if sched_idx is None else sched_idx},
        "step_hbm": {"achieved": step_bytes / (ms / 1000) / 1e9, "peak": hbm_peak,
                     "unit": "GB/s", "frac": step_bytes / (ms / 1000) / 1e9 / hbm_peak,
                     "frac_nominal": step_bytes / (ms / 1000) / 1e9 / nominal,
                     "algorithmic_bytes_per_step": step_bytes},
        "repeats": {"n": len(rep_ms), "steps_each": args.steps,
                    "ms_per_step_median": statistics.median(rep_ms),
                    "ms_per_step_min": min(rep_ms), "ms_per_step_max": max(rep_ms),
                    "value_is": "the median timed region (max over ranks)"},
        "kernel_ms": {"index_scores": 1000 * t_idx, "topk": 1000 * t_topk,
                      "sparse_attn_all_layers": 1000 * t_attn,
                      "eager_step": eager_ms,
                      "timed_as": "eager calls with CUDA events, the whole batch on one stream"},
        "schedule": {"micro_batches": max(1, M), "streams": max(1, M),
                     "index_sms": args.index_sms if M > 1 else None,
                     "attention_split": bool(args.attn_split) if M > 1 else True,
                     "indexers_serialised": M > 1,
                     "steps_per_graph": graph_steps if M > 1 else 1},
        "single_stream": {"value": B * world * args.steps / single_max,
                          "ms_per_step": 1000 * single_max / args.steps,
                          "schedule": "whole batch per kernel on one stream, two-CTA readout "
                                      "split, every SM for the indexer; one CUDA graph per step"},
        "e2e": {"value": B * world * e2e_steps / e2e_elapsed, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelining": e2e_note,
                "repeats": {"n": len(e2e_reps), "steps_each": e2e_steps,
                            "value_min": B * world * e2e_steps / max(e2e_reps),
                            "value_max": B * world * e2e_steps / min(e2e_reps)}},
        "gpu_launches": launches_per_step * args.steps,
        "hsi_reindex": hsi,
        "bf16_scores": bf16,
        "readout_epilogue": epi,
        "paper_cache": paper,
        "configs": configs,
        "decoder": decoder,
        "clocks": clocks,
    }
    if clocks.get("sm_mhz"):
        # time x clock: a clock-normalised step time, comparable across runs
        # whose SM clock differs
        clocks["ms_per_step_x_sm_mhz"] = ms * clocks["sm_mhz"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds, args.layout)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure_paper_cache(C, W, wl, dev, stream, iters, hbm_peak):
    """The same decode step over the cache formats the V4.1 report gives:
    main KV E2M1 with one E4M3 scale per 16 channels (288 B/entry), indexer
    keys and queries in MXFP4 (68 B/entry), window rows in FP8 (584 B/row).
    Timed as a CUDA graph replay of index + top-k + every layer's readout."""
    import torch
    B, L = wl.batch, wl.layers
    n_ent = wl.n_entries()
    cfg = C.config(ratio=wl.ratio, layout=1, idx_layout=1)
    cache = C.Cache(cfg, [int(x) for x in n_ent], device=dev)
    W.fill_cache(wl, cache)
    q_idx, w = W.dev_q_idx(wl), W.dev_w(wl)
    qs = [W.dev_q(wl, l) for l in range(L)]
    swas = [C.csa2_swa_fp8_quantise(W.dev_swa(wl, l)) for l in range(L)]
    topk = torch.empty(B, 512, dtype=torch.int32, device=dev)
    ws = torch.empty(C.csa2_index_workspace_bytes(cache, B), dtype=torch.uint8, device=dev)
    attn_ws = torch.empty(max(16, C.csa2_sparse_attn_workspace_bytes(cache, B)),
                          dtype=torch.uint8, device=dev)
    outs = [torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    scale = 512 ** -0.5

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        C.csa2_index_topk_decode(cache, q_idx, w, topk_idx=topk, workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        C.csa2_sparse_attn_decode_layers(cache, qs, None, topk, scale, outs, None,
                                         workspace=attn_ws, swa_fp8s=swas)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(iters):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / iters
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(iters)]
    for i in range(iters):
        step(evs[i])
    torch.cuda.synchronize()
    t_sel = sum(e[0].elapsed_time(e[1]) for e in evs) / iters
    t_attn = sum(e[1].elapsed_time(e[2]) for e in evs) / iters
    # the MXFP4 indexer alone (its dominant kernel)
    sc = torch.empty(B, (int(n_ent.max()) + 3) // 4 * 4, dtype=torch.float32, device=dev)
    hist = torch.empty(B, 2048, dtype=torch.int32, device=dev)
    t_ix = statistics.median(per_step_ms(
        lambda: C.csa2_index_scores_decode(cache, q_idx, w, sc, key_hist=hist), iters, stream))
    if cache.device_error() != 0:
        raise RuntimeError("device error word set during the paper-cache measurement")
    tot = int(n_ent.sum())
    idx_bytes = tot * 68 + B * (32 * 128 * 2 + 32 * 4)
    attn_bytes = L * B * (512 * 288 + 128 * 584 + 2 * 64 * 512 * 2)
    step_bytes = idx_bytes + attn_bytes
    del cache
    return {"formats": "main KV E2M1 + E4M3/16 (288 B), indexer K MXFP4 (68 B), "
                       "window FP8 (584 B/row)",
            "ms_per_step": ms, "value": B / (ms / 1000), "unit": "query-tokens/s",
            "selection_ms": t_sel, "readout_all_layers_ms": t_attn,
            "index_ms": t_ix,
            "index_roofline": {"kernel": "k_index_fp4 (block-scaled MXFP4 MMAs)",
                               "bound": "hbm", "algorithmic_bytes_per_launch": idx_bytes,
                               "achieved": idx_bytes / (t_ix / 1000) / 1e9, "peak": hbm_peak,
                               "unit": "GB/s",
                               "frac": idx_bytes / (t_ix / 1000) / 1e9 / hbm_peak},
            "algorithmic_bytes_per_step": step_bytes,
            "step_hbm_gbs": step_bytes / (ms / 1000) / 1e9,
            "step_hbm_frac": step_bytes / (ms / 1000) / 1e9 / hbm_peak,
            "timed_as": "cuda graph replay (selection and readout split: eager events)"}


def measure_epilogue(C, cache, d, attn_ws, scale, wl, dev, stream, iters):
    """One layer's readout with the V4 blog reading's section 4.3 variants
    (a per-head sink logit and the output RoPE(-i) on the last 64 channels)
    against the plain readout, same inputs, events around each call."""
    import torch
    B = wl.batch
    sink = torch.linspace(-2.0, 2.0, 64, device=dev)
    pos = torch.full((B,), int(wl.ctx) - 1, dtype=torch.int64, device=dev)
    out = torch.empty_like(d["outs"][0])

    def timed(**kw):
        for _ in range(3):
            C.csa2_sparse_attn_decode(cache, d["qs"][0], d["swas"][0], d["topk"], scale, out=out,
                                      workspace=attn_ws, **kw)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(iters):
            C.csa2_sparse_attn_decode(cache, d["qs"][0], d["swas"][0], d["topk"], scale, out=out,
                                      workspace=attn_ws, **kw)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters

    plain = timed()
    variants = timed(sink=sink, rope_pos=pos)
    if cache.device_error() != 0:
        raise RuntimeError("device error word set during the epilogue measurement")
    return {"plain_layer_ms": plain, "sink_rope_layer_ms": variants,
            "timed_as": "eager calls, one layer, the same inputs every call (their 26 MB "
                        "stay in L2: a relative figure)"}


def measure_bf16_scores(C, cache, wl, q_idx, w, n_valid, fp32_idx, key_hist, topk_ws, dev,
                        stream, iters, t_idx32, t_topk32):
    """The Full layer's selection on bf16-rounded scores (the V4 blog
    reading's section 7): index scores stored as bf16, top-k over them.
    Reports its time next to the fp32 selection's, and the recall of the
    fp32 selection (the step's own top-k of the last timed step)."""
    import torch
    B = wl.batch
    ld = (max(n_valid) + 7) // 8 * 8
    s16 = torch.empty(B, ld, dtype=torch.bfloat16, device=dev)
    idx16 = torch.empty(B, 512, dtype=torch.int32, device=dev)

    def run(ev=None):
        if ev is not None:
            ev[0].record(stream)
        C.csa2_index_scores_decode_bf16(cache, q_idx, w, s16, key_hist=key_hist)
        if ev is not None:
            ev[1].record(stream)
        C.csa2_topk_bf16(s16, n_valid, 512, idx_out=idx16, key_hist=key_hist, workspace=topk_ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(iters)]
    for i in range(iters):
        run(evs[i])
    torch.cuda.synchronize()
    t_idx = sum(e[0].elapsed_time(e[1]) for e in evs) / iters
    t_topk = sum(e[1].elapsed_time(e[2]) for e in evs) / iters
    # recall of the fp32 selection, per query (both lists ascending, -1 padded)
    a = fp32_idx.long()
    b = idx16.long()
    hit = torch.zeros(B, device=dev)
    for r in range(B):
        ar = a[r][a[r] >= 0]
        br = b[r][b[r] >= 0]
        hit[r] = torch.isin(ar, br).float().mean() if ar.numel() else 1.0
    if cache.device_error() != 0:
        raise RuntimeError("device error word set during the bf16-score measurement")
    return {"index_ms": t_idx, "topk_ms": t_topk,
            "fp32_index_ms": 1000 * t_idx32, "fp32_topk_ms": 1000 * t_topk32,
            "topk_speedup": (1000 * t_topk32) / t_topk if t_topk > 0 else None,
            "recall_mean": float(hit.mean()), "recall_min": float(hit.min()),
            "recall_of": "the fp32 top-512 of the same scores (seeded N(0,1) inputs)"}


def measure_hsi(C, W, wl, cache, scores, n_valid, dev, stream, iters, hbm_peak,
                max_blocks=2048):
    """Hierarchical Sparse Indexer on the same batch: the candidate pool from
    the Full layer's scores (block maxima + top-2048 blocks), then one
    Reindex layer's selection (its own indexer query over the 16,384 pool
    positions, top-512).  Timed as a CUDA graph replay (both calls) and per
    call with events; not part of the headline step, which is the configured
    Full + Reuse group."""
    import torch
    B = wl.batch
    pool = torch.empty(B, max_blocks, dtype=torch.int32, device=dev)
    pool_ws = torch.empty(max(16, int(C.lib.csa2_hsi_pool_workspace_bytes(B, max(n_valid)))),
                          dtype=torch.uint8, device=dev)
    re_ws = torch.empty(max(16, int(C.lib.csa2_index_reindex_workspace_bytes(
        cache.handle, B, max_blocks))), dtype=torch.uint8, device=dev)
    q2 = W.dev_q_idx(wl, layer=1)
    w2 = W.dev_w(wl, layer=1)
    re_idx = torch.empty(B, 512, dtype=torch.int32, device=dev)

    def run(ev=None):
        if ev is not None:
            ev[0].record(stream)
        C.csa2_hsi_pool(scores, n_valid, max_blocks, pool_blocks=pool, workspace=pool_ws)
        if ev is not None:
            ev[1].record(stream)
        C.csa2_index_topk_reindex_decode(cache, q2, w2, pool, topk_idx=re_idx, workspace=re_ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        run()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        g.replay()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(iters):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    graph_ms = a.elapsed_time(b) / iters
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(iters)]
    for i in range(iters):
        run(evs[i])
    torch.cuda.synchronize()
    t_pool = sum(e[0].elapsed_time(e[1]) for e in evs) / iters
    t_re = sum(e[1].elapsed_time(e[2]) for e in evs) / iters
    if cache.device_error() != 0:
        raise RuntimeError("device error word set during the HSI measurement")
    slots = max_blocks * 8
    pool_bytes = sum(n_valid) * 4                       # block maxima read the Full scores
    re_bytes = B * (slots * 256 + 32 * 128 * 2 + 32 * 4)  # pool keys + query + weights
    return {"max_blocks": max_blocks, "block": 8, "pool_positions": slots,
            "graph_ms": graph_ms, "pool_ms": t_pool, "reindex_ms": t_re,
            "reindex_qtok_s": B / (t_re / 1000),
            "pool_algorithmic_bytes": pool_bytes, "reindex_algorithmic_bytes": re_bytes,
            "reindex_hbm_gbs": re_bytes / (t_re / 1000) / 1e9,
            "reindex_hbm_frac": re_bytes / (t_re / 1000) / 1e9 / hbm_peak,
            "launches": "pool: block max + top-k; reindex: pool-mode indexer + top-k "
                        "segments + top-k + slot map"}


def make_l2_flush(dev, nbytes=512 << 20):
    """Writes a buffer of 4x the 129 MB L2 (torch's fill kernel, outside the
    timed events), so that a timed step finds none of its inputs in L2."""
    import torch
    buf = torch.empty(nbytes // 4, dtype=torch.int32, device=dev)
    return lambda: buf.fill_(1)


def per_step_ms(run, n, stream, flush=None):
    """Device time (ms) of each of n calls of `run`, CUDA events on the
    launching stream around each; the L2 flushed before each when `flush`."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        if flush is not None:
            flush()
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def capture(run, stream):
    """`run` captured as a CUDA graph (warmed on a side stream first)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        run()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    return g


def measure_decode_config(C, W, wid, dev, stream, iters, hbm_peak, flush):
    """One decode step of workload `wid` at full size (Full layer index +
    top-k, then every layer's readout), the whole batch on one stream as a
    CUDA graph; the L2 is flushed before every timed step (the small
    workloads' inputs fit in L2).  Roofline: HBM on the algorithmic bytes of
    the step (indexer keys + queries, and per query and layer the selected
    entries, the window rows, q and out)."""
    import torch
    wl = W.WORKLOADS[wid]
    B, L = wl.batch, wl.layers
    n_ent = [int(x) for x in wl.n_entries()]
    cache = C.Cache(C.config(ratio=wl.ratio), n_ent, device=dev)
    W.fill_cache(wl, cache)
    q_idx, w = W.dev_q_idx(wl), W.dev_w(wl)
    qs = [W.dev_q(wl, l) for l in range(L)]
    swas = [W.dev_swa(wl, l) for l in range(L)]
    ld = max(4, (max(n_ent) + 3) // 4 * 4)
    scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
    hist = torch.empty(B, 2048, dtype=torch.int32, device=dev)
    tws = torch.empty(max(16, C.csa2_topk_workspace_bytes(B, max(n_ent))), dtype=torch.uint8,
                      device=dev)
    aws = torch.empty(max(16, C.csa2_sparse_attn_workspace_bytes(cache, B)), dtype=torch.uint8,
                      device=dev)
    topk = torch.empty(B, 512, dtype=torch.int32, device=dev)
    outs = [torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    scale = 512 ** -0.5

    def index():
        C.csa2_index_scores_decode(cache, q_idx, w, scores, key_hist=hist)

    def select():
        C.csa2_topk(scores, n_ent, 512, idx_out=topk, key_hist=hist, workspace=tws)

    def readout():
        C.csa2_sparse_attn_decode_layers(cache, qs, swas, topk, scale, outs, None, workspace=aws)

    def step():
        index()
        select()
        readout()

    for _ in range(3):
        step()
    g = capture(step, stream)
    for _ in range(3):
        g.replay()
    t = per_step_ms(g.replay, iters, stream, flush)
    t_idx = per_step_ms(index, iters, stream, flush)
    t_sel = per_step_ms(lambda: (index(), select()), iters, stream, flush)
    t_att = per_step_ms(readout, iters, stream, flush)
    if cache.device_error() != 0:
        raise RuntimeError(f"device error word set during workload {wid}")
    ms = statistics.median(t)
    ms_idx = statistics.median(t_idx)
    ms_sel = max(0.0, statistics.median(t_sel) - ms_idx)
    ms_att = statistics.median(t_att)
    idx_bytes = sum(n_ent) * 256 + B * (32 * 128 * 2 + 32 * 4)
    attn_bytes = L * sum(min(512, n) * 272 + 128 * 1024 + 2 * 64 * 1024 for n in n_ent)
    step_bytes = idx_bytes + attn_bytes
    gbs = step_bytes / (ms / 1000) / 1e9
    parts = {"index_scores": ms_idx, "topk": ms_sel, "sparse_attn_all_layers": ms_att}
    top = max(parts, key=parts.get)
    del cache
    return {"workload": wl.name, "batch": B, "entries_per_seq": n_ent if wl.ragged else n_ent[0],
            "ratio": wl.ratio, "layers": f"1 Full + {L - 1} Reuse", "layout": "L32_UE8M0",
            "ms_per_step": ms, "ms_per_step_min": min(t), "ms_per_step_max": max(t),
            "value": B / (ms / 1000), "unit": UNIT, "steps": iters,
            "roofline": {"bound": "hbm", "algorithmic_bytes_per_step": step_bytes,
                         "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "frac_nominal": gbs / 8000.0},
            "kernel_ms": parts,
            "dominant": {"part": top, "share": parts[top] / sum(parts.values())},
            "timed_as": "median of per-step CUDA events, one CUDA graph per step, the L2 "
                        "flushed (512 MB written) before every step; parts timed eagerly the "
                        "same way (top-k = index + top-k minus index)"}


def measure_prefill(C, W, wid, layout, dev, stream, steps, warmup):
    """Chunked prefill of one sequence: the Full layer's causal index scores
    (with each token's score-key histogram, built by the indexer's epilogue)
    and top-512 of every new token from them, then the readout of the Full
    and the Reuse layers (one launch).  Roofline: the dense bf16 tensor pipe (sustained figure) on
    the step's FLOPs (indexer over the visible entries, attention over the
    selected entries and the causal window)."""
    import torch
    wl = W.WORKLOADS[wid]
    L, T = wl.layers, wl.n_queries()
    n_ent = int(wl.n_entries()[0])
    cache = C.Cache(C.config(ratio=wl.ratio, layout=layout), [n_ent], device=dev)
    W.fill_cache(wl, cache)
    q_idx, w = W.dev_q_idx(wl), W.dev_w(wl)
    qs = [W.dev_q(wl, l) for l in range(L)]
    rows = [W.dev_swa(wl, l) for l in range(L)]
    ld = (n_ent + 3) // 4 * 4
    scores = torch.empty(T, ld, dtype=torch.float32, device=dev)
    topk = torch.empty(T, 512, dtype=torch.int32, device=dev)
    hist = torch.empty(T, 2048, dtype=torch.int32, device=dev)
    outs = [torch.empty(T, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    n_valid = [min(n_ent, (wl.pos0 + i + 1) // wl.ratio) for i in range(T)]
    scale = 512 ** -0.5

    def index():
        C.csa2_index_scores_prefill(cache, 0, wl.pos0, q_idx, w, scores, key_hist=hist)

    def select():
        C.csa2_topk(scores, n_valid, 512, idx_out=topk, key_hist=hist)

    def readout():
        C.csa2_sparse_attn_prefill_layers(cache, 0, wl.pos0, qs, rows, wl.swa_pos0, topk, scale,
                                          outs)

    for _ in range(warmup):
        index()
        select()
        readout()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in evs:
        e[0].record(stream)
        index()
        e[1].record(stream)
        select()
        e[2].record(stream)
        readout()
        e[3].record(stream)
    torch.cuda.synchronize()
    if cache.device_error() != 0:
        raise RuntimeError("device error word set during the prefill measurement")
    ms = statistics.median(e[0].elapsed_time(e[3]) for e in evs)
    t_idx = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    t_sel = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    t_att = statistics.median(e[2].elapsed_time(e[3]) for e in evs)
    idx_flops = 2.0 * 32 * 128 * sum(n_valid)            # visible entries only
    cand = [min(512, n) + min(128, wl.pos0 + i - wl.swa_pos0 + 1) for i, n in enumerate(n_valid)]
    attn_flops = L * 64 * 512 * 4.0 * sum(cand)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(peaks.get("bf16_tflops_sustained", 1700.0))
    peak_kind = "measured bf16 cuBLAS, sustained" if "bf16_tflops_sustained" in peaks \
        else "fallback"
    tf = lambda f, t: f / (t / 1000) / 1e12
    parts = {"index_scores": t_idx, "topk": t_sel, "sparse_attn_all_layers": t_att}
    top = max(parts, key=parts.get)
    del cache
    return {"workload": wl.name, "batch": 1, "new_tokens": T, "prefix_tokens": wl.ctx,
            "entries": n_ent, "ratio": wl.ratio, "layers": f"1 Full + {L - 1} Reuse",
            "layout": "L32_UE8M0" if layout == 0 else "L16_E4M3",
            "ms_per_step": ms, "value": T / (ms / 1000), "unit": UNIT, "steps": steps,
            "roofline": {"bound": "tensor", "flops_per_step": idx_flops + attn_flops,
                         "achieved": tf(idx_flops + attn_flops, ms), "peak": peak,
                         "unit": "TFLOP/s", "frac": tf(idx_flops + attn_flops, ms) / peak,
                         "peak_kind": peak_kind},
            "parts_tensor_frac": {"index_scores": tf(idx_flops, t_idx) / peak,
                                  "sparse_attn_all_layers": tf(attn_flops, t_att) / peak},
            "kernel_ms": parts,
            "dominant": {"part": top, "share": parts[top] / sum(parts.values())},
            "timed_as": "median of per-step CUDA events around eager calls (inputs larger "
                        "than L2: 2.3 GB of scores per step)"}


def run_prefill(args):
    """Chunked prefill of one sequence (workload 4) as its own line: 8192 new
    tokens on a 131072-token prefix, ratio 2."""
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import fp4_kv_cache_index_gb300 as C
    from csa2_synth import workloads as W
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local).start()
    barrier(world)
    r = measure_prefill(C, W, args.workload, args.layout, dev, stream, args.steps, args.warmup)
    barrier(world)
    clocks = sampler.stop()
    ms = max_over_ranks(r["ms_per_step"], world, dev)
    wl = W.WORKLOADS[args.workload]
    line = {
        "metric": "CSA2 prefill query-tokens/s, 8192 tokens on a 128K prefix; tensor-pipe "
                  "TFLOP/s vs peak",
        "value": r["new_tokens"] * world / (ms / 1000), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {k: r[k] for k in ("workload", "batch", "new_tokens", "prefix_tokens",
                                     "entries", "ratio", "layers", "layout")},
        "roofline": r["roofline"], "parts_tensor_frac": r["parts_tensor_frac"],
        "kernel_ms": r["kernel_ms"],
        # the indexer, one top-k launch per 1024 rows, one readout launch
        "gpu_launches": args.steps * (1 + (wl.n_queries() + 1023) // 1024 + 1),
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def measure_decoder(C, W, dev, stream, iters, hbm_peak, max_blocks=2048):
    """The pages' decoder (V4.1 report, section 4.2.1: 20 CSA2 layers at
    ratio 1 in five groups of four; group 1 = Full + 3 Reuse, groups 2-5 =
    Reindex + 3 Reuse; a Hierarchical Sparse Indexer pool of 2048 blocks of
    8) over the pages' cache formats (main KV E2M1 + E4M3/16, indexer keys
    and queries MXFP4, FP8 window rows), one decode step for batch 64 at
    128K context: Full index + top-k + pool, 4 x Reindex selection, 20
    readouts.  The step runs as two micro-batches of 32 sequences on two
    streams (the single-stream step is reported beside it; for the one group
    of the paper-cache step the same split was slower, 0.234 against 0.223
    ms, so that step stays on one stream).  Timed as one CUDA graph per
    step, median over `iters`."""
    import torch
    wl = W.WORKLOADS[2]
    B = wl.batch
    n_ent = [int(x) for x in wl.n_entries()]
    cache = C.Cache(C.config(ratio=wl.ratio, layout=1, idx_layout=1), n_ent, device=dev)
    W.fill_cache(wl, cache)
    n_layers, n_groups = 20, 5
    qi = [W.dev_q_idx(wl, layer=g) for g in range(n_groups)]
    wi = [W.dev_w(wl, layer=g) for g in range(n_groups)]
    qs = [W.dev_q(wl, l) for l in range(n_layers)]
    swas = [C.csa2_swa_fp8_quantise(W.dev_swa(wl, l)) for l in range(n_layers)]
    ld = (max(n_ent) + 3) // 4 * 4
    scores = torch.empty(B, ld, dtype=torch.float32, device=dev)
    hist = torch.empty(B, 2048, dtype=torch.int32, device=dev)
    tws = torch.empty(max(16, C.csa2_topk_workspace_bytes(B, max(n_ent))), dtype=torch.uint8,
                      device=dev)
    aws = torch.empty(max(16, C.csa2_sparse_attn_workspace_bytes(cache, B)), dtype=torch.uint8,
                      device=dev)
    pool = torch.empty(B, max_blocks, dtype=torch.int32, device=dev)
    pws = torch.empty(max(16, int(C.lib.csa2_hsi_pool_workspace_bytes(B, max(n_ent)))),
                      dtype=torch.uint8, device=dev)
    rws = torch.empty(max(16, int(C.lib.csa2_index_reindex_workspace_bytes(
        cache.handle, B, max_blocks))), dtype=torch.uint8, device=dev)
    topks = [torch.empty(B, 512, dtype=torch.int32, device=dev) for _ in range(n_groups)]
    outs = [torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    scale = 512 ** -0.5

    def select(g):
        if g == 0:
            C.csa2_index_scores_decode(cache, qi[0], wi[0], scores, key_hist=hist)
            C.csa2_topk(scores, n_ent, 512, idx_out=topks[0], key_hist=hist, workspace=tws)
            C.csa2_hsi_pool(scores, n_ent, max_blocks, pool_blocks=pool, workspace=pws)
        else:
            C.csa2_index_topk_reindex_decode(cache, qi[g], wi[g], pool, topk_idx=topks[g],
                                             workspace=rws)

    def readout(g):
        ls = slice(4 * g, 4 * g + 4)
        C.csa2_sparse_attn_decode_layers(cache, qs[ls], None, topks[g], scale, outs[ls], None,
                                         workspace=aws, swa_fp8s=swas[ls])

    def step():
        for g in range(n_groups):
            select(g)
            readout(g)

    # the schedule: two micro-batches of 32 sequences on two streams, each
    # through the groups in order, so that one micro-batch's readouts
    # (latency-bound) run beside the other's selections (bandwidth-bound);
    # the readouts unsplit, as in the headline schedule
    M = 2
    streams = [torch.cuda.Stream() for _ in range(M)]
    no_split = torch.empty(0, dtype=torch.uint8, device=dev)
    mbs = []
    for m in range(M):
        lo, hi = B * m // M, B * (m + 1) // M
        n = hi - lo
        nv = n_ent[lo:hi]
        mbs.append(dict(
            seq=list(range(lo, hi)), nv=nv, qi=[t[lo:hi] for t in qi], wi=[t[lo:hi] for t in wi],
            qs=[t[lo:hi] for t in qs],
            swas=[tuple(x[lo * 128:hi * 128] for x in f) for f in swas],
            scores=torch.empty(n, ld, dtype=torch.float32, device=dev),
            hist=torch.empty(n, 2048, dtype=torch.int32, device=dev),
            tws=torch.empty(max(16, C.csa2_topk_workspace_bytes(n, max(nv))), dtype=torch.uint8,
                            device=dev),
            pool=torch.empty(n, max_blocks, dtype=torch.int32, device=dev),
            pws=torch.empty(max(16, int(C.lib.csa2_hsi_pool_workspace_bytes(n, max(nv)))),
                            dtype=torch.uint8, device=dev),
            rws=torch.empty(max(16, int(C.lib.csa2_index_reindex_workspace_bytes(
                cache.handle, n, max_blocks))), dtype=torch.uint8, device=dev),
            topks=[torch.empty(n, 512, dtype=torch.int32, device=dev) for _ in range(n_groups)],
            outs=[torch.empty(n, 64, 512, dtype=torch.bfloat16, device=dev)
                  for _ in range(n_layers)]))

    def mb_select(d, g):
        if g == 0:
            C.csa2_index_scores_decode(cache, d["qi"][0], d["wi"][0], d["scores"], seq_ids=d["seq"],
                                       key_hist=d["hist"])
            C.csa2_topk(d["scores"], d["nv"], 512, idx_out=d["topks"][0], key_hist=d["hist"],
                        workspace=d["tws"])
            C.csa2_hsi_pool(d["scores"], d["nv"], max_blocks, pool_blocks=d["pool"],
                            workspace=d["pws"])
        else:
            C.csa2_index_topk_reindex_decode(cache, d["qi"][g], d["wi"][g], d["pool"],
                                             seq_ids=d["seq"], topk_idx=d["topks"][g],
                                             workspace=d["rws"])

    def mb_readout(d, g):
        ls = slice(4 * g, 4 * g + 4)
        C.csa2_sparse_attn_decode_layers(cache, d["qs"][ls], None, d["topks"][g], scale,
                                         d["outs"][ls], None, seq_ids=d["seq"],
                                         workspace=no_split, swa_fp8s=d["swas"][ls])

    def step_mb():
        # each micro-batch on its stream through the groups in order (capping
        # the indexers' grids or ordering the selections across the
        # micro-batches, as the headline schedule does, was slower here)
        main = torch.cuda.current_stream()
        for s_ in streams:
            s_.wait_stream(main)
        for g in range(n_groups):
            for s_, d in zip(streams, mbs):
                with torch.cuda.stream(s_):
                    mb_select(d, g)
                    mb_readout(d, g)
        for s_ in streams:
            main.wait_stream(s_)

    for _ in range(3):
        step()
    gr1 = capture(step, stream)
    for _ in range(3):
        step_mb()
    gr = capture(step_mb, stream)
    for _ in range(3):
        gr1.replay()
        gr.replay()
    t = per_step_ms(gr.replay, iters, stream)
    t1 = per_step_ms(gr1.replay, iters, stream)
    t_full = per_step_ms(lambda: select(0), iters, stream)
    t_re = per_step_ms(lambda: select(1), iters, stream)
    t_rd = per_step_ms(lambda: readout(1), iters, stream)
    if cache.device_error() != 0:
        raise RuntimeError("device error word set during the decoder measurement")
    ms = statistics.median(t)
    q_bytes = B * (32 * 128 * 2 + 32 * 4)
    full_bytes = sum(n_ent) * 68 + q_bytes + sum(n_ent) * 4          # keys, queries, pool's scores
    re_bytes = B * (max_blocks * 8 * 68) + q_bytes
    rd_bytes = B * (512 * 288 + 128 * 584 + 2 * 64 * 1024)
    step_bytes = full_bytes + (n_groups - 1) * re_bytes + n_layers * rd_bytes
    gbs = step_bytes / (ms / 1000) / 1e9
    del cache
    return {"layout": "decoder of 20 layers: [Full + 3 Reuse] + 4 x [Reindex + 3 Reuse], "
                      "pool of 2048 blocks x 8",
            "formats": "main KV E2M1 + E4M3/16 (288 B), indexer K MXFP4 (68 B), window FP8 "
                       "(584 B/row)",
            "batch": B, "entries_per_seq": n_ent[0],
            "ms_per_step": ms, "ms_per_step_min": min(t), "ms_per_step_max": max(t),
            "value": B / (ms / 1000), "unit": "query-tokens/s through the 20 decoder layers",
            "schedule": "two micro-batches of 32 on two streams, each through the five groups "
                        "in order, one micro-batch's readouts beside the other's selections",
            "single_stream_ms": statistics.median(t1),
            "roofline": {"bound": "hbm", "algorithmic_bytes_per_step": step_bytes,
                         "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "frac_nominal": gbs / 8000.0},
            "parts_ms": {"full_selection_and_pool": statistics.median(t_full),
                         "reindex_selection": statistics.median(t_re),
                         "readout_4_layers": statistics.median(t_rd)},
            "timed_as": "median of per-step CUDA events, one CUDA graph per step (keys 17x "
                        "larger than L2, read evict-first); parts eager"}


def run_pages_formats_only(args):
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import fp4_kv_cache_index_gb300 as C
    from csa2_synth import workloads as W
    hbm_peak, _ = measured_peaks()
    stream = torch.cuda.current_stream()
    iters = max(3, args.steps)
    r = {"paper_cache": measure_paper_cache(C, W, W.WORKLOADS[2], dev, stream, iters, hbm_peak),
         "decoder": measure_decoder(C, W, dev, stream, iters, hbm_peak)}
    print(json.dumps(r), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.pages_formats_only:
        return run_pages_formats_only(args)
    from csa2_synth.workloads import WORKLOADS
    if WORKLOADS[args.workload].prefill:
        return run_prefill(args)
    return run_csa2(args)


if __name__ == "__main__":
    sys.exit(main())
