#!/usr/bin/env python3
"""Benchmark of one LoGRA optimiser step on GB300: sketch every microbatch of
every compressed matrix, then apply RowAdam from the sketch.

A step covers, for each layer and each projection matrix (q, k, v, o, gate,
up, down): zero S and one logra_sketch_accumulate per microbatch; then, per
layer, one logra_rowadam_apply_group call over the layer's seven matrices
(fp32 master W, bf16 working copy, v, norms; --apply-mode single: one
logra_rowadam_apply_ex per matrix instead).  Inputs
(bf16 X and dY for every microbatch) are resident in HBM before timing; they
are far larger than L2, so no L2 flush is needed between steps.

Default workload: the 7B-class model, all 28 decoder layers (q/o 3584x3584,
k/v 512x3584, gate/up 18944x3584, down 3584x18944), r = 256, 8 microbatches x
8192 tokens, 25% padding rows.  Its inputs (330 GB of bf16 X and dY per step)
do not fit in one GPU's memory, so they come from a resident pool of
--input-layers layers' inputs (default 4, 47 GB): layer l reads pool slot
l mod P.  Every layer still has its own weights, sketch, v and sign matrices
(per-matrix seeds), so the kernel work per layer is unchanged; only the input
values repeat, 47 GB apart, far beyond L2.  --workload layers27b (4 layers of
27B-class shapes, 16 x 8192 tokens, r in {128, 256, 512}) and the smaller
workloads remain available.  The metric is sketch TFLOP/s over the whole step (algorithmic
sketch FLOPs 2 n r (k + d) per matrix-microbatch, divided by the step time
including the apply), with the apply's GB/s and both kernels' roofline
fractions alongside.  The matrices are independent, so the step issues them
round robin on --streams CUDA streams (default 16, 8 for workloads of fewer than 16
matrices); per-call durations (the
components and the dominant call's roofline) come from one extra step on a
single stream right after the timed region; the apply component also reports all of a
step's apply calls issued at once on up to --apply-streams streams (default 7), and
the whole step is captured once in a CUDA graph whose replays are timed as a
further component (--graph times the step that way instead).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank sketches its own microbatches (weak
scaling), all-reduces each S, then applies; rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sketch TFLOP/s + fused RowAdam-apply GB/s per GB300; % of roofline"

# DRAM bytes (read + write) of one logra_sketch_accumulate call, summed over
# its three launches, from one ncu capture per shape of the kernels as they
# stood when captured (the profile summaries name the capture): key
# (n, d, k, r) -> (bytes, what was captured).  Shapes without an entry report
# null traffic.
SKETCH_TRAFFIC_PER_CALL = {
    # one stream: project 67.18 + 0.00 MB, split 8.40 + 0 MB, accumulate (CTA pairs) 338.2 + 8.6 MB
    # (incl. re-zeroing P^T); under the concurrency hint the call moves 397.1 MB (no split, X read once)
    (8192, 18944, 3584, 256): (422.4e6, "ncu dram__bytes_read.sum + dram__bytes_write.sum of the three launches "
                                        "of one 18944x3584 gate call on one stream, kernels as they stand"),
    # one stream: project 92.35 + 0.10 MB, split 8.40 + 0 MB, accumulate (CTA pairs) 516.65 + 31.62 MB
    (8192, 27648, 5120, 256): (649.1e6, "ncu dram__bytes_read.sum + dram__bytes_write.sum of the three launches "
                                        "of one 27648x5120 gate call on one stream, kernels as they stand"),
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="model7b")
    p.add_argument("--rank", type=int, default=None, help="sketch rank r (default: the workload's)")
    p.add_argument("--layers", type=int, default=None, help="override the workload's layer count")
    p.add_argument("--microbatches", type=int, default=None,
                   help="override the workload's microbatches per step (small profiling cases)")
    p.add_argument("--input-layers", type=int, default=4,
                   help="distinct layers of resident inputs; layer l reads the inputs of slot l mod this "
                        "(0: every layer its own inputs)")
    p.add_argument("--streams", type=int, default=None,
                   help="CUDA streams the matrices are issued on, round robin (each keeps its own workspace); "
                        "default 16 for workloads of at least 16 matrices per step, else 8")
    p.add_argument("--hint", type=int, default=None,
                   help="concurrency hint given to the library (default: the stream count)")
    p.add_argument("--apply-streams", type=int, default=7,
                   help="streams for the all-applies-at-once measurement (each with its own workspace)")
    p.add_argument("--spread", choices=("auto", "on", "off"), default="auto",
                   help="issue a matrix's microbatch calls round robin over the streams (they add into the same "
                        "S with atomic reductions); auto: when the workload has at most half as many matrices as "
                        "streams")
    p.add_argument("--apply-mode", choices=("group", "single"), default="group",
                   help="group: one logra_rowadam_apply_group call per layer (its matrices in shared launches); "
                        "single: one logra_rowadam_apply_ex call per matrix")
    p.add_argument("--graph", action="store_true",
                   help="time the step as replays of one CUDA graph (value); by default the graph-replayed "
                        "step is reported as a component after the eager timed region")
    p.add_argument("--no-graph", action="store_true", help="skip the CUDA graph component")
    p.add_argument("--e2e-steps", type=int, default=2)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    return p.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_config(w, layers, nmb, r, world, pool):
    """The `config` object of the JSON line: what defines the workload, identical in both arms."""
    return {"workload": w.name, "layers": layers, "matrices": [list(x) for x in w.matrices],
            "microbatches": nmb, "tokens": w.tokens, "r": r, "mask_frac": w.mask_frac,
            "input_pool_layers": pool, "l2": "inputs larger than L2, no flush", "parallelism": f"dp{world}"}


# ----------------------------------------------------------------------------- work accounting
def sketch_work(n, d, k, r):
    """Algorithmic FLOPs and bytes of one matrix-microbatch sketch (bf16 X, dY; fp32 S RMW)."""
    return 2.0 * n * r * (k + d), 2.0 * n * (k + d) + 2.0 * d * r * 4


def apply_work(d, k, r):
    """Algorithmic FLOPs and bytes of one apply: W fp32 RMW + bf16 copy + S read + v RMW."""
    return 2.0 * d * k * r, d * k * (4 + 4 + 2) + d * r * 4 + 2.0 * d * 4


# ----------------------------------------------------------------------------- clocks
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            # start timing only once the sampler is producing rows (nvidia-smi takes a moment to start)
            deadline = time.time() + 5.0
            while time.time() < deadline and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
                time.sleep(0.02)
            self.skip = 0
            with open(self.path) as f:
                self.skip = sum(1 for _ in f)        # rows taken before the timed region
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for i, line in enumerate(f):
                if i < getattr(self, "skip", 0):
                    continue
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle timing
def time_oracle(w, r, seconds, host_seed=0):
    """Time the fp64 oracle on a bounded sample of the workload: microbatches of
    the q matrix (d = k = hidden) until ``seconds`` pass, plus one apply of that
    matrix; extrapolate to the step's ratio of microbatches to applies."""
    import numpy as np
    from oracle import logra_oracle as O
    from rank_gradient_sketching_02_gb300 import synth
    name, d, k = w.matrices[0]
    n = w.tokens
    X, dY, _ = synth.host_microbatch(n, d, k, dy_kind=w.dy_kind, dy_std=w.dy_std, mask_frac=w.mask_frac,
                                     key=(host_seed, 0, 0, 0))
    X64 = synth.to_bf16_bits(X).double().numpy()
    dY64 = synth.to_bf16_bits(dY).double().numpy()
    S = np.zeros((d, r))
    t0 = time.perf_counter()
    mbs = 0
    while True:
        S = O.sketch_accumulate(S, X64, dY64, 1, 0, r)
        mbs += 1
        if time.perf_counter() - t0 >= seconds * 0.75:
            break
    t_mb = (time.perf_counter() - t0) / mbs
    W = np.zeros((d, k))
    t1 = time.perf_counter()
    O.rowadam_apply(W, S, np.zeros(d), 1, 0, 0.999, 1e-8, 1e-6, 1.0)
    t_apply = time.perf_counter() - t1
    f_mb, _ = sketch_work(n, d, k, r)
    _, b_apply = apply_work(d, k, r)
    t_unit = w.microbatches * t_mb + t_apply        # one matrix, one step
    value = w.microbatches * f_mb / t_unit / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": (f"fp64 numpy oracle on the {name} matrix ({d}x{k}, r={r}): {mbs} microbatch sketches of "
                       f"{n} tokens ({t_mb:.2f} s each) and one apply ({t_apply:.2f} s, "
                       f"{b_apply / t_apply / 1e9:.2f} GB/s); value = {w.microbatches} microbatches' sketch "
                       f"FLOPs / ({w.microbatches} sketches + 1 apply)")}


def time_oracle_one_thread(workload, r, seconds):
    """The same bounded oracle sample in a child process whose BLAS and OpenMP pools have one thread."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS"):
        env[var] = "1"
    code = ("import json, sys; sys.path.insert(0, %r); import bench; from rank_gradient_sketching_02_gb300 import "
            "synth; print(json.dumps(bench.time_oracle(synth.WORKLOADS[%r], %d, %f)))" % (ROOT, workload, r, seconds))
    try:
        p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT,
                           timeout=max(60.0, 10 * seconds))
        if p.returncode != 0:
            return None
        res = json.loads(p.stdout.strip().splitlines()[-1])
        res["cores"] = 1
        return res
    except Exception:  # noqa: BLE001 - a missing one-thread figure does not fail the bench
        return None


def run_reference(args):
    """Reference arm: the fp64 CPU oracle, as it stands, on the machine's host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from rank_gradient_sketching_02_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    r = args.rank or w.r
    layers = args.layers or w.layers
    pool = layers if args.input_layers <= 0 else min(layers, args.input_layers)
    per_step = max(2.0, args.cpu_seconds / 2)
    for _ in range(args.warmup):
        time_oracle(w, r, 0.5)
    vals = []
    t0 = time.perf_counter()
    res = None
    for _ in range(args.steps):
        res = time_oracle(w, r, per_step)
        vals.append(res["value"])
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(w, layers, args.microbatches or w.microbatches, r, args.gpus, pool),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": res["cores"], "kind": "oracle",
                             "sample": res["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import __graft_entry__
    __graft_entry__.build()
    import rank_gradient_sketching_02_gb300 as L
    from rank_gradient_sketching_02_gb300 import dp, synth

    w = synth.WORKLOADS[args.workload]
    r = args.rank or w.r
    layers = args.layers or w.layers
    n, nmb = w.tokens, args.microbatches or w.microbatches
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = torch.device("cuda", local)
    beta2, eps, lr, c = synth.BETA2, synth.EPS, synth.LR, synth.C

    # ---- resident state and inputs (the input generation is timed on its own, outside the step)
    # Inputs of `pool` distinct layers stay resident; layer l reads slot l mod pool (every layer
    # keeps its own W, S, v and seeds, so the work per layer is the same as with its own inputs).
    # The projections that read one activation share it (q/k/v, gate/up: synth.input_group), and
    # every tensor of a microbatch has the same padding rows.
    pool = layers if args.input_layers <= 0 else min(layers, args.input_layers)
    mats = []
    x_inputs, dy_inputs = {}, {}
    gen_ms = 0.0
    # each layer's sketches are views of one buffer (dp.SketchArena): zeroed and, under torchrun,
    # summed over the ranks as one collective per layer
    arenas = [dp.SketchArena([d for _, d, _ in w.matrices], r, device=dev, bucket_bytes=1 << 62)
              for _ in range(layers)]
    for layer in range(layers):
        for mi, (name, d, k) in enumerate(w.matrices):
            gen = torch.Generator(device=dev)
            gen.manual_seed(1000 + 16 * layer + mi)
            W = torch.empty((d, k), dtype=torch.float32, device=dev).normal_(0.0, 0.02, generator=gen)
            ls, grp = layer % pool, synth.input_group(name)
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record()
            if (ls, grp) not in x_inputs:
                Xs = torch.empty((nmb, n, k), dtype=dt, device=dev)
                for mb in range(nmb):
                    synth.device_activations(n, k, mask_frac=w.mask_frac, key=(2026, rank, ls, grp, mb),
                                             mb_key=(2026, rank, ls, mb), dtype=dt, device=dev, out=Xs[mb])
                x_inputs[(ls, grp)] = Xs
            if (ls, mi) not in dy_inputs:
                Ys = torch.empty((nmb, n, d), dtype=dt, device=dev)
                for mb in range(nmb):
                    synth.device_output_grads(n, d, dy_kind=w.dy_kind, dy_std=w.dy_std, mask_frac=w.mask_frac,
                                              key=(2027, rank, ls, mi, mb), mb_key=(2026, rank, ls, mb), dtype=dt,
                                              device=dev, out=Ys[mb])
                dy_inputs[(ls, mi)] = Ys
            g1.record()
            g1.synchronize()
            gen_ms += g0.elapsed_time(g1)
            m = {"name": name, "layer": layer, "d": d, "k": k, "seed": synth.matrix_seed(2026, layer, mi), "W": W,
                 "Wb": W.to(torch.bfloat16), "v": torch.zeros(d, dtype=torch.float32, device=dev),
                 "S": arenas[layer][mi], "arena": arenas[layer],
                 "norms": torch.zeros(2, dtype=torch.float64, device=dev),
                 "group": grp, "X": x_inputs[(ls, grp)], "dY": dy_inputs[(ls, mi)]}
            mats.append(m)
    torch.cuda.synchronize()
    layer_mats = [[m for m in mats if m["layer"] == li] for li in range(layers)]

    def group_items(ms):
        return [{"W": m["W"], "S": m["S"], "v": m["v"], "seed": m["seed"], "lr": lr, "c": c,
                 "norms_out": m["norms"], "W_bf16_out": m["Wb"]} for m in ms]
    input_bytes = sum(t.numel() * t.element_size() for t in list(x_inputs.values()) + list(dy_inputs.values()))
    # one X per (layer, input group) and one dY per matrix, every microbatch
    step_input_bytes = 0
    for lm in layer_mats:
        seen = set()
        for mm in lm:
            step_input_bytes += mm["dY"].numel() * mm["dY"].element_size()
            if mm["group"] not in seen:
                seen.add(mm["group"])
                step_input_bytes += mm["X"].numel() * mm["X"].element_size()

    # a side stream as the step's main stream (a CUDA graph cannot be captured on the legacy
    # default stream, and the library's per-stream workspaces must be the ones warmed up)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    # pre-size the per-stream workspace so no allocation happens while timing
    ws = max(max(L.lib().logra_sketch_workspace_bytes(n, m["d"], m["k"], r, 1 if dt == torch.bfloat16 else 0),
                 L.lib().logra_apply_workspace_bytes(m["d"], m["k"], r)) for m in mats)
    ws = max([ws] + [L.logra_apply_group_workspace_bytes(group_items(lm)) for lm in layer_mats])
    # The matrices are independent, so they are issued round robin on `--streams` CUDA streams (each
    # with its own library workspace): one matrix's launches fill the SMs that another's leave idle
    # in its tails and launch gaps.  Each matrix's own calls stay in order on one stream.
    nstreams = args.streams or (16 if len(mats) >= 16 else 8)
    streams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(max(1, nstreams) - 1)]
    hint = args.hint or len(streams)
    for st in streams:
        with torch.cuda.stream(st):
            L.logra_reserve_workspace(ws)

    def timed(ev, kind, st, fn, *tag):
        if ev is None:
            fn()
            return
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        ev[kind].append((a, b) + tag)

    # auto: only when at least half of the streams would otherwise sit idle (one or two matrices);
    # spreading costs an event round trip per call, which a host-bound step of many matrices feels
    spread = (2 * len(mats) <= len(streams)) if args.spread == "auto" else (args.spread == "on")

    def one_step(step_idx, ev=None, sts=None):
        sts = sts or streams
        for st in sts[1:]:
            st.wait_stream(stream)
        i = 0
        for li, lm in enumerate(layer_mats):
            used = []
            for m in lm:
                st = sts[i % len(sts)]
                used.append(st)
                if spread and len(sts) > 1:
                    # the matrix's microbatches round robin over the streams, after S is zeroed on the
                    # matrix's own stream; the others join it before the all-reduce and the apply
                    with torch.cuda.stream(st):
                        m["S"].zero_()
                    zeroed = torch.cuda.Event()
                    zeroed.record(st)
                    mb_streams = []
                    for mb in range(nmb):
                        smb = sts[(i + mb) % len(sts)]
                        if smb is not st and smb not in mb_streams:
                            smb.wait_event(zeroed)
                        mb_streams.append(smb)
                        with torch.cuda.stream(smb):
                            L.logra_sketch_accumulate(m["X"][mb], m["dY"][mb], m["S"], m["seed"], step_idx)
                    for smb in set(mb_streams):
                        if smb is not st:
                            st.wait_stream(smb)
                    i += 1
                    with torch.cuda.stream(st):
                        if args.apply_mode == "single":
                            dp.allreduce_sketch(m["S"])
                            L.logra_rowadam_apply_ex(m["W"], m["S"], m["v"], m["seed"], step_idx, beta2, eps, lr,
                                                     c, m["norms"], m["Wb"], None)
                    continue
                i += 1
                with torch.cuda.stream(st):
                    m["S"].zero_()
                    for mb in range(nmb):
                        timed(ev, "sketch", st, lambda: L.logra_sketch_accumulate(
                            m["X"][mb], m["dY"][mb], m["S"], m["seed"], step_idx), m["d"], m["k"])
                    if args.apply_mode == "single":
                        dp.allreduce_sketch(m["S"])
                        timed(ev, "apply", st, lambda: L.logra_rowadam_apply_ex(
                            m["W"], m["S"], m["v"], m["seed"], step_idx, beta2, eps, lr, c, m["norms"], m["Wb"],
                            None), m["d"], m["k"])
            if args.apply_mode == "group":
                # the layer's applies as one call, on the stream of its last matrix, once all of the
                # layer's sketches (on the other streams) are done
                ast = used[-1]
                for st in set(used):
                    if st is not ast:
                        ast.wait_stream(st)
                with torch.cuda.stream(ast):
                    arenas[li].allreduce()
                    timed(ev, "apply", ast, lambda: L.logra_rowadam_apply_group(
                        group_items(lm), step_idx, beta2, eps), li, len(lm))
        for st in sts[1:]:
            stream.wait_stream(st)

    def barrier():
        if world > 1:
            dist.barrier()

    # the step issues sketch calls on len(streams) streams at once: tell the library, so that
    # each call's accumulate leaves SMs to the other streams (the launch shape only)
    L.logra_set_concurrency(hint)
    for s in range(args.warmup):
        one_step(s)
    torch.cuda.synchronize()
    if L.logra_get_status() != 0:
        raise RuntimeError("device status word set during warm-up")
    def capture_step(step_idx):
        """One whole step (every stream's work, fork and join) captured in a CUDA graph; the
        graph's sign matrices are those of `step_idx`, and every replay runs all of the step's
        kernels again on the same resident inputs and state."""
        g = torch.cuda.CUDAGraph()
        l0 = L.logra_launch_count()
        with torch.cuda.graph(g, stream=stream):
            one_step(step_idx)
        n_launch = L.logra_launch_count() - l0
        g.replay()                          # one untimed replay after instantiation
        torch.cuda.synchronize()
        if L.logra_get_status() != 0:
            raise RuntimeError("device status word set by the captured step")
        return g, n_launch

    graph = None
    if args.graph:
        graph, graph_launches = capture_step(args.warmup)
    barrier()
    torch.cuda.synchronize()

    clocks = Clocks(local)
    launches0 = L.logra_launch_count()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            one_step(args.warmup + s)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    launches = L.logra_launch_count() - launches0
    if graph is not None:
        launches = graph_launches * args.steps

    # Per-call durations come from one more step issued on a single stream right after the
    # timed region, with CUDA events around every call on that stream: inside the multi-stream
    # step a call's event span would also cover the other streams' kernels.
    ev = {"sketch": [], "apply": []}
    L.logra_set_concurrency(1)
    one_step(args.warmup + args.steps, ev, [stream])
    torch.cuda.synchronize()

    # The applies of a step are independent too: one more measurement issues all of them at
    # once on the same streams (fork/join on the main stream, CUDA events there), so one
    # matrix's short prep / row-norm launches overlap another's update pass.
    ap_streams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(max(1, args.apply_streams) - 1)]
    for st in ap_streams[1:]:
        with torch.cuda.stream(st):
            L.logra_reserve_workspace(ws)

    def apply_phase(step_idx):
        for st in ap_streams[1:]:
            st.wait_stream(stream)
        if args.apply_mode == "group":
            for li, lm in enumerate(layer_mats):
                with torch.cuda.stream(ap_streams[li % len(ap_streams)]):
                    L.logra_rowadam_apply_group(group_items(lm), step_idx, beta2, eps)
        else:
            for i, m in enumerate(mats):
                with torch.cuda.stream(ap_streams[i % len(ap_streams)]):
                    L.logra_rowadam_apply_ex(m["W"], m["S"], m["v"], m["seed"], step_idx, beta2, eps, lr, c,
                                             m["norms"], m["Wb"], None)
        for st in ap_streams[1:]:
            stream.wait_stream(st)

    apply_phase(args.warmup + args.steps)
    ap_runs = []
    for rep_i in range(3):
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        apply_phase(args.warmup + args.steps + 1 + rep_i)
        a1.record(stream)
        torch.cuda.synchronize()
        ap_runs.append(a0.elapsed_time(a1))
    ap_conc_ms = statistics.median(ap_runs)

    # The same step from the main stream alone through logra_sketch_accumulate_group: per layer one
    # call with every matrix x microbatch sketch (the library spreads them over its own side
    # streams and joins them back), then the layer's grouped apply.  What a caller that issues the
    # backward pass on one stream gets.
    group_comp = None
    if dt == torch.bfloat16 and world == 1:
        def group_step(step_idx):
            for lm in layer_mats:
                for m in lm:
                    m["S"].zero_()
                L.logra_sketch_accumulate_group([{"X": m["X"][mb], "dY": m["dY"][mb], "S": m["S"],
                                                  "seed": m["seed"]} for m in lm for mb in range(nmb)], step_idx)
                lm[0]["arena"].allreduce()
                L.logra_rowadam_apply_group(group_items(lm), step_idx, beta2, eps)

        group_step(args.warmup + args.steps + 20)
        torch.cuda.synchronize()
        q0 = torch.cuda.Event(enable_timing=True)
        q1 = torch.cuda.Event(enable_timing=True)
        gsteps = max(1, min(args.steps, 3))
        q0.record(stream)
        for i in range(gsteps):
            group_step(args.warmup + args.steps + 21 + i)
        q1.record(stream)
        torch.cuda.synchronize()
        group_comp = {"ms_per_step": q0.elapsed_time(q1) / gsteps, "steps": gsteps,
                      "timing": "one logra_sketch_accumulate_group call per layer (all matrices x microbatches) and "
                                "the layer's grouped apply, all issued on the main stream; CUDA events there"}

    # The same step as a CUDA graph (one capture, K timed replays): what launching from the host
    # costs on top of the GPU work.
    graph_comp = None
    if not args.graph and not args.no_graph and world == 1:
        L.logra_set_concurrency(hint)
        g, g_launch = capture_step(args.warmup + args.steps + 8)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph_comp = {"ms_per_step": g0.elapsed_time(g1) / args.steps, "launches_per_step": g_launch,
                      "timing": f"{args.steps} replays of one captured step, CUDA events on the main stream"}
        del g
    # The backward of the largest matrix's Linear layer for one microbatch, as one library call
    # (dX = dY W on the library's tensor-core kernel, then the sketch) against the separate calls a
    # caller would otherwise make (dX through torch.matmul, i.e. cuBLAS, then the sketch); one
    # stream, CUDA events, median of 5 after 3 warm-ups.  Outside the timed step.
    lb_comp = None
    if dt == torch.bfloat16 and world == 1:
        L.logra_set_concurrency(1)
        mb_big = max(mats, key=lambda m: m["d"] * m["k"] + 0.5 * m["d"])
        Xb, dYb, Wb = mb_big["X"][0], mb_big["dY"][0], mb_big["Wb"]
        dXb = torch.empty((n, mb_big["k"]), dtype=torch.bfloat16, device=dev)
        Sb = torch.zeros_like(mb_big["S"])

        def med(fn):
            for _ in range(3):
                fn()
            out = []
            for _ in range(5):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize()
                out.append(e0.elapsed_time(e1))
            return statistics.median(out)

        sd, st_ = mb_big["seed"], args.warmup + args.steps + 40
        t_fused = med(lambda: L.logra_linear_backward(dYb, W=Wb, dX=dXb, X=Xb, S=Sb, seed=sd, step=st_))
        t_sep = med(lambda: (torch.matmul(dYb, Wb, out=dXb), L.logra_sketch_accumulate(Xb, dYb, Sb, sd, st_)))
        t_dx = med(lambda: L.logra_linear_backward(dYb, W=Wb, dX=dXb))
        t_cublas = med(lambda: torch.matmul(dYb, Wb, out=dXb))
        t_sk = med(lambda: L.logra_sketch_accumulate(Xb, dYb, Sb, sd, st_))
        dx_flop = 2.0 * n * mb_big["d"] * mb_big["k"]
        lb_comp = {"shape": {"n": n, "d": mb_big["d"], "k": mb_big["k"], "r": r},
                   "fused_ms": t_fused, "separate_ms": t_sep, "fused_over_separate": t_fused / t_sep,
                   "dx_ms": t_dx, "dx_tflops": dx_flop / (t_dx * 1e-3) / 1e12,
                   "dx_cublas_ms": t_cublas, "dx_cublas_tflops": dx_flop / (t_cublas * 1e-3) / 1e12,
                   "sketch_ms": t_sk,
                   "timing": "fused: one logra_linear_backward call (dX + sketch); separate: torch.matmul "
                             "(cuBLAS) for dX then logra_sketch_accumulate; one stream, CUDA events, "
                             "median of 5 after 3 warm-ups"}
        del dXb, Sb
        L.logra_set_concurrency(hint)

    elapsed_ms = t_start.elapsed_time(t_end)
    if world > 1:
        t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ms_step = elapsed_ms / args.steps
    status = L.logra_get_status()

    # ---- accounting
    sk_f = sk_b = ap_f = ap_b = 0.0
    for m in mats:
        f, b = sketch_work(n, m["d"], m["k"], r)
        sk_f += nmb * f
        sk_b += nmb * b
        f, b = apply_work(m["d"], m["k"], r)
        ap_f += f
        ap_b += b
    sk_ms = sum(a.elapsed_time(b) for a, b, _, _ in ev["sketch"])
    ap_ms = sum(a.elapsed_time(b) for a, b, _, _ in ev["apply"])
    peaks, peak_kind = load_peaks()
    hbm, tc = float(peaks["hbm_gbs"]), float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    value = world * sk_f / (ms_step * 1e-3) / 1e12
    if graph_comp is not None:
        graph_comp["tflops"] = world * sk_f / (graph_comp["ms_per_step"] * 1e-3) / 1e12
    if group_comp is not None:
        group_comp["tflops"] = sk_f / (group_comp["ms_per_step"] * 1e-3) / 1e12

    sk_tflops = sk_f / (sk_ms * 1e-3) / 1e12
    sk_gbs = sk_b / (sk_ms * 1e-3) / 1e9
    ap_gbs = ap_b / (ap_ms * 1e-3) / 1e9
    sk_roof_ms = 1e3 * max(sk_f / (tc * 1e12), sk_b / (hbm * 1e9))
    ap_roof_ms = 1e3 * max(ap_f / (tc * 1e12), ap_b / (hbm * 1e9))

    # Roofline of the dominant call, on the workload's largest matrix shape:
    # algorithmic bytes / FLOPs of one call over its average event-timed duration.
    dmax, kmax = max(((m["d"], m["k"]) for m in mats), key=lambda x: x[0] * x[1] + 0.5 * x[0])
    big = [a.elapsed_time(b) for a, b, d_, k_ in ev["sketch"] if (d_, k_) == (dmax, kmax)]
    call_ms = sum(big) / len(big)
    f1, b1 = sketch_work(n, dmax, kmax, r)
    bound = "tensor" if f1 / (tc * 1e12) > b1 / (hbm * 1e9) else "hbm"
    if bound == "hbm":
        ach = b1 / (call_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm}
    else:
        ach = f1 / (call_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": tc, "unit": "TFLOP/s", "frac": ach / tc}
    traffic = SKETCH_TRAFFIC_PER_CALL.get((n, dmax, kmax, r))
    roof.update({"traffic": traffic[0] if traffic else None,
                 "traffic_source": traffic[1] if traffic else "no ncu capture of this shape: null",
                 "algorithmic_bytes_per_call": b1, "flops_per_call": f1, "ms_per_call": call_ms,
                 "kernel": f"logra_sketch_accumulate on the {dmax}x{kmax} matrix, n={n}, r={r} "
                           "(project + split + accumulate launches)",
                 "peak_source": f"{peak_kind} ({'MEASURED_PEAKS.json' if peak_kind == 'measured' else 'fallback'})"})

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; torch Philox on device)",
        "config": workload_config(w, layers, nmb, r, world, pool),
        "run": {"input_bytes_resident": input_bytes, "input_bytes_per_step": step_input_bytes,
                "shared_activations": "q/k/v read one X, gate/up one X (per layer and microbatch)",
                "input_pool": (f"layer l reads the inputs of resident slot l mod {pool}; W, S, v and the "
                               "sign matrices are per layer") if pool < layers else "every layer its own inputs",
                "input_generation_ms": gen_ms,
                "streams": len(streams), "apply_mode": args.apply_mode,
                "microbatches_spread_over_streams": bool(spread), "concurrency_hint": hint,
                "cuda_graph": bool(args.graph),
                "component_timing": "components and roofline: CUDA events around each call in one "
                "extra step issued on a single stream right after the timed region"},
        "components": {
            "sketch": {"ms_per_step": sk_ms, "tflops": sk_tflops, "gbs": sk_gbs,
                       "frac_of_roofline": sk_roof_ms / sk_ms, "roofline_ms": sk_roof_ms},
            "apply": {"ms_per_step": ap_ms, "gbs": ap_gbs, "frac_hbm": ap_gbs / hbm,
                      "frac_of_roofline": ap_roof_ms / ap_ms, "roofline_ms": ap_roof_ms,
                      "calls_per_step": len(ev["apply"]),
                      "all_applies_on_streams": {"streams": min(len(ap_streams), len(ev["apply"])),
                                                 "ms_per_step": ap_conc_ms,
                                                 "gbs": ap_b / (ap_conc_ms * 1e-3) / 1e9,
                                                 "frac_hbm": ap_b / (ap_conc_ms * 1e-3) / 1e9 / hbm,
                                                 "timing": "median of 3; every apply call of a step issued "
                                                           "round robin on the streams, events on the "
                                                           "main stream around fork and join"}},
        },
        "roofline": roof,
        "cuda_graph_step": graph_comp,
        "one_stream_group_step": group_comp,
        "linear_backward": lb_comp,
        "gpu_launches": launches,
        "clocks": clk,
        "device_status": status,
    }

    # ---- end to end through the public API from pinned host memory
    if not args.no_e2e:
        L.logra_set_concurrency(1)      # one stream
        line["e2e"] = run_e2e(args, L, dp, mats, w, r, dt, dev, stream, sk_f, world, layer_mats, group_items)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(w, r, args.cpu_seconds)
        one = time_oracle_one_thread(w.name, r, max(2.0, args.cpu_seconds / 3))
        if one is not None:
            line["cpu_baseline"]["one_thread"] = {"value": one["value"], "unit": one["unit"], "cores": 1,
                                                  "sample": one["sample"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(args, L, dp, mats, w, r, dt, dev, stream, sk_f, world, layer_mats, group_items):
    """Same step, but every microbatch's inputs come from pinned host memory and the norms go
    back to the host.  Per layer and microbatch the step's inputs are one X per input group
    (q/k/v share one, gate/up one) and one dY per matrix; they are copied on two side streams
    into one of two device slots (double-buffered: the next microbatch's copies overlap this
    one's sketches)."""
    import torch
    from rank_gradient_sketching_02_gb300 import synth
    beta2, eps, lr, c = synth.BETA2, synth.EPS, synth.LR, synth.C
    n, nmb = w.tokens, args.microbatches or w.microbatches
    lm0 = layer_mats[0]
    groups = list(dict.fromkeys(m["group"] for m in lm0))
    # pinned host copies of one microbatch's inputs (re-sent for every layer and microbatch)
    host_x = {g: next(m for m in lm0 if m["group"] == g)["X"][0].cpu().pin_memory() for g in groups}
    host_dy = [m["dY"][0].cpu().pin_memory() for m in lm0]
    slots = [({g: torch.empty_like(host_x[g], device=dev) for g in groups},
              [torch.empty_like(t, device=dev) for t in host_dy]) for _ in range(2)]
    # two copy streams, each moving half of every tensor, so two copy engines work at once
    copies = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    norms_h = torch.empty((len(mats), 2), dtype=torch.float64).pin_memory()
    h2d = d2h = 0

    def e2e_step(step_idx):
        nonlocal h2d, d2h
        done = [None, None]
        i = 0
        for lm in layer_mats:
            for m in lm:
                m["S"].zero_()
            for mb in range(nmb):
                slot = i % 2
                xs, dys = slots[slot]
                readies = []
                for half, cs in enumerate(copies):
                    with torch.cuda.stream(cs):
                        if done[slot] is not None:
                            cs.wait_event(done[slot])
                        lo, hi = (0, n // 2) if half == 0 else (n // 2, n)
                        for g in groups:
                            xs[g][lo:hi].copy_(host_x[g][lo:hi], non_blocking=True)
                        for j in range(len(lm)):
                            dys[j][lo:hi].copy_(host_dy[j][lo:hi], non_blocking=True)
                        ev_r = torch.cuda.Event()
                        ev_r.record(cs)
                        readies.append(ev_r)
                h2d += sum(t.numel() * t.element_size() for t in list(host_x.values()) + host_dy)
                for ev_r in readies:
                    stream.wait_event(ev_r)
                for j, m in enumerate(lm):
                    L.logra_sketch_accumulate(xs[m["group"]], dys[j], m["S"], m["seed"], step_idx)
                ev = torch.cuda.Event()
                ev.record(stream)
                done[slot] = ev
                i += 1
            lm[0]["arena"].allreduce()
            if args.apply_mode == "single":
                for m in lm:
                    L.logra_rowadam_apply_ex(m["W"], m["S"], m["v"], m["seed"], step_idx, beta2, eps, lr, c,
                                             m["norms"], m["Wb"], None)
            else:
                L.logra_rowadam_apply_group(group_items(lm), step_idx, beta2, eps)
            for m in lm:
                norms_h[mats.index(m)].copy_(m["norms"], non_blocking=True)
                d2h += 16
        return norms_h

    e2e_step(10_000)
    torch.cuda.synchronize()
    h2d = d2h = 0
    steps = max(1, args.e2e_steps)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        e2e_step(10_001 + s)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    return {"value": world * sk_f / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d // steps, "d2h_bytes_per_step": d2h // steps,
            "h2d_gbs": (h2d / steps) / (ms * 1e-3) / 1e9,
            "host_inputs": "pinned host copy of one microbatch's inputs of a layer (one X per input group, one "
                           "dY per matrix), re-sent for every layer and microbatch"}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
