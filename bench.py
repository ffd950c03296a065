"""Benchmark of the segmented speculative-verify step on GB300.

One "step" is the whole verify path over one batch: 30 conv layers
(tf_conv_rows), 10 attention layers (tf_attn_partials + tf_attn_merge), the
greedy pick (tf_argmax_rows) and the accept step (tf_accept), captured in one
CUDA graph. Metric: verified rows per second (rows of every stream's window,
all ranks) and the achieved HBM bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..6] [--per-config 3,4,5,6]
                    [--impl tf|reference]
    python bench.py --row markov|block [--workload 3|5] [--steps K] [--warmup W]

Default workload: 64 streams of 16-row windows (1,024 rows), 30 conv + 10
attention layers, key counts log-uniform on [16, 32768]: the largest workload
by rows. The other workloads (1-4, and 6: workload 5 with its rows not
rescaled) are selectable. The same run also times workloads 3, 4, 5 and 6
(``--per-config``), each with its own inputs, table and graph, and reports
them under ``per_config`` (step time, rows/s, HBM fraction, attention fraction).
``--impl reference`` times the float64 CPU oracle on the host cores (one
process per core) on a bounded sample of the same workload.

``--row`` measures one of the draft side's operations on a workload's table of
windows instead of the verify step (default workload 5, the 64 x 16-row
table): ``markov`` the Markov head's chain over every draft row
(tf_markov_chain: the whole chain in one launch for tables of up to 128
streams), ``block`` one layer of the
non-causal block attention (tf_attn_block), ``prompt`` one conv and one
attention layer of a prompt (prefill) call of one stream (tf_prompt_build;
2,048 rows after 14,336 cached keys by default). Each prints its own JSON line.
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
sys.path.insert(0, ROOT)

METRIC = "verified rows/s per segmented verify step"
UNIT = "rows/s"
L2_FLUSH_BYTES = 256 << 20      # > 129 MB L2


class L2Flush:
    """Evicts the step's data from L2 between timed steps (outside the events):
    256 MB written; with mode "clean" (the default) a second 256 MB buffer is
    then read, so the dirty lines of the write are written back before the
    timed region instead of inside it."""

    def __init__(self, torch, dev, mode):
        self.mode = mode
        self.wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.rbuf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev) if mode == "clean" else None
        self.desc = ("flushed: 256 MB written, then 256 MB of another buffer read, between timed steps, "
                     "outside the events" if mode == "clean"
                     else "flushed: 256 MB written between timed steps, outside the events")

    def __call__(self):
        self.wbuf.zero_()
        if self.rbuf is not None:
            self.rbuf.max()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5, 6],
                    help="the headline workload (default 5: 64 streams x 16 rows, the largest by rows)")
    ap.add_argument("--per-config", default="3,4,5,6",
                    help="workloads also timed in the same run (own inputs, table and graph each), "
                         "comma-separated; empty for none")
    ap.add_argument("--row", default="verify", choices=["verify", "markov", "block", "prompt"])
    ap.add_argument("--prompt-rows", type=int, default=2048, help="--row prompt: rows of the prompt chunk")
    ap.add_argument("--prompt-cached", type=int, default=14336, help="--row prompt: keys cached before it")
    ap.add_argument("--impl", default="tf", choices=["tf", "reference"])
    ap.add_argument("--flush", default="clean", choices=["clean", "write"],
                    help="L2 flush between timed steps: write 256 MB then read another 256 MB (clean), "
                         "or only write (leaves the write's dirty lines to the timed step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--conv-layers", type=int, default=None, help="override (small profiling runs)")
    ap.add_argument("--attn-layers", type=int, default=None, help="override (small profiling runs)")
    args = ap.parse_args()
    args.per_config = [int(x) for x in args.per_config.split(",") if x.strip()]
    return args


# ------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(x, world, device="cpu"):
    """Max of a float over ranks (identity on one rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(rows_per_rank, ms_local, world, device="cpu"):
    """Whole-job throughput: the rows every rank verified per step over the
    slowest rank's step time. Returns (rows/s, max ms per step)."""
    ms_max = dist_max(ms_local, world, device=device)
    return rows_per_rank * world / (ms_max * 1e-3), ms_max


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 20 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(ts=ts, sm=float(parts[1]), smax=float(parts[2]), util=float(parts[4]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        if not rows:
            return None
        window = [r for r in rows if t0 - 0.25 <= r["ts"] <= t1 + 0.25]
        loaded = [r for r in window if r["util"] > 0] or window or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded)}


# ----------------------------------------------------------- helpers

def clocks_bad(summary):
    """A clock record that rejects a measurement: a hardware or thermal
    slowdown, or SM clocks well below their maximum with no reason given (a
    clock lock left by someone). sw_power_cap is kept (noted in reasons)."""
    if not summary:
        return False
    if {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"} & set(summary["reasons"]):
        return True
    return not summary["reasons"] and summary["sm_mhz"] < 0.9 * summary["sm_max_mhz"]


def timed_replays(torch, replay, flush, steps, stream, world, clocks):
    """K replays, L2 flushed before each (outside its events), one event pair
    per replay on the launch stream, barrier + synchronize around the loop.
    A run whose clock record rejects it is measured once more (every rank
    decides alike). Returns (ms per replay, wall start, wall end, remeasured)."""
    def loop():
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        dist_barrier(world)
        torch.cuda.synchronize()
        w0 = time.time()
        for k in range(steps):
            flush()
            ev[k][0].record(stream)
            replay()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        w1 = time.time()
        dist_barrier(world)
        return [a.elapsed_time(b) for a, b in ev], w0, w1

    ms, w0, w1 = loop()
    time.sleep(0.3)   # the sampler's last lines of the window
    bad = dist_max(1.0 if clocks_bad(clocks.summary(w0, w1)) else 0.0, world,
                   device=stream.device if world > 1 else "cpu")
    if bad > 0:
        ms, w0, w1 = loop()
        time.sleep(0.3)
        return ms, w0, w1, True
    return ms, w0, w1, False


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the attention kernels' sources, comments and blank space left
    out (a recorded ncu traffic figure is reported only while it matches: any
    change of the code itself makes it stale)."""
    import re
    h = hashlib.sha256()
    for name in ("attn.cu", "attn_tc.cu", "attn_item.cuh", "tc_ptx.cuh", "tf_internal.cuh"):
        with open(os.path.join(ROOT, "stream_speculative_decode_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload_index):
    """Per-launch DRAM bytes of the partials kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "attn_partials_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256_16") != kernel_source_hash():
        return None
    ent = rec.get("per_workload", {}).get(str(workload_index))
    return None if ent is None else float(ent["dram_bytes_per_launch"])


def _units(w, parts):
    """The work of one conv + one attention layer and the head, split over
    ``parts`` processes: conv and head by stream (stream s to part s % parts);
    attention by stream when there are at least as many streams as parts, else
    by (stream, window row) pair, the pairs dealt out in turn."""
    S = len(w.rows)
    if S >= parts:
        attn = [[(s, None) for s in range(S) if s % parts == p] for p in range(parts)]
    else:
        pairs = [(s, i) for s in range(S) for i in range(w.rows[s])]
        attn = [pairs[p::parts] for p in range(parts)]
    conv = [[s for s in range(S) if s % parts == p] for p in range(parts)]
    return conv, attn


def oracle_child(workload_index, part, parts, repeats):
    """(Child process.) Time part ``part`` of ``parts`` of one whole conv layer,
    one whole attention layer and the head (greedy pick + accept) of the
    workload on the oracle (``_units`` says which streams and rows). Inputs are
    drawn for the streams this part touches (same shapes and distributions as
    the workload's). Prints JSON with per-repeat seconds of each part."""
    import json as _json
    from stream_speculative_decode_gb300 import inputs as I
    from oracle import step as O
    w = I.workload(workload_index)
    conv_u, attn_u = _units(w, parts)
    mine_c, mine_a = conv_u[part], attn_u[part]
    touched = sorted(set(mine_c) | {s for s, _ in mine_a})
    res = dict(conv=[0.0] * repeats, attn=[0.0] * repeats, head=[0.0] * repeats, rows=sum(w.rows))
    if touched:
        sub = I.Workload("sample", [w.rows[s] for s in touched], [w.keys[s] for s in touched], 1, 1,
                         vocab=w.vocab, drafts=w.drafts, inf_frac=w.inf_frac, seed=w.seed)
        inp = I.make_inputs(sub, backend="numpy")
        j_of = {s: j for j, s in enumerate(touched)}
        for k in range(repeats):
            t0 = time.perf_counter()
            for s in mine_c:
                r, off, _ = inp.streams[j_of[s]]
                O.short_conv_stream(inp.bcx[0][off:off + r], inp.w[0], inp.state[0][j_of[s]])
            t1 = time.perf_counter()
            for s, i in mine_a:
                j = j_of[s]
                r, off, keys = inp.streams[j]
                if i is None:    # the stream's whole window
                    O.attention_stream(inp.q[0][off:off + r], inp.K[0][j], inp.V[0][j], keys, r)
                else:            # one window row: its causal count of keys
                    O.attention_stream(inp.q[0][off + i:off + i + 1], inp.K[0][j], inp.V[0][j],
                                       keys - r + i + 1, 1)
            t2 = time.perf_counter()
            for s in mine_c:
                r, off, keys = inp.streams[j_of[s]]
                pick, flag = O.argmax_rows(inp.logits[off:off + r])
                O.accept_stream(inp.ids[off:off + r], pick, flag, r, keys, w.vocab)
            t3 = time.perf_counter()
            res["conv"][k], res["attn"][k], res["head"][k] = t1 - t0, t2 - t1, t3 - t2
    print(_json.dumps(res))


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(workload_index, repeats, procs=1):
    """One whole conv layer, one whole attention layer and the head of the
    workload on the oracle, split over ``procs`` fresh child processes that run
    at once (one BLAS thread each). Per repeat the step time is the layer
    counts times the slowest part of each layer, plus the slowest head part.
    Returns (per-repeat step seconds, rows of a step)."""
    from stream_speculative_decode_gb300 import inputs as I
    w = I.workload(workload_index)
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[v] = "1"
    kids = []
    for p in range(procs):
        code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
                f"bench.oracle_child({workload_index}, {p}, {procs}, {repeats})")
        kids.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                     stderr=subprocess.PIPE, text=True))
    outs = []
    for k in kids:
        so, se = k.communicate(timeout=3600)
        if k.returncode != 0:
            raise RuntimeError("oracle sample failed: " + se[-2000:])
        outs.append(json.loads(so.strip().splitlines()[-1]))
    per_repeat = [w.n_conv * max(o["conv"][j] for o in outs) + w.n_attn * max(o["attn"][j] for o in outs)
                  + max(o["head"][j] for o in outs) for j in range(repeats)]
    return per_repeat, outs[0]["rows"]


def sample_desc(w, procs=1):
    par = (f"split over {procs} processes running at once (one per host core, one BLAS thread each; "
           f"conv and head by stream, attention by stream or, with fewer streams than processes, by "
           f"window row)" if procs > 1 else "1 process, 1 BLAS thread")
    return (f"float64 numpy oracle, {par}: one whole conv layer and one whole attention layer over all "
            f"{len(w.rows)} streams ({sum(w.rows)} rows, {sum(w.keys)} keys), then the greedy pick + accept; "
            f"step = {w.n_conv} x conv layer + {w.n_attn} x attention layer + head, each layer's time that "
            f"of its slowest process")


# -------------------------------------------------------------- arms

def run_reference(args, rank, world):
    from stream_speculative_decode_gb300 import inputs as I
    if rank != 0:
        return 0
    w = I.workload(args.workload)
    procs = host_cores()
    times, rows = oracle_sample(args.workload, args.warmup + args.steps, procs)
    timed = times[args.warmup:]
    sec = sum(timed) / max(len(timed), 1)
    value = rows / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": procs, "kind": "oracle",
                         "sample": sample_desc(w, procs)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": w.name, "streams": len(w.rows), "rows": sum(w.rows), "keys_total": sum(w.keys),
            "conv_layers": w.n_conv, "attn_layers": w.n_attn, "vocab": w.vocab,
            "widths": "H=2048, conv in 6144 (B,C,x), kw=3, 32 q / 8 kv heads, d=64"}


def attn_b2b_ms(torch, d, n_attn, flush, stream, dev, replays):
    """Median duration of one attention call with the step's attention calls
    back to back: a graph of the step's attention layers alone, replayed with
    the L2 flushed before each replay, one event pair per replay on the launch
    stream; the median replay over the layers."""
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for l in range(n_attn):
                d.attn(l, torch.cuda.current_stream(dev))
    stream.wait_stream(cap)
    ts = []
    for _ in range(replays):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / n_attn)
    return statistics.median(ts)


def attn_alg_bytes(streams, R):
    """One attention call: every stream's K and V (bf16), the queries in
    (bf16), the output out (fp32)."""
    return sum(k for _, _, k in streams) * 8 * 64 * 2 * 2 + R * 32 * 64 * (2 + 4)


def measure_workload(torch, index, steps, warmup, flush, stream, dev, world, clocks, peak):
    """One workload's step (its own inputs, table and graph), timed like the
    headline: W warm-up replays, then K replays with the L2 flushed before
    each. Returns the per-config record; frees everything it allocated."""
    from stream_speculative_decode_gb300 import inputs as I
    from stream_speculative_decode_gb300.step import DeviceStep, algorithmic_bytes
    w = I.workload(index)
    inp = I.make_inputs(w, backend="torch", device=dev)
    d = DeviceStep(inp, device=dev)
    ab = algorithmic_bytes(inp.streams, w.n_conv, w.n_attn, w.vocab)
    d.run()
    torch.cuda.synchronize()
    d.capture()
    for _ in range(warmup):
        flush()
        d.graph.replay()
    torch.cuda.synchronize()
    step_ms, w0, w1, remeasured = timed_replays(torch, d.graph.replay, flush, steps, stream, world, clocks)
    ms = sum(step_ms) / len(step_ms)
    b2b = attn_b2b_ms(torch, d, w.n_attn, flush, stream, dev, min(steps, 50))
    attn_alg = attn_alg_bytes(inp.streams, inp.R)
    cs = clocks.summary(w0, w1)
    rec = {"workload": w.name, "rows": inp.R, "streams": len(w.rows), "steps": steps, "warmup": warmup,
           "ms_per_step": ms, "rows_s": inp.R / (ms * 1e-3),
           "step_algorithmic_bytes": ab["total"], "hbm_gbs": ab["total"] / (ms * 1e-3) / 1e9,
           "hbm_frac": ab["total"] / (ms * 1e-3) / 1e9 / peak,
           "attn_ms_back_to_back": b2b, "attn_frac": attn_alg / (b2b * 1e-3) / 1e9 / peak,
           "attn_launches_per_call": d.seg.plan["attn_kernels"] + d.seg.plan["attn_merge_launch"],
           "clocks": dict(cs or {}, remeasured=remeasured)}
    d.free()
    del d, inp
    torch.cuda.empty_cache()
    return rec


def run_tf(args, rank, world):
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import inputs as I
    from stream_speculative_decode_gb300 import tf
    from stream_speculative_decode_gb300.step import DeviceStep, algorithmic_bytes

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    w = I.workload(args.workload, n_conv=args.conv_layers, n_attn=args.attn_layers)
    inp = I.make_inputs(w, backend="torch", device=dev)
    d = DeviceStep(inp, device=dev)
    ab = algorithmic_bytes(inp.streams, w.n_conv, w.n_attn, w.vocab)
    R = inp.R

    # per-launch timing of the dominant kernel, recorded inside the graph
    try:
        evs = {"attn": [(torch.cuda.Event(enable_timing=True, external=True),
                                  torch.cuda.Event(enable_timing=True, external=True))
                                 for _ in range(w.n_attn)]}
        graph_events = True
    except TypeError:
        evs, graph_events = None, False
    # warm the kernels once outside capture
    d.run()
    torch.cuda.synchronize()
    # the timed step: a graph without event nodes (an event record between
    # two launches ends their programmatic overlap); the per-launch attention
    # times come from a second graph of the same step with events around each
    # attention call, replayed in a loop of its own
    g_ev = d.capture(events=evs) if graph_events else None
    d.capture()
    flush = L2Flush(torch, dev, args.flush)
    stream = torch.cuda.current_stream(dev)

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    for _ in range(args.warmup):
        flush()
        d.graph.replay()
    torch.cuda.synchronize()

    part_ms = []
    # L2 flushed between timed steps (outside the events)
    step_ms, t_wall0, t_wall1, remeasured = timed_replays(torch, d.graph.replay, flush, args.steps, stream, world,
                                                          clocks)
    clocks_sum = clocks.summary(t_wall0, t_wall1)
    if clocks_sum is not None:
        clocks_sum["remeasured"] = remeasured
    if graph_events:                        # the attention calls, timed inside the step
        for _ in range(args.steps):
            flush()
            g_ev.replay()
            torch.cuda.synchronize()
            part_ms.extend(a.elapsed_time(b) for a, b in evs["attn"])
    # the same attention calls back to back (no event between them): the
    # call's duration when the launches overlap as they do in the step
    b2b_ms = attn_b2b_ms(torch, d, w.n_attn, flush, stream, dev, min(args.steps, 50)) if w.n_attn > 0 else None
    ms = sum(step_ms) / len(step_ms)
    value, ms_max = aggregate(R, ms, world, device=dev)

    if not graph_events:
        # no event nodes in graphs on this PyTorch: time eager launches of the same kernel
        for _ in range(min(args.steps, 20)):
            for l in range(w.n_attn):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                d.attn(l)
                b.record(stream)
                torch.cuda.synchronize()
                part_ms.append(a.elapsed_time(b))

    peak, peak_kind = measured_peaks()
    attn_alg = attn_alg_bytes(inp.streams, R)
    part_avg_ms = sum(part_ms) / len(part_ms) if part_ms else float("nan")
    achieved = attn_alg / (part_avg_ms * 1e-3) / 1e9
    if b2b_ms is None:   # no attention layer
        b2b_ms = part_avg_ms
    b2b_achieved = attn_alg / (b2b_ms * 1e-3) / 1e9 if b2b_ms == b2b_ms and b2b_ms else float("nan")
    traffic = recorded_traffic(args.workload)

    # end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(d, args, stream, flush, ab["total"])
    attn_launches = d.seg.plan["attn_kernels"] + d.seg.plan["attn_merge_launch"]
    launches = d.launches_per_step() * args.steps
    d.free()
    del d, inp, g_ev
    torch.cuda.empty_cache()

    # the other multi-layer workloads of the target set, each in its own run
    # of the same timing (more steps than the headline where K is small, so
    # that the clock record covers each)
    per_config = {}
    if args.per_config and args.conv_layers is None and args.attn_layers is None:
        pc_steps = max(args.steps, 200)
        for idx in args.per_config:
            per_config[str(idx)] = measure_workload(torch, idx, pc_steps, max(args.warmup, 3), flush, stream, dev,
                                                    world, clocks, peak)
    clocks.stop()

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        procs = host_cores()
        times1, rows = oracle_sample(args.workload, 1)
        timesn, _ = oracle_sample(args.workload, 3, procs) if procs > 1 else (times1, rows)
        sec1 = sum(times1) / len(times1)
        secn = sum(timesn) / len(timesn)
        cpu = {"value": rows / secn, "unit": UNIT, "cores": procs, "kind": "oracle",
               "sample": sample_desc(w, procs) + "; mean of 3 repeats",
               "single_core": {"value": rows / sec1, "cores": 1, "sample": sample_desc(w, 1) + "; one repeat"}}

    step_gbs = ab["total"] / (ms_max * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(w), l2=flush.desc,
                       graph="one CUDA graph per step", parallelism=f"replicas x{world}"),
        "hbm": {"step_algorithmic_bytes": ab["total"], "achieved_gbs": step_gbs, "peak_gbs": peak,
                "frac": step_gbs / peak, "peak_kind": peak_kind},
        "roofline": {"kernel": "tf_attn (attention partials with the merge folded in)", "bound": "hbm",
                     "achieved": b2b_achieved, "peak": peak,
                     "unit": "GB/s", "frac": b2b_achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": attn_alg, "avg_launch_ms": b2b_ms,
                     "launches_per_call": attn_launches,
                     "peak_kind": peak_kind,
                     "timing": "the step's attention calls back to back: a graph of the step's attention layers "
                               "alone, replayed after the timed region with the L2 flushed between replays, one "
                               "CUDA event pair per replay on the launch stream; avg_launch_ms = median replay / "
                               "layers (one call = launches_per_call launches)",
                     "per_call_events": {"avg_call_ms": part_avg_ms, "achieved": achieved, "frac": achieved / peak,
                                         "launches_timed": len(part_ms),
                                         "timing": "CUDA events around each attention call inside a copy of the "
                                                   "step graph, replayed K times after the timed region: the pair "
                                                   "costs the call its overlap with the launches before and after"
                                         if graph_events else
                                         "CUDA events around eager launches after the timed region"}},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks_sum,
        "wall_s_timed": t_wall1 - t_wall0,
        "per_config": per_config,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


L2_BYTES = 129 << 20


def run_e2e(d, args, stream, flush, step_bytes):
    """Same metric through the public API with host buffers: every step copies
    its inputs (conv inputs, queries, logits, ids: the step's input buffer)
    from pinned host memory and reads back the picks, flags and per-stream
    accept results (the step's result buffer).

    Serial: copy in, step, copy out, one step at a time, L2 flushed between
    steps (outside the events). Pipelined (the value, where the step's data
    exceed twice the L2, so no flush is needed between steps): the serving
    loop's form, two buffer sets and a copy stream each way, step k+1's inputs
    copied in and step k-1's results read back while step k runs; timed over
    the whole loop."""
    import torch
    host_in = torch.empty(d.in_arena.shape, dtype=torch.uint8, pin_memory=True).copy_(d.in_arena)
    host_out = torch.empty(d.out_arena.shape, dtype=torch.uint8, pin_memory=True)
    h2d = host_in.numel()
    d2h = host_out.numel()
    steps = max(3, min(args.steps, 50))

    def one():
        d.in_arena.copy_(host_in, non_blocking=True)
        d.graph.replay()
        host_out.copy_(d.out_arena, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    serial_ms = sum(ts) / len(ts)
    res = {"value": d.R / (serial_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": serial_ms, "steps": steps, "form": "serial (copy in, step, copy out; L2 flushed between "
                                                             "steps)"}
    if step_bytes <= 2 * L2_BYTES:
        return res

    # pipelined: buffer set b = k % 2 for step k
    g0 = d.graph
    k1 = d.add_io_set()
    d.use_io(k1)
    g1 = d.capture()
    d.use_io(0)
    d.graph = g0
    graphs = [g0, g1]
    arenas_in = [d._io[0]["in_arena"], d._io[k1]["in_arena"]]
    arenas_out = [d._io[0]["out_arena"], d._io[k1]["out_arena"]]
    hosts_out = [host_out, torch.empty(d.out_arena.shape, dtype=torch.uint8, pin_memory=True)]
    s_in, s_out = torch.cuda.Stream(device=stream.device), torch.cuda.Stream(device=stream.device)
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]

    def loop(n):
        for k in range(n):
            b = k % 2
            if k >= 2:
                s_in.wait_event(done[b])      # step k-2 has read this input buffer
            with torch.cuda.stream(s_in):
                arenas_in[b].copy_(host_in, non_blocking=True)
            copied[b].record(s_in)
            stream.wait_event(copied[b])
            if k >= 2:
                stream.wait_event(read[b])    # step k-2's results are read back
            graphs[b].replay()
            done[b].record(stream)
            s_out.wait_event(done[b])
            with torch.cuda.stream(s_out):
                hosts_out[b].copy_(arenas_out[b], non_blocking=True)
            read[b].record(s_out)
        stream.wait_event(read[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(read[(n - 2) % 2])

    loop(4)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    s_in.wait_event(a)
    s_out.wait_event(a)
    loop(steps)
    b.record(stream)
    b.synchronize()
    ms = a.elapsed_time(b) / steps
    res.update({"value": d.R / (ms * 1e-3), "ms_per_step": ms,
                "form": "pipelined: two buffer sets, step k+1's inputs copied in and step k-1's results read "
                        "back while step k runs (a copy stream each way); the step's data exceed twice the L2, "
                        "so no flush between steps; timed over the whole loop",
                "serial": {"value": d.R / (serial_ms * 1e-3), "ms_per_step": serial_ms}})
    return res


def run_row(args, rank, world):
    """One draft-side operation on the workload's windows (see the module
    docstring). Per step: one tf_markov_chain (every Markov step of every
    stream) or one tf_attn_block layer, in a CUDA graph, L2 flushed between
    steps."""
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from stream_speculative_decode_gb300 import inputs as I
    from stream_speculative_decode_gb300 import tf
    from stream_speculative_decode_gb300.step import DeviceStep

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = measured_peaks()
    if args.row == "markov":
        w = I.workload(args.workload, n_conv=0, n_attn=0)
        n = sum(r - 1 for r in w.rows)
        if n == 0:
            raise SystemExit("--row markov needs a workload with drafts (3, 4 or 5)")
        dr = I.make_draft_inputs(w, backend="torch", device=dev)
        off, streams = 0, []
        for r in w.rows:
            streams.append((r, off, r, 64))
            off += r
        seg = tf.tf_segments_build(streams, [], None, [], [], 0, 0)
        prev = torch.from_numpy(dr.prev).to(dev)
        pick = torch.empty(n, dtype=torch.int32, device=dev)
        flag = torch.empty(n, dtype=torch.uint8, device=dev)
        steps_per_call = max(w.rows) - 1

        def call(st):
            tf.tf_markov_chain(seg, dr.W1, dr.W2, w.vocab, dr.base, w.vocab, prev, pick, flag, st)

        units, metric, unit = n, "Markov draft rows/s (drafter head chain)", "rows/s"
        # compulsory bytes: W2 once (steps after the first may find it in L2), every base row,
        # the gathered W1 rows, picks and flags
        alg = w.vocab * I.MK * 2 + n * w.vocab * 2 + n * I.MK * 2 + n * 5
        path = os.environ.get("TF_MARKOV_PATH", "")
        S = len(w.rows)
        if path == "step" or S > 128:
            kname = "markov_step_kernel (tcgen05 W2 . W1[tok] + argmax), one launch a step"
        elif path == "chain" or S > 64:
            kname = "markov_chain_kernel (tcgen05, W2 streamed every step), whole chain in one launch"
        else:
            kname = (f"markov_hold_kernel<{32 if S <= 32 else 64}> (tcgen05, W2 held in tensor and shared "
                     "memory), whole chain in one launch")
        launches = steps_per_call
        extra = {"markov_steps": steps_per_call, "w2_bytes": w.vocab * I.MK * 2,
                 "w2_reads_if_no_l2_reuse": steps_per_call * w.vocab * I.MK * 2}
    elif args.row == "prompt":
        rows, cached = args.prompt_rows, args.prompt_cached
        w = I.prompt_workload(rows, cached, n_conv=1, n_attn=1)
        inp = I.make_inputs(w, backend="torch", device=dev)
        d = DeviceStep(inp, device=dev, prompt=True)

        def call(st):
            tf.tf_conv_rows(d.seg, 0, d.bcx[0], d.w[0], d.y[0], st)
            tf.tf_attn(d.seg, 0, d.q[0], d.partials, d.out[0], st)

        units, metric, unit = rows, "prompt rows/s per conv + attention layer pair", "rows/s"
        # causal attention: row i sees cached + i + 1 keys; q.K and P.V are 2*64 flops each per
        # (row, head, key)
        flops = 4.0 * 64 * 32 * sum(cached + i + 1 for i in range(rows))
        alg = flops
        wr = tf.TF_PROMPT_WINDOW_ROWS
        kname = f"tf_attn over the prompt's {wr}-row windows (+ one tf_conv_rows)"
        launches = 1 + d.seg.plan["attn_kernels"] + d.seg.plan["attn_merge_launch"]
        extra = {"prompt_rows": rows, "cached_keys": cached, "windows": (rows + wr - 1) // wr,
                 "compulsory_hbm_bytes": (cached + rows) * 8 * 64 * 2 * 2 + rows * (6144 * 2 + 2048 * 4)
                 + rows * 32 * 64 * (2 + 4)}
    else:
        w = I.workload(args.workload, n_conv=0, n_attn=1)
        inp = I.make_inputs(w, backend="torch", device=dev)
        d = DeviceStep(inp, device=dev)
        out = torch.empty_like(d.out[0])

        def call(st):
            tf.tf_attn_block(d.seg, 0, d.q[0], d.partials, out, st)

        units, metric, unit = inp.R, "block-attention rows/s per layer (FULL, non-causal)", "rows/s"
        alg = sum(k for _, _, k in inp.streams) * 8 * 64 * 2 * 2 + inp.R * 32 * 64 * (2 + 4)
        kname = "tf_attn_block (partials with the merge folded in)"
        launches = d.seg.plan["attn_kernels"] + d.seg.plan["attn_merge_launch"]
        extra = {}
    call(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.graph(g, stream=cap):
        call(cap)
    flush = L2Flush(torch, dev, args.flush)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    for _ in range(args.warmup):
        flush()
        g.replay()
    torch.cuda.synchronize()
    step_ms, t0, t1, remeasured = timed_replays(torch, g.replay, flush, args.steps, stream, world, clocks)
    clocks.stop()
    ms = sum(step_ms) / args.steps
    value, ms_max = aggregate(units, ms, world, device=dev)
    achieved = alg / (ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "unit": "GB/s", "peak": peak, "peak_kind": peak_kind}
    if args.row == "prompt":   # prefill attention is a contraction: FLOP/s against the bf16 tensor peak
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                tpk, tkind = float(json.load(f)["bf16_tflops"]), "measured"
        except (OSError, KeyError, ValueError):
            tpk, tkind = 1900.0, "fallback"
        achieved = alg / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "unit": "TFLOP/s", "peak": tpk, "peak_kind": tkind}
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(w), row=args.row,
                       l2=flush.desc,
                       graph="one CUDA graph per step", parallelism=f"replicas x{world}", **extra),
        "roofline": {"kernel": kname, "bound": roof["bound"], "achieved": achieved, "peak": roof["peak"],
                     "unit": roof["unit"], "frac": achieved / roof["peak"], "traffic": None,
                     ("algorithmic_flops_per_call" if args.row == "prompt" else "algorithmic_bytes_per_call"): alg,
                     "avg_call_ms": ms, "peak_kind": roof["peak_kind"],
                     "timing": "CUDA events around each graph replay (one call)"},
        "gpu_launches": launches * args.steps,
        "clocks": dict(clocks.summary(t0, t1) or {}, remeasured=remeasured),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    rank, world, _ = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.row != "verify":
        return run_row(args, rank, world)
    return run_tf(args, rank, world)


if __name__ == "__main__":
    sys.exit(main())
