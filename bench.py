"""Benchmark of the fused-dequant decode attention on the Llama-3.1-8B-shaped
128k-token 2-bit GQA cache (batch 1, 32 query heads over 8 KV heads, head_dim
128, 131008 quantized tokens + 64-token fp16 tail, group 32).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one kvq_decode_attn call over the whole cache (the metric's unit);
the prefill of that cache and the per-token append are timed too and reported
beside it.  Inputs are seeded synthetic tensors (no model weights, no dataset).
The timed region replays a CUDA graph of decode launches that rotate over
cache replicas whose total size is several times the L2, so every step reads
its cache from HBM.  One JSON line is printed by rank 0.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-dequant decode attn: µs/step, achieved HBM GB/s vs peak (Llama-3.1-8B, 128k)"
UNIT = "us/step"
FALLBACK_HBM_GBS = 6800.0
MIN_TIMED_S = 0.5  # shortest timed region (clock samples under load)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=25000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--bits", type=int, default=2, choices=[2, 4])
    ap.add_argument("--rope", type=float, default=0.0,
                    help="uniform cache: keys stored before RoPE and rotated in the decode with this "
                         "rotary base (e.g. 500000); 0 = plain decode")
    ap.add_argument("--sink", type=int, default=0,
                    help="uniform cache: keep the first S tokens fp16 (attention-sink window)")
    ap.add_argument("--workload", default="uniform",
                    choices=["uniform", "llama2_13b", "trizone", "serving", "rdkv"],
                    help="uniform: the Llama-3.1-8B 128k-token uniform cache (default); llama2_13b: "
                         "the Llama-2-13B MHA cache (8 sequences x 40 heads x 4,096 tokens, "
                         "4,064 quantized + 32 fp16); trizone: the "
                         "mixed-width cache, 4 sequences x 65,408 old + 128 fresh tokens; "
                         "serving: 16 ragged sequences of 8k-32k tokens, 4-bit, one "
                         "append + decode per step; rdkv: the bit allocation (token weights "
                         "+ widths) of the mixed-width workload's 4 x 65,536-token prompts")
    ap.add_argument("--rdkv-tokens", type=int, default=0,
                    help="rdkv workload: prompt positions per sequence (default: the workload's 65,536; "
                         "a smaller prompt is for profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def workload(bits, name="uniform"):
    from quantized_kv_cache_11_gb300 import synthetic as S
    if name == "llama2_13b":
        w = S.LLAMA2_13B
        return w if bits == 2 else w.scaled(name=w.name.replace("2bit", f"{bits}bit"), bits=bits)
    return S.LLAMA31_8B_128K if bits == 2 else S.LLAMA31_8B_128K_4BIT


def dtype_label(bits) -> str:
    """The arithmetic the decode path computes in."""
    return f"int{bits} codes x fp16 operands on tensor cores, fp32 accumulate and softmax"


def algorithmic_bytes(w, n_quant, n_tail, n_sink=0) -> int:
    """Bytes one decode step must move: packed K/V codes, fp16 scale + zero of
    every group, the fp16 tail and sink tokens, q in and the fp32 output."""
    D, H, b = w.head_dim, w.n_kv_heads, w.bits
    per_tok = 2 * D * b // 8 + (2 * D // 32) * 2  # codes K+V, V meta (fp16 scale + zero per 32 ch)
    k_meta = (n_quant // 32) * 2 * D * 2  # per key group: scale + zero per channel
    fp16 = (n_tail + n_sink) * D * 2 * 2
    return w.batch * H * (n_quant * per_tok + k_meta + fp16) + w.batch * w.n_q_heads * D * (2 + 4)


def with_sink(inp, sink):
    """The workload's tail shortened so that the tokens after an S-token sink
    window still end in whole groups (the quantized region keeps its length)."""
    if sink == 0:
        return inp
    L = inp["seq_len"].astype(int)
    ns = np.minimum(sink, L)
    nq = np.maximum(0, -(-(L - ns - inp["n_tail"]) // 32) * 32)
    nt = L - ns - nq
    if (nt < 0).any():
        raise ValueError("the sink window does not fit the workload's tail")
    return dict(inp, n_tail=nt.astype(np.int32))


def prefill_algorithmic_bytes(w, n_quant, n_tail, n_sink=0) -> int:
    """Prefill reads the fp16 K and V of every token and writes the packed cache
    (codes and fp16 metadata) plus the fp16 tail and sinks."""
    read = 2 * w.batch * (n_quant + n_tail + n_sink) * w.n_kv_heads * w.head_dim * 2
    write = algorithmic_bytes(w, n_quant, n_tail, n_sink) - w.batch * w.n_q_heads * w.head_dim * 6
    return read + write


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("hbm_gbs"):
            return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- the oracle on the host cores: one code path for the GPU arm's cpu_baseline
# and the reference arm.  Each (sequence, KV head) segment of the cache is one
# unit of work; worker processes (spawned, one per core, single-threaded BLAS)
# each hold a round-robin share of the sampled segments, quantize them once, and
# then run the oracle's fp64 decode attention over them on every step.

def _oracle_worker(conn, bits, sm_scale, rope):
    from oracle import kvq_oracle as O
    held, states = [], []
    while True:
        msg = conn.recv()
        if msg[0] == "stop":
            conn.close()
            return
        if msg[0] == "load":
            held.append(msg[1:])
            conn.send(("ok",))
        elif msg[0] == "quantize":
            t0 = time.perf_counter()
            states = [(qh, O.quantize_sequence(k, v, n, nt, bits, n_sink_cap=ns))
                      for (k, v, qh, n, nt, ns) in held]
            conn.send((time.perf_counter() - t0,))
        elif msg[0] == "attend":
            t0 = time.perf_counter()
            for qh, st in states:
                if rope:
                    O.sequence_attention_rope(qh, st, sm_scale, rope)
                else:
                    O.sequence_attention(qh, st, sm_scale)
            conn.send((time.perf_counter() - t0,))


class OraclePool:
    """n spawned worker processes with single-threaded BLAS (spawn: safe after
    CUDA has been initialised in this process)."""

    def __init__(self, n, bits, sm_scale, rope):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.conns, self.procs = [], []
            for _ in range(n):
                a, b = ctx.Pipe()
                pr = ctx.Process(target=_oracle_worker, args=(b, bits, sm_scale, rope), daemon=True)
                pr.start()
                self.conns.append(a)
                self.procs.append(pr)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def load(self, segs):
        for i, sg in enumerate(segs):
            self.conns[i % len(self.conns)].send(("load", *sg))
        for i, _ in enumerate(segs):
            self.conns[i % len(self.conns)].recv()

    def phase(self, cmd) -> float:
        """Wall seconds of one phase run by every worker at once."""
        t0 = time.perf_counter()
        for c in self.conns:
            c.send((cmd,))
        for c in self.conns:
            c.recv()
        return time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            c.send(("stop",))
        for pr in self.procs:
            pr.join(timeout=30)


def oracle_segments(w, inp, n_sink_cap=0, limit=None):
    """(K, V, q of the GQA group, length, tail, sink window) of the first `limit`
    (sequence, KV head) segments, in batch-major order."""
    out = []
    G = w.gqa
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            if limit is not None and len(out) >= limit:
                return out
            n = int(inp["seq_len"][b])
            out.append((np.ascontiguousarray(inp["K"][b, :, h:h + 1]), np.ascontiguousarray(inp["V"][b, :, h:h + 1]),
                        np.ascontiguousarray(inp["q"][b][h * G:(h + 1) * G]), n, int(inp["n_tail"][b]),
                        min(n_sink_cap, n)))
    return out


class OracleStep:
    """The oracle's decode step on this host's cores.  A single-threaded probe of
    one segment sizes the sample: every segment when a whole step fits the
    budget, else whole rounds of one segment per core (the time is then scaled
    to all segments and flagged as extrapolated)."""

    def __init__(self, w, inp, sink=0, rope=0.0, step_budget_s=2.0):
        self.w, self.rope = w, rope
        self.S = w.batch * w.n_kv_heads
        self.cores = os.cpu_count() or 1
        probe = OraclePool(1, w.bits, w.sm_scale, rope)
        probe.load(oracle_segments(w, inp, sink, limit=1))
        self.t_quant1 = probe.phase("quantize")
        self.t_attn1 = min(probe.phase("attend") for _ in range(2))
        probe.close()
        rounds = max(1, int(step_budget_s / max(self.t_attn1, 1e-6)))
        self.m = min(self.S, self.cores * rounds)
        self.pool = OraclePool(min(self.cores, self.m), w.bits, w.sm_scale, rope)
        self.pool.load(oracle_segments(w, inp, sink, limit=self.m))
        self.t_quant = self.pool.phase("quantize")

    def step_us(self) -> float:
        """One decode step (attention over the sampled segments on every core),
        scaled to all segments; microseconds."""
        return self.pool.phase("attend") * self.S / self.m * 1e6

    def describe(self, values) -> dict:
        S, m = self.S, self.m
        what = "all" if m == S else f"{m} of"
        return {
            "value": statistics.mean(values), "unit": UNIT, "kind": "oracle", "cores": self.cores,
            "nproc": self.cores, "threads_per_process": 1,
            "extrapolated": m < S, "sampled_fraction": m / S,
            "all_cores": {"attention_us_per_step": statistics.mean(values),
                          "quantize_ms_per_cache": self.t_quant * S / m * 1e3},
            "single_thread": {"attention_us_per_step": self.t_attn1 * S * 1e6,
                              "quantize_ms_per_cache": self.t_quant1 * S * 1e3,
                              "from": "one segment timed alone, x segments"},
            "sample": f"oracle fp64 decode attention{' with RoPE' if self.rope else ''} over {what} {S} "
                      f"(sequence, KV head) segments per step on {min(self.cores, m)} worker processes "
                      f"(os.cpu_count() = {self.cores}, one BLAS thread each), mean of {len(values)} steps"
                      + ("" if m == S else f", scaled x{S / m:.2f} to the full step") +
                      "; quantizer timed once per segment (the prefill of the cache)",
        }

    def close(self):
        self.pool.close()


def cpu_baseline(w, inp, sink=0, rope=0.0, n_steps=3):
    """The GPU arm's CPU figure: the same oracle step as the reference arm."""
    ost = OracleStep(w, inp, sink=sink, rope=rope)
    try:
        vals = [ost.step_us() for _ in range(n_steps)]
        return ost.describe(vals)
    finally:
        ost.close()


def uniform_config(w, args, n_quant, n_tail, n_sink) -> dict:
    """The keys naming a uniform-cache decode workload (both arms print them)."""
    return {"workload": w.name + ("_prerope" if args.rope else ""), "batch": w.batch,
            "n_q_heads": w.n_q_heads, "rope_base": args.rope or None,
            "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "context": w.context,
            "n_quant": n_quant, "n_tail": n_tail, "n_sink": n_sink, "bits": w.bits, "group": 32}


def serving_config(w, mean_tokens) -> dict:
    """The keys naming the ragged serving workload (both arms print them)."""
    return {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "bits": w.bits, "lengths": f"U[{w.ragged[0]}, {w.ragged[1]}]",
            "mean_tokens": mean_tokens, "step": "one append + one decode"}


def run_reference(args):
    """The oracle on the host cores, same metric/config: each step times the
    oracle on a slice of one KV head's context, sized so the run ends in minutes,
    and is scaled to a full decode step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from quantized_kv_cache_11_gb300 import synthetic as S
    if args.workload == "trizone":
        run_reference_trizone(args)
        return
    if args.workload == "rdkv":
        run_reference_rdkv(args)
        return
    serving = args.workload == "serving"
    w = S.SERVING if serving else workload(args.bits, args.workload)
    inp = S.generate(w) if serving else with_sink(S.generate(w), args.sink)
    n = int(inp["seq_len"][0])
    nt = int(inp["n_tail"][0])
    n_sink = 0 if serving else min(args.sink, n)
    nq = n - nt - n_sink
    # per-step budget so the whole run ends in a few minutes
    ost = OracleStep(w, inp, sink=n_sink, rope=args.rope,
                     step_budget_s=min(4.0, 150.0 / max(1, args.steps + args.warmup)))
    times = []
    for i in range(args.warmup + args.steps):
        t = ost.step_us()
        if i >= args.warmup:
            times.append(t)
    cb = ost.describe(times)
    ost.close()
    if serving:
        config = serving_config(w, float(inp["seq_len"].mean()))
    else:
        config = uniform_config(w, args, nq, nt, n_sink)
    config.update({"l2": "n/a (host cores)", "launch": "oracle calls on the host"})
    value = cb["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1000.0,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config, "extrapolated": cb["extrapolated"],
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_trizone(args):
    """The oracle on the host cores for the mixed-width cache: each step times
    dequantize + fp64 attention of one (sequence, KV head) segment (several
    segments rotate), scaled to all segments."""
    from oracle import kvq_oracle as O
    from quantized_kv_cache_11_gb300 import synthetic as S
    import torch
    w = S.TRIZONE
    inp = S.generate(w)
    tzs = [O.trizone_quantize(inp["K"][b, :, h], inp["V"][b, :, h], inp["v_width"][b, h],
                              inp["k_width"][b, h]) for b, h in ((0, 0), (1, 3), (3, 7))]
    times = []
    for i in range(args.warmup + args.steps):
        b, h = ((0, 0), (1, 3), (3, 7))[i % 3]
        t0 = time.perf_counter()
        O.trizone_attention(inp["q"][b][h * w.gqa:(h + 1) * w.gqa], [tzs[i % 3]], w.sm_scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    segs = w.batch * w.n_kv_heads
    value = statistics.mean(times) * segs * 1e6
    sample = f"oracle dequant + fp64 attention of 1 of {segs} segments per step, scaled x{segs}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1000.0,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name},
        "cpu_baseline": {"kind": "oracle", "cores": torch.get_num_threads(), "sample": sample,
                         "value": value, "unit": UNIT},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def time_graph(launch, n_rep, steps_wanted, world, local):
    """Capture launch(i) for i < per_graph in a CUDA graph (rotating the n_rep
    replicas), replay it until >= steps_wanted launches, and time the replays with
    CUDA events on the current stream, sampling clocks meanwhile.  Returns
    (us per launch, launches timed, clock summary); max over ranks."""
    import torch
    import torch.distributed as dist
    per_graph = n_rep * max(1, 256 // n_rep)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per_graph):
            launch(i)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g.replay()
    torch.cuda.synchronize()
    t_replay = time.perf_counter() - t0
    # at least the requested launches, and at least MIN_TIMED_S of timed work so
    # that the clock sampler sees the GPU under load
    reps = max(1, math.ceil(steps_wanted / per_graph), math.ceil(MIN_TIMED_S / max(t_replay, 1e-6)))
    steps = reps * per_graph
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), torch.device("cuda", local))
    return elapsed_ms * 1000.0 / steps, steps, clk.summary()


def time_single(launch, n_rep, n=64):
    """Median (and 10th / 90th percentile) of n separately timed launches, each
    bracketed by its own CUDA events on the current stream, eager (no graph),
    rotating the replicas; microseconds."""
    import torch
    for i in range(3):
        launch(i)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(ev):
        a.record()
        launch(i)
        b.record()
    torch.cuda.synchronize()
    t = np.array([a.elapsed_time(b) * 1000.0 for a, b in ev])
    return {"median_us": float(np.median(t)), "p10_us": float(np.percentile(t, 10)),
            "p90_us": float(np.percentile(t, 90)), "launches": n}


def max_over_ranks(value: float, device) -> float:
    """The largest of the ranks' values (every rank gets it); the value itself
    when there is one rank.  Each rank runs its own replica of the workload, so
    the job's time per step is the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_e2e(launch, q_host, q_dev, out_host, outs, n_rep, n):
    """Public-API loop, every step inside the timed region: the step's q copied
    from pinned host memory to the device, the decode, and its fp32 output copied
    back to pinned host memory.  Uploads and downloads run on two more streams
    (q double buffered, one output buffer per cache replica) so that step i's
    download and step i+1's upload overlap the decodes, with events ordering every
    copy against the decode that uses it.  The steps are captured in a CUDA graph (what a
    serving loop does to keep the host out of the way) and the graph is replayed
    until >= n steps; returns us per step."""
    import torch
    comp = torch.cuda.current_stream()
    up = torch.cuda.Stream(device=q_dev.device)
    down = torch.cuda.Stream(device=q_dev.device)
    qd = [q_dev, torch.empty_like(q_dev)]
    oh = [out_host, torch.empty_like(out_host).pin_memory()]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(n_rep)]
    ev_q_free = [torch.cuda.Event() for _ in range(2)]
    ev_o_free = [torch.cuda.Event() for _ in range(n_rep)]

    def step(i, cs):
        j, r = i % 2, i % n_rep
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(ev_q_free[j])  # the decode that read qd[j] is done
            qd[j].copy_(q_host, non_blocking=True)
            ev_in[j].record(up)
        cs.wait_event(ev_in[j])
        if i >= n_rep:
            cs.wait_event(ev_o_free[r])  # outs[r] has been downloaded
        launch(i, qd[j])
        ev_q_free[j].record(cs)
        ev_out[r].record(cs)
        with torch.cuda.stream(down):
            down.wait_event(ev_out[r])
            oh[i % 2].copy_(outs[r], non_blocking=True)
            ev_o_free[r].record(down)

    per_graph = n_rep * max(1, 128 // n_rep)
    for i in range(per_graph):  # warm-up outside the graph
        step(i, comp)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        up.wait_stream(cs)
        down.wait_stream(cs)
        for i in range(per_graph):
            step(i, cs)
        cs.wait_stream(up)
        cs.wait_stream(down)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    reps = max(1, math.ceil(n / per_graph))
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(comp)
    for _ in range(reps):
        g.replay()
    x1.record(comp)
    torch.cuda.synchronize()
    return x0.elapsed_time(x1) * 1000.0 / (reps * per_graph)


def read_traffic(name, workload_name, sha):
    """Per-launch DRAM bytes from a committed ncu summary, while the kernel source
    is the one the counters were taken from (else None)."""
    tf = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(tf):
        return None
    rec = {}
    with open(tf) as f:
        for ln in f:
            if ":" in ln and not ln.lstrip().startswith("#"):
                k, v = ln.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("workload") == workload_name and rec.get("kernel_source_sha") == sha:
        return int(rec["dram_bytes_per_launch"])
    return None


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload == "trizone":
        main_trizone(args)
        return
    if args.workload == "serving":
        main_serving(args)
        return
    if args.workload == "rdkv":
        main_rdkv(args)
        return
    import torch
    import torch.distributed as dist
    from quantized_kv_cache_11_gb300 import kvq
    from quantized_kv_cache_11_gb300 import synthetic as S

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvq.load_library()

    w = workload(args.bits, args.workload)
    inp = with_sink(S.generate(w), args.sink)
    n_sink = min(args.sink, int(inp["seq_len"][0]))
    n_quant = int(inp["seq_len"][0] - inp["n_tail"][0]) - n_sink
    n_tail = int(inp["n_tail"][0])
    K = torch.from_numpy(inp["K"]).to(dev)
    V = torch.from_numpy(inp["V"]).to(dev)
    q = torch.from_numpy(inp["q"]).to(dev)

    # ---- cache replicas: total well above the 129 MB L2
    probe = kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, w.bits, w.context, w.tail_cap,
                                 device=dev, sink_cap=args.sink)
    n_rep = max(4, math.ceil(3 * 128e6 / probe.nbytes) + 1)
    caches = [probe] + [kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, w.bits, w.context,
                                             w.tail_cap, device=dev, sink_cap=args.sink)
                        for _ in range(n_rep - 1)]
    stream = torch.cuda.current_stream(dev)
    # prefill timing (first replica, repeated), then fill every replica
    pre_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for c in caches:
        c.prefill(K, V, inp["seq_len"].tolist(), inp["n_tail"].tolist())
    torch.cuda.synchronize()
    pre_ev[0].record()
    for _ in range(5):
        caches[0].prefill(K, V, inp["seq_len"].tolist(), inp["n_tail"].tolist())
    pre_ev[1].record()
    torch.cuda.synchronize()
    prefill_us = pre_ev[0].elapsed_time(pre_ev[1]) * 1000 / 5
    prefill_bytes = prefill_algorithmic_bytes(w, n_quant, n_tail, n_sink)

    # ---- append timing on a separate cache (keeps the replicas unchanged)
    app = kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, w.bits, w.context + 4096,
                               w.tail_cap, device=dev, sink_cap=args.sink)
    app.prefill(K, V, inp["seq_len"].tolist(), inp["n_tail"].tolist())
    kn = torch.randn(w.batch, w.n_kv_heads, w.head_dim, device=dev).half()
    vn = torch.randn(w.batch, w.n_kv_heads, w.head_dim, device=dev).half()
    for _ in range(8):
        app.append(kn, vn)
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_app = 256
    a0.record()
    for _ in range(n_app):
        app.append(kn, vn)
    a1.record()
    torch.cuda.synchronize()
    append_us = a0.elapsed_time(a1) * 1000 / n_app
    del app

    # ---- decode: warm up, quick parity sample, graph of launches over the replicas
    outs = [torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev)
            for _ in caches]
    if args.rope:
        table = caches[0].rope_table(args.rope)  # one table serves every replica (same geometry)

        def dec(c, qq, out):
            c.decode_rope(qq, table, w.sm_scale, out=out)
    else:
        def dec(c, qq, out):
            c.decode(qq, w.sm_scale, out=out)
    for i in range(max(args.warmup, 3)):
        dec(caches[i % n_rep], q, outs[i % n_rep])
    torch.cuda.synchronize()
    parity = None
    if rank == 0:
        from oracle import kvq_oracle as O
        st = O.quantize_sequence(inp["K"][0][:, :1], inp["V"][0][:, :1], int(inp["seq_len"][0]),
                                 n_tail, w.bits, n_sink_cap=args.sink)
        if args.rope:
            ref = O.sequence_attention_rope(inp["q"][0][:w.gqa], st, w.sm_scale, args.rope)
        else:
            ref = O.sequence_attention(inp["q"][0][:w.gqa], st, w.sm_scale)
        got = outs[0][0, :w.gqa].double().cpu().numpy()
        parity = {"kv_heads_checked": 1, "max_abs": float(np.abs(got - ref).max())}
    us_step, steps, clocks = time_graph(
        lambda i: dec(caches[i % n_rep], q, outs[i % n_rep]), n_rep, args.steps, world, local)
    single = time_single(lambda i: dec(caches[i % n_rep], q, outs[i % n_rep]), n_rep)

    # ---- end to end through the public API: pinned host q in, fp32 output out
    q_host = torch.from_numpy(inp["q"]).pin_memory()
    out_host = torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(q)
    e2e_us = time_e2e(lambda i, qd: dec(caches[i % n_rep], qd, outs[i % n_rep]),
                      q_host, q_dev, out_host, outs, n_rep, min(steps, 4000))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = load_peaks()
    nbytes = algorithmic_bytes(w, n_quant, n_tail, n_sink)
    achieved = nbytes / (us_step * 1e-6) / 1e9
    if args.sink:
        traffic = None
    elif args.rope:
        traffic = read_traffic(f"decode_traffic_{w.name}_prerope.txt", w.name + "_prerope",
                               _kernel_sha(ROPE_FILES))
    else:
        traffic = read_traffic(f"decode_traffic_{w.name}.txt", w.name, _kernel_sha())
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": us_step / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(w.bits), "data": "synthetic",
        "config": {**uniform_config(w, args, n_quant, n_tail, n_sink),
                   "l2": f"inputs larger than L2: {n_rep} cache replicas "
                         f"({n_rep * probe.nbytes / 1e6:.0f} MB) rotated every step",
                   "launch": "CUDA graph of " + ("kvq_decode_attn_rope" if args.rope else "kvq_decode_attn") +
                             " calls"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes": nbytes},
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": out_host.numel() * 4},
        "gpu_launches": steps,
        "clocks": clocks,
        "path": {"decode_us": us_step, "decode_per_launch": single, "prefill_us": prefill_us,
                 "prefill_gbs": prefill_bytes / (prefill_us * 1e-6) / 1e9, "append_us": append_us},
        "parity_sample": parity,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, sink=args.sink, rope=args.rope)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


TZ_FILES = ("kvq_trizone_decode.cu", "kvq_trizone_internal.h", "kvq_common.cuh")


def trizone_bytes(w, v_width, k_width, n_fresh) -> dict:
    """Bytes one decode step of the mixed-width cache must move, from the drawn
    widths (the pages' layout, no padding): per kept old token the key codes at
    each channel's width and the value codes at the token's width (+ an fp16
    scale and zero per 32 channels) or its fp16 row; per 32-token block an fp16
    scale and zero per channel; the fp16 fresh rows; q in, fp32 out."""
    D = w.head_dim
    k_bits = np.zeros(v_width.shape[:2])
    for c in (2, 4, 8):
        k_bits += (k_width == c).sum(-1) * c
    total = 0
    kept_total = 0
    for b in range(v_width.shape[0]):
        for h in range(v_width.shape[1]):
            n = {c: int((v_width[b, h] == c).sum()) for c in (2, 4, 8, 16)}
            kept = sum(n.values())
            blocks = sum(-(-x // 32) for x in n.values())
            total += kept * int(k_bits[b, h]) // 8 + blocks * D * 4
            total += sum(n[c] * (D * c // 8 + (D // 32) * 4) for c in (2, 4, 8)) + n[16] * D * 2
            total += n_fresh * D * 4
            kept_total += kept
    total += w.batch * w.n_q_heads * D * (2 + 4)
    return {"decode": total, "kept": kept_total}


def trizone_cpu_baseline(w, inp, budget_s=12.0):
    """The oracle as it stands: dequantize + fp64 attention of one (sequence, KV
    head) of the mixed-width cache, repeated for ~budget_s, scaled to a step."""
    from oracle import kvq_oracle as O
    import torch
    t_old = w.context - w.trizone_fresh
    tz = O.trizone_quantize(inp["K"][0, :, 0], inp["V"][0, :, 0], inp["v_width"][0, 0],
                            inp["k_width"][0, 0])
    q = inp["q"][0][:w.gqa]
    times = []
    t_end = time.perf_counter() + budget_s
    while time.perf_counter() < t_end or len(times) < 2:
        t0 = time.perf_counter()
        O.trizone_attention(q, [tz], w.sm_scale)
        times.append(time.perf_counter() - t0)
    segs = w.batch * w.n_kv_heads
    return {"value": statistics.median(times) * segs * 1e6, "unit": UNIT, "kind": "oracle",
            "cores": torch.get_num_threads(),
            "sample": f"1 of {segs} (sequence, KV head) segments ({w.gqa} query heads, {t_old} old + "
                      f"{w.trizone_fresh} fresh tokens), median of {len(times)} runs, x{segs}"}


def main_trizone(args):
    """The mixed-width cache: 4 sequences x 8 KV heads x (65,408 old tokens with
    value widths {0,2,4,8,16} and key widths {2,4,8} drawn per token / channel,
    + 128 fresh fp16 tokens).  A step is one kvq_trizone_decode_attn call."""
    import torch
    import torch.distributed as dist
    from quantized_kv_cache_11_gb300 import kvq
    from quantized_kv_cache_11_gb300 import synthetic as S

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvq.load_library()
    w = S.TRIZONE
    inp = S.generate(w)
    B, H = w.batch, w.n_kv_heads
    t_old, nf = w.context - w.trizone_fresh, w.trizone_fresh
    K = torch.from_numpy(inp["K"]).to(dev)
    V = torch.from_numpy(inp["V"]).to(dev)
    vw = torch.from_numpy(inp["v_width"]).to(dev)
    kw = torch.from_numpy(inp["k_width"]).to(dev)
    q = torch.from_numpy(inp["q"]).to(dev)
    nb = trizone_bytes(w, inp["v_width"], inp["k_width"], nf)

    def make():
        c = kvq.TriZoneCache(B, H, t_old, nf, device=dev)
        c.build(K, V, vw, kw, [t_old] * B, [nf] * B)
        return c

    probe = make()
    used = int(probe.views()["index"][:, :, 104:108].contiguous().view(torch.int32).sum())
    n_rep = max(4, math.ceil(3 * 128e6 / used) + 1)
    caches = [probe] + [make() for _ in range(n_rep - 1)]
    torch.cuda.synchronize()
    # build timing (first replica, repeated)
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record()
    for _ in range(5):
        caches[0].build(K, V, vw, kw, [t_old] * B, [nf] * B)
    b1.record()
    torch.cuda.synchronize()
    build_us = b0.elapsed_time(b1) * 1000 / 5
    # build moves: the kept and fresh K/V rows in, widths in, the records and the
    # token order out
    build_bytes = (nb["kept"] + B * H * nf) * w.head_dim * 2 * 2 + vw.numel() + kw.numel() + \
        used + nb["kept"] * 4 + B * H * 512

    outs = [torch.empty(B, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev) for _ in caches]
    for i in range(max(args.warmup, 3)):
        caches[i % n_rep].decode(q, w.sm_scale, out=outs[i % n_rep])
    torch.cuda.synchronize()
    parity = None
    if rank == 0:
        from oracle import kvq_oracle as O
        tz = O.trizone_quantize(inp["K"][0, :, 0], inp["V"][0, :, 0], inp["v_width"][0, 0],
                                inp["k_width"][0, 0])
        ref = O.trizone_attention(inp["q"][0][:w.gqa], [tz], w.sm_scale)
        got = outs[0][0, :w.gqa].double().cpu().numpy()
        parity = {"segments_checked": 1, "max_abs": float(np.abs(got - ref).max())}
    us_step, steps, clocks = time_graph(
        lambda i: caches[i % n_rep].decode(q, w.sm_scale, out=outs[i % n_rep]),
        n_rep, args.steps, world, local)
    single = time_single(lambda i: caches[i % n_rep].decode(q, w.sm_scale, out=outs[i % n_rep]), n_rep)
    q_host = torch.from_numpy(inp["q"]).pin_memory()
    out_host = torch.empty(B, w.n_q_heads, w.head_dim, dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(q)
    e2e_us = time_e2e(lambda i, qd: caches[i % n_rep].decode(qd, w.sm_scale, out=outs[i % n_rep]),
                      q_host, q_dev, out_host, outs, n_rep, min(steps, 4000))
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = load_peaks()
    achieved = nb["decode"] / (us_step * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": us_step / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int2/int4/int8 codes and fp16 rows x fp16 operands on tensor cores, fp32 accumulate and softmax",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": B, "n_q_heads": w.n_q_heads, "n_kv_heads": H,
                   "head_dim": w.head_dim, "old_tokens": t_old, "fresh_tokens": nf,
                   "kept_tokens_mean": nb["kept"] / (B * H),
                   "v_width_probs": list(w.v_width_probs), "k_width_probs": list(w.k_width_probs),
                   "stored_bytes": used,
                   "l2": f"inputs larger than L2: {n_rep} cache replicas ({n_rep * used / 1e6:.0f} MB "
                         f"stored) rotated every step",
                   "launch": "CUDA graph of kvq_trizone_decode_attn calls"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": read_traffic("trizone_decode_traffic.txt", w.name, _kernel_sha(TZ_FILES)),
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes": nb["decode"]},
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": out_host.numel() * 4},
        "gpu_launches": steps,
        "clocks": clocks,
        "path": {"decode_us": us_step, "decode_per_launch": single, "build_us": build_us,
                 "build_gbs": build_bytes / (build_us * 1e-6) / 1e9},
        "parity_sample": parity,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = trizone_cpu_baseline(w, inp)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main_serving(args):
    """Serving: 16 sequences (32 query heads over 8 KV heads, head_dim 128, 4-bit)
    with lengths L ~ U[8192, 32768].  Reports the prefill of 16 full 32,768-token
    chunks (rate and time), and times steps of one kvq_append_token (with its
    flushes) + one kvq_decode_attn over the ragged caches; the decode alone is
    timed too for the roofline."""
    import torch
    import torch.distributed as dist
    from quantized_kv_cache_11_gb300 import kvq
    from quantized_kv_cache_11_gb300 import synthetic as S

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvq.load_library()
    w = S.SERVING
    inp = S.generate(w)
    B, H, D, T = w.batch, w.n_kv_heads, w.head_dim, w.context
    K = torch.from_numpy(inp["K"]).to(dev)
    V = torch.from_numpy(inp["V"]).to(dev)
    q = torch.from_numpy(inp["q"]).to(dev)
    # (i) prefill of the full chunks
    full = kvq.QuantizedKVCache(B, H, D, w.bits, T, w.tail_cap, device=dev)
    full.prefill(K, V, [T] * B, [0] * B)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record()
    for _ in range(5):
        full.prefill(K, V, [T] * B, [0] * B)
    p1.record()
    torch.cuda.synchronize()
    prefill_us = p0.elapsed_time(p1) * 1000 / 5
    prefill_bytes = prefill_algorithmic_bytes(w, T, 0) * 1  # all 16 sequences of T tokens
    del full
    torch.cuda.empty_cache()
    # (ii) the ragged caches, then append + decode steps
    seq, nt = inp["seq_len"].astype(int), inp["n_tail"].astype(int)
    cache = kvq.QuantizedKVCache(B, H, D, w.bits, T + 8192, w.tail_cap, device=dev)
    cache.prefill(K, V, seq.tolist(), nt.tolist())
    kn = torch.randn(B, H, D, device=dev).half()
    vn = torch.randn(B, H, D, device=dev).half()
    out = torch.empty(B, w.n_q_heads, D, dtype=torch.float32, device=dev)

    def step():
        cache.append(kn, vn)
        cache.decode(q, w.sm_scale, out=out)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    per_graph = 64
    steps_wanted = min(args.steps, 4096)  # the caches hold 8192 more tokens per sequence
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            step()
    reps = max(1, math.ceil(steps_wanted / per_graph))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
    steps = reps * per_graph
    step_us = max_over_ranks(e0.elapsed_time(e1), dev) * 1000.0 / steps
    # the decode alone over the caches as they now are
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd):
        for _ in range(per_graph):
            cache.decode(q, w.sm_scale, out=out)
    gd.replay()
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record()
    for _ in range(8):
        gd.replay()
    d1.record()
    torch.cuda.synchronize()
    decode_us = max_over_ranks(d0.elapsed_time(d1), dev) * 1000.0 / (8 * per_graph)
    assert cache.device_errors() == 0
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    nq = cache.n_quant.cpu().numpy().astype(int)
    ntl = cache.n_tail.cpu().numpy().astype(int)
    dbytes = sum(algorithmic_bytes(w.scaled(batch=1), int(a), int(b)) for a, b in zip(nq, ntl))
    dbytes -= (B - 1) * w.n_q_heads * D * 6  # q and out counted once per batch above
    peak, peak_kind = load_peaks()
    achieved = dbytes / (decode_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": step_us, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": step_us / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(w.bits), "data": "synthetic",
        "config": {**serving_config(w, float(inp["seq_len"].mean())),
                   "l2": f"inputs larger than L2: {dbytes / 1e6:.0f} MB read per decode",
                   "launch": "CUDA graph of kvq_append_token + kvq_decode_attn"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "decode_kernel<128,4,4>",
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes": dbytes},
        "gpu_launches": 2 * steps,
        "clocks": clk.summary(),
        "path": {"step_us": step_us, "decode_us": decode_us, "append_us": step_us - decode_us,
                 "prefill_us": prefill_us, "prefill_gbs": prefill_bytes / (prefill_us * 1e-6) / 1e9,
                 "prefill_bytes": prefill_bytes, "mean_tokens_at_end": float((nq + ntl).mean())},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp)  # the decode over the caches as prefilled
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


RDKV_METRIC = "RDKV bit allocation (token weights + V/K widths): ms per prompt batch"
RDKV_SAMPLE_T = 1536  # prompt positions of the oracle's sample segment


def rdkv_flops(w) -> float:
    """Algorithmic tensor flops of one token-weight pass: the causal score matrix
    of every (sequence, query head), 2 D flops per (query, key <= query) pair."""
    T = w.context
    return float(w.batch * w.n_q_heads) * T * (T + 1) / 2 * 2 * w.head_dim


def rdkv_oracle_sample(w, q, inp, T):
    """The oracle's three phases on the first T prompt positions of one segment;
    returns (seconds, scale to the full workload by the causal pair count)."""
    from oracle import rdkv_oracle as R
    G = w.gqa
    t0 = time.perf_counter()
    R.segment_allocation(q[0, :T, 0:G], inp["K"][0, :T, 0], inp["V"][0, :T, 0], T - w.trizone_fresh,
                         w.sm_scale, 3.0, 4.0)
    dt = time.perf_counter() - t0
    scale = w.batch * w.n_kv_heads * (w.context * (w.context + 1)) / (T * (T + 1))
    return dt, scale


def main_rdkv(args):
    """RDKV allocation of the mixed-width workload's prompts (4 sequences x 65,536
    positions, 32 query heads over 8 KV heads): a step is kvq_rdkv_token_weights
    (two tensor-core passes over the causal scores) + kvq_rdkv_allocate (costs,
    Lagrangian V widths of the 65,408 old tokens, channel statistics, K widths),
    at 3 bits per old token and 4 bits per channel."""
    import torch
    import torch.distributed as dist
    from quantized_kv_cache_11_gb300 import kvq
    from quantized_kv_cache_11_gb300 import synthetic as S

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvq.load_library()
    w = S.TRIZONE
    if args.rdkv_tokens:
        w = w.scaled(name=f"llama31_8b_trizone_b4_t{args.rdkv_tokens}", context=args.rdkv_tokens)
    inp = S.generate(w)
    qn = S.prompt_queries(w)
    B, H, T, D = w.batch, w.n_kv_heads, w.context, w.head_dim
    t_old = T - w.trizone_fresh
    nt, to = [T] * B, [t_old] * B
    vb, kb = 3.0, 4.0
    q = torch.from_numpy(qn).to(dev)
    k = torch.from_numpy(inp["K"]).to(dev)
    v = torch.from_numpy(inp["V"]).to(dev)
    a = kvq.RDKVAllocator(B, w.n_q_heads, H, T, t_old, device=dev)
    warm, steps = min(max(args.warmup, 3), 5), max(1, min(args.steps, 5))
    for _ in range(warm):
        a.run(q, k, v, nt, to, vb, kb, w.sm_scale)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for e in ev:
            e[0].record()
            a.token_weights(q, k, nt, w.sm_scale)
            e[1].record()
            a.allocate(q, k, v, nt, to, vb, kb)
            e[2].record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    tw_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    al_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    step_ms = max_over_ranks(ev[0][0].elapsed_time(ev[-1][2]) / steps, dev)
    # end to end: prompt tensors from pinned host memory, widths back to the host
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (qn, inp["K"], inp["V"]))
    vwh = torch.empty(a.v_width.shape, dtype=torch.uint8).pin_memory()
    kwh = torch.empty(a.k_width.shape, dtype=torch.uint8).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(2):
        q.copy_(qh, non_blocking=True)
        k.copy_(kh, non_blocking=True)
        v.copy_(vh, non_blocking=True)
        a.run(q, k, v, nt, to, vb, kb, w.sm_scale)
        vwh.copy_(a.v_width, non_blocking=True)
        kwh.copy_(a.k_width, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / 2
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    # parity sample: weights of the last 16 keys of one segment, widths given the costs
    from oracle import rdkv_oracle as R
    G = w.gqa
    kk = inp["K"][0, :, 0].astype(np.float64)
    tail = np.zeros(16)
    for tau in range(T - 16, T):
        for g in range(G):
            sc = w.sm_scale * (kk[:tau + 1] @ qn[0, tau, g].astype(np.float64))
            p = np.exp(sc - sc.max())
            p /= p.sum()
            tail[:tau + 1 - (T - 16)] += p[T - 16:tau + 1]
    got = a.w[0, 0, T - 16:].double().cpu().numpy()
    ref_vw, _ = R.allocate(a.W_t[0, 0, :t_old].cpu().numpy(), R.V_WIDTHS, R.budget_bits(vb, t_old))
    ref_kw, _ = R.allocate(a.W_c[0, 0].cpu().numpy(), R.K_WIDTHS, R.budget_bits(kb, D))
    parity = {"segments_checked": 1, "last_keys_weight_max_rel": float(np.abs(got / tail - 1).max()),
              "v_widths_equal": bool((a.v_width[0, 0, :t_old].cpu().numpy() == ref_vw).all()),
              "k_widths_equal": bool((a.k_width[0, 0].cpu().numpy() == ref_kw).all())}
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        pk = json.load(f)
    peak = float(pk.get("bf16_tflops_sustained") or pk["bf16_tflops"])
    flops = 2 * rdkv_flops(w)  # both passes compute the causal scores
    achieved = flops / (tw_ms * 1e-3) / 1e12
    vwd = np.bincount(a.v_width.cpu().numpy().ravel(), minlength=17)[[0, 2, 4, 8, 16]]
    line = {
        "metric": RDKV_METRIC, "value": step_ms, "unit": "ms/step", "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": step_ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 in, f32 accumulate", "data": "synthetic",
        "config": {"workload": "rdkv_" + w.name, "batch": B, "n_q_heads": w.n_q_heads, "n_kv_heads": H,
                   "head_dim": D, "prompt_tokens": T, "old_tokens": t_old, "v_avg_bits": vb, "k_avg_bits": kb,
                   "l2": f"inputs larger than L2: {q.numel() * 2 / 1e9:.2f} GB of prompt queries per step"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "attn_tc_kernel<1> + attn_tc_kernel<2> (tcgen05)",
                     "peak_source": "measured bf16_tflops_sustained (fp16 has the bf16 rate)",
                     "algorithmic_flops": flops},
        "e2e": {"value": e2e_ms, "unit": "ms/step", "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel()) * 2,
                "d2h_bytes_per_step": a.v_width.numel() + a.k_width.numel()},
        "gpu_launches": steps * 7,
        "clocks": clk.summary(),
        "path": {"token_weights_ms": tw_ms, "allocate_ms": al_ms,
                 "v_width_counts_0_2_4_8_16": vwd.tolist(),
                 "v_bits_per_old_token": float((vwd * np.array([0, 2, 4, 8, 16])).sum() / (B * H * t_old))},
        "parity_sample": parity,
    }
    if world == 1 and not args.no_cpu_baseline:
        import torch as _t
        dt, scale = rdkv_oracle_sample(w, qn, inp, RDKV_SAMPLE_T)
        line["cpu_baseline"] = {"value": dt * scale * 1e3, "unit": "ms/step", "cores": _t.get_num_threads(),
                                "kind": "oracle",
                                "sample": f"oracle token weights + allocation of 1 of {B * H} segments on its "
                                          f"first {RDKV_SAMPLE_T} prompt positions, scaled x{scale:.0f} by the "
                                          f"causal pair count"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_rdkv(args):
    """The oracle on the host cores for the RDKV allocation: each step runs the
    three phases on a sample segment, scaled to the full workload."""
    from quantized_kv_cache_11_gb300 import synthetic as S
    import torch
    w = S.TRIZONE
    inp = S.generate(w)
    qn = S.prompt_queries(w, batches=[0])
    times, scale = [], 1.0
    for i in range(args.warmup + args.steps):
        dt, scale = rdkv_oracle_sample(w, qn, inp, 512)
        if i >= args.warmup:
            times.append(dt)
    value = statistics.mean(times) * scale * 1e3
    sample = (f"oracle token weights + allocation of 1 of {w.batch * w.n_kv_heads} segments on its first 512 "
              f"prompt positions per step, scaled x{scale:.0f} by the causal pair count")
    print(json.dumps({
        "impl": "reference", "metric": RDKV_METRIC, "value": value, "unit": "ms/step", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "rdkv_" + w.name},
        "cpu_baseline": {"kind": "oracle", "cores": torch.get_num_threads(), "sample": sample,
                         "value": value, "unit": "ms/step"},
        "e2e": {"value": value, "unit": "ms/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


DECODE_FILES = ("kvq_decode_impl.cuh", "kvq_decode.cu", "kvq_decode_cps2.cu", "kvq_decode_cps4.cu", "kvq_common.cuh")
ROPE_FILES = ("kvq_decode_impl.cuh", "kvq_decode_rope.cu", "kvq_common.cuh")


def _kernel_sha(files=DECODE_FILES) -> str:
    """Hash of the kernel's code: the sources with comments and whitespace removed,
    so that a traffic record stays tied to the code it was measured on."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "quantized_kv_cache_11_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)                 # line comments
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
