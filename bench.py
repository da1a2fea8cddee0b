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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=25000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--bits", type=int, default=2, choices=[2, 4])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def workload(bits):
    from quantized_kv_cache_11_gb300 import synthetic as S
    return S.LLAMA31_8B_128K if bits == 2 else S.LLAMA31_8B_128K_4BIT


def algorithmic_bytes(w, n_quant, n_tail) -> int:
    """Bytes one decode step must move: packed K/V codes, fp16 scale + zero of
    every group, the fp16 tail, q in and the fp32 output."""
    D, H, b = w.head_dim, w.n_kv_heads, w.bits
    per_tok = 2 * D * b // 8 + (2 * D // 32) * 2  # codes K+V, V meta (fp16 scale + zero per 32 ch)
    k_meta = (n_quant // 32) * 2 * D * 2  # per key group: scale + zero per channel
    tail = n_tail * D * 2 * 2
    return w.batch * H * (n_quant * per_tok + k_meta + tail) + w.batch * w.n_q_heads * D * (2 + 4)


def prefill_algorithmic_bytes(w, n_quant, n_tail) -> int:
    """Prefill reads the fp16 K and V of every token and writes the packed cache
    (codes and fp16 metadata) plus the fp16 tail."""
    read = 2 * w.batch * (n_quant + n_tail) * w.n_kv_heads * w.head_dim * 2
    write = algorithmic_bytes(w, n_quant, n_tail) - w.batch * w.n_q_heads * w.head_dim * 6
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


def cpu_baseline(w, inp, budget_s=12.0):
    """The oracle as it stands on this host: dequantize + fp64 attention for one
    KV head (its 4 query heads) over the whole context, repeated for ~budget_s,
    scaled by the number of KV heads to one full decode step."""
    from oracle import kvq_oracle as O
    import torch
    st = O.quantize_sequence(inp["K"][0][:, :1], inp["V"][0][:, :1], int(inp["seq_len"][0]),
                             int(inp["n_tail"][0]), w.bits)
    q = inp["q"][0][:w.gqa]
    times = []
    t_end = time.perf_counter() + budget_s
    while time.perf_counter() < t_end or len(times) < 2:
        t0 = time.perf_counter()
        O.sequence_attention(q, st, w.sm_scale)
        times.append(time.perf_counter() - t0)
    per_head = statistics.median(times)
    return {"value": per_head * w.n_kv_heads * 1e6, "unit": UNIT, "kind": "oracle",
            "cores": torch.get_num_threads(),
            "sample": f"1 of {w.n_kv_heads} KV heads ({w.gqa} query heads) over all "
                      f"{int(inp['seq_len'][0])} tokens, median of {len(times)} runs, "
                      f"x{w.n_kv_heads}; numpy fp64 (BLAS threads as the host sets them)"}


def run_reference(args):
    """The oracle on the host cores, same metric/config: each step times the
    oracle on a slice of one KV head's context, sized so the run ends in minutes,
    and is scaled to a full decode step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import kvq_oracle as O
    from quantized_kv_cache_11_gb300 import synthetic as S
    import torch
    w = workload(args.bits)
    inp = S.generate(w)
    n = int(inp["seq_len"][0])
    nt = int(inp["n_tail"][0])
    st = O.quantize_sequence(inp["K"][0][:, :1], inp["V"][0][:, :1], n, nt, w.bits)
    # per-step budget ~ 150 s / (steps + warmup), slice length a multiple of 32
    per_step = 150.0 / max(1, args.steps + args.warmup)
    t0 = time.perf_counter()
    sl = 1024
    O.decode_attention(inp["q"][0][:w.gqa],
                       O.dequantize_keys(st["k_codes"][:, :sl], st["k_scale"][:, :sl // 32],
                                         st["k_zero"][:, :sl // 32]),
                       O.dequantize_values(st["v_codes"][:, :sl], st["v_scale"][:, :sl],
                                           st["v_zero"][:, :sl]), w.sm_scale)
    t_blk = max(time.perf_counter() - t0, 1e-5)
    tokens = int(min(n - nt, max(32, (per_step / t_blk * sl) // 32 * 32)))
    nblk = (n - nt) // tokens
    q = inp["q"][0][:w.gqa]
    times = []
    for i in range(args.warmup + args.steps):
        j = i % max(1, nblk)
        a, e = j * tokens, (j + 1) * tokens
        t0 = time.perf_counter()
        kk = O.dequantize_keys(st["k_codes"][:, a:e], st["k_scale"][:, a // 32:e // 32],
                               st["k_zero"][:, a // 32:e // 32])
        vv = O.dequantize_values(st["v_codes"][:, a:e], st["v_scale"][:, a:e], st["v_zero"][:, a:e])
        O.decode_attention(q, kk, vv, w.sm_scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    scale = w.n_kv_heads * (n - nt) / tokens
    value = statistics.mean(times) * scale * 1e6
    sample = (f"oracle dequant + fp64 attention on {tokens} of {n - nt} quantized tokens of 1 of "
              f"{w.n_kv_heads} KV heads per step, scaled x{scale:.1f} to a full step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1000.0,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "bits": w.bits},
        "cpu_baseline": {"kind": "oracle", "cores": torch.get_num_threads(), "sample": sample,
                         "value": value, "unit": UNIT},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
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

    w = workload(args.bits)
    inp = S.generate(w)
    n_quant = int(inp["seq_len"][0] - inp["n_tail"][0])
    n_tail = int(inp["n_tail"][0])
    K = torch.from_numpy(inp["K"]).to(dev)
    V = torch.from_numpy(inp["V"]).to(dev)
    q = torch.from_numpy(inp["q"]).to(dev)

    # ---- cache replicas: total well above the 129 MB L2
    probe = kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, w.bits, w.context, w.tail_cap,
                                 device=dev)
    n_rep = max(4, math.ceil(3 * 128e6 / probe.nbytes) + 1)
    caches = [probe] + [kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, w.bits, w.context,
                                             w.tail_cap, device=dev) for _ in range(n_rep - 1)]
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
    prefill_bytes = prefill_algorithmic_bytes(w, n_quant, n_tail)

    # ---- append timing on a separate cache (keeps the replicas unchanged)
    app = kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, w.bits, w.context + 4096,
                               w.tail_cap, device=dev)
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
    for i in range(max(args.warmup, 3)):
        caches[i % n_rep].decode(q, w.sm_scale, out=outs[i % n_rep])
    torch.cuda.synchronize()
    parity = None
    if rank == 0:
        from oracle import kvq_oracle as O
        st = O.quantize_sequence(inp["K"][0][:, :1], inp["V"][0][:, :1], int(inp["seq_len"][0]),
                                 n_tail, w.bits)
        ref = O.sequence_attention(inp["q"][0][:w.gqa], st, w.sm_scale)
        got = outs[0][0, :w.gqa].double().cpu().numpy()
        parity = {"kv_heads_checked": 1, "max_abs": float(np.abs(got - ref).max())}
    per_graph = n_rep * max(1, 256 // n_rep)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per_graph):
            caches[i % n_rep].decode(q, w.sm_scale, out=outs[i % n_rep])
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    reps = max(1, math.ceil(args.steps / per_graph))
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
    elapsed_ms = e0.elapsed_time(e1)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    us_step = elapsed_ms * 1000.0 / steps

    # ---- end to end through the public API: pinned host q in, fp32 output out
    q_host = torch.from_numpy(inp["q"]).pin_memory()
    out_host = torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(q)
    n_e2e = min(steps, 4000)
    for i in range(16):
        q_dev.copy_(q_host, non_blocking=True)
        caches[i % n_rep].decode(q_dev, w.sm_scale, out=outs[i % n_rep])
        out_host.copy_(outs[i % n_rep], non_blocking=True)
    torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record()
    for i in range(n_e2e):
        q_dev.copy_(q_host, non_blocking=True)
        caches[i % n_rep].decode(q_dev, w.sm_scale, out=outs[i % n_rep])
        out_host.copy_(outs[i % n_rep], non_blocking=True)
    x1.record()
    torch.cuda.synchronize()
    e2e_us = x0.elapsed_time(x1) * 1000.0 / n_e2e

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = load_peaks()
    nbytes = algorithmic_bytes(w, n_quant, n_tail)
    achieved = nbytes / (us_step * 1e-6) / 1e9
    traffic = None
    tf = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    if os.path.exists(tf):
        rec = {}
        with open(tf) as f:
            for ln in f:
                if ":" in ln and not ln.lstrip().startswith("#"):
                    k, v = ln.split(":", 1)
                    rec[k.strip()] = v.strip()
        # only while the kernel source is the one the counters were taken from
        if rec.get("workload") == w.name and rec.get("kernel_source_sha") == _kernel_sha():
            traffic = int(rec["dram_bytes_per_launch"])
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": us_step / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "context": w.context,
                   "n_quant": n_quant, "n_tail": n_tail, "bits": w.bits, "group": 32,
                   "l2": f"inputs larger than L2: {n_rep} cache replicas "
                         f"({n_rep * probe.nbytes / 1e6:.0f} MB) rotated every step",
                   "launch": "CUDA graph of kvq_decode_attn calls"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes": nbytes},
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": out_host.numel() * 4},
        "gpu_launches": steps,
        "clocks": clocks,
        "path": {"decode_us": us_step, "prefill_us": prefill_us,
                 "prefill_gbs": prefill_bytes / (prefill_us * 1e-6) / 1e9, "append_us": append_us},
        "parity_sample": parity,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _kernel_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("kvq_decode.cu", "kvq_common.cuh"):
        with open(os.path.join(ROOT, "quantized_kv_cache_11_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
