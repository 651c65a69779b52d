"""Benchmark of the W4A16 decode GEMV library on GB300.

One step = one replay of the CUDA graph that streams a whole Qwen-7B-shaped
decode step's INT4 projection weights: 28 layers x {[q;k;v], o, [gate;up],
down}, M = 1 (112 GEMV launches, 3.37 GB of packed weights and scales).
The metric is achieved GB/s of algorithmic bytes (packed weights + fp16
scales + fp16 activations + fp16 outputs); the weights (3.37 GB) are far
larger than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  Besides the contract keys it reports
  roofline      the dominant kernel against the measured HBM copy bandwidth
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
  e2e           the same metric through w4a16_layer_seq_run_host: host x in,
                every output back, copies inside the timed region
  configs       per-workload-shape us/GEMV and GB/s with cold L2 (weights
                rotated over >= 4 x L2), warm L2 and single-launch latency,
                as fractions of the measured peak and the nominal 8 TB/s,
                including the M = 1..16 down sweep
  clocks        SM clock and throttle reasons sampled during the timed region

--impl reference times the CPU oracle (the only reference implementation
there is) on the same config, metric and unit.  --gpus N under torchrun runs
N independent replicas (the GEMV has no data-path exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT4 GEMV achieved HBM GB/s and % of GB300 roofline (µs/GEMV, M=1..16)"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-shape table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--case", default=None,
                    help="profiling mode: run one workload GEMV (tiny, q_proj, kv_proj, gate_up, "
                         "down_m1 .. down_m16), seqN (an N-layer M=1 layer sequence), attn "
                         "(decode attention, T = 8192) or q4k ([gate; up] as GGUF Q4_K blocks), "
                         "--launches times and exit")
    ap.add_argument("--launches", type=int, default=4)
    return ap.parse_args()


# ---------------------------------------------------------------- workload

def workload_gemvs(M=1):
    """The GEMVs of one decode step: (name, N, K, M) per launch, in order
    ([q; k; v] and [gate; up] are one launch each)."""
    import synth
    H, KV, F = synth.HIDDEN, synth.KV_DIM, synth.FFN
    one = [("qkv", H + 2 * KV, H), ("o", H, H), ("gate_up", 2 * F, H), ("down", H, F)]
    return [(n, N, K, M) for _ in range(synth.N_LAYERS) for (n, N, K) in one]


def gemv_bytes(N, K, M, group=128):
    """Algorithmic bytes of one GEMV: packed weights, fp16 scales, x, y."""
    return N * K // 2 + 2 * N * (K // group) + 2 * M * K + 2 * M * N


def config_block():
    import synth
    g = workload_gemvs()
    return {
        "workload": "Qwen-7B-shaped decode weight stream: 28 layers x {q,k,v,o,gate,up,down} "
                    "INT4 g128 GEMVs at M=1 ([q;k;v] and [gate;up] one GEMV each), one "
                    "CUDA-graph replay per step (one persistent task-list launch)",
        "layers": synth.N_LAYERS, "hidden": synth.HIDDEN, "kv_dim": synth.KV_DIM, "ffn": synth.FFN,
        "M": 1, "group": 128, "gemvs_per_step": len(g),
        "bytes_per_step": sum(gemv_bytes(N, K, M) for _, N, K, M in g),
        "l2_policy": "inputs larger than L2 (3.37 GB of weights vs 129 MB L2); no flush",
        "inputs": "seeded synthetic: W ~ N(0, 0.02) quantised to INT4 g128, x ~ N(0, 1) fp16",
    }


# ---------------------------------------------------------------- helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback"


# The sources the step's kernel (the M = 1 task-list launch) is built and
# launched from: its kernel, the shared device helpers and declarations, the
# host code that builds the task table, and the public header.
STEP_KERNEL_SOURCES = ("int4_weight_only_gemv_gb300/csrc/gemv_m1.cu", "int4_weight_only_gemv_gb300/csrc/ptx.cuh",
                       "int4_weight_only_gemv_gb300/csrc/kernels.h", "int4_weight_only_gemv_gb300/csrc/api.cu",
                       "include/w4a16.h")


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in STEP_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(rel.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per step from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") == kernel_source_hash():
            return d.get("dram_bytes_per_step")
    except Exception:  # noqa: BLE001
        pass
    return None


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of x over all ranks (the slowest replica's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbps(bytes_per_step: int, ms_per_step: float, world: int) -> float:
    """Whole-job GB/s: every replica streams bytes_per_step per step."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"w4a16_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [t.strip() for t in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- CPU oracle

def oracle_sample_plan(budget_s, steps):
    """Rows of layer 0's projections the oracle computes per step, sized so
    `steps` steps take about budget_s seconds; returns (plan, bytes)."""
    import numpy as np

    import oracle
    import synth
    rate = _oracle_mac_rate()
    macs = rate * budget_s / max(steps, 1)
    shapes = [(name, *synth.proj_shape(name)) for name in synth.PROJ_NAMES]
    total_macs = sum(N * K for _, N, K in shapes)
    frac = min(1.0, macs / total_macs)
    plan, nbytes = [], 0
    for pj, (name, N, K) in enumerate(shapes):
        nrows = max(1, int(N * frac))
        w = synth.weights(N, K, synth.layer_seed(0, pj))
        qw, sc = oracle.quantize(w.numpy())
        x = synth.activations(1, K, synth.layer_seed(0, 7)).numpy().view(np.uint16)
        rows = np.linspace(0, N - 1, nrows).astype(np.int64)
        plan.append((qw, sc, x, rows))
        nbytes += nrows * (K // 2 + 2 * (K // 128) + 2) + 2 * K
    return plan, nbytes, frac


def _oracle_mac_rate():
    import numpy as np

    import oracle
    import synth
    w = synth.weights(64, 3584, 1).numpy()
    qw, sc = oracle.quantize(w)
    x = synth.activations(1, 3584, 1).numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle.gemv(qw, sc, x)
    dt = time.perf_counter() - t0
    return 64 * 3584 / dt


def run_oracle_steps(plan, steps):
    import oracle
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        for qw, sc, x, rows in plan:
            oracle.gemv_rows(qw, sc, x, rows)
        times.append(time.perf_counter() - t0)
    return times


def cpu_baseline(budget_s=15.0):
    plan, nbytes, frac = oracle_sample_plan(budget_s, 1)
    t = run_oracle_steps(plan, 1)[0]
    # a whole layer takes less than the budget: repeat it to fill the budget
    passes = max(1, int(budget_s / t)) if frac >= 1.0 else 1
    if passes > 1:
        t += sum(run_oracle_steps(plan, passes - 1))
    line = {"value": nbytes * passes / t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"single-threaded C oracle (FP64) on {frac:.4f} of the rows of each of "
                      f"layer 0's 7 projections ({nbytes} algorithmic bytes), {passes} pass(es), "
                      f"{t:.1f} s; the oracle uses 1 of the host's cores"}
    line.update(host_cpu())
    line["per_config"] = oracle_config_timing()
    return line


def bench_reference(args, rank, world):
    """The reference arm: the CPU oracle, timed on the host, rank 0 only."""
    if rank != 0:
        return None
    budget = 100.0
    plan, nbytes, frac = oracle_sample_plan(budget, args.steps + args.warmup)
    run_oracle_steps(plan, args.warmup)
    times = run_oracle_steps(plan, args.steps)
    total = sum(times)
    value = nbytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step: {frac:.5f} of the rows of each of layer 0's "
                                   f"7 projections ({nbytes} algorithmic bytes)", **host_cpu()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


# ---------------------------------------------------------------- GPU arm

def build_weights(dev, n_layers=None):
    """n_layers (default 28) layers of packed weights, drawn on the GPU and
    quantised there; the q, k, v weights of a layer are stacked in one
    allocation, and so are gate and up, so that each stack is one GEMV."""
    import torch

    import int4_weight_only_gemv_gb300 as w4
    import synth
    layers = []
    for l in range(synth.N_LAYERS if n_layers is None else n_layers):
        lw = {}
        for names, idx, key in ((("q", "k", "v"), (0, 1, 2), "qkv"), (("gate", "up"), (4, 5), "gate_up"),
                                (("o",), (3,), None), (("down",), (6,), None)):
            ws = [synth.weights(*synth.proj_shape(synth.PROJ_NAMES[i]), synth.layer_seed(l, i), dev)
                  for i in idx]
            qw, sc = w4.w4a16_quantize(torch.cat(ws) if len(ws) > 1 else ws[0])
            del ws
            r = 0
            for name, i in zip(names, idx):
                n = synth.proj_shape(synth.PROJ_NAMES[i])[0]
                lw[name] = (qw[r:r + n], sc[r:r + n])
                r += n
            if key:
                lw[key] = (qw, sc)
        layers.append(lw)
    torch.cuda.synchronize()
    if w4.w4a16_device_status(clear=True):
        raise RuntimeError("quantisation flagged bad input")
    return layers


def make_io(dev, M=1, n_layers=None):
    import torch

    import synth
    L, H, KV, F = synth.N_LAYERS if n_layers is None else n_layers, synth.HIDDEN, synth.KV_DIM, synth.FFN
    x = torch.cat([synth.activations(M, H, synth.layer_seed(l, 7), dev) for l in range(L)])
    io = {"x": x.view(L, M, H)}
    for name, width in (("y_q", H), ("y_k", KV), ("y_v", KV), ("y_o", H), ("y_gu", 2 * F),
                        ("y_down", H)):
        io[name] = torch.empty((L, M, width), dtype=torch.float16, device=dev)
    return io


def time_graph_replays(seq, stream, steps, dist_barrier):
    import torch
    torch.cuda.synchronize()
    dist_barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        seq.run(stream)
    end.record(stream)
    torch.cuda.synchronize()
    dist_barrier()
    return start.elapsed_time(end)


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal


def host_cpu():
    """Model name and logical core count of this host."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:  # noqa: BLE001
            pass
    import platform
    return {"host_cores": os.cpu_count(), "cpu_model": model or platform.machine()}


def gemv_line(qw, sc, M, dev, gemv=None, reps=5, seed=77):
    """One GEMV shape measured three ways:
      cold     -- a CUDA graph of max(200, R) GEMVs cycling over R distinct
                  copies of the weights with R * weight bytes >= 4 x L2, so
                  every launch streams its weights from HBM;
      warm     -- a graph of 200 GEMVs on one copy (L2-resident when it fits);
      single   -- an event pair around one launch outside any graph (median
                  of 20), the per-call latency a caller sees.
    Returns us per GEMV and GB/s of algorithmic bytes, with the fraction of
    the measured HBM peak and of the nominal 8 TB/s."""
    import math

    import torch

    import int4_weight_only_gemv_gb300 as w4
    import synth
    gemv = gemv or w4.w4a16_gemv
    N, K = qw.shape[0], qw.shape[1] * 8
    wbytes = qw.numel() * 4 + sc.numel() * 2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(4 * l2 / wbytes))
    G = max(200, R)
    copies = [(qw.clone(), sc.clone()) for _ in range(R)]
    xs = [synth.activations(M, K, seed + i, dev) for i in range(8)]
    ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for _ in range(8)]
    stream = torch.cuda.Stream()

    def graph_of(which):
        with torch.cuda.stream(stream):
            for i in range(min(G, 8)):
                gemv(*copies[which(i)], xs[i % 8], ys[i % 8])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                gemv(*copies[which(i)], xs[i % 8], ys[i % 8])
        return g

    def time_graph(g, n):
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()
        s.record(cur)
        for _ in range(reps):
            g.replay()
        e.record(cur)
        torch.cuda.synchronize()
        return 1e3 * s.elapsed_time(e) / (reps * n)

    cold = time_graph(graph_of(lambda i: i % R), G)
    warm = time_graph(graph_of(lambda i: 0), G)
    singles = []
    cur = torch.cuda.current_stream()
    for i in range(20):
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(cur)
        gemv(*copies[i % R], xs[i % 8], ys[i % 8])
        e.record(cur)
        torch.cuda.synchronize()
        singles.append(1e3 * s.elapsed_time(e))
    b = gemv_bytes(N, K, M)
    peak, _ = measured_peak()
    gbps = b / cold / 1e3
    del copies
    return {"M": M, "N": N, "K": K, "bytes": b, "us_per_gemv": round(cold, 3), "GBps": round(gbps, 1),
            "frac_measured": round(gbps / peak, 4), "frac_nominal_8TBps": round(gbps / NOMINAL_HBM_GBS, 4),
            "warm_us": round(warm, 3), "single_launch_us": round(statistics.median(singles), 3),
            "rotation": f"{R} weight copies ({R * wbytes / 1e6:.0f} MB >= 4 x {l2 / 1e6:.0f} MB L2), "
                        f"graph of {G} GEMVs"}


def oracle_config_timing(budget_s=0.25):
    """The single-threaded C oracle on each workload GEMV shape, timed on a
    row sample sized to take about budget_s seconds, median of 3 runs, and
    extrapolated to us per full GEMV (the oracle's cost is linear in rows)."""
    import numpy as np

    import oracle
    import synth
    rate = _oracle_mac_rate()
    out = {}
    for cfg in synth.ALL_GEMVS:
        nrows = max(1, min(cfg.N, int(rate * budget_s / (cfg.M * cfg.K))))
        w = synth.weights(nrows, cfg.K, cfg.seed).numpy()
        qw, sc = oracle.quantize(w)
        x = synth.activations(cfg.M, cfg.K, cfg.seed).numpy().view(np.uint16)
        times = []
        for _ in range(3):
            t0 = time.perf_counter()
            oracle.gemv(qw, sc, x)
            times.append(time.perf_counter() - t0)
        t = statistics.median(times) * cfg.N / nrows
        out[cfg.name] = {"us_per_gemv": round(1e6 * t, 1), "rows_timed": nrows,
                         "GBps": round(gemv_bytes(cfg.N, cfg.K, cfg.M) / t / 1e9, 4)}
    return out


def per_config_table(layers, dev, reps=5):
    """Per workload shape: us/GEMV and GB/s with cold L2 (rotation over >= 4 x
    L2 of weight copies), warm L2, and single-launch latency (gemv_line); the
    configured shapes use their own seeds, the stacked [q; k; v] and the W4A8
    lines the step's layer-0 weights."""
    import int4_weight_only_gemv_gb300 as w4
    import synth
    out = {}
    for cfg in synth.ALL_GEMVS:
        qw, sc = w4.w4a16_quantize(synth.weights(cfg.N, cfg.K, cfg.seed, dev))
        out[cfg.name] = gemv_line(qw, sc, cfg.M, dev, reps=reps, seed=cfg.seed)
        del qw, sc
    out["qkv"] = gemv_line(*layers[0]["qkv"], 1, dev, reps=reps)
    # the W4A8 variant on the M = 1 shapes (activations quantised in-kernel)
    for label, key in (("q_proj_a8", "q"), ("gate_up_a8", "gate_up"), ("down_m1_a8", "down")):
        out[label] = gemv_line(*layers[0][key], 1, dev, gemv=w4.w4a16_gemv_a8, reps=reps)
        out[label]["note"] = "W4A8: int8 activations, per-64 block scales computed in the kernel"
    out["gate_up_q4k"] = q4k_line(dev, 20)
    out["down_q4k"] = q4k_line(dev, 20, N=synth.HIDDEN, K=synth.FFN)
    out["attn_decode_T8192"] = attn_decode_line(dev, 20)
    out["layer_seq_qkv_bias_swiglu"] = epilogue_step(layers, dev, 20, ("q", "k", "v"))
    out["layer_seq_bias_swiglu"] = epilogue_step(layers, dev, 20, synth.PROJ_NAMES)
    out["layer_seq_w4a8"] = epilogue_step(layers, dev, 20, (), act_int8=True)
    return out


def q4k_line(dev, reps, N=None, K=None):
    """A projection as GGUF Q4_K blocks at M = 1, by default the [gate; up]
    shape (N = 37888, K = 3584): a CUDA graph of 28 GEMVs over 28 distinct
    block sets (cold L2), us per GEMV and GB/s over the block bytes plus x
    and y."""
    import torch

    import int4_weight_only_gemv_gb300 as w4
    import synth
    N = 2 * synth.FFN if N is None else N
    K = synth.HIDDEN if K is None else K
    nb = N * (K // 256)
    g = torch.Generator(device=dev).manual_seed(4)
    sets = []
    for _ in range(synth.N_LAYERS):
        b = torch.randint(0, 256, (nb, 144), generator=g, dtype=torch.uint8, device=dev)
        d = (torch.rand((nb, 2), generator=g, device=dev) * 0.05 + 1e-3).half()
        b[:, 0:4] = d.view(torch.uint8).view(nb, 4)
        sets.append(b.view(-1))
    xs = [synth.activations(1, K, 90 + i, dev).view(-1) for i in range(len(sets))]
    ys = [torch.empty((N,), dtype=torch.float16, device=dev) for _ in sets]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for b, x, y in zip(sets, xs, ys):
            w4.w4a16_q4k_gemv(b, x, N, K, y=y)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for b, x, y in zip(sets, xs, ys):
            w4.w4a16_q4k_gemv(b, x, N, K, y=y)
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    s.record(cur)
    for _ in range(reps):
        gr.replay()
    e.record(cur)
    torch.cuda.synchronize()
    us = 1e3 * s.elapsed_time(e) / (reps * len(sets))
    bts = nb * 144 + 2 * K + 2 * N
    return {"M": 1, "N": N, "K": K, "us_per_gemv": round(us, 3), "GBps": round(bts / us / 1e3, 1), "bytes": bts,
            "note": "GGUF Q4_K blocks (4.5 bits per weight), read as stored"}


def attn_decode_line(dev, reps, T=8192):
    """Decode attention of one token over an fp16 KV cache of T keys with the
    Qwen-7B head layout (28 query heads over 4 KV heads, head dimension 128):
    a CUDA graph of 28 calls over 28 distinct caches (cold L2: 28 x 16.8 MB),
    one workspace for all of them, us per call and GB/s over the cache bytes
    plus q and o."""
    import torch

    import int4_weight_only_gemv_gb300 as w4
    import synth
    H, Hkv, D = synth.HIDDEN // 128, synth.KV_DIM // 128, 128
    g = torch.Generator(device=dev).manual_seed(8192)
    caches = [(torch.randn((Hkv, T, D), generator=g, device=dev).half(),
               torch.randn((Hkv, T, D), generator=g, device=dev).half()) for _ in range(synth.N_LAYERS)]
    qs = [torch.randn((H, D), generator=g, device=dev).half() for _ in caches]
    os_ = [torch.empty((H, D), dtype=torch.float16, device=dev) for _ in caches]
    ws = w4.attn_decode_new_workspace(H, Hkv, T, dev)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for (k, v), q, o in zip(caches, qs, os_):
            w4.w4a16_attn_decode(q, k, v, T, o=o, workspace=ws)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for (k, v), q, o in zip(caches, qs, os_):
            w4.w4a16_attn_decode(q, k, v, T, o=o, workspace=ws)
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    s.record(cur)
    for _ in range(reps):
        gr.replay()
    e.record(cur)
    torch.cuda.synchronize()
    if w4.w4a16_device_status(clear=True):
        raise RuntimeError("a kernel flagged a failure")
    us = 1e3 * s.elapsed_time(e) / (reps * len(caches))
    b = 2 * Hkv * T * D * 2 + 2 * H * D * 2
    return {"H": H, "Hkv": Hkv, "T": T, "us_per_call": round(us, 3), "GBps": round(b / us / 1e3, 1),
            "bytes": b, "note": "fp16 KV cache, 28 rotated caches (cold L2), partial + merge launches"}


def epilogue_step(layers, dev, reps, bias_on, act_int8=False):
    """The 28-layer M = 1 step with the fused epilogues (output biases on the
    projections bias_on, SwiGLU between [gate; up] and down), or with
    act_int8 and nothing else the plain step as W4A8: ms per step and GB/s
    over the same algorithmic bytes plus the bias bytes."""
    import torch

    import int4_weight_only_gemv_gb300 as w4
    import synth
    H, KV, F = synth.HIDDEN, synth.KV_DIM, synth.FFN
    width = {"q": H, "k": KV, "v": KV, "o": H, "gate": F, "up": F, "down": H}
    g = torch.Generator().manual_seed(5)
    biases = [{n: (torch.randn(width[n], generator=g) * 0.1).to(torch.float16).to(dev) for n in bias_on}
              for _ in layers]
    io = make_io(dev)
    seq = w4.LayerSeq([{k: lw[k] for k in synth.PROJ_NAMES} for lw in layers], io, 1, H, KV, F,
                      biases=biases if bias_on else None, swiglu=not act_int8, act_int8=act_int8)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        seq.run(stream)
    ms = time_graph_replays(seq, stream, reps, lambda: None) / reps
    seq.close()
    b = config_block()["bytes_per_step"] + 2 * sum(width[n] for n in bias_on) * len(layers)
    note = ("W4A8: every GEMV with int8 activations quantised in-kernel" if act_int8 else
            "biases on " + "/".join(bias_on) + ", SwiGLU in the up projection's epilogue")
    return {"M": 1, "layers": len(layers), "ms_per_step": round(ms, 4), "GBps": round(b / ms / 1e6, 1),
            "bytes": b, "note": note}


def bench_ours(args, rank, world):
    import torch
    import torch.distributed as dist

    import int4_weight_only_gemv_gb300 as w4
    import synth
    from int4_weight_only_gemv_gb300 import build as wbuild

    wbuild.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if world > 1:
            dist.barrier()

    layers = build_weights(dev)
    io = make_io(dev)
    seq = w4.LayerSeq([{k: lw[k] for k in synth.PROJ_NAMES} for lw in layers], io, 1,
                      synth.HIDDEN, synth.KV_DIM, synth.FFN)
    stream = torch.cuda.current_stream()
    cfg = config_block()
    bytes_step = cfg["bytes_per_step"]

    for _ in range(args.warmup):
        seq.run(stream)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = time_graph_replays(seq, stream, args.steps, barrier)
    clocks = clk.summary()
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / args.steps
    value = aggregate_gbps(bytes_step, ms_step, world)

    # end to end: host x in, every output back, through the C ABI
    host = {"x": io["x"].cpu().pin_memory()}
    for k in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        host[k] = torch.empty(io[k].shape, dtype=torch.float16).pin_memory()
    h2d = host["x"].numel() * 2
    d2h = sum(host[k].numel() * 2 for k in host if k != "x")
    for _ in range(min(args.warmup, 5)):
        seq.run_host(host, stream)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        seq.run_host(host, stream)
    seq.sync()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps, world, dev)
    barrier()
    e2e_value = aggregate_gbps(bytes_step, 1e3 * e2e_s, world)
    if w4.w4a16_device_status(clear=True):
        raise RuntimeError("a kernel flagged a failure during the bench")

    configs = None if args.no_configs or rank != 0 else per_config_table(layers, dev)
    peak, peak_kind = measured_peak()
    achieved = bytes_step / (ms_step * 1e-3) / 1e9
    traffic = recorded_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "w4a16", "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "kernel": "gemv_m1_kernel (the step's task-list launch; per-launch "
                               "time = step time)"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * seq.num_launches,
        "clocks": clocks,
        "configs": configs,
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline()
    seq.close()
    return line if rank == 0 else None


def run_case(args):
    """One workload GEMV, or an N-layer M = 1 layer sequence (seqN), launched
    --launches times on the default stream (a small, self-contained command
    for ncu captures)."""
    import torch

    import int4_weight_only_gemv_gb300 as w4
    import synth
    from int4_weight_only_gemv_gb300 import build as wbuild
    wbuild.build()
    if args.case.startswith("seq"):
        n = int(args.case[3:])
        dev = torch.device("cuda", 0)
        layers = build_weights(dev, n)
        io = make_io(dev, 1, n)
        seq = w4.LayerSeq([{k: lw[k] for k in synth.PROJ_NAMES} for lw in layers], io, 1,
                          synth.HIDDEN, synth.KV_DIM, synth.FFN)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.launches):
            seq.run()
        e.record()
        torch.cuda.synchronize()
        if w4.w4a16_device_status(clear=True):
            raise RuntimeError("a kernel flagged a failure")
        per_layer = sum(gemv_bytes(N, K, M) for _, N, K, M in workload_gemvs()) // synth.N_LAYERS
        print(json.dumps({"case": args.case, "layers": n, "launches_per_replay": seq.num_launches,
                          "replays": args.launches, "bytes_per_replay": per_layer * n,
                          "us_per_replay": 1e3 * s.elapsed_time(e) / args.launches}))
        seq.close()
        return
    if args.case == "attn":
        # one decode-attention call (Qwen-7B heads, T = 8192), launched `launches` times
        dev = torch.device("cuda", 0)
        H, Hkv, D, T = synth.HIDDEN // 128, synth.KV_DIM // 128, 128, 8192
        gen = torch.Generator(device=dev).manual_seed(1)
        k = torch.randn((Hkv, T, D), generator=gen, device=dev).half()
        v = torch.randn((Hkv, T, D), generator=gen, device=dev).half()
        q = torch.randn((H, D), generator=gen, device=dev).half()
        o = torch.empty((H, D), dtype=torch.float16, device=dev)
        ws = w4.attn_decode_new_workspace(H, Hkv, T, dev)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.launches):
            w4.w4a16_attn_decode(q, k, v, T, o=o, workspace=ws)
        e.record()
        torch.cuda.synchronize()
        if w4.w4a16_device_status(clear=True):
            raise RuntimeError("a kernel flagged a failure")
        print(json.dumps({"case": "attn", "H": H, "Hkv": Hkv, "T": T, "launches": args.launches,
                          "us_per_call_warm_l2": 1e3 * s.elapsed_time(e) / args.launches}))
        return
    if args.case == "q4k":
        # the [gate; up] shape as GGUF Q4_K blocks (random bytes, d and dmin
        # in [1e-3, 0.051]), M = 1, launched `launches` times
        dev = torch.device("cuda", 0)
        N, K = 2 * synth.FFN, synth.HIDDEN
        nb = N * (K // 256)
        gen = torch.Generator(device=dev).manual_seed(4)
        b = torch.randint(0, 256, (nb, 144), generator=gen, dtype=torch.uint8, device=dev)
        d = (torch.rand((nb, 2), generator=gen, device=dev) * 0.05 + 1e-3).half()
        b[:, 0:4] = d.view(torch.uint8).view(nb, 4)
        x = synth.activations(1, K, 90, dev).view(-1)
        y = torch.empty((N,), dtype=torch.float16, device=dev)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.launches):
            w4.w4a16_q4k_gemv(b.view(-1), x, N, K, y=y)
        e.record()
        torch.cuda.synchronize()
        if w4.w4a16_device_status(clear=True):
            raise RuntimeError("a kernel flagged a failure")
        print(json.dumps({"case": "q4k", "N": N, "K": K, "launches": args.launches, "bytes": nb * 144 + 2 * K + 2 * N,
                          "us_per_gemv_warm_l2": 1e3 * s.elapsed_time(e) / args.launches}))
        return
    cfg = {c.name: c for c in synth.ALL_GEMVS}[args.case]
    dev = torch.device("cuda", 0)
    qw, sc = w4.w4a16_quantize(synth.weights(cfg.N, cfg.K, cfg.seed, dev))
    x = synth.activations(cfg.M, cfg.K, cfg.seed, dev)
    y = torch.empty((cfg.M, cfg.N), dtype=torch.float16, device=dev)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.launches):
        w4.w4a16_gemv(qw, sc, x, y)
    e.record()
    torch.cuda.synchronize()
    if w4.w4a16_device_status(clear=True):
        raise RuntimeError("a kernel flagged a failure")
    us = 1e3 * s.elapsed_time(e) / args.launches
    print(json.dumps({"case": cfg.name, "M": cfg.M, "N": cfg.N, "K": cfg.K, "launches": args.launches,
                      "us_per_gemv_warm_l2": us, "bytes": gemv_bytes(cfg.N, cfg.K, cfg.M)}))


def main():
    args = parse_args()
    if args.case:
        run_case(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = bench_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            dist.init_process_group("nccl")
        line = bench_ours(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
