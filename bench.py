"""Benchmark of the DSA decode step on one GB300 (or N independent replicas).

Workload (default): long-context single-stream decode, L = 307200 cached
positions, 11 DSA layers run back to back, each layer with its own seeded
caches: indexer 64 heads x 128 (int8), top-k 2048, MLA attention with 64
heads over a 576-wide bf16 latent (512 value columns).  A step is one token:
the fused decode step of all 11 layers.  The metric is microseconds per layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--kv bf16|fp8]

"--kv fp8" runs the same workload over an FP8 E4M3 latent cache (one fp32
scale per row), written from the same bf16 rows.

One JSON line on stdout (rank 0).  The 11 layers hold 4.3 GB of inputs, far
above the 129 MB L2, so every layer's keys and latent rows come from HBM.
"--impl reference" times the CPU oracle (the only reference there is) on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# The CPU oracle's float64 matrix products must not spread over several BLAS
# threads behind a "cores" count: every process that runs it uses one thread
# (spawned workers inherit this environment).
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dsa_inputs as gen  # noqa: E402

METRIC = "DSA decode-step us/layer at L=300k (11 layers back to back); achieved HBM GB/s vs GB300 peak"
UNIT = "us/layer"
LAYERS = 11
L_LONG = 307200


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_ms(ms, world, device):
    """The job's time: the slowest rank's (max over ranks), seen by every rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_us_per_layer(ms_per_step, n_layers, world):
    """Whole-job time per layer: `world` independent replicas each run a step
    of n_layers in ms_per_step, so the job finishes world x n_layers layers."""
    return ms_per_step * 1000.0 / n_layers / world


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def kv_row_bytes(x):
    """Bytes of one cached latent row as stored (FP8: codes plus the row's scale)."""
    return x.D_k + 4 if x.kv_format == "e4m3" else x.D_k * 2


def make_layers(n_layers, L, device, kv="bf16"):
    """n_layers independent layers whose inputs sit in one device tensor per
    kind (layer i is slice i), so a step can move every layer's inputs with
    one copy per kind."""
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    xs = [gen.l300k(layer=layer, L=L) if L == L_LONG else gen.l64k(layer=layer, L=L)
          for layer in range(n_layers)]
    if kv == "fp8":
        xs = [gen.fp8_cache(x) for x in xs]
    x0 = xs[0]
    fp8 = x0.kv_format == "e4m3"

    def stack(name, arr_of, dtype):
        host = np.stack([np.ascontiguousarray(arr_of(x)) for x in xs])
        return torch.from_numpy(host).to(device=device, dtype=dtype)

    packed = {
        "q_idx": stack("q_idx", lambda x: x.q_idx, torch.int8),
        "w_idx": stack("w_idx", lambda x: x.w_idx, torch.int32),
        "k_idx": stack("k_idx", lambda x: x.k_idx, torch.int8),
        "q": stack("q", lambda x: np.asarray(x.q).view(np.int16), torch.int16),
        "kv": (stack("kv", lambda x: x.kv, torch.uint8) if fp8 else
               stack("kv", lambda x: np.asarray(x.kv).view(np.int16), torch.int16)),
    }
    if fp8:
        packed["kv_scale"] = stack("kv_scale", lambda x: x.kv_scale, torch.float32)
    offsets = torch.from_numpy(x0.offsets).to(device)
    row_offsets = torch.from_numpy(x0.row_offsets).to(device)
    row_len = torch.from_numpy(x0.row_len).to(device)
    layers = []
    for i, x in enumerate(xs):
        # The caller declares its int8 value range (here the data's own bound).
        qk = int(max(np.abs(x.q_idx.astype(np.int32)).max(), np.abs(x.k_idx.astype(np.int32)).max()))
        t = {k: v[i] for k, v in packed.items()}
        prob = dsa.Problem.from_tensors(k=x.k, D_v=x.D_v, softmax_scale=x.softmax_scale,
                                        L_max=int(np.max(x.row_len)), L_total=int(x.offsets[-1]),
                                        qk_abs_max=qk, offsets=offsets, row_offsets=row_offsets,
                                        row_len=row_len, kv_fp8=fp8, **t)
        layers.append((x, prob, t))
    layers[0][2]["_packed"] = packed
    ws = dsa.alloc_workspace(layers[0][1], device=device)   # same sizes for every layer
    k = x0.k
    H_q, D_v = x0.H_q, x0.D_v
    idx = torch.empty((n_layers, 1, k), dtype=torch.int32, device=device)
    nsel = torch.empty((n_layers, 1), dtype=torch.int32, device=device)
    out = torch.empty((n_layers, 1, H_q, D_v), dtype=torch.int16, device=device)
    return layers, ws, idx, nsel, out


def kernels_per_step(prob):
    import dsa_sparse_attention_03_gb300 as dsa
    return dsa.dsa_decode_step_kernels(prob)


def bench_ours(args):
    import torch
    import torch.distributed as dist
    import dsa_sparse_attention_03_gb300 as dsa

    world, rank, local = _dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")
    stream = torch.cuda.Stream(device=device)
    sp = stream.cuda_stream

    n_layers = args.layers
    layers, ws, idx, nsel, out = make_layers(n_layers, L_LONG, device, kv=args.kv)
    x0 = layers[0][0]
    kvb = kv_row_bytes(x0)

    def step():
        for i, (_, prob, _) in enumerate(layers):
            dsa.dsa_decode_step(prob, idx[i], nsel[i], out[i], ws, stream=sp)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(2):
                graph.replay()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                step()
        ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    ms = job_ms(ms, world, device)
    ms_per_step = ms / args.steps
    us_per_layer = job_us_per_layer(ms_per_step, n_layers, world)
    status = dsa.dsa_read_device_status(ws, stream=sp)
    spread = replay_spread(graph, step, stream, n_layers) if not args.no_extras else None

    # Dominant kernel: the indexer alone, back to back over the layers (a CUDA
    # graph of 3 x n_layers launches, so host enqueue time never shows), with
    # CUDA events on its stream around each replay.
    scores = torch.empty((1, L_LONG), dtype=torch.int32, device=device)

    def index_all():
        for _ in range(3):
            for _, prob, _ in layers:
                dsa.dsa_index_scores(prob, scores, ws, stream=sp)

    with torch.cuda.stream(stream):
        index_all()
    torch.cuda.synchronize()
    if args.no_graph:
        igraph = None
    else:
        igraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(igraph, stream=stream):
            index_all()
    idx_ms = []
    with torch.cuda.stream(stream):
        for rep in range(6):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if igraph is not None:
                igraph.replay()
            else:
                index_all()
            e1.record(stream)
            idx_ms.append((e0, e1))
    torch.cuda.synchronize()
    idx_avg_ms = statistics.mean(a.elapsed_time(b) for a, b in idx_ms[1:]) / (3 * n_layers)
    del igraph
    idx_bytes = L_LONG * x0.D_i + x0.H_i * x0.D_i + x0.H_i * 4
    idx_gbs = idx_bytes / (idx_avg_ms * 1e-3) / 1e9
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    step_bytes = n_layers * (L_LONG * x0.D_i + x0.k * kvb + x0.H_q * x0.D_k * 2)
    # The dominant kernel (ncu launch-list share, profiles/decode_step_l300k_launches.md)
    # is the single-row selection-and-attention kernel.  It runs inside
    # dsa_decode_step right after the indexer, so its live duration is the
    # step's per-layer time minus the indexer's back-to-back launch time, both
    # timed with CUDA events on the launching stream.  Its algorithmic bytes:
    # the gathered latent rows, the row's scores, the queries and the output.
    row_bytes = x0.k * kvb + L_LONG * 4 + x0.H_q * x0.D_k * 2 + x0.H_q * x0.D_v * 2
    row_us = us_per_layer - idx_avg_ms * 1000.0
    row_gbs = row_bytes / (row_us * 1e-6) / 1e9 if row_us > 0 else None
    fused = kernels_per_step(layers[0][1]) == 2
    row_roofline = {"kernel": "decode_row_kernel" if fused else "top-k + attention",
                    "bound": "hbm", "achieved": None if row_gbs is None else round(row_gbs, 1),
                    "peak": hbm_peak, "unit": "GB/s",
                    "frac": None if row_gbs is None else round(row_gbs / hbm_peak, 4),
                    "peak_source": peak_src,
                    "traffic": profiled_traffic("decode_row_l300k_full.md", "decode_row.cu") if fused else None,
                    "traffic_source": "profiles/decode_row_l300k_full.md (ncu, same kernel source)",
                    "algorithmic_bytes_per_launch": row_bytes,
                    "avg_launch_us": round(row_us, 3),
                    "duration_source": "step us/layer minus the indexer's back-to-back us/launch (CUDA events)",
                    "note": "latency-bound: a chain of dependent L2 round trips and a grid barrier"}
    in_bytes = n_layers * L_LONG * (x0.D_i + kvb)
    step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9

    stages = bench_stages(layers, ws, idx, nsel, out, stream) if not args.no_extras else None
    e2e = bench_e2e(args, layers, ws, idx, nsel, out, stream, device) if not args.no_extras else None

    # The L = 65536 single-layer point of the metric: 12 independent layers
    # (1.0 GB, > 4x L2) rotated, one decode step per layer.
    sec = bench_l64k(args, stream, device, kv=args.kv) if not args.no_extras else None

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None
    res = {
        "metric": METRIC + ("" if args.kv == "bf16" else "; FP8 E4M3 latent cache"),
        "value": round(us_per_layer, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8+bf16" if args.kv == "bf16" else "int8+e4m3/bf16", "data": "synthetic",
        "config": {"workload": f"l300k: 1 query, L=307200, {n_layers} layers back to back; indexer 64x128 "
                               "int8 (10% near-parallel keys), k=2048, 64 heads x 576 "
                               + ("bf16 latent" if args.kv == "bf16" else
                                  "FP8 E4M3 latent with fp32 row scales") +
                               " (D_v=512), scale 1/24",
                   "kv": args.kv,
                   "layers": n_layers, "L": L_LONG, "k": x0.k, "batch": 1,
                   "l2": f"inputs {in_bytes / 1e9:.1f} GB > L2 (129 MB); not flushed", "cuda_graph": graph is not None,
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(1e6 / (us_per_layer * n_layers * world) * world, 2),
        "step_gbs": round(step_gbs, 1),
        "roofline": row_roofline,
        "roofline_indexer": {"kernel": "indexer (" + ("tc" if dsa.indexer_kind(layers[0][1]) == "tc" else "dp4a") + ")",
                             "bound": "hbm", "achieved": round(idx_gbs, 1), "peak": hbm_peak,
                             "unit": "GB/s", "frac": round(idx_gbs / hbm_peak, 4),
                             "peak_source": peak_src, "traffic": profiled_traffic(),
                             "traffic_source": "profiles/indexer_tc_l300k_full.md (ncu, same kernel source)",
                             "algorithmic_bytes_per_launch": idx_bytes,
                             "avg_launch_us": round(idx_avg_ms * 1000, 3)},
        "replay_us_per_layer": spread,
        "stages_us_per_layer": stages,
        "secondary": sec,
        "e2e": e2e,
        "gpu_launches": args.steps * n_layers * kernels_per_step(layers[0][1]),
        "clocks": clk,
        "device_status": status,
    }
    if not args.no_cpu_baseline and not args.no_extras and world == 1:
        res["cpu_baseline"] = cpu_baseline()
    return res


def replay_spread(graph, step, stream, n_layers, n=200):
    """Per-step distribution: n steps timed one by one (CUDA events around each
    replay), in us per layer."""
    import torch
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(n):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if graph is not None:
                graph.replay()
            else:
                step()
            e1.record(stream)
            evs.append((e0, e1))
    torch.cuda.synchronize()
    v = np.array([a.elapsed_time(b) * 1000.0 / n_layers for a, b in evs])
    return {"n": n, "p10": round(float(np.percentile(v, 10)), 3), "p50": round(float(np.median(v)), 3),
            "p90": round(float(np.percentile(v, 90)), 3), "min": round(float(v.min()), 3),
            "max": round(float(v.max()), 3)}


def profiled_traffic(summary="indexer_tc_l300k_full.md", source="indexer_tc.cu"):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is still the one it was captured from (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", summary)
    src = os.path.join(ROOT, "dsa_sparse_attention_03_gb300", "csrc", source)
    try:
        lines = open(path).read().splitlines()
        want = [l.split(":", 1)[1].strip() for l in lines if l.startswith(f"source sha256 {source}:")]
        val = [l.split(":", 1)[1].strip() for l in lines if l.startswith("dram bytes per launch:")]
        have = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    if not want or not val or want[0] != have:
        return None
    return int(val[0])


def bench_stages(layers, ws, idx, nsel, out, stream):
    """Per-stage device time (CUDA events around each public call, all layers,
    no graph): where a decode step's time goes."""
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    sp = stream.cuda_stream
    x0 = layers[0][0]
    scores = torch.empty((1, x0.L_max), dtype=torch.int32, device=ws.device)
    names = ("index_scores", "topk", "sparse_attn")
    tot = {n: 0.0 for n in names}
    reps = 5
    with torch.cuda.stream(stream):
        for rep in range(reps + 1):
            evs = []
            for i, (_, prob, _) in enumerate(layers):
                e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                e[0].record(stream)
                dsa.dsa_index_scores(prob, scores, ws, stream=sp)
                e[1].record(stream)
                dsa.dsa_topk(prob, scores, idx[i], nsel[i], ws, stream=sp)
                e[2].record(stream)
                dsa.dsa_sparse_attn(prob, idx[i], nsel[i], out[i], None, ws, stream=sp)
                e[3].record(stream)
                evs.append(e)
            torch.cuda.synchronize()
            if rep == 0:
                continue
            for e in evs:
                for j, n in enumerate(names):
                    tot[n] += e[j].elapsed_time(e[j + 1]) * 1000.0
    n = reps * len(layers)
    return {k: round(v / n, 3) for k, v in tot.items()}


def bench_e2e(args, layers, ws, idx, nsel, out, stream, device):
    """The same step through the public API with host buffers: every step copies
    each layer's query inputs and the new token's cache row (indexer key and
    latent row, appended at the last position) from pinned host memory, runs
    the decode step, and reads back the output and the selected indices."""
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    sp = stream.cuda_stream
    packed = layers[0][2]["_packed"]
    xs = [x for x, _, _ in layers]
    # Pinned host inputs of every layer: the query side and the new token's
    # cache rows (indexer key and latent row, appended at the last position).
    host_in = {
        "q_idx": torch.from_numpy(np.stack([x.q_idx for x in xs])).pin_memory(),
        "w_idx": torch.from_numpy(np.stack([x.w_idx for x in xs])).pin_memory(),
        "q": torch.from_numpy(np.stack([np.asarray(x.q).view(np.int16) for x in xs])).pin_memory(),
        "k_row": torch.from_numpy(np.stack([x.k_idx[-1] for x in xs])).pin_memory(),
        "kv_row": torch.from_numpy(np.stack([np.asarray(x.kv[-1]).view(np.int16) if x.kv_format == "bf16"
                                             else np.asarray(x.kv[-1]) for x in xs])).pin_memory(),
    }
    if "kv_scale" in packed:
        host_in["kv_scale_row"] = torch.from_numpy(np.stack([x.kv_scale[-1:] for x in xs])).pin_memory()
    host_out = {"out": torch.empty(tuple(out.shape), dtype=torch.int16).pin_memory(),
                "idx": torch.empty(tuple(idx.shape), dtype=torch.int32).pin_memory()}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    def step():
        packed["q_idx"].copy_(host_in["q_idx"], non_blocking=True)
        packed["w_idx"].copy_(host_in["w_idx"], non_blocking=True)
        packed["q"].copy_(host_in["q"], non_blocking=True)
        packed["k_idx"][:, -1].copy_(host_in["k_row"], non_blocking=True)
        packed["kv"][:, -1].copy_(host_in["kv_row"], non_blocking=True)
        if "kv_scale_row" in host_in:
            packed["kv_scale"][:, -1:].copy_(host_in["kv_scale_row"], non_blocking=True)
        for i, (x, prob, t) in enumerate(layers):
            dsa.dsa_decode_step(prob, idx[i], nsel[i], out[i], ws, stream=sp)
        host_out["out"].copy_(out, non_blocking=True)
        host_out["idx"].copy_(idx, non_blocking=True)

    def timed(run, steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                run()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step()
    torch.cuda.synchronize()
    steps = max(3, args.steps // 2)
    eager_ms = timed(step, steps)
    # The same step as a user would run a decode loop: captured once in a CUDA
    # graph whose memcpy nodes copy from / to the pinned host buffers on every
    # replay.
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
    # Five consecutive runs of steps / 5 replays each, and their median: the
    # host copies share the host's memory path with other work on the box, and
    # a disturbance during one run then moves one of the five, not the value.
    if graph is not None:
        runs = [timed(graph.replay, max(1, steps // 5)) for _ in range(5)]
        ms = float(np.median(runs))
    else:
        runs, ms = [eager_ms], eager_ms
    per_layer = [round(r * 1000.0 / len(layers), 3) for r in runs]
    return {"value": round(ms * 1000.0 / len(layers), 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "cuda_graph": graph is not None,
            "runs_us_per_layer": per_layer, "eager_value": round(eager_ms * 1000.0 / len(layers), 3)}


def bench_l64k(args, stream, device, kv="bf16"):
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    n = 12
    layers, ws, idx, nsel, out = make_layers(n, 65536, device, kv=kv)
    sp = stream.cuda_stream

    def step(i):
        _, prob, _ = layers[i % n]
        dsa.dsa_decode_step(prob, idx[i % n], nsel[i % n], out[i % n], ws, stream=sp)

    def all_layers():
        for i in range(n):
            step(i)

    with torch.cuda.stream(stream):
        all_layers()
    torch.cuda.synchronize()
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            all_layers()
    run = graph.replay if graph is not None else all_layers
    reps = max(2, min(args.steps, 500))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        run()
        e0.record(stream)
        for _ in range(reps):
            run()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / (reps * n)
    x0 = layers[0][0]
    nbytes = 65536 * x0.D_i + x0.k * kv_row_bytes(x0) + x0.H_q * x0.D_k * 2
    in_gb = n * 65536 * (x0.D_i + kv_row_bytes(x0)) / 1e9
    del layers, ws
    return {"workload": f"l64k: 1 query, L=65536, 1 layer (12 rotated layer buffers, {in_gb:.1f} GB)",
            "us_per_layer": round(us, 3), "step_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "cuda_graph": graph is not None}


def _oracle_layer_worker(args):
    """One spawned worker: draw layer `layer` of the L=307200 workload, wait for
    the others, time one oracle decode step.  Returns (start, end) on the
    system-wide monotonic clock."""
    layer, barrier = args
    import oracle
    x = gen.l300k(layer=layer)
    barrier.wait()
    t0 = time.perf_counter()
    oracle.decode_step(x)
    return t0, time.perf_counter()


_BARRIER = None


def _pool_init(b):
    global _BARRIER
    _BARRIER = b


def _oracle_layer_task(layer):
    return _oracle_layer_worker((layer, _BARRIER))


def _oracle_layers_parallel(n_proc):
    """n_proc layers, one per spawned process (one BLAS thread each), all
    started together; returns the wall time from the first start to the last
    end."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    b = ctx.Barrier(n_proc)
    with ctx.Pool(n_proc, initializer=_pool_init, initargs=(b,)) as pool:
        spans = pool.map(_oracle_layer_task, range(n_proc))
    return max(e for _, e in spans) - min(s for s, _ in spans)


def cpu_baseline():
    """The CPU oracle, as it stands, on a bounded sample of the workload: full
    decode steps of single L=307200 layers, on one core and on all host cores
    (one layer per process, spawned, one BLAS thread per process)."""
    cores = os.cpu_count() or 1
    n_all = max(1, min(cores, 16))
    t1 = _oracle_layers_parallel(1)
    tn = _oracle_layers_parallel(n_all) if n_all > 1 else t1
    return {"value": round(tn * 1e6 / n_all, 1), "unit": UNIT, "cores": n_all, "kind": "oracle",
            "host_cores": cores,
            "sample": f"{n_all} of the L=307200 layers (layers 0..{n_all - 1}), one full decode step each, "
                      f"one per process on {n_all} cores at once (numpy int64 scores, stable sort, float64 "
                      f"attention, one BLAS thread per process); value = wall time / layers",
            "seconds": round(tn, 2),
            "single_core": {"value": round(t1 * 1e6, 1), "unit": UNIT, "cores": 1,
                            "sample": "layer 0, one full decode step, one process, one BLAS thread"}}


def _prefix(x, n):
    """The first n cached positions of a single-request problem (same query)."""
    import dataclasses
    return dataclasses.replace(x, k_idx=x.k_idx[:n], kv=x.kv[:n],
                               offsets=np.array([0, n], dtype=np.int32),
                               row_len=np.array([n], dtype=np.int32))


def bench_workload(args):
    """One decode step of another workload (tiny, l64k, batch32, causal64, or a
    2048-row prefill chunk), replayed from a CUDA graph; reported per step (all
    rows of the step)."""
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    world, rank, local = _dist_env()
    if rank != 0:
        return None
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    x = {"tiny": gen.tiny, "l64k": gen.l64k, "batch32": gen.batch32, "causal64": gen.causal64,
         "prefill": gen.prefill}[args.workload]()
    if args.kv == "fp8":
        x = gen.fp8_cache(x)
    qk = int(max(np.abs(x.q_idx.astype(np.int32)).max(), np.abs(x.k_idx.astype(np.int32)).max()))
    prob, t = dsa.upload_inputs(x, device=device, qk_abs_max=qk)
    ws = dsa.alloc_workspace(prob, device=device)
    idx = torch.empty((x.R, x.k), dtype=torch.int32, device=device)
    nsel = torch.empty((x.R,), dtype=torch.int32, device=device)
    out = torch.empty((x.R, x.H_q, x.D_v), dtype=torch.int16, device=device)
    stream = torch.cuda.Stream(device=device)
    sp = stream.cuda_stream

    def step():
        dsa.dsa_decode_step(prob, idx, nsel, out, ws, stream=sp)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    reps = max(10, min(args.steps, 300))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / reps
    status = dsa.dsa_read_device_status(ws, stream=sp)
    n = nsel.cpu().numpy().astype(np.int64)
    nbytes = int(x.L_total) * x.D_i + int(n.sum()) * kv_row_bytes(x) + x.R * x.H_q * x.D_k * 2
    in_bytes = int(x.L_total) * (x.D_i + kv_row_bytes(x))
    return {"metric": f"DSA decode-step us per step, {args.workload}" + ("" if args.kv == "bf16" else ", FP8 cache"),
            "value": round(us, 3),
            "unit": "us/step", "n_gpus": 1, "steps": reps, "warmup": args.warmup,
            "higher_is_better": False, "dtype": "int8+bf16" if args.kv == "bf16" else "int8+e4m3/bf16",
            "data": "synthetic",
            "config": {"workload": args.workload, "kv": args.kv, "R": x.R, "B": x.B, "L_total": int(x.L_total),
                       "k": x.k, "H_i": x.H_i, "D_i": x.D_i, "H_q": x.H_q, "D_k": x.D_k,
                       "indexer": dsa.indexer_kind(prob), "cuda_graph": True,
                       "l2": f"inputs {in_bytes / 1e6:.1f} MB ({'>' if in_bytes > 129e6 else '<'} L2, 129 MB); not flushed"},
            "step_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "gpu_launches": reps * kernels_per_step(prob), "device_status": status}


def bench_front_end(args):
    """The indexer front end (dsa_indexer_front_end) of one decode row: hidden
    width 6144, 64 indexer heads x 128, 8-bit affine weights (54 MB with their
    scales and biases); four weight sets rotated (216 MB > L2), 20 calls per
    CUDA graph.  Roofline: the weight, scale, bias and hidden-row bytes of a
    call over its time, against the measured HBM copy bandwidth."""
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    world, rank, local = _dist_env()
    if rank != 0:
        return None
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    R, d, H_i, D_i = 1, 6144, 64, 128
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    sets = []
    for sd in range(4):
        f = gen.front_end(R=R, d=d, H_i=H_i, D_i=D_i, seed=0x5EED + sd)
        sets.append(([t(f.wq[0]), t(f.wq[1].view(np.int16)), t(f.wq[2].view(np.int16))],
                     [t(f.ww[0]), t(f.ww[1].view(np.int16)), t(f.ww[2].view(np.int16))],
                     t(f.x.view(np.int16))))
    prob = dsa.Problem(R=R, B=1, H_i=H_i, D_i=D_i, H_q=1, D_k=16, D_v=16, k=1, L_max=1, L_total=1,
                       softmax_scale=1.0, qk_abs_max=10, w_abs_max=4)
    ws = torch.empty(dsa.dsa_front_end_workspace_size(prob, d), dtype=torch.uint8, device=device)
    q_idx = torch.empty((R, H_i, D_i), dtype=torch.int8, device=device)
    w_idx = torch.empty((R, H_i), dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device=device)
    sp = stream.cuda_stream
    per_graph = 20

    def calls():
        for i in range(per_graph):
            wq, ww, x = sets[i % 4]
            dsa.dsa_indexer_front_end(prob, d, x, wq, ww, q_idx, w_idx, ws, stream=sp)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            calls()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    reps = max(5, min(args.steps, 100))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / (reps * per_graph)
    status = dsa.dsa_read_device_status(ws, stream=sp)
    O = H_i * D_i + H_i
    nbytes = O * d + O * (d // 64) * 4 + R * d * 2 + R * (H_i * D_i + H_i * 4)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"metric": "indexer front end us per call (one decode row)", "value": round(us, 3),
            "unit": "us/call", "n_gpus": 1, "steps": reps, "warmup": args.warmup,
            "higher_is_better": False, "dtype": "u8 affine weights x bf16 -> fp32 -> int8/int32",
            "data": "synthetic",
            "config": {"workload": "front end: R=1, d=6144, H_i=64, D_i=128, q_max=10, w_max=4",
                       "l2": "4 weight sets (216 MB) rotated > L2; not flushed", "cuda_graph": True},
            "roofline": {"kernel": "front_end_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                         "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                         "algorithmic_bytes_per_launch": nbytes,
                         "note": "time per call includes the memset node of the call's counters"},
            "gpu_launches": reps * per_graph, "device_status": status}


def bench_ab(args):
    """Paired A/B of two variants of the headline step, run in ABBA order: each
    round times A, B, B, A (one graph replay of all layers each, CUDA events
    around each replay) and takes the ratio (B1 + B2) / (A1 + A2), so that
    clock or thermal drift within a round cancels.  Reports the per-round
    ratio's median and spread, and each arm's median us/layer."""
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    world, rank, local = _dist_env()
    if rank != 0:
        return None
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=device)
    sp = stream.cuda_stream
    n_layers = args.layers
    if args.ab == "indexer":
        names = ("tc", "dp4a")
        arms = []
        for ix in names:
            layers, ws, idx, nsel, out = make_layers(n_layers, L_LONG, device)
            for _, prob, _ in layers:
                prob.set(flags=(prob.c.flags & ~0xF) | dsa.INDEXERS[ix])
            arms.append((layers, ws, idx, nsel, out))
    else:
        names = ("bf16", "fp8")
        arms = [make_layers(n_layers, L_LONG, device, kv=kv) for kv in names]
    graphs = []
    for layers, ws, idx, nsel, out in arms:
        def step(layers=layers, ws=ws, idx=idx, nsel=nsel, out=out):
            for i, (_, prob, _) in enumerate(layers):
                dsa.dsa_decode_step(prob, idx[i], nsel[i], out[i], ws, stream=sp)
        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        graphs.append(g)
    rounds = max(20, min(args.steps, 200))
    evs = []
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()
        for _ in range(rounds):
            for arm in (0, 1, 1, 0):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graphs[arm].replay()
                e1.record(stream)
                evs.append((arm, e0, e1))
    torch.cuda.synchronize()
    t = np.array([a.elapsed_time(b) * 1000.0 / n_layers for _, a, b in evs]).reshape(rounds, 4)
    ratio = (t[:, 1] + t[:, 2]) / (t[:, 0] + t[:, 3])
    statuses = [dsa.dsa_read_device_status(arm[1], stream=sp) for arm in arms]
    return {"metric": f"paired ABBA ratio {names[1]} / {names[0]} of the L=300k decode step (us/layer)",
            "value": round(float(np.median(ratio)), 4), "unit": "ratio", "n_gpus": 1,
            "rounds": rounds, "higher_is_better": False, "data": "synthetic",
            "ratio_p10": round(float(np.percentile(ratio, 10)), 4),
            "ratio_p90": round(float(np.percentile(ratio, 90)), 4),
            "arms": {names[0]: round(float(np.median(np.r_[t[:, 0], t[:, 3]])), 3),
                     names[1]: round(float(np.median(np.r_[t[:, 1], t[:, 2]])), 3)},
            "config": {"workload": f"l300k, {n_layers} layers per replay, CUDA graph per arm", "ab": args.ab},
            "device_status": statuses}


def bench_reference(args):
    """The oracle, as it stands, on the host cores.  One timed step is a decode
    step of one L=307200 layer, or -- when --steps is large -- of its first L'
    positions (L' >= 8192, chosen so all steps take about two minutes), with
    the time scaled by L / L' (scoring and sorting are linear in L up to a log
    factor; the attention over k rows is a small constant)."""
    world, rank, local = _dist_env()
    if rank != 0:
        return None
    layers = [gen.l300k(layer=i) for i in range(min(LAYERS, 2))]
    import oracle
    t0 = time.perf_counter()
    oracle.decode_step(layers[0])                 # warm-up, also the per-layer estimate
    t_full = time.perf_counter() - t0
    L = layers[0].L_max
    frac = min(1.0, 120.0 / max(1, args.steps) / max(t_full, 1e-3))
    n_pos = L if frac >= 1.0 else max(8192, int(L * frac) // 4096 * 4096)
    samples = [x if n_pos == L else _prefix(x, n_pos) for x in layers]
    for _ in range(max(0, args.warmup - 1)):
        oracle.decode_step(samples[0])
    t0 = time.perf_counter()
    n = 0
    for s in range(args.steps):
        oracle.decode_step(samples[s % len(samples)])
        n += 1
    dt = time.perf_counter() - t0
    us = dt * 1e6 / n * (L / n_pos)
    sample = (f"{n} single-layer decode steps of the L=307200 workload" if n_pos == L else
              f"{n} decode steps over the first {n_pos} of the 307200 positions of a layer, "
              f"time scaled by {L / n_pos:.2f}")
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1000.0 / n, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "int64+f64", "data": "synthetic",
            "config": {"workload": "l300k: 1 query, L=307200 (one layer per timed step: a "
                                   "bounded sample of the 11-layer token)", "layers": LAYERS},
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--workload", default="l300k",
                    choices=["l300k", "l64k", "tiny", "batch32", "causal64", "prefill", "front_end"],
                    help="l300k: the metric's 11-layer long-context step (default); the others time one "
                         "decode step of that workload")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="latent cache format: bf16 (default) or FP8 E4M3 with fp32 row scales")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="layers per token (the headline workload runs 11)")
    ap.add_argument("--ab", choices=["indexer", "kv"],
                    help="paired ABBA comparison instead of the headline: tensor-core vs dp4a indexer, "
                         "or bf16 vs FP8 latent cache")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the headline timing (no e2e, L=64k point or CPU baseline); for profiling")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        res = bench_reference(args)
    elif args.ab:
        res = bench_ab(args)
    elif args.workload == "front_end":
        res = bench_front_end(args)
    elif args.workload != "l300k":
        res = bench_workload(args)
    else:
        res = bench_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
