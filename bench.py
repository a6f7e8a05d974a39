"""Benchmark of the spark2_5 decode attention block on GB300.

One step = one decode of every layer of the workload for every sequence of its
batch: RMSNorm + q_k_v_proj/g_proj, split + rope + cache write, split-K GQA
attention, gate + o_proj + residual, per layer, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line.  The default workload is the 64-sequence ragged batch
(contexts uniform in [512, 32768], one full and one sliding layer), the
largest that fits one GPU.  ``value`` is decode tokens/s of the whole job
(steps/s times the batch, summed over ranks) with every input resident in HBM;
the weights and caches of several copies of the workload are rotated so the
bytes a step reads are never in L2 from the step before (one copy when a step
alone reads more than four times the L2).  ``e2e`` is the same metric through
the public call with the step's input ``h`` copied from pinned host memory and
the output read back every step.  ``roofline`` is for the kernel with the
largest share of the step.  ``targets`` times, in the same process, the
8-sequence 131072-context workload: its full layer's attention kernel and its
whole step against the HBM roofline.  ``cpu_baseline`` (and ``--impl
reference``) time the float64 CPU oracle on a bounded sample of the workload.
Without WORLD_SIZE in the environment, ``--gpus N`` (N > 1) starts N ranks
itself, one per GPU, each an independent replica.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from decode_attention_block_gb300 import build_lib, synth  # noqa: E402

DEFAULT_WORKLOAD = "full+sliding_bf16_b64_ctx512-32768"
# the workload of --prefill (one sequence) and --decoder unless --workload is given
DEFAULT_CHUNK_WORKLOAD = "full+sliding_bf16_b1_pos700"
# the long-context workload the HBM targets are stated on, timed beside the
# default one: its full layer's attention kernel and its whole step
TARGET_WORKLOAD = "full+sliding_bf16_b8_ctx131072"
TARGET_ATTENTION_FRAC = 0.70
TARGET_STEP_FRAC = 0.60
METRIC = "decode attn-block steps/s & tokens/s; achieved HBM GB/s vs ~8 TB/s peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; the path shards by sequence, so
# ranks run independent replicas and only the timing is reduced)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def free_port() -> int:
    import socket
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        return s_.getsockname()[1]


def spawn_ranks(n: int, argv: list, script: str = None) -> int:
    """Start n ranks of `script` (this file by default) with `argv`, one
    process per GPU, rank r on device r, rendezvous on 127.0.0.1; rank 0's
    output passes through, the others' stdout is dropped.  Returns the first
    non-zero exit status, else 0."""
    port = free_port()
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, script or os.path.abspath(__file__)] + list(argv),
                                      env=env, stdout=None if r == 0 else subprocess.DEVNULL))
    rcs = [p_.wait() for p_ in procs]
    return next((rc for rc in rcs if rc != 0), 0)


def job_tokens_per_s(batch: int, world: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput: every rank decodes `steps` steps of its own
    `batch` sequences (weak scaling), timed by the slowest rank."""
    return batch * world * steps / (ms_max * 1e-3)


# ---------------------------------------------------------------------------
# bytes and peaks
# ---------------------------------------------------------------------------

def step_bytes(wl: synth.Workload) -> dict:
    """Algorithmic HBM bytes of one step: every weight byte once, every KV row
    a token attends to once (K and V).  h and out are not counted."""
    w = wl.weight_bytes_per_layer()
    q_dim, kv_dim, H, es = wl.n_q * wl.head_dim, wl.n_kv * wl.head_dim, wl.hidden, wl.elem_bytes
    per = {"qkv_gate": 0, "attention": 0, "gate_oproj": 0, "attention_full": 0, "attention_sliding": 0}
    for li, spec in enumerate(wl.layers):
        per["qkv_gate"] += ((q_dim + 2 * kv_dim + wl.n_q) * H + H) * es
        per["gate_oproj"] += H * q_dim * es
        kv = sum(wl.rows_read(li, b) for b in range(wl.batch)) * wl.kv_row_bytes()
        per["attention"] += kv
        per["attention_full" if spec.is_full else "attention_sliding"] += kv
    total = len(wl.layers) * w + per["attention"]
    assert total == per["qkv_gate"] + per["gate_oproj"] + per["attention"]
    return {"total": total, "per_kernel": per}


# DRAM bytes (read + write) per launch of the current kernels, from ncu
# captures (dram__bytes_read.sum + dram__bytes_write.sum, the mean over the
# captured launches) of these workloads;
# the profile summaries give each capture's command.  Attention traffic
# follows the rows read, so other workloads scale the captured ratio.
TRAFFIC = {
    ("full+sliding_bf16_b1_pos700", "qkv_rope"): 31_586_240,
    ("full+sliding_bf16_b1_pos700", "gate_oproj"): 21_047_232,
    ("full+sliding_bf16_b1_pos700", "decode_stack"): 113_560_576,
    ("full_bf16_b1_ctx131072", "attention_full"): 541_030_912,
    ("full_bf16_b16_ctx512-32768", "attention_full"): 1_119_880_448,
}
# DRAM bytes per algorithmic byte of the attention kernel in two captures:
# one sequence of 131072 rows (537 MB read), and the first 16 sequences of
# the ragged 64-sequence batch (1.11 GB over contexts of 6568 to 28494 rows)
ATTN_TRAFFIC_RATIO = 541_030_912 / 536_875_008
ATTN_RAGGED_TRAFFIC_RATIO = 1_119_880_448 / 1_111_035_904
# workloads whose attention scales the ragged capture (the same sequences' rows)
RAGGED_ATTENTION = ("full+sliding_bf16_b64_ctx512-32768",)


def measured_traffic(workload: str, kernel: str, bytes_per_launch: float):
    """(traffic per launch, how it was obtained) or (None, reason)."""
    if (workload, kernel) in TRAFFIC:
        return TRAFFIC[(workload, kernel)], "ncu capture of this workload"
    if kernel == "attention_full" and workload in RAGGED_ATTENTION:
        return (int(bytes_per_launch * ATTN_RAGGED_TRAFFIC_RATIO),
                "ncu capture of its first 16 sequences (full_bf16_b16_ctx512-32768), scaled by rows read")
    if kernel.startswith("attention"):
        return int(bytes_per_launch * ATTN_TRAFFIC_RATIO), "ncu capture at 131072 rows, scaled by rows read"
    return None, "no capture of this kernel on this workload"


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx = float(parts[1])
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Copy:
    """One full set of a workload's inputs resident on the device."""

    def __init__(self, wl, B, device):
        self.layers = []
        for li, spec in enumerate(wl.layers):
            w = synth.make_weights(wl, li, device)
            k, v = synth.make_cache(wl, li, device)
            self.layers.append((spec, B.LayerWeights(**w), B.KvLayer(k, v, spec.ring_capacity)))
        self.h = synth.make_h(wl, device)
        self.buf = [torch.empty_like(self.h), torch.empty_like(self.h)]


def run_step(B, geom, wl, cp, ws, stream=None, path="stack"):
    """One decode step of every layer through the public calls: one
    spark_attn_decode_stack call for the whole stack, or spark_attn_decode
    layer by layer."""
    if path == "stack":
        B.spark_attn_decode_stack(geom, cp.h, [w for _, w, _ in cp.layers], [kv for _, _, kv in cp.layers],
                                  [B.SPARK_FULL if s.is_full else B.SPARK_SLIDING for s, _, _ in cp.layers],
                                  wl.positions, cp.buf[0], ws, stream)
        return cp.buf[0]
    cur = cp.h
    for i, (spec, w, kv) in enumerate(cp.layers):
        out = cp.buf[i % 2]
        B.spark_attn_decode(geom, cur, w, kv, B.SPARK_FULL if spec.is_full else B.SPARK_SLIDING,
                            wl.positions, out, ws, stream)
        cur = out
    return cur


def projection_launches(wl) -> int:
    """Kernels one projection (q_k_v_proj or o_proj) of one layer launches:
    the GEMV kernel per 4 sequences up to batch 4 or with fp32 weights, else
    a prologue and a tensor-core GEMM per 128 sequences."""
    if wl.batch <= 4 or wl.dtype != "bf16":
        return -(-wl.batch // 4)
    return 2 * -(-wl.batch // 128)


def stack_is_fused(wl) -> bool:
    """Whether spark_attn_decode_stack runs this workload as one persistent
    kernel (bf16, batch <= 4, spark2_5 geometry) rather than layer by layer."""
    return wl.dtype == "bf16" and wl.batch <= 4


STAGES = ("qkv_rope", "attention_full", "attention_sliding", "gate_oproj")


def stage_layers(wl, stage) -> list:
    """Indices of the layers a stage's timing launches: every layer for the
    projections, the layers of one class for attention."""
    if stage == "attention_full":
        return [i for i, s_ in enumerate(wl.layers) if s_.is_full]
    if stage == "attention_sliding":
        return [i for i, s_ in enumerate(wl.layers) if not s_.is_full]
    return list(range(len(wl.layers)))


def stage_launcher(B, geom, wl, cp, ws, bufs, stage):
    """Launch one stage kernel for the stage's layers of a copy (the same work
    that stage does inside run_step)."""
    layers = stage_layers(wl, stage)

    def go():
        for i in layers:
            spec, w, kv = cp.layers[i]
            cur, out = (cp.h if i == 0 else cp.buf[(i - 1) % 2]), cp.buf[i % 2]
            cls = B.SPARK_FULL if spec.is_full else B.SPARK_SLIDING
            if stage == "qkv_rope":
                B.spark_dbg_qkv_rope(geom, cur, w, kv, cls, wl.positions, bufs["q_rot"], bufs["g"], ws)
            elif stage.startswith("attention"):
                B.spark_dbg_attention(geom, bufs["q_rot"], kv, cls, wl.positions, bufs["a"], ws, 0)
            else:
                B.spark_dbg_gate_oproj(geom, bufs["a"], bufs["g"], cur, w, out, ws)
    return go


def capture(fn):
    """Record fn's launches (made on the current stream) in a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                      # first call outside capture (function attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        fn()
    torch.cuda.synchronize()
    return g


def measure_decode(args, wl, B, geom, device, world, steps, with_e2e=True):
    """Time `steps` decode steps of a workload (graph replay, inputs resident,
    rotating copies against L2), each stage's launches on their own, and,
    with `with_e2e`, the public call end to end from pinned host memory."""
    stream = torch.cuda.current_stream(device)
    sb = step_bytes(wl)
    L = len(wl.layers)
    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 129 * 2 ** 20) or 129 * 2 ** 20
    copies = args.copies or max(1, math.ceil(4 * l2 / sb["total"]))
    cps = [Copy(wl, B, device) for _ in range(copies)]
    ws = B.make_workspace(geom, wl.batch, device)
    H, q_dim = wl.hidden, wl.n_q * wl.head_dim
    bufs = {"q_rot": torch.zeros((wl.batch, q_dim), device=device),
            "g": torch.zeros((wl.batch, wl.n_q), device=device),
            "a": torch.zeros((wl.batch, q_dim), device=device)}
    torch.cuda.synchronize()

    # one CUDA graph per copy: a step's launches replayed without host overhead
    use_graph = not args.no_graph
    path = args.path
    fused = path == "stack" and stack_is_fused(wl)
    if use_graph:
        graphs = [capture(lambda cp=cp: run_step(B, geom, wl, cp, ws, None, path)) for cp in cps]
        step = lambda i: graphs[i % copies].replay()  # noqa: E731
    else:
        step = lambda i: run_step(B, geom, wl, cps[i % copies], ws, stream, path)  # noqa: E731

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    if steps <= 0:   # auto: about two seconds of timed work
        t0 = time.perf_counter()
        for i in range(20):
            step(i)
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 20
        steps = int(min(50000, max(50, 2.0 / max(per, 1e-6))))

    # timed region: exactly `steps` steps
    sampler = ClockSampler(device.index or 0)
    with sampler:
        time.sleep(0.3)
        barrier(world)
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(steps):
            step(i)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    clocks = sampler.summary()
    ms_total = max_over_ranks(start.elapsed_time(end), world, device)
    ms_per_step = ms_total / steps
    kernels_per_step = -(-L // 40) if fused else L * (2 * projection_launches(wl) + 1)

    # per-stage durations: each stage's launches (its layers, all copies)
    # replayed back to back in a graph between two events on this stream
    kavg, per_launch, launches = {}, {}, {}
    bytes_key = {"qkv_rope": "qkv_gate", "gate_oproj": "gate_oproj"}
    for stage in STAGES:
        n = len(stage_layers(wl, stage))
        if n == 0:
            continue
        fns = [stage_launcher(B, geom, wl, cp, ws, bufs, stage) for cp in cps]
        g = capture(lambda: [f() for f in fns])
        reps = max(3, min(200, int(2000 / (n * copies))))
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        kavg[stage] = e0.elapsed_time(e1) / (reps * n * copies)   # ms per launch
        per_launch[stage] = sb["per_kernel"][bytes_key.get(stage, stage)] / n
        launches[stage] = n
    if fused:
        # one persistent kernel per step (per 40 layers): its duration is the step
        kavg = {"decode_stack": ms_per_step / kernels_per_step, **{"layer_" + k: v for k, v in kavg.items()}}
        per_launch = {"decode_stack": sb["total"] / kernels_per_step,
                      **{"layer_" + k: v for k, v in per_launch.items()}}
        launches = {"decode_stack": kernels_per_step, **{"layer_" + k: 0 for k in launches}}
    share = {k: kavg[k] * launches[k] for k in kavg}
    tot = sum(share.values())
    top = max(share, key=share.get)
    kernels = {k: {"avg_us": round(kavg[k] * 1e3, 3), "launches_per_step": launches[k],
                   "share": round(share[k] / tot, 4) if tot else None,
                   "bytes_per_launch": int(per_launch[k]),
                   "gbs": round(per_launch[k] / (kavg[k] * 1e-3) / 1e9, 1)} for k in kavg}

    e2e = None
    if with_e2e:
        # end to end through the public call: h from pinned host, out read back
        h_host = [synth.make_h(wl, "cpu").pin_memory() for _ in range(2)]
        out_host = torch.empty((wl.batch, H), dtype=torch.float32).pin_memory()
        e2e_steps = max(10, min(steps, 2000))
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            cp = cps[i % copies]
            cp.h.copy_(h_host[i % 2], non_blocking=True)
            res = run_step(B, geom, wl, cp, ws, stream, path)
            out_host.copy_(res, non_blocking=True)
            stream.synchronize()
        e2e_s = max_over_ranks(time.perf_counter() - t0, world, device)
        e2e = {"value": round(wl.batch * world * e2e_steps / e2e_s, 3), "unit": "tokens/s",
               "h2d_bytes_per_step": wl.batch * H * 4, "d2h_bytes_per_step": wl.batch * H * 4,
               "launch": "direct calls, synchronised every step"}
    err = B.spark_attn_error_word(ws)
    if err != 0:
        raise RuntimeError(f"device error word {err:#x}")
    return {"steps": steps, "ms_per_step": ms_per_step, "ms_total": ms_total, "clocks": clocks,
            "kavg": kavg, "per_launch": per_launch, "kernels": kernels, "top": top, "copies": copies,
            "l2": l2, "fused": fused, "kernels_per_step": kernels_per_step, "use_graph": use_graph,
            "bytes": sb["total"], "e2e": e2e}


def roofline_of(wl_name: str, m: dict, peaks: dict, kernel: str = None) -> dict:
    """The roofline object of one kernel of a measurement: algorithmic bytes
    per launch over its average launch time, against the measured copy
    bandwidth, with the DRAM traffic of a capture where one exists."""
    k = kernel or m["top"]
    achieved = m["per_launch"][k] / (m["kavg"][k] * 1e-3) / 1e9
    traffic, traffic_src = measured_traffic(wl_name, k, m["per_launch"][k])
    return {"kernel": k, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "peak_source": peaks["source"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic, "traffic_source": traffic_src, "bytes_per_launch": int(m["per_launch"][k]),
            "avg_launch_us": round(m["kavg"][k] * 1e3, 3)}


def measure_targets(args, B, geom, device, world, peaks) -> dict:
    """The long-context workload's full-layer attention kernel and whole step
    against the HBM roofline, timed in this process."""
    wl = synth.workloads()[TARGET_WORKLOAD]
    m = measure_decode(args, wl, B, geom, device, world, max(args.steps, 20) if args.steps > 0 else 0,
                       with_e2e=False)
    att = roofline_of(wl.name, m, peaks, "attention_full")
    gbs = m["bytes"] / (m["ms_per_step"] * 1e-3) / 1e9
    step_frac = gbs / peaks["hbm_gbs"]
    return {"workload": wl.name, "description": wl.description, "steps": m["steps"],
            "full_layer_attention": {**att, "target_frac": TARGET_ATTENTION_FRAC,
                                     "met": att["frac"] >= TARGET_ATTENTION_FRAC},
            "whole_step": {"ms_per_step": round(m["ms_per_step"], 6), "hbm_bytes_per_step": m["bytes"],
                           "hbm_gbs": round(gbs, 1), "frac": round(step_frac, 4),
                           "target_frac": TARGET_STEP_FRAC, "met": step_frac >= TARGET_STEP_FRAC,
                           "tokens_per_s": round(wl.batch * 1e3 / m["ms_per_step"], 3)},
            "kernels": m["kernels"], "clocks": m["clocks"]}


def bench_ours(args, wl, rank, local, world):
    from decode_attention_block_gb300 import binding as B

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    build_lib.build()
    B.load()
    geom = B.spark_geom_default()
    L = len(wl.layers)
    peaks = measured_peaks()
    m = measure_decode(args, wl, B, geom, device, world, args.steps)
    steps, ms_per_step, copies = m["steps"], m["ms_per_step"], m["copies"]
    value = job_tokens_per_s(wl.batch, world, steps, m["ms_total"])
    gbs = m["bytes"] / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) activations and caches, N(0,1/fan_in) weights; no checkpoint)",
        "config": {"workload": wl.name, "description": wl.description, "batch": wl.batch,
                   "positions": wl.positions if wl.batch <= 8 else
                   {"min": min(wl.positions), "max": max(wl.positions), "sum": sum(wl.positions)},
                   "n_layers": L,
                   "layers": ["full" if s.is_full else "sliding" for s in wl.layers][:8]
                   + (["..."] if L > 8 else []),
                   "parallelism": f"replicas x{world} (independent sequences, no collective)",
                   "launch": "CUDA graph per step" if m["use_graph"] else "direct calls",
                   "path": ("one persistent kernel per step (spark_attn_decode_stack)" if m["fused"]
                            else "three kernels per layer" if projection_launches(wl) == 1 else
                            "five kernels per layer (tensor-core projections)"),
                   "l2": f"{copies} rotating copies of weights+caches ({copies * m['bytes'] / 1e6:.0f} MB) "
                         f"vs {m['l2'] / 1e6:.0f} MB L2"},
        "steps_per_s": round(1e3 / ms_per_step * world, 3),
        "hbm_bytes_per_step": m["bytes"],
        "hbm_gbs": round(gbs, 1),
        "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
        "roofline": roofline_of(wl.name, m, peaks),
        "kernels": m["kernels"],
        "e2e": m["e2e"],
        "gpu_launches": m["kernels_per_step"] * steps,
        "clocks": m["clocks"],
    }
    if not args.no_targets and wl.name != TARGET_WORKLOAD:
        torch.cuda.empty_cache()
        line["targets"] = measure_targets(args, B, geom, device, world, peaks)
    elif wl.name == TARGET_WORKLOAD:
        att = roofline_of(wl.name, m, peaks, "attention_full")
        line["targets"] = {"workload": wl.name, "full_layer_attention": {
            **att, "target_frac": TARGET_ATTENTION_FRAC, "met": att["frac"] >= TARGET_ATTENTION_FRAC},
            "whole_step": {"frac": line["hbm_frac"], "target_frac": TARGET_STEP_FRAC,
                           "met": line["hbm_frac"] >= TARGET_STEP_FRAC}}
    return line


# ---------------------------------------------------------------------------
# the oracle (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

_ORACLE_LAYERS = {}


def oracle_layer_sample(wl: synth.Workload, li: int, seqs: list):
    """One layer's inputs for the oracle's timed sample, drawn once per
    process: the weights and the caches of the sampled sequences only (each
    [1, capacity, n_kv, d], the rows the device copy holds)."""
    key = (wl.name, li, tuple(seqs))
    if key not in _ORACLE_LAYERS:
        w = {k: synth.to_numpy(v) for k, v in synth.make_weights(wl, li, "cpu").items()}
        caches = {}
        for b in seqs:
            k, v = synth.make_sequence_cache(wl, li, b, "cpu")
            caches[b] = (synth.to_numpy(k), synth.to_numpy(v))
        _ORACLE_LAYERS[key] = (w, caches)
    return _ORACLE_LAYERS[key]


def oracle_sequences(wl: synth.Workload, n: int = 4) -> list:
    """The sequences the oracle's sample takes: up to n, evenly spread over the
    batch (a ragged batch's short and long histories alike)."""
    k = max(1, min(wl.batch, n))
    return sorted({(i * wl.batch) // k for i in range(k)})


def time_oracle(wl: synth.Workload, budget_s: float) -> dict:
    """Time the float64 CPU oracle on (layer, sequence) units of one step
    until `budget_s` is spent (passes over the sampled units, layer by layer;
    at least one unit), and report the rate scaled to a whole step: units
    timed / units of a step / seconds.  The sampled inputs (up to 4 sequences
    per layer) are drawn once and reused by later calls."""
    import oracle

    geom = oracle.OracleGeometry(hidden=wl.hidden, n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim,
                                 window=wl.window)
    h = synth.to_numpy(synth.make_h(wl, "cpu")).astype(np.float64)
    units_total = len(wl.layers) * wl.batch
    units = 0
    elapsed = 0.0
    seqs = oracle_sequences(wl)
    done = False
    while not done:
        for li, spec in enumerate(wl.layers):
            w, caches = oracle_layer_sample(wl, li, seqs)
            for b in seqs:
                kn, vn = caches[b]
                t0 = time.perf_counter()
                oracle.decode_step(geom, h[b:b + 1], w, kn, vn, spec.is_full, [wl.positions[b]],
                                   spec.ring_capacity)
                elapsed += time.perf_counter() - t0
                units += 1
                if elapsed >= budget_s:
                    done = True
                    break
            if done:
                break
    steps_per_s = (units / units_total) / elapsed
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(steps_per_s * wl.batch, 6), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{units} timed (layer, sequence) decode units, in passes over the "
                      f"{len(wl.layers) * len(seqs)} of sequences {seqs} (a step has {units_total}); "
                      f"{elapsed:.1f} s, numpy float64, BLAS threads up to {cores} cores"}


def time_oracle_prefill(wl: synth.Workload, m: int, budget_s: float) -> dict:
    """The float64 oracle on the first tokens of a chunk (prefill_chunk on a
    prefix of the chunk, each layer on its own inputs), until `budget_s` is
    spent; the rate is tokens/s through every layer."""
    import oracle

    geom = oracle.OracleGeometry(hidden=wl.hidden, n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim,
                                 window=wl.window)
    p0 = int(wl.positions[0])
    t_tok = 0.0
    n_tok = 0
    for mm in (1, 2, 4, 8, 16):
        per_layer = []
        for li, spec in enumerate(wl.layers):
            w = {k: synth.to_numpy(v) for k, v in synth.make_weights(wl, li, "cpu").items()}
            cap = spec.ring_capacity if spec.ring_capacity > 0 else p0 + mm
            g = torch.Generator().manual_seed(wl.seed * 31 + li)
            dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
            k = synth.to_numpy(torch.randn((cap, wl.n_kv, wl.head_dim), generator=g).to(dt))
            v = synth.to_numpy(torch.randn((cap, wl.n_kv, wl.head_dim), generator=g).to(dt))
            h = np.random.default_rng(li).standard_normal((mm, wl.hidden))
            t0 = time.perf_counter()
            oracle.prefill_chunk(geom, h, w, k, v, spec.is_full, p0, spec.ring_capacity)
            per_layer.append(time.perf_counter() - t0)
        t_tok, n_tok = t_tok + sum(per_layer), n_tok + mm
        if t_tok >= budget_s or mm >= m:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(n_tok / t_tok, 6), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_tok} tokens in chunks of 1..{mm} from position {p0} through every layer "
                      f"({t_tok:.1f} s, numpy float64, BLAS threads up to {cores} cores)"}


def time_oracle_decoder(wl: synth.Workload, inter: int, vocab: int) -> dict:
    """The float64 oracle on one sequence of one decoder step: the attention
    block and MLP half of the first layers (at most 4, the time scaled to
    every layer), then the head."""
    import oracle

    geom = oracle.OracleGeometry(hidden=wl.hidden, n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim,
                                 window=wl.window)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    h = synth.to_numpy(synth.make_h(wl, "cpu")).astype(np.float64)[:1]
    pos = [wl.positions[0]]
    elapsed = 0.0
    n_l = min(len(wl.layers), 4)
    for li, spec in enumerate(wl.layers[:n_l]):
        w = {k: synth.to_numpy(v) for k, v in synth.make_weights(wl, li, "cpu").items()}
        k, v = synth.make_sequence_cache(wl, li, 0, "cpu")
        mw = {k_: synth.to_numpy(v_) for k_, v_ in
              synth.make_mlp_weights(wl.seed * 100 + li, wl.hidden, inter, dt, "cpu").items()}
        t0 = time.perf_counter()
        r = oracle.decode_step(geom, h, w, synth.to_numpy(k), synth.to_numpy(v), spec.is_full, pos,
                               spec.ring_capacity)
        h = oracle.mlp_block(geom, r["out"], mw)["out"]
        elapsed += time.perf_counter() - t0
    elapsed *= len(wl.layers) / n_l
    hd = {k_: synth.to_numpy(v_) for k_, v_ in synth.make_head(wl.seed, wl.hidden, vocab, dt, "cpu").items()}
    t0 = time.perf_counter()
    oracle.head_logits(geom, h, hd["norm_w"], hd["embed"])
    elapsed += time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(1.0 / elapsed, 6), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"one sequence through {n_l} of {len(wl.layers)} layers (attention block + MLP half, "
                      f"time scaled to every layer) and the head "
                      f"({elapsed:.1f} s, numpy float64, BLAS threads up to {cores} cores)"}


def bench_reference(args, wl, rank, world):
    """The reference arm: the float64 CPU oracle as it stands, on the host
    cores, each step a bounded sample of the workload; rank 0 only."""
    if rank != 0:
        return None
    k_steps = args.steps if args.steps > 0 else 3
    per_step = max(1.0, min(15.0, 120.0 / (k_steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(wl, 0.0)               # one (layer, sequence) unit each
    runs = [time_oracle(wl, per_step) for _ in range(k_steps)]
    value = float(np.median([r["value"] for r in runs]))
    base = dict(runs[-1])
    base["value"] = round(value, 6)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "tokens/s",
            "n_gpus": world, "steps": k_steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "description": wl.description, "batch": wl.batch},
            "cpu_baseline": base,
            "e2e": {"value": round(value, 6), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def bench_prefill(args, wl):
    """`--prefill M`: chunks of M consecutive tokens of the workload's one
    sequence, starting at its decode position, through every layer of the
    workload (spark_attn_prefill per layer, each layer's output feeding the
    next).  Reports tokens/s, the HBM bytes a chunk must move (each layer's
    weights and its distinct KV rows read or written, once) and the FLOPs
    of its projections and attention."""
    from decode_attention_block_gb300 import binding as B

    if wl.batch != 1:
        raise SystemExit("--prefill takes a one-sequence workload")
    M, p0 = int(args.prefill), int(wl.positions[0])
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    build_lib.build()
    B.load()
    geom = B.spark_geom_default()
    layers, kv_bytes, att_flops = [], 0, 0
    for li, spec in enumerate(wl.layers):
        w = B.LayerWeights(**synth.make_weights(wl, li, device))
        cap = spec.ring_capacity if spec.ring_capacity > 0 else p0 + M
        gen = torch.Generator(device=device)
        gen.manual_seed(wl.seed * 31 + li)
        dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        k = torch.randn((1, cap, wl.n_kv, wl.head_dim), generator=gen, device=device).to(dt)
        v = torch.randn((1, cap, wl.n_kv, wl.head_dim), generator=gen, device=device).to(dt)
        layers.append((spec, w, B.KvLayer(k, v, spec.ring_capacity)))
        first = 0 if spec.is_full else max(0, p0 + 1 - wl.window)
        row_bytes = 2 * wl.n_kv * wl.head_dim * (2 if wl.dtype == "bf16" else 4)
        kv_bytes += (p0 + M - first) * row_bytes + M * row_bytes   # distinct rows read + rows written
        for t in range(M):
            lo = 0 if spec.is_full else max(0, p0 + t + 1 - wl.window)
            att_flops += (p0 + t + 1 - lo) * wl.n_q * wl.head_dim * 4
    nbytes = wl.weight_bytes_per_layer() * len(wl.layers) + kv_bytes
    proj_flops = 2 * M * ((wl.n_q + 2 * wl.n_kv) * wl.head_dim * wl.hidden + wl.n_q * wl.hidden
                          + wl.hidden * wl.n_q * wl.head_dim) * len(wl.layers)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed * 7 + 5)
    h = torch.randn((M, wl.hidden), generator=gen, device=device)
    bufs = [torch.empty_like(h), torch.empty_like(h)]
    ws = B.make_workspace(geom, M, device)
    stream = torch.cuda.current_stream(device)

    def chunk():
        cur = h
        for i, (spec, w, kv) in enumerate(layers):
            out = bufs[i % 2]
            B.spark_attn_prefill(geom, cur, w, kv, B.SPARK_FULL if spec.is_full else B.SPARK_SLIDING, p0,
                                 out, ws, stream)
            cur = out

    for _ in range(args.warmup):
        chunk()
    torch.cuda.synchronize()
    steps = args.steps or 50
    sampler = ClockSampler(0)
    with sampler:
        time.sleep(0.3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            chunk()
        e1.record(stream)
        torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    ms = e0.elapsed_time(e1) / steps
    peaks = measured_peaks()
    return {"metric": f"prefill tokens/s (chunks of {M} consecutive tokens of one sequence)",
            "value": round(M / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": f"{wl.name}, prefill chunk of {M} from position {p0}", "chunk": M,
                       "p0": p0, "layers": ["full" if s_.is_full else "sliding" for s_ in wl.layers]},
            "hbm_bytes_per_step": nbytes, "hbm_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "flops_per_step": proj_flops + att_flops,
            "tflops": round((proj_flops + att_flops) / (ms * 1e-3) / 1e12, 2),
            # the chunk's algorithmic FLOPs (projections and attention, without
            # the hi/lo operand split) against the dense bf16 tensor peak
            "roofline": {"kernel": "whole chunk (projection GEMMs + grouped attention)", "bound": "tensor",
                         "achieved": round((proj_flops + att_flops) / (ms * 1e-3) / 1e12, 2),
                         "peak": peaks["bf16_tflops"], "peak_source": peaks["source"], "unit": "TFLOP/s",
                         "frac": round((proj_flops + att_flops) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                         "traffic": None},
            "cpu_baseline": None if args.no_cpu_baseline else time_oracle_prefill(wl, M, 10.0),
            "clocks": sampler.summary()}


def bench_decoder(args, wl):
    """`--decoder`: whole decode steps of a model with the workload's layers --
    per layer the attention block (spark_attn_decode) and the MLP half
    (spark_mlp_decode, intermediate synth.INTERMEDIATE), then the final norm and
    the tied head (spark_head_logits, vocabulary synth.VOCAB) -- replayed from
    a CUDA graph.  Reports tokens/s, the step's HBM bytes (every weight once,
    the KV rows read) and each stage's time per launch against its bytes."""
    from decode_attention_block_gb300 import binding as B

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    build_lib.build()
    B.load()
    geom = B.spark_geom_default()
    stream = torch.cuda.current_stream(device)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    eb = 2 if wl.dtype == "bf16" else 4
    I, V, H, L = synth.INTERMEDIATE, synth.VOCAB, wl.hidden, len(wl.layers)
    sb = step_bytes(wl)
    mlp_bytes = (3 * I * H + H) * eb
    head_bytes = (V * H + H) * eb
    total = sb["total"] + L * mlp_bytes + head_bytes
    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 129 * 2 ** 20) or 129 * 2 ** 20
    copies = args.copies or max(1, math.ceil(4 * l2 / total))
    cps = []
    for c in range(copies):
        cp = Copy(wl, B, device)
        cp.mlp = [B.MlpWeights(**synth.make_mlp_weights(wl.seed * 100 + li, H, I, dt, device)) for li in range(L)]
        hd = synth.make_head(wl.seed, H, V, dt, device)
        cp.head = (hd["norm_w"], hd["embed"])
        cp.logits = torch.empty((wl.batch, V), device=device)
        cps.append(cp)
    ws = B.make_workspace(geom, wl.batch, device)
    wsm = B.make_mlp_workspace(geom, I, wl.batch, device)

    # launches go to the current stream (the capturing one inside capture())
    def attn(cp, li, cur, out):
        spec, w, kv = cp.layers[li]
        B.spark_attn_decode(geom, cur, w, kv, B.SPARK_FULL if spec.is_full else B.SPARK_SLIDING, wl.positions,
                            out, ws)

    def mlp(cp, li, buf):
        B.spark_mlp_decode(geom, buf, cp.mlp[li], buf, wsm, 0)

    def head(cp, cur):
        B.spark_head_logits(geom, cur, cp.head[0], cp.head[1], cp.logits, wsm, 0)

    def step_of(cp):
        cur = cp.h
        for li in range(L):
            out = cp.buf[li % 2]
            attn(cp, li, cur, out)
            mlp(cp, li, out)
            cur = out
        head(cp, cur)
        return cp.logits

    graphs = [capture(lambda cp=cp: step_of(cp)) for cp in cps]
    for i in range(args.warmup):
        graphs[i % copies].replay()
    torch.cuda.synchronize()
    steps = args.steps or 200
    sampler = ClockSampler(0)
    with sampler:
        time.sleep(0.3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            graphs[i % copies].replay()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps

    # each stage's launches (all layers, all copies) replayed back to back
    stages = {
        "attention_block": (lambda cp: [attn(cp, li, cp.buf[li % 2], cp.buf[(li + 1) % 2]) for li in range(L)],
                            L, sb["total"] / L),
        "mlp": (lambda cp: [mlp(cp, li, cp.buf[li % 2]) for li in range(L)], L, mlp_bytes),
        "head": (lambda cp: head(cp, cp.buf[0]), 1, head_bytes),
    }
    kern = {}
    for name, (fn, n, nbytes) in stages.items():
        g = capture(lambda: [fn(cp) for cp in cps])
        reps = max(3, min(100, int(400 / (n * copies))))
        g.replay()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            g.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        us = a0.elapsed_time(a1) / (reps * n * copies) * 1e3
        kern[name] = {"avg_us": round(us, 3), "launches_per_step": n, "bytes_per_launch": int(nbytes),
                      "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}
    tot = sum(k["avg_us"] * k["launches_per_step"] for k in kern.values())
    for k in kern.values():
        k["share"] = round(k["avg_us"] * k["launches_per_step"] / tot, 4)
    top = max(kern, key=lambda k: kern[k]["share"])

    # end to end: h from pinned host memory, the logits read back
    h_host = synth.make_h(wl, "cpu").pin_memory()
    lg_host = torch.empty((wl.batch, V), dtype=torch.float32).pin_memory()
    n_e2e = max(10, min(steps, 200))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        cp = cps[i % copies]
        cp.h.copy_(h_host, non_blocking=True)
        lg_host.copy_(step_of(cp), non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    for w_ in (ws, wsm):
        if B.spark_attn_error_word(w_) != 0:
            raise RuntimeError("device error word set")
    peaks = measured_peaks()
    ach = kern[top]["gbs"]
    # tensor cores: a prologue and two GEMMs per 128 sequences; GEMV: up per 4, down per 2
    mlp_launches = (3 * -(-wl.batch // 128)) if (wl.batch > 4 and wl.dtype == "bf16") else \
        (-(-wl.batch // 4) + -(-wl.batch // 2))
    head_launches = (2 * -(-wl.batch // 128)) if (wl.batch > 4 and wl.dtype == "bf16") else -(-wl.batch // 4)
    launches = L * (2 * projection_launches(wl) + 1 + mlp_launches) + head_launches
    return {"metric": "decoder step tokens/s (per layer the attention block and the MLP half, then the "
                      "final norm and the tied head)",
            "value": round(wl.batch / (ms * 1e-3), 3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded; no checkpoint)",
            "config": {"workload": f"{wl.name} + MLP (intermediate {I}) per layer + head (vocab {V})",
                       "batch": wl.batch, "n_layers": L, "intermediate": I, "vocab": V,
                       "launch": "CUDA graph per step",
                       "l2": f"{copies} rotating copies ({copies * total / 1e6:.0f} MB) vs {l2 / 1e6:.0f} MB L2"},
            "hbm_bytes_per_step": total, "hbm_gbs": round(total / (ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(total / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "roofline": {"kernel": top, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                         "peak_source": peaks["source"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                         "traffic": None, "traffic_source": "no capture of this stage on this workload",
                         "bytes_per_launch": kern[top]["bytes_per_launch"], "avg_launch_us": kern[top]["avg_us"]},
            "kernels": kern,
            "e2e": {"value": round(wl.batch * n_e2e / e2e_s, 3), "unit": "tokens/s",
                    "h2d_bytes_per_step": wl.batch * H * 4, "d2h_bytes_per_step": wl.batch * V * 4,
                    "launch": "direct calls, synchronised every step"},
            "gpu_launches": launches * steps,
            "cpu_baseline": None if args.no_cpu_baseline else time_oracle_decoder(wl, I, V),
            "clocks": sampler.summary()}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: about two seconds' worth)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None, choices=sorted(synth.workloads()),
                    help=f"default: {DEFAULT_WORKLOAD}; with --prefill or --decoder: {DEFAULT_CHUNK_WORKLOAD}")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copies", type=int, default=0, help="rotating input copies (0: enough to beat L2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch steps directly instead of graph replay")
    ap.add_argument("--path", default="layers", choices=["stack", "layers"],
                    help="one call per layer (default, the faster path measured) or the whole step in one call")
    ap.add_argument("--decoder", action="store_true",
                    help="time whole decoder steps: attention block + MLP per layer, then the head")
    ap.add_argument("--prefill", type=int, default=0,
                    help="time chunks of this many consecutive tokens (spark_attn_prefill) instead of decode")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the long-context workload's attention and step fractions")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU, each an independent replica of the workload
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:]))
    rank, local, world = dist_env()
    if args.gpus > 1 and world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE is {world}")
    if args.workload is None:
        args.workload = DEFAULT_CHUNK_WORKLOAD if (args.prefill > 0 or args.decoder) else DEFAULT_WORKLOAD
    wl = synth.workloads()[args.workload]

    if args.impl == "reference":
        line = bench_reference(args, wl, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if args.prefill > 0:
        print(json.dumps(bench_prefill(args, wl)), flush=True)
        return
    if args.decoder:
        print(json.dumps(bench_decoder(args, wl)), flush=True)
        return

    dist_init(world, "nccl")
    line = bench_ours(args, wl, rank, local, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = time_oracle(wl, float(os.environ.get("SPARK_ORACLE_BUDGET_S", "15")))
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
