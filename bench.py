"""Benchmark of the edge-packed multi-head attention forward pass on GB300.

One step = one full forward pass (projections, edge attention, merge of split
targets, out_proj) over one batch of the skewed n = 20,000 workload
(B = 16 samples, embed_dim 128, 8 heads, 400,000 live edges with Zipf-like
in-degrees up to 8,000), inputs resident in HBM. L2 is flushed between timed
steps by writing a 512 MiB buffer (untimed). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The headline steps run with the library's stage timer off; stage times and
the dominant kernel's roofline come from a separate pass of the same steps.
`per_workload` adds every other workload of the pages' shapes (tiny fp32,
gene-regulatory n=2,000, bipartite 500 -> 20,000 with averaged weights,
complete n=1,024): layer time, stages, roofline and the oracle on a bounded
sample (rank 0 only).

Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path; a barrier and a max over ranks of the step time only).
--impl reference times the fp64 CPU oracle on the host cores instead (rank 0
only), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

WORKLOAD_ID = 3  # default: the skewed n = 20,000 workload (--workload picks another)
METRIC = "edge·head·sample scores/s and layer fwd µs at n=20k; % HBM / tensor roofline"
UNIT = "scores/s"
FLUSH_BYTES = 512 << 20
E2E_STREAMS = 3  # end-to-end leg: steps in flight (own workspace, output and stream each)
PROFILE_DIR = os.path.join(ROOT, "profiles")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def algorithmic_bytes(stage: str, w: synth.Workload, B: int, nnz: int, wmode: str = "none") -> float | None:
    """Compulsory HBM bytes of one launch: every tensor the kernel must touch,
    read or written once (gathered re-reads served by L2 are not counted).
    With weights requested the edge kernel also writes every raw score
    (B, nnz, H) fp32 and the (m, l) pairs, and a weights pass turns them into
    weights."""
    E, L, S, H = w.embed_dim, w.query_features, w.key_features, w.num_heads
    bf = 2
    if stage == "edge_attn":
        scores = (B * nnz * H * 4 + B * L * H * 8) if wmode != "none" else 0
        return (B * L * E * bf          # q rows
                + B * S * 2 * E * bf    # k and v rows, each at least once
                + B * L * E * bf        # mixed, written
                + nnz * 4               # source index per CSR position
                + (L + 1) * 4           # row pointers
                + scores)
    if stage == "edge_attn_out":
        # the edge kernel with out_proj inside: q, k and v rows in, output rows
        # out (the mixed rows it passes through L2 are not compulsory)
        scores = (B * nnz * H * 4 + B * L * H * 8) if wmode != "none" else 0
        return (B * L * E * bf + B * S * 2 * E * bf + E * E * bf + E * bf + B * L * E * bf
                + nnz * 4 + (L + 1) * 4 + scores)
    if stage == "weights":
        out = B * nnz * (H if wmode == "per_head" else 1) * 4
        return B * nnz * H * 4 + B * L * H * 8 + nnz * 4 + out
    if stage == "dense_attn":
        return B * L * E * bf + B * S * 2 * E * bf + B * L * E * bf  # q, k, v^T once; mixed
    if stage == "transpose_v":
        return 2 * B * S * E * bf
    if stage == "proj_qkv":
        return B * L * E * bf + 3 * E * E * bf + B * L * 3 * E * bf
    if stage == "proj_q":
        return B * L * E * bf + E * E * bf + B * L * E * bf
    if stage == "proj_kv":
        return B * S * E * bf + 2 * E * E * bf + B * S * 2 * E * bf
    if stage == "out_proj":
        return B * L * E * bf + E * E * bf + B * L * E * bf
    return None


def stage_flops(stage: str, w: synth.Workload, B: int) -> float | None:
    E, L, S = w.embed_dim, w.query_features, w.key_features
    if stage == "proj_qkv":
        return 2.0 * B * L * E * 3 * E
    if stage == "proj_q":
        return 2.0 * B * L * E * E
    if stage == "proj_kv":
        return 2.0 * B * S * E * 2 * E
    if stage == "out_proj":
        return 2.0 * B * L * E * E
    if stage == "dense_attn":
        return 4.0 * B * L * S * E  # Q K^T and P V over every (target, source) pair and head
    return None


TENSOR_BOUND = {"dense_attn"}  # stages whose roofline is the tensor pipe, not HBM


def source_digest(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "edge_attn": ["graph_sparse_head_gb300/csrc/edge_ring.cuh", "graph_sparse_head_gb300/csrc/edge_attn_ring.cu",
                  "graph_sparse_head_gb300/csrc/edge_stream.cuh"],
    "proj_qkv": ["graph_sparse_head_gb300/csrc/gemm_tc.cu", "graph_sparse_head_gb300/csrc/tc_util.cuh"],
    "out_proj": ["graph_sparse_head_gb300/csrc/gemm_tc.cu", "graph_sparse_head_gb300/csrc/tc_util.cuh"],
    "edge_attn_out": ["graph_sparse_head_gb300/csrc/edge_ring.cuh", "graph_sparse_head_gb300/csrc/edge_out.cuh",
                      "graph_sparse_head_gb300/csrc/edge_attn_ring_out.cu", "graph_sparse_head_gb300/csrc/edge_stream.cuh"],
    "dense_attn": ["graph_sparse_head_gb300/csrc/dense_attn.cu", "graph_sparse_head_gb300/csrc/tc_util.cuh"],
}


def ncu_traffic(stage: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel and on this workload; else None."""
    p = os.path.join(PROFILE_DIR, "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(stage)
    if not e or e.get("source_digest") != source_digest(KERNEL_SOURCES[stage]):
        return None
    if e.get("workload", "").split(",")[0].strip() != workload:
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return len(self.lines)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def query_once(self):
        """One read-only sample, taken now (for a timed region too short for
        the sampling interval)."""
        try:
            r = subprocess.run(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                "-i", str(self.gpu)], capture_output=True, text=True, timeout=10)
            if r.returncode == 0 and r.stdout.strip():
                self.lines.append((time.time(), r.stdout.strip().splitlines()[0]))
                return True
        except (OSError, ValueError, subprocess.TimeoutExpired):
            pass
        return False

    def summary(self, first: int, last: int | None = None):
        """Samples [first, last): the timed region. A region that caught none
        falls back to every sample of the run so far, then to one sample taken
        now, and says which."""
        window = "timed region"
        rows = [l.split(",") for _, l in self.lines[first:last]]
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if not rows:
            window = "whole run (the timed region was shorter than the sampling interval)"
            rows = [[c.strip() for c in l.split(",")] for _, l in self.lines]
            rows = [r for r in rows if len(r) >= 9]
        if not rows and self.query_once():
            window = "one sample right after the timed region"
            rows = [[c.strip() for c in self.lines[-1][1].split(",")]]
            rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "window": "none (nvidia-smi gave no sample)"}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None,
                "window": window}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_seed(rank: int) -> int:
    """Each rank draws its own batch of tokens (weak scaling); rank 0 uses the
    workload's own token stream."""
    return rank


def make_rank_inputs(rank: int, batch: int, wid: int | None = None):
    """(query tokens, key/value tokens, params); key/value is the query for
    attention within one graph."""
    wid = WORKLOAD_ID if wid is None else wid
    w = synth.workload(wid)
    xq, xkv, params = synth.make_inputs(wid, batch)
    if shard_seed(rank):
        rng = np.random.default_rng([1000 + wid, shard_seed(rank)])
        xq = synth.make_tokens(rng, batch, w.query_features, w.embed_dim, w.dtype)
        if xkv is not None:
            xkv = synth.make_tokens(rng, batch, w.key_features, w.embed_dim, w.dtype)
    return xq, (xq if xkv is None else xkv), params


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's value (the job finishes when every rank has)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    on_cpu = dist.get_backend() == "gloo" or device is None
    t = torch.tensor([x], dtype=torch.float64, device="cpu" if on_cpu else device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_cpu_baseline(budget_s: float, src, tgt, w, xq, xkv, params):
    """The oracle as it stands, on whole samples of the workload, until about
    budget_s seconds of CPU time have passed (at least one sample)."""
    import oracle
    cores = oracle.num_threads()
    done, t_total = 0, 0.0
    while done < xq.shape[0]:
        x, kv = xq[done:done + 1], xkv[done:done + 1]
        t0 = time.perf_counter()
        oracle.forward(x, kv, kv, params, src, tgt, w.num_heads, need_weights=False)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total >= budget_s:
            break
    scores = done * len(src) * w.num_heads
    return {"value": scores / t_total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} of {xq.shape[0]} samples of the workload (full graph, all {len(src)} edges), "
                      f"fp64 C oracle, OpenMP over (sample, target), {t_total:.2f} s"}


def bench_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = synth.workload(WORKLOAD_ID)
    src, tgt = synth.make_graph(WORKLOAD_ID)
    xq, xkv, params = make_rank_inputs(0, w.batch)
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    times = []
    for i in range(args.warmup + args.steps):
        b = i % w.batch
        x, kv = xq[b:b + 1], xkv[b:b + 1]
        t0 = time.perf_counter()
        oracle.forward(x, kv, kv, params, src, tgt, w.num_heads, need_weights=False)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    per_sample = sum(times) / len(times)
    value = len(src) * w.num_heads / per_sample
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_sample * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "batch_per_step": 1, "batch": w.batch, "nnz": len(src),
                   "embed_dim": w.embed_dim, "num_heads": w.num_heads, "n": w.query_features},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step one sample (1 of {w.batch}) of the workload, full graph"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _timed(torch, stream, flush, steps, fn):
    """CUDA-event time (ms) of each of `steps` calls of fn on `stream`, with L2
    flushed (untimed) before each."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (e0, e1) in enumerate(ev):
        flush.fill_(i & 0xFF)  # evict L2 between steps (not timed)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


def _stage_pass(pmha, torch, stream, flush, steps, fn):
    """Per-stage CUDA-event times from a pass of their own (the library's stage
    timer records events around each launch, so the headline steps run
    without it)."""
    pmha.pmha_profile_enable(True)
    pmha.pmha_profile_read()
    try:
        _timed(torch, stream, flush, steps, fn)
    finally:
        pmha.pmha_profile_enable(False)
    prof = pmha.pmha_profile_read()
    stages = {k: {"launches": v[0], "total_ms": v[1], "avg_us": 1e3 * v[1] / max(v[0], 1)} for k, v in prof.items()}
    total = sum(v["total_ms"] for v in stages.values()) or 1.0
    for v in stages.values():
        v["share"] = v["total_ms"] / total
    return stages


def _roofline(stages, w, B, nnz, peaks, wmode="none"):
    """Roofline line of the dominant stage (the one with the largest total
    time), and per-stage HBM / tensor fractions in place."""
    for k, v in stages.items():
        alg = algorithmic_bytes(k, w, B, nnz, wmode)
        if alg is not None:
            v["hbm_gbs_algorithmic"] = alg / (v["avg_us"] / 1e6) / 1e9
            v["hbm_frac"] = v["hbm_gbs_algorithmic"] / peaks["hbm_gbs"]
        fl = stage_flops(k, w, B)
        if fl is not None:
            v["tflops"] = fl / (v["avg_us"] / 1e6) / 1e12
            v["tensor_frac"] = v["tflops"] / peaks["bf16_tflops"]
    dom = max(stages, key=lambda k: stages[k]["total_ms"]) if stages else None
    if dom is None:
        return None
    avg_s = stages[dom]["avg_us"] / 1e6
    alg = algorithmic_bytes(dom, w, B, nnz, wmode)
    fl = stage_flops(dom, w, B)
    # a GEMM is tensor-bound when its arithmetic intensity passes the ridge
    # point of the two measured peaks (E = 512), else memory-bound (E = 128)
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor_bound = fl is not None and (dom in TENSOR_BOUND or (alg is not None and fl / alg > ridge))
    if tensor_bound:
        # timed inside a long loop of steps: the sustained tensor peak
        achieved = fl / avg_s / 1e12
        peak = peaks["bf16_tflops_sustained"]
        return {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": ncu_traffic(dom, w.name), "algorithmic_flops_per_launch": fl,
                "algorithmic_bytes_per_launch": alg, "avg_launch_us": stages[dom]["avg_us"],
                "peak_source": f"{peaks['source']} sustained bf16 GEMM (MEASURED_PEAKS.json "
                               "bf16_tflops_sustained; fp16 runs at the bf16 rate)"}
    if alg is not None:
        achieved = alg / avg_s / 1e9
        return {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(dom, w.name),
                "algorithmic_bytes_per_launch": alg, "avg_launch_us": stages[dom]["avg_us"],
                "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"}
    return None


class _Problem:
    """One workload resident on the device: graph, parameters, tokens, output,
    weights and workspace buffers, and one forward step."""

    def __init__(self, pmha, torch, dev, wid, rank, stream):
        self.w = w = synth.workload(wid)
        self.B = B = w.batch
        self.src, self.tgt = synth.make_graph(wid)
        self.xq_np, self.xkv_np, self.prm = make_rank_inputs(rank, B, wid)
        self.self_attn = self.xkv_np is self.xq_np
        self.tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.params = pmha.Params.from_arrays(self.prm, w.num_heads, self.tdt, dev)
        self.graph = pmha.pmha_build_csr(torch.from_numpy(self.src).to(dev), torch.from_numpy(self.tgt).to(dev),
                                         w.query_features, w.key_features)
        self.nnz, self.H = self.graph.nnz, w.num_heads
        self.x = torch.from_numpy(self.xq_np).to(self.tdt).to(dev)
        self.kv = self.x if self.self_attn else torch.from_numpy(self.xkv_np).to(self.tdt).to(dev)
        self.out = torch.empty_like(self.x)
        # the workload's own need_weights (the bipartite map asks for averaged weights)
        self.wmode = w.weights[0] if w.weights else "none"
        shape = (B, self.nnz) if self.wmode == "avg" else (B, self.nnz, self.H)
        self.weights = None if self.wmode == "none" else torch.empty(shape, dtype=torch.float32, device=dev)
        self.ws = torch.empty(pmha.pmha_forward_workspace_size(self.graph, self.params, B, self.wmode),
                              dtype=torch.uint8, device=dev)
        self.pmha, self.stream = pmha, stream

    def step(self, key_padding_mask=None):
        self.pmha.pmha_forward(self.graph, self.params, self.x, self.kv, self.kv, self.wmode, out=self.out,
                               weights=self.weights, workspace=self.ws, stream=self.stream,
                               key_padding_mask=key_padding_mask)

    @property
    def scores(self):
        return float(self.B) * self.nnz * self.H


def measure_workload(pmha, torch, dev, wid, steps, warmup, flush, stream, peaks, cpu_seconds, rank=0):
    """Layer forward time, stage times, the dominant kernel's roofline and the
    oracle on a bounded sample, for one workload (not the headline)."""
    pr = _Problem(pmha, torch, dev, wid, rank, stream)
    for _ in range(warmup):
        pr.step()
    pmha.pmha_device_status()
    ms = statistics.mean(_timed(torch, stream, flush, steps, pr.step))
    stages = _stage_pass(pmha, torch, stream, flush, steps, pr.step)
    pmha.pmha_device_status()
    w = pr.w
    roof = None if wid == 1 else _roofline(stages, w, pr.B, pr.nnz, peaks, pr.wmode)
    cpu = None
    if cpu_seconds > 0:
        cpu = run_cpu_baseline(cpu_seconds, pr.src, pr.tgt, w, pr.xq_np, pr.xkv_np, pr.prm)
    res = {"workload": w.name, "batch": pr.B, "nnz": pr.nnz, "embed_dim": w.embed_dim, "num_heads": w.num_heads,
           "dtype": w.dtype, "need_weights": pr.wmode, "steps": steps, "ms_per_step": ms, "layer_fwd_us": ms * 1e3,
           "value": pr.scores / (ms / 1e3), "unit": UNIT, "stages": stages,
           "roofline": roof if roof is not None else ("none: a latency-bound correctness case (64 nodes)"
                                                       if wid == 1 else None),
           "cpu_baseline": cpu}
    pr.graph.destroy()
    return res


def bench_ours(args):
    import torch

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU: the library has no CPU path")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import graph_sparse_head_gb300 as pmha
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peaks = load_peaks()
    pr = _Problem(pmha, torch, dev, WORKLOAD_ID, rank, stream)
    w, B, nnz, H = pr.w, pr.B, pr.nnz, pr.H
    graph, params, x, kv, out, ws = pr.graph, pr.params, pr.x, pr.kv, pr.out, pr.ws
    xq_np, xkv_np, prm, src, tgt, self_attn = pr.xq_np, pr.xkv_np, pr.prm, pr.src, pr.tgt, pr.self_attn
    step = pr.step

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    pmha.pmha_device_status()

    # ---- the headline: K steps, the library's stage timer off
    sampler = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    first = sampler.mark()
    launches0 = pmha.pmha_launch_count()
    wall0 = time.perf_counter()
    step_ms = _timed(torch, stream, flush, args.steps, step)
    wall = time.perf_counter() - wall0
    launches = pmha.pmha_launch_count() - launches0
    last = sampler.mark()
    if world > 1:
        torch.distributed.barrier()
    pmha.pmha_device_status()
    ms = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms, world, dev)
    scores = pr.scores
    value = world * scores / (ms / 1e3)

    # ---- stage times of the same steps, from a pass of their own
    stage_steps = max(3, min(args.steps, 50))
    stages = _stage_pass(pmha, torch, stream, flush, stage_steps, step)
    pmha.pmha_device_status()
    roof = _roofline(stages, w, B, nnz, peaks, pr.wmode)

    # ---- the same workload with a key_padding_mask: each sample keeps its
    # first n_b ~ U[S/2, S] keys (padding at the end), timed like the steps above
    kpm = torch.from_numpy(synth.padding_mask(np.random.default_rng(7 + rank), B, w.key_features)).to(dev)
    masked_steps = max(3, min(args.steps, 100))
    for _ in range(3):
        step(kpm)
    pmha.pmha_device_status()
    m_ms = max_over_ranks(statistics.mean(_timed(torch, stream, flush, masked_steps, lambda: step(kpm))), world, dev)
    m_stages = _stage_pass(pmha, torch, stream, flush, min(masked_steps, 20), lambda: step(kpm))
    pmha.pmha_device_status()
    masked = {"ms_per_step": m_ms, "value": world * scores / (m_ms / 1e3), "unit": UNIT,
              "steps": masked_steps, "kept_key_fraction": float(1.0 - kpm.float().mean().item()),
              "mask": "per-sample end padding, n_b ~ U[S/2, S] keys kept (value counts every edge)",
              "stages_avg_us": {k: v["avg_us"] for k, v in m_stages.items()}}

    # ---- out_proj inside the edge kernel (PMHA_FUSED_OUT_PROJ=1, not the
    # default), timed the same way
    fused = None
    if not args.no_fused_variant:
        os.environ["PMHA_FUSED_OUT_PROJ"] = "1"
        try:
            for _ in range(3):
                step()
            pmha.pmha_device_status()
            f_steps = max(3, min(args.steps, 50))
            f_ms = max_over_ranks(statistics.mean(_timed(torch, stream, flush, f_steps, step)), world, dev)
            f_stages = _stage_pass(pmha, torch, stream, flush, min(f_steps, 20), step)
            pmha.pmha_device_status()
        finally:
            os.environ.pop("PMHA_FUSED_OUT_PROJ", None)
        fused = {"ms_per_step": f_ms, "value": world * scores / (f_ms / 1e3), "unit": UNIT, "steps": f_steps,
                 "what": "out_proj as tasks of the edge kernel's queue (PMHA_FUSED_OUT_PROJ=1)",
                 "stages_avg_us": {k: v["avg_us"] for k, v in f_stages.items()},
                 "roofline": _roofline(f_stages, w, B, nnz, peaks, pr.wmode)}

    # ---- the backward pass (pmha_backward: forward recompute + gradients of
    # inputs, weights and biases) for a seeded dout, timed the same way
    back = None
    if not args.no_backward:
        g_out = torch.from_numpy(synth.make_tokens(np.random.default_rng(11 + rank), B, w.query_features,
                                                   w.embed_dim, w.dtype)).to(torch.bfloat16).to(dev)
        ws_b = torch.empty(max(1, pmha.pmha_backward_workspace_size(graph, params, B)), dtype=torch.uint8, device=dev)

        def back_step():
            pmha.pmha_backward(graph, params, x, kv, kv, g_out, workspace=ws_b, stream=stream)

        for _ in range(3):
            back_step()
        pmha.pmha_device_status()
        back_steps = max(3, min(args.steps, 30))
        b_ms = max_over_ranks(statistics.mean(_timed(torch, stream, flush, back_steps, back_step)), world, dev)
        b_calls = min(back_steps, 10)
        b_stages = _stage_pass(pmha, torch, stream, flush, b_calls, back_step)
        pmha.pmha_device_status()
        back = {"ms_per_step": b_ms, "value": world * scores / (b_ms / 1e3), "unit": UNIT,
                "steps": back_steps, "what": "pmha_backward: forward recompute, input, weight and bias gradients",
                "stages_avg_us": {k: v["avg_us"] for k, v in b_stages.items()},
                "stages_us_per_call": {k: 1e3 * v["total_ms"] / b_calls for k, v in b_stages.items()}}

    # ---- end to end through the C ABI with host buffers (pinned), per step:
    # copy the step's tokens in, run, copy the output back. Steps rotate over
    # E2E_STREAMS streams, each with its own workspace and output buffer, so
    # one step's copies overlap other steps' kernels (as a serving loop with
    # several requests in flight would); the serial figure (one stream) is
    # reported beside it.
    xh = torch.from_numpy(xq_np).to(torch.bfloat16).pin_memory()
    kvh = xh if self_attn else torch.from_numpy(xkv_np).to(torch.bfloat16).pin_memory()
    streams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(E2E_STREAMS - 1)]
    outs = [torch.empty_like(xh).pin_memory() for _ in range(E2E_STREAMS)]
    ws_need = pmha.pmha_forward_host_workspace_size(graph, params, B, "none")
    wss = [torch.empty(ws_need, dtype=torch.uint8, device=dev) for _ in range(E2E_STREAMS)]
    e2e_steps = max(4, min(args.steps, 20))

    def host_step(i):
        k = i % E2E_STREAMS
        pmha.pmha_forward_host(graph, params, xh, kvh, kvh, outs[k], "none", workspace=wss[k], stream=streams[k])

    for i in range(4):
        host_step(i)
    torch.cuda.synchronize()
    # serial: one stream
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        pmha.pmha_forward_host(graph, params, xh, kvh, kvh, outs[0], "none", workspace=wss[0], stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    # overlapped: the whole run timed from the first copy to the last result
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(streams[0])
    for st_ in streams[1:]:
        st_.wait_event(e0)
    for i in range(e2e_steps):
        host_step(i)
    for st_ in streams[1:]:
        ev = torch.cuda.Event()
        ev.record(st_)
        streams[0].wait_event(ev)
    e1.record(streams[0])
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    e2e_value = world * scores / (e2e_ms / 1e3)
    oh = outs[0]
    h2d = xh.numel() * xh.element_size() + (0 if self_attn else kvh.numel() * kvh.element_size())
    d2h = oh.numel() * oh.element_size()
    clocks = sampler.summary(first, last)
    sampler.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cpu = run_cpu_baseline(args.cpu_seconds, src, tgt, w, xq_np, xkv_np, prm)

    # ---- every other workload of the pages' shapes, on rank 0
    per_workload = None
    if rank == 0 and not args.no_per_workload:
        per_workload = {}
        for wid in sorted(synth.WORKLOADS):
            if wid == WORKLOAD_ID:
                continue
            per_workload[synth.workload(wid).name] = measure_workload(
                pmha, torch, dev, wid, max(3, min(args.steps, 20)), 3, flush, stream, peaks,
                0.0 if args.no_cpu_baseline else args.cpu_seconds_per_workload)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "layer_fwd_us": ms * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "batch": B, "n": w.query_features, "nnz": nnz,
                       "embed_dim": w.embed_dim, "num_heads": H, "max_in_degree": graph.max_in_degree,
                       "need_weights": pr.wmode,
                       "l2": "flushed between timed steps (512 MiB write, untimed)",
                       "parallelism": f"replicas x{world}, own batch per rank, no collective"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "serial_ms_per_step": e2e_serial_ms,
                    "api": f"pmha_forward_host (pinned host buffers), steps rotating over {E2E_STREAMS} streams"},
            "gpu_launches": launches,
            "roofline": roof,
            "stages": stages,
            "stage_timing": f"a separate pass of {stage_steps} steps with the stage timer on (L2 flushed "
                            "between steps); the headline steps run without it",
            "variants": {"key_padding_mask": masked, "backward": back, "fused_out_proj": fused},
            "per_workload": per_workload,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)
    graph.destroy()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    global WORKLOAD_ID
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip timing the backward pass")
    ap.add_argument("--no-fused-variant", action="store_true",
                    help="skip timing out_proj inside the edge kernel (PMHA_FUSED_OUT_PROJ=1)")
    ap.add_argument("--no-per-workload", action="store_true", help="skip the other workloads' lines")
    ap.add_argument("--cpu-seconds-per-workload", type=float, default=3.0,
                    help="budget of the oracle CPU baseline of each other workload")
    ap.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=sorted(synth.WORKLOADS),
                    help="synthetic workload id (default: the skewed n=20,000 graph the metric is quoted on)")
    args = ap.parse_args(argv)
    WORKLOAD_ID = args.workload
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return bench_reference(args)
    return bench_ours(args)


if __name__ == "__main__":
    sys.exit(main())
