"""Benchmark of the edge-packed multi-head attention forward pass on GB300.

One step = one full forward pass (projections, edge attention, merge of split
targets, out_proj) over one batch of the skewed n = 20,000 workload
(B = 16 samples, embed_dim 128, 8 heads, 400,000 live edges with Zipf-like
in-degrees up to 8,000), inputs resident in HBM. L2 is flushed between timed
steps by writing a 512 MiB buffer (untimed). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

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


def algorithmic_bytes(stage: str, w: synth.Workload, B: int, nnz: int) -> float | None:
    """Compulsory HBM bytes of one launch: every tensor the kernel must touch,
    read or written once (gathered re-reads served by L2 are not counted)."""
    E, L, S = w.embed_dim, w.query_features, w.key_features
    bf = 2
    if stage == "edge_attn":
        return (B * L * E * bf          # q rows
                + B * S * 2 * E * bf    # k and v rows, each at least once
                + B * L * E * bf        # mixed, written
                + nnz * 4               # source index per CSR position
                + (L + 1) * 4)          # row pointers
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

    def summary(self, first: int):
        rows = [l.split(",") for _, l in self.lines[first:]]
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_seed(rank: int) -> int:
    """Each rank draws its own batch of tokens (weak scaling); rank 0 uses the
    workload's own token stream."""
    return rank


def make_rank_inputs(rank: int, batch: int):
    """(query tokens, key/value tokens, params); key/value is the query for
    attention within one graph."""
    w = synth.workload(WORKLOAD_ID)
    xq, xkv, params = synth.make_inputs(WORKLOAD_ID, batch)
    if shard_seed(rank):
        rng = np.random.default_rng([1000 + WORKLOAD_ID, shard_seed(rank)])
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
    w = synth.workload(WORKLOAD_ID)
    B = w.batch
    src, tgt = synth.make_graph(WORKLOAD_ID)
    xq_np, xkv_np, prm = make_rank_inputs(rank, B)
    self_attn = xkv_np is xq_np
    params = pmha.Params.from_arrays(prm, w.num_heads, torch.bfloat16, dev)
    graph = pmha.pmha_build_csr(torch.from_numpy(src).to(dev), torch.from_numpy(tgt).to(dev),
                                w.query_features, w.key_features)
    nnz, H = graph.nnz, w.num_heads
    x = torch.from_numpy(xq_np).to(torch.bfloat16).to(dev)
    kv = x if self_attn else torch.from_numpy(xkv_np).to(torch.bfloat16).to(dev)
    out = torch.empty_like(x)
    ws = torch.empty(pmha.pmha_forward_workspace_size(graph, params, B, "none"), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        pmha.pmha_forward(graph, params, x, kv, kv, "none", out=out, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    pmha.pmha_device_status()

    sampler = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    sampler.start()
    first = sampler.mark()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = pmha.pmha_launch_count()
    pmha.pmha_profile_enable(True)
    pmha.pmha_profile_read()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)  # evict L2 between steps (not timed)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    pmha.pmha_profile_enable(False)
    prof = pmha.pmha_profile_read()
    launches = pmha.pmha_launch_count() - launches0
    clocks = sampler.summary(first)
    sampler.stop()
    pmha.pmha_device_status()

    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms, world, dev)
    scores = float(B) * nnz * H
    value = world * scores / (ms / 1e3)

    # ---- the same workload with a key_padding_mask: each sample keeps its
    # first n_b ~ U[S/2, S] keys (padding at the end), timed like the steps above
    kpm = torch.from_numpy(synth.padding_mask(np.random.default_rng(7 + rank), B, w.key_features)).to(dev)
    masked_steps = max(3, min(args.steps, 100))
    for _ in range(3):
        pmha.pmha_forward(graph, params, x, kv, kv, "none", out=out, workspace=ws, stream=stream,
                          key_padding_mask=kpm)
    pmha.pmha_device_status()
    pmha.pmha_profile_enable(True)
    pmha.pmha_profile_read()
    m_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(masked_steps)]
    for i, (e_start, e_end) in enumerate(m_ev):
        flush.fill_(i & 0xFF)
        e_start.record(stream)
        pmha.pmha_forward(graph, params, x, kv, kv, "none", out=out, workspace=ws, stream=stream,
                          key_padding_mask=kpm)
        e_end.record(stream)
    torch.cuda.synchronize()
    pmha.pmha_profile_enable(False)
    m_prof = pmha.pmha_profile_read()
    pmha.pmha_device_status()
    m_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in m_ev) / masked_steps, world, dev)
    masked = {"ms_per_step": m_ms, "value": world * float(B) * nnz * H / (m_ms / 1e3), "unit": UNIT,
              "steps": masked_steps, "kept_key_fraction": float(1.0 - kpm.float().mean().item()),
              "mask": "per-sample end padding, n_b ~ U[S/2, S] keys kept (value counts every edge)",
              "stages_avg_us": {k: 1e3 * v[1] / max(v[0], 1) for k, v in m_prof.items()}}

    # ---- the backward pass (pmha_backward: forward recompute + gradients of
    # inputs, weights and biases) for a seeded dout, timed the same way
    back = None
    if not args.no_backward:
        g_out = torch.from_numpy(synth.make_tokens(np.random.default_rng(11 + rank), B, w.query_features,
                                                   w.embed_dim, w.dtype)).to(torch.bfloat16).to(dev)
        ws_b = torch.empty(max(1, pmha.pmha_backward_workspace_size(graph, params, B)), dtype=torch.uint8, device=dev)
        for _ in range(3):
            pmha.pmha_backward(graph, params, x, kv, kv, g_out, workspace=ws_b, stream=stream)
        pmha.pmha_device_status()
        back_steps = max(3, min(args.steps, 30))
        pmha.pmha_profile_enable(True)
        pmha.pmha_profile_read()
        b_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(back_steps)]
        for i, (e_start, e_end) in enumerate(b_ev):
            flush.fill_(i & 0xFF)
            e_start.record(stream)
            pmha.pmha_backward(graph, params, x, kv, kv, g_out, workspace=ws_b, stream=stream)
            e_end.record(stream)
        torch.cuda.synchronize()
        pmha.pmha_profile_enable(False)
        b_prof = pmha.pmha_profile_read()
        pmha.pmha_device_status()
        b_ms = max_over_ranks(sum(e0_.elapsed_time(e1_) for e0_, e1_ in b_ev) / back_steps, world, dev)
        back = {"ms_per_step": b_ms, "value": world * float(B) * nnz * H / (b_ms / 1e3), "unit": UNIT,
                "steps": back_steps, "what": "pmha_backward: forward recompute, input, weight and bias gradients",
                "stages_avg_us": {k: 1e3 * v[1] / max(v[0], 1) for k, v in b_prof.items()}}

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

    # ---- roofline of the dominant kernel
    peaks = load_peaks()
    stages = {k: {"launches": v[0], "total_ms": v[1], "avg_us": 1e3 * v[1] / max(v[0], 1)} for k, v in prof.items()}
    total_stage_ms = sum(v["total_ms"] for v in stages.values()) or 1.0
    for v in stages.values():
        v["share"] = v["total_ms"] / total_stage_ms
    dom = max(stages, key=lambda k: stages[k]["total_ms"]) if stages else None
    roof = None
    if dom is not None:
        avg_s = stages[dom]["avg_us"] / 1e6
        alg = algorithmic_bytes(dom, w, B, nnz)
        fl = stage_flops(dom, w, B)
        # a GEMM is tensor-bound when its arithmetic intensity passes the ridge
        # point of the two measured peaks (E = 512), else memory-bound (E = 128)
        ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        tensor_bound = fl is not None and (dom in TENSOR_BOUND or (alg is not None and fl / alg > ridge))
        if tensor_bound:
            # timed inside a long loop of steps: the sustained tensor peak
            achieved = fl / avg_s / 1e12
            peak = peaks["bf16_tflops_sustained"]
            roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": ncu_traffic(dom, w.name), "algorithmic_flops_per_launch": fl,
                    "algorithmic_bytes_per_launch": alg, "avg_launch_us": stages[dom]["avg_us"],
                    "peak_source": f"{peaks['source']} sustained bf16 GEMM (MEASURED_PEAKS.json "
                                   "bf16_tflops_sustained; fp16 runs at the bf16 rate)"}
        elif alg is not None:
            achieved = alg / avg_s / 1e9
            roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(dom, w.name),
                    "algorithmic_bytes_per_launch": alg, "avg_launch_us": stages[dom]["avg_us"],
                    "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"}
    for k, v in stages.items():
        alg = algorithmic_bytes(k, w, B, nnz)
        if alg is not None:
            v["hbm_gbs_algorithmic"] = alg / (v["avg_us"] / 1e6) / 1e9
            v["hbm_frac"] = v["hbm_gbs_algorithmic"] / peaks["hbm_gbs"]
        fl = stage_flops(k, w, B)
        if fl is not None:
            v["tflops"] = fl / (v["avg_us"] / 1e6) / 1e12
            v["tensor_frac"] = v["tflops"] / peaks["bf16_tflops"]

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cpu = run_cpu_baseline(args.cpu_seconds, src, tgt, w, xq_np, xkv_np, prm)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "layer_fwd_us": ms * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "batch": B, "n": w.query_features, "nnz": nnz,
                       "embed_dim": w.embed_dim, "num_heads": H, "max_in_degree": graph.max_in_degree,
                       "l2": "flushed between timed steps (512 MiB write, untimed)",
                       "parallelism": f"replicas x{world}, own batch per rank, no collective"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "serial_ms_per_step": e2e_serial_ms,
                    "api": f"pmha_forward_host (pinned host buffers), steps rotating over {E2E_STREAMS} streams"},
            "gpu_launches": launches,
            "roofline": roof,
            "stages": stages,
            "variants": {"key_padding_mask": masked, "backward": back},
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
