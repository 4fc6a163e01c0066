#!/usr/bin/env python
"""Benchmark: weight-stream GB/s of the MXFP4 MoE decode layer sweep on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one decode token through 24 gpt-oss-style MoE layers. Each layer
(qmv_moe_layer, two kernel launches) gathers 4 of 32 experts for gate and up
(2880 x 2880 MXFP4, shared bf16 activation) with SwiGLU fused into that
launch, then gathers the same 4 experts of down (per-slot activation) -- 12
expert matrices, 52,876,800 weight bytes per layer. Router
ids are fresh each step. The weight bytes of a step (1.27 GB) exceed L2, so
nothing is served from L2 across steps. `value` = weight bytes of all steps on
all ranks / max-over-ranks device time (CUDA events, CUDA-graph replay).

Multi-GPU: the workload does not shard; every rank runs an independent replica
(weak scaling) and rank 0 reports the aggregate.

--impl reference times the CPU oracle (single-threaded numpy, the repository's
reference definition of the method) on the same workload, one expert matvec
per step.
"""
from __future__ import annotations

import os

# The CPU legs time the oracle single-threaded; pin BLAS before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import threading  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import qmv_inputs as qi  # noqa: E402

LAYERS = qi.CONFIG1_LAYERS
E, N, K, TOP_K = 32, 2880, 2880, 4
MATRIX_BYTES = 4406400                     # 2880*1440 code bytes + 2880*90 E8M0 bytes
LAYER_BYTES = 12 * MATRIX_BYTES            # gate, up, down x 4 experts
STEP_BYTES = LAYERS * LAYER_BYTES
GATHER_BYTES = TOP_K * MATRIX_BYTES        # one gather launch (4 distinct experts)

WORKLOAD = ("gpt-oss MoE decode layer sweep: 24 layers x (gate, up, down) MXFP4 E2M1/E8M0-g32 "
            "2880x2880 expert gathers, E=32, top_k=4 fresh ids per step, 1 token, bf16 activations, "
            "SwiGLU between")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# Clock sampling (nvidia-smi) during the timed window
# ---------------------------------------------------------------------------

def gpu_uuid(dev) -> str:
    import torch
    u = str(torch.cuda.get_device_properties(dev).uuid)
    return u if u.startswith("GPU-") else "GPU-" + u


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [r for t, r in self.rows if t0 <= t <= t1] or [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------

def oracle_expert_matvecs(canon, scales, x_bits, budget_s: float, min_calls: int = 1):
    """Run the oracle's MXFP4 matvec on consecutive pool experts until the time budget is spent.

    The oracle decodes the canonical bytes itself (unpack, E2M1, E8M0) inside
    the timed loop, as a CPU implementation of the same call would.
    """
    import oracle
    calls, t0 = 0, time.perf_counter()
    while calls < min_calls or time.perf_counter() - t0 < budget_s:
        e = calls % len(canon)
        oracle.mxfp4_matvec(oracle.unpack_nibbles(canon[e]), scales[e], x_bits)
        calls += 1
    return calls, time.perf_counter() - t0


def _oracle_rows_worker(args):
    """One process of the row-parallel oracle leg: the oracle's MXFP4 matvec on
    a block of rows of consecutive pool experts until the budget is spent.
    Returns (weight bytes processed, seconds)."""
    canon_rows, scale_rows, x_bits, budget_s = args
    sys.path.insert(0, ROOT)
    import oracle
    n_rows = canon_rows.shape[1]
    calls, t0 = 0, time.perf_counter()
    while calls < 1 or time.perf_counter() - t0 < budget_s:
        e = calls % canon_rows.shape[0]
        oracle.mxfp4_matvec(oracle.unpack_nibbles(canon_rows[e]), scale_rows[e], x_bits)
        calls += 1
    return calls * n_rows * (K // 2 + K // 32), time.perf_counter() - t0


def cpu_baseline(canon, scales, x_bits, budget_s=12.0):
    """The oracle timed on the host cores: single-threaded, then row-parallel
    (one process per core, each the unchanged oracle on a block of output
    rows; a spawned pool, since the parent holds a CUDA context)."""
    calls, dt = oracle_expert_matvecs(canon, scales, x_bits, budget_s)
    single = calls * MATRIX_BYTES / dt / 1e9
    import multiprocessing as mp
    cores = max(1, os.cpu_count() or 1)
    bounds = np.linspace(0, N, cores + 1).astype(int)
    jobs = [(canon[:, a:b], scales[:, a:b], x_bits, budget_s) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with mp.get_context("spawn").Pool(len(jobs)) as pool:
        res = pool.map(_oracle_rows_worker, jobs)
    parallel = sum(b for b, _ in res) / max(t for _, t in res) / 1e9
    return {"value": parallel, "unit": "GB/s", "cores": len(jobs), "kind": "oracle",
            "single_thread_value": single,
            "sample": f"float64 oracle (incl. decode) on 2880x2880 MXFP4 expert matvecs of the config workload: "
                      f"{len(jobs)} spawned processes over output-row blocks for ~{budget_s:.0f} s each "
                      f"(row-parallel), and {calls} whole matvecs in {dt:.1f} s single-threaded "
                      f"({single:.4f} GB/s)"}


def make_pool(n: int, seed: int):
    """n experts of canonical MXFP4 code bytes [n][N][K/2], E8M0 scales and one bf16 activation."""
    g = qi.rng(seed)
    canon = qi.canonical_uniform_codes(g, (n, N), K, 4)
    scales = qi.e8m0(g, (n, N, K // 32))
    x = qi.normal_bf16_bits(g, (1, K))
    return canon, scales, x


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed (string
    literals kept), so that comment edits leave the digest unchanged."""
    import re
    pat = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'', re.S)
    text = pat.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", text)
    return " ".join(text.split())


# Sources that compile into the step's kernel (matvec_kernel<MXFP4, 1, false>).
STEP_KERNEL_SOURCES = ("qmv_device.cuh", "qmv_internal.h", "qmv_layout.h", "qmv_matvec.cuh",
                       "qmv_matvec_mxfp4.cu")


def kernel_source_digest() -> str:
    """sha256 over the code (comments stripped) of the sources that compile
    into the step's kernel: the kernel identity the committed ncu summary
    refers to."""
    import hashlib
    d = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_quantized_moe_gb300", "csrc")
    for f in STEP_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            d.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return d.hexdigest()


def traffic_for_current_kernel():
    """DRAM bytes per launch of the step's kernel from the committed ncu
    summary, if it was taken on the current kernel sources; otherwise None."""
    import re
    p = os.path.join(ROOT, "profiles", "mxfp4_gather_2880_top4.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", txt)
    if not m or not h or h.group(1) != kernel_source_digest():
        return None
    return float(m.group(1))


# ---------------------------------------------------------------------------
# Distributed helpers
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over the process group (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(bytes_per_step_per_rank: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job GB/s: the bytes every rank streamed over the slowest rank's time."""
    return bytes_per_step_per_rank * steps * world / max_seconds / 1e9


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    canon, scales, x = make_pool(4, qi.CONFIG1_GATE.seed)
    for _ in range(args.warmup):
        oracle_expert_matvecs(canon, scales, x, 0.0)
    t0 = time.perf_counter()
    calls, _ = oracle_expert_matvecs(canon, scales, x, 0.0, min_calls=args.steps)
    dt = time.perf_counter() - t0
    value = calls * MATRIX_BYTES / dt / 1e9
    sample = (f"one 2880x2880 MXFP4 expert matvec (4,406,400 weight bytes) per step, float64 oracle, "
              f"single-threaded numpy, {calls} steps in {dt:.1f} s")
    line = {
        "impl": "reference", "metric": "quantized matvec weight-stream GB/s (MXFP4 MoE decode layer sweep)",
        "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / calls * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded uniform codes, E8M0 in [120,130], N(0,1) bf16 activations)",
        "config": {"workload": WORKLOAD, "step": "one expert matvec of the workload"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch

    import bit_quantized_moe_gb300 as qmv

    L = args.layers
    step_bytes = L * LAYER_BYTES
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # --- weights: pools of distinct packed experts (fused gate/up and down)
    # replicated over the layers; content repeats, addresses do not.
    pool_n = 32
    g_canon, g_scales, x_bits = make_pool(pool_n, qi.CONFIG1_GATE.seed)
    u_canon, u_scales, _ = make_pool(pool_n, qi.CONFIG1_UP.seed + 100)
    d_canon, d_scales, _ = make_pool(pool_n, qi.CONFIG1_DOWN.seed + 200)
    desc_gu = qmv.wdesc("mxfp4", N, K, E)
    desc_dn = qmv.wdesc("mxfp4", K, N, E)
    eb_gu = qmv.qmv_packed_gate_up_expert_bytes(desc_gu)
    eb_dn = qmv.qmv_packed_expert_bytes(desc_dn)
    pool_gu = torch.from_numpy(qmv.qmv_pack_gate_up(qmv.wdesc("mxfp4", N, K, pool_n), g_canon, g_scales,
                                                    u_canon, u_scales)).to(dev).view(pool_n, eb_gu)
    pool_dn = torch.from_numpy(qmv.qmv_pack_weights(qmv.wdesc("mxfp4", K, N, pool_n), d_canon,
                                                    d_scales)).to(dev).view(pool_n, eb_dn)
    W_gu = torch.empty(L * E, eb_gu, dtype=torch.uint8, device=dev)
    W_gu.view(-1, pool_n, eb_gu).copy_(pool_gu.unsqueeze(0).expand(L * E // pool_n, pool_n, eb_gu))
    W_dn = torch.empty(L * E, eb_dn, dtype=torch.uint8, device=dev)
    W_dn.view(-1, pool_n, eb_dn).copy_(pool_dn.unsqueeze(0).expand(L * E // pool_n, pool_n, eb_dn))
    W_gu, W_dn = W_gu.view(L, E * eb_gu), W_dn.view(L, E * eb_dn)
    del pool_gu, pool_dn

    x_dev = torch.from_numpy(x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    total_steps = args.warmup + args.steps
    g = qi.rng(1000 + rank)
    ids_host = np.stack([np.stack([qi.topk_ids(g, 1, TOP_K, E) for _ in range(L)]) for _ in range(total_steps)])
    ids_all = torch.from_numpy(ids_host).to(dev)               # [steps][layers][1][4]
    ids_sel = torch.empty(1, L, 1, TOP_K, dtype=torch.int32, device=dev)
    ids_buf = ids_sel[0]                                       # the step's ids, [layers][1][4]
    step_idx = torch.zeros(1, dtype=torch.long, device=dev)
    ws = torch.zeros(qmv.qmv_moe_layer_workspace_bytes(desc_gu, 1, TOP_K), dtype=torch.uint8, device=dev)
    layer_flags = qmv.QMV_FLAG_PREFETCH_INPUTS
    per_layer = 2
    y = torch.empty(L, 1, TOP_K, K, dtype=torch.bfloat16, device=dev)

    def step():
        """One decode token through all layers (fused gate/up/SwiGLU, then down).
        The weights and the step's ids are not written by the kernel right
        before any layer's launch, so every layer may prefetch them while the
        preceding kernel drains."""
        for l in range(L):
            qmv.qmv_moe_layer(desc_gu, W_gu[l], desc_dn, W_dn[l], x_dev, ids_buf[l], 1, TOP_K, ws, y[l],
                              layer_flags)

    def graph_step():
        """The step as captured: the step's router ids are picked on the device
        (ids_all[step_idx], standing in for the router producing them in the
        same stream), then the counter advances -- in that order, so the
        kernel right before the first layer does not write the ids -- then
        the layers."""
        torch.index_select(ids_all, 0, step_idx, out=ids_sel)
        step_idx.add_(1).remainder_(total_steps)
        step()

    # eager warm-up (sets kernel attributes), then capture one step in a CUDA graph
    ids_buf.copy_(ids_all[0])
    step()
    torch.cuda.synchronize()
    if args.profile:
        for i in range(args.steps):
            ids_buf.copy_(ids_all[i % total_steps])
            step()
        torch.cuda.synchronize()
        print(f"profile run: {args.steps} eager steps over {L} layers, device status "
              f"{qmv.qmv_device_status(clear=True)}", flush=True)
        return 0
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graph_step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        graph_step()
    step_idx.zero_()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_uuid(dev))
    sampler.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        graph.replay()                                 # steps 0 .. W-1
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    ev0.record()
    for i in range(args.steps):
        graph.replay()                                 # steps W .. W+K-1
    ev1.record()
    torch.cuda.synchronize()
    barrier()
    wall1 = time.time()
    # keep the same work running until the sampler has seen >= 1.5 s of it
    while time.time() - wall0 < 1.5:
        for i in range(20):
            graph.replay()
        torch.cuda.synchronize()
    wall2 = time.time()
    sampler.stop()
    dt_ms = ev0.elapsed_time(ev1)
    dt_max = max_over_ranks(dt_ms / 1e3, world, dev)
    value = aggregate_value(step_bytes, args.steps, world, dt_max)
    clocks = sampler.summary(wall0, wall2)
    clocks["window_s"] = round(wall2 - wall0, 3)
    clocks["timed_s"] = round(wall1 - wall0, 3)

    # --- dominant kernel: every launch of the step is matvec_kernel<MXFP4,1>
    # (L fused gate/up/SwiGLU gathers of 35.25 MB and L down gathers of
    # 17.63 MB), so its average launch time is the step time over the step's
    # 2L launches and its average algorithmic bytes per launch are
    # LAYER_BYTES / 2.
    launch_ms = dt_max * 1e3 / args.steps / (per_layer * L)
    hbm, peak_kind = peaks()
    bytes_per_launch = LAYER_BYTES // per_layer
    achieved = bytes_per_launch / (launch_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic_for_current_kernel(), "kernel": "matvec_kernel<MXFP4,1> (qmv_moe_layer)",
                "peak_kind": f"{peak_kind} hbm_gbs (burst copy)", "launch_us_mean": launch_ms * 1e3,
                "launches_timed": args.steps * per_layer * L, "algorithmic_bytes_per_launch": bytes_per_launch,
                "timing": "CUDA events around the timed step graphs; every launch in them is this kernel"}

    # --- e2e: host buffers, h2d of x and ids, graph step, d2h of every layer's output
    x_host = torch.from_numpy(x_bits.view(np.int16)).pin_memory()
    ids_host_p = torch.from_numpy(ids_host).pin_memory()
    y_host = torch.empty(y.shape, dtype=torch.bfloat16).pin_memory()
    n_e2e = min(args.steps, 50)
    torch.cuda.synchronize()
    cur = int(step_idx.item())                         # the id slot the next replay reads
    t0 = time.perf_counter()
    for i in range(n_e2e):
        x_dev.view(torch.int16).copy_(x_host, non_blocking=True)
        ids_all[cur].copy_(ids_host_p[args.warmup + i], non_blocking=True)
        graph.replay()
        cur = (cur + 1) % total_steps
        y_host.copy_(y, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    t_e2e = time.perf_counter() - t0
    t_e2e = max_over_ranks(t_e2e, world, dev)
    e2e = {"value": aggregate_value(step_bytes, n_e2e, world, t_e2e), "unit": "GB/s",
           "h2d_bytes_per_step": x_host.numel() * 2 + ids_buf.numel() * 4,
           "d2h_bytes_per_step": y_host.numel() * 2, "steps": n_e2e}
    status = qmv.qmv_device_status(clear=True)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(g_canon[:4], g_scales[:4], x_bits)

    if rank == 0:
        line = {
            "metric": "quantized matvec weight-stream GB/s (MXFP4 MoE decode layer sweep)",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt_max * 1e3 / args.steps, "us_per_moe_layer": dt_max * 1e6 / args.steps / L,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "frac_of_hbm_peak": value / world / hbm,
            "dtype": "mxfp4(e2m1,e8m0) x bf16 -> f32 accumulate",
            "data": "synthetic (seeded uniform E2M1 codes, E8M0 in [120,130], N(0,1) bf16 activations)",
            "config": {"workload": WORKLOAD, "layers": L, "experts": E, "top_k": TOP_K, "N": N, "K": K,
                       "ntok": 1, "weight_bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2: 1.27 GB of expert weights per step, fresh ids every step",
                       "launch": f"one CUDA graph per step: the step's router ids picked on the device (index_select at a device step counter), then {2 * L} kernels ({L} fused gate/up/SwiGLU gathers + {L} down gathers, qmv_moe_layer), programmatic dependent launch with weight/id prefetch",
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline, "clocks": clocks, "e2e": e2e,
            "gpu_launches": args.steps * L * per_layer, "cpu_baseline": cpu, "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# Per-config measurements (--configs): every config of the workload set, the
# same way as the headline line (CUDA-graph replay, inputs larger than L2,
# CUDA events), one JSON line each. Not the default line.
# ---------------------------------------------------------------------------

L2_BYTES = 132 * 1000 * 1000


def _replicated(qmv, torch, dev, desc_pool, pack, n_total: int, eb: int):
    """A device buffer of n_total experts (eb bytes each): a packed pool of
    distinct experts repeated; content repeats, addresses do not."""
    pool = torch.from_numpy(pack()).to(dev).view(desc_pool.n_experts, eb)
    w = torch.empty(n_total, eb, dtype=torch.uint8, device=dev)
    reps = (n_total + desc_pool.n_experts - 1) // desc_pool.n_experts
    w.copy_(pool.repeat(reps, 1)[:n_total])
    return w


def _graph_time(torch, calls, replays: int = 20):
    """Seconds per replay of a CUDA graph of `calls` (median of 3 batches)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        calls()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    res = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(replays):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        res.append(e0.elapsed_time(e1) / 1e3 / replays)
    return statistics.median(res), s


def run_configs(args):
    import torch

    import bit_quantized_moe_gb300 as qmv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm, peak_kind = peaks()
    PF = qmv.QMV_FLAG_PREFETCH_INPUTS
    g = qi.rng(77)
    pool = 8

    def emit(cfg, call, bytes_per_call, sec_per_call, extra=None):
        gbs = bytes_per_call / sec_per_call / 1e9
        line = {"config": cfg, "call": call, "us_per_call": sec_per_call * 1e6, "GB/s": gbs,
                "frac_of_hbm_peak": gbs / hbm, "peak": hbm, "peak_kind": f"{peak_kind} hbm_gbs",
                "weight_bytes_per_call": bytes_per_call, "status": qmv.qmv_device_status(clear=True)}
        line.update(extra or {})
        print(json.dumps(line), flush=True)

    def canon(fmt, n, N_, K_):
        gg = qi.rng(int(g.integers(1 << 30)))
        return (qi.canonical_uniform_codes(gg, (n, N_), K_, qi.FORMAT_BITS[fmt]),
                qi.e8m0(gg, (n, N_, K_ // qi.FORMAT_GROUP[fmt])))

    def luts(fmt):
        return {"cb2": qi.LUT_CB2, "cb3": qi.LUT_CB3, "cb4": qi.LUT_CB4}.get(fmt)

    # --- config 0: dense MXFP4 2880 x 2880, 1 token, copies rotated past L2
    d0 = qmv.wdesc("mxfp4", 2880, 2880, 1)
    b0 = qmv.qmv_packed_bytes(d0)
    n0 = -(-4 * L2_BYTES // b0)
    c0, s0 = canon("mxfp4", pool, 2880, 2880)
    W0 = _replicated(qmv, torch, dev, qmv.wdesc("mxfp4", 2880, 2880, pool),
                     lambda: qmv.qmv_pack_weights(qmv.wdesc("mxfp4", 2880, 2880, pool), c0, s0), n0, b0)
    x0 = torch.from_numpy(qi.normal_bf16_bits(g, (1, 2880)).view(np.int16)).to(dev).view(torch.bfloat16)
    y0 = torch.empty(n0, 2880, dtype=torch.bfloat16, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_dense_ex(d0, W0[i], x0, 1, y0[i], PF) for i in range(n0)])
    emit(0, "qmv_dense MXFP4 2880x2880 ntok=1", 4406400, t / n0, {"calls_per_graph": n0})
    del W0

    # --- configs 2 and 3 and the DS4 layer: E=256 resident expert sets, fresh ids per call
    E2, top_k = 256, 4
    dgu = qmv.wdesc("cb2", 2048, 7168, E2, luts("cb2"))
    egu = qmv.qmv_packed_gate_up_expert_bytes(dgu)
    cg, sg = canon("cb2", pool, 2048, 7168)
    cu, su = canon("cb2", pool, 2048, 7168)
    Wgu = _replicated(qmv, torch, dev, qmv.wdesc("cb2", 2048, 7168, pool, luts("cb2")),
                      lambda: qmv.qmv_pack_gate_up(qmv.wdesc("cb2", 2048, 7168, pool, luts("cb2")), cg, sg, cu, su),
                      E2, egu).view(-1)
    ddn = qmv.wdesc("cb3", 7168, 2048, E2, luts("cb3"))
    edn = qmv.qmv_packed_expert_bytes(ddn)
    cd, sd = canon("cb3", pool, 7168, 2048)
    Wdn = _replicated(qmv, torch, dev, qmv.wdesc("cb3", 7168, 2048, pool, luts("cb3")),
                      lambda: qmv.qmv_pack_weights(qmv.wdesc("cb3", 7168, 2048, pool, luts("cb3")), cd, sd),
                      E2, edn).view(-1)
    C = 32
    x2 = torch.from_numpy(qi.normal_f32(g, (1, 7168))).to(dev)
    xq2 = torch.empty(qmv.qmv_act_q8_bytes(1, 7168), dtype=torch.uint8, device=dev)
    qmv.qmv_quantize_act_q8(x2, 1, 7168, xq2)
    ids2 = torch.from_numpy(np.stack([qi.topk_ids(g, 1, top_k, E2) for _ in range(C)])).to(dev)
    h2 = torch.empty(C, 1, top_k, 2048, dtype=torch.float32, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_gate_up_swiglu(dgu, Wgu, xq2, ids2[i], 1, top_k, h2[i], PF)
                                       for i in range(C)])
    emit(2, "qmv_moe_gate_up_swiglu CB2 2048x7168 gate+up E=256 top4 ntok=1, q8_1 x", 8 * 4587520, t / C,
         {"calls_per_graph": C})
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_gate_up_swiglu(dgu, Wgu, x2, ids2[i], 1, top_k, h2[i],
                                                                  PF | qmv.QMV_FLAG_X_F32) for i in range(C)])
    emit(2, "qmv_moe_gate_up_swiglu CB2 2048x7168 gate+up E=256 top4 ntok=1, fp32 x (QMV_FLAG_X_F32)",
         8 * 4587520, t / C, {"calls_per_graph": C})
    xqs = torch.empty(C, qmv.qmv_act_q8_bytes(1, 7168), dtype=torch.uint8, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_quantize_act_q8(x2, 1, 7168, xqs[i]) for i in range(C)])
    emit(2, "qmv_quantize_act_q8 K=7168 ntok=1 (activation bytes, not weights)", 7168 * 4, t / C,
         {"calls_per_graph": C})

    C3 = 16
    ids3 = np.stack([qi.topk_ids(g, 4, top_k, E2) for _ in range(C3)])
    distinct = [len(set(r.reshape(-1).tolist())) for r in ids3]
    ids3d = torch.from_numpy(ids3).to(dev)
    xq3 = torch.empty(16, qmv.qmv_act_q8_bytes(1, 2048), dtype=torch.uint8, device=dev)
    qmv.qmv_quantize_act_q8(torch.from_numpy(qi.normal_f32(g, (16, 2048))).to(dev), 16, 2048, xq3)
    y3 = torch.empty(C3, 4, top_k, 7168, dtype=torch.float32, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_gather_ex(ddn, Wdn, xq3, 1, ids3d[i], 4, top_k, y3[i], PF)
                                       for i in range(C3)])
    emit(3, "qmv_moe_gather CB3 7168x2048 down E=256 top4 ntok=4 per-slot x", sum(distinct) * 6422528 / C3,
         t / C3, {"calls_per_graph": C3, "distinct_experts_mean": sum(distinct) / C3})

    # DS4 layer (CB2 gate/up -> SwiGLU -> q8_1 -> CB3 down), both launch structures
    CL = 16
    idsL = torch.from_numpy(np.stack([qi.topk_ids(g, 1, top_k, E2) for _ in range(CL)])).to(dev)
    wsL = torch.zeros(qmv.qmv_moe_layer_workspace_bytes(dgu, 1, top_k), dtype=torch.uint8, device=dev)
    yL = torch.empty(CL, 1, top_k, 7168, dtype=torch.float32, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_layer(dgu, Wgu, ddn, Wdn, xq2, idsL[i], 1, top_k, wsL,
                                                         yL[i], PF) for i in range(CL)])
    emit("ds4-layer", "qmv_moe_layer CB2 gate/up + CB3 down E=256 top4 ntok=1 (2 launches)",
         8 * 4587520 + 4 * 6422528, t / CL, {"calls_per_graph": CL})
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_layer(dgu, Wgu, ddn, Wdn, x2, idsL[i], 1, top_k, wsL,
                                                         yL[i], PF | qmv.QMV_FLAG_X_F32) for i in range(CL)])
    emit("ds4-layer", "qmv_moe_layer CB2 gate/up + CB3 down E=256 top4 ntok=1, fp32 x (2 launches, no quantize launch)",
         8 * 4587520 + 4 * 6422528, t / CL, {"calls_per_graph": CL})
    del Wgu, Wdn

    # --- config 4: dense CB4 7168x7168 and 2048x7168, ntok 1..4, copies rotated past L2
    for (N4, K4) in qi.CONFIG4_SHAPES:
        d4 = qmv.wdesc("cb4", N4, K4, 1, luts("cb4"))
        b4 = qmv.qmv_packed_bytes(d4)
        alg = N4 * K4 // 2 + N4 * (K4 // 32)
        n4 = -(-4 * L2_BYTES // b4)
        c4, s4 = canon("cb4", 2, N4, K4)
        W4 = _replicated(qmv, torch, dev, qmv.wdesc("cb4", N4, K4, 2, luts("cb4")),
                         lambda: qmv.qmv_pack_weights(qmv.wdesc("cb4", N4, K4, 2, luts("cb4")), c4, s4), n4, b4)
        for ntok in qi.CONFIG4_NTOKS:
            xq4 = torch.empty(qmv.qmv_act_q8_bytes(ntok, K4), dtype=torch.uint8, device=dev)
            qmv.qmv_quantize_act_q8(torch.from_numpy(qi.normal_f32(g, (ntok, K4))).to(dev), ntok, K4, xq4)
            y4 = torch.empty(n4, ntok, N4, dtype=torch.float32, device=dev)
            t, _ = _graph_time(torch, lambda: [qmv.qmv_dense_ex(d4, W4[i], xq4, ntok, y4[i], PF) for i in range(n4)])
            emit(4, f"qmv_dense CB4 {N4}x{K4} ntok={ntok}", alg, t / n4, {"calls_per_graph": n4})
        del W4

    # --- verify batches (f3): dense 8 and 16 tokens (one weight stream per 4 tokens, side by side)
    for fmt, (Nv, Kv) in (("mxfp4", (2880, 2880)), ("mxfp8", (2880, 2880)), ("mxfp4", (7168, 7168)),
                          ("mxfp8", (7168, 7168)), ("cb4", (7168, 7168))):
        dv = qmv.wdesc(fmt, Nv, Kv, 1, luts(fmt))
        bv = qmv.qmv_packed_bytes(dv)
        algv = Nv * Kv * qi.FORMAT_BITS[fmt] // 8 + Nv * (Kv // 32)
        nv_ = -(-4 * L2_BYTES // bv)
        cv, sv = canon(fmt, 2, Nv, Kv)
        if fmt == "mxfp8":
            sv = sv - 8
        Wv = _replicated(qmv, torch, dev, qmv.wdesc(fmt, Nv, Kv, 2, luts(fmt)),
                         lambda: qmv.qmv_pack_weights(qmv.wdesc(fmt, Nv, Kv, 2, luts(fmt)), cv, sv), nv_, bv)
        for ntok in (8, 16):
            if fmt in ("mxfp4", "mxfp8"):
                xv = torch.from_numpy(qi.normal_bf16_bits(g, (ntok, Kv)).view(np.int16)).to(dev).view(torch.bfloat16)
                yv = torch.empty(nv_, ntok, Nv, dtype=torch.bfloat16, device=dev)
            else:
                xv = torch.empty(qmv.qmv_act_q8_bytes(ntok, Kv), dtype=torch.uint8, device=dev)
                qmv.qmv_quantize_act_q8(torch.from_numpy(qi.normal_f32(g, (ntok, Kv))).to(dev), ntok, Kv, xv)
                yv = torch.empty(nv_, ntok, Nv, dtype=torch.float32, device=dev)
            t, _ = _graph_time(torch, lambda: [qmv.qmv_dense_ex(dv, Wv[i], xv, ntok, yv[i], PF) for i in range(nv_)])
            emit("f3", f"qmv_dense {fmt.upper()} {Nv}x{Kv} verify ntok={ntok}", algv, t / nv_,
                 {"calls_per_graph": nv_, "weights_x_tokens_per_s": Nv * Kv * ntok / (t / nv_)})
        del Wv

    # --- config 1 layer, both launch structures (the headline bench line uses the default)
    dgm, ddm = qmv.wdesc("mxfp4", N, K, E), qmv.wdesc("mxfp4", K, N, E)
    egm, edm = qmv.qmv_packed_gate_up_expert_bytes(dgm), qmv.qmv_packed_expert_bytes(ddm)
    Lm = 24
    gc, gs = canon("mxfp4", pool, N, K)
    uc, us_ = canon("mxfp4", pool, N, K)
    dc, ds = canon("mxfp4", pool, K, N)
    Wgm = _replicated(qmv, torch, dev, qmv.wdesc("mxfp4", N, K, pool),
                      lambda: qmv.qmv_pack_gate_up(qmv.wdesc("mxfp4", N, K, pool), gc, gs, uc, us_), Lm * E, egm)
    Wdm = _replicated(qmv, torch, dev, qmv.wdesc("mxfp4", K, N, pool),
                      lambda: qmv.qmv_pack_weights(qmv.wdesc("mxfp4", K, N, pool), dc, ds), Lm * E, edm)
    Wgm, Wdm = Wgm.view(Lm, -1), Wdm.view(Lm, -1)
    xm = torch.from_numpy(qi.normal_bf16_bits(g, (1, K)).view(np.int16)).to(dev).view(torch.bfloat16)
    idsm = torch.from_numpy(np.stack([qi.topk_ids(g, 1, TOP_K, E) for _ in range(Lm)])).to(dev)
    wsm = torch.zeros(qmv.qmv_moe_layer_workspace_bytes(dgm, 1, TOP_K), dtype=torch.uint8, device=dev)
    ym = torch.empty(Lm, 1, TOP_K, K, dtype=torch.bfloat16, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_layer(dgm, Wgm[l], ddm, Wdm[l], xm, idsm[l], 1, TOP_K, wsm,
                                                         ym[l], PF) for l in range(Lm)])
    emit(1, "qmv_moe_layer MXFP4 2880 E=32 top4 ntok=1 (2 launches)", LAYER_BYTES, t / Lm, {"calls_per_graph": Lm})
    # an 8-token verify batch through the same layers (32 routed slots per layer)
    ids8 = torch.from_numpy(np.stack([qi.topk_ids(g, 8, TOP_K, E) for _ in range(Lm)])).to(dev)
    x8 = torch.from_numpy(qi.normal_bf16_bits(g, (8, K)).view(np.int16)).to(dev).view(torch.bfloat16)
    ws8 = torch.zeros(qmv.qmv_moe_layer_workspace_bytes(dgm, 8, TOP_K), dtype=torch.uint8, device=dev)
    y8m = torch.empty(Lm, 8, TOP_K, K, dtype=torch.bfloat16, device=dev)
    distinct8 = [len(set(r.reshape(-1).tolist())) for r in ids8.cpu().numpy()]
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_layer(dgm, Wgm[l], ddm, Wdm[l], x8, ids8[l], 8, TOP_K, ws8,
                                                         y8m[l], PF) for l in range(Lm)])
    emit("f3", "qmv_moe_layer MXFP4 2880 E=32 top4 verify ntok=8 (32 routed slots, 2 launches)",
         3 * MATRIX_BYTES * sum(distinct8) / Lm, t / Lm,
         {"calls_per_graph": Lm, "distinct_experts_mean": sum(distinct8) / Lm})
    # sorted gathers (f3): 16 tokens x top-8 = 128 routed slots over the layer's 32 experts
    ids16 = torch.from_numpy(np.stack([qi.topk_ids(g, 16, 8, E) for _ in range(Lm)])).to(dev)
    x16b = torch.from_numpy(qi.normal_bf16_bits(g, (16, K)).view(np.int16)).to(dev).view(torch.bfloat16)
    xs128 = torch.from_numpy(qi.normal_bf16_bits(g, (128, K)).view(np.int16)).to(dev).view(torch.bfloat16)
    y128 = torch.empty(Lm, 16, 8, K, dtype=torch.bfloat16, device=dev)
    distinct16 = [len(set(r.reshape(-1).tolist())) for r in ids16.cpu().numpy()]
    sg_bytes = MATRIX_BYTES * sum(distinct16) / Lm
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_gather_ex(ddm, Wdm[l], x16b, 0, ids16[l], 16, 8, y128[l], PF)
                                       for l in range(Lm)])
    emit("f3", "qmv_moe_gather MXFP4 2880x2880 E=32 sorted, 16 tokens x top-8 (128 slots), shared x", sg_bytes,
         t / Lm, {"calls_per_graph": Lm, "distinct_experts_mean": sum(distinct16) / Lm})
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_gather_ex(ddm, Wdm[l], xs128, 1, ids16[l], 16, 8, y128[l], PF)
                                       for l in range(Lm)])
    emit("f3", "qmv_moe_gather MXFP4 2880x2880 E=32 sorted, 16 tokens x top-8 (128 slots), per-slot x", sg_bytes,
         t / Lm, {"calls_per_graph": Lm, "distinct_experts_mean": sum(distinct16) / Lm})
    # fp16 activations (QMV_FLAG_X_F16): same weights, x, h and y in fp16; x is
    # scaled by 2^-10 so that h and y stay inside fp16's range with these weights
    x16 = (qi.normal_f32(g, (1, K)) * np.float32(2.0 ** -10)).astype(np.float16)
    xm16 = torch.from_numpy(x16.view(np.int16)).to(dev).view(torch.float16)
    ym16 = torch.empty(Lm, 1, TOP_K, K, dtype=torch.float16, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_layer(dgm, Wgm[l], ddm, Wdm[l], xm16, idsm[l], 1, TOP_K, wsm,
                                                         ym16[l], PF | qmv.QMV_FLAG_X_F16) for l in range(Lm)])
    emit("f4", "qmv_moe_layer MXFP4 2880 E=32 top4 ntok=1, fp16 x/h/y (2 launches)", LAYER_BYTES, t / Lm,
         {"calls_per_graph": Lm})
    # the same layer with the router-weighted combine of its top-k outputs
    rw = torch.from_numpy(np.stack([qi.router_weights(g, 1, TOP_K) for _ in range(Lm)])).to(dev)
    wsc = torch.zeros(qmv.qmv_moe_layer_combine_workspace_bytes(dgm, ddm, 1, TOP_K), dtype=torch.uint8, device=dev)
    yc = torch.empty(Lm, 1, K, dtype=torch.bfloat16, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_layer_combine(dgm, Wgm[l], ddm, Wdm[l], xm, idsm[l], rw[l], 1,
                                                                 TOP_K, wsc, yc[l], PF) for l in range(Lm)])
    emit(1, "qmv_moe_layer_combine MXFP4 2880 E=32 top4 ntok=1 (3 launches)", LAYER_BYTES, t / Lm,
         {"calls_per_graph": Lm})
    del Wgm, Wdm

    # --- MXFP8 (E4M3 + E8M0/32): dense 2880x2880 and the gpt-oss-shaped layer
    d8 = qmv.wdesc("mxfp8", N, K, 1)
    b8 = qmv.qmv_packed_bytes(d8)
    alg8 = N * K + N * (K // 32)
    n8 = -(-4 * L2_BYTES // b8)
    c8, s8 = canon("mxfp8", pool, N, K)
    s8 = s8 - 8                                  # E4M3 magnitudes reach 448: scales 8 binades lower
    W8 = _replicated(qmv, torch, dev, qmv.wdesc("mxfp8", N, K, pool),
                     lambda: qmv.qmv_pack_weights(qmv.wdesc("mxfp8", N, K, pool), c8, s8), n8, b8)
    y8 = torch.empty(n8, K, dtype=torch.bfloat16, device=dev)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_dense_ex(d8, W8[i], xm, 1, y8[i], PF) for i in range(n8)])
    emit("f4", "qmv_dense MXFP8 2880x2880 ntok=1", alg8, t / n8, {"calls_per_graph": n8})
    del W8
    dg8, dd8 = qmv.wdesc("mxfp8", N, K, E), qmv.wdesc("mxfp8", K, N, E)
    eg8, ed8 = qmv.qmv_packed_gate_up_expert_bytes(dg8), qmv.qmv_packed_expert_bytes(dd8)
    gc, gs = canon("mxfp8", pool, N, K)
    uc, us_ = canon("mxfp8", pool, N, K)
    dc, ds = canon("mxfp8", pool, K, N)
    Wg8 = _replicated(qmv, torch, dev, qmv.wdesc("mxfp8", N, K, pool),
                      lambda: qmv.qmv_pack_gate_up(qmv.wdesc("mxfp8", N, K, pool), gc, gs - 8, uc, us_ - 8),
                      Lm * E, eg8).view(Lm, -1)
    Wd8 = _replicated(qmv, torch, dev, qmv.wdesc("mxfp8", K, N, pool),
                      lambda: qmv.qmv_pack_weights(qmv.wdesc("mxfp8", K, N, pool), dc, ds - 8),
                      Lm * E, ed8).view(Lm, -1)
    t, _ = _graph_time(torch, lambda: [qmv.qmv_moe_layer(dg8, Wg8[l], dd8, Wd8[l], xm, idsm[l], 1, TOP_K, wsm,
                                                         ym[l], PF) for l in range(Lm)])
    emit("f4", "qmv_moe_layer MXFP8 2880 E=32 top4 ntok=1 (2 launches)", 12 * alg8, t / Lm,
         {"calls_per_graph": Lm})
    return 0


def run_profile_config(args):
    """A few eager calls of one config's call on a small resident expert set
    (16 experts, 32 for the MXFP8 layer; full-size matrices), for ncu
    captures of the codebook, dense and MXFP8 kernels. Prints one status
    line, no JSON."""
    import torch

    import bit_quantized_moe_gb300 as qmv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = qi.rng(88)
    cfg = args.profile_config
    luts = {"cb2": qi.LUT_CB2, "cb3": qi.LUT_CB3, "cb4": qi.LUT_CB4}

    def packed(fmt, n, N_, K_):
        d = qmv.wdesc(fmt, N_, K_, n, luts.get(fmt))
        c = qi.canonical_uniform_codes(g, (n, N_), K_, qi.FORMAT_BITS[fmt])
        sc = qi.e8m0(g, (n, N_, K_ // qi.FORMAT_GROUP[fmt]))
        return torch.from_numpy(qmv.qmv_pack_weights(d, c, sc)).to(dev), d

    def q8(nvec, K_):
        xq = torch.empty(qmv.qmv_act_q8_bytes(nvec, K_), dtype=torch.uint8, device=dev)
        qmv.qmv_quantize_act_q8(torch.from_numpy(qi.normal_f32(g, (nvec, K_))).to(dev), nvec, K_, xq)
        return xq

    E, calls = 16, 6
    if cfg == 0:
        w, d = packed("mxfp4", 1, 2880, 2880)
        x = torch.from_numpy(qi.normal_bf16_bits(g, (1, 2880)).view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty(1, 2880, dtype=torch.bfloat16, device=dev)
        fn = lambda i: qmv.qmv_dense(d, w, x, 1, y)
    elif cfg == 2:
        dg = qmv.wdesc("cb2", 2048, 7168, E, qi.LUT_CB2)
        c1 = qi.canonical_uniform_codes(g, (E, 2048), 7168, 2)
        c2 = qi.canonical_uniform_codes(g, (E, 2048), 7168, 2)
        s1, s2 = qi.e8m0(g, (E, 2048, 7168 // 16)), qi.e8m0(g, (E, 2048, 7168 // 16))
        w = torch.from_numpy(qmv.qmv_pack_gate_up(dg, c1, s1, c2, s2)).to(dev)
        xq = q8(1, 7168)
        ids = torch.from_numpy(np.stack([qi.topk_ids(g, 1, 4, E) for _ in range(calls)])).to(dev)
        h = torch.empty(1, 4, 2048, dtype=torch.float32, device=dev)
        fn = lambda i: qmv.qmv_moe_gate_up_swiglu(dg, w, xq, ids[i], 1, 4, h)
    elif cfg == 5:
        # MXFP8 gpt-oss-shaped layer: fused gate/up/SwiGLU then down, 32 experts
        E8, N8 = 32, 2880
        dg = qmv.wdesc("mxfp8", N8, N8, E8)
        c1 = qi.canonical_uniform_codes(g, (E8, N8), N8, 8)
        c2 = qi.canonical_uniform_codes(g, (E8, N8), N8, 8)
        s1, s2 = qi.e8m0(g, (E8, N8, N8 // 32), 112, 122), qi.e8m0(g, (E8, N8, N8 // 32), 112, 122)
        wg = torch.from_numpy(qmv.qmv_pack_gate_up(dg, c1, s1, c2, s2)).to(dev)
        w, d = packed("mxfp8", E8, N8, N8)
        x = torch.from_numpy(qi.normal_bf16_bits(g, (1, N8)).view(np.int16)).to(dev).view(torch.bfloat16)
        ids = torch.from_numpy(np.stack([qi.topk_ids(g, 1, 4, E8) for _ in range(calls)])).to(dev)
        ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(dg, 1, 4), dtype=torch.uint8, device=dev)
        y = torch.empty(1, 4, N8, dtype=torch.bfloat16, device=dev)
        fn = lambda i: qmv.qmv_moe_layer(dg, wg, d, w, x, ids[i], 1, 4, ws, y, qmv.QMV_FLAG_PREFETCH_INPUTS)
    elif cfg == 6:
        # verify batch: dense MXFP4 7168 x 7168, 16 tokens (tensor-core path)
        w, d = packed("mxfp4", 1, 7168, 7168)
        x = torch.from_numpy(qi.normal_bf16_bits(g, (16, 7168)).view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty(16, 7168, dtype=torch.bfloat16, device=dev)
        fn = lambda i: qmv.qmv_dense_ex(d, w, x, 16, y, qmv.QMV_FLAG_PREFETCH_INPUTS)
    elif cfg == 7:
        # verify batch: dense CB4 7168 x 7168, 16 q8_1 tokens (tensor-core path)
        w, d = packed("cb4", 1, 7168, 7168)
        xq = q8(16, 7168)
        y = torch.empty(16, 7168, dtype=torch.float32, device=dev)
        fn = lambda i: qmv.qmv_dense_ex(d, w, xq, 16, y, qmv.QMV_FLAG_PREFETCH_INPUTS)
    elif cfg == 3:
        w, d = packed("cb3", E, 7168, 2048)
        xq = q8(16, 2048)
        ids = torch.from_numpy(np.stack([qi.topk_ids(g, 4, 4, E) for _ in range(calls)])).to(dev)
        y = torch.empty(4, 4, 7168, dtype=torch.float32, device=dev)
        fn = lambda i: qmv.qmv_moe_gather(d, w, xq, 1, ids[i], 4, 4, y)
    else:
        w, d = packed("cb4", 1, 7168, 7168)
        xq = q8(1, 7168)
        y = torch.empty(1, 7168, dtype=torch.float32, device=dev)
        fn = lambda i: qmv.qmv_dense(d, w, xq, 1, y)
    for i in range(calls):
        fn(i)
    torch.cuda.synchronize()
    print(f"profile-config {cfg}: {calls} calls, device status {qmv.qmv_device_status(clear=True)}", flush=True)
    return 0


# ---------------------------------------------------------------------------
# Secondary ALU roofline: the matvec inner loop's compute rate
# ---------------------------------------------------------------------------

# weight bytes per weight of each format (codes + E8M0 bytes)
BYTES_PER_WEIGHT = {"mxfp4": 4.25 / 8, "mxfp8": 8.25 / 8, "cb2": 2.5 / 8, "cb3": 3.5 / 8, "cb4": 4.25 / 8}
ALU_CASES = (("mxfp4", 1), ("mxfp4", 2), ("mxfp4", 4), ("mxfp8", 1), ("mxfp8", 4), ("cb2", 1), ("cb3", 1),
             ("cb3", 2), ("cb4", 1), ("cb4", 3), ("cb4", 4))


def run_alu(args):
    """For each (format, vectors per entry): the chunk routine's weights per
    clock per SM at the production launch shape (two CTAs per SM), with no
    copies or waits (qmv_debug_chunk_rate), beside the rate the measured HBM
    bandwidth delivers for that format. Clocks are sampled during the runs;
    the rate uses the median sampled SM clock."""
    import torch

    import bit_quantized_moe_gb300 as qmv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    hbm, hbm_kind = peaks()
    sampler = ClockSampler(gpu_uuid(dev))
    sampler.start()
    time.sleep(0.3)
    iters = 256
    rows = []
    wall0 = time.time()
    for fmt, nv in ALU_CASES:
        w, th = qmv.qmv_debug_chunk_rate(fmt, nv, 2, iters)
        sink = torch.empty(th, dtype=torch.float32, device=dev)
        for _ in range(3):
            qmv.qmv_debug_chunk_rate(fmt, nv, 2, iters, sink)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        ev0.record()
        for _ in range(reps):
            qmv.qmv_debug_chunk_rate(fmt, nv, 2, iters, sink)
        ev1.record()
        torch.cuda.synchronize()
        rows.append((fmt, nv, w * reps / (ev0.elapsed_time(ev1) * 1e-3)))
    # the time must scale with the iteration count (a loop the compiler
    # shortened would not): one case at 4x the iterations
    scale = {}
    for it in (iters, 4 * iters):
        w, th = qmv.qmv_debug_chunk_rate("mxfp4", 1, 2, it)
        sink = torch.empty(th, dtype=torch.float32, device=dev)
        qmv.qmv_debug_chunk_rate("mxfp4", 1, 2, it, sink)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        qmv.qmv_debug_chunk_rate("mxfp4", 1, 2, it, sink)
        ev1.record()
        torch.cuda.synchronize()
        scale[it] = ev0.elapsed_time(ev1) * 1e3
    time.sleep(0.3)
    wall1 = time.time()
    sampler.stop()
    clocks = sampler.summary(wall0, wall1)
    mhz = clocks.get("sm_mhz") or 2070.0
    print(f"mxfp4 nv=1 launch time at {iters} / {4 * iters} iterations: {scale[iters]:.1f} / "
          f"{scale[4 * iters]:.1f} us (ratio {scale[4 * iters] / scale[iters]:.2f})", flush=True)
    out = []
    for fmt, nv, wps in rows:
        rate = wps / sms / (mhz * 1e6)
        need = hbm * 1e9 / BYTES_PER_WEIGHT[fmt] / sms / (mhz * 1e6)
        out.append({"fmt": fmt, "vectors": nv, "weights_per_clk_per_sm": round(rate, 2),
                    "hbm_rate_weights_per_clk_per_sm": round(need, 2), "compute_over_hbm": round(rate / need, 3)})
        print(f"{fmt:6s} nv={nv}  {rate:7.2f} weights/clk/SM (compute only)   HBM at {hbm:.0f} GB/s ({hbm_kind}) "
              f"needs {need:6.2f}   ratio {rate / need:5.2f}", flush=True)
    print(json.dumps({"alu_roofline": out, "sm_mhz": mhz, "clocks": clocks, "sms": sms,
                      "launch": "2 CTAs per SM of the production shape, chunk routine on a resident tile, "
                                f"{iters} iterations per warp"}), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Phase probe: where the time of each launch of the step goes
# ---------------------------------------------------------------------------

PROBE_LAYERS = (10, 11, 12, 13)    # 8 launches: the probe buffer's 8 slots


def run_phase_probe(args):
    """Builds the phase-probe variant of the library (build.py --phase-probe)
    and runs the step's graph in a child process that loads it: the launches
    of four consecutive layers record per-warp %globaltimer stamps at the
    phases of the matvec kernel. Prints, per launch, each phase's min /
    median / max over all warps in us from the first probed launch's start,
    then one JSON line of per-launch spans."""
    if not os.environ.get("QMV_LIB"):
        import importlib.util
        spec = importlib.util.spec_from_file_location(
            "qmv_build", os.path.join(ROOT, "bit_quantized_moe_gb300", "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        lib = mod.build(phase_probe=True)
        env = dict(os.environ, QMV_LIB=lib)
        cmd = [sys.executable, os.path.abspath(__file__), "--phase-probe", "--warmup", str(args.warmup),
               "--layers", str(args.layers)]
        return subprocess.call(cmd, env=env)
    import torch

    import bit_quantized_moe_gb300 as qmv
    L = args.layers
    assert L > max(PROBE_LAYERS), "the probed layers must exist"
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pool_n = 32
    g_canon, g_scales, x_bits = make_pool(pool_n, qi.CONFIG1_GATE.seed)
    u_canon, u_scales, _ = make_pool(pool_n, qi.CONFIG1_UP.seed + 100)
    d_canon, d_scales, _ = make_pool(pool_n, qi.CONFIG1_DOWN.seed + 200)
    desc_gu, desc_dn = qmv.wdesc("mxfp4", N, K, E), qmv.wdesc("mxfp4", K, N, E)
    eb_gu, eb_dn = qmv.qmv_packed_gate_up_expert_bytes(desc_gu), qmv.qmv_packed_expert_bytes(desc_dn)
    pool_gu = torch.from_numpy(qmv.qmv_pack_gate_up(qmv.wdesc("mxfp4", N, K, pool_n), g_canon, g_scales,
                                                    u_canon, u_scales)).to(dev).view(pool_n, eb_gu)
    pool_dn = torch.from_numpy(qmv.qmv_pack_weights(qmv.wdesc("mxfp4", K, N, pool_n), d_canon,
                                                    d_scales)).to(dev).view(pool_n, eb_dn)
    W_gu = torch.empty(L * E, eb_gu, dtype=torch.uint8, device=dev)
    W_gu.view(-1, pool_n, eb_gu).copy_(pool_gu.unsqueeze(0).expand(L * E // pool_n, pool_n, eb_gu))
    W_dn = torch.empty(L * E, eb_dn, dtype=torch.uint8, device=dev)
    W_dn.view(-1, pool_n, eb_dn).copy_(pool_dn.unsqueeze(0).expand(L * E // pool_n, pool_n, eb_dn))
    W_gu, W_dn = W_gu.view(L, E * eb_gu), W_dn.view(L, E * eb_dn)
    x_dev = torch.from_numpy(x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    g = qi.rng(1000)
    ids = torch.from_numpy(np.stack([qi.topk_ids(g, 1, TOP_K, E) for _ in range(L)])).to(dev)
    ws = torch.zeros(qmv.qmv_moe_layer_workspace_bytes(desc_gu, 1, TOP_K), dtype=torch.uint8, device=dev)
    y = torch.empty(L, 1, TOP_K, K, dtype=torch.bfloat16, device=dev)

    def step(probe):
        for l in range(L):
            if probe:
                qmv.qmv_debug_phase_probe(l in PROBE_LAYERS)
            qmv.qmv_moe_layer(desc_gu, W_gu[l], desc_dn, W_dn[l], x_dev, ids[l], 1, TOP_K, ws, y[l],
                              qmv.QMV_FLAG_PREFETCH_INPUTS)
        if probe:
            qmv.qmv_debug_phase_probe(False)

    step(False)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(False)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(True)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    qmv.qmv_debug_phase_read("mxfp4", clear=True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    graph.replay()
    ev1.record()
    torch.cuda.synchronize()
    t = qmv.qmv_debug_phase_read("mxfp4", clear=True).astype(np.int64)
    print(f"phase probe: {L} layers, step {ev0.elapsed_time(ev1) * 1e3:.1f} us "
          f"({ev0.elapsed_time(ev1) * 1e3 / L:.2f} us per layer, probe build); layers {PROBE_LAYERS} probed, "
          f"us from the first probed launch's earliest start; min / median / max over warps", flush=True)
    starts = t[0, :, :, 0]
    base = starts[starts > 0].min()
    spans = []
    for slot in range(8):
        a = t[slot]
        w = a[a[:, :, 0] > 0]
        kind = "gate/up" if slot % 2 == 0 else "down"
        print(f"launch {slot} ({kind}, layer {PROBE_LAYERS[slot // 2]}): {int((a[:, 0, 0] > 0).sum())} CTAs, "
              f"{len(w)} warps")
        row = {"launch": slot, "kind": kind}
        for k, name in enumerate(qmv.PHASES):
            c = w[:, k]
            c = c[c > 0]
            if len(c) == 0:
                continue
            lo, med, hi = (c.min() - base) / 1e3, (np.median(c) - base) / 1e3, (c.max() - base) / 1e3
            row[name] = [round(lo, 2), round(med, 2), round(hi, 2)]
            print(f"  {name:12s} n={len(c):5d} {lo:8.2f} {med:8.2f} {hi:8.2f}")
        spans.append(row)
    print(json.dumps({"phase_probe": spans}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="eager run of --steps steps over --layers layers for ncu captures; prints no JSON")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="layers held on the device (the reported workload is 24; smaller for ncu captures)")
    ap.add_argument("--digest", action="store_true", help="print the kernel source digest and exit")
    ap.add_argument("--alu", action="store_true",
                    help="the chunk routine's compute rate per format (secondary ALU roofline) and exit")
    ap.add_argument("--phase-probe", action="store_true",
                    help="build the phase-probe variant and print where each launch's time goes")
    ap.add_argument("--configs", action="store_true",
                    help="measure every config of the workload set (one JSON line per call type) and exit")
    ap.add_argument("--profile-config", type=int, choices=[0, 2, 3, 4, 5, 6, 7], default=None,
                    help="a few eager calls of one config on a small resident set, for ncu captures "
                         "(5: the MXFP8 layer; 6 / 7: a 16-token MXFP4 / CB4 7168x7168 verify batch)")
    args = ap.parse_args(argv)
    if args.digest:
        print(kernel_source_digest())
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.phase_probe:
        return run_phase_probe(args)
    if args.alu:
        return run_alu(args)
    if args.configs:
        return run_configs(args)
    if args.profile_config is not None:
        return run_profile_config(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
