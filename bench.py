#!/usr/bin/env python
"""Benchmark of the routed ReLU^2 MoE layer on GB300: MoE-layer tokens/s and the
fraction of the HBM roofline (decode) or of the dense tensor peak (prefill)
reached.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload nano_decode] [--tokens 64] [--points all|none|<workload>]

A step is one full layer forward (router, dispatch, experts up, experts down,
combine, shared expert; latent projections for latent shapes) over one batch
of T synthetic tokens.  Weights come in several seeded replicas that the steps
rotate through, so no step finds the previous step's weights in L2.  Prints
one JSON line (rank 0): the headline workload (Nano decode, T = 64) with its
dominant kernel's roofline, the end-to-end figure through the host-buffer
entry point and the oracle on the host cores, plus ``per_workload``: every
workload at every token count it is defined for.  Multi-GPU (torchrun): every
rank runs its own layer replica on its own tokens (no collective on the data
path; weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 2 ** 20
CSRC = os.path.join(ROOT, "routed_relu_expert_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.md")
# the sources a kernel family is compiled from: a recorded DRAM traffic figure
# holds only while their hash is unchanged
KERNEL_SOURCES = {
    "gemv": ("gemv.cu", "epilogue.cuh", "nvfp4.cuh", "common.cuh", "internal.h"),
    "tc": ("gemm_tc.cu", "tc_common.cuh", "epilogue.cuh", "nvfp4.cuh", "common.cuh", "internal.h"),
    "fp4": ("gemm_fp4.cu", "tc_common.cuh", "epilogue.cuh", "nvfp4.cuh", "common.cuh", "internal.h"),
}
ACT_TERMS = 3            # the library's default NVFP4 activation terms


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="nano_decode")
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--replicas", type=int, default=0, help="weight replicas (0 = enough to defeat L2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--points", default="all",
                    help="per_workload entries: all, none, or one workload name")
    ap.add_argument("--eager", action="store_true", help="time eager calls instead of CUDA-graph replays")
    ap.add_argument("--no-backward", dest="backward", action="store_false",
                    help="skip the backward timings")
    ap.add_argument("--no-blocks", dest="blocks", action="store_false",
                    help="skip the MoE-block chains (RMSNorm + layer + residual) at the verify shapes")
    ap.add_argument("--nvfp4-act-terms", type=int, default=-1,
                    help="NVFP4 experts: activation terms on the FP4 tensor path (1-4), 0 = FP16 path; "
                         "-1 = the library's default")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while a timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        rows = [l.strip().split(",") for l in open(self.f.name) if l.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank processes its own tokens (weak scaling)."""
    return world * tokens_per_rank / seconds


# ---------------------------------------------------------------------------
def expert_bytes(shape) -> int:
    """HBM bytes of one routed expert (up + down; NVFP4: values, block scales
    and the two FP32 per-tensor scales)."""
    de, I = shape.d_e, shape.d_expert
    if shape.expert_dtype == 2:
        return 2 * (I * de // 2 + I * de // 16) + 8
    return 2 * I * de * (4 if shape.expert_dtype == 0 else 2)


def layer_bytes(shape, n_active: int, T: int) -> dict:
    """Algorithmic HBM bytes of one layer step: weights of the experts that
    received routes, shared expert, router, latent pair, and the activations in
    and out."""
    ab = 4 if shape.act_dtype == 0 else 2
    de, d, S, E = shape.d_e, shape.d_model, shape.d_shared, shape.n_experts
    b = {"experts": n_active * expert_bytes(shape), "shared": 2 * d * S * ab, "router": E * d * 4 + E * 4,
         "latent": 2 * d * shape.d_latent * ab, "activations": 2 * T * d * ab}
    b["total"] = sum(b.values())
    return b


def layer_flops(shape, T: int) -> int:
    de, I, d, S, E, K = shape.d_e, shape.d_expert, shape.d_model, shape.d_shared, shape.n_experts, shape.top_k
    per_tok = 2 * E * d + K * 4 * de * I + 4 * d * S + 4 * d * shape.d_latent
    return per_tok * T


def product_ledger(shape, n_active: int, T: int, which: str) -> dict:
    """Algorithmic bytes and FLOPs of one grouped expert product over a batch:
    ``up`` reads the active experts' up weights and the R = T*K routed rows and
    writes h [R, I]; ``down`` reads the down weights and h and writes the FP32
    routed rows u [R, de] (plus the routing weight of every row)."""
    ab = 4 if shape.act_dtype == 0 else 2
    de, I, R = shape.d_e, shape.d_expert, T * shape.top_k
    w1 = expert_bytes(shape) // 2 if shape.expert_dtype != 2 else (I * de // 2 + I * de // 16 + 4)
    if which == "up":
        b = n_active * w1 + R * de * ab + R * I * ab
    else:
        b = n_active * w1 + R * I * ab + R * de * 4 + R * 4
    return {"bytes": int(b), "flops": int(2 * R * de * I)}


def routing_stats(ids, n_experts, tile_rows=128):
    """Load skew of one batch's routing, from its [T, K] expert ids (the load
    statistics of page "M6.1 Routed Capacity", section on load balance): routes
    per expert -> experts with routes, max/mean, CV^2 (variance / mean^2 over
    all experts), entropy of the route shares normalised by log E, the slope of
    log(count) against log(rank) over the experts with routes (about -s for a
    Zipf(s) popularity), and the share of padded rows when every expert's rows
    are cut into tiles of `tile_rows` (the grouped GEMM's tail waste)."""
    c = np.bincount(np.asarray(ids).reshape(-1).astype(np.int64), minlength=n_experts).astype(np.float64)
    total = c.sum()
    mean = total / n_experts
    p = c[c > 0] / total
    srt = np.sort(c[c > 0])[::-1]
    slope = None
    if len(srt) >= 3 and srt[0] > srt[-1]:
        slope = round(float(np.polyfit(np.log(np.arange(1, len(srt) + 1)), np.log(srt), 1)[0]), 3)
    padded = float((np.ceil(c / tile_rows) * tile_rows).sum())
    return {"experts_with_routes": int((c > 0).sum()), "max_over_mean": round(float(c.max() / mean), 2),
            "cv2": round(float(c.var() / mean ** 2), 3),
            "norm_entropy": round(float(-(p * np.log(p)).sum() / np.log(n_experts)), 3),
            "loglog_slope": slope, f"tail_waste_{tile_rows}_row_tiles": round(float(1.0 - total / padded), 3)}


def roofline_fractions(shape, T: int, n_active: int, ms: float, pk: dict) -> dict:
    """A layer step's bytes and FLOPs over its time, against the measured peaks;
    the binding one is the larger ideal time (bytes at the copy bandwidth,
    FLOPs at the burst bf16 peak)."""
    lb = layer_bytes(shape, n_active, T)
    fl = layer_flops(shape, T)
    s = ms / 1e3
    gbs = lb["total"] / s / 1e9
    tf = fl / s / 1e12
    tensor = fl / (pk["bf16_tflops"] * 1e12) > lb["total"] / (pk["hbm_gbs"] * 1e9)
    return {"bound": "tensor" if tensor else "hbm", "bytes_per_step": int(lb["total"]), "flops_per_step": int(fl),
            "hbm_gb_per_s": round(gbs, 1), "hbm_frac": round(gbs / pk["hbm_gbs"], 4), "tflops": round(tf, 1),
            "tensor_frac_burst": round(tf / pk["bf16_tflops"], 4),
            "tensor_frac_sustained": round(tf / pk["bf16_tflops_sustained"], 4)}


# ---------------------------------------------------------------------------
def sources_sha16(family: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, family: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, or None when there is none or the kernel's sources changed since
    it was taken (rows: | kernel | workload | bytes | sources sha16 |)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, None
    want = sources_sha16(family)
    for line in open(TRAFFIC_FILE):
        cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload:
            try:
                b = int(cells[2].replace(",", ""))
            except ValueError:
                continue
            return (b if cells[3] == want else None), cells[3]
    return None, None


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


# ---------------------------------------------------------------------------
class _Rows:
    """weights[name][e] as float64 numpy (CPU tensors are converted on access)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        v = self.t[e]
        return v.numpy() if v.dtype == __import__("torch").uint8 else v.float().numpy().astype(np.float64)


def oracle_inputs(w):
    out = {}
    for k, v in w.items():
        v = v.cpu()
        if k in ("w_up", "w_down", "w_up_q", "w_down_q", "w_up_sf", "w_down_sf"):
            out[k] = _Rows(v)
        elif k in ("w_router", "bias"):
            out[k] = v.numpy()
        else:
            out[k] = v.float().numpy().astype(np.float64)
    return out


def time_oracle(shape, w, x, budget_s: float, min_tokens: int = 1):
    """Tokens/s of the oracle on the first rows of x, growing the sample until
    it takes at least budget_s (bounded)."""
    from oracle import moe_oracle as O
    ow = oracle_inputs(w)
    xn = x.float().cpu().numpy().astype(np.float64)
    n = min_tokens
    done_t, done_s = 0, 0.0
    while True:
        rows = xn[done_t % xn.shape[0]:][:n]
        t0 = time.perf_counter()
        O.full_layer(rows, ow, shape.n_experts, shape.top_k, shape.n_group, shape.topk_group,
                     shape.norm_topk_prob, shape.routed_scaling_factor, bf16_points=shape.act_dtype == 1)
        done_s += time.perf_counter() - t0
        done_t += rows.shape[0]
        if done_s >= budget_s or done_t >= xn.shape[0]:
            break
        n = min(2 * n, xn.shape[0] - done_t)
    return done_t / done_s, done_t, done_s


_ONE_THREAD = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import torch
torch.set_num_threads(int(sys.argv[4]))          # the draws may use every core
import bench
from synth import WORKLOADS, make_weights, make_x
shape = WORKLOADS[sys.argv[2]]
w = make_weights(shape, "cpu")
x = make_x(shape, int(sys.argv[3]), "cpu")
torch.set_num_threads(1)
tps, nt, secs = bench.time_oracle(shape, w, x, float(sys.argv[5]))
print(json.dumps({"value": tps, "tokens": nt, "seconds": secs}))
"""


def time_oracle_one_thread(shape, T: int, budget_s: float):
    """The oracle with its BLAS held to one thread, in a fresh interpreter
    (started after this process has used the GPU, so spawned, not forked)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, "-c", _ONE_THREAD, ROOT, shape.name, str(T), str(cpu_cores()),
                            str(budget_s)], capture_output=True, text=True, env=env, timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


# ---------------------------------------------------------------------------
def n_replicas(shape, T: int, requested: int = 0) -> int:
    """Weight replicas that together exceed 4x L2 for the bytes a step reads."""
    if requested:
        return requested
    per_step = layer_bytes(shape, min(T * shape.top_k, shape.n_experts), T)["total"]
    return max(2, min(8, -(-4 * L2_BYTES // per_step) + 1))


class Runner:
    """Device-side timing of the layer through the C ABI binding."""

    def __init__(self, M, dev, world, eager=False):
        import torch
        self.torch, self.M, self.dev, self.world, self.eager = torch, M, dev, world, eager
        self.stream = torch.cuda.current_stream()

    def timed(self, fn, K):
        """Milliseconds of K calls of fn, CUDA events on the launching stream,
        barrier + synchronize on both sides, max over ranks."""
        torch = self.torch
        if self.world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for i in range(K):
            fn(i)
        e1.record(self.stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), self.world, self.dev)
        if self.world > 1:
            torch.distributed.barrier()
        return ms

    def layers(self, shape, n_rep):
        from synth import make_weights
        reps = [make_weights(shape, self.dev, replica=r) for r in range(n_rep)]
        return reps, [self.M.MoELayer(self.M.config_from(shape), w) for w in reps]

    def step_fn(self, layers, x, y, warmup):
        """A step function replaying one CUDA graph of the whole layer per
        weight replica (eager calls with --eager), and kernel launches per step."""
        torch, M = self.torch, self.M
        n_rep = len(layers)
        ws = M.new_workspace(layers[0].cfg, x.shape[0], self.dev)
        for L in layers:
            L._ws = ws

        def eager(i):
            layers[i % n_rep].forward(x, y)

        for i in range(max(warmup, n_rep)):
            eager(i)
        torch.cuda.synchronize()
        if self.eager:
            c0 = M.load().moe_launch_count()
            eager(0)
            return eager, M.load().moe_launch_count() - c0, ws, eager
        graphs, per = [], 0
        for r in range(n_rep):
            g = torch.cuda.CUDAGraph()
            c0 = M.load().moe_launch_count()
            with torch.cuda.graph(g):
                layers[r].forward(x, y)
            per = M.load().moe_launch_count() - c0
            graphs.append(g)
        for i in range(max(3, warmup)):
            graphs[i % n_rep].replay()
        torch.cuda.synchronize()
        return (lambda i: graphs[i % n_rep].replay()), per, ws, eager

    def steps_for(self, fn, target_ms=150.0, lo=20, hi=2000):
        est = self.timed(fn, 5) / 5
        return int(max(lo, min(hi, target_ms / max(est, 1e-3))))

    def active_and_routing(self, layer, x, y, shape):
        T = x.shape[0]
        ids = self.torch.empty((T, shape.top_k), dtype=self.torch.int32, device=self.dev)
        layer.forward(x, y, ids_out=ids)
        ids_np = ids.cpu().numpy()
        return int(np.unique(ids_np).size), routing_stats(ids_np, shape.n_experts), ids


def measure_products(run: Runner, shape, T, layers, x, n_active, pk):
    """The two grouped expert products timed alone on the launching stream
    (moe_experts_up, moe_experts_down), each over >= 20 launches rotating the
    weight replicas; algorithmic bytes / FLOPs per launch over the mean time."""
    torch, M = run.torch, run.M
    cfg = layers[0].cfg
    K_, R = shape.top_k, T * shape.top_k
    ws = M.new_workspace(cfg, T, run.dev)
    ids = torch.empty((T, K_), dtype=torch.int32, device=run.dev)
    topw = torch.empty((T, K_), dtype=torch.float32, device=run.dev)
    x_e = x
    if shape.d_latent:
        x_e = torch.empty((T, shape.d_latent), dtype=x.dtype, device=run.dev)
        M.moe_latent_down(cfg, x, layers[0].weights, x_e, ws)
    w0 = layers[0].weights.tensors
    M.moe_router(cfg, x, w0["w_router"], w0["router_bias"], ids, topw, ws)
    counts = torch.empty(shape.n_experts, dtype=torch.int32, device=run.dev)
    offsets = torch.empty(shape.n_experts + 1, dtype=torch.int32, device=run.dev)
    rt = torch.empty(R, dtype=torch.int32, device=run.dev)
    rs = torch.empty(R, dtype=torch.int32, device=run.dev)
    tsr = torch.empty((T, K_), dtype=torch.int32, device=run.dev)
    xp = torch.empty((R, shape.d_e), dtype=x.dtype, device=run.dev) if T > 64 else None
    M.moe_dispatch(cfg, ids, counts, offsets, rt, rs, tsr, ws, x_e=x_e if xp is not None else None, x_packed=xp)
    h = torch.empty((R, shape.d_expert), dtype=x.dtype, device=run.dev)
    u = torch.empty((R, shape.d_e), dtype=torch.float32, device=run.dev)
    n_rep = len(layers)

    def up(i):
        M.moe_experts_up(cfg, T, rt, offsets, layers[i % n_rep].weights, h, ws, x_e=x_e, x_packed=xp)

    def down(i):
        M.moe_experts_down(cfg, T, h, offsets, rt, rs, topw, layers[i % n_rep].weights, u, ws)

    out = {}
    for name, fn in (("up", up), ("down", down)):
        for i in range(3):
            fn(i)
        k = 40
        c0 = M.load().moe_launch_count()
        ms = run.timed(fn, k) / k
        launches = (M.load().moe_launch_count() - c0) // k
        led = product_ledger(shape, n_active, T, name)
        tensor = led["flops"] / (pk["bf16_tflops"] * 1e12) > led["bytes"] / (pk["hbm_gbs"] * 1e9)
        out[name] = {"ms": ms, "launches": int(launches), "bytes": led["bytes"], "flops": led["flops"],
                     "gbs": led["bytes"] / (ms / 1e3) / 1e9, "tflops": led["flops"] / (ms / 1e3) / 1e12,
                     "tensor": tensor}
    return out


def fp4_tile_rows(rows_per_seg, segs, N, sms=152):
    """Rows per tile of the FP4 grouped GEMM (the library's rule)."""
    bn = 16 if rows_per_seg <= 16 else 32 if rows_per_seg <= 32 else 64
    while bn > 16 and -(-rows_per_seg // bn) * segs * -(-N // 128) < 2 * sms:
        bn -= 16
    return bn


def product_kernel_name(shape, T, which, act_terms=ACT_TERMS):
    """The kernel that runs a grouped expert product at this size (names as the
    profiler prints their template arguments); act_terms: the NVFP4
    activation terms the library uses at T (0: the FP16 path)."""
    if shape.expert_dtype == 2 and act_terms > 0:
        R = T * shape.top_k
        segs = min(shape.n_experts, R)
        N = shape.d_expert if which == "up" else shape.d_e
        bn = fp4_tile_rows(-(-R // segs), segs, N)
        bnmax = 16 if bn <= 16 else 32 if bn <= 32 else 64
        return f"fp4_gemm_kernel<{0 if which == 'up' else 1}, {0 if which == 'up' else 1}, {bnmax}, {act_terms}>", "fp4"
    if T > 64:
        # (the step entry points hand NVFP4 products BF16 rows: FP4A = 1)
        cg = 1 if shape.expert_dtype == 2 else 2
        fp4 = 1 if shape.expert_dtype == 2 else 0
        return f"tc_gemm_kernel<{0 if which == 'up' else 1}, {0 if which == 'up' else 1}, {fp4}, {cg}>", "tc"
    if shape.expert_dtype == 2:
        K = shape.d_e if which == "up" else shape.d_expert
        wpg = 1 if K <= 1536 else 2
        return (f"gemv_nvfp4_bulk_kernel<{0 if which == 'up' else 1}, {0 if which == 'up' else 1}, 0, {wpg}>",
                "gemv")
    K = shape.d_e if which == "up" else shape.d_expert
    N = shape.d_expert if which == "up" else shape.d_e
    fpc = 32 if K <= 2048 and N % 32 == 0 else 16
    return f"gemv_bf16_kernel<{0 if which == 'up' else 1}, {0 if which == 'up' else 1}, {fpc}>", "gemv"


def measure_point(run: Runner, shape, T, layers, warmup):
    """One workload point: the whole layer step timed as graph replays."""
    from synth import make_x
    torch, M = run.torch, run.M
    x = make_x(shape, T, run.dev)
    y = torch.empty_like(x)
    fn, per, ws, _ = run.step_fn(layers, x, y, warmup)
    K = run.steps_for(fn)
    ms = run.timed(fn, K) / K
    err = M.moe_get_device_error(ws)
    n_active, routing, _ = run.active_and_routing(layers[0], x, y, shape)
    return {"ms": ms, "steps": K, "launches_per_step": int(per), "n_active": n_active, "routing": routing,
            "err": err}


VERIFY_ROWS = (1, 2, 4, 8, 16)   # verify-block shapes the block chain is timed at


def dead_groups(run: Runner, shape, T, layer, x):
    """(dead, total) (expert, 16-neuron group) pairs of one step of `layer` on
    x: groups whose h values are zero in every row of the expert, the part of
    W_down the ReLU^2-sparse down projection does not read."""
    torch, M = run.torch, run.M
    from routed_relu_expert_gb300 import _native as N
    cfg = layer.cfg
    layer.forward(x, torch.empty_like(x))
    ws = layer.workspace(T, x.device)
    R, I = T * shape.top_k, shape.d_expert

    def region(r, dt):
        off, nb = M.workspace_region(cfg, T, r)
        return ws[off:off + nb].view(dt)
    h = (region(N.MOE_WS_H, torch.int16).view(R, I).cpu().numpy() & 0x7FFF) != 0
    offs = region(N.MOE_WS_OFFSETS, torch.int32).cpu().numpy()
    dead = tot = 0
    for e in range(shape.n_experts):
        a, b = int(offs[e]), int(offs[e + 1])
        if b > a:
            live = h[a:b].reshape(b - a, I // 16, 16).any(axis=(0, 2))
            dead += int((~live).sum())
            tot += live.size
    return dead, tot


BACKWARD_POINTS = {"nano_decode": (64,), "nano_prefill": (2048, 8192), "super_latent": (256, 4096)}


def backward_flops(shape, T: int) -> int:
    """Algorithmic FLOPs of the backward: two products (input and weight
    gradient) for each forward product of the experts, shared expert and
    latent pair; the router's backward touches only the chosen logits
    (2 T K d for dW_r and again for dx)."""
    de, I, d, S, K = shape.d_e, shape.d_expert, shape.d_model, shape.d_shared, shape.top_k
    fwd = K * 4 * de * I + 4 * d * S + 4 * d * shape.d_latent
    return int(T * (2 * fwd + 4 * K * d))


def measure_backward(run: Runner, shape, T, layers, pk):
    """moe_layer_backward of one forward (its state in the workspace), timed as
    CUDA-graph replays rotating the weight replicas; FLOPs / time against the
    BF16 tensor peak."""
    torch, M = run.torch, run.M
    from synth import make_x
    n = len(layers)
    cfg = layers[0].cfg
    x = make_x(shape, T, run.dev)
    g = torch.Generator(device=run.dev)
    g.manual_seed(77)
    dy = torch.randn((T, shape.d_model), generator=g, device=run.dev).to(torch.bfloat16)
    E, K = shape.n_experts, shape.top_k
    states = []
    for L in layers:
        ws = M.new_workspace(cfg, T, run.dev)
        L._ws = ws
        st = {"ids": torch.empty((T, K), dtype=torch.int32, device=run.dev),
              "topw": torch.empty((T, K), dtype=torch.float32, device=run.dev),
              "scores": torch.empty((T, E), dtype=torch.float32, device=run.dev), "ws": ws}
        L.forward(x, torch.empty_like(x), ids_out=st["ids"], topw_out=st["topw"], scores_out=st["scores"])
        states.append(st)
    z = lambda *sh: torch.zeros(sh, dtype=torch.float32, device=run.dev)
    de, I, d, S, Ld = shape.d_e, shape.d_expert, shape.d_model, shape.d_shared, shape.d_latent
    grads = {"d_router": z(E, d), "d_up": z(E, I, de), "d_down": z(E, de, I)}
    if Ld:
        grads["d_lat_down"], grads["d_lat_up"] = z(Ld, d), z(d, Ld)
    if S:
        grads["d_sh_up"], grads["d_sh_down"] = z(S, d), z(d, S)
    dx = torch.empty((T, d), dtype=torch.float32, device=run.dev)
    bws = M.new_backward_workspace(cfg, T, run.dev)

    def call(i):
        st = states[i % n]
        M.moe_layer_backward(cfg, x, layers[i % n].weights, dy, st["ids"], st["topw"], st["scores"], dx, grads,
                             st["ws"], bws)

    for i in range(n):
        call(i)
    torch.cuda.synchronize()
    graphs = []
    c0 = M.load().moe_launch_count()
    for i in range(n):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            call(i)
        graphs.append(gr)
    per = (M.load().moe_launch_count() - c0) // n

    def fn(i):
        graphs[i % n].replay()

    for i in range(3):
        fn(i)
    K_ = run.steps_for(fn, target_ms=150.0, lo=10, hi=500)
    ms = run.timed(fn, K_) / K_
    fl = backward_flops(shape, T)
    return {"ms_per_backward": round(ms, 5), "tokens_per_s": round(T / (ms / 1e3), 1), "timed_steps": K_,
            "launches_per_backward": int(per), "algorithmic_flops": fl,
            "tflops": round(fl / (ms / 1e3) / 1e12, 2),
            "tensor_frac_bf16_burst": round(fl / (ms / 1e3) / 1e12 / pk["bf16_tflops"], 4),
            "kernel": "gemm_bwd_kernel (mma.sync m16n8k16, 64x64x32 tiles)"}


def measure_sparse_point(run: Runner, shape, T, layers, pk):
    """The layer with the plain and with the group-major (ReLU^2-sparse) down
    weights at one decode size: step times, the dead-group fraction, the bytes
    the sparse step reads, and the down product alone (moe_experts_down)."""
    torch, M = run.torch, run.M
    from synth import make_x
    dense = measure_point(run, shape, T, layers, 3)
    saved = [L.weights for L in layers]
    for L in layers:
        L.enable_sparse_down()
    try:
        sparse = measure_point(run, shape, T, layers, 3)
        x = make_x(shape, T, run.dev)
        dead, tot = dead_groups(run, shape, T, layers[0], x)
        prods = {}
        if shape.expert_dtype != 2:
            sp = measure_products(run, shape, T, layers, x, dense["n_active"], pk)["down"]
            for L, w in zip(layers, saved):
                L.weights = w
            dp = measure_products(run, shape, T, layers, x, dense["n_active"], pk)["down"]
            prods = {"down_dense_ms": round(dp["ms"], 5), "down_sparse_ms": round(sp["ms"], 5)}
    finally:
        for L, w in zip(layers, saved):
            L.weights = w
    elt = 0.5 + 1.0 / 16 if shape.expert_dtype == 2 else 2.0
    skipped = dead * shape.d_e * 16 * elt
    led = layer_bytes(shape, dense["n_active"], T)
    read = led["total"] - skipped
    return {"ms_dense": round(dense["ms"], 5), "ms_sparse": round(sparse["ms"], 5),
            "speedup": round(dense["ms"] / sparse["ms"], 3), "dead_group_frac": round(dead / max(tot, 1), 4),
            "experts_active": dense["n_active"], "bytes_dense": int(led["total"]), "bytes_read_sparse": int(read),
            "hbm_frac_dense_bytes": round(led["total"] / (sparse["ms"] / 1e3) / 1e9 / pk["hbm_gbs"], 4),
            "hbm_frac_bytes_read": round(read / (sparse["ms"] / 1e3) / 1e9 / pk["hbm_gbs"], 4),
            "launches_per_step": sparse["launches_per_step"], "device_error_word": sparse["err"], **prods}


def measure_block_chain(run: Runner, shape, T, layers, warmup):
    """The MoE block (RMSNorm, layer, residual) chained over the weight
    replicas: block r reads block r-1's output, all captured in one CUDA graph;
    ms per block = replay time / number of blocks."""
    from synth import make_norm_weight, make_x
    torch, M = run.torch, run.M
    n = len(layers)
    blocks = [M.MoEBlock(L.cfg, L.weights.tensors, make_norm_weight(shape, run.dev, r), 1e-5)
              for r, L in enumerate(layers)]
    ws = M.new_workspace(blocks[0].cfg, T, run.dev)
    for b in blocks:
        b._ws = ws
    x = make_x(shape, T, run.dev)
    bufs = [torch.empty_like(x) for _ in range(n)]

    def chain():
        cur = x
        for r in range(n):
            blocks[r].forward(cur, bufs[r])
            cur = bufs[r]

    for _ in range(max(1, warmup)):
        chain()
    torch.cuda.synchronize()
    c0 = M.load().moe_launch_count()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    per = M.load().moe_launch_count() - c0
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()

    def fn(i):
        g.replay()

    K = max(10, run.steps_for(fn) // n)
    ms = run.timed(fn, K) / K
    return {"ms_per_block": ms / n, "blocks_per_graph": n, "steps": K, "launches_per_block": per // n,
            "err": M.moe_get_device_error(ws)}


def run_ours(args, rank, world, dev):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import routed_relu_expert_gb300 as M
    from synth import WORKLOADS, make_x

    pk = peaks()
    if args.nvfp4_act_terms >= 0:
        M.set_nvfp4_act_terms(args.nvfp4_act_terms)
    run = Runner(M, dev, world, eager=args.eager)
    shape = WORKLOADS[args.workload]
    T = args.tokens
    n_rep = n_replicas(shape, T, args.replicas)
    reps, layers = run.layers(shape, n_rep)
    x = make_x(shape, T, dev)
    y = torch.empty_like(x)
    fn, per_step_launches, ws, eager_fn = run.step_fn(layers, x, y, args.warmup)
    err = M.moe_get_device_error(ws)

    clocks = ClockSampler(torch.cuda.current_device() if not os.environ.get("CUDA_VISIBLE_DEVICES") else 0)
    clocks.start()
    ms = run.timed(fn, args.steps)
    clk = clocks.stop()
    ms_step = ms / args.steps
    value = job_throughput(T, world, ms_step / 1e3)
    ms_eager = None
    if not args.eager:
        ke = max(10, min(args.steps, 200))
        ms_eager = run.timed(eager_fn, ke) / ke
    n_active, routing, _ = run.active_and_routing(layers[0], x, y, shape)
    prods = measure_products(run, shape, T, layers, x, n_active, pk)

    # end to end through the C ABI with host buffers (copies inside the timed region)
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    x_dev = torch.empty_like(x)
    for i in range(3):
        M.moe_layer_forward_host(layers[0].cfg, xh, x_dev, layers[i % n_rep].weights, y, yh, ws)
    k_e2e = max(10, args.steps // 4)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(k_e2e):
        M.moe_layer_forward_host(layers[0].cfg, xh, x_dev, layers[i % n_rep].weights, y, yh, ws)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / k_e2e, world, dev)

    # every workload at every token count it is defined for
    per_workload, pw_clocks = {}, None
    if args.points != "none":
        names = [n for n in ("tiny_fp32", "nano_decode", "nano_prefill", "super_latent", "super_nvfp4",
                             "nano_decode_relu_sparse", "super_nvfp4_relu_sparse")
                 if args.points in ("all", n)]
        sampler = ClockSampler(torch.cuda.current_device() if not os.environ.get("CUDA_VISIBLE_DEVICES") else 0)
        sampler.start()
        for name in names:
            sh = WORKLOADS[name]
            need = n_replicas(sh, min(sh.tokens))
            if sh is shape and len(layers) >= need:
                lay = layers
            else:
                lay = None
                torch.cuda.empty_cache()
                lay = run.layers(sh, need)[1]
            if sh.relu_sparsity > 0:
                # ReLU^2-sparse decode: the same layer with plain and with group-major down weights
                for Ts in sh.tokens:
                    per_workload[f"{name} T={Ts}"] = measure_sparse_point(run, sh, Ts, lay, pk)
                del lay
                continue
            for Ts in sh.tokens:
                p = measure_point(run, sh, Ts, lay, 3)
                entry = {"ms_per_step": round(p["ms"], 5), "tokens_per_s": round(Ts / (p["ms"] / 1e3), 1),
                         "timed_steps": p["steps"], "weight_replicas": len(lay), "experts_active": p["n_active"],
                         "launches_per_step": p["launches_per_step"], "device_error_word": p["err"]}
                entry.update(roofline_fractions(sh, Ts, p["n_active"], p["ms"], pk))
                entry["routing"] = p["routing"]
                per_workload[f"{name} T={Ts}"] = entry
            if args.backward:
                for Ts in BACKWARD_POINTS.get(name, ()):
                    per_workload[f"{name} backward T={Ts}"] = measure_backward(run, sh, Ts, lay, pk)
            if name in ("nano_decode", "super_latent", "super_nvfp4") and args.blocks:
                # the MoE block (RMSNorm + layer + residual) at the verify shapes,
                # a chain of blocks with independent weights in one graph
                for Ts in VERIFY_ROWS:
                    b = measure_block_chain(run, sh, Ts, lay, 3)
                    ids = torch.empty((Ts, sh.top_k), dtype=torch.int32, device=dev)
                    xb = make_x(sh, Ts, dev)
                    lay[0].forward(xb, torch.empty_like(xb), ids_out=ids)
                    n_act = int(np.unique(ids.cpu().numpy()).size)
                    entry = {"ms_per_block": round(b["ms_per_block"], 5),
                             "tokens_per_s": round(Ts / (b["ms_per_block"] / 1e3), 1),
                             "blocks_per_graph": b["blocks_per_graph"], "timed_replays": b["steps"],
                             "launches_per_block": b["launches_per_block"], "device_error_word": b["err"],
                             "experts_active_first_block": n_act}
                    entry.update(roofline_fractions(sh, Ts, n_act, b["ms_per_block"], pk))
                    per_workload[f"{name} block-chain T={Ts}"] = entry
            if lay is not layers:
                del lay
        pw_clocks = sampler.stop()

    return {
        "value": value, "ms_per_step": ms_step, "n_active": n_active, "clocks": clk,
        "launches": int(per_step_launches) * args.steps, "err": err, "ms_eager": ms_eager,
        "prods": prods, "routing": routing, "peaks": pk, "e2e_s": e2e_s, "n_rep": n_rep, "shape": shape, "T": T,
        "rep_bytes": layer_bytes(shape, shape.n_experts, T)["total"], "per_workload": per_workload,
        "act_terms": M.nvfp4_act_terms_for(T),
        "per_workload_clocks": pw_clocks,
    }


# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, as the reference arm."""
    if rank != 0:
        return None
    from synth import WORKLOADS, make_weights, make_x
    shape = WORKLOADS[args.workload]
    T = args.tokens
    w = make_weights(shape, "cpu")
    x = make_x(shape, T, "cpu")
    budget = 150.0
    per_step = []
    t_start = time.perf_counter()
    steps_done = 0
    for i in range(args.warmup + args.steps):
        tps, nt, secs = time_oracle(shape, w, x[i % T:][:1], 0.0)
        if i >= args.warmup:
            per_step.append(secs / nt)
            steps_done += 1
        if time.perf_counter() - t_start > budget and steps_done >= 1:
            break
    s_per_tok = sum(per_step) / len(per_step)
    value = 1.0 / s_per_tok
    line = {
        "impl": "reference", "metric": "MoE-layer tokens/s", "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": steps_done, "warmup": args.warmup, "ms_per_step": round(s_per_tok * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{shape.name} T={T}", "sample": "one token of the batch per step",
                   "runs_on": "host cores of rank 0 (the oracle uses no GPU)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{steps_done} steps of 1 token ({shape.name}, T={T} batch rows)",
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def roofline_entry(r, shape, T, pk):
    """The dominant kernel: the longer of the two grouped expert products."""
    prods = r["prods"]
    which = max(prods, key=lambda k: prods[k]["ms"])
    p = prods[which]
    kname, family = product_kernel_name(shape, T, which, r["act_terms"])
    workload = f"{shape.name} T={T}"
    traffic, sha = recorded_traffic(kname, workload, family)
    if p["tensor"]:
        roof = {"bound": "tensor", "achieved": round(p["tflops"], 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(p["tflops"] / pk["bf16_tflops"], 4), "algorithmic_flops_per_launch": p["flops"]}
    else:
        roof = {"bound": "hbm", "achieved": round(p["gbs"], 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(p["gbs"] / pk["hbm_gbs"], 4)}
    roof.update({
        "kernel": f"grouped expert {which} projection ({kname}, through moe_experts_{which})",
        "traffic": traffic,
        "traffic_source": (f"ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, profiles/"
                           f"roofline_traffic.md (kernel sources {sha})" if traffic else
                           "no ncu capture of the current kernel sources"),
        "algorithmic_bytes_per_launch": p["bytes"], "avg_launch_ms": round(p["ms"], 5),
        "launches_per_call": p["launches"],
        "peak_source": pk["source"] + (" (cuBLAS bf16 burst)" if p["tensor"] else " (burst copy)"),
        "other_product": {k: {"avg_launch_ms": round(v["ms"], 5), "gb_per_s": round(v["gbs"], 1),
                              "hbm_frac": round(v["gbs"] / pk["hbm_gbs"], 4), "tflops": round(v["tflops"], 1),
                              "algorithmic_bytes_per_launch": v["bytes"]}
                          for k, v in prods.items() if k != which},
    })
    return roof


# ---------------------------------------------------------------------------
def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local)
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    r = run_ours(args, rank, world, dev)
    shape = r["shape"]
    T = r["T"]
    pk = r["peaks"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from synth import make_weights, make_x
        # same workload on the host: weights drawn on the CPU (same recipe), oracle timed on a bounded sample
        wc = make_weights(shape, "cpu")
        xc = make_x(shape, T, "cpu")
        tps, nt, secs = time_oracle(shape, wc, xc, 12.0)
        del wc
        one = time_oracle_one_thread(shape, T, 6.0)
        cpu = {"value": round(tps, 3), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{nt} of the {T} tokens of one {shape.name} batch, {secs:.1f} s",
               "cpu_model": cpu_model(),
               "one_thread": ({"value": round(one["value"], 3), "unit": "tokens/s", "cores": 1,
                               "sample": f"{one['tokens']} tokens, {one['seconds']:.1f} s, BLAS held to one thread"}
                              if one else None)}
    ab = 2 if shape.act_dtype != 0 else 4
    if rank == 0:
        layer = roofline_fractions(shape, T, r["n_active"], r["ms_per_step"], pk)
        layer["bytes_breakdown"] = layer_bytes(shape, r["n_active"], T)
        line = {
            "metric": "MoE-layer tokens/s", "value": round(r["value"], 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(r["ms_per_step"], 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if shape.act_dtype else "f32", "data": "synthetic",
            "config": {"workload": f"{shape.name} T={T}", "tokens_per_step_per_gpu": T,
                       "d_model": shape.d_model, "experts": shape.n_experts, "top_k": shape.top_k,
                       "d_expert": shape.d_expert, "d_shared": shape.d_shared, "d_latent": shape.d_latent,
                       "parallelism": f"replicas x{world}",
                       "l2": f"weights rotate over {r['n_rep']} seeded replicas "
                             f"({r['rep_bytes'] / 1e9:.2f} GB each); no step reads the previous step's weights",
                       "experts_active": r["n_active"], "routing": r["routing"]},
            "roofline": roofline_entry(r, shape, T, pk),
            "layer_roofline": layer,
            "clocks": r["clocks"],
            "gpu_launches": r["launches"],
            "execution": ("CUDA graph of the layer per weight replica, replayed each step"
                          if not args.eager else "eager C-ABI calls"),
            "eager_ms_per_step": round(r["ms_eager"], 5) if r["ms_eager"] else None,
            "device_error_word": r["err"],
            "e2e": {"value": round(world * T / r["e2e_s"], 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": T * shape.d_model * ab, "d2h_bytes_per_step": T * shape.d_model * ab,
                    "api": "moe_layer_forward_host (pinned host x and y)"},
            "cpu_baseline": cpu,
        }
        if r["per_workload"]:
            line["per_workload"] = r["per_workload"]
            line["per_workload_clocks"] = r["per_workload_clocks"]
            line["per_workload_note"] = ("graph replays; bound = the larger ideal time (bytes at the measured copy "
                                         "bandwidth, FLOPs at the burst bf16 peak); tensor fractions against both "
                                         "the burst and the sustained measured bf16 peaks")
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
