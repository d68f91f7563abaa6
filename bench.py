#!/usr/bin/env python3
"""Benchmark of one routed MoE layer (route -> bucket -> MXFP4 SwiGLU expert FFN
-> combine) on GB300, through the k3moe C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode] [--impl k3moe|reference]

A step is one whole MoE layer over one batch of synthetic input (the default
workload: 1 token, H=7168, I=2048, 896 experts, top-16, all 21 GB of MXFP4
weights resident in HBM).  Steps rotate over --sets input sets (different
tokens, so different experts) and a 256 MiB buffer is written between timed
steps to flush L2 unless every step already reads more than twice the L2 in
expert weights (then the rotating inputs keep L2 cold; --l2-flush forces the
write).  Prints one JSON line (rank 0).  With N>1 (torchrun) each
rank runs an independent replica on its own GPU (no collectives on the data
path); value = tokens of all ranks / the slowest rank's time.

--impl reference times the float64 C oracle on the host's cores instead."""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import platform
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gen  # noqa: E402

METRIC = "MoE-layer tokens/s + achieved HBM GB/s (decode), FP4 TFLOPS (prefill)"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 126 << 20  # GB300 L2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--config", default="decode", choices=sorted(gen.CONFIGS))
    p.add_argument("--impl", default="k3moe", choices=["k3moe", "reference"])
    p.add_argument("--mode", type=int, default=0, help="expert FFN mode (0 auto, 1 gemv, 3 gemm, 4 w4a4; 2, the retired stream mode, runs gemv)")
    p.add_argument("--sets", type=int, default=64, help="rotating input sets")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle sample budget")
    p.add_argument("--l2-flush", action="store_true",
                   help="write a 256 MiB buffer between timed steps even when the inputs exceed L2")
    p.add_argument("--experts", type=int, default=0,
                   help="override E (small cases for profiling; 0 = the workload's own)")
    p.add_argument("--tokens", type=int, default=0,
                   help="override T (small cases for profiling; 0 = the workload's own)")
    p.add_argument("--no-graphs", dest="graphs", action="store_false",
                   help="time each step as a k3moe_layer call instead of the replay of its captured CUDA graph")
    p.add_argument("--calls-per-graph", type=int, default=8,
                   help="consecutive k3moe_layer calls (one per step, each on its own input set) per captured "
                        "graph, as a model's layers follow each other; 1 = one graph per step")
    p.add_argument("--legs", default="all", choices=["all", "none", "router"],
                   help="also time the other workloads (batch8, speculative-verify batches, prefill, "
                        "skewed, probe) into the line's workloads object; router: the router entry point "
                        "alone on the decode, batch8 and prefill tokens (its own 896 x 7168 router matrix, "
                        "whatever --experts is)")
    p.add_argument("--leg-steps", type=int, default=20, help="timed steps per extra workload (at most --steps)")
    p.add_argument("--leg-cpu-seconds", type=float, default=2.0, help="oracle sample budget per extra workload")
    p.add_argument("--no-stack", action="store_true",
                   help="skip the 92-layer decode over host-resident experts (31 GB of page-locked host memory)")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def slowest_rank_ms(local_ms: float, ws: int, device) -> float:
    """The longest of the ranks' timed regions (every rank calls it; a MAX
    all_reduce of the timing only, no data crosses ranks)."""
    if ws == 1:
        return float(local_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, slowest_ms: float, ws: int) -> float:
    """Units all replicas processed per second of the slowest replica's time."""
    return ws * units_per_rank / (slowest_ms / 1e3)


def host_cpu() -> dict:
    """The host the oracle is timed on: logical CPUs and the CPU model (lscpu's
    "Model name", else /proc/cpuinfo, else the machine type)."""
    model = None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.split(":")[0].strip().lower() == "model name":
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "hardware", "cpu model"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "model": model or platform.machine(), "oracle_threads": 1}


def expert_bytes(s) -> int:
    """Packed MXFP4 bytes of one expert: 3 matrices x H*I x (1/2 code + 1/32 scale)."""
    return 3 * s.H * s.I * 17 // 32


def input_set(name, s, i):
    seed = gen.INPUT_SEED + 1000 * i
    return gen.make_logits(name, s, seed=seed), gen.make_x(s, seed=seed)



def routed_experts(s, logits):
    """Expert ids each token picks (top-k by logit, ties to the lower index).
    Used only to size the reported byte counts."""
    order = np.lexsort((np.broadcast_to(np.arange(s.E), logits.shape), -logits.astype(np.float64)), axis=1)
    return order[:, : s.k]


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = os.path.join(tempfile.gettempdir(), f"k3moe_clocks_{os.getpid()}.csv")
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        """End sampling and keep the samples; returns the summary of [t0, t1]."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        self.rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                self.rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except Exception:
                continue
        os.unlink(self.path)
        return self.window(self.t0, self.t1)

    def window(self, t0, t1):
        """Median SM clock, maximum clock and throttle reasons seen in [t0, t1]."""
        rows = getattr(self, "rows", None)
        if not rows:
            return None
        lo, hi = (t0 or 0) - 1.0, (t1 or 1e18) + 1.0
        sel = [r for r in rows if lo <= r[0] <= hi] or rows
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in sel:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median([r[1] for r in sel])), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": sorted(reasons), "samples": len(sel)}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def kernel_source_hash(files=None) -> str:
    """Hash of the CUDA sources (all of csrc/, or the listed file names in it)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mxfp4_expert_ffn_router_gb300", "csrc")
    paths = sorted(glob.glob(os.path.join(csrc, "*"))) if files is None else [os.path.join(csrc, f) for f in sorted(files)]
    for f in paths:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str):
    """DRAM bytes per launch of the expert FFN from the committed ncu summary, or
    None when the kernels changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    ent = d.get(config)
    if not ent:
        return None
    try:
        now = kernel_source_hash(ent.get("source_files"))
    except OSError:
        return None
    if ent.get("source_hash") != now:
        return None
    return ent.get("dram_bytes_per_call")


# ----------------------------------------------------------------------------- oracle
def oracle_sample(name, s, sets, budget_s, whole_layers=None, a4=False):
    """Time the float64 oracle on whole layers of the first input sets (decode-
    sized workloads) or on a token sample (route+bucket of every token, then the
    FFN and combine token by token), within ~budget_s seconds, one thread."""
    import oracle
    t_tokens, t_sec, n = 0, 0.0, 0
    whole = s.T <= 8 if whole_layers is None else whole_layers
    tag = " (A4 path)" if a4 else ""
    if whole:
        for logits, xbits in sets:
            ids = np.unique(routed_experts(s, logits))
            W = oracle.Weights(s.E, {int(e): tuple(z[0] for z in gen.expert_arrays(s.H, s.I, int(e), int(e) + 1))
                                     for e in ids})
            t = time.perf_counter()
            oracle.moe_layer(s, logits, xbits, W, a4=a4)
            t_sec += time.perf_counter() - t
            t_tokens += s.T
            n += 1
            if t_sec >= budget_s:
                break
        return t_tokens / t_sec, f"{n} whole layers of {s.T} token(s) ({name}){tag}, 1 thread"
    logits, xbits = sets[0]
    t = time.perf_counter()
    idx, w, _ = oracle.route(s, logits)
    oracle.bucket(s, idx)
    t_rb = time.perf_counter() - t
    cache = {}
    for tok in range(s.T):
        for e in idx[tok]:
            if int(e) not in cache:
                cache[int(e)] = tuple(z[0] for z in gen.expert_arrays(s.H, s.I, int(e), int(e) + 1))
        W = oracle.Weights(s.E, {int(e): cache[int(e)] for e in idx[tok]})
        t = time.perf_counter()
        oracle.moe_token(s, xbits[tok], idx[tok], w[tok], W, a4=a4)
        t_sec += time.perf_counter() - t
        n += 1
        if t_sec >= budget_s:
            break
    per_tok = t_sec / n + t_rb / s.T
    return 1.0 / per_tok, (f"route+bucket of all {s.T} tokens plus the FFN+combine of {n} tokens "
                           f"({name}){tag}, 1 thread")


def workload_shape(a):
    s = gen.CONFIGS[a.config]
    if a.experts:
        s = gen.Shape(s.T, s.H, s.I, a.experts, min(s.k, a.experts))
    if a.tokens:
        s = gen.Shape(a.tokens, s.H, s.I, s.E, s.k)
    return s


def run_reference(a):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    s = workload_shape(a)
    nsets = max(1, min(a.sets, a.steps + a.warmup)) if s.T <= 8 else 1
    sets = [input_set(a.config, s, i) for i in range(nsets)]
    import oracle
    cache = {}

    def weights_for(logits):
        ids = [int(e) for e in np.unique(routed_experts(s, logits))]
        for e in ids:
            if e not in cache:
                cache[e] = tuple(z[0] for z in gen.expert_arrays(s.H, s.I, e, e + 1))
        return oracle.Weights(s.E, {e: cache[e] for e in ids})

    def one_step(i):
        logits, xbits = sets[i % len(sets)]
        if s.T <= 8:
            W = weights_for(logits)
            t = time.perf_counter()
            oracle.moe_layer(s, logits, xbits, W)
            return time.perf_counter() - t, s.T
        # prefill-sized: one step = route+bucket of all tokens + FFN of 2 tokens (bounded sample)
        t = time.perf_counter()
        idx, w, _ = oracle.route(s, logits)
        oracle.bucket(s, idx)
        rb = time.perf_counter() - t
        tok = i % s.T
        W = weights_for(logits[tok:tok + 1])
        t = time.perf_counter()
        oracle.moe_token(s, xbits[tok], idx[tok], w[tok], W)
        ffn = time.perf_counter() - t
        return rb / s.T + ffn, 1

    a.l2_mode = l2_policy(a, s, sets)[1]
    for i in range(a.warmup):
        one_step(i)
    tot, toks = 0.0, 0
    for i in range(a.steps):
        dt, nt = one_step(a.warmup + i)
        tot += dt
        toks += nt
    value = toks / tot
    sample = (f"{a.steps} whole layers of {s.T} token(s)" if s.T <= 8 else
              f"{a.steps} steps of route+bucket (amortised per token) plus one token's FFN+combine")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * tot / a.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(a, s),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample, "host": host_cpu()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def l2_policy(a, s, sets):
    """L2 between timed steps.  The inputs rotate over the sets (different routed
    experts); when every set reads more than twice the L2 in expert weights the
    steps need no flush, else a 256 MiB buffer is written between them."""
    min_step_bytes = min(len(np.unique(routed_experts(s, l))) for l, _ in sets) * expert_bytes(s)
    do_flush = a.l2_flush or min_step_bytes < 2 * L2_BYTES
    text = (f"{L2_FLUSH_BYTES >> 20} MiB buffer written between timed steps" if do_flush else
            f"inputs larger than L2: each step reads >= {min_step_bytes / 1e6:.0f} MB of expert weights "
            f"(L2 {L2_BYTES >> 20} MiB), no flush")
    return do_flush, text


def resolved_mode(s, mode):
    """The expert FFN mode the library resolves AUTO (0) to for this shape."""
    if mode == 2:
        return 1  # the retired STREAM mode runs the GEMV kernels
    if mode != 0:
        return mode
    A = s.T * s.k
    gemm_ok = s.H % 128 == 0 and s.I % 128 == 0
    return 3 if gemm_ok and 5 * A >= 4 * s.E else 1


def ffn_kernel_count(s, mode):
    """Kernels one k3moe_expert_ffn call launches."""
    return {1: 4, 3: 6, 4: 6}[resolved_mode(s, mode)]


def layer_kernel_count(s, mode):
    """Kernels one k3moe_layer call launches: the single-block front (route, bucket
    and GEMV prep) + gate/up + h16 + down + combine for small GEMV batches, else
    route + bucket (1 or 3) + the expert FFN's kernels + combine."""
    A = s.T * s.k
    if resolved_mode(s, mode) == 1 and s.T <= 4 and s.E <= 1024 and A <= 128:
        return 5
    return 1 + (1 if A <= 4096 else 3) + ffn_kernel_count(s, mode) + 1


def ffn_kernel_label(s, mode):
    """The kernels of one k3moe_expert_ffn call in the mode the library resolves."""
    mode = resolved_mode(s, mode)
    return {1: "k3moe_expert_ffn, GEMV mode (gemv_prep + gemv_rows gate/up + gemv_h16 + gemv_rows down)",
            3: "k3moe_expert_ffn, GEMM mode (gemm_prep + gemm_sched + rows_to_f16 + ffn_gemm_kernel gate/up "
               "+ rows_to_f16 + ffn_gemm_kernel down; kind::f16 after in-kernel e2m1 dequantisation)",
            4: "k3moe_expert_ffn, W4A4 mode (gemm_prep + gemm_sched + rows_to_mxfp4 + ffn_gemm_mxf4_kernel "
               "gate/up + rows_to_mxfp4 + ffn_gemm_mxf4_kernel down; kind::mxf4)"}[mode]


def tensor_figures(s, mode, ffn_s):
    """Tensor-pipe view of a GEMM-mode expert FFN: FLOPs 2 A (2I H + H I) per call
    and the dense peak of the MMA kind the mode runs: the measured bf16 peak for
    kind::f16 (GEMM mode), times the nominal fp4/bf16 ratio 6 for kind::mxf4
    (W4A4 mode)."""
    mode = resolved_mode(s, mode)
    if mode not in (3, 4):
        return None
    A = s.T * s.k
    flops = 2.0 * A * 3 * s.H * s.I
    peaks = measured_peaks()
    bf16 = float(peaks["bf16_tflops"]) if peaks and "bf16_tflops" in peaks else 1900.0
    ratio = 1.0 if mode == 3 else 6.0
    tf = flops / ffn_s / 1e12
    src = "measured" if peaks else "fallback"
    return {"kind": "f16 (bf16 x bf16 after dequantisation)" if mode == 3 else "mxf4 (e2m1 x e2m1)",
            "tflops": tf, "peak_tflops": bf16 * ratio,
            "peak_source": f"{src} bf16" + ("" if mode == 3 else " x 6 (nominal fp4/bf16)"),
            "frac": tf / (bf16 * ratio), "fp4_dense_frac": tf / (bf16 * 6.0)}


def launch_note(a, calls_per_graph=None):
    if not getattr(a, "graphs", False):
        return "each timed step is one k3moe_layer call"
    g = calls_per_graph if calls_per_graph is not None else max(1, getattr(a, "calls_per_graph", 1))
    if g <= 1:
        return "each timed step replays a CUDA graph holding one captured k3moe_layer call"
    return (f"each timed step is one k3moe_layer call on its own input set; the calls are replayed from CUDA "
            f"graphs holding {g} consecutive calls each (their kernels keep programmatic-launch edges, also "
            f"from one call to the next), timed per graph and divided evenly among its calls")


def workload_config(a, s, name=None):
    name = name or a.config
    return {"workload": f"{name}: T={s.T} tokens, H={s.H}, I={s.I}, E={s.E}, top-{s.k}, "
                        f"MXFP4 experts resident",
            "tokens": s.T, "hidden": s.H, "intermediate": s.I, "experts": s.E, "top_k": s.k,
            "l2": f"{getattr(a, 'l2_mode', 'L2 flushed between steps')}; inputs rotate over {a.sets} sets",
            "launch": launch_note(a, getattr(a, "calls_per_graph_used", None)),
            "parallelism": f"replicas x{a.gpus}"}


def hbm_peak():
    peaks = measured_peaks()
    if peaks and "hbm_gbs" in peaks:
        return float(peaks["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def ffn_bytes_per_call(s, n_unique):
    """Algorithmic bytes of one expert FFN call: the routed experts' MXFP4 codes
    and scales (each read once), x read (bf16), h written and read (bf16), Y
    written (fp32)."""
    A = s.T * s.k
    return n_unique * expert_bytes(s) + s.T * s.H * 2 + A * s.I * 4 + A * s.H * 4


def per_expert_roofline_s(s, counts, mode):
    """Roofline time of one expert FFN call taken expert by expert: each routed
    expert costs the longer of streaming its weights (B_e / HBM peak) and its
    FLOPs (n_e * 6 H I / tensor peak of the mode's MMA kind); the activation, h
    and Y bytes add their HBM time.  GEMV and STREAM run on the CUDA cores: their
    bound is the HBM term alone."""
    bw = hbm_peak()[0] * 1e9
    m = resolved_mode(s, mode)
    peaks = measured_peaks()
    bf16 = float(peaks["bf16_tflops"]) if peaks and "bf16_tflops" in peaks else 1900.0
    f_peak = {3: bf16, 4: 6.0 * bf16}.get(m)
    be = expert_bytes(s)
    t = 0.0
    for n in counts[counts > 0]:
        t_w = be / bw
        t_f = n * 6.0 * s.H * s.I / (f_peak * 1e12) if f_peak else 0.0
        t += max(t_w, t_f)
    A = s.T * s.k
    return t + (s.T * s.H * 2 + A * s.I * 4 + A * s.H * 4) / bw


def mode_name(s, mode):
    return {1: "gemv", 3: "gemm_w4a16", 4: "w4a4"}[resolved_mode(s, mode)]


# ----------------------------------------------------------------------------- GPU arm
class LayerBench:
    """One workload's timed steps through the C ABI: route -> bucket -> expert
    FFN -> combine on the launching stream, inputs rotating over host-generated
    sets that are uploaded once (resident in HBM when the timed region starts)."""

    def __init__(self, a, name, s, mode, W, nsets, dev, flush_always=False):
        import torch

        import mxfp4_expert_ffn_router_gb300 as k3
        self.k3, self.a, self.name, self.s, self.mode, self.W, self.dev = k3, a, name, s, mode, W, dev
        self.sets = [input_set(name, s, i) for i in range(nsets)]
        self.nsets = nsets
        A = s.T * s.k
        self.logits_d = [torch.from_numpy(l).to(dev) for l, _ in self.sets]
        self.x_d = [torch.from_numpy(x.view(np.int16)).to(dev) for _, x in self.sets]
        picks = [routed_experts(s, l) for l, _ in self.sets]
        self.uniq = [len(np.unique(p)) for p in picks]
        self.counts = [np.bincount(p.ravel(), minlength=s.E) for p in picks]
        i32, f32 = torch.int32, torch.float32
        self.st = torch.zeros(1, dtype=i32, device=dev)
        self.idx = torch.empty((s.T, s.k), dtype=i32, device=dev)
        self.w = torch.empty((s.T, s.k), dtype=f32, device=dev)
        self.cnt = torch.empty(s.E, dtype=i32, device=dev)
        self.offsets = torch.empty(s.E + 1, dtype=i32, device=dev)
        self.perm = torch.empty(A, dtype=i32, device=dev)
        self.inv = torch.empty(A, dtype=i32, device=dev)
        self.wsb = torch.empty(max(1, k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_BUCKET)), dtype=torch.uint8,
                               device=dev)
        self.wsf = torch.empty(max(1, k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, mode)),
                               dtype=torch.uint8, device=dev)
        self.wsl = torch.empty(max(1, k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_LAYER, mode)),
                               dtype=torch.uint8, device=dev)
        self.Y = torch.empty((A, s.H), dtype=f32, device=dev)
        self.out = torch.empty((s.T, s.H), dtype=torch.bfloat16, device=dev)
        self.do_flush, self.l2_mode = l2_policy(a, s, self.sets)
        self.do_flush = self.do_flush or flush_always
        self.flush = torch.empty(L2_FLUSH_BYTES if self.do_flush else 1, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream()
        self.launches_per_step = layer_kernel_count(s, mode)

    def layer(self, i, ev=None, phases=False):
        """One step; ev[0] / ev[3] bracket it.  A timed step is one k3moe_layer
        call; with phases the four calls run instead, with ev[1] / ev[2]
        bracketing the expert FFN call (events between calls end the launch
        overlap of the kernels around them, so only the phase pass has them)."""
        k3, s, st, stream = self.k3, self.s, self.st, self.stream
        j = i % self.nsets
        if ev is not None:
            ev[0].record(stream)
        if not phases:
            k3.k3moe_layer(s, self.logits_d[j], self.x_d[j], self.W, self.idx, self.w, self.cnt, self.offsets,
                           self.perm, self.inv, self.Y, self.out, None, self.mode, self.wsl, st, stream=stream)
            if ev is not None:
                ev[3].record(stream)
            return
        k3.k3moe_route(s, self.logits_d[j], self.idx, self.w, st, stream=stream)
        k3.k3moe_bucket(s, self.idx, self.cnt, self.offsets, self.perm, self.inv, self.wsb, st, stream=stream)
        if phases:
            ev[1].record(stream)
        k3.k3moe_expert_ffn(s, self.x_d[j], self.W, self.offsets, self.perm, self.Y, self.mode, self.wsf, st,
                            stream=stream)
        if phases:
            ev[2].record(stream)
        k3.k3moe_combine(s, self.Y, self.w, self.inv, self.out, None, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    def capture(self):
        """One CUDA graph per input set holding that set's k3moe_layer call (its
        kernels keep their programmatic-launch edges in the graph), so that a timed
        step is one graph launch on the host instead of a ctypes call and five
        kernel launches: the host cannot fall behind the GPU."""
        import torch
        k3, s = self.k3, self.s

        def call(j):
            k3.k3moe_layer(s, self.logits_d[j], self.x_d[j], self.W, self.idx, self.w, self.cnt, self.offsets,
                           self.perm, self.inv, self.Y, self.out, None, self.mode, self.wsl, self.st)

        self.graphs = []
        for j in range(self.nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call(j)
            self.graphs.append(g)
        # graphs of G consecutive calls (sets b G .. b G + G - 1), when the sets divide into them and no L2
        # flush has to run between steps
        G = max(1, getattr(self.a, "calls_per_graph", 1))
        self.G = G if G > 1 and self.nsets % G == 0 and not self.do_flush else 1
        self.ggraphs = []
        if self.G > 1:
            for b in range(self.nsets // self.G):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for j in range(b * self.G, (b + 1) * self.G):
                        call(j)
                self.ggraphs.append(g)
        torch.cuda.synchronize()

    def run(self, steps, warmup, clocks=None, barrier=None):
        """Warm-up, then K timed steps (events around each step only; each step a
        graph replay when the graphs were captured), then the same K steps again as
        separate calls with the expert FFN call bracketed (phase split)."""
        import torch
        for i in range(warmup):
            if self.do_flush:
                self.flush.fill_(i & 0xFF)
            self.layer(i)
        torch.cuda.synchronize()
        if int(self.st.item()) != 0:
            raise RuntimeError(f"{self.name}: device status {int(self.st.item())} during warm-up")
        self.graphs = None
        self.G = 1
        if getattr(self.a, "graphs", False):
            self.capture()
            for i in range(warmup):
                self.graphs[i % self.nsets].replay()
            for g in self.ggraphs:
                g.replay()
            torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        pevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        if barrier:
            barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        t_wall = time.perf_counter()
        spans = []  # (first step, steps) per timed launch
        i = 0
        while i < steps:
            if self.do_flush:
                self.flush.fill_((i + 1) & 0xFF)
            j = (warmup + i) % self.nsets
            n = self.G if (self.graphs is not None and self.G > 1 and j % self.G == 0 and i + self.G <= steps) else 1
            if self.graphs is not None:
                ev = evs[i]
                ev[0].record(self.stream)
                if n > 1:
                    self.ggraphs[j // self.G].replay()
                else:
                    self.graphs[j].replay()
                ev[3].record(self.stream)
            else:
                self.layer(warmup + i, evs[i])
            spans.append((i, n))
            i += n
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        for i in range(steps):
            if self.do_flush:
                self.flush.fill_((i + 1) & 0xFF)
            self.layer(warmup + i, pevs[i], phases=True)
        torch.cuda.synchronize()
        t1 = time.time()
        if barrier:
            barrier()
        if int(self.st.item()) != 0:
            raise RuntimeError(f"{self.name}: device status {int(self.st.item())} in the timed steps")
        self.step_ms = np.zeros(steps)
        for i0, n in spans:
            self.step_ms[i0:i0 + n] = evs[i0][0].elapsed_time(evs[i0][3]) / n
        self.calls_per_graph = self.G
        self.rb_ms = np.array([e[0].elapsed_time(e[1]) for e in pevs])
        self.ffn_ms = np.array([e[1].elapsed_time(e[2]) for e in pevs])
        self.comb_ms = np.array([e[2].elapsed_time(e[3]) for e in pevs])
        self.pstep_ms = np.array([e[0].elapsed_time(e[3]) for e in pevs])
        self.steps, self.warmup, self.t_wall, self.t0, self.t1 = steps, warmup, t_wall, t0, t1

    def roofline(self):
        s = self.s
        sel = [(self.warmup + i) % self.nsets for i in range(self.steps)]
        ffn_bytes = np.array([ffn_bytes_per_call(s, self.uniq[j]) for j in sel], dtype=np.float64)
        achieved = float(ffn_bytes.sum() / (self.ffn_ms.sum() / 1e3) / 1e9)
        peak, src = hbm_peak()
        t_roof = np.array([per_expert_roofline_s(s, self.counts[j], self.mode) for j in sel])
        med = float(np.median(self.ffn_ms)) / 1e3
        return {"bound": "hbm", "kernel": ffn_kernel_label(s, self.mode), "achieved": achieved, "peak": peak,
                "peak_source": src, "unit": "GB/s", "frac": achieved / peak,
                "bytes_per_call": float(ffn_bytes.mean()), "ffn_us_median": med * 1e6,
                "per_expert_roofline": {"t_us": float(t_roof.mean() * 1e6),
                                        "frac": float(t_roof.sum() / (self.ffn_ms.sum() / 1e3))},
                "tensor": tensor_figures(s, self.mode, med)}


def run_leg(a, name, mode, W, dev, ws, clocks, cpu_cache, rank):
    """One entry of the line's "workloads" object."""
    s = gen.CONFIGS[name]
    nsets = max(1, min(a.sets, 64 if s.T <= 64 else 4 if s.T <= 4096 else 2))
    lb = LayerBench(a, name, s, mode, W, nsets, dev)
    steps = max(1, min(a.steps, a.leg_steps))
    warmup = max(3, min(a.warmup, 5))
    lb.run(steps, warmup)
    tot_ms = slowest_rank_ms(float(lb.step_ms.sum()), ws, dev)
    ent = {"mode": mode_name(s, mode), "tokens": s.T, "experts": s.E, "top_k": s.k,
           "tokens_per_s": whole_job_rate(s.T * steps, tot_ms, ws), "ms_per_step": tot_ms / steps,
           "steps": steps, "warmup": warmup, "unique_experts_mean": float(np.mean(lb.uniq)),
           "expert_ffn_us_median": float(np.median(lb.ffn_ms) * 1e3),
           "phase_us_median": {"route_bucket": float(np.median(lb.rb_ms) * 1e3),
                               "expert_ffn": float(np.median(lb.ffn_ms) * 1e3),
                               "combine": float(np.median(lb.comb_ms) * 1e3)},
           "roofline": lb.roofline(), "gpu_launches": lb.launches_per_step * steps, "l2": lb.l2_mode,
           "timed_window": (lb.t0, lb.t1)}
    a4 = resolved_mode(s, mode) == 4
    if rank == 0 and not a.no_cpu_baseline:
        key = (name, a4)
        if key not in cpu_cache:
            v, sample = oracle_sample(name, s, lb.sets[:1], a.leg_cpu_seconds, whole_layers=False, a4=a4)
            cpu_cache[key] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample}
        ent["cpu_baseline"] = cpu_cache[key]
    del lb
    return ent


def run_router_leg(a, name, dev, ws, rank):
    """The router entry point alone (scores x . wr^T, then the top-k route) on a
    workload's tokens: tokens/s, and its roofline -- HBM bytes (router matrix,
    x, logits) below 64 tokens (CUDA-core kernel), bf16 tensor FLOPs 2 T E H from
    64 tokens (tcgen05 kernel)."""
    import torch

    import mxfp4_expert_ffn_router_gb300 as k3
    s = gen.CONFIGS[name]
    wr = torch.from_numpy(gen.make_router(s).view(np.int16)).to(dev)
    nsets = 8 if s.T <= 64 else 2
    xs = [torch.from_numpy(gen.make_x(s, seed=gen.INPUT_SEED + 1000 * i).view(np.int16)).to(dev)
          for i in range(nsets)]
    logits = torch.empty((s.T, s.E), dtype=torch.float32, device=dev)
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device=dev)
    w = torch.empty((s.T, s.k), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    steps = max(1, min(a.steps, a.leg_steps))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(3 + steps):
        flush.fill_(i & 0xFF)  # the router matrix (12.8 MB) would otherwise stay in L2
        if i >= 3:
            evs[i - 3][0].record(stream)
        k3.k3moe_router(s, xs[i % nsets], wr, logits, idx, w, st, stream=stream)
        if i >= 3:
            evs[i - 3][1].record(stream)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"router {name}: device status {int(st.item())}")
    ms = np.array([e[0].elapsed_time(e[1]) for e in evs])
    tot = slowest_rank_ms(float(ms.sum()), ws, dev)
    med = float(np.median(ms)) / 1e3
    ent = {"tokens": s.T, "experts": s.E, "hidden": s.H, "top_k": s.k, "steps": steps, "warmup": 3,
           "tokens_per_s": whole_job_rate(s.T * steps, tot, ws), "us_median": med * 1e6,
           "l2": f"{L2_FLUSH_BYTES >> 20} MiB buffer written between timed calls"}
    if s.T < 64:
        by = s.E * s.H * 2 + s.T * s.H * 2 + s.T * s.E * 4
        peak, src = hbm_peak()
        ent["roofline"] = {"bound": "hbm", "kernel": "router_gemv_kernel + route_kernel", "bytes_per_call": by,
                           "achieved": by / med / 1e9, "peak": peak, "peak_source": src, "unit": "GB/s",
                           "frac": by / med / 1e9 / peak}
    else:
        fl = 2.0 * s.T * s.E * s.H
        peaks = measured_peaks()
        bf16 = float(peaks["bf16_tflops"]) if peaks and "bf16_tflops" in peaks else 1900.0
        ent["roofline"] = {"bound": "tensor", "kernel": "router_gemm_kernel (tcgen05 kind::f16, bf16) + route_kernel",
                           "flops_per_call": fl, "achieved": fl / med / 1e12, "peak": bf16,
                           "peak_source": "measured bf16" if peaks else "fallback", "unit": "TFLOP/s",
                           "frac": fl / med / 1e12 / bf16}
    return ent


def run_stack_leg(a, dev, ws, budgets_gb=(8, 32, 64, 128), layers=92, physical=2, warm_tokens=6,
                  timed_tokens=4):
    """The pages' per-token expert workload: 92 MoE layers (I = 1536, 896 experts,
    top-16, one token) whose experts live in page-locked host memory, through one
    LRU arena of expert slots in HBM, at several arena budgets.  Per layer and
    token the inputs are drawn from the generator (logits N(0, sigma 2), x N(0,1);
    the attention that would produce them is not part of the path).  Reports
    seconds per token, bytes read from host memory per token, raw and true
    resident hit rates, and the host-to-arena copy rate."""
    import torch

    from mxfp4_expert_ffn_router_gb300.stack import CachedMoEStack, HostExpertStore
    s = gen.Shape(1, 7168, 1536, 896, 16)

    def fill(p, ptrs):
        gen.fill_experts(s.H, s.I, 0, s.E, *ptrs, seed=gen.WEIGHT_SEED + p)

    t0 = time.perf_counter()
    store = HostExpertStore(s.H, s.I, s.E, physical, layers, fill, device=dev)
    setup_s = time.perf_counter() - t0
    # distinct inputs for every (token, layer): no routing repeats across tokens
    n_in = (warm_tokens + timed_tokens) * layers
    lg_all = gen.normal_f32(500, gen.stream(gen.KIND_LOGITS), n_in * s.E, 2.0).reshape(n_in, 1, s.E)
    x_all = gen.normal_bf16_bits(500, gen.stream(gen.KIND_X), n_in * s.H).reshape(n_in, 1, s.H)
    lg_d = torch.from_numpy(lg_all).to(dev)
    x_d = torch.from_numpy(x_all.view(np.int16)).to(dev)
    inputs = [(lg_d[i], x_d[i]) for i in range(n_in)]
    out = torch.empty((1, s.H), dtype=torch.bfloat16, device=dev)
    be = expert_bytes(s)
    # reference for the arena fill: the copy engines' host -> HBM rate on 2 GB of the store
    src = store.arrays[0].view(-1)[: 2 << 30]
    dst = torch.empty(src.numel(), dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dst.copy_(src, non_blocking=True)
    e0.record()
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    e1.record()
    e1.synchronize()
    dma_gbs = 3 * src.numel() / (e0.elapsed_time(e1) / 1e3) / 1e9
    del dst
    res = {"layers": layers, "physical_layers_in_host_memory": physical, "host_to_hbm_dma_gbs": dma_gbs,
           "host_store_gb": store.bytes / 1e9, "host_store_setup_s": setup_s,
           "expert_bytes": be, "requests_per_token": layers * s.k, "budgets": {}}
    stream = torch.cuda.current_stream()
    for gb in budgets_gb:
        slots = int(gb * 1e9 // be)
        stack = CachedMoEStack(s, store, slots, device=dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tok_ms = []
        for tkn in range(warm_tokens + timed_tokens):
            if tkn == warm_tokens:
                torch.cuda.synchronize()
                before = stack.counters()
            ev0.record(stream)
            for l in range(layers):
                lg, x = inputs[tkn * layers + l]
                stack.layer(l, lg, x, out, stream=stream)
            ev1.record(stream)
            ev1.synchronize()
            if tkn >= warm_tokens:
                tok_ms.append(ev0.elapsed_time(ev1))
        if int(stack.status.item()) != 0:
            raise RuntimeError(f"stack: device status {int(stack.status.item())}")
        after = stack.counters()
        d = {key: after[key] - before[key] for key in after}
        tot_ms = slowest_rank_ms(float(sum(tok_ms)), ws, dev)
        res["budgets"][f"{gb}GB"] = {
            "slots": slots, "s_per_token": tot_ms / 1e3 / timed_tokens,
            "tokens_per_s": whole_job_rate(timed_tokens, tot_ms, ws),
            "bytes_from_host_per_token": d["bytes_from_host"] / timed_tokens,
            "requests_per_token": d["requests"] / timed_tokens,
            "raw_hit_rate": d["raw_hits"] / max(1, d["requests"]),
            "true_resident_hit_rate": d["true_resident_hits"] / max(1, d["requests"]),
            "host_to_hbm_gbs": d["bytes_from_host"] / (tot_ms / 1e3) / 1e9,
            "warm_tokens": warm_tokens, "timed_tokens": timed_tokens}
        del stack
        torch.cuda.empty_cache()
    del store
    return res


LEGS = [("batch8", 0), ("batch8", 3), ("spec2", 1), ("spec2", 3), ("spec4", 1), ("spec4", 3),
        ("spec12", 1), ("spec12", 3), ("spec16", 1), ("spec16", 3),
        ("prefill", 0), ("prefill", 4), ("skewed", 0), ("skewed", 4), ("probe", 4), ("probe", 3)]


def run_gpu(a):
    import torch

    import mxfp4_expert_ffn_router_gb300 as k3
    from gen.device import DeviceExperts
    from mxfp4_expert_ffn_router_gb300 import build as k3build

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        k3build.build()
    if ws > 1:
        dist.barrier()
    barrier = dist.barrier if ws > 1 else None
    s = workload_shape(a)
    nsets = max(1, a.sets)
    experts = DeviceExperts(s.H, s.I, s.E, device=dev)
    W = k3.Weights.from_stacked(*experts.tensors)
    lb = LayerBench(a, a.config, s, a.mode, W, nsets, dev)
    a.l2_mode = lb.l2_mode
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    lb.run(a.steps, a.warmup, barrier=barrier)
    a.calls_per_graph_used = getattr(lb, "calls_per_graph", 1)
    clocks.t0, clocks.t1 = lb.t0, lb.t1
    tot_ms = slowest_rank_ms(float(lb.step_ms.sum()), ws, dev)
    value = whole_job_rate(s.T * a.steps, tot_ms, ws)
    roof = lb.roofline()
    roof["traffic"] = recorded_traffic(a.config)
    head_launches = lb.launches_per_step * a.steps
    head_step_us = {"median": float(np.median(lb.step_ms) * 1e3), "min": float(lb.step_ms.min() * 1e3),
                    "max": float(lb.step_ms.max() * 1e3)}
    head_phases = {"route_bucket": float(np.median(lb.rb_ms) * 1e3),
                   "expert_ffn": float(np.median(lb.ffn_ms) * 1e3),
                   "combine": float(np.median(lb.comb_ms) * 1e3),
                   "step_with_phase_events": float(np.median(lb.pstep_ms) * 1e3),
                   "note": "a second pass of the same K steps with events around the "
                           "expert FFN call; value and step_us come from the first pass"}
    head_wall = lb.t_wall
    head_sets = lb.sets

    # ------------------------------------------------------------- end to end (host buffers)
    e2e = None
    if not a.no_e2e:
        lg_h = [torch.from_numpy(l).pin_memory() for l, _ in lb.sets]
        x_h = [torch.from_numpy(x.view(np.int16)).pin_memory() for _, x in lb.sets]
        out_h = torch.empty((s.T, s.H), dtype=torch.bfloat16).pin_memory()
        lg_dev = torch.empty_like(lb.logits_d[0])
        x_dev = torch.empty_like(lb.x_d[0])
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, min(a.steps, 500))
        stream = lb.stream

        def e2e_step(j, strm):
            lg_dev.copy_(lg_h[j], non_blocking=True)
            x_dev.copy_(x_h[j], non_blocking=True)
            k3.k3moe_layer(s, lg_dev, x_dev, W, lb.idx, lb.w, lb.cnt, lb.offsets, lb.perm, lb.inv, lb.Y, lb.out,
                           None, a.mode, lb.wsl, lb.st, stream=strm)
            out_h.copy_(lb.out, non_blocking=True)

        # one CUDA graph per input set holding the step's two host-to-device copies,
        # its k3moe_layer call and the device-to-host copy of out: one launch per step
        # from the host; every step is still synchronised before the next is issued
        e2e_graphs = None
        if getattr(a, "graphs", False):
            e2e_graphs = []
            for j in range(nsets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    e2e_step(j, None)
                e2e_graphs.append(g)
            torch.cuda.synchronize()
        tot = 0.0
        for i in range(n_e2e + 3):
            j = i % nsets
            if lb.do_flush:
                lb.flush.fill_(i & 0xFF)
            ev0.record(stream)
            if e2e_graphs is not None:
                with torch.cuda.stream(stream):
                    e2e_graphs[j].replay()
            else:
                e2e_step(j, stream)
            ev1.record(stream)
            ev1.synchronize()
            if i >= 3:
                tot += ev0.elapsed_time(ev1)
        e2e_val = whole_job_rate(s.T * n_e2e, slowest_rank_ms(tot, ws, dev), ws)
        e2e = {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": s.T * s.E * 4 + s.T * s.H * 2,
               "d2h_bytes_per_step": s.T * s.H * 2, "steps": n_e2e,
               "launch": ("each step replays a CUDA graph of its two host-to-device copies, the k3moe_layer call "
                          "and the device-to-host copy of out, and is synchronised before the next step is issued"
                          if e2e_graphs is not None else
                          "each step: two host-to-device copies, the k3moe_layer call and the device-to-host copy of "
                          "out, synchronised before the next step is issued")}

    # ------------------------------------------------------------- the other workloads
    workloads = None
    legs = [] if a.legs != "all" or a.experts or a.tokens else LEGS
    if legs and (s.H, s.I, s.E) != (7168, 2048, 896):
        legs = []
    if legs:
        del lb
        torch.cuda.empty_cache()
        workloads = {}
        cpu_cache = {}
        for name, mode in legs:
            ls = gen.CONFIGS[name]
            Wl = W if ls.E == s.E else k3.Weights.from_stacked(*[t[: ls.E] for t in experts.tensors])
            key = f"{name}/{mode_name(ls, mode)}"
            workloads[key] = run_leg(a, name, mode, Wl, dev, ws, clocks, cpu_cache, rank)
            torch.cuda.empty_cache()
        for name in ("decode", "batch8", "prefill"):
            workloads[f"router/{name}"] = run_router_leg(a, name, dev, ws, rank)
        if not a.no_stack:
            del W, Wl, experts
            torch.cuda.empty_cache()
            workloads["stack92/decode_i1536_host_experts"] = run_stack_leg(a, dev, ws)
    if a.legs == "router":
        workloads = {f"router/{name}": run_router_leg(a, name, dev, ws, rank) for name in ("decode", "batch8", "prefill")}
    time.sleep(0.2)
    clk = clocks.stop()
    for ent in (workloads or {}).values():  # clocks seen during each workload's timed steps
        if "timed_window" in ent:
            ent["clocks"] = clocks.window(*ent.pop("timed_window"))

    cpu = None
    if rank == 0 and not a.no_cpu_baseline:
        v, sample = oracle_sample(a.config, s, head_sets, a.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample, "host": host_cpu()}
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": a.steps,
                "warmup": a.warmup, "ms_per_step": tot_ms / a.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "e2m1*bf16->f32",
                "data": "synthetic", "config": workload_config(a, s),
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "clocks": clk,
                "gpu_launches": head_launches, "step_us": head_step_us, "phase_us_median": head_phases,
                "wall_s_timed_region": head_wall, "workloads": workloads,
                "clocks_all_timed_regions": clocks.window(None, None)}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_gpu(a)


if __name__ == "__main__":
    main()
