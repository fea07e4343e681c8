#!/usr/bin/env python
"""Benchmark of the GB300 block-sparse fused LM-head.

One step = the whole hot path over one batch: active spans built on the device
from the loss mask, the fused forward (target logprob, entropy, lse of the
active tokens) and the backward (d-logits of active tiles, dHidden, dW).  The
default workload is the largest one-GPU configuration, long_256k (T=262144
tokens, H=8192, V=128256, bf16; 32 sequences of 8192 tokens whose first
2458..4096 prompt tokens are inactive, about 60 % active), with its dense-mask
ablation (every token active) timed alongside.  rl_16k (T=16384, H=4096,
V=128256) is timed as a secondary line inside the same JSON.  Metric: active
tokens per second of fwd+bwd, and the fraction of the GB300 dense-bf16 tensor
peak achieved on active FLOPs (8 * Ta * H * V per step: forward logits,
backward recompute, dHidden and dW, each 2 * Ta * H * V).  Every fraction is
given against four denominators: the measured sustained and burst cuBLAS bf16
rates, the nominal dense-bf16 peak (2250 TFLOP/s), and the tensor peak at the
SM clock sampled during that timed region (SMs x 8192 flop/clk x MHz).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long_256k] [--secondary rl_16k|none]
                    [--max-gap 128] [--vocab-chunk 0]

Prints one JSON line on rank 0.  --impl reference times the CPU oracle (fp64
NumPy) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
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

from entropy_active_span_gb300 import workloads as W  # noqa: E402

METRIC = "active tokens/sec fwd+bwd; % of GB300 bf16 tensor peak on active FLOPs"
UNIT = "active tokens/s"
NOMINAL_BF16_TFLOPS = 2250.0     # GB300 dense bf16, nominal
FLOP_PER_CLK_SM = 8192           # dense bf16 tensor flop per SM per clock (tcgen05)
GEMM_KINDS = ("fwd_gemm_tc", "dlogits_gemm_tc", "bwd_chunk_gemm_tc", "dproj_gemm_tc")


def kind_flops(name: str, Ta: int, H: int, V: int, chunk: int) -> float:
    """Algorithmic FLOPs per step of each traced tensor-core launch kind.

    Every contraction is 2 * Ta * H * (vocabulary columns it covers).  The
    backward runs d-logits of chunk 0 alone, then launches that hold dW and
    dHidden of chunk c-1 with the d-logits of chunk c, then dW and dHidden of
    the last chunk."""
    vc = min(chunk, V)
    n = -(-V // vc)
    live = [min(vc, V - c * vc) for c in range(n)]
    u = 2.0 * Ta * H
    if name == "fwd_gemm_tc":
        return u * V
    if name == "dlogits_gemm_tc":
        return u * live[0]
    if name == "bwd_chunk_gemm_tc":
        return u * sum(2 * live[c - 1] + live[c] for c in range(1, n))
    if name == "dproj_gemm_tc":
        return u * 2 * live[-1]
    return 0.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="long_256k", choices=sorted(W.ALL_WORKLOADS))
    p.add_argument("--secondary", default="rl_16k",
                   help="workload timed as a secondary line ('none' to skip)")
    p.add_argument("--ablation-steps", type=int, default=10,
                   help="timed steps of the dense, forward-only and secondary passes "
                        "(at most --steps)")
    p.add_argument("--max-gap", type=int, default=128)
    p.add_argument("--vocab-chunk", type=int, default=0)
    p.add_argument("--rows", choices=("active", "span"), default="active")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-dense", action="store_true")
    p.add_argument("--no-forward-only", action="store_true")
    p.add_argument("--no-e4m3-training", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle sample (cpu_baseline)")
    p.add_argument("--ref-step-seconds", type=float, default=2.0,
                   help="target CPU time of one --impl reference step")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(bf16=d["bf16_tflops"], bf16_sustained=d["bf16_tflops_sustained"],
                    hbm=d["hbm_gbs"], source="measured")
    return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


def fractions(tflops: float, pk: dict, sm_mhz, sms: int, peak_scale: float = 1.0) -> dict:
    """`tflops` against the four denominators.  peak_scale multiplies every
    bf16 peak (2 for e4m3 operands: the nominal dense fp8/bf16 ratio)."""
    out = {"frac_sustained": tflops / (peak_scale * pk["bf16_sustained"]),
           "frac_burst": tflops / (peak_scale * pk["bf16"]),
           "frac_nominal": tflops / (peak_scale * NOMINAL_BF16_TFLOPS),
           "frac_per_clock": None, "per_clock_peak_tflops": None, "sm_mhz_median": sm_mhz}
    if sm_mhz:
        pc = peak_scale * sms * FLOP_PER_CLK_SM * sm_mhz * 1e6 / 1e12
        out["per_clock_peak_tflops"] = pc
        out["frac_per_clock"] = tflops / pc
    return out


def source_sha() -> str:
    """sha256[:16] of the tensor-core kernel sources and of the host code that
    sets their launch shapes and rasters (identifies a capture's build)."""
    import hashlib
    csrc = os.path.join(ROOT, "entropy_active_span_gb300", "csrc")
    src = "".join(open(os.path.join(csrc, f)).read()
                  for f in ("eas_gemm_tc.cu", "eas_device.cuh", "eas_kernels.h", "eas_api.cu"))
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def recorded_traffic(kernel: str, shape: str):
    """DRAM bytes per launch of `kernel` at launch shape `shape` (a workload
    name and its vocabulary chunk, e.g. 'long_256k/c16384') from a committed
    ncu summary, with that summary's file name; (None, None) if there is none.

    Summaries under profiles/ carry lines 'traffic <kernel> <shape> <bytes>
    <sha>', where sha is source_sha() at capture time: a figure taken from
    another kernel build, another launch shape or another workload is never
    reported."""
    import glob
    sha = source_sha()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(path):
            parts = line.split()
            if (len(parts) == 5 and parts[0] == "traffic" and parts[1] == kernel
                    and parts[2] == shape and parts[4] == sha):
                return int(parts[3]), os.path.basename(path)
    return None, None


def aggregate_ranks(ms: float, tokens: float, device) -> tuple[float, float]:
    """Whole-job view of one timed region: the slowest rank's milliseconds and
    the active tokens of all ranks (each rank processes its own batch)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, tokens
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([tokens], dtype=torch.float64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- CPU oracle

def _oracle_rows(inp, rows, Wf):
    """One oracle fwd+bwd over the given active rows; returns seconds."""
    import oracle
    h = W.to_f64(inp["hidden"][rows])
    t0 = time.perf_counter()
    oracle.lmhead_forward_rows(h, Wf, inp["targets"][rows])
    oracle.lmhead_backward_rows_weighted(h, Wf, inp["targets"][rows],
                                         inp["g_logprob"][rows], inp["g_entropy"][rows])
    return time.perf_counter() - t0


def oracle_cost_fit(inp, Wf, rng) -> tuple[float, float]:
    """(a, b) with the oracle's fwd+bwd time for a batch of n active rows
    close to a + b*n on this host: a is the part that does not depend on n
    (its passes over the fp64 copy of W, which dominate small batches), b the
    per-row work.  Fitted from two probe batches of 8 and 64 rows; b = 0 when
    the workload has no more than 8 active rows."""
    act = np.flatnonzero(inp["mask"])

    def probe(n):
        rows = np.sort(rng.choice(act, size=min(n, len(act)), replace=False))
        return len(rows), _oracle_rows(inp, rows, Wf)

    n1, t1 = probe(8)
    n2, t2 = probe(64)
    if n2 <= n1:
        return t1, 0.0
    b = max((t2 - t1) / (n2 - n1), 1e-9)
    return max(t1 - b * n1, 0.0), b


def oracle_sample_size(inp, Wf, target_s: float, rng) -> int:
    """Active rows whose oracle fwd+bwd takes about target_s on this host."""
    n_act = int(np.count_nonzero(inp["mask"]))
    a, b = oracle_cost_fit(inp, Wf, rng)
    if b <= 0.0:
        return n_act
    return int(max(8, min(n_act, (target_s - a) / b)))


def oracle_sample_rate(inp, target_s: float):
    """Times the fp64 oracle's fwd+bwd on a sample of active rows sized to
    about target_s seconds.  Returns (rows, seconds)."""
    act = np.flatnonzero(inp["mask"])
    Wf = W.to_f64(inp["weight"])
    rng = np.random.default_rng(0)
    n = oracle_sample_size(inp, Wf, target_s, rng)
    rows = np.sort(rng.choice(act, size=n, replace=False))
    return n, _oracle_rows(inp, rows, Wf)


def reference_arm(args, rank):
    """--impl reference: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    w = W.ALL_WORKLOADS[args.workload]
    inp = W.make_inputs(w)
    act = np.flatnonzero(inp["mask"])
    Wf = W.to_f64(inp["weight"])
    rng = np.random.default_rng(1)
    # One step = a sample of active rows.  Its target time is --ref-step-seconds
    # or four times the oracle's per-call fixed cost, whichever is larger, so
    # that the per-row work dominates the rate; capped so that all warm-up and
    # timed steps take about three minutes at most.
    a, b = oracle_cost_fit(inp, Wf, rng)
    target = max(args.ref_step_seconds, 4.0 * a)
    target = min(target, max(args.ref_step_seconds, 180.0 / max(1, args.steps + args.warmup)))
    n = len(act) if b <= 0.0 else int(max(8, min(len(act), (target - a) / b)))
    times = []
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(act, size=n, replace=False))
        t = _oracle_rows(inp, rows, Wf)
        if i >= args.warmup:
            times.append(t)
    total = sum(times)
    value = n * len(times) / total
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "T": w.T, "H": w.H, "V": w.V,
                   "active_tokens": int(len(act)), "max_gap": args.max_gap},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} random active rows per step at full H={w.H}, V={w.V}: "
                                   "fp64 forward + d-logits + dHidden + dW contribution"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "clocks.mem,temperature.gpu")

    def __init__(self, uuid: str | None):
        self.proc = None
        self.path = None
        self.window = None      # (start, end) of the timed region, local wall clock
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if uuid:
                cmd += ["-i", uuid]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def wait_first(self, limit_s: float = 5.0):
        """Blocks until nvidia-smi has written its first sample (or limit_s)."""
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < limit_s:
            if self.proc.poll() is not None:
                return
            try:
                if os.path.getsize(self.path) > 0:
                    return
            except OSError:
                return
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None
            parts = parts[1:]
            try:
                r = {"ts": ts, "sm": float(parts[0]), "max": float(parts[1]), "pw": float(parts[2]),
                     "why": {n for n, v in zip(names, parts[4:8]) if v.lower() == "active"}}
                if len(parts) >= 10:
                    r["mem"], r["temp"] = float(parts[8]), float(parts[9])
            except ValueError:
                continue
            rows.append(r)
        os.unlink(self.path)
        if not rows:
            return None
        # samples of the timed region (when there are enough of them), else
        # every sample under load: power above 60 % of the highest draw seen
        # (the sampler starts before the warm-up; its first sample can be idle)
        sel, basis = rows, "all samples"
        if self.window is not None:
            w0, w1 = self.window
            inside = [r for r in rows if r["ts"] is not None and w0 <= r["ts"] <= w1]
            if len(inside) >= 3:
                sel, basis = inside, "timed region"
        top = max(r["pw"] for r in sel)
        loaded = [r for r in sel if r["pw"] >= 0.6 * top] or sel
        reasons = set().union(*(r["why"] for r in loaded))
        out = {"sm_mhz": statistics.median(r["sm"] for r in loaded),
               "sm_max_mhz": rows[-1]["max"], "reasons": sorted(reasons),
               "samples": len(rows), "samples_used": len(loaded),
               "basis": basis + ", under load",
               "power_w_median": statistics.median(r["pw"] for r in loaded)}
        mem = [r["mem"] for r in loaded if "mem" in r]
        if mem:
            out["mem_mhz"] = statistics.median(mem)
            out["temp_c_max"] = max(r["temp"] for r in rows if "temp" in r)
        return out


# -------------------------------------------------------------- our arm

class Problem:
    """Device-resident inputs, outputs and workspaces of one workload."""

    def __init__(self, w, rank, args, dev, eas):
        import torch
        self.w = w
        wr = w.replace(seed=w.seed + 1000 * rank)     # each rank: its own batch (weak scaling)
        self.inp = W.make_inputs(wr)
        self.T, self.H, self.V = w.T, w.H, w.V
        self.Ta = int(self.inp["mask"].sum())
        self.flags = eas.EAS_ROWS_SPAN if args.rows == "span" else eas.EAS_ROWS_ACTIVE
        self.args, self.dev, self.eas = args, dev, eas
        T, H, V = self.T, self.H, self.V

        def d(x):
            t = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
            return t.view(torch.bfloat16) if x.dtype == np.uint16 else t

        inp = self.inp
        self.hidden, self.weight = d(inp["hidden"]), d(inp["weight"])
        self.targets, self.mask = d(inp["targets"]), d(inp["mask"])
        self.glp, self.gh = d(inp["g_logprob"]), d(inp["g_entropy"])
        cap = (T + 1) // 2
        self.spans = torch.empty((cap, 2), dtype=torch.int32, device=dev)
        self.ns = torch.empty(1, dtype=torch.int32, device=dev)
        self.sws = eas.workspace(eas.spans_workspace_size(T), dev)
        self.ws_bytes = eas.lmhead_workspace_size(T, H, V, torch.bfloat16, args.vocab_chunk)
        self.ws = eas.workspace(self.ws_bytes, dev)
        self.lp, self.ent, self.lse = (torch.empty(T, dtype=torch.float32, device=dev)
                                       for _ in range(3))
        self.dh = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((V, H), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def step(self, m=None, marks=None, d_in=None):
        """One pass of the hot path.  marks: three timing events recorded at
        the step's start, after the span build and after the forward (phase
        split of the timed region).  d_in: other device inputs (end to end)."""
        eas, a = self.eas, self.args
        x = d_in or {"hidden": self.hidden, "weight": self.weight, "targets": self.targets,
                     "mask": self.mask if m is None else m, "g_logprob": self.glp,
                     "g_entropy": self.gh}
        if marks is not None:
            marks[0].record(self.stream)
        eas.build_active_spans(x["mask"], a.max_gap, spans=self.spans, num_spans=self.ns,
                               ws=self.sws)
        if marks is not None:
            marks[1].record(self.stream)
        eas.lmhead_fwd(x["hidden"], x["weight"], x["targets"], x["mask"], self.spans, self.ns,
                       self.flags, ws=self.ws, out=(self.lp, self.ent, self.lse))
        if marks is not None:
            marks[2].record(self.stream)
        # the backward reuses the row schedule and packed rows the forward
        # just left in the same workspace
        eas.lmhead_bwd(x["g_logprob"], x["g_entropy"], x["hidden"], x["weight"], x["targets"],
                       x["mask"], self.spans, self.ns, self.lse, self.ent,
                       self.flags | eas.EAS_REUSE_FWD_ROWS, a.vocab_chunk, ws=self.ws,
                       dhidden=self.dh, dweight=self.dw)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return

    import torch
    import torch.distributed as dist

    import entropy_active_span_gb300 as eas

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")

    w = W.ALL_WORKLOADS[args.workload]
    if w.dtype != "bf16":
        raise SystemExit("bench measures the bf16 tensor-core path")
    abl_steps = max(1, min(args.steps, args.ablation_steps))
    chunk = args.vocab_chunk or 16384
    pk = peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    uuid = None
    try:
        uuid = str(props.uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None

    def barrier():
        if world > 1:
            dist.barrier()

    def timed(fn, k, stream, trace=False, marks=None, clocks=True):
        """Warm-up, then k timed calls bracketed by barrier + synchronize;
        returns (ms per call over the slowest rank, trace records, clocks).
        The clock sampler runs from before the warm-up (also under load) to
        the end of the timed calls, so that short regions still get samples."""
        sampler = ClockSampler(uuid) if (clocks and rank == 0) else None
        if sampler:
            sampler.wait_first()
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if trace:
            eas.trace_enable(True)
        t_start = datetime.datetime.now()
        e0.record(stream)
        for i in range(k):
            if marks is None:
                fn()
            else:
                fn(marks=marks[i])
        e1.record(stream)
        torch.cuda.synchronize()
        if sampler:
            sampler.window = (t_start, datetime.datetime.now())
        clk = sampler.stop() if sampler else None
        recs = None
        if trace:
            eas.trace_enable(False)
            recs = eas.trace_read()
        barrier()
        torch.cuda.synchronize()
        ms, _ = aggregate_ranks(e0.elapsed_time(e1), 0.0, dev)
        return ms / k, recs, clk

    def mhz(clk):
        return clk["sm_mhz"] if clk else None

    def rate_block(tflops, clk, peak_scale=1.0):
        f = fractions(tflops, pk, mhz(clk), sms, peak_scale)
        return {"tflops": tflops, "frac_of_peak": f["frac_sustained"],
                "frac_of_burst": f["frac_burst"], "frac_of_nominal": f["frac_nominal"],
                "frac_per_clock": f["frac_per_clock"], "sm_mhz_median": f["sm_mhz_median"],
                "power_w_median": clk.get("power_w_median") if clk else None}

    def breakdown(P, recs, steps, ms, clk):
        """Per-kernel times from the library's event trace, the roofline of
        the dominant tensor-core launch kind, and the launch count."""
        by = {}
        for name, t in recs:
            e = by.setdefault(name, [0, 0.0])
            e[0] += 1
            e[1] += t
        launches = sum(c for n, (c, _) in by.items() if n != "memset")
        gemm = {k: v for k, v in by.items() if k in GEMM_KINDS}
        top = max(gemm.items(), key=lambda kv: kv[1][1]) if gemm else None
        roofline = None
        if top is not None:
            name, (count, tot_ms) = top
            flops_kind = kind_flops(name, P.Ta, P.H, P.V, chunk) * steps
            achieved = flops_kind / (tot_ms / 1000.0) / 1e12
            f = fractions(achieved, pk, mhz(clk), sms)
            shape = f"{P.w.name}/c{chunk}" + ("/span" if args.rows == "span" else "")
            traffic, tsrc = recorded_traffic(name, shape)
            roofline = {"bound": "tensor", "kernel": name, "achieved": achieved,
                        "peak": pk["bf16_sustained"], "unit": "TFLOP/s",
                        "frac": achieved / pk["bf16_sustained"],
                        "peak_kind": f"bf16_tflops_sustained ({pk['source']}): the kernel runs "
                                     "inside a seconds-long, power-capped step",
                        "frac_burst": f["frac_burst"], "peak_burst": pk["bf16"],
                        "frac_nominal": f["frac_nominal"], "peak_nominal": NOMINAL_BF16_TFLOPS,
                        "frac_per_clock": f["frac_per_clock"],
                        "peak_per_clock": f["per_clock_peak_tflops"],
                        "sm_mhz_median": f["sm_mhz_median"],
                        "per_clock_rule": f"{sms} SMs x {FLOP_PER_CLK_SM} flop/clk x median "
                                          "SM MHz sampled during this timed region",
                        "traffic": traffic, "traffic_shape": shape,
                        "traffic_source": (f"profiles/{tsrc}" if tsrc else
                                           "no capture of this kernel build at this launch "
                                           "shape"),
                        "algorithmic_flops_per_launch": flops_kind / count,
                        "launches_per_step": count / steps,
                        "ms_per_launch": tot_ms / count}
        kernels = {k: round(v[1] / steps, 4) for k, v in sorted(by.items())}
        gemm_tflops = {k: round(kind_flops(k, P.Ta, P.H, P.V, chunk) * steps
                                / (v[1] / 1000.0) / 1e12, 1) for k, v in gemm.items()}
        return roofline, kernels, gemm_tflops, launches

    # ---- headline workload: main timed region (device-resident inputs)
    P = Problem(w, rank, args, dev, eas)
    T, H, V, Ta = P.T, P.H, P.V, P.Ta
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    ms, recs, clocks = timed(P.step, args.steps, P.stream, trace=True, marks=marks)
    assert eas.read_device_status(P.ws) == 0 and eas.read_device_status(P.sws) == 0

    _, tokens_all = aggregate_ranks(0.0, float(Ta), dev)
    value = tokens_all / (ms / 1000.0)
    flops_step = 8.0 * Ta * H * V
    tflops = flops_step / (ms / 1000.0) / 1e12
    roofline, kernels, gemm_tflops, launches = breakdown(P, recs, args.steps, ms, clocks)

    # phase split of the same timed steps: span build, forward, backward
    ends = [marks[i + 1][0] for i in range(args.steps - 1)]
    span_ms = statistics.fmean(m[0].elapsed_time(m[1]) for m in marks)
    fwd_ms = statistics.fmean(m[1].elapsed_time(m[2]) for m in marks)
    bwd_ms = statistics.fmean(m[2].elapsed_time(e) for m, e in zip(marks[:-1], ends)) \
        if args.steps > 1 else ms - span_ms - fwd_ms
    u = 2.0 * Ta * H * V
    phases = {"spans_ms": round(span_ms, 4), "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
              "tflops_fwd": u / (fwd_ms / 1000.0) / 1e12,
              "tflops_bwd": 3 * u / (bwd_ms / 1000.0) / 1e12,
              "tflops_6HV": 3 * u / (ms / 1000.0) / 1e12,
              "note": "fwd credits 2*Ta*H*V, bwd 6*Ta*H*V (recompute, dHidden, dW); tflops_6HV "
                      "is the whole step on 6*Ta*H*V, i.e. without crediting the recompute"}

    # ---- end to end: host (pinned) inputs in, results out, through the API.
    # Measured right after the main timed region, before the ablations below,
    # so both headline numbers see the same thermal and power state.
    # Every step copies all of its inputs (hidden, W, targets, mask, g_logprob,
    # g_entropy) from pinned host memory and reads its logprob and entropy
    # back.  The inputs of step i+1 are copied on a second stream while step i
    # computes (two device input buffers), as a training loop prefetches its
    # next batch.
    e2e = None
    if not args.no_e2e:
        names = ("hidden", "weight", "targets", "mask", "g_logprob", "g_entropy")
        host = {k: torch.from_numpy(np.ascontiguousarray(P.inp[k])).pin_memory() for k in names}
        first = {"hidden": P.hidden, "weight": P.weight, "targets": P.targets, "mask": P.mask,
                 "g_logprob": P.glp, "g_entropy": P.gh}
        bufs = [first, {k: torch.empty_like(v) for k, v in first.items()}]
        out_lp = torch.empty(T, dtype=torch.float32).pin_memory()
        out_ent = torch.empty(T, dtype=torch.float32).pin_memory()
        copy_stream = torch.cuda.Stream(dev)
        ready = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        stream = P.stream

        def run_e2e(k, start_event=None):
            for i in range(k):
                b = i % 2
                with torch.cuda.stream(copy_stream):
                    if i == 0 and start_event is not None:
                        copy_stream.wait_event(start_event)
                    if i >= 2:
                        copy_stream.wait_event(free[b])
                    for name in names:
                        bufs[b][name].view(torch.uint8).view(-1).copy_(
                            host[name].view(torch.uint8).view(-1), non_blocking=True)
                    ready[b].record(copy_stream)
                stream.wait_event(ready[b])
                P.step(d_in=bufs[b])
                free[b].record(stream)
                out_lp.copy_(P.lp, non_blocking=True)
                out_ent.copy_(P.ent, non_blocking=True)

        run_e2e(args.warmup)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_e2e(args.steps, start_event=e0)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems, _ = aggregate_ranks(e0.elapsed_time(e1), 0.0, dev)
        ems /= args.steps
        assert np.isfinite(out_lp.numpy()).all()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = 2 * T * 4
        e2e = {"value": tokens_all / (ems / 1000.0), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems,
               "note": "every step copies hidden, W, targets, mask, g_logprob, g_entropy from "
                       "pinned host memory and reads logprob and entropy back; step i+1's "
                       "inputs are copied on a second stream while step i computes; "
                       "gradients stay on the device"}
        del bufs, host

    # ---- dense-mask ablation (same kernels, every token active): the
    # skip-vs-dense comparison of the same workload
    dense = None
    if not args.no_dense:
        ones = torch.ones(T, dtype=torch.uint8, device=dev)
        dms, _, dclk = timed(lambda: P.step(ones), abl_steps, P.stream)
        dense = {"ms_per_step": dms, "steps": abl_steps,
                 "active_tokens_per_s": world * T / (dms / 1000.0),
                 **rate_block(8.0 * T * H * V / (dms / 1000.0) / 1e12, dclk),
                 "skip_speedup": dms / ms,
                 "note": "all T tokens active; ms_per_step / the sparse step's is what skipping "
                         "the inactive tokens saves"}
        del ones

    # ---- forward-only scoring (no lse kept): bf16 operands, and e4m3 operands
    # with W quantised once and hidden quantised inside every step
    fwd_only = None
    if not args.no_forward_only:
        ws_fwd = eas.workspace(eas.lmhead_workspace_size(T, H, V, torch.bfloat16), dev)

        def score_bf16():
            eas.build_active_spans(P.mask, args.max_gap, spans=P.spans, num_spans=P.ns,
                                   ws=P.sws)
            eas.lmhead_fwd(P.hidden, P.weight, P.targets, P.mask, P.spans, P.ns, P.flags,
                           ws=ws_fwd, out=(P.lp, P.ent, P.lse), want_lse=False)

        w8, wsc = eas.quantize_rows_e4m3(P.weight)
        h8 = torch.empty((T, H), dtype=torch.uint8, device=dev)
        hsc = torch.empty(T, dtype=torch.float32, device=dev)
        ws8 = eas.workspace(eas.lmhead_workspace_size(T, H, V, torch.uint8), dev)

        def score_fp8():
            eas.quantize_rows_e4m3(P.hidden, out=h8, scale=hsc)
            eas.build_active_spans(P.mask, args.max_gap, spans=P.spans, num_spans=P.ns,
                                   ws=P.sws)
            eas.lmhead_fwd_fp8(h8, hsc, w8, wsc, P.targets, P.mask, P.spans, P.ns, P.flags,
                               ws=ws8, out=(P.lp, P.ent, P.lse), want_lse=False)

        fwd_only = {}
        for name, fn, scale in (("bf16", score_bf16, 1.0), ("e4m3", score_fp8, 2.0)):
            fms, _, fclk = timed(fn, abl_steps, P.stream)
            tf = 2.0 * Ta * H * V / (fms / 1000.0) / 1e12
            fwd_only[name] = {"ms_per_step": fms, "steps": abl_steps,
                              "active_tokens_per_s": tokens_all / (fms / 1000.0),
                              **rate_block(tf, fclk, scale)}
        fwd_only["e4m3"]["peak_kind"] = ("every bf16 denominator x 2 (nominal dense fp8/bf16 "
                                         "ratio 4.5/2.25)")
        del ws_fwd, ws8, h8, w8

    # ---- training on e4m3 logits: hidden and W quantised every step (W
    # changes every optimizer step), the e4m3 forward, and the e4m3 backward
    # (d-logits recomputed from the e4m3 operands, dHidden and dW in bf16).
    # Two of the four GEMMs run at the e4m3 rate, so the peak for its active
    # FLOPs is 4/3 of every bf16 peak: 8u / (2u/P + 2u/(2P)).
    e4m3_train = None
    if not args.no_e4m3_training and H % 128 == 0:
        h8 = torch.empty((T, H), dtype=torch.uint8, device=dev)
        hsc = torch.empty(T, dtype=torch.float32, device=dev)
        w8 = torch.empty((V, H), dtype=torch.uint8, device=dev)
        wsc = torch.empty(V, dtype=torch.float32, device=dev)
        ws8 = eas.workspace(eas.lmhead_workspace_size(T, H, V, torch.uint8), dev)
        wsb = eas.workspace(eas.lmhead_bwd_fp8_workspace_size(T, H, V, args.vocab_chunk), dev)

        def train_e4m3():
            eas.quantize_rows_e4m3(P.hidden, out=h8, scale=hsc)
            eas.quantize_rows_e4m3(P.weight, out=w8, scale=wsc)
            eas.build_active_spans(P.mask, args.max_gap, spans=P.spans, num_spans=P.ns,
                                   ws=P.sws)
            eas.lmhead_fwd_fp8(h8, hsc, w8, wsc, P.targets, P.mask, P.spans, P.ns, P.flags,
                               ws=ws8, out=(P.lp, P.ent, P.lse))
            eas.lmhead_bwd_fp8(P.glp, P.gh, P.hidden, P.weight, h8, hsc, w8, wsc, P.targets,
                               P.mask, P.spans, P.ns, P.lse, P.ent, P.flags, args.vocab_chunk,
                               ws=wsb, dhidden=P.dh, dweight=P.dw)

        tms, trecs, tclk = timed(train_e4m3, abl_steps, P.stream, trace=True)
        assert eas.read_device_status(wsb) == 0
        tby = {}
        for name, t in trecs:
            tby[name] = tby.get(name, 0.0) + t / abl_steps
        tf = 8.0 * Ta * H * V / (tms / 1000.0) / 1e12
        e4m3_train = {"ms_per_step": tms, "steps": abl_steps,
                      "active_tokens_per_s": tokens_all / (tms / 1000.0),
                      **rate_block(tf, tclk, 4.0 / 3.0),
                      "speedup_vs_bf16_step": ms / tms,
                      "kernels_ms_per_step": {k: round(v, 3) for k, v in sorted(tby.items())},
                      "peak_kind": "every bf16 denominator x 4/3 (forward and recompute at the "
                                   "nominal e4m3 rate, 2x bf16; dHidden and dW in bf16)",
                      "note": "includes quantising hidden and W every step"}
        del ws8, wsb, h8, w8

    cpu_inp = P.inp
    del P

    # ---- secondary workload: the main timed region only
    secondary = None
    if args.secondary != "none" and args.secondary != args.workload:
        s = Problem(W.ALL_WORKLOADS[args.secondary], rank, args, dev, eas)
        sms_, srecs, sclk = timed(s.step, args.steps, s.stream, trace=True)
        assert eas.read_device_status(s.ws) == 0
        _, stok = aggregate_ranks(0.0, float(s.Ta), dev)
        srf, skern, sgemm, _ = breakdown(s, srecs, args.steps, sms_, sclk)
        secondary = {s.w.name: {"value": stok / (sms_ / 1000.0), "unit": UNIT,
                                "ms_per_step": sms_, "steps": args.steps,
                                "config": {"T": s.T, "H": s.H, "V": s.V,
                                           "active_tokens_per_rank": s.Ta},
                                **rate_block(8.0 * s.Ta * s.H * s.V / (sms_ / 1000.0) / 1e12,
                                             sclk),
                                "roofline": srf, "kernels_ms_per_step": skern,
                                "gemm_tflops": sgemm, "clocks": sclk}}
        del s

    # ---- CPU oracle baseline (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, t = oracle_sample_rate(cpu_inp, args.cpu_seconds)
        cpu = {"value": n / t, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{n} random active rows at full H={H}, V={V}: fp64 forward + "
                         f"d-logits + dHidden + dW contribution, {t:.1f} s"}

    if rank == 0:
        rb = rate_block(tflops, clocks)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "T": T, "H": H, "V": V,
                       "active_tokens_per_rank": Ta, "max_gap": args.max_gap,
                       "rows": args.rows, "vocab_chunk": chunk,
                       "workspace_bytes": eas.lmhead_workspace_size(T, H, V, torch.bfloat16,
                                                                    args.vocab_chunk),
                       "parallelism": f"replicas x{world} (independent batches)",
                       "l2": "inputs larger than L2 (W alone is %.2f GB)" % (V * H * 2 / 1e9)},
            "tflops_active": tflops,
            "frac_of_peak": rb["frac_of_peak"],
            "peak_tflops": pk["bf16_sustained"],
            "peak_kind": f"bf16_tflops_sustained ({pk['source']})",
            "frac_of_burst": rb["frac_of_burst"], "peak_burst_tflops": pk["bf16"],
            "frac_of_nominal": rb["frac_of_nominal"], "peak_nominal_tflops": NOMINAL_BF16_TFLOPS,
            "frac_per_clock": rb["frac_per_clock"],
            "roofline": roofline,
            "kernels_ms_per_step": kernels,
            "gemm_tflops": gemm_tflops,
            "phases": phases,
            "gpu_launches": launches,
            "dense_ablation": dense,
            "forward_only": fwd_only,
            "e4m3_training": e4m3_train,
            "secondary": secondary,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
