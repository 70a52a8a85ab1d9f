#!/usr/bin/env python3
"""Throughput of the sparse MoE feed-forward layer on B300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

A step is one pass of the whole layer (router/top-2/softmax -> grouping -> expert
up-projection with SwiGLU -> down-projection -> gate-weighted combine; for the stacked
workload, RMSNorm + layer + residual for each of its 4 layers) over one batch of seeded
synthetic input, through the C ABI of libmoe.so.  Inputs are resident in HBM when the
timed region starts; the expert weights (2.82 GB per layer) are larger than the 126 MB
L2, so no flush is needed between steps.  `value` is tokens/s of the whole job (all ranks).

Default workload: the largest single-layer configuration, 16384 tokens with skewed routing
(d=4096, f=14336, 8 experts, top-2; tensor-core bound).  The same line carries, under
"decode", the 32-token decode batch (HBM bound) measured in the same process the same way.
`--impl reference` times the fp64 CPU oracle instead (the slow reference arm), on a bounded
sample of the same workload.
Under torchrun each rank runs an independent replica on its own GPU (the layer needs no
exchange between ranks), timed with a barrier on both sides and the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MoE-layer tokens/s and TFLOP/s (or HBM GB/s) on 1 B300 vs roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", type=int, default=4, choices=sorted(workloads.WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-decode", action="store_true",
                   help="forward pass of a workload other than the decode batch: do not add the "
                        "decode batch's measurement under \"decode\"")
    p.add_argument("--pass", dest="which", default="forward",
                   choices=["forward", "backward", "train", "attention", "decoder"],
                   help="time the layer's forward (default), its backward (moe_layer_backward), "
                        "a training step (moe_layer_forward_train + moe_layer_backward_saved), or "
                        "the causal grouped-query attention of the layer's other sub-block, or one "
                        "whole decoder layer (attention sub-block + MoE sub-block)")
    p.add_argument("--ep", action="store_true",
                   help="expert parallelism: the N ranks hold n/N experts each and exchange token "
                        "rows by NCCL all-to-all (sparse_mixture_experts_56_b300.ep); every rank "
                        "routes T tokens of its own")
    p.add_argument("--seq-len", type=int, default=0,
                   help="--pass attention: tokens per sequence (0: the workload's T)")
    return p.parse_args()


# ----------------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU)
# ----------------------------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as td
            td.init_process_group(backend=backend)
            self.pg = td

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------------------------
# clocks during the timed region (NVML reads only)
# ----------------------------------------------------------------------------------------------
REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
           0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
           0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    """SM clock and clock-event reasons sampled every few ms during the timed region, through
    NVML when the Python bindings are present, else through `nvidia-smi -lms`."""

    def __init__(self, torch_dev):
        import torch
        self.samples = []
        self.mode = None
        self.max_mhz = None
        self._stop = threading.Event()
        self._thr = None
        self._proc = None
        uuid = str(torch.cuda.get_device_properties(torch_dev).uuid)
        self.uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        try:
            import pynvml
            pynvml.nvmlInit()
            self.h = pynvml.nvmlDeviceGetHandleByUUID(self.uuid)
            self.nv = pynvml
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception:
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "nvidia-smi"

    def _run_nvml(self):
        nv = self.nv
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            try:
                self.samples.append((nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM), int(fn(self.h))))
            except Exception:
                pass
            time.sleep(0.002)

    def _run_smi(self):
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            try:
                mhz, mx, reasons = float(parts[0]), float(parts[1]), int(parts[2], 16)
            except (ValueError, IndexError):
                continue
            self.max_mhz = mx
            self.samples.append((mhz, reasons))

    def start(self):
        if self.mode == "nvml":
            self._thr = threading.Thread(target=self._run_nvml, daemon=True)
        elif self.mode == "nvidia-smi":
            import subprocess
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid,
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._thr = threading.Thread(target=self._run_smi, daemon=True)
            time.sleep(1.0)   # nvidia-smi's start-up is over before the timed region
        if self._thr:
            self._thr.start()

    def stop(self):
        self._stop.set()
        if self._proc:
            self._proc.terminate()
            self._proc.wait()
        if self._thr:
            self._thr.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": self.mode}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        names = [n for b, n in REASONS.items() if bits & b and n != "gpu_idle"]
        return {"sm_mhz": float(statistics.median(mhz)),
                "sm_max_mhz": float(self.max_mhz) if self.max_mhz else None,
                "reasons": names, "samples": len(self.samples), "source": self.mode}


def tensor_peak(pk, clocks):
    """The bf16 denominator of a tensor-bound line: cuBLAS's burst figure (a GEMM timed
    alone at full clock), the right peak for a layer step of a few milliseconds.  The
    sustained figure (cuBLAS held for seconds at the power cap) is returned beside it, so
    that lines can also say how they compare with cuBLAS under the cap."""
    burst = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sus = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    kind = "burst" + (" (the power cap was active in the timed region)" if capped else "")
    return burst, kind, burst, sus


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    source of the kernel (profiles/<kernel>__<workload>.md holds 'traffic_bytes_per_launch:'
    and 'source_sha256:' lines, and optionally 'source_file:', the kernel's file under csrc/,
    grouped_tc.cu if absent); None otherwise."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip().lstrip("-* ").strip("`")] = v.strip().strip("`")
    name = os.path.basename(fields.get("source_file", "grouped_tc.cu"))
    src = os.path.join(ROOT, "sparse_mixture_experts_56_b300", "csrc", name)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    if fields.get("source_sha256") != sha:
        return None
    try:
        return float(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------------------------
# inputs
# ----------------------------------------------------------------------------------------------
def host_inputs(w, seed):
    """Per layer: dict of stored tensors (bf16 bit patterns or fp32) + the activations."""
    layers = [workloads.make_inputs(w, seed=seed, layer=l, tensors=("wg", "w1", "w3", "w2"))
              for l in range(w.layers)]
    x = workloads.make_inputs(w, seed=seed, tensors=("x",))["x"]
    bias = workloads.logit_bias_vector(w.n) if w.skew_bias else None
    return x, layers, bias


def to_dev(a, w, dev):
    import torch
    if w.dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


# ----------------------------------------------------------------------------------------------
# the oracle arm (CPU)
# ----------------------------------------------------------------------------------------------
def oracle_prepare(w, x, layers, bias):
    """Expands the stored inputs to float64 once (input preparation, outside any timing)."""
    xf = workloads.as_f32(x, w).astype(np.float64)
    lf = []
    for L in layers:
        lf.append({k: workloads.as_f32(L[k], w).astype(np.float64) for k in ("wg", "w1", "w3", "w2")})
    return xf, lf, bias


def oracle_step(w, xf, lf, bias, tokens):
    import oracle
    if w.layers == 1:
        return oracle.moe_layer(xf, lf[0]["wg"], lf[0]["w1"], lf[0]["w3"], lf[0]["w2"], w.k, bias,
                                tokens=tokens)
    h = xf[tokens]
    for L in lf:
        h = oracle.stacked_layer(h, L["wg"], L["w1"], L["w3"], L["w2"], w.k, w.rms_eps)
    return h


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample_tokens(w, budget_tokens: int, rng):
    return np.sort(rng.choice(w.T, size=min(w.T, budget_tokens), replace=False))


def run_cpu_baseline(w, xf, lf, bias, target_s=10.0):
    """Times the oracle on a bounded sample of the workload's tokens."""
    rng = np.random.default_rng(1234)
    n_tok = {1: 64, 2: 32, 3: 256, 4: 256, 5: 64}.get(w.wid, 64)
    tokens = oracle_sample_tokens(w, n_tok, rng)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_step(w, xf, lf, bias, tokens)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s or (w.wid != 1 and reps >= 1 and el * (reps + 1) / reps > 30):
            break
    return {"value": reps * len(tokens) / el, "unit": "tokens/s", "cores": cpu_cores(),
            "kind": "oracle",
            "sample": f"{len(tokens)} of the {w.T} tokens x {reps} repetition(s), fp64 NumPy "
                      f"({el:.1f} s); inputs expanded to float64 before timing"}


def reference_arm(args, w, dist):
    if dist.rank != 0:
        return
    x, layers, bias = host_inputs(w, args.seed)
    xf, lf, _ = oracle_prepare(w, x, layers, bias)
    del layers
    rng = np.random.default_rng(4321)
    per_step = w.T if w.wid == 1 else 1
    for _ in range(args.warmup):
        oracle_step(w, xf, lf, bias, oracle_sample_tokens(w, per_step, rng))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, xf, lf, bias, oracle_sample_tokens(w, per_step, rng))
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "d_model": w.d, "d_ff": w.f, "n_experts": w.n,
                       "top_k": w.k, "layers": w.layers, "tokens_per_step": per_step},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} token(s) of the {w.T}-token batch per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------------
def ours_arm(args, w, dist):
    import torch
    import sparse_mixture_experts_56_b300 as moe

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    moe._native.lib()
    line = forward_line(args, w, dist, dev, with_cpu=True)
    if w.wid != 2 and not args.no_decode:
        # the HBM-bound decode batch, measured the same way (its own inputs, timed region,
        # clocks, roofline and end-to-end figure), carried in the same line; a decode step is
        # half a millisecond, so it is timed over at least 400 steps (the number is reported)
        torch.cuda.empty_cache()
        dargs = argparse.Namespace(**vars(args))
        dargs.steps = max(args.steps, 400)
        dec = forward_line(dargs, workloads.workload(2), dist, dev, with_cpu=False)
        line["decode"] = {k: dec[k] for k in ("value", "unit", "steps", "ms_per_step", "tflops",
                                              "roofline", "e2e", "clocks", "gpu_launches", "config",
                                              "expert_counts") if k in dec}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def forward_line(args, w, dist, dev, with_cpu):
    """Times `args.steps` layer steps of workload `w` and returns the JSON line as a dict."""
    import torch
    import sparse_mixture_experts_56_b300 as moe

    x_h, layers_h, bias_h = host_inputs(w, args.seed)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    esz = 2 if w.dtype == "bf16" else 4
    x = to_dev(x_h, w, dev)
    layers = [{k: to_dev(L[k], w, dev) for k in ("wg", "w1", "w3", "w2")} for L in layers_h]
    bias = torch.from_numpy(bias_h).to(dev) if bias_h is not None else None
    T, d, f, n, k = w.T, w.d, w.f, w.n, w.k
    A = T * k
    ws = moe.workspace(T, d, f, n, k, tdt, dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gw = torch.empty((T, k), dtype=torch.float32, device=dev)
    off = torch.empty(n + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(A, dtype=torch.int32, device=dev)
    inv = torch.empty(A, dtype=torch.int32, device=dev)
    hbuf = torch.empty((A, f), dtype=tdt, device=dev)
    yp = torch.empty((A, d), dtype=tdt, device=dev)
    hs = [x.clone() for _ in range(2)]
    xn = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    def layer(inp, L, out, residual, marks=None):
        moe.moe_router_topk(inp, L["wg"], k, bias, topk_idx=idx, topk_w=gw)
        moe.moe_permute(idx, n, ws, expert_offsets=off, perm=perm, inv_perm=inv)
        if marks:
            marks[0].record(stream)
        moe.moe_expert_up(inp, perm, off, L["w1"], L["w3"], k, ws, h=hbuf)
        if marks:
            marks[1].record(stream)
        moe.moe_expert_down(hbuf, off, L["w2"], k, ws, y_perm=yp)
        if marks:
            marks[2].record(stream)
        moe.moe_combine(yp, inv, gw, residual, y=out)

    def step(marks=None):
        if w.layers == 1:
            layer(x, layers[0], hs[0], None, marks)
            return
        h_in = x
        for li, L in enumerate(layers):
            moe.moe_rmsnorm(h_in, w.rms_eps, x=xn)
            out = hs[li % 2]
            layer(xn, L, out, h_in, marks if li == 0 else None)
            h_in = out

    launches_per_layer = 1 + (1 if A <= 32768 else 3) + 1 + 1 + 1 + 1
    launches_per_step = w.layers * (launches_per_layer + (1 if w.layers > 1 else 0))

    for _ in range(max(3, args.warmup)):
        step()
    st = moe.moe_check_device_error(ws)
    if st != 0:
        raise SystemExit(f"device status {st} after warm-up")

    sampler = ClockSampler(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    start.record(stream)
    for i in range(args.steps):
        step(ev[i])
    stop.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    clk = sampler.summary()
    dist.barrier()
    ms_total = start.elapsed_time(stop)
    st = moe.moe_check_device_error(ws)
    if st != 0:
        raise SystemExit(f"device status {st} in the timed region")
    ms_total = dist.max(ms_total)
    up_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    down_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)

    value = T * dist.world * args.steps / (ms_total / 1e3)
    flops_step = workloads.active_flops(w) * w.layers
    counts = np.diff(off.cpu().numpy())
    touched = int((counts > 0).sum())

    # roofline of the dominant kernel: the w1|w3 up-projection with SwiGLU (moe_expert_up:
    # row gather + grouped tcgen05 GEMM), per launch
    up_bytes = touched * 2 * f * d * esz + A * d * esz + A * f * esz   # w1, w3 of touched experts + x rows + h
    up_flops = 2.0 * A * d * 2 * f
    pk, pk_kind = peaks()
    hbm_peak = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tc_peak = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    ai = up_flops / up_bytes
    ridge = tc_peak * 1e12 / (hbm_peak * 1e9)
    if ai < ridge:
        ach = up_bytes / (up_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak}
    else:
        peak, kind, burst, sus = tensor_peak(pk, clk)
        ach = up_flops / (up_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "peak_kind": kind, "frac_of_sustained": ach / sus,
                "step_frac": flops_step / (ms_total / args.steps / 1e3) / 1e12 / peak}
    # batches of at most 64 tokens take the swapped-operand form (weights as the MMA's 128-row
    # side), larger ones the token-rows-as-M form
    form = "swapped-operand " if T <= 64 else ""
    roof.update({"traffic": kernel_traffic("expert_up", w.name),
                 "kernel": f"moe_expert_up (gather + {form}w1|w3 tcgen05 GEMM + SwiGLU)",
                 "algorithmic": up_bytes if roof["bound"] == "hbm" else up_flops,
                 "ms_per_launch": up_ms, "peak_source": f"{pk_kind} (MEASURED_PEAKS.json)" if pk_kind == "measured" else "fallback",
                 "down_ms_per_launch": down_ms})

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded Gaussian, Mixtral-shaped)",
            "config": {"workload": w.name, "T": T, "d_model": d, "d_ff": f, "n_experts": n, "top_k": k,
                       "layers": w.layers, "skewed_bias": w.skew_bias, "global_batch": T * dist.world,
                       "parallelism": f"replicas x{dist.world}",
                       "l2": "no flush: per-step inputs (expert weights, %.2f GB/layer) exceed the 126 MB L2"
                             % (3 * n * d * f * esz / 1e9)},
            "tflops": flops_step * dist.world * args.steps / (ms_total / 1e3) / 1e12,
            "roofline": roof, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk, "expert_counts": counts.tolist()}

    line["routing_stats"] = routing_stats_report(moe, w, step, layer, layers, x, xn, hs, idx, off,
                                                 stream)

    if not args.no_e2e:
        line["e2e"] = e2e_forward(args, w, dist, moe, x_h, layers, bias, ws, stream)

    if with_cpu and dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        xf, lf, _ = oracle_prepare(w, x_h, layers_h, bias_h)
        del layers_h
        line["cpu_baseline"] = run_cpu_baseline(w, xf, lf, bias_h)
    return line


def e2e_forward(args, w, dist, moe, x_h, layers, bias, ws, stream):
    """End to end through the public call, moe_layer_forward, with host buffers: every step
    copies its x from pinned host memory to the device, runs the layer (or the stack) and
    copies y back to pinned host memory.  The copies run on their own streams, one step
    ahead (H2D) and one behind (D2H) the layer, as a serving loop would overlap them; every
    copy of every step is inside the timed region, which ends when the last y is on the
    host."""
    import torch
    k = w.k
    esz = 2 if w.dtype == "bf16" else 4
    x_pin = torch.from_numpy(np.ascontiguousarray(x_h).view(np.int16) if w.dtype == "bf16" else x_h)
    x_pin = (x_pin.view(torch.bfloat16) if w.dtype == "bf16" else x_pin).pin_memory()
    y_pin = [torch.empty_like(x_pin).pin_memory() for _ in range(2)]
    x_dev = [torch.empty(x_pin.shape, dtype=x_pin.dtype, device=ws.device) for _ in range(2)]
    y_dev = [torch.empty_like(x_dev[0]) for _ in range(2)]
    xn = torch.empty_like(x_dev[0])
    hb = [torch.empty_like(x_dev[0]) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    loaded = [ev(), ev()]     # x_dev[b] holds the step's input
    used = [ev(), ev()]       # the layer has finished reading x_dev[b] and writing y_dev[b]
    drained = [ev(), ev()]    # y_dev[b] is on the host

    def layer_step(b):
        if w.layers == 1:
            moe.moe_layer_forward(x_dev[b], layers[0]["wg"], layers[0]["w1"], layers[0]["w3"],
                                  layers[0]["w2"], k, ws, logit_bias=bias, y=y_dev[b])
            return
        h_in = x_dev[b]
        for li, L in enumerate(layers):
            moe.moe_rmsnorm(h_in, w.rms_eps, x=xn)
            out = y_dev[b] if li == len(layers) - 1 else hb[li % 2]
            moe.moe_layer_forward(xn, L["wg"], L["w1"], L["w3"], L["w2"], k, ws, residual=h_in, y=out)
            h_in = out

    def load(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(used[b])          # step i-2 has finished with x_dev[b]
            x_dev[b].copy_(x_pin, non_blocking=True)
            loaded[b].record(h2d)

    def run(steps):
        load(0)
        for i in range(steps):
            b = i % 2
            if i + 1 < steps:
                load(i + 1)
            stream.wait_event(loaded[b])
            if i >= 2:
                stream.wait_event(drained[b])    # y_dev[b] of step i-2 is on the host
            layer_step(b)
            used[b].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(used[b])
                y_pin[b].copy_(y_dev[b], non_blocking=True)
                drained[b].record(d2h)
        for b in range(min(2, steps)):
            stream.wait_event(drained[b])

    run(3)
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_event(e0)
    run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    if moe.moe_check_device_error(ws) != 0:
        raise SystemExit("device status set in the end-to-end loop")
    e_ms = dist.max(e0.elapsed_time(e1))
    return {"value": w.T * dist.world * args.steps / (e_ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": w.T * w.d * esz, "d2h_bytes_per_step": w.T * w.d * esz,
            "ms_per_step": e_ms / args.steps, "api": "moe_layer_forward",
            "copies": "pinned H2D one step ahead and D2H one step behind, on their own streams"}


def routing_stats_report(moe, w, step, layer, layers, x, xn, hs, idx, off, stream):
    """Per-layer expert load and consecutive-token repetition (moe_routing_stats) of one more
    step, outside the timed region, plus the kernel's own time per launch.  Consecutive
    tokens of the decode batch belong to different sequences (no pairs); the other
    workloads are read as sequences of up to 4096 tokens."""
    import math
    import torch
    T, n, k = w.T, w.n, w.k
    seq_len = 1 if w.wid == 2 else min(T, 4096)
    counts = torch.empty((w.layers, n), dtype=torch.int64, device=x.device)
    pairs = torch.empty((w.layers, 3), dtype=torch.int64, device=x.device)
    hist = torch.empty((w.layers, n + 1), dtype=torch.int32, device=x.device)
    h_in = x
    for li, L in enumerate(layers):
        if w.layers == 1:
            layer(x, L, hs[0], None)
        else:
            moe.moe_rmsnorm(h_in, w.rms_eps, x=xn)
            layer(xn, L, hs[li % 2], h_in)
            h_in = hs[li % 2]
        moe.moe_routing_stats(idx, n, seq_len, expert_counts=counts[li], pair_counts=pairs[li])
        hist[li].copy_(off)
    # the kernel is far shorter than a Python call: time a CUDA graph of `reps` launches so
    # that the host does not set the pace
    reps = 200
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        for _ in range(reps):
            moe.moe_routing_stats(idx, n, seq_len, expert_counts=counts[-1], pair_counts=pairs[-1])
    graph.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    del graph
    c, pr, hs_np = counts.cpu().numpy(), pairs.cpu().numpy(), hist.cpu().numpy()
    per_layer = []
    for li in range(w.layers):
        if c[li].tolist() != np.diff(hs_np[li]).tolist():
            raise SystemExit("routing statistics disagree with the grouping offsets")
        p = int(pr[li, 0])
        per_layer.append({"expert_counts": c[li].tolist(), "pairs": p,
                          "first_choice_rate": pr[li, 1] / p if p else None,
                          "shared_expert_rate": pr[li, 2] / p if p else None})
    return {"seq_len": seq_len, "per_layer": per_layer,
            "random_first_choice_rate": 1.0 / n,
            "random_shared_expert_rate": 1.0 - math.comb(n - k, k) / math.comb(n, k),
            "kernel_us_per_launch": us, "bytes_read_per_launch": T * k * 4}


def backward_arm(args, w, dist):
    """Times moe_layer_backward: one step = the gradients of <dy, MoE(x)> with respect to x,
    W_g, the logit bias and every expert's w1, w3, w2 (routing recomputed inside the call).
    With --pass train a step is moe_layer_forward_train followed by moe_layer_backward_saved."""
    import torch
    import sparse_mixture_experts_56_b300 as moe

    if w.dtype != "bf16" or w.layers != 1:
        raise SystemExit("bench.py --pass backward: single-layer bf16 workloads only")
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    moe._native.lib()
    T, d, f, n, k = w.T, w.d, w.f, w.n, w.k
    A = T * k
    inp = workloads.make_inputs(w, seed=args.seed, tensors=("x", "wg", "w1", "w3", "w2", "dy"))
    g = {t: to_dev(inp[t], w, dev) for t in ("x", "wg", "w1", "w3", "w2", "dy")}
    bias = torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None
    ws = moe.backward_workspace(T, d, f, n, k, torch.bfloat16, dev)
    outs = {"dx": torch.empty_like(g["x"]), "dw_gate": torch.empty((d, n), dtype=torch.float32, device=dev),
            "dw1": torch.empty_like(g["w1"]), "dw3": torch.empty_like(g["w3"]),
            "dw2": torch.empty_like(g["w2"]), "dlogit_bias": torch.empty(n, dtype=torch.float32, device=dev)}
    stream = torch.cuda.current_stream()
    train = args.which == "train"
    if train:
        fws = moe.workspace(T, d, f, n, k, torch.bfloat16, dev)
        saved = moe.train_saved(T, d, f, n, k, torch.bfloat16, dev)
        y = torch.empty_like(g["x"])
        lib = moe._native.lib()

    def step(xx=None, dyy=None):
        xx = g["x"] if xx is None else xx
        dyy = g["dy"] if dyy is None else dyy
        if not train:
            moe.moe_layer_backward(xx, g["wg"], g["w1"], g["w3"], g["w2"], k, dyy, ws,
                                   logit_bias=bias, **outs)
            return
        moe.moe_layer_forward_train(xx, g["wg"], g["w1"], g["w3"], g["w2"], k, fws, saved,
                                    logit_bias=bias, y=y)
        st = lib.moe_layer_backward_saved(
            xx.data_ptr(), g["wg"].data_ptr(), g["w1"].data_ptr(), g["w3"].data_ptr(),
            g["w2"].data_ptr(), dyy.data_ptr(), T, d, f, n, k, moe.MOE_BF16, saved.data_ptr(),
            saved.numel(), outs["dx"].data_ptr(), outs["dw_gate"].data_ptr(),
            outs["dlogit_bias"].data_ptr(), outs["dw1"].data_ptr(), outs["dw3"].data_ptr(),
            outs["dw2"].data_ptr(), ws.data_ptr(), ws.numel(), stream.cuda_stream)
        moe._native.check("moe_layer_backward_saved", st)

    for _ in range(max(3, args.warmup)):
        step()
    if moe.moe_check_device_error(ws) != 0:
        raise SystemExit("device status set after warm-up")
    sampler = ClockSampler(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    dist.barrier()
    if moe.moe_check_device_error(ws) != 0:
        raise SystemExit("device status set in the timed region")
    ms = dist.max(e0.elapsed_time(e1)) / args.steps
    # FLOPs of the expert GEMMs: recompute of a|b (4Adf), dy w2 (2Adf), dx (4Adf), three
    # weight gradients (6Adf); a training step is the forward (6Adf) and the backward without
    # the recompute (12Adf); the router's part is negligible
    flops = (18.0 if train else 16.0) * A * d * f
    pk, pk_kind = peaks()
    clk = sampler.summary()
    tc_peak, kind, burst, sus = tensor_peak(pk, clk)
    ach = flops / (ms / 1e3) / 1e12
    line = {"metric": METRIC, "pass": args.which, "value": T * dist.world / (ms / 1e3),
            "unit": "tokens/s", "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded Gaussian, Mixtral-shaped; dy ~ N(0,1))",
            "config": {"workload": w.name, "T": T, "d_model": d, "d_ff": f, "n_experts": n, "top_k": k,
                       "skewed_bias": w.skew_bias, "parallelism": f"replicas x{dist.world}",
                       "l2": "no flush: per-step weights and gradients exceed the 126 MB L2"},
            "tflops": flops * dist.world / (ms / 1e3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": ach / tc_peak, "traffic": None, "peak_kind": kind,
                         "frac_of_burst": ach / burst, "frac_of_sustained": ach / sus,
                         "kernel": ("moe_layer_forward_train + moe_layer_backward_saved (all launches; "
                                    "18*T*K*d*f FLOPs)") if train else
                                   "moe_layer_backward (all launches of the call; 16*T*K*d*f FLOPs)",
                         "peak_source": f"{pk_kind} (MEASURED_PEAKS.json)"},
            "gpu_launches": (21 if train else 14) * args.steps, "clocks": clk}
    if not args.no_e2e and not train:
        x_pin = torch.from_numpy(np.ascontiguousarray(inp["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
        dy_pin = torch.from_numpy(np.ascontiguousarray(inp["dy"]).view(np.int16)).view(torch.bfloat16).pin_memory()
        dx_pin = torch.empty_like(x_pin).pin_memory()
        dwg_pin = torch.empty((d, n), dtype=torch.float32).pin_memory()
        xd, dyd = torch.empty_like(g["x"]), torch.empty_like(g["dy"])

        def e2e_step():
            xd.copy_(x_pin, non_blocking=True)
            dyd.copy_(dy_pin, non_blocking=True)
            step(xd, dyd)
            dx_pin.copy_(outs["dx"], non_blocking=True)
            dwg_pin.copy_(outs["dw_gate"], non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        em = dist.max(e0.elapsed_time(e1)) / args.steps
        line["e2e"] = {"value": T * dist.world / (em / 1e3), "unit": "tokens/s",
                       "h2d_bytes_per_step": 2 * T * d * 2, "d2h_bytes_per_step": T * d * 2 + d * n * 4,
                       "ms_per_step": em, "api": "moe_layer_backward (dx and dW_g copied back)"}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline and not train:
        import oracle
        f64 = {t: workloads.as_f32(inp[t], w).astype(np.float64) for t in ("x", "wg", "w1", "w3", "w2", "dy")}
        rng = np.random.default_rng(99)
        tok = oracle_sample_tokens(w, {2: 32, 3: 64, 4: 64}.get(w.wid, 32), rng)
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.moe_layer_backward(f64["x"][tok], f64["wg"], f64["w1"], f64["w3"], f64["w2"], k,
                                      f64["dy"][tok], inp["bias"])
            reps += 1
            el = time.perf_counter() - t0
            if el >= 10.0 or el * (reps + 1) / reps > 30:
                break
        line["cpu_baseline"] = {"value": reps * len(tok) / el, "unit": "tokens/s", "cores": cpu_cores(),
                                "kind": "oracle",
                                "sample": f"backward of {len(tok)} of the {T} tokens x {reps} repetition(s), "
                                          f"fp64 NumPy ({el:.1f} s)"}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def attention_arm(args, w, dist):
    """Times moe_attention_gqa on the workload's tokens with the pages' head counts (32 query,
    8 key-value heads of 128): one step = causal attention over every sequence."""
    import torch
    import sparse_mixture_experts_56_b300 as moe

    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    moe._native.lib()
    T, hq, hkv, dh = w.T, 32, 8, 128
    seq = args.seq_len if args.seq_len > 0 else T
    g = torch.Generator(device="cpu").manual_seed(args.seed)
    q = torch.randn((T, hq, dh), generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn((T, hkv, dh), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((T, hkv, dh), generator=g).to(torch.bfloat16).to(dev)
    out = torch.empty_like(q)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        moe.moe_attention_gqa(q, k, v, ws, seq, out=out)
    if moe.moe_check_device_error(ws) != 0:
        raise SystemExit("device status set after warm-up")
    sampler = ClockSampler(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0.record(stream)
    for _ in range(args.steps):
        moe.moe_attention_gqa(q, k, v, ws, seq, out=out)
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    dist.barrier()
    if moe.moe_check_device_error(ws) != 0:
        raise SystemExit("device status set in the timed region")
    ms = dist.max(e0.elapsed_time(e1)) / args.steps
    # causal FLOPs: 2 products (Q K^T, P V) x 2 FLOP x dh x the (i, j <= i) pairs, per head
    pairs = 0
    for s0 in range(0, T, seq):
        m = min(seq, T - s0)
        pairs += m * (m + 1) // 2
    flops = 4.0 * dh * hq * pairs
    pk, pk_kind = peaks()
    clk = sampler.summary()
    tc_peak, kind, burst, sus = tensor_peak(pk, clk)
    ach = flops / (ms / 1e3) / 1e12
    line = {"metric": METRIC, "pass": "attention", "value": T * dist.world / (ms / 1e3),
            "unit": "tokens/s", "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (q, k, v ~ N(0,1))",
            "config": {"workload": f"attention-gqa-t{T}-s{seq}", "T": T, "seq_len": seq,
                       "q_heads": hq, "kv_heads": hkv, "head_dim": dh,
                       "parallelism": f"replicas x{dist.world}"},
            "tflops": flops * dist.world / (ms / 1e3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": ach / tc_peak, "traffic": None, "peak_kind": kind,
                         "frac_of_burst": ach / burst, "frac_of_sustained": ach / sus,
                         "kernel": "attention_gqa_kernel (causal FLOPs 4*dh*hq*pairs)",
                         "peak_source": f"{pk_kind} (MEASURED_PEAKS.json)"},
            "gpu_launches": args.steps, "clocks": clk}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def decoder_arm(args, w, dist):
    """Times moe_decoder_layer_forward on the workload's tokens with the pages' attention
    shapes (32 query / 8 key-value heads of 128, d = 4096): RMSNorm, q/k/v projections, causal
    GQA attention, output projection + residual, RMSNorm, the MoE layer + residual."""
    import torch
    import sparse_mixture_experts_56_b300 as moe

    if w.dtype != "bf16" or w.layers != 1:
        raise SystemExit("bench.py --pass decoder: single-layer bf16 workloads only")
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    moe._native.lib()
    T, d, f, n, k, hq, hkv = w.T, w.d, w.f, w.n, w.k, 32, 8
    seq = args.seq_len if args.seq_len > 0 else min(T, 4096)
    inp = workloads.make_inputs(w, seed=args.seed, tensors=("x", "wg", "w1", "w3", "w2"))
    g = {t: to_dev(inp[t], w, dev) for t in ("x", "wg", "w1", "w3", "w2")}
    gen = torch.Generator(device="cpu").manual_seed(args.seed)
    proj = {name: (torch.randn(shape, generator=gen) * shape[1] ** -0.5).to(torch.bfloat16).to(dev)
            for name, shape in (("wq", (hq * 128, d)), ("wk", (hkv * 128, d)), ("wv", (hkv * 128, d)),
                                ("wo", (d, hq * 128)))}
    bias = torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None
    ws = moe.decoder_workspace(T, d, f, n, k, hq, hkv, dev)
    y = torch.empty_like(g["x"])
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_decoder_layer_forward(g["x"], proj["wq"], proj["wk"], proj["wv"], proj["wo"], g["wg"],
                                      g["w1"], g["w3"], g["w2"], k, hq, hkv, ws, seq_len=seq,
                                      logit_bias=bias, y=y)

    for _ in range(max(3, args.warmup)):
        step()
    if moe.moe_check_device_error(ws) != 0:
        raise SystemExit("device status set after warm-up")
    sampler = ClockSampler(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    dist.barrier()
    if moe.moe_check_device_error(ws) != 0:
        raise SystemExit("device status set in the timed region")
    ms = dist.max(e0.elapsed_time(e1)) / args.steps
    pairs = sum(min(seq, T - s0) * (min(seq, T - s0) + 1) // 2 for s0 in range(0, T, seq))
    flops = (2.0 * T * d * (hq + 2 * hkv) * 128 + 2.0 * T * hq * 128 * d + 4.0 * 128 * hq * pairs
             + workloads.active_flops(w))
    pk, pk_kind = peaks()
    clk = sampler.summary()
    tc_peak, kind, burst, sus = tensor_peak(pk, clk)
    ach = flops / (ms / 1e3) / 1e12
    line = {"metric": METRIC, "pass": "decoder", "value": T * dist.world / (ms / 1e3),
            "unit": "tokens/s", "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded Gaussian, Mixtral-shaped)",
            "config": {"workload": f"decoder-layer-{w.name}", "T": T, "seq_len": seq, "d_model": d,
                       "d_ff": f, "n_experts": n, "top_k": k, "q_heads": hq, "kv_heads": hkv,
                       "parallelism": f"replicas x{dist.world}"},
            "tflops": flops * dist.world / (ms / 1e3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": ach / tc_peak, "traffic": None, "peak_kind": kind,
                         "frac_of_sustained": ach / sus,
                         "kernel": "whole decoder layer (projections, causal attention, MoE FLOPs)",
                         "peak_source": f"{pk_kind} (MEASURED_PEAKS.json)"},
            # rmsnorm, span offsets, q, k, v, attention, o, residual add, rmsnorm, then the MoE
            # layer's router, grouping (1 or 3), gather, up, down, combine
            "gpu_launches": (9 + 5 + (1 if T * k <= 32768 else 3)) * args.steps, "clocks": clk}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def ep_arm(args, w, dist):
    """Times the expert-parallel layer pass: rank r of N holds experts [r*n/N, (r+1)*n/N) and
    T tokens of its own (seeded per rank); one step = route, group, the count and row
    all-to-alls, the local experts, the return all-to-all and the combine, on every rank."""
    import torch
    import sparse_mixture_experts_56_b300 as moe
    from sparse_mixture_experts_56_b300 import ep

    if w.dtype != "bf16" or w.layers != 1:
        raise SystemExit("bench.py --ep: single-layer bf16 workloads only")
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    moe._native.lib()
    G, r = dist.world, dist.rank
    blk = ep.expert_block(r, w.n, G)
    weights = workloads.make_inputs(w, seed=args.seed, tensors=("wg", "w1", "w3", "w2"))
    x = to_dev(workloads.make_inputs(w, seed=args.seed + r, tensors=("x",))["x"], w, dev)
    wg = to_dev(weights["wg"], w, dev)
    wl = {t: to_dev(np.ascontiguousarray(weights[t][blk.start:blk.stop]), w, dev) for t in ("w1", "w3", "w2")}
    del weights
    bias = torch.from_numpy(workloads.logit_bias_vector(w.n)).to(dev) if w.skew_bias else None
    comm = ep.TorchComm() if dist.world > 1 or dist.pg else None
    if comm is None:
        import torch.distributed as td
        td.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % _free_port(), rank=0,
                              world_size=1, device_id=dev)
        dist.pg = td
        comm = ep.TorchComm()
    ops = ep.NativeOps(dev)
    stream = torch.cuda.current_stream()

    def step():
        return ep.ep_layer_forward(comm, ops, x, wg, wl["w1"], wl["w3"], wl["w2"], w.k, w.n, bias)

    for _ in range(max(3, args.warmup)):
        _, stats = step()
    sampler = ClockSampler(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0.record(stream)
    for _ in range(args.steps):
        _, stats = step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    dist.barrier()
    ms = dist.max(e0.elapsed_time(e1)) / args.steps
    rows = torch.tensor([stats["expert_rows"]], dtype=torch.int64, device=dev)
    if G > 1:
        allr = [torch.empty_like(rows) for _ in range(G)]
        dist.pg.all_gather(allr, rows)
        load = [int(t.item()) for t in allr]
    else:
        load = [int(rows.item())]
    flops = workloads.active_flops(w) * G
    pk, pk_kind = peaks()
    clk = sampler.summary()
    tc_peak, kind, burst, sus = tensor_peak(pk, clk)
    ach = flops / (ms / 1e3) / 1e12
    line = {"metric": METRIC, "pass": "forward-ep", "value": w.T * G / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": G, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded Gaussian, Mixtral-shaped; tokens seeded per rank)",
            "config": {"workload": w.name, "T_per_rank": w.T, "d_model": w.d, "d_ff": w.f,
                       "n_experts": w.n, "top_k": w.k, "skewed_bias": w.skew_bias,
                       "parallelism": f"ep{G} (experts {w.n // G} per rank, NCCL all-to-all)",
                       "l2": "no flush: per-step weights exceed the 126 MB L2"},
            "tflops": ach,
            "roofline": {"bound": "tensor", "achieved": ach, "peak": tc_peak * G, "unit": "TFLOP/s",
                         "frac": ach / (tc_peak * G), "traffic": None, "peak_kind": kind,
                         "kernel": "whole EP layer pass on every rank (active FLOPs 6*T*K*d*f per rank)",
                         "peak_source": f"{pk_kind} (MEASURED_PEAKS.json), times the ranks"},
            "ep": {"ranks": G, "expert_rows_per_rank": load,
                   "imbalance_max_over_mean": max(load) / (sum(load) / len(load)) if sum(load) else None},
            # router, grouping (1 or 3), gather, regroup, up (gather + GEMM), down, gather back,
            # combine; NCCL's own kernels are not counted
            "gpu_launches": (9 + (2 if w.T * w.k > 32768 else 0)) * args.steps, "clocks": clk}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def main():
    args = parse()
    w = workloads.workload(args.workload)
    dist = Dist()
    if args.impl == "reference":
        reference_arm(args, w, dist)   # rank 0 only; the other ranks exit without work
        return
    import torch
    dist.init("nccl" if torch.cuda.is_available() else "gloo")
    try:
        if args.ep:
            ep_arm(args, w, dist)
        elif args.which in ("backward", "train"):
            backward_arm(args, w, dist)
        elif args.which == "attention":
            attention_arm(args, w, dist)
        elif args.which == "decoder":
            decoder_arm(args, w, dist)
        else:
            ours_arm(args, w, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
