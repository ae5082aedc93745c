"""Benchmark of the tensor-parallel MLP block (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5|c3]
                    [--mode splitk|buffers] [--impl ours|reference]

A step is one forward + backward pass of the whole block over one batch of
seeded synthetic input: the column-parallel GEMM with the fused activation, the
row-parallel GEMM with the shard sum, and the backward (activation gradient,
both weight gradients, dX with its shard sum), all N shards as virtual ranks on
one GPU. Inputs and weights are resident in HBM before the timed region; every
input is larger than L2 (129 MB) or read once per step, so no L2 flush is
inserted. Under torchrun every rank runs its own replica on its own batch (data
parallel, no collective on the data path): weak scaling, value = all ranks'
FLOPs / the slowest rank's time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (token rows), on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sharded MLP fwd+bwd TFLOP/s (% BF16 peak); decode GEMV HBM GB/s (% peak)"

WORKLOADS = {
    "c5": dict(desc="large prefill/training SwiGLU MLP fwd+bwd: b=1 s=8192 h=8192 ffn=28672 N=4",
               b=1, s=8192, h=8192, f=28672, N=4, act="swiglu", cfg=5),
    "c3": dict(desc="mid training erf-GELU MLP fwd+bwd: b=4 s=2048 h=4096 ffn=16384 N=8",
               b=4, s=2048, h=4096, f=16384, N=8, act="gelu", cfg=3),
    "c1": dict(desc="tiny fp32 erf-GELU MLP fwd+bwd: b=2 s=16 h=128 ffn=512 N=2 (CUDA cores, no TF32)",
               b=2, s=16, h=128, f=512, N=2, act="gelu", cfg=1, dtype="f32"),
    "c2": dict(desc="page-2-sized pre-LN transformer layer fwd+bwd: b=8 s=128 h=128 heads=8 "
                    "ffn=512 N=2", b=8, s=128, h=128, f=512, N=2, heads=8, act="gelu", cfg=2,
               layer=True),
    "c3-sp": dict(desc="sequence-parallel pre-LN erf-GELU MLP block fwd+bwd (LN on each rank's "
                       "rows, reduce-scatter + all-gather): b=4 s=2048 h=4096 ffn=16384 N=8",
                  b=4, s=2048, h=4096, f=16384, N=8, act="gelu", cfg=3, sp=True),
    "gpt": dict(desc="small tensor-parallel GPT training (vocabulary-parallel embedding and "
                     "cross-entropy, tied output layer, AdamW): vocab=256 h=128 heads=8 ffn=512 "
                     "layers=2 b=4 s=32 N=2, fp32", b=4, s=32, h=128, f=512, N=2, heads=8,
                vocab=256, layers=2, act="gelu", cfg=6, gpt=True, dtype="f32"),
    "gqa": dict(desc="head-sharded grouped-query attention block fwd+bwd (LN, QKV, attention, "
                     "W_o, shard sum): b=4 s=512 h=2048 heads=32 kv_heads=8 N=16 (each key/value "
                     "head replicated on 2 shards)", b=4, s=512, h=2048, f=0, heads=32,
                kv_heads=8, N=16, act="none", cfg=7, gqa=True),
    # reduced-token case of c5 for ncu captures (a few GB on the device, inputs > L2)
    "c5-2k": dict(desc="profiling case: SwiGLU MLP fwd+bwd b=1 s=2048 h=8192 ffn=28672 N=4",
                  b=1, s=2048, h=8192, f=28672, N=4, act="swiglu", cfg=5),
}

DECODE = dict(desc="decode GEMV sweep: SwiGLU MLP forward, h=8192 ffn=28672 N=8 "
                   "(W_gate/W_up column-split, W_down row-split), shard sum via fp32 partials",
              h=8192, f=28672, N=8, tokens=(1, 8, 32, 64), cfg=4)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def layer_flops(w):
    """Algorithmic FLOPs of the pre-LN layer forward + backward (backward = 2 x forward):
    QKV 2*M*h*3h, scores and P V 4*b*heads*s*s*d, W_o 2*M*h*h, MLP 4*M*h*f."""
    M, h, f = w["b"] * w["s"], w["h"], w["f"]
    fwd = 6 * M * h * h + 4 * w["b"] * w["s"] * w["s"] * h + 2 * M * h * h + 4 * M * h * f
    return 3.0 * fwd


def mlp_flops(w, M=None):
    M = w["b"] * w["s"] if M is None else M
    per = 6 if w["act"] == "swiglu" else 4
    return 3.0 * per * M * w["h"] * w["f"]  # backward = 2 x forward


def col_gemm_flops(w):
    M = w["b"] * w["s"]
    return (4.0 if w["act"] == "swiglu" else 2.0) * M * w["h"] * w["f"]


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one column-GEMM launch,
# from an ncu capture of the full-size workload, valid only for the kernel source it
# was taken on (sha256 of csrc/gemm_tc.cu + csrc/ptx.cuh + csrc/epi_math.cuh); see profiles/.
COL_GEMM_TRAFFIC = {
    "c5": {"bytes": 6.647e9 + 1.398e9, "src": "d417b4ec8df59967"},
    "c3": {"bytes": 1.123e9 + 0.502e9, "src": "d417b4ec8df59967"},
}


# Tensor-pipe activity of the same launch (sm__pipe_tensor_cycles_active and
# sm__pipe_tc_cycles_active, % of peak over the elapsed cycles) from a one-pass ncu
# capture of the full-size workload, under the same source-hash rule. See profiles/.
COL_GEMM_TENSOR_PIPE = {
    "c5": {"tensor": 90.03, "tc": 90.24, "case": "c5", "src": "d417b4ec8df59967"},
    "c3": {"tensor": 74.10, "tc": 74.92, "case": "c3", "src": "d417b4ec8df59967"},
}


def _kernel_source_hash():
    """Hash of the tensor-core GEMM's source (kernel and its PTX wrappers): a stored
    traffic figure is reported only while the kernel it was measured on is unchanged."""
    import hashlib
    h = hashlib.sha256()
    for name in ("gemm_tc.cu", "ptx.cuh", "epi_math.cuh"):
        with open(os.path.join(ROOT, "attention_gemms_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def col_gemm_traffic(workload):
    t = COL_GEMM_TRAFFIC.get(workload)
    if not t or t["src"] != _kernel_source_hash():
        return None
    return t["bytes"]


def col_gemm_tensor_pipe(workload):
    t = COL_GEMM_TENSOR_PIPE.get(workload)
    if not t or t["src"] != _kernel_source_hash():
        return None
    return {"sm__pipe_tensor_cycles_active_pct": t["tensor"],
            "sm__pipe_tc_cycles_active_pct": t["tc"], "captured_on": t["case"]}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(backend):
    """One process group over the ranks, with a bounded timeout (TP_DIST_TIMEOUT_S,
    default 300 s): a rank that has left makes the others' next barrier or timing
    reduction raise instead of waiting forever."""
    import datetime
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        timeout = datetime.timedelta(seconds=float(os.environ.get("TP_DIST_TIMEOUT_S", "300")))
        dist.init_process_group(backend=backend, timeout=timeout)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Timing only: the slowest rank's value (no data-path collective)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed_offset(rank: int) -> int:
    """Each data-parallel replica gets its own batch (X, dZ streams)."""
    return 100 * rank


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ inputs

def make_inputs(w, rank, device):
    import torch
    from attention_gemms_gb300 import synth
    M, h, f = w["b"] * w["s"], w["h"], w["f"]
    c = w["cfg"]
    off = rank_seed_offset(rank)

    dt = w.get("dtype", "bf16")

    def dev(shape, name, sigma, extra=0):
        a = synth.normal(shape, synth.seed_of(c, name) + extra, sigma, dt)
        if dt == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device), a
        return torch.from_numpy(a).to(device), a

    X, Xh = dev((M, h), "X", 1.0, off)
    dZ, dZh = dev((M, h), "dZ", 1.0, off)
    W1, W1h = dev((h, f), "Wg", 0.02)
    W1u, W1uh = dev((h, f), "Wu", 0.02) if w["act"] == "swiglu" else (None, None)
    W2, W2h = dev((f, h), "Wd", 0.02)
    host = {"X": Xh, "dZ": dZh, "W1": W1h, "W1u": W1uh, "W2": W2h}
    return {"X": X, "dZ": dZ, "W1": W1, "W1u": W1u, "W2": W2}, host


# ------------------------------------------------------------------ our arm

def overlapped_e2e(stream, steps, step_on, ins, ins_host, outs, outs_host):
    """Time `steps` end-to-end steps: every step copies its inputs in from pinned host
    memory (ins_host -> a device input set) and its results out (a device output set ->
    outs_host). Copies run on a second stream and overlap the neighbouring steps'
    compute; inputs and outputs are double-buffered (ins / outs are the first sets, a
    second set is allocated like them) and events order each copy after the step that
    frees its buffer. step_on(in_set, out_set) enqueues one step on `stream`.
    Returns ms per step (CUDA events on `stream`)."""
    import torch
    ins_b = [list(ins), [torch.empty_like(t) for t in ins]]
    outs_b = [list(outs), [torch.empty_like(t) for t in outs]]
    copy = torch.cuda.Stream(device=stream.device)
    ev = torch.cuda.Event
    torch.cuda.synchronize()
    e0, e1 = ev(enable_timing=True), ev(enable_timing=True)
    e0.record(stream)
    copy.wait_event(e0)
    in_ready, step_done, out_read = [ev(), ev()], [None, None], [None, None]

    def copy_in(k):
        with torch.cuda.stream(copy):
            for dst, src in zip(ins_b[k], ins_host):
                dst.copy_(src, non_blocking=True)
        in_ready[k] = ev()
        in_ready[k].record(copy)

    copy_in(0)
    for k in range(steps):
        cur = k % 2
        if k + 1 < steps:  # next step's inputs, once the step that used that buffer is done
            if step_done[1 - cur] is not None:
                copy.wait_event(step_done[1 - cur])
            copy_in(1 - cur)
        stream.wait_event(in_ready[cur])
        if out_read[cur] is not None:
            stream.wait_event(out_read[cur])
        step_on(ins_b[cur], outs_b[cur])
        step_done[cur] = ev()
        step_done[cur].record(stream)
        copy.wait_event(step_done[cur])
        with torch.cuda.stream(copy):
            for dst, src in zip(outs_host, outs_b[cur]):
                dst.copy_(src, non_blocking=True)
        out_read[cur] = ev()
        out_read[cur].record(copy)
    stream.wait_stream(copy)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


VENDOR_PEAKS = {"bf16_tflops": 2250.0, "hbm_gbs": 7900.0,
                "label": "nominal dense bf16 2.25 PFLOP/s and HBM3e 7.9 TB/s (vendor class)"}


def timed_steps(stream, steps, step):
    """Time `steps` calls of step(i) on `stream`: one event pair brackets all of them
    (the mean) and one pair per step gives the per-step distribution (the median).
    Returns (mean ms, median ms)."""
    import torch
    ev = lambda: torch.cuda.Event(enable_timing=True)
    t0, t1 = ev(), ev()
    per = [(ev(), ev()) for _ in range(steps)]
    t0.record(stream)
    for i in range(steps):
        per[i][0].record(stream)
        step(i)
        per[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    med = float(np.median([a.elapsed_time(b) for a, b in per]))
    return t0.elapsed_time(t1) / steps, med


def run_ours(args, w):
    import torch
    from attention_gemms_gb300 import build as B
    from attention_gemms_gb300 import tpmlp as T

    ws_, rank, local = dist_env()
    if ws_ > 1:
        torch.cuda.set_device(local)
    dist_init("nccl")
    B.build()
    T.lib()
    device = torch.device("cuda", torch.cuda.current_device())
    if w.get("layer"):
        return run_layer(args, w, T, device, rank, ws_)
    if w.get("sp"):
        return run_sp(args, w, T, device, rank, ws_)
    if w.get("gpt"):
        return run_gpt(args, w, T, device, rank, ws_)
    if w.get("gqa"):
        return run_gqa(args, w, T, device, rank, ws_)
    M, h, f, N = w["b"] * w["s"], w["h"], w["f"], w["N"]
    sw = w["act"] == "swiglu"
    act = T.Act.SWIGLU if sw else T.Act.GELU
    modes = {"splitk": T.Reduce.SPLITK, "buffers": T.Reduce.BUFFERS}
    f32 = w.get("dtype") == "f32"
    BF = T.DType.F32 if f32 else T.DType.BF16
    bf = torch.float32 if f32 else torch.bfloat16
    t_gen = time.time()
    d, hostin = make_inputs(w, rank, device)
    t_gen = time.time() - t_gen
    e = lambda *s: torch.empty(*s, dtype=bf, device=device)
    Y, Yu, H = e(M, f), (e(M, f) if sw else None), e(M, f)
    Z, dX = e(M, h), e(M, h)
    dW1, dW1u, dW2 = e(h, f), (e(h, f) if sw else None), e(f, h)
    wsb = max(T.tp_workspace_size(T.Op.ROW_LINEAR, M, f, h, N, BF, T.Act.NONE, m)
              for m in modes.values())
    wsb = max([wsb] + [T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, N, BF, act, m)
                       for m in modes.values()])
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    flops = mlp_flops(w)
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_s = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    pin = lambda: torch.empty((M, h), dtype=bf, pin_memory=True)
    Xp, dZp = pin(), pin()
    if f32:
        Xp.numpy()[:] = hostin["X"]
        dZp.numpy()[:] = hostin["dZ"]
    else:
        Xp.view(torch.int16).numpy()[:] = hostin["X"].view(np.int16)
        dZp.view(torch.int16).numpy()[:] = hostin["dZ"].view(np.int16)
    outs_host = [pin(), pin()]

    def measure(mode_name):
        """Warm-up, the timed steps (device-resident inputs) and the end-to-end steps of
        one shard-sum variant; per-rank ms, the column GEMM's ms and the launch count."""
        mode = modes[mode_name]
        col_ev = []

        def step_on(Xs, dZs, Zs, dXs, record=False):
            if record:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
            T.tp_col_linear(Xs, d["W1"], d["W1u"], Y, Yu, H, M, h, f, N, BF, act, stream)
            if record:
                b.record(stream)
                col_ev.append((a, b))
            T.tp_row_linear(H, d["W2"], None, Zs, M, f, h, N, BF, mode, ws, ws.numel(), stream)
            T.tp_mlp_bwd(Xs, d["W1"], d["W1u"], d["W2"], Y, Yu, H, dZs, dXs, dW1, dW1u, dW2,
                         M, h, f, N, BF, act, mode, ws, ws.numel(), stream)

        for _ in range(args.warmup):
            step_on(d["X"], d["dZ"], Z, dX)
        torch.cuda.synchronize()
        if T.tp_check_status(stream) != 0:
            raise RuntimeError("device wait timeout during warm-up: " + T.tp_last_error())
        barrier()
        torch.cuda.synchronize()
        n0 = T.tp_launch_count()
        ms, med = timed_steps(stream, args.steps,
                              lambda i: step_on(d["X"], d["dZ"], Z, dX, record=True))
        barrier()
        launches = T.tp_launch_count() - n0
        col_ms = sum(a.elapsed_time(b) for a, b in col_ev) / len(col_ev)
        if T.tp_check_status(stream) != 0:
            raise RuntimeError("device wait timeout in the timed region: " + T.tp_last_error())
        # end to end: inputs in from pinned host memory and results out, every step,
        # copies overlapped with the neighbouring steps' compute (overlapped_e2e)
        barrier()
        e2e_ms = overlapped_e2e(stream, args.steps, lambda i, o: step_on(i[0], i[1], o[0], o[1]),
                                [d["X"], d["dZ"]], [Xp, dZp], [Z, dX], outs_host)
        barrier()
        if T.tp_check_status(stream) != 0:
            raise RuntimeError("device wait timeout in the end-to-end steps: " + T.tp_last_error())
        return {"ms": max_over_ranks(ms, device), "median": max_over_ranks(med, device),
                "col": max_over_ranks(col_ms, device), "e2e": max_over_ranks(e2e_ms, device),
                "launches": launches}

    def interleaved():
        """Steps of the two variants alternated (per-step CUDA events), so that clock
        drift under the power cap weighs on both alike: per-variant median ms."""
        ev = lambda: torch.cuda.Event(enable_timing=True)
        per = {name: [] for name in modes}
        barrier()
        torch.cuda.synchronize()
        for _ in range(args.steps):
            for name, mode in modes.items():
                a, b = ev(), ev()
                a.record(stream)
                T.tp_col_linear(d["X"], d["W1"], d["W1u"], Y, Yu, H, M, h, f, N, BF, act, stream)
                T.tp_row_linear(H, d["W2"], None, Z, M, f, h, N, BF, mode, ws, ws.numel(), stream)
                T.tp_mlp_bwd(d["X"], d["W1"], d["W1u"], d["W2"], Y, Yu, H, d["dZ"], dX, dW1, dW1u,
                             dW2, M, h, f, N, BF, act, mode, ws, ws.numel(), stream)
                b.record(stream)
                per[name].append((a, b))
        torch.cuda.synchronize()
        barrier()
        return {name: max_over_ranks(float(np.median([a.elapsed_time(b) for a, b in v])), device)
                for name, v in per.items()}

    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    main_r = measure(args.mode)
    others, inter = {}, {}
    if args.variants and not f32:
        for name in modes:
            if name != args.mode:
                others[name] = measure(name)
        inter = interleaved()
    clk = clocks.stop()

    ms_max, e2e_max, col_max = main_r["ms"], main_r["e2e"], main_r["col"]
    value = flops * ws_ / (ms_max * 1e-3) / 1e12
    e2e_val = flops * ws_ / (e2e_max * 1e-3) / 1e12
    col_tf = col_gemm_flops(w) / (col_max * 1e-3) / 1e12
    traffic = col_gemm_traffic(args.workload)
    vp = VENDOR_PEAKS["bf16_tflops"]
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "ms_per_step_median": round(main_r["median"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if f32 else "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights; random init)",
        "config": {"workload": w["desc"], "tokens": M, "h": h, "ffn": f, "shards": N,
                   "act": w["act"], "shard_sum": args.mode, "global_batch": w["b"] * ws_,
                   "seq_len": w["s"], "parallelism": f"tp{N} virtual ranks per GPU, dp{ws_}",
                   "l2": "inputs larger than L2 (no flush)"},
        "pct_of_peak": round(100 * value / ws_ / peak, 2),
        "pct_of_vendor_peak": round(100 * value / ws_ / vp, 2),
        "roofline": {"bound": "tensor", "kernel": "gemm_tc2_kernel (column-parallel GEMM + fused "
                     + ("SwiGLU" if sw else "GELU") + " epilogue)",
                     "achieved": round(col_tf, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(col_tf / peak, 4), "frac_of_sustained": round(col_tf / peak_s, 4),
                     "frac_of_vendor": round(col_tf / vp, 4),
                     "peak_source": f"{src} bf16 dense (burst)",
                     "vendor_peak": {"value": vp, "label": VENDOR_PEAKS["label"]},
                     "traffic": traffic,
                     "tensor_pipe_active": col_gemm_tensor_pipe(args.workload),
                     "algorithmic_flops_per_launch": col_gemm_flops(w),
                     "avg_launch_ms": round(col_max, 4)},
        "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 2 * M * h * (4 if f32 else 2),
                "d2h_bytes_per_step": 2 * M * h * (4 if f32 else 2),
                "ms_per_step": round(e2e_max, 4)},
        "gpu_launches": int(main_r["launches"]),
        "clocks": clk,
        "input_gen_s": round(t_gen, 1),
    }
    if others:
        var = {}
        for name, r in [(args.mode, main_r)] + list(others.items()):
            tf = flops * ws_ / (r["ms"] * 1e-3) / 1e12
            var[name] = {"ms_per_step": round(r["ms"], 4), "ms_per_step_median": round(r["median"], 4),
                         "TFLOPs": round(tf, 2), "pct_of_peak": round(100 * tf / ws_ / peak, 2),
                         "e2e_TFLOPs": round(flops * ws_ / (r["e2e"] * 1e-3) / 1e12, 2),
                         "column_gemm_ms": round(r["col"], 4), "gpu_launches": int(r["launches"])}
            if name in inter:
                tf_i = flops * ws_ / (inter[name] * 1e-3) / 1e12
                var[name]["interleaved_ms_median"] = round(inter[name], 4)
                var[name]["interleaved_TFLOPs"] = round(tf_i, 2)
                var[name]["interleaved_pct_of_peak"] = round(100 * tf_i / ws_ / peak, 2)
        var["note"] = ("splitk: the row-parallel sums folded as split-K into one accumulator; "
                       "buffers: per-shard fp32 partials summed by the shard-reduce kernel (the "
                       "backward's dX sum on a side stream beside the weight-gradient GEMMs); "
                       "each timed in its own bracketed run, then in one run of alternating "
                       "steps (interleaved_*, per-step medians)")
        out["shard_sum_variants"] = var
    if f32:
        out["roofline"] = {"bound": "alu", "note": "fp32 FFMA path at a latency-bound size; "
                           "no roofline fraction is claimed", "achieved": None, "peak": None,
                           "unit": "TFLOP/s", "frac": None, "traffic": None}
    if args.shard_sum:
        out["reduce_ln"] = run_shard_sum(args, w, device, T)
    if args.decode and not f32:
        out["decode"] = run_decode(args, device, T)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, hostin, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_sp(args, w, T, device, rank, nranks):
    """The sequence-parallel pre-LN MLP block, forward + backward, per step. The MLP
    FLOPs are the work counted; the same block without sequence parallelism (LN on
    the replicated rows, the ordinary all-reduce, replicated LN gradients) is timed
    beside it, and the column GEMM of the block on its own gives the roofline."""
    import torch
    M, h, f, N = w["b"] * w["s"], w["h"], w["f"], w["N"]
    sw = w["act"] == "swiglu"
    A = T.Act.SWIGLU if sw else T.Act.GELU
    mode = T.Reduce.SPLITK if args.mode == "splitk" else T.Reduce.BUFFERS
    BF, bf, f32 = T.DType.BF16, torch.bfloat16, torch.float32
    t_gen = time.time()
    d, hostin = make_inputs(w, rank, device)
    t_gen = time.time() - t_gen
    e = lambda *sh, dt=bf: torch.empty(sh, dtype=dt, device=device)
    g, b = torch.ones(h, device=device), torch.zeros(h, device=device)
    xn, mean, rstd = e(M, h), e(M, dt=f32), e(M, dt=f32)
    Y, Yu, H, out, dx = e(M, f), (e(M, f) if sw else None), e(M, f), e(M, h), e(M, h)
    dg, db, dgr, dbr = e(h, dt=f32), e(h, dt=f32), e(N, h, dt=f32), e(N, h, dt=f32)
    dW1, dWu, dW2 = e(h, f), (e(h, f) if sw else None), e(f, h)
    wsb = max(T.tp_workspace_size(T.Op.SP_MLP_FWD, M, h, f, N, BF, A, mode),
              T.tp_workspace_size(T.Op.SP_MLP_BWD, M, h, f, N, BF, A, mode),
              T.tp_workspace_size(T.Op.MLP_FWD, M, h, f, N, BF, A, mode),
              T.tp_workspace_size(T.Op.MLP_BWD, M, h, f, N, BF, A, mode),
              T.tp_workspace_size(T.Op.LAYERNORM_BWD, M, h, 0, 1, BF))
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=device)
    dxn = e(M, h)
    stream = torch.cuda.current_stream()
    X, W1, W1u, W2, dZ = d["X"], d["W1"], d["W1u"], d["W2"], d["dZ"]

    def sp_step():
        T.tp_sp_mlp_fwd(X, g, b, W1, W1u, W2, xn, mean, rstd, Y, Yu, H, out, M, h, f, N, BF, A,
                        mode, ws, ws.numel(), stream)
        T.tp_sp_mlp_bwd(X, g, W1, W1u, W2, xn, mean, rstd, Y, Yu, H, dZ, dx, dg, db, dgr, dbr,
                        dW1, dWu, dW2, M, h, f, N, BF, A, mode, ws, ws.numel(), stream)

    def tp_step():  # LN replicated on every rank, all-reduce, replicated LN gradients
        T.tp_layernorm_fwd(X, g, b, xn, mean, rstd, M, h, 1e-5, BF, stream)
        T.tp_mlp_fwd(xn, W1, W1u, W2, X, Y, Yu, H, out, M, h, f, N, BF, A, mode, ws, ws.numel(),
                     stream)
        T.tp_mlp_bwd(xn, W1, W1u, W2, Y, Yu, H, dZ, dxn, dW1, dWu, dW2, M, h, f, N, BF, A, mode,
                     ws, ws.numel(), stream)
        T.tp_layernorm_bwd(X, g, mean, rstd, dxn, dZ, dx, dg, db, M, h, BF, ws, ws.numel(),
                           stream)

    def timed(fn, steps):
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        z.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(z) / steps

    for _ in range(args.warmup):
        sp_step()
        tp_step()
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    n0 = T.tp_launch_count()
    ms = timed(sp_step, args.steps)
    launches = T.tp_launch_count() - n0
    barrier()
    tp_ms = timed(tp_step, args.steps)
    col_ms = timed(lambda: T.tp_col_linear(xn, W1, W1u, Y, Yu, H, M, h, f, N, BF, A, stream),
                   args.steps)
    # end to end: x and dout in from pinned host memory, out and dx back, every step
    # (copies overlapped with the neighbouring steps' compute)
    pin = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    Xp, dZp = pin(hostin["X"]), pin(hostin["dZ"])
    hostbuf = lambda: torch.empty((M, h), dtype=bf, pin_memory=True)

    def sp_step_on(i, o):
        T.tp_sp_mlp_fwd(i[0], g, b, W1, W1u, W2, xn, mean, rstd, Y, Yu, H, o[0], M, h, f, N, BF,
                        A, mode, ws, ws.numel(), stream)
        T.tp_sp_mlp_bwd(i[0], g, W1, W1u, W2, xn, mean, rstd, Y, Yu, H, i[1], o[1], dg, db, dgr,
                        dbr, dW1, dWu, dW2, M, h, f, N, BF, A, mode, ws, ws.numel(), stream)
    barrier()
    e2e_ms = overlapped_e2e(stream, args.steps, sp_step_on, [X, dZ], [Xp, dZp], [out, dx],
                            [hostbuf(), hostbuf()])
    clk = clocks.stop()
    if T.tp_check_status(stream) != 0:
        raise RuntimeError("device wait timeout: " + T.tp_last_error())
    ms_max, e2e_max = max_over_ranks(ms, device), max_over_ranks(e2e_ms, device)
    tp_max, col_max = max_over_ranks(tp_ms, device), max_over_ranks(col_ms, device)
    flops = mlp_flops(w)
    value = flops * nranks / (ms_max * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    col_tf = col_gemm_flops(w) / (col_max * 1e-3) / 1e12
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": nranks,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights; LN gamma=1, beta=0)",
        "config": {"workload": w["desc"], "tokens": M, "h": h, "ffn": f, "shards": N,
                   "act": w["act"], "shard_sum": args.mode, "sequence_parallel": True,
                   "global_batch": w["b"] * nranks, "seq_len": w["s"],
                   "parallelism": f"tp{N}+sp virtual ranks per GPU, dp{nranks}",
                   "l2": "inputs larger than L2 (no flush)"},
        "pct_of_peak": round(100 * value / nranks / peak, 2),
        "without_sp_ms_per_step": round(tp_max, 4),
        "roofline": {"bound": "tensor", "kernel": "gemm_tc2_kernel (column-parallel GEMM + fused "
                     + ("SwiGLU" if sw else "GELU") + " epilogue), timed on its own at the "
                     "block's shape", "achieved": round(col_tf, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(col_tf / peak, 4),
                     "peak_source": f"{src} bf16 dense (burst)",
                     "traffic": col_gemm_traffic(args.workload.replace("-sp", "")),
                     "algorithmic_flops_per_launch": col_gemm_flops(w),
                     "avg_launch_ms": round(col_max, 4)},
        "e2e": {"value": round(flops * nranks / (e2e_max * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 2 * M * h * 2, "d2h_bytes_per_step": 2 * M * h * 2,
                "ms_per_step": round(e2e_max, 4)},
        "gpu_launches": int(launches),
        "clocks": clk,
        "input_gen_s": round(t_gen, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, hostin, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(res), flush=True)


def gpt_flops(w):
    """Algorithmic FLOPs of one training step: 3 x the forward's matrix products
    (layers' linear maps and attention, output layer)."""
    M, h, f, v, L = w["b"] * w["s"], w["h"], w["f"], w["vocab"], w["layers"]
    per_layer = 2 * M * h * (3 * h + h + 2 * f) + 4 * w["b"] * w["s"] * w["s"] * h
    return 3.0 * (L * per_layer + 2 * M * h * v)


def run_vocab_ce(device, T, M=8192, v=50304, N=8, reps=20):
    """Vocabulary-parallel cross-entropy, forward + backward (in place), bf16 logits at
    a GPT-2-sized vocabulary: HBM-bound; algorithmic bytes = the logits read by the
    forward, read and written by the backward (+ targets, lse, row losses)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(77)
    L = (torch.randn((M, v), generator=g, device=device) * 2).to(torch.bfloat16)
    tg = torch.randint(0, v, (M,), generator=g, device=device, dtype=torch.int32)
    f = lambda *sh: torch.empty(sh, dtype=torch.float32, device=device)
    lse, rows, shards, loss = f(M), f(M), f(N), f(1)
    stream = torch.cuda.current_stream()
    BF = T.DType.BF16

    def fwd():
        T.tp_vocab_ce_fwd(L, tg, lse, rows, shards, loss, M, v, N, BF, stream)

    def bwd():
        T.tp_vocab_ce_bwd(L, tg, lse, L, M, v, N, 1.0 / M, BF, stream)
    out = {"shape": {"M": M, "vocab": v, "N": N, "dtype": "bf16"}, "unit": "GB/s"}
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    for name, fn, nbytes in (("fwd", fwd, M * v * 2 + 16 * M), ("bwd", bwd, 2 * M * v * 2 + 8 * M)):
        for _ in range(3):
            fwd()
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            fwd()  # the backward needs the forward's lse; both rewrite nothing they read
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            z.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(z))
        us = float(np.median(ts)) * 1e3
        out[name] = {"us": round(us, 2), "algorithmic_bytes": int(nbytes),
                     "achieved": round(nbytes / us / 1e3, 1), "frac": round(nbytes / us / 1e3 / hbm, 4)}
    out["peak"], out["peak_source"] = hbm, f"{src} HBM copy"
    del L
    torch.cuda.empty_cache()
    return out


def run_vocab_ce_only(args):
    """The vocabulary-parallel cross-entropy (forward + backward) alone, for profiling."""
    import torch
    from attention_gemms_gb300 import build as B
    from attention_gemms_gb300 import tpmlp as T
    ws_, rank, local = dist_env()
    if ws_ > 1:
        torch.cuda.set_device(local)
    dist_init("nccl")
    B.build()
    T.lib()
    device = torch.device("cuda", torch.cuda.current_device())
    ce = run_vocab_ce(device, T, reps=max(args.steps, 1))
    tot_us = ce["fwd"]["us"] + ce["bwd"]["us"]
    nbytes = ce["fwd"]["algorithmic_bytes"] + ce["bwd"]["algorithmic_bytes"]
    if rank == 0:
        print(json.dumps({
            "metric": "vocabulary-parallel cross-entropy fwd+bwd GB/s", "unit": "GB/s",
            "value": round(nbytes / tot_us / 1e3 * ws_, 1), "n_gpus": ws_, "steps": args.steps,
            "warmup": 3, "ms_per_step": round(tot_us / 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "vocab-ce", **ce["shape"]},
            "roofline": {"bound": "hbm", "kernel": "vocab_ce_bwd_vec_kernel",
                         "achieved": ce["bwd"]["achieved"], "peak": ce["peak"], "unit": "GB/s",
                         "frac": ce["bwd"]["frac"], "traffic": None},
            "vocab_ce": ce}), flush=True)


def run_gpt(args, w, T, device, rank, nranks):
    """The small GPT's training step (forward, backward, AdamW) on one seeded batch,
    the page's 50-step run, plus the vocabulary-parallel cross-entropy at a large
    vocabulary for its HBM roofline."""
    import torch
    from attention_gemms_gb300 import gpt as GP
    from attention_gemms_gb300 import synth
    mode = T.Reduce.SPLITK if args.mode == "splitk" else T.Reduce.BUFFERS
    steps_run = 50
    t_gen = time.time()
    p, ids, tg = synth.gpt_inputs(w["cfg"], w["vocab"], w["h"], w["f"], w["layers"], w["b"], w["s"])
    t_gen = time.time() - t_gen
    m = GP.SmallGPT(w["vocab"], w["h"], w["heads"], w["f"], w["layers"], w["b"], w["s"], w["N"],
                    mode=mode, steps=steps_run, device=device)
    m.load(p)
    m.set_batch(ids, tg)
    stream = torch.cuda.current_stream()
    # the page's run from the loaded parameters: 50 steps, losses kept on the device
    for _ in range(steps_run):
        m.step(stream=stream)
    torch.cuda.synchronize()
    trajectory = m.losses.cpu().numpy().tolist()
    # one step's launches, then the step captured once as a CUDA graph: the step count
    # and the loss history live in device memory, so every replay is a whole step
    n0 = T.tp_launch_count()
    m.step(stream=stream)
    per_step = T.tp_launch_count() - n0
    torch.cuda.synchronize()
    m.capture()
    for _ in range(args.warmup):
        m.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    ms, ms_med = timed_steps(stream, args.steps, lambda i: m.replay())
    launches = per_step * args.steps
    # end to end: the batch's ids and targets in from pinned host memory, the loss out
    idp = torch.from_numpy(np.asarray(ids, np.int32).reshape(-1)).pin_memory()
    tgp = torch.from_numpy(np.asarray(tg, np.int32).reshape(-1)).pin_memory()
    lossp = torch.empty(1, dtype=torch.float32, pin_memory=True)
    barrier()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        m.ids.copy_(idp, non_blocking=True)
        m.targets.copy_(tgp, non_blocking=True)
        m.replay()
        lossp.copy_(m.loss_now, non_blocking=True)
    z.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(z) / args.steps
    clk = clocks.stop()
    if T.tp_check_status(stream) != 0:
        raise RuntimeError("device wait timeout: " + T.tp_last_error())
    ce = run_vocab_ce(device, T)
    ms_max, e2e_max = max_over_ranks(ms, device), max_over_ranks(e2e_ms, device)
    M = w["b"] * w["s"]
    tok = M * nranks / (ms_max * 1e-3)
    res = {
        "metric": "small GPT training tokens/s (vocabulary-parallel embedding + cross-entropy)",
        "value": round(tok, 1), "unit": "tokens/s", "n_gpus": nranks, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "ms_per_step_median": round(max_over_ranks(ms_med, device), 4),
        "cuda_graph": "the whole training step (forward, backward, step counter, AdamW) "
                      "replayed from one CUDA graph",
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded random tokens and targets; E ~ U(-1/sqrt(h), 1/sqrt(h)), "
                "weights ~ N(0, 0.02^2))",
        "config": {"workload": w["desc"], "tokens": M, "vocab": w["vocab"], "h": w["h"],
                   "ffn": w["f"], "layers": w["layers"], "heads": w["heads"], "shards": w["N"],
                   "shard_sum": args.mode, "parallelism": f"tp{w['N']} virtual ranks per GPU, "
                   f"dp{nranks}", "l2": "whole model L2-resident (latency-bound size)"},
        "tflops": round(gpt_flops(w) * nranks / (ms_max * 1e-3) / 1e12, 4),
        "loss_trajectory_every_10": [round(x, 4) for x in trajectory[::10]] + [round(trajectory[-1], 4)],
        "roofline": {"bound": "hbm", "kernel": "vocab_ce_bwd_kernel (vocabulary-parallel "
                     "cross-entropy gradient, bf16 logits, M=8192 v=50304 N=8, timed on its own)",
                     "achieved": ce["bwd"]["achieved"], "peak": ce["peak"], "unit": "GB/s",
                     "frac": ce["bwd"]["frac"], "traffic": None,
                     "note": "the GPT step itself is launch/latency-bound at this size"},
        "vocab_ce": ce,
        "e2e": {"value": round(M * nranks / (e2e_max * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * M * 4, "d2h_bytes_per_step": 4,
                "ms_per_step": round(e2e_max, 4)},
        "gpu_launches": int(launches),
        "clocks": clk,
        "input_gen_s": round(t_gen, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = gpt_cpu_baseline(w, p, ids, tg)
    if rank == 0:
        print(json.dumps(res), flush=True)


def gpt_cpu_baseline(w, p, ids, tg, steps=3):
    """The fp64 oracle's training step (forward, backward, AdamW) on the same batch."""
    from oracle import gpt_oracle as G
    f64 = {k: np.asarray(a, np.float64) for k, a in p.items()}
    params = {"E": f64["E"], "gammaf": f64["gammaf"], "betaf": f64["betaf"],
              "layers": [{k: f64[f"L{li}.{k}"] for k in G.LAYER_KEYS} for li in range(w["layers"])]}
    cfg = dict(b=w["b"], s=w["s"], heads=w["heads"], N=w["N"])
    c0, t0 = time.process_time(), time.perf_counter()
    G.gpt_train(params, ids, tg, cfg, steps)
    dt, dc = (time.perf_counter() - t0) / steps, (time.process_time() - c0) / steps
    M = w["b"] * w["s"]
    return {"value": round(M / dt, 1), "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "threads_effective": round(dc / dt, 1), "kind": "oracle",
            "sample": f"fp64 oracle training steps (forward, backward, AdamW) on the full batch, "
                      f"{steps} steps, {dt * 1e3:.0f} ms each"}


def gqa_flops(w):
    """Algorithmic FLOPs of the GQA block forward + backward, counted on the unsharded
    model (replicated key/value projections are redundant work, not counted):
    projections 2 M h (H + 2 Hkv) d + 2 M h h, attention 4 b H s^2 d; backward 2x."""
    M, h, H, Hkv, b, s = w["b"] * w["s"], w["h"], w["heads"], w["kv_heads"], w["b"], w["s"]
    d = h // H
    fwd = 2 * M * h * (H + 2 * Hkv) * d + 2 * M * h * h + 4 * b * H * s * s * d
    return 3.0 * fwd, 4.0 * b * H * s * s * d


def run_gqa(args, w, T, device, rank, nranks):
    """The head-sharded GQA block, forward + backward per step. The dominant kernel of
    the step is the pair GEMM (four 2048-wide launches: W_o forward, dO, dW_o, dx_n);
    its roofline is taken on the dO GEMM (M x h x h) timed alone through tp_gemm. The
    tensor-core attention core (forward, and backward with its scratch) is timed alone
    as well and reported under "attention"."""
    import torch
    from attention_gemms_gb300 import synth
    b, s, h, H, Hkv, N = w["b"], w["s"], w["h"], w["heads"], w["kv_heads"], w["N"]
    M, d = b * s, h // H
    BF = T.DType.BF16
    mode = T.Reduce.SPLITK if args.mode == "splitk" else T.Reduce.BUFFERS
    Wc = T.tp_gqa_qkv_cols(h, H, Hkv, N)
    c = w["cfg"]
    sig = 1.0 / math.sqrt(h)
    dev = lambda shape, name, sigma: torch.from_numpy(
        synth.normal(shape, synth.seed_of(c, name), sigma, "bf16").view(np.int16)).view(
        torch.bfloat16).to(device)
    t_gen = time.time()
    x, dout = dev((M, h), "X", 1.0), dev((M, h), "dZ", 1.0)
    Wq, Wk = dev((h, H * d), "Wqkv", sig), dev((h, Hkv * d), "Wg", sig)
    Wv, Wo = dev((h, Hkv * d), "Wu", sig), dev((h, h), "Wo", sig)
    t_gen = time.time() - t_gen
    g, be = torch.ones(h, device=device), torch.zeros(h, device=device)
    e = lambda *sh, dt=torch.bfloat16: torch.empty(sh, dtype=dt, device=device)
    f32 = torch.float32
    Wsh = e(h, Wc)
    T.tp_gqa_pack_qkv(Wq, Wk, Wv, Wsh, h, H, Hkv, N, BF)
    xn, mean, rstd, qkv, o, lse, out = (e(M, h), e(M, dt=f32), e(M, dt=f32), e(M, Wc), e(M, h),
                                        e(b, H, s, dt=f32), e(M, h))
    dx, dg, db, dW, dWo = e(M, h), e(h, dt=f32), e(h, dt=f32), e(h, Wc), e(h, h)
    ws = torch.empty(max(T.tp_gqa_workspace_size(1, M, h, H, Hkv, N, BF, mode),
                         T.tp_gqa_workspace_size(0, M, h, H, Hkv, N, BF, mode), 256),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step_on(x, dout, out, dx):
        T.tp_gqa_attn_proj_fwd(x, g, be, Wsh, Wo, xn, mean, rstd, qkv, o, lse, out, b, s, h, H,
                               Hkv, N, 0, BF, mode, ws, ws.numel(), stream)
        T.tp_gqa_attn_proj_bwd(x, g, Wsh, Wo, xn, mean, rstd, qkv, o, lse, dout, dx, dg, db, dW,
                               dWo, b, s, h, H, Hkv, N, 0, BF, mode, ws, ws.numel(), stream)

    def step():
        step_on(x, dout, out, dx)

    def timed(fn, steps):
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        z.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(z) / steps

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    n0 = T.tp_launch_count()
    ms = timed(step, args.steps)
    launches = T.tp_launch_count() - n0
    attn_ms = timed(lambda: T.tp_gqa_attention_fwd(qkv, o, lse, b, s, h, H, Hkv, N, 0, BF, stream),
                    args.steps)
    dO_t, dqkv_t = e(M, h), e(M, Wc)
    dO_t.copy_(dout)
    awsb = T.tp_gqa_attention_bwd_workspace_size(b, s, H)
    aws = torch.empty(awsb, dtype=torch.uint8, device=device)
    attn_bwd_ms = timed(lambda: T.tp_gqa_attention_bwd(qkv, o, lse, dO_t, dqkv_t, b, s, h, H, Hkv,
                                                       N, 0, BF, aws, awsb, stream), args.steps)
    gemm_ms = timed(lambda: T.tp_gemm(dout, Wo, dO_t, M, h, h, 0, 1, BF, stream), args.steps)
    xp = torch.empty((M, h), dtype=torch.bfloat16, pin_memory=True)
    dp = torch.empty((M, h), dtype=torch.bfloat16, pin_memory=True)
    xp.copy_(x)
    dp.copy_(dout)
    outp = torch.empty((M, h), dtype=torch.bfloat16, pin_memory=True)
    dxp = torch.empty((M, h), dtype=torch.bfloat16, pin_memory=True)

    barrier()
    e2e_ms = overlapped_e2e(stream, args.steps, lambda i, o: step_on(i[0], i[1], o[0], o[1]),
                            [x, dout], [xp, dp], [out, dx], [outp, dxp])
    clk = clocks.stop()
    if T.tp_check_status(stream) != 0:
        raise RuntimeError("device wait timeout: " + T.tp_last_error())
    ms_max, e2e_max = max_over_ranks(ms, device), max_over_ranks(e2e_ms, device)
    attn_max = max_over_ranks(attn_ms, device)
    attn_bwd_max = max_over_ranks(attn_bwd_ms, device)
    gemm_max = max_over_ranks(gemm_ms, device)
    total, attn_fwd = gqa_flops(w)
    attn_tf = attn_fwd / (attn_max * 1e-3) / 1e12
    attn_bwd_tf = 2.0 * attn_fwd / (attn_bwd_max * 1e-3) / 1e12
    gemm_flops = 2.0 * M * h * h
    gemm_tf = gemm_flops / (gemm_max * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    res = {
        "metric": "head-sharded GQA attention block fwd+bwd TFLOP/s",
        "value": round(total * nranks / (ms_max * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "n_gpus": nranks, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0, 1/h) weights; LN gamma=1, beta=0)",
        "config": {"workload": w["desc"], "tokens": M, "h": h, "heads": H, "kv_heads": Hkv,
                   "shards": N, "qkv_columns_sharded": Wc,
                   "qkv_columns_unreplicated": (H + 2 * Hkv) * d, "shard_sum": args.mode,
                   "parallelism": f"tp{N} virtual ranks per GPU, dp{nranks}",
                   "l2": "activations larger than L2 (no flush)"},
        "roofline": {"bound": "tensor", "kernel": "gemm_tc2_kernel (pair tcgen05 GEMM, 256 x 256 "
                     "tiles on CTA pairs; 44 % of the step's GPU time, its four 2048-wide "
                     "launches 27 %), timed on its own as the dO GEMM "
                     f"(M {M} x N {h} x K {h}) through tp_gemm",
                     "achieved": round(gemm_tf, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(gemm_tf / peak, 4),
                     "peak_source": f"{src} bf16 dense (burst)",
                     "traffic": col_gemm_traffic("gqa-dO"),
                     "algorithmic_flops_per_launch": gemm_flops,
                     "avg_launch_ms": round(gemm_max, 4)},
        "attention": {"kernels": "attn_fwd_tc_kernel; attn_bwd_dsum_kernel + attn_bwd_dkdv_tc_kernel "
                      "+ attn_bwd_dq_tc_kernel (tcgen05, bf16 head_dim 64), each pass timed on "
                      "its own, non-causal",
                      "fwd_tflops": round(attn_tf, 2), "fwd_frac": round(attn_tf / peak, 4),
                      "fwd_ms": round(attn_max, 4), "bwd_tflops": round(attn_bwd_tf, 2),
                      "bwd_frac": round(attn_bwd_tf / peak, 4), "bwd_ms": round(attn_bwd_max, 4),
                      "flops": {"fwd": attn_fwd, "bwd": 2.0 * attn_fwd}},
        "e2e": {"value": round(total * nranks / (e2e_max * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 2 * M * h * 2, "d2h_bytes_per_step": 2 * M * h * 2,
                "ms_per_step": round(e2e_max, 4)},
        "gpu_launches": int(launches), "clocks": clk, "input_gen_s": round(t_gen, 1),
    }
    if rank == 0:
        print(json.dumps(res), flush=True)


# ------------------------------------------------------------------ page-2 layer

def layer_inputs(w, rank):
    """Seeded inputs of the pre-LN layer: x, dout ~N(0,1); W_qkv, W_o, W1, W2 ~N(0,0.02^2);
    LayerNorm gamma = 1, beta = 0 (the framework's initial values)."""
    from attention_gemms_gb300 import synth
    b, s, h, f, c = w["b"], w["s"], w["h"], w["f"], w["cfg"]
    M, off = b * s, rank_seed_offset(rank)
    g = lambda shape, name, sigma, extra=0: synth.normal(shape, synth.seed_of(c, name) + extra,
                                                         sigma, "bf16")
    return {"x": g((M, h), "X", 1.0, off), "dout": g((M, h), "dZ", 1.0, off),
            "Wqkv": g((h, 3 * h), "Wqkv", 0.02), "Wo": g((h, h), "Wo", 0.02),
            "W1": g((h, f), "W1", 0.02), "W2": g((f, h), "W2", 0.02),
            "gamma1": np.ones(h, np.float32), "beta1": np.zeros(h, np.float32),
            "gamma2": np.ones(h, np.float32), "beta2": np.zeros(h, np.float32)}


def run_layer(args, w, T, device, rank, nranks):
    import torch
    b, s, h, f, N, heads = w["b"], w["s"], w["h"], w["f"], w["N"], w["heads"]
    M = b * s
    BF, bf, f32 = T.DType.BF16, torch.bfloat16, torch.float32
    mode = T.Reduce.SPLITK if args.mode == "splitk" else T.Reduce.BUFFERS
    hin = layer_inputs(w, rank)
    to = lambda a: (torch.from_numpy(a.view(np.int16)).view(bf) if a.dtype == np.uint16
                    else torch.from_numpy(a)).to(device)
    d = {k: to(v) for k, v in hin.items()}
    e = lambda *sh, dty=bf: torch.empty(*sh, dtype=dty, device=device)
    sv = dict(xn1=e(M, h), mean1=e(M, dty=f32), rstd1=e(M, dty=f32), qkv=e(M, 3 * h), o=e(M, h),
              lse=e(b, heads, s, dty=f32), x1=e(M, h), xn2=e(M, h), mean2=e(M, dty=f32),
              rstd2=e(M, dty=f32), y=e(M, f), hh=e(M, f))
    gr = dict(dWqkv=e(h, 3 * h), dWo=e(h, h), dW1=e(h, f), dW2=e(f, h), dgamma1=e(h, dty=f32),
              dbeta1=e(h, dty=f32), dgamma2=e(h, dty=f32), dbeta2=e(h, dty=f32))
    W = T.make_struct(T.LayerWeights, **{k: d[k] for k in ("Wqkv", "Wo", "W1", "W2", "gamma1",
                                                             "beta1", "gamma2", "beta2")})
    S = T.make_struct(T.LayerSaved, **sv)
    G = T.make_struct(T.LayerGrads, **gr)
    wsb = max(T.tp_workspace_size(T.Op.LAYER_FWD, M, h, f, N, BF, T.Act.GELU, mode),
              T.tp_workspace_size(T.Op.LAYER_BWD, M, h, f, N, BF, T.Act.GELU, mode))
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=device)
    out, dx = e(M, h), e(M, h)

    def step():
        T.tp_layer_fwd(d["x"], W, S, out, b, s, h, f, heads, N, 0, BF, mode, ws, ws.numel())
        T.tp_layer_bwd(d["x"], W, S, d["dout"], dx, G, b, s, h, f, heads, N, 0, BF, mode, ws,
                       ws.numel())

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    n0 = T.tp_launch_count()
    step()
    per_step_launches = T.tp_launch_count() - n0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(max(args.warmup, 20)):
        g.replay()
    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier()
    ms = t0.elapsed_time(t1) / args.steps
    # end to end through the C ABI: x and dout in from pinned memory, out and dx back
    xp = torch.empty((M, h), dtype=bf, pin_memory=True)
    dp = torch.empty((M, h), dtype=bf, pin_memory=True)
    xp.view(torch.int16).numpy()[:] = hin["x"].view(np.int16)
    dp.view(torch.int16).numpy()[:] = hin["dout"].view(np.int16)
    op, dxp = torch.empty_like(xp, pin_memory=True), torch.empty_like(xp, pin_memory=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        d["x"].copy_(xp, non_blocking=True)
        d["dout"].copy_(dp, non_blocking=True)
        step()
        op.copy_(out, non_blocking=True)
        dxp.copy_(dx, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop()
    if T.tp_check_status() != 0:
        raise RuntimeError("device wait timeout in the layer: " + T.tp_last_error())
    ms_max, e2e_max = max_over_ranks(ms, device), max_over_ranks(e2e_ms, device)
    fl = layer_flops(w)
    res = {
        "metric": METRIC, "value": round(fl * nranks / (ms_max * 1e-3) / 1e12, 3),
        "unit": "TFLOP/s", "n_gpus": nranks, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; LN gamma=1, beta=0)",
        "config": {"workload": w["desc"], "tokens": M, "h": h, "ffn": f, "heads": heads,
                   "shards": N, "shard_sum": args.mode, "replay": "CUDA graph of one step",
                   "launches_per_step": int(per_step_launches),
                   "parallelism": f"tp{N} virtual ranks per GPU, dp{nranks}"},
        "roofline": {"bound": "latency", "note": "launch/latency-bound size (M=1024, h=128): "
                     "the step time is reported, no roofline fraction is claimed",
                     "achieved": None, "peak": None, "unit": "TFLOP/s", "frac": None,
                     "traffic": None},
        "e2e": {"value": round(fl * nranks / (e2e_max * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 2 * M * h * 2, "d2h_bytes_per_step": 2 * M * h * 2,
                "ms_per_step": round(e2e_max, 4), "replay": "eager launches"},
        "gpu_launches": int(per_step_launches) * args.steps,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = layer_cpu_baseline(w, hin)
    if rank == 0:
        print(json.dumps(res), flush=True)


def layer_cpu_baseline(w, hin, reps=3):
    from attention_gemms_gb300 import synth
    from oracle import tp_oracle as O
    f64 = lambda a: synth.to_f64(a, "bf16") if a.dtype == np.uint16 else a.astype(np.float64)
    p = {k: f64(hin[k]) for k in ("Wqkv", "Wo", "W1", "W2", "gamma1", "beta1", "gamma2", "beta2")}
    x, dout = f64(hin["x"]), f64(hin["dout"])
    c0, t0 = time.process_time(), time.perf_counter()
    for _ in range(reps):
        O.layer_bwd(x, w["b"], w["s"], p, w["heads"], w["N"], dout)  # runs the forward too
    dt, dc = (time.perf_counter() - t0) / reps, (time.process_time() - c0) / reps
    return {"value": round(layer_flops(w) / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "threads_effective": round(dc / dt, 1),
            "kind": "oracle", "sample": f"fp64 oracle layer forward+backward on the whole "
                                        f"workload, {reps} repetitions, {dt:.2f} s each"}


# ------------------------------------------------------------------ decode sweep

def decode_bytes(T, h, f, N):
    """Algorithmic HBM bytes of one decode forward: the three weight matrices once,
    x in, A = SiLU(x Wg) * (x Wu) out and back in, the fp32 shard partials out and
    back in, Z out."""
    weights = 3 * h * f * 2
    acts = T * h * 2 + 2 * T * f * 2 + T * h * 2
    partials = 2 * N * T * h * 4
    return weights + acts + partials, 3 * h * f * 2, 2 * h * f * 2 + T * h * 2 + T * f * 2


def run_shard_sum(args, w, device, T, reps=20):
    """The shard sum at the workload's size, on its own (variant A's reduction of the
    fp32 partials) and followed by LayerNorm, fused into one pass and unfused
    (reduce, then LN reading the sum back). HBM-bound: GB/s of algorithmic bytes
    against the measured copy bandwidth. Inputs (the partials) are larger than L2."""
    import torch
    M, h, N = w["b"] * w["s"], w["h"], w["N"]
    f32 = w.get("dtype") == "f32"
    BF = T.DType.F32 if f32 else T.DType.BF16
    bf = torch.float32 if f32 else torch.bfloat16
    e = 4 if f32 else 2
    g = torch.Generator(device=device)
    g.manual_seed(4242)
    P = torch.randn((N, M, h), generator=g, device=device, dtype=torch.float32)
    R = torch.randn((M, h), generator=g, device=device, dtype=torch.float32).to(bf)
    gamma = torch.ones(h, device=device, dtype=torch.float32)
    beta = torch.zeros(h, device=device, dtype=torch.float32)
    S, Y = torch.empty((M, h), device=device, dtype=bf), torch.empty((M, h), device=device, dtype=bf)
    mean = torch.empty(M, device=device, dtype=torch.float32)
    rstd = torch.empty(M, device=device, dtype=torch.float32)
    stream = torch.cuda.current_stream()
    calls = {
        "reduce": (lambda: T.tp_shard_reduce(P, R, S, N, M, h, BF, stream),
                   N * M * h * 4 + 2 * M * h * e),
        "reduce_ln_fused": (lambda: T.tp_shard_reduce_ln(P, R, gamma, beta, S, Y, mean, rstd, N, M,
                                                         h, 1e-5, BF, stream),
                            N * M * h * 4 + 3 * M * h * e + 8 * M),
        "reduce_then_ln": (lambda: (T.tp_shard_reduce(P, R, S, N, M, h, BF, stream),
                                    T.tp_layernorm_fwd(S, gamma, beta, Y, mean, rstd, M, h, 1e-5,
                                                       BF, stream)),
                           N * M * h * 4 + 3 * M * h * e + 8 * M),
    }
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    out = {"unit": "GB/s", "peak": hbm, "peak_source": f"{src} HBM copy",
           "shape": {"N": N, "M": M, "h": h}, "l2": "partials larger than L2 (no flush)"}
    for name, (fn, nbytes) in calls.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / reps
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"us": round(us, 2), "algorithmic_bytes": int(nbytes), "achieved": round(gbs, 1),
                     "frac": round(gbs / hbm, 4)}
    if T.tp_check_status(stream) != 0:
        raise RuntimeError("device error in the shard-sum measurement: " + T.tp_last_error())
    del P, R, S, Y
    torch.cuda.empty_cache()
    return out


def run_decode(args, device, T):
    import torch
    from attention_gemms_gb300 import synth
    w = DECODE
    h, f, N, c = w["h"], w["f"], w["N"], w["cfg"]
    BF = T.DType.BF16
    mode = T.Reduce.BUFFERS

    def dev(shape, name, sigma, extra=0):
        a = synth.normal(shape, synth.seed_of(c, name) + extra, sigma, "bf16")
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)

    Wg, Wu, Wd = dev((h, f), "Wg", 0.02), dev((h, f), "Wu", 0.02), dev((f, h), "Wd", 0.02)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    res = {"workload": w["desc"], "unit": "GB/s", "peak": hbm,
           "peak_source": f"{src} HBM copy bandwidth", "cuda_graph": True, "per_tokens": {}}
    stream = torch.cuda.current_stream()
    for nt in w["tokens"]:
        X = dev((nt, h), "X", 1.0, nt)
        A = torch.empty((nt, f), dtype=torch.bfloat16, device=device)
        Z = torch.empty((nt, h), dtype=torch.bfloat16, device=device)
        wsb = T.tp_workspace_size(T.Op.ROW_LINEAR, nt, f, h, N, BF, T.Act.NONE, mode)
        ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=device)
        def fwd():
            T.tp_col_linear(X, Wg, Wu, None, None, A, nt, h, f, N, BF, T.Act.SWIGLU)
            T.tp_row_linear(A, Wd, None, Z, nt, f, h, N, BF, mode, ws, ws.numel())

        for _ in range(args.warmup):
            fwd()
        torch.cuda.synchronize()
        # one step's launches in a CUDA graph (the tensor maps are kernel parameters)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fwd()
        # warm up for at least 200 ms of replays: clocks (SM and HBM) drop while the
        # GPU idles, e.g. during the CPU baseline, and take a moment to come back
        t_w = time.time()
        n_w = 0
        while n_w < args.warmup or time.time() - t_w < args.decode_warmup_ms * 1e-3:
            g.replay()
            n_w += 1
            if n_w % 50 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.steps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / args.steps
        # the gate/up GEMM alone, launched eagerly between events (weights > L2)
        col_ms = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            T.tp_col_linear(X, Wg, Wu, None, None, A, nt, h, f, N, BF, T.Act.SWIGLU)
            e1.record()
            torch.cuda.synchronize()
            col_ms.append(e0.elapsed_time(e1))
        col = float(np.median(col_ms))
        total, wbytes, col_bytes = decode_bytes(nt, h, f, N)
        if T.tp_check_status(stream) != 0:
            raise RuntimeError("device wait timeout in decode: " + T.tp_last_error())
        gbs = total / (ms * 1e-3) / 1e9
        res["per_tokens"][str(nt)] = {
            "ms_per_step": round(ms, 4), "GBps": round(gbs, 1),
            "pct_of_peak": round(100 * gbs / hbm, 1),
            "weight_GBps": round(wbytes / (ms * 1e-3) / 1e9, 1),
            "TFLOPs": round(2 * nt * 3 * h * f / (ms * 1e-3) / 1e12, 2),
            "roofline": {"bound": "hbm",
                         "kernel": ("gemv_kernel<1, EPI_SWIGLU, paired> (gate/up + SwiGLU)" if nt == 1
                                    else "gemm_tc_kernel<128, EPI_SWIGLU, decode> (gate/up + SwiGLU)"),
                         "achieved": round(col_bytes / (col * 1e-3) / 1e9, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(col_bytes / (col * 1e-3) / 1e9 / hbm, 4),
                         "avg_launch_ms": round(col, 4), "algorithmic_bytes": col_bytes},
        }
        del g
    return res


def run_decode_only(args):
    """The decode sweep as the main line: value = the lowest GB/s over the token counts."""
    import torch
    from attention_gemms_gb300 import build as B
    from attention_gemms_gb300 import tpmlp as T
    ws_, rank, local = dist_env()
    if ws_ > 1:
        torch.cuda.set_device(local)
    dist_init("nccl")
    B.build()
    T.lib()
    device = torch.device("cuda", torch.cuda.current_device())
    barrier()
    d = run_decode(args, device, T)
    worst = min(v["GBps"] for v in d["per_tokens"].values())
    worst = max_over_ranks(-worst, device) * -1.0
    if rank == 0:
        peak = d["peak"]
        print(json.dumps({"metric": METRIC, "value": round(worst * ws_, 1), "unit": "GB/s",
                          "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "bf16", "data": "synthetic (seeded)",
                          "config": {"workload": DECODE["desc"], "tokens": list(DECODE["tokens"])},
                          "pct_of_peak": round(100 * worst / peak, 1), "decode": d}), flush=True)


# ------------------------------------------------------------------ CPU oracle

def _oracle_sample(w, hostin, rows, Wf):
    """One forward + backward of the oracle on `rows` token rows (full weights)."""
    from attention_gemms_gb300 import synth
    from oracle import tp_oracle as O
    dt = w.get("dtype", "bf16")
    X = synth.to_f64(hostin["X"][:rows], dt)
    dZ = synth.to_f64(hostin["dZ"][:rows], dt)
    if w.get("sp"):  # rows is a multiple of N: each virtual rank holds rows / N of them
        g, b = np.ones(X.shape[1]), np.zeros(X.shape[1])
        O.sp_mlp_block_bwd(X, g, b, Wf["W1"], Wf["W2"], w["N"], dZ, w["act"], Wf["W1u"])
        return
    if w["act"] == "swiglu":
        O.mlp_swiglu_fwd(X, Wf["W1"], Wf["W1u"], Wf["W2"], w["N"])
        O.mlp_swiglu_bwd(X, Wf["W1"], Wf["W1u"], Wf["W2"], dZ, w["N"])
    else:
        O.mlp_gelu_fwd(X, Wf["W1"], Wf["W2"], w["N"])
        O.mlp_gelu_bwd(X, Wf["W1"], Wf["W2"], dZ, w["N"])


def _weights_f64(hostin, dt="bf16"):
    from attention_gemms_gb300 import synth
    return {k: (synth.to_f64(hostin[k], dt) if hostin[k] is not None else None)
            for k in ("W1", "W1u", "W2")}


def cpu_baseline(w, hostin, budget_s=15.0):
    Wf = _weights_f64(hostin, w.get("dtype", "bf16"))
    rows = 8
    while True:
        c0, t0 = time.process_time(), time.perf_counter()
        _oracle_sample(w, hostin, rows, Wf)
        dt, dc = time.perf_counter() - t0, time.process_time() - c0
        if dt * 2 > budget_s or rows >= w["b"] * w["s"]:
            break
        rows = min(w["b"] * w["s"], int(rows * max(2.0, budget_s / max(dt, 1e-3) * 0.5)))
        rows -= rows % w["N"] if w.get("sp") else 0
    return {"value": round(mlp_flops(w, rows) / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)),
            "threads_effective": round(dc / dt, 1), "kind": "oracle",
            "sample": f"fp64 oracle forward+backward on {rows} of {w['b'] * w['s']} token rows, "
                      f"full weights, {dt:.1f} s; FLOPs scaled by the row fraction",
            "wall_s": round(dt, 2)}


def run_reference(args, w):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    t_gen = time.time()
    from attention_gemms_gb300 import synth
    M, h, f = w["b"] * w["s"], w["h"], w["f"]
    c = w["cfg"]
    dtp = w.get("dtype", "bf16")
    metric, unit, scale = METRIC, "TFLOP/s", 1e12
    if w.get("gqa"):
        from oracle import gqa_oracle as Q
        H, Hkv, N, d = w["heads"], w["kv_heads"], w["N"], h // w["heads"]
        sig = 1.0 / math.sqrt(h)
        nrm = lambda shape, name, sg: synth.to_f64(synth.normal(shape, synth.seed_of(c, name), sg,
                                                                "bf16"), "bf16")
        x, dout = nrm((w["s"], h), "X", 1.0), nrm((w["s"], h), "dZ", 1.0)  # one sequence
        Wsh = Q.gqa_pack(nrm((h, H * d), "Wqkv", sig), nrm((h, Hkv * d), "Wg", sig),
                         nrm((h, Hkv * d), "Wu", sig), H, Hkv, N)
        Wo = nrm((h, h), "Wo", sig)
        g1, b1 = np.ones(h), np.zeros(h)
        run = lambda: Q.gqa_block_bwd(x, 1, w["s"], g1, b1, Wsh, Wo, H, Hkv, N, dout)
        flops = gqa_flops(dict(w, b=1))[0]
        metric = "head-sharded GQA attention block fwd+bwd TFLOP/s"
        sample = (f"fp64 oracle GQA block forward+backward on 1 of {w['b']} sequences "
                  f"(s={w['s']}); FLOPs of that sequence")
    elif w.get("gpt"):
        from oracle import gpt_oracle as G
        pr, ids, tg = synth.gpt_inputs(c, w["vocab"], h, f, w["layers"], w["b"], w["s"])
        f64 = {k: np.asarray(a, np.float64) for k, a in pr.items()}
        params = {"E": f64["E"], "gammaf": f64["gammaf"], "betaf": f64["betaf"],
                  "layers": [{k: f64[f"L{li}.{k}"] for k in G.LAYER_KEYS}
                             for li in range(w["layers"])]}
        gcfg = dict(b=w["b"], s=w["s"], heads=w["heads"], N=w["N"])
        run = lambda: G.gpt_train(params, ids, tg, gcfg, 1)
        flops = M  # tokens per step
        metric = "small GPT training tokens/s (vocabulary-parallel embedding + cross-entropy)"
        unit, scale = "tokens/s", 1.0
        sample = "fp64 oracle training step (forward, backward, AdamW) on the whole batch"
    elif w.get("layer"):
        from oracle import tp_oracle as O
        hin = layer_inputs(w, 0)
        f64 = lambda a: synth.to_f64(a, "bf16") if a.dtype == np.uint16 else a.astype(np.float64)
        p = {k: f64(hin[k]) for k in ("Wqkv", "Wo", "W1", "W2", "gamma1", "beta1", "gamma2",
                                      "beta2")}
        x, dout = f64(hin["x"]), f64(hin["dout"])
        run = lambda: O.layer_bwd(x, w["b"], w["s"], p, w["heads"], w["N"], dout)
        flops = layer_flops(w)
        sample = "fp64 oracle layer forward+backward on the whole workload per step"
    else:
        hostin = {"X": synth.normal((M, h), synth.seed_of(c, "X"), 1.0, dtp),
                  "dZ": synth.normal((M, h), synth.seed_of(c, "dZ"), 1.0, dtp),
                  "W1": synth.normal((h, f), synth.seed_of(c, "Wg"), 0.02, dtp),
                  "W1u": (synth.normal((h, f), synth.seed_of(c, "Wu"), 0.02, dtp)
                          if w["act"] == "swiglu" else None),
                  "W2": synth.normal((f, h), synth.seed_of(c, "Wd"), 0.02, dtp)}
        Wf = _weights_f64(hostin, dtp)
        rows = min(args.ref_rows, M)
        if w.get("sp"):
            rows = max(w["N"], rows - rows % w["N"])
        run = lambda: _oracle_sample(w, hostin, rows, Wf)
        flops = mlp_flops(w, rows)
        sample = (f"fp64 oracle forward+backward on {rows} of {M} token rows per step, full "
                  f"weights; FLOPs scaled by the row fraction")
    t_gen = time.time() - t_gen
    for _ in range(args.warmup):
        run()
    c0, t0 = time.process_time(), time.perf_counter()
    for _ in range(args.steps):
        run()
    dt, dc = (time.perf_counter() - t0) / args.steps, (time.process_time() - c0) / args.steps
    val = flops / dt / scale
    print(json.dumps({
        "metric": metric, "value": round(val, 6), "unit": unit, "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "impl": "reference",
        "config": {"workload": w["desc"], "tokens": M, "h": h, "ffn": f, "shards": w["N"],
                   "act": w["act"]},
        "cpu_baseline": {"value": round(val, 6), "unit": unit, "kind": "oracle",
                         "cores": len(os.sched_getaffinity(0)),
                         "threads_effective": round(dc / dt, 1), "sample": sample},
        "e2e": {"value": round(val, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "input_gen_s": round(t_gen, 1),
    }), flush=True)


def _ref_line(args, metric, val, unit, dt, dc, sample, config, t_gen):
    ws_, _, _ = dist_env()
    print(json.dumps({
        "metric": metric, "value": round(val, 6), "unit": unit, "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "impl": "reference", "config": config,
        "cpu_baseline": {"value": round(val, 6), "unit": unit, "kind": "oracle",
                         "cores": len(os.sched_getaffinity(0)),
                         "threads_effective": round(dc / dt, 1), "sample": sample},
        "e2e": {"value": round(val, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "input_gen_s": round(t_gen, 1)}), flush=True)


def _time_ref(args, run):
    for _ in range(args.warmup):
        run()
    c0, t0 = time.process_time(), time.perf_counter()
    for _ in range(args.steps):
        run()
    return (time.perf_counter() - t0) / args.steps, (time.process_time() - c0) / args.steps


def run_reference_hbm(args):
    """Oracle arms of the HBM-bound lines, each on a bounded sample (rank 0 only):
    c4 -- the fp64 SwiGLU decode forward of one token on one shard's slice of the
    weights (1/8 of them); vocab-ce -- the vocabulary-parallel cross-entropy forward +
    backward on 32 of the 8192 rows. GB/s of the bf16 bytes the GPU line counts, scaled
    to the sample."""
    _, rank, _ = dist_env()
    if rank != 0:
        return
    from attention_gemms_gb300 import synth
    t_gen = time.time()
    if args.workload == "c4":
        from oracle import tp_oracle as O
        h, f, N = DECODE["h"], DECODE["f"], DECODE["N"]
        fs = f // N
        c = DECODE["cfg"]
        x = synth.to_f64(synth.normal((1, h), synth.seed_of(c, "X"), 1.0, "bf16"), "bf16")
        Wg = synth.to_f64(synth.normal((h, fs), synth.seed_of(c, "Wg"), 0.02, "bf16"), "bf16")
        Wu = synth.to_f64(synth.normal((h, fs), synth.seed_of(c, "Wu"), 0.02, "bf16"), "bf16")
        Wd = synth.to_f64(synth.normal((fs, h), synth.seed_of(c, "Wd"), 0.02, "bf16"), "bf16")
        run = lambda: O.mlp_swiglu_fwd(x, Wg, Wu, Wd, 1)
        nbytes = 3 * h * fs * 2
        metric = METRIC  # the decode line's metric (its value is GB/s)
        sample = (f"fp64 oracle SwiGLU forward of 1 token on one shard's slice ({fs} of {f} "
                  f"columns) of the weights; bytes = that slice in bf16")
        config = {"workload": DECODE["desc"], "tokens": 1}
    else:
        from oracle import gpt_oracle as G
        rows, v, N = 32, 50304, 8
        L = synth.to_f64(synth.normal((rows, v), 9001, 2.0, "bf16"), "bf16")
        tg = synth.integers((rows,), 9002, v)

        def run():
            _, lse, _, _ = G.vocab_ce_fwd(L, tg, N)
            G.vocab_ce_bwd(L, tg, lse, N, 1.0 / rows)
        nbytes = 3 * rows * v * 2
        metric = "vocabulary-parallel cross-entropy fwd+bwd GB/s"
        sample = f"fp64 oracle cross-entropy forward + backward on {rows} of 8192 rows (v={v}, N={N})"
        config = {"workload": "vocab-ce", "M": 8192, "vocab": v, "N": N}
    t_gen = time.time() - t_gen
    dt, dc = _time_ref(args, run)
    _ref_line(args, metric, nbytes / dt / 1e9, "GB/s", dt, dc, sample, config, t_gen)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="c5", choices=sorted(WORKLOADS) + ["c4", "vocab-ce"],
                    help="c5 (default): large SwiGLU MLP; c3: GELU MLP; c2: page-2 layer; "
                         "c1: tiny fp32 MLP; c4: decode sweep only; c5-2k: profiling case; "
                         "c3-sp: sequence-parallel MLP block; gpt: small GPT training; "
                         "gqa: head-sharded grouped-query attention block; vocab-ce: the "
                         "vocabulary-parallel cross-entropy alone (M=8192, v=50304, N=8)")
    ap.add_argument("--mode", default="splitk", choices=["splitk", "buffers"],
                    help="shard-sum variant of the main line (the other is timed beside it)")
    ap.add_argument("--no-variants", dest="variants", action="store_false", default=True,
                    help="time only --mode, not the other shard-sum variant")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode", dest="decode", action="store_true", default=True,
                    help="also run the decode GEMV sweep (default)")
    ap.add_argument("--no-decode", dest="decode", action="store_false")
    ap.add_argument("--no-shard-sum", dest="shard_sum", action="store_false", default=True,
                    help="skip the shard-sum / fused reduce + LayerNorm measurement")
    ap.add_argument("--decode-warmup-ms", type=float, default=200.0,
                    help="minimum warm-up time of each decode token count (clocks ramp up)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference" and args.workload in ("c4", "vocab-ce"):
        return run_reference_hbm(args)
    if args.workload == "c4":
        return run_decode_only(args)
    if args.workload == "vocab-ce":
        return run_vocab_ce_only(args)
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
