"""Benchmark of the indexer backward on GB300: one step = score-grad + gemm
stage (dQ, dW, dK) over one batch of seeded synthetic inputs of the anchor
workload (B=1, H=64, D=128, S_k=4096, S_q=8192, topk=1024, causal top-k ids).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--mode atomic|det]
                  [--workload anchor] [--impl reference]

Prints one JSON line (rank 0).  `value` is nominal gemm-stage TFLOP/s of the
whole step (6*S_q*topk*H*D per step, all ranks), inputs resident in HBM;
`e2e` is the same metric through the public API with pinned-host inputs and
results copied inside the timed region; `roofline` covers the gemm-stage
kernel; `cpu_baseline` times the fp64 oracle on a bounded row sample.
`--impl reference` times the oracle itself as the reference arm.
`other_configs` adds, measured in the same run, the gemm-stage and score-grad
kernel times of the other contract configurations (both dK modes of the
anchor and the window workload, the S_q = 4096 top-k 512 shape, the dense
variant).
With N > 1 every rank runs an independent replica (weak scaling); the path
has no exchange step between replicas.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "indexer-bwd kernel µs & TFLOP/s (frac of bf16 peak), H64 D128 Sq8192 topk1024"

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# ncu captures of the anchor workload in atomic mode, each kept with the hash
# of the source files of the kernels it measured; a change to any of those
# files makes the figure stale and the benchmark then reports null.  The
# captures and their commands are summarised under profiles/.
# the gemm stage's kernels (k conversion, kernel choice, union pass, blocked
# kernel, the per-row kernel's empty launch) and the code they include
GEMM_FILES = ("blk.cu", "blk.h", "blk_pipe.cuh", "blk_pipe.cu", "gemm.cu", "kcommon.cuh", "ptx.cuh", "internal.h")
SCORE_GRAD_FILES = ("score_grad.cu",)
PROFILED_TRAFFIC = {
    # k_to_f16 + select + union + blk + (exiting) per-row kernels of one gemm-stage call
    ("anchor", "atomic", "gemm_stage"): ("45422db0c20962a5d1f7228ba3177a2790d4127ccc7412b939d244f3d7afa49a", 1.062e6 + 4.211e6 + 83.894e6 + 423.134e6 + 0.068e6),
    ("anchor", "atomic", "score_grad"): ("56e45ec7b1c5fb62867535e1ef1414916bef85b0738b22445c9f9c2b9e269420", 102.819e6),
}


def sources_hash(files) -> str:
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "sparse_attention_indexer_bwd_gb300", "csrc")
    for f in files:
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(workload: str, mode: str) -> dict:
    out = {}
    for kernel, files in (("gemm_stage", GEMM_FILES), ("score_grad", SCORE_GRAD_FILES)):
        entry = PROFILED_TRAFFIC.get((workload, mode, kernel))
        if entry and sources_hash(files) == entry[0]:
            out[kernel] = entry[1]
    return out


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="anchor", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mode", default="atomic", choices=["atomic", "det"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-extra", action="store_true", help="skip the other contract configurations")
    ap.add_argument("--extra-steps", type=int, default=20)
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]), "hbm_gbs": float(p["hbm_gbs"]), "src": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "src": "fallback"}


# ------------------------------------------------------------ distributed ---

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, td, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if td is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def dist_init(ws, backend):
    import torch.distributed as td
    if ws > 1 and not td.is_initialized():
        td.init_process_group(backend)
    return td if ws > 1 else None


# ------------------------------------------------------------ oracle legs ---

def oracle_sample(wl: synth.Workload, x: dict, I: np.ndarray, rows: np.ndarray):
    """Runs the oracle's score-grad and gemm stage on the given query rows
    (B == 1 workloads).  Returns the nominal FLOPs of the sample."""
    import oracle
    q = x["q"][:, rows]
    w = x["w"][:, rows]
    if wl.dense:
        raise ValueError("row samples of the dense workload are not supported")
    idx = x["idx"][:, rows]
    dI = oracle.score_grad_sparse(I[:, rows], x["attn"][:, rows], idx, wl.S_k)
    # the scale 1/S_q of the full problem: score_grad_sparse divides by the
    # sample's row count, so rescale to the workload's
    dI *= len(rows) / wl.S_q
    oracle.gemm_sparse(q, x["k"], w, dI, idx, wl.S_k)
    return 6.0 * len(rows) * wl.topk * wl.H * wl.D


def cpu_baseline(wl, x, I, seconds):
    import oracle
    cores = oracle.set_threads(0)
    rng = np.random.default_rng(0)
    order = rng.permutation(wl.S_q)
    flops = 0.0
    done = 0
    t0 = time.perf_counter()
    chunk = 256
    while done < wl.S_q and time.perf_counter() - t0 < seconds:
        rows = np.sort(order[done:done + chunk])
        flops += oracle_sample(wl, x, I, rows)
        done += len(rows)
    el = time.perf_counter() - t0
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} of {wl.S_q} query rows (random, full rows), score-grad + gemm stage, fp64, "
                      f"{el:.1f} s"}


def run_reference(args, wl):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    x = synth.make_inputs(wl)
    # index_score = the forward logits, from the oracle's own forward (the
    # reference arm runs nothing but the oracle)
    rng = np.random.default_rng(1)
    cores = oracle.set_threads(0)
    # calibrate: seconds per row, then size each step's sample so that the
    # whole run takes about a minute
    cal = np.sort(rng.permutation(wl.S_q)[:32])
    Ic = np.zeros((wl.B, wl.S_q, wl.topk), np.float32)
    Ic[:, cal] = oracle.forward_sparse(x["q"][:, cal], x["k"], x["w"][:, cal], x["idx"][:, cal], wl.S_k)
    t0 = time.perf_counter()
    oracle_sample(wl, x, Ic, cal)
    per_row = (time.perf_counter() - t0) / len(cal)
    total_steps = args.steps + args.warmup
    nrows = int(max(8, min(wl.S_q, 60.0 / max(total_steps, 1) / max(per_row, 1e-6))))
    times, flops = [], 0.0
    for s in range(total_steps):
        rows = np.sort(rng.permutation(wl.S_q)[:nrows])
        I = np.zeros((wl.B, wl.S_q, wl.topk), np.float32)
        I[:, rows] = oracle.forward_sparse(x["q"][:, rows], x["k"], x["w"][:, rows], x["idx"][:, rows], wl.S_k)
        t0 = time.perf_counter()
        f = oracle_sample(wl, x, I, rows)
        el = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(el)
            flops += f
    total = sum(times)
    val = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / max(len(times), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: B={wl.B} H={wl.H} D={wl.D} S_q={wl.S_q} S_k={wl.S_k} topk={wl.topk}",
                   "sample_rows_per_step": nrows},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{nrows} random full query rows per step of {wl.S_q}, "
                                   "score-grad + gemm stage, fp64"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm ---

class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                smax = float(row[2])
            except ValueError:
                continue
            for n, v in zip(names, row[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# The other contract configurations, measured in the same run (gemm-stage
# and score-grad kernel times only; no end-to-end or CPU legs).
EXTRA_CONFIGS = (("anchor", "det"), ("sq4096_topk512", "atomic"), ("window_topk2048", "atomic"),
                 ("window_topk2048", "det"), ("dense_s4096", "atomic"), ("dense_s4096", "det"))


def measure_config(ibwd, torch, dev, name, mode_name, steps, warmup, pk):
    """Score-grad and gemm-stage kernel times of one workload and dK mode,
    timed with CUDA events on the launching stream over `steps` steps (each
    with a fresh attn_score copy; inputs larger than L2)."""
    wl = synth.WORKLOADS[name]
    mode = ibwd.IBWD_DK_DETERMINISTIC if mode_name == "det" else ibwd.IBWD_DK_ATOMIC
    x = synth.make_inputs(wl)
    q = torch.from_numpy(x["q"].view(np.int16)).to(dev).view(torch.bfloat16)
    k = torch.from_numpy(x["k"].view(np.int16)).to(dev).view(torch.bfloat16)
    w = torch.from_numpy(x["w"]).to(dev)
    idx = None if wl.dense else torch.from_numpy(x["idx"]).to(dev)
    attn0 = torch.from_numpy(x["attn"]).to(dev)
    I = ibwd.indexer_fwd_dense(q, k, w) if wl.dense else ibwd.indexer_fwd(q, k, w, idx)
    B, S_q, H, D = q.shape
    dq = torch.empty((B, S_q, H, D), dtype=torch.float32, device=dev)
    dw = torch.empty((B, S_q, H), dtype=torch.float32, device=dev)
    dk = torch.empty((B, wl.S_k, D), dtype=torch.float32, device=dev)
    wsb = torch.empty(ibwd.indexer_bwd_dense_gemm_workspace_size(B, S_q, H, D, mode) if wl.dense else
                      ibwd.indexer_bwd_gemm_workspace_size(B, S_q, wl.S_k, H, D, wl.topk, mode),
                      dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    attn = [attn0.clone() for _ in range(2)]
    sg, gm = [], []
    for i in range(warmup + steps):
        a = attn[i & 1]
        a.copy_(attn0)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        zero = dk if mode == ibwd.IBWD_DK_ATOMIC else None
        ev[0].record(stream)
        if wl.dense:
            ibwd.indexer_bwd_dense_score_grad(I, a, 1.0, zero, stream)
        else:
            ibwd.indexer_bwd_score_grad(I, a, idx, wl.S_k, 1.0, zero, stream)
        ev[1].record(stream)
        if wl.dense:
            ibwd.indexer_bwd_dense_gemm(q, k, w, a, dq, dw, dk, mode, wsb, stream)
        else:
            ibwd.indexer_bwd_gemm(q, k, w, a, idx, dq, dw, dk, mode, wsb, stream)
        ev[2].record(stream)
        torch.cuda.synchronize()
        if i >= warmup:
            sg.append(ev[0].elapsed_time(ev[1]))
            gm.append(ev[1].elapsed_time(ev[2]))
    st = ibwd.indexer_bwd_last_device_status(stream)
    if st != ibwd.IBWD_OK:
        raise SystemExit(f"device status after {name}/{mode_name}: {ibwd.status_string(st)}")
    flops = wl.flops()
    valid = 1.0 if wl.dense else float((x["idx"] >= 0).mean())
    zero_bytes = 4.0 * wl.B * wl.S_k * wl.D if mode == ibwd.IBWD_DK_ATOMIC else 0.0
    sg_bytes = (8.0 * wl.B * wl.S_q * (wl.S_q + 1) / 2 + 4.0 * wl.B * wl.S_q * wl.S_q if wl.dense else
                16.0 * wl.B * wl.S_q * wl.topk) + zero_bytes
    gmed = float(np.median(gm))
    sgmed = float(np.median(sg))
    return {
        "workload": f"{wl.name}: B={wl.B} H={wl.H} D={wl.D} S_q={wl.S_q} S_k={wl.S_k} "
                    + ("every causal key (dense)" if wl.dense else f"topk={wl.topk}, {wl.ids} top-k ids"),
        "dk_mode": mode_name, "steps": steps,
        "gemm_stage_us": {"median": 1e3 * gmed, "min": 1e3 * float(np.min(gm)), "p90": 1e3 * float(np.percentile(gm, 90))},
        "tflops": flops / (gmed * 1e-3) / 1e12,
        "frac_nominal": flops / (gmed * 1e-3) / 1e12 / pk["bf16_tflops"],
        "frac_valid_slots": valid * flops / (gmed * 1e-3) / 1e12 / pk["bf16_tflops"],
        "valid_slot_fraction": round(valid, 4),
        "score_grad_us": 1e3 * sgmed,
        "score_grad_gbs": sg_bytes / (sgmed * 1e-3) / 1e9,
    }


def run_ours(args, wl):
    import torch
    import sparse_attention_indexer_bwd_gb300 as ibwd

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    td = dist_init(ws, "nccl")
    mode = ibwd.IBWD_DK_DETERMINISTIC if args.mode == "det" else ibwd.IBWD_DK_ATOMIC

    # ---- inputs (seeded, synthetic; resident in HBM before timing)
    x = synth.make_inputs(wl)
    q = torch.from_numpy(x["q"].view(np.int16)).to(dev).view(torch.bfloat16)
    k = torch.from_numpy(x["k"].view(np.int16)).to(dev).view(torch.bfloat16)
    w = torch.from_numpy(x["w"]).to(dev)
    idx = None if wl.dense else torch.from_numpy(x["idx"]).to(dev)
    attn0 = torch.from_numpy(x["attn"]).to(dev)
    # index_score: the forward of the same q, k, w (input preparation, untimed)
    I = ibwd.indexer_fwd_dense(q, k, w) if wl.dense else ibwd.indexer_fwd(q, k, w, idx)
    B, S_q, H, D = q.shape
    dq = torch.empty((B, S_q, H, D), dtype=torch.float32, device=dev)
    dw = torch.empty((B, S_q, H), dtype=torch.float32, device=dev)
    dk = torch.empty((B, wl.S_k, D), dtype=torch.float32, device=dev)
    wsb = torch.empty(ibwd.indexer_bwd_dense_gemm_workspace_size(B, S_q, H, D, mode) if wl.dense else
                      ibwd.indexer_bwd_gemm_workspace_size(B, S_q, wl.S_k, H, D, wl.topk, mode),
                      dtype=torch.uint8, device=dev)
    # score-grad overwrites attn_score with dI: every step gets its own copy
    nbuf = args.steps + args.warmup
    attn = [attn0.clone() for _ in range(nbuf)]
    stream = torch.cuda.current_stream()
    # this library's kernels per step: score-grad, k copy, then
    # sparse: kernel choice, union pass, blocked and per-row kernels (atomic)
    # or union pass, key scan, placement, blocked kernel, segment sum (det);
    # dense: scale pass, blocked kernel (+ key offsets, segment sum: det)
    if wl.dense:
        launches_per_step = 4 if mode == ibwd.IBWD_DK_ATOMIC else 6
    else:
        launches_per_step = 6 if mode == ibwd.IBWD_DK_ATOMIC else 7

    def step(a, ev=None):
        if ev is not None:
            ev[0].record(stream)
        zero = dk if mode == ibwd.IBWD_DK_ATOMIC else None
        if wl.dense:
            ibwd.indexer_bwd_dense_score_grad(I, a, 1.0, zero, stream)
        else:
            ibwd.indexer_bwd_score_grad(I, a, idx, wl.S_k, 1.0, zero, stream)
        if ev is not None:
            ev[1].record(stream)
        if wl.dense:
            ibwd.indexer_bwd_dense_gemm(q, k, w, a, dq, dw, dk, mode, wsb, stream)
        else:
            ibwd.indexer_bwd_gemm(q, k, w, a, idx, dq, dw, dk, mode, wsb, stream)
        if ev is not None:
            ev[2].record(stream)

    def whole(a):
        ibwd.indexer_backward(q, k, w, I, a, idx, dk_mode=mode, workspace=wsb, out=(dq, dw, dk), stream=stream)

    # ---- timed region: K steps of the whole backward through its one-call
    # entry point (indexer_bwd: the score-grad, then the gemm stage's kernels
    # launched programmatically behind it), barrier + synchronize on both sides
    for i in range(args.warmup):
        whole(attn[i])
    st = ibwd.indexer_bwd_last_device_status(stream)
    if st != ibwd.IBWD_OK:
        raise SystemExit(f"device status after warm-up: {ibwd.status_string(st)}")
    clocks = Clocks(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                    if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local)
    if td:
        td.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        whole(attn[args.warmup + i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if td:
        td.barrier()
    total_ms = t_start.elapsed_time(t_end)
    st = ibwd.indexer_bwd_last_device_status(stream)
    if st != ibwd.IBWD_OK:
        raise SystemExit(f"device status after the timed region: {ibwd.status_string(st)}")
    if td:
        total_ms = max_over_ranks(total_ms, td, dev)

    # the same steps as the pair of calls with events between the two
    # kernels: the per-kernel split (an event between them also ends their
    # programmatic overlap, so the pair's step is a little longer)
    for a in attn:
        a.copy_(attn0)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        step(attn[i])
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for i in range(args.steps):
        step(attn[args.warmup + i], evs[i])
    p1.record(stream)
    torch.cuda.synchronize()
    pair_ms = p0.elapsed_time(p1) / args.steps
    sg_ms = [e[0].elapsed_time(e[1]) for e in evs]
    gm_ms = [e[1].elapsed_time(e[2]) for e in evs]
    st = ibwd.indexer_bwd_last_device_status(stream)
    if st != ibwd.IBWD_OK:
        raise SystemExit(f"device status after the pair-of-calls steps: {ibwd.status_string(st)}")
    del attn

    flops = wl.flops()
    ms_step = total_ms / args.steps
    value = ws * flops / (ms_step * 1e-3) / 1e12
    pk = peaks()
    gm_avg = statistics.mean(gm_ms)
    sg_avg = statistics.mean(sg_ms)
    achieved = flops / (gm_avg * 1e-3) / 1e12
    zero_bytes = 4.0 * wl.B * wl.S_k * wl.D if mode == ibwd.IBWD_DK_ATOMIC else 0.0
    if wl.dense:
        valid = (wl.S_q + 1) / (2.0 * wl.S_q)
        # read index_score and attn_score on and below the diagonal, write the full dI rows
        sg_bytes = 8.0 * wl.B * wl.S_q * (wl.S_q + 1) / 2 + 4.0 * wl.B * wl.S_q * wl.S_q + zero_bytes
    else:
        valid = float((x["idx"] >= 0).mean())
        sg_bytes = 16.0 * wl.B * wl.S_q * wl.topk + zero_bytes

    # ---- end to end through the public API from pinned host memory
    e2e = None
    if not args.no_e2e:
        arrays = [("q", x["q"].view(np.int16)), ("k", x["k"].view(np.int16)), ("w", x["w"]), ("attn", x["attn"])]
        if not wl.dense:
            arrays.append(("idx", x["idx"]))
        h = {n: torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for n, a in arrays}
        h["I"] = I.cpu().pin_memory()
        # Steps are pipelined the way a training loop would run them: step i+1's
        # inputs are copied in while step i computes and step i-1's results are
        # read back, on three streams with two device buffer sets.  Every step
        # still moves its own inputs in and its own results out inside the
        # timed region.
        nb = 2
        hout = [[torch.empty(t.shape, dtype=torch.float32).pin_memory() for t in (dq, dw, dk)] for _ in range(nb)]
        dbuf = [{n: torch.empty(t.shape, dtype=t.dtype, device=dev) for n, t in h.items()} for _ in range(nb)]
        dout = [[torch.empty_like(t) for t in (dq, dw, dk)] for _ in range(nb)]
        h2d = sum(t.numel() * t.element_size() for t in h.values())
        d2h = sum(t.numel() * t.element_size() for t in hout[0])
        ksteps = max(4, min(20, args.steps))
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(nb)]
        ev_comp = [torch.cuda.Event() for _ in range(nb)]
        ev_out = [torch.cuda.Event() for _ in range(nb)]
        started = [False] * nb

        def e2e_step(i):
            b = i % nb
            if started[b]:
                s_in.wait_event(ev_comp[b])     # the inputs of buffer b were consumed
                stream.wait_event(ev_out[b])    # its results were read back
            with torch.cuda.stream(s_in):
                for n, t in h.items():
                    dbuf[b][n].copy_(t, non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            d = dbuf[b]
            ibwd.indexer_backward(d["q"].view(torch.bfloat16), d["k"].view(torch.bfloat16), d["w"], d["I"],
                                  d["attn"], d.get("idx"), dk_mode=mode, workspace=wsb, out=tuple(dout[b]),
                                  stream=stream)
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for ho, do in zip(hout[b], dout[b]):
                    ho.copy_(do, non_blocking=True)
            ev_out[b].record(s_out)
            started[b] = True

        for i in range(nb):
            e2e_step(i)
        torch.cuda.synchronize()
        if td:
            td.barrier()
        t0 = time.perf_counter()
        for i in range(ksteps):
            e2e_step(nb + i)
        torch.cuda.synchronize()
        e_ms = (time.perf_counter() - t0) * 1e3 / ksteps
        if td:
            e_ms = max_over_ranks(e_ms, td, dev)
        e2e = {"value": ws * flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms, "steps": ksteps,
               "note": "host wall clock over the steps; copies in, compute and copies out of consecutive "
                       "steps overlap on three streams"}

    # the forward kernel on its own (not part of the step): CUDA events around
    # each launch, inputs resident
    fwd_flops = (2.0 * wl.B * wl.H * wl.D * wl.S_q * (wl.S_q + 1) / 2.0 if wl.dense else
                 2.0 * wl.B * wl.S_q * wl.topk * wl.H * wl.D)
    fwd_ms = []
    for it in range(13):
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        if wl.dense:
            ibwd.indexer_fwd_dense(q, k, w, out=I, stream=stream)
        else:
            ibwd.indexer_fwd(q, k, w, idx, out=I, stream=stream)
        f1.record(stream)
        torch.cuda.synchronize()
        if it >= 3:
            fwd_ms.append(f0.elapsed_time(f1))
    fwd_avg = statistics.mean(fwd_ms)
    forward = {"us": 1e3 * fwd_avg, "tflops": fwd_flops / (fwd_avg * 1e-3) / 1e12,
               "note": "forward kernel alone (index_score), 2*slots*H*D FLOP; not part of the step"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not wl.dense:
        cpu = cpu_baseline(wl, x, I.cpu().numpy(), args.cpu_seconds)

    # the other contract configurations (one GPU runs; rank 0 of a replica job)
    extra = None
    if rank == 0 and not args.no_extra:
        extra = []
        for name, mname in EXTRA_CONFIGS:
            if name == wl.name and mname == args.mode:
                continue
            extra.append(measure_config(ibwd, torch, dev, name, mname, args.extra_steps, 3, peaks()))
            torch.cuda.empty_cache()

    if rank != 0:
        return
    traffic = profiled_traffic(wl.name, args.mode)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 tensor-core operands, fp32 accumulate (bf16 inputs)",
        "data": "synthetic (seeded; index_score = this library's forward of the seeded q, k, w)",
        "config": {"workload": f"{wl.name}: B={wl.B} H={wl.H} D={wl.D} S_q={wl.S_q} S_k={wl.S_k} "
                               + ("every causal key (dense)" if wl.dense else f"topk={wl.topk}, {wl.ids} top-k ids"),
                   "dk_mode": args.mode, "l2": "inputs larger than L2 (q alone is 134 MB); "
                                               "a fresh attn_score copy per step",
                   "valid_slot_fraction": round(valid, 4)},
        "us_per_step": 1e3 * ms_step,
        # valid slots only (the dense count is already over s <= t)
        "tflops_valid_slots": value * (1.0 if wl.dense else valid),
        "kernels_us": {"score_grad": 1e3 * sg_avg, "gemm_stage": 1e3 * gm_avg},
        "kernels_us_stats": {name: {"median": 1e3 * float(np.median(v)), "min": 1e3 * float(np.min(v)),
                                    "p90": 1e3 * float(np.percentile(v, 90))}
                             for name, v in (("score_grad", sg_ms), ("gemm_stage", gm_ms))},
        "score_grad_gbs": sg_bytes / (sg_avg * 1e-3) / 1e9,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / pk["bf16_tflops"], "frac_valid_slots": achieved * valid / pk["bf16_tflops"],
                     "traffic": traffic.get("gemm_stage"),
                     "note": f"gemm-stage call (fp16 copy of k + main kernel), nominal 6*S_q*topk*H*D FLOP; "
                             f"peak = {pk['src']} dense bf16 burst (fp16 dense rate is the same)"},
        "roofline_score_grad": {"bound": "hbm", "achieved": sg_bytes / (sg_avg * 1e-3) / 1e9,
                                "peak": pk["hbm_gbs"], "unit": "GB/s",
                                "frac": sg_bytes / (sg_avg * 1e-3) / 1e9 / pk["hbm_gbs"],
                                "traffic": traffic.get("score_grad"), "algorithmic_bytes": sg_bytes},
        "pair_of_calls": {"us_per_step": 1e3 * pair_ms, "tflops": flops / (pair_ms * 1e-3) / 1e12,
                          "steps": args.steps,
                          "note": "the same steps as indexer_bwd_score_grad + indexer_bwd_gemm with events between "
                                  "them (kernels_us), timed after the region above"},
        "forward": forward,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "other_configs": extra,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
