"""Benchmark of one DFlash 2 draft-verify cycle on GB300.

A step is one whole cycle for B sequences: conv + LM head + top-16 +
logsumexp, pair scores, lattice walk, verify with residual / bonus draw —
the four calls of the C ABI.  Default workload: B=32, K=8, V=151936,
H=2048, r=256, bf16, T=1 (the b32k8 synthetic workload).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl ours|reference]

Prints one JSON line.  ``value`` = draft-verify cycles/s over all ranks
(device-timed, inputs resident in HBM); ``e2e`` = the same through the
public API with host buffers (H2D of the step's inputs and D2H of its
results inside the timed region).  Under torchrun each rank runs its own
batch (replicas, weak scaling) and rank 0 reports.  ``--impl reference``
times the CPU oracle on a bounded sample of the same workload.
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


def _set_blas_threads(argv):
    """The oracle's BLAS thread count, fixed before numpy loads: the value
    after --oracle-threads, else every host core for the oracle runs
    (--impl reference, --oracle-sample)."""
    n = None
    if "--oracle-threads" in argv:
        n = argv[argv.index("--oracle-threads") + 1]
    elif "reference" in argv or "--oracle-sample" in argv:
        n = str(os.cpu_count())
    if n is not None:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS",
                    "MKL_NUM_THREADS"):
            os.environ[var] = n


if __name__ == "__main__":
    _set_blas_threads(sys.argv)

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

C = 16
GRAPH_STEPS = 100    # cycles captured per CUDA graph in the timed region
METRIC = ("draft-verify cycles/s and verified tokens/s at B=32,K=8,V=151936;"
          " % HBM/TC roofline")
UNIT = "cycles/s"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="b32k8")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="bounded CPU work for the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", action="store_true",
                    help="(internal) time the oracle on a sample of the "
                         "workload and print its JSON; run as a child "
                         "process so that its thread count is its own")
    ap.add_argument("--oracle-threads", type=int, default=None)
    ap.add_argument("--sweep", default=None,
                    help="time the sweep grid instead (one JSON line per "
                         "point): 'all' or a comma list of point names")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)
# --------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(base: int, rank: int) -> int:
    """Philox seed of a rank: every replica draws its own uniforms."""
    return base * 1000003 + rank


def aggregate(cycles_per_rank: int, seconds_per_rank, world: int):
    """Whole-job throughput: all ranks' cycles over the slowest rank."""
    t = max(seconds_per_rank)
    return world * cycles_per_rank / t, t


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------
# peaks and clocks
# --------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling, started ahead of the timed
    region; only samples whose own timestamps fall inside [mark_start(),
    mark_end()] are summarised."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv",
                                                    delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f")
                if self.t0 and self.t1 and not (self.t0 <= ts <= self.t1):
                    continue
                sm.append(float(r[2]))
                smax.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# workload synthesis (outside every timed region)
# --------------------------------------------------------------------------
def synth_target_torch(w, x, dev):
    """Target logits of workload ``w``: its transform of the drafter's fp32
    logits, which are computed here with plain torch ops on the device
    (input synthesis only)."""
    import torch
    torch.backends.cuda.matmul.allow_tf32 = False
    h = x["h"].to(dev).float()                       # [B, K+1, H]
    H = w.H
    if x["w_conv"] is not None:
        wc = x["w_conv"].to(dev).float()
        w0 = h @ wc[:H].T
        w1 = h @ wc[H:].T
        prev = torch.zeros_like(h)
        prev[:, 1:] = h[:, :-1]
        y = w0 * h + w1 * prev
    else:
        y = h
    if w.dtype == "bf16":
        y = y.to(torch.bfloat16)
    y = y.float().reshape(-1, H)
    wl = x["w_lm"].to(dev)
    U = torch.empty(y.shape[0], w.V, dtype=torch.float32, device=dev)
    step = 16384
    for v0 in range(0, w.V, step):
        U[:, v0:v0 + step] = y @ wl[v0:v0 + step].float().T
    d = U.reshape(w.B, w.K + 1, w.V).cpu().numpy()
    return synth.target_logits(w, d)


def bench_config(w, world: int) -> dict:
    """The workload as both arms report it (same keys and values)."""
    return {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "H": w.H,
            "r": w.r, "T": w.T, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (W_lm streamed each cycle)",
            "recipe": synth.describe(w)}


# --------------------------------------------------------------------------
# algorithmic bytes and flops per launch
# --------------------------------------------------------------------------
def lmhead_algorithmic(w):
    """Bytes and flops of one LM-head launch (the step's dominant kernel):
    read W_lm and y once (as E4M3 codes plus row scales for the 8-bit
    head), write topv/topi/lse."""
    es = 1 if w.lm_e4m3 else (2 if w.dtype == "bf16" else 4)
    M = w.M
    by = w.V * w.H * es + M * w.H * es + M * (C * 8 + 4)
    if w.lm_e4m3:
        by += (w.V + M) * 4
    fl = 2.0 * M * w.V * w.H
    return by, fl


def verify_roofline(w, n_mean, verify_us, hbm_gbs):
    """The verify stage against the HBM rate.  It reads rows 0..n of each
    sequence (n accepted drafts), the draw row again, and of the later rows
    only what it streams before the earlier rejection is known: the main
    figure is the bytes the accepted lengths need; every target row's bytes
    (what a verify reading all rows would move in the same time) beside
    it."""
    vb = verify_algorithmic(w, n_mean)
    ab = w.B * (w.K + 1) * w.V * 4
    t = verify_us * 1e-6
    return {"bytes": vb, "GB/s": vb / t / 1e9,
            "frac": vb / t / 1e9 / hbm_gbs,
            "all_rows_bytes": ab, "all_rows_GB/s": ab / t / 1e9,
            "frac_all_rows": ab / t / 1e9 / hbm_gbs,
            "note": "rows after a sequence's first rejection stop being "
                    "read once it is known; bytes = rows 0..n of each "
                    "sequence and the draw row again; all_rows_bytes = "
                    "every B*(K+1) target row"}


def verify_algorithmic(w, n_mean):
    """Bytes the verify needs: target rows 0..n of each sequence (n
    accepted drafts), at T > 0 the draw row once more (the inverse CDF
    walks it after its total is known), plus the drafts, candidates and
    q."""
    rows = w.B * (n_mean + 1) + (w.B if w.T > 0 else 0)
    return rows * w.V * 4 + w.M * C * 8 + w.M * 4


# --------------------------------------------------------------------------
# CPU oracle timing (bounded sample of the same workload)
# --------------------------------------------------------------------------
def oracle_w8(w, x):
    """The oracle's E4M3 codes and scales of W_lm for an 8-bit-head
    workload and their dequantized matrix (weight preparation, done once,
    outside the timed sample, as the CUDA path quantizes W_lm once)."""
    if not w.lm_e4m3:
        return None
    import oracle
    codes, scale = oracle.quantize_e4m3_rows(x["w_lm"].float().numpy())
    return codes, scale, oracle.dequantize_e4m3_rows(codes, scale)


def time_oracle(w, x, L, seconds: float, seed: int, w8=None):
    """Whole cycles of the oracle on the first sequences of the workload,
    one sequence at a time, until ``seconds`` of work; returns cycles/s
    scaled to the full batch, and a description of the sample."""
    import oracle
    f64 = lambda t: None if t is None else t.float().numpy().astype(np.float64)
    W = {k: f64(x[k]) for k in ("w_conv", "w_lm", "w_gate", "e_in", "e_out")}
    h = f64(x["h"])[:, :w.K]
    Lc = L.numpy() if hasattr(L, "numpy") else L
    anchor = x["anchor"].numpy()
    done, t0 = 0, time.perf_counter()
    while True:
        b = done % w.B
        oracle.draft_verify_cycle(h[b:b + 1], W["w_conv"], W["w_lm"],
                                  W["w_gate"], W["e_in"], W["e_out"],
                                  anchor[b:b + 1], Lc[b:b + 1], w.T, seed, 0,
                                  w.dtype, w_lm_e4m3=w8)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds or done >= w.B:
            break
    seq_per_s = done / el
    return {"value": seq_per_s / w.B, "unit": UNIT,
            "cores": oracle_threads(), "kind": "oracle",
            "sample": (f"{done} of {w.B} sequences of one cycle ({el:.1f} s, "
                       f"float64 numpy; cycles/s = sequences/s / B)")}


def oracle_threads() -> int:
    """Threads the oracle's BLAS runs on in this process (set by
    _set_blas_threads before numpy loaded; else every core)."""
    v = os.environ.get("OPENBLAS_NUM_THREADS")
    return int(v) if v and v.isdigit() else os.cpu_count()


def reference_inputs(w):
    """The workload's inputs, with the target logits of the first
    sequences (those a bounded sample reaches) from the oracle's own
    drafter logits; the rest of the target rows are zero."""
    import oracle
    x = synth.make_inputs(w)
    f64 = lambda t: None if t is None else t.float().numpy().astype(np.float64)
    nseq = max(1, min(w.B, 4))
    h = f64(x["h"][:nseq])
    y = oracle.to_storage(oracle.conv2tap(h, f64(x["w_conv"])), w.dtype)
    _, _, _, U = oracle.lmhead_topk(
        y.reshape(-1, w.H).astype(np.float64), f64(x["w_lm"]),
        want_logits=True)
    d = np.zeros((w.B, w.K + 1, w.V), np.float32)
    d[:nseq] = U.reshape(nseq, w.K + 1, w.V)
    return x, synth.target_logits(w, d)


def run_oracle_sample(args):
    """Child process of the CPU baseline: the oracle on a bounded sample of
    the workload, with its own BLAS thread count; prints one JSON dict."""
    w = synth.get(args.config)
    x, L = reference_inputs(w)
    r = time_oracle(w, x, L, args.cpu_seconds, w.seed, oracle_w8(w, x))
    print(json.dumps(r))
    return 0


def cpu_baseline(args):
    """The oracle timed on the host cores in child processes: all cores
    (the reported value) and one thread."""
    out = {}
    for name, n in (("all", os.cpu_count()), ("one", 1)):
        cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample",
               "--config", args.config, "--cpu-seconds",
               str(args.cpu_seconds / 2), "--oracle-threads", str(n)]
        env = dict(os.environ)
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS",
                    "MKL_NUM_THREADS"):
            env[var] = str(n)
        try:
            r = subprocess.run(cmd, capture_output=True, text=True,
                               env=env, timeout=600)
            out[name] = json.loads(r.stdout.strip().splitlines()[-1])
        except (subprocess.SubprocessError, ValueError, IndexError) as exc:
            out[name] = {"error": str(exc)[:200]}
    res = dict(out["all"])
    res["single_thread"] = out["one"]
    res["threads_how"] = ("BLAS threads fixed by OPENBLAS_NUM_THREADS / "
                          "OMP_NUM_THREADS in a child process")
    return res


# --------------------------------------------------------------------------
# the reference arm: the CPU oracle
# --------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = synth.get(args.config)
    x, L = reference_inputs(w)
    per = max(2.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    w8 = oracle_w8(w, x)
    for _ in range(args.warmup):
        time_oracle(w, x, L, per, w.seed, w8)
    vals = [time_oracle(w, x, L, per, w.seed, w8) for _ in range(args.steps)]
    v = statistics.median(r["value"] for r in vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(w, ws),
            "cpu_baseline": {"value": v, "unit": UNIT,
                             "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"]},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------
# sweep: per-stage rooflines over the K x B x T grid
# --------------------------------------------------------------------------
def run_sweep(args):
    """Each sweep point: cycles/s over CUDA-graph replays and per-stage
    event times, one JSON line per point.  Inputs are drawn on the device
    with seeded torch generators from the same distributions as synth (the
    grid's 4.5 GB of target logits would take minutes to draw on the host);
    the weights are shared by all points."""
    import torch
    import block_drafter_verify_gb300 as dv_mod
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    torch.backends.cuda.matmul.allow_tf32 = False
    pts = synth.sweep_points()
    if args.sweep != "all":
        want = set(args.sweep.split(","))
        pts = [p for p in pts if p.name in want]
    g = torch.Generator(device=dev).manual_seed(pts[0].seed)
    w0 = pts[0]

    def normal(shape, sd, dt=torch.bfloat16):
        return (torch.randn(shape, generator=g, device=dev) * sd).to(dt)
    weights = {"w_conv": normal((2 * w0.H, w0.H), w0.conv_sd),
               "w_lm": normal((w0.V, w0.H), w0.w_lm_sd),
               "w_gate": normal((w0.r, w0.H), w0.sel_sd),
               "e_in": normal((w0.V, w0.r), w0.sel_sd),
               "e_out": normal((w0.V, w0.r), w0.sel_sd)}
    pk = peaks()
    for w in pts:
        h_all = normal((w.B, w.K + 1, w.H), 1.0)
        anchor = torch.randint(0, w.V, (w.B,), generator=g, device=dev,
                               dtype=torch.int32)
        # target = 0.9 * drafter logits + N(0, 1), drafter logits in fp32
        hf = h_all.float()
        wc = weights["w_conv"].float()
        prev = torch.zeros_like(hf)
        prev[:, 1:] = hf[:, :-1]
        y = ((hf @ wc[:w.H].T) * hf + (hf @ wc[w.H:].T) * prev).to(
            torch.bfloat16).float().reshape(-1, w.H)
        L = torch.empty(y.shape[0], w.V, device=dev)
        for v0 in range(0, w.V, 16384):
            L[:, v0:v0 + 16384] = y @ weights["w_lm"][v0:v0 + 16384].float().T
        L.mul_(w.target[1]).add_(torch.randn(L.shape, generator=g,
                                             device=dev) * w.target[2])
        L = L.reshape(w.B, w.K + 1, w.V)
        del hf, prev, y
        h = h_all[:, :w.K].contiguous()
        dv = dv_mod.DraftVerify(w.B, w.K, w.H, w.V, w.r, weights, device=dev)
        for i in range(3):
            dv.cycle(h, anchor, L, w.T, w.seed, i)
        torch.cuda.synchronize(dev)
        dv_mod.dflash_check()
        G, R = 20, 5
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for i in range(G):
                dv.cycle(h, anchor, L, w.T, w.seed, 3 + i)
        gr.replay()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(R):
            gr.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / (G * R)
        stages = dv_mod.STAGES
        ev = [(torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in stages]
        for b_, e_ in ev:
            b_.record()
            e_.record()
        tim = {n: [] for n in stages}
        n_sum = 0
        for i in range(5):
            for si in range(len(stages)):
                dv_mod.dflash_profile_stage(si, ev[si][0], ev[si][1])
            dv.cycle(h, anchor, L, w.T, w.seed, 100 + i)
            torch.cuda.synchronize(dev)
            n_sum += int(dv.n.sum().item())
            for si, n in enumerate(stages):
                tim[n].append(ev[si][0].elapsed_time(ev[si][1]) * 1e3)
        for si in range(len(stages)):
            dv_mod.dflash_profile_stage(si, None, None)
        dv_mod.dflash_check()
        names = {"conv": "conv+gate", "lmhead": "lmhead",
                 "pair_score": "merge+pair_score+walk", "verify": "verify"}
        stage_us = {names[n]: float(np.mean(tim[n])) for n in names}
        by, fl = lmhead_algorithmic(w)
        t_lm = stage_us["lmhead"] * 1e-6
        ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
        lm = ({"bound": "hbm", "frac": by / t_lm / 1e9 / pk["hbm_gbs"],
               "tensor_frac": fl / t_lm / 1e12 / pk["bf16_tflops"]}
              if fl / by < ridge else
              {"bound": "tensor", "frac": fl / t_lm / 1e12 / pk["bf16_tflops"],
               "hbm_frac": by / t_lm / 1e9 / pk["hbm_gbs"]})
        sb = stage_bytes(w, True)
        n_mean = n_sum / (5 * w.B)
        # the verify reads rows 0..n of each sequence (and the draw row),
        # not every target row: its fraction is of those bytes
        all_rows = sb["verify"]
        sb["verify"] = verify_algorithmic(w, n_mean)
        line = {"sweep_point": w.name, "B": w.B, "K": w.K, "T": w.T,
                "V": w.V, "H": w.H, "cycles_per_s": 1e3 / ms,
                "ms_per_cycle": ms, "mean_accepted": n_mean,
                "stage_us": stage_us,
                "stage_timing": "events around each kernel, 5 eager cycles",
                "lmhead": lm,
                "stage_hbm_frac": {k: sb[k] / (stage_us[k] * 1e-6) / 1e9 /
                                   pk["hbm_gbs"] for k in sb
                                   if k in stage_us},
                "verify_all_rows_frac": all_rows / (stage_us["verify"] *
                                                    1e-6) / 1e9 /
                                        pk["hbm_gbs"],
                "data": "synthetic (device-drawn, same distributions)",
                "peak_source": pk["source"]}
        print(json.dumps(line), flush=True)
        del dv, L, h, h_all, gr
        torch.cuda.empty_cache()
    return 0


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import block_drafter_verify_gb300 as dv_mod

    w = synth.get(args.config)
    x = synth.make_inputs(w)
    L_cpu = synth_target_torch(w, x, dev)
    weights = {k: (None if x[k] is None else x[k].to(dev).contiguous())
               for k in ("w_conv", "w_lm", "w_gate", "e_in", "e_out")}
    h = x["h"][:, :w.K].contiguous().to(dev)
    anchor = x["anchor"].to(dev)
    L = L_cpu.to(dev)
    seed = rank_seed(w.seed, rank)
    dv = dv_mod.DraftVerify(w.B, w.K, w.H, w.V, w.r, weights, device=dev,
                            lm_e4m3=w.lm_e4m3)
    stream = torch.cuda.current_stream(dev)

    # Warm-up, then the timed region: the K cycles are captured into CUDA
    # graphs (at most GRAPH_STEPS cycles per graph, each cycle with its own
    # Philox cycle counter) and replayed, so host launch overhead is not
    # timed; the work on the device is exactly the eager path's.
    stages = dv_mod.STAGES
    K = args.steps
    for i in range(args.warmup):
        dv.cycle(h, anchor, L, w.T, seed, i)
    torch.cuda.synchronize(dev)
    dv_mod.dflash_check()

    def capture(first, count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(count):
                dv.cycle(h, anchor, L, w.T, seed, first + i)
        return g

    clk = ClockSampler(dev.index or 0).__enter__()
    G = min(K, GRAPH_STEPS)
    graphs = []
    use_graph, graph_error = True, ""
    try:
        g_full = capture(args.warmup, G)
        graphs = [g_full] * (K // G)
        if K % G:
            graphs.append(capture(args.warmup + (K // G) * G, K % G))
        graphs[0].replay()            # one untimed replay of the captured work
        torch.cuda.synchronize(dev)
    except RuntimeError as exc:       # capture refused: time the eager calls
        use_graph = False
        graph_error = str(exc).splitlines()[0][:200]
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    # an event after every graph replay: per-cycle time percentiles
    marks = [torch.cuda.Event(enable_timing=True) for _ in graphs]
    barrier()
    torch.cuda.synchronize(dev)
    clk.mark_start()
    t_start.record(stream)
    if use_graph:
        for g, mk_ in zip(graphs, marks):
            g.replay()
            mk_.record(stream)
    else:
        for i in range(K):
            dv.cycle(h, anchor, L, w.T, seed, args.warmup + i)
    t_stop.record(stream)
    torch.cuda.synchronize(dev)
    clk.mark_end()
    clk.__exit__(None, None, None)
    barrier()
    dv_mod.dflash_check()
    secs = t_start.elapsed_time(t_stop) / 1e3
    secs_max = max_over_ranks(secs, dev)
    value, _ = aggregate(K, [secs_max], world)
    cycle_ms = None
    if use_graph and len(graphs) >= 2:
        per = []
        prev = t_start
        for g, mk_ in zip(graphs, marks):
            n_c = G if g is g_full else K % G
            per.append(prev.elapsed_time(mk_) / n_c)
            prev = mk_
        q = np.percentile(per, [10, 50, 90])
        cycle_ms = {"p10": float(q[0]), "p50": float(q[1]),
                    "p90": float(q[2]), "graphs": len(per),
                    "cycles_per_graph": G}

    # per-kernel times: CUDA events the library records around each launch,
    # on the launching stream, over eager cycles (not part of the timed K)
    KS = min(K, 20)

    def mk():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e
    ev = [[(mk(), mk()) for _ in stages] for _ in range(KS)]
    n_sum = torch.zeros((), dtype=torch.int64, device=dev)
    torch.cuda.synchronize(dev)
    for i in range(KS):
        for si in range(len(stages)):
            dv_mod.dflash_profile_stage(si, ev[i][si][0], ev[i][si][1])
        dv.cycle(h, anchor, L, w.T, seed, args.warmup + i)
        n_sum += dv.n.sum()
    torch.cuda.synchronize(dev)
    for si in range(len(stages)):
        dv_mod.dflash_profile_stage(si, None, None)
    dv_mod.dflash_check()
    n_mean_cycles = float(n_sum.item()) / (KS * w.B)
    # dflash_draft with bf16 storage and a conv runs three kernels: the conv
    # (with the context gate), the LM head, and one launch that merges the
    # LM head's partials, scores the pairs and walks (recorded as the
    # pair-score stage); otherwise the per-step kernels
    fused = w.dtype == "bf16" and w.conv_sd is not None
    names = ({"conv": "conv+gate", "lmhead": "lmhead",
              "pair_score": "merge+pair_score+walk", "verify": "verify"}
             if fused else {n: n for n in stages if n != "quant"})
    if w.lm_e4m3:
        names["quant"] = "quantize_y"
    stage_us_eager = {}
    for si, name in enumerate(stages):
        if name == "conv" and w.conv_sd is None:
            continue
        if name not in names:
            continue
        stage_us_eager[names[name]] = statistics.mean(
            ev[i][si][0].elapsed_time(ev[i][si][1]) * 1e3 for i in range(KS))
    # The same events recorded inside one CUDA graph of KS cycles: event
    # nodes around every kernel, so a kernel neither overlaps its
    # neighbours (programmatic launch) nor includes a host launch gap.
    # These are the per-kernel times the roofline divides by; the eager
    # times are kept beside them.
    stage_us = stage_us_eager
    stage_timing = "eager cycles"
    if use_graph:
        evg = [[(mk(), mk()) for _ in stages] for _ in range(KS)]
        torch.cuda.synchronize(dev)
        try:
            gs = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gs):
                for i in range(KS):
                    for si in range(len(stages)):
                        dv_mod.dflash_profile_stage(si, evg[i][si][0],
                                                    evg[i][si][1])
                    dv.cycle(h, anchor, L, w.T, seed, 5 * 10**5 + i)
        except RuntimeError:
            gs = None
        for si in range(len(stages)):
            dv_mod.dflash_profile_stage(si, None, None)
        if gs is not None:
            for _ in range(2):
                gs.replay()
            torch.cuda.synchronize(dev)
            dv_mod.dflash_check()
            stage_us = {}
            for si, name in enumerate(stages):
                if names.get(name) in stage_us_eager:
                    stage_us[names[name]] = statistics.mean(
                        evg[i][si][0].elapsed_time(evg[i][si][1]) * 1e3
                        for i in range(KS))
            stage_timing = ("events around each kernel inside a CUDA graph "
                            f"of {KS} cycles")

    # roofline of the dominant kernel (the LM head)
    pk = peaks()
    by, fl = lmhead_algorithmic(w)
    t_lm = stage_us["lmhead"] * 1e-6
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    hbm_bound = (fl / by) < ridge
    traffic = None
    tr_file = os.path.join(ROOT, "profiles", "lmhead_traffic.json")
    if os.path.exists(tr_file):
        with open(tr_file) as f:
            tr = json.load(f)
        for e in (tr if isinstance(tr, list) else [tr]):
            if e.get("workload") == w.name and e.get("kernel_rev") == \
                    lmhead_kernel_rev():
                traffic = e.get("bytes_per_launch")
    tensor_peak, tensor_src = pk["bf16_tflops"], pk["source"]
    if w.lm_e4m3:   # E4M3 MMA: the measured bf16 rate x the nominal 2x
        tensor_peak = 2.0 * pk["bf16_tflops"]
        tensor_src = pk["source"] + " bf16 x 2 (nominal e4m3 / bf16 ratio)"
        ridge = tensor_peak * 1e12 / (pk["hbm_gbs"] * 1e9)
        hbm_bound = (fl / by) < ridge
    if hbm_bound:
        achieved = by / t_lm / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                "traffic": traffic, "peak_source": pk["source"],
                "kernel": "lmhead",
                "tensor_frac": fl / t_lm / 1e12 / tensor_peak,
                "tensor_peak_source": tensor_src}
    else:
        achieved = fl / t_lm / 1e12
        roof = {"bound": "tensor", "achieved": achieved,
                "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": achieved / tensor_peak, "traffic": traffic,
                "peak_source": tensor_src, "kernel": "lmhead",
                "hbm_frac": by / t_lm / 1e9 / pk["hbm_gbs"]}

    # the loop: cycles with the commit step, the anchor handed over from
    # cycle to cycle (same hidden states and target logits every cycle, as
    # the drafter and target forwards are not part of this path)
    loop = None
    if use_graph:
        anchor_l = anchor.clone()
        cap = 16 + 2 * G * (w.K + 1)
        tokens_l = torch.empty(w.B, cap, dtype=torch.int32, device=dev)
        length_l = torch.zeros(w.B, dtype=torch.int32, device=dev)
        stats_l = torch.zeros(dv_mod.COMMIT_STATS, dtype=torch.int64,
                              device=dev)
        gl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gl):
            for i in range(G):
                dv.cycle(h, anchor_l, L, w.T, seed, 7 * 10**5 + i)
                dv.commit(anchor_l, tokens_l, length_l, stats_l)
        gl.replay()                       # untimed
        torch.cuda.synchronize(dev)
        length_l.zero_()
        stats_l.zero_()
        l0 = torch.cuda.Event(enable_timing=True)
        l1 = torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        gl.replay()
        l1.record(stream)
        torch.cuda.synchronize(dev)
        dv_mod.dflash_check()
        st_ = stats_l.cpu().numpy()
        lsecs = l0.elapsed_time(l1) / 1e3
        loop = {"cycles": G, "cycles_per_s": G / lsecs,
                "emitted_tokens_per_s": float(st_[2]) / lsecs,
                "mean_acceptance_length": float(st_[0]) / float(st_[1]),
                "with": "dflash_cycle + dflash_commit, "
                        "anchor handed over every cycle"}

    sel = selector_report(dv_mod, dv, w, h, anchor, L, seed, stream, dev,
                          pk)

    # achieved bandwidth of the other stages (algorithmic bytes per launch
    # / mean event time), against the measured HBM peak
    stage_roof = {}
    for name, nbytes in stage_bytes(w, fused).items():
        if name in stage_us and stage_us[name] > 0:
            gbs = nbytes / (stage_us[name] * 1e-6) / 1e9
            stage_roof[name] = {"bytes": nbytes, "GB/s": gbs,
                                "frac": gbs / pk["hbm_gbs"]}
    if "verify" in stage_roof:
        stage_roof["verify"] = verify_roofline(w, n_mean_cycles,
                                               stage_us["verify"],
                                               pk["hbm_gbs"])

    # end to end through the public API with host buffers
    e2e_steps = args.e2e_steps or max(3, min(K, 20))
    h_host = x["h"][:, :w.K].contiguous().pin_memory()
    a_host = x["anchor"].pin_memory()
    L_host = L_cpu.pin_memory()
    n_host = torch.empty(w.B, dtype=torch.int32).pin_memory()
    o_host = torch.empty(w.B, w.K + 1, dtype=torch.int32).pin_memory()
    # two sets of device inputs: the copies of step i + 1 (on their own
    # stream) run while step i computes; a set is refilled only after the
    # cycle that read it
    bufs = [(torch.empty_like(h), torch.empty_like(anchor),
             torch.empty_like(L)) for _ in range(2)]
    # the target logits (the bulk of the bytes) in NCOPY row ranges, one
    # copy stream each, so that several copy engines share them
    NCOPY = 4
    copy_s = [torch.cuda.Stream(dev) for _ in range(NCOPY)]
    copied = [[torch.cuda.Event() for _ in range(NCOPY)] for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]
    Lh_flat = L_host.view(-1, w.V)
    rows = Lh_flat.shape[0]
    cuts = [rows * c // NCOPY for c in range(NCOPY + 1)]
    barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for cs in copy_s:
        cs.wait_stream(stream)
    for i in range(e2e_steps):
        j = i % 2
        h_d, a_d, L_d = bufs[j]
        Ld_flat = L_d.view(-1, w.V)
        for c, cs in enumerate(copy_s):
            with torch.cuda.stream(cs):
                if i >= 2:
                    cs.wait_event(freed[j])
                if c == 0:
                    h_d.copy_(h_host, non_blocking=True)
                    a_d.copy_(a_host, non_blocking=True)
                Ld_flat[cuts[c]:cuts[c + 1]].copy_(
                    Lh_flat[cuts[c]:cuts[c + 1]], non_blocking=True)
                copied[j][c].record(cs)
        for c in range(NCOPY):
            stream.wait_event(copied[j][c])
        n, out = dv.cycle(h_d, a_d, L_d, w.T, seed, 10**6 + i)
        n_host.copy_(n, non_blocking=True)
        o_host.copy_(out, non_blocking=True)
        freed[j].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, dev)
    e2e_value = world * e2e_steps / e2e_secs
    h2d = h_host.numel() * h_host.element_size() + a_host.numel() * 4 + \
        L_host.numel() * 4
    d2h = n_host.numel() * 4 + o_host.numel() * 4

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args)

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    n_mean = n_mean_cycles
    launches_per_step = (4 if w.dtype == "bf16" and w.conv_sd is not None
                         else (3 if w.conv_sd is not None else 2) + 3)
    if w.lm_e4m3:
        launches_per_step += 1      # the quantization of y
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": 1e3 * secs_max / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype + ("+e4m3 LM head" if w.lm_e4m3 else ""),
        "data": "synthetic",
        "config": bench_config(w, world),
        "timing": ("CUDA graph replay of the K cycles" if use_graph
                   else "eager calls: " + graph_error),
        "verified_tokens_per_s": value * w.B * (n_mean + 1),
        "mean_accepted": n_mean,
        "mean_emitted": n_mean + 1,
        "cycle_ms": cycle_ms,
        "loop": loop,
        "selectors": sel,
        "stage_us": stage_us,
        "stage_us_eager": stage_us_eager,
        "stage_timing": stage_timing,
        "stage_roofline": stage_roof,
        "clocks": clk.summary(),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "h2d_GB/s": h2d * e2e_steps / e2e_secs / 1e9,
                "overlap": "inputs of the next cycle copied on 4 copy "
                           "streams (double-buffered) while the cycle runs"},
        "gpu_launches": launches_per_step * K,
        "roofline": roof,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    return 0


def selector_report(dv_mod, dv, w, h, anchor, L, seed, stream, dev, pk,
                    reps=20):
    """The T = 0 selector variants on the bench lattice, outside the timed
    cycles: mean accepted drafts under greedy verification with the greedy
    walk and with the Viterbi walk (same pair scores), recall@16 of the
    target's argmax by position and the acceptance a perfect selector would
    reach, and the two kernels' event times (recall: algorithmic bytes / time
    against the HBM peak).  The recall launch follows dflash_draft, whose
    W_lm stream has evicted the target logits from L2."""
    import torch
    B, K, C = w.B, w.K, 16
    topi = dv.topi.view(B, K, C)
    arg = torch.empty(B, K, dtype=torch.int32, device=dev)
    hit = torch.empty_like(arg)
    n_g = torch.zeros((), dtype=torch.int64, device=dev)
    n_v = torch.zeros((), dtype=torch.int64, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
          for _ in range(reps)]
    torch.cuda.synchronize(dev)
    for i in range(reps):
        c = 2 * 10**6 + i
        dv.draft_all(h, anchor, 0.0, seed, c)
        ev[i][0].record(stream)
        dv_mod.dflash_top16_recall(L, topi, arg, hit)
        ev[i][1].record(stream)
        dv.verify(L, 0.0, seed, c)
        n_g += dv.n.sum()
        ev[i][2].record(stream)
        dv_mod.dflash_path_viterbi(dv.scores, topi, dv.slot, dv.draft, dv.q)
        ev[i][3].record(stream)
        dv.verify(L, 0.0, seed, c)
        n_v += dv.n.sum()
    torch.cuda.synchronize(dev)
    dv_mod.dflash_check()
    t_rec = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
    t_vit = statistics.mean(e[2].elapsed_time(e[3]) for e in ev) * 1e3
    rec_bytes = B * K * (w.V * 4 + C * 4 + 8)
    vit_bytes = B * K * (C * C * 4 + C * 4 + 8 + C * 4)
    recall, perfect = recall_by_position(hit)
    gbs = rec_bytes / (t_rec * 1e-6) / 1e9
    return {"T": 0.0,
            "mean_accepted_greedy_walk": float(n_g.item()) / (reps * B),
            "mean_accepted_viterbi_walk": float(n_v.item()) / (reps * B),
            "mean_accepted_perfect_selector": float(perfect),
            "recall16_by_position": [round(float(v), 4) for v in recall],
            "viterbi_us": t_vit,
            "viterbi_GB/s": vit_bytes / (t_vit * 1e-6) / 1e9,
            "recall_us": t_rec,
            "recall_roofline": {"bound": "hbm", "bytes": rec_bytes,
                                "achieved": gbs, "peak": pk["hbm_gbs"],
                                "unit": "GB/s", "frac": gbs / pk["hbm_gbs"]}}


def recall_by_position(in_top16):
    """Recall@16 per drafted position, and the acceptance length a perfect
    selector would reach under greedy verification (leading positions whose
    target token is among the candidates), from dflash_top16_recall's
    in_top16 [B,K] (a report of the diagnostic's flags, not a step of
    the path)."""
    import torch
    f = in_top16.to(torch.int64)
    recall = f.double().mean(dim=0)
    miss = (f == 0)
    first = torch.where(miss.any(dim=1), miss.int().argmax(dim=1),
                        torch.full_like(miss[:, 0], f.shape[1],
                                        dtype=torch.int64))
    return recall, first.double().mean()


def stage_bytes(w, fused):
    """Algorithmic bytes per launch of the stages other than the LM head
    (each input read once, each output written once)."""
    M, H, V, r = w.B * w.K, w.H, w.V, w.r
    e = 2 if w.dtype == "bf16" else 4
    out = {}
    if w.conv_sd is not None:
        conv = 2 * H * H * e + M * H * e * 2
        if fused:
            conv += r * H * e + M * r * 4
        out["conv+gate" if fused else "conv"] = conv
    scores = M * 32 * r * e + M * 256 * 4 + M * 16 * 8
    if fused:
        # strip partials: one (16 values, 16 ids, max, sum) list per row and
        # vocab strip, as many strips as the LM head's grid has units
        strips = lmhead_strips(w)
        out["merge+pair_score+walk"] = (M * strips * 136 + M * r * 4 +
                                        scores + M * 16 * 4)
    else:
        out["pair_score"] = scores + M * H * e + r * H * e
    out["verify"] = w.B * (w.K + 1) * V * 4
    if w.lm_e4m3:
        out["quantize_y"] = M * H * e + M * H + M * 4
    return out


def lmhead_strips(w, sms=152):
    """Vocab strips of the tensor-core LM head's grid (CTA pairs when the
    rows span two or more 128-row tiles)."""
    rt = (w.B * w.K + 127) // 128
    vt = (w.V + 255) // 256
    units = sms // 2 if rt >= 2 else sms
    rg = (rt + 1) // 2 if rt >= 2 else rt
    return max(1, min(units // rg, vt, 160))


def lmhead_kernel_rev() -> str:
    """Revision tag of the LM-head kernel source (hash of its files with
    comments and blank space removed), so that a stored ncu traffic figure
    is only used for the code it measured."""
    import hashlib
    import re
    p = os.path.join(ROOT, "block_drafter_verify_gb300", "csrc")
    h = hashlib.sha1()
    for name in sorted(os.listdir(p)):
        if name.startswith("lmhead"):
            with open(os.path.join(p, name)) as f:
                src = f.read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            src = re.sub(r"//[^\n]*", "", src)
            h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:12]


def main(argv=None):
    args = parse(argv)
    if args.oracle_sample:
        return run_oracle_sample(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
