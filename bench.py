#!/usr/bin/env python
"""Benchmark of the Mamba-3 SSM layer core on B300: prefill and decode tokens/s, % of roofline.

Headline (``value``): prefill tokens/s of the SISO 1.5B-layer workload
(B 8, T 4096, H 32, P 64, N 128, bf16 inputs, fp32 accumulation, y written in the
input dtype), inputs resident in HBM; the same prefill with fp32 y is timed beside it.  The same line carries the dominant kernel's roofline,
the fp64 CPU oracle's throughput on a bounded sample, an end-to-end number
through the C ABI with host buffers, the decode legs (B 256 x H 32, 1000
steps from a 512-token prefill state; SISO N 128 and MIMO R 4 N 64), the
16384-token prefill + 256 decode steps, SM clocks during the timed regions,
and the count of library kernel launches.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Several GPUs run independent replicas (torchrun, one rank per GPU): each rank
draws its own inputs; a barrier and a max over ranks bracket the timed region.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Mamba-3 SSM prefill tokens/s & decode tokens/s, % of B300 roofline"
HEADLINE = "siso-prefill-bf16-b8-t4096-h32-p64-n128"
SISO_DEC = "siso-decode-bf16-b256-h32-p64-n128"
MIMO_DEC = "mimo-r4-decode-bf16-b256-h32-p64-n64"
MIMO_PRE = "mimo-r4-prefill-bf16-b8-t4096-h32-p64-n64"
LONG = "long-siso-prefill-bf16-b1-t16384-h32-p64-n128"
L2_BYTES = 126 * 1024 * 1024
CHUNK_ROWS = 128  # (token, rank) rows per chunk of the tensor-core prefill


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# ------------------------------------------------------------------ algorithmic counts


def prefill_bytes(w, out_bytes=4) -> int:
    """Mandatory HBM traffic of one prefill call from a fresh state, returning h_T."""
    tok = w.B * w.T * w.H
    inp = tok * (w.R * w.P * 2 + 2 * w.R * w.N * 2 + 2 * 2 + (w.N // 2) * 2)
    out = tok * w.R * w.P * out_bytes
    state = w.B * w.H * (w.N * w.P * 4 + (w.N // 2) * 4 + w.R * w.N * 2 + w.R * w.P * 2)
    return inp + out + state + w.H * 4


B300_SMS = 148
FP32_LANES_PER_SM = 128
SM_MAX_MHZ = 2032
BWD_CHUNK = 32  # tokens per chunk of the backward at (token, rank) rows <= 64


def backward_fmas(w, c=BWD_CHUNK) -> int:
    """fp32 multiply-adds of the chunked backward, dense M x M chunk products (M = c R rows):
    per chunk 2 M N P (the chunk's own state terms) + 3 M N P (B~ Gout, dY Hp^T, X Gout^T)
    + M^2 (3 N + 2 P) (C~ B~^T, dY X^T, dC~, dB~, dX)."""
    while c * w.R > 64:
        c //= 2
    M = c * w.R
    per_chunk = 5 * M * w.N * w.P + M * M * (3 * w.N + 2 * w.P)
    return w.B * w.H * (w.T // c) * per_chunk


def fp32_peak_tflops(mhz=SM_MAX_MHZ) -> float:
    """CUDA-core fp32 peak: SMs x fp32 lanes x 2 flops per multiply-add x SM clock."""
    return B300_SMS * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def prefill_flops(w, rows=CHUNK_ROWS) -> int:
    """Flops of the chunked masked form at the kernel's chunk (full rows x rows score tiles)."""
    c_tok = rows // w.R
    per_chunk = 2 * rows * rows * w.N + 2 * rows * rows * w.P + 4 * rows * w.N * w.P
    return w.B * w.H * per_chunk * (-(-w.T // c_tok))


def ssd_prefill_bytes(w, out_bytes=4) -> int:
    """Mandatory HBM traffic of the Mamba-2 special case (no lambda, theta, angle or previous
    token): x, B, C, dt in, y out, h_T."""
    tok = w.B * w.T * w.H
    return tok * (w.P * 2 + 2 * w.N * 2 + 2 + w.P * out_bytes) + w.B * w.H * w.N * w.P * 4 + w.H * 4


def ssd_decode_bytes(w, out_bytes=4) -> int:
    """One Mamba-2 decode step: state read + write, x, B, C, dt in, y out."""
    bh = w.B * w.H
    return bh * (2 * w.N * w.P * 4 + w.P * 2 + 2 * w.N * 2 + 2 + w.P * out_bytes) + w.H * 4


def decode_bytes(w, out_bytes=4) -> int:
    """Mandatory HBM traffic of one decode step: state read + write, token inputs, y."""
    bh = w.B * w.H
    state = 2 * bh * (w.N * w.P * 4 + (w.N // 2) * 4 + w.R * w.N * 2 + w.R * w.P * 2)
    inp = bh * (w.R * w.P * 2 + 2 * w.R * w.N * 2 + 2 * 2 + (w.N // 2) * 2)
    return state + inp + bh * w.R * w.P * out_bytes + w.H * 4


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons; keeps samples inside marked windows."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.windows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                pass

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def summary(self):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [s for s in self.samples
                  if any(a - 0.05 <= s[0] <= b + 0.05 for a, b in self.windows)]
        use = inside or self.samples
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in use for n, v in zip(names, s[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[1] for s in use),
                "sm_max_mhz": max(s[2] for s in use), "reasons": reasons, "samples": len(use),
                "in_timed_regions": bool(inside)}


# ------------------------------------------------------------------ helpers


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in ("m3_prefill_tc.cu", "m3_ptx.cuh"):
        with open(os.path.join(ROOT, "state_space_sequence_trapezoidal_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, sha: str):
    """Per-launch DRAM bytes from a committed ncu summary, only if taken on this kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_sha") != sha:
        return None
    return e.get("dram_bytes_per_launch")


def gen_inputs_parallel(w, seeds, A_seed, dtype="bf16"):
    """Per-step decode inputs, drawn in host threads (one seeded generator per step)."""
    from concurrent.futures import ThreadPoolExecutor

    from state_space_sequence_trapezoidal_b300 import synth

    def one(s):
        return synth.make_inputs(w.B, 1, w.H, w.P, w.N, w.R, s, dtype, A_seed=A_seed)

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        return list(ex.map(one, seeds))


def to_dev(inp, dev, torch):
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(
        dev, torch.float32 if k == "A" else torch.bfloat16) for k, v in inp.items()}


# ------------------------------------------------------------------ the oracle arm


def oracle_throughput(w, inp, budget_s: float, start: int = 0, min_slices: int = 0):
    """Time the fp64 CPU oracle on whole (b, h) sequences of workload ``w`` (inputs ``inp``),
    taking distinct sequences from index ``start`` on, in batches over all host cores, until
    ``budget_s`` seconds of oracle time (and at least ``min_slices`` sequences).
    Returns (tokens/s, threads used, sequences done, seconds)."""
    import oracle

    ncores = os.cpu_count() or 1
    batch = max(8, ncores)
    total = w.B * w.H
    done, spent, used = 0, 0.0, 1
    while (spent < budget_s or done < min_slices) and done < total:
        ids = [(start + done + i) % total for i in range(min(batch, total - done))]
        sl = [(i // w.H, i % w.H) for i in ids]
        g = oracle.gather(inp, sl)
        t0 = time.perf_counter()
        _, _, used = oracle.scan(g["x"], g["Bm"], g["Cm"], g["dt"], g["A"], g["lam"], g["theta"],
                                 nthreads=ncores)
        spent += time.perf_counter() - t0
        done += len(sl)
    tokens = done * w.T / w.H  # a token carries all H heads
    return tokens / spent, used, done, spent


def oracle_single_thread(w, inp, budget_s: float):
    """The fp64 oracle on one host thread: whole (b, h) sequences one at a time until
    ``budget_s`` seconds.  Returns (tokens/s, sequences done, seconds)."""
    import oracle

    total = w.B * w.H
    done, spent = 0, 0.0
    while spent < budget_s and done < total:
        sl = [(done // w.H, done % w.H)]
        g = oracle.gather(inp, sl)
        t0 = time.perf_counter()
        oracle.scan(g["x"], g["Bm"], g["Cm"], g["dt"], g["A"], g["lam"], g["theta"], nthreads=1)
        spent += time.perf_counter() - t0
        done += 1
    return done * w.T / w.H / spent, done, spent


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded sample (a batch of whole
    sequences) of the headline workload, timed on the host cores."""
    from state_space_sequence_trapezoidal_b300 import dist as D
    from state_space_sequence_trapezoidal_b300 import synth

    rank, world, _ = D.env_rank()
    if rank != 0:
        return 0
    w = synth.WORKLOADS[HEADLINE]
    inp = synth.make_inputs(w.B, w.T, w.H, w.P, w.N, w.R, w.seed, w.dtype)
    n_per_step = max(8, os.cpu_count() or 1)
    tok, sec, used, pos = 0.0, 0.0, 1, 0
    for i in range(args.warmup + args.steps):
        _, used, done, spent = oracle_throughput(w, inp, budget_s=0.0, start=pos,
                                                 min_slices=n_per_step)
        pos += done
        if i >= args.warmup:
            tok += done * w.T / w.H
            sec += spent
    value = tok / sec
    desc = (f"each step: {n_per_step} whole (b,h) sequences x {w.T} tokens of {w.name} "
            f"(fp64, OpenMP over sequences); tokens counted as sequences x T / H")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "P": w.P, "N": w.N, "R": w.R},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--skip-extras", action="store_true", help="headline prefill only")
    ap.add_argument("--profile-prefill", choices=["headline", "mimo", "long", "backward"],
                    default=None,
                    help="run only --steps plain calls of one prefill workload (the backward: "
                         "of the headline shape cut to --profile-T tokens), for profilers; "
                         "prints their time, no bench line")
    ap.add_argument("--profile-B", type=int, default=0, help="batch rows of --profile-prefill "
                    "(0: the workload's own)")
    ap.add_argument("--profile-T", type=int, default=0, help="tokens of --profile-prefill "
                    "(0: the workload's own)")
    ap.add_argument("--profile-decode", choices=["siso", "mimo"], default=None,
                    help="run only --decode-steps plain decode steps of one decode workload "
                         "(for profilers); prints their time, no bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch

    import state_space_sequence_trapezoidal_b300 as m3
    from state_space_sequence_trapezoidal_b300 import dist as D
    from state_space_sequence_trapezoidal_b300 import synth

    rank, world, local = D.init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    m3.load()
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    clocks = ClockSampler(f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local))
    stream = torch.cuda.current_stream(dev)

    def capture(fn):
        """Record the library launches fn makes (on the current stream) as a CUDA graph."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize(dev)
        return g

    def timed(fn, n):
        """Run fn n times between two events on the launching stream; returns ms per call."""
        D.barrier()
        torch.cuda.synchronize(dev)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        s.record(stream)
        for _ in range(n):
            fn()
        e.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(t0, time.time())
        D.barrier()
        return s.elapsed_time(e) / n

    if args.profile_prefill:
        name = {"headline": HEADLINE, "mimo": MIMO_PRE, "long": LONG,
                "backward": HEADLINE}[args.profile_prefill]
        wp = synth.WORKLOADS[name]
        Bp, Tp = args.profile_B or wp.B, args.profile_T or wp.T
        dp = to_dev(synth.make_inputs(Bp, Tp, wp.H, wp.P, wp.N, wp.R, wp.seed, wp.dtype), dev,
                    torch)
        if args.profile_prefill == "backward":
            dyp = torch.randn(Bp, Tp, wp.H, wp.R, wp.P, dtype=torch.float32, device=dev)

            def one():
                m3.m3_ssm_prefill_backward(dp["x"], dp["B"], dp["C"], dp["dt"], dp["A"],
                                           dp["lambda"], dp["theta"], dyp)
        else:
            yp = torch.empty(Bp, Tp, wp.H, wp.R, wp.P, dtype=torch.bfloat16, device=dev)
            hp = m3.State.zeros(Bp, wp.H, wp.N, wp.P, wp.R, device=dev)
            wsp = m3.prefill_workspace(dp["x"], dp["dt"], dp["theta"], torch.bfloat16)

            def one():
                m3.m3_ssm_prefill(dp["x"], dp["B"], dp["C"], dp["dt"], dp["A"], dp["lambda"],
                                  dp["theta"], y=yp, hT=hp, workspace=wsp,
                                  out_dtype=torch.bfloat16)

        for _ in range(args.warmup):
            one()
        ms = timed(one, args.steps)
        if rank == 0:
            print(json.dumps({"profile_prefill": args.profile_prefill, "workload": name, "B": Bp,
                              "T": Tp, "ms_per_call_host_launched": ms}), flush=True)
        return 0

    if args.profile_decode:
        wd = synth.WORKLOADS[SISO_DEC if args.profile_decode == "siso" else MIMO_DEC]
        inp = to_dev(synth.make_inputs(wd.B, 1, wd.H, wd.P, wd.N, wd.R, wd.seed, wd.dtype), dev,
                     torch)
        q = {k: (v[:, 0].contiguous() if k != "A" else v) for k, v in inp.items()}
        st = m3.State.zeros(wd.B, wd.H, wd.N, wd.P, wd.R, device=dev)
        st.h.normal_(0.0, 0.01)
        yt = torch.empty(wd.B, wd.H, wd.R, wd.P, dtype=torch.float32, device=dev)

        def one():
            m3.m3_ssm_decode_step(st, q["x"], q["B"], q["C"], q["dt"], q["A"], q["lambda"],
                                  q["theta"], y_t=yt)

        for _ in range(args.warmup):
            one()
        ms = timed(one, args.decode_steps)
        if rank == 0:
            # plain launches from Python, for profiling only: not a bench figure
            print(json.dumps({"profile_decode": wd.name, "us_per_step_host_launched": ms * 1e3}),
                  flush=True)
        return 0

    # -------------------------------------------------------------- headline prefill
    # y in the input dtype (bf16), as the method's write-out step states; the fp32-y variant
    # is timed beside it.
    w = synth.WORKLOADS[HEADLINE]
    inp = synth.make_inputs(w.B, w.T, w.H, w.P, w.N, w.R, D.rank_seed(w.seed, rank), w.dtype)
    d = to_dev(inp, dev, torch)
    y = torch.empty(w.B, w.T, w.H, w.R, w.P, dtype=torch.bfloat16, device=dev)
    hT = m3.State.zeros(w.B, w.H, w.N, w.P, w.R, device=dev)
    ws = m3.prefill_workspace(d["x"], d["dt"], d["theta"], torch.bfloat16)

    def prefill_step():
        m3.m3_ssm_prefill(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"], d["theta"], y=y,
                          hT=hT, workspace=ws, out_dtype=torch.bfloat16)

    for _ in range(args.warmup):
        prefill_step()
    ms = timed(prefill_step, args.steps)
    if m3.m3_ssm_device_status(ws) != m3.M3_OK:
        raise RuntimeError("device status reports a timed-out wait in the prefill kernel")
    ms_max = D.max_over_ranks(ms, dev)
    tokens = w.B * w.T
    value = D.aggregate_throughput(tokens, world, ms_max / 1e3)
    pb = prefill_bytes(w, out_bytes=2)
    achieved = pb / (ms / 1e3) / 1e9
    sha = kernel_source_sha()
    kname = "prefill_tc_kernel<128,1,0,1>"
    pf = prefill_flops(w)
    in_bytes = sum(v.numel() * v.element_size() for v in d.values())

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "P": w.P, "N": w.N, "R": w.R,
                   "chunk_tokens": CHUNK_ROWS // w.R, "in_dtype": "bf16", "out_dtype": "bf16",
                   "parallelism": f"replicas x{world}",
                   "l2": (f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB per step vs "
                          f"{L2_BYTES / 1e6:.0f} MB)")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic(kname, sha),
                     "kernel": kname, "algorithmic_bytes_per_launch": pb,
                     "bytes_per_token_head": "x 128 + B, C 512 + theta 128 + dt, lambda 4 + y 128 "
                                             "(bf16) = 900 B, plus the exit state once",
                     "peak_source": peaks["source"],
                     "tensor_view": {"algorithmic_tflops": pf / (ms / 1e3) / 1e12,
                                     "peak": peaks["bf16_tflops"],
                                     "frac": pf / (ms / 1e3) / 1e12 / peaks["bf16_tflops"]}},
        "gpu_launches": args.steps,
    }

    if not args.skip_extras:
        # ---------------------------------------------------------- fp32 y at the same shape
        y32 = torch.empty(w.B, w.T, w.H, w.R, w.P, dtype=torch.float32, device=dev)

        def prefill_f32y():
            m3.m3_ssm_prefill(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"], d["theta"],
                              y=y32, hT=hT, workspace=ws)

        for _ in range(3):
            prefill_f32y()
        ms32 = D.max_over_ranks(timed(prefill_f32y, 20), dev)
        pb32 = prefill_bytes(w, out_bytes=4)
        line["fp32_y"] = {"ms": ms32, "tokens_per_s": D.aggregate_throughput(tokens, world,
                                                                             ms32 / 1e3),
                          "algorithmic_bytes": pb32,
                          "hbm_frac": pb32 / (ms32 / 1e3) / 1e9 / peaks["hbm_gbs"]}
        line["gpu_launches"] += 20
        del y32

        # ---------------------------------------------------------- end to end (host buffers)
        # Pinned host inputs and outputs; the batch is cut into parts that alternate between
        # two streams, so that one part's host-to-device copy, another's kernels and a third's
        # device-to-host copy overlap.  Every byte still crosses the host link each step.
        parts = 4
        pb_rows = w.B // parts
        hin = {k: v.cpu().pin_memory() for k, v in d.items()}
        hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        hh = torch.empty(hT.h.shape, dtype=torch.float32).pin_memory()
        streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        dd = {k: torch.empty_like(v) for k, v in d.items()}
        part_dims = m3.M3Dims(pb_rows, w.T, w.H, w.P, w.N, w.R, 0, m3.M3_BF16, m3.M3_BF16)
        wss = [m3.workspace_for(part_dims, dev) for _ in streams]
        launches_per_part = 1 if wss[0].numel() <= 256 else 3
        hstates = [m3.State(hT.h[i * pb_rows:(i + 1) * pb_rows], hT.phi[i * pb_rows:(i + 1) * pb_rows],
                            hT.prev_B[i * pb_rows:(i + 1) * pb_rows],
                            hT.prev_x[i * pb_rows:(i + 1) * pb_rows]) for i in range(parts)]

        def e2e_step():
            cur = torch.cuda.current_stream(dev)
            dd["A"].copy_(hin["A"], non_blocking=True)
            for i in range(parts):
                s_ = streams[i % 2]
                s_.wait_stream(cur)
                with torch.cuda.stream(s_):
                    rows = slice(i * pb_rows, (i + 1) * pb_rows)
                    for k, v in hin.items():
                        if k != "A":
                            dd[k][rows].copy_(v[rows], non_blocking=True)
                    m3.m3_ssm_prefill(dd["x"][rows], dd["B"][rows], dd["C"][rows], dd["dt"][rows],
                                      dd["A"], dd["lambda"][rows], dd["theta"][rows], y=y[rows],
                                      hT=hstates[i], workspace=wss[i % 2],
                                      out_dtype=torch.bfloat16, stream=s_)
                    hy[rows].copy_(y[rows], non_blocking=True)
                    hh[rows].copy_(hT.h[rows], non_blocking=True)
            for s_ in streams:
                cur.wait_stream(s_)

        for _ in range(3):
            e2e_step()
        ne = max(3, min(20, args.steps))
        ms_e2e = D.max_over_ranks(timed(e2e_step, ne), dev)
        line["e2e"] = {"value": D.aggregate_throughput(tokens, world, ms_e2e / 1e3),
                       "unit": "tokens/s", "h2d_bytes_per_step": in_bytes,
                       "d2h_bytes_per_step": y.numel() * 2 + hT.h.numel() * 4,
                       "ms_per_step": ms_e2e,
                       "how": (f"batch cut into {parts} parts of {pb_rows} rows on 2 streams: "
                               "H2D of a part, its prefill and D2H of its y and h_T overlap "
                               "with the other parts'")}
        line["gpu_launches"] += ne * parts * launches_per_part
        del hin, hy, hh, dd, wss

        # ---------------------------------------------------------- fused BCNorm + bias prologue
        # The headline prefill on raw B, C projection outputs, normalised, weighted and
        # biased inside the kernel, against the plain prefill above (inputs already
        # normalised).  Same HBM bytes (the parameters are 1 KB).
        prm = synth.make_bcnorm_params(w.N, w.H, w.R, D.rank_seed(w.seed, rank) + 7)
        raw = synth.make_raw_bc({k: inp[k] for k in ("B", "C")}, D.rank_seed(w.seed, rank) + 8)
        rb = {k: torch.from_numpy(raw[k]).to(dev, torch.bfloat16) for k in ("B", "C")}
        norm = m3.BCNorm(**{k: torch.from_numpy(prm[k]).to(dev, torch.bfloat16)
                            for k in ("B_weight", "B_bias", "C_weight", "C_bias")}, eps=prm["eps"])

        def prefill_bcnorm():
            m3.m3_ssm_prefill_bcnorm(d["x"], rb["B"], rb["C"], d["dt"], d["A"], d["lambda"],
                                     d["theta"], norm, y=y, hT=hT, workspace=ws,
                                     out_dtype=torch.bfloat16)

        for _ in range(3):
            prefill_bcnorm()
        msn = D.max_over_ranks(timed(prefill_bcnorm, 20), dev)
        line["bcnorm"] = {"workload": w.name, "fused_ms": msn, "plain_ms": ms_max,
                          "fused_over_plain": msn / ms_max,
                          "tokens_per_s": D.aggregate_throughput(tokens, world, msn / 1e3),
                          "hbm_frac": pb / (msn / 1e3) / 1e9 / peaks["hbm_gbs"],
                          "note": "raw B, C in; RMS norm over N, weight, per-head bias applied "
                                  "in the transform warps"}
        line["gpu_launches"] += 20
        del rb, raw

        # ---------------------------------------------------------- MIMO prefill
        wm = synth.WORKLOADS[MIMO_PRE]
        dm = to_dev(synth.make_inputs(wm.B, wm.T, wm.H, wm.P, wm.N, wm.R,
                                      D.rank_seed(wm.seed, rank), wm.dtype), dev, torch)
        ym = torch.empty(wm.B, wm.T, wm.H, wm.R, wm.P, dtype=torch.bfloat16, device=dev)
        hm = m3.State.zeros(wm.B, wm.H, wm.N, wm.P, wm.R, device=dev)

        wsm = m3.prefill_workspace(dm["x"], dm["dt"], dm["theta"], torch.bfloat16)

        def fm():
            m3.m3_ssm_prefill(dm["x"], dm["B"], dm["C"], dm["dt"], dm["A"], dm["lambda"],
                              dm["theta"], y=ym, hT=hm, workspace=wsm, out_dtype=torch.bfloat16)

        for _ in range(3):
            fm()
        msm = D.max_over_ranks(timed(fm, 20), dev)
        bm = prefill_bytes(wm, out_bytes=2)
        line["mimo_prefill"] = {
            "workload": wm.name, "ms": msm, "out_dtype": "bf16", "algorithmic_bytes": bm,
            "tokens_per_s": D.aggregate_throughput(wm.B * wm.T, world, msm / 1e3),
            "achieved_gbs": bm / (msm / 1e3) / 1e9, "hbm_frac": bm / (msm / 1e3) / 1e9 / peaks["hbm_gbs"],
            "algorithmic_tflops": prefill_flops(wm) / (msm / 1e3) / 1e12}
        line["gpu_launches"] += 20
        del dm, ym, hm

        # ---------------------------------------------------------- decode loops
        dec = {}
        for name in (SISO_DEC, MIMO_DEC):
            wd = synth.WORKLOADS[name]
            seed = D.rank_seed(wd.seed, rank)
            pre = to_dev(synth.make_inputs(wd.B, wd.prefill_T_for_decode, wd.H, wd.P, wd.N, wd.R,
                                           seed, wd.dtype), dev, torch)
            st = m3.State.zeros(wd.B, wd.H, wd.N, wd.P, wd.R, device=dev)

            wsd = m3.prefill_workspace(pre["x"], pre["dt"], pre["theta"])

            def reset_state():
                m3.m3_ssm_prefill(pre["x"], pre["B"], pre["C"], pre["dt"], pre["A"], pre["lambda"],
                                  pre["theta"], hT=st, workspace=wsd)

            nsteps = args.decode_steps
            dsteps = []
            for c0 in range(0, nsteps, 64):  # draw on the host in batches, keep on the device
                seeds = [synth.decode_step_seed(seed, s) for s in range(c0, min(nsteps, c0 + 64))]
                for si in gen_inputs_parallel(wd, seeds, A_seed=seed):
                    t = to_dev(si, dev, torch)
                    dsteps.append({k: (v[:, 0].contiguous() if k != "A" else v)
                                   for k, v in t.items()})
            yt = torch.empty(wd.B, wd.H, wd.R, wd.P, dtype=torch.float32, device=dev)

            def step(q):
                m3.m3_ssm_decode_step(st, q["x"], q["B"], q["C"], q["dt"], q["A"], q["lambda"],
                                      q["theta"], y_t=yt)

            def loop():
                for q in dsteps:
                    step(q)

            reset_state()
            for q in dsteps[:3]:  # warm-up steps, then back to the prefill state
                step(q)
            torch.cuda.synchronize(dev)
            graph = capture(loop)  # the whole step loop as one CUDA graph, as a server runs it
            reset_state()
            ms_loop = D.max_over_ranks(timed(graph.replay, 1), dev)
            per = ms_loop / nsteps
            db = decode_bytes(wd)
            dec[name] = {"steps": nsteps, "ms_total": ms_loop, "us_per_step": per * 1e3,
                         "tokens_per_s": D.aggregate_throughput(wd.B, world, per / 1e3),
                         "achieved_gbs": db / (per / 1e3) / 1e9,
                         "hbm_frac": db / (per / 1e3) / 1e9 / peaks["hbm_gbs"],
                         "algorithmic_bytes_per_step": db,
                         "state_bytes": wd.B * wd.H * wd.N * wd.P * 4}
            line["gpu_launches"] += nsteps
            del dsteps, pre, st
        line["decode"] = dec

        # ---------------------------------------------------------- Mamba-2 special case
        # The same shapes through m3_ssd_* (lambda = 1, theta = 0: no trapezoid term, no
        # rotation, state h alone), as in the paper's Mamba-2 versus Mamba-3 decode table.
        sx = {k: d[k][:, :, :, 0].contiguous() for k in ("x", "B", "C")}
        ys = torch.empty(w.B, w.T, w.H, 1, w.P, dtype=torch.bfloat16, device=dev)
        hs = torch.zeros(w.B, w.H, w.N, w.P, dtype=torch.float32, device=dev)

        def fs():
            m3.m3_ssd_prefill(sx["x"], sx["B"], sx["C"], d["dt"], d["A"], None, y=ys, hT=hs,
                              workspace=ws, out_dtype=torch.bfloat16)

        for _ in range(3):
            fs()
        mss = D.max_over_ranks(timed(fs, 20), dev)
        bs = ssd_prefill_bytes(w, out_bytes=2)
        wd = synth.WORKLOADS[SISO_DEC]
        seed = D.rank_seed(wd.seed, rank)
        nsteps = args.decode_steps
        ssteps = []
        for c0 in range(0, nsteps, 64):
            seeds = [synth.decode_step_seed(seed, s) for s in range(c0, min(nsteps, c0 + 64))]
            for si in gen_inputs_parallel(wd, seeds, A_seed=seed):
                t = to_dev(si, dev, torch)
                ssteps.append({k: (v[:, 0, :, 0].contiguous() if k in ("x", "B", "C") else
                                   (v[:, 0].contiguous() if k == "dt" else v))
                               for k, v in t.items() if k in ("x", "B", "C", "dt", "A")})
        hsd = torch.zeros(wd.B, wd.H, wd.N, wd.P, dtype=torch.float32, device=dev)
        ysd = torch.empty(wd.B, wd.H, 1, wd.P, dtype=torch.float32, device=dev)

        def sloop():
            for q in ssteps:
                m3.m3_ssd_decode_step(hsd, q["x"], q["B"], q["C"], q["dt"], q["A"], y_t=ysd)

        for q in ssteps[:3]:
            m3.m3_ssd_decode_step(hsd, q["x"], q["B"], q["C"], q["dt"], q["A"], y_t=ysd)
        torch.cuda.synchronize(dev)
        sgraph = capture(sloop)
        hsd.normal_(0.0, 0.05)
        ms_sl = D.max_over_ranks(timed(sgraph.replay, 1), dev)
        sper = ms_sl / nsteps
        sdb = ssd_decode_bytes(wd)
        m3_dec_us = dec[SISO_DEC]["us_per_step"]
        line["mamba2"] = {
            "prefill": {"workload": w.name, "ms": mss,
                        "tokens_per_s": D.aggregate_throughput(w.B * w.T, world, mss / 1e3),
                        "hbm_frac": bs / (mss / 1e3) / 1e9 / peaks["hbm_gbs"],
                        "algorithmic_bytes": bs},
            "decode": {"workload": wd.name, "steps": nsteps, "us_per_step": sper * 1e3,
                       "tokens_per_s": D.aggregate_throughput(wd.B, world, sper / 1e3),
                       "hbm_frac": sdb / (sper / 1e3) / 1e9 / peaks["hbm_gbs"],
                       "algorithmic_bytes_per_step": sdb},
            "mamba3_over_mamba2": {"prefill_time": ms_max / mss,
                                   "decode_step_time": m3_dec_us / (sper * 1e3)}}
        line["gpu_launches"] += 20 + nsteps
        del sx, ys, hs, ssteps, hsd

        # ---------------------------------------------------------- backward of the prefill
        # Gradients of every input for the headline shape (fp32 CUDA-core chunked adjoint: six
        # launches); dy in fp32.
        dyb = torch.randn(w.B, w.T, w.H, w.R, w.P, dtype=torch.float32, device=dev)
        n_bws = m3.load().m3_ssm_prefill_backward_workspace(ctypes.byref(m3.M3Dims(
            w.B, w.T, w.H, w.P, w.N, w.R, 0, m3.M3_BF16, m3.M3_F32)))
        wsb = torch.empty((n_bws + 15) // 16 * 16, dtype=torch.uint8, device=dev)

        def fb():
            return m3.m3_ssm_prefill_backward(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"],
                                              d["theta"], dyb, workspace=wsb)

        fb()
        msb = D.max_over_ranks(timed(fb, 3), dev)
        tokh = w.B * w.T * w.H
        bb = tokh * (w.R * w.P * 2 + 2 * w.R * w.N * 2 + 2 * 2 + (w.N // 2) * 2   # inputs
                     + w.R * w.P * 4                                             # dy
                     + (w.R * w.P + 2 * w.R * w.N + 2 + w.N // 2) * 4) + w.H * 8 # gradients
        fmab = backward_fmas(w)
        line["backward"] = {"workload": w.name, "ms": msb,
                            "tokens_per_s": D.aggregate_throughput(w.B * w.T, world, msb / 1e3),
                            "bound": "alu",
                            "fp32_fmas": fmab,
                            "achieved_tflops": 2 * fmab / (msb / 1e3) / 1e12,
                            "peak_tflops": fp32_peak_tflops(),
                            "peak_source": "148 SMs x 128 fp32 lanes x 2 x 2032 MHz",
                            "alu_frac": 2 * fmab / (msb / 1e3) / 1e12 / fp32_peak_tflops(),
                            "hbm_frac": bb / (msb / 1e3) / 1e9 / peaks["hbm_gbs"],
                            "algorithmic_bytes": bb, "workspace_bytes": n_bws}
        line["gpu_launches"] += 3 * 6  # three timed calls of six launches
        del dyb, wsb

        # ---------------------------------------------------------- 16384-token prefill + decode
        wl = synth.WORKLOADS[LONG]
        lseed = D.rank_seed(wl.seed, rank)
        dl = to_dev(synth.make_inputs(wl.B, wl.T, wl.H, wl.P, wl.N, wl.R, lseed, wl.dtype), dev,
                    torch)
        yl = torch.empty(wl.B, wl.T, wl.H, wl.R, wl.P, dtype=torch.bfloat16, device=dev)
        sl = m3.State.zeros(wl.B, wl.H, wl.N, wl.P, wl.R, device=dev)

        wsl = m3.prefill_workspace(dl["x"], dl["dt"], dl["theta"], torch.bfloat16)
        long_launches = 1 if wsl.numel() <= 256 else 3  # segmented: first pass, scan, second pass

        def fl():
            m3.m3_ssm_prefill(dl["x"], dl["B"], dl["C"], dl["dt"], dl["A"], dl["lambda"],
                              dl["theta"], y=yl, hT=sl, workspace=wsl, out_dtype=torch.bfloat16)

        for _ in range(3):
            fl()
        msl = D.max_over_ranks(timed(fl, 10), dev)
        ldec = to_dev(synth.make_inputs(wl.B, wl.decode_steps, wl.H, wl.P, wl.N, wl.R, lseed + 100,
                                        wl.dtype, A_seed=lseed), dev, torch)
        lsteps = [{k: (v[:, s].contiguous() if k != "A" else v) for k, v in ldec.items()}
                  for s in range(wl.decode_steps)]
        ylt = torch.empty(wl.B, wl.H, wl.R, wl.P, dtype=torch.float32, device=dev)

        def lloop():
            for q in lsteps:
                m3.m3_ssm_decode_step(sl, q["x"], q["B"], q["C"], q["dt"], q["A"], q["lambda"],
                                      q["theta"], y_t=ylt)

        lgraph = capture(lloop)
        fl()  # back to the prefill's exit state
        msld = D.max_over_ranks(timed(lgraph.replay, 1), dev)
        line["long"] = {"workload": wl.name, "prefill_ms": msl,
                        "prefill_tokens_per_s": D.aggregate_throughput(wl.B * wl.T, world, msl / 1e3),
                        "prefill_hbm_frac": prefill_bytes(wl, 2) / (msl / 1e3) / 1e9 / peaks["hbm_gbs"],
                        "prefill_algorithmic_bytes": prefill_bytes(wl, 2), "out_dtype": "bf16",
                        "decode_steps": wl.decode_steps,
                        "decode_us_per_step": msld / wl.decode_steps * 1e3,
                        "end_to_end_ms": msl + msld}
        line["gpu_launches"] += 10 * long_launches + wl.decode_steps

    line["clocks"] = clocks.summary()

    # -------------------------------------------------------------- CPU oracle baseline
    if rank == 0 and world == 1 and not args.skip_extras:
        v, used, done, spent = oracle_throughput(w, inp, budget_s=10.0)
        v1, done1, spent1 = oracle_single_thread(w, inp, budget_s=3.0)
        line["cpu_baseline"] = {
            "value": v, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": (f"{done} of {w.B * w.H} (b,h) sequences x {w.T} tokens of the same "
                       f"workload, {spent:.1f} s of fp64 oracle time; tokens counted as "
                       f"sequences x T / H"),
            "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{done1} (b,h) sequences x {w.T} tokens, {spent1:.1f} s"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    D.barrier()
    return 0


if __name__ == "__main__":
    sys.exit(main())
