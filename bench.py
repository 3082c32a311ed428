#!/usr/bin/env python
"""Benchmark of the active-shape AG-GEMM / GEMM-RS path on one GB300 per rank.

One step = one pass of the whole hot path over the 16 packed-sequence microbatches
of the SwiGLU MLP workload (tp=4 virtual ranks, hidden=4096, ffn=14336, capacity
8192 tokens, T ~ U{1024..8192 step 4}): per microbatch, set the active shape, then
  fc1  AG-GEMM + SwiGLU  A_0 = swiglu(concat_r X_r @ W1^T)  (X_r [T/4, 4096], W1 [7168, 4096])
  fc2  GEMM-RS           Y_r = rows_r sum_j A_j @ B_j^T      (A_j [T, 3584],   B_j [4096, 3584])
fc1 is virtual rank 0's column shard; its activated output is rank 0's fc2 input and
the other ranks' A_j are inputs (``--mlp unfused`` writes fc1's [T, 7168] output
instead). Every activation is distinct per microbatch (far larger than L2) and the
weights are shared. FLOPs are algorithmic: 2*T*H*N for AG, 2*T*K*H*tp for RS.

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference] [--sweep]

Prints one JSON line (rank 0); its ``sweep`` key holds the active-T sweep of the metric
(fc1 / fc2 of the SwiGLU MLP, the QKV projection and the large configuration's GEMM-RS
at a ladder of T, each point one whole call with L2 flushed before it, against the
roofline). ``--impl reference`` times the CPU oracle instead, on a bounded row sample
of the same workload. ``--sweep`` additionally prints one JSON line per (op, T) point
of a longer ladder.
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import shutil
import signal
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gemm_overlap_gemms_gb300 import synth  # noqa: E402

METRIC = "AG-GEMM / GEMM-RS TFLOP/s and % of GB300 bf16 peak vs active token count T"
WORKLOAD = "swiglu"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the sources of the tile kernels: the kernels and their device-side building blocks
KERNEL_SRC = [os.path.join(ROOT, "gemm_overlap_gemms_gb300", "csrc", f) for f in ("ub_gemm.cu", "ub_device.cuh")]
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one ncu capture per op,
# per active token of the captured launch, and the kernel source they were taken on.
# Traffic is reported as null once the kernel source no longer matches.
NCU_TRAFFIC = {
    "rs": {"sha256_16": "87b9fffd489eae7b", "bytes": 1248.18e6, "T": 8192,
           "source": "profiles/ub_gemm_pair_kernel_rs_swiglu_fc2_T8192.md"},
    "ag_swiglu": {"sha256_16": "87b9fffd489eae7b", "bytes": 484.98e6, "T": 8192,
                  "source": "profiles/ub_gemm_pair_kernel_ag_glu_swiglu_fc1_T8192.md"},
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", action="store_true",
                    help="also print one JSON line per point of the extended active-T ladder")
    ap.add_argument("--no-sweep", action="store_true",
                    help="leave the active-T sweep out of the JSON line")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mlp", choices=["fused", "unfused"], default="fused",
                    help="fused: fc1 runs with the SwiGLU epilogue and feeds virtual rank 0's fc2 "
                         "input (default); unfused: plain fc1 output [T, 7168]")
    ap.add_argument("--no-bulk", action="store_true",
                    help="skip the bulk-overlap measurement")
    ap.add_argument("--no-padded", action="store_true",
                    help="skip the padded-to-capacity comparator")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--case", choices=["ag", "rs", "ag_swiglu", "ag_kn", "rs_kn", "wgrad_g", "wgrad_s",
                                       "bulk_rs", "bulk_ag"],
                    default=None,
                    help="time one op of the workload at one T only (small profiling case)")
    ap.add_argument("--case-T", type=int, default=8192)
    ap.add_argument("--case-workload", choices=["swiglu", "qkv", "large"], default="swiglu",
                    help="the shapes of --case: hidden, tp, AG N and RS K of this workload")
    ap.add_argument("--case-N", type=int, default=0, help="AG output width of --case (0: the workload's)")
    ap.add_argument("--case-K", type=int, default=0, help="RS K per shard of --case (0: the workload's)")
    ap.add_argument("--case-reps", type=int, default=3)
    ap.add_argument("--sm-margin", type=int, default=0)
    ap.add_argument("--gather-kernel", type=int, default=-1, choices=[-1, 0, 1, 2],
                    help="-1: the library's choice by T (default); 0: driver copies; 1: the all-gather "
                         "is one kernel launch; 2: inside the GEMM kernel")
    ap.add_argument("--timeout-ms", type=float, default=None,
                    help="bound of the device-side waits (default: the library's 1 s)")
    ap.add_argument("--cta-pair", type=int, default=-1, choices=[-1, 0, 1],
                    help="-1: chosen per call (default); 1: 256x256 tiles on CTA pairs; 0: single CTAs")
    ap.add_argument("--copy-streams", type=int, default=4)
    ap.add_argument("--gather-ahead", type=int, default=0, choices=[0, 1, 2],
                    help="1: each microbatch's all-gather runs on a second stream beside the previous "
                         "microbatch's GEMM-RS, and its fc1 runs on the gathered buffer "
                         "(ag_gemm_from_buffer); 2: the same on one stream, the all-gather in beside mode "
                         "(UB_OPT_BULK_BESIDE) right after the GEMM-RS; 0: fc1 gathers inside its own "
                         "call (default)")
    ap.add_argument("--pdl", type=int, default=1, choices=[0, 1],
                    help="1: kernels launched with programmatic dependent launch (default); 0: plain")
    ap.add_argument("--skinny", type=int, default=-1, choices=[-1, 0, 1],
                    help="few-token kernel: -1 whenever usable (default), 0 never, 1 whenever usable")
    ap.add_argument("--streamk", type=int, default=-1, choices=[-1, 0, 1, 2, 3, 4, 5, 6, 7, 8],
                    help="-1: chosen per call (default); 1: the last wave of pair tiles cut into as many k-pieces as allowed; 2..8: at most that many; 0: whole tiles")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def _peak_value(d, *keys):
    for k in keys:
        v = d.get(k)
        if isinstance(v, (int, float)):
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "median", "tflops", "gbs"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


def kernel_traffic(op: str, avg_T: float):
    """ncu DRAM traffic of one launch of `op`, scaled from the captured launch to the
    mean active T of the benchmark's launches (traffic grows with T: A and Y are
    proportional, and the weight re-reads follow the number of M-tile waves)."""
    rec = NCU_TRAFFIC.get(op)
    if not rec or not all(os.path.exists(f) for f in KERNEL_SRC):
        return None
    if kernel_src_sha() != rec["sha256_16"]:
        return None
    return {"bytes_per_launch": rec["bytes"] * avg_T / rec["T"], "captured_T": rec["T"],
            "scaled_to_mean_T": avg_T, "source": rec["source"]}


def kernel_src_sha() -> str:
    """sha256 prefix of the tile kernels' sources, concatenated in KERNEL_SRC order."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SRC:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def step_flops(Ts, w):
    H, N, K, tp = w.hidden, w.ag_n[0], w.rs_k[0], w.tp
    ag = sum(2.0 * T * H * N for T in Ts)
    rs = sum(2.0 * T * K * H * tp for T in Ts)
    return ag, rs


# ---------------------------------------------------------------- distributed plumbing

def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = None

    def start(self):
        smi = shutil.which("nvidia-smi")
        if not smi:
            return
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = subprocess.Popen([smi, "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                      "--format=csv,noheader,nounits", "-lms", "50"],
                                     stdout=self.out, stderr=subprocess.DEVNULL)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)  # one more sample, without a run of idle ones after the timed region
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        lines = [l.strip() for l in self.out.read().splitlines() if l.strip()]
        self.out.close()
        os.unlink(self.out.name)
        return parse_clocks(lines)


def parse_clocks(lines):
    """Summary of nvidia-smi samples in ClockSampler.FIELDS order (csv, no header, no
    units): median SM clock, the highest max clock, and the throttle reasons seen
    active in any sample; None without a usable sample."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for l in lines:
        f = [x.strip() for x in l.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
            "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm

class SwigluWorkload:
    """Device-resident inputs of the 16 microbatches plus the shared weights."""

    def __init__(self, device, seed=synth.SEED):
        from gemm_overlap_gemms_gb300 import ub
        self.w = w = synth.WORKLOADS[WORKLOAD]
        self.Ts = synth.token_counts(WORKLOAD, seed)
        g = synth.generator(device, seed)
        H, N, K, tp = w.hidden, w.ag_n[0], w.rs_k[0], w.tp
        self.W1 = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g, device)
        self.B = [synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g, device) for _ in range(tp)]
        self.X, self.A = [], []
        for T in self.Ts:
            self.X.append(synth.normal_bf16((T, H), 1.0, g, device))
            self.A.append([synth.normal_bf16((T, K), 1.0, g, device) for _ in range(tp)])
        cap = w.max_tokens
        self.Y1 = torch.empty((cap, N), dtype=torch.bfloat16, device=device)
        self.Yz = torch.empty((cap, N // 2), dtype=torch.bfloat16, device=device)
        self.Yrs = torch.empty((cap, H), dtype=torch.bfloat16, device=device)
        self.buf = ub.UserBuffer([cap, H], tp)
        self.buf.set_option("cta_pair", CTA_PAIR)
        self.buf.set_option("streamk", STREAMK)
        self.buf.set_option("pdl", PDL)

    def shards(self, i):
        T, tp = self.Ts[i], self.w.tp
        c = T // tp
        return [self.X[i][r * c:(r + 1) * c] for r in range(tp)]

    def out_shards(self, i):
        T, tp = self.Ts[i], self.w.tp
        c = T // tp
        return [self.Yrs[r * c:(r + 1) * c] for r in range(tp)]

    def run_mb(self, i, stream):
        T = self.Ts[i]
        self.buf.set_active_shape([T, self.w.hidden])
        if MLP == "fused":
            # fc1 with the SwiGLU epilogue writes virtual rank 0's fc2 input directly
            self.buf.ag_gemm_swiglu(self.shards(i), self.W1, self.A[i][0], stream=stream)
        else:
            self.buf.ag_gemm(self.shards(i), self.W1, self.Y1, stream=stream)
        self.buf.gemm_rs(self.A[i], self.B, self.out_shards(i), stream=stream)

    def step(self, stream):
        if GATHER_AHEAD:
            self.step_gather_ahead(stream)
            return
        for i in range(len(self.Ts)):
            self.run_mb(i, stream)

    def step_gather_ahead(self, stream):
        """The same microbatches with each all-gather moved off fc1's critical path: it
        runs on a second stream once the previous fc1 has read the buffer, beside the
        previous microbatch's GEMM-RS, and fc1 then reads the gathered buffer. With
        GATHER_AHEAD = 2 everything is on one stream and the all-gather runs beside the
        GEMM-RS in beside mode (launched once the GEMM-RS's CTAs hold their SMs, which is
        after the fc1 before it has completed)."""
        if GATHER_AHEAD == 2:
            H, n = self.w.hidden, len(self.Ts)
            self.buf.set_active_shape([self.Ts[0], H])
            self.buf.allgather(self.shards(0), stream=stream)
            for i in range(n):
                self.buf.set_active_shape([self.Ts[i], H])
                if MLP == "fused":
                    self.buf.ag_gemm_from_buffer(self.W1, self.A[i][0], swiglu=True, stream=stream)
                else:
                    self.buf.ag_gemm_from_buffer(self.W1, self.Y1, stream=stream)
                self.buf.gemm_rs(self.A[i], self.B, self.out_shards(i), stream=stream)
                if i + 1 < n:
                    self.buf.set_active_shape([self.Ts[i + 1], H])
                    self.buf.set_option("bulk_beside", 1)
                    self.buf.allgather(self.shards(i + 1), stream=stream)
                    self.buf.set_option("bulk_beside", 0)
            return
        if not hasattr(self, "side"):
            self.side = torch.cuda.Stream(stream.device)
            self.ev_read = [torch.cuda.Event() for _ in self.Ts]
            self.ev_landed = [torch.cuda.Event() for _ in self.Ts]
        H, n = self.w.hidden, len(self.Ts)
        self.buf.set_active_shape([self.Ts[0], H])
        self.buf.allgather(self.shards(0), stream=stream)
        for i in range(n):
            self.buf.set_active_shape([self.Ts[i], H])
            if i > 0:
                stream.wait_event(self.ev_landed[i])
            if MLP == "fused":
                self.buf.ag_gemm_from_buffer(self.W1, self.A[i][0], swiglu=True, stream=stream)
            else:
                self.buf.ag_gemm_from_buffer(self.W1, self.Y1, stream=stream)
            self.ev_read[i].record(stream)
            if i + 1 < n:
                self.buf.set_active_shape([self.Ts[i + 1], H])
                self.side.wait_event(self.ev_read[i])
                self.buf.allgather(self.shards(i + 1), stream=self.side)
                self.ev_landed[i + 1].record(self.side)
                self.buf.set_active_shape([self.Ts[i], H])
            self.buf.gemm_rs(self.A[i], self.B, self.out_shards(i), stream=stream)


class no_gc:
    """Python's cyclic garbage collector kept off across warm-up and timed regions: a
    collection pauses the thread that issues the step's launches and copies, and the GPU
    then runs out of queued work. Measured on GB300: about one end-to-end region in three
    took ~1.8x the others (19.7-20.9 against 11.5 ms per step) with the collector on; with
    it off, 15 regions of three runs all took 11.48-11.56 ms (slow regions still come now
    and then -- another run: 13.9 and 17.6 among five -- from outside the process, which
    the median leaves out). Entered with the collector
    on, it collects once and disables it (use it before the warm-up steps, so that the GPU
    is busy again when the timer starts); entered with it off, it does nothing."""

    def __enter__(self):
        self.was = gc.isenabled()
        if self.was:
            gc.collect()
            gc.disable()
        return self

    def __exit__(self, *exc):
        if self.was:
            gc.enable()
        return False


def time_steps(fn, steps, warmup, stream, world):
    with no_gc():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    return e0.elapsed_time(e1)  # ms


def time_calls(fn, calls, warmup, stream, graph=True):
    """Time one call, `fn(st)` issuing it on stream `st`. Returns (median ms, mean ms,
    eager ms): with `graph`, the call is captured once into a CUDA graph and replayed
    `calls` times on `stream`, each replay between CUDA events, after `warmup` replays --
    what the call costs the GPU, with no host work (argument marshalling, launch calls)
    between calls to starve it; eager = `calls` calls issued back to back from Python,
    events at both ends only (a host slower than the GPU shows up here). Without
    `graph`, median and mean are None."""
    fn(stream)
    torch.cuda.synchronize()
    eager = time_steps(lambda: fn(stream), calls, 3, stream, 1) / calls
    if not graph:
        return None, None, eager
    cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fn(cap)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(calls + 1)]
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        ev[0].record(stream)
        for i in range(calls):
            g.replay()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(calls)]
    del g
    return float(np.median(ms)), float(np.mean(ms)), eager


SWEEP_CALLS, SWEEP_WARMUP = 50, 10   # per point: median of 50 timed graph replays after 10 warm-ups

# The active-T sweep carried in the default JSON line: (name, workload, op, T ladder).
# fc1 / fc2 of the SwiGLU MLP, the QKV projection, and the large configuration's two
# GEMM-RS (attention-out K = 1024, fc2 K = 3584 per shard).
DEFAULT_SWEEP = (
    ("fc1_ag_swiglu", "swiglu", "ag_swiglu", (4, 64, 128, 512, 1024, 2048, 4096, 8192)),
    ("fc2_rs", "swiglu", "rs", (4, 64, 128, 512, 1024, 2048, 4096, 8192)),
    ("qkv_ag", "qkv", "ag", (4, 512, 1024, 2048, 4096, 8192)),
    ("large_rs_k1024", "large", "rs", (8, 2048, 16384)),
    ("large_rs_k3584", "large", "rs", (8, 2048, 16384)),
)
DEFAULT_SWEEP_CALLS, DEFAULT_SWEEP_WARMUP = 20, 5
L2_FLUSH_BYTES = 256 << 20   # written before every timed call: twice the 129 MB L2


def op_flops_bytes(op, T, H, tp, N=0, K=0):
    """Algorithmic FLOPs and HBM bytes of one call. AG: 2*T*H*N FLOPs; bytes = the weight
    once, the shards read, the gathered buffer written, Y written (SwiGLU: N/2 columns).
    RS: 2*T*K*H*tp FLOPs; bytes = the tp weights once, the tp A_j read, the tp row blocks
    written."""
    if op == "rs":
        return 2.0 * T * K * H * tp, 2.0 * (tp * K * H + tp * T * K + T * H)
    n_out = N // 2 if op == "ag_swiglu" else N
    return 2.0 * T * H * N, 2.0 * (N * H + 2 * T * H + T * n_out)


def roofline_point(flops, nbytes, sec, tensor_peak, hbm_peak):
    """TFLOP/s and GB/s of one call against the roofline min(tensor peak, I * HBM peak),
    I = FLOPs / byte: `bound` names the roof that limits this shape."""
    tf = flops / sec / 1e12
    gbs = nbytes / sec / 1e9
    intensity = flops / nbytes
    attainable = min(tensor_peak, intensity * hbm_peak / 1e3)
    return {"tflops": tf, "frac_of_peak": tf / tensor_peak, "hbm_gbs": gbs, "hbm_frac": gbs / hbm_peak,
            "flop_per_byte": intensity, "bound": "tensor" if attainable >= tensor_peak else "hbm",
            "frac_of_roofline": tf / attainable}


def time_graph_flushed(fn, stream, flush, calls, warmup, clean=False):
    """Median and minimum time of one call, `fn(st)` issuing it on stream `st`: the call is
    captured once into a CUDA graph and replayed `calls` times on `stream`, each replay
    between CUDA events and preceded by a write of `flush` (larger than L2) outside the
    events, after `warmup` replays. The write leaves L2 full of dirty lines, which the
    call then writes back to HBM as it evicts them; with `clean`, `flush` is also read
    back after the write (outside the events), so that the call starts from a cold L2 of
    clean lines, as after a kernel that read rather than wrote."""
    fn(stream)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fn(cap)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        sink = torch.empty((), dtype=flush.dtype, device=flush.device)
        for a, b in ev:
            flush.zero_()
            if clean:
                torch.sum(flush, dim=0, out=sink)
            a.record(stream)
            g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    del g
    return float(np.median(ms)), float(np.min(ms))


READ_FLOOR_MAX_T = 512  # few-token points: the weight read is the work


def read_floor(buf, weights, stream, flush, clean=False):
    """Median time of one plain read of the weight bytes (`ub_stream_read`: one kernel,
    one CTA per SM, bulk copies into shared memory, nothing computed), timed exactly as a
    sweep call is (graph replay, L2 flushed before each): what reading the same bytes in
    one isolated kernel costs on this GPU, launch and ramp included."""
    med, _ = time_graph_flushed(lambda st: buf.stream_read(weights, stream=st), stream, flush,
                                DEFAULT_SWEEP_CALLS, DEFAULT_SWEEP_WARMUP, clean)
    return med


def default_sweep(stream):
    """The active-T sweep of the metric ("TFLOP/s and % of bf16 peak vs active token
    count T"): every point is one whole call (AG: the gather, its flag waits and joins
    included) on a handle registered at the workload's capacity, timed as the median of
    DEFAULT_SWEEP_CALLS graph replays with L2 flushed before each, with the kernel path
    the library took. Fractions are of the measured burst bf16 peak (an isolated call)
    and of the measured HBM bandwidth (algorithmic bytes). Few-token points (T <= 512)
    also carry the time a bare streaming kernel takes to read the same weight bytes
    under the same timing (`read_floor_us`, `ub_stream_read`): the floor an isolated call
    of that size meets before any GEMM work."""
    from gemm_overlap_gemms_gb300 import ub
    pk, src = peaks()
    tensor_peak = _peak_value(pk, "bf16_tflops") or FALLBACK["bf16_tflops"]
    hbm_peak = _peak_value(pk, "hbm_gbs") or FALLBACK["hbm_gbs"]
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    points = []
    t_start = time.perf_counter()
    for wname in ("swiglu", "qkv", "large"):
        w = synth.WORKLOADS[wname]
        H, tp, cap = w.hidden, w.tp, w.max_tokens
        g = synth.generator(dev, 31)
        buf = ub.UserBuffer([cap, H], tp)
        X = synth.normal_bf16((cap, H), 1.0, g, dev)
        Yrs = torch.empty((cap, H), dtype=torch.bfloat16, device=dev)
        for name, wl_name, op, Ts in DEFAULT_SWEEP:
            if wl_name != wname:
                continue
            if op == "rs":
                K = int(name.rsplit("_k", 1)[1]) if "_k" in name else w.rs_k[0]
                A = [synth.normal_bf16((cap, K), 1.0, g, dev) for _ in range(tp)]
                B_all = synth.normal_bf16((tp * H, K), 1.0 / math.sqrt(K), g, dev)  # the tp weights, end to end
                Bt = list(B_all.split(H))
                N = 0
                weights = B_all
            else:
                N, K = w.ag_n[0], 0
                Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g, dev)
                weights = Wt
                Y = torch.empty((cap, N // 2 if op == "ag_swiglu" else N), dtype=torch.bfloat16, device=dev)
            floor = None
            for T in Ts:
                c = T // tp
                buf.set_active_shape([T, H])
                if op == "rs":
                    a_T = [a[:T] for a in A]
                    outs = [Yrs[r * c:(r + 1) * c] for r in range(tp)]
                    fn = lambda st, a_T=a_T, outs=outs: buf.gemm_rs(a_T, Bt, outs, stream=st)
                else:
                    shards = [X[r * c:(r + 1) * c] for r in range(tp)]
                    call = buf.ag_gemm_swiglu if op == "ag_swiglu" else buf.ag_gemm
                    fn = lambda st, shards=shards, call=call: call(shards, Wt, Y, stream=st)
                med, best = time_graph_flushed(fn, stream, flush, DEFAULT_SWEEP_CALLS, DEFAULT_SWEEP_WARMUP)
                cnt = buf.counters()
                flops, nbytes = op_flops_bytes(op, T, H, tp, N, K)
                pt = {"op": name, "T": T, "us": med * 1e3, "us_min": best * 1e3}
                pt.update(roofline_point(flops, nbytes, med / 1e3, tensor_peak, hbm_peak))
                pt["kernel"] = ub.KERNELS.get(cnt["last_kernel"], "?")
                pt["k_pieces"] = cnt["last_pieces"]
                if op != "rs":
                    pt["gather"] = ub.GATHERS.get(cnt["last_gather"], "?")
                if T <= READ_FLOOR_MAX_T:
                    if floor is None:
                        floor = read_floor(buf, weights, stream, flush)
                        floor_clean = read_floor(buf, weights, stream, flush, clean=True)
                    pt["read_floor_us"] = floor * 1e3
                    pt["frac_of_read_floor"] = floor / med
                    # the same call and floor after a flush that leaves L2 clean (written,
                    # then read back): a few-token call writes back the flush's dirty lines
                    # as it streams its weights, which a call after a read-only kernel
                    # would not
                    med_c, _ = time_graph_flushed(fn, stream, flush, DEFAULT_SWEEP_CALLS, DEFAULT_SWEEP_WARMUP,
                                                  clean=True)
                    pt["clean_l2"] = {"us": med_c * 1e3, "hbm_frac": nbytes / (med_c / 1e3) / 1e9 / hbm_peak,
                                      "read_floor_us": floor_clean * 1e3, "frac_of_read_floor": floor_clean / med_c}
                points.append(pt)
            if op == "rs":
                del A, Bt, B_all, weights
            else:
                del Wt, Y, weights
        assert buf.query_status() == ub.UB_OK, "device status %d" % buf.query_status()
        buf.close()
        del X, Yrs
    del flush
    return {"points": points, "timing": "median of %d CUDA-graph replays of one whole call, L2 flushed (%d MiB "
                                        "written) before each, after %d warm-up replays; `clean_l2` (T <= %d): "
                                        "the same with the flush buffer read back after the write, so that L2 "
                                        "holds clean lines" % (DEFAULT_SWEEP_CALLS, L2_FLUSH_BYTES >> 20,
                                                               DEFAULT_SWEEP_WARMUP, READ_FLOOR_MAX_T),
            "peaks": {"bf16_tflops": tensor_peak, "hbm_gbs": hbm_peak,
                      "source": "%s burst bf16 and HBM copy (%s)" % (src, "MEASURED_PEAKS.json" if src == "measured"
                                                                      else "recipe fallback")},
            "seconds": time.perf_counter() - t_start}


def e2e_measure(wl, steps, warmup, stream, world, reps=7):
    """Same step, with each microbatch's activations copied in from pinned host memory
    and its outputs copied back, inside the timed region. Copies run on their own
    streams so that microbatch i+1's inputs and microbatch i-1's outputs move while
    microbatch i computes (outputs alternate between two device buffers). A microbatch's
    input copy waits only until the previous step has computed that microbatch, so the
    host link streams without a break from one timed step to the next, as a training
    loop's prefetch would; no copy of the timed steps starts before the timer's start
    event, and the timer stops after the last output has landed in host memory. The
    timed region runs `reps` times (ms of each returned), each with the garbage
    collector off (no_gc): the host link and the host thread that issues the copies can
    still see other work on the machine, which the median leaves out."""
    fused = MLP == "fused"
    a0 = 1 if fused else 0      # fused: A[i][0] is produced on the device by fc1
    hX = [x.cpu().pin_memory() for x in wl.X]
    hA = [[a.cpu().pin_memory() for a in As[a0:]] for As in wl.A]
    N, H, cap = wl.w.ag_n[0], wl.w.hidden, wl.w.max_tokens
    hY1 = [] if fused else [torch.empty((T, N), dtype=torch.bfloat16).pin_memory() for T in wl.Ts]
    hY2 = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for T in wl.Ts]
    h2d = sum(x.numel() * 2 for x in hX) + sum(a.numel() * 2 for As in hA for a in As)
    d2h = sum(y.numel() * 2 for y in hY1) + sum(y.numel() * 2 for y in hY2)
    dev = wl.W1.device
    Y1 = [wl.Y1, torch.empty((cap, N), dtype=torch.bfloat16, device=dev)]
    Y2 = [wl.Yrs, torch.empty((cap, H), dtype=torch.bfloat16, device=dev)]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    n = len(wl.Ts)
    computed = [torch.cuda.Event() for _ in range(n)]
    landed = [torch.cuda.Event() for _ in range(n)]
    drained = [torch.cuda.Event() for _ in range(2)]
    for e in computed + drained:
        e.record(stream)
    tp = wl.w.tp

    def step():
        for i, T in enumerate(wl.Ts):
            b = i & 1
            c = T // tp
            with torch.cuda.stream(s_in):
                s_in.wait_event(computed[i])          # the previous step is done with X[i], A[i]
                wl.X[i].copy_(hX[i], non_blocking=True)
                for j in range(a0, tp):
                    wl.A[i][j].copy_(hA[i][j - a0], non_blocking=True)
                landed[i].record(s_in)
            stream.wait_event(landed[i])
            stream.wait_event(drained[b])              # output buffer b has been read back
            wl.buf.set_active_shape([T, H])
            if fused:
                wl.buf.ag_gemm_swiglu(wl.shards(i), wl.W1, wl.A[i][0], stream=stream)
            else:
                wl.buf.ag_gemm(wl.shards(i), wl.W1, Y1[b], stream=stream)
            wl.buf.gemm_rs(wl.A[i], wl.B, [Y2[b][r * c:(r + 1) * c] for r in range(tp)], stream=stream)
            computed[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[i])
                if not fused:
                    hY1[i].copy_(Y1[b][:T], non_blocking=True)
                hY2[i].copy_(Y2[b][:T], non_blocking=True)
                drained[b].record(s_out)

    with no_gc():  # before the warm-up: the GPU is busy when timing starts
        for _ in range(warmup):
            s_in.wait_stream(stream)
            step()
            stream.wait_stream(s_out)
        times = []
        for _ in range(reps):
            torch.cuda.synchronize()
            barrier(world)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            s_in.wait_event(e0)            # nothing of the timed steps starts before the timer
            for _ in range(steps):
                step()
            stream.wait_stream(s_out)      # the last outputs are in host memory
            e1.record(stream)
            torch.cuda.synchronize()
            barrier(world)
            times.append(e0.elapsed_time(e1))
    return times, h2d, d2h


def padded_measure(wl, steps, warmup, stream, world):
    """The same microbatches padded to capacity, the fallback the pages describe when
    buffers are sized for the maximum token count: every microbatch runs at
    T = max_tokens, its real tokens first and zeros after them. Returns ms per step."""
    w = wl.w
    cap, H, K, tp = w.max_tokens, w.hidden, w.rs_k[0], w.tp
    dev = wl.W1.device
    Xp, Ap = [], []
    for i, T in enumerate(wl.Ts):
        x = torch.zeros((cap, H), dtype=torch.bfloat16, device=dev)
        x[:T].copy_(wl.X[i])
        Xp.append(x)
        As = []
        for j in range(tp):
            a = torch.zeros((cap, K), dtype=torch.bfloat16, device=dev)
            a[:T].copy_(wl.A[i][j])
            As.append(a)
        Ap.append(As)
    c = cap // tp
    outs = [wl.Yrs[r * c:(r + 1) * c] for r in range(tp)]

    def step():
        wl.buf.set_active_shape([cap, H])
        for i in range(len(wl.Ts)):
            sh = [Xp[i][r * c:(r + 1) * c] for r in range(tp)]
            if MLP == "fused":
                wl.buf.ag_gemm_swiglu(sh, wl.W1, Ap[i][0], stream=stream)
            else:
                wl.buf.ag_gemm(sh, wl.W1, wl.Y1, stream=stream)
            wl.buf.gemm_rs(Ap[i], wl.B, outs, stream=stream)

    ms = time_steps(step, steps, warmup, stream, world)
    del Xp, Ap
    return ms


def interleaved_medians(fns, rounds=5):
    """Each timing function called once per round, in turn, for `rounds` rounds; the
    median of each one's results. Single timings of a pair of kernels vary by several us,
    and a GEMM's time drifts with the clocks over a run, which would bias whichever
    timing came first if each were repeated on its own."""
    results = [[f() for f in fns] for _ in range(rounds)]
    return [float(np.median([r[i] for r in results])) for i in range(len(fns))]


def split_around(steps: int):
    """The steps of the per-kernel event regions before and after the headline region:
    half each (the extra one after)."""
    return steps // 2, steps - steps // 2


def median_region(times_ms, steps: int):
    """The median of several timed regions of `steps` steps each, and a note listing them
    per step (the end-to-end measurement: the host link and the issuing thread see other
    work on the machine, so one region can be slow for reasons outside the step)."""
    med = float(np.median(times_ms))
    note = "median of %d regions of %d steps each: %s ms per step" % (
        len(times_ms), steps, ", ".join("%.2f" % (t / steps) for t in times_ms))
    return med, note


def bulk_measure(wl, stream, T=4096, reps=20):
    """The "bulk" method at one microbatch of the workload: an independent collective
    beside an unrelated GEMM. fc1 backward: its input-gradient GEMM (gemm_rs_kn over
    dZ_j Wt_j) beside the bulk all-gather of its input X (needed by its weight gradient);
    then its weight-gradient GEMM beside a bulk reduce-scatter of tp bf16 partials
    [T, hidden]. `overlapped_ms`: beside mode (UB_OPT_BULK_BESIDE: the collective on the
    GEMM's stream right after it, launched once the GEMM's CTAs hold their SMs);
    `two_streams_overlapped_ms`: the collective on a second stream, the GEMM issued
    first. Times are ms per pair of operations (20 back to back per timing), each the
    median of five timings interleaved with the others'."""
    w = wl.w
    H, F, tp = w.hidden, w.rs_k[0], w.tp
    dev = wl.W1.device
    g = synth.generator(dev, 17)
    c = T // tp
    X = synth.normal_bf16((T, H), 1.0, g, dev)
    dZ = [synth.normal_bf16((T, F), 1.0, g, dev) for _ in range(tp)]
    Wt = [synth.normal_bf16((F, H), 1.0 / math.sqrt(H), g, dev) for _ in range(tp)]
    P = [synth.normal_bf16((T, H), 1.0, g, dev) for _ in range(tp)]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    outs = [out[r * c:(r + 1) * c] for r in range(tp)]
    Ys = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ys = [Ys[r * c:(r + 1) * c] for r in range(tp)]
    dW = torch.empty((F, H), dtype=torch.bfloat16, device=dev)
    shards = [X[r * c:(r + 1) * c] for r in range(tp)]
    side = torch.cuda.Stream(dev)
    buf = wl.buf
    buf.set_active_shape([T, H])
    buf.allgather(shards, stream=stream)      # the buffer holds X for the wgrad runs

    def timed(fn):
        return time_steps(fn, reps, 2, stream, 1) / reps

    def both(gemm, coll):
        def fn():
            side.wait_stream(stream)
            gemm()
            coll()
            stream.wait_stream(side)
        return fn

    def beside(gemm, coll):
        def fn():
            gemm()
            coll()
        return fn

    def timed_beside(fn):
        buf.set_option("bulk_beside", 1)
        try:
            return timed(fn)
        finally:
            buf.set_option("bulk_beside", 0)

    dgrad = lambda: buf.gemm_rs_kn(dZ, Wt, outs, stream=stream)
    ag_side = lambda: buf.allgather(shards, stream=side)
    ag_alone = lambda: buf.allgather(shards, stream=stream)
    wgrad = lambda: buf.wgrad(dZ[0], out=dW, stream=stream)
    rs_side = lambda: buf.reduce_scatter(P, ys, stream=side)
    rs_alone = lambda: buf.reduce_scatter(P, ys, stream=stream)
    res = {"T": T}
    for name, gemm, coll_side, coll_alone, coll_bytes in (
            ("allgather_beside_dgrad", dgrad, ag_side, ag_alone, 2 * T * H * 2),
            ("reduce_scatter_beside_wgrad", wgrad, rs_side, rs_alone, (tp + 1) * T * H * 2)):
        t_g, t_c, t_b, t_2 = interleaved_medians([lambda: timed(gemm), lambda: timed(coll_alone),
                                                  lambda: timed_beside(beside(gemm, coll_alone)),
                                                  lambda: timed(both(gemm, coll_side))])
        hidden = lambda t: (t_g + t_c - t) / t_c if t_c > 0 else None
        res[name] = {"gemm_ms": t_g, "collective_ms": t_c, "sequential_ms": t_g + t_c,
                     "overlapped_ms": t_b, "hidden_fraction": hidden(t_b),
                     "two_streams_overlapped_ms": t_2, "two_streams_hidden_fraction": hidden(t_2),
                     "collective_gbs": coll_bytes / (t_c / 1e3) / 1e9}
    assert buf.query_status() == 0
    return res


def cpu_baseline(wl, seconds):
    """The oracle as it stands, on a row sample of one microbatch of the workload."""
    import oracle
    i = len(wl.Ts) // 2
    T, w = wl.Ts[i], wl.w
    H, N, K, tp = w.hidden, w.ag_n[0], w.rs_k[0], w.tp
    X = synth.to_u16(wl.X[i])
    W1 = synth.to_u16(wl.W1)
    B = [synth.to_u16(b) for b in wl.B]
    A = [synth.to_u16(a) for a in wl.A[i]]
    rng = np.random.default_rng(0)
    G = np.full((T, H), 0xFFFF, dtype=np.uint16)
    c = T // tp
    oracle.allgather([X[r * c:(r + 1) * c] for r in range(tp)], G, T)

    def run(nrows):
        rows = np.sort(rng.choice(T, size=nrows, replace=False))
        t0 = time.perf_counter()
        y1 = oracle.gemm_rows(G, W1, rows)
        if MLP == "fused":
            oracle.swiglu(y1)
        oracle.gemm_rs_rows([a[rows] for a in A], B, rows, T)
        return time.perf_counter() - t0, nrows * (2.0 * H * N + 2.0 * K * H * tp)

    dt, _ = run(4)
    per_row = max(dt / 4, 1e-4)
    n = int(min(T, max(4, seconds / per_row)))
    dt, flops = run(n)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": "%d of %d rows of microbatch %d (T=%d): fc1 AG-GEMM rows plus fc2 GEMM-RS "
                      "rows, fp64 loops, %.1f s" % (n, T, i, T, dt)}


def run_ours(args):
    from gemm_overlap_gemms_gb300 import ub
    rank, world, local = dist_init(args)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.Stream(device)
    wl = SwigluWorkload(device)
    w = wl.w
    ag_flops, rs_flops = step_flops(wl.Ts, w)
    flops = ag_flops + rs_flops

    with torch.cuda.stream(stream):
        pass
    clocks = ClockSampler(local)

    def step():
        wl.step(stream)

    ag_op = "ag_swiglu" if MLP == "fused" else "ag"
    with no_gc():  # before the warm-up, kept off through every region
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        # The headline: K steps with nothing on the stream but the step's own work. The
        # per-kernel durations for the roofline come from K more steps with a CUDA event
        # recorded on the stream before and after every GEMM launch (UB_OPT_PROFILE). An event
        # between two kernels removes their programmatic launch (the second kernel's launch
        # and prologue no longer overlap the end of the first; ~1.5 % of the step on GB300),
        # so the events stay out of the headline region; they run in two halves, just before
        # and just after it, so that their kernels see the GPU's clocks and power state on
        # both sides of the headline (under the power cap, the clocks drift over a run).
        k_before, k_after = split_around(args.steps)
        ag_ms = rs_ms = ms_events = 0.0
        ag_n = rs_n = 0
        clocks.start()

        def events_region(k):
            nonlocal ag_ms, rs_ms, ms_events, ag_n, rs_n
            if k == 0:
                return
            wl.buf.set_option("profile", 1)
            wl.buf.kernel_time(ag_op)
            wl.buf.kernel_time("rs")
            ms_events += max_over_ranks(time_steps(step, k, 0, stream, world), world)
            a, an = wl.buf.kernel_time(ag_op)
            r, rn = wl.buf.kernel_time("rs")
            ag_ms, ag_n, rs_ms, rs_n = ag_ms + a, ag_n + an, rs_ms + r, rs_n + rn
            wl.buf.set_option("profile", 0)

        events_region(k_before)
        ms = time_steps(step, args.steps, 0, stream, world)
        events_region(k_after)
        clk = clocks.stop()
    assert wl.buf.query_status() == ub.UB_OK, "device status %d" % wl.buf.query_status()
    ms = max_over_ranks(ms, world)
    total_flops = flops * args.steps * world
    value = total_flops / (ms / 1e3) / 1e12

    pk, src = peaks()
    tensor_peak = _peak_value(pk, "bf16_tflops_sustained", "bf16_tflops") or FALLBACK["bf16_tflops_sustained"]
    kernels = {
        "ag": {"launches": ag_n, "avg_us": 1e3 * ag_ms / max(ag_n, 1),
               "tflops": (ag_flops * args.steps) / (ag_ms / 1e3) / 1e12 if ag_ms > 0 else None},
        "rs": {"launches": rs_n, "avg_us": 1e3 * rs_ms / max(rs_n, 1),
               "tflops": (rs_flops * args.steps) / (rs_ms / 1e3) / 1e12 if rs_ms > 0 else None},
        "timed_region": "%d + %d steps just before and just after the headline's %d, with a CUDA "
                        "event before and after every GEMM launch on its stream: %.3f ms per step there"
                        % (k_before, k_after, args.steps, ms_events / args.steps),
    }
    dom = "rs" if rs_ms >= ag_ms else "ag"
    achieved = kernels[dom]["tflops"]
    tr = kernel_traffic("ag_swiglu" if (dom == "ag" and MLP == "fused") else dom, float(np.mean(wl.Ts)))
    roofline = {"bound": "tensor",
                "kernel": "ub_gemm_pair_kernel<%s>" % ("MODE_RS" if dom == "rs" else
                                                       ("MODE_AG_GLU" if MLP == "fused" else "MODE_AG")),
                "achieved": achieved, "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": achieved / tensor_peak if achieved else None,
                "traffic": tr["bytes_per_launch"] if tr else None, "traffic_detail": tr,
                "peak_source": "%s bf16 sustained (%s)" % (src, "MEASURED_PEAKS.json" if src == "measured"
                                                             else "no MEASURED_PEAKS.json: recipe fallback")}

    e2e = None
    if not args.no_e2e:
        e_steps = max(2, min(args.steps, 10))
        e_all, h2d, d2h = e2e_measure(wl, e_steps, max(3, args.warmup), stream, world)
        e_all = [max_over_ranks(t, world) for t in e_all]
        e_ms, e_note = median_region(e_all, e_steps)
        e2e = {"value": flops * e_steps * world / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / e_steps, "timed_regions": e_note}

    padded = None
    if not args.no_padded:
        p_steps = max(2, min(args.steps, 5))
        p_ms = max_over_ranks(padded_measure(wl, p_steps, 1, stream, world), world) / p_steps
        padded = {"ms_per_step": p_ms, "useful_tflops": flops * world / (p_ms / 1e3) / 1e12,
                  "active_speedup": p_ms / (ms / args.steps),
                  "what": "same microbatches padded to max_tokens=%d (real tokens first, zeros "
                          "after); useful FLOPs only" % w.max_tokens}
    bulk = bulk_measure(wl, stream) if not args.no_bulk and rank == 0 else None
    active_sweep = default_sweep(stream) if not args.no_sweep and rank == 0 else None
    sweep = sweep_points(wl, stream) + sweep_other_configs(stream) if args.sweep and rank == 0 else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; packed-sequence token counts, N(0,1) activations, "
                "N(0,1/fan_in) weights)",
        "config": {"workload": "SwiGLU MLP: tp=4 virtual shards, hidden=4096, ffn=14336, "
                               "max_tokens=8192, 16 microbatches T~U{1024..8192 step 4}; "
                               "fc1 AG-GEMM N=7168 + fc2 GEMM-RS K=3584",
                   "mlp": ("fc1 with fused SwiGLU epilogue writes virtual rank 0's fc2 input"
                           if MLP == "fused" else "fc1 output [T, 7168] unfused"),
                   "gather": ("each all-gather beside the previous microbatch's GEMM-RS, fc1 on the "
                              "gathered buffer" if GATHER_AHEAD else "inside each fc1 AG-GEMM call"),
                   "tp": w.tp, "hidden": w.hidden, "max_tokens": w.max_tokens,
                   "microbatches": len(wl.Ts), "tokens_per_step": int(sum(wl.Ts)),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: 2.7 GB of distinct activations per step; "
                         "weights shared across microbatches"},
        "gpu_launches": ag_n + rs_n + (len(wl.Ts) * args.steps if GATHER_AHEAD else 0),
        "kernels": kernels,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "padded_comparator": padded,
        "bulk_overlap": bulk,
        "sweep": active_sweep,
        "clocks": clk,
        "flops_per_step": {"ag": ag_flops, "rs": rs_flops},
    }
    if rank == 0:
        if sweep:
            for p in sweep:
                print(json.dumps(p))
        print(json.dumps(line))
    wl.buf.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def sweep_points(wl, stream):
    """TFLOP/s of each op at a ladder of active T on the benchmark's handle."""
    w = wl.w
    H, N, K, tp = w.hidden, w.ag_n[0], w.rs_k[0], w.tp
    out = []
    Xmax = wl.X[int(np.argmax(wl.Ts))]
    Amax = wl.A[int(np.argmax(wl.Ts))]
    Tmax = max(wl.Ts)
    pk, src = peaks()
    tensor_peak = _peak_value(pk, "bf16_tflops") or FALLBACK["bf16_tflops"]
    hbm_peak = _peak_value(pk, "hbm_gbs") or FALLBACK["hbm_gbs"]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=Xmax.device)
    for T in (4, 64, 128, 256, 512, 1024, 2048, 4096, 6144, 8192):
        if T > Tmax:
            X = synth.normal_bf16((T, H), 1.0, synth.generator(Xmax.device, 5), Xmax.device)
            A = [synth.normal_bf16((T, K), 1.0, synth.generator(Xmax.device, 6 + j), Xmax.device)
                 for j in range(tp)]
        else:
            X, A = Xmax[:T], [a[:T].contiguous() for a in Amax]
        c = T // tp
        shards = [X[r * c:(r + 1) * c] for r in range(tp)]
        outs = [wl.Yrs[r * c:(r + 1) * c] for r in range(tp)]
        wl.buf.set_active_shape([T, H])
        for op in ("ag", "ag_swiglu", "ag_swiglu_no_overlap", "rs"):
            if op == "ag":
                fn = lambda st: wl.buf.ag_gemm(shards, wl.W1, wl.Y1, stream=st)
            elif op.startswith("ag_swiglu"):
                fn = lambda st: wl.buf.ag_gemm_swiglu(shards, wl.W1, wl.Yz, stream=st)
            else:
                fn = lambda st: wl.buf.gemm_rs(A, wl.B, outs, stream=st)
            # the no-overlap comparator puts the gather copies on the GEMM's stream, ahead
            # of it (driver copies and stream flag writes: timed eagerly, no graph)
            no_overlap = op == "ag_swiglu_no_overlap"
            wl.buf.set_option("copy_streams", 0 if no_overlap else 4)
            wl.buf.set_option("gather_kernel", 0 if no_overlap else -1)
            _, _, eager = time_calls(fn, SWEEP_CALLS, SWEEP_WARMUP, stream, graph=False)
            ms = eager if no_overlap else time_graph_flushed(fn, stream, flush, SWEEP_CALLS, SWEEP_WARMUP)[0]
            wl.buf.set_option("copy_streams", 4)
            wl.buf.set_option("gather_kernel", -1)
            fl = 2.0 * T * H * N if op != "rs" else 2.0 * T * K * H * tp
            tf = fl / (ms / 1e3) / 1e12
            # algorithmic HBM bytes: weights once, activations in, results out (AG: the
            # shards read and the gathered buffer written as well)
            if op == "rs":
                nbytes = 2.0 * (tp * K * H + tp * T * K + T * H)
            else:
                n_out = N // 2 if op.startswith("ag_swiglu") else N
                nbytes = 2.0 * (N * H + 2 * T * H + T * n_out)
            out.append({"sweep": op, "T": T, "us": ms * 1e3, "us_eager": eager * 1e3,
                        "timing": "eager, back to back" if no_overlap else "graph replay, L2 flushed",
                        "tflops": tf, "frac_of_peak": tf / tensor_peak,
                        "hbm_gbs": nbytes / (ms / 1e3) / 1e9, "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                        "note": ("gather copies on the GEMM's stream, before it (no overlap)"
                                 if op == "ag_swiglu_no_overlap" else
                                 "includes the gather copies, overlapped" if op != "rs" else "")})
    del flush
    return out


def sweep_other_configs(stream):
    """The other throughput configs on their own handles: QKV (AG-GEMM, N = 3072, tp 4,
    hidden 4096) and large (GEMM-RS, tp 8, hidden 8192, attention-out K = 1024 and fc2
    K = 3584 per shard), over a ladder of active T (median of 50 graph replays per point,
    L2 flushed before each; and 50 calls back to back)."""
    from gemm_overlap_gemms_gb300 import ub
    pk, _ = peaks()
    tensor_peak = _peak_value(pk, "bf16_tflops") or FALLBACK["bf16_tflops"]
    hbm_peak = _peak_value(pk, "hbm_gbs") or FALLBACK["hbm_gbs"]
    dev = torch.device("cuda", torch.cuda.current_device())
    g = synth.generator(dev, 7)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = []

    def point(name, T, fn, fl, nbytes):
        _, _, eager = time_calls(fn, SWEEP_CALLS, SWEEP_WARMUP, stream, graph=False)
        ms = time_graph_flushed(fn, stream, flush, SWEEP_CALLS, SWEEP_WARMUP)[0]
        tf = fl / (ms / 1e3) / 1e12
        out.append({"sweep": name, "T": T, "us": ms * 1e3, "us_eager": eager * 1e3,
                    "timing": "graph replay, L2 flushed", "tflops": tf, "frac_of_peak": tf / tensor_peak,
                    "hbm_gbs": nbytes / (ms / 1e3) / 1e9, "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                    "note": "includes the gather" if name.startswith("qkv") else ""})

    w = synth.WORKLOADS["qkv"]
    H, N, tp = w.hidden, w.ag_n[0], w.tp
    Wq = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g, dev)
    X = synth.normal_bf16((w.max_tokens, H), 1.0, g, dev)
    Y = torch.empty((w.max_tokens, N), dtype=torch.bfloat16, device=dev)
    buf = ub.UserBuffer([w.max_tokens, H], tp)
    for T in (4, 64, 512, 1024, 2048, 4096, 8192):
        c = T // tp
        buf.set_active_shape([T, H])
        shards = [X[r * c:(r + 1) * c] for r in range(tp)]
        point("qkv_ag", T, lambda st: buf.ag_gemm(shards, Wq, Y[:T], stream=st), 2.0 * T * H * N,
              2.0 * (N * H + 2 * T * H + T * N))
    buf.close()
    del Wq, X, Y

    w = synth.WORKLOADS["large"]
    H, tp = w.hidden, w.tp
    buf = ub.UserBuffer([w.max_tokens, H], tp)
    Yl = torch.empty((w.max_tokens, H), dtype=torch.bfloat16, device=dev)
    for K in w.rs_k:
        B = [synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g, dev) for _ in range(tp)]
        A = [synth.normal_bf16((w.max_tokens, K), 1.0, g, dev) for _ in range(tp)]
        for T in (8, 512, 2048, 8192, 16384):
            c = T // tp
            buf.set_active_shape([T, H])
            a_T = [a[:T] for a in A]
            outs = [Yl[r * c:(r + 1) * c] for r in range(tp)]
            point("large_rs_k%d" % K, T, lambda st: buf.gemm_rs(a_T, B, outs, stream=st), 2.0 * T * K * H * tp,
                  2.0 * (tp * K * H + tp * T * K + T * H))
        del A, B
    buf.close()
    return out


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = synth.WORKLOADS[WORKLOAD]
    Ts = synth.token_counts(WORKLOAD)
    H, N, K, tp = w.hidden, w.ag_n[0], w.rs_k[0], w.tp
    g = synth.generator("cpu")
    W1 = synth.to_u16(synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g))
    B = [synth.to_u16(synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g)) for _ in range(tp)]
    rng = np.random.default_rng(0)
    nrows = oracle.threads()          # one sampled row per oracle thread

    def one_mb(i):
        T = Ts[i]
        x = synth.to_u16(synth.normal_bf16((nrows, H), 1.0, g))
        a = [synth.to_u16(synth.normal_bf16((nrows, K), 1.0, g)) for _ in range(tp)]
        rows = np.sort(rng.choice(T, size=nrows, replace=False))
        t0 = time.perf_counter()
        y1 = oracle.gemm_rows(x, W1, np.arange(nrows))
        if MLP == "fused":
            oracle.swiglu(y1)
        oracle.gemm_rs_rows(a, B, rows, T)
        return time.perf_counter() - t0, nrows * (2.0 * H * N + 2.0 * K * H * tp)

    t_mb, _ = one_mb(0)
    budget = 150.0 / max(1, args.steps + args.warmup)    # whole run within a few minutes
    per_step = int(max(1, min(len(Ts), budget / max(t_mb, 1e-3))))
    cursor = [0]

    def one_step():
        # a bounded sample of one step: `nrows` rows of fc1 and fc2 in `per_step`
        # microbatches, cycling through all of them across steps
        dt = fl = 0.0
        for _ in range(per_step):
            d, f = one_mb(cursor[0] % len(Ts))
            cursor[0] += 1
            dt += d
            fl += f
        return dt, fl

    for _ in range(args.warmup):
        one_step()
    tot_dt = tot_fl = 0.0
    for _ in range(args.steps):
        dt, fl = one_step()
        tot_dt += dt
        tot_fl += fl
    value = tot_fl / tot_dt / 1e12
    sample = ("per step %d rows (one per thread) of fc1 AG-GEMM and fc2 GEMM-RS in each of %d "
              "of the %d microbatches, cycling; fp64 loops" % (nrows, per_step, len(Ts)))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "SwiGLU MLP: tp=4 virtual shards, hidden=4096, ffn=14336, "
                               "max_tokens=8192, 16 microbatches T~U{1024..8192 step 4}; "
                               "fc1 AG-GEMM N=7168 + fc2 GEMM-RS K=3584"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_case(args):
    """One op of the workload at one active T: a warm-up launch, then `case_reps`
    launches (the small case the profiler captures; holds well under 1 GB)."""
    from gemm_overlap_gemms_gb300 import ub
    w = synth.WORKLOADS[args.case_workload]
    dev = torch.device("cuda", 0)
    T = args.case_T
    H, tp = w.hidden, w.tp
    N = args.case_N or (w.ag_n[0] if w.ag_n else 2 * H)
    K = args.case_K or (w.rs_k[0] if w.rs_k else H)
    g = synth.generator(dev)
    buf = ub.UserBuffer([w.max_tokens, H], tp)
    buf.set_option("cta_pair", args.cta_pair)
    buf.set_option("streamk", args.streamk)
    buf.set_option("copy_streams", args.copy_streams)
    if args.timeout_ms:
        buf.set_option("timeout_ns", int(args.timeout_ms * 1e6))
    buf.set_option("sm_margin", args.sm_margin)
    buf.set_option("gather_kernel", args.gather_kernel)
    buf.set_option("skinny", args.skinny)
    buf.set_option("pdl", args.pdl)
    buf.set_active_shape([T, H])
    c = T // tp
    nbytes = None
    if args.case in ("bulk_rs", "bulk_ag"):
        # the bulk method's collectives alone: bytes moved per call
        if args.case == "bulk_rs":
            P = [synth.normal_bf16((T, H), 1.0, g, dev) for _ in range(tp)]
            Ys = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
            ys = [Ys[r * c:(r + 1) * c] for r in range(tp)]
            fn = lambda: buf.reduce_scatter(P, ys)
            nbytes = (tp + 1) * T * H * 2
        else:
            X = synth.normal_bf16((T, H), 1.0, g, dev)
            shards = [X[r * c:(r + 1) * c] for r in range(tp)]
            fn = lambda: buf.allgather(shards)
            nbytes = 2 * T * H * 2
        flops = 0.0
    elif args.case in ("ag_kn", "rs_kn", "wgrad_g", "wgrad_s"):
        # backward of the workload's MLP: fc2 dgrad (AG of dY times Bt [H, K]), fc1 dgrad
        # (RS over dZ_j Wt_j, Wt_j [N, H] with K = N/2 per rank as in the fused fc1),
        # fc1 wgrad dWt = dZ^T G, fc2 wgrad dBt = dS^T A
        F = K
        if args.case == "ag_kn":
            dY = synth.normal_bf16((T, H), 1.0, g, dev)
            Bt = synth.normal_bf16((H, F), 1.0 / math.sqrt(F), g, dev)
            out = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
            shards = [dY[r * c:(r + 1) * c] for r in range(tp)]
            fn = lambda: buf.ag_gemm_kn(shards, Bt, out)
            flops = 2.0 * T * H * F
        elif args.case == "rs_kn":
            dZ = [synth.normal_bf16((T, F), 1.0, g, dev) for _ in range(tp)]
            Wt = [synth.normal_bf16((F, H), 1.0 / math.sqrt(H), g, dev) for _ in range(tp)]
            Ys = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
            outs = [Ys[r * c:(r + 1) * c] for r in range(tp)]
            fn = lambda: buf.gemm_rs_kn(dZ, Wt, outs)
            flops = 2.0 * T * F * H * tp
        else:
            X = synth.normal_bf16((T, H), 1.0, g, dev)
            W1 = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g, dev)
            buf.ag_gemm([X[r * c:(r + 1) * c] for r in range(tp)], W1)   # gathers G
            Dm = synth.normal_bf16((T, N if args.case == "wgrad_g" else F), 1.0, g, dev)
            fn = (lambda: buf.wgrad(Dm)) if args.case == "wgrad_g" else (lambda: buf.wgrad(Dm, ub_is_a=True))
            flops = 2.0 * T * H * Dm.shape[1]
    elif args.case in ("ag", "ag_swiglu"):
        X = synth.normal_bf16((T, H), 1.0, g, dev)
        W1 = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g, dev)
        shards = [X[r * c:(r + 1) * c] for r in range(tp)]
        if args.case == "ag":
            Y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: buf.ag_gemm(shards, W1, Y)
        else:
            Z = torch.empty((T, N // 2), dtype=torch.bfloat16, device=dev)
            fn = lambda: buf.ag_gemm_swiglu(shards, W1, Z)
        flops = 2.0 * T * H * N
    else:
        A = [synth.normal_bf16((T, K), 1.0, g, dev) for _ in range(tp)]
        B = [synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g, dev) for _ in range(tp)]
        Ys = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        outs = [Ys[r * c:(r + 1) * c] for r in range(tp)]
        fn = lambda: buf.gemm_rs(A, B, outs)
        flops = 2.0 * T * K * H * tp
    buf.set_option("profile", 1)
    fn()
    torch.cuda.synchronize()
    op_name = {"wgrad_g": "wgrad", "wgrad_s": "wgrad", "bulk_rs": "reduce_scatter"}.get(args.case, args.case)
    if args.case == "bulk_ag":
        # no kernel of ours to time: CUDA events around the whole call on the stream
        torch.cuda.synchronize()
        t_ms = time_steps(fn, args.case_reps, 2, torch.cuda.current_stream(), 1) / args.case_reps
        print(json.dumps({"case": args.case, "T": T, "gather_kernel": args.gather_kernel, "us": 1e3 * t_ms,
                          "gbs": nbytes / (t_ms / 1e3) / 1e9}))
        buf.close()
        return
    first_ms, _ = buf.kernel_time(op_name)
    first_status = buf.query_status()
    for _ in range(args.case_reps):
        fn()
    torch.cuda.synchronize()
    ms, n = buf.kernel_time(op_name)
    buf.set_option("profile", 0)
    # whole calls (gather copies, flag writes, joins included), CUDA events on the stream
    call_ms = time_steps(fn, args.case_reps, 1, torch.cuda.current_stream(), 1) / args.case_reps
    # host time to enqueue one call (no synchronisation inside the loop)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.case_reps):
        fn()
    host_us = 1e6 * (time.perf_counter() - t0) / args.case_reps
    torch.cuda.synchronize()
    # the same call captured once into a CUDA graph and replayed: no host work per call
    cs = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            fn()
    graph_ms = time_steps(graph.replay, args.case_reps, 2, torch.cuda.current_stream(), 1) / args.case_reps
    del graph
    status = buf.query_status()
    buf.close()
    print(json.dumps({"case": args.case, "workload": args.case_workload, "T": T, "N": N, "K": K,
                      "cta_pair": args.cta_pair, "streamk": args.streamk,
                      "copy_streams": args.copy_streams, "sm_margin": args.sm_margin,
                      "gather_kernel": args.gather_kernel, "launches": n, "avg_us": 1e3 * ms / max(n, 1),
                      "tflops": flops * n / (ms / 1e3) / 1e12 if ms > 0 and flops else None,
                      "gbs": nbytes * n / (ms / 1e3) / 1e9 if ms > 0 and nbytes else None,
                      "call_us": 1e3 * call_ms, "host_us": host_us, "graph_us": 1e3 * graph_ms,
                      "first_us": 1e3 * first_ms, "first_status": first_status, "status": status}))
    if status != ub.UB_OK:
        sys.exit("device status %d (%s)" % (status, ub.ERRORS.get(status, "?")))


CTA_PAIR = -1
STREAMK = -1
PDL = 1
MLP = "fused"
GATHER_AHEAD = 0


def main():
    global CTA_PAIR, STREAMK, PDL, MLP, GATHER_AHEAD
    args = parse()
    GATHER_AHEAD = args.gather_ahead
    CTA_PAIR = args.cta_pair
    STREAMK = args.streamk
    PDL = args.pdl
    MLP = args.mlp
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
