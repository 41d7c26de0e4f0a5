#!/usr/bin/env python
"""Benchmark of Fibottention's sparse self-attention hot path on GB300.

One step = one pass of the whole path over one batch of the workload:
support build (host), forward (O, LSE) and backward (dQ, dK, dV), through
the C ABI of libfibatt.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores

The headline workload is the largest single-GPU configuration (long:
B=2, H=16, N=16385, fwd+bwd, bf16).  The same line carries, per workload
(tiny, vitb, vitb_nodiag, video, train, long), the forward and backward
kernel times, pairs/s, GB/s and the fraction of the binding roofline.

Timing: W untimed steps, then exactly K steps between two CUDA events,
bracketed by a barrier and torch.cuda.synchronize(); max over ranks.  Inputs
rotate over enough copies that each step's tensors are evicted from L2 (129
MB) by the steps in between.  Per-kernel durations come from back-to-back
loops of one call kind on the same rotating sets (CUDA events at the ends).
nvidia-smi samples the clocks from the start of the timed region to the end
of the per-kernel loops.  With --gpus N > 1 and no torchrun environment,
bench.py starts the N ranks itself (one process per GPU).
"""
from __future__ import annotations

import argparse
import ctypes
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_head_self_gb300 import _native, api  # noqa: E402
from sparse_head_self_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = ("attended query-key pairs/sec and achieved HBM GB/s (% of GB300 peak), "
          "fwd and fwd+bwd")
UNIT = "pairs/s"
FALLBACK_HBM_GBS = 6800.0
HEADLINE = "long"   # the largest configuration that fits one GPU
RECORD_WORKLOADS = ("tiny", "vitb", "vitb_nodiag", "video", "train", "long")


# ------------------------------------------------------------------ helpers

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    p.add_argument("--profile-run", action="store_true",
                   help="warm-up and timed steps of the workload only (no per-workload records, end-to-end "
                        "run or CPU baseline): the command profiled by ncu")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--block", action="store_true",
                   help="time the attention layer (QKV projection, Fibottention, output projection) fwd+bwd "
                        "instead of the attention core, next to the same layer with masked dense attention")
    p.add_argument("--global-token", action="store_true",
                   help="token 0 global in every head (README Algorithm 2's class token)")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    return p.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (a timing reduction, not a data path)."""
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: int, steps: int, world: int, max_elapsed_ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (each rank runs its own batch; weak scaling)."""
    return world * units_per_rank * steps / (max_elapsed_ms / 1e3)


def algorithmic_bytes(wl, backward: bool) -> int:
    """Minimum HBM bytes of one call: every input row read once, every output
    row written once (Q,K,V -> O,LSE forward; Q,K,V,O,dO,LSE -> dQ,dK,dV backward)."""
    e = wl.B * wl.H * wl.N * wl.D
    s = 4 if wl.dtype == "f32" else 2
    rows = wl.B * wl.H * wl.N
    return (8 * e * s + 4 * rows) if backward else (4 * e * s + 4 * rows)


# Secondary roofline: FP32 arithmetic.  Per attended pair the forward does
# 2 x 64 multiply-adds (the score and the row update), the backward 5 x 64
# (two scores, three row updates); the peak is the GB300's FP32 FMA rate,
# 152 SMs x 128 lanes x 2 flops at the 2070 MHz maximum SM clock.
FLOPS_PER_PAIR = {"fwd": 2 * 2 * 64, "bwd": 5 * 2 * 64}
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "sparse_head_self_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM traffic of one call from the committed ncu record, or None when
    the kernel sources changed since it was taken.

    Reads are ``dram__bytes_read.sum``.  A kernel's writes mostly end in L2
    as dirty lines that reach DRAM after the kernel has ended (ncu then
    counts them nowhere), so the write side is the larger of
    ``dram__bytes_write.sum`` and the bytes the SMs wrote into L2
    (``lts__t_sectors_op_write.sum`` x 32 B): every byte written into L2
    goes to DRAM once.  Returns {"read", "write", "total", ...}."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d[workload][kernel]
        if ent.get("source_hash") != kernel_source_hash():
            return None
        rd = int(ent["dram_read"])
        wr = max(int(ent["dram_write"]), int(ent["l2_write"]))
        out = {"read": rd, "write": wr, "total": rd + wr, "dram_write": int(ent["dram_write"]),
               "l2_write": int(ent["l2_write"]), "capture": ent.get("capture")}
        if "l2_to_sm_read" in ent:   # reads that missed L1 (l1tex__m_xbar2l1tex_read_bytes.sum)
            out["l2_to_sm_read"] = int(ent["l2_to_sm_read"])
        if "scaled_from" in ent:
            out["scaled_from"] = ent["scaled_from"]
        return out
    except Exception:
        return None


def roofline_record(wl, kind: str, ms: float, pairs: int, hbm_peak: float, peak_kind: str):
    """Roofline of one call kind ("fwd" or "bwd") of a workload: achieved HBM
    GB/s (algorithmic bytes over the measured time) and FP32 TFLOP/s (flops
    per attended pair over the same time), each against its peak, and which
    of the two roofs binds (the larger ideal time)."""
    nbytes = algorithmic_bytes(wl, kind == "bwd")
    flops = pairs * FLOPS_PER_PAIR[kind]
    t_hbm = nbytes / (hbm_peak * 1e9)
    t_alu = flops / (FP32_PEAK_TFLOPS * 1e12)
    gbs = nbytes / ms / 1e6
    tfl = flops / (ms / 1e3) / 1e12
    return {"ms": round(ms, 5), "pairs_per_s": pairs / (ms / 1e3), "GB_s": round(gbs, 1),
            "frac_hbm": round(gbs / hbm_peak, 4), "TFLOP_s": round(tfl, 2),
            "frac_alu": round(tfl / FP32_PEAK_TFLOPS, 4), "algorithmic_bytes": nbytes, "flops": flops,
            "bound": "alu" if t_alu > t_hbm else "hbm", "hbm_peak_kind": peak_kind}


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        if not self.rows:
            return None
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# --------------------------------------------------------------- gb300 arm

class Step:
    """Raw C-ABI calls for one step on one rotating buffer set."""

    def __init__(self, wl, dev, rotate: int, seed: int = 0, global_token: bool = False):
        self.global_token = global_token
        self.lib = _native.lib()
        self.wl = wl
        H = wl.H
        ab = [api.wythoff_row(i) for i in range(1, H + 1)]
        w = api.window_schedule(H, wl.w_min, wl.w_max)
        self.a = (ctypes.c_int64 * H)(*[x[0] for x in ab])
        self.b = (ctypes.c_int64 * H)(*[x[1] for x in ab])
        self.w = (ctypes.c_int64 * H)(*w)
        self.dt = _native.F32 if wl.dtype == "f32" else _native.BF16
        q, k, v, do = make_inputs(wl, seed)
        self.host = (q, k, v, do)
        self.sets = []
        sup = api.Support.wythoff(H, wl.N, wl.w_min, wl.w_max, wl.diag).set_global_token(global_token)
        self.pairs = sup.total_pairs(wl.B)
        ws_bytes = sup.bwd_workspace_bytes(wl.B)
        for r in range(rotate):
            t = {n: x.to(dev) for n, x in zip(("Q", "K", "V", "dO"), (q, k, v, do))}
            t["O"] = torch.empty_like(t["Q"])
            t["LSE"] = torch.empty((wl.B, H, wl.N), dtype=torch.float32, device=dev)
            for n in ("dQ", "dK", "dV"):
                t[n] = torch.empty_like(t["Q"])
            t["ws"] = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
            t["ws_bytes"] = ws_bytes
            self.sets.append(t)
        self.ptr = [{n: (x.data_ptr() if isinstance(x, torch.Tensor) else x) for n, x in t.items()}
                    for t in self.sets]

    def bytes_per_set(self) -> int:
        t = self.sets[0]
        return sum(x.numel() * x.element_size() for x in t.values() if isinstance(x, torch.Tensor))

    def run(self, r: int, stream: int, ev=None):
        L, wl, p = self.lib, self.wl, self.ptr[r]
        h = ctypes.c_void_p()
        _native.check(L.fibatt_support_build(wl.H, wl.N, self.a, self.b, self.w, int(wl.diag),
                                             ctypes.byref(h)))
        _native.check(L.fibatt_support_set_global_token(h, int(self.global_token)))
        if ev is not None:
            ev[0].record()
        _native.check(L.fibatt_fwd(h, wl.B, wl.D, self.dt, p["Q"], p["K"], p["V"], wl.scale, p["O"],
                                   p["LSE"], stream))
        if ev is not None:
            ev[1].record()
        _native.check(L.fibatt_bwd(h, wl.B, wl.D, self.dt, p["Q"], p["K"], p["V"], p["O"], p["LSE"],
                                   p["dO"], wl.scale, p["dQ"], p["dK"], p["dV"], p["ws"],
                                   p["ws_bytes"], stream))
        if ev is not None:
            ev[2].record()
        L.fibatt_support_destroy(h)

    def kernel_ms(self, rotate: int, stream: int, n: int = 0, seconds: float = 0.25):
        """Average device time of one forward and of one backward call, each
        measured over back-to-back calls on the rotating sets (CUDA events on
        the launching stream around the whole run): n calls, or (n = 0) as
        many as take about `seconds` (at least 20), from a short calibration."""
        L, wl = self.lib, self.wl
        h = ctypes.c_void_p()
        _native.check(L.fibatt_support_build(wl.H, wl.N, self.a, self.b, self.w, int(wl.diag),
                                             ctypes.byref(h)))
        _native.check(L.fibatt_support_set_global_token(h, int(self.global_token)))
        out, calls = [], []
        for kind in ("fwd", "bwd"):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for i in range(5):
                self._call(kind, h, i % rotate, stream)
            e.record()
            e.synchronize()
            cnt = n if n > 0 else int(min(20000, max(20, seconds / max(s.elapsed_time(e) / 5e3, 1e-7))))
            s.record()
            for i in range(cnt):
                self._call(kind, h, i % rotate, stream)
            e.record()
            e.synchronize()
            out.append(s.elapsed_time(e) / cnt)
            calls.append(cnt)
        L.fibatt_support_destroy(h)
        self.calls = calls
        return out[0], out[1]

    def _call(self, kind, h, r, stream):
        L, wl, p = self.lib, self.wl, self.ptr[r]
        if kind == "fwd":
            _native.check(L.fibatt_fwd(h, wl.B, wl.D, self.dt, p["Q"], p["K"], p["V"], wl.scale, p["O"],
                                       p["LSE"], stream))
        else:
            _native.check(L.fibatt_bwd(h, wl.B, wl.D, self.dt, p["Q"], p["K"], p["V"], p["O"], p["LSE"],
                                       p["dO"], wl.scale, p["dQ"], p["dK"], p["dV"], p["ws"],
                                       p["ws_bytes"], stream))


def run_e2e(step: Step, dev, steps: int):
    """Same step through the public Python API, with the inputs copied from
    pinned host memory and every output read back to pinned host memory.

    Steps are pipelined two deep: step i's host-to-device copies (copy
    stream), fwd + bwd (compute stream) and device-to-host copies (second
    copy stream) overlap with those of steps i - 1 and i + 1, on two device
    buffer sets; events keep every buffer from being overwritten before its
    last reader is done."""
    wl = step.wl
    q, k, v, do = (x.pin_memory() for x in step.host)
    out_sets = []
    for _ in range(2):
        outs = {n: torch.empty((wl.B, wl.H, wl.N, wl.D), dtype=wl.torch_dtype).pin_memory()
                for n in ("O", "dQ", "dK", "dV")}
        outs["LSE"] = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32).pin_memory()
        out_sets.append(outs)
    sets = step.sets[:2]
    h2d = sum(x.numel() * x.element_size() for x in (q, k, v, do))
    d2h = sum(x.numel() * x.element_size() for x in out_sets[0].values())
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def one(i):
        c = i % 2
        t, outs = sets[c], out_sets[c]
        sup = api.Support.wythoff(wl.H, wl.N, wl.w_min, wl.w_max, wl.diag).set_global_token(step.global_token)
        with torch.cuda.stream(s_in):
            if used[c]:
                s_in.wait_event(ev_cmp[c])      # step i-2 done reading these inputs
            for n, x in zip(("Q", "K", "V", "dO"), (q, k, v, do)):
                t[n].copy_(x, non_blocking=True)
            ev_in[c].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[c])
            if used[c]:
                s_cmp.wait_event(ev_out[c])     # step i-2's outputs read back
            api.fwd(sup, t["Q"], t["K"], t["V"], wl.scale, O=t["O"], LSE=t["LSE"], stream=s_cmp)
            api.bwd(sup, t["Q"], t["K"], t["V"], t["O"], t["LSE"], t["dO"], wl.scale, dQ=t["dQ"],
                    dK=t["dK"], dV=t["dV"], workspace=t["ws"], stream=s_cmp)
            ev_cmp[c].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[c])
            for n in ("O", "LSE", "dQ", "dK", "dV"):
                outs[n].copy_(t[n], non_blocking=True)
            ev_out[c].record(s_out)
        used[c] = True
        sup.close()

    for i in range(4):
        one(i)
    torch.cuda.synchronize(dev)
    main = torch.cuda.current_stream(dev)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(main)
    s_in.wait_stream(main)
    for i in range(steps):
        one(i)
    main.wait_stream(s_out)
    main.wait_stream(s_cmp)
    e.record(main)
    torch.cuda.synchronize(dev)
    ms = s.elapsed_time(e) / steps
    return ms, h2d, d2h


def _oracle_heads(wl, global_token: bool):
    import oracle
    w = oracle.windows(wl.H, wl.w_min, wl.w_max)
    return [oracle.Head.fibottention(*oracle.wythoff_row(i + 1), w[i], wl.diag, global_token)
            for i in range(wl.H)]


def _row_pairs(N, table, global_token, rows):
    """Attended pairs of the listed query rows: the banded ones read off the
    signed table, plus what the global first token adds (every key for row 0,
    key 0 for a row whose band misses it)."""
    offs = [int(d) for d in table]
    n = 0
    for j in rows:
        band = sum(1 for d in offs if 0 <= j + d < N)
        if global_token:
            band = N if j == 0 else band + (0 if -j in offs else 1)
        n += band
    return n


def cpu_baseline(wl, target_s: float, global_token: bool = False):
    """The fp64 oracle as it stands, on the host cores, on a bounded sample of
    the workload: forward and backward of blocks of query/key rows, one head
    after another (heads 1, 2, ..., each sampled at evenly spread rows), for
    about target_s seconds.  The unit is attended pairs of the sampled query
    rows per second (each sampled row's forward, its dQ and the dK, dV of the
    key row with the same index)."""
    import oracle
    cores = oracle.set_threads(oracle.max_threads())
    q, k, v, do = make_inputs(wl.with_batch(1), 0)
    heads = _oracle_heads(wl, global_token)
    tables = [oracle.signed_table(wl.N, hd) for hd in heads]
    block = max(1, min(wl.N, 4 * cores))
    done_pairs, done_rows, t0, i = 0, 0, time.perf_counter(), 0
    while True:
        h = i % wl.H
        start = (i // wl.H) * 7919 % wl.N   # spread the blocks over the sequence
        rows = sorted({(start + t * max(1, wl.N // block)) % wl.N for t in range(block)})
        oracle.fwd_head(q[0, h], k[0, h], v[0, h], heads[h], wl.scale, rows=rows)
        oracle.bwd_head(q[0, h], k[0, h], v[0, h], do[0, h], heads[h], wl.scale, qrows=rows, krows=rows)
        done_pairs += _row_pairs(wl.N, tables[h], global_token, rows)
        done_rows += len(rows)
        i += 1
        el = time.perf_counter() - t0
        if el >= target_s or done_rows >= wl.B * wl.H * wl.N:
            break
    return {"value": done_pairs / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"fp64 oracle fwd+bwd of {done_rows} query/key rows ({i} blocks of up to {block} rows spread "
                       f"over heads 1..{min(i, wl.H)} of batch element 0) of the {wl.name} workload, "
                       f"{done_pairs} attended pairs, {el:.1f} s")}


def _rotation(step_probe_bytes: int, l2: int) -> int:
    """Input/output sets to rotate so that every set is evicted from L2 by
    the others before it is used again (at most 64 sets)."""
    return int(min(64, max(2, math.ceil(3 * l2 / step_probe_bytes) + 1)))


def _make_step(wl, dev, l2, global_token):
    probe = Step(wl, dev, 1, global_token=global_token)
    per_set = probe.bytes_per_set()
    del probe
    rotate = _rotation(per_set, l2)
    return Step(wl, dev, rotate, global_token=global_token), rotate, per_set


def workload_record(step, rotate, sptr, hbm_peak, peak_kind, seconds=0.25):
    """Forward and backward kernel times of one workload (back-to-back loops)
    and their rooflines."""
    wl = step.wl
    fwd_ms, bwd_ms = step.kernel_ms(rotate, sptr, seconds=seconds)
    fwd = roofline_record(wl, "fwd", fwd_ms, step.pairs, hbm_peak, peak_kind)
    bwd = roofline_record(wl, "bwd", bwd_ms, step.pairs, hbm_peak, peak_kind)
    fb, bb = fwd["algorithmic_bytes"], bwd["algorithmic_bytes"]
    rec = {"B": wl.B, "H": wl.H, "N": wl.N, "dtype": wl.dtype, "diag": wl.diag,
           "w": [wl.w_min, wl.w_max], "pairs": step.pairs, "fwd": fwd, "bwd": bwd,
           "fwd_bwd": {"ms": round(fwd_ms + bwd_ms, 5),
                       "pairs_per_s": step.pairs / ((fwd_ms + bwd_ms) / 1e3),
                       "GB_s": round((fb + bb) / (fwd_ms + bwd_ms) / 1e6, 1),
                       "frac_hbm": round((fb + bb) / (fwd_ms + bwd_ms) / 1e6 / hbm_peak, 4)},
           "calls_timed": {"fwd": step.calls[0], "bwd": step.calls[1]},
           "l2": f"{rotate} rotating sets"}
    if wl.name == "tiny":
        rec["note"] = "launch-bound (0.2 MB per call): parity case, no roofline claim"
    return rec, fwd_ms, bwd_ms


def gb300_arm(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the gb300 arm")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    wl = WORKLOADS[args.workload]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    step, rotate, per_set = _make_step(wl, dev, l2, args.global_token)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    for i in range(args.warmup):
        step.run(i % rotate, sptr)
    torch.cuda.synchronize(dev)

    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    barrier(world)
    torch.cuda.synchronize(dev)
    if not args.profile_run:
        clocks.start()
    launches0 = step.lib.fibatt_launch_count()
    # the timed region: K whole steps back to back (no event between the
    # kernels, so each launch may overlap the previous kernel's drain)
    start.record()
    for i in range(K):
        step.run(i % rotate, sptr)
    end.record()
    torch.cuda.synchronize(dev)
    launches = step.lib.fibatt_launch_count() - launches0
    barrier(world)
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    if args.profile_run:
        if rank == 0:
            print(json.dumps({"profile_run": wl.name, "steps": K, "ms_per_step": elapsed_ms / K}), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    t_loops = time.perf_counter()
    # per-kernel durations of the headline workload, then of every other
    # workload (each allocated in turn), the clock sampler still running
    head_rec, fwd_ms, bwd_ms = workload_record(step, rotate, sptr, peak, peak_kind)
    records = {}
    for name in RECORD_WORKLOADS:
        if name == wl.name:
            records[name] = head_rec
            continue
        sub, srot, _ = _make_step(WORKLOADS[name], dev, l2, args.global_token)
        records[name], _, _ = workload_record(sub, srot, sptr, peak, peak_kind)
        del sub
        torch.cuda.empty_cache()
    loops_s = time.perf_counter() - t_loops
    dev_err = ctypes.c_uint(0)
    _native.check(step.lib.fibatt_device_error(1, ctypes.byref(dev_err)))
    if dev_err.value:
        raise SystemExit(f"device error word set during the timed region: {dev_err.value:#x}")
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = (f"from the start of the timed region to the end of the per-kernel loops of every "
                         f"workload ({loops_s:.1f} s)")

    ms_step = elapsed_ms / K
    value = whole_job_value(step.pairs, K, world, elapsed_ms)
    dominant = "bwd" if bwd_ms >= fwd_ms else "fwd"
    d = head_rec[dominant]
    kname = f"fibatt_{dominant}"
    traffic = recorded_traffic(kname, wl.name)
    if traffic is not None and "l2_to_sm_read" in traffic:
        traffic["l2_to_sm_GB_s"] = round(traffic["l2_to_sm_read"] / d["ms"] / 1e6, 1)   # at the bench's time
    hbm_line = {"bound": "hbm", "kernel": kname, "achieved": d["GB_s"], "peak": peak, "peak_kind": peak_kind,
                "unit": "GB/s", "frac": d["frac_hbm"], "traffic": None if traffic is None else traffic["total"],
                "traffic_detail": traffic, "algorithmic_bytes": d["algorithmic_bytes"], "avg_ms": d["ms"]}
    alu_line = {"bound": "alu", "kernel": kname, "achieved": d["TFLOP_s"], "peak": round(FP32_PEAK_TFLOPS, 1),
                "peak_kind": "derived: 152 SMs x 128 FP32 lanes x 2 flops x 2.07 GHz", "unit": "TFLOP/s",
                "frac": d["frac_alu"], "traffic": None if traffic is None else traffic["total"],
                "flops_per_pair": FLOPS_PER_PAIR[dominant], "flops": d["flops"], "avg_ms": d["ms"]}
    roofline, secondary = (alu_line, hbm_line) if d["bound"] == "alu" else (hbm_line, alu_line)

    e2e_ms, h2d, d2h = run_e2e(step, dev, args.e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": (f"{wl.name}: B={wl.B} H={wl.H} N={wl.N} d={wl.D} {wl.dtype}, "
                                f"Wythoff rows 1..{wl.H}, w {wl.w_min}..{wl.w_max}, "
                                f"diag={'on' if wl.diag else 'off'}"
                                + (", global token 0" if args.global_token else "")),
                   "B_per_gpu": wl.B, "H": wl.H, "N": wl.N,
                   "step": "support build + fwd + bwd (all hot-path rows)",
                   "pairs_per_step_per_gpu": step.pairs,
                   "l2": (f"{rotate} rotating input/output sets of {per_set / 1e6:.0f} MB "
                          f"(> {l2 / 1e6:.0f} MB L2 between reuses)"),
                   "parallelism": f"replicas over B, {world} GPU(s), no collective"},
        "fwd": head_rec["fwd"],
        "bwd": head_rec["bwd"],
        "fwd_bwd": head_rec["fwd_bwd"],
        "roofline": roofline,
        "roofline_secondary": secondary,
        "workloads": records,
        "e2e": {"value": world * step.pairs / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": args.e2e_steps},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds, args.global_token)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------- reference arm

def reference_arm(args):
    """The fp64 oracle, as it stands, timed on host cores: each step is a
    bounded sample (a block of query/key rows of one (b, h) head, forward and
    backward), sized so that the whole run ends within a few minutes."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    wl = WORKLOADS[args.workload]
    cores = oracle.set_threads(oracle.max_threads())
    q, k, v, do = make_inputs(wl.with_batch(1), 0)
    heads = _oracle_heads(wl, args.global_token)
    tables = [oracle.signed_table(wl.N, hd) for hd in heads]

    def row_pairs(h, rows):
        return _row_pairs(wl.N, tables[h], args.global_token, rows)

    def one(i, nrows):
        h = i % wl.H
        r0 = (i * nrows) % wl.N
        rows = [(r0 + t) % wl.N for t in range(nrows)]
        oracle.fwd_head(q[0, h], k[0, h], v[0, h], heads[h], wl.scale, rows=rows)
        oracle.bwd_head(q[0, h], k[0, h], v[0, h], do[0, h], heads[h], wl.scale, qrows=rows, krows=rows)
        return row_pairs(h, rows)

    # size a step so that warmup + steps take about 120 s
    t0 = time.perf_counter()
    one(0, 4)
    per_row = max((time.perf_counter() - t0) / 4, 1e-6)
    budget = 120.0 / max(1, args.steps + args.warmup)
    nrows = int(max(1, min(wl.N, budget / per_row)))
    for i in range(args.warmup):
        one(i, nrows)
    pairs, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        pairs += one(i, nrows)
    el = time.perf_counter() - t0
    value = pairs / el
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": wl.name, "B_per_gpu": wl.B, "H": wl.H, "N": wl.N,
                      "step": f"fwd+bwd of {nrows} query/key rows of one (b,h) head"},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": f"{nrows} rows of one head per step, fp64 C oracle"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def block_arm(args):
    """The attention layer of a ViT block (sparse_head_self_gb300.block) as a
    training step: forward and backward through autograd, synthetic input of
    the workload's shape, dim = H * 64; next to it the same layer with its
    attention core written as torch scaled-dot-product attention under the
    support's boolean mask (dense work, same result)."""
    from sparse_head_self_gb300.block import FibottentionSelfAttention
    import oracle
    wl = WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    torch.manual_seed(0)
    layer = FibottentionSelfAttention(wl.H * 64, wl.H, wl.N, wl.w_min, wl.w_max, wl.diag,
                                      global_token=args.global_token).to(dev, wl.torch_dtype)
    x = torch.randn(wl.B, wl.N, wl.H * 64, device=dev, dtype=wl.torch_dtype, requires_grad=True)
    g = torch.randn_like(x)
    heads = _oracle_heads(wl, args.global_token)
    mask = torch.stack([torch.from_numpy(oracle.support_mask(wl.N, h).astype(bool)) for h in heads]).to(dev)

    def dense_layer(xx):
        B, N, dim = xx.shape
        qkv = layer.qkv(xx).view(B, N, 3, wl.H, 64).permute(2, 0, 3, 1, 4)
        o = torch.nn.functional.scaled_dot_product_attention(qkv[0], qkv[1], qkv[2], attn_mask=mask[None],
                                                             scale=layer.scale)
        return layer.proj(o.transpose(1, 2).reshape(B, N, dim))

    def time_steps(fn, n):
        for _ in range(max(3, args.warmup)):
            fn(x).backward(g)
        torch.cuda.synchronize(dev)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(n):
            fn(x).backward(g)
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / n

    K = min(args.steps, 500)
    ms = time_steps(layer, K)
    ms_dense = time_steps(dense_layer, K)
    # the same layer with its forward and backward captured as CUDA graphs
    # (no host launch overhead; the kernels neither allocate nor synchronise)
    graphed = torch.cuda.make_graphed_callables(layer, (x,))
    ms_graph = time_steps(graphed, K)
    tokens = wl.B * wl.N
    out = {"metric": "attention layer training step (QKV projection, attention, output projection; fwd+bwd)",
           "value": tokens / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": max(3, args.warmup),
           "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": wl.dtype, "data": "synthetic",
           "config": {"workload": f"{wl.name}: B={wl.B} N={wl.N} dim={wl.H * 64} heads={wl.H}"
                                  + (", global token 0" if args.global_token else ""),
                      "layer": "Linear(dim, 3 dim) -> Fibottention -> Linear(dim, dim)"},
           "cuda_graph": {"ms_per_step": ms_graph, "tokens_per_s": tokens / (ms_graph / 1e3)},
           "dense_masked_sdpa": {"ms_per_step": ms_dense, "tokens_per_s": tokens / (ms_dense / 1e3)}}
    print(json.dumps(out), flush=True)


def _rank_entry(rank: int, world: int, port: int, target, args):
    """One rank started by launch_ranks: the torchrun environment, then the arm."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), LOCAL_WORLD_SIZE=str(world))
    target(args)


def launch_ranks(world: int, target, args) -> None:
    """Start `world` ranks of `target(args)` as processes on this node (one per
    GPU, rank r on cuda:r), rendezvous on 127.0.0.1, and wait for all of them;
    what torchrun would do for `bench.py --gpus N`."""
    import multiprocessing as mp
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_entry, args=(r, world, port, target, args)) for r in range(world)]
    for pr in procs:
        pr.start()
    codes = []
    for pr in procs:
        pr.join()
        codes.append(pr.exitcode)
    if any(c != 0 for c in codes):
        raise SystemExit(f"bench ranks exited with codes {codes}")


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        arm = reference_arm
    elif args.block:
        arm = block_arm
    else:
        arm = gb300_arm
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is not None and int(env_world) != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={env_world}: launch one rank per GPU "
                         f"(torchrun --nproc-per-node {args.gpus}, or no torchrun at all)")
    if env_world is None and args.gpus > 1:
        if arm is block_arm:
            raise SystemExit("--block runs on one GPU")
        launch_ranks(args.gpus, arm, args)
        return
    arm(args)


if __name__ == "__main__":
    main()
