"""Benchmark of the ReplaySSM decode hot path on one GB300 (or N, one process per GPU).

A step is one standard decode step of one Mamba-2 layer at B = 256
(nheads 128, headdim 64, dstate 128, ngroups 8, FP32 checkpoint, L = 16)
through the C ABI, with inputs already resident in HBM; the 1 GiB state is
larger than L2, so no L2 flush is needed between steps.  Timing starts at a
window boundary and covers exactly --steps launches, so the timed region
holds floor-or-ceil(K / 16) flush steps; `natural_window` restates the rate
at the natural 15 : 1 mix from the per-launch means.  Per-launch CUDA events
on the launching stream give the roofline of the decode kernel.  Extra
objects time the Gated DeltaNet layer (B = 256), speculative verify + commit
(B = 512, T = 4), the FP8 / NVFP4 read copies (with their per-window error
against the exact output), the conventional read-modify-write and
snapshot-per-draft kernels on the same GPU (and the ratios), a batch sweep
and a window-length sweep.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --impl reference the CPU oracle (the conventional per-token recurrence
in float64) is timed on the host cores on a bounded sample of the same
workload.  Multi-GPU runs (torchrun) shard sequences: every rank runs its own
B = 256 batch with no communication on the data path.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SSM decode seq·steps/s per layer at B=256 (Mamba-2/GDN); HBM GB/s vs 8 TB/s"
UNIT = "seq·steps/s"
FALLBACK_HBM_GBS = 6800.0
E2E_STEPS = 320  # host-buffer leg: 20 whole windows, whatever --steps is


# ----------------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in ("decode128.cu", "common.cuh", "internal.h"):
        h.update(open(os.path.join(ROOT, "checkpoint_input_replay_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_record(name: str):
    """The ncu DRAM figures in profiles/<name>.json (written beside the summary of the
    same name) when they were taken on the current decode kernel source, else None."""
    p = os.path.join(ROOT, "profiles", name + ".json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))
    if rec.get("kernel_sha") != kernel_sha():
        return None
    return rec


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self, skip_first: int = 2):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        rows = rows[skip_first:] or rows
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for name, v in zip(names, r[2:]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------- workloads

def m2_bytes(shape, h: int, flush: bool) -> int:
    """Algorithmic HBM bytes of one Mamba-2 decode step per sequence with h records buffered."""
    H, G, P, N = shape.n_heads, shape.n_groups, shape.d_head, shape.d_state
    state = H * P * N * 4
    record = H * P * 2 + H * 2 + H * 4 + G * N * 2          # x, dt, log a, B
    inputs = H * P * 2 + H * 2 + 2 * G * N * 2               # x, dt, B, C
    out = H * P * 4
    b = state + h * record + inputs + out
    return b + (state if flush else record)


def gdn_bytes(shape, h: int, flush: bool) -> int:
    H, G, P, N = shape.n_heads, shape.n_groups, shape.d_head, shape.d_state
    state = H * P * N * 4
    record = H * P * 4 + H * 4 + G * N * 2                   # u, g, k
    inputs = 2 * G * N * 2 + H * P * 2 + 2 * H * 4           # q, k, v, g, beta
    out = H * P * 4
    b = state + h * record + inputs + out
    return b + (state if flush else record)


def kda_bytes(shape, h: int, flush: bool) -> int:
    """Per-channel-gate layer: records carry a log decay per key channel."""
    H, G, P, N = shape.n_heads, shape.n_groups, shape.d_head, shape.d_state
    state = H * P * N * 4
    record = H * P * 4 + H * N * 4 + G * N * 2               # u, g, k
    inputs = 2 * G * N * 2 + H * P * 2 + H * N * 4 + H * 4     # q, k, v, g, beta
    out = H * P * 4
    b = state + h * record + inputs + out
    return b + (state if flush else record)


def upload(inp: dict, dev) -> dict:
    import torch
    out = {}
    for k, v in inp.items():
        if v.dtype == np.uint16:
            out[k] = torch.from_numpy(v.view(np.int16).copy()).to(dev).view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(dev)
    return out


class Shard:
    """Sequences [b0, b1) of a workload whose batch is the whole job's: rank r of N
    takes the r-th slice (the generator is a pure function of the sequence index,
    so a slice equals the same rows of the whole job's inputs)."""

    def __init__(self, wl, b0: int, b1: int):
        self.wl, self.b0, self.b1 = wl, b0, b1
        self.shape = wl.shape.with_batch(b1 - b0)
        self.s0_std = wl.s0_std

    def _range(self, lo, hi):
        hi = self.shape.batch if hi is None else hi
        return self.b0 + lo, self.b0 + hi

    def step(self, t, lo=0, hi=None):
        return self.wl.step(t, *self._range(lo, hi))

    def S0(self, lo=0, hi=None):
        return self.wl.S0(*self._range(lo, hi))

    def draft(self, s, T, lo=0, hi=None):
        return self.wl.draft(s, T, *self._range(lo, hi))

    def accepted(self, s, T, lo=0, hi=None):
        return self.wl.accepted(s, T, *self._range(lo, hi))

    def __getattr__(self, name):  # A(), c() and the like: per layer, not per sequence
        if name in ("wl", "b0", "b1"):
            raise AttributeError(name)
        return getattr(self.wl, name)


def shard_of(wl, rank: int, world: int) -> Shard:
    """This rank's equal slice of the whole job's batch."""
    per = wl.shape.batch // world
    if per * world != wl.shape.batch:
        raise ValueError("the job's batch must be a multiple of the number of ranks")
    return Shard(wl, rank * per, (rank + 1) * per)


class nvtx_range:
    """An NVTX range around a bench leg (for nsys / ncu range filters); a no-op when
    the torch build has no NVTX."""

    def __init__(self, name: str):
        self.name = name

    def __enter__(self):
        try:
            import torch
            torch.cuda.nvtx.range_push(self.name)
            self.on = True
        except Exception:
            self.on = False
        return self

    def __exit__(self, *exc):
        if self.on:
            import torch
            torch.cuda.nvtx.range_pop()
        return False


def job_value(world: int, batch_per_rank: int, steps: int, elapsed_ms_max: float) -> float:
    """Whole-job sequence-steps per second: every rank's units over the slowest rank's time."""
    return world * batch_per_rank * steps / (elapsed_ms_max / 1e3)


def make_cache(wl, dev, read_mode=None, seed=0):
    """Cache with a seeded synthetic initial state N(0, s0_std) drawn on the device."""
    import torch
    from checkpoint_input_replay_gb300 import ReplayCache
    cache = ReplayCache.for_shape(wl.shape, read_mode=read_mode, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + seed)
    ck = cache.ckpt
    for b0 in range(0, wl.shape.batch, 32):
        ck[b0:b0 + 32].normal_(0.0, wl.s0_std, generator=g)
    if read_mode is not None:
        cache.flush()
    torch.cuda.synchronize(dev)
    return cache


def run_decode_loop(cache, steps_inputs, K, W, dev, barrier):
    import torch
    stream = torch.cuda.current_stream(dev)
    D = len(steps_inputs)
    for t in range(W):
        inp, y = steps_inputs[t % D]
        cache.decode_step(inp, y, stream=stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for t in range(K):
        inp, y = steps_inputs[(W + t) % D]
        ev[t][0].record(stream)
        cache.decode_step(inp, y, stream=stream)
        ev[t][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    return start.elapsed_time(end), [a.elapsed_time(b) for a, b in ev]


def decode_leg(wl, dev, K, W, L, bytes_fn, barrier, distinct=16, seed=0):
    """Decode steps of one layer; warm-up W rounded up so timing starts at a window boundary."""
    import torch
    W = int(math.ceil(W / L) * L)
    cache = make_cache(wl, dev, seed=seed)
    A = torch.from_numpy(wl.A()).to(dev) if hasattr(wl, "A") else None
    steps = []
    for t in range(distinct):
        inp = upload(wl.step(t), dev)
        if A is not None:
            inp["A"] = A
        y = torch.empty(wl.shape.batch, wl.shape.n_heads, wl.shape.d_head, dtype=torch.float32, device=dev)
        steps.append((inp, y))
    elapsed, per = run_decode_loop(cache, steps, K, W, dev, barrier)
    err = cache.device_error()
    nbytes = [bytes_fn(wl.shape, (W + t) % L, (W + t) % L == L - 1) * wl.shape.batch for t in range(K)]
    flush_ms = [p for t, p in enumerate(per) if (W + t) % L == L - 1]
    nonflush_ms = [p for t, p in enumerate(per) if (W + t) % L != L - 1]
    flush_b = [b for t, b in enumerate(nbytes) if (W + t) % L == L - 1]
    nonflush_b = [b for t, b in enumerate(nbytes) if (W + t) % L != L - 1]
    res = {
        "elapsed_ms": elapsed, "launch_ms_total": sum(per), "bytes_total": sum(nbytes),
        "nonflush_gbs": sum(nonflush_b) / (sum(nonflush_ms) * 1e6) if nonflush_ms else None,
        "flush_gbs": sum(flush_b) / (sum(flush_ms) * 1e6) if flush_ms else None,
        "nonflush_us": 1e3 * statistics.mean(nonflush_ms) if nonflush_ms else None,
        "flush_us": 1e3 * statistics.mean(flush_ms) if flush_ms else None,
        "device_error": err, "launches": K, "flush_launches": len(flush_ms),
        "gap_us": 1e3 * (elapsed - sum(per)) / K,
    }
    res["natural_window"] = natural_window(res, wl.shape, L, bytes_fn)
    del cache, steps
    torch.cuda.empty_cache()
    return res


def natural_window(res, shape, L, bytes_fn):
    """The decode rate at the natural mix of one window (L - 1 non-flush steps, one
    flush), from the per-launch means and the mean gap between launches; and the
    window's algorithmic bytes over the summed launch times."""
    if res["flush_us"] is None or (L > 1 and res["nonflush_us"] is None):
        return None
    nf = res["nonflush_us"] if L > 1 else 0.0
    us = (L - 1) * nf + res["flush_us"] + L * res["gap_us"]
    nbytes = sum(bytes_fn(shape, h, h == L - 1) for h in range(L)) * shape.batch
    kern_us = (L - 1) * nf + res["flush_us"]
    return {"value": shape.batch * L / (us * 1e-6), "unit": UNIT, "us_per_step": us / L,
            "achieved_gbs": nbytes / (kern_us * 1e3), "window_bytes": nbytes,
            "note": f"{L - 1} non-flush + 1 flush launch at their mean times plus the mean launch gap"}


def e2e_leg(wl, dev, K, W):
    """Same metric through the C ABI's host-buffer call (rs_pipe_decode_step, via
    ReplayCache.decode_step_from_host): every step its pinned host inputs are copied in and y
    copied back to pinned host memory, the copies overlapping the neighbouring steps' kernels."""
    import torch
    cache = make_cache(wl, dev)
    host = []
    for t in range(16):
        raw = wl.step(t)
        h = {}
        for k, v in raw.items():
            ten = torch.from_numpy(v.view(np.int16).copy()).view(torch.bfloat16) if v.dtype == np.uint16 \
                else torch.from_numpy(np.ascontiguousarray(v))
            h[k] = ten.pin_memory()
        h["A"] = torch.from_numpy(wl.A()).pin_memory()
        host.append(h)
    y_host = torch.empty(wl.shape.batch, wl.shape.n_heads, wl.shape.d_head, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(dev)
    for t in range(W):
        cache.decode_step_from_host(host[t % 16], y_host, stream=stream)
    cache.host_sync(stream)
    torch.cuda.synchronize(dev)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for t in range(K):
        cache.decode_step_from_host(host[(W + t) % 16], y_host, stream=stream)
    cache.host_sync(stream)  # the last step's y is in host memory when `e` completes
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = s.elapsed_time(e)
    h2d = sum(v.numel() * v.element_size() for v in host[0].values())
    d2h = y_host.numel() * 4
    assert cache.device_error() == 0
    return {"value": wl.shape.batch * K / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / K}


def verify_leg(wl, dev, rounds, W, barrier):
    """Verify (T = 4) + commit rounds at B = 512; returns throughput and verify-kernel bandwidth."""
    import torch
    T = 4
    cache = make_cache(wl, dev)
    s = wl.shape
    is_m2 = s.kind == 0
    A = torch.from_numpy(wl.A()).to(dev) if is_m2 else None
    drafts, accs = [], []
    for r in range(4):
        inp = upload(wl.draft(r, T), dev)
        if A is not None:
            inp["A"] = A
        drafts.append(inp)
        accs.append(torch.from_numpy(wl.accepted(r, T)).to(dev))
    y = torch.empty(s.batch, T, s.n_heads, s.d_head, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for r in range(W):
        cache.verify(T, drafts[r % 4], y, stream=stream)
        cache.commit(accs[r % 4], stream=stream)
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(rounds)]
    barrier()
    for r in range(rounds):
        ev[r][0].record(stream)
        cache.verify(T, drafts[r % 4], y, stream=stream)
        ev[r][1].record(stream)
        cache.commit(accs[r % 4], stream=stream)
        ev[r][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ver = [a.elapsed_time(b) for a, b, _ in ev]
    com = [b.elapsed_time(c) for _, b, c in ev]
    total = ev[0][0].elapsed_time(ev[-1][2])
    # verify reads the state once plus ~mean ring (h ~ L/2) and the drafts
    H, P, N, G = s.n_heads, s.d_head, s.d_state, s.n_groups
    state = H * P * N * 4
    vbytes = s.batch * (state + T * H * P * 4)
    assert cache.device_error() == 0
    del cache
    torch.cuda.empty_cache()
    return {"workload": f"{'mamba2' if is_m2 else 'gdn'} verify T=4 + commit, B={s.batch}",
            "tokens_per_s": s.batch * T * rounds / (total / 1e3),
            "verify_us": 1e3 * statistics.mean(ver), "commit_us": 1e3 * statistics.mean(com),
            "verify_state_gbs": vbytes / (statistics.mean(ver) * 1e6), "rounds": rounds}


def read_copy_leg(wl, dev, mode, K, W):
    """Non-flush decode with the low-precision read copy (config 1 shape)."""
    import torch
    s = wl.shape
    cache = make_cache(wl, dev, read_mode=mode)
    A = torch.from_numpy(wl.A()).to(dev)
    steps = []
    for t in range(16):
        inp = upload(wl.step(t), dev)
        inp["A"] = A
        steps.append((inp, torch.empty(s.batch, s.n_heads, s.d_head, dtype=torch.float32, device=dev)))
    L = s.ring_len
    W = int(math.ceil(W / L) * L)
    elapsed, per = run_decode_loop(cache, steps, K, W, dev, lambda: None)
    nf = [(t, p) for t, p in enumerate(per) if (W + t) % L != L - 1]
    nonflush = [p for _, p in nf]
    fl = [p for t, p in enumerate(per) if (W + t) % L == L - 1]
    H, P, N = s.n_heads, s.d_head, s.d_state
    state = H * P * N * 4
    rc = H * P * N + H * P * 4 if mode == "fp8" else H * P * N // 2 + H * P * N // 16 + H * 4
    # all algorithmic bytes of a non-flush launch: the copy in place of the FP32 state,
    # plus the buffered records, this token's inputs, the output and the appended record
    nf_bytes = sum((m2_bytes(s, (W + t) % L, False) - state + rc) * s.batch for t, _ in nf)
    assert cache.device_error() == 0
    del cache
    torch.cuda.empty_cache()
    return {"mode": mode, "nonflush_us": 1e3 * statistics.mean(nonflush),
            "flush_us": 1e3 * statistics.mean(fl) if fl else None,
            "window_us_per_step": 1e3 * (sum(nonflush) / len(nonflush) * (L - 1) + (statistics.mean(fl) if fl else 0)) / L,
            "nonflush_gbs": nf_bytes / (sum(nonflush) * 1e6),
            "copy_bytes_per_seq": rc, "seq_steps_per_s": s.batch * K / (elapsed / 1e3)}


def _timed_launches(fn, K, W, dev):
    """W untimed calls, then K calls each bracketed by CUDA events on the current stream;
    returns (elapsed ms over the K calls, per-call ms)."""
    import torch
    stream = torch.cuda.current_stream(dev)
    for t in range(W):
        fn(t)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for t in range(K):
        ev[t][0].record(stream)
        fn(W + t)
        ev[t][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    return start.elapsed_time(end), [a.elapsed_time(b) for a, b in ev]


def _random_state(t, std, seed):
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    for b0 in range(0, t.shape[0], 32):
        t[b0:b0 + 32].normal_(0.0, std, generator=g)


def _uploaded_steps(wl, dev, n):
    import torch
    A = torch.from_numpy(wl.A()).to(dev) if wl.shape.kind == 0 else None
    out = []
    for t in range(n):
        inp = upload(wl.step(t), dev)
        if A is not None:
            inp["A"] = A
        out.append(inp)
    return out


def conventional_decode_leg(wl, dev, K, W):
    """The conventional read-modify-write decode step on the same GPU: the whole state is
    read and written back every token (rs_conventional_decode_step)."""
    import torch
    from checkpoint_input_replay_gb300 import ConventionalLayer
    s = wl.shape
    layer = ConventionalLayer.for_shape(s, device=dev)
    _random_state(layer.state, wl.s0_std, 2000)
    steps = _uploaded_steps(wl, dev, 16)
    y = torch.empty(s.batch, s.n_heads, s.d_head, dtype=torch.float32, device=dev)
    elapsed, per = _timed_launches(lambda t: layer.decode_step(steps[t % 16], y), K, W, dev)
    H, G, P, N = s.n_heads, s.n_groups, s.d_head, s.d_state
    inputs = (H * P * 2 + H * 2 + 2 * G * N * 2) if s.kind == 0 else (2 * G * N * 2 + H * P * 2 + 2 * H * 4)
    nbytes = s.batch * (2 * H * P * N * 4 + inputs + H * P * 4)
    us = 1e3 * statistics.mean(per)
    del layer, steps
    torch.cuda.empty_cache()
    return {"us_per_step": us, "achieved_gbs": nbytes / (us * 1e3), "bytes_per_step": nbytes,
            "value": s.batch * K / (elapsed / 1e3), "unit": UNIT, "launches": K}


def snapshot_leg(wl, dev, rounds, W):
    """Snapshot-per-draft speculative verify (one state read, T = 4 snapshot writes) and
    rollback by slot select, on the same GPU (rs_snapshot_verify / rs_snapshot_commit)."""
    import torch
    from checkpoint_input_replay_gb300 import SnapshotLayer
    T = 4
    s = wl.shape
    layer = SnapshotLayer.for_shape(s, device=dev)
    _random_state(layer.pool[:, 0], wl.s0_std, 3000)
    A = torch.from_numpy(wl.A()).to(dev) if s.kind == 0 else None
    drafts, accs = [], []
    for r in range(4):
        inp = upload(wl.draft(r, T), dev)
        if A is not None:
            inp["A"] = A
        drafts.append(inp)
        accs.append(torch.from_numpy(wl.accepted(r, T)).to(dev))
    y = torch.empty(s.batch, T, s.n_heads, s.d_head, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def one(r):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        layer.verify(T, drafts[r % 4], y, stream=stream)
        e1.record(stream)
        layer.commit(accs[r % 4], stream=stream)
        e2.record(stream)
        return e0, e1, e2
    for r in range(W):
        one(r)
    torch.cuda.synchronize(dev)
    evs = [one(W + r) for r in range(rounds)]
    torch.cuda.synchronize(dev)
    ver = [a.elapsed_time(b) for a, b, _ in evs]
    com = [b.elapsed_time(c) for _, b, c in evs]
    total = evs[0][0].elapsed_time(evs[-1][2])
    H, P, N = s.n_heads, s.d_head, s.d_state
    vbytes = s.batch * ((1 + T) * H * P * N * 4 + T * H * P * 4)
    assert layer.device_error() == 0
    del layer
    torch.cuda.empty_cache()
    return {"verify_us": 1e3 * statistics.mean(ver), "commit_us": 1e3 * statistics.mean(com),
            "verify_gbs": vbytes / (statistics.mean(ver) * 1e6), "round_us": 1e3 * total / rounds,
            "tokens_per_s": s.batch * T * rounds / (total / 1e3), "rounds": rounds}


def tree_verify_leg(wl, dev, rounds, W):
    """Tree-shaped speculation (four drafts: draft 0, two alternatives 1 and 2 after it,
    draft 3 after draft 1) verified in one pass, then each sequence's accepted
    root-to-draft path committed by index list; B = 512, same workload as the chain
    verify leg.  The accepted path per sequence and round comes from the workload's
    accepted count: 0 -> [], 1 -> [0], 2 -> [0, 1] or [0, 2] by sequence parity,
    3 or 4 -> [0, 1, 3]."""
    import torch
    T = 4
    parents = [-1, 0, 0, 1]
    cache = make_cache(wl, dev)
    s = wl.shape
    A = torch.from_numpy(wl.A()).to(dev) if s.kind == 0 else None
    drafts, lens, paths = [], [], []
    for r in range(4):
        inp = upload(wl.draft(r, T), dev)
        if A is not None:
            inp["A"] = A
        drafts.append(inp)
        acc = wl.accepted(r, T)
        pl = np.zeros(s.batch, dtype=np.int32)
        pt = np.zeros((s.batch, cache.T_max), dtype=np.int32)
        for b in range(s.batch):
            a = int(acc[b])
            path = [] if a == 0 else [0] if a == 1 else ([0, 1] if b % 2 == 0 else [0, 2]) if a == 2 else [0, 1, 3]
            pl[b] = len(path)
            pt[b, :len(path)] = path
        lens.append(torch.from_numpy(pl).to(dev))
        paths.append(torch.from_numpy(pt).to(dev))
    y = torch.empty(s.batch, T, s.n_heads, s.d_head, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for r in range(W):
        cache.verify_tree(T, parents, drafts[r % 4], y, stream=stream)
        cache.commit_path(lens[r % 4], paths[r % 4], stream=stream)
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(rounds)]
    for r in range(rounds):
        ev[r][0].record(stream)
        cache.verify_tree(T, parents, drafts[r % 4], y, stream=stream)
        ev[r][1].record(stream)
        cache.commit_path(lens[r % 4], paths[r % 4], stream=stream)
        ev[r][2].record(stream)
    torch.cuda.synchronize(dev)
    ver = [a.elapsed_time(b) for a, b, _ in ev]
    com = [b.elapsed_time(c) for _, b, c in ev]
    total = ev[0][0].elapsed_time(ev[-1][2])
    assert cache.device_error() == 0
    del cache
    torch.cuda.empty_cache()
    return {"workload": f"{'mamba2' if s.kind == 0 else 'gdn'} tree verify (parents {parents}) + path commit, "
                        f"B={s.batch}",
            "verify_us": 1e3 * statistics.mean(ver), "commit_us": 1e3 * statistics.mean(com),
            "round_us": 1e3 * total / rounds, "rounds": rounds}


def read_copy_error_leg(wl, dev, mode, steps):
    """Per-window rel-L2 of the read-copy outputs against the FP32-checkpoint outputs of
    the same kernels on the same inputs (two caches side by side; the FP32 path itself
    matches the float64 recurrence within 2e-4 in the tests), and the non-flush launch's
    algorithmic bytes over its time."""
    import torch
    s = wl.shape
    L = s.ring_len
    from checkpoint_input_replay_gb300 import ReplayCache
    exact = make_cache(wl, dev, seed=7)
    quant = ReplayCache.for_shape(s, read_mode=mode, device=dev)
    quant.ckpt.copy_(exact.ckpt)
    quant.flush()
    steps_in = _uploaded_steps(wl, dev, 16)
    y0 = torch.empty(s.batch, s.n_heads, s.d_head, dtype=torch.float32, device=dev)
    y1 = torch.empty_like(y0)
    nw = steps // L
    num = torch.zeros(nw, dtype=torch.float64, device=dev)
    den = torch.zeros(nw, dtype=torch.float64, device=dev)
    for t in range(steps):
        exact.decode_step(steps_in[t % 16], y0)
        quant.decode_step(steps_in[t % 16], y1)
        w = t // L
        num[w] += ((y1 - y0).double() ** 2).sum()
        den[w] += (y0.double() ** 2).sum()
    per_window = torch.sqrt(num / den).cpu().numpy()
    assert exact.device_error() == 0 and quant.device_error() == 0
    del exact, quant
    torch.cuda.empty_cache()
    return {"per_window_rel_l2_first8": [round(float(x), 6) for x in per_window[:8]],
            "per_window_rel_l2_last4": [round(float(x), 6) for x in per_window[-4:]],
            "windows": nw, "max_window_ge1": float(per_window[1:].max()),
            "aggregate_rel_l2": float(np.sqrt(num.sum().item() / den.sum().item())),
            "first8_mean": float(per_window[1:9].mean()), "last8_mean": float(per_window[-8:].mean()),
            "inputs": "16 distinct seeded input steps cycled; initial state N(0,0.1)"}


def mixed_phase_leg(wl, dev, K, W, uniform=False):
    """Decode with the sequences at staggered window positions (after step k of the first
    window, the sequences b with b % L == k are folded by rs_flush), so that every launch
    mixes flush and non-flush sequences, about one in L folding."""
    import torch
    s = wl.shape
    L = s.ring_len
    if uniform:  # the even split of units over the CTAs, for comparison
        os.environ["RS_DEBUG_UNIFORM_SPLIT"] = "1"
    try:
        cache = make_cache(wl, dev, seed=11)
    finally:
        os.environ.pop("RS_DEBUG_UNIFORM_SPLIT", None)
    steps = _uploaded_steps(wl, dev, 16)
    y = torch.empty(s.batch, s.n_heads, s.d_head, dtype=torch.float32, device=dev)
    for k in range(L):
        cache.decode_step(steps[k % 16], y)
        mask = torch.tensor([1 if b % L == k else 0 for b in range(s.batch)], dtype=torch.uint8, device=dev)
        cache.flush(mask)
    elapsed, per = _timed_launches(lambda t: cache.decode_step(steps[t % 16], y), K, W, dev)
    folding = int(cache.cursor[:, 2].sum().item())
    assert cache.device_error() == 0
    del cache, steps
    torch.cuda.empty_cache()
    us = 1e3 * elapsed / K
    return {"us_per_step": us, "value": s.batch * K / (elapsed / 1e3), "unit": UNIT, "launches": K,
            "folding_last_step": folding,
            "note": f"sequences at {L} staggered window positions; every launch folds about 1/{L} of them"}


def graph_window_leg(wl, dev, windows, warm):
    """One window of decode steps (L launches) captured once as a CUDA graph and replayed."""
    import torch
    s = wl.shape
    L = s.ring_len
    cache = make_cache(wl, dev, seed=12)
    steps = _uploaded_steps(wl, dev, L)
    ys = [torch.empty(s.batch, s.n_heads, s.d_head, dtype=torch.float32, device=dev) for _ in range(L)]
    for t in range(L):  # eager first window: every kernel configured before the capture
        cache.decode_step(steps[t], ys[t])
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            for t in range(L):
                cache.decode_step(steps[t], ys[t], stream=cs)
    torch.cuda.current_stream(dev).wait_stream(cs)
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(windows):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    assert cache.device_error() == 0
    del g, cache, steps
    torch.cuda.empty_cache()
    return {"us_per_step": 1e3 * ms / (windows * L), "value": s.batch * windows * L / (ms / 1e3), "unit": UNIT,
            "windows": windows, "note": f"one captured window of {L} decode launches, replayed"}


def sweep_leg(dev, kind, batch, L, K, W, with_conventional=True):
    """One point of the batch / window-length sweeps: the ReplaySSM decode at its natural
    window mix and, at the same shape, the conventional decode step."""
    import dataclasses as dc
    from workloads import configs
    base = configs.CONFIG1 if kind == 0 else configs.CONFIG2
    shape = dc.replace(base, batch=batch, ring_len=L)
    wl = configs.Mamba2Workload(shape, seed=1, s0_std=0.1) if kind == 0 else \
        configs.GdnWorkload(shape, seed=2, s0_std=0.05)
    r = decode_leg(wl, dev, K, W, L, m2_bytes if kind == 0 else gdn_bytes, lambda: None)
    nat = r["natural_window"]
    out = {"batch": batch, "L": L, "value": nat["value"], "us_per_step": nat["us_per_step"],
           "nonflush_us": r["nonflush_us"], "flush_us": r["flush_us"], "achieved_gbs": nat["achieved_gbs"]}
    if with_conventional:
        c = conventional_decode_leg(wl, dev, max(K // 2, 4), 3)
        out["conventional_us_per_step"] = c["us_per_step"]
        out["speedup_vs_conventional"] = c["us_per_step"] / nat["us_per_step"]
    return out


# ----------------------------------------------------------------------------- oracle arm

def oracle_sample(wl, steps: int, seqs: list[int]):
    """Time the float64 oracle's conventional decode on a few sequences of the workload."""
    from oracle.layer import OracleLayer
    inputs = [{k: v for k, v in wl.step(t, seqs[0], seqs[-1] + 1).items()} for t in range(steps)]
    S0 = wl.S0(seqs[0], seqs[-1] + 1)
    lay = OracleLayer(wl.shape, seqs, S0, A=wl.A() if hasattr(wl, "A") else None)
    t0 = time.perf_counter()
    for t in range(steps):
        lay.decode(inputs[t])
    dt = time.perf_counter() - t0
    return len(seqs) * steps / dt, dt


def _oracle_worker(args):
    """One host process of the CPU baseline: the oracle on one sequence of the
    config-1 workload (runs in a spawned process, one BLAS thread)."""
    seq, steps = args
    from workloads import configs
    return oracle_sample(configs.config1(), steps, [seq])


def cpu_baseline_leg(steps_single=512, steps_each=256):
    """The float64 oracle timed on the host: one core on one sequence (>= 1 s of work),
    then one spawned process per host core, each on its own sequence, run together."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    env_keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env_keep:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(1) as pool:
            rate1, secs1 = pool.map(_oracle_worker, [(0, steps_single)])[0]
        with ctx.Pool(cores) as pool:
            res = pool.map(_oracle_worker, [(i, steps_each) for i in range(cores)])
    finally:
        for k, v in env_keep.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    wall = max(r[1] for r in res)
    return {"value": cores * steps_each / wall, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{steps_each} decode steps of each of sequences 0-{cores - 1} of the B=256 config-1 "
                      f"workload, one float64 numpy process per host core, run together "
                      f"(slowest process {wall:.1f} s)",
            "single_core": {"value": rate1, "unit": UNIT, "cores": 1,
                            "sample": f"{steps_single} decode steps of sequence 0 ({secs1:.1f} s)"}}


def window_state_ratio(win, shape):
    """Measured state bytes of one L = 16 window over (L + 1) |S|: the ncu DRAM bytes of the
    window's 16 decode launches (one capture, B = win["batch"]) minus their non-state
    algorithmic bytes (records, tokens, outputs), divided by L + 1 state reads/writes."""
    L = shape.ring_len
    state = shape.n_heads * shape.d_head * shape.d_state * 4
    launches = sorted(win["launches"], key=lambda r: r["pos"])
    dram = sum(r["dram_bytes"] for r in launches)
    alg = sum(m2_bytes(shape, r["pos"], r["pos"] == L - 1) for r in launches) * shape.batch
    state_alg = (L + 1) * state * shape.batch
    return {"window_state_ratio": (dram - (alg - state_alg)) / state_alg,
            "window_traffic_over_algorithmic": dram / alg,
            "window_capture": f"ncu DRAM bytes of the {len(launches)} decode launches of one window at "
                              f"B={shape.batch} ({win['summary']})"}


def extras(line, args, dev, hbm, m2):
    """The other legs: GDN decode, verify + commit, read copies, the conventional kernels
    and the ratios, the batch and window-length sweeps."""
    from workloads import configs
    W = args.warmup
    Kx = 64  # four windows per leg
    with nvtx_range("decode gdn"):
        gdn = decode_leg(configs.config2(), dev, Kx, W, 16, gdn_bytes, lambda: None)
    line["gdn"] = {"workload": "gdn decode, 1 layer: B=256 Hv=32 Hk=16 dk=dv=128, L=16",
                   "value": configs.config2().shape.batch * Kx / (gdn["elapsed_ms"] / 1e3),
                   "unit": UNIT, "achieved_gbs": gdn["bytes_total"] / (gdn["launch_ms_total"] * 1e6),
                   "nonflush_gbs": gdn["nonflush_gbs"], "flush_gbs": gdn["flush_gbs"],
                   "nonflush_us": gdn["nonflush_us"], "flush_us": gdn["flush_us"],
                   "frac": gdn["bytes_total"] / (gdn["launch_ms_total"] * 1e6) / hbm,
                   "natural_window": gdn["natural_window"]}
    with nvtx_range("decode per-channel gate"):
        kda = decode_leg(configs.config_kda(), dev, Kx, W, 16, kda_bytes, lambda: None)
    line["kda"] = {"workload": "decode, delta rule with a per-key-channel gate, 1 layer: B=256 Hv=32 Hk=16 "
                               "dk=dv=128, L=16", "unit": UNIT, "natural_window": kda["natural_window"],
                   "nonflush_us": kda["nonflush_us"], "flush_us": kda["flush_us"],
                   "nonflush_gbs": kda["nonflush_gbs"], "flush_gbs": kda["flush_gbs"],
                   "frac": kda["natural_window"]["achieved_gbs"] / hbm}
    with nvtx_range("verify + commit"):
        ver = [verify_leg(configs.config3_mamba2(), dev, 64, 4, lambda: None),
               verify_leg(configs.config3_gdn(), dev, 64, 4, lambda: None)]
    for v in ver:
        v["verify_frac"] = v["verify_state_gbs"] / hbm
    line["verify"] = ver
    with nvtx_range("tree verify + path commit"):
        line["tree_verify"] = [tree_verify_leg(configs.config3_mamba2(), dev, 32, 4),
                               tree_verify_leg(configs.config3_gdn(), dev, 32, 4)]
    rc = []
    for mode in ("fp8", "nvfp4"):
        with nvtx_range(f"decode read copy {mode}"):
            r = read_copy_leg(configs.config4(), dev, mode, Kx, W)
        r["nonflush_frac"] = r["nonflush_gbs"] / hbm
        r["speedup_vs_fp32_nonflush"] = m2["nonflush_us"] / r["nonflush_us"]
        with nvtx_range(f"read copy error {mode}"):
            r["error_vs_fp32_outputs"] = read_copy_error_leg(configs.config4(), dev, mode, 4096)
        rc.append(r)
    line["read_copy"] = rc
    with nvtx_range("conventional kernels"):
        cm2 = conventional_decode_leg(configs.config1(), dev, 32, W)
        cgdn = conventional_decode_leg(configs.config2(), dev, 32, W)
        sm2 = snapshot_leg(configs.config3_mamba2(), dev, 32, 4)
        sgdn = snapshot_leg(configs.config3_gdn(), dev, 32, 4)
        # the same read-modify-write per token, run by the ReplaySSM decode kernel at L = 1
        # (every step folds its one record and writes the state)
        l1m2 = sweep_leg(dev, 0, 256, 1, 16, 16, with_conventional=False)
        l1gdn = sweep_leg(dev, 1, 256, 1, 16, 16, with_conventional=False)
    for c in (sm2, sgdn):
        c["verify_frac"] = c["verify_gbs"] / hbm
    for c in (cm2, cgdn):
        c["frac"] = c["achieved_gbs"] / hbm
    best_m2 = min(cm2["us_per_step"], l1m2["us_per_step"])
    best_gdn = min(cgdn["us_per_step"], l1gdn["us_per_step"])
    line["conventional"] = {
        "decode_mamba2": cm2, "decode_gdn": cgdn, "snapshot_spec_mamba2": sm2, "snapshot_spec_gdn": sgdn,
        "decode_mamba2_as_window_1": l1m2, "decode_gdn_as_window_1": l1gdn,
        "decode_speedup_mamba2": best_m2 / m2["natural_window"]["us_per_step"],
        "decode_speedup_gdn": best_gdn / gdn["natural_window"]["us_per_step"],
        "spec_speedup_mamba2": ver[0]["tokens_per_s"] / sm2["tokens_per_s"],
        "spec_speedup_gdn": ver[1]["tokens_per_s"] / sgdn["tokens_per_s"],
        "note": "same GPU, same shapes: decode at the natural 15:1 window mix vs the faster of the two "
                "read-modify-write steps (the conventional kernel, and the ReplaySSM kernel at L=1); "
                "speculative T=4 verify + commit rounds at B=512 vs snapshot-per-draft verify + "
                "slot-select commit"}
    with nvtx_range("mixed window positions"):
        mp = mixed_phase_leg(configs.config1(), dev, 64, 16)
        mp_even = mixed_phase_leg(configs.config1(), dev, 64, 16, uniform=True)
    mp["vs_synchronized_window"] = m2["natural_window"]["us_per_step"] / mp["us_per_step"]
    mp["even_split_us_per_step"] = mp_even["us_per_step"]
    mp["weighted_split_speedup"] = mp_even["us_per_step"] / mp["us_per_step"]
    line["mixed_phase"] = mp
    with nvtx_range("cuda graph window"):
        gw = graph_window_leg(configs.config1(), dev, 8, 2)
    gw["vs_eager_window"] = m2["natural_window"]["us_per_step"] / gw["us_per_step"]
    line["graph_window"] = gw
    with nvtx_range("batch sweep"):
        line["batch_sweep"] = [sweep_leg(dev, 0, b, 16, 32, 16) for b in (1, 16, 64, 256, 1024)]
    with nvtx_range("window sweep"):
        line["window_sweep"] = [sweep_leg(dev, kind, 256, L, 2 * L, L, with_conventional=False)
                                for kind in (0, 1) for L in (4, 8, 16, 32)]
        for r, kind in zip(line["window_sweep"], [0] * 4 + [1] * 4):
            r["kind"] = "mamba2" if kind == 0 else "gdn"


# ----------------------------------------------------------------------------- main

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reference_arm(args, world, rank):
    """--impl reference: the oracle on the host cores, same metric and workload."""
    from workloads import configs
    if rank != 0:
        return 0
    wl = configs.config1()
    per_step_seqs = [0]
    for _ in range(args.warmup):
        oracle_sample(wl, 1, per_step_seqs)
    total = 0.0
    from oracle.layer import OracleLayer
    inputs = [wl.step(t, 0, 1) for t in range(16)]
    lay = OracleLayer(wl.shape, [0], wl.S0(0, 1), A=wl.A())
    t0 = time.perf_counter()
    for t in range(args.steps):
        lay.decode(inputs[t % 16])
    total = time.perf_counter() - t0
    value = args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "mamba2 decode, config-1 layer (H128 P64 N128 G8 L16), one sequence per step",
                       "batch": 1},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} decode steps of sequence 0 of the B=256 workload "
                                       "(float64 numpy, one thread)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3200)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the GDN / verify / read-copy objects")
    ap.add_argument("--batch", type=int, default=256,
                    help="sequences per GPU of the Mamba-2 decode leg (the metric is quoted at 256)")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the Mamba-2 decode leg (a small profiling case with --batch)")
    ap.add_argument("--verify-only", choices=["mamba2", "gdn"],
                    help="time only one verify + commit leg, at --verify-batch sequences (a profiling case)")
    ap.add_argument("--verify-batch", type=int, default=512)
    ap.add_argument("--gdn-decode-only", action="store_true",
                    help="time only the GDN decode leg, at --batch sequences (a profiling case)")
    ap.add_argument("--read-copy-only", choices=["fp8", "nvfp4"],
                    help="time only the non-flush decode with a read copy, at --batch sequences (a profiling case)")
    ap.add_argument("--kda-decode-only", action="store_true",
                    help="time only the per-channel-gate decode leg, at --batch sequences (a profiling case)")
    ap.add_argument("--conventional-only", choices=["mamba2", "gdn"],
                    help="time only the conventional read-modify-write decode step, at --batch sequences "
                         "(a profiling case)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    from workloads import configs
    import checkpoint_input_replay_gb300  # noqa: F401  (fails loudly if the library is missing)

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.verify_only:
        wl = (configs.config3_mamba2 if args.verify_only == "mamba2" else configs.config3_gdn)(args.verify_batch)
        res = verify_leg(wl, dev, args.steps, args.warmup, lambda: None)
        if rank == 0:
            print(json.dumps({"verify": res}))
        return 0
    if args.gdn_decode_only:
        wl = configs.config2(batch=args.batch)
        r = decode_leg(wl, dev, args.steps, args.warmup, 16, gdn_bytes, lambda: None)
        if rank == 0:
            print(json.dumps({"gdn": {"batch": args.batch, "nonflush_us": r["nonflush_us"], "flush_us": r["flush_us"],
                                      "nonflush_gbs": r["nonflush_gbs"], "launches": r["launches"]}}))
        return 0
    if args.kda_decode_only:
        wl = configs.config_kda(batch=args.batch)
        r = decode_leg(wl, dev, args.steps, args.warmup, 16, kda_bytes, lambda: None)
        if rank == 0:
            print(json.dumps({"kda": {"batch": args.batch, "nonflush_us": r["nonflush_us"], "flush_us": r["flush_us"],
                                      "nonflush_gbs": r["nonflush_gbs"], "natural_window": r["natural_window"],
                                      "launches": r["launches"]}}))
        return 0
    if args.conventional_only:
        wl = (configs.config1 if args.conventional_only == "mamba2" else configs.config2)(batch=args.batch)
        res = conventional_decode_leg(wl, dev, args.steps, args.warmup)
        if rank == 0:
            print(json.dumps({"conventional": res}))
        return 0
    if args.read_copy_only:
        res = read_copy_leg(configs.config1(batch=args.batch), dev, args.read_copy_only, args.steps, args.warmup)
        if rank == 0:
            print(json.dumps({"read_copy": res}))
        return 0
    if world > 1:
        import torch.distributed as dist
        barrier = lambda: dist.barrier()
    else:
        barrier = lambda: None

    K, W = args.steps, args.warmup
    # each rank decodes its own slice of a world x B job (weak scaling, no exchange)
    wl1 = shard_of(configs.config1(batch=world * args.batch), rank, world)
    with ClockSampler(local) as clk:
        with nvtx_range("decode mamba2 (headline)"):
            m2 = decode_leg(wl1, dev, K, W, 16, m2_bytes, barrier, seed=rank)
    elapsed = max_over_ranks(m2["elapsed_ms"], world, dev)
    value = job_value(world, wl1.shape.batch, K, elapsed)

    hbm, peak_kind = peaks()
    achieved = m2["bytes_total"] / (m2["launch_ms_total"] * 1e6)
    # DRAM bytes per launch: the mean over one captured L = 16 window of the same
    # workload (ncu, uncached), like `achieved`, which is over whole-window mixes
    win = ncu_record("decode_mamba2_window_b256") if wl1.shape.batch == 256 else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": (sum(r["dram_bytes"] for r in win["launches"]) / len(win["launches"])) if win else None,
                "peak_kind": peak_kind,
                "nonflush_gbs": m2["nonflush_gbs"], "nonflush_frac": m2["nonflush_gbs"] / hbm,
                "flush_gbs": m2["flush_gbs"], "nonflush_us": m2["nonflush_us"], "flush_us": m2["flush_us"]}
    if win:
        roofline.update(window_state_ratio(win, configs.CONFIG1.with_batch(win["batch"])))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": elapsed / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": "mamba2 decode, 1 layer: B=256 nheads=128 headdim=64 dstate=128 ngroups=8, "
                                   "FP32 checkpoint, bf16 x/dt/B/C, L=16 (15 non-flush + 1 flush per window)",
                       "batch_per_gpu": wl1.shape.batch, "global_batch": world * wl1.shape.batch, "ring_len": 16,
                       "timed_launches": K, "flush_launches_timed": m2["flush_launches"],
                       "l2": "no flush: the %d MiB state per step exceeds the 129 MB L2" % (wl1.shape.batch * 4),
                       "inputs": "16 distinct seeded input steps resident in HBM, cycled; initial state N(0,0.1)"},
            "natural_window": m2["natural_window"],
            "roofline": roofline, "gpu_launches": m2["launches"], "clocks": clk.summary(),
            "device_error": m2["device_error"]}
    if rank == 0 and args.decode_only:
        print(json.dumps(line), flush=True)
    elif rank == 0:
        with nvtx_range("decode mamba2 from host buffers"):
            line["e2e"] = e2e_leg(wl1, dev, E2E_STEPS, W)
        line["e2e"]["steps"] = E2E_STEPS
        if world == 1:
            line["cpu_baseline"] = cpu_baseline_leg()
        if not args.no_extra:
            extras(line, args, dev, hbm, m2)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
