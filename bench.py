#!/usr/bin/env python3
"""Benchmark of the KDA chunked packed-varlen prefill on one GB300.

Workload: the production packed chunk -- 16 sequences with seeded Dirichlet(1)
lengths summing to 8192 rows, H = 32, dk = dv = 128, bf16 q/k/v/out, fp32
g/beta, nonzero fp32 initial states, fp32 final states (kern-k3-pp-prefill
README, "P: the packed prefill").  One step is one kda_chunk_prefill call over
the whole chunk.  Metric: rows (tokens) per second, plus the achieved fraction
of the HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints ONE JSON line.  --impl reference times the fp64 CPU oracle on the host
cores instead (the reference arm of this build).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA packed-prefill tokens/s on 1 GB300 (8192-row chunk) + % of roofline"
WORKLOAD = "packed16_8192"
KERNEL_NAME = "kda_tc_kernel"
BYTES_PER_TOKEN_HEAD = 1540          # q, k, v, out bf16 (4 x 256 B) + g fp32 (512 B) + beta (4 B)


def algorithmic_bytes(w, with_initial=True, with_final=True) -> int:
    per_state = w.dk * w.dv * 4
    b = w.T * w.H * BYTES_PER_TOKEN_HEAD
    b += w.N * w.H * per_state * (int(with_initial) + int(with_final))
    return b


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# the sources a kernel is compiled from (its launcher included)
KERNEL_SOURCES = ("kda_common.cuh", "kda_internal.h", "kda_sm100.cuh", "kda_tc.cu")
DECODE_SOURCES = ("kda_common.cuh", "kda_decode.h", "kda_decode.cu")
CONV_SOURCES = ("kda_common.cuh", "kda_conv.h", "kda_conv.cu")


def code_only(text: str) -> str:
    """C/C++ source without comments, trailing blanks and empty lines: what the
    compiler sees (comment edits do not invalidate a recorded measurement)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_sha(sources=None) -> str:
    csrc = os.path.join(ROOT, "kda_linear_attention_chunk_gb300", "csrc")
    h = hashlib.sha256()
    for f in sources or KERNEL_SOURCES:
        h.update(code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str = None, sources=None):
    """DRAM bytes per launch from a committed ncu summary (profiles/traffic.txt for
    the prefill, profiles/traffic_<workload>.txt otherwise), if it was taken on
    the kernel sources as they are now; else None."""
    workload = workload or WORKLOAD
    name = "traffic.txt" if workload == WORKLOAD else f"traffic_{workload}.txt"
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    d = {}
    for line in open(path):
        if ":" in line and not line.lstrip().startswith("#"):
            key, val = line.split(":", 1)
            d[key.strip()] = val.strip()
    if d.get("kernel_source_sha") != kernel_source_sha(sources) or d.get("workload") != workload:
        return None
    return int(d["dram_bytes_per_launch"]) if "dram_bytes_per_launch" in d else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.tmp, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.p = None

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.tmp.flush()
        rows = []
        for line in open(self.tmp.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 9:
                rows.append(parts)
        os.unlink(self.tmp.name)
        return rows


def summarize_clocks(rows):
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
    def num(x):
        try:
            return float(x)
        except ValueError:
            return None
    sm = [num(r[1]) for r in rows if num(r[1]) is not None]
    mx = [num(r[2]) for r in rows if num(r[2]) is not None]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(rows)}


def make_device_inputs(w, seed_offset, torch, np):
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    w2 = syn.Workload(w.name, w.lengths, w.H, w.dk, w.dv, w.qkv_dtype, w.init_state, seed=w.seed + seed_offset)
    x = syn.draw(w2)
    s0 = syn.draw_initial_state(w2)
    pin = {}
    for k, v in x.items():
        t = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16 else torch.from_numpy(v)
        pin[k] = t.pin_memory()
    pin["s0"] = torch.from_numpy(s0).pin_memory()
    pin["cu"] = torch.from_numpy(w.cu_seqlens()).pin_memory()
    dev = {k: v.cuda() for k, v in pin.items()}
    return pin, dev


DECODE_N, DECODE_H = 64, 32   # decode: 64 running requests, one token each, 32 heads


def decode_bytes(n_live: int, n: int, h: int) -> int:
    """Algorithmic bytes of one decode step: each live (sequence, head) reads and
    writes its 64 KiB state; per row-head q, k, v, out (256 B each), g (512 B),
    beta (4 B); the slot table."""
    return n_live * h * 2 * 128 * 128 * 4 + n * h * (4 * 256 + 512 + 4) + 4 * n


def measure_decode(torch, np, kda, stream, steps: int = 100, warmup: int = 10):
    """kda_decode on DECODE_N sequences x DECODE_H heads: a pool of 2 x DECODE_N
    entries, the steps alternating between two slot tables that name disjoint
    halves of it (each half 134 MB, above L2), CUDA events on the stream."""
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    n, h = DECODE_N, DECODE_H
    w = syn.Workload("decode64_h32", [1] * n, H=h, dk=128, dv=128, seed=77)
    x = syn.draw(w)
    d = {k: (torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16
             else torch.from_numpy(v)).cuda() for k, v in x.items()}
    rng = np.random.default_rng(77)
    pool = torch.from_numpy((0.02 * rng.standard_normal((2 * n, h, 128, 128))).astype(np.float32)).cuda()
    perm = rng.permutation(2 * n).astype(np.int32)
    tables = [torch.from_numpy(np.sort(perm[:n])).cuda(), torch.from_numpy(np.sort(perm[n:])).cuda()]
    out = torch.empty((n, h, 128), dtype=torch.bfloat16, device="cuda")

    def step(i):
        kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, state_slots=tables[i % 2], out=out,
                   stream=stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    alg = decode_bytes(n, n, h)
    peak, peak_kind = peaks()
    achieved = alg / (ms / 1e3) / 1e9
    return {"workload": "decode64_h32", "kernel": "kda_decode_kernel", "N": n, "H": h, "steps": steps,
            "us_per_step": ms * 1e3, "tokens_per_s": n / (ms / 1e3),
            "l2": "2 slot tables over disjoint halves of a 2 x 64-entry pool (134 MB each)",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "algorithmic_bytes_per_launch": alg,
                         "traffic": recorded_traffic("decode64_h32", DECODE_SOURCES)}}


def decode_conv_bytes(n: int, h: int) -> int:
    """Algorithmic bytes of one fused conv + decode step: the decode step's
    (the projections in place of q, k, v), plus per sequence its window entry
    read and written (3 taps x 3 streams x H x 128 bf16 each way), the filters
    (3 x H x 128 x 4 fp32) and the window slot table."""
    return decode_bytes(n, n, h) + n * 2 * 9 * h * 128 * 2 + 3 * h * 128 * 4 * 4 + 4 * n


def measure_decode_conv(torch, np, kda, stream, steps: int = 100, warmup: int = 10):
    """kda_decode_conv (SiLU) on the decode step's shape: state and window pools
    of 2 x DECODE_N entries, the steps alternating between two pairs of slot
    tables over disjoint halves of them (134 MB of states each, above L2)."""
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    n, h = DECODE_N, DECODE_H
    w = syn.Workload("decode_conv64_h32", [1] * n, H=h, dk=128, dv=128, seed=78)
    x = syn.draw(w)
    d = {k: (torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16
             else torch.from_numpy(v)).cuda() for k, v in x.items()}
    rng = np.random.default_rng(78)
    pool = torch.from_numpy((0.02 * rng.standard_normal((2 * n, h, 128, 128))).astype(np.float32)).cuda()
    cpool = torch.from_numpy(rng.standard_normal((2 * n, 3, 3, h * 128)).astype(np.float32)).to(torch.bfloat16).cuda()
    cw = torch.from_numpy((0.5 * rng.standard_normal((3, h * 128, 4))).astype(np.float32)).cuda()
    perm = rng.permutation(2 * n).astype(np.int32)
    tables = [torch.from_numpy(np.sort(perm[:n])).cuda(), torch.from_numpy(np.sort(perm[n:])).cuda()]
    ctables = [tables[1].flip(0).contiguous(), tables[0].flip(0).contiguous()]
    out = torch.empty((n, h, 128), dtype=torch.bfloat16, device="cuda")

    def step(i):
        kda.decode_conv(d["q"], d["k"], d["v"], cw, cpool, d["g"], d["beta"], pool, conv_slots=ctables[i % 2],
                        state_slots=tables[i % 2], activation="silu", out=out, stream=stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    # the same step as two calls: the short conv on the N one-row sequences, then
    # the decode step on its bf16 q, k, v
    cu1 = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    qkv = tuple(torch.empty_like(d["q"]) for _ in range(3))

    def two_calls(i):
        kda.short_conv(d["q"], d["k"], d["v"], cw, cu1, cpool, conv_slots=ctables[i % 2], activation="silu",
                       out=qkv, stream=stream)
        kda.decode(qkv[0], qkv[1], qkv[2], d["g"], d["beta"], pool, state_slots=tables[i % 2], out=out,
                   stream=stream)

    for i in range(warmup):
        two_calls(i)
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(steps):
        two_calls(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms2 = ev0.elapsed_time(ev1) / steps
    alg = decode_conv_bytes(n, h)
    peak, peak_kind = peaks()
    achieved = alg / (ms / 1e3) / 1e9
    return {"workload": "decode_conv64_h32", "kernel": "kda_decode_conv_kernel", "N": n, "H": h, "steps": steps,
            "activation": "silu", "us_per_step": ms * 1e3, "tokens_per_s": n / (ms / 1e3),
            "two_calls_us_per_step": ms2 * 1e3,
            "l2": "2 pairs of slot tables over disjoint halves of 2 x 64-entry state and window pools",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "algorithmic_bytes_per_launch": alg,
                         "traffic": recorded_traffic("decode_conv64_h32", DECODE_SOURCES)}}


def conv_bytes(lengths, h: int) -> int:
    """Algorithmic bytes of one short-conv prologue call: per row-head the q, k,
    v projections in and q, k, v out (256 B each); the filters (3 x H x 128 x 4
    fp32); per sequence with rows its window entry read and written (3 taps x
    3 streams x H x 128 bf16 each way); cu_seqlens and the slot table."""
    t = int(sum(lengths))
    live = sum(1 for n in lengths if n > 0)
    n = len(lengths)
    return t * h * 6 * 256 + 3 * h * 128 * 4 * 4 + live * 2 * 9 * h * 128 * 2 + 4 * (2 * n + 1)


def measure_conv(torch, np, kda, stream, steps: int = 100, warmup: int = 10):
    """kda_short_conv (SiLU) on the packed 8192-row workload's lengths at H = 32:
    two rotating input sets (each call moves 403 MB, above L2), windows in a
    pool of 2 x 16 entries, the calls alternating between its halves."""
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    n_heads = 32
    lengths = list(syn.workloads()[WORKLOAD].lengths)
    rng = np.random.default_rng(79)
    t_rows = int(sum(lengths))
    sets = []
    for _ in range(2):
        xs = [torch.from_numpy((rng.standard_normal((t_rows, n_heads, 128))).astype(np.float32)).to(torch.bfloat16).cuda()
              for _ in range(3)]
        outs = tuple(torch.empty_like(xs[0]) for _ in range(3))
        sets.append((xs, outs))
    w = torch.from_numpy((0.5 * rng.standard_normal((3, n_heads * 128, 4))).astype(np.float32)).cuda()
    n = len(lengths)
    pool = torch.zeros((2 * n, 3, 3, n_heads * 128), dtype=torch.bfloat16, device="cuda")
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).cuda()
    tables = [torch.arange(0, n, dtype=torch.int32, device="cuda"), torch.arange(n, 2 * n, dtype=torch.int32, device="cuda")]

    def step(i):
        xs, outs = sets[i % 2]
        kda.short_conv(xs[0], xs[1], xs[2], w, cu, pool, conv_slots=tables[(i // 2) % 2], activation="silu",
                       out=outs, stream=stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    alg = conv_bytes(lengths, n_heads)
    peak, _ = peaks()
    achieved = alg / (ms / 1e3) / 1e9
    return {"workload": "conv_packed16_8192_h32", "kernel": "kda_conv_kernel",
            "T": t_rows, "N": n, "H": n_heads, "activation": "silu", "steps": steps, "us_per_call": ms * 1e3,
            "tokens_per_s": t_rows / (ms / 1e3), "l2": "2 rotating input sets of 201 MB (projections) each",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "algorithmic_bytes_per_launch": alg,
                         "traffic": recorded_traffic("conv_packed16_8192_h32", CONV_SOURCES)}}


def conv_prefill_bytes(lengths, h: int) -> int:
    """Algorithmic bytes of one fused layer call: per row-head the x_q, x_k, x_v
    projections (256 B each), g (512 B), beta (4 B) and out (256 B); every
    sequence's state entry read and written (64 KiB each way) and its window
    entry read and written (9 x H x 128 bf16 each way); the filters."""
    t = int(sum(lengths))
    live = sum(1 for n in lengths if n > 0)
    return (t * h * (3 * 256 + 512 + 4 + 256) + live * h * 2 * 128 * 128 * 4 + live * 2 * 9 * h * 128 * 2 +
            3 * h * 128 * 4 * 4)


def measure_conv_prefill(torch, np, kda, stream, steps: int = 100, warmup: int = 10):
    """kda_chunk_prefill_conv (SiLU) on the packed 8192-row workload at H = 32,
    against the same layer as two calls (kda_short_conv, then
    kda_chunk_prefill_slots): two rotating input sets, state and window pools
    of 2 x 16 entries with the calls alternating between their halves."""
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    n_heads = 32
    w_ = syn.workloads()[WORKLOAD]
    lengths = list(w_.lengths)
    rng = np.random.default_rng(83)
    t_rows = int(sum(lengths))
    n = len(lengths)
    sets = []
    for i in range(2):
        xs = [torch.from_numpy(rng.standard_normal((t_rows, n_heads, 128)).astype(np.float32)).to(torch.bfloat16).cuda()
              for _ in range(3)]
        g = torch.from_numpy((-0.2 * rng.random((t_rows, n_heads, 128))).astype(np.float32)).cuda()
        beta = torch.from_numpy(rng.random((t_rows, n_heads)).astype(np.float32)).cuda()
        out = torch.empty((t_rows, n_heads, 128), dtype=torch.bfloat16, device="cuda")
        qkv = tuple(torch.empty_like(xs[0]) for _ in range(3))
        sets.append((xs, g, beta, out, qkv))
    w = torch.from_numpy((0.5 * rng.standard_normal((3, n_heads * 128, 4))).astype(np.float32)).cuda()
    pool = torch.zeros((2 * n, 3, 3, n_heads * 128), dtype=torch.bfloat16, device="cuda")
    spool = torch.from_numpy((0.02 * rng.standard_normal((2 * n, n_heads, 128, 128))).astype(np.float32)).cuda()
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).cuda()
    tables = [torch.arange(0, n, dtype=torch.int32, device="cuda"), torch.arange(n, 2 * n, dtype=torch.int32, device="cuda")]

    def fused(i):
        xs, g, beta, out, _ = sets[i % 2]
        kda.chunk_prefill_conv(xs[0], xs[1], xs[2], w, g, beta, cu, pool, spool, slots=tables[(i // 2) % 2],
                               activation="silu", out=out, stream=stream)

    def two_calls(i):
        xs, g, beta, out, qkv = sets[i % 2]
        sl = tables[(i // 2) % 2]
        q, k, v = kda.short_conv(xs[0], xs[1], xs[2], w, cu, pool, conv_slots=sl, activation="silu", out=qkv,
                                 stream=stream)
        kda.chunk_prefill_slots(q, k, v, g, beta, cu, sl, spool, out=out, stream=stream)

    def timed(fn):
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(steps):
            fn(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / steps

    ms = timed(fused)
    ms2 = timed(two_calls)
    alg = conv_prefill_bytes(lengths, n_heads)
    peak, _ = peaks()
    achieved = alg / (ms / 1e3) / 1e9
    return {"workload": "conv_prefill_packed16_8192_h32", "kernel": "kda_tc_kernel (fused prologue)",
            "T": t_rows, "N": n, "H": n_heads, "activation": "silu", "steps": steps, "us_per_call": ms * 1e3,
            "tokens_per_s": t_rows / (ms / 1e3), "two_calls_us_per_step": ms2 * 1e3,
            "l2": "2 rotating input sets of 470 MB each",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "algorithmic_bytes_per_launch": alg,
                         "traffic": recorded_traffic("conv_prefill_packed16_8192_h32", KERNEL_SOURCES)}}


FOLD_W = 8   # speculative window: 8 draft tokens a sequence


def fold_bytes(accepted, h: int, w: int) -> int:
    """Algorithmic bytes of one fold: each (sequence, head) with accepted > 0 reads
    and writes its 64 KiB state and reads k, v (256 B each), g (512 B) and beta
    (4 B) of its accepted tokens; the accepted counts and slot table."""
    n = len(accepted)
    live = int((accepted > 0).sum())
    toks = int(accepted.sum())
    return live * h * 2 * 128 * 128 * 4 + toks * h * (2 * 256 + 512 + 4) + 8 * n


def measure_fold(torch, np, kda, stream, steps: int = 100, warmup: int = 10):
    """kda_fold_commit on DECODE_N sequences x DECODE_H heads with windows of
    FOLD_W tokens and seeded accepted counts in [0, FOLD_W]; the steps alternate
    between two slot tables over disjoint halves of the pool (above L2)."""
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    n, h, w = DECODE_N, DECODE_H, FOLD_W
    wl = syn.Workload("fold64_w8_h32", [w] * n, H=h, dk=128, dv=128, seed=78)
    x = syn.draw(wl)
    d = {}
    for k in ("k", "v", "g", "beta"):
        v = x[k]
        t = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16 else torch.from_numpy(v)
        d[k] = t.reshape((n, w) + tuple(t.shape[1:])).contiguous().cuda()
    rng = np.random.default_rng(78)
    accepted = rng.integers(0, w + 1, n).astype(np.int32)
    acc_t = torch.from_numpy(accepted).cuda()
    pool = torch.from_numpy((0.02 * rng.standard_normal((2 * n, h, 128, 128))).astype(np.float32)).cuda()
    perm = rng.permutation(2 * n).astype(np.int32)
    tables = [torch.from_numpy(np.sort(perm[:n])).cuda(), torch.from_numpy(np.sort(perm[n:])).cuda()]

    def step(i):
        kda.fold_commit(d["k"], d["v"], d["g"], d["beta"], acc_t, pool, state_slots=tables[i % 2], stream=stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    alg = fold_bytes(accepted, h, w)
    peak, _ = peaks()
    achieved = alg / (ms / 1e3) / 1e9
    return {"workload": "fold64_w8_h32", "kernel": "kda_fold_kernel", "N": n, "H": h, "window": w,
            "accepted_tokens": int(accepted.sum()), "steps": steps, "us_per_step": ms * 1e3,
            "l2": "2 slot tables over disjoint halves of a 2 x 64-entry pool (134 MB each)",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "algorithmic_bytes_per_launch": alg,
                         "traffic": recorded_traffic("fold64_w8_h32", DECODE_SOURCES)}}


def max_over_ranks(values, world: int, dist=None, device="cpu"):
    """Every rank's timings -> their maximum over the ranks (each rank gets it):
    the job takes as long as its slowest replica."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def replica_throughput(rows_per_replica: int, world: int, ms_per_step: float) -> float:
    """Whole-job rows/s: every replica processes its own copy of the workload."""
    return world * rows_per_replica / (ms_per_step / 1e3)


def config_bytes(w, rows: int, with_initial: bool) -> int:
    """Algorithmic bytes of one call over `rows` rows of workload w: per row-head
    q, k, v, out, g, beta (1540 B at bf16 d = 128; 1284 B at fp32 d = 64), plus
    the states read (if any) and written."""
    per_row_head = (w.dk + w.dk + w.dv + w.dv) * (2 if w.qkv_dtype == "bf16" else 4) + 4 * w.dk + 4
    n = 1 if w.calls > 1 else w.N
    return rows * w.H * per_row_head + n * w.H * w.dk * w.dv * 4 * (int(with_initial) + 1)


def tc_mode(w, rows: int, num_sms: int) -> str:
    """Which form of the tensor-core prefill a call of this workload runs
    (kda.h, "Split"): split for few units (N * H at most half the SMs) and
    T >= 1024 rows, with two chain CTAs a unit ("split-half") where N * H is
    at most a fifth of the SMs, unless KDA_SPLIT says otherwise; else the
    fused kernel."""
    if w.qkv_dtype != "bf16" or w.dk != 128 or w.dv != 128:
        return "cuda-core"
    n = 1 if w.calls > 1 else w.N
    env = os.environ.get("KDA_SPLIT", "")
    ok = 2 * n * w.H <= num_sms and n <= 256 and rows >= 1
    if env.startswith("0") or not ok:
        return "fused"
    if not (env.startswith("1") or env in ("full", "half") or rows >= 1024):
        return "fused"
    u = n * w.H
    half_ok = 4 * u <= num_sms
    if env == "full" or not half_ok:
        return "split"
    if env == "half" or 5 * u <= num_sms:
        return "split-half"
    return "split"


def measure_configs(torch, np, kda, stream, reps: int = 3, only=None, rows_override: int = 0):
    """The other four workloads, one line each: time per call (CUDA events, after
    one warm-up), tokens/s and the fraction of the HBM roofline.  The context of
    262,144 rows runs as its 32 chained calls of 8192 rows with the state carried;
    for timing, every call reads the same 8192-row input set (each call's inputs
    exceed L2, so nothing is served from a previous call).  `only` times one
    workload alone (profiler captures); rows_override then shortens a
    single-sequence workload to that many rows."""
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    peak, _ = peaks()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    res = {}
    for name, w in syn.workloads().items():
        if name == WORKLOAD or (only is not None and name != only):
            continue
        if rows_override and w.N == 1 and w.calls == 1:
            w = syn.Workload(f"{name[:name.rfind('_')]}_{rows_override}", [rows_override], H=w.H, dk=w.dk,
                             dv=w.dv, qkv_dtype=w.qkv_dtype, init_state=w.init_state, seed=w.seed)
        rows = w.T // w.calls
        x = syn.draw(w, 0, rows)
        dt = torch.bfloat16 if w.qkv_dtype == "bf16" else torch.float32
        d = {k: (torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16
                 else torch.from_numpy(v)).cuda() for k, v in x.items()}
        cu = torch.tensor(w.cu_seqlens() if w.calls == 1 else [0, rows], dtype=torch.int32, device="cuda")
        n = 1 if w.calls > 1 else w.N
        s0 = syn.draw_initial_state(w)
        s0 = torch.from_numpy(s0).cuda() if s0 is not None else None
        out = torch.empty((rows, w.H, w.dv), dtype=dt, device="cuda")
        fin = [torch.empty((n, w.H, w.dv, w.dk), dtype=torch.float32, device="cuda") for _ in range(2)]

        def run():
            state = s0
            for c in range(w.calls):
                kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, initial_state=state, out=out,
                                  final_state=fin[c % 2], stream=stream)
                state = fin[c % 2]

        def timed() -> float:
            run()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                run()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / (reps * w.calls)

        ms_call = timed()
        alg = sum(config_bytes(w, rows, with_initial=(s0 is not None) or c > 0) for c in range(w.calls)) / w.calls
        mode = tc_mode(w, rows, sms)
        res[w.name] = {"calls": w.calls, "rows_per_call": rows, "us_per_call": ms_call * 1e3,
                       "tokens_per_s": rows / (ms_call / 1e3),
                       "roofline_frac": alg / (ms_call / 1e3) / 1e9 / peak,
                       "units": n * w.H, "kernel": mode}
        if mode.startswith("split") and only is None:
            # the same calls on the fused kernel and in the other split form
            # where the SMs allow both, for comparison (KDA_SPLIT is read on
            # every call)
            old = os.environ.get("KDA_SPLIT")
            other = [("full_chain_us_per_call", "full")] if mode == "split-half" else (
                [("half_chain_us_per_call", "half")] if 4 * n * w.H <= sms else [])
            try:
                for key, env in [("fused_us_per_call", "0")] + other:
                    os.environ["KDA_SPLIT"] = env
                    res[w.name][key] = timed() * 1e3
            finally:
                if old is None:
                    os.environ.pop("KDA_SPLIT", None)
                else:
                    os.environ["KDA_SPLIT"] = old
        del d, out, fin, s0
        torch.cuda.empty_cache()
    return res


def run_gpu_arm(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import kda_linear_attention_chunk_gb300 as kda
    from kda_linear_attention_chunk_gb300 import synthetic as syn

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    w = syn.workloads()[WORKLOAD]
    sets = [make_device_inputs(w, i, torch, np) for i in range(2)]   # 2 rotating sets (> L2 each)
    stream = torch.cuda.current_stream()
    outs = [torch.empty((w.T, w.H, w.dv), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    fins = [torch.empty((w.N, w.H, w.dv, w.dk), dtype=torch.float32, device="cuda") for _ in range(2)]

    def step(i):
        d = sets[i % 2][1]
        kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], initial_state=d["s0"],
                          out=outs[i % 2], final_state=fins[i % 2], stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local)
    time.sleep(0.25)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    kernel_ms = ev0.elapsed_time(ev1) / args.steps

    # end to end through the public API: every step copies its inputs from pinned
    # host memory, runs the call and reads its results back to pinned host memory.
    # Steps are pipelined over three streams (inputs in, compute, results out)
    # with two device buffer sets, so one step's inputs travel in while the
    # previous step's results travel out (the host link carries both directions).
    host_out = [torch.empty((w.T, w.H, w.dv), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    host_fin = [torch.empty((w.N, w.H, w.dv, w.dk), dtype=torch.float32).pin_memory() for _ in range(2)]
    dev_in = [{k: torch.empty_like(v, device="cuda") for k, v in sets[0][0].items()} for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in sets[0][0].values())
    d2h = host_out[0].numel() * 2 + host_fin[0].numel() * 4
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]       # inputs of buffer b landed
    ev_k = [torch.cuda.Event() for _ in range(2)]        # call on buffer b done
    ev_out = [torch.cuda.Event() for _ in range(2)]      # results of buffer b read back

    def e2e_step(i):
        b = i % 2
        pin = sets[i % 2][0]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_k[b])                 # buffer b's previous call has read its inputs
            for k, v in pin.items():
                dev_in[b][k].copy_(v, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])                 # buffer b's previous results are read back
        kda.chunk_prefill(dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"], dev_in[b]["g"], dev_in[b]["beta"],
                          dev_in[b]["cu"], initial_state=dev_in[b]["s0"], out=outs[b], final_state=fins[b],
                          stream=stream)
        ev_k[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_k[b])
            host_out[b].copy_(outs[b], non_blocking=True)
            host_fin[b].copy_(fins[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 50))
    # device timing: the input stream starts after e0; e1 follows the last read-back
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(ev_out[(e2e_steps - 1) % 2])
    stream.wait_event(ev_out[e2e_steps % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    clocks = summarize_clocks(sampler.stop())
    decode = measure_decode(torch, np, kda, stream) if not args.no_decode else None
    fold = measure_fold(torch, np, kda, stream) if not args.no_decode else None
    conv = measure_conv(torch, np, kda, stream) if not args.no_decode else None
    conv_prefill = measure_conv_prefill(torch, np, kda, stream) if not args.no_decode else None
    decode_conv = measure_decode_conv(torch, np, kda, stream) if not args.no_decode else None
    configs = measure_configs(torch, np, kda, stream) if not args.no_configs else None
    assert kda.device_error() == 0, "device error word set during the bench"

    kernel_ms, e2e_ms = max_over_ranks([kernel_ms, e2e_ms], world, dist, device="cuda")
    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    value = replica_throughput(w.T, world, kernel_ms)
    alg = algorithmic_bytes(w)
    peak, peak_kind = peaks()
    achieved = alg / (kernel_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": kernel_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded splitmix64 inputs, workload shapes of the packed prefill)",
        "config": {"workload": WORKLOAD, "N": w.N, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "lengths": w.lengths, "initial_state": "N(0,0.02) fp32", "final_state": True,
                   "l2": "inputs larger than L2: 2 rotating input sets of %.0f MB" % (alg / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "e2e": {"value": replica_throughput(w.T, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(),
                     "kernel": KERNEL_NAME, "algorithmic_bytes_per_launch": alg,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "clocks": clocks,
    }
    if decode is not None:
        line["decode"] = decode
    if fold is not None:
        line["fold"] = fold
    if conv is not None:
        line["conv"] = conv
        line["conv_prefill"] = conv_prefill
    if decode_conv is not None:
        line["decode_conv"] = decode_conv
    if configs is not None:
        line["configs"] = configs
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, heads=args.cpu_heads)
    if world > 1:
        dist.destroy_process_group()
    return line


def cpu_baseline(w, heads: int, min_seconds: float = 10.0):
    """The oracle (fp64 token recurrence, plain C, all host cores) on a bounded
    sample of the same workload: all 8192 rows for `heads` of the H heads."""
    import oracle
    from kda_linear_attention_chunk_gb300 import synthetic as syn

    hs = list(range(heads))
    x = syn.draw(w, heads=hs)
    s0 = syn.draw_initial_state(w, heads=hs)
    cores = os.cpu_count() or 1
    oracle.load()
    reps, dt = 0, 0.0
    while reps < 1 or (dt < min_seconds and reps < 200):   # repeat the sample to about min_seconds
        t0 = time.perf_counter()
        oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], w.cu_seqlens(), initial_state=s0,
                   nthreads=cores)
        dt += time.perf_counter() - t0
        reps += 1
    return {"value": reps * w.T * (heads / w.H) / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "seconds": dt, "repeats": reps,
            "sample": f"all {w.T} rows of the {WORKLOAD} workload for {heads} of {w.H} heads, run {reps} "
                      f"times back to back; tokens/s counts a row as {heads}/{w.H} of a token"}


def run_reference_arm(args):
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    import oracle

    w = syn.workloads()[WORKLOAD]
    heads = args.ref_heads
    hs = list(range(heads))
    x = syn.draw(w, heads=hs)
    s0 = syn.draw_initial_state(w, heads=hs)
    cores = os.cpu_count() or 1
    oracle.load()
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], w.cu_seqlens(), initial_state=s0,
                   nthreads=cores)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = w.T * (heads / w.H) / (ms / 1e3)
    sample = (f"each step: all {w.T} rows of the {WORKLOAD} workload for {heads} of {w.H} heads; "
              f"tokens/s counts a row as {heads}/{w.H} of a token")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": w.N, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--cpu-heads", type=int, default=32)
    ap.add_argument("--ref-heads", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode-step, fold and short-conv measurements")
    ap.add_argument("--no-configs", action="store_true", help="skip the other four workloads")
    ap.add_argument("--profile-config", default=None,
                    help="time only this one of the other workloads (for profiler captures), nothing else")
    ap.add_argument("--profile-rows", type=int, default=0,
                    help="with --profile-config: a single-sequence workload shortened to this many rows")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_config:
        import numpy as np
        import torch
        import kda_linear_attention_chunk_gb300 as kda
        res = measure_configs(torch, np, kda, torch.cuda.current_stream(), reps=args.steps, only=args.profile_config,
                              rows_override=args.profile_rows)
        assert kda.device_error() == 0, "device error word set"
        print(json.dumps({"profile_config": res}), flush=True)
        return
    line = run_reference_arm(args) if args.impl == "reference" else run_gpu_arm(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
