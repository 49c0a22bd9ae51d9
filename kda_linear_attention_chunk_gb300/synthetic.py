"""Seeded synthetic inputs for the KDA chunked packed-varlen prefill.

This module only draws inputs.  It holds none of the method's arithmetic, so
both the CUDA path and the CPU oracle take their inputs from it.  The element
generator is the small C helper synthetic_gen.c (built here with gcc on first
use): a counter-based splitmix64 with Box-Muller normals, where every value is
a pure function of (seed, stream, flat index), so any row range or head
subset of a tensor can be drawn on its own and agrees with the full tensor.

Input recipe (the production packed prefill of the kern-k3-pp-prefill README,
section "P: the packed prefill": up to 16 sequences in an 8192-row chunk,
contexts to 262144, per-sequence states):

* q, k ~ N(0, 1), then L2-normalised over each head's dk channels;
* v ~ N(0, 1);
* g = log(alpha) ~ U[-0.2, 0] per token, head and channel;
* beta = sigmoid(N(0, 1)) per token and head;
* initial state ~ N(0, 0.02) (standard deviation) where the workload has one;
* q, k, v rounded to bf16 (round to nearest even) unless the workload is fp32;
* sequence lengths of the 16-sequence chunk: a seeded Dirichlet(1, ..., 1)
  split of 8192 rows, each at least 1.

Values are computed in double precision with the C library's log/cos/exp, so
the bits are reproducible on one machine (where both arms run) and agree
almost always across machines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synthetic_gen.c")
_LIB = os.path.join(_HERE, "_build", "libsynth.so")

KIND_Q, KIND_K, KIND_V, KIND_G, KIND_BETA, KIND_STATE = range(6)
STREAM_LENS = 7
STREAM_PROFILE = 11   # uniforms that pick the entries a decay profile changes
_gen = None


def build_generator() -> str:
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"],
                   check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _gen
    if _gen is None:
        if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            build_generator()
        lib = ctypes.CDLL(_LIB)
        lib.syn_fill.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
        lib.syn_fill.restype = ctypes.c_int
        lib.syn_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]
        lib.syn_uniform.restype = ctypes.c_int
        _gen = lib
    return _gen


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _lib().syn_uniform(seed, stream, n, out.ctypes.data)
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bit pattern (uint16), round to nearest even via fp32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    b = f.view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b).astype(np.uint32) << np.uint32(16)).view(np.float32)


def dirichlet_lengths(total: int, parts: int, seed: int) -> List[int]:
    """Split ``total`` rows into ``parts`` lengths, each >= 1, by a seeded
    Dirichlet(1, ..., 1) draw (normalised exponentials).  Each part gets
    1 + floor(p_i * (total - parts)); the rows left over go one each to the
    largest fractional remainders (ties to the lower index)."""
    e = -np.log(uniform(seed, STREAM_LENS, parts))
    p = e / e.sum()
    share = p * (total - parts)
    base = np.floor(share).astype(np.int64)
    left = total - parts - int(base.sum())
    order = sorted(range(parts), key=lambda i: (-(share[i] - base[i]), i))
    for i in order[:left]:
        base[i] += 1
    lens = [int(1 + b) for b in base]
    assert sum(lens) == total and min(lens) >= 1
    return lens


@dataclass
class Workload:
    """One synthetic workload: packed sequence lengths plus tensor shapes."""

    name: str
    lengths: List[int]
    H: int
    dk: int
    dv: int
    qkv_dtype: str = "bf16"          # "bf16" or "f32"
    init_state: bool = False          # N(0, 0.02) initial states if True
    calls: int = 1                    # >1: the rows are split into equal calls
    seed: int = 0
    note: str = ""

    @property
    def N(self) -> int:
        return len(self.lengths)

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)


def workloads() -> Dict[str, Workload]:
    """The five workloads: tiny fp32, 4-sequence varlen, the 8192-row
    production packed chunk, one 65536-row sequence and a 262144-row context
    carried across 32 calls of 8192 rows."""
    return {
        "tiny_fp32_256": Workload("tiny_fp32_256", [256], H=2, dk=64, dv=64, qkv_dtype="f32",
                                  note="1 x 256 rows, H=2, d=64, fp32 q/k/v, zero initial state"),
        "varlen4_4096": Workload("varlen4_4096", [1000, 513, 64, 2519], H=16, dk=128, dv=128,
                                 init_state=True,
                                 note="lengths [1000,513,64,2519], H=16, d=128, bf16, N(0,0.02) states"),
        "packed16_8192": Workload("packed16_8192", dirichlet_lengths(8192, 16, 0), H=32, dk=128,
                                  dv=128, init_state=True,
                                  note="16 Dirichlet(1) lengths summing to 8192, H=32, d=128, bf16, "
                                       "N(0,0.02) states"),
        "long_65536": Workload("long_65536", [65536], H=32, dk=128, dv=128,
                               note="1 x 65536 rows, H=32, d=128, bf16, zero initial state"),
        "context_262144": Workload("context_262144", [262144], H=32, dk=128, dv=128, calls=32,
                                   note="1 x 262144 rows as 32 calls of 8192 rows, state carried"),
    }


def _heads(w: Workload, heads: Optional[Sequence[int]]) -> np.ndarray:
    return np.arange(w.H, dtype=np.int32) if heads is None else np.asarray(list(heads), dtype=np.int32)


def _fill(kind, w, row_lo, nrows, hs, d, shape, dtype, out_code):
    out = np.empty(shape, dtype=dtype)
    rc = _lib().syn_fill(kind, w.seed, row_lo, nrows, hs.ctypes.data, len(hs), w.H, d,
                         out.ctypes.data, out_code, _threads())
    if rc != 0:
        raise ValueError("synthetic generator rejected its arguments")
    return out


def draw(w: Workload, row_lo: int = 0, row_hi: Optional[int] = None,
         heads: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Draw rows [row_lo, row_hi) of the workload for the listed heads.

    Returns q, k, v as uint16 bf16 bits (or float32 for fp32 workloads), each
    [rows][nh][d]; g float32 [rows][nh][dk]; beta float32 [rows][nh].  The
    values are those of the full [T][H][d] tensors at those positions."""
    if row_hi is None:
        row_hi = w.T
    hs = _heads(w, heads)
    n = row_hi - row_lo
    bf = w.qkv_dtype == "bf16"
    dt, code = (np.uint16, 0) if bf else (np.float32, 1)
    return {
        "q": _fill(KIND_Q, w, row_lo, n, hs, w.dk, (n, len(hs), w.dk), dt, code),
        "k": _fill(KIND_K, w, row_lo, n, hs, w.dk, (n, len(hs), w.dk), dt, code),
        "v": _fill(KIND_V, w, row_lo, n, hs, w.dv, (n, len(hs), w.dv), dt, code),
        "g": _fill(KIND_G, w, row_lo, n, hs, w.dk, (n, len(hs), w.dk), np.float32, 1),
        "beta": _fill(KIND_BETA, w, row_lo, n, hs, 1, (n, len(hs)), np.float32, 1),
    }


def draw_initial_state(w: Workload, heads: Optional[Sequence[int]] = None) -> Optional[np.ndarray]:
    """[N][nh][dv][dk] float32 initial states, or None for a zero start.  With
    dk != dv the state is the [dv][dk] corner of the d x d draw, d = max."""
    if not w.init_state:
        return None
    hs = _heads(w, heads)
    d = max(w.dk, w.dv)
    s = _fill(KIND_STATE, w, 0, w.N, hs, d, (w.N, len(hs), d, d), np.float32, 1)
    return np.ascontiguousarray(s[:, :, :w.dv, :w.dk])


DECAY_PROFILES = ("u02", "u05", "u1", "u3", "alpha0", "mixed")


def decay_profile(g: np.ndarray, profile: str, seed: int = 0) -> np.ndarray:
    """Another gate distribution from g as drawn (U[-0.2, 0], [T][H][dk]), for
    tests of the decay range; a copy, float32:

    * u02: unchanged;  u05, u1, u3: U[-a, 0] for a = 0.5, 1, 3 (g scaled);
    * alpha0: about 3% of the (head, channel) pairs held at g = -20 on every
      row (alpha = e^-20, a channel that forgets at once), the rest unchanged;
    * mixed: about 5% of the entries replaced by U[0, 0.5] (a growing gate),
      the rest unchanged.

    The entries are picked by seeded uniforms over the whole tensor."""
    g = np.array(g, dtype=np.float32)
    T, H, dk = g.shape
    if profile == "u02":
        return g
    if profile in ("u05", "u1", "u3"):
        a = {"u05": 0.5, "u1": 1.0, "u3": 3.0}[profile]
        return (g * np.float32(a / 0.2)).astype(np.float32)
    if profile == "alpha0":
        pick = uniform(seed, STREAM_PROFILE, H * dk).reshape(H, dk) < 0.03
        g[:, pick] = -20.0
        return g
    if profile == "mixed":
        u = uniform(seed, STREAM_PROFILE + 1, T * H * dk).reshape(T, H, dk)
        pos = u < 0.05
        g[pos] = (u[pos] * (0.5 / 0.05)).astype(np.float32)
        return g
    raise ValueError(f"unknown decay profile {profile!r}")


def random_lengths(total: int, parts: int, seed: int, allow_empty: bool = False) -> List[int]:
    """Seeded ragged lengths for edge-case tests (zeros allowed if asked)."""
    if parts == 1:
        return [total]
    u = uniform(seed, STREAM_LENS + 100, parts - 1)
    cuts = np.sort((u * (total + 1)).astype(np.int64).clip(0, total))
    lens = [int(x) for x in np.diff(np.concatenate([[0], cuts, [total]]))]
    if not allow_empty:
        lens = [max(1, x) for x in lens]
        lens[int(np.argmax(lens))] -= sum(lens) - total
    return lens
