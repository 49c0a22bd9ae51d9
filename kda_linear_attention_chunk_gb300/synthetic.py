"""Seeded synthetic inputs for the KDA chunked packed-varlen prefill.

This module only draws inputs.  It holds none of the method's arithmetic, so
both the CUDA path and the CPU oracle can take their inputs from it.

Generator: a counter-based splitmix64.  Element ``i`` of stream ``s`` under
seed ``seed`` is ``mix64(mix64(seed) + s * 2**48 + i)``, where ``mix64`` is the
splitmix64 output function (add the golden-ratio increment, then the two
xor-shift-multiply rounds and a final xor-shift).  Because every element is a
pure function of its flat index, any row range or head subset of a tensor can
be drawn on its own and agrees with the full tensor.  Normal deviates use the
Box-Muller transform on the uniforms of indices ``2i`` and ``2i + 1``.

Input recipe (the production packed prefill of the kern-k3-pp-prefill README,
section "P: the packed prefill": up to 16 sequences in an 8192-row chunk,
contexts to 262144, per-sequence states):

* q, k ~ N(0, 1), then L2-normalised over each head's dk channels;
* v ~ N(0, 1);
* g = log(alpha) ~ U[-0.2, 0] per token, head and channel;
* beta = sigmoid(N(0, 1)) per token and head;
* initial state ~ N(0, 0.02) (standard deviation) where the workload has one;
* q, k, v rounded to bf16 (round to nearest even) unless the workload is fp32.

The random values are computed in float64; numpy's elementwise log/cos/exp
may differ in the last ulp between machines, so the bits are reproducible on
one machine (where both arms run) and agree almost always across machines.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

STREAM_Q, STREAM_K, STREAM_V, STREAM_G, STREAM_BETA, STREAM_INIT, STREAM_LENS = 1, 2, 3, 4, 5, 6, 7


def _mix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, stream: int, index: np.ndarray) -> np.ndarray:
    key = _mix64(np.array([seed], dtype=np.uint64))[0]
    with np.errstate(over="ignore"):
        ctr = key + np.uint64(stream) * np.uint64(1 << 48) + index.astype(np.uint64)
    return _mix64(ctr)


def uniform(seed: int, stream: int, index: np.ndarray) -> np.ndarray:
    """Uniform deviates in the open interval (0, 1), float64."""
    bits = raw_u64(seed, stream, index) >> np.uint64(11)
    return (bits.astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, index: np.ndarray) -> np.ndarray:
    """Standard normal deviates (Box-Muller, cosine branch), float64."""
    idx = index.astype(np.uint64) * np.uint64(2)
    u1 = uniform(seed, stream, idx)
    u2 = uniform(seed, stream, idx + np.uint64(1))
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bit pattern (uint16), round to nearest even via fp32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    b = f.view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def dirichlet_lengths(total: int, parts: int, seed: int) -> List[int]:
    """Split ``total`` rows into ``parts`` lengths, each >= 1, by a seeded
    Dirichlet(1, ..., 1) draw (normalised exponentials).  Each part gets
    1 + floor(p_i * (total - parts)); the rows left over go one each to the
    largest fractional remainders (ties to the lower index)."""
    e = -np.log(uniform(seed, STREAM_LENS, np.arange(parts, dtype=np.uint64)))
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


def _flat_index(rows: np.ndarray, heads: np.ndarray, H: int, d: int) -> np.ndarray:
    r = rows.astype(np.uint64)[:, None, None]
    h = heads.astype(np.uint64)[None, :, None]
    c = np.arange(d, dtype=np.uint64)[None, None, :]
    return (r * np.uint64(H) + h) * np.uint64(d) + c


def draw(w: Workload, row_lo: int = 0, row_hi: Optional[int] = None,
         heads: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Draw rows [row_lo, row_hi) of the workload for the listed heads.

    Returns q, k, v as uint16 bf16 bits (or float32 for fp32 workloads), each
    [rows][nh][d]; g float32 [rows][nh][dk]; beta float32 [rows][nh].  The
    values are those of the full [T][H][d] tensors at those positions."""
    if row_hi is None:
        row_hi = w.T
    hs = np.arange(w.H) if heads is None else np.asarray(list(heads), dtype=np.int64)
    rows = np.arange(row_lo, row_hi, dtype=np.int64)
    out: Dict[str, np.ndarray] = {}
    for name, stream, d in (("q", STREAM_Q, w.dk), ("k", STREAM_K, w.dk), ("v", STREAM_V, w.dv)):
        x = normal(w.seed, stream, _flat_index(rows, hs, w.H, d))
        if name in ("q", "k"):
            x = x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
        out[name] = to_bf16_bits(x) if w.qkv_dtype == "bf16" else x.astype(np.float32)
    u = uniform(w.seed, STREAM_G, _flat_index(rows, hs, w.H, w.dk))
    out["g"] = (-0.2 * u).astype(np.float32)
    bidx = (rows.astype(np.uint64)[:, None] * np.uint64(w.H) + hs.astype(np.uint64)[None, :])
    out["beta"] = (1.0 / (1.0 + np.exp(-normal(w.seed, STREAM_BETA, bidx)))).astype(np.float32)
    return out


def draw_initial_state(w: Workload, heads: Optional[Sequence[int]] = None) -> Optional[np.ndarray]:
    """[N][nh][dv][dk] float32 initial states, or None for a zero start."""
    if not w.init_state:
        return None
    hs = np.arange(w.H) if heads is None else np.asarray(list(heads), dtype=np.int64)
    n = np.arange(w.N, dtype=np.uint64)[:, None, None, None]
    h = hs.astype(np.uint64)[None, :, None, None]
    v = np.arange(w.dv, dtype=np.uint64)[None, None, :, None]
    c = np.arange(w.dk, dtype=np.uint64)[None, None, None, :]
    idx = ((n * np.uint64(w.H) + h) * np.uint64(w.dv) + v) * np.uint64(w.dk) + c
    return (0.02 * normal(w.seed, STREAM_INIT, idx)).astype(np.float32)


def random_lengths(total: int, parts: int, seed: int, allow_empty: bool = False) -> List[int]:
    """Seeded ragged lengths for edge-case tests (may include zeros)."""
    if parts == 1:
        return [total]
    u = uniform(seed, STREAM_LENS + 100, np.arange(parts - 1, dtype=np.uint64))
    cuts = np.sort((u * (total + 1)).astype(np.int64).clip(0, total))
    edges = np.concatenate([[0], cuts, [total]])
    lens = [int(x) for x in np.diff(edges)]
    if not allow_empty:
        lens = [max(1, x) for x in lens]
        diff = sum(lens) - total
        i = int(np.argmax(lens))
        lens[i] -= diff
    return lens
