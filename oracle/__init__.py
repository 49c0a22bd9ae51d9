"""ctypes loader for the fp64 CPU oracle (oracle/kda_oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and the
cpu_baseline leg of bench.py are the only users.  The CUDA library never
imports, links or calls anything here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

BF16, F32, F64 = 0, 1, 2
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags: Sequence[str] = ()) -> str:
    """Compile the oracle with gcc (plain C11, -O2, POSIX threads)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread",
           *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale(lib: str, src: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


def load(path: Optional[str] = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if _stale(_LIB, _SRC):
            build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.kda_oracle_recurrent.argtypes = [P, P, P, I, P, P, I, P, P, P, P,
                                         I, I, I, I, I, P, I, I]
    lib.kda_oracle_recurrent.restype = I
    lib.kda_oracle_chunked.argtypes = [P, P, P, I, P, P, I, P, P, P, P,
                                       I, I, I, I, I, P, I, I, I]
    lib.kda_oracle_chunked.restype = I
    return lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported oracle input dtype {a.dtype}")


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def run(q, k, v, g, beta, cu_seqlens, initial_state=None, heads=None, chunk: int = 0,
        nthreads: Optional[int] = None, lib=None, want_state: bool = True
        ) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """Run the oracle.

    q, k: [T][H][dk]; v: [T][H][dv] (uint16 bf16 bits, float32 or float64);
    g: [T][H][dk], beta: [T][H] (float32 or float64, same dtype);
    cu_seqlens: [N+1] int; initial_state: None or [N][nsel][dv][dk] (float);
    heads: indices of the heads to compute (default: all).
    chunk = 0 runs the token recurrence, chunk >= 1 the chunked form.
    Returns out [T][nsel][dv] float64 and final_state [N][nsel][dv][dk] float64.
    """
    lib = lib or load()
    q, k, v = (np.ascontiguousarray(x) for x in (q, k, v))
    g, beta = np.ascontiguousarray(g), np.ascontiguousarray(beta)
    if g.dtype != beta.dtype:
        beta = beta.astype(g.dtype)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu.shape[0] - 1
    hs = np.arange(H, dtype=np.int32) if heads is None else np.ascontiguousarray(heads, dtype=np.int32)
    nsel = hs.shape[0]
    init = None if initial_state is None else np.ascontiguousarray(initial_state, dtype=np.float64)
    if init is not None:
        assert init.shape == (N, nsel, dv, dk), init.shape
    out = np.zeros((T, nsel, dv), dtype=np.float64)
    fin = np.zeros((N, nsel, dv, dk), dtype=np.float64) if want_state else None
    nt = nthreads or os.cpu_count() or 1
    args = [_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(g), _ptr(beta), _dtype_code(g),
            _ptr(cu), _ptr(init), _ptr(out), _ptr(fin), N, T, H, dk, dv, _ptr(hs), nsel]
    if chunk == 0:
        rc = lib.kda_oracle_recurrent(*args, nt)
    else:
        rc = lib.kda_oracle_chunked(*args, chunk, nt)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out, fin


def run_slots(q, k, v, g, beta, cu_seqlens, state_slots, state_pool, out=None, heads=None,
              chunk: int = 0, nthreads: Optional[int] = None, lib=None):
    """Slot-indexed states (kern-k3-pp-prefill README, section "D inside
    SGLang": a KDA layer's recurrent state sits in a pool laid out
    [slot][head][v][k] f32, reached through a table of slot ids, and padded
    entries carry slot -1, which the kernel skips).

    Sequence n starts from state_pool[state_slots[n]] and its final state
    replaces that entry.  A sequence whose slot id is -1 is padding: nothing
    of it is computed, its rows of `out` keep what they held and the pool is
    not touched.  An id outside [-1, num_slots) is handled like -1 and
    reported.  Valid ids must be distinct (two sequences cannot own one
    state).

    Inputs as run(); state_slots: [N] int; state_pool: [num_slots][nsel][dv][dk];
    out: [T][nsel][dv] values kept in the skipped rows (default NaN).
    Returns (out [T][nsel][dv], pool [num_slots][nsel][dv][dk], both float64,
    and the list of sequence indices whose id was out of range).
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    slots = np.asarray(state_slots, dtype=np.int64)
    pool = np.array(state_pool, dtype=np.float64)          # a copy: updated below
    num_slots = pool.shape[0]
    N = cu.shape[0] - 1
    assert slots.shape == (N,), slots.shape
    T = q.shape[0]
    nsel = pool.shape[1]
    dv = v.shape[2]
    res = (np.full((T, nsel, dv), np.nan) if out is None else np.array(out, dtype=np.float64))
    bad = [n for n in range(N) if slots[n] < -1 or slots[n] >= num_slots]
    live = [n for n in range(N) if 0 <= slots[n] < num_slots]
    if len(set(int(slots[n]) for n in live)) != len(live):
        raise ValueError("two sequences name the same state slot")
    if not live:
        return res, pool, bad
    # The live sequences, packed back to back, form one ordinary call whose
    # initial states are gathered from the pool.
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in live]).astype(np.int64)
    lens = [int(cu[n + 1] - cu[n]) for n in live]
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sub_out, fin = run(q[rows], k[rows], v[rows], g[rows], beta[rows], sub_cu,
                       initial_state=pool[slots[live]], heads=heads, chunk=chunk,
                       nthreads=nthreads, lib=lib)
    res[rows] = sub_out
    pool[slots[live]] = fin
    return res, pool, bad


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the exact float64 values they encode."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def short_conv(xq, xk, xv, conv_weight, cu_seqlens, conv_pool, conv_slots=None, activation: str = "silu",
               eps: float = 1e-6):
    """The short-conv + L2-norm prologue of a KDA layer (kern-k3-pp-prefill
    README: section "P: the packed prefill" runs the KDA layers with
    per-sequence conv windows and states; section "D inside SGLang" keeps the
    window in the engine's pool laid out [slot][tap][q | k | v] bf16, indexed
    by the same slot ids as the state).

    The pages fix the window layout only.  Readings: the window carries the
    three rows before a sequence's first row, so the causal conv has four
    taps; the weights [3][H*D][4] (tap 3 weighs the row itself) and the
    activation (none or SiLU) are the caller's; q and k are scaled to unit L2
    norm per head, y / sqrt(|y|^2 + eps); v is not.

    For sequence n with window entry s = conv_slots[n] (n if None), rows
    t = 0 .. L-1 and each stream (q, k, v), in this order:
      1. the input sequence is [taps 0, 1, 2 of the entry ; its L rows];
      2. y_t = sum_j w[j] * input[t + j] over j = 0 .. 3, channel by channel;
      3. the activation;
      4. for q and k, the per-head L2 normalisation;
      5. the entry's taps become the last three rows of that input sequence.
    A sequence whose id is -1 is padding: nothing of it is computed or written.
    An id outside [-1, num_slots) is handled like -1 and reported.

    xq, xk, xv: uint16 bf16 bits [T][H][D]; conv_weight: float [3][H*D][4];
    conv_pool: uint16 bf16 bits [num_slots][3][3][H*D].
    Returns (q, k, v) float64 [T][H][D] (NaN in rows not computed), the new
    pool (uint16 bits) and the list of sequence indices whose id was out of
    range.
    """
    xs = [np.asarray(a, dtype=np.uint16) for a in (xq, xk, xv)]
    T, H, D = xs[0].shape
    C = H * D
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    w = np.asarray(conv_weight, dtype=np.float64).reshape(3, C, 4)
    pool = np.array(conv_pool, dtype=np.uint16)             # a copy: updated below
    num_slots = pool.shape[0]
    assert pool.shape == (num_slots, 3, 3, C), pool.shape
    slots = np.arange(N) if conv_slots is None else np.asarray(conv_slots, dtype=np.int64)
    outs = [np.full((T, C), np.nan) for _ in range(3)]
    bad = [n for n in range(N) if slots[n] < -1 or slots[n] >= num_slots]
    for n in range(N):
        slot = int(slots[n])
        if not 0 <= slot < num_slots:
            continue
        b, e = int(cu[n]), int(cu[n + 1])
        L = e - b
        if L <= 0:
            continue
        for s in range(3):
            seq_bits = np.concatenate([pool[slot, :, s, :], xs[s].reshape(T, C)[b:e]], axis=0)   # [3 + L][C]
            seq = bf16_bits_to_f64(seq_bits)
            y = sum(w[s, :, j] * seq[j:j + L] for j in range(4))                              # [L][C]
            if activation == "silu":
                y = y / (1.0 + np.exp(-y))
            elif activation != "none":
                raise ValueError(activation)
            if s < 2:
                yh = y.reshape(L, H, D)
                y = (yh / np.sqrt((yh * yh).sum(axis=2, keepdims=True) + eps)).reshape(L, C)
            outs[s][b:e] = y
            pool[slot, :, s, :] = seq_bits[L:L + 3]
    return tuple(o.reshape(T, H, D) for o in outs), pool, bad
