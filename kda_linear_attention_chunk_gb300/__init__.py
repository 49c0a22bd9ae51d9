"""Python binding of libkda.so, the GB300 KDA chunked packed-varlen prefill.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI of include/kda.h.  PyTorch supplies device memory
and streams.  There is no fallback: if the library is not built, the entry
points raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")

KDA_OK, KDA_ERR_NULL, KDA_ERR_SHAPE, KDA_ERR_UNSUPPORTED = 0, 1, 2, 3
KDA_ERR_ALIGN, KDA_ERR_ALIAS, KDA_ERR_CUDA, KDA_ERR_DEVICE = 4, 5, 6, 7
KDA_ERR_NOALLOC_LIMIT = 8
KDA_NOALLOC_MAX_SEQS = 16384

EXPORTED = ("kda_chunk_prefill", "kda_chunk_prefill_f32", "kda_chunk_prefill_fullrange", "kda_status_string",
            "kda_device_error", "kda_chunk_prefill_noalloc", "kda_chunk_prefill_slots", "kda_chunk_prefill_conv",
            "kda_decode", "kda_fold_commit", "kda_short_conv", "kda_decode_conv")
# device error word bits (kda_device_error)
ERR_WAIT_TIMEOUT = 1    # a bounded wait ran out; the kernel wound down early
ERR_BAD_SEQLENS = 2     # a cu_seqlens entry broke its contract (clamped)
ERR_BAD_SLOT = 8        # a state slot id outside [-1, num_slots)
ERR_BAD_ACCEPTED = 16   # an accepted count outside [0, window]
ERR_DECAY_RANGE = 32    # the tensor-core prefill met a decay beyond its fp16 operand range

_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}" if where else status_string(status))


def load(path: str = LIB_PATH):
    """Load libkda.so (built by __graft_entry__.build()); raises if missing."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkda.so is not built ({path}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    sig = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, P]
    for name in ("kda_chunk_prefill", "kda_chunk_prefill_f32", "kda_chunk_prefill_fullrange",
                 "kda_chunk_prefill_noalloc"):
        fn = getattr(lib, name)
        fn.argtypes = sig
        fn.restype = I
    lib.kda_chunk_prefill_slots.argtypes = [P, P, P, P, P, P, P, P, I, P, I, I, I, I, I, P]
    lib.kda_chunk_prefill_slots.restype = I
    lib.kda_chunk_prefill_conv.argtypes = [P, P, P, P, P, P, P, P, P, I, P, I, P, I, I, I, I, I, I,
                                           ctypes.c_float, P]
    lib.kda_chunk_prefill_conv.restype = I
    lib.kda_decode.argtypes = [P, P, P, P, P, P, P, I, P, I, I, I, I, P]
    lib.kda_decode.restype = I
    lib.kda_fold_commit.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P]
    lib.kda_fold_commit.restype = I
    lib.kda_short_conv.argtypes = [P, P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, ctypes.c_float, P]
    lib.kda_short_conv.restype = I
    lib.kda_decode_conv.argtypes = [P, P, P, P, P, P, I, P, P, P, P, I, P, I, I, I, I, I, ctypes.c_float, P]
    lib.kda_decode_conv.restype = I
    lib.kda_status_string.argtypes = [I]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_device_error.argtypes = [ctypes.POINTER(ctypes.c_int), I]
    lib.kda_device_error.restype = I
    if path == LIB_PATH:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().kda_status_string(int(status)).decode()
    except RuntimeError:
        return f"kda_status {status}"


def kda_chunk_prefill(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                      N: int, T: int, H: int, dk: int, dv: int, stream) -> int:
    """Raw C-ABI call: integer device pointers (0 = NULL) and sizes."""
    return load().kda_chunk_prefill(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                                    N, T, H, dk, dv, stream)


def kda_chunk_prefill_f32(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                          N: int, T: int, H: int, dk: int, dv: int, stream) -> int:
    """Raw C-ABI call for fp32 q/k/v/out."""
    return load().kda_chunk_prefill_f32(q, k, v, g, beta, cu_seqlens, initial_state, out,
                                        final_state, N, T, H, dk, dv, stream)


def kda_chunk_prefill_fullrange(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                                N: int, T: int, H: int, dk: int, dv: int, stream) -> int:
    """Raw C-ABI call of the bf16 prefill on the CUDA-core kernel, which takes
    any decay (no fp16 operand range)."""
    return load().kda_chunk_prefill_fullrange(q, k, v, g, beta, cu_seqlens, initial_state, out,
                                              final_state, N, T, H, dk, dv, stream)


def kda_chunk_prefill_noalloc(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                              N: int, T: int, H: int, dk: int, dv: int, stream) -> int:
    """Raw C-ABI call of the entry point that allocates nothing (up to
    KDA_NOALLOC_MAX_SEQS sequences; its scheduling table lives inside the
    library, for callers that cannot allocate device memory per call)."""
    return load().kda_chunk_prefill_noalloc(q, k, v, g, beta, cu_seqlens, initial_state, out,
                                            final_state, N, T, H, dk, dv, stream)


def kda_chunk_prefill_slots(q, k, v, g, beta, cu_seqlens, state_slots, state_pool, num_slots: int, out,
                            N: int, T: int, H: int, dk: int, dv: int, stream) -> int:
    """Raw C-ABI call with the states in a slot-addressed pool."""
    return load().kda_chunk_prefill_slots(q, k, v, g, beta, cu_seqlens, state_slots, state_pool,
                                          num_slots, out, N, T, H, dk, dv, stream)


def kda_chunk_prefill_conv(xq, xk, xv, conv_weight, g, beta, cu_seqlens, slots, conv_pool, conv_num_slots: int,
                           state_pool, num_slots: int, out, N: int, T: int, H: int, dk: int, dv: int,
                           activation: int, eps: float, stream) -> int:
    """Raw C-ABI call: the short-conv prologue fused into the prefill."""
    return load().kda_chunk_prefill_conv(xq, xk, xv, conv_weight, g, beta, cu_seqlens, slots, conv_pool,
                                         conv_num_slots, state_pool, num_slots, out, N, T, H, dk, dv, activation,
                                         eps, stream)


def kda_decode(q, k, v, g, beta, state_slots, state_pool, num_slots: int, out, N: int, H: int, dk: int, dv: int,
               stream) -> int:
    """Raw C-ABI call: one recurrence step per sequence on a slot-addressed pool."""
    return load().kda_decode(q, k, v, g, beta, state_slots, state_pool, num_slots, out, N, H, dk, dv, stream)


def kda_fold_commit(k, v, g, beta, accepted, state_slots, state_pool, num_slots: int, N: int, W: int, H: int,
                    dk: int, dv: int, stream) -> int:
    """Raw C-ABI call: fold the accepted tokens of each window into the pool."""
    return load().kda_fold_commit(k, v, g, beta, accepted, state_slots, state_pool, num_slots, N, W, H, dk, dv,
                                  stream)


def kda_short_conv(xq, xk, xv, conv_weight, cu_seqlens, conv_slots, conv_pool, num_slots: int, q_out, k_out,
                   v_out, N: int, T: int, H: int, d: int, activation: int, eps: float, stream) -> int:
    """Raw C-ABI call: short conv + L2 norm prologue, conv windows in a slot-addressed pool."""
    return load().kda_short_conv(xq, xk, xv, conv_weight, cu_seqlens, conv_slots, conv_pool, num_slots, q_out,
                                 k_out, v_out, N, T, H, d, activation, eps, stream)


def kda_decode_conv(xq, xk, xv, conv_weight, conv_slots, conv_pool, conv_num_slots: int, g, beta, state_slots,
                    state_pool, num_slots: int, out, N: int, H: int, dk: int, dv: int, activation: int, eps: float,
                    stream) -> int:
    """Raw C-ABI call: the decode step with the short conv fused in front of it."""
    return load().kda_decode_conv(xq, xk, xv, conv_weight, conv_slots, conv_pool, conv_num_slots, g, beta,
                                  state_slots, state_pool, num_slots, out, N, H, dk, dv, activation, eps, stream)


def device_error(reset: bool = False) -> int:
    word = ctypes.c_int(0)
    st = load().kda_device_error(ctypes.byref(word), int(reset))
    if st != KDA_OK:
        raise KdaError(st, "kda_device_error")
    return word.value


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def chunk_prefill(q, k, v, g, beta, cu_seqlens, initial_state=None, out=None, final_state=None,
                  output_final_state: bool = True, stream=None,
                  full_range: bool = False) -> Tuple[object, Optional[object]]:
    """KDA chunked packed-varlen prefill on torch CUDA tensors.

    q, k: [T][H][dk], v: [T][H][dv] (bfloat16 or float32; dk, dv in {64, 128});
    g: [T][H][dk] float32; beta: [T][H] float32; cu_seqlens: [N+1] int32 on
    the device; initial_state: [N][H][dv][dk] float32 or None.  Returns
    (out [T][H][dv] in q's dtype, final_state [N][H][dv][dk] float32 or None).
    Runs asynchronously on ``stream`` (default: torch's current stream).
    ``full_range`` (bfloat16 only) selects kda_chunk_prefill_fullrange, for
    decays beyond the tensor-core kernel's range (ERR_DECAY_RANGE).
    """
    import torch

    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.shape[0] - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("cu_seqlens", cu_seqlens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    handle = int(s.cuda_stream) if hasattr(s, "cuda_stream") else int(s)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), _ptr(initial_state),
            _ptr(out), _ptr(final_state), N, T, H, dk, dv, handle)
    if q.dtype == torch.bfloat16:
        st = kda_chunk_prefill_fullrange(*args) if full_range else kda_chunk_prefill(*args)
    elif q.dtype == torch.float32:
        st = kda_chunk_prefill_f32(*args)
    else:
        raise ValueError(f"unsupported q dtype {q.dtype}")
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_prefill")
    return out, final_state


def chunk_prefill_slots(q, k, v, g, beta, cu_seqlens, state_slots, state_pool, out=None, stream=None):
    """KDA prefill with slot-addressed states, on torch CUDA tensors.

    q, k, v: [T][H][128] bfloat16; g: [T][H][128] float32; beta: [T][H]
    float32; cu_seqlens: [N+1] int32 and state_slots: [N] int32 on the device
    (-1 = padded sequence, skipped); state_pool: [num_slots][H][128][128]
    float32, read and updated in place.  Returns out [T][H][128] bfloat16
    (rows of padded sequences keep what ``out`` held; a fresh ``out`` is
    uninitialised there).  Runs asynchronously on ``stream``.
    """
    import torch

    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.shape[0] - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("cu_seqlens", cu_seqlens),
                    ("state_slots", state_slots), ("state_pool", state_pool)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if q.dtype != torch.bfloat16:
        raise ValueError("chunk_prefill_slots takes bfloat16 q/k/v")
    if state_slots.dtype != torch.int32 or tuple(state_slots.shape) != (N,):
        raise ValueError("state_slots must be int32 [N]")
    if state_pool.dtype != torch.float32 or tuple(state_pool.shape[1:]) != (H, dv, dk):
        raise ValueError("state_pool must be float32 [num_slots][H][dv][dk]")
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    handle = int(s.cuda_stream) if hasattr(s, "cuda_stream") else int(s)
    st = kda_chunk_prefill_slots(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                 _ptr(state_slots), _ptr(state_pool), int(state_pool.shape[0]), _ptr(out),
                                 N, T, H, dk, dv, handle)
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_prefill_slots")
    return out


def decode(q, k, v, g, beta, state_pool, state_slots=None, out=None, stream=None):
    """One KDA recurrence step per sequence (decode) on torch CUDA tensors.

    q, k, v: [N][H][128] bfloat16 (row n = sequence n's new token); g:
    [N][H][128] float32; beta: [N][H] float32; state_pool:
    [num_slots][H][128][128] float32, updated in place; state_slots: [N] int32
    on the device (-1 = padded row, skipped) or None for entry n.  Returns out
    [N][H][128] bfloat16 (rows of padded sequences keep what ``out`` held).
    """
    import torch

    N, H, dk = q.shape
    dv = v.shape[2]
    tensors = [("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("state_pool", state_pool)]
    if state_slots is not None:
        tensors.append(("state_slots", state_slots))
    for name, t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if q.dtype != torch.bfloat16:
        raise ValueError("decode takes bfloat16 q/k/v")
    if state_slots is not None and (state_slots.dtype != torch.int32 or tuple(state_slots.shape) != (N,)):
        raise ValueError("state_slots must be int32 [N]")
    if state_pool.dtype != torch.float32 or tuple(state_pool.shape[1:]) != (H, dv, dk):
        raise ValueError("state_pool must be float32 [num_slots][H][dv][dk]")
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    handle = int(s.cuda_stream) if hasattr(s, "cuda_stream") else int(s)
    st = kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_slots), _ptr(state_pool),
                    int(state_pool.shape[0]), _ptr(out), N, H, dk, dv, handle)
    if st != KDA_OK:
        raise KdaError(st, "kda_decode")
    return out


def fold_commit(k, v, g, beta, accepted, state_pool, state_slots=None, stream=None):
    """Commit of a speculative round on torch CUDA tensors: the first accepted[n]
    tokens of sequence n's window are folded into its state.

    k, v: [N][W][H][128] bfloat16; g: [N][W][H][128] float32; beta: [N][W][H]
    float32; accepted: [N] int32 on the device; state_pool:
    [num_slots][H][128][128] float32, updated in place; state_slots: [N] int32
    (-1 = skip) or None for entry n.
    """
    import torch

    N, W, H, dk = k.shape
    dv = v.shape[3]
    tensors = [("k", k), ("v", v), ("g", g), ("beta", beta), ("accepted", accepted), ("state_pool", state_pool)]
    if state_slots is not None:
        tensors.append(("state_slots", state_slots))
    for name, t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k.dtype != torch.bfloat16:
        raise ValueError("fold_commit takes bfloat16 k/v")
    if accepted.dtype != torch.int32 or tuple(accepted.shape) != (N,):
        raise ValueError("accepted must be int32 [N]")
    if state_pool.dtype != torch.float32 or tuple(state_pool.shape[1:]) != (H, dv, dk):
        raise ValueError("state_pool must be float32 [num_slots][H][dv][dk]")
    s = stream if stream is not None else torch.cuda.current_stream(k.device)
    handle = int(s.cuda_stream) if hasattr(s, "cuda_stream") else int(s)
    st = kda_fold_commit(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(accepted), _ptr(state_slots),
                         _ptr(state_pool), int(state_pool.shape[0]), N, W, H, dk, dv, handle)
    if st != KDA_OK:
        raise KdaError(st, "kda_fold_commit")


ACTIVATIONS = {"none": 0, "silu": 1}


def short_conv(xq, xk, xv, conv_weight, cu_seqlens, conv_pool, conv_slots=None, activation: str = "silu",
               eps: float = 1e-6, out=None, stream=None):
    """Short conv + L2 norm prologue on torch CUDA tensors.

    xq, xk, xv: [T][H][128] bfloat16; conv_weight: [3][H*128][4] float32 (tap
    3 weighs the row itself); cu_seqlens: [N+1] int32; conv_pool:
    [num_slots][3][3][H*128] bfloat16, updated in place; conv_slots: [N] int32
    (-1 = padded, skipped) or None for entry n.  activation "none" or "silu".
    Returns (q, k, v), each [T][H][128] bfloat16 (q and k with unit L2 norm
    per head).
    """
    import torch

    T, H, d = xq.shape
    N = int(cu_seqlens.shape[0]) - 1
    tensors = [("xq", xq), ("xk", xk), ("xv", xv), ("conv_weight", conv_weight), ("cu_seqlens", cu_seqlens),
               ("conv_pool", conv_pool)]
    if conv_slots is not None:
        tensors.append(("conv_slots", conv_slots))
    for name, t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if xq.dtype != torch.bfloat16 or xk.dtype != torch.bfloat16 or xv.dtype != torch.bfloat16:
        raise ValueError("short_conv takes bfloat16 projections")
    if conv_weight.dtype != torch.float32 or tuple(conv_weight.shape) != (3, H * d, 4):
        raise ValueError("conv_weight must be float32 [3][H*d][4]")
    if conv_pool.dtype != torch.bfloat16 or tuple(conv_pool.shape[1:]) != (3, 3, H * d):
        raise ValueError("conv_pool must be bfloat16 [num_slots][3][3][H*d]")
    if conv_slots is not None and (conv_slots.dtype != torch.int32 or tuple(conv_slots.shape) != (N,)):
        raise ValueError("conv_slots must be int32 [N]")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    if out is None:
        out = tuple(torch.empty_like(xq) for _ in range(3))
    q, k, v = out
    s = stream if stream is not None else torch.cuda.current_stream(xq.device)
    handle = int(s.cuda_stream) if hasattr(s, "cuda_stream") else int(s)
    st = kda_short_conv(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(conv_weight), _ptr(cu_seqlens), _ptr(conv_slots),
                        _ptr(conv_pool), int(conv_pool.shape[0]), _ptr(q), _ptr(k), _ptr(v), N, T, H, d,
                        ACTIVATIONS[activation], float(eps), handle)
    if st != KDA_OK:
        raise KdaError(st, "kda_short_conv")
    return q, k, v


def chunk_prefill_conv(xq, xk, xv, conv_weight, g, beta, cu_seqlens, conv_pool, state_pool, slots=None,
                       activation: str = "silu", eps: float = 1e-6, out=None, stream=None):
    """A KDA layer's prefill with the short-conv + L2-norm prologue fused in,
    on torch CUDA tensors.

    xq, xk, xv: [T][H][128] bfloat16 projections; conv_weight: [3][H*128][4]
    float32; g: [T][H][128] float32; beta: [T][H] float32; cu_seqlens: [N+1]
    int32; conv_pool: [conv_num_slots][3][3][H*128] bfloat16 and state_pool:
    [num_slots][H][128][128] float32, both updated in place; slots: [N] int32
    (-1 = padded, skipped) or None for entry n of both pools.  Returns out
    [T][H][128] bfloat16 (rows of padded sequences keep what ``out`` held).
    """
    import torch

    T, H, d = xq.shape
    N = int(cu_seqlens.shape[0]) - 1
    tensors = [("xq", xq), ("xk", xk), ("xv", xv), ("conv_weight", conv_weight), ("g", g), ("beta", beta),
               ("cu_seqlens", cu_seqlens), ("conv_pool", conv_pool), ("state_pool", state_pool)]
    if slots is not None:
        tensors.append(("slots", slots))
        if slots.dtype != torch.int32 or tuple(slots.shape) != (N,):
            raise ValueError("slots must be int32 [N]")
    for name, t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if xq.dtype != torch.bfloat16 or xk.dtype != torch.bfloat16 or xv.dtype != torch.bfloat16:
        raise ValueError("chunk_prefill_conv takes bfloat16 projections")
    if conv_weight.dtype != torch.float32 or tuple(conv_weight.shape) != (3, H * d, 4):
        raise ValueError("conv_weight must be float32 [3][H*d][4]")
    if conv_pool.dtype != torch.bfloat16 or tuple(conv_pool.shape[1:]) != (3, 3, H * d):
        raise ValueError("conv_pool must be bfloat16 [num_slots][3][3][H*d]")
    if state_pool.dtype != torch.float32 or tuple(state_pool.shape[1:]) != (H, d, d):
        raise ValueError("state_pool must be float32 [num_slots][H][d][d]")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    if out is None:
        out = torch.empty((T, H, d), dtype=xq.dtype, device=xq.device)
    s = stream if stream is not None else torch.cuda.current_stream(xq.device)
    handle = int(s.cuda_stream) if hasattr(s, "cuda_stream") else int(s)
    st = kda_chunk_prefill_conv(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(conv_weight), _ptr(g), _ptr(beta),
                                _ptr(cu_seqlens), _ptr(slots), _ptr(conv_pool), int(conv_pool.shape[0]),
                                _ptr(state_pool), int(state_pool.shape[0]), _ptr(out), N, T, H, d, d,
                                ACTIVATIONS[activation], float(eps), handle)
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_prefill_conv")
    return out


def decode_conv(xq, xk, xv, conv_weight, conv_pool, g, beta, state_pool, conv_slots=None, state_slots=None,
                activation: str = "silu", eps: float = 1e-6, out=None, stream=None):
    """The decode step with the short conv + L2 norm prologue fused in front of
    it, on torch CUDA tensors.

    xq, xk, xv: [N][H][128] bfloat16 (row n = sequence n's new token, before
    the conv); conv_weight: [3][H*128][4] float32; conv_pool:
    [conv_num_slots][3][3][H*128] bfloat16 and state_pool:
    [num_slots][H][128][128] float32, both updated in place; conv_slots,
    state_slots: [N] int32 (-1 = padded row, skipped) or None for entry n;
    g: [N][H][128] float32; beta: [N][H] float32.  Returns out [N][H][128]
    bfloat16 (rows of padded sequences keep what ``out`` held).
    """
    import torch

    N, H, d = xq.shape
    tensors = [("xq", xq), ("xk", xk), ("xv", xv), ("conv_weight", conv_weight), ("conv_pool", conv_pool),
               ("g", g), ("beta", beta), ("state_pool", state_pool)]
    for name, t in (("conv_slots", conv_slots), ("state_slots", state_slots)):
        if t is not None:
            tensors.append((name, t))
            if t.dtype != torch.int32 or tuple(t.shape) != (N,):
                raise ValueError(f"{name} must be int32 [N]")
    for name, t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if xq.dtype != torch.bfloat16 or xk.dtype != torch.bfloat16 or xv.dtype != torch.bfloat16:
        raise ValueError("decode_conv takes bfloat16 projections")
    if conv_weight.dtype != torch.float32 or tuple(conv_weight.shape) != (3, H * d, 4):
        raise ValueError("conv_weight must be float32 [3][H*d][4]")
    if conv_pool.dtype != torch.bfloat16 or tuple(conv_pool.shape[1:]) != (3, 3, H * d):
        raise ValueError("conv_pool must be bfloat16 [num_slots][3][3][H*d]")
    if state_pool.dtype != torch.float32 or tuple(state_pool.shape[1:]) != (H, d, d):
        raise ValueError("state_pool must be float32 [num_slots][H][dv][dk]")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    if out is None:
        out = torch.empty((N, H, d), dtype=xq.dtype, device=xq.device)
    s = stream if stream is not None else torch.cuda.current_stream(xq.device)
    handle = int(s.cuda_stream) if hasattr(s, "cuda_stream") else int(s)
    st = kda_decode_conv(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(conv_weight), _ptr(conv_slots), _ptr(conv_pool),
                         int(conv_pool.shape[0]), _ptr(g), _ptr(beta), _ptr(state_slots), _ptr(state_pool),
                         int(state_pool.shape[0]), _ptr(out), N, H, d, d, ACTIVATIONS[activation], float(eps),
                         handle)
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_conv")
    return out
