"""kda_chunk_prefill_noalloc, the entry point that allocates nothing, against
kda_chunk_prefill, through the C ABI.

Some callers cannot allocate device memory per call: a serving runtime that
lays out all of its device memory when a model is loaded, or a layer library
that is handed only its tensors.  For them the scheduling table that a large
packed batch needs lives in a static array inside the library, shared by
every call.  The GPU test therefore makes calls in a row, on different
batches -- up to KDA_NOALLOC_MAX_SEQS sequences, the size of that array --
and checks each against the regular entry point bit for bit: the per-sequence
arithmetic does not depend on which SM runs a sequence or when, so the two
entry points must give the same bytes.  The largest batch is also checked
against the fp64 oracle on sampled sequences.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest

import kda_linear_attention_chunk_gb300 as kda
from kda_linear_attention_chunk_gb300 import synthetic as syn


def _workloads():
    rng = np.random.default_rng(5)
    many = [int(x) for x in rng.integers(0, 96, size=600)]      # 600 short sequences, some empty
    many[17] = 0
    many[300] = 200
    edge = [int(x) for x in rng.integers(0, 9, size=kda.KDA_NOALLOC_MAX_SEQS)]   # the limit itself
    edge[0] = 0
    edge[-1] = 0
    edge[5000] = 130
    return [syn.Workload("many600", many, H=2, dk=128, dv=128, init_state=True, seed=21),
            syn.Workload("packed16", [90, 45, 1397, 48, 1088, 385, 352, 1002, 0, 209, 317, 563, 50, 154, 667, 491],
                         H=4, dk=128, dv=128, init_state=True, seed=22),
            syn.Workload("edge16384", edge, H=2, dk=128, dv=128, init_state=True, seed=23)]


def _noalloc_call(t, d, cu, s0, w):
    out = t.empty((w.T, w.H, w.dv), dtype=t.bfloat16, device="cuda")
    fin = t.empty((w.N, w.H, w.dv, w.dk), dtype=t.float32, device="cuda")
    stream = t.cuda.current_stream()
    st = kda.kda_chunk_prefill_noalloc(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(),
                                       d["beta"].data_ptr(), cu.data_ptr(), s0.data_ptr(), out.data_ptr(),
                                       fin.data_ptr(), w.N, w.T, w.H, w.dk, w.dv, int(stream.cuda_stream))
    assert st == kda.KDA_OK, kda.status_string(st)
    return out, fin


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_on_calls_in_a_row():
    from gpu_util import OUT_TOL, STATE_TOL, inputs_to_dev, oracle_run, out_to_f64, rel_l2, run_gpu, to_dev, torch
    t = torch()
    results = []
    for w in _workloads():
        x = syn.draw(w)
        d = inputs_to_dev(x)
        s0 = to_dev(syn.draw_initial_state(w))
        cu = t.from_numpy(np.asarray(w.cu_seqlens(), dtype=np.int32)).cuda()
        o_na, f_na = _noalloc_call(t, d, cu, s0, w)
        o_ref, f_ref = run_gpu(d, cu, s0=s0)
        results.append((w, x, o_na, f_na, o_ref, f_ref))
    t.cuda.synchronize()
    assert kda.device_error(reset=True) == 0
    for w, x, o_na, f_na, o_ref, f_ref in results:
        assert t.equal(o_na, o_ref), w.name
        assert t.equal(f_na, f_ref), w.name
    # the batch at the limit against the oracle, on sampled sequences
    w, x, o_na, f_na, _, _ = results[-1]
    cu = w.cu_seqlens()
    s0 = syn.draw_initial_state(w)
    picks = [5000] + [int(n) for n in np.random.default_rng(9).choice(w.N, size=24, replace=False)]
    o = out_to_f64(o_na)
    f = f_na.cpu().numpy().astype(np.float64)
    for n in picks:
        lo, hi = int(cu[n]), int(cu[n + 1])
        xs = {k: v[lo:hi] for k, v in x.items()}
        o_ref, f_ref = oracle_run(xs, np.array([0, hi - lo], dtype=np.int32), s0[n:n + 1])
        if hi > lo:
            assert rel_l2(o[lo:hi], o_ref) <= OUT_TOL, n
        assert rel_l2(f[n:n + 1], f_ref) <= STATE_TOL, n


def test_noalloc_rejects_too_many_sequences():
    """N above the library-held table's size is refused before anything runs
    (the other checks, which come first, pass on these never-dereferenced
    addresses)."""
    lib = kda.load()
    n = kda.KDA_NOALLOC_MAX_SEQS + 1
    T, H, d = 64, 2, 128
    base, step = 1 << 24, 1 << 22          # distinct, 16-byte aligned, far apart
    q, k, v, g, beta, cu, out = (ctypes.c_void_p(base + i * step) for i in range(7))
    st = lib.kda_chunk_prefill_noalloc(q, k, v, g, beta, cu, None, out, None, n, T, H, d, d, None)
    assert st == kda.KDA_ERR_NOALLOC_LIMIT
    assert "KDA_NOALLOC_MAX_SEQS" in kda.status_string(st)
