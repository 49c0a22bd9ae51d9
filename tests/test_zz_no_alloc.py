"""kda_chunk_prefill_noalloc, the entry point that allocates nothing, against
kda_chunk_prefill, through the C ABI.

Some callers cannot allocate device memory per call: a serving runtime that
lays out all of its device memory when a model is loaded, or a layer library
that is handed only its tensors.  For them the scheduling table that a large
packed batch needs lives in a static array inside the library, shared by
every call.  The GPU test therefore makes two calls in a row, on different
batches, and checks each against the regular entry point within the parity
tolerances of the other GPU tests.  This file is collected last.
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
    return [syn.Workload("many600", many, H=2, dk=128, dv=128, init_state=True, seed=21),
            syn.Workload("packed16", [90, 45, 1397, 48, 1088, 385, 352, 1002, 0, 209, 317, 563, 50, 154, 667, 491],
                         H=4, dk=128, dv=128, init_state=True, seed=22)]


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
def test_noalloc_matches_regular_entry_on_two_calls_in_a_row():
    from gpu_util import OUT_TOL, STATE_TOL, inputs_to_dev, out_to_f64, rel_l2, run_gpu, to_dev, torch
    t = torch()
    results = []
    for w in _workloads():
        d = inputs_to_dev(syn.draw(w))
        s0 = to_dev(syn.draw_initial_state(w))
        cu = t.from_numpy(np.asarray(w.cu_seqlens(), dtype=np.int32)).cuda()
        o_na, f_na = _noalloc_call(t, d, cu, s0, w)
        o_ref, f_ref = run_gpu(d, cu, s0=s0)
        results.append((w.name, o_na, f_na, o_ref, f_ref))
    t.cuda.synchronize()
    assert kda.device_error(reset=True) == 0
    for name, o_na, f_na, o_ref, f_ref in results:
        assert rel_l2(out_to_f64(o_na), out_to_f64(o_ref)) <= OUT_TOL, name
        assert rel_l2(f_na.cpu().numpy(), f_ref.cpu().numpy()) <= STATE_TOL, name


def test_noalloc_rejects_too_many_sequences():
    """N above the library-held table's size is refused before anything runs."""
    lib = kda.load()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    n = kda.KDA_NOALLOC_MAX_SEQS + 1
    st = lib.kda_chunk_prefill_noalloc(fake, fake, fake, fake, fake, fake, None, fake, None,
                                       n, 64, 2, 128, 128, None)
    assert st == kda.KDA_ERR_NOALLOC_LIMIT
    assert "KDA_NOALLOC_MAX_SEQS" in kda.status_string(st)
