"""Failure detection on the GPU: a bounded wait that runs out.

Every wait of the tensor-core kernel gives up after a bounded number of
polls, sets bit 1 of the device error word, stops the other roles of its CTA
and winds down: every MMA and TMA copy already in flight lands before TMEM is
freed and the CTA exits, so the GPU stays usable.  This test builds a copy of
the library in which the chain's wait for MMA1 has a limit of zero polls: the
wait gives up at once although its MMA does complete, which drives every CTA
through that path -- in split mode the chain CTAs, whose abort then stops
the producer CTAs waiting on them.  The call must return, the copy's error word must hold
bit 1, and a normal call afterwards (the regular library, same process and
context) must still meet the parity bounds.
"""
import ctypes

import numpy as np
import pytest

import kda_linear_attention_chunk_gb300 as kda
from kda_linear_attention_chunk_gb300 import build as kbuild
from kda_linear_attention_chunk_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("split", ["0", "full", "half"])
def test_wait_timeout_sets_bit_and_leaves_the_gpu_usable(split, monkeypatch):
    from gpu_util import (OUT_TOL, STATE_TOL, check_elementwise, inputs_to_dev, oracle_run, out_to_f64, rel_l2,
                          run_gpu, to_dev, torch)
    # the fused kernel, or split mode with one or two chain CTAs a unit (their MMA1 wait)
    monkeypatch.setenv("KDA_SPLIT", split)
    t = torch()
    lib = kda.load(kbuild.build_variant("wait0", ["KDA_WAIT_LIMIT_MMA1=0"]))
    w = syn.Workload("timeout", [300, 64, 1, 129], H=4, dk=128, dv=128, init_state=True, seed=41)
    x = syn.draw(w)
    d = inputs_to_dev(x)
    s0 = to_dev(syn.draw_initial_state(w))
    cu = t.from_numpy(w.cu_seqlens()).cuda()
    out = t.empty((w.T, w.H, w.dv), dtype=t.bfloat16, device="cuda")
    fin = t.empty((w.N, w.H, w.dv, w.dk), dtype=t.float32, device="cuda")
    word = ctypes.c_int(0)
    assert lib.kda_device_error(ctypes.byref(word), 1) == kda.KDA_OK
    st = lib.kda_chunk_prefill(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(),
                               d["beta"].data_ptr(), cu.data_ptr(), s0.data_ptr(), out.data_ptr(), fin.data_ptr(),
                               w.N, w.T, w.H, w.dk, w.dv, int(t.cuda.current_stream().cuda_stream))
    assert st == kda.KDA_OK
    t.cuda.synchronize()                                  # the kernel returned
    assert lib.kda_device_error(ctypes.byref(word), 1) == kda.KDA_OK
    assert word.value & kda.ERR_WAIT_TIMEOUT, f"error word {word.value:#x}"
    # the context is intact: the regular library still computes the right thing
    o, f = run_gpu(d, cu, s0=s0)
    t.cuda.synchronize()
    o_ref, f_ref = oracle_run(x, w.cu_seqlens(), syn.draw_initial_state(w))
    o, f = out_to_f64(o), f.cpu().numpy().astype(np.float64)
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
    check_elementwise(o, o_ref, "tc_out")
    check_elementwise(f, f_ref, "tc_state")
