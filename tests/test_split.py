"""Split mode of the tensor-core prefill: for calls with few (sequence, head)
units, the chunk preparation runs on most SMs and each unit's state chain on
an SM of its own, the two handing chunks over through a ring in device memory.

The chain computes exactly the fused kernel's operations on exactly its
operands (the producers run the fused kernel's prep code), so the split and
the fused kernel must give the same bytes -- with one chain CTA a unit, or
two that keep half of the value channels each.  KDA_SPLIT=0 / full / half
(read on every call) forces a mode; half falls back to full where the SMs do
not allow two chains a unit.  Parity against the oracle is covered here on a
ragged batch with a long sequence, and by test_parity's varlen4_4096,
long_65536 and context_262144 workloads (64 and 32 units: split by default).
"""
import os

import numpy as np
import pytest

import kda_linear_attention_chunk_gb300 as kda
from gpu_util import (OUT_TOL, STATE_TOL, check_elementwise, inputs_to_dev, oracle_run, out_to_f64, rel_l2, run_gpu,
                      to_dev, torch)
from kda_linear_attention_chunk_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def run_mode(mode, fn):
    old = os.environ.get("KDA_SPLIT")
    os.environ["KDA_SPLIT"] = mode
    try:
        return fn()
    finally:
        if old is None:
            del os.environ["KDA_SPLIT"]
        else:
            os.environ["KDA_SPLIT"] = old


def dense_call(w, x, s0):
    t = torch()
    d = inputs_to_dev(x)
    s0d = to_dev(s0)
    cu = w.cu_seqlens()

    def go():
        kda.device_error(reset=True)
        o, f = run_gpu(d, cu, s0=s0d)
        t.cuda.synchronize()
        assert kda.device_error(reset=True) == 0
        return o.view(t.int16).cpu().numpy(), f.cpu().numpy()
    return go


@pytest.mark.parametrize("lens,H", [([700], 2), ([300, 1, 0, 64, 65, 129, 5], 3), ([64 * 20 + 3, 17], 8),
                                    ([2519, 1000, 513, 64], 16), ([64 * 40 + 31, 0, 1], 12)])
def test_split_equals_fused_bit_for_bit(lens, H):
    w = syn.Workload("split", lens, H=H, dk=128, dv=128, init_state=True, seed=51)
    x = syn.draw(w)
    go = dense_call(w, x, syn.draw_initial_state(w))
    o_f, s_f = run_mode("0", go)
    for mode in ("full", "half"):
        o_s, s_s = run_mode(mode, go)
        np.testing.assert_array_equal(o_s, o_f, err_msg=mode)
        np.testing.assert_array_equal(s_s, s_f, err_msg=mode)


def test_split_slots_equals_fused_bit_for_bit():
    t = torch()
    lens = [400, 3, 0, 190]
    H, entries = 4, 9
    w = syn.Workload("split_slots", lens, H=H, dk=128, dv=128, init_state=False, seed=52)
    x = syn.draw(w)
    d = inputs_to_dev(x)
    cu = t.from_numpy(w.cu_seqlens()).cuda()
    rng = np.random.default_rng(52)
    pool0 = (0.02 * rng.standard_normal((entries, H, 128, 128))).astype(np.float32)
    slots = t.tensor([5, -1, 2, 7], dtype=t.int32, device="cuda")

    def go():
        pool = t.from_numpy(pool0.copy()).cuda()
        out = t.zeros((w.T, H, 128), dtype=t.bfloat16, device="cuda")
        kda.device_error(reset=True)
        kda.chunk_prefill_slots(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, slots, pool, out=out)
        t.cuda.synchronize()
        assert kda.device_error(reset=True) == 0
        return out.view(t.int16).cpu().numpy(), pool.cpu().numpy()
    o_f, p_f = run_mode("0", go)
    for mode in ("full", "half"):
        o_s, p_s = run_mode(mode, go)
        np.testing.assert_array_equal(o_s, o_f, err_msg=mode)
        np.testing.assert_array_equal(p_s, p_f, err_msg=mode)
        untouched = [0, 1, 3, 4, 6, 8]
        np.testing.assert_array_equal(p_s[untouched], pool0[untouched])


@pytest.mark.parametrize("mode", ["full", "half"])
def test_split_parity_ragged_long(mode):
    """Against the oracle, element by element: a long sequence with short ones."""
    w = syn.Workload("split_parity", [64 * 24 + 37, 5, 130, 64], H=4, dk=128, dv=128, init_state=True, seed=53)
    x = syn.draw(w)
    s0 = syn.draw_initial_state(w)
    d = inputs_to_dev(x)

    def go():
        o, f = run_gpu(d, w.cu_seqlens(), s0=to_dev(s0))
        torch().cuda.synchronize()
        return out_to_f64(o), f.cpu().numpy().astype(np.float64)
    o, f = run_mode(mode, go)
    o_ref, f_ref = oracle_run(x, w.cu_seqlens(), s0)
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
    check_elementwise(o, o_ref, "tc_out")
    check_elementwise(f, f_ref, "tc_state")


@pytest.mark.parametrize("mode", ["full", "half"])
def test_split_repeated_calls_identical(mode):
    """The ring and its flags are fresh each call: back-to-back calls on one
    stream give the same bytes."""
    w = syn.Workload("split_repeat", [2000, 300], H=6, dk=128, dv=128, init_state=True, seed=54)
    x = syn.draw(w)
    go = dense_call(w, x, syn.draw_initial_state(w))
    first = run_mode(mode, go)
    for _ in range(3):
        again = run_mode(mode, go)
        np.testing.assert_array_equal(again[0], first[0])
        np.testing.assert_array_equal(again[1], first[1])
