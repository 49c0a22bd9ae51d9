"""The decay range of the tensor-core kernel, and kda_chunk_prefill_fullrange.

The tensor-core kernel splits every in-chunk decay exp(G_i - G_j) around the
chunk's middle row m into two fp16 factors.  include/kda.h states the range
in which that holds (|G_r - G_m| <= 15 ln 2 per chunk and key channel) and
that a chunk outside it sets bit 32 of the device error word.  These tests
draw gates of several strengths (synthetic.decay_profile: U[-a, 0] for
a = 0.2, 0.5, 1, 3; channels held at g = -20; 5% of the entries positive)
and check on the same inputs -- with the tensor-core kernel fused and in
split mode (environment variable KDA_SPLIT) -- that

* the bit is set when the inputs leave the range and clear when they stay
  inside it (the extent is computed here in fp64 from g; calls within 1% of
  the limit may go either way);
* inside the range the tensor-core results meet the parity bounds;
* kda_chunk_prefill_fullrange meets the fp32 bounds on every profile and
  never sets the bit, and keeps the packing and call-splitting identities.
"""
import numpy as np
import pytest

import kda_linear_attention_chunk_gb300 as kda
from gpu_util import (OUT_TOL, STATE_TOL, TC_MAX_FACTOR_LOG2, check_elementwise, inputs_to_dev, oracle_run,
                      out_to_f64, rel_l2, run_gpu, tc_decay_extent, to_dev, torch)
from kda_linear_attention_chunk_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

W = syn.Workload("decay", [1000, 513, 64, 300, 7, 129], H=4, dk=128, dv=128, init_state=True, seed=7)


def draw(profile, w=W):
    x = syn.draw(w)
    x["g"] = syn.decay_profile(x["g"], profile, seed=w.seed)
    return x, w.cu_seqlens(), syn.draw_initial_state(w)


def gpu_call(x, cu, s0, full_range):
    kda.device_error(reset=True)
    out, fin = run_gpu(inputs_to_dev(x), cu, s0=to_dev(s0), full_range=full_range)
    torch().cuda.synchronize()
    return out_to_f64(out), fin.cpu().numpy().astype(np.float64), kda.device_error(reset=True)


@pytest.mark.parametrize("split", ["0", "full", "half"])
@pytest.mark.parametrize("profile", syn.DECAY_PROFILES)
def test_tensor_core_range_bit_and_parity(profile, split, monkeypatch):
    # the fused kernel, and split mode (whose producers run the same decay scan)
    monkeypatch.setenv("KDA_SPLIT", split)
    x, cu, s0 = draw(profile)
    extent = tc_decay_extent(x["g"], cu)
    o, f, word = gpu_call(x, cu, s0, full_range=False)
    flagged = bool(word & kda.ERR_DECAY_RANGE)
    if extent > TC_MAX_FACTOR_LOG2 * 1.01:
        assert flagged, f"extent {extent:.2f} beyond the range but not reported"
        return
    if extent < TC_MAX_FACTOR_LOG2 * 0.99:
        assert not flagged, f"extent {extent:.2f} inside the range but reported"
    if flagged:
        return
    o_ref, f_ref = oracle_run(x, cu, s0)
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
    check_elementwise(o, o_ref, "tc_out")
    check_elementwise(f, f_ref, "tc_state")


def test_the_profiles_cover_both_sides_of_the_range():
    """The strong profiles leave the range, the default stays well inside."""
    cu = W.cu_seqlens()
    g = syn.draw(W)["g"]
    assert tc_decay_extent(g, cu) < 0.5 * TC_MAX_FACTOR_LOG2
    for p in ("u1", "u3", "alpha0"):
        assert tc_decay_extent(syn.decay_profile(g, p, seed=W.seed), cu) > 1.5 * TC_MAX_FACTOR_LOG2, p


@pytest.mark.parametrize("profile", syn.DECAY_PROFILES)
def test_fullrange_parity(profile):
    x, cu, s0 = draw(profile)
    o, f, word = gpu_call(x, cu, s0, full_range=True)
    assert not (word & kda.ERR_DECAY_RANGE)
    assert np.isfinite(o).all() and np.isfinite(f).all()
    o_ref, f_ref = oracle_run(x, cu, s0)
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
    check_elementwise(o, o_ref, "f32_bf16out")
    check_elementwise(f, f_ref, "f32")


def test_fullrange_packing_and_split_are_bit_exact():
    """A sequence alone equals its rows of the packed call, and a sequence cut
    into two calls at a multiple of 64 rows (state carried) equals one call."""
    t = torch()
    x, cu, s0 = draw("alpha0")
    d = inputs_to_dev(x)
    out, fin = run_gpu(d, cu, s0=to_dev(s0), full_range=True)
    n = 3                                                        # rows 1577 .. 1876
    lo, hi = int(cu[n]), int(cu[n + 1])
    one = {k: v[lo:hi].contiguous() for k, v in d.items()}
    o1, f1 = run_gpu(one, [0, hi - lo], s0=to_dev(s0[n:n + 1]), full_range=True)
    assert t.equal(o1, out[lo:hi]) and t.equal(f1[0], fin[n])
    cut = 128
    a = {k: v[:cut].contiguous() for k, v in one.items()}
    b = {k: v[cut:].contiguous() for k, v in one.items()}
    oa, fa = run_gpu(a, [0, cut], s0=to_dev(s0[n:n + 1]), full_range=True)
    ob, fb = run_gpu(b, [0, hi - lo - cut], s0=fa, full_range=True)
    t.cuda.synchronize()
    assert t.equal(t.cat([oa, ob]), o1) and t.equal(fb, f1)
