"""GPU parity against the fp64 oracle, through the C ABI (via the binding).

Tolerances (relative L2 over the whole tensor): 2e-3 on outputs, 1e-3 on
final states.  bf16 outputs alone carry about 1.66e-3 of round-to-nearest
error against the fp64 result; the kernel's own error (fp16 MMA operands,
fp32 accumulation) must fit in the rest.

The small cases are also checked element by element, to catch localised
corruption (a wrong row, head or index is off by about 100% of the tensor's
RMS) rather than to restate the L2 contract: |gpu - ref| <= 2^-8 |ref| +
0.05 rms(ref) for bf16 outputs (half an ulp of bf16, plus 5% of the RMS for
the kernel's worst-case operand roundings, where a sum of fp16-rounded terms
partly cancels) and <= 0.05 rms(ref) for fp32 outputs and states.
"""
import numpy as np
import pytest

from gpu_util import (OUT_TOL, STATE_TOL, inputs_to_dev, oracle_run, out_to_f64, rel_l2, run_gpu,
                      to_dev, torch)
from kda_linear_attention_chunk_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def check_elementwise(gpu, ref, bf16):
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = (2.0 ** -8) * np.abs(ref) + 0.05 * rms if bf16 else 0.05 * rms
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{int(bad.sum())} elements out of bound; worst {np.max(np.abs(gpu - ref)):.3e}"


def run_case(w, heads_for_oracle=None):
    x = syn.draw(w)
    cu = w.cu_seqlens()
    s0 = syn.draw_initial_state(w)
    out, fin = run_gpu(inputs_to_dev(x), cu, s0=to_dev(s0))
    torch().cuda.synchronize()
    o = out_to_f64(out)
    f = fin.cpu().numpy().astype(np.float64)
    if heads_for_oracle is None:
        o_ref, f_ref = oracle_run(x, cu, s0)
        return o, f, o_ref, f_ref
    hs = list(heads_for_oracle)
    xs = syn.draw(w, heads=hs)
    o_ref, f_ref = oracle_run(xs, cu, None if s0 is None else s0[:, hs])
    return o[:, hs], f[:, hs], o_ref, f_ref


@pytest.mark.parametrize("lens,H", [([1, 63, 64, 65, 130, 0, 200, 7], 3), ([64 * 3 + 17], 2), ([5] * 40, 2)])
def test_small_ragged_elementwise(lens, H):
    w = syn.Workload("small", lens, H=H, dk=128, dv=128, init_state=True, seed=3)
    o, f, o_ref, f_ref = run_case(w)
    assert rel_l2(o, o_ref) <= OUT_TOL
    assert rel_l2(f, f_ref) <= STATE_TOL
    check_elementwise(o, o_ref, bf16=True)
    check_elementwise(f, f_ref, bf16=False)


def test_tiny_fp32_256():
    w = syn.workloads()["tiny_fp32_256"]
    o, f, o_ref, f_ref = run_case(w)
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
    check_elementwise(o, o_ref, bf16=False)


def test_varlen4_4096():
    o, f, o_ref, f_ref = run_case(syn.workloads()["varlen4_4096"])
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL


def test_packed16_8192():
    o, f, o_ref, f_ref = run_case(syn.workloads()["packed16_8192"])
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
    # per-sequence diagnostic bound (each sequence's rows, all heads)
    cu = syn.workloads()["packed16_8192"].cu_seqlens()
    for n in range(len(cu) - 1):
        assert rel_l2(o[cu[n]:cu[n + 1]], o_ref[cu[n]:cu[n + 1]]) <= 2 * OUT_TOL


def test_long_65536_sampled_heads():
    w = syn.workloads()["long_65536"]
    o, f, o_ref, f_ref = run_case(w, heads_for_oracle=[0, 21])
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
    # long-range behaviour: the last 4096 rows alone are still within tolerance
    assert rel_l2(o[-4096:], o_ref[-4096:]) <= OUT_TOL


def test_context_262144_carried_state():
    w = syn.workloads()["context_262144"]
    rows = w.T // w.calls
    t = torch()
    cu = t.tensor([0, rows], dtype=t.int32, device="cuda")
    state = None
    hs = [5, 30]
    outs = []
    for c in range(w.calls):
        x = syn.draw(w, c * rows, (c + 1) * rows)
        out, state = run_gpu(inputs_to_dev(x), cu, s0=state)
        outs.append(out_to_f64(out)[:, hs])
    f = state.cpu().numpy().astype(np.float64)[:, hs]
    xs = syn.draw(w, heads=hs)
    o_ref, f_ref = oracle_run(xs, w.cu_seqlens())
    o = np.concatenate(outs)
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
