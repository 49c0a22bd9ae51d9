"""Every head size the boundary accepts, for both dtypes, against the oracle.

dk, dv in {64, 128} in all four combinations, bf16 (kda_chunk_prefill) and
fp32 (kda_chunk_prefill_f32) q/k/v, on a ragged packed batch with empty and
one-row sequences and nonzero initial states.  bf16 with dk = dv = 128 runs
on the tensor-core kernel and is held to its bounds; everything else runs on
the fp32 CUDA-core kernel and is held to the fp32 bounds (plus the bf16
rounding of the outputs).  The slot-addressed call is checked bit for bit
against the dense call on the CUDA-core kernel's head sizes.
"""
import numpy as np
import pytest

import kda_linear_attention_chunk_gb300 as kda
from gpu_util import (OUT_TOL, STATE_TOL, check_elementwise, inputs_to_dev, oracle_run, out_to_f64, rel_l2,
                      run_gpu, to_dev, torch)
from kda_linear_attention_chunk_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

LENS = [1, 63, 64, 65, 130, 0, 200, 7]
SIZES = [(64, 64), (64, 128), (128, 64), (128, 128)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", SIZES)
def test_head_size_parity(dtype, dk, dv):
    w = syn.Workload("sizes", LENS, H=3, dk=dk, dv=dv, qkv_dtype=dtype, init_state=True, seed=11)
    x = syn.draw(w)
    cu = w.cu_seqlens()
    s0 = syn.draw_initial_state(w)
    out, fin = run_gpu(inputs_to_dev(x), cu, s0=to_dev(s0))
    torch().cuda.synchronize()
    assert tuple(out.shape) == (w.T, w.H, dv) and tuple(fin.shape) == (w.N, w.H, dv, dk)
    o = out_to_f64(out)
    f = fin.cpu().numpy().astype(np.float64)
    o_ref, f_ref = oracle_run(x, cu, s0)
    assert rel_l2(o, o_ref) <= OUT_TOL and rel_l2(f, f_ref) <= STATE_TOL
    if dtype == "bf16" and dk == 128 and dv == 128:
        check_elementwise(o, o_ref, "tc_out")
        check_elementwise(f, f_ref, "tc_state")
    else:
        check_elementwise(o, o_ref, "f32_bf16out" if dtype == "bf16" else "f32")
        check_elementwise(f, f_ref, "f32")


@pytest.mark.parametrize("dk,dv", SIZES[:3])
def test_slots_on_other_head_sizes_equal_dense(dk, dv):
    t = torch()
    w = syn.Workload("sizes", LENS, H=2, dk=dk, dv=dv, init_state=True, seed=12)
    d = inputs_to_dev(syn.draw(w))
    cu = w.cu_seqlens()
    s0 = syn.draw_initial_state(w)
    out, fin = run_gpu(d, cu, s0=to_dev(s0))
    slots = np.array([4, 0, 7, 2, 9, 1, 3, 5], dtype=np.int32)
    pool = np.zeros((10, w.H, dv, dk), dtype=np.float32)
    pool[slots] = s0
    pool_t = to_dev(pool)
    cu_t = t.from_numpy(cu).cuda()
    out2 = kda.chunk_prefill_slots(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_t,
                                   t.from_numpy(slots).cuda(), pool_t)
    t.cuda.synchronize()
    assert t.equal(out2, out)
    assert t.equal(pool_t[t.from_numpy(slots).long().cuda()], fin)
    untouched = [6, 8]
    assert t.equal(pool_t[untouched], to_dev(pool)[untouched])
