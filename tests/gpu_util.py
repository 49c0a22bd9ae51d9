"""Helpers for the GPU tests: move synthetic inputs to the device, call the
library through its binding, and compare against the oracle."""
import numpy as np

import oracle
from kda_linear_attention_chunk_gb300 import synthetic as syn

OUT_TOL = 2e-3     # relative L2 on outputs (bf16 outputs carry ~1.66e-3 of rounding)
STATE_TOL = 1e-3   # relative L2 on final states

# ---- element-wise bounds -------------------------------------------------------
# Every element e = gpu - ref (ref the fp64 oracle) must satisfy
#     |e| <= r * |ref| + kappa * u * rms(ref)
# with r the output rounding (bf16 round-to-nearest: at most 2^-8 of |ref|,
# the half ulp at the bottom of a binade; 0 for fp32 outputs and states), u
# the unit roundoff of the arithmetic that feeds the result and kappa a
# budget for how such roundings add up (derivation in the design notes):
#
#  * tensor-core kernel: fp16 MMA operands (u = 2^-11), fp32 accumulation.  A
#    result is a sum of products of two rounded operands (relative error of a
#    product <= 2u, RMS about u sqrt(2/3)) over 64 or 128 terms, chained
#    through A, the inverse, W and U, Delta and the outputs; the RMS of the
#    error comes out near u * rms(ref) (measured: 0.4-0.9 u for outputs and
#    states on every workload), and kappa = 16 (outputs) and 20 (states)
#    leave about 20 sigma of that for the largest of up to 10^7 elements
#    (measured largest: 8-13 u for outputs, 9-14 u for states).
#  * CUDA-core kernel: fp32 throughout (u = 2^-24); its results are exact to
#    a few parts in 10^6, so kappa * u = 2^-14 (6.1e-5) of rms(ref) bounds
#    them with room for the fp32 cumulative sums behind strong decays.
#  * states of the tensor-core kernel fed by the short-conv prologue: the
#    conv mixes four consecutive rows and SiLU gives v a nonzero mean, so the
#    delta rule predicts the rows well and Delta = U - S'^T W'^T is a small
#    difference of two large terms; the fp16 rounding of S' (the MMA1
#    operand) then shows against a state smaller than those terms.  Measured
#    16-33 u on such inputs (the same bytes for the fused kernel and for the
#    prologue and the prefill as two calls); kappa = 48.
U_F16 = 2.0 ** -11
BF16_HALF_ULP = 2.0 ** -8
TC_OUT_KAPPA = 16
TC_STATE_KAPPA = 20
TC_STATE_PROLOGUE_KAPPA = 48
F32_ABS = 2.0 ** -14


def elementwise_excess(gpu, ref, rounding, abs_tol):
    """Largest |gpu - ref| / (rounding |ref| + abs_tol rms(ref)): <= 1 passes."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = rounding * np.abs(ref) + abs_tol * (rms if rms > 0 else 1.0)
    return float(np.max(np.abs(gpu - ref) / bound)) if ref.size else 0.0


def check_elementwise(gpu, ref, kind):
    """kind: 'tc_out' (bf16 outputs of the tensor-core kernel), 'tc_state',
    'tc_state_prologue' (its states when the short-conv prologue made q, k,
    v), 'f32_bf16out' (bf16 outputs of the CUDA-core kernel), 'f32' (fp32
    outputs or states of the CUDA-core kernel)."""
    rounding, abs_tol = {
        "tc_out": (BF16_HALF_ULP, TC_OUT_KAPPA * U_F16),
        "tc_state": (0.0, TC_STATE_KAPPA * U_F16),
        "tc_state_prologue": (0.0, TC_STATE_PROLOGUE_KAPPA * U_F16),
        "f32_bf16out": (BF16_HALF_ULP, F32_ABS),
        "f32": (0.0, F32_ABS),
    }[kind]
    x = elementwise_excess(gpu, ref, rounding, abs_tol)
    assert np.isfinite(x) and x <= 1.0, f"{kind}: element-wise error {x:.3f} x its bound"


# ---- the tensor-core kernel's decay range ----------------------------------------
TC_MAX_FACTOR_LOG2 = 15.0   # documented: |G_r - G_m| <= 15 ln 2 per chunk and key channel


def tc_decay_extent(g, cu_seqlens):
    """Largest |G_r - G_m| / ln 2 over every chunk, head and key channel of a
    call, in fp64 (G the in-chunk cumulative sum of g, m = (L - 1) // 2 the
    chunk's middle row): the quantity the tensor-core kernel checks."""
    g = np.asarray(g, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    worst = 0.0
    for n in range(len(cu) - 1):
        for c0 in range(int(cu[n]), int(cu[n + 1]), 64):
            L = min(64, int(cu[n + 1]) - c0)
            G = np.cumsum(g[c0:c0 + L], axis=0)
            worst = max(worst, float(np.max(np.abs(G - G[(L - 1) // 2]))))
    return worst / np.log(2.0)


def sampled_heads(w, count, salt=0):
    """Heads of workload w to check against the oracle: a seeded draw that
    changes with the workload's seed and with KDA_TEST_SEED (default 0)."""
    import os
    run = int(os.environ.get("KDA_TEST_SEED", "0"))
    u = syn.uniform(w.seed * 1009 + run * 7919 + salt, 900, 4 * count)
    hs = []
    for x in u:
        h = int(x * w.H)
        if h not in hs:
            hs.append(h)
        if len(hs) == count:
            break
    return sorted(hs)


def torch():
    import torch as t
    return t


def to_dev(x, bf16=True):
    t = torch()
    if x is None:
        return None
    if x.dtype == np.uint16:
        return t.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(t.bfloat16).cuda()
    return t.from_numpy(np.ascontiguousarray(x)).cuda()


def inputs_to_dev(x):
    return {k: to_dev(v) for k, v in x.items()}


def run_gpu(d, cu, s0=None, out=None, final_state=None, stream=None, full_range=False):
    import kda_linear_attention_chunk_gb300 as kda
    t = torch()
    cu_t = t.from_numpy(np.asarray(cu, dtype=np.int32)).cuda() if not hasattr(cu, "is_cuda") else cu
    return kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_t,
                             initial_state=s0, out=out, final_state=final_state, stream=stream,
                             full_range=full_range)


def out_to_f64(o):
    t = torch()
    if o.dtype == t.bfloat16:
        return o.float().cpu().numpy().astype(np.float64)
    return o.cpu().numpy().astype(np.float64)


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def oracle_run(x, cu, s0=None, heads=None, nthreads=None):
    return oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, initial_state=s0,
                      heads=heads, nthreads=nthreads)
