"""Helpers for the GPU tests: move synthetic inputs to the device, call the
library through its binding, and compare against the oracle."""
import numpy as np

import oracle
from kda_linear_attention_chunk_gb300 import synthetic as syn

OUT_TOL = 2e-3     # relative L2 on outputs (bf16 outputs carry ~1.66e-3 of rounding)
STATE_TOL = 1e-3   # relative L2 on final states


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


def run_gpu(d, cu, s0=None, out=None, final_state=None, stream=None):
    import kda_linear_attention_chunk_gb300 as kda
    t = torch()
    cu_t = t.from_numpy(np.asarray(cu, dtype=np.int32)).cuda() if not hasattr(cu, "is_cuda") else cu
    return kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_t,
                             initial_state=s0, out=out, final_state=final_state, stream=stream)


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
