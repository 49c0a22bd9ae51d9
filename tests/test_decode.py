"""The decode step on the GPU (kda_decode): one recurrence step per sequence on
states in a slot-addressed pool, padded rows (slot -1) skipped (kern-k3-pp-
prefill README, section "D inside SGLang").  A decode step is the prefill of
one row per sequence, so the oracle is its slot-indexed form on
cu_seqlens = 0, 1, ..., N."""
import numpy as np
import pytest

import oracle
from gpu_util import out_to_f64, rel_l2, to_dev, torch, OUT_TOL, STATE_TOL
from kda_linear_attention_chunk_gb300 import synthetic as syn
import kda_linear_attention_chunk_gb300 as kda

pytestmark = pytest.mark.gpu


def make_pool(num_slots, H, seed):
    rng = np.random.default_rng(seed)
    return (0.02 * rng.standard_normal((num_slots, H, 128, 128))).astype(np.float32)


def step_inputs(N, H, seed):
    """One token per sequence, drawn like the prefill workloads' rows."""
    w = syn.Workload("decode", [1] * N, H=H, dk=128, dv=128, seed=seed)
    return syn.draw(w)


def gpu_step(x, pool_t, slots=None, out=None):
    t = torch()
    d = {k: to_dev(v) for k, v in x.items()}
    sl = None if slots is None else t.from_numpy(np.asarray(slots, dtype=np.int32)).cuda()
    if out is None:
        N, H = x["q"].shape[:2]
        out = t.full((N, H, 128), float("nan"), dtype=t.bfloat16, device="cuda")
    kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], pool_t, state_slots=sl, out=out)
    t.cuda.synchronize()
    return out


def oracle_step(x, slots, pool, heads=None):
    N = x["q"].shape[0]
    return oracle.run_slots(x["q"], x["k"], x["v"], x["g"], x["beta"], np.arange(N + 1), slots, pool,
                            heads=heads)


def test_decode_parity_with_padding():
    N, H, num_slots = 37, 4, 50
    x = step_inputs(N, H, seed=31)
    rng = np.random.default_rng(31)
    slots = rng.permutation(num_slots)[:N].astype(np.int32)
    slots[[2, 9, 30]] = -1
    pool = make_pool(num_slots, H, seed=8)
    pool_t = to_dev(pool)
    out = gpu_step(x, pool_t, slots)
    o_ref, pool_ref, bad = oracle_step(x, slots, pool)
    assert bad == [] and (kda.device_error() & kda.ERR_BAD_SLOT) == 0
    live = slots >= 0
    assert rel_l2(out_to_f64(out)[live], o_ref[live]) <= OUT_TOL
    assert bool(torch().isnan(out[torch().from_numpy(~live).cuda()].float()).all())
    after = pool_t.cpu().numpy()
    assert rel_l2(after[slots[live]], pool_ref[slots[live]]) <= STATE_TOL
    unnamed = np.setdiff1d(np.arange(num_slots), slots[live])
    assert np.array_equal(after[unnamed], pool[unnamed])


def test_decode_dense_entries_without_a_table():
    N, H = 20, 2
    x = step_inputs(N, H, seed=32)
    pool = make_pool(N, H, seed=9)
    pool_t = to_dev(pool)
    out = gpu_step(x, pool_t, slots=None)
    o_ref, pool_ref, _ = oracle_step(x, np.arange(N), pool)
    assert rel_l2(out_to_f64(out), o_ref) <= OUT_TOL
    assert rel_l2(pool_t.cpu().numpy(), pool_ref) <= STATE_TOL


def test_decode_bad_ids_reported_and_skipped():
    N, H, num_slots = 6, 2, 4
    x = step_inputs(N, H, seed=33)
    slots = np.array([0, 4, 1, -3, 2, 3], dtype=np.int32)
    pool = make_pool(num_slots, H, seed=10)
    pool_t = to_dev(pool)
    kda.device_error(reset=True)
    out = gpu_step(x, pool_t, slots)
    assert kda.device_error(reset=True) & kda.ERR_BAD_SLOT
    o_ref, pool_ref, bad = oracle_step(x, slots, pool)
    assert bad == [1, 3]
    live = np.array([0, 2, 4, 5])
    assert rel_l2(out_to_f64(out)[live], o_ref[live]) <= OUT_TOL
    assert bool(torch().isnan(out[[1, 3]].float()).all())
    assert rel_l2(pool_t.cpu().numpy(), pool_ref) <= STATE_TOL


def test_decode_steps_continue_a_prefill():
    """A prefill of 100 rows per sequence, then 12 decode steps on the same
    pool, against the oracle's single pass over all 112 rows."""
    t = torch()
    N, H, P, D = 5, 2, 100, 12
    w = syn.Workload("ctx", [P + D] * N, H=H, dk=128, dv=128, seed=34)
    x = syn.draw(w)
    cu = w.cu_seqlens()
    slots = np.array([3, 0, 6, 2, 5], dtype=np.int32)
    pool = make_pool(8, H, seed=11)
    o_ref, pool_ref, _ = oracle.run_slots(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, slots, pool)
    pool_t = to_dev(pool)
    pre_rows = np.concatenate([np.arange(cu[n], cu[n] + P) for n in range(N)])
    pre = {k: to_dev(v[pre_rows]) for k, v in x.items()}
    sl = t.from_numpy(slots).cuda()
    kda.chunk_prefill_slots(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"],
                            t.from_numpy(np.arange(0, N * P + 1, P, dtype=np.int32)).cuda(), sl, pool_t)
    for step in range(D):
        rows = cu[:-1] + P + step
        out = gpu_step({k: v[rows] for k, v in x.items()}, pool_t, slots)
        assert rel_l2(out_to_f64(out), o_ref[rows]) <= OUT_TOL, f"step {step}"
    assert rel_l2(pool_t.cpu().numpy()[slots], pool_ref[slots]) <= STATE_TOL


def test_decode_batch64_h32_sampled_heads():
    """64 running requests, 32 heads, a pool of 256 entries (8 rows padded);
    every head checked through the final states, four heads' outputs too."""
    N, H, num_slots = 64, 32, 256
    x = step_inputs(N, H, seed=35)
    rng = np.random.default_rng(35)
    slots = rng.permutation(num_slots)[:N].astype(np.int32)
    slots[rng.permutation(N)[:8]] = -1
    pool = make_pool(num_slots, H, seed=12)
    pool_t = to_dev(pool)
    out = gpu_step(x, pool_t, slots)
    o_ref, pool_ref, _ = oracle_step(x, slots, pool)
    live = slots >= 0
    heads = [0, 7, 19, 31]
    assert rel_l2(out_to_f64(out)[live][:, heads], o_ref[live][:, heads]) <= OUT_TOL
    after = pool_t.cpu().numpy()
    assert rel_l2(after[slots[live]], pool_ref[slots[live]]) <= STATE_TOL
