"""The commit of a speculative round on the GPU (kda_fold_commit, the
ReplaySSM exact fold: SGLang PR #32890, prhub report, speculative-decoding
file list).  The state takes exactly the first accepted[n] tokens of
sequence n's window.  Checked against the oracle (those rows as a prefill)
and, bit for bit, against the same tokens applied by kda_decode one step at a
time."""
import numpy as np
import pytest

import oracle
from gpu_util import STATE_TOL, check_elementwise, rel_l2, to_dev, torch
from kda_linear_attention_chunk_gb300 import synthetic as syn
import kda_linear_attention_chunk_gb300 as kda

pytestmark = pytest.mark.gpu


def windows(N, W, H, seed):
    """N windows of W tokens: [N][W][H][...] arrays (rows drawn like prefill rows)."""
    w = syn.Workload("spec", [W] * N, H=H, dk=128, dv=128, seed=seed)
    x = syn.draw(w)
    return {k: v.reshape((N, W) + v.shape[1:]) for k, v in x.items()}


def make_pool(num_slots, H, seed):
    rng = np.random.default_rng(seed)
    return (0.02 * rng.standard_normal((num_slots, H, 128, 128))).astype(np.float32)


def gpu_fold(x, acc, pool_t, slots):
    t = torch()
    d = {k: to_dev(np.ascontiguousarray(v)) for k, v in x.items()}
    kda.fold_commit(d["k"], d["v"], d["g"], d["beta"], t.from_numpy(np.asarray(acc, dtype=np.int32)).cuda(),
                    pool_t, state_slots=None if slots is None else t.from_numpy(np.asarray(slots, np.int32)).cuda())
    t.cuda.synchronize()


def oracle_fold(x, acc, slots, pool):
    N, W = x["k"].shape[:2]
    flat = {k: v.reshape((N * W,) + v.shape[2:]) for k, v in x.items()}
    a = np.clip(np.asarray(acc), 0, W)
    rows = np.concatenate([np.arange(n * W, n * W + a[n]) for n in range(N)]).astype(np.int64)
    cu = np.concatenate([[0], np.cumsum(a)]).astype(np.int32)
    sel = {k: v[rows] for k, v in flat.items()}
    _, pool_ref, bad = oracle.run_slots(sel["k"], sel["k"], sel["v"], sel["g"], sel["beta"], cu, slots, pool)
    return pool_ref, bad


def test_fold_parity_with_oracle():
    N, W, H, num_slots = 24, 8, 4, 30
    x = windows(N, W, H, seed=41)
    rng = np.random.default_rng(41)
    acc = rng.integers(0, W + 1, N)
    slots = rng.permutation(num_slots)[:N].astype(np.int32)
    slots[[5, 17]] = -1
    pool = make_pool(num_slots, H, seed=13)
    pool_t = to_dev(pool)
    gpu_fold(x, acc, pool_t, slots)
    pool_ref, bad = oracle_fold(x, acc, slots, pool)
    assert bad == [] and (kda.device_error() & (kda.ERR_BAD_SLOT | kda.ERR_BAD_ACCEPTED)) == 0
    after = pool_t.cpu().numpy()
    touched = slots[(slots >= 0) & (acc > 0)]                    # entries the call folds tokens into
    assert rel_l2(after[touched], pool_ref[touched]) <= STATE_TOL
    check_elementwise(after[touched], pool_ref[touched], "f32")
    for n in np.nonzero((acc == 0) | (slots < 0))[0]:          # nothing folded: untouched, bit for bit
        if slots[n] >= 0:
            assert np.array_equal(after[slots[n]], pool[slots[n]])
    unnamed = np.setdiff1d(np.arange(num_slots), slots[slots >= 0])
    assert np.array_equal(after[unnamed], pool[unnamed])


def test_fold_equals_decode_steps_bitwise():
    t = torch()
    N, W, H, num_slots = 16, 6, 4, 20
    x = windows(N, W, H, seed=42)
    rng = np.random.default_rng(42)
    acc = rng.integers(0, W + 1, N)
    acc[0], acc[1] = 0, W
    slots = rng.permutation(num_slots)[:N].astype(np.int32)
    pool = make_pool(num_slots, H, seed=14)
    folded = to_dev(pool)
    gpu_fold(x, acc, folded, slots)
    stepped = to_dev(pool)
    for step in range(W):
        live = np.where(acc > step, slots, -1).astype(np.int32)
        d = {k: to_dev(np.ascontiguousarray(v[:, step])) for k, v in x.items()}
        kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], stepped,
                   state_slots=t.from_numpy(live).cuda())
    t.cuda.synchronize()
    assert t.equal(folded, stepped)


def test_fold_bad_counts_are_clamped_and_reported():
    N, W, H = 4, 5, 2
    x = windows(N, W, H, seed=43)
    acc = np.array([2, W + 3, -1, W], dtype=np.int32)
    pool = make_pool(N, H, seed=15)
    pool_t = to_dev(pool)
    kda.device_error(reset=True)
    gpu_fold(x, acc, pool_t, None)
    assert kda.device_error(reset=True) & kda.ERR_BAD_ACCEPTED
    pool_ref, _ = oracle_fold(x, acc, np.arange(N), pool)
    after = pool_t.cpu().numpy()
    touched = [0, 1, 3]                                          # counts 2, W + 3 (clamped to W) and W
    assert rel_l2(after[touched], pool_ref[touched]) <= STATE_TOL
    check_elementwise(after[touched], pool_ref[touched], "f32")
    assert np.array_equal(after[2], pool[2])                     # -1 clamps to 0: untouched
