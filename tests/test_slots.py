"""Slot-addressed states on the GPU (kda_chunk_prefill_slots).

A serving engine keeps each request's recurrent state in a pool laid out
[slot][head][v][k] fp32 and names it by slot id; padded entries carry -1 and
are skipped (kern-k3-pp-prefill README, section "D inside SGLang").  These
tests compare the kernel with the oracle's slot-indexed form, check that a
sequence's results are bit for bit those of the dense-state call, that
padded sequences and unnamed pool entries are left alone, that ids outside
the pool are reported and skipped, and that the pool carries the state
across calls."""
import numpy as np
import pytest

import oracle
from gpu_util import inputs_to_dev, out_to_f64, rel_l2, run_gpu, to_dev, torch, OUT_TOL, STATE_TOL
from kda_linear_attention_chunk_gb300 import synthetic as syn
import kda_linear_attention_chunk_gb300 as kda

pytestmark = pytest.mark.gpu


def make_pool(num_slots, H, seed):
    rng = np.random.default_rng(seed)
    return (0.02 * rng.standard_normal((num_slots, H, 128, 128))).astype(np.float32)


def slots_call(d, cu, slots, pool_t, out=None):
    t = torch()
    cu_t = t.from_numpy(np.asarray(cu, dtype=np.int32)).cuda()
    sl_t = t.from_numpy(np.asarray(slots, dtype=np.int32)).cuda()
    if out is None:
        T, H = d["q"].shape[:2]
        out = t.full((T, H, 128), float("nan"), dtype=t.bfloat16, device="cuda")
    kda.chunk_prefill_slots(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_t, sl_t, pool_t, out=out)
    t.cuda.synchronize()
    return out


def dense_call(d, cu, slots, pool):
    """The dense-state call on the same rows, each sequence starting from its
    pool entry (zeros for padded ones, whose results are ignored)."""
    s0 = np.zeros((len(slots),) + pool.shape[1:], dtype=np.float32)
    for n, s in enumerate(slots):
        if 0 <= s < pool.shape[0]:
            s0[n] = pool[s]
    out, fin = run_gpu(d, cu, s0=to_dev(s0))
    torch().cuda.synchronize()
    return out, fin


def live(slots, num_slots):
    return [n for n, s in enumerate(slots) if 0 <= s < num_slots]


def check_against_dense(w, x, slots, pool, out, pool_after):
    """Live sequences: out rows and pool entries equal the dense call bitwise;
    padded sequences: rows still NaN; entries nobody names: unchanged."""
    t = torch()
    cu = w.cu_seqlens()
    o_d, f_d = dense_call(inputs_to_dev(x), cu, slots, pool)
    named = set()
    for n, s in enumerate(slots):
        rows = slice(int(cu[n]), int(cu[n + 1]))
        if 0 <= s < pool.shape[0]:
            named.add(int(s))
            assert t.equal(out[rows], o_d[rows]), f"sequence {n} rows"
            assert t.equal(pool_after[s], f_d[n]), f"sequence {n} state (slot {s})"
        else:
            assert bool(t.isnan(out[rows].float()).all()), f"padded sequence {n} was written"
    for s in range(pool.shape[0]):
        if s not in named:
            assert t.equal(pool_after[s], t.from_numpy(pool[s]).cuda()), f"unnamed slot {s} changed"


def test_slots_parity_with_oracle():
    lens = [300, 1, 64, 0, 129, 700, 65]
    slots = [7, 2, -1, 5, 11, -1, 0]
    w = syn.Workload("slots", lens, H=4, dk=128, dv=128, seed=21)
    x = syn.draw(w)
    pool = make_pool(12, 4, seed=3)
    pool_t = to_dev(pool)
    out = slots_call(inputs_to_dev(x), w.cu_seqlens(), slots, pool_t)
    o_ref, pool_ref, bad = oracle.run_slots(x["q"], x["k"], x["v"], x["g"], x["beta"], w.cu_seqlens(),
                                            slots, pool)
    assert bad == [] and (kda.device_error() & kda.ERR_BAD_SLOT) == 0
    cu = w.cu_seqlens()
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in live(slots, 12)])
    o = out_to_f64(out)
    assert rel_l2(o[rows], o_ref[rows]) <= OUT_TOL
    named = [s for s in slots if s >= 0]
    assert rel_l2(pool_t.cpu().numpy()[named], pool_ref[named]) <= STATE_TOL
    check_against_dense(w, x, slots, pool, out, pool_t)
    # the zero-row sequence's entry is left as it was
    assert torch().equal(pool_t[5], torch().from_numpy(pool[5]).cuda())


def test_slots_bad_ids_reported_and_skipped():
    lens = [100, 64, 200, 33]
    slots = [3, 4, -7, 1]         # 4 and -7 lie outside a pool of 4 entries
    w = syn.Workload("badslot", lens, H=2, dk=128, dv=128, seed=22)
    x = syn.draw(w)
    pool = make_pool(4, 2, seed=4)
    pool_t = to_dev(pool)
    kda.device_error(reset=True)
    out = slots_call(inputs_to_dev(x), w.cu_seqlens(), slots, pool_t)
    assert kda.device_error(reset=True) & kda.ERR_BAD_SLOT
    check_against_dense(w, x, slots, pool, out, pool_t)


def test_slots_many_sequences():
    """More sequences than the kernel sorts in shared memory: the unsorted
    deal, with a fifth of the entries padded."""
    rng = np.random.default_rng(23)
    N = 300
    lens = syn.random_lengths(6000, N, seed=23, allow_empty=True)
    slots = rng.permutation(400)[:N].astype(np.int32)
    slots[rng.random(N) < 0.2] = -1
    w = syn.Workload("many", lens, H=2, dk=128, dv=128, seed=23)
    x = syn.draw(w)
    pool = make_pool(400, 2, seed=5)
    pool_t = to_dev(pool)
    out = slots_call(inputs_to_dev(x), w.cu_seqlens(), slots, pool_t)
    check_against_dense(w, x, list(slots), pool, out, pool_t)
    o_ref, pool_ref, _ = oracle.run_slots(x["q"], x["k"], x["v"], x["g"], x["beta"], w.cu_seqlens(),
                                          slots, pool)
    cu = w.cu_seqlens()
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in live(slots, 400)])
    assert rel_l2(out_to_f64(out)[rows], o_ref[rows]) <= OUT_TOL
    named = slots[slots >= 0]
    assert rel_l2(pool_t.cpu().numpy()[named], pool_ref[named]) <= STATE_TOL


def test_slots_packed16_8192_full_size():
    """The 16-sequence, 8192-row, 32-head batch in a pool of 64 entries, two
    sequences padded: bit for bit the dense call, and two heads against the
    oracle."""
    w = syn.workloads()["packed16_8192"]
    x = syn.draw(w)
    rng = np.random.default_rng(24)
    slots = rng.permutation(64)[:w.N].astype(np.int32)
    slots[[3, 11]] = -1
    pool = make_pool(64, w.H, seed=6)
    pool_t = to_dev(pool)
    out = slots_call(inputs_to_dev(x), w.cu_seqlens(), slots, pool_t)
    check_against_dense(w, x, list(slots), pool, out, pool_t)
    heads = [0, 17]
    o_ref, pool_ref, _ = oracle.run_slots(x["q"], x["k"], x["v"], x["g"], x["beta"], w.cu_seqlens(),
                                          slots, pool[:, heads], heads=heads)
    cu = w.cu_seqlens()
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in live(slots, 64)])
    assert rel_l2(out_to_f64(out)[rows][:, heads], o_ref[rows]) <= OUT_TOL
    named = slots[slots >= 0]
    assert rel_l2(pool_t.cpu().numpy()[named][:, heads], pool_ref[named]) <= STATE_TOL


def test_slots_pool_carries_state_across_calls_bitwise():
    """Sequences split into two calls at multiples of 64 rows, sharing the pool,
    give the bits of one call (the carried state stays fp32)."""
    t = torch()
    lens = [256, 130, 64]
    cut = [128, 64, 64]
    slots = [2, 0, 5]
    w = syn.Workload("carry", lens, H=4, dk=128, dv=128, seed=25)
    x = syn.draw(w)
    pool = make_pool(6, 4, seed=7)
    one = to_dev(pool)
    out_one = slots_call(inputs_to_dev(x), w.cu_seqlens(), slots, one)
    two = to_dev(pool)
    out_two = t.full_like(out_one, float("nan"))
    cu = w.cu_seqlens()
    for first in (True, False):
        rows, sub = [], []
        for n in range(len(lens)):
            lo, hi = (cu[n], cu[n] + cut[n]) if first else (cu[n] + cut[n], cu[n + 1])
            rows.append(np.arange(lo, hi))
            sub.append(hi - lo)
        rows = np.concatenate(rows)
        part = inputs_to_dev({k: v[rows] for k, v in x.items()})
        sub_cu = np.concatenate([[0], np.cumsum(sub)]).astype(np.int32)
        o = slots_call(part, sub_cu, slots, two)
        out_two[t.from_numpy(rows).cuda()] = o
    assert t.equal(out_one, out_two)
    assert t.equal(one, two)
