"""Pins for the oracle's slot-indexed form (no GPU).

The states of a serving engine live in a pool, [slot][head][v][k] fp32, and a
call names each sequence's entry by a slot id; -1 marks padding that is
skipped (kern-k3-pp-prefill README, section "D inside SGLang").  These pins
tie oracle.run_slots to properties the definition fixes, independently of how
run_slots routes the data: with the identity table it is the plain call; any
placement of the states in a larger pool gives the same outputs and moves
the final states with them; padded sequences leave their rows and the pool
alone without changing anyone else's result (the sequences are independent);
and a sequence split across two calls that share the pool equals one pass
(the state is carried through the pool, in place).
"""
import numpy as np
import pytest

import oracle

from test_oracle import random_case, rel_l2


def plain(case, **kw):
    return oracle.run(case["q"], case["k"], case["v"], case["g"], case["beta"], case["cu_seqlens"],
                      initial_state=case["initial_state"], **kw)


def slots_run(case, slots, pool, **kw):
    return oracle.run_slots(case["q"], case["k"], case["v"], case["g"], case["beta"],
                            case["cu_seqlens"], slots, pool, **kw)


@pytest.mark.parametrize("chunk", [0, 16])
def test_identity_table_is_the_plain_call(chunk):
    case = random_case([37, 64, 1, 90], H=2, dk=16, dv=8, seed=31)
    o, s = plain(case, chunk=chunk)
    o2, pool, bad = slots_run(case, np.arange(4), case["initial_state"], chunk=chunk)
    assert bad == []
    assert np.array_equal(o2, o) and np.array_equal(pool, s)


def test_states_placed_anywhere_in_a_larger_pool():
    lens = [50, 3, 128, 70, 0]
    case = random_case(lens, H=3, dk=8, dv=12, seed=32)
    o, s = plain(case)
    rng = np.random.default_rng(5)
    num_slots = 11
    slots = rng.permutation(num_slots)[:len(lens)]
    pool = rng.standard_normal((num_slots, 3, 12, 8))
    pool[slots] = case["initial_state"]
    o2, pool2, bad = slots_run(case, slots, pool)
    assert bad == []
    assert rel_l2(o2, o) <= 1e-14
    assert rel_l2(pool2[slots], s) <= 1e-14
    others = np.setdiff1d(np.arange(num_slots), slots)
    assert np.array_equal(pool2[others], pool[others])


def test_padded_sequences_are_skipped():
    lens = [40, 25, 64, 9]
    case = random_case(lens, H=2, dk=8, dv=8, seed=33)
    o, s = plain(case)
    cu = case["cu_seqlens"]
    slots = np.array([2, -1, 0, -1])
    pool = np.zeros((3, 2, 8, 8))
    pool[2], pool[0] = case["initial_state"][0], case["initial_state"][2]
    canary = np.full(o.shape, 7.25)
    o2, pool2, bad = slots_run(case, slots, pool, out=canary)
    assert bad == []
    for n in (1, 3):
        assert np.all(o2[cu[n]:cu[n + 1]] == 7.25)
    for n, sl in ((0, 2), (2, 0)):
        assert rel_l2(o2[cu[n]:cu[n + 1]], o[cu[n]:cu[n + 1]]) <= 1e-14
        assert rel_l2(pool2[sl], s[n]) <= 1e-14
    assert np.array_equal(pool2[1], pool[1])


def test_pool_carries_the_state_across_calls():
    """A sequence split at any row and run as two calls that share the pool
    equals one pass: the first call leaves the state in the slot, the second
    starts from it."""
    lens = [130, 77, 5]
    case = random_case(lens, H=2, dk=16, dv=16, seed=34)
    o, s = plain(case, chunk=64)
    cu = case["cu_seqlens"]
    cut = [61, 1, 5]   # rows of each sequence in the first call
    slots = np.array([4, 1, 2])
    pool = np.zeros((5, 2, 16, 16))
    pool[slots] = case["initial_state"]
    out = np.zeros(o.shape)
    for first in (True, False):
        rows, sub_lens = [], []
        for n in range(len(lens)):
            lo, hi = (cu[n], cu[n] + cut[n]) if first else (cu[n] + cut[n], cu[n + 1])
            rows.append(np.arange(lo, hi))
            sub_lens.append(hi - lo)
        rows = np.concatenate(rows)
        part = {key: case[key][rows] for key in ("q", "k", "v", "g", "beta")}
        part["cu_seqlens"] = np.concatenate([[0], np.cumsum(sub_lens)]).astype(np.int32)
        o_part, pool, bad = slots_run(part, slots, pool, chunk=64)
        assert bad == []
        out[rows] = o_part
    assert rel_l2(out, o) <= 1e-13
    assert rel_l2(pool[slots], s) <= 1e-13


def test_out_of_range_ids_are_reported_and_skipped():
    case = random_case([10, 12, 6], H=1, dk=4, dv=4, seed=35)
    pool = np.ones((3, 1, 4, 4))
    o, pool2, bad = slots_run(case, [3, -2, 1], pool)
    assert bad == [0, 1]
    assert np.isnan(o[:22]).all() and not np.isnan(o[22:]).any()
    assert np.array_equal(pool2[[0, 2]], pool[[0, 2]])


def test_shared_slot_is_rejected():
    case = random_case([10, 12], H=1, dk=4, dv=4, seed=36)
    with pytest.raises(ValueError):
        slots_run(case, [1, 1], np.zeros((2, 1, 4, 4)))


# --------------------------------------------------------------------------
# Planted mistakes in a copy of run_slots must fail the pins above.
# --------------------------------------------------------------------------
SLOT_MUTANTS = {
    "write_back_by_sequence": ("pool[slots[live]] = fin", "pool[np.array(live)] = fin"),
    "gather_by_sequence": ("initial_state=pool[slots[live]]", "initial_state=pool[np.array(live)]"),
    "padding_wraps_to_last_slot": ("if 0 <= slots[n] < num_slots]", "if slots[n] < num_slots]"),
    "padding_rows_cleared": ("np.full((T, nsel, dv), np.nan) if out is None else np.array(out, dtype=np.float64)",
                             "np.zeros((T, nsel, dv))"),
}


def _variant(edit):
    import inspect
    src = inspect.getsource(oracle.run_slots)
    if edit is not None:
        assert edit[0] in src, edit[0]
        src = src.replace(*edit)
    ns = dict(vars(oracle))
    exec(compile(src, "<run_slots variant>", "exec"), ns)
    return ns["run_slots"]


def _battery(fn) -> bool:
    ok = True
    lens = [50, 3, 0, 70]
    case = random_case(lens, H=2, dk=8, dv=8, seed=41)
    o, s = plain(case)
    cu = case["cu_seqlens"]
    args = [case[n] for n in ("q", "k", "v", "g", "beta", "cu_seqlens")]
    # states placed in a larger pool, one sequence padded
    slots = np.array([5, 0, 2, -1])
    pool = np.random.default_rng(6).standard_normal((6, 2, 8, 8))
    pool[slots[:3]] = case["initial_state"][:3]
    o2, pool2, bad = fn(*args, slots, pool, out=np.full(o.shape, 3.5))
    ok &= bad == []
    ok &= bool(rel_l2(o2[:cu[3]], o[:cu[3]]) <= 1e-14 and np.all(o2[cu[3]:] == 3.5))
    ok &= bool(rel_l2(pool2[slots[:3]], s[:3]) <= 1e-14)
    ok &= bool(np.array_equal(pool2[[1, 3, 4]], pool[[1, 3, 4]]))
    return ok


def test_unmutated_run_slots_passes_the_battery():
    assert _battery(_variant(None))


@pytest.mark.parametrize("name", sorted(SLOT_MUTANTS))
def test_run_slots_mutant_is_caught(name):
    assert not _battery(_variant(SLOT_MUTANTS[name])), f"mutant {name} survived"
