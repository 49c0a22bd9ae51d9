"""Bit-exact indexing and edge cases on the GPU (through the C ABI binding).

The kernel's arithmetic for one (sequence, head) does not depend on its
neighbours, so packing, ordering and the split of a context into calls must
not change a single bit of the results."""
import numpy as np
import pytest

from gpu_util import inputs_to_dev, oracle_run, out_to_f64, rel_l2, run_gpu, to_dev, torch, OUT_TOL
from kda_linear_attention_chunk_gb300 import synthetic as syn
import kda_linear_attention_chunk_gb300 as kda

pytestmark = pytest.mark.gpu

LENS = [1, 64, 65, 200, 0, 37, 128, 3]


def case(lens=LENS, H=4, seed=7, init=True):
    w = syn.Workload("idx", lens, H=H, dk=128, dv=128, init_state=init, seed=seed)
    return w, syn.draw(w), syn.draw_initial_state(w)


def packed_run(w, x, s0):
    out, fin = run_gpu(inputs_to_dev(x), w.cu_seqlens(), s0=to_dev(s0))
    torch().cuda.synchronize()
    return out, fin


@pytest.mark.parametrize("split", ["0", "full", "half"])
def test_each_sequence_alone_equals_packed_bitwise(split, monkeypatch):
    # the fused kernel, or split mode (one or two chain CTAs a unit) wherever a call allows it
    monkeypatch.setenv("KDA_SPLIT", split)
    w, x, s0 = case()
    out, fin = packed_run(w, x, s0)
    cu = w.cu_seqlens()
    for n, L in enumerate(w.lengths):
        xn = {k: v[cu[n]:cu[n + 1]] for k, v in x.items()}
        wn = syn.Workload("one", [L], H=w.H, dk=128, dv=128)
        o1, f1 = packed_run(wn, xn, s0[n:n + 1])
        if L:
            assert torch().equal(o1, out[cu[n]:cu[n + 1]]), f"sequence {n}"
        assert torch().equal(f1[0], fin[n]), f"state {n}"


@pytest.mark.parametrize("split", ["0", "full", "half"])
def test_sequence_order_permutation_bitwise(split, monkeypatch):
    monkeypatch.setenv("KDA_SPLIT", split)
    w, x, s0 = case()
    out, fin = packed_run(w, x, s0)
    cu = w.cu_seqlens()
    perm = [3, 0, 7, 5, 1, 6, 2, 4]
    xs = {k: np.concatenate([v[cu[p]:cu[p + 1]] for p in perm]) for k, v in x.items()}
    wp = syn.Workload("perm", [w.lengths[p] for p in perm], H=w.H, dk=128, dv=128)
    op, fp = packed_run(wp, xs, s0[perm])
    cup = wp.cu_seqlens()
    for i, p in enumerate(perm):
        assert torch().equal(op[cup[i]:cup[i + 1]], out[cu[p]:cu[p + 1]])
        assert torch().equal(fp[i], fin[p])


def test_canaries_every_row_written_and_guard_untouched():
    t = torch()
    w, x, s0 = case()
    T, H = w.T, w.H
    guard = 64
    big = t.full((T + guard, H, 128), float("nan"), dtype=t.bfloat16, device="cuda")
    fin = t.full((w.N + 1, H, 128, 128), float("nan"), dtype=t.float32, device="cuda")
    run_gpu(inputs_to_dev(x), w.cu_seqlens(), s0=to_dev(s0), out=big[:T], final_state=fin[:w.N])
    t.cuda.synchronize()
    assert not t.isnan(big[:T].float()).any()
    assert t.isnan(big[T:].float()).all()
    assert not t.isnan(fin[:w.N]).any()
    assert t.isnan(fin[w.N:]).all()


def test_zero_length_sequences_copy_state():
    t = torch()
    w, x, s0 = case(lens=[0, 5, 0], H=2)
    out, fin = packed_run(w, x, s0)
    assert t.equal(fin[0].cpu(), t.from_numpy(s0[0])) and t.equal(fin[2].cpu(), t.from_numpy(s0[2]))
    w2, x2, _ = case(lens=[0, 5, 0], H=2, init=False)
    _, fin2 = packed_run(w2, x2, None)
    assert t.count_nonzero(fin2[0]) == 0 and t.count_nonzero(fin2[2]) == 0


def test_all_empty_call():
    t = torch()
    w = syn.Workload("empty", [0, 0], H=2, dk=128, dv=128, init_state=True)
    s0 = syn.draw_initial_state(w)
    empty = {k: t.empty((0, 2, 128) if k != "beta" else (0, 2),
                        dtype=t.bfloat16 if k in "qkv" else t.float32, device="cuda")
             for k in ("q", "k", "v", "g", "beta")}
    out, fin = run_gpu(empty, w.cu_seqlens(), s0=to_dev(s0))
    t.cuda.synchronize()
    assert t.equal(fin.cpu(), t.from_numpy(s0))


def test_deterministic_and_zero_initial_equals_null():
    t = torch()
    w, x, _ = case(init=False)
    d = inputs_to_dev(x)
    o1, f1 = run_gpu(d, w.cu_seqlens())
    o2, f2 = run_gpu(d, w.cu_seqlens(), s0=t.zeros((w.N, w.H, 128, 128), device="cuda"))
    o3, f3 = run_gpu(d, w.cu_seqlens())
    t.cuda.synchronize()
    assert t.equal(o1, o3) and t.equal(f1, f3)
    assert t.equal(o1, o2) and t.equal(f1, f2)


def test_in_place_state_update_and_null_final_state():
    t = torch()
    w, x, s0 = case()
    d = inputs_to_dev(x)
    o1, f1 = run_gpu(d, w.cu_seqlens(), s0=to_dev(s0))
    st = to_dev(s0)
    o2, f2 = run_gpu(d, w.cu_seqlens(), s0=st, final_state=st)
    o3, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"],
                              t.from_numpy(w.cu_seqlens()).cuda(), initial_state=to_dev(s0),
                              output_final_state=False)
    t.cuda.synchronize()
    assert t.equal(o1, o2) and t.equal(f1, st) and t.equal(o1, o3)


def test_side_stream():
    t = torch()
    w, x, s0 = case()
    d = inputs_to_dev(x)
    o1, f1 = run_gpu(d, w.cu_seqlens(), s0=to_dev(s0))
    s = t.cuda.Stream()
    with t.cuda.stream(s):
        o2, f2 = run_gpu(d, w.cu_seqlens(), s0=to_dev(s0), stream=s)
    s.synchronize()
    t.cuda.synchronize()
    assert t.equal(o1, o2) and t.equal(f1, f2)


@pytest.mark.parametrize("one_mode,chain_mode", [("", ""), ("full", "0"), ("0", "half"), ("half", "full")])
def test_chained_calls_equal_single_call_bitwise(one_mode, chain_mode, monkeypatch):
    """A context split into calls of 8192 rows (a multiple of the 64-row chunk)
    with the fp32 state carried gives the same bits as one call -- also with the
    one call in split mode and the chained calls on the fused kernel, the other
    way round, and with half chains against whole ones."""
    t = torch()
    w = syn.Workload("chain", [4 * 8192], H=4, dk=128, dv=128, seed=11)
    x = syn.draw(w)
    d = inputs_to_dev(x)
    if one_mode:
        monkeypatch.setenv("KDA_SPLIT", one_mode)
    o_one, f_one = run_gpu(d, w.cu_seqlens())
    if chain_mode:
        monkeypatch.setenv("KDA_SPLIT", chain_mode)
    cu = t.tensor([0, 8192], dtype=t.int32, device="cuda")
    state = None
    for c in range(4):
        part = {k: v[c * 8192:(c + 1) * 8192].contiguous() for k, v in d.items()}
        o, state = run_gpu(part, cu, s0=state)
        assert t.equal(o, o_one[c * 8192:(c + 1) * 8192]), f"call {c}"
    assert t.equal(state, f_one)


def test_bad_cu_seqlens_stay_in_bounds():
    """A table that breaks its contract is clamped: no fault, the guard region
    stays untouched, and the device error word reports it."""
    t = torch()
    w, x, s0 = case(lens=[40, 40], H=2)
    kda.device_error(reset=True)
    big = t.full((w.T + 64, 2, 128), float("nan"), dtype=t.bfloat16, device="cuda")
    bad = t.tensor([0, 100000, 80], dtype=t.int32, device="cuda")
    run_gpu(inputs_to_dev(x), bad, s0=to_dev(s0), out=big[:w.T])
    t.cuda.synchronize()
    assert t.isnan(big[w.T:].float()).all()
    assert kda.device_error(reset=True) & 2


def test_many_units_per_cta_equal_each_sequence_alone_bitwise():
    """More (sequence, head) units than CTAs, so every CTA changes units
    several times -- the finished unit's state leaves TMEM and the next one's
    initial state comes in -- with initial states and ragged lengths: every
    sampled sequence must come out exactly as in a call of its own (one unit a
    CTA, no change)."""
    t = torch()
    rng = np.random.default_rng(61)
    lens = [int(x) for x in rng.integers(1, 300, size=120)]
    lens[7] = 0
    lens[50] = 64
    w, x, s0 = case(lens=lens, H=4, seed=61)   # 480 units on at most 152 CTAs
    out, fin = packed_run(w, x, s0)
    cu = w.cu_seqlens()
    for n in [0, 1, 7, 13, 50, 64, 99, 119]:
        L = w.lengths[n]
        xn = {k: v[cu[n]:cu[n + 1]] for k, v in x.items()}
        wn = syn.Workload("one", [L], H=w.H, dk=128, dv=128)
        o1, f1 = packed_run(wn, xn, s0[n:n + 1])
        if L:
            assert t.equal(o1, out[cu[n]:cu[n + 1]]), f"sequence {n}"
        assert t.equal(f1[0], fin[n]), f"state {n}"
