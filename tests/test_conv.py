"""The short-conv + L2-norm prologue on the GPU (kda_short_conv) against the
oracle: ragged packed batches with windows in a slot-addressed pool, padding
and bad ids, chained calls, and the packed 8192-row workload at H = 32
(kern-k3-pp-prefill README, sections "P: the packed prefill" and "D inside
SGLang").  Outputs are bf16, so the bound is relative L2 2e-3 (bf16 rounding
alone leaves about 1.1e-3); the windows are copies of input rows and must
match bit for bit."""
import numpy as np
import pytest

import oracle
from gpu_util import rel_l2, torch

import kda_linear_attention_chunk_gb300 as kda

pytestmark = pytest.mark.gpu

CONV_TOL = 2e-3


def bf16_bits(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def draw(lens, H, num_slots, seed, scale=1.0):
    """Projections ~ N(0, scale^2), filters ~ N(0, 0.5^2), windows ~ N(0, scale^2)."""
    rng = np.random.default_rng(seed)
    T = int(sum(lens))
    xs = [bf16_bits(scale * rng.standard_normal((T, H, 128))) for _ in range(3)]
    w = (0.5 * rng.standard_normal((3, H * 128, 4))).astype(np.float32)
    pool = bf16_bits(scale * rng.standard_normal((num_slots, 3, 3, H * 128)))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return xs, w, pool, cu


def dev_bf16(bits):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t.bfloat16).cuda()


def host_bits(tensor):
    return tensor.view(torch().int16).cpu().numpy().view(np.uint16)


def gpu_conv(xs, w, pool_t, cu, slots=None, activation="silu", eps=1e-6, fill=float("nan")):
    t = torch()
    T, H = xs[0].shape[:2]
    x_t = [dev_bf16(x) for x in xs]
    outs = tuple(t.full((T, H, 128), fill, dtype=t.bfloat16, device="cuda") for _ in range(3))
    sl = None if slots is None else t.from_numpy(np.asarray(slots, dtype=np.int32)).cuda()
    kda.short_conv(*x_t, t.from_numpy(w).cuda(), t.from_numpy(cu).cuda(), pool_t, conv_slots=sl,
                   activation=activation, eps=eps, out=outs)
    t.cuda.synchronize()
    return [o.float().cpu().numpy().astype(np.float64) for o in outs]


@pytest.mark.parametrize("activation", ["silu", "none"])
def test_conv_parity_ragged(activation):
    lens = [0, 1, 2, 3, 5, 64, 70, 129, 33, 31, 32]
    H, num_slots = 3, 16
    xs, w, pool, cu = draw(lens, H, num_slots, seed=11)
    rng = np.random.default_rng(11)
    slots = rng.permutation(num_slots)[:len(lens)].astype(np.int32)
    slots[6] = -1
    pool_t = dev_bf16(pool)
    kda.device_error(reset=True)
    got = gpu_conv(xs, w, pool_t, cu, slots, activation=activation)
    assert kda.device_error(reset=True) == 0
    ref, new_pool, bad = oracle.short_conv(*xs, w, cu, pool, slots, activation=activation)
    assert bad == []
    live = ~np.isnan(ref[0][:, 0, 0])
    assert live.sum() == sum(lens) - lens[6]
    for g, r in zip(got, ref):
        assert np.isnan(g[~live]).all()                # padded rows are not written
        assert rel_l2(g[live], r[live]) <= CONV_TOL
    np.testing.assert_array_equal(host_bits(pool_t), new_pool)


def test_conv_chained_calls_equal_one_call_bit_for_bit():
    lens = [40, 3, 97, 1]
    H, num_slots = 2, 6
    xs, w, pool, cu = draw(lens, H, num_slots, seed=12)
    slots = np.array([4, 1, 0, 5], dtype=np.int32)
    t = torch()
    pool_a = dev_bf16(pool)
    whole = gpu_conv(xs, w, pool_a, cu, slots)
    cut = [n // 3 for n in lens]
    first = np.concatenate([np.arange(cu[i], cu[i] + cut[i]) for i in range(len(lens))])
    second = np.concatenate([np.arange(cu[i] + cut[i], cu[i + 1]) for i in range(len(lens))])
    cu1 = np.concatenate([[0], np.cumsum(cut)]).astype(np.int32)
    cu2 = np.concatenate([[0], np.cumsum([lens[i] - cut[i] for i in range(len(lens))])]).astype(np.int32)
    pool_b = dev_bf16(pool)
    a = gpu_conv([x[first] for x in xs], w, pool_b, cu1, slots)
    b = gpu_conv([x[second] for x in xs], w, pool_b, cu2, slots)
    for s in range(3):
        np.testing.assert_array_equal(whole[s][first], a[s])
        np.testing.assert_array_equal(whole[s][second], b[s])
    assert t.equal(pool_a, pool_b)


def test_conv_bad_ids_reported_and_skipped():
    lens = [5, 6, 7]
    H, num_slots = 2, 3
    xs, w, pool, cu = draw(lens, H, num_slots, seed=13)
    slots = np.array([0, 7, 2], dtype=np.int32)
    pool_t = dev_bf16(pool)
    kda.device_error(reset=True)
    got = gpu_conv(xs, w, pool_t, cu, slots)
    assert kda.device_error(reset=True) & kda.ERR_BAD_SLOT
    ref, new_pool, bad = oracle.short_conv(*xs, w, cu, pool, slots)
    assert bad == [1]
    assert np.isnan(got[0][5:11]).all()
    live = np.r_[0:5, 11:18]
    for g, r in zip(got, ref):
        assert rel_l2(g[live], r[live]) <= CONV_TOL
    np.testing.assert_array_equal(host_bits(pool_t), new_pool)


def test_conv_dense_entries_without_a_table():
    lens = [17, 0, 45]
    H = 1
    xs, w, pool, cu = draw(lens, H, 3, seed=14)
    pool_t = dev_bf16(pool)
    got = gpu_conv(xs, w, pool_t, cu, None, activation="none", eps=0.0)
    ref, new_pool, _ = oracle.short_conv(*xs, w, cu, pool, None, activation="none", eps=0.0)
    for g, r in zip(got, ref):
        assert rel_l2(g, r) <= CONV_TOL
    np.testing.assert_array_equal(host_bits(pool_t), new_pool)


def test_conv_packed16_8192_h32():
    """The packed 8192-row workload's lengths at H = 32 (16 sequences)."""
    lens = [90, 45, 1397, 48, 1088, 385, 352, 1002, 1334, 209, 317, 563, 50, 154, 667, 491]
    H, num_slots = 32, 32
    xs, w, pool, cu = draw(lens, H, num_slots, seed=15)
    slots = np.arange(0, 32, 2, dtype=np.int32)
    pool_t = dev_bf16(pool)
    got = gpu_conv(xs, w, pool_t, cu, slots)
    ref, new_pool, _ = oracle.short_conv(*xs, w, cu, pool, slots)
    for g, r in zip(got, ref):
        assert rel_l2(g, r) <= CONV_TOL
    np.testing.assert_array_equal(host_bits(pool_t), new_pool)


@pytest.mark.parametrize("seed", [16, 17, 18])
def test_conv_short_sequences_at_every_block_offset(seed):
    """Many sequences of 1 to 6 rows among longer ones, so that sequences start
    at (nearly) every offset within the kernel's 64-row blocks, the last three
    rows before a block edge included (a sequence starting there has its
    window read by the warp of the earlier block only)."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(1, 7, 200)]
    for pos in (10, 60, 120, 170):
        lens[pos] = int(rng.integers(30, 140))
    H = 2
    num_slots = len(lens) + 5
    xs, w, pool, cu = draw(lens, H, num_slots, seed=seed)
    slots = rng.permutation(num_slots)[:len(lens)].astype(np.int32)
    pool_t = dev_bf16(pool)
    got = gpu_conv(xs, w, pool_t, cu, slots)
    ref, new_pool, _ = oracle.short_conv(*xs, w, cu, pool, slots)
    for g, r in zip(got, ref):
        assert rel_l2(g, r) <= CONV_TOL
    np.testing.assert_array_equal(host_bits(pool_t), new_pool)


def test_conv_then_prefill_matches_the_oracle_chain():
    """The prologue's q, k, v fed to the prefill (as a layer runs them) against
    the oracle's prologue, rounded to bf16, fed to the oracle's recurrence."""
    from gpu_util import OUT_TOL, STATE_TOL, to_dev
    t = torch()
    lens = [70, 1, 130, 5, 64]
    H = 2
    xs, w, pool, cu = draw(lens, H, len(lens), seed=19)
    rng = np.random.default_rng(19)
    T = int(cu[-1])
    g = (-0.2 * rng.random((T, H, 128))).astype(np.float32)
    beta = rng.random((T, H)).astype(np.float32)
    s0 = (0.02 * rng.standard_normal((len(lens), H, 128, 128))).astype(np.float32)
    pool_t = dev_bf16(pool)
    x_t = [dev_bf16(x) for x in xs]
    q, k, v = kda.short_conv(*x_t, t.from_numpy(w).cuda(), t.from_numpy(cu).cuda(), pool_t, activation="silu")
    out, fin = kda.chunk_prefill(q, k, v, to_dev(g), to_dev(beta), t.from_numpy(cu).cuda(),
                                 initial_state=to_dev(s0))
    t.cuda.synchronize()
    (qr, kr, vr), _, _ = oracle.short_conv(*xs, w, cu, pool, None, activation="silu")
    qb, kb, vb = (bf16_bits(a.astype(np.float32)) for a in (qr, kr, vr))
    o_ref, f_ref = oracle.run(qb, kb, vb, g, beta, cu, initial_state=s0)
    assert rel_l2(out.float().cpu().numpy(), o_ref) <= OUT_TOL
    assert rel_l2(fin.cpu().numpy(), f_ref) <= STATE_TOL
    from gpu_util import check_elementwise
    check_elementwise(out.float().cpu().numpy(), o_ref, "tc_out")
    check_elementwise(fin.cpu().numpy(), f_ref, "tc_state_prologue")


@pytest.mark.parametrize("pattern", ["one_row", "about_20_rows"])
def test_conv_short_blocks_for_short_sequences(pattern):
    """Short mean lengths run in short row blocks (4 rows per warp for one-row
    sequences, 16 for about 20): parity, padding and windows as for long ones."""
    rng = np.random.default_rng(20 if pattern == "one_row" else 21)
    lens = [1] * 64 if pattern == "one_row" else [int(x) for x in rng.integers(1, 40, 50)]
    H = 4
    num_slots = len(lens) + 3
    xs, w, pool, cu = draw(lens, H, num_slots, seed=22)
    slots = rng.permutation(num_slots)[:len(lens)].astype(np.int32)
    slots[5] = -1
    pool_t = dev_bf16(pool)
    got = gpu_conv(xs, w, pool_t, cu, slots)
    ref, new_pool, _ = oracle.short_conv(*xs, w, cu, pool, slots)
    live = ~np.isnan(ref[0][:, 0, 0])
    for g, r in zip(got, ref):
        assert np.isnan(g[~live]).all()
        assert rel_l2(g[live], r[live]) <= CONV_TOL
    np.testing.assert_array_equal(host_bits(pool_t), new_pool)
