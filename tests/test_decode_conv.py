"""The decode step with the short conv fused in front of it (kda_decode_conv)
on the GPU against the oracle's prologue feeding the oracle's recurrence
(kern-k3-pp-prefill README, section "D inside SGLang": the decode step runs
the conv on the step's rows with the windows in the engine's pool, then the
recurrence on the slot-addressed states).  The fused kernel keeps q, k and v in
fp32 between the two, so the oracle's are not rounded either.  Tolerances as
for the decode step; the windows are copies of input rows and must match bit
for bit."""
import numpy as np
import pytest

import oracle
from gpu_util import OUT_TOL, STATE_TOL, rel_l2, to_dev, torch
from test_conv import bf16_bits, dev_bf16, host_bits

import kda_linear_attention_chunk_gb300 as kda

pytestmark = pytest.mark.gpu


def draw(N, H, num_slots, conv_num_slots, seed):
    rng = np.random.default_rng(seed)
    xs = [bf16_bits(rng.standard_normal((N, H, 128))) for _ in range(3)]
    w = (0.5 * rng.standard_normal((3, H * 128, 4))).astype(np.float32)
    cpool = bf16_bits(rng.standard_normal((conv_num_slots, 3, 3, H * 128)))
    g = (-0.2 * rng.random((N, H, 128))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))).astype(np.float32)
    pool = (0.02 * rng.standard_normal((num_slots, H, 128, 128))).astype(np.float32)
    return xs, w, cpool, g, beta, pool


def reference(xs, w, cpool, g, beta, pool, conv_slots, state_slots, activation="silu", eps=1e-6):
    """The oracle chain; a row is skipped when either of its ids is -1 or bad."""
    N = xs[0].shape[0]
    cu = np.arange(N + 1, dtype=np.int32)
    cs, ss = np.array(conv_slots, dtype=np.int64), np.array(state_slots, dtype=np.int64)
    dead = (cs < 0) | (cs >= cpool.shape[0]) | (ss < 0) | (ss >= pool.shape[0])
    cs[dead], ss[dead] = -1, -1
    (q, k, v), new_cpool, _ = oracle.short_conv(*xs, w, cu, cpool, cs, activation=activation, eps=eps)
    out, new_pool, _ = oracle.run_slots(q, k, v, g, beta, cu, ss, pool)
    return out, new_pool, new_cpool, dead


def run_gpu(xs, w, cpool, g, beta, pool, conv_slots, state_slots, activation="silu", eps=1e-6):
    t = torch()
    x_t = [dev_bf16(x) for x in xs]
    cpool_t, pool_t = dev_bf16(cpool), to_dev(pool)
    cs = None if conv_slots is None else t.from_numpy(np.asarray(conv_slots, dtype=np.int32)).cuda()
    ss = None if state_slots is None else t.from_numpy(np.asarray(state_slots, dtype=np.int32)).cuda()
    out = t.full(xs[0].shape, float("nan"), dtype=t.bfloat16, device="cuda")
    kda.decode_conv(*x_t, t.from_numpy(w).cuda(), cpool_t, to_dev(g), to_dev(beta), pool_t, conv_slots=cs,
                    state_slots=ss, activation=activation, eps=eps, out=out)
    t.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), pool_t.cpu().numpy(), host_bits(cpool_t)


@pytest.mark.parametrize("activation", ["silu", "none"])
def test_decode_conv_parity_with_padding(activation):
    N, H = 37, 3
    xs, w, cpool, g, beta, pool = draw(N, H, num_slots=45, conv_num_slots=41, seed=31)
    rng = np.random.default_rng(31)
    conv_slots = rng.permutation(41)[:N].astype(np.int32)
    state_slots = rng.permutation(45)[:N].astype(np.int32)
    conv_slots[4], state_slots[9] = -1, -1
    kda.device_error(reset=True)
    out, new_pool, new_cpool = run_gpu(xs, w, cpool, g, beta, pool, conv_slots, state_slots, activation)
    assert kda.device_error(reset=True) == 0
    ref_out, ref_pool, ref_cpool, dead = reference(xs, w, cpool, g, beta, pool, conv_slots, state_slots, activation)
    assert dead.sum() == 2
    assert np.isnan(out[dead]).all()                     # skipped rows are not written
    assert rel_l2(out[~dead], ref_out[~dead]) <= OUT_TOL
    live_states = state_slots[~dead]
    assert rel_l2(new_pool[live_states], ref_pool[live_states]) <= STATE_TOL
    untouched = np.setdiff1d(np.arange(45), live_states)
    np.testing.assert_array_equal(new_pool[untouched], pool[untouched])
    np.testing.assert_array_equal(new_cpool, ref_cpool)  # windows: bit for bit, untouched entries included


def test_decode_conv_bad_ids_reported_and_skipped():
    N, H = 6, 2
    xs, w, cpool, g, beta, pool = draw(N, H, num_slots=6, conv_num_slots=6, seed=32)
    conv_slots = np.array([0, 9, 2, 3, 4, 5], dtype=np.int32)
    state_slots = np.array([5, 4, 3, -7, 1, 0], dtype=np.int32)
    kda.device_error(reset=True)
    out, new_pool, new_cpool = run_gpu(xs, w, cpool, g, beta, pool, conv_slots, state_slots)
    assert kda.device_error(reset=True) & kda.ERR_BAD_SLOT
    ref_out, ref_pool, ref_cpool, dead = reference(xs, w, cpool, g, beta, pool, conv_slots, state_slots)
    assert list(np.flatnonzero(dead)) == [1, 3]
    assert np.isnan(out[dead]).all()
    assert rel_l2(out[~dead], ref_out[~dead]) <= OUT_TOL
    np.testing.assert_array_equal(new_cpool, ref_cpool)
    assert rel_l2(new_pool, ref_pool) <= STATE_TOL


def test_decode_conv_dense_entries_without_tables():
    N, H = 5, 1
    xs, w, cpool, g, beta, pool = draw(N, H, num_slots=5, conv_num_slots=5, seed=33)
    out, new_pool, new_cpool = run_gpu(xs, w, cpool, g, beta, pool, None, None, activation="none", eps=0.0)
    ref_out, ref_pool, ref_cpool, _ = reference(xs, w, cpool, g, beta, pool, np.arange(N), np.arange(N),
                                                activation="none", eps=0.0)
    assert rel_l2(out, ref_out) <= OUT_TOL
    assert rel_l2(new_pool, ref_pool) <= STATE_TOL
    np.testing.assert_array_equal(new_cpool, ref_cpool)


def test_prefill_prologue_then_fused_decode_steps():
    """A prompt through kda_short_conv and kda_chunk_prefill_slots, then three
    fused decode steps on the same two pools: the windows equal the oracle's
    conv over the prompt and the three tokens, bit for bit, and the states and
    outputs follow the oracle chain (the prompt's q, k, v rounded to bf16 as the
    prefill path stores them)."""
    t = torch()
    lens = [70, 3, 129]
    N, H, steps = len(lens), 2, 3
    rng = np.random.default_rng(34)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    xs = [bf16_bits(rng.standard_normal((T, H, 128))) for _ in range(3)]
    xd = [[bf16_bits(rng.standard_normal((N, H, 128))) for _ in range(3)] for _ in range(steps)]
    w = (0.5 * rng.standard_normal((3, H * 128, 4))).astype(np.float32)
    cpool = bf16_bits(rng.standard_normal((5, 3, 3, H * 128)))
    pool = (0.02 * rng.standard_normal((4, H, 128, 128))).astype(np.float32)
    g = (-0.2 * rng.random((T, H, 128))).astype(np.float32)
    beta = rng.random((T, H)).astype(np.float32)
    gd = [(-0.2 * rng.random((N, H, 128))).astype(np.float32) for _ in range(steps)]
    bd = [rng.random((N, H)).astype(np.float32) for _ in range(steps)]
    cslots, sslots = np.array([4, 0, 2], dtype=np.int32), np.array([1, 3, 0], dtype=np.int32)
    # GPU
    cpool_t, pool_t = dev_bf16(cpool), to_dev(pool)
    cs_t, ss_t = (t.from_numpy(a).cuda() for a in (cslots, sslots))
    w_t = t.from_numpy(w).cuda()
    q, k, v = kda.short_conv(*[dev_bf16(x) for x in xs], w_t, t.from_numpy(cu).cuda(), cpool_t, conv_slots=cs_t)
    kda.chunk_prefill_slots(q, k, v, to_dev(g), to_dev(beta), t.from_numpy(cu).cuda(), ss_t, pool_t)
    outs = [kda.decode_conv(*[dev_bf16(x) for x in xd[i]], w_t, cpool_t, to_dev(gd[i]), to_dev(bd[i]), pool_t,
                            conv_slots=cs_t, state_slots=ss_t) for i in range(steps)]
    t.cuda.synchronize()
    # oracle: the prompt's prologue (rounded to bf16, as stored) and recurrence,
    # then each step's prologue (fp32 in the fused kernel: not rounded) and step
    (qr, kr, vr), cp, _ = oracle.short_conv(*xs, w, cu, cpool, cslots)
    qb, kb, vb = (bf16_bits(a.astype(np.float32)) for a in (qr, kr, vr))
    _, sp, _ = oracle.run_slots(qb, kb, vb, g, beta, cu, sslots, pool)
    cud = np.arange(N + 1, dtype=np.int32)
    for i in range(steps):
        (qd, kd, vd), cp, _ = oracle.short_conv(*xd[i], w, cud, cp, cslots)
        o_ref, sp, _ = oracle.run_slots(qd, kd, vd, gd[i], bd[i], cud, sslots, sp)
        assert rel_l2(outs[i].float().cpu().numpy(), o_ref) <= OUT_TOL
    np.testing.assert_array_equal(host_bits(cpool_t), cp)
    assert rel_l2(pool_t.cpu().numpy()[sslots], sp[sslots]) <= STATE_TOL


def test_decode_conv_64_sequences_h32():
    """The decode workload's shape: 64 sequences x 32 heads in pools of 128."""
    N, H = 64, 32
    xs, w, cpool, g, beta, pool = draw(N, H, num_slots=128, conv_num_slots=128, seed=35)
    slots = np.arange(1, 128, 2, dtype=np.int32)
    out, new_pool, new_cpool = run_gpu(xs, w, cpool, g, beta, pool, slots, slots[::-1].copy())
    ref_out, ref_pool, ref_cpool, _ = reference(xs, w, cpool, g, beta, pool, slots, slots[::-1].copy())
    assert rel_l2(out, ref_out) <= OUT_TOL
    assert rel_l2(new_pool[slots], ref_pool[slots]) <= STATE_TOL
    np.testing.assert_array_equal(new_cpool, ref_cpool)
