"""kda_chunk_prefill_conv: the short-conv + L2-norm prologue fused into the
tensor-core prefill (kern-k3-pp-prefill README, "P: the packed prefill": the
KDA layers run with per-sequence conv windows and states; "D inside SGLang":
both live in the engine's pools under the same slot ids).

The reference chain is the oracle's: oracle.short_conv (fp64), its q, k, v
rounded to bf16 (the fused kernel rounds them in shared memory just as
kda_short_conv rounds its outputs), then the oracle's recurrence.  Outputs are
held to the tensor-core kernel's bound, states to its bound for inputs made by
the prologue (gpu_util: the delta rule predicts such rows well, and the
rounding of the state operand shows against a smaller state); the windows
are copies of input rows and must match bit for bit.  The fused call gives
the same bytes as kda_short_conv followed by kda_chunk_prefill_slots.
"""
import numpy as np
import pytest

import oracle
import kda_linear_attention_chunk_gb300 as kda
from gpu_util import (OUT_TOL, STATE_TOL, check_elementwise, rel_l2, sampled_heads, to_dev, torch)
from kda_linear_attention_chunk_gb300 import synthetic as syn
from test_conv import bf16_bits, dev_bf16, draw, host_bits

pytestmark = pytest.mark.gpu


def layer_inputs(lens, H, entries, seed):
    xs, w, pool, cu = draw(lens, H, entries, seed=seed)
    rng = np.random.default_rng(seed + 1000)
    T = int(cu[-1])
    g = (-0.2 * rng.random((T, H, 128))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))).astype(np.float32)
    spool = (0.02 * rng.standard_normal((entries, H, 128, 128))).astype(np.float32)
    return xs, w, pool, cu, g, beta, spool


def fused(xs, w, pool, cu, g, beta, spool, slots=None, activation="silu", fill=float("nan")):
    t = torch()
    T, H = xs[0].shape[:2]
    pool_t, spool_t = dev_bf16(pool), to_dev(spool)
    out = t.full((T, H, 128), fill, dtype=t.bfloat16, device="cuda")
    sl = None if slots is None else t.from_numpy(np.asarray(slots, dtype=np.int32)).cuda()
    kda.chunk_prefill_conv(*[dev_bf16(x) for x in xs], t.from_numpy(w).cuda(), to_dev(g), to_dev(beta),
                           t.from_numpy(cu).cuda(), pool_t, spool_t, slots=sl, activation=activation, out=out)
    t.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), spool_t.cpu().numpy(), host_bits(pool_t)


def oracle_chain(xs, w, pool, cu, g, beta, spool, slots=None, activation="silu", heads=None):
    (qr, kr, vr), new_pool, bad = oracle.short_conv(*xs, w, cu, pool, slots, activation=activation)
    qb, kb, vb = (bf16_bits(np.nan_to_num(a).astype(np.float32)) for a in (qr, kr, vr))
    sl = np.arange(len(cu) - 1) if slots is None else np.asarray(slots)
    hs = list(range(xs[0].shape[1])) if heads is None else list(heads)
    out, spool_ref, _ = oracle.run_slots(qb[:, hs], kb[:, hs], vb[:, hs], g[:, hs], beta[:, hs], cu, sl,
                                         spool[:, hs])
    return out, spool_ref, new_pool, bad


@pytest.mark.parametrize("activation", ["silu", "none"])
def test_fused_matches_the_oracle_chain(activation):
    lens = [70, 1, 130, 5, 64, 0, 200, 2, 3, 129]
    H = 3
    xs, w, pool, cu, g, beta, spool = layer_inputs(lens, H, len(lens), seed=31)
    kda.device_error(reset=True)
    out, spool_after, pool_after = fused(xs, w, pool, cu, g, beta, spool, activation=activation)
    assert kda.device_error(reset=True) == 0
    o_ref, s_ref, new_pool, _ = oracle_chain(xs, w, pool, cu, g, beta, spool, activation=activation)
    assert rel_l2(out, o_ref) <= OUT_TOL and rel_l2(spool_after, s_ref) <= STATE_TOL
    check_elementwise(out, o_ref, "tc_out")
    check_elementwise(spool_after, s_ref, "tc_state_prologue")
    np.testing.assert_array_equal(pool_after, new_pool)


def test_fused_slots_padding_and_untouched_entries():
    lens = [40, 0, 3, 97, 1, 66, 2]
    H, entries = 2, 12
    xs, w, pool, cu, g, beta, spool = layer_inputs(lens, H, entries, seed=32)
    rng = np.random.default_rng(32)
    slots = rng.permutation(entries)[:len(lens)].astype(np.int32)
    slots[3] = -1
    out, spool_after, pool_after = fused(xs, w, pool, cu, g, beta, spool, slots=slots)
    o_ref, s_ref, new_pool, bad = oracle_chain(xs, w, pool, cu, g, beta, spool, slots=slots)
    assert bad == []
    live = ~np.isnan(o_ref[:, 0, 0])
    assert np.isnan(out[~live]).all()                           # padded rows are not written
    assert rel_l2(out[live], o_ref[live]) <= OUT_TOL
    named = slots[slots >= 0]
    assert rel_l2(spool_after[named], s_ref[named]) <= STATE_TOL
    others = np.setdiff1d(np.arange(entries), named)
    assert np.array_equal(spool_after[others], spool[others])   # padded and unnamed entries untouched
    assert np.array_equal(spool_after[slots[1]], spool[slots[1]])   # an empty sequence leaves its entry
    np.testing.assert_array_equal(pool_after, new_pool)


def test_fused_equals_the_two_calls():
    """The same layer as kda_short_conv followed by kda_chunk_prefill_slots:
    the same bytes (the prologue's arithmetic is the same in both, in the same
    order), windows included."""
    t = torch()
    lens = [300, 17, 64, 129]
    H = 4
    xs, w, pool, cu, g, beta, spool = layer_inputs(lens, H, len(lens), seed=33)
    out, spool_after, pool_after = fused(xs, w, pool, cu, g, beta, spool)
    pool_t, spool_t = dev_bf16(pool), to_dev(spool)
    cu_t = t.from_numpy(cu).cuda()
    q, k, v = kda.short_conv(*[dev_bf16(x) for x in xs], t.from_numpy(w).cuda(), cu_t, pool_t)
    slots = t.arange(len(lens), dtype=t.int32, device="cuda")
    out2 = kda.chunk_prefill_slots(q, k, v, to_dev(g), to_dev(beta), cu_t, slots, spool_t)
    t.cuda.synchronize()
    assert np.array_equal(out, out2.float().cpu().numpy().astype(np.float64))
    assert np.array_equal(spool_after, spool_t.cpu().numpy())
    np.testing.assert_array_equal(pool_after, host_bits(pool_t))


def test_fused_chained_calls_equal_one_call_bit_for_bit():
    """A sequence cut at a multiple of 64 rows into two calls, window and state
    carried in the pools, gives the bytes of one call."""
    lens = [300]
    H = 2
    xs, w, pool, cu, g, beta, spool = layer_inputs(lens, H, 1, seed=34)
    one, s_one, p_one = fused(xs, w, pool, cu, g, beta, spool)
    cut = 192
    a = fused([x[:cut] for x in xs], w, pool, np.array([0, cut], np.int32), g[:cut], beta[:cut], spool)
    b = fused([x[cut:] for x in xs], w, a[2], np.array([0, 300 - cut], np.int32), g[cut:], beta[cut:], a[1])
    assert np.array_equal(np.concatenate([a[0], b[0]]), one)
    assert np.array_equal(b[1], s_one)
    np.testing.assert_array_equal(b[2], p_one)


def test_fused_packed16_8192_sampled_heads():
    """The production shape: the 16-sequence 8192-row chunk at H = 32."""
    w_ = syn.workloads()["packed16_8192"]
    lens = w_.lengths
    H = 32
    xs, w, pool, cu, g, beta, spool = layer_inputs(lens, H, len(lens), seed=35)
    out, spool_after, pool_after = fused(xs, w, pool, cu, g, beta, spool)
    hs = sampled_heads(w_, 3, salt=2)
    o_ref, s_ref, _, _ = oracle_chain(xs, w, pool, cu, g, beta, spool, heads=hs)
    assert rel_l2(out[:, hs], o_ref) <= OUT_TOL and rel_l2(spool_after[:, hs], s_ref) <= STATE_TOL
    check_elementwise(out[:, hs], o_ref, "tc_out")
    check_elementwise(spool_after[:, hs], s_ref, "tc_state_prologue")
    _, new_pool, _ = oracle.short_conv(*xs, w, cu, pool, None)
    np.testing.assert_array_equal(pool_after, new_pool)
