"""Pins for the fp64 CPU oracle (no GPU).

The pages print no KDA worked example, so the oracle is pinned against what
the mathematics fixes: exact rational brute force on tiny cases, closed forms
of the degenerate cases (beta = 0; alpha = 1 and beta = 0; one-hot keys,
which reduce to plain causal linear attention; a single token's rank-1
update), the delta-rule invariant, continuity of the state across calls,
linearity, equivariance, and agreement of two independent routes (token
recurrence and chunked WY form).  test_oracle_mutants.py plants mistakes in a
copy of the oracle and checks that these pins catch them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def random_case(lens, H, dk, dv, seed=0, init=True, g_lo=-0.2, unit_k=True):
    rng = np.random.default_rng(seed)
    T = int(sum(lens))
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = rng.uniform(g_lo, 0.0, (T, H, dk))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    s0 = 0.02 * rng.standard_normal((len(lens), H, dv, dk)) if init else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=cu, initial_state=s0)


def run(case, **kw):
    args = dict(case)
    args.update(kw)
    return oracle.run(**args)


# --------------------------------------------------------------------------
# P2: exact rational brute force -- the definition as explicit matrices
# --------------------------------------------------------------------------
def brute_force_exact(q, k, v, alpha, beta, s0):
    """S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T, o_t = S_t^T q_t,
    all in exact rational arithmetic with explicit dk x dk matrices."""
    T, dk = len(q), len(q[0])
    dv = len(v[0])
    S = [[Fraction(s0[c][j]) for j in range(dv)] for c in range(dk)]
    outs = []
    for t in range(T):
        E = [[(Fraction(1) if a == b else Fraction(0)) - beta[t] * k[t][a] * k[t][b]
              for b in range(dk)] for a in range(dk)]
        M = [[E[a][b] * alpha[t][b] for b in range(dk)] for a in range(dk)]   # (I - b k k^T) Diag(alpha)
        S = [[sum(M[a][b] * S[b][j] for b in range(dk)) + beta[t] * k[t][a] * v[t][j]
              for j in range(dv)] for a in range(dk)]
        outs.append([sum(S[a][j] * q[t][a] for a in range(dk)) for j in range(dv)])
    return outs, S


@pytest.mark.parametrize("route", [0, 1, 2, 4])
def test_p2_exact_brute_force(route):
    rng = np.random.default_rng(7)
    dk = dv = 3
    T = 6
    quarter = lambda: Fraction(int(rng.integers(-4, 5)), 4)
    q = [[quarter() for _ in range(dk)] for _ in range(T)]
    k = [[quarter() for _ in range(dk)] for _ in range(T)]
    v = [[quarter() for _ in range(dv)] for _ in range(T)]
    alpha = [[Fraction(int(rng.integers(1, 5)), 4) for _ in range(dk)] for _ in range(T)]
    beta = [Fraction(int(rng.integers(0, 5)), 4) for _ in range(T)]
    s0 = [[quarter() for _ in range(dv)] for _ in range(dk)]
    outs, S = brute_force_exact(q, k, v, alpha, beta, s0)

    f = lambda m: np.array([[float(x) for x in row] for row in m])
    qa, ka, va = (f(x)[:, None, :] for x in (q, k, v))
    ga = np.log(f(alpha))[:, None, :]
    ba = np.array([float(b) for b in beta])[:, None]
    init = f(s0).T[None, None]                               # [N][H][dv][dk]
    out, fin = oracle.run(qa, ka, va, ga, ba, [0, T], initial_state=init, chunk=route)
    exp_out = f(outs)
    exp_fin = f(S).T
    assert np.max(np.abs(out[:, 0, :] - exp_out)) <= 1e-14 * max(1.0, np.max(np.abs(exp_out)))
    assert np.max(np.abs(fin[0, 0] - exp_fin)) <= 1e-14 * max(1.0, np.max(np.abs(exp_fin)))


# --------------------------------------------------------------------------
# P1: chunked route == token recurrence (C = 1 is the recurrence itself)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
def test_p1_chunked_matches_recurrence(chunk):
    case = random_case([37, 1, 130, 64, 0, 95], H=2, dk=32, dv=24, seed=chunk)
    o_ref, s_ref = run(case)
    o, s = run(case, chunk=chunk)
    assert rel_l2(o, o_ref) <= 1e-12
    assert rel_l2(s, s_ref) <= 1e-12


def test_p1_full_width_chunk64():
    case = random_case([200, 77], H=1, dk=128, dv=128, seed=3)
    o_ref, s_ref = run(case)
    o, s = run(case, chunk=64)
    assert rel_l2(o, o_ref) <= 1e-12
    assert rel_l2(s, s_ref) <= 1e-12


def strong_gates(g, kind, rng):
    """Gate regimes beyond U[-0.2, 0]: U[-3, 0]; a few channels at -20 on
    every row (alpha ~ 2e-9); 5% of the entries positive, U[0, 0.5]."""
    g = np.array(g)
    if kind == "u3":
        return g * 15.0
    if kind == "alpha0":
        g[:, :, rng.choice(g.shape[2], 3, replace=False)] = -20.0
        return g
    pos = rng.uniform(size=g.shape) < 0.05
    g[pos] = rng.uniform(0.0, 0.5, size=int(pos.sum()))
    return g


@pytest.mark.parametrize("kind", ["u3", "alpha0", "mixed"])
@pytest.mark.parametrize("chunk", [16, 64])
def test_p1_chunked_matches_recurrence_for_strong_and_mixed_gates(kind, chunk):
    """P1 again where the per-pair decays exp(G_i - G_j) span hundreds of
    e-folds (or grow): the chunked route forms each one directly."""
    case = random_case([37, 130, 64, 95], H=2, dk=32, dv=24, seed=20 + chunk)
    case["g"] = strong_gates(case["g"], kind, np.random.default_rng(chunk))
    o_ref, s_ref = run(case)
    o, s = run(case, chunk=chunk)
    assert np.isfinite(o).all() and np.isfinite(s).all()
    assert rel_l2(o, o_ref) <= 1e-12
    assert rel_l2(s, s_ref) <= 1e-12


# --------------------------------------------------------------------------
# P3 / P4: beta = 0 leaves the state only decayed; alpha = 1 too: nothing moves
# --------------------------------------------------------------------------
@pytest.mark.parametrize("gates", ["u02", "u3", "alpha0", "mixed"])
@pytest.mark.parametrize("chunk", [0, 64])
def test_p3_beta_zero_only_decays(chunk, gates):
    case = random_case([90, 41], H=2, dk=16, dv=8, seed=5)
    if gates != "u02":
        case["g"] = strong_gates(case["g"], gates, np.random.default_rng(5))
    case["beta"][:] = 0.0
    o, s = run(case, chunk=chunk)
    cu, g, q, s0 = case["cu_seqlens"], case["g"], case["q"], case["initial_state"]
    for n in range(2):
        for h in range(2):
            G = np.cumsum(g[cu[n]:cu[n + 1], h], axis=0)                   # [L][dk]
            expect_o = (q[cu[n]:cu[n + 1], h] * np.exp(G)) @ s0[n, h].T      # [L][dv]
            expect_s = s0[n, h] * np.exp(G[-1])[None, :]                     # [dv][dk]
            assert rel_l2(o[cu[n]:cu[n + 1], h], expect_o) <= 1e-13
            assert rel_l2(s[n, h], expect_s) <= 1e-13


@pytest.mark.parametrize("chunk", [0, 16])
def test_p4_identity_step(chunk):
    case = random_case([50], H=1, dk=8, dv=8, seed=6)
    case["beta"][:] = 0.0
    case["g"][:] = 0.0
    o, s = run(case, chunk=chunk)
    s0 = case["initial_state"][0, 0]
    assert np.array_equal(s[0, 0], s0)
    np.testing.assert_allclose(o[:, 0], case["q"][:, 0] @ s0.T, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# P5: one-hot keys, zero state -> gated / plain causal linear attention
# --------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [0, 8])
@pytest.mark.parametrize("gated", [False, True])
def test_p5_one_hot_keys_linear_attention(chunk, gated):
    rng = np.random.default_rng(11)
    T, dk, dv = 24, 32, 5
    chans = rng.permutation(dk)[:T]
    k = np.zeros((T, 1, dk))
    k[np.arange(T), 0, chans] = 1.0
    q = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = rng.uniform(-0.3, 0.0, (T, 1, dk)) if gated else np.zeros((T, 1, dk))
    beta = rng.uniform(0.1, 1.0, (T, 1))
    out, _ = oracle.run(q, k, v, g, beta, [0, T], chunk=chunk)
    G = np.cumsum(g[:, 0], axis=0)
    expect = np.zeros((T, dv))
    for t in range(T):
        for i in range(t + 1):
            c = chans[i]
            w = beta[i, 0] * np.exp(G[t, c] - G[i, c]) * q[t, 0, c]
            expect[t] += w * v[i, 0]
    if not gated:   # plain causal linear attention on beta-scaled values
        la = np.tril(q[:, 0] @ k[:, 0].T) @ (beta[:, 0, None] * v[:, 0])
        np.testing.assert_allclose(expect, la, rtol=1e-13, atol=1e-13)
    assert rel_l2(out[:, 0], expect) <= 1e-13


# --------------------------------------------------------------------------
# P6: one token is one rank-1 update of the decayed state
# --------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [0, 64])
def test_p6_single_token_rank1(chunk):
    case = random_case([1], H=1, dk=128, dv=128, seed=12)
    o, s = run(case, chunk=chunk)
    k = case["k"][0, 0]
    q = case["q"][0, 0]
    v = case["v"][0, 0]
    a = np.exp(case["g"][0, 0])
    b = case["beta"][0, 0]
    S0 = case["initial_state"][0, 0].T                           # [dk][dv]
    S1 = (np.eye(128) - b * np.outer(k, k)) @ np.diag(a) @ S0 + b * np.outer(k, v)
    assert rel_l2(s[0, 0], S1.T) <= 1e-14
    assert rel_l2(o[0, 0], S1.T @ q) <= 1e-14


# --------------------------------------------------------------------------
# P7: delta-rule invariant for unit keys; beta = 1 stores v exactly
# --------------------------------------------------------------------------
def test_p7_delta_rule_invariant():
    case = random_case([12], H=1, dk=16, dv=8, seed=13)
    case["beta"][5, 0] = 1.0
    state = case["initial_state"]
    for t in range(12):
        step = {key: (val[t:t + 1] if key in ("q", "k", "v", "g", "beta") else val)
                for key, val in case.items()}
        step["cu_seqlens"] = np.array([0, 1], dtype=np.int32)
        step["initial_state"] = state
        _, new_state = run(step)
        k = case["k"][t, 0]
        a = np.exp(case["g"][t, 0])
        b = case["beta"][t, 0]
        prev = state[0, 0].T                                     # [dk][dv]
        lhs = k @ new_state[0, 0].T
        rhs = (1.0 - b) * (k * a) @ prev + b * case["v"][t, 0]
        np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-13)
        if b == 1.0:
            np.testing.assert_allclose(lhs, case["v"][t, 0], rtol=1e-12, atol=1e-13)
        state = new_state


# --------------------------------------------------------------------------
# P8: state continuity -- a sequence split across calls equals one pass
# --------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [0, 64])
def test_p8_continuity(chunk):
    case = random_case([300], H=2, dk=32, dv=32, seed=14)
    o_all, s_all = run(case, chunk=chunk)
    state = case["initial_state"]
    outs = []
    for lo, hi in [(0, 1), (1, 64), (64, 65), (65, 211), (211, 300)]:
        part = {key: (val[lo:hi] if key in ("q", "k", "v", "g", "beta") else val)
                for key, val in case.items()}
        part["cu_seqlens"] = np.array([0, hi - lo], dtype=np.int32)
        part["initial_state"] = state
        o, state = run(part, chunk=chunk)
        outs.append(o)
    assert rel_l2(np.concatenate(outs), o_all) <= 1e-13
    assert rel_l2(state, s_all) <= 1e-13


# --------------------------------------------------------------------------
# P9: linearity in (V, S0) for fixed keys, decays and betas
# --------------------------------------------------------------------------
def test_p9_linearity():
    c1 = random_case([70, 33], H=2, dk=16, dv=12, seed=15)
    c2 = random_case([70, 33], H=2, dk=16, dv=12, seed=16)
    for key in ("q", "k", "g", "beta"):
        c2[key] = c1[key]
    o1, s1 = run(c1)
    o2, s2 = run(c2)
    c3 = dict(c1)
    c3["v"] = 2.5 * c1["v"] - 0.75 * c2["v"]
    c3["initial_state"] = 2.5 * c1["initial_state"] - 0.75 * c2["initial_state"]
    o3, s3 = run(c3)
    assert rel_l2(o3, 2.5 * o1 - 0.75 * o2) <= 1e-13
    assert rel_l2(s3, 2.5 * s1 - 0.75 * s2) <= 1e-13


# --------------------------------------------------------------------------
# P10: equivariance -- dv permutation, head independence, packing
# --------------------------------------------------------------------------
def test_p10_dv_permutation():
    case = random_case([80, 20], H=2, dk=16, dv=16, seed=17)
    o, s = run(case)
    perm = np.random.default_rng(3).permutation(16)
    c2 = dict(case)
    c2["v"] = case["v"][:, :, perm]
    c2["initial_state"] = case["initial_state"][:, :, perm, :]
    o2, s2 = run(c2)
    assert np.array_equal(o2, o[:, :, perm])
    assert np.array_equal(s2, s[:, :, perm, :])


def test_p10_heads_and_packing_independent():
    lens = [33, 64, 1, 150]
    case = random_case(lens, H=3, dk=16, dv=8, seed=18)
    o, s = run(case, chunk=16)
    c2 = dict(case)
    c2["k"] = case["k"].copy()
    c2["k"][:, 1] = -case["k"][:, 1] + 0.5      # disturb head 1 only
    o2, s2 = run(c2, chunk=16)
    for h in (0, 2):
        assert np.array_equal(o2[:, h], o[:, h]) and np.array_equal(s2[:, h], s[:, h])
    cu = case["cu_seqlens"]
    for n in range(len(lens)):
        part = {key: (val[cu[n]:cu[n + 1]] if key in ("q", "k", "v", "g", "beta") else val)
                for key, val in case.items()}
        part["cu_seqlens"] = np.array([0, lens[n]], dtype=np.int32)
        part["initial_state"] = case["initial_state"][n:n + 1]
        on, sn = run(part, chunk=16)
        assert np.array_equal(on, o[cu[n]:cu[n + 1]])
        assert np.array_equal(sn[0], s[n])


def test_head_subset_matches_full():
    case = random_case([40, 24], H=4, dk=8, dv=8, seed=19, init=False)
    o, s = run(case)
    o2, s2 = run(case, heads=[3, 1])
    assert np.array_equal(o2[:, 0], o[:, 3]) and np.array_equal(o2[:, 1], o[:, 1])
    assert np.array_equal(s2[:, 0], s[:, 3])


def test_zero_length_sequence_keeps_state():
    case = random_case([0, 5, 0], H=1, dk=4, dv=4, seed=20)
    o, s = run(case, chunk=4)
    s0 = case["initial_state"]
    assert np.array_equal(s[0], s0[0]) and np.array_equal(s[2], s0[2])


def test_rejects_bad_cu_seqlens():
    case = random_case([4, 4], H=1, dk=4, dv=4, seed=21)
    case["cu_seqlens"] = np.array([0, 5, 4], dtype=np.int32)
    with pytest.raises(ValueError):
        run(case)


def test_bf16_and_f32_inputs_upcast_exactly():
    from kda_linear_attention_chunk_gb300 import synthetic as syn
    w = syn.Workload("t", [20, 7], H=2, dk=8, dv=8, init_state=True)
    x = syn.draw(w)
    o_bits, s_bits = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], w.cu_seqlens(),
                                initial_state=syn.draw_initial_state(w))
    up = {n: syn.bf16_bits_to_f32(x[n]).astype(np.float64) for n in ("q", "k", "v")}
    o64, s64 = oracle.run(up["q"], up["k"], up["v"], x["g"].astype(np.float64),
                          x["beta"].astype(np.float64), w.cu_seqlens(),
                          initial_state=syn.draw_initial_state(w))
    assert np.array_equal(o_bits, o64) and np.array_equal(s_bits, s64)


def test_golden_regression_fixture():
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_rational.json")
    doc = json.load(open(path))
    x = doc["inputs"]
    arr = lambda n: np.array(x[n], dtype=np.float64)
    out, fin = oracle.run(arr("q"), arr("k"), arr("v"), np.log(arr("alpha")), arr("beta"),
                          np.array(x["cu_seqlens"], dtype=np.int32), initial_state=arr("initial_state"))
    assert np.array_equal(out, np.array(doc["out"]))
    assert np.array_equal(fin, np.array(doc["final_state"]))
