"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (no GPU).

Each mutant is one textual edit of oracle/kda_oracle.c (a wrong sign, a
dropped term, a swapped index, a transposed layout, an off-by-one), compiled
to a temporary library.  A short battery of the oracle pins runs against it;
the test passes only when the battery fails.  The unmodified copy must pass
the same battery, so the battery itself is sound.
"""
import os
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle
from test_oracle import brute_force_exact, random_case, rel_l2

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "kda_oracle.c")

MUTANTS = {
    # recurrence
    "erase_sign": ("e[v] = b * (vv[v] - e[v]);", "e[v] = b * (vv[v] + e[v]);"),
    "beta_on_v_only": ("e[v] = b * (vv[v] - e[v]);", "e[v] = b * vv[v] - e[v];"),
    "decay_sign": ("al[c] = exp(at3(J, J->g, J->gb_dtype, t, h, c, dk));",
                   "al[c] = exp(-at3(J, J->g, J->gb_dtype, t, h, c, dk));"),
    "readout_before_write": ("o[v] += qq[c] * S[c * dv + v];",
                             "o[v] += qq[c] * (S[c * dv + v] - kk[c] * e[v]);"),
    "state_layout_transposed": ("S[c * dv + v] = src[v * dk + c];", "S[c * dv + v] = src[c * dv + v];"),
    # chunked form
    "exclusive_cumsum": ("acc += at3(J, J->g, J->gb_dtype, s0 + r, h, c, dk);\n                G[r * dk + c] = acc;",
                         "G[r * dk + c] = acc;\n                acc += at3(J, J->g, J->gb_dtype, s0 + r, h, c, dk);"),
    "akk_decay_transposed": ("s += K[i * dk + c] * K[j * dk + c] * exp(G[i * dk + c] - G[j * dk + c]);",
                             "s += K[i * dk + c] * K[j * dk + c] * exp(G[j * dk + c] - G[i * dk + c]);"),
    "akk_beta_column": ("A[i * C + j] = bt[i] * s;", "A[i * C + j] = bt[j] * s;"),
    "inverse_sign": ("Tm[i * C + l] -= a * Tm[j * C + l];", "Tm[i * C + l] += a * Tm[j * C + l];"),
    "w_without_beta": ("s += Tm[i * C + j] * bt[j] * K[j * dk + c] * exp(G[j * dk + c]);",
                       "s += Tm[i * C + j] * K[j * dk + c] * exp(G[j * dk + c]);"),
    "aqk_strict_lower": ("if (i <= r)", "if (i < r)"),
    "state_decay_wrong_row": ("const double *Gl = G + (size_t)(L - 1) * dk;",
                              "const double *Gl = G + (size_t)(L > 1 ? L - 2 : 0) * dk;"),
    "output_drops_inter_chunk": ("s += Q[r * dk + c] * exp(G[r * dk + c]) * S[c * dv + v];",
                                 "s += 0.0 * S[c * dv + v];"),
}


def battery(lib) -> bool:
    """True when every check passes."""
    ok = True
    # P2, exact rational brute force, both routes
    rng = np.random.default_rng(7)
    T, dk, dv = 6, 3, 3
    quarter = lambda: Fraction(int(rng.integers(-4, 5)), 4)
    q = [[quarter() for _ in range(dk)] for _ in range(T)]
    k = [[quarter() for _ in range(dk)] for _ in range(T)]
    v = [[quarter() for _ in range(dv)] for _ in range(T)]
    alpha = [[Fraction(int(rng.integers(1, 5)), 4) for _ in range(dk)] for _ in range(T)]
    beta = [Fraction(int(rng.integers(1, 5)), 4) for _ in range(T)]
    s0 = [[quarter() for _ in range(dv)] for _ in range(dk)]
    outs, S = brute_force_exact(q, k, v, alpha, beta, s0)
    f = lambda m: np.array([[float(x) for x in row] for row in m])
    for route in (0, 4):
        o, s = oracle.run(f(q)[:, None], f(k)[:, None], f(v)[:, None], np.log(f(alpha))[:, None],
                          np.array([float(b) for b in beta])[:, None], [0, T],
                          initial_state=f(s0).T[None, None], chunk=route, lib=lib)
        ok &= bool(np.max(np.abs(o[:, 0] - f(outs))) <= 1e-12)
        ok &= bool(np.max(np.abs(s[0, 0] - f(S).T)) <= 1e-12)
    # P1, chunked vs recurrence on a ragged packed case
    case = random_case([37, 1, 130, 64], H=2, dk=16, dv=12, seed=2)
    o_r, s_r = oracle.run(**case, lib=lib)
    o_c, s_c = oracle.run(**case, chunk=16, lib=lib)
    ok &= bool(rel_l2(o_c, o_r) <= 1e-12 and rel_l2(s_c, s_r) <= 1e-12)
    # P8, continuity across a split
    case = random_case([100], H=1, dk=8, dv=8, seed=3)
    o_all, s_all = oracle.run(**case, lib=lib)
    first = {k_: (v_[:40] if k_ in ("q", "k", "v", "g", "beta") else v_) for k_, v_ in case.items()}
    first["cu_seqlens"] = np.array([0, 40], dtype=np.int32)
    o1, st = oracle.run(**first, lib=lib)
    second = {k_: (v_[40:] if k_ in ("q", "k", "v", "g", "beta") else v_) for k_, v_ in case.items()}
    second["cu_seqlens"] = np.array([0, 60], dtype=np.int32)
    second["initial_state"] = st
    o2, s2 = oracle.run(**second, lib=lib)
    ok &= bool(rel_l2(np.concatenate([o1, o2]), o_all) <= 1e-13 and rel_l2(s2, s_all) <= 1e-13)
    return ok


def build_variant(tmp, name, edit):
    src = open(SRC).read()
    if edit is not None:
        old, new = edit
        assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
        src = src.replace(old, new)
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as fh:
        fh.write(src)
    lib = os.path.join(tmp, f"lib{name}.so")
    oracle.build(src=path, out=lib)
    return oracle.load(lib)


@pytest.fixture(scope="module")
def tmpdir_mod():
    with tempfile.TemporaryDirectory() as d:
        yield d


def test_unmutated_copy_passes(tmpdir_mod):
    assert battery(build_variant(tmpdir_mod, "clean", None))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmpdir_mod, name):
    assert not battery(build_variant(tmpdir_mod, name, MUTANTS[name])), f"mutant {name} survived"
