"""Plant plausible mistakes in a copy of the short-conv oracle
(oracle.short_conv) and check that its pins catch every one of them (no GPU).

Each mutant is one textual edit of the function's source (taps in the wrong
order, the wrong window kept, the norm over the wrong axis or applied to v,
a sign, eps outside the root, padding not skipped, the taps of another
stream), executed into a fresh namespace.  The pins of test_oracle_conv run
against it; the test passes only when one of them fails.  The unmodified copy
must pass all of them, so the battery itself is sound.
"""
import inspect
import textwrap

import numpy as np
import pytest

import oracle
from test_oracle_conv import PINS

SRC = textwrap.dedent(inspect.getsource(oracle.short_conv))

MUTANTS = {
    "taps_reversed": ("w[s, :, j] * seq[j:j + L]", "w[s, :, j] * seq[3 - j:3 - j + L]"),
    "window_keeps_old_taps": ("pool[slot, :, s, :] = seq_bits[L:L + 3]", "pool[slot, :, s, :] = seq_bits[0:3]"),
    "window_newest_first": ("pool[slot, :, s, :] = seq_bits[L:L + 3]",
                            "pool[slot, :, s, :] = seq_bits[L:L + 3][::-1]"),
    "norm_over_all_heads": ("(yh * yh).sum(axis=2, keepdims=True)", "(yh * yh).sum(axis=(1, 2), keepdims=True)"),
    "norm_on_v_too": ("if s < 2:", "if s < 3:"),
    "silu_sign": ("y / (1.0 + np.exp(-y))", "y / (1.0 + np.exp(y))"),
    "eps_outside_root": ("np.sqrt((yh * yh).sum(axis=2, keepdims=True) + eps)",
                         "(np.sqrt((yh * yh).sum(axis=2, keepdims=True)) + eps)"),
    "padding_not_skipped": ("if not 0 <= slot < num_slots:", "if slot >= num_slots:"),
    "taps_of_another_stream": ("pool[slot, :, s, :], xs[s]", "pool[slot, :, (s + 1) % 3, :], xs[s]"),
}


def build(src):
    ns = {"np": np, "bf16_bits_to_f64": oracle.bf16_bits_to_f64}
    exec(compile(src, "<short_conv copy>", "exec"), ns)
    return ns["short_conv"]


def battery(fn) -> bool:
    """True when every pin passes."""
    for pin in PINS:
        try:
            pin(fn)
        except Exception:
            return False
    return True


def test_unmodified_copy_passes_the_battery():
    assert battery(build(SRC))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site of {name} not found once in the oracle"
    assert not battery(build(SRC.replace(old, new))), f"mutant {name} passed every pin"
