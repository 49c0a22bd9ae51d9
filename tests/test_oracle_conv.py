"""Pins of the short-conv + L2-norm oracle (oracle.short_conv) against facts
that do not come from the oracle itself: the identity and pure-delay
filters, numpy's own convolution, scipy's logistic function, the window
contents after short sequences, chained calls, and padding (kern-k3-pp-prefill
README, sections "P: the packed prefill" and "D inside SGLang")."""
import numpy as np
import pytest

import oracle

H, D = 2, 128
C = H * D


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def inputs(T, seed, num_slots=4):
    rng = np.random.default_rng(seed)
    xs = [bf16_bits(rng.standard_normal((T, H, D))) for _ in range(3)]
    pool = bf16_bits(rng.standard_normal((num_slots, 3, 3, C)))
    w = rng.standard_normal((3, C, 4))
    return xs, w, pool


def f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def pin_identity_filter(conv=oracle.short_conv):
    """w = (0, 0, 0, 1), no activation: q and k are the rows scaled to unit L2
    norm per head (numpy's norm), v is the row itself."""
    T = 9
    xs, _, pool = inputs(T, 1)
    w = np.zeros((3, C, 4))
    w[:, :, 3] = 1.0
    (q, k, v), _, _ = conv(*xs, w, [0, 4, 9], pool, [1, 3], activation="none", eps=0.0)
    for got, x in ((q, xs[0]), (k, xs[1])):
        xf = f64(x)
        ref = xf / np.linalg.norm(xf, axis=2, keepdims=True)
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=0)
    np.testing.assert_array_equal(v, f64(xs[2]))


def pin_pure_delay(conv=oracle.short_conv):
    """w = (1, 0, 0, 0): y_t = x_{t-3}, the window's taps for t < 3, in tap
    order (oldest first), then the sequence's own rows."""
    T = 7
    xs, _, pool = inputs(T, 2)
    w = np.zeros((3, C, 4))
    w[:, :, 0] = 1.0
    (_, _, v), _, _ = conv(*xs, w, [0, T], pool, [2], activation="none")
    xv = f64(xs[2]).reshape(T, C)
    taps = f64(pool[2, :, 2, :])
    for t in range(T):
        ref = taps[t] if t < 3 else xv[t - 3]
        np.testing.assert_array_equal(v.reshape(T, C)[t], ref)


def pin_numpy_convolve(conv=oracle.short_conv):
    """Random filters: v channel by channel equals numpy's full convolution of
    [taps ; rows] with the filter, restricted to the rows; q is that result
    normalised per head."""
    T = 23
    xs, w, pool = inputs(T, 3)
    (q, _, v), _, _ = conv(*xs, w, [0, T], pool, [0], activation="none", eps=1e-6)
    for s, got in ((2, v.reshape(T, C)), (0, None)):
        seq = np.concatenate([f64(pool[0, :, s, :]), f64(xs[s]).reshape(T, C)], axis=0)
        ref = np.empty((T, C))
        for c in range(C):
            # np.convolve(a, f)[i] = sum_j a[i - j] f[j]: reversing the filter puts
            # tap 3 on the newest row
            ref[:, c] = np.convolve(seq[:, c], w[s, c, ::-1], mode="valid")
        if got is not None:
            np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
        else:
            rh = ref.reshape(T, H, D)
            refq = rh / np.sqrt((rh ** 2).sum(axis=2, keepdims=True) + 1e-6)
            np.testing.assert_allclose(q, refq, rtol=1e-12, atol=1e-14)


def pin_silu(conv=oracle.short_conv):
    """SiLU on the identity filter: v = x * expit(x) (scipy's logistic)."""
    special = pytest.importorskip("scipy.special")
    T = 5
    xs, _, pool = inputs(T, 4)
    w = np.zeros((3, C, 4))
    w[:, :, 3] = 1.0
    (_, _, v), _, _ = conv(*xs, w, [0, T], pool, [0], activation="silu")
    xv = f64(xs[2])
    np.testing.assert_allclose(v, xv * special.expit(xv), rtol=1e-13, atol=1e-300)


def pin_window(L, conv=oracle.short_conv):
    """The new taps are the last three rows of [old taps ; rows], bit for bit:
    for L < 3 the old taps shift down by L."""
    xs, w, pool = inputs(L, 5)
    _, new, _ = conv(*xs, w, [0, L], pool, [3])
    for s in range(3):
        seq = np.concatenate([pool[3, :, s, :], xs[s].reshape(L, C)], axis=0)
        np.testing.assert_array_equal(new[3, :, s, :], seq[-3:])
    np.testing.assert_array_equal(new[[0, 1, 2]], pool[[0, 1, 2]])   # entries no sequence names


def pin_chained(conv=oracle.short_conv):
    """Two calls over the halves of each sequence, the window carried between
    them, give the outputs and the window of one call over the whole."""
    lens = [9, 2, 14]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    xs, w, pool = inputs(T, 6)
    slots = [2, 0, 3]
    (q, k, v), new, _ = conv(*xs, w, cu, pool, slots)
    cut = [n // 2 for n in lens]
    first = np.concatenate([np.arange(cu[i], cu[i] + cut[i]) for i in range(3)])
    second = np.concatenate([np.arange(cu[i] + cut[i], cu[i + 1]) for i in range(3)])
    cu1 = np.concatenate([[0], np.cumsum(cut)])
    cu2 = np.concatenate([[0], np.cumsum([lens[i] - cut[i] for i in range(3)])])
    (q1, k1, v1), mid, _ = conv(*(x[first] for x in xs), w, cu1, pool, slots)
    (q2, k2, v2), fin, _ = conv(*(x[second] for x in xs), w, cu2, mid, slots)
    for whole, a, b in ((q, q1, q2), (k, k1, k2), (v, v1, v2)):
        np.testing.assert_array_equal(whole[first], a)
        np.testing.assert_array_equal(whole[second], b)
    np.testing.assert_array_equal(new, fin)


def pin_padding(conv=oracle.short_conv):
    """Id -1: nothing computed, entry untouched; an id outside the pool is
    handled the same way and reported; an empty sequence leaves its entry."""
    lens = [3, 4, 0, 2]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    xs, w, pool = inputs(T, 7, num_slots=4)
    (q, k, v), new, bad = conv(*xs, w, cu, pool, [-1, 9, 1, 2])
    assert bad == [1]
    assert np.isnan(q[:7]).all() and np.isnan(v[:7]).all()
    assert not np.isnan(q[7:]).any()
    np.testing.assert_array_equal(new[[0, 1, 3]], pool[[0, 1, 3]])
    assert not np.array_equal(new[2], pool[2])


PINS = [pin_identity_filter, pin_pure_delay, pin_numpy_convolve, pin_silu, pin_chained, pin_padding] + \
    [lambda conv, L=L: pin_window(L, conv) for L in (1, 2, 3, 4, 11)]


def test_identity_filter_gives_normalised_inputs():
    pin_identity_filter()


def test_pure_delay_reads_the_window_then_the_rows():
    pin_pure_delay()


def test_matches_numpy_convolve():
    pin_numpy_convolve()


def test_silu_is_x_times_logistic():
    pin_silu()


@pytest.mark.parametrize("L", [1, 2, 3, 4, 11])
def test_window_after_short_and_long_sequences(L):
    pin_window(L)


def test_chained_calls_equal_one_call():
    pin_chained()


def test_padding_and_bad_ids():
    pin_padding()
