"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/kda.h declares, and rejects bad arguments
synchronously with the documented status, before touching any device.

Fake, never-dereferenced addresses are only passed in calls that must fail
validation; calls that would pass it run only on machines without a GPU."""
import os
import re

import pytest

import kda_linear_attention_chunk_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_expected_calls():
    assert declared_entry_points() == sorted(kda.EXPORTED)


def test_library_exports_every_declared_symbol(kda_lib):
    for name in declared_entry_points():
        assert hasattr(kda_lib, name), name


def test_status_strings(kda_lib):
    for s in range(8):
        assert kda_lib.kda_status_string(s).decode().startswith("KDA_")
    assert b"unknown" in kda_lib.kda_status_string(99)


A = 1 << 20   # fake, 16-byte aligned, never dereferenced addresses


def call(fn="kda_chunk_prefill", **over):
    T, H, d, N = 64, 2, 128, 1
    rows = T * H * d
    args = dict(q=A, k=A + 2 * rows * 4, v=A + 4 * rows * 4, g=A + 6 * rows * 4, beta=A + 10 * rows * 4,
                cu=A + 11 * rows * 4, s0=0, out=A + 12 * rows * 4, s1=0, N=N, T=T, H=H, dk=d, dv=d,
                stream=0)
    if fn == "kda_chunk_prefill_f32":
        args["dk"] = args["dv"] = 64
    args.update(over)
    order = ["q", "k", "v", "g", "beta", "cu", "s0", "out", "s1", "N", "T", "H", "dk", "dv", "stream"]
    return getattr(kda, fn)(*[args[n] for n in order])


PREFILL_ENTRIES = ["kda_chunk_prefill", "kda_chunk_prefill_f32", "kda_chunk_prefill_fullrange",
                   "kda_chunk_prefill_noalloc"]


@pytest.mark.parametrize("fn", PREFILL_ENTRIES)
def test_validation_statuses(kda_lib, fn):
    assert call(fn, q=0) == kda.KDA_ERR_NULL
    assert call(fn, cu=0) == kda.KDA_ERR_NULL
    assert call(fn, N=0) == kda.KDA_ERR_SHAPE
    assert call(fn, T=-1) == kda.KDA_ERR_SHAPE
    assert call(fn, H=0) == kda.KDA_ERR_SHAPE
    assert call(fn, dk=96, dv=96) == kda.KDA_ERR_UNSUPPORTED
    assert call(fn, dk=128, dv=32) == kda.KDA_ERR_UNSUPPORTED
    assert call(fn, dk=256, dv=128) == kda.KDA_ERR_UNSUPPORTED
    assert call(fn, q=A + 8) == kda.KDA_ERR_ALIGN
    assert call(fn, beta=A + 2) == kda.KDA_ERR_ALIGN
    assert call(fn, out=A + 16) == kda.KDA_ERR_ALIAS                                  # out overlaps q
    assert call(fn, s0=A + (40 << 20), s1=A + (40 << 20) + 64) == kda.KDA_ERR_ALIAS   # partial overlap


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
def test_exact_state_alias_passes_validation(kda_lib):
    assert call(s0=A + (40 << 20), s1=A + (40 << 20)) == kda.KDA_ERR_DEVICE


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
@pytest.mark.parametrize("fn", PREFILL_ENTRIES)
def test_every_head_size_and_many_sequences_pass_validation(kda_lib, fn):
    """dk, dv in {64, 128} in every combination, for both dtypes, and more
    than 1024 sequences: all pass the checks (and reach the device check)."""
    for dk in (64, 128):
        for dv in (64, 128):
            assert call(fn, dk=dk, dv=dv) == kda.KDA_ERR_DEVICE, (dk, dv)
    assert call(fn, N=2000) == kda.KDA_ERR_DEVICE


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
def test_noalloc_checks_arguments_before_its_limit(kda_lib):
    """The no-allocation entry checks its arguments as kda_chunk_prefill does,
    then its own limit on N."""
    n = kda.KDA_NOALLOC_MAX_SEQS + 1
    cu = A + (80 << 20)                   # room for N + 1 entries
    assert call("kda_chunk_prefill_noalloc", N=n, cu=cu, q=0) == kda.KDA_ERR_NULL
    assert call("kda_chunk_prefill_noalloc", N=n, cu=cu, q=A + 8) == kda.KDA_ERR_ALIGN
    assert call("kda_chunk_prefill_noalloc", N=n, cu=cu, out=A + 16) == kda.KDA_ERR_ALIAS
    assert call("kda_chunk_prefill_noalloc", N=n, cu=cu) == kda.KDA_ERR_NOALLOC_LIMIT
    assert call("kda_chunk_prefill_noalloc", N=n - 1, cu=cu) == kda.KDA_ERR_DEVICE


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
def test_empty_rows_allow_null_tensors(kda_lib):
    assert call(q=0, k=0, v=0, g=0, beta=0, out=0, T=0) == kda.KDA_ERR_DEVICE


def call_slots(**over):
    T, H, d, N = 64, 2, 128, 3
    rows = T * H * d
    args = dict(q=A, k=A + 2 * rows * 4, v=A + 4 * rows * 4, g=A + 6 * rows * 4, beta=A + 10 * rows * 4,
                cu=A + 11 * rows * 4, slots=A + 11 * rows * 4 + 64, pool=A + (40 << 20), num_slots=5,
                out=A + 12 * rows * 4, N=N, T=T, H=H, dk=d, dv=d, stream=0)
    args.update(over)
    order = ["q", "k", "v", "g", "beta", "cu", "slots", "pool", "num_slots", "out", "N", "T", "H", "dk", "dv",
             "stream"]
    return kda.kda_chunk_prefill_slots(*[args[n] for n in order])


def test_slots_validation_statuses(kda_lib):
    pool_bytes = 5 * 2 * 128 * 128 * 4
    assert call_slots(slots=0) == kda.KDA_ERR_NULL
    assert call_slots(pool=0) == kda.KDA_ERR_NULL
    assert call_slots(num_slots=0) == kda.KDA_ERR_SHAPE
    assert call_slots(N=0) == kda.KDA_ERR_SHAPE
    assert call_slots(dk=96, dv=64) == kda.KDA_ERR_UNSUPPORTED
    assert call_slots(slots=A + (1 << 19) + 2) == kda.KDA_ERR_ALIGN
    assert call_slots(pool=A + (40 << 20) + 8) == kda.KDA_ERR_ALIGN
    assert call_slots(pool=A) == kda.KDA_ERR_ALIAS                                     # pool over q
    assert call_slots(slots=A + (40 << 20) + pool_bytes - 4) == kda.KDA_ERR_ALIAS      # slots inside the pool
    assert call_slots(out=A + (60 << 20), slots=A + (60 << 20) + 16) == kda.KDA_ERR_ALIAS   # slots inside out


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
def test_slots_valid_call_passes_validation(kda_lib):
    assert call_slots() == kda.KDA_ERR_DEVICE
    assert call_slots(pool=A + (40 << 20) + 5 * 2 * 128 * 128 * 4) == kda.KDA_ERR_DEVICE   # pool just past
    assert call_slots(dk=64, dv=64) == kda.KDA_ERR_DEVICE
    assert call_slots(dk=64, dv=128) == kda.KDA_ERR_DEVICE
    assert call_slots(N=2000) == kda.KDA_ERR_DEVICE


def call_decode(**over):
    N, H, d = 4, 2, 128
    rows = N * H * d
    args = dict(q=A, k=A + 2 * rows, v=A + 4 * rows, g=A + 6 * rows, beta=A + 10 * rows, slots=A + 11 * rows,
                pool=A + (40 << 20), num_slots=6, out=A + 12 * rows, N=N, H=H, dk=d, dv=d, stream=0)
    args.update(over)
    order = ["q", "k", "v", "g", "beta", "slots", "pool", "num_slots", "out", "N", "H", "dk", "dv", "stream"]
    return kda.kda_decode(*[args[n] for n in order])


def test_decode_validation_statuses(kda_lib):
    assert call_decode(q=0) == kda.KDA_ERR_NULL
    assert call_decode(pool=0) == kda.KDA_ERR_NULL
    assert call_decode(N=0) == kda.KDA_ERR_SHAPE
    assert call_decode(num_slots=0) == kda.KDA_ERR_SHAPE
    assert call_decode(slots=0, num_slots=3) == kda.KDA_ERR_SHAPE          # entry n needs num_slots >= N
    assert call_decode(dk=64, dv=64) == kda.KDA_ERR_UNSUPPORTED
    assert call_decode(q=A + 8) == kda.KDA_ERR_ALIGN
    assert call_decode(slots=A + 11 * 1024 + 2) == kda.KDA_ERR_ALIGN
    assert call_decode(pool=A) == kda.KDA_ERR_ALIAS                        # pool over q
    assert call_decode(out=A + 6 * 1024) == kda.KDA_ERR_ALIAS              # out over v


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
def test_decode_valid_call_passes_validation(kda_lib):
    assert call_decode() == kda.KDA_ERR_DEVICE
    assert call_decode(slots=0, num_slots=4) == kda.KDA_ERR_DEVICE


def call_fold(**over):
    N, W, H, d = 4, 3, 2, 128
    rows = N * W * H * d
    args = dict(k=A, v=A + 2 * rows, g=A + 4 * rows, beta=A + 8 * rows, acc=A + 8 * rows + 4096,
                slots=A + 8 * rows + 8192, pool=A + (40 << 20), num_slots=6, N=N, W=W, H=H, dk=d, dv=d, stream=0)
    args.update(over)
    order = ["k", "v", "g", "beta", "acc", "slots", "pool", "num_slots", "N", "W", "H", "dk", "dv", "stream"]
    return kda.kda_fold_commit(*[args[n] for n in order])


def test_fold_validation_statuses(kda_lib):
    assert call_fold(k=0) == kda.KDA_ERR_NULL
    assert call_fold(acc=0) == kda.KDA_ERR_NULL
    assert call_fold(W=0) == kda.KDA_ERR_SHAPE
    assert call_fold(slots=0, num_slots=3) == kda.KDA_ERR_SHAPE
    assert call_fold(dk=64, dv=64) == kda.KDA_ERR_UNSUPPORTED
    assert call_fold(k=A + 8) == kda.KDA_ERR_ALIGN
    assert call_fold(acc=A + 8 * 3072 * 4 + 4098) == kda.KDA_ERR_ALIGN
    assert call_fold(pool=A) == kda.KDA_ERR_ALIAS


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
def test_fold_valid_call_passes_validation(kda_lib):
    assert call_fold() == kda.KDA_ERR_DEVICE


def call_conv(**over):
    N, T, H, d = 3, 40, 2, 128
    xb = T * H * d * 2
    args = dict(xq=A, xk=A + xb, xv=A + 2 * xb, w=A + 3 * xb, cu=A + 3 * xb + 16384, slots=A + 3 * xb + 20480,
                pool=A + (8 << 20), num_slots=5, q=A + (16 << 20), k=A + (16 << 20) + xb, v=A + (16 << 20) + 2 * xb,
                N=N, T=T, H=H, d=d, act=1, eps=1e-6, stream=0)
    args.update(over)
    order = ["xq", "xk", "xv", "w", "cu", "slots", "pool", "num_slots", "q", "k", "v", "N", "T", "H", "d", "act",
             "eps", "stream"]
    return kda.kda_short_conv(*[args[n] for n in order])


def test_conv_validation_statuses(kda_lib):
    assert call_conv(xq=0) == kda.KDA_ERR_NULL
    assert call_conv(w=0) == kda.KDA_ERR_NULL
    assert call_conv(pool=0) == kda.KDA_ERR_NULL
    assert call_conv(N=0) == kda.KDA_ERR_SHAPE
    assert call_conv(num_slots=0) == kda.KDA_ERR_SHAPE
    assert call_conv(slots=0, num_slots=2) == kda.KDA_ERR_SHAPE            # entry n needs num_slots >= N
    assert call_conv(act=2) == kda.KDA_ERR_SHAPE
    assert call_conv(eps=-1.0) == kda.KDA_ERR_SHAPE
    assert call_conv(eps=float("nan")) == kda.KDA_ERR_SHAPE
    assert call_conv(d=64) == kda.KDA_ERR_UNSUPPORTED
    assert call_conv(xk=A + 40 * 2 * 128 * 2 + 8) == kda.KDA_ERR_ALIGN
    assert call_conv(cu=A + 3 * 40 * 2 * 128 * 2 + 16386) == kda.KDA_ERR_ALIGN
    assert call_conv(pool=A) == kda.KDA_ERR_ALIAS                          # pool over xq
    assert call_conv(v=A + 40 * 2 * 128 * 2) == kda.KDA_ERR_ALIAS          # v_out over xk
    assert call_conv(k=A + (16 << 20)) == kda.KDA_ERR_ALIAS                # k_out over q_out
    assert call_conv(q=A + (8 << 20)) == kda.KDA_ERR_ALIAS                 # q_out over the pool


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
def test_conv_empty_rows_allow_null_tensors(kda_lib):
    assert call_conv(xq=0, xk=0, xv=0, q=0, k=0, v=0, T=0) == kda.KDA_ERR_DEVICE


@pytest.mark.skipif(_has_gpu(), reason="valid call with fake addresses: CPU-only check")
def test_conv_valid_call_passes_validation(kda_lib):
    assert call_conv() == kda.KDA_ERR_DEVICE
    assert call_conv(slots=0, num_slots=3, act=0, eps=0.0) == kda.KDA_ERR_DEVICE


def call_decode_conv(**over):
    N, H = 3, 2
    xb = N * H * 128 * 2
    args = dict(xq=A, xk=A + xb, xv=A + 2 * xb, w=A + 3 * xb, cslots=A + 3 * xb + 16384, cpool=A + (8 << 20),
                cnum=5, g=A + (1 << 20), beta=A + (1 << 20) + 8192, slots=A + (1 << 20) + 12288,
                pool=A + (16 << 20), num_slots=4, out=A + (2 << 20), N=N, H=H, dk=128, dv=128, act=1, eps=1e-6,
                stream=0)
    args.update(over)
    order = ["xq", "xk", "xv", "w", "cslots", "cpool", "cnum", "g", "beta", "slots", "pool", "num_slots", "out",
             "N", "H", "dk", "dv", "act", "eps", "stream"]
    return kda.kda_decode_conv(*[args[n] for n in order])


def test_decode_conv_validation_statuses(kda_lib):
    assert call_decode_conv(xq=0) == kda.KDA_ERR_NULL
    assert call_decode_conv(cpool=0) == kda.KDA_ERR_NULL
    assert call_decode_conv(pool=0) == kda.KDA_ERR_NULL
    assert call_decode_conv(N=0) == kda.KDA_ERR_SHAPE
    assert call_decode_conv(cnum=0) == kda.KDA_ERR_SHAPE
    assert call_decode_conv(cslots=0, cnum=2) == kda.KDA_ERR_SHAPE          # entry n needs conv_num_slots >= N
    assert call_decode_conv(slots=0, num_slots=2) == kda.KDA_ERR_SHAPE      # and num_slots >= N
    assert call_decode_conv(act=2) == kda.KDA_ERR_SHAPE
    assert call_decode_conv(eps=float("nan")) == kda.KDA_ERR_SHAPE
    assert call_decode_conv(dk=64, dv=64) == kda.KDA_ERR_UNSUPPORTED
    assert call_decode_conv(xk=A + 3 * 2 * 128 * 2 + 8) == kda.KDA_ERR_ALIGN
    assert call_decode_conv(cslots=A + 3 * 3 * 2 * 128 * 2 + 16386) == kda.KDA_ERR_ALIGN
    assert call_decode_conv(cpool=A) == kda.KDA_ERR_ALIAS                   # window pool over xq
    assert call_decode_conv(out=A + (1 << 20)) == kda.KDA_ERR_ALIAS         # out over g
    assert call_decode_conv(pool=A + (8 << 20)) == kda.KDA_ERR_ALIAS        # state pool over the window pool


@pytest.mark.skipif(_has_gpu(), reason="on a GPU box a valid call would launch on these fake addresses")
def test_decode_conv_valid_call_passes_validation(kda_lib):
    assert call_decode_conv() == kda.KDA_ERR_DEVICE
    assert call_decode_conv(slots=0, cslots=0, num_slots=3, cnum=3) == kda.KDA_ERR_DEVICE
