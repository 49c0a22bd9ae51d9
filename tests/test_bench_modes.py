"""The bench's record of which form of the tensor-core prefill each workload
runs (bench.tc_mode) follows the library's choice (kda.h, "Split"): the fused
kernel for many units, split mode for few units and T >= 1024 rows, half
chains where the units are at most a fifth of the SMs, and the KDA_SPLIT
overrides.  Host logic only (no GPU)."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from kda_linear_attention_chunk_gb300 import synthetic as syn  # noqa: E402

SMS = 152


def mode(lens, H, rows=None, env="", dk=128, dtype="bf16", monkeypatch=None):
    w = syn.Workload("m", lens, H=H, dk=dk, dv=dk, qkv_dtype=dtype)
    if env:
        monkeypatch.setenv("KDA_SPLIT", env)
    else:
        monkeypatch.delenv("KDA_SPLIT", raising=False)
    return bench.tc_mode(w, rows if rows is not None else w.T, SMS)


def test_default_forms(monkeypatch):
    assert mode([1024] * 16, 32, monkeypatch=monkeypatch) == "fused"            # 512 units
    assert mode([4096], 32, monkeypatch=monkeypatch) == "split"                 # 32 units > SMs / 5
    assert mode([4096], 30, monkeypatch=monkeypatch) == "split-half"            # 30 units <= 152 / 5
    assert mode([4096], 16, monkeypatch=monkeypatch) == "split-half"
    assert mode([1000, 513, 64, 2519], 16, monkeypatch=monkeypatch) == "split"  # 64 units: no room for two chains
    assert mode([512], 16, monkeypatch=monkeypatch) == "fused"                  # T < 1024
    assert mode([4096], 77, monkeypatch=monkeypatch) == "fused"                 # 77 units > SMs / 2
    assert mode([256], 2, dk=64, dtype="f32", monkeypatch=monkeypatch) == "cuda-core"


def test_overrides(monkeypatch):
    assert mode([4096], 16, env="0", monkeypatch=monkeypatch) == "fused"
    assert mode([4096], 16, env="full", monkeypatch=monkeypatch) == "split"
    assert mode([4096], 32, env="half", monkeypatch=monkeypatch) == "split-half"   # 32 units: 4 * 32 <= 152
    assert mode([4096], 40, env="half", monkeypatch=monkeypatch) == "split"        # 4 * 40 > 152: falls back
    assert mode([512], 16, env="1", monkeypatch=monkeypatch) == "split-half"       # "1" also below 1024 rows
    assert mode([4096], 77, env="1", monkeypatch=monkeypatch) == "fused"           # not possible at all


@pytest.mark.parametrize("name", ["long_65536", "context_262144", "varlen4_4096", "packed16_8192"])
def test_bench_workloads(name, monkeypatch):
    monkeypatch.delenv("KDA_SPLIT", raising=False)
    w = syn.workloads()[name]
    rows = w.T // w.calls
    expect = {"long_65536": "split", "context_262144": "split", "varlen4_4096": "split",
              "packed16_8192": "fused"}[name]
    assert bench.tc_mode(w, rows, SMS) == expect
