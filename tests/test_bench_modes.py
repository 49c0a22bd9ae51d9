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


def test_traffic_records_follow_the_kernel_sources(tmp_path, monkeypatch):
    """A committed ncu traffic figure is reported only while the kernel sources
    it was captured on are the current ones (comments aside), and only for its
    own workload; every committed record parses."""
    for name in sorted(os.listdir(os.path.join(bench.ROOT, "profiles"))):
        if name.startswith("traffic") and name.endswith(".txt"):
            keys = {}
            for line in open(os.path.join(bench.ROOT, "profiles", name)):
                if ":" in line and not line.lstrip().startswith("#"):
                    k, v = line.split(":", 1)
                    keys[k.strip()] = v.strip()
            assert {"kernel", "workload", "kernel_source_sha", "dram_bytes_per_launch"} <= set(keys), name
            assert int(keys["dram_bytes_per_launch"]) > 0 and len(keys["kernel_source_sha"]) == 16, name

    src = "int f(int x) {  // twice\n    return 2 * x;\n}\n"
    edited = "/* doubles */\nint f(int x) {\n\n    return 2 * x;   \n}\n"
    assert bench.code_only(src) == bench.code_only(edited)            # comments and blanks do not count
    assert bench.code_only(src) != bench.code_only(src.replace("2 *", "3 *"))

    csrc = tmp_path / "kda_linear_attention_chunk_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(src)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha(("k.cu",))
    record = f"# a capture\nkernel: k\nworkload: w1\nkernel_source_sha: {sha}\ndram_bytes_per_launch: 1234\n"
    (tmp_path / "profiles" / "traffic_w1.txt").write_text(record)
    assert bench.recorded_traffic("w1", ("k.cu",)) == 1234
    assert bench.recorded_traffic("w2", ("k.cu",)) is None                 # no record for that workload
    (tmp_path / "profiles" / "traffic_w2.txt").write_text(record)           # a record naming another workload
    assert bench.recorded_traffic("w2", ("k.cu",)) is None
    (csrc / "k.cu").write_text(edited)
    assert bench.recorded_traffic("w1", ("k.cu",)) == 1234                  # a comment edit keeps it
    (csrc / "k.cu").write_text(src.replace("2 *", "3 *"))
    assert bench.recorded_traffic("w1", ("k.cu",)) is None                  # a code change drops it
