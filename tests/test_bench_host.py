"""Host logic of bench.py, without a GPU: the GEMM source digest that guards
the committed ncu counters, the parsing of those counters, and the reference
arm's bounded sampling (with a stand-in for the oracle, so that it runs in
milliseconds)."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

CODE = """// a kernel
__global__ void k(int *p) {  /* one
   block comment */
    p[0] = 1;   // trailing

}
"""


def test_code_digest_ignores_comments_and_blank_lines():
    base = bench.code_digest([CODE])
    edited = CODE.replace("// a kernel", "// a kernel, reworded").replace(
        "/* one\n   block comment */", "/* two */") + "\n\n// appended\n"
    assert bench.code_digest([edited]) == base


def test_code_digest_sees_code_changes():
    base = bench.code_digest([CODE])
    assert bench.code_digest([CODE.replace("p[0] = 1", "p[0] = 2")]) != base
    assert bench.code_digest([CODE, CODE]) != base


def test_profiled_traffic_matches_the_committed_summary():
    per = bench.profiled_traffic()
    assert per is not None, "the ncu summary's source digest differs from the GEMM source"
    assert set(per) == {"qkv", "fc", "proj"}
    assert all(isinstance(v, int) and v > 0 for v in per.values())


def test_profiled_traffic_is_none_for_another_source(monkeypatch):
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic() is None


class FakeOracle:
    """Stands in for the oracle: each call 'takes' time proportional to its
    rows, and counts the rows it was given."""

    def __init__(self):
        self.rows = []

    def num_threads(self):
        return 3

    def bsgemm_i8(self, a, b, relu):
        self.rows.append(("gemm", a.shape[0]))
        return None, 0

    def probe_hash(self, seed, M, N, K):
        self.rows.append(("probe", M))
        return b"\0" * 32, 0


def small_data():
    rng = np.random.default_rng(0)
    return [(rng.standard_normal((8192, 8), dtype=np.float32),
             rng.standard_normal((8, 4), dtype=np.float32), False) for _ in range(3)]


def fake_clock(monkeypatch, per_row):
    """Each oracle part 'takes' per_row seconds for each row it processes."""
    orig_part = bench.oracle_part

    def part(orc, data, p, rows):
        ops, _ = orig_part(orc, data, p, rows)
        return ops, rows * per_row
    monkeypatch.setattr(bench, "oracle_part", part)


def test_sample_rows_scale_to_the_budget(monkeypatch):
    fake_clock(monkeypatch, per_row=1e-3)        # 256 rows take 0.256 s
    orc = FakeOracle()
    rows = bench.sample_rows(orc, small_data(), seconds=0.5)
    assert rows[:3] == [496, 496, 496]           # 256 * 0.5 / 0.256, down to a multiple of 8
    assert rows[3] == 496
    rows = bench.sample_rows(orc, small_data(), seconds=100.0)
    assert rows[:3] == [8192] * 3 and rows[3] == 1024   # capped at the full sizes
    rows = bench.sample_rows(orc, small_data(), seconds=1e-6)
    assert rows == [8, 8, 8, 8]                  # at least 8 rows


def test_reference_arm_is_bounded_and_complete(monkeypatch):
    import oracle
    fake = FakeOracle()
    monkeypatch.setattr(oracle, "load", lambda: fake)
    monkeypatch.setattr(bench, "oracle_inputs", small_data)
    fake_clock(monkeypatch, per_row=1e-3)
    args = type("A", (), {"steps": 1000, "warmup": 5})()
    line = bench.run_reference(args, 0, 1)
    assert bench.run_reference(args, 1, 2) is None          # only rank 0 runs it
    json.dumps(line)
    assert line["impl"] == "reference" and line["steps"] == 1000
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 3
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["value"] > 0 and line["higher_is_better"] is True
    # the whole run stays near its two-minute budget of (fake) oracle time
    timed = sum(r for kind, r in fake.rows) * 1e-3
    assert timed < 200.0
    # step i ran part i mod 4: the probe every fourth step
    probe_calls = sum(1 for kind, _ in fake.rows if kind == "probe")
    assert 250 <= probe_calls <= 260


def test_config_line_names_the_workload():
    cfg = bench.config_dict(1)
    assert cfg["workload"].startswith("gpt2_small_linears_M8192")
    names = [g["name"] for g in cfg["gemms"]]
    assert names == ["qkv", "fc", "proj", "probe"]
