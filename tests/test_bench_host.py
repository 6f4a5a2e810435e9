"""Host logic of bench.py, without a GPU: the GEMM source digest that guards
the committed ncu counters, the parsing of those counters, the reference
arm's bounded sampling (with a stand-in for the oracle, so that it runs in
milliseconds), and the JSON line's contract built from synthetic stage
times."""
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


@pytest.mark.parametrize("profile,names", [
    (bench.GEMM_PROFILE, {"sq4096", "sq8192", "sq16384", "ragged_adversarial"}),
    (bench.SMALL_GEMM_PROFILE, {"qkv", "fc", "proj"})])
def test_committed_ncu_summaries_parse(profile, names):
    src, per = bench.parse_profile(profile)
    if src is None:
        pytest.skip(f"{profile} not committed")
    assert len(src) == 16
    assert set(per) == names
    assert all(isinstance(v, int) and v > 0 for v in per.values())


def test_profiled_traffic_is_none_for_another_source(monkeypatch):
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic() is None


class FakeClock:
    def __init__(self):
        self.t = 0.0

    def __call__(self):
        return self.t


class FakeOracle:
    """Stands in for the oracle: each call advances a fake clock in
    proportion to its work and records the block it was given."""

    def __init__(self, clock, per_mac=1e-9):
        self.clock = clock
        self.per_mac = per_mac
        self.calls = []

    def num_threads(self):
        return 3

    def bsgemm_i8(self, a, b, relu):
        self.calls.append(("gemm", a.shape[0], b.shape[1]))
        self.clock.t += a.shape[0] * b.shape[1] * a.shape[1] * self.per_mac
        return None, 0

    def probe_hash(self, seed, M, N, K):
        self.calls.append(("probe", M, N))
        self.clock.t += M * N * K * self.per_mac
        return b"\0" * 32, 0


def small_data():
    """Stand-ins with the step's shapes along M and N but K = 8."""
    rng = np.random.default_rng(0)
    out = {}
    for name, M, N, K, relu, _ in bench.unit_list("large"):
        out[name] = (rng.standard_normal((M, 8), dtype=np.float32),
                     rng.standard_normal((8, N), dtype=np.float32), relu)
    return out


def fake(monkeypatch, per_mac=1e-9):
    clock = FakeClock()
    monkeypatch.setattr(bench, "CLOCK", clock)
    return FakeOracle(clock, per_mac)


def test_sample_sizes_scale_to_the_budget(monkeypatch):
    orc = fake(monkeypatch, per_mac=1e-8)
    smp = bench.OracleSample(orc, small_data())
    # a 64 x 64 x 8 block takes 327.68 us: r grows as the square root of the budget
    rows = smp.sizes(seconds=0.01)
    assert rows[:4] == [352] * 4             # 64 * sqrt(0.01 / 327.68e-6), multiple of 8
    rows = smp.sizes(seconds=100.0)
    assert rows[:4] == [4096, 8192, 16384, 12289 // 8 * 8]   # capped at the larger side
    assert rows[4] == 1024                   # the probe: at most all 1024 rows
    rows = smp.sizes(seconds=1e-9)
    assert rows == [8] * 5                   # at least 8


def test_sample_blocks_take_leading_rows_and_columns(monkeypatch):
    orc = fake(monkeypatch)
    data = small_data()
    smp = bench.OracleSample(orc, data)
    ops, t = smp.run(3, 5000)                # ragged: M = 4097 caps the rows
    assert orc.calls[-1] == ("gemm", 4097, 5000)
    assert ops == 2 * 4097 * 5000 * 8 and t > 0
    a, b, _ = smp.cache[(3, 5000)]
    assert np.array_equal(a, data["ragged_adversarial"][0][:4097])
    assert np.array_equal(b, data["ragged_adversarial"][1][:, :5000])


def test_reference_arm_is_bounded_and_complete(monkeypatch):
    import oracle
    orc = fake(monkeypatch)
    monkeypatch.setattr(oracle, "load", lambda: orc)
    monkeypatch.setattr(bench, "oracle_inputs", small_data)
    args = type("A", (), {"steps": 100, "warmup": 5})()
    line = bench.run_reference(args, 0, 1)
    assert bench.run_reference(args, 1, 2) is None          # only rank 0 runs it
    json.dumps(line)
    assert line["impl"] == "reference" and line["steps"] == 100
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 3
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["value"] > 0 and line["higher_is_better"] is True
    # the whole run stays near its two-minute budget of (fake) oracle time
    assert orc.clock.t < 200.0
    # step i ran part i mod 5: the probe every fifth step (+ calibration)
    probe_calls = sum(1 for c in orc.calls if c[0] == "probe")
    assert 20 <= probe_calls <= 23


def test_config_line_names_the_workload():
    cfg = bench.config_dict(1)
    assert cfg["workload"].startswith("large_gemms_4096^3+8192^3+16384^3+ragged")
    names = [g["name"] for g in cfg["gemms"]]
    assert names == ["sq4096", "sq8192", "sq16384", "ragged_adversarial", "probe"]
    small = bench.config_dict(1, "small")
    assert [g["name"] for g in small["gemms"]] == ["qkv", "fc", "proj", "probe"]


def test_quantize_bytes_count_codes_not_f16_operands():
    assert bench.quant_algo_bytes(2, 3, 4) == 5 * (8 + 12) + 4 * 5


def _fake_workload(kind):
    from types import SimpleNamespace
    units = [dict(name=n, M=M, N=N, K=K) for n, M, N, K, _, _ in bench.unit_list(kind)]
    return SimpleNamespace(units=units)


def test_bench_line_keeps_the_contract():
    """The JSON line built from synthetic stage times: every key of the
    contract, the throughput arithmetic, and one line of JSON."""
    W = _fake_workload("large")
    ms = {"sq4096": 0.1, "sq8192": 0.6, "sq16384": 4.4, "ragged_adversarial": 0.5}
    qms = {"sq4096": 0.05, "sq8192": 0.17, "sq16384": 0.68, "ragged_adversarial": 0.19}
    stage_ms = {}
    for u in W.units:
        stage_ms["gemm_" + u["name"]] = [ms[u["name"]]] * 3
        stage_ms["quantize_" + u["name"]] = [qms[u["name"]]] * 3
    stage_ms["probe"] = [0.08]
    peaks = {"bf16_tflops": 1908.6, "bf16_tflops_sustained": 1695.1, "hbm_gbs": 6789.3}
    roof, quant, probe_ms = bench.summarize(W, [6.7], stage_ms, peaks, "measured", 6.7, 1,
                                            bench.GEMM_PROFILE)
    ops = sum(2 * u["M"] * u["N"] * u["K"] for u in W.units)
    assert roof["achieved"] == pytest.approx(ops / (sum(ms.values()) * 1e-3) / 1e12, rel=1e-6)
    assert roof["frac"] == pytest.approx(roof["achieved"] / 1908.6, abs=1e-4)
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] == 1908.6
    assert roof["traffic"] is None or isinstance(roof["traffic"], int)
    qbytes = sum(bench.quant_algo_bytes(u["M"], u["N"], u["K"]) for u in W.units)
    assert quant["achieved_gbs"] == pytest.approx(qbytes / (sum(qms.values()) * 1e-3) / 1e9,
                                                  abs=0.1)
    args = type("A", (), {"steps": 100, "warmup": 5})()
    clk = {"sm_mhz": 1790.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    line = bench.build_line(args, 1, 6.7, roof, quant, probe_ms, 2100.0, clk, 2010, 6000, 400,
                            0.9, (18.3, 27.4), [18.3] * 20, 3355443192, 1610678308, None, "ab",
                            "ab", True, 0, 0, 0.165, roof, quant)
    text = json.dumps(line)
    assert "\n" not in text
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["value"] == pytest.approx(bench.step_ops("large") / (6.7e-3) / 1e12, rel=1e-6)
    assert line["unit"] == "TOPS" and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["n_gpus"] == 1 and line["steps"] == 100 and line["warmup"] == 5
    assert line["config"]["workload"] == bench.WORKLOAD
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in line["roofline"], key
    e2e = line["e2e"]
    assert e2e["unit"] == "TOPS" and e2e["h2d_bytes_per_step"] == 3355443192
    assert e2e["d2h_bytes_per_step"] == 1610678308
    assert e2e["value"] == pytest.approx(bench.step_ops("large") / 18.3e-3 / 1e12, rel=1e-3)
    assert line["gpu_launches"] == 2010 and line["clocks"]["sm_mhz"] == 1790.0


def test_clock_log_summary(tmp_path, monkeypatch):
    """The clocks key from an nvidia-smi log in the sampler's format: the
    median SM clock, the maximum, and every throttle reason seen active
    (malformed lines skipped)."""
    monkeypatch.setenv("BSG_CLOCKS_DIR", str(tmp_path))
    s = bench.ClockSampler(0)
    rows = ["0, 2070, 2070, 176.67, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1785, 2070, 1390.2, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1770, 2070, 1401.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage",
            "0, 1650, 2070, 1399.9, 0x8, Active, Not Active, Not Active, Active"]

    class Proc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.f = open(s.path, "w")
    s.f.write("\n".join(rows) + "\n")
    s.proc = Proc()
    clk = s.stop()
    assert clk["samples"] == 4
    assert clk["sm_mhz"] == pytest.approx((1770 + 1785) / 2)
    assert clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["hw_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(1)
    assert empty.stop()["reasons"] == ["nvidia-smi unavailable"]
