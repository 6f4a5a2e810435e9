"""The item list of the one-read column kernels, walked on the host.

The kernels' bounded waits end because of how the list is ordered (each
quantize item waits for its panel's max items, and CTAs take items in list
order): every (panel, slice) must appear exactly once as a max item and once
as a quantize item, and all of a panel's max items must come before any of its
quantize items.  The quantize items of panel p follow the max items of panel
p + L (the lag), so that the max items have had L panels' worth of time.

This compiles a small host program against the library's own `lag_item` and
`colq_lag` (lag_list.cuh) with nvcc, so the code checked is the code the
kernels run.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "verifiable_quantize_rows_gb300", "csrc")

PROGRAM = r"""
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "lag_list.cuh"

static int walk(int64_t P, int64_t S, int64_t L) {
    std::vector<int64_t> maxpos(P * S, -1), qpos(P * S, -1);
    std::vector<int64_t> lastmax(P, -1), firstq(P, LLONG_MAX);
    for (int64_t it = 0; it < 2 * P * S; ++it) {
        bool q;
        int64_t panel, slice;
        bsg::lag_item(it, P, S, L, q, panel, slice);
        if (panel < 0 || panel >= P || slice < 0 || slice >= S) return 1;
        std::vector<int64_t> &pos = q ? qpos : maxpos;
        if (pos[panel * S + slice] != -1) return 2;   // an item twice
        pos[panel * S + slice] = it;
        if (q) {
            if (it < firstq[panel]) firstq[panel] = it;
        } else if (it > lastmax[panel]) {
            lastmax[panel] = it;
        }
    }
    for (int64_t p = 0; p < P; ++p) {
        if (lastmax[p] < 0 || firstq[p] == LLONG_MAX) return 3;  // a missing item
        if (!(lastmax[p] < firstq[p])) return 4;                 // a quantize item too early
        const int64_t ahead = p + L < P ? p + L : P - 1;
        if (!(lastmax[ahead] < firstq[p])) return 5;             // the lag not kept
    }
    return 0;
}

int main() {
    const int64_t Ps[] = {1, 2, 3, 5, 8, 33, 128, 393};
    const int64_t Ss[] = {1, 2, 3, 6, 64, 128};
    const int64_t Ls[] = {1, 2, 3, 4, 8, 16, 85, 4096};
    int cases = 0;
    for (int64_t P : Ps)
        for (int64_t S : Ss)
            for (int64_t L : Ls) {
                const int r = walk(P, S, L);
                if (r) {
                    std::printf("FAIL %d P=%lld S=%lld L=%lld\n", r, (long long)P, (long long)S,
                                (long long)L);
                    return 1;
                }
                ++cases;
            }
    std::printf("ok %d\n", cases);
    const int64_t rows[] = {16384, 8192, 4097, 768, 64, 1};
    for (int64_t r : rows) std::printf("lag %lld %lld\n", (long long)r, (long long)bsg::colq_lag(r));
    return 0;
}
"""


@pytest.fixture(scope="module")
def lag_program(tmp_path_factory):
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("lag_list")
    src = d / "walk.cu"
    src.write_text(PROGRAM)
    exe = d / "walk"
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe), str(src)],
                   check=True, capture_output=True, text=True)
    return str(exe)


def run(exe, env_lag=None):
    env = dict(os.environ)
    env.pop("BSG_COLQ_LAG", None)
    if env_lag is not None:
        env["BSG_COLQ_LAG"] = env_lag
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.split("\n")
    lags = {int(a): int(b) for _, a, b in (ln.split() for ln in lines if ln.startswith("lag "))}
    return lines[0], lags


def test_every_item_once_and_max_items_first(lag_program):
    first, _ = run(lag_program)
    assert first == "ok %d" % (8 * 6 * 8)


def test_default_lag_holds_about_32_MiB_of_X(lag_program):
    # 128-column panels of f32: rows * 512 bytes each; the lag rounds
    # 32 MiB / panel to the nearest whole panel, at least 2
    _, lags = run(lag_program)
    assert lags == {16384: 4, 8192: 8, 4097: 16, 768: 85, 64: 1024, 1: 65536}
    for rows, L in lags.items():
        assert L >= 2
        assert abs(L * rows * 512 - (32 << 20)) <= rows * 512 / 2


def test_lag_override_and_its_bounds(lag_program):
    _, lags = run(lag_program, "3")
    assert set(lags.values()) == {3}
    _, lags = run(lag_program, "0")      # out of range: the default
    assert lags[16384] == 4
    _, lags = run(lag_program, "5000")   # out of range: the default
    assert lags[8192] == 8
