"""The GEMM's tile-width choice, checked on the host through the library's
own code (bsg_gemm_tile_width): the width with the fewest idle SMs in the
last wave, weighted by the narrower tiles' lower efficiency."""
import pytest

import verifiable_quantize_rows_gb300 as bsg
from verifiable_quantize_rows_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return bsg.load()


def test_widths_are_valid():
    for M in (1, 100, 1024, 4097, 8192):
        for N in (1, 65, 768, 2304, 3072, 12289, 50304):
            for sms in (1, 148, 152):
                assert bsg.gemm_tile_width(M, N, sms) in (64, 128, 192, 256)


@pytest.mark.parametrize("M,N,want", [
    (8192, 50304, 256),   # LM head: many waves, the wide tile is best
    (8192, 8192, 256),
    (8192, 768, 192),     # proj: 96 pair tiles of 256 need 2 waves of 76; 128 of 192 too, each 3/4 the work
    (8192, 2304, 256),    # qkv: 288 pair tiles, 3.8 waves
    (1024, 1024, 64),     # probe: 32 wide tiles would use a fifth of the SMs
])
def test_choice_on_the_workloads(M, N, want):
    assert bsg.gemm_tile_width(M, N, 152) == want


def test_bad_arguments():
    assert bsg.load().bsg_gemm_tile_width(0, 5, 152) == -1
