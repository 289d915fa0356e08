"""The arithmetic-unit microbenchmark (fa_measure_unit_rates): it runs, and
the rates it reports are consistent with each other: a lane's FFMA issues at
most once per clock per SM sub-partition (4 x 32 per SM), the exp2 unit is
slower than the FP32 pipe, and the two-lane FFMA2 does at least as many
FMAs per clock as FFMA."""

import pytest

pytestmark = pytest.mark.gpu


def test_unit_rates_are_consistent(cuda_lib):
    r = cuda_lib.fa_measure_unit_rates(1024)
    assert cuda_lib.fa_last_device_status() == cuda_lib.FA_OK
    ex2, ffma, ffma2 = (r["ex2_per_clk_per_sm"], r["ffma_per_clk_per_sm"],
                        r["ffma2_fma_per_clk_per_sm"])
    assert 0 < ffma <= 128 * 1.02, r
    assert 0 < ex2 < ffma, r
    assert ffma2 >= 0.9 * ffma, r

