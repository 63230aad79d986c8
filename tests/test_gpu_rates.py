"""gemm_f32_unit_rates: the per-SM unit rates the roofline is built on."""
import pytest

from tests._gpu import lib

pytestmark = pytest.mark.gpu


def test_unit_rates_are_measured_and_plausible():
    g = lib()
    r = g.gemm_f32_unit_rates()
    # a kind::tf32 MMA of M = 128, N = 256, K = 8 is 524288 FLOP; any rate
    # between one such MMA per 512 clocks and one per 32 clocks is a
    # measurement, not a unit mismatch
    assert 1024 <= r["tf32_flop_per_clk_sm"] <= 16384
    # the pair MMA does per SM what the single one does, or more
    assert r["tf32_pair_flop_per_clk_sm"] >= 0.9 * r["tf32_flop_per_clk_sm"]
    # 128 fp32 lanes x 2 FLOP per clock, within what issue can give
    assert 64 <= r["ffma_flop_per_clk_sm"] <= 512
    assert 200 <= r["sm_mhz"] <= 3000
    assert r["num_sms"] >= 2
    # the probe leaves the device usable and the library's error word clear
    assert g.gemm_f32_status(None) == (g.GEMM_F32_OK, 0)
