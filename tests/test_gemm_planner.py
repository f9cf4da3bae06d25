"""The GEMM's tile choice (mx_gemm_tile_for) against a measured tile sweep, on
the CPU: no GPU is needed.

Every supported tile was timed on one GB300 (152 SMs) at N = 6144 for the M
values below (CUDA graphs of launches over operands rotating beyond L2, us per
launch, K = 2048 / 3072).  The planner's choice must be within 4 % of the
fastest tile at every point: it is a cost model of per-K-step cycles, waves
of tiles over the SMs or SM pairs, and a fixed per-tile cost, so this pins the
model to the measurements it was fitted on."""

import pytest

import mxfp8_norm_quant_gb300 as mx

TILES = [(128, 64), (128, 128), (128, 192), (256, 128), (256, 192), (256, 256)]
# M: ((K=2048 us per tile in TILES order), (K=3072 us ...))
SWEEP = {
    128: ((8.47, 9.58, 10.76, 9.18, 9.77, 10.84), (10.48, 11.96, 13.82, 11.28, 11.90, 13.27)),
    256: ((13.35, 9.57, 10.69, 9.30, 9.90, 10.98), (17.35, 11.99, 13.58, 11.34, 12.02, 13.41)),
    512: ((17.82, 14.67, 10.94, 14.02, 10.40, 11.23), (23.68, 19.32, 13.91, 18.14, 12.54, 13.75)),
    768: ((22.16, 15.04, 16.69, 14.67, 14.97, 11.73), (30.07, 19.39, 21.97, 18.63, 19.28, 14.44)),
    1024: ((30.42, 19.66, 16.85, 18.66, 15.31, 19.88), (42.26, 25.96, 22.06, 24.29, 19.39, 24.48)),
    1536: ((39.39, 24.30, 22.59, 22.91, 20.01, 20.21), (55.16, 32.84, 29.81, 30.77, 25.81, 25.04)),
    2048: ((52.07, 33.02, 28.07, 30.83, 24.21, 27.94), (73.58, 45.50, 37.69, 42.62, 32.43, 35.22)),
    4096: ((95.05, 55.94, 45.45, 52.06, 38.13, 51.84), (136.62, 79.30, 63.00, 74.06, 53.13, 66.33)),
    32768: ((709.0, 381.8, 341.3, 384.8, 272.8, 354.1), (1027.8, 553.1, 487.9, 541.9, 402.8, 486.4)),
}


@pytest.mark.parametrize("m", sorted(SWEEP))
@pytest.mark.parametrize("ki,k", [(0, 2048), (1, 3072)])
def test_choice_is_within_4_percent_of_the_fastest_tile(m, ki, k):
    times = dict(zip(TILES, SWEEP[m][ki]))
    tile = mx.mx_gemm_tile_for(m, 6144, k, 152)
    assert tile in times, tile
    assert times[tile] <= 1.04 * min(times.values()), (tile, times[tile], min(times.values()))


def test_choice_is_a_supported_tile_everywhere():
    for sms in (148, 152, 160):
        for m in (1, 64, 128, 129, 255, 256, 300, 512, 700, 768, 1000, 1024, 2000, 4096, 10000, 32768, 1 << 20):
            for n in (16, 64, 192, 2048, 6144, 6176, 1 << 20):
                for k in (32, 2048, 3072, 1 << 20):
                    assert mx.mx_gemm_tile_for(m, n, k, sms) in TILES


@pytest.mark.parametrize("args", [(-1, 6144, 2048, 152), (128, 8, 2048, 152), (128, 6144, 48, 152),
                                  (128, 6144, 2048, 1), (128, (1 << 20) + 16, 2048, 152)])
def test_invalid_arguments(args):
    with pytest.raises(mx.MxError):
        mx.mx_gemm_tile_for(*args)
