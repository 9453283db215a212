"""The skewed-load workload: the fitted router-bias scale gives a Zipf(1.1)
load profile under the oracle's routing, on seeds other than the calibration
seed."""
import pytest

from oracle.fit_zipf_alpha import TARGET, load_slope
from sparse_moe_transformer_02_b300 import inputs as I


@pytest.mark.parametrize("seed", [0, 7])
def test_realised_load_slope(seed):
    assert abs(load_slope(I.ZIPF_ALPHA, seed=seed) - TARGET) < 0.1


def test_bias_zero_is_flat():
    assert abs(load_slope(0.0, seed=3)) < 0.3
