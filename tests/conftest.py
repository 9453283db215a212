import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size case (minutes on the host)")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


# ---------------------------------------------------------------- shared GPU fixtures
@pytest.fixture(scope="session")
def flint_bf16():
    """Flint-shaped bf16 layer (d=2048, 256 experts + shared, F=512, top-6), seed 0: host and device."""
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import inputs as I
    spec = I.FLINT_BF16
    L = I.make_layer(spec, seed=0)
    return spec, L, B.upload_layer(L)


@pytest.fixture(scope="session")
def flint_nvfp4():
    """The same draws quantised to NVFP4 (e2m1 + e4m3 per 16 + fp32 per matrix)."""
    from sparse_moe_transformer_02_b300 import binding as B
    from sparse_moe_transformer_02_b300 import inputs as I
    spec = I.FLINT_NVFP4
    L = I.make_layer(spec, seed=0)
    return spec, L, B.upload_layer(L)
