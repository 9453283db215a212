"""NVFP4 expert weights (decoded in registers) against the oracle."""
import numpy as np
import pytest
import torch

from parity import check_layer, to_torch_x
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL = I.LayerSpec(d=1024, ffn=512, shared_ffn=512, num_experts=16, top_k=4, weight="nvfp4")


def run(spec, dev, x_np, max_tokens, **kw):
    layer = B.layer_from_spec(spec, dev, max_tokens, **kw)
    x = to_torch_x(x_np)
    T = x.shape[0]
    y = torch.empty_like(x)
    idx = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    layer.forward(x, y, idx, gate)
    torch.cuda.synchronize()
    assert layer.check() == B.MOE_OK
    return y, idx, gate


@pytest.mark.parametrize("T", [1, 16, 70])
def test_small_nvfp4(T):
    L = I.make_layer(SMALL, seed=3)
    dev = B.upload_layer(L)
    x = I.make_tokens(SMALL, seed=T, T=T)
    y, idx, gate = run(SMALL, dev, x, 128)
    print("small nvfp4", T, check_layer(L, x, y, idx, gate, SMALL.top_k, "nvfp4"))


def test_flint_nvfp4_decode_32(flint_nvfp4):
    spec, L, dev = flint_nvfp4
    x = I.make_tokens(spec, seed=32, T=32)
    y, idx, gate = run(spec, dev, x, 64)
    print("flint nvfp4 32", check_layer(L, x, y, idx, gate, spec.top_k, "nvfp4"))
