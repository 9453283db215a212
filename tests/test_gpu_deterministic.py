"""The deterministic combine mode of the tcgen05 paths: the down passes store
gate-weighted per-slot rows (each once) and the finalise sums each token's
rows in selection order, then the shared expert's row and x.  Repeated calls
agree bit for bit; the result matches the oracle element by element and the
accumulate mode within its fp32 rounding order.  Weight-major (T < 512) and
token-major (T >= 512) bf16 down passes and the NVFP4 tensor-core path."""
import numpy as np
import pytest
import torch

from parity import check_layer, to_torch_x
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL4 = I.LayerSpec(d=1024, ffn=512, shared_ffn=512, num_experts=16, top_k=4, weight="nvfp4")
NOSHARED = I.LayerSpec(d=512, ffn=256, shared_ffn=0, num_experts=32, top_k=4)


def forward(layer, x, k):
    T = x.shape[0]
    y = torch.empty_like(x)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    layer.forward(x, y, idx, gate)
    torch.cuda.synchronize()
    assert layer.check() == B.MOE_OK
    return y, idx, gate


def run_modes(spec, L, dev, T, seed, residual=False, fmt="bf16"):
    x_np = I.make_tokens(spec, seed=seed, T=T)
    x = to_torch_x(x_np)
    det = B.layer_from_spec(spec, dev, T, path=B.MOE_PATH_TC, deterministic=True, add_residual=residual)
    acc = B.layer_from_spec(spec, dev, T, path=B.MOE_PATH_TC, add_residual=residual)
    ys = [forward(det, x, spec.top_k) for _ in range(3)]
    for y2, _, _ in ys[1:]:
        assert torch.equal(y2.view(torch.int16), ys[0][0].view(torch.int16))
    y, idx, gate = ys[0]
    r = check_layer(L, x_np, y, idx, gate, spec.top_k, fmt, residual=residual)
    y_acc, idx_acc, _ = forward(acc, x, spec.top_k)
    assert torch.equal(idx_acc, idx)
    d = (y_acc.double() - y.double()).norm() / y.double().norm()
    assert d < 1e-2, float(d)
    return r


@pytest.mark.parametrize("T,residual", [(40, False), (300, True), (600, False), (1100, True)])
def test_deterministic_bf16(flint_bf16, T, residual):
    spec, L, dev = flint_bf16
    print("deterministic bf16", T, run_modes(spec, L, dev, T, seed=4000 + T, residual=residual))


def test_deterministic_bf16_no_shared_expert():
    L = I.make_layer(NOSHARED, seed=6)
    dev = B.upload_layer(L)
    for T in (64, 700):
        run_modes(NOSHARED, L, dev, T, seed=T)


@pytest.mark.parametrize("T", [48, 300])
def test_deterministic_nvfp4(T):
    L = I.make_layer(SMALL4, seed=12)
    dev = B.upload_layer(L)
    print("deterministic nvfp4", T, run_modes(SMALL4, L, dev, T, seed=T, fmt="nvfp4"))
