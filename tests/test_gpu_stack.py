"""Stacked MoE layers with residual adds and Zipf-skewed routing (full width,
T = 2048), against the oracle on sampled tokens:
  - every layer teacher-forced from the oracle's own input to that layer
    (the GPU runs layer l on the oracle's x_l), within the single-layer bounds;
  - the chain run exactly as the bench runs it (each layer reads the previous
    layer's GPU output), against the oracle's chain, by rel-L2 (bf16 rounding
    of the residual stream may differ by one unit in the last place where the
    two sums straddle a rounding boundary, and such a difference is carried on).
"""
import numpy as np
import pytest
import torch

from parity import check_layer, to_f64, to_torch_x
from oracle.formats import round_to_bf16
from oracle.moe_oracle import LayerWeights, moe_forward, moe_stack
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

N_LAYERS = 4
T = 2048


def bits_of(v: np.ndarray) -> np.ndarray:
    """float64 values that are bf16 values -> uint16 bit patterns (exact)."""
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_stack_of_zipf_layers_with_residual():
    spec = I.FLINT_STACK_ZIPF
    Ls = [I.make_layer(spec, seed=3, layer=l) for l in range(N_LAYERS)]
    layers = [B.layer_from_spec(spec, B.upload_layer(L), T) for L in Ls]
    x_np = I.make_tokens(spec, seed=3, T=T)
    sample = np.sort(np.random.default_rng(1).choice(T, 16, replace=False))
    Ws = [LayerWeights(L) for L in Ls]

    # teacher forcing: layer l on the oracle's own x_l (all T tokens on the GPU,
    # the sampled ones checked)
    xl = x_np
    for l, (layer, W) in enumerate(zip(layers, Ws)):
        idx = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
        y = layer.forward(to_torch_x(xl), idx=idx, gate=gate)
        torch.cuda.synchronize()
        r = check_layer(Ls[l], xl, y, idx, gate, spec.top_k, "bf16", residual=True, tokens=sample)
        print("layer", l, r)
        if l + 1 < N_LAYERS:          # the oracle's x_{l+1} for every token
            yref, _, _ = moe_forward(xl, W, spec.top_k, residual=True)
            xl = bits_of(round_to_bf16(yref))

    # the chain as the bench runs it
    x = to_torch_x(x_np)
    for layer in layers:
        x = layer.forward(x)
    torch.cuda.synchronize()
    for layer in layers:
        assert layer.check() == B.MOE_OK
    ref, _ = moe_stack(x_np, Ws, spec.top_k, tokens=sample)
    yg = to_f64(x)[sample]
    rel = np.linalg.norm(yg - ref) / np.linalg.norm(ref)
    assert np.all(np.isfinite(yg)) and rel <= 1e-2, rel
    print("chained", N_LAYERS, "layers: rel-L2", rel)
