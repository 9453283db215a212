"""The 47-layer stack with residual adds and Zipf-skewed routing (full width,
T = 2048), chained on the GPU exactly as the bench runs it (layer l + 1 reads
layer l's output).  Every layer is checked against the oracle fed the GPU's
own input to that layer, on 64 seeded sampled tokens (teacher forcing), within
the single-layer bounds; the oracle's own 47-layer chain on the same tokens is
compared at the end and its rel-L2 reported (a one-unit bf16 difference in the
residual stream can move a later near-tie, so the per-layer check is the gate).

The Flint stack is 47 MoE layers (swarmz.net, "Recursive Flint: 40B Open
Model, 2.5B Active", section "The architecture, in plain terms").  Layers are
drawn on the device one at a time and freed after use; the oracle reads the
routed experts it needs from the device.
"""
import numpy as np
import pytest
import torch

from parity import check_layer, host_layer, to_f64
from oracle.formats import round_to_bf16
from oracle.moe_oracle import LayerWeights, moe_forward
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

N_LAYERS = 47
T = 2048
N_SAMPLE = 64


def bits_of(v: np.ndarray) -> np.ndarray:
    """float64 values that are bf16 values -> uint16 bit patterns (exact)."""
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def gpu_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def test_stack47_zipf_layers_teacher_forced():
    spec = I.FLINT_STACK_ZIPF
    seed = 3
    x = I.make_tokens_torch(spec, seed=seed, T=T, device="cuda")
    sample = np.sort(np.random.default_rng(1).choice(T, N_SAMPLE, replace=False))
    sample[-1] = T - 1
    x_ref = None                           # the oracle's own chain on the sampled tokens
    worst = {"max_abs": 0.0, "rel_l2": 0.0, "gate_err": 0.0, "near_ties": 0}
    per_layer = []
    for l in range(N_LAYERS):
        dev = I.make_layer_torch(spec, seed=seed, layer=l, device="cuda")
        layer = B.layer_from_spec(spec, dev, T)
        idx = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
        y = layer.forward(x, idx=idx, gate=gate)
        torch.cuda.synchronize()
        assert layer.check() == B.MOE_OK, l
        L = host_layer(dev)
        x_np = gpu_bits(x)
        r = check_layer(L, x_np, y, idx, gate, spec.top_k, "bf16", residual=True, tokens=sample, enforce=False)
        print("layer", l, {kk: (round(v, 6) if isinstance(v, float) else v) for kk, v in r.items()}, flush=True)
        per_layer.append(r)
        for key in ("max_abs", "rel_l2", "gate_err"):
            worst[key] = max(worst[key], r[key])
        worst["near_ties"] += r["near_ties"]
        W = LayerWeights(L)
        xin = x_np[sample] if x_ref is None else bits_of(x_ref)
        yref, _, _ = moe_forward(xin, W, spec.top_k, residual=True)
        x_ref = round_to_bf16(yref)
        layer.close()
        del dev, L, W
        x = y
    yg = to_f64(x)[sample]
    rel = float(np.linalg.norm(yg - x_ref) / np.linalg.norm(x_ref))
    print("stack47 per-layer worst", worst, "| chained rel-L2 after 47 layers", rel)
    assert np.all(np.isfinite(yg))
    for l, r in enumerate(per_layer):
        assert r["err_over_bound"] <= 1.0 and r["rel_l2"] <= 1e-2, (l, r)
