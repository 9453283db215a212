"""Pins for the oracle's stack of MoE layers (residual adds, bf16 residual
stream): a hand-computed scalar stack, the all-zero stack, and invariances.

The stack is the 47 MoE layers of the Flint decoder with a residual add
between them (swarmz.net, "Recursive Flint: 40B Open Model, 2.5B Active",
section "The architecture, in plain terms").  A missing or doubled residual,
a missing bf16 rounding between layers or at the end, or feeding layer l + 1
the unrounded sum fails at least one test here.
"""
import json
import os

import numpy as np

from oracle.formats import round_to_bf16
from oracle.moe_oracle import LayerWeights, moe_forward, moe_stack
from sparse_moe_transformer_02_b300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def scalar_layer(v: dict) -> LayerWeights:
    """One layer of width 1 with one routed expert and a shared expert (float32 storage)."""
    f = lambda key, shape: np.full(shape, v[key], dtype=np.float32)
    return LayerWeights({"router_w": f("router_w", (1, 1)), "router_b": np.zeros(1, np.float32),
                         "w_gate": f("w_gate", (1, 1, 1)), "w_up": f("w_up", (1, 1, 1)),
                         "w_down": f("w_down", (1, 1, 1)), "ws_gate": f("ws_gate", (1, 1)),
                         "ws_up": f("ws_up", (1, 1)), "ws_down": f("ws_down", (1, 1))})


def test_scalar_two_layer_stack_by_hand():
    g = json.load(open(os.path.join(GOLDEN, "stack_scalar_two_layer.json")))
    layers = [scalar_layer(v) for v in g["layers"]]
    x0 = np.array([[g["x0"]]], dtype=np.float32)
    x1, idx1 = moe_stack(x0, layers[:1], k=1)
    assert x1[0, 0] == g["x1"]
    assert idx1[0][0, 0] == 0
    x2, idxs = moe_stack(x0, layers, k=1)
    assert x2[0, 0] == g["x2"]
    assert x2[0, 0] != g["x2_if_layer1_unrounded"]
    assert len(idxs) == 2
    # the unrounded sums the file derives are what one layer adds before rounding
    y1, _, _ = moe_forward(x0, layers[0], 1, residual=True)
    assert y1[0, 0] == g["x1_sum_before_rounding"]
    y2, _, _ = moe_forward(np.array([[g["x1"]]]), layers[1], 1, residual=True)
    assert abs(y2[0, 0] - g["x2_sum_before_rounding"]) <= 4e-16


def zero_layer(spec: I.LayerSpec) -> LayerWeights:
    E, d, F, Fs = spec.num_experts, spec.d, spec.ffn, spec.shared_ffn
    z = lambda *s: np.zeros(s, dtype=np.float32)
    return LayerWeights({"router_w": z(E, d), "router_b": z(E), "w_gate": z(E, F, d), "w_up": z(E, F, d),
                         "w_down": z(E, d, F), "ws_gate": z(Fs, d), "ws_up": z(Fs, d), "ws_down": z(d, Fs)})


def test_all_zero_stack_returns_its_input():
    spec = I.LayerSpec(d=64, ffn=64, shared_ffn=64, num_experts=8, top_k=3, act="bf16")
    x = I.make_tokens(spec, seed=4, T=5)                     # bf16 values
    xf = I.bf16_bits_to_f32(x).astype(np.float64)
    for depth in (1, 2, 5):
        out, idxs = moe_stack(x, [zero_layer(spec)] * depth, k=spec.top_k)
        assert np.array_equal(out, xf), depth
        # equal logits: the k lowest expert indices, in order
        assert all(np.array_equal(i, np.tile(np.arange(spec.top_k), (5, 1))) for i in idxs)


def tiny_stack(n_layers: int, seed: int):
    spec = I.LayerSpec(d=64, ffn=64, shared_ffn=64, num_experts=8, top_k=3, act="bf16", weight="bf16",
                       add_residual=True, sigma_w=0.08, sigma_router=0.3)
    return spec, [LayerWeights(I.make_layer(spec, seed=seed, layer=l)) for l in range(n_layers)]


def test_stack_equals_layers_applied_in_turn_with_bf16_rounding():
    """Each layer's output is a bf16 value (the stream is rounded), and the
    stack of n layers is layer n applied to the stack of n - 1."""
    spec, Ws = tiny_stack(3, seed=6)
    x = I.make_tokens(spec, seed=6, T=7)
    prev = I.bf16_bits_to_f32(x).astype(np.float64)
    for n in range(1, 4):
        out, _ = moe_stack(x, Ws[:n], k=spec.top_k)
        assert np.array_equal(round_to_bf16(out), out)       # a bf16 value after every layer
        y, _, _ = moe_forward(prev, Ws[n - 1], spec.top_k, residual=True)
        assert np.array_equal(out, round_to_bf16(y))
        assert not np.allclose(out, prev, atol=1e-3)         # every layer moves the stream
        prev = out


def test_stack_token_permutation_and_sampling():
    spec, Ws = tiny_stack(3, seed=8)
    x = I.make_tokens(spec, seed=8, T=9)
    out, idxs = moe_stack(x, Ws, k=spec.top_k)
    perm = np.random.default_rng(0).permutation(9)
    out_p, idxs_p = moe_stack(x[perm], Ws, k=spec.top_k)
    assert np.array_equal(out_p, out[perm])
    for a, b in zip(idxs, idxs_p):
        assert np.array_equal(b, a[perm])
    sample = [2, 5, 8]
    out_s, _ = moe_stack(x, Ws, k=spec.top_k, tokens=sample)
    assert np.array_equal(out_s, out[sample])
