"""Pins for the CPU oracle: each test ties it to something other than itself.

Brute force on tiny inputs, closed forms, invariants of the definition, and
library routines for the number formats.  A dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of these.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import formats as F
from oracle.moe_oracle import LayerWeights, expert_ffn, group_slots, moe_dense, moe_forward, \
    moe_forward_with_routing, route, select_topk, silu, topk_gates
from sparse_moe_transformer_02_b300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- formats
def test_bf16_decode_fields():
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x0080: 2.0 ** -126, 0x0000: 0.0}
    for bits, v in cases.items():
        assert F.bf16_to_f64(np.uint16(bits)) == v
    assert np.isinf(F.bf16_to_f64(np.uint16(0x7F80)))
    assert np.isnan(F.bf16_to_f64(np.uint16(0x7FC0)))


def test_bf16_decode_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = F.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_round_to_bf16_vs_torch_on_f32():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(200000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e-39).astype(np.float32),
                        # exact ties: bf16 value + half an ulp
                        (I.bf16_bits_to_f32(I.bf16_bits(rng.standard_normal(1000).astype(np.float32)))
                         * np.float32(1 + 2 ** -8)).astype(np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    assert np.array_equal(F.round_to_bf16(v.astype(np.float64)), ref)


def test_round_to_bf16_single_rounding():
    # ties go to the even mantissa
    assert F.round_to_bf16(1 + 2.0 ** -8) == 1.0
    assert F.round_to_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    # just above a tie: one rounding from float64 rounds up (a detour through
    # float32 would first land on the tie and then round down)
    assert F.round_to_bf16(1 + 2.0 ** -8 + 2.0 ** -40) == 1 + 2.0 ** -7
    assert F.round_to_bf16(-(1 + 2.0 ** -8 + 2.0 ** -40)) == -(1 + 2.0 ** -7)


def test_e2m1_table():
    # the FP4 E2M1 value set (OCP Microscaling Formats spec, table of E2M1 values)
    pos = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = F.e2m1_value(np.arange(16))
    assert list(got[:8]) == pos
    assert list(got[8:]) == [-p for p in pos]


def test_e4m3_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = F.e4m3_value(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()
    assert F.e4m3_value(0x7E) == 448.0 and F.e4m3_value(0x08) == 2.0 ** -6
    assert F.e4m3_value(0x01) == 2.0 ** -9 and F.e4m3_value(0x38) == 1.0


def test_nvfp4_decode_hand_block():
    # row of 32 values = 2 blocks; codes 0..15 then 15..0
    codes = np.array(list(range(16)) + list(range(15, -1, -1)), dtype=np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None, :]
    scales = np.array([[0x38, 0x40]], dtype=np.uint8)          # 1.0 and 2.0
    got = F.nvfp4_to_f64(packed, scales, np.float32(0.5))[0]
    tab = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    want = [tab[c] * 1.0 * 0.5 for c in range(16)] + [tab[c] * 2.0 * 0.5 for c in range(15, -1, -1)]
    assert list(got) == want


def test_nvfp4_quantiser_roundtrip():
    rng = np.random.default_rng(3)
    # an exactly representable matrix: w = q * s_b * s_t, every block holding a
    # +-6 (so its amax fixes s_b) and block (0, 0) using s_b = 448 (so the
    # matrix amax fixes s_t)
    rows, K = 8, 64
    nb = K // 16
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    q = (rng.choice(mags, size=(rows, K)) * rng.choice([-1.0, 1.0], size=(rows, K))).reshape(rows, nb, 16)
    q[:, :, 0] = 6.0
    sb_codes = rng.integers(0x30, 0x50, size=(rows, nb)).astype(np.uint8)
    sb_codes[0, 0] = 0x7E
    s_t = 2.0 ** -9
    w = (q * F.e4m3_value(sb_codes)[:, :, None] * s_t).reshape(rows, K)
    p, s, t = I.quantize_nvfp4(w)
    assert float(t) == s_t and (s == sb_codes).all()
    assert np.array_equal(F.nvfp4_to_f64(p, s, t), w)
    # random N(0, 0.02): each value within one block-scale unit (half the
    # widest e2m1 spacing) of the original
    w = rng.standard_normal((64, 256)) * 0.02
    p, s, t = I.quantize_nvfp4(w)
    back = F.nvfp4_to_f64(p, s, t)
    unit = (F.e4m3_value(s) * float(t)).repeat(16, axis=1)
    assert np.all(np.abs(back - w) <= unit + 1e-12)
    assert np.linalg.norm(back - w) / np.linalg.norm(w) < 0.12


# ---------------------------------------------------------------- routing
def test_topk_matches_brute_force_subsets():
    rng = np.random.default_rng(7)
    E, k = 16, 6
    l = rng.standard_normal((24, E))
    l[3, 5] = l[3, 9]                       # an exact tie inside the selected set
    idx = select_topk(l, k)
    for t in range(l.shape[0]):
        best = max(itertools.combinations(range(E), k),
                   key=lambda S: (sum(l[t, e] for e in S), tuple(-e for e in S)))
        assert set(idx[t]) == set(best)
        assert len(set(idx[t])) == k and all(0 <= e < E for e in idx[t])
        vals = l[t, idx[t]]
        assert all(vals[i] > vals[i + 1] or (vals[i] == vals[i + 1] and idx[t, i] < idx[t, i + 1])
                   for i in range(k - 1))


def test_topk_tie_lower_index_wins():
    l = np.zeros((1, 10))
    l[0, [2, 7]] = 5.0
    l[0, [4, 8]] = 3.0
    assert list(select_topk(l, 3)[0]) == [2, 7, 4]


def test_gates_closed_forms():
    rng = np.random.default_rng(11)
    l = rng.standard_normal((50, 64)) * 2
    idx = select_topk(l, 6)
    g = topk_gates(l, idx)
    assert np.allclose(g.sum(1), 1.0, rtol=0, atol=1e-12)
    assert (g > 0).all() and (np.diff(g, axis=1) <= 0).all()
    full = scipy.special.softmax(l, axis=1)
    sel = np.take_along_axis(full, idx, axis=1)
    assert np.allclose(g, sel / sel.sum(1, keepdims=True), rtol=1e-12, atol=0)
    eq = topk_gates(np.zeros((2, 64)), select_topk(np.zeros((2, 64)), 6))
    assert np.allclose(eq, 1 / 6, rtol=0, atol=1e-15)


def test_gates_from_known_logits():
    # one-hot token, router column = ln p: the logits are ln p and the
    # renormalised top-3 gates are p_j / (p_0 + p_1 + p_2)
    p = np.array([0.05, 0.4, 0.1, 0.3, 0.15])
    L = {"router_w": np.log(p)[:, None] * np.ones((1, 4)) * np.array([[1, 0, 0, 0]]),
         "router_b": np.zeros(5), "w_gate": np.zeros((5, 2, 4)), "w_up": np.zeros((5, 2, 4)),
         "w_down": np.zeros((5, 4, 2))}
    W = LayerWeights(L)
    idx, gate, logits = route(np.array([[1.0, 0, 0, 0]]), W, 3)
    assert list(idx[0]) == [1, 3, 4]
    assert np.allclose(gate[0], [0.4 / 0.85, 0.3 / 0.85, 0.15 / 0.85], rtol=1e-14, atol=0)


def test_router_bias_enters_logits():
    L = {"router_w": np.zeros((4, 3)), "router_b": np.array([0.0, 2.0, 1.0, 3.0]),
         "w_gate": np.zeros((4, 2, 3)), "w_up": np.zeros((4, 2, 3)), "w_down": np.zeros((4, 3, 2))}
    idx, gate, _ = route(np.ones((1, 3)), LayerWeights(L), 2)
    assert list(idx[0]) == [3, 1]
    assert np.allclose(gate[0], [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))])


def test_group_slots_against_loops():
    rng = np.random.default_rng(5)
    T, E, k = 37, 12, 4
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    counts, offsets, tok_of_slot, slot_of = group_slots(idx, E)
    want_tok, want_slot = [], np.zeros((T, k), dtype=int)
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    want_slot[t, j] = len(want_tok)
                    want_tok.append(t)
    assert counts.sum() == T * k and list(offsets[1:] - offsets[:-1]) == list(counts)
    assert list(tok_of_slot) == want_tok and (slot_of == want_slot).all()
    assert sorted(slot_of.reshape(-1)) == list(range(T * k))       # a bijection


# ---------------------------------------------------------------- experts
def test_silu_special_values():
    z = np.array([0.0, 40.0, -40.0, 1.3, -0.7])
    s = silu(z)
    assert s[0] == 0.0 and abs(s[1] - 40.0) < 1e-12 and abs(s[2]) < 1e-15
    assert np.allclose(s, z * scipy.special.expit(z), rtol=1e-15, atol=0)


def test_expert_zero_input_gives_zero():
    rng = np.random.default_rng(0)
    Wg, Wu, Wd = rng.standard_normal((6, 4)), rng.standard_normal((6, 4)), rng.standard_normal((4, 6))
    assert np.all(expert_ffn(Wg, Wu, Wd, np.zeros((3, 4))) == 0)


def test_expert_scalar_case():
    wg, wu, wd, x = 0.7, -1.3, 2.1, 0.9
    y = expert_ffn(np.array([[wg]]), np.array([[wu]]), np.array([[wd]]), np.array([[x]]))
    a = wg * x
    assert abs(y[0, 0] - wd * (a / (1 + math.exp(-a))) * (wu * x)) < 1e-15


def test_expert_with_permutation_weights():
    # Wg = c*I, Wu = P (a permutation), Wd = diag(s) Q: E(x) = s * Q(silu(c x) * P x)
    n, c = 5, 0.8
    P = np.eye(n)[[2, 0, 4, 1, 3]]
    Q = np.eye(n)[[1, 3, 0, 4, 2]]
    s = np.array([1.0, -2.0, 0.5, 3.0, -1.0])
    x = np.array([[0.3, -1.2, 2.0, 0.7, -0.4]])
    y = expert_ffn(c * np.eye(n), P, s[:, None] * Q, x)[0]
    inner = (c * x[0]) * scipy.special.expit(c * x[0]) * x[0][[2, 0, 4, 1, 3]]
    assert np.allclose(y, s * inner[[1, 3, 0, 4, 2]], rtol=1e-14, atol=1e-16)


# ---------------------------------------------------------------- whole layer
@pytest.fixture(scope="module")
def tiny():
    spec = I.TINY_F32
    return spec, I.make_layer(spec, seed=0), I.make_tokens(spec, seed=0, T=16)


def test_dense_identity(tiny):
    spec, L, x = tiny
    W = LayerWeights(L)
    y, _, _ = moe_forward(x, W, spec.top_k)
    yd = moe_dense(x, W, spec.top_k)
    assert np.allclose(y, yd, rtol=1e-12, atol=1e-14)


def test_each_token_hits_k_distinct_experts(tiny):
    spec, L, x = tiny
    _, idx, gate = moe_forward(x, LayerWeights(L), spec.top_k)
    for t in range(idx.shape[0]):
        assert len(set(idx[t])) == spec.top_k
    assert np.allclose(gate.sum(1), 1.0, rtol=0, atol=1e-12)


def test_k_equals_E_with_equal_logits_is_mean(tiny):
    spec, L, x = tiny
    L2 = dict(L, router_w=np.zeros_like(L["router_w"]), router_b=np.zeros_like(L["router_b"]))
    W = LayerWeights(L2)
    y, _, gate = moe_forward(x, W, spec.num_experts)
    assert np.allclose(gate, 1.0 / spec.num_experts, rtol=0, atol=1e-15)
    xf = x.astype(np.float64)
    mean = sum(expert_ffn(*W.expert(e), xf) for e in range(spec.num_experts)) / spec.num_experts
    assert np.allclose(y, mean + expert_ffn(*W.shared(), xf), rtol=1e-12, atol=1e-15)


def test_token_permutation_and_batch_invariance(tiny):
    spec, L, x = tiny
    W = LayerWeights(L)
    y, idx, _ = moe_forward(x, W, spec.top_k)
    perm = np.random.default_rng(2).permutation(x.shape[0])
    yp, idxp, _ = moe_forward(x[perm], W, spec.top_k)
    assert np.allclose(yp, y[perm], rtol=1e-13, atol=1e-16) and (idxp == idx[perm]).all()
    y5, _, _ = moe_forward(x[5:6], W, spec.top_k)
    assert np.allclose(y5[0], y[5], rtol=1e-13, atol=1e-16)


def test_expert_relabelling_invariance(tiny):
    spec, L, x = tiny
    W = LayerWeights(L)
    y, idx, _ = moe_forward(x, W, spec.top_k)
    pi = np.random.default_rng(9).permutation(spec.num_experts)     # new expert n is old pi[n]
    L2 = dict(L, router_w=L["router_w"][pi], router_b=L["router_b"][pi],
              w_gate=L["w_gate"][pi], w_up=L["w_up"][pi], w_down=L["w_down"][pi])
    y2, idx2, _ = moe_forward(x, LayerWeights(L2), spec.top_k)
    assert np.allclose(y2, y, rtol=1e-12, atol=1e-15)
    assert (pi[idx2] == idx).all()


def test_shared_expert_always_active(tiny):
    spec, L, x = tiny
    L0 = dict(L, w_gate=np.zeros_like(L["w_gate"]))
    W = LayerWeights(L0)
    y, _, _ = moe_forward(x, W, spec.top_k)
    assert np.allclose(y, expert_ffn(*W.shared(), x.astype(np.float64)), rtol=1e-14, atol=0)


def test_linear_in_down_projection_and_residual(tiny):
    spec, L, x = tiny
    y, _, _ = moe_forward(x, LayerWeights(L), spec.top_k)
    L2 = dict(L, w_down=L["w_down"] * 2, ws_down=L["ws_down"] * 2)
    y2, _, _ = moe_forward(x, LayerWeights(L2), spec.top_k)
    assert np.allclose(y2, 2 * y, rtol=1e-13, atol=0)
    yr, _, _ = moe_forward(x, LayerWeights(L), spec.top_k, residual=True)
    assert np.allclose(yr - y, x.astype(np.float64), rtol=0, atol=1e-14)


def test_forward_with_given_routing_matches(tiny):
    spec, L, x = tiny
    W = LayerWeights(L)
    y, idx, gate = moe_forward(x, W, spec.top_k)
    assert np.allclose(moe_forward_with_routing(x, W, idx, gate), y, rtol=1e-14, atol=0)


# ---------------------------------------------------------------- pages' structure
def test_flint_structure_and_parameter_budget():
    g = json.load(open(os.path.join(GOLDEN, "flint_structure.json")))
    spec = I.FLINT_BF16
    assert spec.num_experts == g["routed_experts_per_layer"]["value"]
    assert spec.top_k == g["experts_selected_per_token"]["value"]
    assert g["shared_experts_always_active"]["value"] == 1 and spec.shared_ffn > 0
    d, Fw = spec.d, spec.ffn
    per_expert = 3 * d * Fw
    n_moe = g["moe_layers"]["value"]
    heads = g["attention_heads"]["value"]
    attn = (heads["q"] * heads["head_dim"] * d * 2 + 2 * heads["kv"] * heads["head_dim"] * d)
    n_layers = n_moe + g["dense_layers"]["value"]
    routed_total = n_moe * spec.num_experts * per_expert
    body_total = routed_total + n_moe * per_expert + n_layers * attn
    # the assumed widths are consistent with the card's totals (embeddings not given)
    assert 0.95 * 39.8e9 < body_total < g["total_params_billion"]["value"] * 1e9
    active = n_moe * (spec.top_k + 1) * per_expert + n_layers * attn
    assert abs(active / (g["active_body_params_billion"]["value"] * 1e9) - 1) < 0.15
