"""Pins for the oracle's sliding-window GQA decode attention: a hand-worked
one-head step, RoPE and RMSNorm properties, sinks at their limits, the window
boundary, single-key attention, and GQA against the equivalent multi-head
layout."""
import json
import os

import numpy as np
import scipy.special

from oracle.attention import attention_decode, rms_norm_heads, rope, window_positions
from sparse_moe_transformer_02_b300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_step():
    g = json.load(open(os.path.join(GOLDEN, "attention_hand.json")))
    W = {n: np.array(g[n], dtype=np.float32) for n in ("wq", "wk", "wv", "wo")}
    W.update(q_norm=np.ones(2, np.float32), k_norm=np.ones(2, np.float32),
             sinks=np.array([g["sink"]], np.float32))
    kc = I.bf16_bits(np.array(g["cache_k"], np.float32))
    vc = I.bf16_bits(np.array(g["cache_v"], np.float32))
    out, k_new, v_new = attention_decode(np.array(g["x"], np.float32), g["pos"], kc, vc, W, n_q=1, n_kv=1, hd=2,
                                         window=3, eps=0.0, use_rope=False)
    assert np.allclose(out, g["out"], rtol=0, atol=1e-15)
    assert np.array_equal(I.bf16_bits_to_f32(k_new).reshape(-1), np.array([0.0, 1.4140625], np.float32))
    assert np.array_equal(I.bf16_bits_to_f32(v_new).reshape(-1), np.array([0.5, 0.0], np.float32))


def test_rope_properties():
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal((4, 128)), rng.standard_normal((4, 128))
    assert np.array_equal(rope(q, 0, 10000.0), q)
    assert np.allclose(np.linalg.norm(rope(q, 77, 10000.0), axis=-1), np.linalg.norm(q, axis=-1))
    # scores depend on the position difference only
    a = np.sum(rope(q, 130, 10000.0) * rope(k, 100, 10000.0), axis=-1)
    b = np.sum(rope(q, 1030, 10000.0) * rope(k, 1000, 10000.0), axis=-1)
    assert np.allclose(a, b, rtol=1e-9, atol=1e-9)
    # pair (0, 64) at pos 1 turns by exactly 1 radian
    e = np.zeros((1, 128))
    e[0, 0] = 1.0
    r = rope(e, 1, 10000.0)
    assert np.allclose([r[0, 0], r[0, 64]], [np.cos(1.0), np.sin(1.0)])


def test_rms_norm_properties():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((3, 128)) * 5
    n = rms_norm_heads(v, np.ones(128), 0.0)
    assert np.allclose(np.sqrt(np.mean(n ** 2, axis=-1)), 1.0)
    assert np.allclose(rms_norm_heads(7.0 * v, np.ones(128), 0.0), n)
    gam = rng.standard_normal(128)
    assert np.allclose(rms_norm_heads(v, gam, 0.0), n * gam)


def small_case(seed, n_q=4, n_kv=2, hd=128, d=64, window=5):
    rng = np.random.default_rng(seed)
    f = lambda *s: (rng.standard_normal(s) * 0.2).astype(np.float32)
    W = {"wq": f(n_q * hd, d), "wk": f(n_kv * hd, d), "wv": f(n_kv * hd, d), "wo": f(d, n_q * hd),
         "q_norm": (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32),
         "k_norm": (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32),
         "sinks": rng.standard_normal(n_q).astype(np.float32)}
    kc = I.bf16_bits(rng.standard_normal((window, n_kv, hd)).astype(np.float32))
    vc = I.bf16_bits(rng.standard_normal((window, n_kv, hd)).astype(np.float32))
    x = I.bf16_bits(rng.standard_normal(d).astype(np.float32))
    return W, kc, vc, x


def test_sinks_at_their_limits_and_plain_softmax():
    W, kc, vc, x = small_case(2, n_q=1, n_kv=1)
    pos, window = 9, 5
    W0 = dict(W, sinks=np.array([-1e30], np.float32))
    out, kn, vn = attention_decode(x, pos, kc, vc, W0, 1, 1, 128, window)
    # the same step written as a plain softmax over the window (no sink)
    xf = I.bf16_bits_to_f32(x).astype(np.float64)
    q = rope(rms_norm_heads((W["wq"].astype(np.float64) @ xf).reshape(1, 128), W["q_norm"].astype(np.float64),
                            1e-6), pos, 10000.0)
    kcf = I.bf16_bits_to_f32(kc).astype(np.float64)
    vcf = I.bf16_bits_to_f32(vc).astype(np.float64)
    kcf[pos % window] = I.bf16_bits_to_f32(kn)
    vcf[pos % window] = I.bf16_bits_to_f32(vn)
    z = kcf[:, 0, :] @ q[0] / np.sqrt(128)
    o = scipy.special.softmax(z) @ vcf[:, 0, :]
    assert np.allclose(out, W["wo"].astype(np.float64) @ o, rtol=1e-12, atol=1e-12)
    big = dict(W, sinks=np.array([1e4], np.float32))
    out_big, _, _ = attention_decode(x, pos, kc, vc, big, 1, 1, 128, window)
    assert np.max(np.abs(out_big)) < 1e-100


def test_window_boundary_and_single_key():
    W, kc, vc, x = small_case(3)
    # pos 2 with window 5: slots 3 and 4 hold no reached position and must not matter
    out, _, _ = attention_decode(x, 2, kc, vc, W, 4, 2, 128, 5)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[3:] = I.bf16_bits(np.full((2, 2, 128), 9.0, np.float32))
    vc2[3:] = I.bf16_bits(np.full((2, 2, 128), -9.0, np.float32))
    out2, _, _ = attention_decode(x, 2, kc2, vc2, W, 4, 2, 128, 5)
    assert np.array_equal(out, out2)
    assert list(window_positions(2, 5)) == [0, 1, 2] and list(window_positions(700, 513)) == list(range(188, 701))
    # position 0 with the sinks at -inf: each head returns its own new value exactly
    Wn = dict(W, sinks=np.full(4, -1e30, np.float32))
    out0, _, vn = attention_decode(x, 0, kc, vc, Wn, 4, 2, 128, 5)
    vnf = I.bf16_bits_to_f32(vn).astype(np.float64)
    o = np.stack([vnf[h // 2] for h in range(4)]).reshape(-1)
    assert np.allclose(out0, W["wo"].astype(np.float64) @ o, rtol=1e-12, atol=1e-12)


def test_gqa_equals_expanded_multi_head():
    W, kc, vc, x = small_case(4, n_q=4, n_kv=2)
    out, _, _ = attention_decode(x, 7, kc, vc, W, 4, 2, 128, 5)
    # four key/value heads, each a copy of its group's head
    rep = lambda w: np.repeat(w.reshape(2, 128, -1), 2, axis=0).reshape(4 * 128, -1)
    We = dict(W, wk=rep(W["wk"]), wv=rep(W["wv"]))
    kce, vce = np.repeat(kc, 2, axis=1), np.repeat(vc, 2, axis=1)
    out_e, _, _ = attention_decode(x, 7, kce, vce, We, 4, 4, 128, 5)
    assert np.allclose(out, out_e, rtol=1e-13, atol=1e-13)
