"""Pins for the oracle's 4-bit output layer: a hand-built NVFP4 head with
logits worked out by hand, random codes decoded through torch's e4m3 type,
and row selection."""
import json
import os

import numpy as np

from oracle.lm_head import head_weights, lm_head_logits
from sparse_moe_transformer_02_b300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def pack(codes: np.ndarray) -> np.ndarray:
    """Codes [rows][K] -> bytes [rows][K/2], element 2i in the low nibble."""
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def hand_head():
    g = json.load(open(os.path.join(GOLDEN, "lm_head_hand.json")))
    codes = np.zeros((3, 32), dtype=np.uint8)
    codes[0, :16] = 0x2
    codes[1, 0] = 0xF
    codes[1, 16] = 0x7
    codes[2, 0::2] = 0x1
    codes[2, 1::2] = 0x9
    scales = np.array([r["scales"] for r in g["rows"]], dtype=np.uint8)
    return g, pack(codes), scales, np.float32(g["tscale"])


def test_hand_built_head():
    g, packed, scales, ts = hand_head()
    W = head_weights(packed, scales, ts)
    assert np.array_equal(W[0], np.r_[np.ones(16), np.zeros(16)])
    assert W[1, 0] == -3.0 and W[1, 16] == 1.5 and np.count_nonzero(W[1]) == 2
    assert np.array_equal(W[2], np.tile([1.0, -1.0], 16))
    x = np.stack([np.ones(32), np.arange(32.0)]).astype(np.float32)
    assert np.array_equal(lm_head_logits(x, packed, scales, ts), np.array(g["logits"]))
    # bf16 activations: the same values as bit patterns
    xb = I.bf16_bits(x)
    assert np.array_equal(lm_head_logits(xb, packed, scales, ts), np.array(g["logits"]))


def test_random_head_against_torch_formats_and_row_selection():
    """Random codes and block scales decoded through torch's float8_e4m3fn and
    the e2m1 value list; the logits are that matrix times x."""
    import torch
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, size=(8, 64), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, size=(8, 4), dtype=np.uint8)        # finite e4m3 codes
    ts = np.float32(0.375)
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])
    sc = torch.from_numpy(scales.view(np.int8).copy()).view(torch.float8_e4m3fn).double().numpy()
    w = e2m1[codes] * np.repeat(sc, 16, axis=1) * 0.375
    packed = pack(codes)
    assert np.array_equal(head_weights(packed, scales, ts), w)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    full = lm_head_logits(x, packed, scales, ts)
    assert np.allclose(full, x.astype(np.float64) @ w.T, rtol=0, atol=1e-12)
    assert np.array_equal(lm_head_logits(x, packed, scales, ts, rows=[5, 1]), full[:, [5, 1]])
