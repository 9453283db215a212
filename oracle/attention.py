"""Plain float64 definition of one sliding-window GQA attention step at decode.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix (swarmz.net, "Recursive Flint: 40B Open Model, 2.5B
Active", section "The architecture, in plain terms"; futurpulse.com, section
"How does Flint use 39.8B parameters efficiently?"; evermx.com review, Feature
Overview, "Sparse architecture"):
- 35 of the 49 layers use sliding-window attention over the current token and
  the 512 before it (a 513-token window);
- 32 query heads share 4 key/value heads (grouped-query attention), head
  dimension 128;
- queries and keys get a per-head RMSNorm;
- each head has a learned attention sink;
- the sliding-window layers apply rotary position embeddings (RoPE).

Readings taken where the pages are silent:
- projections q = Wq x, k = Wk x, v = Wv x and out = Wo o, no biases;
- the per-head RMSNorm normalises each head's 128 values by their root mean
  square (epsilon 1e-6) and multiplies by a learned 128-vector (one for
  queries, one for keys, shared by the heads);
- RoPE rotates the pairs (i, i + 64), i < 64, of every query and key head by
  the angle pos * base^(-2 i / 128), base 10,000, after the norm;
- the sink of head h is one more logit s_h in that head's softmax
  denominator, with no value: p_j = exp(z_j) / (exp(s_h) + sum_j' exp(z_j'));
- scores z_j = q . k_j / sqrt(128);
- the key/value cache holds bf16 values (the activation type); the new
  token's key and value are rounded to bf16 when stored and the attention
  reads all window entries, the new one included, from the cache;
- query head h uses key/value head h // (32 / 4).
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_to_f64, round_to_bf16


def _f64(a):
    a = np.asarray(a)
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def rms_norm_heads(v: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """v [..., heads, hd] -> v / sqrt(mean(v^2 over hd) + eps) * gamma."""
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * gamma


def rope(v: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotate the pairs (i, i + hd/2) of every head v [heads, hd] by pos * base^(-2 i / hd)."""
    hd = v.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    ang = pos * base ** (-2.0 * i / hd)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., :half], v[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def window_positions(pos: int, window: int) -> np.ndarray:
    """Positions the token at `pos` attends to: max(0, pos - window + 1) .. pos."""
    return np.arange(max(0, pos - window + 1), pos + 1)


def attention_decode(x, pos: int, k_cache, v_cache, W: dict, n_q: int, n_kv: int, hd: int, window: int,
                     rope_base: float = 10000.0, eps: float = 1e-6, use_rope: bool = True, residual: bool = False):
    """One decode step for one sequence.

    x [d] (bf16 bits, f32 or f64); k_cache, v_cache [window][n_kv][hd] bf16
    bits, the entry of position p' in slot p' % window (slots of positions not
    yet reached are ignored); W: wq [n_q hd][d], wk, wv [n_kv hd][d], wo
    [d][n_q hd] (bf16 bits or floats), q_norm, k_norm [hd], sinks [n_q].
    Returns (out [d] float64, k_new [n_kv][hd] and v_new bf16 bit patterns as
    stored in slot pos % window).
    """
    xf = _f64(x)
    wq, wk, wv, wo = (_f64(W[n]) for n in ("wq", "wk", "wv", "wo"))
    q = (wq @ xf).reshape(n_q, hd)
    k = (wk @ xf).reshape(n_kv, hd)
    v = (wv @ xf).reshape(n_kv, hd)
    q = rms_norm_heads(q, _f64(W["q_norm"]), eps)
    k = rms_norm_heads(k, _f64(W["k_norm"]), eps)
    if use_rope:
        q = rope(q, pos, rope_base)
        k = rope(k, pos, rope_base)
    k_new = round_to_bf16(k)
    v_new = round_to_bf16(v)
    kc = _f64(k_cache).copy()
    vc = _f64(v_cache).copy()
    kc[pos % window] = k_new
    vc[pos % window] = v_new
    slots = window_positions(pos, window) % window
    sinks = _f64(W["sinks"])
    group = n_q // n_kv
    o = np.zeros((n_q, hd))
    for h in range(n_q):
        g = h // group
        z = kc[slots, g, :] @ q[h] / np.sqrt(hd)
        m = max(np.max(z), sinks[h])
        p = np.exp(z - m)
        denom = np.exp(sinks[h] - m) + np.sum(p)
        o[h] = (p @ vc[slots, g, :]) / denom
    out = wo @ o.reshape(-1)
    if residual:
        out = out + xf
    to_bits = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return out, to_bits(k_new), to_bits(v_new)
