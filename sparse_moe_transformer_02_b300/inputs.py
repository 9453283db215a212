"""Seeded synthetic inputs for one sparse Mixture-of-Experts FFN layer.

This module only *makes inputs*: Gaussian draws, their rounding to the
storage format (bf16 or NVFP4), and the router bias that skews expert load.
It holds none of the layer's arithmetic (no routing, no expert FFN), so both
the CUDA path and the CPU oracle can be fed from it without sharing code.

Shapes follow the Flint model card as reported on the evermx.com review
("Recursive Flint: Open-Weight MoE Coding Model", section "Sparse
architecture"): 256 routed experts per MoE layer, 6 selected per token, one
always-active shared expert, 47 MoE layers.  The pages give counts, not
widths; the widths used here (hidden 2048, expert FFN 512) are assumptions.

Random streams are keyed by (seed, layer, tensor id, expert) through
numpy's SeedSequence, so any expert's slice can be regenerated alone.
All floating-point draws are float32 N(0, 1) scaled by sigma in float32,
then rounded to the storage format.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

# Stream ids: one per logical tensor of a layer.
TID_X, TID_ROUTER_W, TID_ROUTER_B, TID_GATE, TID_UP, TID_DOWN = 0, 1, 2, 3, 4, 5
TID_SGATE, TID_SUP, TID_SDOWN, TID_ZIPF_PERM = 6, 7, 8, 9

# Router-bias scale for the Zipf(1.1) skewed-load workload.  Fitted once by
# oracle/fit_zipf_alpha.py on a calibration seed (seed 1000) so that the
# realised per-expert load of N(0, 1) tokens, ranked, falls with a log-log
# slope of -1.1 over the 64 most loaded experts.
ZIPF_S = 1.1
ZIPF_ALPHA = 0.5324


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape and storage format of one MoE layer (and its synthetic draws)."""
    d: int = 2048               # hidden width
    ffn: int = 512              # routed expert FFN width
    shared_ffn: int = 512       # shared expert FFN width, 0 = no shared expert
    num_experts: int = 256
    top_k: int = 6
    act: str = "bf16"           # "f32" | "bf16"
    weight: str = "bf16"        # "f32" | "bf16" | "nvfp4"
    add_residual: bool = False
    sigma_w: float = 0.02       # expert weights
    sigma_router: float = 0.02  # router weights
    sigma_x: float = 1.0        # activations
    bias: str = "zero"          # "zero" | "zipf"


# The five workloads; names are what the tests and the bench call them.
TINY_F32 = LayerSpec(d=512, ffn=128, shared_ffn=128, num_experts=64, top_k=6,
                     act="f32", weight="f32", sigma_router=0.05)
FLINT_BF16 = LayerSpec()
FLINT_NVFP4 = LayerSpec(weight="nvfp4")
# The stack's expert weights are drawn N(0, 0.01): the stack's description
# gives no weight scale, and with N(0, 0.02) experts and only a residual add
# between layers the residual stream diverges (each layer adds about
# (0.24 x_rms^2)^2 to x_rms^2, measured on B300 and the oracle: rms 1 -> 5.4 by
# layer 17, overflow near layer 18).  At 0.01 a layer's output is 8x smaller
# and the stream stays at unit scale through 47 layers (rms about 1.02).
FLINT_STACK_ZIPF = LayerSpec(add_residual=True, bias="zipf", sigma_w=0.01)


def _rng(seed: int, layer: int, tensor: int, expert: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=int(seed), spawn_key=(int(layer), int(tensor), int(expert)))
    return np.random.default_rng(ss)


def normal_f32(seed: int, layer: int, tensor: int, shape, sigma: float, expert: int = 0) -> np.ndarray:
    """float32 draws N(0, sigma^2): standard normal draw times sigma, both float32."""
    z = _rng(seed, layer, tensor, expert).standard_normal(shape, dtype=np.float32)
    z *= np.float32(sigma)
    return z


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact float32 value of bfloat16 bit patterns (for building float views of stored weights)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# NVFP4 encoding (e2m1 values, one e4m3 scale per 16 consecutive values along
# the reduction dimension, one float32 scale per matrix).  The pages name the
# NVFP4 checkpoint only (evermx.com review, section "Quantization"); the
# layout and the recipe below are the plainest reading of that format name.
# ---------------------------------------------------------------------------
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _encode_e2m1(v: np.ndarray) -> np.ndarray:
    """Nearest e2m1 code (ties to the even code), saturating at +-6; v float64."""
    mag = np.minimum(np.abs(v), 6.0)
    hi = np.searchsorted(_E2M1_MAG, mag, side="left").clip(0, 7)   # first value >= mag
    lo = (hi - 1).clip(0, 7)
    dlo = mag - _E2M1_MAG[lo]
    dhi = _E2M1_MAG[hi] - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = ((v < 0) & (code != 0)).astype(np.uint8) << 3
    return code | sign


def _encode_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest non-negative e4m3 (finite-only variant) code, ties to even, saturating at 448."""
    v = np.minimum(np.asarray(v, dtype=np.float64), 448.0)
    out = np.zeros(v.shape, dtype=np.uint8)
    sub = v < 2.0 ** -6
    m_sub = np.rint(v[sub] / 2.0 ** -9)                     # 0..8; 8 becomes the smallest normal
    out[sub] = m_sub.astype(np.uint8)
    nv = v[~sub]
    m, e = np.frexp(nv)                                      # nv = m * 2^e, m in [0.5, 1)
    e = e - 1                                                # nv = (2m) * 2^e, 2m in [1, 2)
    mant = np.rint((2.0 * m - 1.0) * 8.0)
    carry = mant >= 8
    mant = np.where(carry, 0, mant)
    e = np.where(carry, e + 1, e)
    code = ((e + 7) << 3) | mant.astype(np.int64)
    out[~sub] = np.minimum(code, 0x7E).astype(np.uint8)
    return out


def _e4m3_code_value(c: np.ndarray) -> np.ndarray:
    c = c.astype(np.int64)
    e = (c >> 3) & 0xF
    m = c & 7
    return np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))


def quantize_nvfp4(w: np.ndarray, s_t=None):
    """Quantise one matrix w[rows][K] (K % 16 == 0) to NVFP4.

    Recipe: tensor scale s_t = amax(w) / (6 * 448); block scale
    s_b = e4m3(amax(block) / (6 * s_t)); value code q = e2m1(w / (s_b * s_t)).
    Returns (packed uint8 [rows][K/2] with element 2i in the low nibble,
    block scales uint8 [rows][K/16] as e4m3 codes, tensor scale as float32).
    ``s_t`` given: quantise rows of a larger matrix whose tensor scale is known.
    """
    w = np.asarray(w, dtype=np.float64)
    rows, K = w.shape
    assert K % 16 == 0
    if s_t is None:
        amax = float(np.max(np.abs(w))) if w.size else 0.0
        s_t = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    s_t = np.float32(s_t)
    blocks = w.reshape(rows, K // 16, 16)
    bmax = np.max(np.abs(blocks), axis=2)
    sb_code = _encode_e4m3(bmax / (6.0 * float(s_t)))
    sb_val = _e4m3_code_value(sb_code)
    denom = sb_val[:, :, None] * float(s_t)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(denom > 0, blocks / np.where(denom > 0, denom, 1.0), 0.0)
    q = _encode_e2m1(ratio).reshape(rows, K)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, sb_code.astype(np.uint8), np.float32(s_t)


# ---------------------------------------------------------------------------
# Layer and token construction
# ---------------------------------------------------------------------------
def _pool():
    return ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))


def _expert_stack(seed, layer, tensor, E, shape, sigma, fmt):
    """E independent per-expert draws, stored as fmt: f32 -> float32, bf16 -> uint16 bits."""
    def one(e):
        z = normal_f32(seed, layer, tensor, shape, sigma, expert=e)
        return bf16_bits(z) if fmt == "bf16" else z
    dtype = np.uint16 if fmt == "bf16" else np.float32
    out = np.empty((E,) + tuple(shape), dtype=dtype)
    with _pool() as ex:
        for e, arr in enumerate(ex.map(one, range(E))):
            out[e] = arr
    return out


def _nvfp4_stack(seed, layer, tensor, E, shape, sigma):
    """Per-expert NVFP4 quantisation of the same float32 draws the bf16 format would use."""
    rows, K = shape

    def one(e):
        return quantize_nvfp4(normal_f32(seed, layer, tensor, shape, sigma, expert=e))
    packed = np.empty((E, rows, K // 2), dtype=np.uint8)
    scales = np.empty((E, rows, K // 16), dtype=np.uint8)
    tsc = np.empty((E,), dtype=np.float32)
    with _pool() as ex:
        for e, (p, s, t) in enumerate(ex.map(one, range(E))):
            packed[e], scales[e], tsc[e] = p, s, t
    return {"packed": packed, "scales": scales, "tscale": tsc}


def zipf_bias(seed: int, layer: int, E: int, s: float = ZIPF_S, alpha: float = ZIPF_ALPHA) -> np.ndarray:
    """Router bias that skews expert load towards a Zipf(s) rank profile.

    Rank r = 1..E gets target share p_r proportional to r^-s; ranks are dealt
    to experts by a seeded permutation; b_e = alpha * ln p_rank(e).
    """
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    perm = _rng(seed, layer, TID_ZIPF_PERM).permutation(E)   # perm[e] = rank index of expert e
    return (alpha * np.log(p[perm])).astype(np.float32)


def make_layer(spec: LayerSpec, seed: int, layer: int = 0) -> dict:
    """All weights of one layer as numpy arrays in their storage format.

    Keys: router_w f32 [E][d], router_b f32 [E]; w_gate, w_up [E][F][d] and
    w_down [E][d][F]; ws_gate, ws_up [Fs][d] and ws_down [d][Fs] (absent when
    shared_ffn == 0).  bf16 tensors are uint16 bit patterns; nvfp4 tensors are
    dicts {"packed", "scales", "tscale"}.
    """
    E, d, F, Fs = spec.num_experts, spec.d, spec.ffn, spec.shared_ffn
    L = {"spec": spec}
    L["router_w"] = normal_f32(seed, layer, TID_ROUTER_W, (E, d), spec.sigma_router)
    if spec.bias == "zipf":
        L["router_b"] = zipf_bias(seed, layer, E)
    else:
        L["router_b"] = np.zeros((E,), dtype=np.float32)
    for name, tid, shape, n in (("w_gate", TID_GATE, (F, d), E), ("w_up", TID_UP, (F, d), E),
                                ("w_down", TID_DOWN, (d, F), E)):
        if spec.weight == "nvfp4":
            L[name] = _nvfp4_stack(seed, layer, tid, n, shape, spec.sigma_w)
        else:
            L[name] = _expert_stack(seed, layer, tid, n, shape, spec.sigma_w, spec.weight)
    if Fs > 0:
        for name, tid, shape in (("ws_gate", TID_SGATE, (Fs, d)), ("ws_up", TID_SUP, (Fs, d)),
                                 ("ws_down", TID_SDOWN, (d, Fs))):
            if spec.weight == "nvfp4":
                st = _nvfp4_stack(seed, layer, tid, 1, shape, spec.sigma_w)
                L[name] = {"packed": st["packed"][0], "scales": st["scales"][0], "tscale": st["tscale"][:1]}
            else:
                L[name] = _expert_stack(seed, layer, tid, 1, shape, spec.sigma_w, spec.weight)[0]
    return L


# The 4-bit output layer.  The pages put about 0.3B parameters in the output
# head (about 2.5B active with it, about 2.2B without it: evermx.com review,
# Feature Overview, "Sparse architecture"); over the assumed hidden width 2048
# that is a vocabulary of about 146k entries, taken as 146,432 (a multiple of
# 256).  The head is quantised to NVFP4 from N(0, sigma^2) draws.
HEAD_VOCAB = 146432
TID_HEAD = 10


def make_head(seed: int, V: int = HEAD_VOCAB, d: int = 2048, sigma: float = 0.02, chunk: int = 8192) -> dict:
    """NVFP4 output layer [V][d]: {"packed" [V][d/2], "scales" [V][d/16], "tscale" [1]}.
    Rows are drawn in chunks (each chunk its own stream) and quantised with the
    matrix's tensor scale."""
    starts = list(range(0, V, chunk))

    def draw(i):
        return normal_f32(seed, 0, TID_HEAD, (min(chunk, V - starts[i]), d), sigma, expert=i)
    with _pool() as ex:
        amax = max(ex.map(lambda i: float(np.max(np.abs(draw(i)))), range(len(starts))))
    s_t = np.float32(amax / (6.0 * 448.0))
    packed = np.empty((V, d // 2), dtype=np.uint8)
    scales = np.empty((V, d // 16), dtype=np.uint8)

    def one(i):
        p, sc, _ = quantize_nvfp4(draw(i), s_t=s_t)
        r0 = starts[i]
        packed[r0:r0 + p.shape[0]] = p
        scales[r0:r0 + p.shape[0]] = sc
    with _pool() as ex:
        list(ex.map(one, range(len(starts))))
    return {"packed": packed, "scales": scales, "tscale": np.array([s_t], dtype=np.float32)}


def make_tokens(spec: LayerSpec, seed: int, T: int, layer: int = 0) -> np.ndarray:
    """Activations x[T][d], N(0, sigma_x^2): float32, or uint16 bf16 bits when spec.act == 'bf16'."""
    z = normal_f32(seed, layer, TID_X, (T, spec.d), spec.sigma_x)
    return bf16_bits(z) if spec.act == "bf16" else z


def tied_router(spec: LayerSpec, seed: int, layer: int, pairs) -> dict:
    """Layer whose router rows are duplicated for each (src, dst) in pairs, so logits tie exactly."""
    L = make_layer(spec, seed, layer)
    for src, dst in pairs:
        L["router_w"][dst] = L["router_w"][src]
        L["router_b"][dst] = L["router_b"][src]
    return L


def make_layer_torch(spec: LayerSpec, seed: int, layer: int, device) -> dict:
    """One layer drawn on a torch device (bf16 or fp32 storage), keyed by the
    moe_weights field names: same distributions as ``make_layer`` but torch's
    generator, so full-size stacks are made in seconds.  Router weights are
    fp32; the Zipf bias, when asked for, is the same as ``make_layer``'s."""
    import torch
    assert spec.weight in ("bf16", "f32")
    E, d, F, Fs = spec.num_experts, spec.d, spec.ffn, spec.shared_ffn
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000 + int(layer))
    dt = torch.bfloat16 if spec.weight == "bf16" else torch.float32
    w = {"router_w": torch.randn(E, d, generator=g, device=device) * spec.sigma_router}
    if spec.bias == "zipf":
        w["router_b"] = torch.from_numpy(zipf_bias(seed, layer, E)).to(device)
    else:
        w["router_b"] = torch.zeros(E, device=device)
    shapes = [("w_gate", (E, F, d)), ("w_up", (E, F, d)), ("w_down", (E, d, F))]
    if Fs > 0:
        shapes += [("ws_gate", (Fs, d)), ("ws_up", (Fs, d)), ("ws_down", (d, Fs))]
    for name, shape in shapes:
        w[name] = (torch.randn(*shape, generator=g, device=device) * spec.sigma_w).to(dt)
    return w


def make_tokens_torch(spec: LayerSpec, seed: int, T: int, device):
    """Activations x[T][d] N(0, sigma_x^2) drawn on a torch device, in the spec's activation type."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 7919 + 17)
    x = torch.randn(T, spec.d, generator=g, device=device) * spec.sigma_x
    return x.to(torch.bfloat16) if spec.act == "bf16" else x


# ---------------------------------------------------------------------------
# Sliding-window attention of the Flint decoder (swarmz.net, "Recursive Flint:
# 40B Open Model, 2.5B Active", section "The architecture, in plain terms"):
# 32 query heads over 4 key/value heads of dimension 128, a 513-token window.
# ---------------------------------------------------------------------------
FLINT_ATTN = {"d": 2048, "n_q": 32, "n_kv": 4, "hd": 128, "window": 513}
TID_WQ, TID_WK, TID_WV, TID_WO, TID_QN, TID_KN, TID_SINK, TID_KC, TID_VC = 20, 21, 22, 23, 24, 25, 26, 27, 28


def make_attention(seed: int, layer: int = 0, d: int = 2048, n_q: int = 32, n_kv: int = 4, hd: int = 128,
                   sigma: float = 0.02) -> dict:
    """Attention weights: wq [n_q hd][d], wk, wv [n_kv hd][d], wo [d][n_q hd] as bf16 bit patterns
    (N(0, sigma^2)); q_norm, k_norm [hd] float32 around 1 (1 + N(0, 0.1^2)); sinks [n_q] float32 N(0, 1)."""
    W = {}
    for name, tid, shape in (("wq", TID_WQ, (n_q * hd, d)), ("wk", TID_WK, (n_kv * hd, d)),
                             ("wv", TID_WV, (n_kv * hd, d)), ("wo", TID_WO, (d, n_q * hd))):
        W[name] = bf16_bits(normal_f32(seed, layer, tid, shape, sigma))
    W["q_norm"] = (1.0 + normal_f32(seed, layer, TID_QN, (hd,), 0.1)).astype(np.float32)
    W["k_norm"] = (1.0 + normal_f32(seed, layer, TID_KN, (hd,), 0.1)).astype(np.float32)
    W["sinks"] = normal_f32(seed, layer, TID_SINK, (n_q,), 1.0)
    return W


def make_kv_cache(seed: int, B: int, window: int, n_kv: int = 4, hd: int = 128, layer: int = 0):
    """Key and value ring buffers [B][window][n_kv][hd] as bf16 bit patterns: keys N(0, 1) (the scale of
    normalised keys), values N(0, 0.8^2) (the scale of Wv x for N(0, 1) activations and N(0, 0.02^2) weights)."""
    k = bf16_bits(normal_f32(seed, layer, TID_KC, (B, window, n_kv, hd), 1.0))
    v = bf16_bits(normal_f32(seed, layer, TID_VC, (B, window, n_kv, hd), 0.8))
    return k, v
