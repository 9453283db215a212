"""Sliding-window GQA decode attention (moe_attn_decode) against the oracle:
the Flint attention shape (32 query heads over 4 key/value heads of 128, a
513-token window, per-head QK RMSNorm, sinks, RoPE), batches of sequences at
positions from 0 (one key) through the window boundary to the model's
262,144-token context, every output element and the new cache entries.

Bounds: y is bf16 with the layer tolerances (max-abs 2e-2, rel-L2 1e-2); the
new key/value entries are bf16 roundings of fp32 values, so each lies within
one bf16 unit of the oracle's rounding of its float64 value, and the rest of
the cache is untouched.
"""
import numpy as np
import pytest
import torch

from oracle.attention import attention_decode
from parity import to_torch_x
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

A = I.FLINT_ATTN
POS = [0, 5, 511, 512, 513, 1000, 4097, 262143]


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module")
def flint_attn():
    W = I.make_attention(seed=0)
    return W, {k: dev(v) for k, v in W.items()}


def run_case(W, Wd, Bn, pos, use_rope=True, residual=False, seed=1):
    attn = B.MoeAttn(Wd, A["d"], A["n_q"], A["n_kv"], A["window"], max_batch=8, use_rope=use_rope,
                     add_residual=residual)
    kc, vc = I.make_kv_cache(seed, Bn, A["window"])
    x = I.make_tokens(I.FLINT_BF16, seed=seed, T=Bn)
    kd, vd = dev(kc), dev(vc)
    y = attn.decode(to_torch_x(x), dev(np.array(pos, np.int32)), kd, vd)
    torch.cuda.synchronize()
    assert attn.check() == B.MOE_OK
    yg = y.double().cpu().numpy()
    kg, vg = bits(kd), bits(vd)
    worst = {"max_abs": 0.0, "rel_l2": 0.0}
    for b in range(Bn):
        ref, k_new, v_new = attention_decode(x[b], pos[b], kc[b], vc[b], W, A["n_q"], A["n_kv"], A["hd"],
                                             A["window"], use_rope=use_rope, residual=residual)
        err = yg[b] - ref
        rel = np.linalg.norm(err) / np.linalg.norm(ref)
        assert np.max(np.abs(err)) <= 2e-2 and rel <= 1e-2, (b, pos[b], np.max(np.abs(err)), rel)
        worst["max_abs"] = max(worst["max_abs"], float(np.max(np.abs(err))))
        worst["rel_l2"] = max(worst["rel_l2"], float(rel))
        slot = pos[b] % A["window"]
        for got, want in ((kg[b, slot], k_new), (vg[b, slot], v_new)):
            g32 = I.bf16_bits_to_f32(got).astype(np.float64)
            w32 = I.bf16_bits_to_f32(want).astype(np.float64)
            ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(w32), 2.0 ** -126))) - 7)
            assert np.all(np.abs(g32 - w32) <= ulp), (b, np.max(np.abs(g32 - w32) / ulp))
        other = np.ones(A["window"], bool)
        other[slot] = False
        assert np.array_equal(kg[b, other], kc[b, other]) and np.array_equal(vg[b, other], vc[b, other])
    attn.close()
    return worst


@pytest.mark.parametrize("Bn", [1, 3, 8])
def test_flint_attention_decode(flint_attn, Bn):
    W, Wd = flint_attn
    pos = POS[:Bn] if Bn > 1 else [1000]
    print("attention B", Bn, run_case(W, Wd, Bn, pos))


def test_attention_without_rope_with_residual(flint_attn):
    W, Wd = flint_attn
    print("attention no-rope residual", run_case(W, Wd, 4, [3, 600, 70000, 512], use_rope=False, residual=True,
                                                 seed=2))


def test_attention_deterministic_and_graph_replay(flint_attn):
    W, Wd = flint_attn
    attn = B.MoeAttn(Wd, A["d"], A["n_q"], A["n_kv"], A["window"], max_batch=8)
    kc, vc = I.make_kv_cache(3, 2, A["window"])
    x = to_torch_x(I.make_tokens(I.FLINT_BF16, seed=3, T=2))
    pos = dev(np.array([700, 20], np.int32))
    k1, v1 = dev(kc), dev(vc)
    y1 = attn.decode(x, pos, k1, v1)
    s = torch.cuda.Stream()
    k2, v2 = dev(kc), dev(vc)
    y2 = torch.empty_like(x)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        attn.decode(x, pos, k2, v2, y2, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert attn.check() == B.MOE_OK
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    # the same graph at new positions (pos lives in device memory)
    pos.copy_(dev(np.array([701, 21], np.int32)))
    g.replay()
    torch.cuda.synchronize()
    assert attn.check() == B.MOE_OK
    attn.close()
