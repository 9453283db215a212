"""NVFP4 expert weights against the oracle: the tensor-core path (codes decoded
into tensor memory, f16 MMAs) and the weight-streaming GEMV path (decoded in
registers)."""
import numpy as np
import pytest
import torch

from parity import check_layer, to_torch_x
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL = I.LayerSpec(d=1024, ffn=512, shared_ffn=512, num_experts=16, top_k=4, weight="nvfp4")


def run(spec, dev, x_np, max_tokens, **kw):
    layer = B.layer_from_spec(spec, dev, max_tokens, **kw)
    x = to_torch_x(x_np)
    T = x.shape[0]
    y = torch.empty_like(x)
    idx = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    layer.forward(x, y, idx, gate)
    torch.cuda.synchronize()
    assert layer.check() == B.MOE_OK
    return y, idx, gate


PATHS = {"tc": B.MOE_PATH_TC, "gemv": B.MOE_PATH_GEMV}


@pytest.fixture(scope="module")
def small():
    L = I.make_layer(SMALL, seed=3)
    return L, B.upload_layer(L)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("T", [1, 16, 70, 300])
def test_small_nvfp4(small, T, path):
    # T = 300: about 75 slots per expert, so routed tiles of 64 tokens split
    L, dev = small
    x = I.make_tokens(SMALL, seed=T, T=T)
    y, idx, gate = run(SMALL, dev, x, 300, path=PATHS[path])
    print("small nvfp4", path, T, check_layer(L, x, y, idx, gate, SMALL.top_k, "nvfp4"))


@pytest.mark.parametrize("path", list(PATHS))
def test_flint_nvfp4_decode_32(flint_nvfp4, path):
    spec, L, dev = flint_nvfp4
    x = I.make_tokens(spec, seed=32, T=32)
    y, idx, gate = run(spec, dev, x, 64, path=PATHS[path])
    print("flint nvfp4 32", path, check_layer(L, x, y, idx, gate, spec.top_k, "nvfp4"))


def test_nvfp4_paths_agree(flint_nvfp4):
    """Tensor-core and GEMV paths on the same 64 tokens: same routing, outputs
    equal to within the two paths' rounding of intermediates (f16 vs fp32)."""
    spec, L, dev = flint_nvfp4
    x = I.make_tokens(spec, seed=64, T=64)
    y_tc, idx_tc, _ = run(spec, dev, x, 64, path=B.MOE_PATH_TC)
    y_gv, idx_gv, _ = run(spec, dev, x, 64, path=B.MOE_PATH_GEMV)
    assert torch.equal(idx_tc, idx_gv)
    d = (y_tc.double() - y_gv.double()).norm() / y_gv.double().norm()
    assert d < 1e-2, d.item()


def test_nvfp4_large_activations(small):
    """Activations 2^12 times larger (|x| up to ~10^4, |h| ~ 10^7: far outside
    f16).  The tensor-core path scales each f16 row of x by a power of two and
    keeps h / xs^2 in f16, so nothing saturates and the result still matches
    the oracle, relative to the output's magnitude.  The routing is the
    library's (logits of ~10^3 have fp32 rounding far above the near-tie
    gap), checked to be valid: k distinct experts per token, each inside the
    float64 top-k up to the fp32 rounding of those logits.  Gates are
    recomputed in float64 for that routing."""
    from oracle.moe_oracle import LayerWeights, moe_forward_with_routing, router_logits, topk_gates
    from oracle.moe_oracle import _widen
    L, dev = small
    x = I.make_tokens(SMALL, seed=5, T=40)
    xb = (x.astype(np.uint32) + (12 << 7)).astype(np.uint16)       # bf16 exponent + 12: exactly x * 2^12
    y, idx, gate = run(SMALL, dev, xb, 64, path=B.MOE_PATH_TC)
    W = LayerWeights(L)
    xf = _widen(xb)
    ig = idx.cpu().numpy().astype(np.int64)
    l = router_logits(xf, W.Wr, W.b)
    # fp32 logits of this size are exact to about |x| |w| d 2^-24 each
    tol = 4.0 * 2.0 ** -24 * (np.abs(xf) @ np.abs(W.Wr).T).max()
    kth = -np.sort(-l, axis=1)[:, SMALL.top_k - 1]
    for t in range(ig.shape[0]):
        assert len(set(ig[t].tolist())) == SMALL.top_k and ig[t].min() >= 0 and ig[t].max() < SMALL.num_experts
        assert np.all(l[t, ig[t]] >= kth[t] - tol), (t, ig[t])
    y_ref = moe_forward_with_routing(xf, W, ig, topk_gates(l, ig))
    err = y.double().cpu().numpy() - y_ref
    scale = np.abs(y_ref).max()
    assert np.abs(err).max() <= 2e-2 * scale
    assert np.linalg.norm(err) <= 5e-2 * np.linalg.norm(y_ref)


def test_nvfp4_f16_range_is_reported(small):
    """A per-matrix scale large enough to push h / xs^2 past the f16 range:
    the call completes, saturates and moe_check reports MOE_ERR_RANGE."""
    L, dev = small
    dev2 = dict(dev)
    dev2["t_up"] = dev["t_up"] * 1e9
    layer = B.layer_from_spec(SMALL, dev2, 16, path=B.MOE_PATH_TC)
    x = to_torch_x(I.make_tokens(SMALL, seed=7, T=16))
    y = torch.empty_like(x)
    layer.forward(x, y)
    torch.cuda.synchronize()
    assert layer.check() == B.MOE_ERR_RANGE
    assert layer.check() == B.MOE_OK          # the error word is cleared by the check
