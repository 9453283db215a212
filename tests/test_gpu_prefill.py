"""Prefill-sized batches (tcgen05 grouped-GEMM path) against the oracle."""
import numpy as np
import pytest
import torch

from parity import check_layer, check_routing, to_torch_x
from oracle.moe_oracle import LayerWeights, group_slots, router_logits
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL = I.LayerSpec(d=256, ffn=256, shared_ffn=128, num_experts=16, top_k=4)
NOSHARED = I.LayerSpec(d=256, ffn=128, shared_ffn=0, num_experts=8, top_k=2)


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
    return layer, y, idx, gate


@pytest.fixture(scope="module")
def small():
    L = I.make_layer(SMALL, seed=1)
    return L, B.upload_layer(L)


@pytest.mark.parametrize("T", [1, 17, 100, 300])
def test_small_tc_path(small, T):
    L, dev = small
    x = I.make_tokens(SMALL, seed=T, T=T)
    _, y, idx, gate = run(SMALL, dev, x, 300, path=B.MOE_PATH_TC)
    r = check_layer(L, x, y, idx, gate, SMALL.top_k, "bf16")
    print("small tc", T, r)


def test_no_shared_expert_tc_and_gemv():
    L = I.make_layer(NOSHARED, seed=2)
    dev = B.upload_layer(L)
    x = I.make_tokens(NOSHARED, seed=2, T=200)
    for path in (B.MOE_PATH_TC, B.MOE_PATH_GEMV):
        _, y, idx, gate = run(NOSHARED, dev, x, 200, path=path)
        check_layer(L, x, y, idx, gate, NOSHARED.top_k, "bf16")


def test_tc_and_gemv_paths_agree(flint_bf16):
    spec, L, dev = flint_bf16
    x = I.make_tokens(spec, seed=9, T=64)
    _, y_tc, idx_tc, _ = run(spec, dev, x, 64, path=B.MOE_PATH_TC)
    _, y_gv, idx_gv, gate = run(spec, dev, x, 64, path=B.MOE_PATH_GEMV)
    assert torch.equal(idx_tc, idx_gv)
    check_layer(L, x, y_tc, idx_gv, gate, spec.top_k, "bf16")
    d = (y_tc.double() - y_gv.double()).norm() / y_gv.double().norm()
    assert d < 1e-2


def test_flint_prefill_4096(flint_bf16):
    spec, L, dev = flint_bf16
    T = 4096
    x = I.make_tokens(spec, seed=4096, T=T)
    layer, y, idx, gate = run(spec, dev, x, T)
    # routing, grouping and outputs on every token
    W = LayerWeights(L)
    l = router_logits(x.astype(np.float64) if x.dtype != np.uint16 else
                      (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64), W.Wr, W.b)
    ig = idx.cpu().numpy().astype(np.int64)
    check_routing(l, ig, gate.cpu().numpy().astype(np.float64), spec.top_k)
    offs, tos, so = layer.grouping(T, "cuda")
    counts, offsets, tok_of_slot, slot_of = group_slots(ig, spec.num_experts)
    assert np.array_equal(offs.cpu().numpy(), offsets)
    assert np.array_equal(tos.cpu().numpy(), tok_of_slot)
    assert np.array_equal(so.cpu().numpy(), slot_of)
    r = check_layer(L, x, y, idx, gate, spec.top_k, "bf16")          # every token
    print("flint prefill 4096", r)


def test_flint_prefill_ragged_with_residual(flint_bf16):
    spec, L, dev = flint_bf16
    T = 1000
    x = I.make_tokens(spec, seed=1000, T=T)
    _, y, idx, gate = run(spec, dev, x, T, add_residual=True)
    check_layer(L, x, y, idx, gate, spec.top_k, "bf16", residual=True, tokens=np.arange(0, T, 31))


@pytest.mark.parametrize("which", ["tensor_core_router", "tensor_core_router_2048", "tensor_core_router_100",
                                   "simt_router"])
def test_route_and_grouping_large_batch(flint_bf16, small, which):
    """Routing and grouping on every token: the tensor-core router at T = 100,
    777 and 2048 (one, seven and sixteen 128-token blocks), the SIMT router
    at T = 300; repeated calls give bit-identical routing."""
    if which.startswith("tensor_core_router"):
        spec, L, dev = flint_bf16                # E = 256: tensor-core router
        T = {"tensor_core_router": 777, "tensor_core_router_2048": 2048, "tensor_core_router_100": 100}[which]
    else:
        spec, (L, dev) = SMALL, small            # E = 16: fp32 SIMT router
        T = 300
    x_np = I.make_tokens(spec, seed=55, T=T)
    layer = B.layer_from_spec(spec, dev, T)
    x = to_torch_x(x_np)
    idx, gate, cnt = layer.route(x)
    offs, tos, so = layer.grouping(T, "cuda")
    idx2, gate2, _ = layer.route(x)                  # bit-identical repeats
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2) and torch.equal(gate, gate2)
    W = LayerWeights(L)
    xf = (x_np.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    l = router_logits(xf, W.Wr, W.b)
    ig = idx.cpu().numpy().astype(np.int64)
    check_routing(l, ig, gate.cpu().numpy().astype(np.float64), spec.top_k)
    counts, offsets, tok_of_slot, slot_of = group_slots(ig, spec.num_experts)
    assert np.array_equal(cnt.cpu().numpy(), counts)
    assert np.array_equal(offs.cpu().numpy(), offsets)
    assert np.array_equal(tos.cpu().numpy(), tok_of_slot)
    assert np.array_equal(so.cpu().numpy(), slot_of)


WIDE = I.LayerSpec(d=384, ffn=256, shared_ffn=128, num_experts=16, top_k=4)


@pytest.mark.parametrize("T", [511, 512, 900])
def test_token_major_down_pass_boundary(small, T):
    """From 512 tokens on the down pass runs token-major (256 Wd rows per tile)."""
    L, dev = small
    x = I.make_tokens(SMALL, seed=T, T=T)
    _, y, idx, gate = run(SMALL, dev, x, 900, path=B.MOE_PATH_TC)
    check_layer(L, x, y, idx, gate, SMALL.top_k, "bf16")


def test_down_pass_layouts_agree(small):
    """The same 511 tokens through the weight-major (T = 511) and the token-major
    (T = 512, one extra token) down pass: same routing, outputs equal to fp32
    accumulation order."""
    L, dev = small
    x = I.make_tokens(SMALL, seed=77, T=512)
    _, y_a, idx_a, _ = run(SMALL, dev, x[:511], 512, path=B.MOE_PATH_TC)
    _, y_b, idx_b, _ = run(SMALL, dev, x, 512, path=B.MOE_PATH_TC)
    assert torch.equal(idx_a, idx_b[:511])
    a, b = y_a.double(), y_b[:511].double()
    assert ((a - b).norm() / b.norm()).item() < 2e-3


@pytest.mark.parametrize("spec", [NOSHARED, WIDE], ids=["no_shared", "d384"])
def test_token_major_no_shared_and_narrow_d(spec):
    """No shared expert (token-major pass on routed tiles only), and d = 384
    (not a multiple of 256: the weight-major pass stays in use)."""
    L = I.make_layer(spec, seed=3)
    dev = B.upload_layer(L)
    x = I.make_tokens(spec, seed=3, T=700)
    _, y, idx, gate = run(spec, dev, x, 700, path=B.MOE_PATH_TC)
    check_layer(L, x, y, idx, gate, spec.top_k, "bf16")


def test_token_major_large_batch(small):
    """A large token-major batch (64 slot tiles per expert; the transposed red
    epilogue on every tile); every token against the oracle."""
    L, dev = small
    T = 8192
    x = I.make_tokens(SMALL, seed=8192, T=T)
    _, y, idx, gate = run(SMALL, dev, x, T, path=B.MOE_PATH_TC)
    check_layer(L, x, y, idx, gate, SMALL.top_k, "bf16")
