"""Decode-sized batches against the oracle: the default path (tcgen05 for bf16
weights, GEMV kernels for fp32) and the weight-streaming GEMV kernels forced
at the Flint shape."""
import numpy as np
import pytest
import torch

from parity import check_layer, check_routing, to_torch_x
from oracle.moe_oracle import LayerWeights, group_slots, router_logits
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu


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
def tiny():
    spec = I.TINY_F32
    L = I.make_layer(spec, seed=0)
    return spec, L, B.upload_layer(L)


@pytest.mark.parametrize("T", [1, 5, 16])
def test_tiny_f32_forward(tiny, T):
    spec, L, dev = tiny
    x = I.make_tokens(spec, seed=0, T=16)[:T]
    _, y, idx, gate = run(spec, dev, x, 16)
    r = check_layer(L, x, y, idx, gate, spec.top_k, "f32")
    print("tiny f32", T, r)


def test_tiny_route_counts_and_grouping(tiny):
    spec, L, dev = tiny
    T = 16
    x_np = I.make_tokens(spec, seed=0, T=T)
    layer = B.layer_from_spec(spec, dev, T)
    x = to_torch_x(x_np)
    idx, gate, cnt = layer.route(x)
    offs, tos, so = layer.grouping(T, "cuda")
    torch.cuda.synchronize()
    W = LayerWeights(L)
    l = router_logits(x_np.astype(np.float64), W.Wr, W.b)
    ig = idx.cpu().numpy().astype(np.int64)
    check_routing(l, ig, gate.cpu().numpy().astype(np.float64), spec.top_k)
    counts, offsets, tok_of_slot, slot_of = group_slots(ig, spec.num_experts)
    assert np.array_equal(cnt.cpu().numpy(), counts)
    assert np.array_equal(offs.cpu().numpy(), offsets)
    assert np.array_equal(tos.cpu().numpy(), tok_of_slot)
    assert np.array_equal(so.cpu().numpy(), slot_of)


def test_tiny_exact_ties_pick_lower_index(tiny):
    spec, _, _ = tiny
    # experts (3, 40), (7, 8) and (12, 60) get identical router rows
    L = I.tied_router(spec, seed=0, layer=0, pairs=[(3, 40), (7, 8), (12, 60)])
    dev = B.upload_layer(L)
    x_np = I.make_tokens(spec, seed=5, T=16)
    layer = B.layer_from_spec(spec, dev, 16)
    idx, gate, _ = layer.route(to_torch_x(x_np))
    ig = idx.cpu().numpy()
    W = LayerWeights(L)
    l = router_logits(x_np.astype(np.float64), W.Wr, W.b)
    for t in range(16):
        s = set(ig[t].tolist())
        assert not ({40, 8, 60} & s) or ({3, 7, 12} & s), (t, ig[t])
        for lo, hi in ((3, 40), (7, 8), (12, 60)):
            if hi in s:
                assert lo in s and list(ig[t]).index(lo) < list(ig[t]).index(hi)
    check_routing(l, ig.astype(np.int64), gate.cpu().numpy().astype(np.float64), spec.top_k)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_flint_decode_bf16(flint_bf16, T):
    spec, L, dev = flint_bf16
    x = I.make_tokens(spec, seed=100 + T, T=T)
    _, y, idx, gate = run(spec, dev, x, 64)
    r = check_layer(L, x, y, idx, gate, spec.top_k, "bf16")
    print("flint decode", T, r)


@pytest.mark.parametrize("T", [8, 64])
def test_flint_decode_bf16_gemv_path(flint_bf16, T):
    """The GEMV kernels (tensor-pipe mma.sync weight streaming for bf16) at the
    Flint shape, every output element against the oracle."""
    spec, L, dev = flint_bf16
    x = I.make_tokens(spec, seed=200 + T, T=T)
    _, y, idx, gate = run(spec, dev, x, 64, path=B.MOE_PATH_GEMV)
    r = check_layer(L, x, y, idx, gate, spec.top_k, "bf16")
    print("flint decode gemv", T, r)


def test_flint_decode_residual_and_ragged(flint_bf16):
    spec, L, dev = flint_bf16
    x = I.make_tokens(spec, seed=7, T=37)
    _, y, idx, gate = run(spec, dev, x, 64, add_residual=True)
    check_layer(L, x, y, idx, gate, spec.top_k, "bf16", residual=True)


def test_deterministic_and_host_entry(flint_bf16):
    """The GEMV path combines each token's expert outputs in a fixed order, so
    two runs agree bit for bit (the tcgen05 path adds with unordered reductions
    and promises no bitwise repeatability)."""
    spec, L, dev = flint_bf16
    x_np = I.make_tokens(spec, seed=3, T=24)
    layer, y, idx, gate = run(spec, dev, x_np, 64, path=B.MOE_PATH_GEMV)
    y2 = layer.forward(to_torch_x(x_np))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    xh = to_torch_x(x_np, "cpu").pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, yh)
    assert torch.equal(yh.view(torch.int16), y.cpu().view(torch.int16))


def test_zero_tokens_is_noop(tiny):
    spec, _, dev = tiny
    layer = B.layer_from_spec(spec, dev, 16)
    x = torch.zeros((1, spec.d), device="cuda")
    y = torch.full((1, spec.d), 7.0, device="cuda")
    assert B.moe_forward(layer.h, x.data_ptr(), 0, y.data_ptr()) == B.MOE_OK
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    assert B.moe_forward(layer.h, x.data_ptr(), 17, y.data_ptr()) == B.MOE_ERR_INVALID_ARG
    assert B.moe_forward(layer.h, x.data_ptr(), 1, x.data_ptr()) == B.MOE_ERR_INVALID_ARG


def test_long_batch_on_gemv_path_runs_in_passes(tiny):
    spec, L, dev = tiny
    T = 600                                   # > 256 tokens: three passes
    x = I.make_tokens(spec, seed=11, T=T)
    _, y, idx, gate = run(spec, dev, x, T, path=B.MOE_PATH_GEMV)
    check_layer(L, x, y, idx, gate, spec.top_k, "f32", tokens=np.arange(0, T, 7))


def test_cuda_graph_capture_and_replay(flint_bf16):
    spec, L, dev = flint_bf16
    x_np = I.make_tokens(spec, seed=21, T=8)
    layer = B.layer_from_spec(spec, dev, 64)
    x = to_torch_x(x_np)
    y = torch.empty_like(x)
    idx = torch.empty((8, spec.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((8, spec.top_k), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    layer.forward(x, y, idx, gate, stream=s)          # warm-up outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(x, y, idx, gate, stream=s)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    check_layer(L, x_np, y, idx, gate, spec.top_k, "bf16")


def test_bounded_wait_reports_timeout_and_context_survives(tiny):
    spec, L, dev = tiny
    layer = B.layer_from_spec(spec, dev, 16)
    s = torch.cuda.current_stream().cuda_stream
    assert B.moe_debug_expire_wait(layer.h, 20000, s) == B.MOE_OK
    assert layer.check() == B.MOE_ERR_TIMEOUT
    assert layer.check() == B.MOE_OK                  # the word was cleared
    x = I.make_tokens(spec, seed=0, T=16)
    _, y, idx, gate = run(spec, dev, x, 16)           # the context still works
    check_layer(L, x, y, idx, gate, spec.top_k, "f32")
