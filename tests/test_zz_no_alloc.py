"""moe_route_noalloc -- routing for callers that cannot allocate device memory
-- checked against moe_route (the handle-based entry point) on two calls in a
row, through the C ABI.  Collected last so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from parity import GATE_ATOL, check_routing, to_torch_x
from oracle.moe_oracle import LayerWeights, router_logits
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu


def test_noalloc_route_matches_handle_route_twice():
    spec = I.LayerSpec(d=1024, ffn=128, shared_ffn=128, num_experts=256, top_k=6)
    L = I.make_layer(spec, seed=12)
    dev = B.upload_layer(L)
    layer = B.layer_from_spec(spec, dev, 64)
    s = torch.cuda.current_stream().cuda_stream
    for call, (T, seed) in enumerate(((64, 31), (23, 32))):     # two calls in a row, different sizes
        x = to_torch_x(I.make_tokens(spec, seed=seed, T=T))
        idx_ref, gate_ref, cnt_ref = layer.route(x)
        idx = torch.full((T, spec.top_k), -1, dtype=torch.int32, device="cuda")
        gate = torch.full((T, spec.top_k), -1.0, dtype=torch.float32, device="cuda")
        cnt = torch.full((spec.num_experts,), -1, dtype=torch.int32, device="cuda")
        st = B.moe_route_noalloc(x.data_ptr(), T, spec.d, spec.num_experts, spec.top_k, B.MOE_BF16,
                                 dev["router_w"].data_ptr(), dev["router_b"].data_ptr(), idx.data_ptr(),
                                 gate.data_ptr(), cnt.data_ptr(), s)
        assert st == B.MOE_OK, (call, B.moe_status_string(st))
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref), call
        assert torch.equal(cnt, cnt_ref), call
        assert float((gate - gate_ref).abs().max()) <= GATE_ATOL, call
    layer.close()


def test_noalloc_wide_router_f32_without_bias_or_counts():
    """E = 512 experts (16 logits per lane in the top-k), k = 8, fp32
    activations, no router bias and no counts buffer, right after a handle's
    moe_route has left the shared scratch in another state; checked against
    moe_route and against the oracle's routing (bit-exact where the 8th/9th
    logit gap exceeds 1e-4)."""
    spec = I.LayerSpec(d=512, ffn=128, shared_ffn=128, num_experts=512, top_k=8, act="f32", weight="f32",
                       sigma_router=0.05)
    L = I.make_layer(spec, seed=13)
    dev = B.upload_layer(L)
    dev_nob = dict(dev)
    dev_nob["router_b"] = None
    layer = B.layer_from_spec(spec, dev_nob, 64)
    s = torch.cuda.current_stream().cuda_stream
    W = LayerWeights(L)
    for call, (T, seed) in enumerate(((40, 41), (64, 42))):
        x_np = I.make_tokens(spec, seed=seed, T=T)
        x = to_torch_x(x_np)
        idx_ref, gate_ref, _ = layer.route(x)
        idx = torch.full((T, spec.top_k), -1, dtype=torch.int32, device="cuda")
        gate = torch.full((T, spec.top_k), -1.0, dtype=torch.float32, device="cuda")
        st = B.moe_route_noalloc(x.data_ptr(), T, spec.d, spec.num_experts, spec.top_k, B.MOE_F32,
                                 dev["router_w"].data_ptr(), 0, idx.data_ptr(), gate.data_ptr(), 0, s)
        assert st == B.MOE_OK, (call, B.moe_status_string(st))
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref), call
        assert float((gate - gate_ref).abs().max()) <= GATE_ATOL, call
        l = router_logits(x_np.astype(np.float64), W.Wr, np.zeros(spec.num_experts))
        check_routing(l, idx.cpu().numpy().astype(np.int64), gate.cpu().numpy().astype(np.float64), spec.top_k)
    layer.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    x = torch.zeros((65, 1024), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((256, 1024), dtype=torch.float32, device="cuda")
    idx = torch.empty((65, 6), dtype=torch.int32, device="cuda")
    gate = torch.empty((65, 6), dtype=torch.float32, device="cuda")
    st = B.moe_route_noalloc(x.data_ptr(), 65, 1024, 256, 6, B.MOE_BF16, w.data_ptr(), 0, idx.data_ptr(),
                             gate.data_ptr())
    assert st == B.MOE_ERR_INVALID_ARG
    st = B.moe_route_noalloc(x.data_ptr(), 8, 1024, 1024, 6, B.MOE_BF16, w.data_ptr(), 0, idx.data_ptr(),
                             gate.data_ptr())
    assert st == B.MOE_ERR_INVALID_ARG
