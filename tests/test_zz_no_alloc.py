"""moe_route_noalloc -- routing for callers that cannot allocate device memory
-- checked against moe_route (the handle-based entry point) on two calls in a
row, through the C ABI.  Collected last so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from parity import GATE_ATOL, to_torch_x
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
