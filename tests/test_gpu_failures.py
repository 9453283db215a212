"""Failure paths on the GPU, made on the host: an injected allocation failure
in moe_create (the library must report MOE_ERR_OOM and hold nothing), and a
handle on a second device when one is visible."""
import pytest
import torch

from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

SPEC = I.LayerSpec(d=256, ffn=128, shared_ffn=128, num_experts=16, top_k=4)


def test_create_reports_oom_and_holds_nothing():
    L = I.make_layer(SPEC, seed=1)
    dev = B.upload_layer(L)
    layer = B.layer_from_spec(SPEC, dev, 64)           # warm: the library's first allocation is behind us
    layer.close()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    w = B.moe_weights()
    for name, _ in B.moe_weights._fields_:
        t = dev.get(name)
        setattr(w, name, t.data_ptr() if t is not None else None)
    cfg = B.moe_config(d=SPEC.d, ffn=SPEC.ffn, shared_ffn=SPEC.shared_ffn, num_experts=SPEC.num_experts,
                       top_k=SPEC.top_k, max_tokens=64, act_dtype=B.MOE_BF16, weight_dtype=B.MOE_BF16,
                       add_residual=0, path=0, gemv_max_tokens=0, wait_timeout_ms=0)
    try:
        assert B.moe_debug_fail_alloc(1) == B.MOE_OK
        st, h = B.moe_create(cfg, w, torch.cuda.current_stream().cuda_stream)
    finally:
        B.moe_debug_fail_alloc(0)
    assert st == B.MOE_ERR_OOM and h is None
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    # the injection was used up: the next create succeeds and works
    st, h = B.moe_create(cfg, w, torch.cuda.current_stream().cuda_stream)
    assert st == B.MOE_OK and h
    assert B.moe_destroy(h) == B.MOE_OK


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs a second visible device")
def test_second_device_routes():
    L = I.make_layer(SPEC, seed=2)
    x = I.make_tokens(SPEC, seed=2, T=16)
    outs = []
    for d in (0, 1):
        with torch.cuda.device(d):
            dev = B.upload_layer(L, f"cuda:{d}")
            layer = B.layer_from_spec(SPEC, dev, 16)
            xt = torch.from_numpy(x.view("int16")).view(torch.bfloat16).to(f"cuda:{d}")
            idx, _, _ = layer.route(xt)
            torch.cuda.synchronize()
            outs.append(idx.cpu())
            layer.close()
    assert torch.equal(outs[0], outs[1])
