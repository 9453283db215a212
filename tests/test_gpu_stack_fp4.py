"""A stack of MoE layers with NVFP4 expert weights on the persistent kernel
(every layer in one cooperative launch, T <= 32): bit for bit the same as
chaining the layers one call at a time (the same per-layer arithmetic), the
routing trace equal, and the chain itself against the oracle layer by layer
(teacher-forced: each layer's oracle input is the device's previous output)."""
import numpy as np
import pytest
import torch

from parity import check_layer
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

SPEC = I.LayerSpec(d=1024, ffn=512, shared_ffn=512, num_experts=16, top_k=4, weight="nvfp4", add_residual=True,
                   sigma_w=0.01)
NL = 3


@pytest.fixture(scope="module")
def stack():
    host = [I.make_layer(SPEC, seed=21, layer=l) for l in range(NL)]
    dev = [B.upload_layer(L) for L in host]
    return host, dev


def chain(dev, x):
    """The layers one moe_forward at a time; returns the outputs of every layer."""
    outs, idx = [], []
    cur = x
    for w in dev:
        layer = B.layer_from_spec(SPEC, w, 32, add_residual=True)
        y = torch.empty_like(cur)
        i = torch.empty((cur.shape[0], SPEC.top_k), dtype=torch.int32, device="cuda")
        g = torch.empty((cur.shape[0], SPEC.top_k), dtype=torch.float32, device="cuda")
        layer.forward(cur, y, i, g)
        torch.cuda.synchronize()
        assert layer.check() == B.MOE_OK
        outs.append(y)
        idx.append(i)
        cur = y
    return outs, idx


@pytest.mark.parametrize("T", [1, 8, 32])
def test_fp4_stack_persistent_equals_chain_and_oracle(stack, T):
    host, dev = stack
    st = B.MoeStack(SPEC, dev, max_tokens=32)
    assert st.persistent(T)
    x = I.make_tokens_torch(SPEC, seed=70 + T, T=T, device="cuda")
    y, it, gt = st.forward(x, routing=True)
    torch.cuda.synchronize()
    assert st.check() == B.MOE_OK
    outs, idx = chain(dev, x)
    assert torch.equal(y.view(torch.int16), outs[-1].view(torch.int16))
    for l in range(NL):
        assert torch.equal(it[l], idx[l])
    # teacher-forced oracle check of every layer on the chain's inputs
    ins = [x] + outs[:-1]
    for l in range(NL):
        xn = ins[l].view(torch.int16).cpu().numpy().view(np.uint16)
        check_layer(host[l], xn, outs[l], idx[l], gt[l], SPEC.top_k, "nvfp4", residual=True)


def test_fp4_stack_with_x_trace_runs_per_layer(stack):
    host, dev = stack
    st = B.MoeStack(SPEC, dev, max_tokens=32)
    x = I.make_tokens_torch(SPEC, seed=5, T=16, device="cuda")
    y, xt, it, gt = st.forward(x, trace=True)
    y2 = st.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(xt[-1].view(torch.int16), y.view(torch.int16))
    assert not B.MoeStack(SPEC, dev, max_tokens=64).persistent(33)


def test_flint_fp4_stack_two_layers():
    sp = I.LayerSpec(weight="nvfp4", add_residual=True, sigma_w=0.01)
    dev = [B.upload_layer(I.make_layer(sp, seed=0, layer=l)) for l in range(2)]
    st = B.MoeStack(sp, dev, max_tokens=32)
    x = I.make_tokens_torch(sp, seed=3, T=32, device="cuda")
    y = st.forward(x)
    torch.cuda.synchronize()
    assert st.check() == B.MOE_OK
    cur = x
    for w in dev:
        layer = B.layer_from_spec(sp, w, 32, add_residual=True)
        nxt = torch.empty_like(cur)
        layer.forward(cur, nxt)
        cur = nxt
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), cur.view(torch.int16))
