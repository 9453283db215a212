"""The 47-layer stack through moe_stack_forward: the persistent decode kernel
(every layer in one launch, T <= 8) and the per-layer path (T = 16), on the
Flint shape with Zipf-skewed routing and residual adds.

Every layer is checked against the oracle on all tokens, fed the layer input
the GPU actually used (the kernel's trace of the residual stream), within the
single-layer bounds; routing indices bit-exact where the k-th/(k+1)-th gap
exceeds 1e-4.  The persistent kernel sums each token's expert outputs in a
fixed order, so two runs agree bit for bit.
"""
import numpy as np
import pytest
import torch

from parity import check_layer, host_layer
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

N_LAYERS = 47
SEED = 11


@pytest.fixture(scope="module")
def stack47():
    spec = I.FLINT_STACK_ZIPF
    layers = [I.make_layer_torch(spec, seed=SEED, layer=l, device="cuda") for l in range(N_LAYERS)]
    st = B.MoeStack(spec, layers, max_tokens=64)
    yield spec, layers, st
    st.close()
    del layers
    torch.cuda.empty_cache()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def check_trace(spec, layers, xt, it, gt, label):
    worst = {"max_abs": 0.0, "rel_l2": 0.0, "gate_err": 0.0, "near_ties": 0}
    for l in range(len(layers)):
        r = check_layer(host_layer(layers[l]), bits(xt[l]), xt[l + 1], it[l], gt[l], spec.top_k, "bf16",
                        residual=True)
        for key in ("max_abs", "rel_l2", "gate_err"):
            worst[key] = max(worst[key], r[key])
        worst["near_ties"] += r["near_ties"]
    print(label, worst)


@pytest.mark.parametrize("T", [1, 5, 8])
def test_persistent_stack_against_oracle(stack47, T):
    spec, layers, st = stack47
    assert st.persistent(T)
    x = I.make_tokens_torch(spec, seed=SEED + T, T=T, device="cuda")
    y, xt, it, gt = st.forward(x, trace=True)
    torch.cuda.synchronize()
    assert st.check() == B.MOE_OK
    assert torch.equal(xt[0], x) and torch.equal(xt[-1], y)
    check_trace(spec, layers, xt, it, gt, f"persistent T={T}")


def test_persistent_stack_is_deterministic_and_graph_capturable(stack47):
    spec, layers, st = stack47
    T = 8
    x = I.make_tokens_torch(spec, seed=99, T=T, device="cuda")
    s = torch.cuda.Stream()
    y1 = st.forward(x, stream=s)
    s.synchronize()
    y2 = torch.empty_like(x)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st.forward(x, y2, stream=s)
    for _ in range(2):
        y2.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert st.check() == B.MOE_OK
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_stack_per_layer_path(stack47):
    spec, layers, st = stack47
    T = 16
    assert not st.persistent(T)
    x = I.make_tokens_torch(spec, seed=SEED + T, T=T, device="cuda")
    y, xt, it, gt = st.forward(x, trace=True)
    torch.cuda.synchronize()
    assert st.check() == B.MOE_OK
    assert torch.equal(xt[-1], y)
    check_trace(spec, layers, xt, it, gt, f"per-layer T={T}")
