"""moe_forward at T <= 8 on the default path: the persistent kernel run as a
stack of one layer (routing, gate/up and down in one cooperative launch).
Every output element against the oracle, the residual add on and off, no
shared expert, the grouping it leaves for moe_get_grouping, routing outputs
requested one at a time, bitwise repeatability and agreement with the
tcgen05 path."""
import numpy as np
import pytest
import torch

from parity import check_layer, to_torch_x
from oracle.moe_oracle import LayerWeights, group_slots
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu

# no shared expert, widths in whole 256-value segments, fewer experts
NOSHARED_256 = I.LayerSpec(d=512, ffn=256, shared_ffn=0, num_experts=32, top_k=4)


def fused_launches(layer, fn):
    """Runs fn() with per-launch timing on and returns the launches per kernel."""
    assert B.moe_profile_enable(layer.h, 1, 64) == B.MOE_OK
    fn()
    torch.cuda.synchronize()
    st, r = B.moe_profile_read(layer.h)
    assert st == B.MOE_OK
    B.moe_profile_enable(layer.h, 0, 0)
    return {k: n for k, (_, n) in r.items() if n}


def forward(layer, x, T, k):
    y = torch.empty_like(x)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    layer.forward(x, y, idx, gate)
    return y, idx, gate


@pytest.mark.parametrize("T,residual", [(1, False), (3, True), (8, False), (8, True)])
def test_fused_layer_matches_oracle(flint_bf16, T, residual):
    spec, L, dev = flint_bf16
    x_np = I.make_tokens(spec, seed=900 + T, T=T)
    layer = B.layer_from_spec(spec, dev, 64, add_residual=residual)
    x = to_torch_x(x_np)
    out = {}
    runs = fused_launches(layer, lambda: out.update(zip("yig", forward(layer, x, T, spec.top_k))))
    assert runs == {"fused": 1}, runs
    assert layer.check() == B.MOE_OK
    r = check_layer(L, x_np, out["y"], out["i"], out["g"], spec.top_k, "bf16", residual=residual)
    print("fused", T, residual, r)


def test_fused_grouping_and_partial_routing_outputs(flint_bf16):
    spec, L, dev = flint_bf16
    T = 7
    x_np = I.make_tokens(spec, seed=77, T=T)
    layer = B.layer_from_spec(spec, dev, 64)
    x = to_torch_x(x_np)
    y, idx, gate = forward(layer, x, T, spec.top_k)
    offs, tos, so = layer.grouping(T, "cuda")
    torch.cuda.synchronize()
    counts, offsets, tok_of_slot, slot_of = group_slots(idx.cpu().numpy().astype(np.int64), spec.num_experts)
    assert np.array_equal(offs.cpu().numpy(), offsets)
    assert np.array_equal(tos.cpu().numpy(), tok_of_slot)
    assert np.array_equal(so.cpu().numpy(), slot_of)
    # only idx, then only gate: the same values, the other buffer untouched
    idx2 = torch.full_like(idx, -5)
    gate2 = torch.full_like(gate, 9.0)
    y2 = torch.empty_like(x)
    assert B.moe_forward(layer.h, x.data_ptr(), T, y2.data_ptr(), idx2.data_ptr(), 0) == B.MOE_OK
    y3 = torch.empty_like(x)
    assert B.moe_forward(layer.h, x.data_ptr(), T, y3.data_ptr(), 0, gate2.data_ptr()) == B.MOE_OK
    torch.cuda.synchronize()
    assert torch.equal(idx2, idx) and torch.equal(gate2, gate)
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    assert torch.equal(y3.view(torch.int16), y.view(torch.int16))


def test_fused_is_repeatable_and_agrees_with_tcgen05(flint_bf16):
    """The persistent kernel sums in a fixed order (bit-for-bit repeatable); the
    tcgen05 path computes the same layer within the bf16 tolerance."""
    spec, L, dev = flint_bf16
    T = 8
    x_np = I.make_tokens(spec, seed=31, T=T)
    x = to_torch_x(x_np)
    layer = B.layer_from_spec(spec, dev, 64)
    ys = [forward(layer, x, T, spec.top_k)[0] for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(ys[0].view(torch.int16), yy.view(torch.int16)) for yy in ys[1:])
    tc = B.layer_from_spec(spec, dev, 64, path=B.MOE_PATH_TC)
    y_tc, _, _ = forward(tc, x, T, spec.top_k)
    torch.cuda.synchronize()
    d = (y_tc.double() - ys[0].double()).norm() / ys[0].double().norm()
    assert d < 1e-2, float(d)


def test_fused_without_shared_expert():
    spec = NOSHARED_256
    L = I.make_layer(spec, seed=4)
    dev = B.upload_layer(L)
    layer = B.layer_from_spec(spec, dev, 16)
    for T in (1, 8):
        x_np = I.make_tokens(spec, seed=40 + T, T=T)
        x = to_torch_x(x_np)
        out = {}
        runs = fused_launches(layer, lambda: out.update(zip("yig", forward(layer, x, T, spec.top_k))))
        assert runs == {"fused": 1}, runs
        check_layer(L, x_np, out["y"], out["i"], out["g"], spec.top_k, "bf16")


def test_larger_batches_leave_the_fused_path(flint_bf16):
    spec, L, dev = flint_bf16
    layer = B.layer_from_spec(spec, dev, 64)
    x = to_torch_x(I.make_tokens(spec, seed=9, T=9))
    runs = fused_launches(layer, lambda: forward(layer, x, 9, spec.top_k))
    assert "fused" not in runs and "tc_gateup" in runs, runs
