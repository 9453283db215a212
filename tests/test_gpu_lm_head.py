"""The 4-bit output layer (moe_head_forward) against the oracle, every logit.

Bound, derived from the arithmetic: the kernel's weights are exact (NVFP4
decoded to f16), x is an exact power-of-two rescaling of bf16 values into f16
(exact unless a value falls below the f16 normal range, 2^-14 of the token's
largest: a relative change below 2^-11 of an entry that small), and the
products are exact in the fp32 accumulator, whose rounding over d terms is at
most d 2^-24 sum |x W| and in practice far less; each logit must lie within
64 x 2^-24 x sum_i |x_i W_vi| of the float64 value, and rel-L2 within 1e-5.
"""
import numpy as np
import pytest
import torch

from oracle.lm_head import head_weights
from parity import to_torch_x
from sparse_moe_transformer_02_b300 import binding as B
from sparse_moe_transformer_02_b300 import inputs as I

pytestmark = pytest.mark.gpu


def upload_head(h, device="cuda"):
    return (torch.from_numpy(h["packed"]).to(device), torch.from_numpy(h["scales"]).to(device),
            torch.from_numpy(h["tscale"]).to(device))


def check_logits(h, x_np, logits, chunk=16384):
    got = logits.double().cpu().numpy()
    V = h["packed"].shape[0]
    xf = (x_np.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    worst_rel, err2, ref2 = 0.0, 0.0, 0.0
    for r0 in range(0, V, chunk):
        rows = np.arange(r0, min(V, r0 + chunk))
        W = head_weights(h["packed"][rows], h["scales"][rows], h["tscale"])
        ref = xf @ W.T
        absref = np.abs(xf) @ np.abs(W).T
        err = got[:, rows] - ref
        bound = 64 * 2.0 ** -24 * absref + 1e-30
        assert np.all(np.abs(err) <= bound), float(np.max(np.abs(err) / bound))
        worst_rel = max(worst_rel, float(np.max(np.abs(err) / bound)))
        err2 += float(np.sum(err ** 2))
        ref2 += float(np.sum(ref ** 2))
    rel = (err2 / ref2) ** 0.5
    assert rel <= 1e-5, rel
    return {"rel_l2": rel, "worst_err_over_bound": worst_rel}


@pytest.fixture(scope="module")
def flint_head():
    h = I.make_head(seed=0)
    return h, upload_head(h)


@pytest.mark.parametrize("T", [1, 3, 8, 13])
def test_flint_head_logits(flint_head, T):
    h, (codes, scales, ts) = flint_head
    head = B.LmHead(codes, scales, ts, max_tokens=16)
    spec = I.LayerSpec()
    x_np = I.make_tokens(spec, seed=300 + T, T=T)
    logits = head.forward(to_torch_x(x_np))
    torch.cuda.synchronize()
    assert head.check() == B.MOE_OK
    print("lm_head", T, check_logits(h, x_np, logits))
    head.close()


def test_small_head_and_argument_checks():
    h = I.make_head(seed=5, V=64, d=512, chunk=16)
    codes, scales, ts = upload_head(h)
    head = B.LmHead(codes, scales, ts, max_tokens=8)
    spec = I.LayerSpec(d=512)
    x_np = I.make_tokens(spec, seed=5, T=8)
    # activations spanning many binades: the per-token power-of-two scale must keep them exact
    x_np[3] = (x_np[3].astype(np.uint32) + (20 << 7)).astype(np.uint16)      # x * 2^20
    big = (x_np[5] & 0x7F80) > (31 << 7)
    x_np[5] = np.where(big, (x_np[5].astype(np.uint32) - (30 << 7)), x_np[5]).astype(np.uint16)  # x * 2^-30
    logits = head.forward(to_torch_x(x_np))
    torch.cuda.synchronize()
    assert head.check() == B.MOE_OK
    check_logits(h, x_np, logits)
    x = to_torch_x(x_np)
    out = torch.empty((8, 64), dtype=torch.float32, device="cuda")
    assert B.moe_head_forward(head.h, x.data_ptr(), 9, out.data_ptr()) == B.MOE_ERR_INVALID_ARG
    assert B.moe_head_forward(head.h, x.data_ptr() + 2, 1, out.data_ptr()) == B.MOE_ERR_INVALID_ARG
    assert B.moe_head_forward(head.h, x.data_ptr(), 0, out.data_ptr()) == B.MOE_OK
    head.close()
    assert B.moe_head_create(500, 64, 8, codes.data_ptr(), scales.data_ptr(), ts.data_ptr())[0] == \
        B.MOE_ERR_UNSUPPORTED
    assert B.moe_head_create(512, 48, 8, codes.data_ptr(), scales.data_ptr(), ts.data_ptr())[0] == \
        B.MOE_ERR_UNSUPPORTED
