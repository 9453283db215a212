"""Host-only checks of the C ABI: the library loads, exports every function
include/moe.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

from sparse_moe_transformer_02_b300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from sparse_moe_transformer_02_b300 import build
    build.build()
    return B.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(B.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(7):
        assert B.moe_status_string(s).startswith("MOE_")
    assert "UNKNOWN" in B.moe_status_string(99)


def good_cfg(**kw):
    c = dict(d=512, ffn=128, shared_ffn=128, num_experts=64, top_k=6, max_tokens=16,
             act_dtype=B.MOE_F32, weight_dtype=B.MOE_F32, add_residual=0, path=0,
             gemv_max_tokens=0, wait_timeout_ms=0)
    c.update(kw)
    return B.moe_config(**c)


def fake_weights():
    w = B.moe_weights()
    for i, (n, _) in enumerate(B.moe_weights._fields_):
        setattr(w, n, 0x10000 * (i + 1))      # never dereferenced: validation fails first
    return w


@pytest.mark.parametrize("kw, want", [
    (dict(d=0), B.MOE_ERR_INVALID_ARG),
    (dict(top_k=0), B.MOE_ERR_INVALID_ARG),
    (dict(top_k=7, num_experts=6), B.MOE_ERR_INVALID_ARG),
    (dict(max_tokens=0), B.MOE_ERR_INVALID_ARG),
    (dict(path=7), B.MOE_ERR_INVALID_ARG),
    (dict(deterministic=2), B.MOE_ERR_INVALID_ARG),
    (dict(deterministic=-1), B.MOE_ERR_INVALID_ARG),
    (dict(d=100), B.MOE_ERR_UNSUPPORTED),
    (dict(d=6464), B.MOE_ERR_UNSUPPORTED),           # the router's staging limit is d <= 6400
    (dict(ffn=96), B.MOE_ERR_UNSUPPORTED),
    (dict(num_experts=1024), B.MOE_ERR_UNSUPPORTED),
    (dict(top_k=9, num_experts=64), B.MOE_ERR_UNSUPPORTED),
    (dict(act_dtype=B.MOE_F32, weight_dtype=B.MOE_BF16), B.MOE_ERR_UNSUPPORTED),
    (dict(act_dtype=B.MOE_F32, weight_dtype=B.MOE_NVFP4), B.MOE_ERR_UNSUPPORTED),
    (dict(act_dtype=B.MOE_F32, weight_dtype=B.MOE_F32, path=B.MOE_PATH_TC), B.MOE_ERR_UNSUPPORTED),
    (dict(d=192, act_dtype=B.MOE_BF16, weight_dtype=B.MOE_BF16), B.MOE_ERR_UNSUPPORTED),
    (dict(ffn=192, act_dtype=B.MOE_BF16, weight_dtype=B.MOE_BF16), B.MOE_ERR_UNSUPPORTED),
    (dict(act_dtype=B.MOE_BF16, weight_dtype=B.MOE_NVFP4), B.MOE_ERR_UNSUPPORTED),
    (dict(act_dtype=B.MOE_F32, weight_dtype=B.MOE_F32, path=B.MOE_PATH_GEMV, shared_ffn=256),
     B.MOE_ERR_UNSUPPORTED),
])
def test_create_rejects_bad_config(lib, kw, want):
    st, h = B.moe_create(good_cfg(**kw), fake_weights(), 0)
    assert st == want and h is None


def test_create_rejects_bad_weight_pointers(lib):
    w = fake_weights()
    w.router_w = None
    st, h = B.moe_create(good_cfg(), w, 0)
    assert st == B.MOE_ERR_INVALID_ARG and h is None
    w = fake_weights()
    w.w_up = 0x10008                              # not 16-byte aligned
    assert B.moe_create(good_cfg(), w, 0)[0] == B.MOE_ERR_INVALID_ARG
    w = fake_weights()
    w.ws_down = None                              # shared expert declared but missing
    assert B.moe_create(good_cfg(), w, 0)[0] == B.MOE_ERR_INVALID_ARG
    w = fake_weights()
    w.s_gate = None                               # NVFP4 scales missing
    cfg = good_cfg(d=1024, ffn=512, shared_ffn=512, act_dtype=B.MOE_BF16, weight_dtype=B.MOE_NVFP4)
    assert B.moe_create(cfg, w, 0)[0] == B.MOE_ERR_INVALID_ARG


def test_failure_injection_arguments(lib):
    assert B.moe_debug_fail_alloc(-1) == B.MOE_ERR_INVALID_ARG
    assert B.moe_debug_fail_alloc(0) == B.MOE_OK


def test_noalloc_rejects_bad_sizes_on_the_host(lib):
    # every rejection happens before the library looks at the device
    cases = [dict(T=65), dict(T=-1), dict(d=6464), dict(d=96), dict(E=513), dict(k=9), dict(k=7, E=6),
             dict(act=B.MOE_NVFP4)]
    for c in cases:
        a = dict(T=8, d=1024, E=256, k=6, act=B.MOE_BF16)
        a.update(c)
        st = B.moe_route_noalloc(0x1000, a["T"], a["d"], a["E"], a["k"], a["act"], 0x2000, 0, 0x3000, 0x4000)
        assert st == B.MOE_ERR_INVALID_ARG, c


def test_null_handle_calls(lib):
    assert B.moe_destroy(None) == B.MOE_OK
    assert B.moe_forward(None, 0x1000, 1, 0x2000) == B.MOE_ERR_INVALID_ARG
    assert B.moe_route(None, 0x1000, 1, 0x2000, 0x3000) == B.MOE_ERR_INVALID_ARG
    assert B.moe_check(None) == B.MOE_ERR_INVALID_ARG
    assert B.moe_get_grouping(None, 1) == B.MOE_ERR_INVALID_ARG
    assert B.moe_forward_host(None, 0x1000, 1, 0x2000) == B.MOE_ERR_INVALID_ARG
    assert B.moe_debug_expire_wait(None, 100) == B.MOE_ERR_INVALID_ARG
    rc = B.lib().moe_create(None, None, None, None)
    assert rc == B.MOE_ERR_INVALID_ARG
