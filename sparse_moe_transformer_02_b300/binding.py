"""ctypes binding of libmoe (include/moe.h): same function names, argument
marshalling only.  Every step of the layer runs in the library's CUDA
kernels; there is no Python or CPU fallback, and loading fails loudly when
the shared library is missing.

``MoeLayer`` is a convenience wrapper that keeps torch tensors (device memory
and streams) alive for the handle's lifetime and passes their pointers.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_OOM, MOE_ERR_TIMEOUT, MOE_ERR_RANGE = range(7)
MOE_F32, MOE_BF16, MOE_NVFP4 = 0, 1, 2
MOE_PATH_AUTO, MOE_PATH_GEMV, MOE_PATH_TC = 0, 1, 2

EXPORTED = ["moe_status_string", "moe_create", "moe_destroy", "moe_route", "moe_forward",
            "moe_forward_host", "moe_get_grouping", "moe_check", "moe_debug_expire_wait",
            "moe_profile_enable", "moe_profile_read", "moe_route_noalloc", "moe_debug_fail_alloc",
            "moe_stack_create", "moe_stack_destroy", "moe_stack_uses_persistent", "moe_stack_forward",
            "moe_stack_check", "moe_head_create", "moe_head_forward", "moe_head_check", "moe_head_destroy",
            "moe_attn_create", "moe_attn_decode", "moe_attn_check", "moe_attn_destroy"]
KERNEL_NAMES = ["route", "gemv_gateup", "gemv_down", "tc_gather", "tc_gateup", "tc_down", "tc_finalize",
                "fused"]


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "d", "ffn", "shared_ffn", "num_experts", "top_k", "max_tokens", "act_dtype", "weight_dtype",
        "add_residual", "path", "gemv_max_tokens", "wait_timeout_ms", "deterministic")]


class moe_attn_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("d", "n_q", "n_kv", "head_dim", "window", "max_batch", "use_rope",
                                              "add_residual", "wait_timeout_ms")] + \
               [("rope_base", ctypes.c_float), ("eps", ctypes.c_float)]


class moe_attn_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("wq", "wk", "wv", "wo", "q_norm", "k_norm", "sinks")]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_w", "router_b", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down",
        "s_gate", "s_up", "s_down", "ss_gate", "ss_up", "ss_down",
        "t_gate", "t_up", "t_down", "ts_gate", "ts_up", "ts_down")]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so not found at {LIB_PATH}; build it with "
                               "`python -m sparse_moe_transformer_02_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_create.restype = ctypes.c_int
        L.moe_create.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(moe_weights), vp,
                                 ctypes.POINTER(vp)]
        L.moe_destroy.restype = ctypes.c_int
        L.moe_destroy.argtypes = [vp]
        L.moe_route.restype = ctypes.c_int
        L.moe_route.argtypes = [vp, vp, i32, vp, vp, vp, vp]
        L.moe_forward.restype = ctypes.c_int
        L.moe_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp]
        L.moe_forward_host.restype = ctypes.c_int
        L.moe_forward_host.argtypes = [vp, vp, i32, vp, vp]
        L.moe_get_grouping.restype = ctypes.c_int
        L.moe_get_grouping.argtypes = [vp, i32, vp, vp, vp, vp]
        L.moe_check.restype = ctypes.c_int
        L.moe_check.argtypes = [vp, vp]
        L.moe_debug_expire_wait.restype = ctypes.c_int
        L.moe_debug_expire_wait.argtypes = [vp, i32, vp]
        L.moe_profile_enable.restype = ctypes.c_int
        L.moe_profile_enable.argtypes = [vp, i32, i32]
        L.moe_profile_read.restype = ctypes.c_int
        L.moe_profile_read.argtypes = [vp, vp, vp]
        L.moe_stack_create.restype = ctypes.c_int
        L.moe_stack_create.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(moe_weights), i32, vp,
                                       ctypes.POINTER(vp)]
        L.moe_stack_destroy.restype = ctypes.c_int
        L.moe_stack_destroy.argtypes = [vp]
        L.moe_stack_uses_persistent.restype = ctypes.c_int32
        L.moe_stack_uses_persistent.argtypes = [vp, i32]
        L.moe_stack_forward.restype = ctypes.c_int
        L.moe_stack_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
        L.moe_stack_check.restype = ctypes.c_int
        L.moe_stack_check.argtypes = [vp, vp]
        L.moe_debug_fail_alloc.restype = ctypes.c_int
        L.moe_debug_fail_alloc.argtypes = [i32]
        L.moe_attn_create.restype = ctypes.c_int
        L.moe_attn_create.argtypes = [ctypes.POINTER(moe_attn_config), ctypes.POINTER(moe_attn_weights),
                                      ctypes.POINTER(vp)]
        L.moe_attn_decode.restype = ctypes.c_int
        L.moe_attn_decode.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
        L.moe_attn_check.restype = ctypes.c_int
        L.moe_attn_check.argtypes = [vp, vp]
        L.moe_attn_destroy.restype = ctypes.c_int
        L.moe_attn_destroy.argtypes = [vp]
        L.moe_head_create.restype = ctypes.c_int
        L.moe_head_create.argtypes = [i32, i32, i32, vp, vp, vp, i32, ctypes.POINTER(vp)]
        L.moe_head_forward.restype = ctypes.c_int
        L.moe_head_forward.argtypes = [vp, vp, i32, vp, vp]
        L.moe_head_check.restype = ctypes.c_int
        L.moe_head_check.argtypes = [vp, vp]
        L.moe_head_destroy.restype = ctypes.c_int
        L.moe_head_destroy.argtypes = [vp]
        L.moe_route_noalloc.restype = ctypes.c_int
        L.moe_route_noalloc.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        _lib = L
    return _lib


# ---------------------------------------------------------------- C functions, same names
def moe_status_string(s: int) -> str:
    return lib().moe_status_string(int(s)).decode()


status_string = moe_status_string


def moe_create(cfg: moe_config, w: moe_weights, stream: int = 0):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    st = lib().moe_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.c_void_p(stream), ctypes.byref(h))
    return st, h.value


def moe_destroy(h) -> int:
    return lib().moe_destroy(h)


def moe_route(h, x: int, T: int, idx: int, gate: int, counts: int = 0, stream: int = 0) -> int:
    return lib().moe_route(h, x, T, idx, gate, counts or None, stream)


def moe_forward(h, x: int, T: int, y: int, idx_out: int = 0, gate_out: int = 0, stream: int = 0) -> int:
    return lib().moe_forward(h, x, T, y, idx_out or None, gate_out or None, stream)


def moe_forward_host(h, x_host: int, T: int, y_host: int, stream: int = 0) -> int:
    return lib().moe_forward_host(h, x_host, T, y_host, stream)


def moe_get_grouping(h, T: int, offsets: int = 0, tok_of_slot: int = 0, slot_of: int = 0, stream: int = 0) -> int:
    return lib().moe_get_grouping(h, T, offsets or None, tok_of_slot or None, slot_of or None, stream)


def moe_check(h, stream: int = 0) -> int:
    return lib().moe_check(h, stream)


def moe_debug_expire_wait(h, timeout_us: int, stream: int = 0) -> int:
    return lib().moe_debug_expire_wait(h, timeout_us, stream)


def moe_debug_fail_alloc(nth: int) -> int:
    """Make the library's nth device allocation from now on fail (0 = off)."""
    return lib().moe_debug_fail_alloc(int(nth))


def moe_profile_enable(h, enable: int, max_launches: int = 4096) -> int:
    return lib().moe_profile_enable(h, int(enable), int(max_launches))


def moe_profile_read(h):
    """Returns (status, {kernel name: (total ms, launches)})."""
    n = len(KERNEL_NAMES)
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int32 * n)()
    st = lib().moe_profile_read(h, ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(cnt, ctypes.c_void_p))
    return st, {KERNEL_NAMES[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}


def moe_route_noalloc(x: int, T: int, d: int, num_experts: int, top_k: int, act_dtype: int, router_w: int,
                      router_b: int, idx: int, gate: int, counts: int = 0, stream: int = 0) -> int:
    """Routing with no device allocation (scratch in a fixed static array; see include/moe.h)."""
    return lib().moe_route_noalloc(x, T, d, num_experts, top_k, act_dtype, router_w, router_b or None, idx, gate,
                                   counts or None, stream)


def moe_stack_create(cfg: moe_config, layers, stream: int = 0):
    """layers: a sequence of moe_weights.  Returns (status, handle)."""
    arr = (moe_weights * len(layers))(*layers)
    h = ctypes.c_void_p()
    st = lib().moe_stack_create(ctypes.byref(cfg), arr, len(layers), ctypes.c_void_p(stream), ctypes.byref(h))
    return st, h.value


def moe_stack_destroy(h) -> int:
    return lib().moe_stack_destroy(h)


def moe_stack_uses_persistent(h, T: int) -> int:
    return lib().moe_stack_uses_persistent(h, T)


def moe_stack_forward(h, x: int, T: int, y: int, x_trace: int = 0, idx_trace: int = 0, gate_trace: int = 0,
                      stream: int = 0) -> int:
    return lib().moe_stack_forward(h, x, T, y, x_trace or None, idx_trace or None, gate_trace or None, stream)


def moe_stack_check(h, stream: int = 0) -> int:
    return lib().moe_stack_check(h, stream)


def moe_attn_create(cfg: moe_attn_config, w: moe_attn_weights):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    st = lib().moe_attn_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
    return st, h.value


def moe_attn_decode(h, x: int, B: int, pos: int, k_cache: int, v_cache: int, y: int, stream: int = 0) -> int:
    return lib().moe_attn_decode(h, x, B, pos, k_cache, v_cache, y, stream)


def moe_attn_check(h, stream: int = 0) -> int:
    return lib().moe_attn_check(h, stream)


def moe_attn_destroy(h) -> int:
    return lib().moe_attn_destroy(h)


def moe_head_create(d: int, vocab: int, max_tokens: int, codes: int, scales: int, tscale: int,
                    wait_timeout_ms: int = 0):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    st = lib().moe_head_create(d, vocab, max_tokens, codes or None, scales or None, tscale or None,
                               wait_timeout_ms, ctypes.byref(h))
    return st, h.value


def moe_head_forward(h, x: int, T: int, logits: int, stream: int = 0) -> int:
    return lib().moe_head_forward(h, x, T, logits, stream)


def moe_head_check(h, stream: int = 0) -> int:
    return lib().moe_head_check(h, stream)


def moe_head_destroy(h) -> int:
    return lib().moe_head_destroy(h)


def _ok(st: int, what: str):
    if st != MOE_OK:
        raise MoeError(st, what)


# ---------------------------------------------------------------- torch convenience
_DT = {"f32": MOE_F32, "bf16": MOE_BF16, "nvfp4": MOE_NVFP4}


class MoeLayer:
    """One layer's handle plus the device tensors it borrows.

    ``weights`` maps the moe_weights field names to CUDA tensors (or None).
    """

    def __init__(self, *, d, ffn, shared_ffn, num_experts, top_k, max_tokens, act, weight,
                 weights: dict, add_residual=False, path=MOE_PATH_AUTO, gemv_max_tokens=0,
                 wait_timeout_ms=0, deterministic=False, stream=None):
        import torch
        self.torch = torch
        self.cfg = moe_config(d=d, ffn=ffn, shared_ffn=shared_ffn, num_experts=num_experts, top_k=top_k,
                              max_tokens=max_tokens, act_dtype=_DT[act], weight_dtype=_DT[weight],
                              add_residual=int(bool(add_residual)), path=path,
                              gemv_max_tokens=gemv_max_tokens, wait_timeout_ms=wait_timeout_ms,
                              deterministic=int(bool(deterministic)))
        self.tensors = dict(weights)            # keeps the borrowed memory alive
        w = moe_weights()
        for name, _ in moe_weights._fields_:
            t = self.tensors.get(name)
            setattr(w, name, t.data_ptr() if t is not None else None)
        self.w = w
        s = stream if stream is not None else torch.cuda.current_stream()
        st, self.h = moe_create(self.cfg, w, s.cuda_stream)
        _ok(st, "moe_create")
        self.d, self.k, self.E = d, top_k, num_experts
        self.act = act

    def _stream(self, stream):
        return (stream if stream is not None else self.torch.cuda.current_stream()).cuda_stream

    def forward(self, x, y=None, idx=None, gate=None, stream=None):
        T = x.shape[0]
        if y is None:
            y = self.torch.empty_like(x)
        st = moe_forward(self.h, x.data_ptr(), T, y.data_ptr(), idx.data_ptr() if idx is not None else 0,
                         gate.data_ptr() if gate is not None else 0, self._stream(stream))
        _ok(st, "moe_forward")
        return y

    def route(self, x, stream=None, counts=True):
        torch = self.torch
        T = x.shape[0]
        idx = torch.empty((T, self.k), dtype=torch.int32, device=x.device)
        gate = torch.empty((T, self.k), dtype=torch.float32, device=x.device)
        cnt = torch.empty((self.E,), dtype=torch.int32, device=x.device) if counts else None
        st = moe_route(self.h, x.data_ptr(), T, idx.data_ptr(), gate.data_ptr(),
                       cnt.data_ptr() if cnt is not None else 0, self._stream(stream))
        _ok(st, "moe_route")
        return idx, gate, cnt

    def grouping(self, T, device, stream=None):
        torch = self.torch
        offs = torch.empty((self.E + 1,), dtype=torch.int32, device=device)
        tos = torch.empty((T * self.k,), dtype=torch.int32, device=device)
        so = torch.empty((T, self.k), dtype=torch.int32, device=device)
        _ok(moe_get_grouping(self.h, T, offs.data_ptr(), tos.data_ptr(), so.data_ptr(), self._stream(stream)),
            "moe_get_grouping")
        return offs, tos, so

    def forward_host(self, x_host, y_host, stream=None):
        st = moe_forward_host(self.h, x_host.data_ptr(), x_host.shape[0], y_host.data_ptr(), self._stream(stream))
        _ok(st, "moe_forward_host")
        return y_host

    def check(self, stream=None) -> int:
        return moe_check(self.h, self._stream(stream))

    def close(self):
        if getattr(self, "h", None):
            moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def weights_struct(weights: dict) -> moe_weights:
    """moe_weights with the data pointers of a dict of device tensors (missing keys -> NULL)."""
    w = moe_weights()
    for name, _ in moe_weights._fields_:
        t = weights.get(name)
        setattr(w, name, t.data_ptr() if t is not None else None)
    return w


class MoeStack:
    """A stack handle plus the device tensors of every layer it borrows."""

    def __init__(self, spec, layers: list, max_tokens: int, stream=None, **kw):
        import torch
        self.torch = torch
        self.tensors = [dict(w) for w in layers]
        self.cfg = moe_config(d=spec.d, ffn=spec.ffn, shared_ffn=spec.shared_ffn, num_experts=spec.num_experts,
                              top_k=spec.top_k, max_tokens=max_tokens, act_dtype=_DT[spec.act],
                              weight_dtype=_DT[spec.weight], add_residual=1, path=kw.get("path", MOE_PATH_AUTO),
                              gemv_max_tokens=0, wait_timeout_ms=kw.get("wait_timeout_ms", 0))
        s = stream if stream is not None else torch.cuda.current_stream()
        st, self.h = moe_stack_create(self.cfg, [weights_struct(w) for w in self.tensors], s.cuda_stream)
        _ok(st, "moe_stack_create")
        self.L, self.d, self.k = len(layers), spec.d, spec.top_k

    def _stream(self, stream):
        return (stream if stream is not None else self.torch.cuda.current_stream()).cuda_stream

    def persistent(self, T: int) -> bool:
        return bool(moe_stack_uses_persistent(self.h, T))

    def forward(self, x, y=None, trace=False, routing=False, stream=None):
        """Returns y; (y, x_trace [L+1][T][d], idx [L][T][k], gate [L][T][k]) with trace=True;
        (y, idx, gate) with routing=True (the routing only, no x_trace)."""
        torch = self.torch
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        xt = it = gt = None
        if trace:
            xt = torch.empty((self.L + 1, T, self.d), dtype=x.dtype, device=x.device)
        if trace or routing:
            it = torch.empty((self.L, T, self.k), dtype=torch.int32, device=x.device)
            gt = torch.empty((self.L, T, self.k), dtype=torch.float32, device=x.device)
        st = moe_stack_forward(self.h, x.data_ptr(), T, y.data_ptr(), xt.data_ptr() if xt is not None else 0,
                               it.data_ptr() if it is not None else 0, gt.data_ptr() if gt is not None else 0,
                               self._stream(stream))
        _ok(st, "moe_stack_forward")
        if trace:
            return y, xt, it, gt
        return (y, it, gt) if routing else y

    def check(self, stream=None) -> int:
        return moe_stack_check(self.h, self._stream(stream))

    def close(self):
        if getattr(self, "h", None):
            moe_stack_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoeAttn:
    """A sliding-window attention handle plus the device tensors it borrows
    (keys as in inputs.make_attention, as device tensors)."""

    def __init__(self, weights: dict, d: int, n_q: int, n_kv: int, window: int, max_batch: int = 8,
                 use_rope: bool = True, add_residual: bool = False, rope_base: float = 10000.0, eps: float = 1e-6,
                 wait_timeout_ms: int = 0):
        import torch
        self.torch = torch
        self.tensors = dict(weights)
        self.cfg = moe_attn_config(d=d, n_q=n_q, n_kv=n_kv, head_dim=128, window=window, max_batch=max_batch,
                                   use_rope=int(bool(use_rope)), add_residual=int(bool(add_residual)),
                                   wait_timeout_ms=wait_timeout_ms, rope_base=rope_base, eps=eps)
        w = moe_attn_weights()
        for name, _ in moe_attn_weights._fields_:
            setattr(w, name, self.tensors[name].data_ptr())
        st, self.h = moe_attn_create(self.cfg, w)
        _ok(st, "moe_attn_create")

    def decode(self, x, pos, k_cache, v_cache, y=None, stream=None):
        torch = self.torch
        if y is None:
            y = torch.empty_like(x)
        s = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        _ok(moe_attn_decode(self.h, x.data_ptr(), x.shape[0], pos.data_ptr(), k_cache.data_ptr(),
                            v_cache.data_ptr(), y.data_ptr(), s), "moe_attn_decode")
        return y

    def check(self, stream=None) -> int:
        s = (stream if stream is not None else self.torch.cuda.current_stream()).cuda_stream
        return moe_attn_check(self.h, s)

    def close(self):
        if getattr(self, "h", None):
            moe_attn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LmHead:
    """A 4-bit output-layer handle plus the device tensors it borrows
    (codes uint8 [V][d/2], scales uint8 [V][d/16], tscale float32 [1])."""

    def __init__(self, codes, scales, tscale, max_tokens: int, wait_timeout_ms: int = 0):
        import torch
        self.torch = torch
        self.codes, self.scales, self.tscale = codes, scales, tscale
        self.V, self.d = codes.shape[0], codes.shape[1] * 2
        st, self.h = moe_head_create(self.d, self.V, max_tokens, codes.data_ptr(), scales.data_ptr(),
                                     tscale.data_ptr(), wait_timeout_ms)
        _ok(st, "moe_head_create")

    def forward(self, x, logits=None, stream=None):
        torch = self.torch
        if logits is None:
            logits = torch.empty((x.shape[0], self.V), dtype=torch.float32, device=x.device)
        s = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        _ok(moe_head_forward(self.h, x.data_ptr(), x.shape[0], logits.data_ptr(), s), "moe_head_forward")
        return logits

    def check(self, stream=None) -> int:
        s = (stream if stream is not None else self.torch.cuda.current_stream()).cuda_stream
        return moe_head_check(self.h, s)

    def close(self):
        if getattr(self, "h", None):
            moe_head_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def upload_layer(L: dict, device="cuda") -> dict:
    """Copy a layer made by ``inputs.make_layer`` (numpy, storage formats) to
    the device, keyed by the moe_weights field names."""
    import numpy as np
    import torch

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    out = {"router_w": dev(L["router_w"]), "router_b": dev(L["router_b"])}
    names = {"w_gate": ("s_gate", "t_gate"), "w_up": ("s_up", "t_up"), "w_down": ("s_down", "t_down"),
             "ws_gate": ("ss_gate", "ts_gate"), "ws_up": ("ss_up", "ts_up"), "ws_down": ("ss_down", "ts_down")}
    for k, (sk, tk) in names.items():
        v = L.get(k)
        if v is None:
            continue
        if isinstance(v, dict):
            out[k] = dev(v["packed"])
            out[sk] = dev(v["scales"])
            out[tk] = dev(np.asarray(v["tscale"], dtype=np.float32).reshape(-1))
        else:
            out[k] = dev(v)
    return out


def layer_from_spec(spec, weights: dict, max_tokens: int, **kw) -> MoeLayer:
    """MoeLayer for an ``inputs.LayerSpec`` and device weights from ``upload_layer``."""
    kw.setdefault("add_residual", spec.add_residual)
    return MoeLayer(d=spec.d, ffn=spec.ffn, shared_ffn=spec.shared_ffn, num_experts=spec.num_experts,
                    top_k=spec.top_k, max_tokens=max_tokens, act=spec.act, weight=spec.weight,
                    weights=weights, **kw)
