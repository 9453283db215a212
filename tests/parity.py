"""Comparison of the CUDA layer's outputs with the CPU oracle.

Tolerances (the layer's acceptance bounds):
  - routed expert indices bit-exact for every token whose 6th/7th (k-th /
    (k+1)-th) logit gap exceeds 1e-4; inside a near-tie the library's choice
    must lie in the near-tied set, and that token's reference output is then
    recomputed with the library's routing;
  - gates within 2e-5 absolute of the float64 softmax of the same logits
    (fp32 logits and an fp32 exp/divide: a few units of fp32 rounding);
  - output max-abs <= 2e-2 and rel-L2 <= 1e-2 for bf16 weights, rel-L2 <=
    5e-2 for NVFP4 weights; rel-L2 = ||y_gpu - y_ref||_2 / ||y_ref||_2.
    When the output carries the residual x (values of several units) and is
    stored in bf16, the max-abs bound is 2e-2 plus one bf16 unit in the last
    place of the reference value: the output format's resolution there
    exceeds 2e-2 (2^-5 for |y| in [4, 8)), and a sum computed to fp32
    accuracy may round to either bf16 neighbour of the exact one.
"""
import numpy as np
import torch

from oracle.moe_oracle import LayerWeights, moe_forward_with_routing, router_logits, select_topk, topk_gates
from oracle.moe_oracle import _widen

GAP = 1e-4
GATE_ATOL = 2e-5
MAX_ABS = 2e-2
REL_L2 = {"f32": 1e-2, "bf16": 1e-2, "nvfp4": 5e-2}


class DeviceExperts:
    """A per-expert stack of device weights [E][rows][cols] that the oracle can
    index like a numpy array: item e is copied to the host on demand (bf16 as
    uint16 bit patterns, fp32 as float32).  These are the layer's inputs, drawn
    by the input generator; nothing here comes from the library."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __getitem__(self, e):
        return host_array(self.t[int(e)])


def host_array(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def host_layer(dev: dict) -> dict:
    """Oracle view of a layer held on the device (keys as in inputs.make_layer):
    router and shared expert copied whole, routed experts fetched lazily."""
    L = {"router_w": host_array(dev["router_w"]), "router_b": host_array(dev["router_b"])}
    for n in ("w_gate", "w_up", "w_down"):
        L[n] = DeviceExperts(dev[n])
    for n in ("ws_gate", "ws_up", "ws_down"):
        if dev.get(n) is not None:
            L[n] = host_array(dev[n])
    return L


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return np.exp2(e - 7)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def to_torch_x(x: np.ndarray, device="cuda") -> torch.Tensor:
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(x).to(device)


def check_routing(l: np.ndarray, idx_gpu: np.ndarray, gate_gpu: np.ndarray, k: int, stats: dict = None):
    """Returns (idx_use, gate_use, n_near): the routing the reference output uses.
    ``stats`` (optional) receives the largest gate error seen."""
    T, E = l.shape
    srt = -np.sort(-l, axis=1)
    gap = srt[:, k - 1] - srt[:, k] if E > k else np.full(T, np.inf)
    idx_ref = select_topk(l, k)
    idx_use = idx_ref.copy()
    n_near = 0
    for t in range(T):
        g = idx_gpu[t]
        assert len(set(g.tolist())) == k and all(0 <= e < E for e in g), (t, g)
        if gap[t] > GAP:
            assert set(g.tolist()) == set(idx_ref[t].tolist()), (t, g, idx_ref[t], gap[t])
        else:
            n_near += 1
            assert all(l[t, e] >= srt[t, k - 1] - GAP for e in g), (t, g)
            idx_use[t] = g
        # descending by logit up to the tie tolerance
        lv = l[t, g]
        assert np.all(lv[:-1] >= lv[1:] - 1e-5), (t, g, lv)
    gate_use = topk_gates(l, idx_use)
    # gates, matched by expert
    worst = 0.0
    for t in range(T):
        ref = dict(zip(idx_use[t].tolist(), gate_use[t].tolist()))
        for j in range(k):
            e = int(idx_gpu[t, j])
            if e in ref:
                err = abs(gate_gpu[t, j] - ref[e])
                worst = max(worst, err)
                assert err <= GATE_ATOL, (t, j, gate_gpu[t, j], ref[e])
    if stats is not None:
        stats["gate_err"] = worst
    return idx_use, gate_use, n_near


def check_layer(L: dict, x: np.ndarray, y_gpu: torch.Tensor, idx_gpu: torch.Tensor, gate_gpu: torch.Tensor,
                k: int, fmt: str, residual: bool = False, tokens=None, enforce: bool = True):
    """Full-layer parity on `tokens` (all when None). Returns a dict of error figures.
    With enforce=False the output bounds are measured, not asserted (routing still is)."""
    W = LayerWeights(L)
    xf = _widen(x)
    sel = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    xs = xf[sel]
    l = router_logits(xs, W.Wr, W.b)
    ig = idx_gpu.cpu().numpy()[sel].astype(np.int64)
    gg = gate_gpu.cpu().numpy()[sel].astype(np.float64)
    stats = {}
    idx_use, gate_use, n_near = check_routing(l, ig, gg, k, stats)
    y_ref = moe_forward_with_routing(xs, W, idx_use, gate_use, residual=residual)
    yg = to_f64(y_gpu)[sel]
    err = yg - y_ref
    max_abs = float(np.max(np.abs(err)))
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-30))
    assert np.all(np.isfinite(yg))
    bound = MAX_ABS + (bf16_ulp(y_ref) if residual and y_gpu.dtype == torch.bfloat16 else 0.0)
    over = float(np.max(np.abs(err) / bound))
    moe_ref = y_ref - xs if residual else y_ref
    out = {"max_abs": max_abs, "rel_l2": rel, "near_ties": n_near, "gate_err": stats["gate_err"],
           "err_over_bound": over, "x_rms": float(np.sqrt(np.mean(xs ** 2))),
           "moe_rms": float(np.sqrt(np.mean(moe_ref ** 2))), "moe_max": float(np.max(np.abs(moe_ref))),
           "y_max": float(np.max(np.abs(y_ref)))}
    if enforce:
        assert np.all(np.abs(err) <= bound), (max_abs, rel)
        assert rel <= REL_L2[fmt], (max_abs, rel)
    return out
