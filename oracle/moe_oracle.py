"""Plain float64 definition of one sparse MoE FFN layer's forward pass.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix, and where:
- The FFN is split into parallel expert sub-networks and a gating network
  picks a few of them for each token (kongchang.com, section "Architecture:
  The 40B Total vs. 2.5B Active Trade-off").
- Each MoE layer has 256 routed experts, 6 are selected per token, and one
  shared expert is always active (evermx.com review, section "Sparse
  architecture"; swarmz.net, section "The architecture, in plain terms";
  futurpulse.com, section "How does Flint use 39.8B parameters efficiently?").
- Per generated token the selected experts' weights are read once
  (kongchang.com, section "125+ tokens/s: The Practical Threshold").

What the pages leave open, and the reading taken here:
- router: logits l[t][e] = x_t . Wr[e] + b[e] in float64; softmax over E;
- selection on logits, largest first, lower expert index first on equal
  logits; k = 6;
- the k gates renormalised to sum to 1 (= softmax over the k selected
  logits: the full softmax's denominator cancels);
- experts are SwiGLU without biases: E(x) = Wd (silu(Wg x) * (Wu x)),
  silu(z) = z / (1 + exp(-z));
- the shared expert has the same form and weight 1 (no gate);
- y_t = sum_j g_j E_{idx_j}(x_t) + S(x_t), plus x_t when a residual add is
  asked for; in a stack, the residual stream is rounded to bfloat16 after
  every layer.

Everything stays float64 from the widened inputs to the output; rounding to
the output type is left to the caller (``formats.round_to_bf16``).
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_to_f64, nvfp4_to_f64, round_to_bf16


# ---------------------------------------------------------------------------
# Inputs in their storage formats -> float64
# ---------------------------------------------------------------------------
def _widen(a) -> np.ndarray:
    """float32 / bf16-bits (uint16) / float64 array -> float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_to_f64(a)
    return a.astype(np.float64)


class LayerWeights:
    """Float64 views of one layer's weights, decoded one expert at a time.

    ``layer`` is the dict of storage-format arrays (f32, bf16 bit patterns or
    NVFP4 dicts) with keys router_w, router_b, w_gate, w_up, w_down and,
    optionally, ws_gate, ws_up, ws_down.
    """

    def __init__(self, layer: dict):
        self.L = layer
        self.Wr = np.asarray(layer["router_w"], dtype=np.float64)
        b = layer.get("router_b")
        self.b = np.zeros(self.Wr.shape[0]) if b is None else np.asarray(b, dtype=np.float64)
        self.E = self.Wr.shape[0]
        self.has_shared = layer.get("ws_gate") is not None

    @staticmethod
    def _mat(t, e=None):
        if isinstance(t, dict):
            if e is None:
                return nvfp4_to_f64(t["packed"], t["scales"], np.asarray(t["tscale"]).reshape(-1)[0])
            return nvfp4_to_f64(t["packed"][e], t["scales"][e], t["tscale"][e])
        return _widen(t if e is None else t[e])

    def expert(self, e: int):
        """(Wg [F][d], Wu [F][d], Wd [d][F]) of routed expert e, float64."""
        return tuple(self._mat(self.L[n], e) for n in ("w_gate", "w_up", "w_down"))

    def shared(self):
        return tuple(self._mat(self.L[n]) for n in ("ws_gate", "ws_up", "ws_down"))


# ---------------------------------------------------------------------------
# Router
# ---------------------------------------------------------------------------
def router_logits(xf: np.ndarray, Wr: np.ndarray, b: np.ndarray) -> np.ndarray:
    """l[t][e] = sum_i x[t][i] Wr[e][i] + b[e], float64 (the gating network's scores)."""
    return xf @ Wr.T + b[None, :]


def select_topk(l: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, ordered by (-logit, expert index)."""
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-l[t, e], e))
        idx[t] = order[:k]
    return idx


def topk_gates(l: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """g_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0) over the k selected logits."""
    sel = np.take_along_axis(l, idx, axis=1)
    z = np.exp(sel - sel[:, :1])
    return z / z.sum(axis=1, keepdims=True)


def route(xf: np.ndarray, W: LayerWeights, k: int):
    """(idx [T][k], gate [T][k], logits [T][E]) for float64 activations xf."""
    l = router_logits(xf, W.Wr, W.b)
    idx = select_topk(l, k)
    return idx, topk_gates(l, idx), l


def group_slots(idx: np.ndarray, E: int):
    """Group the T*k token-slots by expert, stably.

    Slot s = t*k + j.  Returns counts[E], offsets[E+1] (exclusive scan),
    tok_of_slot[T*k] (token of the s-th grouped slot) and slot_of[T][k]
    (grouped position of slot (t, j)).  Within one expert the slots keep
    their (t, j) order.
    """
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    order = np.argsort(flat, kind="stable")       # grouped position -> original slot
    tok_of_slot = order // k
    slot_of = np.empty(T * k, dtype=np.int64)
    slot_of[order] = np.arange(T * k)
    return counts, offsets, tok_of_slot, slot_of.reshape(T, k)


# ---------------------------------------------------------------------------
# Experts
# ---------------------------------------------------------------------------
def silu(z):
    return z / (1.0 + np.exp(-z))


def expert_ffn(Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, xf: np.ndarray) -> np.ndarray:
    """SwiGLU expert on rows of xf [n][d]: Wd (silu(Wg x) * (Wu x)) -> [n][d]."""
    a = xf @ Wg.T
    u = xf @ Wu.T
    return (silu(a) * u) @ Wd.T


# ---------------------------------------------------------------------------
# Layer
# ---------------------------------------------------------------------------
def moe_forward_with_routing(x, W: LayerWeights, idx, gate, residual: bool = False,
                             tokens=None) -> np.ndarray:
    """y_t = sum_j gate[t][j] E_{idx[t][j]}(x_t) + S(x_t) (+ x_t), float64.

    ``idx``/``gate`` are per token of ``tokens`` (all tokens when None).  Each
    expert's weights are decoded once and applied to the tokens routed to it;
    the per-token sum then runs over j = 0..k-1 in order, shared expert last.
    """
    xf = _widen(x)
    if tokens is not None:
        xf = xf[np.asarray(tokens)]
    idx = np.asarray(idx)
    gate = np.asarray(gate, dtype=np.float64)
    n, k = idx.shape
    contrib = np.zeros((n, k, xf.shape[1]))
    for e in np.unique(idx):
        rows, js = np.nonzero(idx == e)
        Wg, Wu, Wd = W.expert(int(e))
        contrib[rows, js] = expert_ffn(Wg, Wu, Wd, xf[rows])
    y = np.zeros_like(xf)
    for j in range(k):
        y += gate[:, j:j + 1] * contrib[:, j]
    if W.has_shared:
        y += expert_ffn(*W.shared(), xf)
    if residual:
        y += xf
    return y


def moe_forward(x, W: LayerWeights, k: int, residual: bool = False, tokens=None):
    """Full layer on the tokens in ``tokens`` (all when None): (y, idx, gate)."""
    xf = _widen(x)
    if tokens is not None:
        xf = xf[np.asarray(tokens)]
    idx, gate, _ = route(xf, W, k)
    y = moe_forward_with_routing(xf, W, idx, gate, residual=residual)
    return y, idx, gate


def moe_dense(x, W: LayerWeights, k: int, residual: bool = False) -> np.ndarray:
    """The same layer written densely: y_t = sum_{e<E} G[t][e] E_e(x_t) + S(x_t).

    G is the renormalised top-k gate matrix, zero outside the selected
    experts.  Every expert runs on every token; meant for small shapes only.
    """
    xf = _widen(x)
    idx, gate, _ = route(xf, W, k)
    T = xf.shape[0]
    G = np.zeros((T, W.E))
    for t in range(T):
        for j in range(k):
            G[t, idx[t, j]] = gate[t, j]
    y = np.zeros_like(xf)
    for e in range(W.E):
        y += G[:, e:e + 1] * expert_ffn(*W.expert(e), xf)
    if W.has_shared:
        y += expert_ffn(*W.shared(), xf)
    if residual:
        y += xf
    return y


def moe_stack(x, layers, k: int, tokens=None):
    """Stack of MoE layers with residual adds, tokens independent of each other.

    x_{l+1} = bf16(x_l + moe_l(x_l)); returns the final float64 values (each
    already a bf16 value) and the per-layer routing indices.
    """
    xf = _widen(x)
    if tokens is not None:
        xf = xf[np.asarray(tokens)]
    idxs = []
    for W in layers:
        y, idx, _ = moe_forward(xf, W, k, residual=True)
        xf = round_to_bf16(y)
        idxs.append(idx)
    return xf, idxs
