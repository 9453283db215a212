"""Fit the router-bias scale of the skewed-load workload.

TEST INFRASTRUCTURE (see the package docstring); run by hand:

    python -m oracle.fit_zipf_alpha

The skewed workload gives expert e the router bias b_e = alpha * ln p_r(e),
p_r proportional to r^-1.1 over ranks r = 1..E dealt by a seeded permutation
(``inputs.zipf_bias``).  This script finds alpha by bisection so that the
expert load realised by the oracle's routing of N(0, 1) tokens, ranked, falls
with a log-log slope of -1.1 over the 64 most loaded experts, on a calibration
seed distinct from every seed the tests and the bench use.  It prints the
value that ``inputs.ZIPF_ALPHA`` holds.
"""
import numpy as np

from oracle.moe_oracle import router_logits, select_topk

CAL_SEED = 1000
TARGET = -1.1
TOP_RANKS = 64


def load_slope(alpha: float, T: int = 2048, seed: int = CAL_SEED) -> float:
    from sparse_moe_transformer_02_b300 import inputs as I   # input generator only
    spec = I.FLINT_STACK_ZIPF
    Wr = I.normal_f32(seed, 0, I.TID_ROUTER_W, (spec.num_experts, spec.d), spec.sigma_router).astype(np.float64)
    b = I.zipf_bias(seed, 0, spec.num_experts, alpha=alpha).astype(np.float64)
    xb = I.make_tokens(spec, seed, T)
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    idx = select_topk(router_logits(x, Wr, b), spec.top_k)
    load = np.sort(np.bincount(idx.reshape(-1), minlength=spec.num_experts))[::-1][:TOP_RANKS]
    ranks = np.arange(1, TOP_RANKS + 1)
    keep = load > 0
    return float(np.polyfit(np.log(ranks[keep]), np.log(load[keep]), 1)[0])


def fit(lo: float = 0.0, hi: float = 3.0, iters: int = 16) -> float:
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if load_slope(mid) > TARGET:      # not steep enough: more bias
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


if __name__ == "__main__":
    a = fit()
    print(f"alpha = {a:.4f}  (realised slope {load_slope(a):.3f} over the top {TOP_RANKS} ranks)")
