"""CPU oracle for one sparse Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls, links
or executes anything in this package: only the tests, the smoke check in
``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` use it.  It shares no code with the CUDA library (no kernels,
headers, tables or helpers) and imports nothing from it.

Everything is float64 numpy, written from the definition of the layer as the
pages describe it; see ``moe_oracle``, ``lm_head`` and ``attention`` for the
per-function citations.
"""
from .formats import (bf16_to_f64, round_to_bf16, e2m1_value, e4m3_value,  # noqa: F401
                      nvfp4_to_f64)
from .moe_oracle import (router_logits, select_topk, topk_gates, route, silu,  # noqa: F401
                         expert_ffn, group_slots, LayerWeights, moe_forward,
                         moe_forward_with_routing, moe_dense, moe_stack)
from .lm_head import head_weights, lm_head_logits  # noqa: F401
from .attention import attention_decode, rms_norm_heads, rope, window_positions  # noqa: F401
