"""Plain float64 definition of the 4-bit output layer (lm_head).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages say Flint's output layer was quantised to 4 bits because, with
about 2.5B parameters active per token, it is a large share of the weights
read for each token, and that the shipped low-bit model is NVFP4 (evermx.com
review, Feature Overview, "Quantization"; futurpulse.com, section "How did
Recursive use AI to build Flint?").  The head maps the final hidden state to
one logit per vocabulary entry: logits[t][v] = sum_i x[t][i] W[v][i].

Readings taken where the pages are silent: the head's weights use the same
NVFP4 layout as the experts (e2m1 codes along the hidden dimension, one e4m3
scale per 16 values, one fp32 scale for the matrix); the logits are fp32;
the vocabulary size follows from the parameter counts (about 0.3B head
parameters = 2.5B active with the head - 2.2B without it, over the assumed
hidden width 2048, so V = 146,432).
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_to_f64, nvfp4_to_f64


def head_weights(packed, scales, tscale) -> np.ndarray:
    """W [V][d] float64, decoded from NVFP4 codes, block scales and the matrix scale."""
    return nvfp4_to_f64(packed, scales, float(np.asarray(tscale).reshape(-1)[0]))


def lm_head_logits(x, packed, scales, tscale, rows=None) -> np.ndarray:
    """logits [T][V] (or [T][len(rows)] for the vocabulary rows in `rows`), float64.

    x is float32 / float64, or uint16 bf16 bit patterns.
    """
    x = np.asarray(x)
    xf = bf16_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)
    if rows is not None:
        rows = np.asarray(rows)
        packed, scales = np.asarray(packed)[rows], np.asarray(scales)[rows]
    W = head_weights(packed, scales, tscale)
    return xf @ W.T
