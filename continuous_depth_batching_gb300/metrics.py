"""Speedup bounds of depth-adaptive decoding, for reporting.

"Depth-adaptive Inference of Looped Language Models via Continuous Depth
Batching", §5: with F_r the FLOPs of one recurrent-core application for one
token and F_0 the loop-independent FLOPs of the prelude and coda, the
decode-speedup bound at mean exit depth d is eq. (1)

    S_dec = (F_0 + r_max F_r) / (F_0 + d F_r)  <=  r_max / d,

and with alpha the measured share of time spent on prefill, eq. (2)

    S_e2e = (alpha + (1 - alpha) / S_dec)^-1.

FLOPs count two per multiply-add of the weights a token touches (the
embedding is a gather).  The context-dependent attention term is optional
(`context_len`); eq. (1) treats F_r as a constant.
"""

from __future__ import annotations


def token_flops(shape, context_len: int = 0):
    """(F_0, F_r) per generated token for a model shape (synth.ModelShape fields)."""
    d, f, V = shape.d_model, shape.ffn, shape.vocab
    layer = 2.0 * (4 * d * d + 3 * d * f) + 4.0 * d * context_len
    F_r = shape.n_core * layer + (4.0 * d * d if shape.has_adapter else 0.0)
    F_0 = (shape.n_prelude + shape.n_coda) * layer + 2.0 * V * d
    return F_0, F_r


def s_dec(F_0: float, F_r: float, r_max: int, mean_depth: float) -> float:
    """Eq. (1)."""
    return (F_0 + r_max * F_r) / (F_0 + mean_depth * F_r)


def s_e2e(alpha: float, sdec: float) -> float:
    """Eq. (2)."""
    return 1.0 / (alpha + (1.0 - alpha) / sdec)
