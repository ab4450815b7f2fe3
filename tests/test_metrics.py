"""§5 speedup bounds (continuous_depth_batching_gb300/metrics.py).

Pinned to the oracle's executed FLOP counts (not to the formula itself): the
per-token F_0 / F_r of the closed form must equal what the oracle actually
executes for one decode forward at a known exit depth and context, for a
fully looped and a 2-4-2-style model.  The bound at the Ouro- and
Huginn-shaped configurations is checked against eq. (1) evaluated by hand
from the shapes, and eq. (2) against its limits.
"""

import dataclasses

import numpy as np
import pytest

from continuous_depth_batching_gb300 import metrics
from oracle.model import OracleModel, decode_sequence
from synth import make_weights, model_shape


def micro(**kw):
    base = dict(name="micro", vocab=64, d_model=32, n_heads=4, head_dim=8, ffn=48, n_prelude=0, n_core=2,
                n_coda=0, r_max=4, r_min=2, has_adapter=False, dtype="fp32", init_std=0.2, gate_bias=0.0)
    base.update(kw)
    return dataclasses.replace(model_shape("tiny"), **base)


@pytest.mark.parametrize("variant", ["looped", "huginn_like"])
def test_closed_form_equals_executed_flops(variant):
    shape = micro() if variant == "looped" else micro(n_prelude=1, n_core=1, n_coda=1, has_adapter=True)
    wts = make_weights(shape)
    prompt = np.arange(5, dtype=np.int32)
    e = 3
    om = OracleModel(shape, wts)
    decode_sequence(om, prompt, 1)
    before = dataclasses.asdict(om.flops)
    om2 = OracleModel(shape, wts)
    decode_sequence(om2, prompt, 2, force_exit=np.array([e], dtype=np.int8))
    after = dataclasses.asdict(om2.flops)
    executed = {k: after[k] - before[k] for k in after}
    L = len(prompt) + 1  # the decode forward at position P sees P + 1 keys
    F0, Fr = metrics.token_flops(shape, context_len=L)
    n_attn_boundary = shape.n_prelude + shape.n_coda
    attn_r = 4.0 * shape.d_model * L * shape.n_core
    attn_0 = 4.0 * shape.d_model * L * n_attn_boundary
    assert executed["core"] + e * attn_r == pytest.approx(e * Fr, rel=1e-12)
    assert executed["prelude"] + executed["coda"] + attn_0 == pytest.approx(F0, rel=1e-12)
    assert executed["attention"] == pytest.approx(e * attn_r + attn_0, rel=1e-12)


def test_bound_at_the_model_shapes():
    ouro = model_shape("ouro")
    F0, Fr = metrics.token_flops(ouro)
    d, f, V = 2048, 5632, 49152
    assert Fr == 2 * 24 * (4 * d * d + 3 * d * f)
    assert F0 == 2 * V * d
    assert metrics.s_dec(F0, Fr, 4, 3.0) == pytest.approx((F0 + 4 * Fr) / (F0 + 3 * Fr))
    assert round(metrics.s_dec(F0, Fr, 4, 3.0), 4) == 1.3245
    assert metrics.s_dec(F0, Fr, 4, 3.0) < 4 / 3
    hug = dataclasses.replace(model_shape("huginn"))
    F0h, Frh = metrics.token_flops(hug)
    assert round(metrics.s_dec(F0h, Frh, 32, 12.0), 3) == 2.518
    assert metrics.s_dec(F0h, Frh, 32, 12.0) < 32 / 12


def test_e2e_limits():
    assert metrics.s_e2e(0.0, 1.5) == pytest.approx(1.5)
    assert metrics.s_e2e(1.0, 1.5) == pytest.approx(1.0)
    assert 1.0 < metrics.s_e2e(0.3, 1.5) < 1.5
