"""The depth-indexed KV cache the engine leaves in its arena, read back and
compared with the oracle's logical cache.

"Depth-adaptive Inference of Looped Language Models via Continuous Depth
Batching", §4.2: every core layer keeps one KV slot per loop step, and a
position that left the loop after step e was computed only up to e; a later
row at step r reads that position's entry of step min(r, e) (the depth clamp).

One sequence decodes alone in a new engine, so it holds the pool's first
blocks in order (cdb_test_kv_pool).  Then, for every cached position p, core
layer l and loop step r:

* r <= e_p: the engine's K and V rows equal the oracle's within the dtype's
  tolerance (the oracle's entry exists);
* r > e_p: the oracle has no entry, and the engine's slot holds a bit-exact
  copy of step e_p's entry (the exit-gap fill that realises the clamp).

bf16 runs the decode attention that forms each token's own K and V rows from
the QKV projection's partials; fp32 the separate RoPE / KV-write kernel.
"""

import dataclasses

import numpy as np
import pytest

from oracle.model import OracleModel, decode_sequence
from synth import make_weights, model_shape
from tests.gpu_util import force_tables

pytestmark = pytest.mark.gpu

NEAR = 1e-3


def _shape(dtype):
    return dataclasses.replace(model_shape("tiny"), name="kv", vocab=1024, d_model=256, n_heads=2, head_dim=128,
                               ffn=512, n_prelude=0, n_core=2, n_coda=0, r_max=5, r_min=2, has_adapter=False,
                               dtype=dtype, gate_bias=0.12)


@pytest.mark.parametrize("dtype,tol,gap", [("fp32", 1e-4, 1e-3), ("bf16", 2e-2, 1e-2)])
def test_kv_pool_holds_the_oracle_cache(dtype, tol, gap):
    from continuous_depth_batching_gb300 import binding
    shape = _shape(dtype)
    wts = make_weights(shape)
    rng = np.random.default_rng(61)
    P, gen = 40, 8
    prompt = rng.integers(0, shape.vocab, P).astype(np.int32)
    tr = decode_sequence(OracleModel(shape, wts), prompt, gen, "adaptive", keep_kv=True, near_tol=NEAR)
    n_pos = P + gen - 1  # the last generated token is never fed back
    max_ctx = (n_pos + 15) // 16 * 16
    eng = binding.Engine(shape, binding.device_weights(shape, wts), mode="refill", W=1, M=8192, K=1,
                         max_ctx=max_ctx, max_new_cap=gen, kv_blocks=max_ctx // 16)
    fe, ft = force_tables(tr, None, gap)
    eng.admit(0, prompt, gen, fe, ft)
    eng.run()
    out = eng.drain()
    assert list(out[0]["tokens"]) == tr.tokens and list(out[0]["exit_depths"]) == tr.exit_depths
    pool = eng.kv_pool().float().cpu().numpy().astype(np.float64)  # [blk, slot, K|V, H, 16, hd]
    eng.close()

    d, r_max = shape.d_model, shape.r_max
    ok = gaps = 0
    worst = 0.0
    for p in range(n_pos):
        e = r_max if p < P else tr.exit_depths[p - P]
        for l in range(shape.n_core):
            step_e = None
            for r in range(1, r_max + 1):
                s = shape.n_prelude + l * r_max + r - 1
                eng_kv = pool[p // 16, s, :, :, p % 16, :].reshape(2, d)
                ora_kv = np.stack([tr.kv.K[s, p], tr.kv.V[s, p]]).astype(np.float64)
                if r <= e:
                    assert np.isfinite(ora_kv).all(), (p, l, r)
                    err = float(np.max(np.abs(eng_kv - ora_kv)))
                    worst = max(worst, err)
                    assert err <= tol, (p, l, r, e, err)
                    if r == e:
                        step_e = eng_kv
                    ok += 1
                else:
                    assert np.isnan(ora_kv).all(), (p, l, r, e)
                    np.testing.assert_array_equal(eng_kv, step_e, err_msg=f"gap p={p} l={l} r={r} e={e}")
                    gaps += 1
    print(f"{dtype}: {ok} cached entries within {worst:.2e}, {gaps} exit-gap copies")
    assert gaps > 0, "the sequence should exit early at least once"
