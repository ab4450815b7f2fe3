"""Noise floor of the bf16 model at full depth: two correct oracles compared.

TEST INFRASTRUCTURE ONLY.  Decodes one sequence of the Ouro-shaped workload
(the shortest prompt, first 8 generated tokens) twice with the same bf16
rounding points: once with every matrix product reduced in float64 (the
oracle) and once with the linear layers reduced in float32 (an equally valid
order and precision of summation).  Their disagreement bounds how closely any
correct implementation can match the oracle; the full-size GPU parity test
derives its tolerances and forcing bands from it.

Measured (16-core box and 8-core container agree): logits 0.050, hidden
0.69 (RMS 9.7), gate logit 0.013 max abs; tokens and exit depths equal.

``floor`` computes the same disagreement for any model and request list; the
bf16 parity tests take their tolerances from it.

Usage: python -m oracle.noise_floor
"""

import numpy as np

from synth import make_requests, make_weights, model_shape, workload
from oracle.model import OracleModel, decode_sequence


def floor(shape, weights, requests, T):
    """Largest disagreement of the two oracles over the first T generated
    tokens of each request: dict with max abs logit, hidden-state and gate
    differences and the hidden-state RMS.  The float32-reduction run follows
    the float64 run's exit depths and tokens (requests may carry replayed
    depths under "replay"), so both see the same sequence."""
    om = OracleModel(shape, weights)
    w32 = {id(v): v.astype(np.float32) for v in om.w.values()}

    class Fp32Reductions(OracleModel):
        def linear(self, x, W, stage):
            return (x.astype(np.float32) @ w32[id(W)].T).astype(np.float64)

    om2 = Fp32Reductions.__new__(Fp32Reductions)
    om2.__dict__.update(om.__dict__)
    out = dict(logits=0.0, hidden=0.0, gate=0.0, hidden_rms=0.0)
    for r in requests:
        n = min(T, r["gen_len"])
        a = decode_sequence(om, r["prompt"], n, keep_logits=n, force_exit=r.get("replay"))
        b = decode_sequence(om2, r["prompt"], n, keep_logits=n, force_exit=np.array(a.exit_depths, np.int8),
                            force_token=np.array(a.tokens, np.int32))
        ha = np.array(a.hidden)
        out["logits"] = max(out["logits"], float(np.abs(np.array(a.logits) - np.array(b.logits)).max()))
        out["hidden"] = max(out["hidden"], float(np.abs(ha - np.array(b.hidden)).max()))
        out["hidden_rms"] = max(out["hidden_rms"], float(np.sqrt((ha ** 2).mean())))
        za = [z for zs in a.gate_logits for z in zs]
        zb = [z for zs in b.gate_logits for z in zs]
        if za:
            out["gate"] = max(out["gate"], float(np.abs(np.array(za) - np.array(zb)).max()))
    return out


def main(T=8):
    wl = workload("ouro")
    shape = model_shape("ouro")
    wts = make_weights(shape)
    r = sorted(make_requests(wl, shape.vocab), key=lambda r: len(r["prompt"]))[0]
    f = floor(shape, wts, [dict(prompt=r["prompt"], gen_len=T)], T)
    print("sequence", r["seq_id"], "prompt", len(r["prompt"]), f)


if __name__ == "__main__":
    main()
