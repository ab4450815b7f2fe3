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

Usage: python -m oracle.noise_floor
"""

import numpy as np

from synth import make_requests, make_weights, model_shape, workload
from oracle.model import OracleModel, decode_sequence


def main(T=8):
    wl = workload("ouro")
    shape = model_shape("ouro")
    wts = make_weights(shape)
    r = sorted(make_requests(wl, shape.vocab), key=lambda r: len(r["prompt"]))[0]
    om = OracleModel(shape, wts)
    a = decode_sequence(om, r["prompt"], T, keep_logits=T)
    w32 = {id(v): v.astype(np.float32) for v in om.w.values()}

    class Fp32Reductions(OracleModel):
        def linear(self, x, W, stage):
            return (x.astype(np.float32) @ w32[id(W)].T).astype(np.float64)

    om2 = Fp32Reductions.__new__(Fp32Reductions)
    om2.__dict__.update(om.__dict__)
    b = decode_sequence(om2, r["prompt"], T, keep_logits=T)
    la, lb = np.array(a.logits), np.array(b.logits)
    ha, hb = np.array(a.hidden), np.array(b.hidden)
    za = np.concatenate([np.array(z) for z in a.gate_logits if z])
    zb = np.concatenate([np.array(z) for z in b.gate_logits if z])
    print("sequence", r["seq_id"], "prompt", len(r["prompt"]), "tokens equal", a.tokens == b.tokens,
          "exits equal", a.exit_depths == b.exit_depths)
    print("logits max abs", float(np.abs(la - lb).max()), "hidden max abs", float(np.abs(ha - hb).max()),
          "hidden rms", float(np.sqrt((ha ** 2).mean())), "gate max abs", float(np.abs(za - zb).max()))


if __name__ == "__main__":
    main()
