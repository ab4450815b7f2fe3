"""Calibrate the exit-gate bias of each synthetic model on the CPU oracle.

TEST INFRASTRUCTURE ONLY.  Writes ``synth/gate_bias.json``, the frozen bias
both the oracle and the CUDA library read as an input.

The models are random-initialised, so the exit head of the paper (App. E.2,
Ouro's trained gate) is replaced by a linear probe whose bias sets how often
tokens exit.  The bias is chosen from the gate logits of a fixed-depth pilot
run (every token runs r_max loops and its logit z_d is recorded after each
step d).  With the lookahead rule of §4.3 a token's exit depth for bias b is
min(r_max, 1 + min{d in [r_min-1, r_max-2] : z_d + b > logit(q)}).

* tiny: the bias that spreads exit depths most evenly over 2..r_max
  (largest entropy of the depth histogram on a grid of step 0.005).
* ouro: the bias whose live-gate mean exit depth over a sample of the job
  (6 sequences spread over its prompt lengths, each decoded for all 256
  generated tokens, since exits grow shallower along a sequence) is closest
  to 3.
* huginn: exit depths are replayed (App. C.2), the bias stays 0.

Usage: python -m oracle.calibrate_gate [tiny|ouro ...]
"""

from __future__ import annotations

import json
import os
import sys

import numpy as np

from synth import make_requests, make_weights, model_shape, workload
from synth.configs import replace as _replace  # dataclasses.replace re-exported
from oracle.model import OracleModel, decode_sequence

_OUT = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "synth", "gate_bias.json")


def exit_depths(Z: np.ndarray, b: float, r_min: int, r_max: int, theta: float):
    lo, hi = r_min - 1, r_max - 2          # deciding steps d (1-based)
    g = (Z[:, lo - 1:hi] + b) > theta
    first = np.where(g.any(1), g.argmax(1) + lo, r_max)   # d of first positive gate
    return np.minimum(first + 1, r_max)


def pilot_logits(name: str, n_seqs: int, gen: int) -> np.ndarray:
    shape = _replace(model_shape(name), gate_bias=0.0)
    wl = workload(name)
    reqs = make_requests(wl, shape.vocab, shape.r_max, shape.r_min)
    reqs = sorted(reqs, key=lambda r: len(r["prompt"]))[:n_seqs]
    om = OracleModel(shape, make_weights(shape))
    Z = []
    for r in reqs:
        tr = decode_sequence(om, r["prompt"], gen, mode="fixed")
        Z += tr.gate_logits
    return np.array(Z)


def calibrate(name: str) -> float:
    shape = model_shape(name)
    if name == "huginn":
        return 0.0
    if name == "tiny":
        Z = pilot_logits(name, workload(name).n_seqs, 16)
        best, best_h = 0.0, -1.0
        for b in np.arange(-1.0, 1.0, 0.005):
            e = exit_depths(Z, b, shape.r_min, shape.r_max, shape.gate_threshold_logit)
            p = np.bincount(e, minlength=shape.r_max + 1)[shape.r_min:] / len(e)
            h = -np.sum(p[p > 0] * np.log(p[p > 0]))
            if h > best_h + 1e-12:
                best, best_h = float(b), h
        return round(best, 3)
    if name == "ouro":
        return calibrate_mean(name, 3.0)
    raise KeyError(name)


def job_sample(name: str, n_seqs: int):
    """n_seqs requests spread evenly over the workload's sequence ids (prompt
    lengths are independent draws, so this spans the prompt-length range)."""
    wl = workload(name)
    reqs = make_requests(wl, model_shape(name).vocab)
    step = max(1, wl.n_seqs // n_seqs)
    return [reqs[i] for i in range(0, wl.n_seqs, step)][:n_seqs]


def adaptive_mean(shape, weights, reqs, gen: int, b: float) -> float:
    """Mean exit depth of the live gate with bias b (each request decoded alone)."""
    om = OracleModel(_replace(shape, gate_bias=b), weights)
    e = []
    for r in reqs:
        e += decode_sequence(om, r["prompt"], gen).exit_depths
    return float(np.mean(e))


def calibrate_mean(name: str, target: float, n_seqs: int = 6, gen: int = 256) -> float:
    """Bias whose mean exit depth over a sample of the job is closest to target.

    A fixed-depth pilot gives every token's logits z_1..z_{r_max-1}, hence the
    mean exit depth m(b) of any bias under the lookahead rule.  Exits change
    later tokens' states through the depth clamp, so the live-gate mean at the
    pilot's bias b0 is measured with adaptive runs and the bias is moved along
    the pilot's m(b) curve by the difference (one correction step, then the
    better of the two)."""
    shape = _replace(model_shape(name), gate_bias=0.0)
    weights = make_weights(shape)
    reqs = job_sample(name, n_seqs)
    om = OracleModel(shape, weights)
    Z = []
    for r in reqs:
        Z += decode_sequence(om, r["prompt"], gen, mode="fixed").gate_logits
    Z = np.array(Z)
    del om
    bs = np.arange(-3.0, 3.0, 0.005)
    curve = np.array([exit_depths(Z, b, shape.r_min, shape.r_max, shape.gate_threshold_logit).mean() for b in bs])

    def bias_for(m):
        return float(bs[int(np.argmin(np.abs(curve - m)))])

    b0 = bias_for(target)
    m0 = adaptive_mean(shape, weights, reqs, gen, b0)
    b1 = bias_for(target + (target - m0))
    m1 = adaptive_mean(shape, weights, reqs, gen, b1)
    print(f"{name}: pilot bias {b0:.3f} -> live mean {m0:.3f}; corrected bias {b1:.3f} -> live mean {m1:.3f}")
    return round(b0 if abs(m0 - target) <= abs(m1 - target) else b1, 3)


def main(names):
    data = {}
    if os.path.exists(_OUT):
        with open(_OUT) as f:
            data = json.load(f)
    for n in names:
        data[n] = calibrate(n)
        print(n, data[n])
    with open(_OUT, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main(sys.argv[1:] or ["tiny", "ouro", "huginn"])
