"""Recurrent-step latency versus batch size and context length.

"Depth-adaptive Inference of Looped Language Models via Continuous Depth
Batching", §5 and Appendix B: B equal-length requests of context L decode at
full depth (no early exit), all starting together after their prefill; the
latency of one recurrent step is fitted per context length with eq. (4),

    t(B) = delta + (gamma + alpha L) B,     B* = delta / (gamma + alpha L),

delta being the weight-reload cost, gamma the per-token compute and alpha the
per-KV-entry streaming cost.  The pages separate the loop step from the
prelude/coda cost by varying r and fitting eq. (3); this library runs the
loop step as its own call (cdb_step_core), so tau_r is timed directly with
CUDA events around each core step and tau_0 (coda + prelude) around the
boundary calls.  Cells whose KV does not fit the memory budget are skipped.

    python -m continuous_depth_batching_gb300.step_latency --model ouro
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def step_bytes_flops(shape, B, L):
    """Algorithmic bytes and FLOPs of one recurrent step (core weights once,
    one KV row per key per core layer, KV writes, fp32 state in and out)."""
    d, f, es = shape.d_model, shape.ffn, shape.elem_bytes
    P = shape.n_core * (4 * d * d + 3 * d * f) + (2 * d * d if shape.has_adapter else 0)
    kv = shape.n_core * 2 * d * es * B * L
    by = P * es + kv + B * shape.n_core * 2 * d * es + 16 * B * d
    fl = 2.0 * P * B + 4.0 * shape.n_core * d * B * L
    return by, fl


def measure_cell(shape, dw, B, L, tokens=16, warm_tokens=2, seed=7):
    import numpy as np
    import torch

    from continuous_depth_batching_gb300 import binding

    gen = warm_tokens + tokens + 1
    max_ctx = (L + gen + 15) // 16 * 16
    eng = binding.Engine(shape, dw, mode="fixed_depth", W=B, M=8192, K=1, max_ctx=max_ctx, max_new_cap=gen,
                         kv_blocks=B * (max_ctx // 16))
    rng = np.random.default_rng(seed)
    for i in range(B):
        eng.admit(i, rng.integers(0, shape.vocab, L).astype(np.int32), gen)
    s = eng.stream
    core_ms, bound_ms = [], []
    cores = 0  # every token runs r_max core steps at full depth
    while True:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        rc, info = eng.step_boundary()
        b.record(s)
        if rc == binding.DONE:
            break
        if rc == binding.IDLE:
            c = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            c.record(s)
            eng.step_core()
            e.record(s)
            core_ms.append((cores // shape.r_max, c, e))
            cores += 1
        elif cores > 0 and info.stage != 1:  # coda / prelude of the decode loop (not prefill)
            bound_ms.append(((cores - 1) // shape.r_max, a, b))
    torch.cuda.synchronize()
    eng.close()
    lo, hi = warm_tokens, warm_tokens + tokens
    tc = [c.elapsed_time(e) for t, c, e in core_ms if lo <= t < hi]
    tb = [a.elapsed_time(b) for t, a, b in bound_ms if lo <= t < hi]
    tau_r = statistics.median(tc) if tc else float("nan")
    tau_0 = sum(tb) / max(tokens, 1)
    return tau_r, tau_0, len(tc)


def fit_line(xs, ys):
    n = len(xs)
    mx, my = sum(xs) / n, sum(ys) / n
    sxx = sum((x - mx) ** 2 for x in xs)
    slope = sum((x - mx) * (y - my) for x, y in zip(xs, ys)) / sxx if sxx > 0 else 0.0
    return my - slope * mx, slope


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--model", default="ouro")
    ap.add_argument("--batches", default="1,8,16,32,64,128,256,512")
    ap.add_argument("--contexts", default="128,512,2048,8192")
    ap.add_argument("--kv-gb", type=float, default=220.0, help="KV budget per cell")
    ap.add_argument("--tokens", type=int, default=16)
    ap.add_argument("--kv-slots", type=int, default=0,
                    help="KV slots per core layer (App. E.1): 0 depth-indexed, 1 single slot, 2 first-then-shared")
    args = ap.parse_args()

    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.build import build
    from synth import make_weights, model_shape

    build()
    import dataclasses
    shape = dataclasses.replace(model_shape(args.model), kv_slots=args.kv_slots)
    dw = binding.device_weights(shape, make_weights(shape))
    kv_tok = binding.kv_bytes_per_token(shape)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {"hbm_gbs": 6779.4, "bf16_tflops_sustained": 1709.3}
    bw, tf = peaks["hbm_gbs"] * 1e9, peaks["bf16_tflops_sustained"] * 1e12
    rows = []
    for L in [int(v) for v in args.contexts.split(",")]:
        cells = []
        for B in [int(v) for v in args.batches.split(",")]:
            if B * (L + args.tokens + 16) * kv_tok > args.kv_gb * 1e9:
                continue
            tau_r, tau_0, n = measure_cell(shape, dw, B, L, tokens=args.tokens)
            by, fl = step_bytes_flops(shape, B, L)
            t_roof = max(by / bw, fl / tf) * 1e3
            cell = dict(L=L, B=B, tau_r_ms=round(tau_r, 4), tau_0_ms=round(tau_0, 4), steps=n,
                        roofline_ms=round(t_roof, 4), frac_of_roofline=round(t_roof / tau_r, 3))
            print(json.dumps(cell), flush=True)
            cells.append(cell)
        if len(cells) >= 2:
            delta, slope = fit_line([c["B"] for c in cells], [c["tau_r_ms"] for c in cells])
            rows.append(dict(L=L, delta_ms=round(delta, 4), slope_ms_per_token=round(slope, 5),
                             B_star=round(delta / slope, 1) if slope > 0 else None))
            print(json.dumps(dict(fit=rows[-1])), flush=True)
    print(json.dumps(dict(model=args.model, fits=rows)))


if __name__ == "__main__":
    main()
