"""A small decode case for kernel profiling (ncu), with the bench's per-launch shapes.

Runs the Ouro-shaped model and workload of bench.py (d 2048, 16x128 heads,
SwiGLU 5632, W = 64, prompts 128..1024) but with --layers core layers instead
of 24, so every attention and projection launch has exactly the bench's
shape while the depth-indexed KV pool stays a few GB.  Prints the kernel-class
timing of the decode steps.  Not a benchmark: bench.py is.

    python -m continuous_depth_batching_gb300.profile_case --layers 1 --steps 4
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--workload", default="ouro")
    ap.add_argument("--split", type=int, default=0, help="keys per split-KV partial (0: library default)")
    ap.add_argument("--W", type=int, default=0, help="core slots (0: the workload's)")
    ap.add_argument("--prompt-len", type=int, default=0, help="every prompt this long (0: the workload's lengths)")
    ap.add_argument("--gen", type=int, default=0, help="tokens generated per request (0: the workload's)")
    ap.add_argument("--kv-slots", type=int, default=0)
    args = ap.parse_args()

    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.build import build
    from synth import make_requests, make_weights, model_shape, workload

    build()
    wl = workload(args.workload)
    over = {}
    if args.W:
        over.update(W=args.W, n_seqs=max(wl.n_seqs, args.W))
    if args.prompt_len:
        over.update(prompt_lo=args.prompt_len, prompt_hi=args.prompt_len)
    if args.gen:
        over.update(gen_lo=args.gen, gen_hi=args.gen)
    wl = wl.with_(**over)
    shape = dataclasses.replace(model_shape(wl.model), n_core=args.layers, kv_slots=args.kv_slots)
    dw = binding.device_weights(shape, make_weights(shape))
    reqs = make_requests(wl, shape.vocab, shape.r_max, shape.r_min)
    max_ctx = (wl.prompt_hi + wl.gen_hi - 1 + 15) // 16 * 16
    eng = binding.Engine(shape, dw, mode="refill", W=wl.W, M=wl.M, K=wl.K, max_ctx=max_ctx,
                         max_new_cap=wl.gen_hi, attn_split=args.split)
    for r in reqs:
        eng.admit(r["seq_id"], r["prompt"], r["gen_len"], r["replay"])

    def advance(n):
        done = 0
        while done < n:
            rc, _ = eng.step_boundary()
            if rc == binding.DONE:
                break
            if rc == binding.IDLE:
                eng.step_core()
                done += 1

    # Per decode step (one decode-attention launch per step with one layer):
    # the launch's index among the decode-attention launches (prefill chunks
    # use their own kernel) and its algorithmic bytes, so an ncu capture
    # (-k k_attn_tma -s INDEX) can be matched.
    eng.profile_enable(True)
    n_attn = 0
    per_step = []
    total = {}
    for i in range(args.warmup + args.steps):
        advance(1)
        st = eng.profile_read()
        if st["attention"]["launches"]:
            per_step.append({"step": i, "attn_index": n_attn, "attn_launches": st["attention"]["launches"],
                             "attn_bytes": st["attention"]["bytes"], "attn_ms": st["attention"]["ms"]})
        n_attn += st["attention"]["launches"]
        if i >= args.warmup:
            for k, v in st.items():
                t = total.setdefault(k, dict(launches=0, ms=0.0, bytes=0.0, flops=0.0))
                for f in t:
                    t[f] += v[f]
    eng.close()
    for r in per_step:
        print(json.dumps(r))
    print(json.dumps({k: dict(v, GBps=(v["bytes"] / v["ms"] / 1e6) if v["ms"] else None)
                      for k, v in total.items()}))


if __name__ == "__main__":
    main()
