"""Online serving: Poisson arrivals, normalised latency, refill vs no-refill vs fixed depth.

"Depth-adaptive Inference of Looped Language Models via Continuous Depth
Batching", §6.3 and Fig. 6 (App. D): requests arrive by a Poisson process at
rate lambda; a request's normalised latency is its end-to-end time divided by
its output length; the serving capacity is the rate at which normalised
latency starts to rise sharply.  The synthetic requests have prompts
U[64, 2048] and outputs U[32, 512] tokens; the rate of each point is
calibrated so the mean recurrent batch is near a target (Little's law:
concurrency = rate x time in system, so the rate is rescaled by target /
measured from short refill-mode pilot runs).

Time is wall-clock: a request is admitted once its arrival time has passed,
the engine is stepped between admissions, and finished requests are
collected without stalling the device queue (cdb_poll).  Requests are
measured if they arrive inside the window; the run continues until they
finish.

    python -m continuous_depth_batching_gb300.online --model ouro --targets 1,8,32,128
"""

from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def poisson_arrivals(rate: float, window: float, seed: int) -> np.ndarray:
    """Arrival times in [0, window) of a Poisson process with `rate` per second."""
    rng = np.random.default_rng(seed)
    out, t = [], 0.0
    while True:
        t += rng.exponential(1.0 / rate)
        if t >= window:
            return np.asarray(out, dtype=np.float64)
        out.append(t)


def make_online_requests(n: int, vocab: int, seed: int, prompt=(64, 2048), gen=(32, 512)):
    rng = np.random.default_rng(seed)
    plen = rng.integers(prompt[0], prompt[1] + 1, n)
    glen = rng.integers(gen[0], gen[1] + 1, n)
    return [dict(seq_id=i, prompt=rng.integers(0, vocab, int(plen[i])).astype(np.int32), gen_len=int(glen[i]))
            for i in range(n)]


def normalized_latency(arrive, finish, out_len) -> np.ndarray:
    """End-to-end seconds per output token of each request."""
    return (np.asarray(finish, np.float64) - np.asarray(arrive, np.float64)) / np.asarray(out_len, np.float64)


def latency_stats(lat) -> dict:
    lat = np.asarray(lat, np.float64)
    if lat.size == 0:
        return {"n": 0}
    return {"n": int(lat.size), "mean_ms": float(lat.mean() * 1e3), "p50_ms": float(np.percentile(lat, 50) * 1e3),
            "p90_ms": float(np.percentile(lat, 90) * 1e3), "p99_ms": float(np.percentile(lat, 99) * 1e3)}


def rescale_rate(rate: float, measured_batch: float, target_batch: float, lo=0.25, hi=4.0) -> float:
    """Little's law step: concurrency scales with the rate below saturation (bounded step)."""
    if measured_batch <= 0:
        return rate * hi
    return rate * min(hi, max(lo, target_batch / measured_batch))


def run_point(make_engine, reqs, arrive, window, mode, drain_limit=120.0):
    """Serve `reqs` arriving at `arrive` (seconds) with a fresh engine in `mode`."""
    from continuous_depth_batching_gb300 import binding
    eng = make_engine(mode)
    n = len(arrive)
    finish = np.full(n, np.nan)
    batches = []
    i = 0
    t0 = time.perf_counter()
    try:
        while True:
            now = time.perf_counter() - t0
            while i < n and arrive[i] <= now:
                r = reqs[i]
                eng.admit(i, r["prompt"], r["gen_len"])
                i += 1
            rc, _ = eng.step_boundary()
            if rc == binding.IDLE:
                _, info = eng.step_core()
                if info.batch:
                    batches.append(info.batch)
            for r in eng.poll():
                finish[r["seq_id"]] = time.perf_counter() - t0
            if rc == binding.DONE:
                if i >= n:
                    break
                time.sleep(max(0.0, arrive[i] - (time.perf_counter() - t0)))
            if time.perf_counter() - t0 > window + drain_limit:
                break
        eng.sync()
        for r in eng.drain():
            finish[r["seq_id"]] = time.perf_counter() - t0
        wall = time.perf_counter() - t0
    finally:
        eng.close()
    done = ~np.isnan(finish)
    out = np.array([reqs[k]["gen_len"] for k in range(n)], np.float64)
    lat = normalized_latency(arrive[done], finish[done], out[done])
    return {"mode": mode, "requests": int(n), "finished": int(done.sum()), "wall_s": wall,
            "mean_core_batch": float(np.mean(batches)) if batches else 0.0, "core_steps": len(batches),
            "tokens_per_s": float(out[done].sum() / wall) if wall > 0 else 0.0,
            "normalized_latency": latency_stats(lat)}


def predict_points(shape, lm, points, seed=4, depth_probs=None, kv_gb=150.0, modes=("refill", "no_refill",
                                                                                      "fixed_depth")):
    """Predicted online serving (include/cdb_plan.h, cdb_predict_online) at (target, rate, window) points.

    The requests and arrivals are those the measured driver draws; exit
    depths, which the live gate decides on the GPU, are drawn from
    `depth_probs` over r_min, r_min + 1, ... (a stand-in with the measured
    mean).  Returns one dict per (point, mode) with the predicted mean and
    p50 normalised latency and the mean recurrent batch."""
    from continuous_depth_batching_gb300 import binding
    pool = make_online_requests(20000, shape.vocab, seed + 1)
    rng = np.random.default_rng(seed + 2)
    probs = np.asarray(depth_probs if depth_probs is not None else [1.0], np.float64)
    probs = probs / probs.sum()
    depths = np.arange(shape.r_min, shape.r_min + len(probs))
    out = []
    kv_tok = shape.n_kv_slots * 2 * shape.d_model * shape.elem_bytes
    for target, rate, window in points:
        arr = poisson_arrivals(rate, window, seed + 100 * target + 7)
        reqs = []
        for i in range(len(arr)):
            g = pool[i]["gen_len"]
            reqs.append(dict(prompt_len=len(pool[i]["prompt"]), gen_len=g,
                             exit_depths=rng.choice(depths, g - 1, p=probs).astype(np.int8)))
        W = min(512, max(64, 2 * target))
        K = 1 if shape.n_prelude + shape.n_coda == 0 else max(1, W // 4)
        job = binding.PlanJob(reqs, W=W, M=8192, r_max=shape.r_max, r_min=shape.r_min,
                              kv_blocks=int(kv_gb * 1e9 / (16 * kv_tok)), max_ctx=2048 + 512, max_new_cap=512)
        for mode in modes:
            fin, pred = binding.predict_online(job, arr, mode, K, lm)
            lat = normalized_latency(arr, fin, [r["gen_len"] for r in reqs])
            st = latency_stats(lat)
            out.append({"target_batch": target, "rate_per_s": rate, "mode": mode, "requests": len(reqs),
                        "predicted_mean_ms": st.get("mean_ms"), "predicted_p50_ms": st.get("p50_ms"),
                        "predicted_mean_core_batch": pred["mean_core_batch"]})
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--model", default="ouro")
    ap.add_argument("--targets", default="1,8,32,128")
    ap.add_argument("--modes", default="refill,no_refill,fixed_depth")
    ap.add_argument("--window", type=float, default=15.0, help="seconds of arrivals per measured point")
    ap.add_argument("--min-requests", type=int, default=24)
    ap.add_argument("--pilot", type=float, default=6.0)
    ap.add_argument("--kv-gb", type=float, default=150.0)
    ap.add_argument("--seed", type=int, default=4)
    ap.add_argument("--kv-slots", type=int, default=0,
                    help="KV slots per core layer (App. E.1): 0 depth-indexed, 1 single slot, 2 first-then-shared")
    ap.add_argument("--predict-fit", default="",
                    help="no GPU: predict with this latency fit (schedule_select --save-fit; 'roofline' for the "
                         "roofline model) at --rates")
    ap.add_argument("--rates", default="", help="target:rate pairs for --predict-fit, e.g. 8:6.86,32:21.83")
    ap.add_argument("--depth-probs", default="0.45,0.39,0.16",
                    help="exit-depth distribution from r_min up, for --predict-fit")
    args = ap.parse_args()

    if args.predict_fit:
        from continuous_depth_batching_gb300 import binding
        from synth import model_shape
        shape = model_shape(args.model)
        if args.predict_fit == "roofline":
            lm = binding.roofline_latency(shape, 6779.4, 1709.3)
        else:
            lm = binding.LatencyModel.from_dict(json.load(open(args.predict_fit))["fit"])
        points = [(int(t), float(r), args.window) for t, r in (p.split(":") for p in args.rates.split(","))]
        for row in predict_points(shape, lm, points, args.seed, [float(v) for v in args.depth_probs.split(",")],
                                  args.kv_gb, tuple(args.modes.split(","))):
            print(json.dumps(row), flush=True)
        return

    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.build import build
    from synth import make_weights, model_shape

    build()
    import dataclasses
    shape = dataclasses.replace(model_shape(args.model), kv_slots=args.kv_slots)
    dw = binding.device_weights(shape, make_weights(shape))
    max_ctx, gen_cap = 2048 + 512, 512
    kv_tok = binding.kv_bytes_per_token(shape)
    kv_blocks = int(args.kv_gb * 1e9 / (16 * kv_tok))
    pool = make_online_requests(20000, shape.vocab, args.seed + 1)
    mean_tokens = float(np.mean([r["gen_len"] for r in pool]))

    for target in [int(v) for v in args.targets.split(",")]:
        W = min(512, max(64, 2 * target))
        K = 1 if shape.n_prelude + shape.n_coda == 0 else max(1, W // 4)

        def make_engine(mode, W=W, K=K):
            return binding.Engine(shape, dw, mode=mode, W=W, M=8192, K=K, max_ctx=max_ctx, max_new_cap=gen_cap,
                                  kv_blocks=kv_blocks)

        # Pilots: first guess from one request's time in system at about 2 ms per loop step.
        rate = target / (mean_tokens * shape.r_max * 0.75 * 2e-3)
        for p in range(2):
            arr = poisson_arrivals(rate, args.pilot, args.seed + 100 * target + p)
            pt = run_point(make_engine, pool, arr, args.pilot, "refill", drain_limit=20.0)
            print(json.dumps({"target": target, "pilot": p, "rate_per_s": rate,
                              "mean_core_batch": pt["mean_core_batch"]}), flush=True)
            rate = rescale_rate(rate, pt["mean_core_batch"], target)
        window = min(4 * args.window, max(args.window, args.min_requests / rate))
        arr = poisson_arrivals(rate, window, args.seed + 100 * target + 7)
        for mode in args.modes.split(","):
            res = run_point(make_engine, pool, arr, window, mode)
            res.update(target_batch=target, rate_per_s=rate, window_s=window, W=W, K=K, model=shape.name,
                       kv_slots=shape.kv_slots)
            print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
