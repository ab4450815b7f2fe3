"""Refill / no-refill and minimum coda batch K: measured against the planner.

"Depth-adaptive Inference of Looped Language Models via Continuous Depth
Batching", §5 (recurrent-step latency model), §6.2 ("When is refill most
effective?"), §6.4 and Fig. 7 (the K ablation).  Every job replays the same
exit depths (App. C.2): the workload's own replay table, or for a live-gate
workload the depths a first refill run recorded.

1. Whole jobs on the GPU: no-refill, fixed depth and refill at each K of the
   sweep; GPU time from CUDA events around the job.
2. The per-stage latency model delta + gamma * rows + alpha * ctx fitted by
   non-negative least squares to per-call CUDA-event times of the fixed-depth
   and no-refill jobs (large and shrinking batches), rows and ctx taken from
   the step info each call returns.
3. The planner (include/cdb_plan.h) predicts every measured job from the
   fitted model and from the roofline model, and selects a schedule; the
   report shows whether each selection matches the measured best.

    python -m continuous_depth_batching_gb300.schedule_select --workload huginn --seqs 64
"""

from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

STAGE_PREFILL, STAGE_PRELUDE, STAGE_LOOP, STAGE_CODA = 1, 2, 3, 4
COLS = {STAGE_PREFILL: 0, STAGE_PRELUDE: 3, STAGE_LOOP: 6, STAGE_CODA: 9}
NAMES = {0: "prefill", 3: "prelude", 6: "core", 9: "coda"}


def run_job(eng_args, reqs, depths, *, per_call=False):
    """One whole job; returns (gpu seconds, per-call rows [(features, seconds)], exit depths)."""
    import numpy as np
    import torch

    from continuous_depth_batching_gb300 import binding
    eng = binding.Engine(*eng_args[0], **eng_args[1])
    s = eng.stream
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(s)
    for r in reqs:
        fe = depths.get(r["seq_id"]) if depths is not None else None
        eng.admit(r["seq_id"], r["prompt"], r["gen_len"], fe)
    calls = []

    def feats(info):
        x = np.zeros(12)
        for st, b, c, pt in ((info.stage, info.batch, info.ctx, info.prefill_tokens),
                             (info.stage2, info.batch2, info.ctx2, 0)):
            if st in COLS:
                j = COLS[st]
                x[j] += 1
                x[j + 1] += pt if st == STAGE_PREFILL else b
                x[j + 2] += c
        return x

    while True:
        if per_call:
            a = torch.cuda.Event(enable_timing=True)
            a.record(s)
        rc, info = eng.step_boundary()
        if per_call and info.stage:
            b = torch.cuda.Event(enable_timing=True)
            b.record(s)
            calls.append((feats(info), a, b))
        if rc == binding.DONE:
            break
        if rc == binding.IDLE:
            if per_call:
                a = torch.cuda.Event(enable_timing=True)
                a.record(s)
            rc, info = eng.step_core()
            if per_call:
                b = torch.cuda.Event(enable_timing=True)
                b.record(s)
                calls.append((feats(info), a, b))
    res = eng.drain(cap=len(reqs))
    g1.record(s)
    torch.cuda.synchronize()
    eng.close()
    rows = [(x, a.elapsed_time(b) / 1e3) for x, a, b in calls]
    return g0.elapsed_time(g1) / 1e3, rows, {r["seq_id"]: np.asarray(r["exit_depths"], np.int8) for r in res}


def fit_latency(rows):
    """Non-negative least squares of seconds on the 12 stage features."""
    import numpy as np
    from scipy.optimize import nnls
    X = np.array([x for x, _ in rows])
    y = np.array([t for _, t in rows])
    scale = np.maximum(np.abs(X).max(axis=0), 1.0)
    coef, _ = nnls(X / scale, y)
    coef = coef / scale
    model = {NAMES[j]: {"delta": float(coef[j]), "gamma": float(coef[j + 1]), "alpha": float(coef[j + 2])}
             for j in NAMES}
    pred = X @ coef
    rel = float(np.sqrt(np.mean((pred - y) ** 2)) / max(np.mean(y), 1e-12))
    return model, rel


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="huginn")
    ap.add_argument("--seqs", type=int, default=0, help="first N requests of the workload (0: all)")
    ap.add_argument("--W", type=int, default=0)
    ap.add_argument("--ks", default="", help="K values of the refill sweep (default 1, W/8, W/4, W/2, W)")
    ap.add_argument("--save-fit", default="", help="write the fitted latency model (JSON) to this path")
    args = ap.parse_args()

    import dataclasses

    import numpy as np
    import torch

    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.build import build
    from synth import make_requests, make_weights, model_shape, workload

    build()
    wl = workload(args.workload)
    if args.W:
        wl = dataclasses.replace(wl, W=args.W)
    shape = model_shape(wl.model)
    dw = binding.device_weights(shape, make_weights(shape))
    reqs = make_requests(wl, shape.vocab, shape.r_max, shape.r_min)
    if args.seqs:
        reqs = reqs[:args.seqs]
    max_ctx = (wl.prompt_hi + wl.gen_hi - 1 + 15) // 16 * 16
    base = dict(W=wl.W, M=wl.M, max_ctx=max_ctx, max_new_cap=wl.gen_hi)

    def eng(mode, K):
        return ((shape, dw), dict(base, mode=mode, K=K))

    # Exit depths every job replays.
    if reqs[0]["replay"] is not None:
        depths = {r["seq_id"]: np.asarray(r["replay"], np.int8) for r in reqs}
    else:
        _, _, depths = run_job(eng("refill", 1), reqs, None)
    W = wl.W
    ks = [int(k) for k in args.ks.split(",")] if args.ks else sorted({1, max(1, W // 8), max(1, W // 4),
                                                                       max(1, W // 2), W})
    measured = {}
    fit_rows = []
    for name, mode, K, pc in [("fixed_depth", "fixed_depth", 1, True), ("no_refill", "no_refill", 1, True)] + \
            [(f"refill_K{k}", "refill", k, False) for k in ks]:
        t, rows, _ = run_job(eng(mode, K), reqs, depths, per_call=pc)
        if pc:
            fit_rows += rows
            t, _, _ = run_job(eng(mode, K), reqs, depths)  # the job's own time without per-call events
        measured[name] = t
        print(json.dumps({"measured": name, "seconds": round(t, 4)}), flush=True)
    fitted, rel = fit_latency(fit_rows)
    print(json.dumps({"fit": fitted, "rms_rel_error_per_call": round(rel, 4), "calls": len(fit_rows)}), flush=True)
    if args.save_fit:
        with open(args.save_fit, "w") as fh:
            json.dump({"model": shape.name, "fit": fitted}, fh)

    peaks = {"hbm_gbs": 6779.4, "bf16_tflops_sustained": 1709.3}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peaks.update(json.load(open(pk)))
    models = {"fitted": binding.LatencyModel.from_dict(fitted),
              "roofline": binding.roofline_latency(shape, peaks["hbm_gbs"], peaks["bf16_tflops_sustained"])}
    job = binding.PlanJob([dict(prompt_len=len(r["prompt"]), gen_len=r["gen_len"], exit_depths=depths[r["seq_id"]])
                           for r in reqs], W=W, M=wl.M, r_max=shape.r_max, r_min=shape.r_min,
                          kv_blocks=W * (max_ctx // 16), max_ctx=max_ctx, max_new_cap=wl.gen_hi)
    best_meas = min((k for k in measured if k != "fixed_depth"), key=measured.get)
    report = {"workload": wl.name, "seqs": len(reqs), "W": W, "ks": ks, "measured_s": measured,
              "measured_best": best_meas, "models": {}}
    for mname, lm in models.items():
        pred = {}
        for name in measured:
            mode = "refill" if name.startswith("refill") else name
            K = int(name[len("refill_K"):]) if name.startswith("refill") else 1
            pred[name] = binding.predict_job(job, mode, K, lm)["seconds"]
        sel = binding.select_schedule(job, lm)
        pick = "no_refill" if sel["mode"] == "no_refill" else f"refill_K{sel['K']}"
        ranked = min((k for k in pred if k != "fixed_depth"), key=pred.get)
        norm = {k: pred[k] / pred["fixed_depth"] for k in pred}
        meas_norm = {k: measured[k] / measured["fixed_depth"] for k in measured}
        report["models"][mname] = {
            "predicted_s": pred, "predicted_over_fixed": norm, "measured_over_fixed": meas_norm,
            "max_rel_error_over_fixed": max(abs(norm[k] - meas_norm[k]) / meas_norm[k] for k in norm),
            "selection": {"mode": sel["mode"], "K": sel["K"]}, "best_of_measured_set": ranked,
            "matches_measured_best": ranked == best_meas,
            "measured_cost_of_choice": (measured.get(pick, None) / measured[best_meas]) if pick in measured else None,
            "model": lm.as_dict()}
    print(json.dumps(report), flush=True)


if __name__ == "__main__":
    main()
