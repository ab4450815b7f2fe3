#!/usr/bin/env python3
"""Decoded tokens/s of continuous depth batching on one GB300.

Workload: the Ouro-1.4B-shaped fully looped model (d 2048, 16x128 heads,
SwiGLU 5632, 24-layer core looped up to 4 times, bf16, seeded random weights)
decoding 256 synthetic requests (prompt lengths uniform 128..1024, 256
generated tokens each) in refill mode with W = 64 active sequences, M = 8192
prefill tokens, K = 1, 16-token KV blocks.

A step is one recurrent-core loop step of the engine (batch re-formation,
24 shared blocks at each token's own depth, exit gate, compaction) together
with the coda / prelude / prefill stages the scheduler interleaves before it.
`value` counts the tokens generated during K timed steps after W warm-up
steps, with the model and all requests resident (device-timed with CUDA events
on the library's compute stream).  `e2e` runs the whole offline job through
the public API (admit host prompts ... drain host results), wall-clocked.

--impl reference times the CPU oracle (the plain per-sequence decoder) on the
host cores, one generated token per step.
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decoded tokens/sec at 1 GB300 (refill vs fixed-depth); core-step % of roofline"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ouro")
    ap.add_argument("--mode", default="refill", choices=["refill", "no_refill", "fixed_depth"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-modes", action="store_true", help="skip the no-refill and fixed-depth full jobs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=30.0)
    ap.add_argument("--kv-slots", type=int, default=0,
                    help="KV slots per core layer: 0 = r_max (depth-indexed), 1 single-slot, 2 first-then-shared")
    return ap.parse_args()


def attention_traffic_ratio():
    """DRAM traffic / algorithmic bytes of the decode-attention kernel from the
    committed ncu summary, if it was captured from the current source."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "k_attn_tma_ouro_decode.md")
    src = os.path.join(ROOT, "continuous_depth_batching_gb300", "csrc", "attention.cu")
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    kv = {}
    for line in open(prof):
        if ":" in line and not line.startswith(("|", " ", "#")):
            k, _, v = line.partition(":")
            kv[k.strip()] = v.strip()
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if kv.get("source_sha256") != sha or "traffic_ratio_dram_over_algorithmic" not in kv:
        return None
    return float(kv["traffic_ratio_dram_over_algorithmic"])


def weight_gb(shape):
    """Bytes of weights one core step streams (every core layer, plus the adapter), in GB."""
    d, f = shape.d_model, shape.ffn
    per_layer = 4 * d * d + 3 * d * f
    n = shape.n_core * per_layer + (2 * d * d if shape.has_adapter else 0)
    return n * shape.elem_bytes / 1e9


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops_sustained"], "measured"
    return 6800.0, 1700.0, "fallback"


class Clocks:
    """nvidia-smi samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.index = index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(ms: float, tokens: float, world: int, device: str = "cuda"):
    """Whole-job figures over replicas: max of the ranks' times, sum of their tokens."""
    if world <= 1:
        return ms, tokens
    import torch
    import torch.distributed as dist
    mx = torch.tensor([ms], dtype=torch.float64, device=device)
    sm = torch.tensor([tokens], dtype=torch.float64, device=device)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[0])


def cpu_baseline(shape, wts, reqs, seconds, n_seqs=4, n_tokens=16):
    """The oracle as it stands, on a bounded sample of the same workload.

    n_seqs sequences at evenly spaced quantiles of the workload's prompt
    lengths, each decoded alone: prefill, then its first n_tokens generated
    tokens.  A prefill is not interruptible, so prompts are cut to the length
    whose prefills take about half the budget together, estimated from an
    untimed 16-token prefill (long-context workloads would otherwise spend
    tens of minutes in one prompt); the sample says so when it cuts."""
    import numpy as np  # noqa: F401
    from oracle.model import OracleModel, iter_decode
    om = OracleModel(shape, wts)
    order = sorted(reqs, key=lambda r: len(r["prompt"]))
    picks = [order[min(len(order) - 1, int((k + 0.5) * len(order) / n_seqs))] for k in range(n_seqs)]
    t = time.perf_counter()
    next(iter_decode(om, order[0]["prompt"][:16], 2))
    per_tok = (time.perf_counter() - t) / 16
    pmax = max(16, int(0.5 * seconds / n_seqs / max(per_tok, 1e-9)))
    t0 = time.perf_counter()
    tokens, done = 0, []
    for r in picks:
        n = 0
        for _ in iter_decode(om, r["prompt"][:pmax], min(n_tokens, r["gen_len"])):
            n += 1
            tokens += 1
        done.append((r["seq_id"], len(r["prompt"]), n))
    dt = time.perf_counter() - t0
    desc = "; ".join(f"seq {s} (prompt {p}{f', first {pmax} tokens' if p > pmax else ''}): prefill + {n} "
                     f"generated tokens" for s, p, n in done)
    return {"value": tokens / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n_seqs} sequences at the prompt-length quantiles: " + desc +
                      f", {dt:.1f} s, fp64 numpy oracle"}


def run_reference(args):
    rank, world, _ = dist_setup()
    if rank != 0:
        return
    from oracle.model import OracleModel, iter_decode
    from synth import make_requests, make_weights, model_shape, workload
    wl = workload(args.workload)
    shape = dataclasses.replace(model_shape(wl.model), kv_slots=args.kv_slots)
    wts = make_weights(shape)
    reqs = sorted(make_requests(wl, shape.vocab, shape.r_max, shape.r_min), key=lambda r: len(r["prompt"]))
    om = OracleModel(shape, wts)

    def stream():
        for r in reqs:
            for _ in iter_decode(om, r["prompt"], r["gen_len"]):
                yield r["seq_id"]

    g = stream()
    for _ in range(args.warmup):
        next(g)
    t0 = time.perf_counter()
    used = set()
    for _ in range(args.steps):
        used.add(next(g))
    dt = time.perf_counter() - t0
    v = args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(wl, shape, args.mode, "oracle, one generated token per step"),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"sequences {sorted(used)} in prompt-length order, one token per step"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _config(wl, shape, mode, flush):
    return {"workload": f"{wl.name}-shaped offline decode: {wl.n_seqs} seqs, prompts U[{wl.prompt_lo},"
                        f"{wl.prompt_hi}], {wl.gen_hi} generated, W={wl.W}, M={wl.M}, K={wl.K}",
            "model": f"{shape.name}: d{shape.d_model} {shape.n_heads}x{shape.head_dim} ffn{shape.ffn} "
                     f"{shape.n_prelude}-{shape.n_core}-{shape.n_coda} r_max{shape.r_max} {shape.dtype}",
            "mode": mode, "global_batch": wl.W, "seq_len": wl.prompt_hi + wl.gen_hi,
            "kv_layout": {0: "depth-indexed", 1: "single-slot", 2: "first-then-shared"}.get(
                shape.kv_slots if shape.kv_slots < shape.r_max else 0, f"{shape.kv_slots} slots"),
            "parallelism": "replicas", "l2": flush}


def live_core_costs(eng, stream, binding, n_steps):
    """Live core-step time and per-class costs by step deltas.

    CUDA events go around each cdb_step_core call only, so programmatic
    dependent launch stays in effect between the step's kernels.  Steps cycle
    through no repeat and cdb_profile_repeat of each class (its kernels
    launched twice, writing the same values); a class's live cost is the mean
    time of its repeated steps minus the mean time of plain steps.  RMSNorm
    (which folds pending split-K partials in place) is not repeated: it stays
    in "other", the core-step time not attributed to a class.
    """
    import torch
    classes = [None, "attention", "gemm", "rowwise"]
    times = {c: [] for c in classes}
    bound = {}  # boundary calls that did work, by stage: (events, count)
    i = 0
    while i < n_steps * len(classes):
        cls = classes[i % len(classes)]
        eng.profile_repeat(cls)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rc, info = eng.step_boundary()
        if rc == binding.DONE:
            break
        if rc != binding.IDLE:
            b.record(stream)
            bound.setdefault(binding.STAGES.get(info.stage, str(info.stage)), []).append((a, b))
            continue
        a.record(stream)
        eng.step_core()
        b.record(stream)
        times[cls].append((a, b))
        i += 1
    eng.profile_repeat(None)
    torch.cuda.synchronize()
    mean = {c: (sum(a.elapsed_time(b) for a, b in v) / len(v)) if v else float("nan") for c, v in times.items()}
    base = mean[None]
    n_core = sum(len(v) for v in times.values())
    out = {"core_step_ms": base, "steps_per_class": min(len(v) for v in times.values()),
           "boundary_ms_per_core_step": {k: sum(a.elapsed_time(b) for a, b in v) / max(n_core, 1)
                                         for k, v in bound.items()},
           "boundary_calls_per_core_step": {k: len(v) / max(n_core, 1) for k, v in bound.items()}}
    for c in classes[1:]:
        out[c] = mean[c] - base
    out["rowwise_note"] = "the SwiGLU combine (bf16 decode runs RoPE and the KV write inside attention); RMSNorm folds are in other"
    out["other"] = base - sum(out[c] for c in classes[1:])
    return out


def run_ours(args):
    import numpy as np
    import torch

    from continuous_depth_batching_gb300 import binding, metrics
    from continuous_depth_batching_gb300.build import build
    from synth import make_requests, make_weights, model_shape, workload

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build()
    wl = workload(args.workload)
    shape = dataclasses.replace(model_shape(wl.model), kv_slots=args.kv_slots)
    wts = make_weights(shape)
    dw = binding.device_weights(shape, wts)
    reqs = make_requests(wl, shape.vocab, shape.r_max, shape.r_min)
    max_ctx = (wl.prompt_hi + wl.gen_hi - 1 + 15) // 16 * 16
    kw = dict(mode=args.mode, W=wl.W, M=wl.M, K=wl.K, max_ctx=max_ctx, max_new_cap=wl.gen_hi)

    def admit_all(eng):
        for r in reqs:
            eng.admit(r["seq_id"], r["prompt"], r["gen_len"], r["replay"])

    def advance(eng, n_core):
        toks = cores = 0
        while cores < n_core:
            rc, info = eng.step_boundary()
            toks += info.new_tokens
            if rc == binding.DONE:
                break
            if rc == binding.IDLE:
                rc, info = eng.step_core()
                cores += 1
        return toks, cores

    eng = binding.Engine(shape, dw, **kw)
    admit_all(eng)
    advance(eng, args.warmup)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    stream = torch.cuda.current_stream()
    l0 = binding.kernel_launches()
    print(f"launches_before_timed={l0}", file=sys.stderr, flush=True)
    clk = Clocks(local)
    clk.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    toks, cores = advance(eng, args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1)
    launches = binding.kernel_launches() - l0
    # Kernel-class timing: CUDA events around each attention / GEMM launch in
    # the window right after the timed one (events between kernels would break
    # the programmatic-dependent-launch overlap inside the timed window).
    prof_steps = max(1, min(args.steps, 100))
    eng.profile_enable(True, core_only=True)
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    _, pcores = advance(eng, prof_steps)
    p1.record(stream)
    prof = eng.profile_read()
    eng.profile_enable(False)
    prof_ms = p0.elapsed_time(p1)
    live = live_core_costs(eng, stream, binding, max(8, min(args.steps, 200)))
    eng.close()
    ms, tot_toks = aggregate(ms, toks, world)
    value = tot_toks / (ms / 1e3)

    # Roofline of the dominant kernel class (largest device time in the window).
    hbm, tf, src = peaks()
    dom = max((k for k in prof if prof[k]["launches"] > 0), key=lambda k: prof[k]["ms"])
    st = prof[dom]
    per_launch_ms = st["ms"] / st["launches"]
    inten = st["flops"] / max(st["bytes"], 1.0)
    if inten < tf * 1e12 / (hbm * 1e9):
        achieved = st["bytes"] / st["launches"] / (per_launch_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm}
    else:
        achieved = st["flops"] / st["launches"] / (per_launch_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf, "unit": "TFLOP/s", "frac": achieved / tf}
    ratio = attention_traffic_ratio() if dom == "attention" else None
    traffic = ratio * st["bytes"] / st["launches"] if ratio is not None else None
    roof.update({"kernel": dom, "traffic": traffic, "peak_source": src,
                 "traffic_source": ("ncu dram__bytes_read+write of one captured launch over its algorithmic "
                                    "bytes (profiles/k_attn_tma_ouro_decode.md), times this window's algorithmic "
                                    "bytes per launch") if traffic is not None else None,
                 "window": f"{pcores} core steps right after the timed ones, CUDA events on the compute stream",
                 "share_of_step": st["ms"] / prof_ms,
                 "classes": {k: {"launches": v["launches"], "ms": round(v["ms"], 3),
                                 "GBps": (v["bytes"] / (v["ms"] / 1e3) / 1e9) if v["ms"] else None,
                                 "TFps": (v["flops"] / (v["ms"] / 1e3) / 1e12) if v["ms"] else None}
                             for k, v in prof.items()}})
    # Whole core step (the metric's "core-step % of roofline"): the algorithmic
    # bytes and FLOPs of every kernel class per core step, averaged over the
    # profile window, against the unprofiled time per core step of the timed
    # window; the roofline time is max(bytes / HBM peak, FLOPs / tensor peak).
    by_step = sum(v["bytes"] for v in prof.values()) / max(pcores, 1)
    fl_step = sum(v["flops"] for v in prof.values()) / max(pcores, 1)
    t_step = live["core_step_ms"] / 1e3
    t_roof = max(by_step / (hbm * 1e9), fl_step / (tf * 1e12))
    core_step = {"bytes_per_step": by_step, "flops_per_step": fl_step, "s_per_step": t_step,
                 "achieved_GBps": by_step / t_step / 1e9, "achieved_TFps": fl_step / t_step / 1e12,
                 "roofline_s": t_roof, "frac": t_roof / t_step,
                 "bound": "hbm" if by_step / (hbm * 1e9) >= fl_step / (tf * 1e12) else "tensor",
                 "peaks": {"hbm_GBps": hbm, "tensor_TFps": tf, "source": src},
                 "how": "algorithmic bytes and FLOPs of the core steps' launches (profile window, core steps "
                        "only) over the live core-step time (CUDA events around each cdb_step_core, none "
                        "between its kernels)",
                 "live_ms": live}

    def full_job(mode):
        """The whole offline job through the public API: admit host prompts ... drain host results.

        Also returns the prefill share of GPU time (alpha of eq. 2), from CUDA
        events around every boundary call that ran a prefill stage.
        """
        eng2 = binding.Engine(shape, dw, **dict(kw, mode=mode))
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        pairs = []
        t0 = time.perf_counter()
        g0.record(stream)
        admit_all(eng2)
        n_core = 0
        while True:
            a = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            rc, info = eng2.step_boundary()
            if info.stage == binding_stage_prefill:
                b = torch.cuda.Event(enable_timing=True)
                b.record(stream)
                pairs.append((a, b))
            if rc == binding.DONE:
                break
            if rc == binding.IDLE:
                eng2.step_core()
                n_core += 1
        res = eng2.drain(cap=len(reqs))
        g1.record(stream)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        gpu_ms = g0.elapsed_time(g1)
        pre_ms = sum(a.elapsed_time(b) for a, b in pairs)
        gen = sum(len(r["tokens"]) for r in res)
        depth = float(np.mean(np.concatenate([r["exit_depths"] for r in res if len(r["exit_depths"])])))
        h2d, d2h = eng2.io_bytes()
        eng2.close()
        return {"value": gen / dt, "unit": UNIT, "h2d_bytes_per_step": h2d / max(n_core, 1),
                "d2h_bytes_per_step": d2h / max(n_core, 1), "core_steps": n_core, "seconds": dt,
                "tokens": gen, "finished_sequences": len(res), "alpha": pre_ms / gpu_ms,
                "mean_exit_depth": depth}

    binding_stage_prefill = 1
    e2e = None
    modes = None
    if not args.no_e2e:
        e2e = full_job(args.mode)
        if not args.no_modes and args.mode == "refill":
            fixed = full_job("fixed_depth")
            norefill = full_job("no_refill")
            F0, Fr = metrics.token_flops(shape)
            sdec = metrics.s_dec(F0, Fr, shape.r_max, e2e["mean_exit_depth"])
            se2e = metrics.s_e2e(fixed["alpha"], sdec)
            speed = e2e["value"] / fixed["value"]
            modes = {"refill": e2e["value"], "no_refill": norefill["value"], "fixed_depth": fixed["value"],
                     "unit": UNIT, "refill_vs_fixed": speed, "no_refill_vs_fixed": norefill["value"] / fixed["value"],
                     "mean_exit_depth": e2e["mean_exit_depth"], "S_dec": sdec,
                     "alpha_fixed_depth": fixed["alpha"], "alpha_refill": e2e["alpha"], "S_e2e": se2e,
                     "realised_fraction_of_S_e2e": speed / se2e,
                     "note": "whole 256-sequence jobs through the public API, wall clock; S_dec eq. (1) "
                             "with parameter FLOPs, S_e2e eq. (2) with alpha from the fixed-depth job"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(shape, wts, reqs, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / max(cores, 1), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": _config(wl, shape, args.mode,
                                  f"inputs larger than L2 ({weight_gb(shape):.1f} GB of weights per step)"),
                "roofline": roof, "core_step_roofline": core_step, "cpu_baseline": cpu, "e2e": e2e,
                "modes": modes, "gpu_launches": launches,
                "clocks": clocks, "tokens_in_window": tot_toks, "core_steps": cores}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
