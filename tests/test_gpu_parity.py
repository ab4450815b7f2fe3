"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Bar (from the method's invariance: batching does not change predictions or
exit decisions): generated tokens and exit depths identical, with gate logits
within 1e-3 of the threshold and near-tied argmaxes forced to the oracle's
decision; logits, coda inputs and gate logits within 1e-4 (fp32 models) or
2e-2 (bf16 models).
"""

import dataclasses

import numpy as np
import pytest

from synth import make_requests, make_weights, model_shape, workload
from tests.gpu_util import check_forced, compare, gpu_run, oracle_traces

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-4
BF16_TOL = 2e-2
# A bf16 run may pick either token of a top-2 pair closer than the arithmetic
# noise between two correct implementations: the oracle-only noise floor of
# these two-layer bf16 models (float64 against float32 reductions,
# oracle/noise_floor.py) is 0.0034 in logits and 0.0010 in gate logits.  Such
# argmaxes (top-2 gap below three times the floor) are pinned to the oracle's
# choice, counted, and their logits still compared.
BF16_GAP = 1e-2
GAP = {"fp32": 1e-3, "bf16": BF16_GAP}
# Largest share of forced decisions (gate decisions, tokens).  The bands cover
# 0-3% of the tokens of these random-weight models in fp32 and 0-15% in bf16
# (measured on GB300; the single-slot model repeats tokens with small top-2
# gaps and is the highest).
MAX_FORCED = {"fp32": 0.05, "bf16": 0.15}


@pytest.fixture(scope="module")
def tiny():
    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.build import build
    build()
    shape = model_shape("tiny")
    wts = make_weights(shape)
    reqs = make_requests(workload("tiny"), shape.vocab)
    return shape, wts, binding.device_weights(shape, wts), reqs


@pytest.fixture(scope="module")
def tiny_ref(tiny):
    shape, wts, _, reqs = tiny
    return oracle_traces(shape, wts, reqs, "adaptive", keep_logits=16)


def test_tiny_refill_matches_oracle(tiny, tiny_ref):
    shape, _, dw, reqs = tiny
    out, trace = gpu_run(shape, dw, reqs, tiny_ref, mode="refill", W=4, K=1, trace_tokens=16,
                         trace_gate=True, attn_split=16)
    err = compare(out, tiny_ref, FP32_TOL, check_gate=True)
    check_forced(tiny_ref, None, GAP["fp32"], MAX_FORCED["fp32"], label="tiny")
    depths = np.concatenate([o["exit_depths"] for o in out.values()])
    assert set(depths.tolist()) >= {2, 3, 4, 8}, "exit depths should spread"
    assert any(len(r["hist"]) > 1 for r in trace if r["stage"] == "loop"), "refill mixes depths"
    print("tiny refill max err", err)


def test_tiny_no_refill_matches_oracle(tiny, tiny_ref):
    shape, _, dw, reqs = tiny
    out, _ = gpu_run(shape, dw, reqs, tiny_ref, mode="no_refill", W=4, trace_tokens=16, attn_split=16)
    compare(out, tiny_ref, FP32_TOL)


def test_tiny_fixed_depth_matches_oracle(tiny):
    shape, wts, dw, reqs = tiny
    ref = oracle_traces(shape, wts, reqs[:4], "fixed", keep_logits=16)
    out, trace = gpu_run(shape, dw, reqs[:4], ref, mode="fixed_depth", W=4, trace_tokens=16, attn_split=16)
    compare(out, ref, FP32_TOL)
    assert all(len(r["hist"]) == 1 for r in trace if r["stage"] == "loop"), "fixed depth runs cohorts"
    assert all(list(o["exit_depths"]) == [shape.r_max] * 15 for o in out.values())


def test_modes_and_batch_sizes_agree_bit_exactly(tiny, tiny_ref):
    """Refill, no-refill and one-slot sequential runs produce identical bits."""
    shape, _, dw, reqs = tiny
    runs = [gpu_run(shape, dw, reqs, tiny_ref, mode=m, W=w, trace_tokens=16, attn_split=16)[0]
            for m, w in [("refill", 4), ("no_refill", 4), ("refill", 1), ("refill", 8)]]
    for other in runs[1:]:
        for sid in runs[0]:
            np.testing.assert_array_equal(runs[0][sid]["tokens"], other[sid]["tokens"])
            np.testing.assert_array_equal(runs[0][sid]["exit_depths"], other[sid]["exit_depths"])
            np.testing.assert_array_equal(runs[0][sid]["logits"], other[sid]["logits"])


def test_chunked_prefill_matches_oracle(tiny, tiny_ref):
    """Prompts split across prefill batches of M=20 tokens give the same result."""
    shape, _, dw, reqs = tiny
    out, trace = gpu_run(shape, dw, reqs, tiny_ref, mode="refill", W=4, M=20, trace_tokens=16, attn_split=16)
    compare(out, tiny_ref, FP32_TOL)
    assert any(r["stage"] == "prefill" and r["prefill_tokens"] == 20 for r in trace)


def test_single_split_attention_matches(tiny, tiny_ref):
    shape, _, dw, reqs = tiny
    out, _ = gpu_run(shape, dw, reqs[:3], {k: tiny_ref[k] for k in range(3)}, mode="refill", W=4,
                     trace_tokens=16, attn_split=0)
    compare(out, {k: tiny_ref[k] for k in range(3)}, FP32_TOL)


def _mini(dtype, **kw):
    base = dict(name="mini", vocab=1024, d_model=256, n_heads=2, head_dim=128, ffn=512, n_prelude=0,
                n_core=2, n_coda=0, r_max=5, r_min=2, has_adapter=False, dtype=dtype, gate_bias=0.12)
    base.update(kw)
    return dataclasses.replace(model_shape("tiny"), **base)


def _reqs(shape, n, plo, phi, gen, seed=5):
    rng = np.random.default_rng(seed)
    return [dict(seq_id=i, prompt=rng.integers(0, shape.vocab, int(rng.integers(plo, phi + 1))).astype(np.int32),
                 gen_len=gen, replay=None) for i in range(n)]


def test_bf16_model_matches_oracle():
    from continuous_depth_batching_gb300 import binding
    shape = _mini("bf16")
    wts = make_weights(shape)
    reqs = _reqs(shape, 6, 20, 70, 10)
    ref = oracle_traces(shape, wts, reqs, "adaptive", keep_logits=10)
    out, _ = gpu_run(shape, binding.device_weights(shape, wts), reqs, ref, mode="refill", W=3, K=1,
                     trace_tokens=10, trace_gate=True, attn_split=32, gap_band=BF16_GAP)
    err = compare(out, ref, BF16_TOL, check_gate=True)
    check_forced(ref, None, BF16_GAP, MAX_FORCED["bf16"], label="bf16 mini")
    print("bf16 mini max err", err)


@pytest.mark.parametrize("dtype,tol", [("fp32", FP32_TOL), ("bf16", BF16_TOL)])
def test_huginn_like_model_matches_oracle(dtype, tol):
    """Prelude and coda transformer layers, adapter before every loop step, hd 96."""
    from continuous_depth_batching_gb300 import binding
    shape = _mini(dtype, d_model=192, n_heads=2, head_dim=96, ffn=384, n_prelude=1, n_core=2, n_coda=1,
                  has_adapter=True, r_max=6, gate_bias=0.05)
    wts = make_weights(shape)
    reqs = _reqs(shape, 5, 10, 40, 8, seed=9)
    rng = np.random.default_rng(1)
    for r in reqs[:2]:  # two sequences replay recorded depths, the rest use the live gate
        r["replay"] = rng.integers(2, shape.r_max + 1, r["gen_len"] - 1).astype(np.int8)
    ref = oracle_traces(shape, wts, reqs, "adaptive", keep_logits=8)
    out, _ = gpu_run(shape, binding.device_weights(shape, wts), reqs, ref, mode="refill", W=3, K=2,
                     trace_tokens=8, trace_gate=True, attn_split=16, gap_band=GAP[dtype])
    err = compare(out, ref, tol, check_gate=True)
    check_forced(ref, {r["seq_id"]: r["replay"] for r in reqs}, GAP[dtype], MAX_FORCED[dtype],
                 label=f"huginn-like {dtype}")
    print("huginn-like", dtype, "max err", err)


@pytest.mark.parametrize("kv_slots", [1, 2])
@pytest.mark.parametrize("dtype,tol", [("fp32", FP32_TOL), ("bf16", BF16_TOL)])
def test_shared_kv_layouts_match_oracle(kv_slots, dtype, tol):
    """Single-slot and first-then-shared caches (App. E.1) in refill mode.  The
    prefill budget keeps every prompt in one chunk (with a shared cache a
    prompt split across chunks would read its earlier chunk at the last loop
    step, which the sequence-alone oracle does not do)."""
    from continuous_depth_batching_gb300 import binding
    shape = _mini(dtype, kv_slots=kv_slots)
    wts = make_weights(shape)
    reqs = _reqs(shape, 6, 20, 70, 10, seed=21)
    ref = oracle_traces(shape, wts, reqs, "adaptive", keep_logits=10)
    out, _ = gpu_run(shape, binding.device_weights(shape, wts), reqs, ref, mode="refill", W=3, K=1,
                     trace_tokens=10, trace_gate=True, attn_split=32, gap_band=GAP[dtype])
    err = compare(out, ref, tol, check_gate=True)
    check_forced(ref, None, GAP[dtype], MAX_FORCED[dtype], label=f"shared kv s={kv_slots} {dtype}")
    print("shared kv", kv_slots, dtype, "max err", err)


def test_huginn_like_single_slot_cache_matches_oracle():
    """The layout the pages run Huginn with: one KV slot per core layer."""
    from continuous_depth_batching_gb300 import binding
    shape = _mini("bf16", d_model=192, n_heads=2, head_dim=96, ffn=384, n_prelude=1, n_core=2, n_coda=1,
                  has_adapter=True, r_max=6, gate_bias=0.05, kv_slots=1)
    wts = make_weights(shape)
    reqs = _reqs(shape, 5, 10, 40, 8, seed=19)
    ref = oracle_traces(shape, wts, reqs, "adaptive", keep_logits=8)
    out, _ = gpu_run(shape, binding.device_weights(shape, wts), reqs, ref, mode="refill", W=3, K=2,
                     trace_tokens=8, trace_gate=True, attn_split=16, gap_band=BF16_GAP)
    err = compare(out, ref, BF16_TOL, check_gate=True)
    check_forced(ref, None, BF16_GAP, MAX_FORCED["bf16"], label="huginn-like single slot")
    print("huginn-like single slot max err", err)


@pytest.mark.parametrize("variant,dtype,tol,kv_slots", [("looped", "fp32", FP32_TOL, 0),
                                                         ("huginn_like", "bf16", BF16_TOL, 1)])
def test_convergence_gate_matches_oracle(variant, dtype, tol, kv_slots):
    """Huginn's convergence exit (App. E.2) decided live on the GPU: the
    statistics c_d, exit depths and tokens match the oracle.  The bf16 case is
    the pages' Huginn setting: convergence exit over a single-slot cache.  A
    statistic within the gate tolerance of the threshold takes the oracle's
    decision (each side's c may be off by that much).

    With random weights c_d clusters tightly by loop step.  fp32 resolves
    tokens inside a cluster, so its threshold is the median of the deciding
    statistics (exit depths differ between tokens); in bf16 such a threshold
    would make every decision a rounding-noise tie, so the threshold sits in
    the gap between the step-2 and step-3 clusters (every token exits at 4)."""
    from continuous_depth_batching_gb300 import binding
    kw = dict(r_min=3, r_max=6, gate_kind="convergence", kv_slots=kv_slots)
    if variant == "huginn_like":
        kw.update(d_model=192, n_heads=2, head_dim=96, ffn=384, n_prelude=1, n_core=2, n_coda=1,
                  has_adapter=True)
    shape0 = _mini(dtype, conv_tau=0.0, **kw)
    wts = make_weights(shape0)
    reqs = _reqs(shape0, 5, 10, 40, 8, seed=23)
    free = oracle_traces(shape0, wts, reqs[:2])  # never exits: the statistics' range
    zs = np.array([z for tr in free.values() for z in tr.gate_logits])  # [forwards][r_max - 1]
    if dtype == "fp32":
        tau = float(np.median(zs[:, shape0.r_min - 2:shape0.r_max - 2]))
    else:
        tau = float(np.sqrt(zs[:, 1].min() * zs[:, 2].max()))
    shape = dataclasses.replace(shape0, conv_tau=tau)
    band = 1e-3 if dtype == "fp32" else BF16_TOL
    ref = oracle_traces(shape, wts, reqs, "adaptive", keep_logits=8, near_tol=band)
    out, _ = gpu_run(shape, binding.device_weights(shape, wts), reqs, ref, mode="refill", W=3, K=2,
                     trace_tokens=8, trace_gate=True, attn_split=16, gap_band=GAP[dtype])
    err = compare(out, ref, tol, check_gate=True)
    check_forced(ref, None, GAP[dtype], 0.25, label=f"convergence {variant} {dtype}")
    print("convergence", variant, dtype, "max err", err)
    depths = [e for tr in ref.values() for e in tr.exit_depths]
    assert min(depths) >= 3 and len(set(depths)) >= (2 if dtype == "fp32" else 1), depths
    assert sum(sum(tr.near_gate) for tr in ref.values()) <= len(depths) // 4


def test_poll_returns_each_finished_sequence_once(tiny, tiny_ref):
    """cdb_poll between steps hands out finished sequences without waiting;
    poll and the final drain together return every sequence exactly once, with
    the tokens of a run that only drains at the end (the online-serving driver
    relies on this)."""
    from continuous_depth_batching_gb300 import binding
    shape, _, dw, reqs = tiny
    eng = binding.Engine(shape, dw, mode="refill", W=2, M=64, K=1, max_ctx=64, max_new_cap=16, attn_split=16)
    for r in reqs:
        eng.admit(r["seq_id"], r["prompt"], r["gen_len"])
    seen = []
    polled = 0
    while True:
        rc, _ = eng.step_boundary()
        if rc == binding.DONE:
            break
        if rc == binding.IDLE:
            eng.step_core()
        got = eng.poll()
        polled += len(got)
        seen += got
    eng.sync()
    seen += eng.drain()
    eng.close()
    ids = [o["seq_id"] for o in seen]
    assert sorted(ids) == sorted(r["seq_id"] for r in reqs) and len(set(ids)) == len(ids)
    assert polled > 0, "sequences that finished early should come back from poll"
    ref, _ = gpu_run(shape, dw, reqs, None, mode="refill", W=2, M=64, K=1, max_ctx=64, attn_split=16, force=False)
    for o in seen:
        assert list(o["tokens"]) == list(ref[o["seq_id"]]["tokens"])


def test_degenerate_requests_match_oracle(tiny):
    """A one-token prompt, requests that only prefill (one generated token), a
    prompt chunked across prefill batches whose context ends exactly at
    max_ctx, mixed with ordinary requests; and an engine with nothing admitted."""
    from continuous_depth_batching_gb300 import binding
    shape, wts, dw, _ = tiny
    rng = np.random.default_rng(7)
    max_ctx = 48
    spec = [(1, 5), (6, 1), (1, 1), (40, 9), (20, 3)]  # (prompt, generated); 40 + 9 - 1 = max_ctx
    reqs = [dict(seq_id=i, prompt=rng.integers(0, shape.vocab, p).astype(np.int32), gen_len=g, replay=None)
            for i, (p, g) in enumerate(spec)]
    ref = oracle_traces(shape, wts, reqs, "adaptive")
    out, _ = gpu_run(shape, dw, reqs, ref, mode="refill", W=2, M=16, K=1, max_ctx=max_ctx, attn_split=16)
    compare(out, ref, FP32_TOL, check_logits=False)
    assert [len(out[i]["tokens"]) for i in range(len(spec))] == [g for _, g in spec]
    eng = binding.Engine(shape, dw, mode="refill", W=2, M=16, max_ctx=max_ctx, max_new_cap=4)
    assert eng.step_boundary()[0] == binding.DONE and eng.drain() == []
    eng.close()
