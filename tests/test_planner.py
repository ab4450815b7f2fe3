"""The latency planner (include/cdb_plan.h) against closed forms of the schedule.

"Depth-adaptive Inference of Looped Language Models via Continuous Depth
Batching", §5 (t = delta + gamma N_b + alpha N_c per recurrent step), §6.4 /
Fig. 7 (minimum coda batch K) and Algorithms 1-2.  With one cost term switched
on at a time the predicted time counts something the schedule fixes:

* core gamma: loop-step tokens, the sum of all exit depths (any mode);
* core alpha: sum over decode forwards of depth x (position + 1);
* prefill gamma / alpha: prompt tokens / causal pairs sum P (P + 1) / 2;
* coda gamma and prelude gamma: decode forwards, sum (gen_len - 1);
* core delta: core steps.  No-refill with one cohort (W >= requests, equal
  output lengths) runs, per generated token, as many steps as the deepest
  token of the cohort; refill with K = 1 and W >= requests never makes a
  token wait, so it runs as many steps as the longest chain of exit depths.
"""

import dataclasses

import numpy as np
import pytest

from continuous_depth_batching_gb300 import binding
from synth import model_shape


def _reqs(n, gen, r_min, r_max, seed=3, plo=5, phi=40):
    rng = np.random.default_rng(seed)
    return [dict(prompt_len=int(rng.integers(plo, phi + 1)), gen_len=gen,
                 exit_depths=rng.integers(r_min, r_max + 1, gen - 1).astype(np.int8)) for _ in range(n)]


def _lm(**terms):
    d = {}
    for k, v in terms.items():
        stage, term = k.split("_")
        d.setdefault(stage, {})[term] = v
    return binding.LatencyModel.from_dict(d)


@pytest.mark.parametrize("mode", ["refill", "no_refill", "fixed_depth"])
def test_cost_terms_count_the_schedule(mode):
    r_min, r_max = 2, 6
    reqs = _reqs(7, 9, r_min, r_max)
    job = binding.PlanJob(reqs, W=4, M=64, r_max=r_max, r_min=r_min)
    depth = [np.full(r["gen_len"] - 1, r_max) if mode == "fixed_depth" else r["exit_depths"] for r in reqs]
    want_steps = sum(int(e.sum()) for e in depth)
    want_ctx = sum(int((e * (r["prompt_len"] + np.arange(len(e)) + 1)).sum()) for e, r in zip(depth, reqs))
    fwd = sum(r["gen_len"] - 1 for r in reqs)
    P = np.array([r["prompt_len"] for r in reqs])
    assert binding.predict_job(job, mode, 1, _lm(core_gamma=1.0))["seconds"] == want_steps
    assert binding.predict_job(job, mode, 1, _lm(core_alpha=1.0))["seconds"] == want_ctx
    assert binding.predict_job(job, mode, 1, _lm(prefill_gamma=1.0))["seconds"] == P.sum()
    assert binding.predict_job(job, mode, 1, _lm(prefill_alpha=1.0))["seconds"] == (P * (P + 1) // 2).sum()
    assert binding.predict_job(job, mode, 1, _lm(coda_gamma=1.0))["seconds"] == fwd
    assert binding.predict_job(job, mode, 1, _lm(prelude_gamma=1.0))["seconds"] == fwd
    p = binding.predict_job(job, mode, 1, _lm(core_gamma=1.0))
    assert p["tokens"] == sum(r["gen_len"] for r in reqs)
    assert p["core_token_steps"] == want_steps


def test_core_steps_of_one_cohort_and_of_refill():
    r_min, r_max = 2, 5
    reqs = _reqs(6, 8, r_min, r_max, seed=11)
    job = binding.PlanJob(reqs, W=8, M=4096, S=1, r_max=r_max, r_min=r_min)
    E = np.stack([r["exit_depths"] for r in reqs])          # [request][decode forward]
    nr = binding.predict_job(job, "no_refill", 1, _lm(core_delta=1.0))
    assert nr["core_steps"] == E.max(axis=0).sum()
    rf = binding.predict_job(job, "refill", 1, _lm(core_delta=1.0))
    assert rf["core_steps"] == E.sum(axis=1).max()
    fx = binding.predict_job(job, "fixed_depth", 1, _lm(core_delta=1.0))
    assert fx["core_steps"] == r_max * E.shape[1]


def test_roofline_model_of_the_ouro_shape():
    shape = model_shape("ouro")
    lm = binding.roofline_latency(shape, 6000.0, 1500.0).as_dict()
    d, f = shape.d_model, shape.ffn
    core_bytes = shape.n_core * (4 * d * d + 3 * d * f) * 2
    assert lm["core"]["delta"] == pytest.approx(core_bytes / 6000e9)
    assert lm["core"]["alpha"] == pytest.approx(shape.n_core * 2 * d * 2 / 6000e9)
    assert lm["core"]["gamma"] == pytest.approx(2 * core_bytes / 2 / 1500e12)
    assert lm["coda"]["delta"] == pytest.approx(shape.vocab * d * 2 / 6000e9)
    assert lm["prelude"]["delta"] == 0.0
    # Launch cost adds to delta only.
    lm2 = binding.roofline_latency(shape, 6000.0, 1500.0, launch_s=1e-6).as_dict()
    assert lm2["core"]["delta"] > lm["core"]["delta"] and lm2["core"]["gamma"] == lm["core"]["gamma"]


def test_selection_follows_the_regime():
    """Memory-bound core steps (delta dominates): refill wins (§5).  Costly
    boundary stages with compute-bound core steps: no-refill wins (§6.2,
    Huginn).  Costly coda with refill forced on: a larger K wins (§6.4)."""
    r_min, r_max = 2, 8
    reqs = _reqs(32, 12, r_min, r_max, seed=5)
    job = binding.PlanJob(reqs, W=16, M=4096, r_max=r_max, r_min=r_min)
    mem = binding.select_schedule(job, _lm(core_delta=1.0, core_gamma=0.001))
    assert mem["mode"] == "refill" and mem["refill_seconds"] < mem["no_refill_seconds"]
    heavy = binding.select_schedule(job, _lm(core_gamma=0.01, coda_delta=1.0, prelude_delta=1.0))
    assert heavy["mode"] == "no_refill" and heavy["refill_seconds"] >= heavy["no_refill_seconds"]
    ks = {K: binding.predict_job(job, "refill", K, _lm(core_delta=0.1, core_gamma=0.01, coda_delta=1.0))["seconds"]
          for K in (1, 4, 16)}
    assert ks[4] < ks[1]


def test_planner_rejects_bad_jobs():
    reqs = _reqs(2, 4, 2, 4)
    job = binding.PlanJob(reqs, W=2, r_max=4, r_min=2)
    with pytest.raises(binding.CdbError):
        binding.predict_job(job, "refill", 0, _lm(core_delta=1.0))
    with pytest.raises(binding.CdbError):
        binding.predict_job(job, "refill", 1, _lm(core_delta=-1.0))
    bad = [dict(r, exit_depths=np.full(3, 9, np.int8)) for r in reqs]
    with pytest.raises(binding.CdbError):
        binding.predict_job(binding.PlanJob(bad, W=2, r_max=4, r_min=2), "refill", 1, _lm(core_delta=1.0))
    with pytest.raises(ValueError):
        binding.PlanJob([dict(reqs[0], exit_depths=np.zeros(1, np.int8))], W=2)
    huginn = dataclasses.replace(model_shape("huginn"), d_model=0)
    with pytest.raises(binding.CdbError):
        binding.roofline_latency(huginn, 1.0, 1.0)


def test_latency_fit_recovers_a_known_model():
    """The per-call regression of schedule_select (non-negative least squares on
    the twelve stage features) returns the coefficients that generated the
    times, including calls that ran a coda and a prelude together."""
    pytest.importorskip("scipy")
    from continuous_depth_batching_gb300.schedule_select import fit_latency
    true = {"prefill": (1e-3, 2e-6, 1e-9), "prelude": (5e-5, 1e-6, 0.0), "core": (1.4e-3, 1.2e-5, 3e-9),
            "coda": (2e-4, 3e-6, 1e-10)}
    col = {"prefill": 0, "prelude": 3, "core": 6, "coda": 9}
    coef = np.zeros(12)
    for k, (d, g, a) in true.items():
        coef[col[k]:col[k] + 3] = (d, g, a)
    rng = np.random.default_rng(0)
    rows = []
    for _ in range(3000):
        x = np.zeros(12)
        st = col[("prefill", "prelude", "core", "coda")[rng.integers(0, 4)]]
        x[st], x[st + 1] = 1, rng.integers(1, 64)
        x[st + 2] = x[st + 1] * rng.integers(100, 1000)
        if st == 9 and rng.random() < 0.5:      # coda followed by a prelude in one call
            x[3], x[4], x[5] = 1, x[10], x[11] + x[10]
        rows.append((x, float(x @ coef)))
    model, rel = fit_latency(rows)
    assert rel < 1e-6
    for k, (d, g, a) in true.items():
        got = model[k]
        assert got["delta"] == pytest.approx(d, rel=1e-4, abs=1e-9)
        assert got["gamma"] == pytest.approx(g, rel=1e-4, abs=1e-11)
        assert got["alpha"] == pytest.approx(a, rel=1e-4, abs=1e-14)


def test_step_info_reports_context_entries():
    """cdb_step_info.ctx / ctx2: the sum over a stage's rows of (position + 1),
    the cached entries each row's attention reads per layer."""
    P, gen = 10, 4
    sim = binding.Sim("refill", W=1, M=64, K=1, r_max=3, r_min=2)
    sim.admit(0, P, gen, np.array([2, 3, 2], np.int8))
    rc, info = sim.step_boundary()                      # prefill + prelude of the first decode token
    assert info.stage == 1 and info.ctx == P * (P + 1) // 2
    assert info.stage2 == 2 and info.batch2 == 1 and info.ctx2 == P + 1
    rc, info = sim.step_boundary()
    assert rc == binding.IDLE
    rc, info = sim.step_core()                          # the token at position P, loop step 1
    assert info.stage == 3 and info.batch == 1 and info.ctx == P + 1
    sim.step_boundary()
    sim.step_core()                                     # step 2: it exits (depth 2)
    rc, info = sim.step_boundary()                      # coda of position P, prelude of P + 1
    assert info.stage == 4 and info.ctx == P + 1 and info.stage2 == 2 and info.ctx2 == P + 2


@pytest.mark.parametrize("mode", ["refill", "no_refill", "fixed_depth"])
def test_online_prediction_reduces_to_offline_and_to_isolated_requests(mode):
    """All arrivals at 0: the online prediction is the offline one (same busy
    time, the last request finishes at it).  Arrivals far apart: every request
    runs alone, so its latency is the offline prediction of that request."""
    r_min, r_max = 2, 5
    reqs = _reqs(6, 7, r_min, r_max, seed=9)
    lm = _lm(prefill_delta=1e-3, prefill_gamma=1e-6, core_delta=2e-3, core_gamma=1e-5, core_alpha=1e-8,
             coda_delta=3e-4, prelude_delta=5e-5)
    job = binding.PlanJob(reqs, W=4, M=64, r_max=r_max, r_min=r_min)
    off = binding.predict_job(job, mode, 1, lm)
    fin, on = binding.predict_online(job, np.zeros(len(reqs)), mode, 1, lm)
    assert on["seconds"] == pytest.approx(off["seconds"]) and fin.max() == pytest.approx(off["seconds"])
    assert (fin > 0).all()
    gap = 10.0 * off["seconds"]
    arr = gap * np.arange(len(reqs))
    fin, _ = binding.predict_online(job, arr, mode, 1, lm)
    for i, r in enumerate(reqs):
        alone = binding.predict_job(binding.PlanJob([r], W=4, M=64, r_max=r_max, r_min=r_min), mode, 1, lm)
        assert fin[i] - arr[i] == pytest.approx(alone["seconds"])


def test_online_prediction_rejects_bad_arrivals():
    reqs = _reqs(3, 4, 2, 4)
    job = binding.PlanJob(reqs, W=2, r_max=4, r_min=2)
    with pytest.raises(binding.CdbError):
        binding.predict_online(job, [0.0, 2.0, 1.0], "refill", 1, _lm(core_delta=1.0))
    with pytest.raises(binding.CdbError):
        binding.predict_online(job, [-1.0, 0.0, 1.0], "refill", 1, _lm(core_delta=1.0))
    with pytest.raises(ValueError):
        binding.predict_online(job, [0.0, 1.0], "refill", 1, _lm(core_delta=1.0))


def test_roofline_model_of_the_huginn_shape():
    """Adapter in the core, two prelude and two coda blocks, the LM head in the coda."""
    shape = model_shape("huginn")
    lm = binding.roofline_latency(shape, 6000.0, 1500.0).as_dict()
    d, f, V = shape.d_model, shape.ffn, shape.vocab
    block = 4 * d * d + 3 * d * f
    assert lm["core"]["delta"] == pytest.approx((shape.n_core * block + 2 * d * d) * 2 / 6000e9)
    assert lm["prelude"]["delta"] == pytest.approx(shape.n_prelude * block * 2 / 6000e9)
    assert lm["coda"]["delta"] == pytest.approx((shape.n_coda * block + V * d) * 2 / 6000e9)
    assert lm["prelude"]["alpha"] == pytest.approx(shape.n_prelude * 2 * d * 2 / 6000e9)
    applications = shape.n_prelude + shape.r_max * shape.n_core + shape.n_coda
    assert lm["prefill"]["alpha"] == pytest.approx(4 * d * applications / 1500e12)


def test_prefill_chunks_follow_the_token_budget():
    """One prompt of P tokens with budget M is prefilled in ceil(P / M) chunks
    (App. A.1), and the prefill context entries are the causal pairs."""
    P = 100
    for M in (16, 33, 100, 128):
        job = binding.PlanJob([dict(prompt_len=P, gen_len=3, exit_depths=np.array([2, 2], np.int8))],
                              W=1, M=M, r_max=3, r_min=2)
        p = binding.predict_job(job, "refill", 1, _lm(prefill_delta=1.0, prefill_alpha=1e-9))
        assert p["prefill_stages"] == -(-P // M)
        assert p["prefill_seconds"] == pytest.approx(-(-P // M) + 1e-9 * P * (P + 1) / 2)
