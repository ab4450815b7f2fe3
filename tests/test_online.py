"""Host-side helpers of the online-serving driver (continuous_depth_batching_gb300/online.py).

"Depth-adaptive Inference of Looped Language Models via Continuous Depth
Batching", §6.3: Poisson arrivals at rate lambda and normalised latency
(end-to-end time / output tokens).  Checked against the Poisson process's
own laws (count mean lambda*T, exponential gaps of mean 1/lambda), the
definition of normalised latency and Little's law for the rate update.
"""

import numpy as np
import pytest

from continuous_depth_batching_gb300.online import (latency_stats, make_online_requests, normalized_latency,
                                                    poisson_arrivals, rescale_rate)


def test_poisson_arrivals_follow_the_process():
    rate, T = 50.0, 400.0
    a = poisson_arrivals(rate, T, seed=3)
    assert np.all(np.diff(a) > 0) and a[0] > 0 and a[-1] < T
    n = len(a)
    assert abs(n - rate * T) < 4 * np.sqrt(rate * T)           # count ~ Poisson(lambda T)
    gaps = np.diff(np.concatenate([[0.0], a]))
    assert abs(gaps.mean() - 1 / rate) < 4 * (1 / rate) / np.sqrt(n)
    assert abs(np.median(gaps) - np.log(2) / rate) < 0.05 / rate  # exponential median
    assert np.array_equal(a, poisson_arrivals(rate, T, seed=3))


def test_normalized_latency_and_stats():
    lat = normalized_latency([0.0, 1.0, 2.0], [2.0, 2.0, 6.0], [4, 2, 8])
    np.testing.assert_allclose(lat, [0.5, 0.5, 0.5])
    st = latency_stats(np.array([0.001, 0.002, 0.003, 0.004]))
    assert st["n"] == 4 and st["mean_ms"] == pytest.approx(2.5) and st["p50_ms"] == pytest.approx(2.5)
    assert latency_stats([])["n"] == 0


def test_rate_rescaling_is_littles_law_with_bounded_steps():
    assert rescale_rate(10.0, 16.0, 32.0) == pytest.approx(20.0)
    assert rescale_rate(10.0, 64.0, 32.0) == pytest.approx(5.0)
    assert rescale_rate(10.0, 1.0, 512.0) == pytest.approx(40.0)   # step capped at 4x
    assert rescale_rate(10.0, 0.0, 8.0) == pytest.approx(40.0)


def test_online_requests_have_the_stated_lengths():
    reqs = make_online_requests(500, 1000, seed=1)
    p = np.array([len(r["prompt"]) for r in reqs])
    g = np.array([r["gen_len"] for r in reqs])
    assert p.min() >= 64 and p.max() <= 2048 and g.min() >= 32 and g.max() <= 512
    assert all(r["prompt"].max() < 1000 for r in reqs)


def test_predicted_points_run_on_the_cpu():
    """The planner's online prediction over the driver's own requests and arrivals."""
    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.online import predict_points
    from synth import model_shape
    shape = model_shape("ouro")
    lm = binding.roofline_latency(shape, 6779.4, 1709.3)
    rows = predict_points(shape, lm, [(8, 5.0, 4.0)], depth_probs=[0.45, 0.39, 0.16])
    assert [r["mode"] for r in rows] == ["refill", "no_refill", "fixed_depth"]
    for r in rows:
        assert r["requests"] > 0 and np.isfinite(r["predicted_mean_ms"]) and r["predicted_mean_ms"] > 0
    by = {r["mode"]: r["predicted_mean_ms"] for r in rows}
    assert by["fixed_depth"] >= by["refill"]   # fixed depth runs every token r_max loops
