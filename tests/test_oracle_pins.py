"""Pins of the CPU oracle to facts other than itself.

* Fixed depth with a depth-indexed cache is an unrolled pre-norm transformer of
  n_core * r_max layers (each loop step uses its own cache slots; §4.2 of the
  paper), so the oracle's fixed-depth tokens and logits must equal a full-
  sequence, cache-free causal forward computed with torch's own attention.
* With early exits, the oracle must equal a recursive, cache-free
  recomputation that applies the depth-clamp reading directly
  (tests/brute_force.py), including prelude/coda layers and the adapter; the
  same holds for the shared cache layouts of App. E.1, where the brute force
  states which loop step of each key is visible instead of using slots.
* Gate extremes: an always-positive gate exits every token at r_min (§4.3,
  lookahead: r_min = 2), an always-negative gate reproduces fixed depth.
* bf16 rounding equals torch's float32 -> bfloat16 conversion.
* RoPE scores depend only on the relative position.
* Executed FLOPs equal the closed form used by §5 eq. (1).
* Exit gaps of the depth-indexed cache are never written.
* Probe gate (§4.3): a closed form of the probe on a 2-element state, and the
  oracle's gate logits and exit depths equal the probe applied to the brute
  force's loop states (after the step) with the lookahead rule.
* bf16 storage (Table 1, bfloat16): at fixed depth the oracle's bf16 logits
  equal a full-sequence torch forward that casts through torch.bfloat16 at the
  same storage points, and dropping any one point moves the logits far outside
  that tolerance.
* Convergence exit (App. E.2): the oracle's statistics and exit depths equal
  the normalised L2 distances of the brute force's loop states with the
  lookahead rule applied to them; c = 1 exactly at step 1 when s_0 = 0; a
  threshold above every statistic exits at r_min = 3, a zero threshold
  reproduces fixed depth.
"""

import dataclasses
import functools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from synth import make_requests, make_weights, model_shape, workload
from oracle.model import OracleModel, decode_sequence, _bf16
from tests.brute_force import BruteForceLM


def micro(**kw):
    base = dict(name="micro", vocab=64, d_model=32, n_heads=4, head_dim=8, ffn=48,
                n_prelude=0, n_core=2, n_coda=0, r_max=3, r_min=2,
                has_adapter=False, dtype="fp32", init_std=0.2, gate_bias=0.0)
    base.update(kw)
    return dataclasses.replace(model_shape("tiny"), **base)


def prompt_for(shape, n, seed=7):
    rng = np.random.default_rng(seed)
    return rng.integers(0, shape.vocab, n).astype(np.int32)


# ---------------------------------------------------------------------------
# fixed depth == unrolled textbook transformer (torch, float64, no cache)
# ---------------------------------------------------------------------------

def torch_unrolled_logits(shape, weights, tokens):
    w = {k: torch.from_numpy(v.astype(np.float64)) for k, v in weights.items()}
    T = len(tokens)
    d, H, hd = shape.d_model, shape.n_heads, shape.head_dim
    x = w["embed"][torch.as_tensor(tokens, dtype=torch.long)]
    inv = shape.rope_theta ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rope(t):  # [H, T, hd]
        a, b = t[..., : hd // 2], t[..., hd // 2:]
        return torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1)

    def rms(t, g):
        return F.rms_norm(t, (d,), g, eps=shape.rms_eps)

    for _ in range(shape.r_max):
        for l in range(shape.n_core):
            p = f"core.{l}."
            u = rms(x, w[p + "attn_norm"])
            q, k, v = F.linear(u, w[p + "wqkv"]).split(d, dim=-1)
            q = rope(q.view(T, H, hd).transpose(0, 1))
            k = rope(k.view(T, H, hd).transpose(0, 1))
            v = v.view(T, H, hd).transpose(0, 1)
            o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
            x = x + F.linear(o.transpose(0, 1).reshape(T, d), w[p + "wo"])
            u = rms(x, w[p + "mlp_norm"])
            x = x + F.linear(F.silu(F.linear(u, w[p + "wg"])) * F.linear(u, w[p + "wu"]), w[p + "wd"])
    return F.linear(rms(x, w["final_norm"]), w["lm_head"]).numpy()


@pytest.mark.parametrize("r_max", [1, 3])
def test_fixed_depth_is_unrolled_transformer(r_max):
    shape = micro(r_max=r_max, r_min=min(2, r_max))
    wts = make_weights(shape)
    prompt = prompt_for(shape, 9)
    gen = 6
    tr = decode_sequence(OracleModel(shape, wts), prompt, gen, mode="fixed", keep_logits=gen)
    seq = np.concatenate([prompt, np.array(tr.tokens[:-1], dtype=np.int32)])
    ref = torch_unrolled_logits(shape, wts, seq)
    P = len(prompt)
    for t in range(gen):
        np.testing.assert_allclose(tr.logits[t], ref[P - 1 + t], atol=2e-5, rtol=0)
        assert tr.tokens[t] == int(np.argmax(ref[P - 1 + t]))
    assert tr.exit_depths == [r_max] * (gen - 1)


def test_tiny_config_fixed_depth_is_unrolled_transformer():
    shape = model_shape("tiny")
    wts = make_weights(shape)
    req = make_requests(workload("tiny"), shape.vocab)[3]
    gen = 5
    tr = decode_sequence(OracleModel(shape, wts), req["prompt"], gen, mode="fixed", keep_logits=gen)
    seq = np.concatenate([req["prompt"], np.array(tr.tokens[:-1], dtype=np.int32)])
    ref = torch_unrolled_logits(shape, wts, seq)
    P = len(req["prompt"])
    for t in range(gen):
        np.testing.assert_allclose(tr.logits[t], ref[P - 1 + t], atol=2e-5, rtol=0)


# ---------------------------------------------------------------------------
# early exit + depth clamp == cache-free recursion
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("variant", ["looped", "huginn_like"])
def test_adaptive_matches_brute_force(variant):
    if variant == "looped":
        shape = micro(r_max=4)
    else:
        shape = micro(r_max=4, n_prelude=1, n_core=1, n_coda=1, has_adapter=True)
    wts = make_weights(shape)
    prompt = prompt_for(shape, 5, seed=11)
    gen = 7
    rng = np.random.default_rng(5)
    depths = rng.integers(2, shape.r_max + 1, gen - 1).astype(np.int8)
    depths[1] = 2
    depths[2] = shape.r_max
    tr = decode_sequence(OracleModel(shape, wts), prompt, gen, mode="adaptive",
                         force_exit=depths, keep_logits=gen)
    assert tr.exit_depths == [int(x) for x in depths]
    bf = BruteForceLM(shape, wts, prompt, gen, lambda t: int(depths[t - 1]))
    toks, lg = bf.run()
    assert tr.tokens == toks
    for t in range(gen):
        np.testing.assert_allclose(tr.logits[t], lg[t], atol=2e-5, rtol=0)


def test_brute_force_detects_wrong_clamp():
    """Sensitivity: reading exited tokens at the current depth (no clamp) differs."""
    shape = micro(r_max=4)
    wts = make_weights(shape)
    prompt = prompt_for(shape, 5, seed=11)
    gen = 5
    depths = np.array([2, 2, 4, 3], dtype=np.int8)
    tr = decode_sequence(OracleModel(shape, wts), prompt, gen, force_exit=depths, keep_logits=gen)
    # A schedule that pretends every earlier token ran to full depth reads other states.
    bf = BruteForceLM(shape, wts, prompt, gen, lambda t: int(depths[t - 1]))
    bf.exit_depth = lambda i: shape.r_max if i < bf.P else int(depths[i - bf.P])
    honest = bf.run()[1]
    wrong = BruteForceLM(shape, wts, prompt, gen, lambda t: int(depths[t - 1]))
    wrong.exit_depth = lambda i: shape.r_max
    wrong_lg = wrong.run()[1]
    np.testing.assert_allclose(tr.logits[-1], honest[-1], atol=2e-5, rtol=0)
    assert np.max(np.abs(tr.logits[-1] - wrong_lg[-1])) > 1e-3


@pytest.mark.parametrize("kv_slots", [1, 2])
@pytest.mark.parametrize("variant", ["looped", "huginn_like"])
def test_shared_kv_layouts_match_brute_force(variant, kv_slots):
    """Single-slot and first-then-shared caches (App. E.1): the oracle's slot
    overwrites equal the brute force's explicit visible-step rule."""
    if variant == "looped":
        shape = micro(r_max=4, kv_slots=kv_slots)
    else:
        shape = micro(r_max=4, n_prelude=1, n_core=1, n_coda=1, has_adapter=True, kv_slots=kv_slots)
    wts = make_weights(shape)
    prompt = prompt_for(shape, 5, seed=13)
    gen = 6
    depths = np.array([2, 4, 3, 2, 4], dtype=np.int8)
    tr = decode_sequence(OracleModel(shape, wts), prompt, gen, force_exit=depths, keep_logits=gen)
    toks, lg = BruteForceLM(shape, wts, prompt, gen, lambda t: int(depths[t - 1])).run()
    assert tr.tokens == toks
    for t in range(gen):
        np.testing.assert_allclose(tr.logits[t], lg[t], atol=2e-5, rtol=0)
    # The layout matters: the depth-indexed cache gives other logits.
    deep = decode_sequence(OracleModel(dataclasses.replace(shape, kv_slots=0), wts), prompt, gen,
                           force_exit=depths, keep_logits=gen)
    assert max(np.abs(np.array(deep.logits) - np.array(tr.logits)).max(axis=1)) > 1e-3


# ---------------------------------------------------------------------------
# gate special cases, rounding, RoPE, FLOPs, gaps
# ---------------------------------------------------------------------------

def test_gate_extremes():
    shape = micro(r_max=5)
    prompt = prompt_for(shape, 6)
    gen = 6
    wts = make_weights(shape)
    hi = decode_sequence(OracleModel(dataclasses.replace(shape, gate_bias=100.0), wts), prompt, gen)
    assert hi.exit_depths == [2] * (gen - 1)
    hi3 = decode_sequence(OracleModel(dataclasses.replace(shape, gate_bias=100.0, r_min=3), wts),
                          prompt, gen)
    assert hi3.exit_depths == [3] * (gen - 1)
    lo = decode_sequence(OracleModel(dataclasses.replace(shape, gate_bias=-100.0), wts), prompt, gen,
                         keep_logits=gen)
    fx = decode_sequence(OracleModel(shape, wts), prompt, gen, mode="fixed", keep_logits=gen)
    assert lo.exit_depths == [5] * (gen - 1)
    assert lo.tokens == fx.tokens
    for a, b in zip(lo.logits, fx.logits):
        np.testing.assert_array_equal(a, b)


def test_gate_threshold_is_strict_and_in_logit_space():
    shape = micro(r_max=4, gate_q=0.5)
    om = OracleModel(shape, make_weights(shape))
    assert om.theta == 0.0
    assert OracleModel(micro(gate_q=0.2), make_weights(shape)).theta == pytest.approx(math.log(0.25))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 10000), rng.normal(0, 1e-3, 1000),
                        # exact ties between two bf16 neighbours
                        (np.arange(1, 200) * 2 + 1).astype(np.float64) * 2.0 ** -8 + 1.0])
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(_bf16(x32.astype(np.float64)).astype(np.float32), ref)


def test_rope_is_relative():
    shape = micro()
    om = OracleModel(shape, make_weights(shape))
    rng = np.random.default_rng(1)
    q = rng.normal(size=(1, shape.n_heads, shape.head_dim))
    k = rng.normal(size=(1, shape.n_heads, shape.head_dim))
    s1 = np.einsum("nhk,nhk->nh", om.rope(q, [9]), om.rope(k, [4]))
    s2 = np.einsum("nhk,nhk->nh", om.rope(q, [105]), om.rope(k, [100]))
    np.testing.assert_allclose(s1, s2, atol=1e-9)
    np.testing.assert_allclose(np.linalg.norm(om.rope(q, [77])), np.linalg.norm(q), atol=1e-12)


@pytest.mark.parametrize("variant", ["looped", "huginn_like"])
def test_decode_flops_match_closed_form(variant):
    if variant == "looped":
        shape = micro(r_max=4)
    else:
        shape = micro(r_max=4, n_prelude=1, n_core=1, n_coda=1, has_adapter=True)
    wts = make_weights(shape)
    prompt = prompt_for(shape, 5)
    gen = 4
    depths = np.array([2, 4, 3], dtype=np.int8)
    om = OracleModel(shape, wts)
    # prefill alone
    decode_sequence(om, prompt, 1)
    pre = dataclasses.asdict(om.flops)
    om2 = OracleModel(shape, wts)
    decode_sequence(om2, prompt, gen, force_exit=depths)
    got = {k: v - pre[k] for k, v in dataclasses.asdict(om2.flops).items()}
    d, f, V = shape.d_model, shape.ffn, shape.vocab
    layer = 2 * (4 * d * d + 3 * d * f)           # qkv, o, gate/up, down
    adapter = 2 * (2 * d * d) if shape.has_adapter else 0
    P = len(prompt)
    ctx = [P + t for t in range(1, gen)]           # keys seen by decode forward t
    assert got["core"] == sum(int(e) * (shape.n_core * layer + adapter) for e in depths)
    assert got["prelude"] == (gen - 1) * shape.n_prelude * layer
    assert got["coda"] == (gen - 1) * (shape.n_coda * layer + 2 * V * d)
    n_attn = shape.n_prelude + shape.n_coda
    assert got["attention"] == sum(4 * d * L * (int(e) * shape.n_core + n_attn)
                                   for e, L in zip(depths, ctx))


def test_exit_gaps_never_written():
    shape = micro(r_max=4)
    wts = make_weights(shape)
    prompt = prompt_for(shape, 5)
    depths = np.array([2, 3, 4, 2], dtype=np.int8)
    tr = decode_sequence(OracleModel(shape, wts), prompt, 5, force_exit=depths, keep_kv=True)
    K = tr.kv.K
    om = OracleModel(shape, wts)
    P = len(prompt)
    for l in range(shape.n_core):
        for dpt in range(1, shape.r_max + 1):
            sl = om.slot_core(l, dpt)
            assert np.all(np.isfinite(K[sl, :P]))
            for t, e in enumerate(depths, start=1):
                written = np.all(np.isfinite(K[sl, P + t - 1]))
                assert written == (dpt <= e)


# ---------------------------------------------------------------------------
# convergence exit (App. E.2)
# ---------------------------------------------------------------------------

def conv_micro(variant, **kw):
    base = dict(r_max=6, r_min=3, gate_kind="convergence")
    if variant == "huginn_like":
        base.update(n_prelude=1, n_core=1, n_coda=1, has_adapter=True)
    base.update(kw)
    return micro(**base)


def test_convergence_statistic_closed_form():
    om = OracleModel(conv_micro("looped"), make_weights(conv_micro("looped")))
    c = om.convergence(np.array([[3.0, 4.0], [3.0, 4.0], [0.0, 0.0]]),
                       np.array([[0.0, 0.0], [3.0, 0.0], [1.0, 1.0]]))
    assert c[0] == 1.0 and c[1] == pytest.approx(0.8, abs=1e-7) and np.isinf(c[2])
    assert om.gate_fires(om.theta - 1e-3) and not om.gate_fires(om.theta)


@pytest.mark.parametrize("variant", ["looped", "huginn_like"])
def test_convergence_gate_matches_brute_force(variant):
    shape0 = conv_micro(variant, conv_tau=0.0)
    wts = make_weights(shape0)
    prompt = prompt_for(shape0, 5, seed=17)
    gen = 7
    # Statistics of a run that never exits fix a threshold inside their range.
    free = decode_sequence(OracleModel(shape0, wts), prompt, gen)
    deciding = np.array([z for zs in free.gate_logits for z in zs[shape0.r_min - 2:shape0.r_max - 2]])
    tau = float(np.median(deciding))
    shape = dataclasses.replace(shape0, conv_tau=tau)
    tr = decode_sequence(OracleModel(shape, wts), prompt, gen, keep_logits=gen)
    assert len(set(tr.exit_depths)) >= 2, tr.exit_depths

    P = len(prompt)
    bf = None

    def c_of(i, d):
        a, b = bf.state(i, d), bf.state(i, d - 1)
        return float(np.linalg.norm(a - b) / np.linalg.norm(a))

    def exit_of(t):
        # Lookahead: a statistic below tau after step d (r_min-1 <= d <= r_max-2)
        # makes the token run step d+1 and leave.
        i = P + t - 1
        for d in range(shape.r_min - 1, shape.r_max - 1):
            if c_of(i, d) < tau:
                return d + 1
        return shape.r_max

    bf = BruteForceLM(shape, wts, prompt, gen, exit_of)
    toks, lg = bf.run()
    assert tr.exit_depths == [exit_of(t) for t in range(1, gen)]
    assert tr.tokens == toks
    for t in range(1, gen):
        i = P + t - 1
        want = [c_of(i, d) for d in range(1, tr.exit_depths[t - 1])]
        np.testing.assert_allclose(tr.gate_logits[t - 1], want, rtol=1e-5, atol=0)
        margin = min(abs(c - tau) for c in want[shape.r_min - 2:])
        assert margin > 1e-5 or tr.exit_depths[t - 1] == shape.r_min  # no decision within rounding of tau
    for t in range(gen):
        np.testing.assert_allclose(tr.logits[t], lg[t], atol=2e-5, rtol=0)


def test_convergence_gate_extremes():
    shape = conv_micro("huginn_like")
    wts = make_weights(shape)
    prompt = prompt_for(shape, 6)
    gen = 6
    hi = decode_sequence(OracleModel(dataclasses.replace(shape, conv_tau=10.0), wts), prompt, gen)
    assert hi.exit_depths == [3] * (gen - 1)
    lo = decode_sequence(OracleModel(dataclasses.replace(shape, conv_tau=0.0), wts), prompt, gen,
                         keep_logits=gen)
    fx = decode_sequence(OracleModel(shape, wts), prompt, gen, mode="fixed", keep_logits=gen)
    assert lo.exit_depths == [shape.r_max] * (gen - 1)
    assert lo.tokens == fx.tokens
    for a, b in zip(lo.logits, fx.logits):
        np.testing.assert_array_equal(a, b)
    # s_0 = 0 with the adapter: the first statistic is exactly 1.
    assert all(zs[0] == 1.0 for zs in lo.gate_logits)


# ---------------------------------------------------------------------------
# probe gate (§4.3): closed form, and logits from the brute force's loop states
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("eps,want", [(0.0, 0.1 + math.sqrt(2.0)), (12.5, 1.1)])
def test_probe_logit_closed_form(eps, want):
    """h = [3, 4] has mean square 12.5.  With w = [1, 0.5], b = 0.1 and eps = 0
    the unit-RMS state is [3, 4] / sqrt(12.5), so z = 0.1 + 5 / sqrt(12.5) =
    0.1 + sqrt(2); with eps = 12.5 inside the root the divisor is 5 and
    z = 0.1 + 1.  Dropping the normalisation (z = 5.1), adding eps outside the
    root, or a gain other than one gives other values."""
    shape = micro(d_model=2, n_heads=1, head_dim=2, rms_eps=eps, gate_bias=0.1)
    om = OracleModel(shape, {"gate_w": np.array([1.0, 0.5], dtype=np.float32)})
    z = om.gate_logit(np.array([[3.0, 4.0]]))
    assert z.shape == (1,)
    assert z[0] == pytest.approx(want, abs=1e-6)


@pytest.mark.parametrize("variant", ["looped", "huginn_like"])
def test_probe_gate_matches_brute_force(variant):
    """The oracle's gate logits and exit depths equal the probe applied to the
    brute force's cache-free loop states (the state after step d), with the
    lookahead rule applied to them: a logit above logit(q) = 0 after step d,
    r_min - 1 <= d <= r_max - 2, makes the token run step d + 1 and leave."""
    kw = dict(r_max=5)
    if variant == "huginn_like":
        kw.update(n_prelude=1, n_core=1, n_coda=1, has_adapter=True)
    shape0 = micro(**kw)
    wts = make_weights(shape0)
    prompt = prompt_for(shape0, 5, seed=29)
    gen = 7
    # Logits of a run that never exits place the threshold inside their range.
    free = decode_sequence(OracleModel(shape0, wts), prompt, gen, mode="fixed")
    deciding = [z for zs in free.gate_logits for z in zs[shape0.r_min - 2:shape0.r_max - 2]]
    shape = dataclasses.replace(shape0, gate_bias=-float(np.median(deciding)))
    tr = decode_sequence(OracleModel(shape, wts), prompt, gen, keep_logits=gen)
    assert len(set(tr.exit_depths)) >= 3, tr.exit_depths

    P = len(prompt)
    bf = None

    @functools.lru_cache(maxsize=None)
    def exit_of(t):
        i = P + t - 1
        for d in range(shape.r_min - 1, shape.r_max - 1):
            if bf.probe_logit(i, d) > 0.0:
                return d + 1
        return shape.r_max

    bf = BruteForceLM(shape, wts, prompt, gen, exit_of)
    toks, lg = bf.run()
    assert tr.exit_depths == [exit_of(t) for t in range(1, gen)]
    assert tr.tokens == toks
    for t in range(1, gen):
        i = P + t - 1
        want = [bf.probe_logit(i, d) for d in range(1, tr.exit_depths[t - 1])]
        np.testing.assert_allclose(tr.gate_logits[t - 1], want, rtol=0, atol=2e-5)
        # no decision within rounding distance of the threshold
        assert min(abs(z) for z in want[shape.r_min - 2:]) > 1e-4
    for t in range(gen):
        np.testing.assert_allclose(tr.logits[t], lg[t], atol=2e-5, rtol=0)


def test_probe_gate_reads_the_state_after_the_step():
    """Sensitivity of the brute-force pin: the probe on the state that entered
    step d (before it) gives other logits than the oracle records for step d."""
    shape = micro(r_max=4)
    wts = make_weights(shape)
    prompt = prompt_for(shape, 5, seed=29)
    depths = np.array([4, 4, 4], dtype=np.int8)
    tr = decode_sequence(OracleModel(shape, wts), prompt, 4, force_exit=depths)
    bf = BruteForceLM(shape, wts, prompt, 4, lambda t: int(depths[t - 1]))
    i = len(prompt)
    after = [bf.probe_logit(i, d) for d in range(1, 4)]
    state, bf.state = bf.state, lambda j, d: state(j, d - 1)
    before = [bf.probe_logit(i, d) for d in range(1, 4)]
    np.testing.assert_allclose(tr.gate_logits[0], after, atol=2e-5, rtol=0)
    assert np.max(np.abs(np.array(tr.gate_logits[0]) - np.array(before))) > 1e-2


# ---------------------------------------------------------------------------
# bf16 storage points (Table 1, bfloat16): an independent torch forward
# ---------------------------------------------------------------------------

# Values the method stores in bf16 (the rest stays float32): the normalised
# inputs of the QKV, gate/up and LM-head products, q, k and v after RoPE (so
# the KV cache), the attention output, the SwiGLU product and the adapter input.
BF16_POINTS = ("attn_norm", "q", "k", "v", "attn_out", "mlp_norm", "swiglu", "adapter_in", "head_in")


def torch_bf16_fixed_depth_logits(shape, weights, tokens, skip=None):
    """Cache-free causal forward of the whole sequence at fixed depth (every
    token runs r_max loop steps, so with a depth-indexed cache this is the
    unrolled transformer).  Arithmetic in float64 through torch's own ops;
    every result stored as float32, and cast through torch.bfloat16 from
    float32 at the points of BF16_POINTS except `skip` (to show that each point
    matters).  Returns float32-valued logits for every position."""
    w = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(torch.float64)
         for k, v in weights.items()}
    T = len(tokens)
    d, H, hd = shape.d_model, shape.n_heads, shape.head_dim

    def f32(t):
        return t.to(torch.float32).to(torch.float64)

    def bf(t, point):
        return f32(t) if point == skip else t.to(torch.float32).to(torch.bfloat16).to(torch.float64)

    inv = shape.rope_theta ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rope(t):  # [H, T, hd]
        a, b = t[..., : hd // 2], t[..., hd // 2:]
        return torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1)

    def norm(t, g, point):
        return bf(F.rms_norm(t, (d,), g, eps=shape.rms_eps), point)

    def block(p, x):
        u = norm(x, w[p + "attn_norm"], "attn_norm")
        q, k, v = f32(F.linear(u, w[p + "wqkv"])).split(d, dim=-1)
        q = bf(rope(q.view(T, H, hd).transpose(0, 1)), "q")
        k = bf(rope(k.view(T, H, hd).transpose(0, 1)), "k")
        v = bf(v.view(T, H, hd).transpose(0, 1), "v")
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        o = bf(o.transpose(0, 1).reshape(T, d), "attn_out")
        x = f32(x + F.linear(o, w[p + "wo"]))
        u = norm(x, w[p + "mlp_norm"], "mlp_norm")
        mid = bf(f32(F.silu(f32(F.linear(u, w[p + "wg"]))) * f32(F.linear(u, w[p + "wu"]))), "swiglu")
        return f32(x + F.linear(mid, w[p + "wd"]))

    x = w["embed"][torch.as_tensor(tokens, dtype=torch.long)]
    for i in range(shape.n_prelude):
        x = block(f"prelude.{i}.", x)
    e = x
    s = torch.zeros_like(e) if shape.has_adapter else e
    for _ in range(shape.r_max):
        if shape.has_adapter:
            s = f32(F.linear(bf(torch.cat([e, s], dim=-1), "adapter_in"), w["adapter"]))
        for l in range(shape.n_core):
            s = block(f"core.{l}.", s)
    y = s
    for j in range(shape.n_coda):
        y = block(f"coda.{j}.", y)
    return f32(F.linear(norm(y, w["final_norm"], "head_in"), w["lm_head"])).numpy()


def _bf16_case(variant, r_max):
    kw = dict(dtype="bf16", r_max=r_max, r_min=min(2, r_max))
    if variant == "huginn_like":
        kw.update(n_prelude=1, n_core=1, n_coda=1, has_adapter=True)
    shape = micro(**kw)
    wts = make_weights(shape)
    prompt = prompt_for(shape, 8, seed=31)
    gen = 5
    tr = decode_sequence(OracleModel(shape, wts), prompt, gen, mode="fixed", keep_logits=gen)
    seq = np.concatenate([prompt, np.array(tr.tokens[:-1], dtype=np.int32)])
    return shape, wts, seq, tr, len(prompt) - 1


@pytest.mark.parametrize("r_max", [1, 3])
@pytest.mark.parametrize("variant", ["looped", "huginn_like"])
def test_bf16_storage_points_match_torch(variant, r_max):
    shape, wts, seq, tr, p0 = _bf16_case(variant, r_max)
    ref = torch_bf16_fixed_depth_logits(shape, wts, seq)
    for t in range(len(tr.tokens)):
        np.testing.assert_allclose(tr.logits[t], ref[p0 + t], atol=1e-5, rtol=0)


@pytest.mark.parametrize("variant", ["looped", "huginn_like"])
def test_each_bf16_storage_point_matters(variant):
    """Dropping any one rounding point moves the logits far outside the
    tolerance above, so an oracle that missed (or added) one would fail it."""
    shape, wts, seq, tr, p0 = _bf16_case(variant, 3)
    got = np.array(tr.logits)
    for point in BF16_POINTS:
        if point == "adapter_in" and not shape.has_adapter:
            continue
        ref = torch_bf16_fixed_depth_logits(shape, wts, seq, skip=point)[p0:p0 + len(got)]
        assert np.max(np.abs(got - ref)) > 1e-4, point
