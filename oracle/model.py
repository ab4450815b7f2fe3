"""Plain CPU oracle of a depth-adaptive looped LM decoded one sequence at a time.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library.

Source: "Depth-adaptive Inference of Looped Language Models via Continuous
Depth Batching" (arxiv 2608.09444v2).  Continuous depth batching does not
change the model's predictions or exit decisions (§3, last paragraph), so the
result of any batched schedule is, by definition, the result of decoding each
sequence alone, token by token and loop by loop.  That definition is what this
module computes:

* §2: prelude once, shared recurrent core r_t <= r_max times, coda once.
* §4.2: depth-indexed KV cache, one slot per (core layer, loop step); a token
  that exits at e leaves depths e+1..r_max unwritten.  A later token at depth d
  reads earlier token j at depth min(d, e_j) (the last state j wrote), so a gap
  is never read.
* §4.3: lookahead gate; the gate after loop step d decides whether the token
  takes part in step d+2, so a positive gate at d means the token runs d+1 and
  exits; the minimum exit depth is r_min = 2 (§7 "Designing exit gates").
* Appendix A.1: prefill runs every prompt token at full depth; only the last
  prompt position produces a token (A.5 "Attention and output projection").

Arithmetic: every reduction (matrix products, norms, softmax, dot products) is
evaluated in float64 and the result stored as float32.  For bf16 models the
values the method stores in bf16 (A.2 Table 1, numerical precision bfloat16)
are rounded from that float32 value to bf16 with round-to-nearest-even at these
points only: the normalised GEMM inputs, q/k/v after RoPE (so the KV cache),
the attention output, the SwiGLU product and the adapter input.  The residual
stream, softmax, norms, logits and the gate logit stay float32.

Readings where the pages are silent (each also listed in the design notes):
pre-norm RMSNorm blocks (eps 1e-6, gains 1, no biases), rotate-half RoPE with
theta 1e4 at the token's position at every depth, SwiGLU MLP, final RMSNorm
before an untied LM head, greedy argmax with ties to the lowest index, exit
gate z = w_g . rmsnorm(h) + b_g compared with logit(q) (a token exits when
sigmoid(z) > q; z == logit(q) does not exit).  Huginn-shaped models enter every
loop step through x = A [e; s_{d-1}] with s_0 = 0 and e the prelude output.

Convergence exit (App. E.2, Huginn's training-free criterion): after loop step
d the statistic is c_d = ||s_d - s_{d-1}||_2 / ||s_d||_2, with s_{d-1} the
state that entered step d (s_0 = 0 with an adapter, else the prelude output),
and the token exits when c_d < tau (c_d == tau does not exit).  It goes through
the same lookahead as the linear gate, so with r_min = 3 the first deciding
comparison is c_2 (App. E.2: minimum loop count 3 for this criterion).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


# ---------------------------------------------------------------------------
# rounding of stored values
# ---------------------------------------------------------------------------

def _f32(x):
    """Store as float32 (returned as float64 holding the float32 value)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _bf16(x):
    """Store as bfloat16: float32 value rounded to nearest even in the top 16 bits."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _decode_weight(a: np.ndarray) -> np.ndarray:
    """Weights arrive as float32 (fp32 models) or uint16 bf16 bit patterns."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ---------------------------------------------------------------------------
# model
# ---------------------------------------------------------------------------

@dataclass
class FlopCount:
    """Multiply-add FLOPs (2 per MAC) the oracle actually executed, by stage."""
    prelude: float = 0.0
    core: float = 0.0
    coda: float = 0.0
    attention: float = 0.0

    def add(self, stage: str, n: float):
        setattr(self, stage, getattr(self, stage) + n)


class OracleModel:
    """Weights of one looped LM held in float64 plus the per-op definitions."""

    def __init__(self, shape, weights: dict):
        self.m = shape
        self.bf16 = shape.dtype == "bf16"
        self.store = _bf16 if self.bf16 else _f32
        self.w = {k: _decode_weight(v) for k, v in weights.items()}
        self.flops = FlopCount()
        m = shape
        self.convergence_gate = getattr(m, "gate_kind", "probe") == "convergence"
        self.theta = m.conv_tau if self.convergence_gate else math.log(m.gate_q / (1.0 - m.gate_q))
        half = m.head_dim // 2
        # RoPE inverse frequencies theta^(-2i/hd), i < hd/2.
        self.inv_freq = m.rope_theta ** (-2.0 * np.arange(half, dtype=np.float64) / m.head_dim)

    # -- cache slots (§4.2; App. E.1: l0 + lr * s entries per token) --
    # Core layer l keeps s slots per position.  Loop step d writes and reads
    # slot min(d, s): s = r_max is the depth-indexed cache (one slot per step),
    # s = 1 the single-slot shared cache (every step overwrites the slot), s = 2
    # first-then-shared (step 1 private, steps >= 2 share the second slot).
    def slot_prelude(self, i: int) -> int:
        return i

    def slot_core(self, l: int, depth):
        s = self.m.slots_per_core_layer
        return self.m.n_prelude + l * s + (np.minimum(depth, s) - 1)

    def slot_coda(self, j: int) -> int:
        return self.m.n_prelude + self.m.n_core * self.m.slots_per_core_layer + j

    # -- elementary ops --
    def rmsnorm(self, x, g):
        ms = np.mean(x * x, axis=-1, keepdims=True)
        return _f32(x / np.sqrt(ms + self.m.rms_eps) * g)

    def linear(self, x, W, stage):
        self.flops.add(stage, 2.0 * x.shape[0] * W.shape[0] * W.shape[1])
        return x @ W.T

    def rope(self, x, pos):
        """Rotate-half RoPE on [n, H, hd] at integer positions pos[n]."""
        half = self.m.head_dim // 2
        ang = np.asarray(pos, dtype=np.float64)[:, None] * self.inv_freq[None, :]
        c = np.cos(ang)[:, None, :]
        s = np.sin(ang)[:, None, :]
        a, b = x[..., :half], x[..., half:]
        return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)

    def attend(self, q, keys, vals, lens):
        """Row i: softmax(q_i k^T / sqrt(hd)) v over keys[:lens[i]], per head.

        q [n, H, hd]; keys, vals [L, H, hd].
        """
        m = self.m
        n = q.shape[0]
        self.flops.add("attention", 4.0 * float(np.sum(lens)) * m.d_model)
        # optimize=True lets numpy evaluate the float64 contractions with BLAS
        # (same sums, faster for long prompts).
        sc = np.einsum("nhk,lhk->nhl", q, keys, optimize=True) / math.sqrt(m.head_dim)
        visible = np.arange(keys.shape[0])[None, :] < np.asarray(lens)[:, None]
        sc = np.where(visible[:, None, :], sc, -np.inf)
        sc = sc - sc.max(axis=-1, keepdims=True)
        p = np.exp(sc)
        p = p / p.sum(axis=-1, keepdims=True)
        return np.einsum("nhl,lhk->nhk", p, vals, optimize=True)

    def block(self, prefix: str, h, pos, kv, write_slot: int, key_slots, stage):
        """One pre-norm transformer block on rows h [n, d] at positions pos[n].

        The rows' K/V are stored in cache slot write_slot at their positions.
        Key position j is read from slot key_slots[j]; row i sees keys
        0..pos[i] (causal), its own included.
        """
        m = self.m
        n, d = h.shape
        H, hd = m.n_heads, m.head_dim
        w = self.w
        u = self.store(self.rmsnorm(h, w[prefix + "attn_norm"]))
        qkv = _f32(self.linear(u, w[prefix + "wqkv"], stage))
        q = self.store(self.rope(qkv[:, :d].reshape(n, H, hd), pos))
        k = self.store(self.rope(qkv[:, d:2 * d].reshape(n, H, hd), pos))
        v = self.store(qkv[:, 2 * d:].reshape(n, H, hd))
        kv.K[write_slot, pos] = k.reshape(n, d)
        kv.V[write_slot, pos] = v.reshape(n, d)
        L = len(key_slots)
        kpos = np.arange(L)
        keys = kv.K[key_slots, kpos].astype(np.float64).reshape(L, H, hd)
        vals = kv.V[key_slots, kpos].astype(np.float64).reshape(L, H, hd)
        o = self.attend(q, keys, vals, np.asarray(pos) + 1)
        o = self.store(_f32(o.reshape(n, d)))
        h = _f32(h + self.linear(o, w[prefix + "wo"], stage))
        u = self.store(self.rmsnorm(h, w[prefix + "mlp_norm"]))
        g = _f32(self.linear(u, w[prefix + "wg"], stage))
        up = _f32(self.linear(u, w[prefix + "wu"], stage))
        mid = self.store(_f32(g / (1.0 + np.exp(-g)) * up))
        return _f32(h + self.linear(mid, w[prefix + "wd"], stage))

    def embed(self, tokens):
        return _f32(self.w["embed"][np.asarray(tokens)])

    def adapter(self, e, s):
        """Huginn-shaped loop input x = A [e; s]: the concatenation of the prelude output and the loop state (2d -> d)."""
        x = self.store(np.concatenate([e, s], axis=-1))
        return _f32(self.linear(x, self.w["adapter"], "core"))

    def gate_logit(self, h):
        """z = w_g . rmsnorm(h) + b_g with unit gain, float32 result."""
        m = self.m
        ms = np.mean(h * h, axis=-1, keepdims=True)
        hn = h / np.sqrt(ms + m.rms_eps)
        return _f32(hn @ self.w["gate_w"] + m.gate_bias)

    def convergence(self, s, s_prev):
        """c = ||s - s_prev||_2 / ||s||_2 per row, float32 result (inf when s = 0)."""
        num = np.sqrt(np.sum((s - s_prev) ** 2, axis=-1))
        den = np.sqrt(np.sum(s * s, axis=-1))
        with np.errstate(divide="ignore", invalid="ignore"):
            return _f32(np.where(den > 0, num / np.where(den > 0, den, 1.0), np.inf))

    def gate_fires(self, z):
        """Exit decision of one gate value: z > logit(q) for the probe, c < tau for convergence."""
        return z < self.theta if self.convergence_gate else z > self.theta

    def logits(self, h):
        u = self.store(self.rmsnorm(h, self.w["final_norm"]))
        return _f32(self.linear(u, self.w["lm_head"], "coda"))


class SeqKV:
    """Logical KV store of one sequence: [slot][position][d], NaN where unwritten."""

    def __init__(self, model: OracleModel, n_pos: int):
        m = model.m
        self.K = np.full((m.n_kv_slots, n_pos, m.d_model), np.nan, dtype=np.float32)
        self.V = np.full((m.n_kv_slots, n_pos, m.d_model), np.nan, dtype=np.float32)


@dataclass
class SeqTrace:
    """Everything the oracle decided for one sequence."""
    tokens: list = field(default_factory=list)          # generated ids, token 0 from prefill
    exit_depths: list = field(default_factory=list)     # per decode forward (gen_len - 1)
    gate_logits: list = field(default_factory=list)     # per decode forward: z_1..z_{e-1} (c_d for convergence)
    near_gate: list = field(default_factory=list)       # per decode forward: |z_d - theta| < tol at a deciding d
    top2_gap: list = field(default_factory=list)        # per generated token
    logits: list = field(default_factory=list)          # per generated token (if kept)
    hidden: list = field(default_factory=list)          # coda input per generated token (if kept)
    kv: SeqKV | None = None


def decode_sequence(model: OracleModel, prompt, gen_len: int, mode: str = "adaptive",
                    force_exit=None, force_token=None, keep_logits: int = 0,
                    keep_kv: bool = False, near_tol: float = 1e-3) -> SeqTrace:
    """Decode one sequence alone (see iter_decode); returns the full trace."""
    tr = None
    for tr in iter_decode(model, prompt, gen_len, mode, force_exit, force_token, keep_logits,
                          keep_kv, near_tol):
        pass
    return tr


def iter_decode(model: OracleModel, prompt, gen_len: int, mode: str = "adaptive",
                force_exit=None, force_token=None, keep_logits: int = 0,
                keep_kv: bool = False, near_tol: float = 1e-3):
    """Decode one sequence alone, yielding the trace after each generated token.

    mode "adaptive" uses the lookahead gate (or force_exit); "fixed" runs every
    token at r_max loops (token-level continuous batching, §6.1).
    force_exit[t-1] (decode forward t = 1..gen_len-1): 0 = live gate, else the
    exit depth in [2, r_max].  force_token[t]: -1 = live argmax, else the id.
    keep_logits: number of leading generated tokens whose logits and coda
    input are recorded.
    """
    m = model.m
    w = model.w
    P = len(prompt)
    n_pos = P + gen_len - 1
    kv = SeqKV(model, max(n_pos, P))
    e = np.full(max(n_pos, P) + 1, m.r_max, dtype=np.int64)   # exit depth per position
    tr = SeqTrace()

    def emit(logits, t, hidden):
        order = np.argsort(-logits, kind="stable")
        tok = int(order[0])
        gap = float(logits[order[0]] - logits[order[1]]) if len(order) > 1 else float("inf")
        if force_token is not None and force_token[t] >= 0:
            tok = int(force_token[t])
        tr.tokens.append(tok)
        tr.top2_gap.append(gap)
        if t < keep_logits:
            tr.logits.append(logits.astype(np.float32))
            tr.hidden.append(hidden.astype(np.float32))
        return tok

    # ---- prefill: every prompt position at full depth (App. A.1) ----
    pos = np.arange(P)
    h = model.embed(prompt)
    for i in range(m.n_prelude):
        sl = model.slot_prelude(i)
        h = model.block(f"prelude.{i}.", h, pos, kv, sl, np.full(P, sl), "prelude")
    emb = h
    s = np.zeros_like(h) if m.has_adapter else h
    for d in range(1, m.r_max + 1):
        x = model.adapter(emb, s) if m.has_adapter else s
        for l in range(m.n_core):
            sl = model.slot_core(l, d)
            x = model.block(f"core.{l}.", x, pos, kv, sl, np.full(P, sl), "core")
        s = x
    y = s
    for j in range(m.n_coda):
        sl = model.slot_coda(j)
        y = model.block(f"coda.{j}.", y, pos, kv, sl, np.full(P, sl), "coda")
    last = y[-1:]
    tok = emit(model.logits(last)[0], 0, last[0])
    if keep_kv:
        tr.kv = kv
    yield tr

    # ---- decode: one token at a time, one loop step at a time ----
    for t in range(1, gen_len):
        p = P + t - 1
        e[p] = m.r_max                       # in flight: own slot read at current depth
        ppos = np.array([p])
        h = model.embed([tok])

        for i in range(m.n_prelude):
            sl = model.slot_prelude(i)
            h = model.block(f"prelude.{i}.", h, ppos, kv, sl, np.full(p + 1, sl), "prelude")
        emb = h
        s = np.zeros_like(h) if m.has_adapter else h
        forced = 0 if force_exit is None else int(force_exit[t - 1])
        exit_at = forced if (mode == "adaptive" and forced) else m.r_max
        decided = exit_at != m.r_max
        zs, near = [], False
        for d in range(1, m.r_max + 1):
            x = model.adapter(emb, s) if m.has_adapter else s
            # Depth clamp: key j is read at min(d, e_j); e_p = r_max in flight.
            # With a shared layout the slot of that step holds j's latest write.
            read_depth = np.minimum(d, e[:p + 1])
            s_prev = s
            for l in range(m.n_core):
                key_slots = model.slot_core(l, read_depth)
                x = model.block(f"core.{l}.", x, ppos, kv, model.slot_core(l, d),
                                key_slots, "core")
            s = x
            if d == exit_at:
                break
            if model.convergence_gate:
                z = float(model.convergence(s, s_prev)[0])
            else:
                z = float(model.gate_logit(s)[0])
            zs.append(z)
            deciding = m.r_min - 1 <= d <= m.r_max - 2
            if deciding and not decided and not (mode == "adaptive" and forced):
                if abs(z - model.theta) < near_tol:
                    near = True
                if mode == "adaptive" and not decided and model.gate_fires(z):
                    exit_at = d + 1
                    decided = True
        e[p] = d
        tr.exit_depths.append(int(d))
        tr.gate_logits.append(zs)
        tr.near_gate.append(near)
        y = s
        for j in range(m.n_coda):
            sl = model.slot_coda(j)
            y = model.block(f"coda.{j}.", y, ppos, kv, sl, np.full(p + 1, sl), "coda")
        tok = emit(model.logits(y)[0], t, y[0])
        yield tr


def _decode_one(args):
    shape, weights, req, mode, keep_logits = args
    model = OracleModel(shape, weights)
    return decode_sequence(model, req["prompt"], req["gen_len"], mode,
                           req.get("force_exit"), req.get("force_token"), keep_logits)


def decode_workload(model: OracleModel, requests, mode: str = "adaptive",
                    keep_logits: int = 0):
    """Decode each request alone, in order (the definition CDB must reproduce)."""
    return [decode_sequence(model, r["prompt"], r["gen_len"], mode,
                            r.get("force_exit"), r.get("force_token"), keep_logits)
            for r in requests]

