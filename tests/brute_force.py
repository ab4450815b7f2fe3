"""Cache-free recomputation of a looped LM, for pinning the oracle on tiny inputs.

Written independently of ``oracle/``: there is no KV store here.  Every
hidden state is a function of (position, loop step, layer) evaluated by
recursion on the definition of §2 and §4.2 of "Depth-adaptive Inference of
Looped Language Models via Continuous Depth Batching": at loop step d, position
i attends to each earlier position j through the keys and values position j
produced at step min(d, e_j) of the same core layer (its last written state),
and to itself at step d.  Results are memoised per (position, step, layer) so
tiny cases finish quickly; memoisation does not change what is computed.

All arithmetic is float64 without intermediate rounding (compare against the
oracle only for fp32 models, where the oracle's float32 storage is the only
difference).
"""

from __future__ import annotations

import functools
import math

import numpy as np


def _w64(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


class BruteForceLM:
    def __init__(self, shape, weights, prompt, gen_len, exit_depth_of_token):
        """exit_depth_of_token(t) -> exit depth of decode forward t (1-based).

        shape.kv_slots selects the cache layout of App. E.1 (0 or r_max:
        depth-indexed; 1: single slot; 2: first-then-shared); see visible_step.
        """
        self.m = shape
        self.w = {k: _w64(v) for k, v in weights.items()}
        self.P = len(prompt)
        self.gen_len = gen_len
        self.toks = {i: int(t) for i, t in enumerate(prompt)}
        self.exit_of = exit_depth_of_token
        hd = shape.head_dim
        self.freq = 1.0 / (shape.rope_theta ** (np.arange(0, hd, 2) / hd))

    # -- pieces --
    def _norm(self, x, g):
        return x / math.sqrt(float(np.dot(x, x)) / len(x) + self.m.rms_eps) * g

    def _rot(self, v, i):
        m = self.m
        out = np.empty_like(v)
        half = m.head_dim // 2
        for h in range(m.n_heads):
            seg = v[h * m.head_dim:(h + 1) * m.head_dim]
            a, b = seg[:half], seg[half:]
            c, s = np.cos(i * self.freq), np.sin(i * self.freq)
            out[h * m.head_dim:(h + 1) * m.head_dim] = np.concatenate([a * c - b * s, a * s + b * c])
        return out

    def _kv(self, prefix, x, i):
        d = self.m.d_model
        u = self._norm(x, self.w[prefix + "attn_norm"])
        W = self.w[prefix + "wqkv"]
        return self._rot(W[d:2 * d] @ u, i), W[2 * d:] @ u

    def _layer(self, prefix, x, i, kv_of):
        m, d = self.m, self.m.d_model
        u = self._norm(x, self.w[prefix + "attn_norm"])
        q = self._rot(self.w[prefix + "wqkv"][:d] @ u, i)
        ks, vs = [], []
        for j in range(i + 1):
            k, v = kv_of(j)
            ks.append(k)
            vs.append(v)
        ks, vs = np.array(ks), np.array(vs)
        o = np.empty(d)
        for h in range(m.n_heads):
            sl = slice(h * m.head_dim, (h + 1) * m.head_dim)
            sc = ks[:, sl] @ q[sl] / math.sqrt(m.head_dim)
            p = np.exp(sc - sc.max())
            o[sl] = (p / p.sum()) @ vs[:, sl]
        x = x + self.w[prefix + "wo"] @ o
        u = self._norm(x, self.w[prefix + "mlp_norm"])
        g = self.w[prefix + "wg"] @ u
        up = self.w[prefix + "wu"] @ u
        return x + self.w[prefix + "wd"] @ (g / (1.0 + np.exp(-g)) * up)

    # -- definitions by recursion --
    def exit_depth(self, i):
        if i < self.P:
            return self.m.r_max
        return self.exit_of(i - self.P + 1)

    def token(self, i):
        if i not in self.toks:
            self.toks[i] = int(np.argmax(self.logits(i - 1)))
        return self.toks[i]

    @functools.lru_cache(maxsize=None)
    def prelude_in(self, i, l):
        if l == 0:
            return self.w["embed"][self.token(i)].copy()
        pre = f"prelude.{l - 1}."
        return self._layer(pre, self.prelude_in(i, l - 1), i,
                           lambda j: self._kv(pre, self.prelude_in(j, l - 1), j))

    def emb(self, i):
        return self.prelude_in(i, self.m.n_prelude)

    @functools.lru_cache(maxsize=None)
    def state(self, i, d):
        """s_i^d: the core state of position i after d loop steps."""
        m = self.m
        if d == 0:
            return np.zeros(m.d_model) if m.has_adapter else self.emb(i)
        return self.core_in(i, d, m.n_core)

    @functools.lru_cache(maxsize=None)
    def core_in(self, i, d, l):
        """Input of core layer l at loop step d for position i (l = n_core: output)."""
        m = self.m
        if l == 0:
            s = self.state(i, d - 1)
            if m.has_adapter:
                return self.w["adapter"] @ np.concatenate([self.emb(i), s])
            return s
        pre = f"core.{l - 1}."

        def kv_of(j):
            return self._kv(pre, self.core_in(j, self.visible_step(i, j, d), l - 1), j)

        return self._layer(pre, self.core_in(i, d, l - 1), i, kv_of)

    def visible_step(self, i, j, d):
        """Loop step of key j whose K/V position i sees at its loop step d.

        Depth-indexed cache: step d of j, or j's last step e_j if it left
        earlier (the depth clamp).  Shared layouts keep fewer slots, so a key
        shows whatever step last wrote the slot step d reads: with s slots,
        steps below s have private slots (step d itself); the last slot holds
        the key's latest step, which is d while the prompt runs its loop steps
        together in prefill and e_j once the key's token has finished.
        """
        m = self.m
        if j == i:
            return d
        s = m.r_max if m.kv_slots <= 0 else min(m.kv_slots, m.r_max)
        if s == m.r_max:
            return min(d, self.exit_depth(j))
        if d < s:
            return d
        return d if i < self.P else self.exit_depth(j)

    def probe_logit(self, i, d):
        """Linear exit probe on the state after loop step d: the state scaled to
        unit root-mean-square (eps inside the root, unit gain), dotted with the
        gate vector, plus the bias."""
        s = self.state(i, d)
        rms = math.sqrt(sum(float(x) * float(x) for x in s) / len(s) + self.m.rms_eps)
        w = self.w["gate_w"]
        return sum(float(w[c]) * float(s[c]) for c in range(len(s))) / rms + self.m.gate_bias

    @functools.lru_cache(maxsize=None)
    def coda_in(self, i, l):
        if l == 0:
            return self.state(i, self.exit_depth(i))
        pre = f"coda.{l - 1}."
        return self._layer(pre, self.coda_in(i, l - 1), i,
                           lambda j: self._kv(pre, self.coda_in(j, l - 1), j))

    @functools.lru_cache(maxsize=None)
    def logits(self, i):
        h = self.coda_in(i, self.m.n_coda)
        return self.w["lm_head"] @ self._norm(h, self.w["final_norm"])

    def run(self):
        """(tokens[gen_len], logits per generated token)."""
        toks, lg = [], []
        for t in range(self.gen_len):
            i = self.P + t - 1               # position whose forward yields token t
            lg.append(self.logits(i))
            toks.append(self.token(i + 1))
        return toks, lg
