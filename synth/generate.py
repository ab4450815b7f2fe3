"""Counter-based seeded generators for weights and workloads.

Every random value is a pure function of (seed, stream, index) through the
splitmix64 output function (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; constants as in S. Vigna's
public-domain splitmix64.c).  Normals use the Box–Muller transform on the two
32-bit halves of one 64-bit draw.  Because values depend only on the index,
large tensors are generated in parallel chunks with identical results.

Weights of bf16 models are returned as uint16 bit patterns (round to nearest
even from the fp32 draw, once, here); fp32 models get float32 arrays.  Norm
gains are ones.  Nothing in this module evaluates the looped model.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import ModelShape, Workload

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_at(key: int, idx: np.ndarray) -> np.ndarray:
    """The idx-th output (0-based) of the splitmix64 sequence whose state starts at key."""
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx.astype(np.uint64) + np.uint64(1)) * _GAMMA
        return _mix(z)


def _stream_key(seed: int, stream: int) -> int:
    with np.errstate(over="ignore"):
        x = np.array([(seed << 32) ^ stream], dtype=np.uint64)
        return int(_mix(x + _GAMMA)[0])


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _bf16_bits(x32: np.ndarray) -> np.ndarray:
    u = x32.view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _normal_chunk(key: int, lo: int, hi: int, std: float, bf16: bool):
    idx = np.arange(lo, hi, dtype=np.uint64)
    z = splitmix64_at(key, idx)
    u1 = ((z >> np.uint64(32)).astype(np.float64) + 1.0) * (1.0 / 4294967296.0)
    u2 = (z & np.uint64(0xFFFFFFFF)).astype(np.float64) * (1.0 / 4294967296.0)
    n = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    x32 = (n * std).astype(np.float32)
    return _bf16_bits(x32) if bf16 else x32


def normal_tensor(seed: int, stream: int, shape, std: float, bf16: bool) -> np.ndarray:
    """N(0, std^2) tensor; uint16 bf16 bit patterns if bf16 else float32."""
    n = int(np.prod(shape))
    key = _stream_key(seed, stream)
    out = np.empty(n, dtype=np.uint16 if bf16 else np.float32)
    bounds = [(lo, min(n, lo + _CHUNK)) for lo in range(0, n, _CHUNK)]

    def work(b):
        out[b[0]:b[1]] = _normal_chunk(key, b[0], b[1], std, bf16)

    if len(bounds) > 1:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, bounds))
    elif bounds:
        work(bounds[0])
    return out.reshape(shape)


def _ones(shape, bf16: bool) -> np.ndarray:
    if bf16:
        return np.full(shape, 0x3F80, dtype=np.uint16)
    return np.ones(shape, dtype=np.float32)


def weight_names(m: ModelShape):
    """(name, shape, kind) in generation order; kind is 'normal' or 'ones'."""
    d, f, V = m.d_model, m.ffn, m.vocab
    names = [("embed", (V, d), "normal"), ("lm_head", (V, d), "normal"),
             ("final_norm", (d,), "ones"), ("gate_w", (d,), "normal")]
    if m.has_adapter:
        names.append(("adapter", (d, 2 * d), "normal"))
    for kind, count in (("prelude", m.n_prelude), ("core", m.n_core),
                        ("coda", m.n_coda)):
        for i in range(count):
            p = f"{kind}.{i}."
            names += [(p + "attn_norm", (d,), "ones"),
                      (p + "wqkv", (3 * d, d), "normal"),
                      (p + "wo", (d, d), "normal"),
                      (p + "mlp_norm", (d,), "ones"),
                      (p + "wg", (f, d), "normal"),
                      (p + "wu", (f, d), "normal"),
                      (p + "wd", (d, f), "normal")]
    return names


def make_weights(m: ModelShape) -> dict:
    """All weights of model m, keyed by name (see weight_names)."""
    bf16 = m.dtype == "bf16"
    out = {}
    for stream, (name, shape, kind) in enumerate(weight_names(m)):
        if kind == "ones":
            out[name] = _ones(shape, bf16)
        else:
            out[name] = normal_tensor(m.weight_seed, stream, shape, m.init_std, bf16)
    return out


def _uniform_ints(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform on [lo, hi] (multiply-shift on the high 32 bits)."""
    z = splitmix64_at(_stream_key(seed, stream), np.arange(n, dtype=np.uint64))
    span = np.uint64(hi - lo + 1)
    return (((z >> np.uint64(32)) * span) >> np.uint64(32)).astype(np.int64) + lo


def _uniform01(seed: int, stream: int, n: int) -> np.ndarray:
    z = splitmix64_at(_stream_key(seed, stream), np.arange(n, dtype=np.uint64))
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def make_lengths(w: Workload):
    """(prompt_len[n], gen_len[n]) uniform on the workload's inclusive ranges."""
    pl = _uniform_ints(w.length_seed, 0, w.n_seqs, w.prompt_lo, w.prompt_hi)
    gl = _uniform_ints(w.length_seed, 1, w.n_seqs, w.gen_lo, w.gen_hi)
    return pl, gl


def make_prompts(w: Workload, vocab: int, prompt_lens) -> list:
    """Token ids uniform over [0, vocab) for each sequence (one stream per sequence)."""
    return [_uniform_ints(w.prompt_seed, i, int(L), 0, vocab - 1).astype(np.int32)
            for i, L in enumerate(prompt_lens)]


def make_replay_depths(w: Workload, r_max: int, r_min: int, gen_lens) -> list:
    """Replayed exit depths per decode forward: truncated geometric on {r_min..r_max}.

    P(D = k) = p (1-p)^(k - r_min) for k < r_max, the remaining mass at r_max.
    One entry per adaptive decode forward (gen_len - 1 per sequence).
    """
    p = w.replay_p
    out = []
    for i, g in enumerate(gen_lens):
        u = _uniform01(w.replay_seed, i, max(0, int(g) - 1))
        k = np.floor(np.log1p(-u) / np.log1p(-p)).astype(np.int64) + r_min
        out.append(np.minimum(k, r_max).astype(np.int8))
    return out


def make_arrivals(seed: int, n: int, rate: float) -> np.ndarray:
    """Poisson-process arrival times (seconds) at the given rate."""
    u = _uniform01(seed, 0, n)
    gaps = -np.log1p(-u) / rate
    return np.cumsum(gaps)


def make_requests(w: Workload, vocab: int, r_max: int = 0, r_min: int = 2):
    """The workload's requests: list of dicts with prompt, gen_len, replay depths."""
    pl, gl = make_lengths(w)
    prompts = make_prompts(w, vocab, pl)
    depths = (make_replay_depths(w, r_max, r_min, gl) if w.replay_depths
              else [None] * w.n_seqs)
    return [dict(seq_id=i, prompt=prompts[i], gen_len=int(gl[i]),
                 replay=depths[i]) for i in range(w.n_seqs)]
