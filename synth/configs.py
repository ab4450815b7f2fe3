"""Model shapes and workload recipes of the five benchmark configurations.

Shapes follow the looped-LM split of "Depth-adaptive Inference of Looped
Language Models via Continuous Depth Batching" (arxiv 2608.09444, §2: prelude,
recurrent core run up to r_max times, coda) and the two model families of its
§6.1 (Ouro 1.4B, fully looped 0-24-0, r_max 4; Huginn 3.5B, 2-4-2).  Scheduler
parameters follow its Table 1 (W, M, S = max(1, floor(W/8)), 16-token KV
blocks) and §6.1 (minimum coda batch K = 1 for Ouro, floor(W/4) for Huginn).

The exit-gate bias of each model is a frozen input calibrated once on the CPU
oracle (``oracle/calibrate_gate.py`` writes ``gate_bias.json`` beside this
file); it is not computed here.
"""

from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass, replace

_HERE = os.path.dirname(os.path.abspath(__file__))


def _load_bias() -> dict:
    path = os.path.join(_HERE, "gate_bias.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return {}


_BIAS = _load_bias()


@dataclass(frozen=True)
class ModelShape:
    """One looped LM: prelude layers, a shared core looped r times, coda layers.

    dtype "fp32" stores weights, activations and KV in fp32; "bf16" stores
    weights and the KV cache in bf16 (Table 1, numerical precision bfloat16).
    The exit gate is a linear probe over the RMS-normalised core state; a token
    exits when sigmoid(z) > gate_q, compared in logit space.
    """

    name: str
    vocab: int
    d_model: int
    n_heads: int
    head_dim: int
    ffn: int
    n_prelude: int
    n_core: int
    n_coda: int
    r_max: int
    r_min: int
    has_adapter: bool
    dtype: str
    gate_q: float = 0.5
    gate_bias: float = 0.0
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    init_std: float = 0.02
    weight_seed: int = 0
    kv_slots: int = 0  # KV slots per recurrent layer s (App. E.1): 0 = r_max (depth-indexed), 1, 2 = shared
    # Exit policy: "probe" (the linear gate above) or "convergence" (Huginn's
    # training-free criterion, App. E.2: exit once the normalised L2 distance
    # between consecutive loop states falls below conv_tau).
    gate_kind: str = "probe"
    conv_tau: float = 0.0

    @property
    def slots_per_core_layer(self) -> int:
        return self.r_max if self.kv_slots <= 0 else min(self.kv_slots, self.r_max)

    @property
    def gate_threshold_logit(self) -> float:
        q = self.gate_q
        return math.log(q / (1.0 - q))

    @property
    def n_kv_slots(self) -> int:
        """KV entries per token, l0 + lr * s (App. E.1; s = r_max for the depth-indexed cache)."""
        return self.n_prelude + self.n_coda + self.n_core * self.slots_per_core_layer

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "fp32" else 2


@dataclass(frozen=True)
class Workload:
    """A synthetic offline (or online) request set plus scheduler settings."""

    name: str
    model: str
    n_seqs: int
    prompt_lo: int
    prompt_hi: int
    gen_lo: int
    gen_hi: int
    W: int
    M: int
    K: int
    mode: str = "refill"           # refill | no_refill | fixed_depth
    replay_depths: bool = False    # exit depths replayed from a seeded draw
    replay_p: float = 0.0          # truncated-geometric parameter of the draw
    kv_headroom: float = 0.0
    prompt_seed: int = 1
    length_seed: int = 2
    replay_seed: int = 3
    arrival_seed: int = 4

    @property
    def S(self) -> int:
        return max(1, self.W // 8)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _bias(name: str) -> float:
    return float(_BIAS.get(name, 0.0))


MODELS = {
    # Tiny fully looped fp32 model used for exact parity.
    "tiny": ModelShape(
        name="tiny", vocab=512, d_model=256, n_heads=4, head_dim=64, ffn=768,
        n_prelude=0, n_core=2, n_coda=0, r_max=8, r_min=2, has_adapter=False,
        dtype="fp32", gate_bias=_bias("tiny"),
    ),
    # Ouro-1.4B-shaped fully looped model (0-24-0, r_max 4).
    "ouro": ModelShape(
        name="ouro", vocab=49152, d_model=2048, n_heads=16, head_dim=128,
        ffn=5632, n_prelude=0, n_core=24, n_coda=0, r_max=4, r_min=2,
        has_adapter=False, dtype="bf16", gate_bias=_bias("ouro"),
    ),
    # Huginn-3.5B-shaped 2-4-2 model with a concat(embedding, state) adapter.
    "huginn": ModelShape(
        name="huginn", vocab=65536, d_model=5280, n_heads=55, head_dim=96,
        ffn=17920, n_prelude=2, n_core=4, n_coda=2, r_max=32, r_min=2,
        has_adapter=True, dtype="bf16", gate_bias=_bias("huginn"),
    ),
}

# Truncated geometric over {2..32} with mean exactly 12 (p chosen so that
# 2 + (1-p)(1-(1-p)^30)/p = 12.0).
HUGINN_REPLAY_P = 0.08515

WORKLOADS = {
    "tiny": Workload(name="tiny", model="tiny", n_seqs=8, prompt_lo=32,
                     prompt_hi=32, gen_lo=16, gen_hi=16, W=4, M=8192, K=1),
    "ouro": Workload(name="ouro", model="ouro", n_seqs=256, prompt_lo=128,
                     prompt_hi=1024, gen_lo=256, gen_hi=256, W=64, M=8192,
                     K=1),
    "huginn": Workload(name="huginn", model="huginn", n_seqs=128,
                       prompt_lo=256, prompt_hi=512, gen_lo=256, gen_hi=256,
                       W=64, M=8192, K=16, replay_depths=True,
                       replay_p=HUGINN_REPLAY_P),
    "long": Workload(name="long", model="ouro", n_seqs=32, prompt_lo=8192,
                     prompt_hi=8192, gen_lo=128, gen_hi=128, W=8, M=8192,
                     K=1),
    "online_ouro": Workload(name="online_ouro", model="ouro", n_seqs=512,
                            prompt_lo=64, prompt_hi=2048, gen_lo=32,
                            gen_hi=512, W=512, M=8192, K=1),
}


def model_shape(name: str) -> ModelShape:
    return MODELS[name]


def workload(name: str) -> Workload:
    return WORKLOADS[name]
