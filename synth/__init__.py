"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

This package holds model shapes, workload recipes and counter-based random
generators only.  It contains none of the looped model's arithmetic: weights,
prompts, lengths, replayed exit depths and arrival times are produced here and
handed to both sides unchanged.
"""

from .configs import (  # noqa: F401
    ModelShape,
    Workload,
    MODELS,
    WORKLOADS,
    model_shape,
    workload,
)
from .generate import (  # noqa: F401
    splitmix64_at,
    normal_tensor,
    make_weights,
    make_prompts,
    make_lengths,
    make_replay_depths,
    make_arrivals,
    make_requests,
    weight_names,
)
