"""The C-ABI library loads on a CPU machine and exports what include/*.h declares.

No compute calls: only pure host functions (sizes, argument validation that
happens before any CUDA call).  KV bytes per token are pinned to Table 4 of
"Depth-adaptive Inference of Looped Language Models via Continuous Depth
Batching" (Appendix E.1): Ouro 768 KiB (s=4), Huginn 1402 KiB (s=16, r_max 16
as in the paper's Huginn runs).
"""

import ctypes as C
import dataclasses
import os
import re

import pytest

from continuous_depth_batching_gb300 import binding
from continuous_depth_batching_gb300.build import build
from synth import model_shape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build()
    return binding.lib()


def declared_functions():
    names = set()
    for h in sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(cdb_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"cdb_init", "cdb_admit", "cdb_step_core", "cdb_step_boundary", "cdb_drain"} <= names
    for n in sorted(names):
        assert hasattr(L, n), n


# Table 4 prints KiB per token rounded to whole KiB: the depth-indexed cache
# (s = r_max; Huginn at the paper's r_max 16), single-slot (s = 1) and
# first-then-shared (s = 2) layouts, l0 + lr * s entries (App. E.1).  The
# shared rows go through the kv_slots field with the model's own r_max.
TABLE4 = [("ouro", 0, 4, 768), ("ouro", 1, 4, 192), ("ouro", 2, 4, 384),
          ("huginn", 0, 16, 1402), ("huginn", 1, 32, 165), ("huginn", 2, 32, 248)]


@pytest.mark.parametrize("name,s,r_max,kib", TABLE4)
def test_kv_bytes_per_token_table4(L, name, s, r_max, kib):
    shape = dataclasses.replace(model_shape(name), r_max=r_max, kv_slots=s)
    desc = binding.model_desc(shape)
    assert abs(L.cdb_kv_bytes_per_token(C.byref(desc)) / 1024 - kib) <= 0.5
    assert abs(shape.n_kv_slots * 2 * shape.d_model * shape.elem_bytes / 1024 - kib) <= 0.5


def test_core_parameter_counts():
    # Appendix B: the Ouro-1.4B core holds about 1.2B parameters (24 narrow
    # layers) and the Huginn core about 1.6B (4 wide layers).
    def core_params(m):
        d, f = m.d_model, m.ffn
        return m.n_core * (4 * d * d + 3 * d * f)
    assert round(core_params(model_shape("ouro")) / 1e9, 1) == 1.2
    assert round(core_params(model_shape("huginn")) / 1e9, 1) == 1.6


def test_init_rejects_bad_arguments_without_a_gpu(L):
    shape = model_shape("tiny")
    desc = binding.model_desc(shape)
    cfg = binding.SchedCfg(0, 4, 64, 0, 1, 16, 0.0, 64, 16, 0, 0, None, 0, None, None, 0)
    w = binding.Weights()
    ctx = C.c_void_p()
    assert L.cdb_init(C.byref(desc), C.byref(w), C.byref(cfg), C.byref(ctx)) == -1  # no arena, no weights
    bad = binding.model_desc(dataclasses.replace(shape, r_min=1))
    assert L.cdb_init(C.byref(bad), C.byref(w), C.byref(cfg), C.byref(ctx)) == -1
    assert L.cdb_arena_bytes(C.byref(desc), C.byref(cfg)) > 0


def test_sim_rejects_bad_force_exit(L):
    import numpy as np
    sim = binding.Sim("refill", W=2, M=16, r_max=4)
    with pytest.raises(binding.CdbError):
        sim.admit(0, 4, 3, np.array([1, 3], dtype=np.int8))  # depth 1 < r_min
    with pytest.raises(binding.CdbError):
        sim.admit(1, 4, 3, np.array([5, 3], dtype=np.int8))  # depth > r_max


def test_convergence_gate_descriptor():
    shape = dataclasses.replace(model_shape("huginn"), r_min=3, gate_kind="convergence", conv_tau=0.25)
    desc = binding.model_desc(shape)
    assert desc.gate_kind == 1 and desc.gate_threshold == pytest.approx(0.25)
    assert binding.model_desc(model_shape("huginn")).gate_kind == 0
