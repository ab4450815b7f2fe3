"""ctypes binding of the CDB C ABI (include/cdb.h, include/cdb_sim.h).

Argument marshalling only: every stage of the decode path runs inside the
native library.  PyTorch supplies device memory (weights, the arena) and
streams.  Loading fails loudly when the library has not been built.
"""

from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import LIB

MAX_DEPTH = 64

OK, IDLE, DONE = 0, 1, 2
ERRORS = {-1: "CDB_ERR_ARG", -2: "CDB_ERR_ARENA", -3: "CDB_ERR_KV_FULL", -4: "CDB_ERR_CUDA",
          -5: "CDB_ERR_DEVICE_BOUNDS", -6: "CDB_ERR_TIMEOUT", -7: "CDB_ERR_STATE"}
MODES = {"refill": 0, "no_refill": 1, "fixed_depth": 2}
STAGES = {0: "none", 1: "prefill", 2: "prelude", 3: "loop", 4: "coda"}


class ModelDesc(C.Structure):
    _fields_ = [("vocab", C.c_int), ("d_model", C.c_int), ("n_heads", C.c_int), ("head_dim", C.c_int),
                ("ffn", C.c_int), ("n_prelude", C.c_int), ("n_core", C.c_int), ("n_coda", C.c_int),
                ("r_max", C.c_int), ("r_min", C.c_int), ("has_adapter", C.c_int), ("dtype", C.c_int),
                ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("gate_threshold", C.c_float),
                ("gate_bias", C.c_float), ("kv_slots", C.c_int), ("gate_kind", C.c_int)]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("attn_norm", "wqkv", "wo", "mlp_norm", "wg", "wu", "wd")]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("gate_w", C.c_void_p), ("adapter", C.c_void_p), ("prelude", C.POINTER(LayerWeights)),
                ("core", C.POINTER(LayerWeights)), ("coda", C.POINTER(LayerWeights))]


class SchedCfg(C.Structure):
    _fields_ = [("mode", C.c_int), ("W", C.c_int), ("M", C.c_int), ("S", C.c_int), ("K", C.c_int),
                ("kv_blocks", C.c_int), ("kv_headroom", C.c_float), ("max_ctx", C.c_int),
                ("max_new_cap", C.c_int), ("trace_tokens", C.c_int), ("trace_gate", C.c_int),
                ("arena", C.c_void_p), ("arena_bytes", C.c_size_t), ("compute_stream", C.c_void_p),
                ("prep_stream", C.c_void_p), ("attn_split", C.c_int)]


class StepInfo(C.Structure):
    _fields_ = [("stage", C.c_int), ("batch", C.c_int), ("prefill_tokens", C.c_int), ("stage2", C.c_int),
                ("batch2", C.c_int), ("exits", C.c_int), ("q_r", C.c_int), ("q_c", C.c_int), ("q_p", C.c_int),
                ("q_d", C.c_int), ("depth_hist", C.c_int * MAX_DEPTH), ("step_index", C.c_int64),
                ("new_tokens", C.c_int), ("ctx", C.c_int64), ("ctx2", C.c_int64)]

    def as_dict(self):
        d = {f: getattr(self, f) for f, _ in self._fields_ if f != "depth_hist"}
        d["depth_hist"] = list(self.depth_hist)
        return d


class Result(C.Structure):
    _fields_ = [("seq_id", C.c_int64), ("n_tokens", C.c_int), ("tokens", C.POINTER(C.c_int32)),
                ("exit_depths", C.POINTER(C.c_int8)), ("gate_logits", C.POINTER(C.c_float)),
                ("logits", C.POINTER(C.c_float)), ("hidden", C.POINTER(C.c_float))]


class KernelStat(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("launches", C.c_int64), ("ms", C.c_double), ("bytes", C.c_double),
                ("flops", C.c_double)]


class TraceRow(C.Structure):
    _fields_ = [("stage", C.c_int), ("batch", C.c_int), ("prefill_tokens", C.c_int), ("exits", C.c_int),
                ("q_r", C.c_int), ("q_c", C.c_int), ("q_p", C.c_int), ("q_d", C.c_int),
                ("depth_hist", C.c_int * MAX_DEPTH)]

    def as_dict(self):
        hist = {i + 1: n for i, n in enumerate(self.depth_hist) if n}
        return dict(stage=STAGES[self.stage], batch=self.batch, prefill_tokens=self.prefill_tokens,
                    exits=self.exits, q_r=self.q_r, q_c=self.q_c, q_p=self.q_p, q_d=self.q_d, hist=hist)


_lib = None


def lib(path: str | None = None) -> C.CDLL:
    """Load libcdb.so (built by continuous_depth_batching_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(f"CDB library not built ({p}); run continuous_depth_batching_gb300.build.build()")
    L = C.CDLL(p)
    L.cdb_arena_bytes.restype = C.c_size_t
    L.cdb_arena_bytes.argtypes = [C.POINTER(ModelDesc), C.POINTER(SchedCfg)]
    L.cdb_kv_bytes_per_token.restype = C.c_size_t
    L.cdb_kv_bytes_per_token.argtypes = [C.POINTER(ModelDesc)]
    L.cdb_init.argtypes = [C.POINTER(ModelDesc), C.POINTER(Weights), C.POINTER(SchedCfg), C.POINTER(C.c_void_p)]
    L.cdb_admit.argtypes = [C.c_void_p, C.c_int64, C.POINTER(C.c_int32), C.c_int, C.c_int,
                            C.POINTER(C.c_int8), C.POINTER(C.c_int32)]
    L.cdb_step_boundary.argtypes = [C.c_void_p, C.POINTER(StepInfo)]
    L.cdb_step_core.argtypes = [C.c_void_p, C.POINTER(StepInfo)]
    L.cdb_drain.argtypes = [C.c_void_p, C.POINTER(Result), C.c_int, C.POINTER(C.c_int)]
    L.cdb_poll.argtypes = [C.c_void_p, C.POINTER(Result), C.c_int, C.POINTER(C.c_int)]
    L.cdb_sync.argtypes = [C.c_void_p]
    L.cdb_free.argtypes = [C.c_void_p]
    L.cdb_free.restype = None
    L.cdb_last_error.argtypes = [C.c_void_p]
    L.cdb_last_error.restype = C.c_char_p
    L.cdb_trace_enable.argtypes = [C.c_void_p, C.c_int]
    L.cdb_profile_enable.argtypes = [C.c_void_p, C.c_int]
    L.cdb_test_kv_pool.argtypes = [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_int), C.POINTER(C.c_int)]
    L.cdb_profile_repeat.argtypes = [C.c_void_p, C.c_int]
    L.cdb_profile_read.argtypes = [C.c_void_p, C.POINTER(KernelStat), C.c_int, C.POINTER(C.c_int)]
    L.cdb_kernel_launches.restype = C.c_int64
    L.cdb_kernel_launches.argtypes = []
    L.cdb_io_bytes.argtypes = [C.c_void_p, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]
    L.cdb_trace_read.argtypes = [C.c_void_p, C.POINTER(TraceRow), C.c_int, C.POINTER(C.c_int)]
    L.cdb_sim_create.argtypes = [C.c_int] * 8 + [C.c_float, C.c_int, C.c_int, C.POINTER(C.c_void_p)]
    L.cdb_sim_admit.argtypes = [C.c_void_p, C.c_int64, C.c_int, C.c_int, C.POINTER(C.c_int8)]
    L.cdb_sim_step_boundary.argtypes = [C.c_void_p, C.POINTER(StepInfo)]
    L.cdb_sim_step_core.argtypes = [C.c_void_p, C.POINTER(StepInfo)]
    L.cdb_sim_trace_read.argtypes = [C.c_void_p, C.POINTER(TraceRow), C.c_int, C.POINTER(C.c_int)]
    L.cdb_sim_finished.argtypes = [C.c_void_p, C.POINTER(C.c_int64), C.c_int, C.POINTER(C.c_int)]
    L.cdb_sim_free.argtypes = [C.c_void_p]
    L.cdb_sim_free.restype = None
    L.cdb_predict_job.argtypes = [C.POINTER(Job), C.c_int, C.c_int, C.POINTER(LatencyModel), C.POINTER(Prediction)]
    L.cdb_roofline_latency.argtypes = [C.POINTER(ModelDesc), C.c_double, C.c_double, C.c_double,
                                       C.POINTER(LatencyModel)]
    L.cdb_predict_online.argtypes = [C.POINTER(Job), C.POINTER(C.c_double), C.c_int, C.c_int,
                                     C.POINTER(LatencyModel), C.POINTER(C.c_double), C.POINTER(Prediction)]
    L.cdb_select_schedule.argtypes = [C.POINTER(Job), C.POINTER(LatencyModel), C.POINTER(C.c_int),
                                      C.POINTER(C.c_int), C.POINTER(Prediction), C.POINTER(C.c_double),
                                      C.POINTER(C.c_double)]
    _lib = L
    return L


def kernel_launches() -> int:
    return int(lib().cdb_kernel_launches())


class CdbError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(C.POINTER(C.c_int32))


def _i8(a):
    a = np.ascontiguousarray(a, dtype=np.int8)
    return a, a.ctypes.data_as(C.POINTER(C.c_int8))


def model_desc(shape) -> ModelDesc:
    """cdb_model_desc from a shape object with the fields of synth.ModelShape."""
    import math
    q = shape.gate_q
    conv = getattr(shape, "gate_kind", "probe") == "convergence"
    return ModelDesc(shape.vocab, shape.d_model, shape.n_heads, shape.head_dim, shape.ffn, shape.n_prelude,
                     shape.n_core, shape.n_coda, shape.r_max, shape.r_min, int(shape.has_adapter),
                     1 if shape.dtype == "bf16" else 0, shape.rms_eps, shape.rope_theta,
                     shape.conv_tau if conv else math.log(q / (1.0 - q)), shape.gate_bias,
                     int(getattr(shape, "kv_slots", 0)), 1 if conv else 0)


def kv_bytes_per_token(shape) -> int:
    """KV-cache bytes one token occupies for this model (every layer and loop step)."""
    return int(lib().cdb_kv_bytes_per_token(C.byref(model_desc(shape))))


def device_weights(shape, weights: dict, device="cuda") -> dict:
    """Move host weights (float32 or uint16 bf16 bit patterns) to device tensors."""
    import torch
    out = {}
    for k, v in weights.items():
        if v.dtype == np.uint16:
            t = torch.from_numpy(v.view(np.int16)).to(device).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(device)
        out[k] = t.contiguous()
    return out


class Engine:
    """One CDB context on the current CUDA device."""

    def __init__(self, shape, dev_weights: dict, *, mode="refill", W=64, M=8192, S=0, K=1, kv_blocks=None,
                 kv_headroom=0.0, max_ctx=2048, max_new_cap=256, trace_tokens=0, trace_gate=False,
                 attn_split=0, stream=None, prep_stream=None):
        import torch
        self.L = lib()
        self.shape = shape
        self.w = dev_weights
        self.desc = model_desc(shape)
        self.max_new_cap = max_new_cap
        self.trace_tokens = trace_tokens
        self.trace_gate = bool(trace_gate)
        if kv_blocks is None:
            kv_blocks = W * ((max_ctx + 15) // 16)
        self.cfg = SchedCfg(MODES[mode] if isinstance(mode, str) else mode, W, M, S, K, kv_blocks, kv_headroom,
                            max_ctx, max_new_cap, trace_tokens, int(bool(trace_gate)), None, 0, None, None,
                            attn_split)
        n = self.L.cdb_arena_bytes(C.byref(self.desc), C.byref(self.cfg))
        self.arena = torch.empty(n + 256, dtype=torch.uint8, device="cuda")
        base = self.arena.data_ptr()
        self.cfg.arena = (base + 255) // 256 * 256
        self.cfg.arena_bytes = n
        self.stream = stream or torch.cuda.current_stream()
        self.cfg.compute_stream = self.stream.cuda_stream
        self.prep = prep_stream
        self.cfg.prep_stream = prep_stream.cuda_stream if prep_stream is not None else None

        def layers(kind, count):
            arr = (LayerWeights * max(count, 1))()
            for i in range(count):
                p = f"{kind}.{i}."
                arr[i] = LayerWeights(*[dev_weights[p + n].data_ptr() for n in
                                        ("attn_norm", "wqkv", "wo", "mlp_norm", "wg", "wu", "wd")])
            return arr

        self._lw = [layers("prelude", shape.n_prelude), layers("core", shape.n_core),
                    layers("coda", shape.n_coda)]
        ad = dev_weights["adapter"].data_ptr() if shape.has_adapter else None
        self.weights = Weights(dev_weights["embed"].data_ptr(), dev_weights["lm_head"].data_ptr(),
                               dev_weights["final_norm"].data_ptr(), dev_weights["gate_w"].data_ptr(), ad,
                               self._lw[0], self._lw[1], self._lw[2])
        ctx = C.c_void_p()
        rc = self.L.cdb_init(C.byref(self.desc), C.byref(self.weights), C.byref(self.cfg), C.byref(ctx))
        if rc != OK:
            raise CdbError(rc, "cdb_init failed")
        self.ctx = ctx

    def _check(self, rc):
        if rc < 0:
            raise CdbError(rc, self.L.cdb_last_error(self.ctx).decode())
        return rc

    def admit(self, seq_id, prompt, max_new, force_exit=None, force_token=None):
        p, pp = _i32(prompt)
        fe = fp = ft = ftp = None
        if force_exit is not None:
            fe, fp = _i8(force_exit)
        if force_token is not None:
            ft, ftp = _i32(force_token)
        return self._check(self.L.cdb_admit(self.ctx, int(seq_id), pp, len(p), int(max_new), fp, ftp))

    def step_boundary(self):
        info = StepInfo()
        return self._check(self.L.cdb_step_boundary(self.ctx, C.byref(info))), info

    def step_core(self):
        info = StepInfo()
        return self._check(self.L.cdb_step_core(self.ctx, C.byref(info))), info

    def sync(self):
        return self._check(self.L.cdb_sync(self.ctx))

    def drain(self, cap=4096):
        """Finished sequences (waits for their results); see cdb_drain."""
        return self._collect(self.L.cdb_drain, cap)

    def poll(self, cap=16):
        """Finished sequences whose results are already on the host (no wait); see cdb_poll."""
        return self._collect(self.L.cdb_poll, cap)

    def _collect(self, fn, cap):
        s = self.shape
        cap_new = self.max_new_cap
        bufs = []
        res = (Result * cap)()
        for i in range(cap):
            b = dict(tokens=np.zeros(cap_new, np.int32), depths=np.zeros(max(cap_new - 1, 1), np.int8))
            res[i].tokens = b["tokens"].ctypes.data_as(C.POINTER(C.c_int32))
            res[i].exit_depths = b["depths"].ctypes.data_as(C.POINTER(C.c_int8))
            if self.trace_gate:
                b["gate"] = np.full(cap_new * s.r_max, np.nan, np.float32)
                res[i].gate_logits = b["gate"].ctypes.data_as(C.POINTER(C.c_float))
            if self.trace_tokens:
                b["logits"] = np.zeros(self.trace_tokens * s.vocab, np.float32)
                b["hidden"] = np.zeros(self.trace_tokens * s.d_model, np.float32)
                res[i].logits = b["logits"].ctypes.data_as(C.POINTER(C.c_float))
                res[i].hidden = b["hidden"].ctypes.data_as(C.POINTER(C.c_float))
            bufs.append(b)
        n = C.c_int()
        self._check(fn(self.ctx, res, cap, C.byref(n)))
        out = []
        for i in range(n.value):
            nt = res[i].n_tokens
            b = bufs[i]
            r = dict(seq_id=res[i].seq_id, tokens=b["tokens"][:nt].copy(),
                     exit_depths=b["depths"][:max(nt - 1, 0)].astype(np.int64).copy())
            if self.trace_gate:
                r["gate_logits"] = b["gate"][:(nt - 1) * s.r_max].reshape(nt - 1, s.r_max).copy()
            if self.trace_tokens:
                r["logits"] = b["logits"].reshape(self.trace_tokens, s.vocab).copy()
                r["hidden"] = b["hidden"].reshape(self.trace_tokens, s.d_model).copy()
            out.append(r)
        return out

    def profile_enable(self, on=True, core_only=False):
        self._check(self.L.cdb_profile_enable(self.ctx, (2 if core_only else 1) if on else 0))

    def profile_repeat(self, cls=None):
        """Relaunch one kernel class inside every core step (None stops)."""
        code = -1 if cls is None else {"attention": 0, "gemm": 1, "rowwise": 3}[cls]
        self._check(self.L.cdb_profile_repeat(self.ctx, code))

    def profile_read(self):
        st = (KernelStat * 8)()
        n = C.c_int()
        self._check(self.L.cdb_profile_read(self.ctx, st, 8, C.byref(n)))
        return {st[i].name.decode(): dict(launches=st[i].launches, ms=st[i].ms, bytes=st[i].bytes,
                                          flops=st[i].flops) for i in range(n.value)}

    def io_bytes(self):
        a, b = C.c_int64(), C.c_int64()
        self._check(self.L.cdb_io_bytes(self.ctx, C.byref(a), C.byref(b)))
        return a.value, b.value

    def kv_pool(self):
        """The KV cache in the arena as a tensor view [kv_blocks, n_kv_slots, 2, H, 16, hd]."""
        import torch
        p, nb, ns = C.c_void_p(), C.c_int(), C.c_int()
        self._check(self.L.cdb_test_kv_pool(self.ctx, C.byref(p), C.byref(nb), C.byref(ns)))
        s = self.shape
        es = 2 if s.dtype == "bf16" else 4
        n = nb.value * ns.value * 2 * s.n_heads * 16 * s.head_dim
        off = p.value - self.arena.data_ptr()
        raw = self.arena[off:off + n * es]
        t = raw.view(torch.bfloat16 if es == 2 else torch.float32)
        return t.view(nb.value, ns.value, 2, s.n_heads, 16, s.head_dim)

    def trace_enable(self, on=True):
        self._check(self.L.cdb_trace_enable(self.ctx, int(on)))

    def trace(self):
        n = C.c_int()
        self._check(self.L.cdb_trace_read(self.ctx, None, 1 << 30, C.byref(n)))
        cap = max(n.value, 1)
        rows = (TraceRow * cap)()
        self._check(self.L.cdb_trace_read(self.ctx, rows, cap, C.byref(n)))
        return [rows[i].as_dict() for i in range(n.value)]

    def run(self, max_calls=10 ** 9):
        """Driver loop: boundary stages until IDLE, then a core step; until DONE."""
        calls = 0
        while calls < max_calls:
            rc, _ = self.step_boundary()
            calls += 1
            if rc == DONE:
                break
            if rc == IDLE:
                self.step_core()
        self.sync()
        return calls

    def close(self):
        if getattr(self, "ctx", None):
            self.L.cdb_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Sim:
    """Host-only replay of the scheduler (include/cdb_sim.h)."""

    def __init__(self, mode="refill", W=64, M=8192, S=0, K=1, r_max=4, r_min=2, kv_blocks=1 << 20,
                 kv_headroom=0.0, max_ctx=1 << 16, max_new_cap=1 << 14):
        self.L = lib()
        h = C.c_void_p()
        rc = self.L.cdb_sim_create(MODES[mode] if isinstance(mode, str) else mode, W, M, S, K, r_max, r_min,
                                   kv_blocks, kv_headroom, max_ctx, max_new_cap, C.byref(h))
        if rc != OK:
            raise CdbError(rc, "cdb_sim_create")
        self.h = h

    def admit(self, seq_id, prompt_len, max_new, exit_depths=None):
        e = ep = None
        if exit_depths is not None:
            e, ep = _i8(exit_depths)
        rc = self.L.cdb_sim_admit(self.h, int(seq_id), int(prompt_len), int(max_new), ep)
        if rc < 0:
            raise CdbError(rc, "cdb_sim_admit")
        return rc

    def step_boundary(self):
        info = StepInfo()
        return self.L.cdb_sim_step_boundary(self.h, C.byref(info)), info

    def step_core(self):
        info = StepInfo()
        return self.L.cdb_sim_step_core(self.h, C.byref(info)), info

    def run(self, max_calls=10 ** 7):
        for _ in range(max_calls):
            rc, _ = self.step_boundary()
            if rc < 0:
                raise CdbError(rc, "boundary")
            if rc == DONE:
                return
            if rc == IDLE:
                rc, _ = self.step_core()
                if rc < 0:
                    raise CdbError(rc, "core")

    def trace_len(self):
        n = C.c_int()
        self.L.cdb_sim_trace_read(self.h, None, 1 << 30, C.byref(n))
        return n.value

    def trace(self):
        cap = max(self.trace_len(), 1)
        rows = (TraceRow * cap)()
        n = C.c_int()
        self.L.cdb_sim_trace_read(self.h, rows, cap, C.byref(n))
        return [rows[i].as_dict() for i in range(n.value)]

    def finished(self, cap=1 << 20):
        ids = (C.c_int64 * cap)()
        n = C.c_int()
        self.L.cdb_sim_finished(self.h, ids, cap, C.byref(n))
        return list(ids[:n.value])

    def __del__(self):
        try:
            self.L.cdb_sim_free(self.h)
        except Exception:
            pass


# ---------------------------------------------------------------------------
# latency planner (include/cdb_plan.h)
# ---------------------------------------------------------------------------

COST_STAGES = ("prefill", "prelude", "core", "coda")


class StageCost(C.Structure):
    _fields_ = [("delta", C.c_double), ("gamma", C.c_double), ("alpha", C.c_double)]


class LatencyModel(C.Structure):
    _fields_ = [(s, StageCost) for s in COST_STAGES]

    def as_dict(self):
        return {s: {k: getattr(getattr(self, s), k) for k in ("delta", "gamma", "alpha")} for s in COST_STAGES}

    @classmethod
    def from_dict(cls, d):
        lm = cls()
        for s in COST_STAGES:
            c = d.get(s, {})
            setattr(lm, s, StageCost(float(c.get("delta", 0.0)), float(c.get("gamma", 0.0)),
                                     float(c.get("alpha", 0.0))))
        return lm


class Job(C.Structure):
    _fields_ = [("n_seqs", C.c_int), ("prompt_len", C.POINTER(C.c_int32)), ("gen_len", C.POINTER(C.c_int32)),
                ("exit_depths", C.POINTER(C.c_int8)), ("W", C.c_int), ("M", C.c_int), ("S", C.c_int),
                ("r_max", C.c_int), ("r_min", C.c_int), ("kv_blocks", C.c_int), ("kv_headroom", C.c_float),
                ("max_ctx", C.c_int), ("max_new_cap", C.c_int)]


class Prediction(C.Structure):
    _fields_ = [("seconds", C.c_double), ("prefill_seconds", C.c_double), ("prelude_seconds", C.c_double),
                ("core_seconds", C.c_double), ("coda_seconds", C.c_double), ("prefill_stages", C.c_int64),
                ("prelude_stages", C.c_int64), ("core_steps", C.c_int64), ("coda_stages", C.c_int64),
                ("tokens", C.c_int64), ("core_token_steps", C.c_int64), ("mean_core_batch", C.c_double),
                ("mean_coda_batch", C.c_double)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class PlanJob:
    """An offline job for the planner: requests with prompt / output lengths and exit depths."""

    def __init__(self, reqs, W, M=8192, S=0, r_max=4, r_min=2, kv_blocks=1 << 22, kv_headroom=0.0,
                 max_ctx=None, max_new_cap=None):
        import numpy as np
        self._p = np.ascontiguousarray([len(r["prompt"]) if "prompt" in r else r["prompt_len"] for r in reqs],
                                       dtype=np.int32)
        self._g = np.ascontiguousarray([r["gen_len"] for r in reqs], dtype=np.int32)
        ex = [np.asarray(r["replay"] if r.get("replay") is not None else r.get("exit_depths", []), dtype=np.int8)
              for r in reqs]
        for e, g in zip(ex, self._g):
            if len(e) != g - 1:
                raise ValueError("every request needs gen_len - 1 exit depths")
        self._e = np.ascontiguousarray(np.concatenate(ex) if ex else np.zeros(0, np.int8), dtype=np.int8)
        mc = int(max_ctx or int((self._p + self._g - 1).max()))
        mn = int(max_new_cap or int(self._g.max()))
        self.job = Job(len(reqs), self._p.ctypes.data_as(C.POINTER(C.c_int32)),
                       self._g.ctypes.data_as(C.POINTER(C.c_int32)), self._e.ctypes.data_as(C.POINTER(C.c_int8)),
                       W, M, S, r_max, r_min, kv_blocks, kv_headroom, mc, mn)


def predict_job(job: PlanJob, mode, K, lm: LatencyModel) -> dict:
    out = Prediction()
    rc = lib().cdb_predict_job(C.byref(job.job), MODES[mode] if isinstance(mode, str) else mode, K, C.byref(lm),
                               C.byref(out))
    if rc != OK:
        raise CdbError(rc, "cdb_predict_job")
    return out.as_dict()


def roofline_latency(shape, hbm_gbps, tensor_tflops, launch_s=0.0) -> LatencyModel:
    lm = LatencyModel()
    desc = model_desc(shape)
    rc = lib().cdb_roofline_latency(C.byref(desc), hbm_gbps, tensor_tflops, launch_s, C.byref(lm))
    if rc != OK:
        raise CdbError(rc, "cdb_roofline_latency")
    return lm


def select_schedule(job: PlanJob, lm: LatencyModel) -> dict:
    mode, K = C.c_int(), C.c_int()
    best = Prediction()
    r_s, n_s = C.c_double(), C.c_double()
    rc = lib().cdb_select_schedule(C.byref(job.job), C.byref(lm), C.byref(mode), C.byref(K), C.byref(best),
                                   C.byref(r_s), C.byref(n_s))
    if rc != OK:
        raise CdbError(rc, "cdb_select_schedule")
    names = {v: k for k, v in MODES.items()}
    return {"mode": names[mode.value], "K": K.value, "prediction": best.as_dict(),
            "refill_seconds": r_s.value, "no_refill_seconds": n_s.value}


def predict_online(job: PlanJob, arrival_s, mode, K, lm: LatencyModel):
    """Predicted finish time of every request arriving at arrival_s (see cdb_predict_online)."""
    import numpy as np
    arr = np.ascontiguousarray(arrival_s, dtype=np.float64)
    if arr.shape != (job.job.n_seqs,):
        raise ValueError("one arrival time per request")
    fin = np.zeros(job.job.n_seqs, dtype=np.float64)
    out = Prediction()
    rc = lib().cdb_predict_online(C.byref(job.job), arr.ctypes.data_as(C.POINTER(C.c_double)),
                                  MODES[mode] if isinstance(mode, str) else mode, K, C.byref(lm),
                                  fin.ctypes.data_as(C.POINTER(C.c_double)), C.byref(out))
    if rc != OK:
        raise CdbError(rc, "cdb_predict_online")
    return fin, out.as_dict()
