"""Helpers shared by the GPU parity tests (oracle runs, forcing tables, GPU runs)."""

from __future__ import annotations

import numpy as np

from oracle.model import OracleModel, decode_sequence

NEAR = 1e-3  # gate logits / top-2 gaps closer than this are forced to the oracle's decision


def oracle_traces(shape, wts, reqs, mode="adaptive", keep_logits=0, near_tol=NEAR):
    om = OracleModel(shape, wts)
    out = {}
    for r in reqs:
        out[r["seq_id"]] = decode_sequence(om, r["prompt"], r["gen_len"], mode, r.get("replay"),
                                           None, keep_logits=keep_logits, near_tol=near_tol)
    return out


def force_tables(tr, replay=None, gap_band=NEAR):
    """force_exit / force_token arrays that pin near-threshold decisions to the oracle's.

    Gate decisions the oracle flagged as near (its near_tol band) and argmaxes
    whose top-2 gap is below gap_band take the oracle's result.
    """
    if replay is not None:
        fe = np.asarray(replay, dtype=np.int8)
    else:
        fe = np.array([e if near else 0 for e, near in zip(tr.exit_depths, tr.near_gate)], dtype=np.int8)
    ft = np.array([t if g < gap_band else -1 for t, g in zip(tr.tokens, tr.top2_gap)], dtype=np.int32)
    return fe, ft


def gpu_run(shape, dev_w, reqs, traces, *, mode="refill", W=4, M=8192, K=1, S=0, max_ctx=None,
            trace_tokens=0, trace_gate=False, attn_split=0, force=True, gap_band=NEAR, repeat=None):
    from continuous_depth_batching_gb300 import binding
    if max_ctx is None:
        max_ctx = max(len(r["prompt"]) + r["gen_len"] for r in reqs)
    cap = max(r["gen_len"] for r in reqs)
    eng = binding.Engine(shape, dev_w, mode=mode, W=W, M=M, K=K, S=S, max_ctx=max_ctx, max_new_cap=cap,
                         trace_tokens=trace_tokens, trace_gate=trace_gate, attn_split=attn_split)
    eng.trace_enable(True)
    if repeat is not None:
        eng.profile_repeat(repeat)
    for r in reqs:
        fe = ft = None
        if force and traces is not None:
            fe, ft = force_tables(traces[r["seq_id"]], r.get("replay"), gap_band)
        elif r.get("replay") is not None:
            fe = np.asarray(r["replay"], dtype=np.int8)
        eng.admit(r["seq_id"], r["prompt"], r["gen_len"], fe, ft)
    eng.run()
    out = {o["seq_id"]: o for o in eng.drain()}
    trace = eng.trace()
    eng.close()
    return out, trace


def forced_counts(traces, replays=None, gap_band=NEAR):
    """(forced exits, live gate decisions, forced tokens, tokens) of the forcing
    tables force_tables builds for these traces; replayed sequences decide no
    exit live, so their decisions are not counted."""
    fe = ne = ft = nt = 0
    for sid, tr in traces.items():
        if replays is None or replays.get(sid) is None:
            fe += int(sum(tr.near_gate))
            ne += len(tr.exit_depths)
        ft += int(sum(g < gap_band for g in tr.top2_gap))
        nt += len(tr.tokens)
    return fe, ne, ft, nt


def check_forced(traces, replays=None, gap_band=NEAR, max_frac=0.05, label=""):
    """Print the forced decisions and bound them: at most max_frac of the live
    gate decisions and of the tokens (at least one of each is allowed)."""
    fe, ne, ft, nt = forced_counts(traces, replays, gap_band)
    print(f"{label} forced exits {fe}/{ne}, forced tokens {ft}/{nt} (gap band {gap_band:g})")
    assert fe <= max(1, int(max_frac * ne)), (fe, ne)
    assert ft <= max(1, int(max_frac * nt)), (ft, nt)
    return fe, ne, ft, nt


def compare(out, traces, tol, check_logits=True, check_gate=False):
    """Tokens and exit depths exact; logits / hidden / gate logits within tol."""
    worst = 0.0
    assert sorted(out) == sorted(traces)
    for sid, tr in traces.items():
        o = out[sid]
        assert list(o["tokens"]) == tr.tokens, (sid, list(o["tokens"]), tr.tokens)
        assert list(o["exit_depths"]) == tr.exit_depths, (sid, list(o["exit_depths"]), tr.exit_depths)
        if check_logits and tr.logits:
            n = len(tr.logits)
            worst = max(worst, float(np.max(np.abs(o["logits"][:n] - np.array(tr.logits)))))
            worst = max(worst, float(np.max(np.abs(o["hidden"][:n] - np.array(tr.hidden)))))
        if check_gate:
            for t, zs in enumerate(tr.gate_logits):
                if zs:
                    g = o["gate_logits"][t, :len(zs)]
                    worst = max(worst, float(np.max(np.abs(g - np.array(zs)))))
    assert worst <= tol, worst
    return worst
