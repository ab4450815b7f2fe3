"""The host scheduler reproduces the paper's scheduling traces (Tables 2-3).

The traces give stage kinds, batch sizes, per-depth batch composition and
queue sizes, but not the prompt lengths or the exit depth of each token (the
datasets are not available).  Each test therefore chooses prompt lengths that
add up to the traces' own prefill token counts and per-token exit depths
consistent with the traces' exit counts, replays them through the scheduler
(include/cdb_sim.h) and compares every row.  Also checked: the Fig. 1 counts
(refill 6 forward passes, no-refill 8 for three sequences in two slots) with
chosen depths, since the figure does not print them (parity unpinned).
"""

import os

import numpy as np
import pytest

from continuous_depth_batching_gb300.binding import Sim

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def read_table(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append(line.rstrip("\n").split("\t"))
    return rows


def parse_detail(det):
    hist, exits = {}, 0
    body, _, x = det.partition(";x")
    exits = int(x)
    for part in body.split(","):
        r, n = part[1:].split(":")
        hist[int(r)] = int(n)
    return hist, exits


def check(trace, table, no_refill=False):
    assert len(trace) >= len(table)
    for i, (row, exp) in enumerate(zip(trace, table)):
        kind, B = exp[0], int(exp[1])
        where = f"stage {i + 1}: {row} vs {exp}"
        assert row["stage"] == kind, where
        assert row["batch"] == B, where
        if kind == "prefill":
            assert row["prefill_tokens"] == int(exp[2]), where
        if kind == "loop":
            hist, exits = parse_detail(exp[2])
            assert row["hist"] == hist, where
            assert row["exits"] == exits, where
        if no_refill:
            assert (row["q_d"], row["q_p"]) == (int(exp[3]), int(exp[4])), where
        else:
            assert (row["q_r"], row["q_c"], row["q_p"]) == (int(exp[3]), int(exp[4]), int(exp[5])), where


def ouro_lengths():
    # 20x400 + 192 of seq 20 = 8192; 208 + 31x250 + 234 of seq 52 = 8192;
    # 238 + 11x160 = 1998 (Table 2 stages 1, 3, 5).
    L = [400] * 20 + [400] + [250] * 31 + [472] + [160] * 11
    return L + [300] * (256 - len(L))


def huginn_lengths():
    # 20x400 + 192 = 8192; 208 + 32x240 + 304 = 8192; 285 + 10x150 = 1785.
    L = [400] * 20 + [400] + [240] * 32 + [589] + [150] * 10
    return L + [300] * (256 - len(L))


def run(sim, lengths, depth_of, gen=256, r_max=4, stages=20):
    for i, L in enumerate(lengths):
        e = np.array([depth_of(i, t) for t in range(1, gen)], dtype=np.int8)
        sim.admit(i, L, gen, e)
    # run until the trace has enough rows
    for _ in range(10000):
        if sim.trace_len() >= stages:
            break
        rc, _ = sim.step_boundary()
        assert rc >= 0
        if rc == 1:
            rc, _ = sim.step_core()
            assert rc >= 0
    return sim.trace()


def test_table2_ouro_refill_k1():
    def depth(i, t):
        if t == 1:
            return 2 if i == 0 else 3 if i <= 29 else 4
        if t == 2:
            if i == 0 or 1 <= i <= 9 or i == 30:
                return 2
            return 3
        return 4
    tr = run(Sim("refill", W=64, M=8192, K=1, r_max=4), ouro_lengths(), depth)
    check(tr, read_table("table2_ouro_refill_k1.tsv"))


def test_table2_huginn_refill_k1():
    def depth(i, t):
        if t == 1:
            return 7 if i <= 6 else 8 if i <= 28 else 9 if i <= 46 else 12
        return 5
    tr = run(Sim("refill", W=64, M=8192, K=1, r_max=16), huginn_lengths(), depth, r_max=16)
    check(tr, read_table("table2_huginn_refill_k1.tsv"))


def test_table3_ouro_no_refill():
    def depth(i, t):
        counts = {1: (1, 29, 34), 2: (13, 39, 12), 3: (17, 39, 8)}.get(t, (64, 0, 0))
        a, b, _ = counts
        return 2 if i < a else 3 if i < a + b else 4
    tr = run(Sim("no_refill", W=64, M=8192, K=1, r_max=4), ouro_lengths(), depth)
    check(tr, read_table("table3_ouro_norefill.tsv"), no_refill=True)


def test_table3_ouro_refill_k16():
    def depth(i, t):
        if t == 1:
            return 2 if i == 0 else 3 if i <= 29 else 4
        if t == 2:
            if i <= 9 or 30 <= i <= 32:
                return 2
            if 10 <= i <= 26 or 33 <= i <= 54:
                return 3
            return 4
        return 4
    tr = run(Sim("refill", W=64, M=8192, K=16, r_max=4), ouro_lengths(), depth)
    check(tr, read_table("table3_ouro_refill_k16.tsv"))


@pytest.mark.parametrize("mode,passes", [("refill", 6), ("no_refill", 8)])
def test_fig1_toy(mode, passes):
    # Three sequences, two slots, one decode token each (chosen depths 2, 4, 4):
    # refill starts the third sequence in the slot the first exit frees.
    sim = Sim(mode, W=2, M=64, S=1, K=1, r_max=4)
    for i, e in enumerate([2, 4, 4]):
        sim.admit(i, 4, 2, np.array([e], dtype=np.int8))
    sim.run()
    loops = [r for r in sim.trace() if r["stage"] == "loop"]
    assert len(loops) == passes
    assert sorted(sim.finished()) == [0, 1, 2]


@pytest.mark.parametrize("mode", ["refill", "no_refill", "fixed_depth"])
def test_every_sequence_finishes_with_all_loop_work(mode):
    rng = np.random.default_rng(3)
    r_max = 5
    sim = Sim(mode, W=7, M=50, S=0, K=2, r_max=r_max)
    total = 0
    for i in range(23):
        gen = int(rng.integers(1, 9))
        e = rng.integers(2, r_max + 1, max(gen - 1, 0)).astype(np.int8)
        sim.admit(i, int(rng.integers(1, 40)), gen, e)
        total += int(e.sum()) if mode != "fixed_depth" else r_max * (gen - 1)
    sim.run()
    assert sorted(sim.finished()) == list(range(23))
    loops = [r for r in sim.trace() if r["stage"] == "loop"]
    assert sum(sum(r["hist"].values()) for r in loops) == total
    assert max(r["batch"] for r in loops) <= 7


@pytest.mark.parametrize("mode", ["refill", "no_refill", "fixed_depth"])
def test_degenerate_jobs(mode):
    """No requests: the first call reports DONE.  Requests that generate one
    token finish in prefill (the token comes from the prompt's last position,
    App. A.5) and never reach the recurrent core."""
    from continuous_depth_batching_gb300 import binding
    sim = Sim(mode, W=2, M=16, S=1, K=1, r_max=4)
    assert sim.step_boundary()[0] == binding.DONE
    sim = Sim(mode, W=2, M=16, S=1, K=1, r_max=4)
    for i, p in enumerate([1, 16, 33]):            # one token, exactly M, two chunks and a bit
        sim.admit(i, p, 1, np.zeros(0, np.int8))
    sim.run()
    assert sorted(sim.finished()) == [0, 1, 2]
    tr = sim.trace()
    assert not any(r["stage"] in ("loop", "coda", "prelude") for r in tr)
    assert sum(r["prefill_tokens"] for r in tr if r["stage"] == "prefill") == 1 + 16 + 33
