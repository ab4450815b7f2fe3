"""Decode attention over the depth-indexed paged cache (include/cdb_testing.h).

Reference: a float64 torch restatement of the read rule of §4.2 ("Depth-
adaptive Inference of Looped Language Models via Continuous Depth Batching"):
row i at loop step r reads position j from loop step min(r, e_j) through the
sequence's 16-token pages.  Exit gaps (steps above e_j) hold NaN, so a gap read
would poison the output.  Also: split sizes agree, and each row's bits do not
depend on the other rows in the call.
"""

import ctypes as C

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.build import build
    build()
    lib = binding.lib()
    lib.cdb_test_attention.argtypes = ([C.c_void_p, C.c_int] + [C.c_void_p] * 5 + [C.c_int, C.c_void_p] +
                                       [C.c_int] * 8 + [C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p])
    lib.cdb_test_attention_uniform.argtypes = ([C.c_void_p, C.c_int] + [C.c_void_p] * 5 + [C.c_int] * 9 +
                                               [C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p])
    lib.cdb_test_attention_scratch_bytes.restype = C.c_size_t
    lib.cdb_test_attention_scratch_bytes.argtypes = [C.c_int] * 5
    return lib


def make_case(dtype, H, hd, rows=6, r_max=4, n_core=2, layer=1, max_ctx=700, seed=0):
    import torch
    rng = np.random.default_rng(seed)
    d = H * hd
    nsl = n_core * r_max
    max_blocks = (max_ctx + 15) // 16
    kv_blocks = rows * max_blocks + 7
    tdt = torch.bfloat16 if dtype == 1 else torch.float32
    pool = torch.randn(kv_blocks, nsl, 2, H, 16, hd, dtype=torch.float64)
    perm = rng.permutation(kv_blocks)[: rows * max_blocks].reshape(rows, max_blocks)
    bt = torch.from_numpy(perm.astype(np.int32))
    etab = torch.from_numpy(rng.integers(1, r_max + 1, (kv_blocks, 16)).astype(np.uint8))
    pos = rng.integers(0, max_ctx, rows).astype(np.int32)
    pos[0], pos[1] = 0, max_ctx - 1
    depth = rng.integers(0, r_max, rows).astype(np.int32)
    slot = np.arange(rows, dtype=np.int32)
    base = layer * r_max
    for i in range(rows):  # own position is in flight: read at the current step
        b = perm[i, pos[i] // 16]
        etab[b, pos[i] % 16] = r_max
    # exit gaps -> NaN
    for b in range(kv_blocks):
        for o in range(16):
            e = int(etab[b, o])
            pool[b, base + e:base + r_max, :, :, o, :] = float("nan")
    q = torch.randn(rows, d, dtype=torch.float64)
    return dict(pool=pool.to(tdt), bt=bt, etab=etab, pos=pos, depth=depth, slot=slot, q=q.to(tdt), H=H, hd=hd,
                nsl=nsl, base=base, max_blocks=max_blocks, kv_blocks=kv_blocks, max_ctx=max_ctx, r_max=r_max,
                dtype=dtype)


def reference(cs):
    import torch
    pool = cs["pool"].double()
    q = cs["q"].double()
    H, hd = cs["H"], cs["hd"]
    out = torch.zeros_like(q)
    for i in range(len(cs["pos"])):
        r = int(cs["depth"][i]) + 1
        P = int(cs["pos"][i]) + 1
        j = torch.arange(P)
        blk = cs["bt"][int(cs["slot"][i])][j // 16].long()
        off = j % 16
        e = cs["etab"][blk, off].long()
        sl = cs["base"] + torch.clamp(e, max=r) - 1
        K = pool[blk, sl, 0, :, off]  # [P, H, hd]
        V = pool[blk, sl, 1, :, off]
        for h in range(H):
            s = K[:, h] @ q[i, h * hd:(h + 1) * hd] / np.sqrt(hd)
            p = torch.softmax(s, 0)
            out[i, h * hd:(h + 1) * hd] = p @ V[:, h]
    return out


def run(L, cs, split, rows=None):
    import torch
    n = rows or len(cs["pos"])
    dev = {k: cs[k].cuda() for k in ("pool", "bt", "etab", "q")}
    slot = torch.from_numpy(cs["slot"][:n]).cuda()
    pos = torch.from_numpy(cs["pos"][:n]).cuda()
    depth = torch.from_numpy(cs["depth"][:n]).cuda()
    out = torch.zeros(n, cs["H"] * cs["hd"], dtype=cs["q"].dtype, device="cuda")
    nb = L.cdb_test_attention_scratch_bytes(n, cs["H"], cs["hd"], split, cs["max_ctx"])
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = L.cdb_test_attention(dev["q"].data_ptr(), n, slot.data_ptr(), pos.data_ptr(), depth.data_ptr(),
                              dev["pool"].data_ptr(), dev["bt"].data_ptr(), cs["max_blocks"], dev["etab"].data_ptr(),
                              cs["kv_blocks"], cs["nsl"], cs["base"], cs["H"], cs["hd"], cs["dtype"], split,
                              cs["max_ctx"], out.data_ptr(), scratch.data_ptr(), nb, None)
    assert rc == 0, rc
    return out


@pytest.mark.parametrize("dtype,H,hd", [(0, 4, 64), (1, 16, 128), (1, 5, 96), (0, 2, 8), (1, 3, 64), (1, 6, 32),
                                        (1, 2, 16), (1, 3, 8)])
@pytest.mark.parametrize("split", [16, 256])
def test_matches_reference(L, dtype, H, hd, split):
    cs = make_case(dtype, H, hd)
    out = run(L, cs, split).double().cpu()
    ref = reference(cs)
    assert torch_finite(out)
    tol = 2e-5 if dtype == 0 else 1e-2
    err = (out - ref).abs()
    assert (err <= tol * (1 + ref.abs())).all().item(), err.max().item()


def torch_finite(t):
    import torch
    return bool(torch.isfinite(t).all().item())


def test_row_bits_independent_of_batch(L):
    cs = make_case(1, 16, 128, rows=8, seed=3)
    full = run(L, cs, 256)
    part = run(L, cs, 256, rows=3)
    assert (full[:3] == part).all().item()


def make_uniform_case(dtype, H, hd, rows=6, seed=0, max_ctx=700):
    """No exit gaps (every e_j = r_max), so the read rule is slot r for every
    key; positions past each row's own one hold NaN in every slot."""
    cs = make_case(dtype, H, hd, rows=rows, max_ctx=max_ctx, seed=seed)
    pool = cs["pool"].double()
    cs["etab"][:] = cs["r_max"]
    rng = np.random.default_rng(seed + 100)
    pool = torch_randn_like(pool, rng)
    for i in range(rows):
        p = int(cs["pos"][i])
        b = int(cs["bt"][int(cs["slot"][i])][p // 16])
        if p % 16 != 15:
            pool[b, :, :, :, p % 16 + 1:, :] = float("nan")
    cs["pool"] = pool.to(cs["pool"].dtype)
    return cs


def torch_randn_like(t, rng):
    import torch
    return torch.from_numpy(rng.standard_normal(tuple(t.shape))).to(t.dtype)


def run_uniform(L, cs, split):
    import torch
    n = len(cs["pos"])
    dev = {k: cs[k].cuda() for k in ("pool", "bt", "q")}
    slot = torch.from_numpy(cs["slot"]).cuda()
    pos = torch.from_numpy(cs["pos"]).cuda()
    depth = torch.from_numpy(cs["depth"]).cuda()
    out = torch.zeros(n, cs["H"] * cs["hd"], dtype=cs["q"].dtype, device="cuda")
    nb = L.cdb_test_attention_scratch_bytes(n, cs["H"], cs["hd"], split, cs["max_ctx"])
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = L.cdb_test_attention_uniform(dev["q"].data_ptr(), n, slot.data_ptr(), pos.data_ptr(), depth.data_ptr(),
                                      dev["pool"].data_ptr(), dev["bt"].data_ptr(), cs["max_blocks"],
                                      cs["kv_blocks"], cs["nsl"], cs["base"], cs["H"], cs["hd"], cs["dtype"],
                                      split, cs["max_ctx"], out.data_ptr(), scratch.data_ptr(), nb, None)
    assert rc == 0, rc
    return out


@pytest.mark.parametrize("dtype,H,hd", [(1, 16, 128), (1, 5, 96), (1, 3, 64), (1, 6, 32), (1, 2, 16), (0, 4, 64)])
@pytest.mark.parametrize("split", [16, 128, 256])
def test_uniform_matches_reference(L, dtype, H, hd, split):
    cs = make_uniform_case(dtype, H, hd, seed=5)
    out = run_uniform(L, cs, split).double().cpu()
    ref = reference(cs)
    assert torch_finite(out)
    tol = 2e-5 if dtype == 0 else 1e-2
    err = (out - ref).abs()
    assert (err <= tol * (1 + ref.abs())).all().item(), err.max().item()


def test_uniform_equals_clamped_read_after_gap_fill(L):
    """Filling each position's exit gaps with its deepest entry (what the
    engine does when a token leaves the loop) makes the uniform read agree
    with the depth-clamped reference."""
    import torch
    cs = make_case(1, 16, 128, rows=5, max_ctx=400, seed=9)
    ref_clamped = run(L, cs, 128)
    pool = cs["pool"].clone()
    base, r_max = cs["base"], cs["r_max"]
    for b in range(cs["kv_blocks"]):
        for o in range(16):
            e = int(cs["etab"][b, o])
            for rr in range(e + 1, r_max + 1):
                pool[b, base + rr - 1, :, :, o, :] = pool[b, base + e - 1, :, :, o, :]
    cs2 = dict(cs, pool=pool)
    out = run_uniform(L, cs2, 128)
    ref = reference(cs)
    err_u = (out.double().cpu() - ref).abs().max().item()
    err_c = (ref_clamped.double().cpu() - ref).abs().max().item()
    assert torch_finite(out)
    assert err_u <= 1e-2 * (1 + ref.abs().max().item()), (err_u, err_c)


@pytest.mark.parametrize("H,hd", [(16, 128), (5, 96), (3, 64), (2, 32)])
def test_prefill_tiles_match_causal_reference(L, H, hd):
    """Causal prefill attention over query tiles against a float64 reference.
    Three sequences: a fresh prompt, a continuing chunk starting mid-page,
    and one short enough to fit in a single partial tile; positions past each
    sequence's last row hold NaN in the pool."""
    import torch
    L.cdb_test_attention_prefill.argtypes = ([C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p] +
                                             [C.c_int] * 6 + [C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p])
    rng = np.random.default_rng(17)
    d = H * hd
    nsl, slot = 6, 4
    runs = [(0, 0, 150), (1, 37, 170), (2, 0, 9)]  # (sequence slot, first position, rows)
    max_blocks = 16
    kv_blocks = 3 * max_blocks + 5
    perm = rng.permutation(kv_blocks)[: 3 * max_blocks].reshape(3, max_blocks)
    bt = torch.from_numpy(perm.astype(np.int32))
    pool = torch.from_numpy(rng.standard_normal((kv_blocks, nsl, 2, H, 16, hd)))
    last = {sq: p0 + n - 1 for sq, p0, n in runs}
    for sq in range(3):
        for p in range(last[sq] + 1, max_blocks * 16):
            pool[perm[sq, p // 16], :, :, :, p % 16, :] = float("nan")
    row_slot = np.concatenate([np.full(n, sq, np.int32) for sq, p0, n in runs])
    row_pos = np.concatenate([np.arange(p0, p0 + n, dtype=np.int32) for sq, p0, n in runs])
    rows = len(row_pos)
    q = torch.from_numpy(rng.standard_normal((rows, d))).to(torch.bfloat16)
    poolb = pool.to(torch.bfloat16)
    ref = torch.zeros(rows, d, dtype=torch.float64)
    pd, qd = poolb.double(), q.double()
    for i in range(rows):
        sq, p = int(row_slot[i]), int(row_pos[i])
        j = torch.arange(p + 1)
        blk = bt[sq][j // 16].long()
        K = pd[blk, slot, 0, :, j % 16]
        V = pd[blk, slot, 1, :, j % 16]
        for h in range(H):
            w = torch.softmax(K[:, h] @ qd[i, h * hd:(h + 1) * hd] / np.sqrt(hd), 0)
            ref[i, h * hd:(h + 1) * hd] = w @ V[:, h]
    out = torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda")
    scratch = torch.zeros(256 + 16 * (rows + 1), dtype=torch.uint8, device="cuda")
    dq, dp, dbt = q.cuda(), poolb.cuda(), bt.cuda()
    rc = L.cdb_test_attention_prefill(dq.data_ptr(), rows, row_slot.ctypes.data, row_pos.ctypes.data, dp.data_ptr(),
                                      dbt.data_ptr(), max_blocks, kv_blocks, nsl, slot, H, hd, out.data_ptr(),
                                      scratch.data_ptr(), scratch.numel(), None)
    assert rc == 0, rc
    o = out.double().cpu()
    assert torch_finite(o)
    err = (o - ref).abs()
    assert (err <= 1e-2 * (1 + ref.abs())).all().item(), err.max().item()


@pytest.mark.parametrize("uniform", [False, True])
def test_long_context_matches_reference(L, uniform):
    """8320 keys (an 8192-token prompt plus 128 generated tokens): 65 splits of
    128 keys per row, merged by the split-KV combine."""
    cs = (make_uniform_case if uniform else make_case)(1, 4, 128, rows=3, max_ctx=8320, seed=13,
                                                      **({} if uniform else dict(n_core=1, layer=0)))
    out = (run_uniform if uniform else run)(L, cs, 128).double().cpu()
    ref = reference(cs)
    assert torch_finite(out)
    err = (out - ref).abs()
    assert (err <= 1e-2 * (1 + ref.abs())).all().item(), err.max().item()


def test_prefill_tiles_long_prompt_match_causal_reference(L):
    """One 8192-row prompt chunk (128 query tiles of 64 rows) and a chunk that
    continues another prompt from position 700, against a float64 causal
    reference over each sequence's whole key range."""
    import torch
    L.cdb_test_attention_prefill.argtypes = ([C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p] +
                                             [C.c_int] * 6 + [C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p])
    rng = np.random.default_rng(19)
    H, hd = 2, 128
    d = H * hd
    nsl, slot = 2, 1
    runs = [(0, 0, 8192), (1, 700, 300)]
    max_blocks = 512
    kv_blocks = 2 * max_blocks + 3
    perm = rng.permutation(kv_blocks)[: 2 * max_blocks].reshape(2, max_blocks)
    bt = torch.from_numpy(perm.astype(np.int32))
    pool = torch.from_numpy(rng.standard_normal((kv_blocks, nsl, 2, H, 16, hd)).astype(np.float32)).to(torch.bfloat16)
    row_slot = np.concatenate([np.full(n, sq, np.int32) for sq, p0, n in runs])
    row_pos = np.concatenate([np.arange(p0, p0 + n, dtype=np.int32) for sq, p0, n in runs])
    rows = len(row_pos)
    q = torch.from_numpy(rng.standard_normal((rows, d)).astype(np.float32)).to(torch.bfloat16)
    ref = torch.zeros(rows, d, dtype=torch.float64)
    r0 = 0
    for sq, p0, n in runs:
        T = p0 + n
        j = torch.arange(T)
        blk = bt[sq][j // 16].long()
        K = pool[blk, slot, 0, :, j % 16].double().transpose(0, 1)  # [H, T, hd]
        V = pool[blk, slot, 1, :, j % 16].double().transpose(0, 1)
        Q = q[r0:r0 + n].double().view(n, H, hd).transpose(0, 1)    # rows at positions p0..T-1
        s = Q @ K.transpose(1, 2) / np.sqrt(hd)                       # [H, n, T]
        s = s.masked_fill(j[None, None, :] > torch.arange(p0, T)[None, :, None], float("-inf"))
        ref[r0:r0 + n] = (torch.softmax(s, -1) @ V).transpose(0, 1).reshape(n, d)
        r0 += n
    out = torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda")
    scratch = torch.zeros(256 + 16 * (rows + 1), dtype=torch.uint8, device="cuda")
    dq, dp, dbt = q.cuda(), pool.cuda(), bt.cuda()
    rc = L.cdb_test_attention_prefill(dq.data_ptr(), rows, row_slot.ctypes.data, row_pos.ctypes.data, dp.data_ptr(),
                                      dbt.data_ptr(), max_blocks, kv_blocks, nsl, slot, H, hd, out.data_ptr(),
                                      scratch.data_ptr(), scratch.numel(), None)
    assert rc == 0, rc
    o = out.double().cpu()
    assert torch_finite(o)
    err = (o - ref).abs()
    assert (err <= 1e-2 * (1 + ref.abs())).all().item(), err.max().item()
