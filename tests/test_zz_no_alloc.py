"""The allocation-free decode attention entry point (cdb_attention_noalloc).

It exists for callers that must not allocate device memory, such as a plugin
whose host program owns all device memory or a latency-critical path that
cannot absorb an allocation's synchronisation; its scratch lives in a 16 MiB
array built into the library.  This file checks, through the C ABI, that two
calls in a row (different shapes and dtypes, so the second call starts from
the first call's leftover scratch) each equal cdb_test_attention, the same
kernels with the same split order run on caller-provided scratch, bit for
bit; that a request too large for the built-in scratch is refused; and that a
row positioned past the block table is skipped and reported.
Collected last so a failure here cannot stop the other GPU tests.
"""

import ctypes as C

import pytest

from tests.test_gpu_attention import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.build import build
    build()
    lib = binding.lib()
    common = [C.c_void_p, C.c_int] + [C.c_void_p] * 5 + [C.c_int, C.c_void_p] + [C.c_int] * 8
    lib.cdb_test_attention.argtypes = common + [C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
    lib.cdb_test_attention_scratch_bytes.restype = C.c_size_t
    lib.cdb_test_attention_scratch_bytes.argtypes = [C.c_int] * 5
    lib.cdb_attention_noalloc.argtypes = common + [C.c_void_p, C.c_void_p]
    return lib


def device_inputs(cs):
    import torch
    d = {k: cs[k].cuda() for k in ("pool", "bt", "etab", "q")}
    for k in ("slot", "pos", "depth"):
        d[k] = torch.from_numpy(cs[k]).cuda()
    return d


def args(cs, d, split):
    return [d["q"].data_ptr(), len(cs["pos"]), d["slot"].data_ptr(), d["pos"].data_ptr(), d["depth"].data_ptr(),
            d["pool"].data_ptr(), d["bt"].data_ptr(), cs["max_blocks"], d["etab"].data_ptr(), cs["kv_blocks"],
            cs["nsl"], cs["base"], cs["H"], cs["hd"], cs["dtype"], split, cs["max_ctx"]]


def with_caller_scratch(L, cs, d, split):
    import torch
    out = torch.zeros(len(cs["pos"]), cs["H"] * cs["hd"], dtype=cs["q"].dtype, device="cuda")
    nb = L.cdb_test_attention_scratch_bytes(len(cs["pos"]), cs["H"], cs["hd"], split, cs["max_ctx"])
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    assert L.cdb_test_attention(*args(cs, d, split), out.data_ptr(), scratch.data_ptr(), nb, None) == 0
    return out


def without_allocation(L, cs, d, split):
    import torch
    out = torch.full((len(cs["pos"]), cs["H"] * cs["hd"]), float("nan"), dtype=cs["q"].dtype, device="cuda")
    assert L.cdb_attention_noalloc(*args(cs, d, split), out.data_ptr(), None) == 0
    return out


def test_two_calls_in_a_row_match_the_caller_scratch_entry_point(L):
    import torch
    first = make_case(1, 16, 128, rows=9, max_ctx=1300, seed=21)   # bf16, 6 splits of 256
    second = make_case(0, 4, 64, rows=5, max_ctx=200, seed=22)     # fp32, 13 splits of 16
    d1, d2 = device_inputs(first), device_inputs(second)
    ref1 = with_caller_scratch(L, first, d1, 256)
    ref2 = with_caller_scratch(L, second, d2, 16)
    got1 = without_allocation(L, first, d1, 256)
    got2 = without_allocation(L, second, d2, 16)
    assert torch.equal(got1, ref1)
    assert torch.equal(got2, ref2)


def test_request_beyond_the_built_in_scratch_is_refused(L):
    cs = make_case(1, 16, 128, rows=2, max_ctx=64, seed=23)
    d = device_inputs(cs)
    a = args(cs, d, 16)
    a[1] = 4096          # rows: 4096 * 16 heads * 4 splits * 130 floats > 16 MiB
    a[16] = 64
    assert L.cdb_attention_noalloc(*a, d["q"].data_ptr(), None) == -1


def test_row_past_the_block_table_is_reported(L):
    """pos == max_ctx with max_ctx a multiple of 16 and of the split: the row's
    page is past its block-table row and its last split past the partials, so
    the kernels skip it and the call reports CDB_ERR_DEVICE_BOUNDS (-5)."""
    import torch
    cs = make_case(1, 4, 64, rows=3, max_ctx=512, seed=24)
    cs["pos"][2] = cs["max_ctx"]
    d = device_inputs(cs)
    out = torch.zeros(3, cs["H"] * cs["hd"], dtype=cs["q"].dtype, device="cuda")
    assert L.cdb_attention_noalloc(*args(cs, d, 256), out.data_ptr(), None) == -5
    nb = L.cdb_test_attention_scratch_bytes(3, cs["H"], cs["hd"], 256, cs["max_ctx"])
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    assert L.cdb_test_attention(*args(cs, d, 256), out.data_ptr(), scratch.data_ptr(), nb, None) == -5
    # The valid rows are still computed, and the next call starts clean.
    cs["pos"][2] = cs["max_ctx"] - 1
    d = device_inputs(cs)
    ref = with_caller_scratch(L, cs, d, 256)
    assert torch.equal(without_allocation(L, cs, d, 256), ref)
