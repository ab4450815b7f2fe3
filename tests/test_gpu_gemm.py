"""Tensor-core projection GEMM (include/cdb_testing.h) against a float64 product.

Checks every epilogue (store, residual add, SwiGLU), every tensor-core tiling
(decode: 64-, 128- or 256-row tiles with split-K fixed by the weight shape;
prefill: 128- and 256-row tiles; wide decode: 128-, 192- or 256-row tiles
by the batch, split-K on 64- to 256-row tiles for narrow weights),
ragged N and K tails, the split-K shapes of the Ouro-shaped core, agreement
with the CUDA-core kernel, and that a row's result does not depend on how
many other rows are in the batch (bit-exact).
"""

import ctypes as C

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

TOL = 1e-4  # fp32 accumulation of bf16 products vs a float64 reference, outputs O(1)


@pytest.fixture(scope="module")
def L():
    from continuous_depth_batching_gb300 import binding
    from continuous_depth_batching_gb300.build import build
    build()
    lib = binding.lib()
    lib.cdb_test_gemm.argtypes = [C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                                  C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                  C.c_size_t, C.c_void_p]
    lib.cdb_test_gemm_ws_bytes.restype = C.c_size_t
    lib.cdb_test_gemm_ws_bytes.argtypes = [C.c_int] * 5
    return lib


def run(L, epi, tiling, A, W, W2=None, C0=None, a_rows=None):
    import torch
    rows, K = A.shape
    N = W.shape[0]
    a_rows = a_rows or rows
    Abuf = torch.zeros(a_rows, K, dtype=torch.bfloat16, device="cuda")
    Abuf[:rows] = A
    ws_bytes = L.cdb_test_gemm_ws_bytes(N, K, rows, tiling, epi)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    Cf = (C0.clone() if C0 is not None else torch.zeros(rows, N, dtype=torch.float32, device="cuda"))
    Ct = torch.zeros(rows, N, dtype=torch.bfloat16, device="cuda")
    rc = L.cdb_test_gemm(epi, tiling, Abuf.data_ptr(), K, a_rows, W.data_ptr(),
                         W2.data_ptr() if W2 is not None else None, N, K, rows,
                         Cf.data_ptr(), Ct.data_ptr(), N, ws.data_ptr(), ws_bytes, None)
    assert rc == 0, rc
    return Cf, Ct


def rnd(*shape, std=1.0, seed=0):
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).cuda()


SHAPES = [(5, 256, 192), (7, 200, 200), (64, 6144, 2048), (64, 2048, 5632), (33, 384, 1000), (300, 384, 256),
          (100, 6144, 2048), (200, 2048, 5632), (500, 6144, 320), (700, 6144, 200), (333, 1024, 1000)]


@pytest.mark.parametrize("rows,N,K", SHAPES)
@pytest.mark.parametrize("tiling", [0, 1, 3])
def test_store_and_residual(L, rows, N, K, tiling):
    import torch
    A = rnd(rows, K, seed=1)
    W = rnd(N, K, std=1.0 / np.sqrt(K), seed=2)
    ref = A.double() @ W.double().T
    Cf, _ = run(L, 0, tiling, A, W)
    assert (Cf.double() - ref).abs().max().item() <= TOL
    C0 = torch.randn(rows, N, device="cuda")
    Cr, _ = run(L, 1, tiling, A, W, C0=C0)
    assert (Cr.double() - (ref + C0.double())).abs().max().item() <= TOL


@pytest.mark.parametrize("rows,N,K", [(5, 256, 192), (64, 5632, 2048), (200, 300, 128), (400, 5632, 256),
                                      (700, 5632, 192), (2000, 5632, 128), (200, 512, 1024)])
@pytest.mark.parametrize("tiling", [0, 1, 3])
def test_swiglu(L, rows, N, K, tiling):
    import torch
    A = rnd(rows, K, seed=3)
    W = rnd(N, K, std=1.0 / np.sqrt(K), seed=4)
    W2 = rnd(N, K, std=1.0 / np.sqrt(K), seed=5)
    g = A.double() @ W.double().T
    u = A.double() @ W2.double().T
    ref = g / (1 + torch.exp(-g)) * u
    _, Ct = run(L, 2, tiling, A, W, W2)
    # bf16 output: one round-to-nearest (half an ulp, 2^-8 relative) plus fp32 error
    assert ((Ct.double() - ref).abs() <= ref.abs() * 2.0 ** -8 + 1e-4).all().item()


def test_matches_cuda_core_kernel(L):
    A = rnd(48, 1024, seed=6)
    W = rnd(640, 1024, std=0.03, seed=7)
    a, _ = run(L, 0, 0, A, W)
    b, _ = run(L, 0, 2, A, W)
    assert (a - b).abs().max().item() <= TOL


@pytest.mark.parametrize("N,K", [(6144, 2048), (2048, 5632), (49152, 2048)])
@pytest.mark.parametrize("tiling", [0, 3])
def test_row_result_independent_of_batch(L, N, K, tiling):
    # Decode tiling: 200 rows run on 256-row tiles, 1-64 rows on 64-row tiles
    # and 100 on 128-row tiles; the split count is the same for all of them.
    # Wide tiling, N = 6144 (48 feature tiles, one wave): 700 rows on 256-row
    # tiles, 500 on 192-row tiles, up to 384 on 128-row tiles; N = 49152
    # (several waves): 256 rows at 500 and 700, 192 at 300, 128 up to 100;
    # N = 2048 (narrow, four K splits): 256-row tiles at 500, 128 at 700.
    rows = 200 if tiling == 0 else 700
    A = rnd(rows, K, seed=8)
    W = rnd(N, K, std=1.0 / np.sqrt(K), seed=9)
    full, _ = run(L, 0, tiling, A, W, a_rows=rows)
    for r in (1, 17, 64, 100) + ((300, 500) if tiling == 3 else ()):
        part, _ = run(L, 0, tiling, A[:r].contiguous(), W, a_rows=rows)
        assert (part == full[:r]).all().item(), "row results must not depend on batch size"


def test_swiglu_row_result_independent_of_batch(L):
    # Wide tiling, N = 5632 (44 feature tiles): 700 rows run in one wave of
    # 256-row tiles, 400 of 192-row tiles, up to 384 rows of 128-row tiles
    # (one accumulator buffer per CTA each time).
    K, N, rows = 2048, 5632, 700
    A = rnd(rows, K, seed=10)
    W = rnd(N, K, std=1.0 / np.sqrt(K), seed=11)
    W2 = rnd(N, K, std=1.0 / np.sqrt(K), seed=12)
    _, full = run(L, 2, 3, A, W, W2, a_rows=rows)
    for r in (1, 100, 300, 400):
        _, part = run(L, 2, 3, A[:r].contiguous(), W, W2, a_rows=rows)
        assert (part == full[:r]).all().item(), "row results must not depend on batch size"
