/*
 * cdb_testing.h — direct access to one of the library's kernels, for tests
 * and tuning.  Not needed to run the decode path (cdb.h).
 */
#ifndef CDB_TESTING_H
#define CDB_TESTING_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The projection GEMM the core step uses: C = A[rows, K] . W[N, K]^T with
 * fp32 accumulation, bf16 A and W (row-major, device pointers).
 *   epi 0: Cf[r][c] = acc (fp32 out)      epi 1: Cf[r][c] += acc
 *   epi 2: Ct[r][c] = bf16(silu(A.W^T) * (A.W2^T))   (SwiGLU, bf16 out)
 *   tiling 0: tensor cores, decode tiles (64 rows, split-K fixed by N and K)
 *   tiling 1: tensor cores, prefill tiles (128 rows, no split)
 *   tiling 2: the CUDA-core kernel (fp32 FMA), for comparison
 * a_rows: rows allocated in A (>= rows).  ws: zero-filled device memory of at
 * least cdb_test_gemm_ws_bytes() bytes that receives the kernel's status
 * word.  stream: cudaStream_t or NULL.
 * Synchronizes the stream; returns CDB_OK (0), CDB_ERR_ARG (-1) for an
 * unsupported shape, CDB_ERR_CUDA (-4), or CDB_ERR_DEVICE_BOUNDS (-5) when a
 * bounded wait inside the kernel expired. */
int cdb_test_gemm(int epi, int tiling, const void *A, int lda, int a_rows, const void *W, const void *W2,
                  int N, int K, int rows, float *Cf, void *Ct, int ldc, void *ws, size_t ws_bytes,
                  void *stream);
size_t cdb_test_gemm_ws_bytes(int N, int K, int rows, int tiling, int epi);

#ifdef __cplusplus
}
#endif
#endif /* CDB_TESTING_H */
