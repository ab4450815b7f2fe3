/*
 * cdb_testing.h — direct access to one of the library's kernels, for tests
 * and tuning.  Not needed to run the decode path (cdb.h).
 */
#ifndef CDB_TESTING_H
#define CDB_TESTING_H

#include <stddef.h>
#include <stdint.h>

typedef struct cdb_ctx cdb_ctx; /* opaque engine context (cdb.h) */

#ifdef __cplusplus
extern "C" {
#endif

/* The projection GEMM the core step uses: C = A[rows, K] . W[N, K]^T with
 * fp32 accumulation, bf16 A and W (row-major, device pointers).
 *   epi 0: Cf[r][c] = acc (fp32 out)      epi 1: Cf[r][c] += acc
 *   epi 2: Ct[r][c] = bf16(silu(A.W^T) * (A.W2^T))   (SwiGLU, bf16 out)
 *   tiling 0: tensor cores, decode tiles (64, 128 or 256 rows by the batch,
 *             split-K fixed by N and K;
 *             the fp32 partials are summed in split order by a second kernel,
 *             as the engine's consumer kernels do, then the epilogue applied)
 *   tiling 1: tensor cores, persistent prefill tiles (256 rows, 128 for
 *             SwiGLU, when rows > 128; else 128), no split
 *   tiling 2: the CUDA-core kernel (fp32 FMA), for comparison
 *   tiling 3: what engines of 384 or more slots run in decode: weights of
 *             fewer than 32 tiles of 128 features split K (at most 4 splits,
 *             fixed by N and K; partials folded as for tiling 0) on 64-, 128-
 *             or 256-row tiles; other weights run persistent tiles without
 *             split, 128, 192 or 256 rows, whichever needs the fewest waves
 *             of CTAs times operand bytes per tile (SwiGLU: above 128 only in
 *             one wave)
 * a_rows: rows allocated in A (>= rows).  ws: device memory of at least
 * cdb_test_gemm_ws_bytes() bytes: the kernel's status word, then the split-K
 * partials.  stream: cudaStream_t or NULL.
 * Synchronizes the stream; returns CDB_OK (0), CDB_ERR_ARG (-1) for an
 * unsupported shape, CDB_ERR_CUDA (-4), or CDB_ERR_DEVICE_BOUNDS (-5) when a
 * bounded wait inside the kernel expired. */
int cdb_test_gemm(int epi, int tiling, const void *A, int lda, int a_rows, const void *W, const void *W2,
                  int N, int K, int rows, float *Cf, void *Ct, int ldc, void *ws, size_t ws_bytes,
                  void *stream);
size_t cdb_test_gemm_ws_bytes(int N, int K, int rows, int tiling, int epi);

/* Decode attention over the depth-indexed paged KV cache, as in the core step
 * ("Depth-adaptive Inference of Looped Language Models via Continuous Depth
 * Batching", §4.2: row i at loop step r reads cached position j from step
 * min(r, e_j); Appendix A.1: 16-token pages through a block table).
 *   q        [rows][n_heads*head_dim], dtype elements (0 fp32, 1 bf16)
 *   slot, pos, depth  int32 [rows]: sequence slot, own position (keys
 *            0..pos are read), loop steps completed (this step is depth+1)
 *   kv_pool  [kv_blocks][n_kv_slots][2][n_heads][16][head_dim]: per block and
 *            slot, K then V, each head's 16 keys contiguous
 *   block_table int32 [*][max_blocks]; exit_table uint8 [kv_blocks][16]
 *   slot_base: cache slot of loop step 1 of this core layer
 *   split:   keys per split-KV partial (fixed, so results do not depend on
 *            the batch); out [rows][n_heads*head_dim], dtype elements
 *   scratch: device memory of cdb_test_attention_scratch_bytes() bytes for
 *            the split partials (any contents; every value read is written
 *            by the same call)
 * All pointers are device pointers owned by the caller.  Synchronizes the
 * stream.  Returns CDB_OK, CDB_ERR_ARG (bad shape or scratch too small),
 * CDB_ERR_CUDA, or CDB_ERR_DEVICE_BOUNDS (a page or depth out of range). */
int cdb_test_attention(const void *q, int rows, const int32_t *slot, const int32_t *pos,
                       const int32_t *depth, const void *kv_pool, const int32_t *block_table,
                       int max_blocks, const uint8_t *exit_table, int kv_blocks, int n_kv_slots,
                       int slot_base, int n_heads, int head_dim, int dtype, int split, int max_ctx,
                       void *out, void *scratch, size_t scratch_bytes, void *stream);
size_t cdb_test_attention_scratch_bytes(int rows, int n_heads, int head_dim, int split, int max_ctx);

/* The attention the engine runs: the same computation as cdb_test_attention
 * when every key of row i is read from one slot, slot_base + depth[i] (loop
 * step depth[i] + 1).  The engine keeps that true by filling exit gaps when a
 * token leaves the loop (its last computed K and V are copied into the slots
 * of the deeper steps it skipped), which makes the slot of loop step r hold
 * the entry of step min(r, e_j) for every cached position j.  Same arguments
 * as cdb_test_attention without exit_table; the same pool layout; keys past
 * a row's position are never used even when the pool holds NaN there. */
int cdb_test_attention_uniform(const void *q, int rows, const int32_t *slot, const int32_t *pos,
                               const int32_t *depth, const void *kv_pool, const int32_t *block_table,
                               int max_blocks, int kv_blocks, int n_kv_slots, int slot_base, int n_heads,
                               int head_dim, int dtype, int split, int max_ctx, void *out, void *scratch,
                               size_t scratch_bytes, void *stream);

/* The causal prefill attention of a prompt chunk (bf16 only, head_dim 32, 64,
 * 96 or 128): row i (query q[i], sequence slot row_slot[i], position
 * row_pos[i]) attends to positions 0..row_pos[i] of its sequence, every key
 * read from KV slot `slot`.  Rows of one sequence must come as runs of
 * consecutive positions (how the scheduler packs a chunk); the library cuts
 * them into query tiles of up to 64 rows.  row_slot and row_pos are HOST
 * arrays; q, kv_pool (layout of cdb_test_attention), block_table and out are
 * device pointers.  scratch: device memory of at least 256 + 16 * (rows + 1)
 * bytes.  Returns CDB_ERR_ARG for an unsupported shape (nothing launched). */
int cdb_test_attention_prefill(const void *q, int rows, const int32_t *row_slot, const int32_t *row_pos,
                               const void *kv_pool, const int32_t *block_table, int max_blocks, int kv_blocks,
                               int n_kv_slots, int slot, int n_heads, int head_dim, void *out, void *scratch,
                               size_t scratch_bytes, void *stream);

/* The same decode attention for callers that must not allocate device memory
 * (for example a plugin whose host program's memory manager owns all device
 * memory, or a latency-critical path that cannot take an allocation's implicit
 * synchronisation).  The paper has no counterpart to this entry point; it is a
 * deployment convenience of this library.
 * Arguments and results are those of cdb_test_attention without the scratch
 * arguments: the split partials and the status word live in a 16 MiB array
 * built into the library, which every GPU that loads the library keeps
 * reserved until the process exits.  A call whose partials
 * (rows * n_heads * ceil(max_ctx / split) * (head_dim + 2) floats, plus 256
 * bytes) exceed 16 MiB is rejected with CDB_ERR_ARG before any GPU work.
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  With CUDA's lazy module loading (the default) the library's device
 * code, and with it the array, is loaded onto a device the first time any
 * kernel or symbol of this library is used there; if that is this call, the
 * driver takes the array's memory then.  A caller that must keep every call
 * free of that cost makes one warm-up call on each device at set-up (or runs
 * with CUDA_MODULE_LOADING=EAGER).  All calls share the one array and it keeps
 * the previous call's contents, so calls that overlap on the GPU (other
 * streams, other host threads) race; issue them one after another.  A row
 * whose position lies past max_ctx's block table or split partials is skipped
 * and the call returns CDB_ERR_DEVICE_BOUNDS.  Synchronizes the stream. */
/* The KV cache inside an engine's arena, so that tests can read back what the
 * engine cached ("Depth-adaptive Inference of Looped Language Models via
 * Continuous Depth Batching", §4.2: one slot per core layer and loop step).
 * *pool: device pointer to [kv_blocks][n_kv_slots][2][n_heads][16][head_dim]
 * elements of the model's dtype (K then V per block and slot, each head's 16
 * positions contiguous); core layer l, loop step r lives in slot
 * n_prelude + l * s + min(r, s) - 1 (s the model's kv_slots, r_max for the
 * depth-indexed cache).  A sequence's i-th block of 16 positions is the pool
 * block its block table names; the engine hands out free blocks in increasing
 * order, so the first sequence admitted to a new engine holds blocks 0, 1, ...
 * The memory belongs to the caller's arena.  Returns CDB_OK or CDB_ERR_ARG. */
int cdb_test_kv_pool(const cdb_ctx *ctx, void **pool, int *kv_blocks, int *n_kv_slots);

int cdb_attention_noalloc(const void *q, int rows, const int32_t *slot, const int32_t *pos,
                          const int32_t *depth, const void *kv_pool, const int32_t *block_table,
                          int max_blocks, const uint8_t *exit_table, int kv_blocks, int n_kv_slots,
                          int slot_base, int n_heads, int head_dim, int dtype, int split, int max_ctx,
                          void *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* CDB_TESTING_H */
