/*
 * cdb.h — continuous depth batching (CDB) for depth-adaptive looped LMs on one GB300.
 *
 * C ABI of the library.  The operations follow "Depth-adaptive Inference of
 * Looped Language Models via Continuous Depth Batching" (arxiv 2608.09444v2):
 *
 *   - §2 Problem Setup: a looped LM has a prelude, a shared recurrent core run
 *     r_t <= r_max times per token, and a coda; r_t is decided per token.
 *   - §4.1 Stage-wise Scheduling and Appendix A.3 Algorithms 1 and 2: four
 *     stage queues (prompts awaiting prefill, tokens awaiting the prelude,
 *     recurrent items, exited tokens awaiting the coda); no-refill and refill
 *     modes; minimum coda batch size K.
 *   - §4.2 Depth-aware KV Cache: one KV slot per (core layer, loop step).  An
 *     earlier token j is read at depth min(d, e_j), its last written state, so
 *     the slots an early exit leaves empty are never read.
 *   - §4.3 Asynchronous Scheduling: the lookahead gate; the gate after step d
 *     decides whether the token takes part in step d+2 (r_min = 2).
 *   - Appendix A.1/A.2 and Table 1: chunked prefill of at most M tokens at full
 *     depth, at most W active sequences, admission after S free slots, a paged
 *     KV cache of 16-token blocks with headroom rho_KV, no preemption.
 *
 * Threading: a context is used by one host thread at a time.
 * Memory: every device buffer the library uses is carved from one caller-owned
 * device arena (cdb_sched_cfg.arena); weights are borrowed device pointers.
 * The library never calls cudaMalloc during steps.
 * Errors: functions return a cdb_status.  Negative values are errors; the
 * message is available from cdb_last_error().  After CDB_ERR_CUDA or
 * CDB_ERR_DEVICE_BOUNDS the context must be freed; after other errors it stays
 * usable.
 */
#ifndef CDB_H
#define CDB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CDB_MAX_DEPTH 64 /* largest r_max the library accepts */

typedef struct cdb_ctx cdb_ctx; /* opaque */

typedef enum {
  CDB_OK = 0,
  CDB_IDLE = 1,  /* step_boundary: the next stage is a core step (or nothing to do yet) */
  CDB_DONE = 2,  /* every admitted sequence has finished */
  CDB_ERR_ARG = -1,
  CDB_ERR_ARENA = -2,   /* arena too small or misaligned */
  CDB_ERR_KV_FULL = -3, /* a sequence can never fit in the KV pool (no preemption) */
  CDB_ERR_CUDA = -4,
  CDB_ERR_DEVICE_BOUNDS = -5, /* a kernel's bounds check recorded a bad index */
  CDB_ERR_TIMEOUT = -6,
  CDB_ERR_STATE = -7
} cdb_status;

typedef enum { CDB_MODE_REFILL = 0, CDB_MODE_NO_REFILL = 1, CDB_MODE_FIXED_DEPTH = 2 } cdb_mode;
typedef enum { CDB_FP32 = 0, CDB_BF16 = 1 } cdb_dtype;

/* Stage kinds reported in cdb_step_info / trace rows (the rows of Tables 2-3). */
typedef enum {
  CDB_STAGE_NONE = 0,
  CDB_STAGE_PREFILL = 1,
  CDB_STAGE_PRELUDE = 2,
  CDB_STAGE_LOOP = 3,
  CDB_STAGE_CODA = 4
} cdb_stage;

/* Exit policies (gate_kind). */
typedef enum {
  CDB_GATE_PROBE = 0,       /* z = gate_w . rmsnorm(h) + gate_bias; exit when z > gate_threshold */
  CDB_GATE_CONVERGENCE = 1  /* c = ||s_d - s_{d-1}|| / ||s_d||; exit when c < gate_threshold */
} cdb_gate_kind;

/* Model shape.  A pre-norm block is RMSNorm -> QKV (RoPE on q,k) -> causal
 * attention -> O-proj + residual -> RMSNorm -> SwiGLU MLP + residual.  The
 * exit gate is z = gate_w . rmsnorm(h) + gate_bias (unit gain) on the core
 * state after each loop step; a token exits when z > gate_threshold (the
 * logit of the probability threshold q).  has_adapter: every loop step starts
 * from x = adapter . [e; s_{d-1}] (adapter [d_model, 2 d_model]) with e the
 * prelude output and s_0 = 0, as in Huginn-shaped models; otherwise s_0 = e. */
typedef struct {
  int vocab, d_model, n_heads, head_dim, ffn;
  int n_prelude, n_core, n_coda;
  int r_max, r_min; /* 2 <= r_min <= r_max <= CDB_MAX_DEPTH */
  int has_adapter;
  int dtype;        /* cdb_dtype: weights, activations and KV cache */
  float rms_eps, rope_theta;
  float gate_threshold, gate_bias;
  /* KV slots per token of each recurrent-core layer, s (App. E.1): 0 or
   * r_max = the depth-indexed cache (loop step d writes and reads slot d);
   * 1 = single-slot sharing (every step overwrites one slot); 2 =
   * first-then-shared (step 1 keeps a private slot, steps >= 2 share the
   * second); in general step d uses slot min(d, s).  A prompt split across
   * prefill chunks then reads its earlier chunks at their last loop step. */
  int kv_slots;
  /* cdb_gate_kind.  CDB_GATE_CONVERGENCE is Huginn's training-free exit
   * ("Depth-adaptive Inference of Looped Language Models via Continuous Depth
   * Batching", App. E.2): after loop step d, c_d = ||s_d - s_{d-1}||_2 /
   * ||s_d||_2 over the fp32 core state, s_{d-1} being the state that entered
   * step d (s_0 = 0 with an adapter, else the prelude output); the token
   * exits when c_d < gate_threshold (equality does not exit; c is +inf when
   * s_d = 0).  gate_w and gate_bias are unused (gate_w may be NULL) and
   * r_min must be >= 3: the lookahead decision after step d takes effect at
   * d + 2 and the first comparison that does not involve s_0 is after step
   * 2.  gate_logits traces then hold c_d. */
  int gate_kind;
} cdb_model_desc;

/* One transformer block; device pointers, row-major [out, in] like nn.Linear.
 * attn_norm, mlp_norm [d]; wqkv [3d, d] (q rows, then k, then v); wo [d, d];
 * wg, wu [ffn, d]; wd [d, ffn].  Element type is the model dtype. */
typedef struct {
  const void *attn_norm, *wqkv, *wo, *mlp_norm, *wg, *wu, *wd;
} cdb_layer_weights;

/* Device pointers, BORROWED until cdb_free.  embed, lm_head [vocab, d];
 * final_norm [d]; gate_w [d]; adapter [d, 2d] or NULL.  The three layer
 * arrays are HOST arrays of n_prelude / n_core / n_coda entries (copied). */
typedef struct {
  const void *embed, *lm_head, *final_norm, *gate_w, *adapter;
  const cdb_layer_weights *prelude, *core, *coda;
} cdb_weights;

typedef struct {
  int mode;          /* cdb_mode */
  int W;             /* max active sequences = max core batch */
  int M;             /* max prompt tokens per prefill batch */
  int S;             /* min free slots before admitting (0: max(1, W/8)) */
  int K;             /* min coda batch (refill mode) */
  int kv_blocks;     /* physical 16-token blocks in the KV pool */
  float kv_headroom; /* rho_KV: fraction of the pool kept free at admission */
  int max_ctx;       /* longest prompt_len + max_new_tokens - 1 accepted */
  int max_new_cap;   /* largest max_new_tokens accepted */
  int trace_tokens;  /* per sequence, keep logits and coda input of the first N tokens */
  int trace_gate;    /* 1: keep every gate logit z_d of every decode forward */
  void *arena;       /* device memory, >= cdb_arena_bytes(); 256-byte aligned */
  size_t arena_bytes;
  void *compute_stream; /* cudaStream_t (NULL: legacy default stream) */
  void *prep_stream;    /* cudaStream_t for host<->device copies of scheduling data */
  int attn_split;    /* keys per split-KV partial in decode attention, a multiple of 16 (0: 128) */
} cdb_sched_cfg;

/* Per-call report.  For a boundary call that ran two stages (coda or prefill,
 * then prelude) the second stage is in stage2/batch2. */
typedef struct {
  int stage, batch, prefill_tokens;
  int stage2, batch2;
  int exits;                     /* loop: tokens leaving the core after this step */
  int q_r, q_c, q_p, q_d;        /* queue sizes after the call */
  int depth_hist[CDB_MAX_DEPTH]; /* loop: depth_hist[i] tokens ran loop step i+1 */
  int64_t step_index;            /* loop steps issued so far, this one included */
  int new_tokens;                /* tokens generated by this call (coda rows + prompts completed) */
  int64_t ctx, ctx2;             /* context entries of stage / stage2: the sum over its rows of
                                    (position + 1), the keys their attention reads per layer */
} cdb_step_info;

/* One finished sequence.  The caller sets the pointers before cdb_drain; the
 * library fills them.  tokens [max_new_tokens]; exit_depths
 * [max_new_tokens-1] (depth of each adaptive decode forward); gate_logits
 * (nullable, needs trace_gate) [(max_new_tokens-1) * r_max], z after step d of
 * forward t at (t-1)*r_max + d-1, NaN where that step did not run; logits
 * (nullable) [trace_tokens * vocab]; hidden (nullable) [trace_tokens * d] is
 * the core state entering the coda.  Buffers must hold max_new_cap entries. */
typedef struct {
  int64_t seq_id;
  int n_tokens;
  int32_t *tokens;
  int8_t *exit_depths;
  float *gate_logits;
  float *logits;
  float *hidden;
} cdb_result;

/* Device bytes cdb_init needs for this model and configuration. */
size_t cdb_arena_bytes(const cdb_model_desc *m, const cdb_sched_cfg *c);

/* KV-cache bytes per token of the depth-indexed layout: (l0 + lr * r_max)
 * entries of K and V, d_model elements each (App. E.1 and Table 4). */
size_t cdb_kv_bytes_per_token(const cdb_model_desc *m);

/* Validate, carve the arena, fill the KV pool with NaN (so a read of an exit
 * gap would poison the output) and build the RoPE table.  Synchronous. */
int cdb_init(const cdb_model_desc *m, const cdb_weights *w, const cdb_sched_cfg *c,
             cdb_ctx **out);

/* Queue one request (host-only; prompt and force tables are copied).
 * max_new_tokens counts the first token, which prefill produces.
 * force_exit (nullable) [max_new_tokens-1]: 0 = live gate, else the exit depth
 * in [r_min, r_max] of that decode forward (replay, App. C.2).
 * force_token (nullable) [max_new_tokens]: -1 = greedy argmax, else the id. */
int cdb_admit(cdb_ctx *ctx, int64_t seq_id, const int32_t *prompt, int prompt_len,
              int max_new_tokens, const int8_t *force_exit, const int32_t *force_token);

/* Run the next non-core stage the mode's priority rule selects (Alg. 1 / 2):
 * coda (+prelude), prefill (+prelude in refill mode), or a cohort prelude.
 * Returns CDB_IDLE when the next stage is a core step, CDB_DONE when all
 * admitted sequences have finished.  Enqueues GPU work and returns. */
int cdb_step_boundary(cdb_ctx *ctx, cdb_step_info *info);

/* One recurrent-core loop step over every token in the recurrent queue:
 * batch re-formation, n_core shared blocks at each token's own depth, exit
 * gate, compaction of continuing tokens and hand-off of exits to the coda
 * queue.  CDB_IDLE if the queue is empty.  Enqueues GPU work and returns;
 * exit counts in info come from the previous step's lookahead flags. */
int cdb_step_core(cdb_ctx *ctx, cdb_step_info *info);

/* Copy up to cap finished sequences (finish order) into buf; *n_out set.
 * Waits for the device copies of every finished sequence's results. */
int cdb_drain(cdb_ctx *ctx, cdb_result *buf, int cap, int *n_out);

/* cdb_drain without waiting: only sequences whose results have already
 * reached host memory are returned (a sequence not ready now comes back from
 * a later poll or drain), so an online driver can collect finished requests
 * between steps without stalling the device queue.  Each finished sequence is
 * returned exactly once by poll and drain together.  Unlike cdb_drain it does
 * not read the device status word (that needs a stream synchronization);
 * cdb_drain and cdb_sync report a failed bounds check. */
int cdb_poll(cdb_ctx *ctx, cdb_result *buf, int cap, int *n_out);

/* Block until all enqueued work has finished and check device-side status. */
int cdb_sync(cdb_ctx *ctx);

void cdb_free(cdb_ctx *ctx);
const char *cdb_last_error(const cdb_ctx *ctx);

/* Kernel timing.  When enabled, every launch of the timed kernel classes is
 * bracketed by CUDA events on the compute stream; cdb_profile_read
 * synchronizes, returns per class the launch count, summed device time and
 * the algorithmic bytes and FLOPs of those launches (bytes each launch must
 * move at least once: weights, KV rows read, activations in and out), and
 * resets the counters.  Classes: "attention" (split-KV decode attention plus
 * its combine), "gemm" (projections of decode-sized batches), "prefill_gemm"
 * (projections of prefill chunks), "prefill_attention", "rowwise"
 * (RMSNorm with the fold of pending split-K partials, RoPE + KV write, the
 * SwiGLU combine, the residual fold). */
typedef struct {
  char name[32];
  int64_t launches;
  double ms, bytes, flops;
} cdb_kernel_stat;
/* on: 0 off, 1 launches of every stage, 2 launches of core steps only. */
int cdb_profile_enable(cdb_ctx *ctx, int on);
int cdb_profile_read(cdb_ctx *ctx, cdb_kernel_stat *out, int cap, int *n_out);

/* Step-delta timing of a kernel class inside the recurrent-core step: while
 * set, every core step launches the class's kernels twice (class 0 decode
 * attention with its combine, 1 projection GEMMs, 3 RoPE + KV write and the
 * SwiGLU combine; -1 stops).  The repeated launches write the same values
 * again (an in-place residual GEMM epilogue is never repeated), so results are
 * unchanged; the difference between the time of such a step and of a plain
 * one is the class's live cost with programmatic dependent launch in effect.
 * For measurement only: the extra launches cost time.  CDB_ERR_ARG for other
 * classes. */
int cdb_profile_repeat(cdb_ctx *ctx, int cls);

/* Kernel launches issued by the library in this process, all contexts. */
int64_t cdb_kernel_launches(void);

/* Host<->device bytes this context has copied so far: prompts, scheduling
 * tables and lists (h2d); lookahead flags, results and status words (d2h). */
int cdb_io_bytes(const cdb_ctx *ctx, int64_t *h2d, int64_t *d2h);

/* Scheduling trace: one row per executed stage (the columns of Tables 2-3).
 * Rows are kept only while trace recording is on. */
typedef struct {
  int stage, batch, prefill_tokens, exits;
  int q_r, q_c, q_p, q_d;
  int depth_hist[CDB_MAX_DEPTH];
} cdb_trace_row;
int cdb_trace_enable(cdb_ctx *ctx, int on);
int cdb_trace_read(cdb_ctx *ctx, cdb_trace_row *rows, int cap, int *n_out);

#ifdef __cplusplus
}
#endif
#endif /* CDB_H */
