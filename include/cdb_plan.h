/*
 * cdb_plan.h — predicted job latency and the choice of scheduling mode.
 *
 * "Depth-adaptive Inference of Looped Language Models via Continuous Depth
 * Batching", §5 "Recurrent batch size and latency": one recurrent step costs
 * t = delta + gamma * N_b + alpha * N_c (delta the weight reload, gamma the
 * per-token compute, alpha the KV streaming per cached entry); refill pays
 * off while the step is memory bound and matters less once it is compute
 * bound (§5, §6.2 "When is refill most effective?"); batching the coda with
 * a minimum batch K trades coda efficiency against core batch size (§6.4,
 * Fig. 7).  The summary page's claim that a roofline model picks refill or
 * no-refill for the load and hardware is what cdb_select_schedule does.
 *
 * Every stage the scheduler runs is costed with the same linear form,
 * delta + gamma * rows + alpha * ctx, where rows is the number of tokens in
 * the stage (prompt tokens for prefill) and ctx the sum over those rows of
 * (position + 1), the cached entries each row's attention reads per layer.
 * A job is predicted by running the host scheduler of cdb.h (the same code,
 * not a model of it) with the job's recorded exit depths replayed (App. C.2)
 * and adding the stage costs: the GPU runs stages one after another, and the
 * lookahead keeps the host off the critical path (§4.3).
 *
 * Host only; no GPU is touched.  Errors: negative cdb_status values.
 */
#ifndef CDB_PLAN_H
#define CDB_PLAN_H

#include <stdint.h>

#include "cdb.h"

#ifdef __cplusplus
extern "C" {
#endif

/* seconds = delta + gamma * rows + alpha * ctx.  All >= 0. */
typedef struct {
  double delta, gamma, alpha;
} cdb_stage_cost;

typedef struct {
  cdb_stage_cost prefill, prelude, core, coda;
} cdb_latency_model;

/* An offline job (every request known up front, §6.2).  HOST arrays,
 * borrowed for the call: prompt_len[n_seqs], gen_len[n_seqs] (tokens
 * generated, the first by prefill) and exit_depths, the concatenation over
 * requests of gen_len[i] - 1 depths in [r_min, r_max] (ignored for fixed
 * depth).  The scheduler limits are those of cdb_sched_cfg; S = 0 selects
 * max(1, W/8). */
typedef struct {
  int n_seqs;
  const int32_t *prompt_len;
  const int32_t *gen_len;
  const int8_t *exit_depths;
  int W, M, S, r_max, r_min, kv_blocks;
  float kv_headroom;
  int max_ctx, max_new_cap;
} cdb_job;

typedef struct {
  double seconds;  /* predicted GPU time of the whole job */
  double prefill_seconds, prelude_seconds, core_seconds, coda_seconds;
  int64_t prefill_stages, prelude_stages, core_steps, coda_stages;
  int64_t tokens;             /* tokens generated */
  int64_t core_token_steps;   /* sum over core steps of the batch size */
  double mean_core_batch, mean_coda_batch;
} cdb_prediction;

/* Predicted latency of `job` under `mode` (cdb_mode) with minimum coda batch
 * K (refill only; pass 1 otherwise).  Returns CDB_OK, CDB_ERR_ARG (bad job,
 * K < 1, a negative cost) or the scheduler's error (CDB_ERR_KV_FULL when a
 * request cannot fit kv_blocks). */
int cdb_predict_job(const cdb_job *job, int mode, int K, const cdb_latency_model *lm,
                    cdb_prediction *out);

/* The latency model the roofline gives for a model on a GPU with HBM
 * bandwidth hbm_gbps (GB/s) and tensor throughput tensor_tflops (TFLOP/s):
 * delta = weight bytes of the stage / bandwidth + launch_s per kernel the
 * stage launches; gamma = max(2 * parameters / tensor rate, bytes written
 * per row / bandwidth); alpha = K and V bytes of one cached entry over the
 * stage's layers / bandwidth (for prefill: the attention FLOPs of one
 * (query, key) pair over every layer application / tensor rate).  Prefill
 * reads the core weights once per loop step.  Returns CDB_ERR_ARG for a bad
 * shape or non-positive rates. */
int cdb_roofline_latency(const cdb_model_desc *m, double hbm_gbps, double tensor_tflops, double launch_s,
                         cdb_latency_model *out);

/* Online serving (§6.3): request i joins the scheduler when a simulated clock
 * passes arrival_s[i] (HOST array, seconds, non-decreasing, >= 0); every
 * scheduler call advances the clock by the cost of the stages it ran, and
 * with nothing to run the clock jumps to the next arrival.  finish_s[i]
 * (HOST, written) is the end of the stage that produced request i's last
 * token, so (finish_s[i] - arrival_s[i]) / gen_len[i] is its normalised
 * latency.  *out is filled as by cdb_predict_job (busy time; the makespan is
 * the largest finish time).  Same errors as cdb_predict_job, plus CDB_ERR_ARG
 * for missing or decreasing arrival times. */
int cdb_predict_online(const cdb_job *job, const double *arrival_s, int mode, int K,
                       const cdb_latency_model *lm, double *finish_s, cdb_prediction *out);

/* Picks the schedule with the lowest predicted job latency among no-refill
 * and refill with K in {1, 2, 4, ..., W} (then K = W).  Writes the chosen
 * mode and K, its prediction (nullable) and the best refill and no-refill
 * times (nullable).  Ties go to no-refill (refill with K = W often issues
 * the same stages), then to the smaller K.  Returns
 * CDB_OK or the first error of cdb_predict_job. */
int cdb_select_schedule(const cdb_job *job, const cdb_latency_model *lm, int *mode, int *K,
                        cdb_prediction *best, double *refill_seconds, double *no_refill_seconds);

#ifdef __cplusplus
}
#endif
#endif /* CDB_PLAN_H */
