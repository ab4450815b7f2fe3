/*
 * cdb_sim.h — host-only simulation of the CDB scheduler (for tests).
 *
 * Runs exactly the scheduler state machine of cdb.h (stage queues, refill /
 * no-refill / fixed-depth policies of §4.1 and Algorithms 1-2, admission rule
 * CanPrefill(W, S, rho_KV) of Appendix A.2, chunked prefill of Appendix A.1,
 * lookahead exit bookkeeping of §4.3) with an executor that computes nothing:
 * each decode forward's exit depth is replayed from a caller table, the way
 * the paper replays recorded exits (Appendix C.2).  It exists so the
 * scheduling traces of Tables 2-3 and Fig. 1 can be checked without a GPU;
 * it produces no tokens and is not a fallback for cdb.h.
 *
 * Errors: negative cdb_status values; the context stays usable.
 */
#ifndef CDB_SIM_H
#define CDB_SIM_H

#include "cdb.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cdb_sim cdb_sim;

/* mode: cdb_mode.  S = 0 selects max(1, W/8).  kv_blocks: 16-token blocks. */
int cdb_sim_create(int mode, int W, int M, int S, int K, int r_max, int r_min,
                   int kv_blocks, float kv_headroom, int max_ctx, int max_new_cap,
                   cdb_sim **out);

/* exit_depths [max_new_tokens - 1]: depth in [r_min, r_max] of each decode
 * forward (ignored in fixed-depth mode, may be NULL there). Copied. */
int cdb_sim_admit(cdb_sim *s, int64_t seq_id, int prompt_len, int max_new_tokens,
                  const int8_t *exit_depths);

int cdb_sim_step_boundary(cdb_sim *s, cdb_step_info *info);
int cdb_sim_step_core(cdb_sim *s, cdb_step_info *info);

/* Every stage executed so far, in order. */
int cdb_sim_trace_read(cdb_sim *s, cdb_trace_row *rows, int cap, int *n_out);

/* Finished sequence ids in finish order (all of them, not consumed). */
int cdb_sim_finished(cdb_sim *s, int64_t *ids, int cap, int *n_out);

void cdb_sim_free(cdb_sim *s);

#ifdef __cplusplus
}
#endif
#endif /* CDB_SIM_H */
