// Scheduling simulator: the host scheduler driven by the replay executor, for
// checking the scheduling traces of Tables 2-3 on a CPU.
#include <cstring>
#include <memory>

#include "../../include/cdb_sim.h"
#include "replay.h"


struct cdb_sim {
  std::unique_ptr<cdb::ReplayExecutor> ex;
  std::unique_ptr<cdb::Scheduler> sched;
};

extern "C" {

int cdb_sim_create(int mode, int W, int M, int S, int K, int r_max, int r_min, int kv_blocks,
                   float kv_headroom, int max_ctx, int max_new_cap, cdb_sim** out) {
  if (!out || W < 1 || M < 1 || K < 1 || r_min < 2 || r_max < r_min || r_max > CDB_MAX_DEPTH ||
      kv_blocks < 1 || max_ctx < 1 || max_new_cap < 1 || mode < 0 || mode > 2)
    return CDB_ERR_ARG;
  cdb::SchedCfg c;
  c.mode = mode;
  c.W = W;
  c.M = M;
  c.S = S > 0 ? S : (W / 8 > 1 ? W / 8 : 1);
  c.K = K;
  c.r_max = r_max;
  c.r_min = r_min;
  c.kv_blocks = kv_blocks;
  c.kv_headroom = kv_headroom;
  c.max_ctx = max_ctx;
  c.max_new_cap = max_new_cap;
  auto* s = new cdb_sim;
  s->ex.reset(new cdb::ReplayExecutor(mode, W, r_max));
  s->sched.reset(new cdb::Scheduler(c, s->ex.get()));
  s->ex->seqs = &s->sched->seqs();
  s->sched->trace_on = true;
  *out = s;
  return CDB_OK;
}

int cdb_sim_admit(cdb_sim* s, int64_t seq_id, int prompt_len, int max_new_tokens,
                  const int8_t* exit_depths) {
  if (!s) return CDB_ERR_ARG;
  return s->sched->admit(seq_id, nullptr, prompt_len, max_new_tokens, exit_depths, nullptr);
}

int cdb_sim_step_boundary(cdb_sim* s, cdb_step_info* info) {
  if (!s) return CDB_ERR_ARG;
  return s->sched->step_boundary(info);
}

int cdb_sim_step_core(cdb_sim* s, cdb_step_info* info) {
  if (!s) return CDB_ERR_ARG;
  return s->sched->step_core(info);
}

int cdb_sim_trace_read(cdb_sim* s, cdb_trace_row* rows, int cap, int* n_out) {
  if (!s || !n_out) return CDB_ERR_ARG;
  auto& tr = s->sched->trace();
  int n = (int)tr.size() < cap ? (int)tr.size() : cap;
  if (rows && n > 0) std::memcpy(rows, tr.data(), sizeof(cdb_trace_row) * n);
  *n_out = n;
  return CDB_OK;
}

int cdb_sim_finished(cdb_sim* s, int64_t* ids, int cap, int* n_out) {
  if (!s || !n_out) return CDB_ERR_ARG;
  auto& f = s->sched->finished_order();
  int n = 0;
  for (int si : f) {
    if (n >= cap) break;
    if (ids) ids[n] = s->sched->seqs()[si].id;
    ++n;
  }
  *n_out = n;
  return CDB_OK;
}

void cdb_sim_free(cdb_sim* s) { delete s; }

}  // extern "C"
