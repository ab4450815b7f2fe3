// Latency planner: predicted job time from a per-stage linear latency model,
// and the choice of refill / no-refill and the minimum coda batch K.
//
// "Depth-adaptive Inference of Looped Language Models via Continuous Depth
// Batching", §5 (recurrent-step latency t = delta + gamma N_b + alpha N_c),
// §6.2 (refill helps most below the saturation batch size), §6.4 and Fig. 7
// (minimum coda batch K).  The job runs through the host scheduler itself with
// its exit depths replayed (App. C.2); each stage it issues is costed by the
// model and the costs add up, since the GPU executes stages in order.
#include <cstring>
#include <memory>
#include <vector>

#include "../../include/cdb_plan.h"
#include "replay.h"

namespace cdb {
namespace {

double stage_time(const cdb_stage_cost& c, double rows, double ctx) {
  return c.delta + c.gamma * rows + c.alpha * ctx;
}

// Replays exits like ReplayExecutor and adds up the cost of every stage.
class CostExecutor : public ReplayExecutor {
 public:
  CostExecutor(int mode, int W, int r_max, const cdb_latency_model& lm)
      : ReplayExecutor(mode, W, r_max), lm_(lm) {
    std::memset(&p_, 0, sizeof(p_));
  }
  int prefill(const PrefillPlan& p, const std::vector<Seq>&) override {
    double ctx = 0;
    for (const PrefillRow& r : p.rows) ctx += r.pos + 1;
    const double c = stage_time(lm_.prefill, (double)p.rows.size(), ctx);
    p_.prefill_seconds += c;
    call_ += c;
    ++p_.prefill_stages;
    p_.tokens += (int64_t)p.done_seqs.size();
    return CDB_OK;
  }
  int prelude(const PreludePlan& p) override {
    double ctx = 0;
    for (const Tok& t : p.rows) ctx += t.pos + 1;
    const double c = stage_time(lm_.prelude, (double)p.rows.size(), ctx);
    p_.prelude_seconds += c;
    call_ += c;
    ++p_.prelude_stages;
    return CDB_OK;
  }
  int core(const CorePlan& p) override {
    double ctx = 0;
    for (const Tok& t : *p.rows) ctx += t.pos + 1;
    const double c = stage_time(lm_.core, (double)p.B, ctx);
    p_.core_seconds += c;
    call_ += c;
    ++p_.core_steps;
    p_.core_token_steps += p.B;
    return ReplayExecutor::core(p);
  }
  int coda(const std::vector<Tok>& rows) override {
    double ctx = 0;
    for (const Tok& t : rows) ctx += t.pos + 1;
    const double c = stage_time(lm_.coda, (double)rows.size(), ctx);
    p_.coda_seconds += c;
    call_ += c;
    ++p_.coda_stages;
    p_.tokens += (int64_t)rows.size();
    coda_rows_ += (int64_t)rows.size();
    return CDB_OK;
  }
  // A finished sequence ends with the stage that produced its last token:
  // record the cost of the current scheduler call up to that stage.
  int finish(const Seq& s) override {
    finished.push_back({s.id, call_});
    return CDB_OK;
  }
  // Cost of the stages run since the last call, which it resets.
  double take_call_cost() {
    const double c = call_;
    call_ = 0;
    return c;
  }
  std::vector<std::pair<int64_t, double>> finished;  // (sequence id, cost into its call)

  cdb_prediction result() const {
    cdb_prediction r = p_;
    r.seconds = r.prefill_seconds + r.prelude_seconds + r.core_seconds + r.coda_seconds;
    r.mean_core_batch = r.core_steps ? (double)r.core_token_steps / (double)r.core_steps : 0.0;
    r.mean_coda_batch = r.coda_stages ? (double)coda_rows_ / (double)r.coda_stages : 0.0;
    return r;
  }

 private:
  cdb_latency_model lm_;
  cdb_prediction p_;
  int64_t coda_rows_ = 0;
  double call_ = 0;
};

bool cost_ok(const cdb_stage_cost& c) { return c.delta >= 0 && c.gamma >= 0 && c.alpha >= 0; }

bool job_ok(const cdb_job* j) {
  if (!j || j->n_seqs < 0 || (j->n_seqs > 0 && (!j->prompt_len || !j->gen_len)) || j->W < 1 || j->M < 1 ||
      j->S < 0 || j->r_min < 2 || j->r_max < j->r_min || j->r_max > CDB_MAX_DEPTH || j->kv_blocks < 1 ||
      j->max_ctx < 1 || j->max_new_cap < 1 || j->kv_headroom < 0.f || j->kv_headroom >= 1.f)
    return false;
  for (int i = 0; i < j->n_seqs; ++i)
    if (j->prompt_len[i] < 1 || j->gen_len[i] < 1 || j->gen_len[i] > j->max_new_cap ||
        j->prompt_len[i] + j->gen_len[i] - 1 > j->max_ctx)
      return false;
  return true;
}

// Scheduler limits of a job; false for an inconsistent job.
bool job_cfg(const cdb_job* job, int mode, int K, SchedCfg* c) {
  c->mode = mode;
  c->W = job->W;
  c->M = job->M;
  c->S = job->S > 0 ? job->S : (job->W / 8 > 1 ? job->W / 8 : 1);
  c->K = K;
  c->r_max = job->r_max;
  c->r_min = job->r_min;
  c->kv_blocks = job->kv_blocks;
  c->kv_headroom = job->kv_headroom;
  c->max_ctx = job->max_ctx;
  c->max_new_cap = job->max_new_cap;
  return c->S <= c->W;
}

// Exit depths of request i (offset `off` into the concatenated table), or
// nullptr for fixed depth; `bad` is set when a depth is outside [r_min, r_max].
const int8_t* job_exits(const cdb_job* job, int mode, int i, int64_t off, bool* bad) {
  if (mode == CDB_MODE_FIXED_DEPTH || !job->exit_depths) return nullptr;
  const int8_t* e = job->exit_depths + off;
  for (int t = 0; t + 1 < job->gen_len[i]; ++t)
    if (e[t] < job->r_min || e[t] > job->r_max) *bad = true;
  return e;
}

}  // namespace
}  // namespace cdb

extern "C" {

int cdb_predict_job(const cdb_job* job, int mode, int K, const cdb_latency_model* lm, cdb_prediction* out) {
  using namespace cdb;
  if (!job_ok(job) || !lm || !out || K < 1 || mode < 0 || mode > 2 || !cost_ok(lm->prefill) ||
      !cost_ok(lm->prelude) || !cost_ok(lm->core) || !cost_ok(lm->coda))
    return CDB_ERR_ARG;
  if (mode != CDB_MODE_FIXED_DEPTH && job->n_seqs > 0 && !job->exit_depths) return CDB_ERR_ARG;
  SchedCfg c;
  if (!job_cfg(job, mode, K, &c)) return CDB_ERR_ARG;
  CostExecutor ex(mode, job->W, job->r_max, *lm);
  Scheduler sched(c, &ex);
  ex.seqs = &sched.seqs();
  int64_t off = 0, work = 64;
  for (int i = 0; i < job->n_seqs; ++i) {
    bool bad = false;
    const int8_t* e = job_exits(job, mode, i, off, &bad);
    if (bad) return CDB_ERR_ARG;
    int rc = sched.admit(i, nullptr, job->prompt_len[i], job->gen_len[i], e, nullptr);
    if (rc < 0) return rc;
    off += job->gen_len[i] - 1;
    work += (int64_t)job->gen_len[i] * (job->r_max + 3) + job->prompt_len[i] / job->M + 2;
  }
  // Every stage makes progress, so the loop ends within `work` calls; the
  // bound only guards against a scheduler that stops progressing.
  for (int64_t it = 0; it < 4 * work; ++it) {
    cdb_step_info info;
    int rc = sched.step_boundary(&info);
    if (rc == CDB_DONE) {
      *out = ex.result();
      return CDB_OK;
    }
    if (rc < 0) return rc;
    if (rc == CDB_IDLE) {
      rc = sched.step_core(&info);
      if (rc < 0) return rc;
    }
  }
  return CDB_ERR_STATE;
}

int cdb_roofline_latency(const cdb_model_desc* m, double hbm_gbps, double tensor_tflops, double launch_s,
                         cdb_latency_model* out) {
  if (!m || !out || hbm_gbps <= 0 || tensor_tflops <= 0 || launch_s < 0 || m->d_model < 1 || m->ffn < 1 ||
      m->vocab < 1 || m->n_core < 1 || m->n_prelude < 0 || m->n_coda < 0 || m->r_max < 1 ||
      (m->dtype != CDB_FP32 && m->dtype != CDB_BF16))
    return CDB_ERR_ARG;
  const double bw = hbm_gbps * 1e9, tf = tensor_tflops * 1e12;
  const double d = m->d_model, f = m->ffn, V = m->vocab, es = m->dtype == CDB_BF16 ? 2.0 : 4.0;
  const double Pl = 4 * d * d + 3 * d * f;                     // one transformer block
  const double Pa = m->has_adapter ? 2 * d * d : 0.0;          // loop-entry adapter
  const double Pc = m->n_core * Pl + Pa, Pp = m->n_prelude * Pl, Po = m->n_coda * Pl + V * d;
  const double kv_row = 2 * d * es;                            // K and V of one entry, one layer
  auto max2 = [](double a, double b) { return a > b ? a : b; };
  // Kernels per stage: about ten per decode block (norms, projections, RoPE
  // and KV write, attention and its combine, SwiGLU fold) plus the stage's own.
  const double Lc = 10.0 * m->n_core + 4 + (m->has_adapter ? 2 : 0);
  const double Lp = 10.0 * m->n_prelude + 3, Lo = 10.0 * m->n_coda + 4;
  const double A = m->n_prelude + (double)m->r_max * m->n_core + m->n_coda;  // block applications in prefill
  out->core = {Pc * es / bw + launch_s * Lc, max2(2 * Pc / tf, m->n_core * kv_row / bw), m->n_core * kv_row / bw};
  out->prelude = {Pp * es / bw + launch_s * Lp, max2(2 * Pp / tf, (d * es + m->n_prelude * kv_row) / bw),
                  m->n_prelude * kv_row / bw};
  out->coda = {Po * es / bw + launch_s * Lo, max2(2 * Po / tf, (V * 4 + m->n_coda * kv_row) / bw),
               m->n_coda * kv_row / bw};
  const double Pf = Pp + m->r_max * Pc + m->n_coda * Pl;
  out->prefill = {(Pf + V * d) * es / bw + launch_s * (9 * A + (m->has_adapter ? 2.0 * m->r_max : 0) + 5),
                  max2(2 * Pf / tf, A * kv_row / bw), 4 * d * A / tf};
  return CDB_OK;
}

int cdb_select_schedule(const cdb_job* job, const cdb_latency_model* lm, int* mode, int* K, cdb_prediction* best,
                        double* refill_seconds, double* no_refill_seconds) {
  if (!job || !lm || !mode || !K) return CDB_ERR_ARG;
  // No-refill first: refill must be strictly faster to be chosen (refill with
  // K = W often issues the very same stages as no-refill).
  cdb_prediction p, bp;
  int rc = cdb_predict_job(job, CDB_MODE_NO_REFILL, 1, lm, &bp);
  if (rc < 0) return rc;
  const double no_refill = bp.seconds;
  int bm = CDB_MODE_NO_REFILL, bk = 1;
  double best_refill = -1;
  std::vector<int> ks;
  for (int k = 1; k < job->W; k *= 2) ks.push_back(k);
  ks.push_back(job->W);
  for (int k : ks) {
    rc = cdb_predict_job(job, CDB_MODE_REFILL, k, lm, &p);
    if (rc < 0) return rc;
    if (p.seconds < bp.seconds) bp = p, bm = CDB_MODE_REFILL, bk = k;
    if (best_refill < 0 || p.seconds < best_refill) best_refill = p.seconds;
  }
  *mode = bm;
  *K = bk;
  if (best) *best = bp;
  if (refill_seconds) *refill_seconds = best_refill;
  if (no_refill_seconds) *no_refill_seconds = no_refill;
  return CDB_OK;
}

int cdb_predict_online(const cdb_job* job, const double* arrival_s, int mode, int K, const cdb_latency_model* lm,
                       double* finish_s, cdb_prediction* out) {
  using namespace cdb;
  if (!job_ok(job) || !lm || !out || !finish_s || (job->n_seqs > 0 && !arrival_s) || K < 1 || mode < 0 ||
      mode > 2 || !cost_ok(lm->prefill) || !cost_ok(lm->prelude) || !cost_ok(lm->core) || !cost_ok(lm->coda))
    return CDB_ERR_ARG;
  if (mode != CDB_MODE_FIXED_DEPTH && job->n_seqs > 0 && !job->exit_depths) return CDB_ERR_ARG;
  for (int i = 0; i < job->n_seqs; ++i)
    if (!(arrival_s[i] >= 0.0) || (i > 0 && arrival_s[i] < arrival_s[i - 1])) return CDB_ERR_ARG;
  SchedCfg c;
  if (!job_cfg(job, mode, K, &c)) return CDB_ERR_ARG;
  CostExecutor ex(mode, job->W, job->r_max, *lm);
  Scheduler sched(c, &ex);
  ex.seqs = &sched.seqs();
  std::vector<int64_t> off(job->n_seqs + 1, 0);
  int64_t work = 64 + 2 * (int64_t)job->n_seqs;
  for (int i = 0; i < job->n_seqs; ++i) {
    bool bad = false;
    job_exits(job, mode, i, off[i], &bad);
    if (bad) return CDB_ERR_ARG;
    off[i + 1] = off[i] + job->gen_len[i] - 1;
    work += (int64_t)job->gen_len[i] * (job->r_max + 3) + job->prompt_len[i] / job->M + 2;
    finish_s[i] = -1.0;
  }
  // Simulated clock: requests join when it passes their arrival time; each
  // scheduler call advances it by the cost of the stages it ran; with nothing
  // to run it jumps to the next arrival.
  double T = 0.0;
  int next = 0;
  for (int64_t it = 0; it < 4 * work; ++it) {
    while (next < job->n_seqs && arrival_s[next] <= T) {
      bool bad = false;
      const int8_t* e = job_exits(job, mode, next, off[next], &bad);
      int rc = sched.admit(next, nullptr, job->prompt_len[next], job->gen_len[next], e, nullptr);
      if (rc < 0) return rc;
      ++next;
    }
    cdb_step_info info;
    int rc = sched.step_boundary(&info);
    if (rc < 0) return rc;
    if (rc == CDB_IDLE) {
      rc = sched.step_core(&info);
      if (rc < 0) return rc;
    }
    for (const auto& f : ex.finished) finish_s[f.first] = T + f.second;
    ex.finished.clear();
    T += ex.take_call_cost();
    if (rc == CDB_DONE) {
      if (next >= job->n_seqs) {
        *out = ex.result();
        return CDB_OK;
      }
      if (arrival_s[next] > T) T = arrival_s[next];
    }
  }
  return CDB_ERR_STATE;
}

}  // extern "C"
