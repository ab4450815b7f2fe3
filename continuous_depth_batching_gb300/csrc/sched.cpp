// Host scheduler of continuous depth batching (see sched.h for the sources).
#include "sched.h"

#include <algorithm>
#include <cstring>

namespace cdb {

Scheduler::Scheduler(const SchedCfg& c, Executor* ex) : c_(c), ex_(ex) {
  for (int s = c_.W - 1; s >= 0; --s) free_slots_.push_back(s);
  for (int b = c_.kv_blocks - 1; b >= 0; --b) free_blocks_.push_back(b);
}

int Scheduler::fail(int code, const std::string& m) {
  err = m;
  return code;
}

int Scheduler::blocks_per_seq_max() const { return (c_.max_ctx + c_.kv_block - 1) / c_.kv_block; }

static int ctx_positions(const Seq& s) { return s.P + s.max_new - 1; }

int Scheduler::admit(int64_t id, const int32_t* prompt, int P, int max_new,
                     const int8_t* force_exit, const int32_t* force_tok) {
  if (P < 1 || max_new < 1) return fail(CDB_ERR_ARG, "prompt_len and max_new_tokens must be >= 1");
  if (max_new > c_.max_new_cap) return fail(CDB_ERR_ARG, "max_new_tokens exceeds max_new_cap");
  if (P + max_new - 1 > c_.max_ctx) return fail(CDB_ERR_ARG, "prompt_len + max_new_tokens - 1 exceeds max_ctx");
  Seq s;
  s.id = id;
  s.P = P;
  s.max_new = max_new;
  if (prompt) s.prompt.assign(prompt, prompt + P);
  else s.prompt.assign(P, 0);
  if (force_exit && max_new > 1) {
    s.force_exit.assign(force_exit, force_exit + (max_new - 1));
    for (int8_t e : s.force_exit)
      if (e != 0 && (e < c_.r_min || e > c_.r_max))
        return fail(CDB_ERR_ARG, "force_exit entries must be 0 or in [r_min, r_max]");
  }
  if (force_tok) s.force_tok.assign(force_tok, force_tok + max_new);
  int need = (ctx_positions(s) + c_.kv_block - 1) / c_.kv_block;
  if (need > c_.kv_blocks) return fail(CDB_ERR_KV_FULL, "sequence needs more KV blocks than the pool holds");
  seqs_.push_back(std::move(s));
  waiting_.push_back((int)seqs_.size() - 1);
  return CDB_OK;
}

bool Scheduler::kv_admissible(const Seq& s) const {
  long need = (ctx_positions(s) + c_.kv_block - 1) / c_.kv_block;
  long free = (long)free_blocks_.size();
  if (free < need) return false;
  return (double)(free - need) >= (double)c_.kv_headroom * (double)c_.kv_blocks;
}

// CanPrefill(W, S, rho_KV) of Appendix A.2/A.3: a chunked prompt always
// continues; a new prompt starts once at least S of the W sequence slots are
// free and the KV pool keeps its headroom after reserving the sequence.
bool Scheduler::can_prefill() const {
  if (chunked_ >= 0) return true;
  if (waiting_.empty()) return false;
  if (c_.W - active_ < c_.S) return false;
  return kv_admissible(seqs_[waiting_.front()]);
}

int Scheduler::admit_to_active(int si) {
  Seq& s = seqs_[si];
  s.slot = free_slots_.back();
  free_slots_.pop_back();
  int need = (ctx_positions(s) + c_.kv_block - 1) / c_.kv_block;
  s.blocks.clear();
  for (int i = 0; i < need; ++i) {
    s.blocks.push_back(free_blocks_.back());
    free_blocks_.pop_back();
  }
  s.state = kPrefilling;
  ++active_;
  return ex_->admit(s);
}

void Scheduler::fill_queues(cdb_step_info* info) const {
  if (!info) return;
  info->q_r = (int)qr_.size();
  info->q_c = (int)qc_.size();
  info->q_p = (int)waiting_.size();
  info->q_d = (int)qd_.size();
  info->step_index = steps_;
}

void Scheduler::record(int stage, int batch, int ptok, int exits, const int* hist) {
  if (!trace_on) return;
  cdb_trace_row r;
  std::memset(&r, 0, sizeof(r));
  r.stage = stage;
  r.batch = batch;
  r.prefill_tokens = ptok;
  r.exits = exits;
  r.q_r = (int)qr_.size();
  r.q_c = (int)qc_.size();
  r.q_p = (int)waiting_.size();
  r.q_d = (int)qd_.size();
  if (hist) std::memcpy(r.depth_hist, hist, sizeof(r.depth_hist));
  trace_.push_back(r);
}

int Scheduler::finish_seq(int si) {
  Seq& s = seqs_[si];
  int rc = ex_->finish(s);
  if (rc < 0) return rc;
  s.state = kFinished;
  free_slots_.push_back(s.slot);
  for (int b : s.blocks) free_blocks_.push_back(b);
  s.blocks.clear();
  --active_;
  finished_.push_back(si);
  return CDB_OK;
}

int Scheduler::run_prelude(std::vector<Tok>& rows, cdb_step_info* info, bool second) {
  if (rows.empty()) return CDB_OK;
  PreludePlan p;
  p.rows = rows;
  p.dst_off = refill_;
  int rc = ex_->prelude(p);
  if (rc < 0) return fail(rc, ex_->error());
  for (auto& t : rows) qr_.push_back(t);
  refill_ += (int)rows.size();
  record(CDB_STAGE_PRELUDE, (int)rows.size(), 0, 0, nullptr);
  if (info) {
    int64_t ctx = 0;
    for (auto& t : rows) ctx += t.pos + 1;
    if (second) {
      info->stage2 = CDB_STAGE_PRELUDE;
      info->batch2 = (int)rows.size();
      info->ctx2 = ctx;
    } else {
      info->stage = CDB_STAGE_PRELUDE;
      info->batch = (int)rows.size();
      info->ctx = ctx;
    }
  }
  return CDB_OK;
}

// Pack up to M prompt tokens: first the rest of a chunked prompt, then new
// prompts in arrival order while fewer than W sequences are active; the last
// prompt may be split (Appendix A.1, Fig. 8 left).
int Scheduler::run_prefill(cdb_step_info* info) {
  PrefillPlan plan;
  int budget = c_.M;
  auto take = [&](int si) {
    Seq& s = seqs_[si];
    int n = std::min(s.P - s.prefilled, budget);
    for (int k = 0; k < n; ++k)
      plan.rows.push_back({s.slot, s.prefilled + k, s.prompt[s.prefilled + k]});
    s.prefilled += n;
    budget -= n;
    plan.n_seqs++;
    if (s.prefilled == s.P) {
      plan.done_rows.push_back((int)plan.rows.size() - 1);
      plan.done_seqs.push_back(si);
    } else {
      chunked_ = si;
    }
  };
  if (chunked_ >= 0) {
    int si = chunked_;
    chunked_ = -1;
    take(si);
  }
  while (budget > 0 && chunked_ < 0 && !waiting_.empty() && active_ < c_.W &&
         kv_admissible(seqs_[waiting_.front()])) {
    int si = waiting_.front();
    waiting_.pop_front();
    int rc = admit_to_active(si);
    if (rc < 0) return fail(rc, ex_->error());
    take(si);
  }
  if (plan.rows.empty()) return fail(CDB_ERR_STATE, "prefill selected with nothing to pack");
  int rc = ex_->prefill(plan, seqs_);
  if (rc < 0) return fail(rc, ex_->error());
  if (info) {
    info->stage = CDB_STAGE_PREFILL;
    info->batch = plan.n_seqs;
    info->prefill_tokens = (int)plan.rows.size();
    info->new_tokens = (int)plan.done_seqs.size();
    for (auto& r : plan.rows) info->ctx += r.pos + 1;
  }
  std::vector<Tok> next;
  for (int si : plan.done_seqs) {
    Seq& s = seqs_[si];
    s.n_gen = 1;
    s.state = kDecoding;
    if (s.max_new == 1) {
      rc = finish_seq(si);
      if (rc < 0) return fail(rc, ex_->error());
      continue;
    }
    Tok t;
    t.seq = si;
    t.slot = s.slot;
    t.pos = s.P;
    t.t = 1;
    next.push_back(t);
  }
  if (c_.mode == CDB_MODE_REFILL) {
    record(CDB_STAGE_PREFILL, plan.n_seqs, (int)plan.rows.size(), 0, nullptr);
    rc = run_prelude(next, info, true);
    if (rc < 0) return rc;
  } else {
    for (auto& t : next) qd_.push_back(t);
    record(CDB_STAGE_PREFILL, plan.n_seqs, (int)plan.rows.size(), 0, nullptr);
  }
  fill_queues(info);
  return CDB_OK;
}

int Scheduler::run_coda(cdb_step_info* info) {
  std::vector<Tok> rows;
  rows.swap(qc_);
  int rc = ex_->coda(rows);
  if (rc < 0) return fail(rc, ex_->error());
  if (info) {
    info->stage = CDB_STAGE_CODA;
    info->batch = (int)rows.size();
    info->new_tokens = (int)rows.size();
    for (auto& t : rows) info->ctx += t.pos + 1;
  }
  std::vector<Tok> next;
  for (auto& t : rows) {
    Seq& s = seqs_[t.seq];
    s.n_gen = t.t + 1;
    if (s.n_gen >= s.max_new) {
      rc = finish_seq(t.seq);
      if (rc < 0) return fail(rc, ex_->error());
      continue;
    }
    Tok n;
    n.seq = t.seq;
    n.slot = t.slot;
    n.pos = t.pos + 1;
    n.t = t.t + 1;
    next.push_back(n);
  }
  if (c_.mode == CDB_MODE_REFILL) {
    record(CDB_STAGE_CODA, (int)rows.size(), 0, 0, nullptr);
    rc = run_prelude(next, info, true);
    if (rc < 0) return rc;
  } else {
    for (auto& t : next) qd_.push_back(t);
    record(CDB_STAGE_CODA, (int)rows.size(), 0, 0, nullptr);
  }
  fill_queues(info);
  return CDB_OK;
}

bool Scheduler::all_done() const {
  return waiting_.empty() && chunked_ < 0 && active_ == 0 && qr_.empty() && qc_.empty() &&
         qd_.empty();
}

int Scheduler::step_boundary(cdb_step_info* info) {
  if (info) std::memset(info, 0, sizeof(*info));
  if (c_.mode == CDB_MODE_REFILL) {
    // Algorithm 2 priority: coda once K exits wait (or when nothing else can
    // run), then prefill, else the recurrent core.
    if (!qc_.empty() && ((int)qc_.size() >= c_.K || (qr_.empty() && !can_prefill())))
      return run_coda(info);
    if (can_prefill()) return run_prefill(info);
    if (!qr_.empty()) {
      fill_queues(info);
      return CDB_IDLE;
    }
  } else {
    // Algorithm 1: prefill while admissible, prelude the whole decode queue,
    // loop until every token exited, then one coda for the cohort.
    if (cohort_) {
      if (!qr_.empty()) {
        fill_queues(info);
        return CDB_IDLE;
      }
      cohort_ = false;
      if (!qc_.empty()) return run_coda(info);
    }
    if (can_prefill()) return run_prefill(info);
    if (!qd_.empty()) {
      std::vector<Tok> rows;
      rows.swap(qd_);
      int rc = run_prelude(rows, info, false);
      if (rc < 0) return rc;
      cohort_ = true;
      fill_queues(info);
      return CDB_OK;
    }
  }
  fill_queues(info);
  if (all_done()) return CDB_DONE;
  if (active_ == 0 && !waiting_.empty())
    return fail(CDB_ERR_KV_FULL, "waiting sequence does not fit the KV pool headroom");
  return fail(CDB_ERR_STATE, "scheduler has no runnable stage");
}

int Scheduler::step_core(cdb_step_info* info) {
  if (info) std::memset(info, 0, sizeof(*info));
  if (qr_.empty()) {
    fill_queues(info);
    return CDB_IDLE;
  }
  CorePlan p;
  p.step = steps_;
  p.B = (int)qr_.size();
  p.B_cont = cont_;
  p.n_ref = refill_;
  p.qc_off = (int)qc_.size();
  p.rows = &qr_;
  if (p.B_cont + p.n_ref != p.B) return fail(CDB_ERR_STATE, "recurrent queue out of sync");
  int rc = ex_->core(p);
  if (rc < 0) return fail(rc, ex_->error());
  const int64_t this_step = steps_++;
  int64_t ctx = 0;
  for (auto& t : qr_) ctx += t.pos + 1;

  // Lookahead: the gate results of the previous step decide this step's exits.
  bool need = false;
  for (auto& t : qr_)
    if (t.depth >= 1 && t.depth + 1 < c_.r_max) need = true;
  if (need) {
    std::vector<uint8_t> pend;
    rc = ex_->core_flags(this_step - 1, pend);
    if (rc < 0) return fail(rc, ex_->error());
    for (auto& t : qr_)
      if (t.depth >= 1) t.pend = pend[t.slot];
  }
  int hist[CDB_MAX_DEPTH];
  std::memset(hist, 0, sizeof(hist));
  std::vector<Tok> cont;
  int exits = 0;
  for (auto& t : qr_) {
    int d = t.depth + 1;
    hist[d - 1]++;
    bool ex = (t.depth >= 1 && t.pend) || d >= c_.r_max;
    Tok n = t;
    n.depth = d;
    n.pend = 0;
    if (ex) {
      qc_.push_back(n);
      ++exits;
    } else {
      cont.push_back(n);
    }
  }
  qr_.swap(cont);
  cont_ = (int)qr_.size();
  refill_ = 0;
  record(CDB_STAGE_LOOP, p.B, 0, exits, hist);
  if (info) {
    info->stage = CDB_STAGE_LOOP;
    info->batch = p.B;
    info->exits = exits;
    info->ctx = ctx;
    std::memcpy(info->depth_hist, hist, sizeof(hist));
  }
  fill_queues(info);
  return CDB_OK;
}

}  // namespace cdb
