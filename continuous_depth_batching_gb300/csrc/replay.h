// Replay executor: runs the scheduler with exit depths taken from a table, the
// way the paper replays recorded exit decisions (Appendix C.2).  Computes no
// model values.  Shared by the scheduling simulator (sim.cpp) and the latency
// planner (planner.cpp).
#pragma once

#include <map>
#include <vector>

#include "sched.h"

namespace cdb {

class ReplayExecutor : public Executor {
 public:
  ReplayExecutor(int mode, int W, int r_max) : mode_(mode), W_(W), r_max_(r_max) {}
  const std::vector<Seq>* seqs = nullptr;
  int admit(const Seq&) override { return CDB_OK; }
  int prefill(const PrefillPlan&, const std::vector<Seq>&) override { return CDB_OK; }
  int prelude(const PreludePlan&) override { return CDB_OK; }
  int core(const CorePlan& p) override {
    std::vector<uint8_t> f(W_, 0);
    for (const Tok& t : *p.rows) {
      const Seq& s = (*seqs)[t.seq];
      int d = t.depth + 1;  // step being run
      int e = r_max_;
      if (mode_ != CDB_MODE_FIXED_DEPTH && !s.force_exit.empty()) e = s.force_exit[t.t - 1];
      // lookahead: the flag set after step d makes the token exit after d+1
      f[t.slot] = (uint8_t)(d + 1 == e && e < r_max_);
    }
    flags_[p.step] = f;
    return CDB_OK;
  }
  int core_flags(int64_t step, std::vector<uint8_t>& pend) override {
    auto it = flags_.find(step);
    if (it == flags_.end()) return CDB_ERR_STATE;
    pend = it->second;
    flags_.erase(flags_.begin(), it);
    return CDB_OK;
  }
  int coda(const std::vector<Tok>&) override { return CDB_OK; }
  int finish(const Seq&) override { return CDB_OK; }

 private:
  int mode_, W_, r_max_;
  std::map<int64_t, std::vector<uint8_t>> flags_;
};

}  // namespace cdb
