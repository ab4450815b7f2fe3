// Host scheduler of continuous depth batching: the stage queues, the refill /
// no-refill / fixed-depth policies and the admission rule.
//
// "Depth-adaptive Inference of Looped Language Models via Continuous Depth
// Batching", §4.1 (four stage queues), Appendix A.3 Algorithms 1 (no-refill)
// and 2 (refill with minimum coda batch K), Appendix A.2 (CanPrefill(W, S,
// rho_KV)), Appendix A.1 (chunked prefill of at most M prompt tokens, paged KV
// in 16-token blocks).  The scheduler is a pure host state machine: it decides
// which stage runs next and which tokens it contains, and hands each decision
// to an Executor.  The GPU executor is the product; a replay executor in
// sim.cpp drives the same code for tests.
//
// Lookahead (§4.3): exits after loop step r are the tokens whose gate was
// positive after step r-1, plus tokens reaching r_max.  The scheduler learns
// the step r-1 gate results (Executor::core_flags) only after step r has been
// enqueued, so the device is never waiting for the host between steps.
#pragma once

#include <cstdint>
#include <deque>
#include <string>
#include <vector>

#include "../../include/cdb.h"

namespace cdb {

enum SeqState { kWaiting = 0, kPrefilling = 1, kDecoding = 2, kFinished = 3 };

struct SchedCfg {
  int mode = CDB_MODE_REFILL;
  int W = 64, M = 8192, S = 8, K = 1;
  int r_max = 4, r_min = 2;
  int kv_block = 16;
  int kv_blocks = 0;
  float kv_headroom = 0.f;
  int max_ctx = 0;
  int max_new_cap = 0;
};

struct Seq {
  int64_t id = 0;
  std::vector<int32_t> prompt;
  int P = 0, max_new = 0;
  std::vector<int8_t> force_exit;  // empty: live gate
  std::vector<int32_t> force_tok;  // empty: live argmax
  int state = kWaiting;
  int slot = -1;        // sequence slot (0..W-1) while active
  int prefilled = 0;    // prompt tokens already prefilled
  int n_gen = 0;        // generated tokens known to exist
  std::vector<int> blocks;
};

// One token in flight.  Its forward produces generated token t (1-based among
// decode forwards) from input token t-1 at position pos = P + t - 1.
struct Tok {
  int seq = -1, slot = -1, pos = 0, t = 0;
  int depth = 0;      // loop steps completed
  uint8_t pend = 0;   // lookahead flag from the previous step's gate
};

struct PrefillRow {
  int slot, pos;
  int32_t tok;
};

struct PrefillPlan {
  std::vector<PrefillRow> rows;
  std::vector<int> done_rows;  // row of the last prompt position of each completed prompt
  std::vector<int> done_seqs;  // the matching sequence indices
  int n_seqs = 0;              // distinct sequences in the chunk
};

struct PreludePlan {
  std::vector<Tok> rows;  // tokens entering the recurrent queue
  int dst_off = 0;        // first refill row they occupy
};

struct CorePlan {
  int64_t step = 0;
  int B = 0, B_cont = 0, n_ref = 0, qc_off = 0;
  const std::vector<Tok>* rows = nullptr;  // the batch in slot order
};

class Executor {
 public:
  virtual ~Executor() = default;
  virtual int admit(const Seq& s) = 0;
  virtual int prefill(const PrefillPlan& p, const std::vector<Seq>& seqs) = 0;
  virtual int prelude(const PreludePlan& p) = 0;
  virtual int core(const CorePlan& p) = 0;
  // Blocks until the lookahead flags of core step `step` are on the host;
  // pend[slot] = 1 if that sequence's token set its flag at that step.
  virtual int core_flags(int64_t step, std::vector<uint8_t>& pend) = 0;
  virtual int coda(const std::vector<Tok>& rows) = 0;
  virtual int finish(const Seq& s) = 0;
  virtual const char* error() const { return ""; }
};

class Scheduler {
 public:
  Scheduler(const SchedCfg& c, Executor* ex);

  int admit(int64_t id, const int32_t* prompt, int P, int max_new, const int8_t* force_exit,
            const int32_t* force_tok);
  int step_boundary(cdb_step_info* info);
  int step_core(cdb_step_info* info);

  bool all_done() const;
  const std::vector<Seq>& seqs() const { return seqs_; }
  std::vector<int>& finished_order() { return finished_; }
  std::vector<cdb_trace_row>& trace() { return trace_; }
  bool trace_on = false;
  std::string err;
  int blocks_per_seq_max() const;

 private:
  bool can_prefill() const;
  bool kv_admissible(const Seq& s) const;
  int admit_to_active(int si);
  int run_prefill(cdb_step_info* info);
  int run_coda(cdb_step_info* info);
  int run_prelude(std::vector<Tok>& rows, cdb_step_info* info, bool second);
  int finish_seq(int si);
  void record(int stage, int batch, int ptok, int exits, const int* hist);
  void fill_queues(cdb_step_info* info) const;
  int fail(int code, const std::string& m);

  SchedCfg c_;
  Executor* ex_;
  std::vector<Seq> seqs_;
  std::deque<int> waiting_;
  int chunked_ = -1;  // sequence whose prompt is partly prefilled
  int active_ = 0;
  std::vector<int> free_slots_;
  std::vector<int> free_blocks_;
  std::vector<Tok> qr_;   // recurrent queue in device slot order
  std::vector<Tok> qc_;   // exited tokens awaiting coda, in exit order
  std::vector<Tok> qd_;   // no-refill: decode queue awaiting the cohort prelude
  int cont_ = 0;          // rows continuing from the last core step
  int refill_ = 0;        // rows appended by preludes since the last core step
  bool cohort_ = false;   // no-refill: a cohort is looping
  int64_t steps_ = 0;     // core steps issued
  std::vector<int> finished_;
  std::vector<cdb_trace_row> trace_;
};

}  // namespace cdb
