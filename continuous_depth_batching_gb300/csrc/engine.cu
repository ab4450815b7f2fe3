// CDB engine: the C ABI of cdb.h, the arena layout and the GPU executor that
// carries out the scheduler's stages with the kernels of kernels.cuh.
//
// Stage sequencing follows "Depth-adaptive Inference of Looped Language
// Models via Continuous Depth Batching": prefill at full depth with chunking
// (Appendix A.1), prelude after prefill or coda, one recurrent-core step over
// the recurrent queue, coda on exited tokens (§4.1, Algorithms 1-2).  The
// lookahead flags of each core step are copied to the host on a second stream
// (§4.3, "asynchronous batch preparation") while the next stages run.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <deque>
#include <memory>
#include <string>
#include <thread>
#include <vector>

#include "../../include/cdb.h"
#include "kernels.cuh"
#include "sched.h"

namespace cdb {

static constexpr int kRing = 8;           // lookahead flag ring (core steps)
static constexpr int kWideBatch = 384;    // engines with at least this many slots split only narrow weights
static constexpr size_t kAlign = 256;
static constexpr size_t kStageSeg = 1 << 20;  // pinned upload segment
static constexpr int kStageSegs = 8;

static size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t total = 0;
  size_t pool, etab, bt, out_tok, ftok, fexit, out_depth, gtrace, ltrace, htrace, estore, rope, sprev;
  size_t rows[5], meta[5];  // X, Xc, Pb, Cb, Tp
  size_t pend_new, ring, status;
  size_t Xp, Ep, rslot, rpos, rtok, ptiles, done_idx, Cp, Cp_meta;
  size_t lslot, lt, lpos;
  size_t A, QKV, Q, O, Mid, logits, part_o, part_ml, gpart;
  size_t gpart_floats;
  // dims
  int es, nsl, max_blocks, max_splits, split, R, S, cap;
};

// KV slots per token of one recurrent-core layer: s of App. E.1.
static int core_slots(const cdb_model_desc* m) {
  return m->kv_slots <= 0 || m->kv_slots > m->r_max ? m->r_max : m->kv_slots;
}

static bool plan_layout(const cdb_model_desc* m, const cdb_sched_cfg* c, Layout* L) {
  const int es = m->dtype == CDB_BF16 ? 2 : 4;
  const size_t d = m->d_model, H = m->n_heads, hd = m->head_dim, f = m->ffn, V = m->vocab;
  const size_t W = c->W, M = c->M;
  L->es = es;
  L->nsl = m->n_prelude + m->n_core * core_slots(m) + m->n_coda;
  L->max_blocks = (c->max_ctx + 15) / 16;
  L->split = c->attn_split > 0 ? c->attn_split : 128;
  L->max_splits = (c->max_ctx + L->split - 1) / L->split;
  L->R = (int)(M > W ? M : W);
  L->cap = c->max_new_cap;
  L->S = c->S > 0 ? c->S : (c->W / 8 > 1 ? c->W / 8 : 1);
  const size_t R = L->R, cap = c->max_new_cap, T = c->trace_tokens;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L->pool = take((size_t)c->kv_blocks * L->nsl * 2 * 16 * d * es);
  L->etab = take((size_t)c->kv_blocks * 16);
  L->bt = take(W * L->max_blocks * 4);
  L->out_tok = take(W * cap * 4);
  L->ftok = take(W * cap * 4);
  L->fexit = take(W * cap);
  L->out_depth = take(W * cap);
  L->gtrace = take(c->trace_gate ? W * cap * m->r_max * 4 : 0);
  L->ltrace = take(W * T * V * 4);
  L->htrace = take(W * T * d * 4);
  L->estore = take(m->has_adapter ? W * d * 4 : 0);
  L->sprev = take(m->gate_kind == CDB_GATE_CONVERGENCE ? W * d * 4 : 0);  // s_{d-1} of each core row
  L->rope = take((size_t)L->max_blocks * 16 * (hd / 2) * 8);  // every position a block table can hold
  for (int i = 0; i < 5; ++i) {
    L->rows[i] = take(W * d * 4);
    L->meta[i] = take(W * 5 * 4);
  }
  L->pend_new = take(W * 4);
  L->ring = take(kRing * W);
  L->status = take(kStatusBytes);
  L->Xp = take(M * d * 4);
  L->Ep = take(m->has_adapter ? M * d * 4 : 0);
  L->rslot = take(M * 4);
  L->rpos = take(M * 4);
  L->rtok = take(M * 4);
  L->ptiles = take(((size_t)M / kPrefillTileRows + W + 2) * 16);
  L->done_idx = take(W * 4);
  L->Cp = take(W * d * 4);
  L->Cp_meta = take(W * 5 * 4);
  L->lslot = take(W * 4);
  L->lt = take(W * 4);
  L->lpos = take(W * 4);
  L->A = take(R * 2 * d * es);
  L->QKV = take(R * 3 * d * 4);
  L->Q = take(R * d * es);
  L->O = take(R * d * es);
  L->Mid = take(R * f * es);
  L->logits = take(W * V * 4);
  L->part_o = take(W * H * L->max_splits * hd * 4);
  L->part_ml = take(W * H * L->max_splits * 2 * 4);
  // Split-K partials of one decode GEMM ([split][row][ldp], ldp <= max(3d, 2f)).
  // Split-K partials: every decode projection below kWideBatch slots, the
  // narrow weights (at most kWideMaxSplits splits) from kWideBatch on.
  L->gpart_floats = (size_t)(W < kWideBatch ? kGemmMaxSplits : kWideMaxSplits) * W * std::max(3 * d, 2 * f);
  L->gpart = take(L->gpart_floats * 4);
  L->total = o;
  return true;
}

struct LayerW {
  const void *attn_norm, *wqkv, *wo, *mlp_norm, *wg, *wu, *wd;
};

struct PendingResult {
  int64_t id;
  int slot, n_tokens, active;
  cudaEvent_t ev;
};

struct HostResult {
  int64_t id;
  int n_tokens;
  std::vector<int32_t> tokens;
  std::vector<int8_t> depths;
  std::vector<float> gate, logits, hidden;
};

class GpuExecutor;

}  // namespace cdb

struct cdb_ctx {
  cdb_model_desc m;
  cdb_sched_cfg c;
  cdb::Layout L;
  char* base = nullptr;
  std::vector<cdb::LayerW> pre, core, coda;
  const void *embed, *lm_head, *final_norm, *gate_w, *adapter;
  cudaStream_t cs = nullptr, ps = nullptr;
  bool own_cs = false, own_ps = false;
  // pinned host memory
  char* stage = nullptr;  // kStageSegs * kStageSeg
  int seg = 0;
  size_t seg_off = 0;
  cudaEvent_t seg_ev[cdb::kStageSegs];
  uint8_t* pend_host = nullptr;  // kRing * W
  cudaEvent_t ev_core[cdb::kRing], ev_flags[cdb::kRing];
  char* res_host = nullptr;      // per slot result staging
  size_t res_stride = 0;
  std::vector<cdb::PendingResult> pending;  // per slot
  std::deque<cdb::HostResult> ready;
  std::unique_ptr<cdb::GpuExecutor> exec;
  std::unique_ptr<cdb::Scheduler> sched;
  std::string err;
  bool dead = false;
  int64_t io_h2d = 0, io_d2h = 0;
  // kernel timing (cdb_profile_enable, cdb_profile_repeat)
  bool prof_on = false;
  bool prof_core_only = false;  // time launches of core steps only
  int prof_repeat = -1;         // class relaunched inside core steps (step-delta cost), -1 none
  bool in_core = false;         // a core step is being enqueued
  struct ProfEv {
    int cls;
    cudaEvent_t a, b;
    double bytes, flops;
  };
  std::vector<ProfEv> prof_live;
  std::vector<cudaEvent_t> ev_pool;
  struct Stat {
    int64_t launches = 0;
    double ms = 0, bytes = 0, flops = 0;
  } stats[5];
};

namespace cdb {

template <typename P>
static P* at(cdb_ctx* x, size_t off) {
  return reinterpret_cast<P*>(x->base + off);
}

static RowMeta meta_at(cdb_ctx* x, size_t off) {
  int* p = at<int>(x, off);
  const int W = x->c.W;
  return RowMeta{p, p + W, p + 2 * W, p + 3 * W, p + 4 * W};
}

static int cuda_fail(cdb_ctx* x, cudaError_t e, const char* what) {
  x->err = std::string(what) + ": " + cudaGetErrorString(e);
  x->dead = true;
  return CDB_ERR_CUDA;
}

#define CK(expr)                                       \
  do {                                                 \
    cudaError_t _e = (expr);                           \
    if (_e != cudaSuccess) return cuda_fail(x, _e, #expr); \
  } while (0)

// Poll an event with a time limit so a stuck device cannot hang the host.
static int wait_event(cdb_ctx* x, cudaEvent_t ev, double limit_s) {
  auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return CDB_OK;
    if (e != cudaErrorNotReady) return cuda_fail(x, e, "cudaEventQuery");
    double dt = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    if (dt > limit_s) {
      x->err = "timed out waiting for the device";
      return CDB_ERR_TIMEOUT;
    }
    if (dt > 0.001) std::this_thread::yield();
  }
}

// Copy host bytes to a device address through the pinned staging segments.
static int upload(cdb_ctx* x, void* dst, const void* src, size_t n) {
  if (n == 0) return CDB_OK;
  if (n > kStageSeg) {
    x->err = "upload larger than a staging segment";
    return CDB_ERR_ARG;
  }
  if (x->seg_off + n > kStageSeg) {
    CK(cudaEventRecord(x->seg_ev[x->seg], x->cs));
    x->seg = (x->seg + 1) % kStageSegs;
    int rc = wait_event(x, x->seg_ev[x->seg], 600.0);
    if (rc < 0) return rc;
    x->seg_off = 0;
  }
  char* h = x->stage + (size_t)x->seg * kStageSeg + x->seg_off;
  std::memcpy(h, src, n);
  x->seg_off = (x->seg_off + n + 15) / 16 * 16;
  CK(cudaMemcpyAsync(dst, h, n, cudaMemcpyHostToDevice, x->cs));
  x->io_h2d += (int64_t)n;
  return CDB_OK;
}

static const char* kProfNames[5] = {"attention", "gemm", "prefill_attention", "rowwise", "prefill_gemm"};

static cudaEvent_t pool_event(cdb_ctx* x) {
  if (!x->ev_pool.empty()) {
    cudaEvent_t e = x->ev_pool.back();
    x->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Bracket one launch with events when timing is on; returns a handle or -1.
static int prof_begin(cdb_ctx* x, int cls) {
  if (!x->prof_on || (x->prof_core_only && !x->in_core)) return -1;
  cdb_ctx::ProfEv ev{cls, pool_event(x), pool_event(x), 0, 0};
  cudaEventRecord(ev.a, x->cs);
  x->prof_live.push_back(ev);
  return (int)x->prof_live.size() - 1;
}

static void prof_end(cdb_ctx* x, int h, double bytes, double flops) {
  if (h < 0) return;
  auto& ev = x->prof_live[h];
  cudaEventRecord(ev.b, x->cs);
  ev.bytes = bytes;
  ev.flops = flops;
}

// Fold finished event pairs into the per-class totals (after a sync).
static void prof_collect(cdb_ctx* x) {
  for (auto& ev : x->prof_live) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ev.a, ev.b) == cudaSuccess) {
      auto& st = x->stats[ev.cls];
      st.launches += 1;
      st.ms += ms;
      st.bytes += ev.bytes;
      st.flops += ev.flops;
    }
    x->ev_pool.push_back(ev.a);
    x->ev_pool.push_back(ev.b);
  }
  x->prof_live.clear();
}

class GpuExecutor : public Executor {
 public:
  explicit GpuExecutor(cdb_ctx* x) : x_(x) {}
  const char* error() const override { return x_->err.c_str(); }

  int admit(const Seq& s) override {
    cdb_ctx* x = x_;
    const Layout& L = x->L;
    const int cap = x->c.max_new_cap;
    std::vector<int32_t> bt(L.max_blocks, -1);
    for (size_t i = 0; i < s.blocks.size(); ++i) bt[i] = s.blocks[i];
    int rc = upload(x, at<int>(x, L.bt) + (size_t)s.slot * L.max_blocks, bt.data(), bt.size() * 4);
    if (rc < 0) return rc;
    std::vector<int8_t> fe(cap, 0);
    if (x->c.mode != CDB_MODE_FIXED_DEPTH)
      for (size_t i = 0; i < s.force_exit.size(); ++i) fe[i] = s.force_exit[i];
    rc = upload(x, at<int8_t>(x, L.fexit) + (size_t)s.slot * cap, fe.data(), cap);
    if (rc < 0) return rc;
    std::vector<int32_t> ft(cap, -1);
    for (size_t i = 0; i < s.force_tok.size(); ++i) ft[i] = s.force_tok[i];
    rc = upload(x, at<int>(x, L.ftok) + (size_t)s.slot * cap, ft.data(), cap * 4);
    if (rc < 0) return rc;
    if (x->c.trace_gate)
      CK(cudaMemsetAsync(at<float>(x, L.gtrace) + (size_t)s.slot * cap * x->m.r_max, 0xFF,
                         (size_t)cap * x->m.r_max * 4, x->cs));
    return CDB_OK;
  }

  // Returns the number of split-K partials left in the gpart workspace for the
  // consumer to fold (0: the epilogue ran in place).  parts: the caller folds.
  template <typename T>
  int gemm(int epi, const T* A, int lda, const void* W, const void* W2, int N, int K, int rows, float* Cf, T* Ct,
           int ldc, bool parts) {
    cdb_ctx* x = x_;
    const double es = sizeof(T), nw = W2 ? 2.0 : 1.0;
    const int h = prof_begin(x, decode_tiles_ ? 1 : 4);
    int ns = -1;
    // Decode tiling (split-K fixed by the weight shape) for engines of fewer
    // than kWideBatch slots; wider engines split only the narrow weights (at
    // most kWideMaxSplits) and run the others on the persistent kernel
    // without split partials, whose traffic grows with the rows (about 200 MB
    // per Ouro-shaped layer at 512 rows with decode splits).  Either way a
    // row's result does not depend on the other rows.
    const bool split_tiles = decode_tiles_ && x->c.W < kWideBatch;
    const int tiling = split_tiles ? kTileSplit : decode_tiles_ ? kTileWide : kTilePrefill;
    float* const gp = parts && decode_tiles_ ? at<float>(x, x->L.gpart) : nullptr;
    if (sizeof(T) == 2)
      ns = launch_gemm_tc(x->cs, epi, (const __nv_bfloat16*)A, lda, x->L.R, (const __nv_bfloat16*)W,
                          (const __nv_bfloat16*)W2, N, K, rows, Cf, (__nv_bfloat16*)Ct, ldc, tiling, gp,
                          x->L.gpart_floats, at<int>(x, x->L.status));
    if (ns < 0) {
      launch_gemm<T>(x->cs, epi, A, lda, (const T*)W, (const T*)W2, N, K, rows, Cf, Ct, ldc);
      ns = 0;
    } else if (repeat(1) && !(ns == 0 && epi == kEpiResid)) {
      // Step-delta timing: the same launch again writes the same partials
      // (or the same stored output); an in-place residual is not repeated.
      launch_gemm_tc(x->cs, epi, (const __nv_bfloat16*)A, lda, x->L.R, (const __nv_bfloat16*)W,
                     (const __nv_bfloat16*)W2, N, K, rows, Cf, (__nv_bfloat16*)Ct, ldc, tiling, gp,
                     x->L.gpart_floats, at<int>(x, x->L.status));
    }
    const double out_b = epi == kEpiSwiglu ? es : (epi == kEpiResid ? 8.0 : 4.0);
    prof_end(x, h, nw * N * (double)K * es + (double)rows * K * es + (double)rows * N * out_b,
             2.0 * nw * rows * (double)N * K);
    return ns;
  }

  // Pending split-K partials of a residual (mode 1) or store (mode 2) GEMM
  // into X, folded by the next RMSNorm of X or by flush().
  struct Pending {
    float* X = nullptr;
    int rows = 0, ns = 0, mode = 0;
  };
  Pending pend_;

  template <typename T>
  void norm(float* X, const void* g, T* A, int rows) {
    cdb_ctx* x = x_;
    if (pend_.ns && (pend_.X != X || pend_.rows != rows)) flush<T>();
    const int h = prof_begin(x, 3);
    launch_rmsnorm<T>(x->cs, X, (const T*)g, A, rows, x->m.d_model, x->m.rms_eps, x->m.d_model,
                      at<float>(x, x->L.gpart), pend_.ns, pend_.mode);
    prof_end(x, h, (double)rows * x->m.d_model * ((pend_.ns ? 8.0 : 4.0) + sizeof(T)), 0.0);
    pend_ = Pending();
  }

  template <typename T>
  void flush() {
    if (!pend_.ns) return;
    cdb_ctx* x = x_;
    const int h = prof_begin(x, 3);
    launch_fold(x->cs, at<float>(x, x->L.gpart), pend_.ns, pend_.rows, x->m.d_model, pend_.X, x->m.d_model,
                pend_.mode);
    prof_end(x, h, (double)pend_.rows * x->m.d_model * 8.0, 0.0);
    pend_ = Pending();
  }

  template <typename T>
  int block(const LayerW& lw, float* X, int rows, const int* mslot, const int* mpos, const int* mdepth,
            int depth_uniform, int slot_base, int clamp, bool decode, double sumL, int maxL = 0) {
    cdb_ctx* x = x_;
    const Layout& L = x->L;
    const int d = x->m.d_model, f = x->m.ffn, H = x->m.n_heads, hd = x->m.head_dim;
    cudaStream_t s = x->cs;
    T* A = at<T>(x, L.A);
    float* QKV = at<float>(x, L.QKV);
    float* GP = at<float>(x, L.gpart);
    T* Q = at<T>(x, L.Q);
    T* O = at<T>(x, L.O);
    T* Mid = at<T>(x, L.Mid);
    int* st = at<int>(x, L.status);
    KvGeom kv = geom();
    const double es = sizeof(T);
    decode_tiles_ = decode;
    norm<T>(X, lw.attn_norm, A, rows);
    int ns = gemm<T>(kEpiStore, A, d, lw.wqkv, nullptr, 3 * d, d, rows, QKV, nullptr, 3 * d, true);
    const int split = decode ? L.split : (1 << 30);
    // Split partials per (row, head): enough for the longest context in this
    // batch (maxL keys; the arena holds max_ctx), which also decides whether
    // the combine runs.  A row's own arithmetic does not depend on it.
    const int msp = decode ? std::max(1, std::min(L.max_splits, maxL > 0 ? (maxL + split - 1) / split
                                                                         : L.max_splits))
                           : 1;
    // bf16 decode: RoPE and the KV write run inside the attention kernel,
    // which reads q, k and v from the QKV partials.
    bool fused = decode && sizeof(T) == 2 && attention_rope_fusable(kv, H, hd, split);
    if (fused) {
      const int ha = prof_begin(x, 0);
      for (int rr = repeat(0) ? 2 : 1; rr > 0 && fused; --rr)
        fused = launch_attention_rope(s, ns ? GP : QKV, ns, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base,
                                      clamp, H, hd, split, msp, at<float2>(x, L.rope), (__nv_bfloat16*)O,
                                      at<float>(x, L.part_o), at<float>(x, L.part_ml), st);
      // Algorithmic bytes: each row reads each of its key rows (K and V, d
      // elements each) once and writes its own K and V rows and its output
      // (the q, k, v partials it folds are the split-K GEMM's L2 traffic).
      prof_end(x, ha, sumL * 2.0 * d * es + rows * d * 3.0 * es, 4.0 * d * sumL);
    }
    if (!fused) {
      int hr = prof_begin(x, 3);
      for (int rr = repeat(3) ? 2 : 1; rr > 0; --rr)
        launch_rope_kv<T>(s, ns ? GP : QKV, ns, rows, mslot, mpos, mdepth, depth_uniform, slot_base, clamp, Q, kv, H,
                          hd, at<float2>(x, L.rope), st);
      prof_end(x, hr, (double)rows * d * (12.0 + 3.0 * es), 0.0);  // q, k, v in; q, K, V rows out
      const int ha = prof_begin(x, decode ? 0 : 2);
      // Exit gaps are filled at compaction, so every key of a row is read from
      // the row's own slot.  Prefill chunks go through query tiles.
      bool done = false;
      if (!decode && sizeof(T) == 2 && pf_tiles_ > 0 && depth_uniform > 0)
        done = launch_prefill_attention(s, (const __nv_bfloat16*)Q, L.R, at<int4>(x, L.ptiles), pf_tiles_, kv,
                                        slot_base + (clamp ? std::min(depth_uniform, clamp) - 1 : 0), H, hd,
                                        (__nv_bfloat16*)O, st);
      if (!done)
        for (int rr = repeat(0) ? 2 : 1; rr > 0; --rr)
          launch_attention<T>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, hd, split, msp,
                              O, at<float>(x, L.part_o), at<float>(x, L.part_ml), st, true);
      // Decode: each row reads each of its key rows (K and V, d elements each)
      // once.  Prefill tiles: each tile reads the keys up to its last position
      // once for all of its rows.  Plus q in, o out.
      prof_end(x, ha, (done ? pf_key_rows_ : sumL) * 2.0 * d * es + 2.0 * rows * d * es, 4.0 * d * sumL);
    }
    ns = gemm<T>(kEpiResid, O, d, lw.wo, nullptr, d, d, rows, X, nullptr, d, true);
    if (ns) pend_ = Pending{X, rows, ns, 1};
    norm<T>(X, lw.mlp_norm, A, rows);
    ns = gemm<T>(kEpiSwiglu, A, d, lw.wg, lw.wu, f, d, rows, nullptr, Mid, f, true);
    if (ns) {
      const int hr = prof_begin(x, 3);
      for (int rr = repeat(3) ? 2 : 1; rr > 0; --rr) launch_swiglu_combine<T>(s, GP, ns, rows, f, Mid);
      prof_end(x, hr, (double)rows * f * (8.0 + es), 0.0);
    }
    ns = gemm<T>(kEpiResid, Mid, f, lw.wd, nullptr, d, f, rows, X, nullptr, d, true);
    if (ns) pend_ = Pending{X, rows, ns, 1};
    return CDB_OK;
  }

  template <typename T>
  int adapter_step(float* X, int rows, const float* E, int e_per_slot, const int* mslot) {
    cdb_ctx* x = x_;
    const int d = x->m.d_model;
    T* A = at<T>(x, x->L.A);
    flush<T>();
    decode_tiles_ = e_per_slot != 0;
    launch_concat<T>(x->cs, E, e_per_slot, mslot, X, A, rows, d);
    const int ns = gemm<T>(kEpiStore, A, 2 * d, x->adapter, nullptr, d, 2 * d, rows, X, nullptr, d, true);
    if (ns) pend_ = Pending{X, rows, ns, 2};
    return CDB_OK;
  }

  // Final RMSNorm + LM head + argmax over rows of H (the coda output).
  template <typename T>
  int head(const float* Hrows, int n, RowMeta m) {
    cdb_ctx* x = x_;
    const Layout& L = x->L;
    const int d = x->m.d_model, V = x->m.vocab, cap = x->c.max_new_cap;
    T* A = at<T>(x, L.A);
    float* lg = at<float>(x, L.logits);
    decode_tiles_ = true;
    flush<T>();
    launch_rmsnorm<T>(x->cs, const_cast<float*>(Hrows), (const T*)x->final_norm, A, n, d, x->m.rms_eps, d, nullptr, 0,
                      0);
    gemm<T>(kEpiStore, A, d, x->lm_head, nullptr, V, d, n, lg, nullptr, V, false);
    const bool tr = x->c.trace_tokens > 0;
    launch_argmax(x->cs, lg, n, V, m, at<int>(x, L.ftok), cap, at<int>(x, L.out_tok), tr ? at<float>(x, L.ltrace) : nullptr,
                  x->c.trace_tokens, Hrows, tr ? at<float>(x, L.htrace) : nullptr, d, at<int>(x, L.status));
    return CDB_OK;
  }

  int prefill(const PrefillPlan& p, const std::vector<Seq>&) override {
    return x_->m.dtype == CDB_BF16 ? prefill_t<__nv_bfloat16>(p) : prefill_t<float>(p);
  }
  template <typename T>
  int prefill_t(const PrefillPlan& p) {
    cdb_ctx* x = x_;
    const Layout& L = x->L;
    const int n = (int)p.rows.size(), d = x->m.d_model;
    std::vector<int32_t> a(n), b(n), c(n);
    for (int i = 0; i < n; ++i) {
      a[i] = p.rows[i].slot;
      b[i] = p.rows[i].pos;
      c[i] = p.rows[i].tok;
    }
    int* rslot = at<int>(x, L.rslot);
    int* rpos = at<int>(x, L.rpos);
    int* rtok = at<int>(x, L.rtok);
    int rc;
    if ((rc = upload(x, rslot, a.data(), n * 4)) < 0) return rc;
    if ((rc = upload(x, rpos, b.data(), n * 4)) < 0) return rc;
    if ((rc = upload(x, rtok, c.data(), n * 4)) < 0) return rc;
    // Query tiles for the prefill attention: runs of consecutive positions of
    // one sequence, at most prefill_tile_rows(head_dim) rows each.
    const std::vector<int4> tiles = prefill_tiles(a.data(), b.data(), n, x->m.head_dim);
    if ((rc = upload(x, at<int4>(x, L.ptiles), tiles.data(), tiles.size() * sizeof(int4))) < 0) return rc;
    pf_tiles_ = (int)tiles.size();
    pf_key_rows_ = 0;
    for (const int4& t : tiles) pf_key_rows_ += (double)t.w + t.y;
    float* Xp = at<float>(x, L.Xp);
    launch_embed_prefill<T>(x->cs, (const T*)x->embed, d, x->m.vocab, rslot, rpos, rtok, n, Xp, geom(), x->m.r_max,
                            at<int>(x, L.status));
    double sumL = 0;
    for (int i = 0; i < n; ++i) sumL += b[i] + 1;
    const int sc = core_slots(&x->m);
    for (int i = 0; i < x->m.n_prelude; ++i) block<T>(x->pre[i], Xp, n, rslot, rpos, nullptr, 1, i, 0, false, sumL);
    flush<T>();
    float* Ep = at<float>(x, L.Ep);
    if (x->m.has_adapter) {
      launch_copy_rows(x->cs, Xp, Ep, n, d);
      CK(cudaMemsetAsync(Xp, 0, (size_t)n * d * 4, x->cs));
    }
    for (int r = 1; r <= x->m.r_max; ++r) {
      if (x->m.has_adapter) adapter_step<T>(Xp, n, Ep, 0, rslot);
      for (int l = 0; l < x->m.n_core; ++l)
        block<T>(x->core[l], Xp, n, rslot, rpos, nullptr, r, x->m.n_prelude + l * sc, sc, false, sumL);
    }
    const int cbase = x->m.n_prelude + x->m.n_core * sc;
    for (int j = 0; j < x->m.n_coda; ++j)
      block<T>(x->coda[j], Xp, n, rslot, rpos, nullptr, 1, cbase + j, 0, false, sumL);
    flush<T>();
    const int nd = (int)p.done_rows.size();
    if (nd > 0) {
      if ((rc = upload(x, at<int>(x, L.done_idx), p.done_rows.data(), nd * 4)) < 0) return rc;
      RowMeta cm = meta_at(x, L.Cp_meta);
      float* Cp = at<float>(x, L.Cp);
      launch_gather_rows(x->cs, Xp, at<int>(x, L.done_idx), rslot, rpos, nd, Cp, cm, d);
      head<T>(Cp, nd, cm);
    }
    pf_tiles_ = 0;
    pf_key_rows_ = 0;
    CK(cudaGetLastError());
    return CDB_OK;
  }

  int prelude(const PreludePlan& p) override {
    return x_->m.dtype == CDB_BF16 ? prelude_t<__nv_bfloat16>(p) : prelude_t<float>(p);
  }
  template <typename T>
  int prelude_t(const PreludePlan& p) {
    cdb_ctx* x = x_;
    const Layout& L = x->L;
    const int n = (int)p.rows.size(), d = x->m.d_model;
    std::vector<int32_t> a(n), b(n), c(n);
    for (int i = 0; i < n; ++i) {
      a[i] = p.rows[i].slot;
      b[i] = p.rows[i].t;
      c[i] = p.rows[i].pos;
    }
    int rc;
    int *ls = at<int>(x, L.lslot), *lt = at<int>(x, L.lt), *lp = at<int>(x, L.lpos);
    if ((rc = upload(x, ls, a.data(), n * 4)) < 0) return rc;
    if ((rc = upload(x, lt, b.data(), n * 4)) < 0) return rc;
    if ((rc = upload(x, lp, c.data(), n * 4)) < 0) return rc;
    if (x->m.n_prelude == 0 && !x->m.has_adapter) {
      // No prelude layers: the embeddings are the refill rows themselves.
      RowMeta pm = meta_at(x, L.meta[2]);
      pm.slot += p.dst_off;
      pm.pos += p.dst_off;
      pm.t += p.dst_off;
      pm.depth += p.dst_off;
      pm.pend += p.dst_off;
      launch_embed_prelude<T>(x->cs, (const T*)x->embed, d, x->m.vocab, ls, lt, lp, n, at<int>(x, L.out_tok),
                              x->c.max_new_cap, at<float>(x, L.rows[2]) + (size_t)p.dst_off * d, pm, geom(),
                              x->m.r_max, at<int>(x, L.status));
      CK(cudaGetLastError());
      return CDB_OK;
    }
    float* Tp = at<float>(x, L.rows[4]);
    RowMeta tm = meta_at(x, L.meta[4]);
    launch_embed_prelude<T>(x->cs, (const T*)x->embed, d, x->m.vocab, ls, lt, lp, n, at<int>(x, L.out_tok),
                            x->c.max_new_cap, Tp, tm, geom(), x->m.r_max, at<int>(x, L.status));
    double sumL = 0;
    int maxL = 0;
    for (int i = 0; i < n; ++i) sumL += c[i] + 1, maxL = std::max(maxL, c[i] + 1);
    for (int i = 0; i < x->m.n_prelude; ++i)
      block<T>(x->pre[i], Tp, n, tm.slot, tm.pos, nullptr, 1, i, 0, true, sumL, maxL);
    flush<T>();
    launch_prelude_finish(x->cs, Tp, tm, n, at<float>(x, L.rows[2]), meta_at(x, L.meta[2]), p.dst_off,
                          x->m.has_adapter ? at<float>(x, L.estore) : nullptr, d, x->m.has_adapter);
    CK(cudaGetLastError());
    return CDB_OK;
  }

  int core(const CorePlan& p) override {
    return x_->m.dtype == CDB_BF16 ? core_t<__nv_bfloat16>(p) : core_t<float>(p);
  }
  template <typename T>
  int core_t(const CorePlan& p) {
    cdb_ctx* x = x_;
    const Layout& L = x->L;
    const int d = x->m.d_model, B = p.B;
    float* X = at<float>(x, L.rows[0]);
    RowMeta mx = meta_at(x, L.meta[0]);
    const bool conv = x->m.gate_kind == CDB_GATE_CONVERGENCE;
    x->in_core = true;
    struct CoreScope {
      cdb_ctx* c;
      ~CoreScope() { c->in_core = false; }
    } scope{x};
    float* sprev = conv ? at<float>(x, L.sprev) : nullptr;  // s_{d-1}, kept for the convergence exit
    launch_gather_core(x->cs, at<float>(x, L.rows[1]), meta_at(x, L.meta[1]), p.B_cont, at<float>(x, L.rows[2]),
                       meta_at(x, L.meta[2]), p.n_ref, X, mx, d, sprev);
    if (x->m.has_adapter) adapter_step<T>(X, B, at<float>(x, L.estore), 1, mx.slot);
    double sumL = 0;
    int maxL = 0;
    for (const Tok& t : *p.rows) sumL += t.pos + 1, maxL = std::max(maxL, t.pos + 1);
    for (int l = 0; l < x->m.n_core; ++l)
      block<T>(x->core[l], X, B, mx.slot, mx.pos, mx.depth, 0, x->m.n_prelude + l * core_slots(&x->m),
               core_slots(&x->m), true, sumL, maxL);
    flush<T>();
    const int ri = (int)(p.step % kRing);
    uint8_t* ring = at<uint8_t>(x, L.ring) + (size_t)ri * x->c.W;
    launch_gate<T>(x->cs, X, sprev, (const T*)x->gate_w, x->m.gate_bias, x->m.gate_threshold, x->m.rms_eps, B, d,
                   mx, x->c.mode, x->m.r_min, x->m.r_max, at<int8_t>(x, L.fexit), x->c.max_new_cap,
                   at<int>(x, L.pend_new), ring, x->c.trace_gate ? at<float>(x, L.gtrace) : nullptr);
    launch_compact(x->cs, X, mx, at<int>(x, L.pend_new), B, d, x->m.r_max, p.qc_off, at<float>(x, L.rows[1]),
                   meta_at(x, L.meta[1]), at<float>(x, L.rows[3]), meta_at(x, L.meta[3]), geom(),
                   at<int8_t>(x, L.out_depth), x->c.max_new_cap,
                   core_slots(&x->m) == x->m.r_max ? x->m.n_core : 0,  // gaps exist only with one slot per step
                   x->m.n_prelude, x->m.head_dim,
                   (int)sizeof(T), at<int>(x, L.status));
    CK(cudaGetLastError());
    // Lookahead flags to the host on the prep stream.
    CK(cudaEventRecord(x->ev_core[ri], x->cs));
    CK(cudaStreamWaitEvent(x->ps, x->ev_core[ri], 0));
    CK(cudaMemcpyAsync(x->pend_host + (size_t)ri * x->c.W, ring, x->c.W, cudaMemcpyDeviceToHost, x->ps));
    x->io_d2h += x->c.W;
    CK(cudaEventRecord(x->ev_flags[ri], x->ps));
    return CDB_OK;
  }

  int core_flags(int64_t step, std::vector<uint8_t>& pend) override {
    cdb_ctx* x = x_;
    const int ri = (int)(step % kRing);
    int rc = wait_event(x, x->ev_flags[ri], 600.0);
    if (rc < 0) return rc;
    pend.assign(x->pend_host + (size_t)ri * x->c.W, x->pend_host + (size_t)(ri + 1) * x->c.W);
    return CDB_OK;
  }

  int coda(const std::vector<Tok>& rows) override {
    return x_->m.dtype == CDB_BF16 ? coda_t<__nv_bfloat16>(rows) : coda_t<float>(rows);
  }
  template <typename T>
  int coda_t(const std::vector<Tok>& rows) {
    cdb_ctx* x = x_;
    const Layout& L = x->L;
    const int n = (int)rows.size(), d = x->m.d_model;
    float* Cb = at<float>(x, L.rows[3]);
    RowMeta mb = meta_at(x, L.meta[3]);
    const float* Hrows = Cb;
    if (x->m.n_coda > 0) {
      float* Tc = at<float>(x, L.rows[4]);
      launch_copy_rows(x->cs, Cb, Tc, n, d);
      const int cbase = x->m.n_prelude + x->m.n_core * core_slots(&x->m);
      double sumL = 0;
      int maxL = 0;
      for (const Tok& t : rows) sumL += t.pos + 1, maxL = std::max(maxL, t.pos + 1);
      for (int j = 0; j < x->m.n_coda; ++j)
        block<T>(x->coda[j], Tc, n, mb.slot, mb.pos, nullptr, 1, cbase + j, 0, true, sumL, maxL);
      flush<T>();
      Hrows = Tc;
    }
    head<T>(Hrows, n, mb);
    CK(cudaGetLastError());
    return CDB_OK;
  }

  int finish(const Seq& s) override {
    cdb_ctx* x = x_;
    const Layout& L = x->L;
    int rc = harvest_slot(s.slot, true);
    if (rc < 0) return rc;
    const int cap = x->c.max_new_cap, slot = s.slot;
    char* h = x->res_host + (size_t)slot * x->res_stride;
    size_t o = 0;
    CK(cudaMemcpyAsync(h + o, at<int>(x, L.out_tok) + (size_t)slot * cap, cap * 4, cudaMemcpyDeviceToHost, x->cs));
    o += cap * 4;
    CK(cudaMemcpyAsync(h + o, at<int8_t>(x, L.out_depth) + (size_t)slot * cap, cap, cudaMemcpyDeviceToHost, x->cs));
    o += (cap + 15) / 16 * 16;
    if (x->c.trace_gate) {
      size_t n = (size_t)cap * x->m.r_max * 4;
      CK(cudaMemcpyAsync(h + o, at<float>(x, L.gtrace) + (size_t)slot * cap * x->m.r_max, n, cudaMemcpyDeviceToHost,
                         x->cs));
      o += n;
    }
    if (x->c.trace_tokens > 0) {
      size_t n = (size_t)x->c.trace_tokens * x->m.vocab * 4;
      CK(cudaMemcpyAsync(h + o, at<float>(x, L.ltrace) + (size_t)slot * x->c.trace_tokens * x->m.vocab, n,
                         cudaMemcpyDeviceToHost, x->cs));
      o += n;
      n = (size_t)x->c.trace_tokens * x->m.d_model * 4;
      CK(cudaMemcpyAsync(h + o, at<float>(x, L.htrace) + (size_t)slot * x->c.trace_tokens * x->m.d_model, n,
                         cudaMemcpyDeviceToHost, x->cs));
    }
    x->io_d2h += (int64_t)o + (x->c.trace_tokens > 0 ? (int64_t)x->c.trace_tokens * x->m.d_model * 4 : 0);
    PendingResult& pr = x->pending[slot];
    CK(cudaEventRecord(pr.ev, x->cs));
    pr.id = s.id;
    pr.slot = slot;
    pr.n_tokens = s.max_new;
    pr.active = 1;
    return CDB_OK;
  }

  // Move a finished sequence's results from pinned staging to the host list.
  int harvest_slot(int slot, bool block_) {
    cdb_ctx* x = x_;
    PendingResult& pr = x->pending[slot];
    if (!pr.active) return CDB_OK;
    if (!block_ && cudaEventQuery(pr.ev) != cudaSuccess) return CDB_OK;
    int rc = wait_event(x, pr.ev, 600.0);
    if (rc < 0) return rc;
    const int cap = x->c.max_new_cap;
    const char* h = x->res_host + (size_t)slot * x->res_stride;
    HostResult r;
    r.id = pr.id;
    r.n_tokens = pr.n_tokens;
    r.tokens.assign((const int32_t*)h, (const int32_t*)h + pr.n_tokens);
    size_t o = cap * 4;
    r.depths.assign((const int8_t*)(h + o), (const int8_t*)(h + o) + (pr.n_tokens > 0 ? pr.n_tokens - 1 : 0));
    o += (cap + 15) / 16 * 16;
    if (x->c.trace_gate) {
      const float* g = (const float*)(h + o);
      r.gate.assign(g, g + (size_t)(pr.n_tokens - 1) * x->m.r_max);
      o += (size_t)cap * x->m.r_max * 4;
    }
    if (x->c.trace_tokens > 0) {
      const float* g = (const float*)(h + o);
      r.logits.assign(g, g + (size_t)x->c.trace_tokens * x->m.vocab);
      o += (size_t)x->c.trace_tokens * x->m.vocab * 4;
      g = (const float*)(h + o);
      r.hidden.assign(g, g + (size_t)x->c.trace_tokens * x->m.d_model);
    }
    x->ready.push_back(std::move(r));
    pr.active = 0;
    return CDB_OK;
  }

  KvGeom geom() {
    cdb_ctx* x = x_;
    KvGeom g;
    g.pool = x->base + x->L.pool;
    g.bt = at<int>(x, x->L.bt);
    g.etab = at<uint8_t>(x, x->L.etab);
    g.max_blocks = x->L.max_blocks;
    g.kv_blocks = x->c.kv_blocks;
    g.nsl = x->L.nsl;
    g.d = x->m.d_model;
    return g;
  }

 private:
  cdb_ctx* x_;
  bool decode_tiles_ = true;  // GEMM tiling for the rows being processed
  int pf_tiles_ = 0;          // query tiles of the prefill chunk being processed
  double pf_key_rows_ = 0;    // key rows those tiles read (each tile: its last position + 1)
  // Relaunch the kernels of class cls in this core step (cdb_profile_repeat).
  bool repeat(int cls) const { return x_->in_core && x_->prof_repeat == cls; }
};

// Names of the device status bits that are set, for the error message.
static std::string status_text(int st) {
  static const struct {
    int bit;
    const char* name;
  } names[] = {{kStatusBadBlock, "block table entry out of range"},
               {kStatusBadDepth, "loop depth out of range"},
               {kStatusBadToken, "token id out of range"},
               {kStatusBadRow, "row, slot or position out of range"},
               {kStatusNaN, "non-finite value"},
               {kStatusTimeout, "bounded wait expired"},
               {kStatusBadLaunch, "unsupported launch shape"}};
  std::string out;
  for (const auto& n : names)
    if (st & n.bit) out += (out.empty() ? "" : "; ") + std::string(n.name);
  return out.empty() ? "unknown" : out;
}

static int check_status(cdb_ctx* x) {
  int st = 0;
  cudaError_t e = cudaMemcpyAsync(&st, at<int>(x, x->L.status), 4, cudaMemcpyDeviceToHost, x->cs);
  if (e != cudaSuccess) return cuda_fail(x, e, "status copy");
  x->io_d2h += 4;
  e = cudaStreamSynchronize(x->cs);
  if (e != cudaSuccess) return cuda_fail(x, e, "cudaStreamSynchronize");
  if (st != 0) {
    x->err = "device bounds check failed (status " + std::to_string(st) + ": " + status_text(st) + ")";
    x->dead = true;
    return CDB_ERR_DEVICE_BOUNDS;
  }
  return CDB_OK;
}

static bool valid_hd(int hd) { return hd == 8 || hd == 16 || hd == 32 || hd == 64 || hd == 96 || hd == 128; }

}  // namespace cdb

using namespace cdb;

extern "C" {

size_t cdb_arena_bytes(const cdb_model_desc* m, const cdb_sched_cfg* c) {
  if (!m || !c) return 0;
  Layout L;
  plan_layout(m, c, &L);
  return L.total;
}

size_t cdb_kv_bytes_per_token(const cdb_model_desc* m) {
  if (!m) return 0;
  const size_t es = m->dtype == CDB_BF16 ? 2 : 4;
  const size_t slots = (size_t)m->n_prelude + m->n_coda + (size_t)m->n_core * core_slots(m);
  return slots * 2 * (size_t)m->d_model * es;
}

int cdb_init(const cdb_model_desc* m, const cdb_weights* w, const cdb_sched_cfg* c, cdb_ctx** out) {
  if (!m || !w || !c || !out) return CDB_ERR_ARG;
  *out = nullptr;
  if (m->vocab < 2 || m->d_model < 4 || m->n_heads < 1 || m->d_model != m->n_heads * m->head_dim ||
      m->d_model % 4 != 0 || !valid_hd(m->head_dim) || m->ffn < 1 || m->n_core < 1 || m->n_prelude < 0 ||
      m->n_coda < 0 || m->r_min < 2 || m->r_max < m->r_min || m->r_max > CDB_MAX_DEPTH || m->kv_slots < 0 ||
      m->kv_slots > m->r_max || m->gate_kind < CDB_GATE_PROBE || m->gate_kind > CDB_GATE_CONVERGENCE ||
      (m->gate_kind == CDB_GATE_CONVERGENCE && m->r_min < 3) ||
      (m->dtype != CDB_FP32 && m->dtype != CDB_BF16) || (m->has_adapter && !w->adapter))
    return CDB_ERR_ARG;
  if (c->W < 1 || c->M < 1 || c->K < 1 || c->kv_blocks < 1 || c->max_ctx < 1 || c->max_new_cap < 1 ||
      c->mode < 0 || c->mode > 2 || c->trace_tokens < 0 || !c->arena || ((uintptr_t)c->arena % kAlign) != 0 ||
      c->attn_split < 0 || c->attn_split % 16 != 0 || (c->S > c->W))
    return CDB_ERR_ARG;
  if (!w->embed || !w->lm_head || !w->final_norm || (m->gate_kind == CDB_GATE_PROBE && !w->gate_w) ||
      (m->n_core > 0 && !w->core) ||
      (m->n_prelude > 0 && !w->prelude) || (m->n_coda > 0 && !w->coda))
    return CDB_ERR_ARG;
  std::unique_ptr<cdb_ctx> x(new cdb_ctx);
  x->m = *m;
  x->c = *c;
  plan_layout(m, c, &x->L);
  if (c->arena_bytes < x->L.total) return CDB_ERR_ARENA;
  if (x->c.S <= 0) x->c.S = x->L.S;
  x->base = (char*)c->arena;
  auto cp = [](const cdb_layer_weights* a, int n, std::vector<LayerW>& v) {
    for (int i = 0; i < n; ++i)
      v.push_back({a[i].attn_norm, a[i].wqkv, a[i].wo, a[i].mlp_norm, a[i].wg, a[i].wu, a[i].wd});
  };
  cp(w->prelude, m->n_prelude, x->pre);
  cp(w->core, m->n_core, x->core);
  cp(w->coda, m->n_coda, x->coda);
  for (auto* v : {&x->pre, &x->core, &x->coda})
    for (auto& lw : *v)
      if (!lw.attn_norm || !lw.wqkv || !lw.wo || !lw.mlp_norm || !lw.wg || !lw.wu || !lw.wd) return CDB_ERR_ARG;
  x->embed = w->embed;
  x->lm_head = w->lm_head;
  x->final_norm = w->final_norm;
  x->gate_w = w->gate_w;
  x->adapter = w->adapter;
  cdb_ctx* xp = x.get();
  cudaError_t e;
#define CKI(expr)                                   \
  do {                                              \
    e = (expr);                                     \
    if (e != cudaSuccess) {                         \
      cuda_fail(xp, e, #expr);                      \
      return CDB_ERR_CUDA;                          \
    }                                               \
  } while (0)
  x->cs = (cudaStream_t)c->compute_stream;
  x->ps = (cudaStream_t)c->prep_stream;
  if (!x->ps) {
    CKI(cudaStreamCreateWithFlags(&x->ps, cudaStreamNonBlocking));
    x->own_ps = true;
  }
  CKI(cudaMallocHost((void**)&x->stage, (size_t)kStageSegs * kStageSeg));
  for (int i = 0; i < kStageSegs; ++i) CKI(cudaEventCreateWithFlags(&x->seg_ev[i], cudaEventDisableTiming));
  for (int i = 0; i < kStageSegs; ++i) CKI(cudaEventRecord(x->seg_ev[i], x->cs));
  CKI(cudaMallocHost((void**)&x->pend_host, (size_t)kRing * c->W));
  for (int i = 0; i < kRing; ++i) {
    CKI(cudaEventCreateWithFlags(&x->ev_core[i], cudaEventDisableTiming));
    CKI(cudaEventCreateWithFlags(&x->ev_flags[i], cudaEventDisableTiming));
  }
  const size_t cap = c->max_new_cap;
  x->res_stride = cap * 4 + (cap + 15) / 16 * 16 + (c->trace_gate ? cap * m->r_max * 4 : 0) +
                  (size_t)c->trace_tokens * (m->vocab + m->d_model) * 4;
  x->res_stride = (x->res_stride + 255) / 256 * 256;
  CKI(cudaMallocHost((void**)&x->res_host, x->res_stride * c->W));
  x->pending.resize(c->W);
  for (auto& p : x->pending) {
    p.active = 0;
    CKI(cudaEventCreateWithFlags(&p.ev, cudaEventDisableTiming));
  }
  // KV pool to NaN: reading an unwritten exit gap would poison the output.
  const Layout& L = x->L;
  CKI(cudaMemsetAsync(x->base + L.pool, 0xFF, L.etab - L.pool, x->cs));
  CKI(cudaMemsetAsync(x->base + L.etab, 0, L.total - L.etab, x->cs));
  CKI(cudaMemsetAsync(x->base + L.bt, 0xFF, (size_t)c->W * L.max_blocks * 4, x->cs));
  launch_rope_table(x->cs, at<float2>(xp, L.rope), L.max_blocks * 16, m->head_dim, m->rope_theta);
  CKI(cudaGetLastError());
  CKI(cudaStreamSynchronize(x->cs));
#undef CKI
  SchedCfg sc;
  sc.mode = c->mode;
  sc.W = c->W;
  sc.M = c->M;
  sc.S = x->c.S;
  sc.K = c->K;
  sc.r_max = m->r_max;
  sc.r_min = m->r_min;
  sc.kv_blocks = c->kv_blocks;
  sc.kv_headroom = c->kv_headroom;
  sc.max_ctx = c->max_ctx;
  sc.max_new_cap = c->max_new_cap;
  x->exec.reset(new GpuExecutor(xp));
  x->sched.reset(new Scheduler(sc, x->exec.get()));
  *out = x.release();
  return CDB_OK;
}

int cdb_admit(cdb_ctx* x, int64_t seq_id, const int32_t* prompt, int prompt_len, int max_new_tokens,
              const int8_t* force_exit, const int32_t* force_token) {
  if (!x) return CDB_ERR_ARG;
  if (x->dead) return CDB_ERR_STATE;
  if (!prompt) {
    x->err = "prompt is NULL";
    return CDB_ERR_ARG;
  }
  for (int i = 0; i < prompt_len; ++i)
    if (prompt[i] < 0 || prompt[i] >= x->m.vocab) {
      x->err = "prompt token out of range";
      return CDB_ERR_ARG;
    }
  if (force_token)
    for (int i = 0; i < max_new_tokens; ++i)
      if (force_token[i] < -1 || force_token[i] >= x->m.vocab) {
        x->err = "force_token out of range";
        return CDB_ERR_ARG;
      }
  int rc = x->sched->admit(seq_id, prompt, prompt_len, max_new_tokens, force_exit, force_token);
  if (rc < 0) x->err = x->sched->err;
  return rc;
}

int cdb_step_boundary(cdb_ctx* x, cdb_step_info* info) {
  if (!x) return CDB_ERR_ARG;
  if (x->dead) return CDB_ERR_STATE;
  int rc = x->sched->step_boundary(info);
  if (rc < 0) x->err = x->sched->err.empty() ? x->err : x->sched->err;
  return rc;
}

int cdb_step_core(cdb_ctx* x, cdb_step_info* info) {
  if (!x) return CDB_ERR_ARG;
  if (x->dead) return CDB_ERR_STATE;
  int rc = x->sched->step_core(info);
  if (rc < 0) x->err = x->sched->err.empty() ? x->err : x->sched->err;
  return rc;
}

int cdb_sync(cdb_ctx* x) {
  if (!x) return CDB_ERR_ARG;
  if (x->dead) return CDB_ERR_STATE;
  cudaError_t e = cudaStreamSynchronize(x->ps);
  if (e != cudaSuccess) return cuda_fail(x, e, "cudaStreamSynchronize(prep)");
  return check_status(x);
}

static int drain_impl(cdb_ctx* x, cdb_result* buf, int cap, int* n_out, bool block) {
  if (!x || !n_out || (cap > 0 && !buf)) return CDB_ERR_ARG;
  *n_out = 0;
  if (x->dead) return CDB_ERR_STATE;
  int rc = block ? check_status(x) : CDB_OK;  // the status check synchronizes the stream
  if (rc < 0) return rc;
  for (int s = 0; s < x->c.W; ++s) {
    rc = x->exec->harvest_slot(s, block);
    if (rc < 0) return rc;
  }
  int n = 0;
  while (n < cap && !x->ready.empty()) {
    HostResult& r = x->ready.front();
    cdb_result& o = buf[n];
    o.seq_id = r.id;
    o.n_tokens = r.n_tokens;
    if (o.tokens) std::memcpy(o.tokens, r.tokens.data(), r.tokens.size() * 4);
    if (o.exit_depths) std::memcpy(o.exit_depths, r.depths.data(), r.depths.size());
    if (o.gate_logits && !r.gate.empty()) std::memcpy(o.gate_logits, r.gate.data(), r.gate.size() * 4);
    if (o.logits && !r.logits.empty()) std::memcpy(o.logits, r.logits.data(), r.logits.size() * 4);
    if (o.hidden && !r.hidden.empty()) std::memcpy(o.hidden, r.hidden.data(), r.hidden.size() * 4);
    x->ready.pop_front();
    ++n;
  }
  *n_out = n;
  return CDB_OK;
}

int cdb_drain(cdb_ctx* x, cdb_result* buf, int cap, int* n_out) { return drain_impl(x, buf, cap, n_out, true); }

int cdb_poll(cdb_ctx* x, cdb_result* buf, int cap, int* n_out) { return drain_impl(x, buf, cap, n_out, false); }

void cdb_free(cdb_ctx* x) {
  if (!x) return;
  cudaStreamSynchronize(x->cs);
  if (x->ps) cudaStreamSynchronize(x->ps);
  for (int i = 0; i < kStageSegs; ++i) cudaEventDestroy(x->seg_ev[i]);
  for (int i = 0; i < kRing; ++i) {
    cudaEventDestroy(x->ev_core[i]);
    cudaEventDestroy(x->ev_flags[i]);
  }
  for (auto& p : x->pending) cudaEventDestroy(p.ev);
  for (auto& ev : x->prof_live) {
    cudaEventDestroy(ev.a);
    cudaEventDestroy(ev.b);
  }
  for (auto e : x->ev_pool) cudaEventDestroy(e);
  if (x->stage) cudaFreeHost(x->stage);
  if (x->pend_host) cudaFreeHost(x->pend_host);
  if (x->res_host) cudaFreeHost(x->res_host);
  if (x->own_ps) cudaStreamDestroy(x->ps);
  delete x;
}

const char* cdb_last_error(const cdb_ctx* x) { return x ? x->err.c_str() : "null context"; }

int64_t cdb_kernel_launches(void) { return (int64_t)launch_count(); }

int cdb_io_bytes(const cdb_ctx* x, int64_t* h2d, int64_t* d2h) {
  if (!x || !h2d || !d2h) return CDB_ERR_ARG;
  *h2d = x->io_h2d;
  *d2h = x->io_d2h;
  return CDB_OK;
}

int cdb_profile_enable(cdb_ctx* x, int on) {
  if (!x || on < 0 || on > 2) return CDB_ERR_ARG;
  x->prof_on = on != 0;
  x->prof_core_only = on == 2;
  return CDB_OK;
}

int cdb_profile_repeat(cdb_ctx* x, int cls) {
  if (!x || !(cls == -1 || cls == 0 || cls == 1 || cls == 3)) return CDB_ERR_ARG;
  x->prof_repeat = cls;
  return CDB_OK;
}

int cdb_profile_read(cdb_ctx* x, cdb_kernel_stat* out, int cap, int* n_out) {
  if (!x || !n_out || (cap > 0 && !out)) return CDB_ERR_ARG;
  cudaError_t e = cudaStreamSynchronize(x->cs);
  if (e != cudaSuccess) return cuda_fail(x, e, "cudaStreamSynchronize");
  prof_collect(x);
  int n = 0;
  for (int c = 0; c < 5 && n < cap; ++c) {
    std::memset(&out[n], 0, sizeof(out[n]));
    std::strncpy(out[n].name, kProfNames[c], sizeof(out[n].name) - 1);
    out[n].launches = x->stats[c].launches;
    out[n].ms = x->stats[c].ms;
    out[n].bytes = x->stats[c].bytes;
    out[n].flops = x->stats[c].flops;
    x->stats[c] = cdb_ctx::Stat();
    ++n;
  }
  *n_out = n;
  return CDB_OK;
}

int cdb_trace_enable(cdb_ctx* x, int on) {
  if (!x) return CDB_ERR_ARG;
  x->sched->trace_on = on != 0;
  if (!on) x->sched->trace().clear();
  return CDB_OK;
}

int cdb_trace_read(cdb_ctx* x, cdb_trace_row* rows, int cap, int* n_out) {
  if (!x || !n_out) return CDB_ERR_ARG;
  auto& tr = x->sched->trace();
  int n = (int)tr.size() < cap ? (int)tr.size() : cap;
  if (rows && n > 0) std::memcpy(rows, tr.data(), sizeof(cdb_trace_row) * n);
  *n_out = n;
  return CDB_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// cdb_testing.h
// ---------------------------------------------------------------------------
#include "../../include/cdb_testing.h"

extern "C" {

size_t cdb_test_gemm_ws_bytes(int N, int K, int rows, int tiling, int epi) {
  if (N < 1 || K < 1 || rows < 0) return 0;
  (void)K;
  const size_t ldp = epi == 2 ? 2 * (size_t)N : (size_t)N;
  return 256 + (tiling == 0 || tiling == 3 ? (size_t)kGemmMaxSplits * rows * ldp * 4 : 0);
}

int cdb_test_gemm(int epi, int tiling, const void* A, int lda, int a_rows, const void* W, const void* W2, int N,
                  int K, int rows, float* Cf, void* Ct, int ldc, void* ws, size_t ws_bytes, void* stream) {
  if (epi < 0 || epi > 2 || tiling < 0 || tiling > 3 || !A || !W || (epi == 2 && (!W2 || !Ct)) ||
      (epi != 2 && !Cf) || !ws || ws_bytes < cdb_test_gemm_ws_bytes(N, K, rows, tiling, epi))
    return CDB_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int* status = (int*)ws;
  float* parts = (float*)((char*)ws + 256);
  if (cudaMemsetAsync(status, 0, 4, s) != cudaSuccess) return CDB_ERR_CUDA;
  if (tiling == 2) {
    launch_gemm<__nv_bfloat16>(s, epi, (const __nv_bfloat16*)A, lda, (const __nv_bfloat16*)W,
                               (const __nv_bfloat16*)W2, N, K, rows, Cf, (__nv_bfloat16*)Ct, ldc);
  } else {
    // The decode tiling leaves split-K partials for a consumer; fold them here
    // the way the engine's consumers do (split order, then the epilogue).
    const int ns = launch_gemm_tc(s, epi, (const __nv_bfloat16*)A, lda, a_rows, (const __nv_bfloat16*)W,
                                  (const __nv_bfloat16*)W2, N, K, rows, Cf, (__nv_bfloat16*)Ct, ldc,
                                  tiling == 0 ? kTileSplit : tiling == 1 ? kTilePrefill : kTileWide,
                                  tiling == 0 || tiling == 3 ? parts : nullptr, (ws_bytes - 256) / 4, status);
    if (ns < 0) return CDB_ERR_ARG;
    if (ns > 0) {
      if (epi == 2) launch_swiglu_combine<__nv_bfloat16>(s, parts, ns, rows, N, (__nv_bfloat16*)Ct);
      else launch_fold(s, parts, ns, rows, N, Cf, ldc, epi == 1 ? 1 : 2);
    }
  }
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return CDB_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CDB_ERR_CUDA;
  return st ? CDB_ERR_DEVICE_BOUNDS : CDB_OK;
}

size_t cdb_test_attention_scratch_bytes(int rows, int n_heads, int head_dim, int split, int max_ctx) {
  if (rows < 0 || n_heads < 1 || head_dim < 1 || split < 1 || max_ctx < 1) return 0;
  const size_t ms = (size_t)(max_ctx + split - 1) / split;
  const size_t po = (size_t)rows * n_heads * ms * head_dim * 4;
  return 256 + (po + 255) / 256 * 256 + (size_t)rows * n_heads * ms * 2 * 4;
}

static int test_attention(const void* q, int rows, const int32_t* slot, const int32_t* pos, const int32_t* depth,
                          const void* kv_pool, const int32_t* block_table, int max_blocks, const uint8_t* exit_table,
                          int kv_blocks, int n_kv_slots, int slot_base, int n_heads, int head_dim, int dtype, int split,
                          int max_ctx, void* out, void* scratch, size_t scratch_bytes, void* stream, bool uniform) {
  if (!q || rows < 1 || !slot || !pos || !depth || !kv_pool || !block_table || max_blocks < 1 ||
      (!exit_table && !uniform) || kv_blocks < 1 || n_kv_slots < 1 || slot_base < 0 || n_heads < 1 ||
      !valid_hd(head_dim) || (dtype != CDB_FP32 && dtype != CDB_BF16) || split < 16 || split % 16 != 0 ||
      max_ctx < 1 || !out || !scratch ||
      scratch_bytes < cdb_test_attention_scratch_bytes(rows, n_heads, head_dim, split, max_ctx))
    return CDB_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)scratch;
  int* status = (int*)w;
  const size_t ms = (size_t)(max_ctx + split - 1) / split;
  float* part_o = (float*)(w + 256);
  float* part_ml = (float*)(w + 256 + ((size_t)rows * n_heads * ms * head_dim * 4 + 255) / 256 * 256);
  if (cudaMemsetAsync(status, 0, kStatusBytes, s) != cudaSuccess) return CDB_ERR_CUDA;
  KvGeom g;
  g.pool = const_cast<void*>(kv_pool);
  g.bt = block_table;
  g.etab = const_cast<uint8_t*>(exit_table);
  g.max_blocks = max_blocks;
  g.kv_blocks = kv_blocks;
  g.nsl = n_kv_slots;
  g.d = n_heads * head_dim;
  if (dtype == CDB_BF16)
    launch_attention<__nv_bfloat16>(s, (const __nv_bfloat16*)q, rows, slot, pos, depth, 0, g, slot_base, kNoSlotCap, n_heads,
                                    head_dim, split, (int)ms, (__nv_bfloat16*)out, part_o, part_ml, status, uniform);
  else
    launch_attention<float>(s, (const float*)q, rows, slot, pos, depth, 0, g, slot_base, kNoSlotCap, n_heads, head_dim,
                            split, (int)ms, (float*)out, part_o, part_ml, status, uniform);
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return CDB_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CDB_ERR_CUDA;
  return st ? CDB_ERR_DEVICE_BOUNDS : CDB_OK;
}

int cdb_test_attention_prefill(const void* q, int rows, const int32_t* row_slot, const int32_t* row_pos,
                               const void* kv_pool, const int32_t* block_table, int max_blocks, int kv_blocks,
                               int n_kv_slots, int slot, int n_heads, int head_dim, void* out, void* scratch,
                               size_t scratch_bytes, void* stream) {
  if (!q || rows < 1 || !row_slot || !row_pos || !kv_pool || !block_table || max_blocks < 1 || kv_blocks < 1 ||
      n_kv_slots < 1 || slot < 0 || slot >= n_kv_slots || n_heads < 1 || !out || !scratch)
    return CDB_ERR_ARG;
  for (int i = 0; i < rows; ++i)
    if (row_slot[i] < 0 || row_pos[i] < 0 || row_pos[i] >= max_blocks * 16) return CDB_ERR_ARG;
  const std::vector<int4> tiles = prefill_tiles(row_slot, row_pos, rows, head_dim);
  if (scratch_bytes < 256 + tiles.size() * sizeof(int4)) return CDB_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int* status = (int*)scratch;
  int4* dt = (int4*)((char*)scratch + 256);
  if (cudaMemsetAsync(status, 0, kStatusBytes, s) != cudaSuccess ||
      cudaMemcpyAsync(dt, tiles.data(), tiles.size() * sizeof(int4), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return CDB_ERR_CUDA;
  KvGeom g;
  g.pool = const_cast<void*>(kv_pool);
  g.bt = block_table;
  g.etab = nullptr;
  g.max_blocks = max_blocks;
  g.kv_blocks = kv_blocks;
  g.nsl = n_kv_slots;
  g.d = n_heads * head_dim;
  if (!launch_prefill_attention(s, (const __nv_bfloat16*)q, rows, dt, (int)tiles.size(), g, slot, n_heads, head_dim,
                                (__nv_bfloat16*)out, status))
    return CDB_ERR_ARG;
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return CDB_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CDB_ERR_CUDA;
  return st ? CDB_ERR_DEVICE_BOUNDS : CDB_OK;
}

int cdb_test_kv_pool(const cdb_ctx* x, void** pool, int* kv_blocks, int* n_kv_slots) {
  if (!x || !pool || !kv_blocks || !n_kv_slots) return CDB_ERR_ARG;
  *pool = x->base + x->L.pool;
  *kv_blocks = x->c.kv_blocks;
  *n_kv_slots = x->L.nsl;
  return CDB_OK;
}

int cdb_test_attention(const void* q, int rows, const int32_t* slot, const int32_t* pos, const int32_t* depth,
                       const void* kv_pool, const int32_t* block_table, int max_blocks, const uint8_t* exit_table,
                       int kv_blocks, int n_kv_slots, int slot_base, int n_heads, int head_dim, int dtype, int split,
                       int max_ctx, void* out, void* scratch, size_t scratch_bytes, void* stream) {
  return test_attention(q, rows, slot, pos, depth, kv_pool, block_table, max_blocks, exit_table, kv_blocks,
                        n_kv_slots, slot_base, n_heads, head_dim, dtype, split, max_ctx, out, scratch, scratch_bytes,
                        stream, false);
}

int cdb_test_attention_uniform(const void* q, int rows, const int32_t* slot, const int32_t* pos, const int32_t* depth,
                               const void* kv_pool, const int32_t* block_table, int max_blocks, int kv_blocks,
                               int n_kv_slots, int slot_base, int n_heads, int head_dim, int dtype, int split,
                               int max_ctx, void* out, void* scratch, size_t scratch_bytes, void* stream) {
  return test_attention(q, rows, slot, pos, depth, kv_pool, block_table, max_blocks, nullptr, kv_blocks, n_kv_slots,
                        slot_base, n_heads, head_dim, dtype, split, max_ctx, out, scratch, scratch_bytes, stream,
                        true);
}

}  // extern "C"
