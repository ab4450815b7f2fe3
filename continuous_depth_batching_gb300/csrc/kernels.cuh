// Device kernels of the CDB hot path and their host launchers.
//
// Layouts (all device memory, carved from the caller's arena):
//   row buffers   fp32 [rows][d]      residual / core state of each row
//   row metadata  int32 per row       slot (sequence slot), pos, t (decode
//                                     forward index), depth (loop steps
//                                     completed before this step), pend
//                                     (lookahead flag from the previous step)
//   KV pool       T [kv_blocks][NSL][2][16][d]   NSL = n_prelude + n_core*r_max
//                 + n_coda slots per token; core layer l, loop step r lives in
//                 slot n_prelude + l*r_max + r-1 (depth-indexed cache, §4.2 of
//                 "Depth-adaptive Inference of Looped Language Models via
//                 Continuous Depth Batching")
//   exit table    uint8 [kv_blocks][16]  exit depth of each cached position
//                 (r_max for prompt positions and tokens still in flight)
//   block table   int32 [W][max_blocks]  logical block -> physical block
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace cdb {

// Kernel launches issued by the launchers below (process-wide).
void count_launch(int n = 1);
long long launch_count();

struct RowMeta {
  int* slot;
  int* pos;
  int* t;
  int* depth;
  int* pend;
};

// Device status word bits (set by bounds checks instead of trapping).
enum : int {
  kStatusBadBlock = 1,
  kStatusBadDepth = 2,
  kStatusBadToken = 4,
  kStatusBadRow = 8,
  kStatusNaN = 16,
  kStatusTimeout = 32,   // a bounded wait inside a kernel expired
  kStatusBadLaunch = 64, // a kernel was launched in a shape it does not support
};
// The status area is kStatusBytes of zeroed device memory: word 0 holds the
// bits above; words kWorkCounter and kWorkCounter + 1 are the work queue of
// the persistent attention kernel, which leaves them at zero after each launch.
constexpr int kStatusBytes = 256;
constexpr int kWorkCounter = 32;

struct KvGeom {
  void* pool;            // T elements
  const int* bt;         // [W][max_blocks]
  uint8_t* etab;         // [kv_blocks][16]
  int max_blocks, kv_blocks, nsl, d;
};

// ---- elementwise / bookkeeping (kernels.cu) ----
template <typename T>
void launch_embed_prefill(cudaStream_t s, const T* E, int d, int V, const int* rslot,
                          const int* rpos, const int* rtok, int rows, float* X, KvGeom kv,
                          int r_max, int* status);
template <typename T>
void launch_embed_prelude(cudaStream_t s, const T* E, int d, int V, const int* lslot,
                          const int* lt, const int* lpos, int rows, const int* out_tok,
                          int max_new_cap, float* X, RowMeta meta, KvGeom kv, int r_max,
                          int* status);
void launch_prelude_finish(cudaStream_t s, const float* Tp, RowMeta tmeta, int rows, float* Pb,
                           RowMeta pmeta, int dst_off, float* estore, int d, int adapter);
template <typename T>
// A = RMSNorm(X) * g.  With ns > 0 pending GEMM partials P (split stride
// rows * d) are folded into X first: mode 1 X += sum, mode 2 X = sum.  A may be
// null (fold only).
void launch_rmsnorm(cudaStream_t s, float* X, const T* g, T* A, int rows, int d, float eps,
                    int lda, const float* P, int ns, int mode);
// C (row stride ldc) = sum of ns partials [split][row][n] (mode 2) or C + sum (mode 1).
void launch_fold(cudaStream_t s, const float* P, int ns, int rows, int n, float* C, int ldc, int mode);
// Mid = silu(sum of gate partials) * (sum of up partials), from the ns split-K
// partials of the gate/up GEMM ([split][row][2f], up at +f).
template <typename T>
void launch_swiglu_combine(cudaStream_t s, const float* P, int ns, int rows, int f, T* Mid);
template <typename T>
void launch_concat(cudaStream_t s, const float* E, int e_per_slot, const int* mslot,
                   const float* X, T* A, int rows, int d);
template <typename T>
// QKV: ns split-K partials [split][row][3d] (ns <= 1: the plain GEMM output).
void launch_rope_kv(cudaStream_t s, const float* QKV, int ns, int rows, const int* mslot,
                    const int* mpos, const int* mdepth, int depth_uniform, int slot_base,
                    int clamp, T* Q, KvGeom kv, int H, int hd, const float2* rope,
                    int* status);
// Exit gate after a loop step.  Sprev == nullptr: linear probe z = w . rmsnorm(X) + bias, fires
// when z > thr; otherwise the convergence statistic c = ||X - Sprev|| / ||X||, fires when c < thr.
template <typename T>
void launch_gate(cudaStream_t s, const float* X, const float* Sprev, const T* w, float bias, float thr, float eps,
                 int rows, int d, RowMeta meta, int mode, int r_min, int r_max,
                 const int8_t* fexit, int max_new_cap, int* pend_new, uint8_t* ring,
                 float* gtrace);
// Compaction of the core batch after the exit gate, plus the exit-gap fill of
// the n_core core layers (KV slots core_slot0 + l * r_max + r - 1).
void launch_compact(cudaStream_t s, const float* X, RowMeta m, const int* pend_new, int B,
                    int d, int r_max, int qc_off, float* Xc, RowMeta mc, float* Cb,
                    RowMeta mb, KvGeom kv, int8_t* out_depth, int max_new_cap, int n_core,
                    int core_slot0, int hd, int es, int* status);
// Core batch = continuing rows then refills; Sprev (nullable) receives a copy of the gathered states.
void launch_gather_core(cudaStream_t s, const float* Xc, RowMeta mc, int B_cont, const float* Pb,
                        RowMeta mp, int n_ref, float* X, RowMeta mx, int d, float* Sprev);
void launch_gather_rows(cudaStream_t s, const float* src, const int* idx, const int* rslot,
                        const int* rpos, int n, float* dst, RowMeta md, int d);
void launch_argmax(cudaStream_t s, const float* logits, int rows, int V, RowMeta m,
                   const int* ftok, int max_new_cap, int* out_tok, float* ltrace,
                   int trace_T, const float* H, float* htrace, int d, int* status);
void launch_rope_table(cudaStream_t s, float2* tab, int max_ctx, int hd, float theta);
void launch_copy_rows(cudaStream_t s, const float* src, float* dst, int rows, int d);

// Slot of a row at loop step r in a layer whose cache starts at slot_base:
// clamp (the slot cap, s of App. E.1) 0 = the layer's single slot, else
// slot_base + min(r, clamp) - 1.  kNoSlotCap: one slot per loop step.
constexpr int kNoSlotCap = 1 << 20;

// ---- attention (attention.cu) ----
// Decode (and prefill) attention.  uniform: every key of a row is read from
// one slot (slot_base + r - 1 with clamp, slot_base without), which holds
// whenever exit gaps are filled (k_compact); otherwise key j is read from
// step min(r, e_j) through the exit-depth table.
template <typename T>
void launch_attention(cudaStream_t s, const T* Q, int rows, const int* mslot, const int* mpos,
                      const int* mdepth, int depth_uniform, KvGeom kv, int slot_base,
                      int clamp, int H, int hd, int split, int max_splits, T* O,
                      float* part_o, float* part_ml, int* status, bool uniform);
// The same decode attention (bf16, every key of a row from one slot) with the
// RoPE / KV write of its rows folded in: q, k and v come from the QKV GEMM's
// ns split-K partials [split][row][3d] (ns <= 1: the plain output), rotated
// and rounded exactly as launch_rope_kv does; the token's K and V rows are
// stored in the pool.  Returns false (nothing launched) for shapes the fused
// kernel does not cover; the caller then runs launch_rope_kv and
// launch_attention.  attention_rope_fusable: whether it covers this cache
// geometry (decided once per engine, so every step takes the same path).
bool attention_rope_fusable(KvGeom kv, int H, int hd, int split);
bool launch_attention_rope(cudaStream_t s, const float* QKV, int ns, int rows, const int* mslot, const int* mpos,
                           const int* mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int hd,
                           int split, int max_splits, const float2* rope, __nv_bfloat16* O, float* part_o,
                           float* part_ml, int* status);

// Causal prefill attention over query tiles (bf16, head_dim 32/64/96/128):
// tiles[t] = (first row, rows <= prefill_tile_rows(hd), sequence slot,
// position of the first row); rows of a tile are consecutive positions of one
// sequence, and every key is read from KV slot `slot`.  Q and O are
// [q_rows][d].  head_dim 64 and 128 run on the tensor cores (tcgen05, 128-row
// tiles, attention_prefill_tc.cu); 32 and 96 on warp-level MMAs (64-row
// tiles).  Returns false (nothing launched) for shapes it does not cover.
constexpr int kPrefillTileRows = 64;
constexpr int kPrefillTileRowsTc = 128;
inline int prefill_tile_rows(int hd) { return hd == 64 || hd == 128 ? kPrefillTileRowsTc : kPrefillTileRows; }
bool launch_prefill_attention(cudaStream_t s, const __nv_bfloat16* Q, int q_rows, const int4* tiles, int n_tiles,
                              KvGeom kv, int slot, int H, int hd, __nv_bfloat16* O, int* status);
bool launch_prefill_attention_tc(cudaStream_t s, const __nv_bfloat16* Q, int q_rows, const int4* tiles, int n_tiles,
                                 KvGeom kv, int slot, int H, int hd, __nv_bfloat16* O, int* status);
// Query tiles of a prefill chunk (rows given by sequence slot and position,
// runs of consecutive positions of one sequence), longest key range first so
// the heaviest tiles start first.
std::vector<int4> prefill_tiles(const int32_t* row_slot, const int32_t* row_pos, int rows, int hd);

// ---- GEMM (gemm_simt.cu) ----
enum GemmEpi { kEpiStore = 0, kEpiResid = 1, kEpiSwiglu = 2 };
// C = A[rows, K] . W[N, K]^T with fp32 accumulation.  kEpiStore: Cf[r][c] = acc;
// kEpiResid: Cf[r][c] += acc; kEpiSwiglu: Ct[r][c] = silu(A.W^T) * (A.W2^T).
template <typename T>
void launch_gemm(cudaStream_t s, int epi, const T* A, int lda, const T* W, const T* W2, int N,
                 int K, int rows, float* Cf, T* Ct, int ldc);

// ---- tensor-core GEMM (gemm_tc.cu), bf16 only ----
// kTileSplit: split-K fixed by the weight shape; kTileWide: split-K (at most
// kWideMaxSplits, fixed by the weight shape) for narrow weights only;
// kTilePrefill: one split.  With ws (room for ws_floats)
// and more than one split, each split's fp32 partial goes to
// ws[split][row][ldp] (ldp = N, or 2N for SwiGLU with the up projection at
// +N) and the epilogue is left to the consumer (sum the partials in split
// order, then apply it); the return value is then the split count.  Returns 0
// when the epilogue was applied in place, -1 when the shape is unsupported.
// a_rows: rows allocated in A (TMA bounds).
constexpr int kGemmMaxSplits = 16;
constexpr int kWideMaxSplits = 4;

// Split-K partials of a GEMM output: P[split][row][ld] with split stride ss;
// their sum in split order (the reduction every consumer uses, so a value is
// the same whichever kernel folds it).
struct Parts {
  const float* P;
  int ns;     // number of partials (<= kGemmMaxSplits); 0 = nothing to fold
  size_t ss;  // floats between consecutive splits
  int ld;     // floats between consecutive rows
  // Sum of columns c..c+3 of `row` (c and ld multiples of 4): every partial
  // is loaded before the first add, then added in split order.  The loop is
  // unrolled for at most S partials (S >= ns).
  template <int S>
  __device__ __forceinline__ float4 sum4_upto(int row, int c) const {
    const float4* p = reinterpret_cast<const float4*>(P + (size_t)row * ld + c);
    const size_t s4 = ss / 4;
    float4 v[S];
#pragma unroll
    for (int q = 0; q < S; ++q) v[q] = q < ns ? p[q * s4] : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < S; ++q)
      if (q < ns) {
        g.x += v[q].x;
        g.y += v[q].y;
        g.z += v[q].z;
        g.w += v[q].w;
      }
    return g;
  }
  // The same sum; the unroll depth follows ns (uniform across the grid).
  __device__ __forceinline__ float4 sum4(int row, int c) const {
    if (ns <= 4) return sum4_upto<4>(row, c);
    if (ns <= 8) return sum4_upto<8>(row, c);
    return sum4_upto<kGemmMaxSplits>(row, c);
  }
};

// Rotate-half RoPE of the pair (a, b) = (x_j, x_{j + hd/2}) by the angle whose
// (cos, sin) is cs.  Both products are rounded before the add, so every kernel
// that rotates a value gets the same bits.
__device__ __forceinline__ void rope_pair(float a, float b, float2 cs, float& lo, float& hi) {
  lo = __fsub_rn(__fmul_rn(a, cs.x), __fmul_rn(b, cs.y));
  hi = __fadd_rn(__fmul_rn(b, cs.x), __fmul_rn(a, cs.y));
}

// Tilings: kTileSplit = 64-row tiles with split-K (decode batches below the
// wide threshold); kTilePrefill = persistent, 256-row tiles (128 for SwiGLU)
// when rows > 128; kTileWide = wide decode batches: narrow weights split-K
// (with a workspace), else persistent, no split, 128, 192 or 256 rows by
// waves x operand bytes per tile.
enum GemmTiling { kTileSplit = 0, kTilePrefill = 1, kTileWide = 2 };
int gemm_tc_splits(int N, int K, bool decode);
int launch_gemm_tc(cudaStream_t s, int epi, const __nv_bfloat16* A, int lda, int a_rows,
                   const __nv_bfloat16* W, const __nv_bfloat16* W2, int N, int K, int rows,
                   float* Cf, __nv_bfloat16* Ct, int ldc, int tiling, float* ws, size_t ws_floats,
                   int* status);

}  // namespace cdb
