// Bookkeeping and elementwise kernels of one CDB step: embedding (prelude),
// RMSNorm, RoPE + KV write into the depth-indexed cache, the lookahead exit
// gate, prefix-sum compaction of the recurrent batch, batch re-formation,
// greedy argmax (coda) and the RoPE table.
//
// Source: "Depth-adaptive Inference of Looped Language Models via Continuous
// Depth Batching", §2 (prelude / core / coda), §4.2 (depth-indexed KV cache),
// §4.3 (lookahead gate), Algorithm 2 (exits to the coda queue, the rest back to
// the recurrent queue), Appendix A.4 (refill mixes loop depths in one batch).
#include "common.cuh"
#include "kernels.cuh"

#include <atomic>

namespace cdb {

static std::atomic<long long> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
long long launch_count() { return g_launches.load(std::memory_order_relaxed); }

// ---------------------------------------------------------------------------
// prelude: embedding gather
// ---------------------------------------------------------------------------

// Prefill rows: X[i] = E[tok_i]; the position's exit depth is r_max (prompt
// tokens run at full depth, Appendix A.1).
template <typename T>
__global__ void k_embed_prefill(const T* __restrict__ E, int d, int V, const int* __restrict__ rslot,
                                const int* __restrict__ rpos, const int* __restrict__ rtok, int rows,
                                float* __restrict__ X, KvGeom kv, int r_max, int* status) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  if (i >= rows) return;
  int tok = rtok[i];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) atomicOr(status, kStatusBadToken);
    tok = 0;
  }
  const T* e = E + (size_t)tok * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) X[(size_t)i * d + c] = to_f(e[c]);
  if (threadIdx.x == 0) {
    const int pos = rpos[i];
    const int blk = kv.bt[rslot[i] * kv.max_blocks + pos / 16];
    if (blk < 0 || blk >= kv.kv_blocks) atomicOr(status, kStatusBadBlock);
    else kv.etab[blk * 16 + (pos & 15)] = (uint8_t)r_max;
  }
}

// Decode prelude: the input of forward t is generated token t-1 of the slot.
template <typename T>
__global__ void k_embed_prelude(const T* __restrict__ E, int d, int V, const int* __restrict__ lslot,
                                const int* __restrict__ lt, const int* __restrict__ lpos, int rows,
                                const int* __restrict__ out_tok, int cap, float* __restrict__ X,
                                RowMeta m, KvGeom kv, int r_max, int* status) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  if (i >= rows) return;
  const int slot = lslot[i], t = lt[i], pos = lpos[i];
  int tok = out_tok[slot * cap + t - 1];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) atomicOr(status, kStatusBadToken);
    tok = 0;
  }
  const T* e = E + (size_t)tok * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) X[(size_t)i * d + c] = to_f(e[c]);
  if (threadIdx.x == 0) {
    m.slot[i] = slot;
    m.pos[i] = pos;
    m.t[i] = t;
    m.depth[i] = 0;
    m.pend[i] = 0;
    const int blk = kv.bt[slot * kv.max_blocks + pos / 16];
    if (blk < 0 || blk >= kv.kv_blocks) atomicOr(status, kStatusBadBlock);
    else kv.etab[blk * 16 + (pos & 15)] = (uint8_t)r_max;  // in flight
  }
}

// Move prelude outputs into the refill rows.  With an adapter the loop starts
// from s_0 = 0 and the prelude output e is kept per slot.
__global__ void k_prelude_finish(const float* __restrict__ Tp, RowMeta tm, int rows,
                                 float* __restrict__ Pb, RowMeta pm, int dst_off,
                                 float* __restrict__ estore, int d, int adapter) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  if (i >= rows) return;
  const int o = dst_off + i, slot = tm.slot[i];
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float v = Tp[(size_t)i * d + c];
    if (adapter) {
      estore[(size_t)slot * d + c] = v;
      Pb[(size_t)o * d + c] = 0.f;
    } else {
      Pb[(size_t)o * d + c] = v;
    }
  }
  if (threadIdx.x == 0) {
    pm.slot[o] = slot;
    pm.pos[o] = tm.pos[i];
    pm.t[o] = tm.t[i];
    pm.depth[o] = 0;
    pm.pend[o] = 0;
  }
}

// ---------------------------------------------------------------------------
// RMSNorm -> GEMM operand; adapter concat
// ---------------------------------------------------------------------------

// Four consecutive elements in one access (8 bytes for bf16, 16 for fp32).
template <typename T>
__device__ __forceinline__ void store4(T* p, const T (&v)[4]);
template <>
__device__ __forceinline__ void store4<float>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, const __nv_bfloat16 (&v)[4]) {
  __nv_bfloat162 lo, hi;
  lo.x = v[0];
  lo.y = v[1];
  hi.x = v[2];
  hi.y = v[3];
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&lo);
  u.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}
template <typename T>
__device__ __forceinline__ void load4(const T* p, T (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 f = *reinterpret_cast<const float4*>(p);
  v[0] = f.x;
  v[1] = f.y;
  v[2] = f.z;
  v[3] = f.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, __nv_bfloat16 (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  v[0] = lo.x;
  v[1] = lo.y;
  v[2] = hi.x;
  v[3] = hi.y;
}

// With pending partials (mode 1: residual, X += sum; mode 2: store, X = sum)
// X is updated first, then normalised.
// One block per row; each thread keeps KV four-column groups of the row in
// registers from the fold to the normalised store (d and lda multiples of 4).
// The gain is a weight, never written while kernels run, so it is loaded
// before waiting for the previous kernel.
template <typename T, int KV>
__global__ void k_rmsnorm(float* __restrict__ X, const T* __restrict__ g, T* __restrict__ A, int rows, int d,
                          float eps, int lda, Parts pp, int mode) {
  const int n4 = d / 4;
  T gv[KV][4];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int u = threadIdx.x + k * blockDim.x;
    if (A != nullptr && u < n4) load4(g + 4 * u, gv[k]);
  }
  pdl_wait();
  pdl_trigger();
  __shared__ float sh[33];
  const int i = blockIdx.x;
  if (i >= rows) return;
  float* x = X + (size_t)i * d;
  const bool keep = !(pp.ns > 0 && mode == 2);  // mode 2 replaces X by the sum
  float4 o[KV];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int u = threadIdx.x + k * blockDim.x;
    o[k] = u < n4 && keep ? *reinterpret_cast<const float4*>(x + 4 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (pp.ns > 0) {
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int u = threadIdx.x + k * blockDim.x;
      if (u < n4) {
        const float4 v = pp.sum4(i, 4 * u);
        o[k].x += v.x;
        o[k].y += v.y;
        o[k].z += v.z;
        o[k].w += v.w;
        *reinterpret_cast<float4*>(x + 4 * u) = o[k];
      }
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    ss = fmaf(o[k].x, o[k].x, ss);
    ss = fmaf(o[k].y, o[k].y, ss);
    ss = fmaf(o[k].z, o[k].z, ss);
    ss = fmaf(o[k].w, o[k].w, ss);
  }
  ss = block_sum(ss, sh);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
  if (A == nullptr) return;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int u = threadIdx.x + k * blockDim.x;
    if (u < n4) {
      const float w[4] = {o[k].x, o[k].y, o[k].z, o[k].w};
      T out[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) out[e] = from_f<T>(w[e] * inv * to_f(gv[k][e]));
      store4(A + (size_t)i * lda + 4 * u, out);
    }
  }
}

// C[i][c] (row stride ldc) = sum of the partials (mode 2) or C + sum (mode 1).
// Grid (rows, column blocks of 4 * blockDim).
__global__ void k_fold(Parts pp, int rows, int n, float* __restrict__ C, int ldc, int mode) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int c = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (i >= rows || c >= n) return;
  const float4 v = pp.sum4(i, c);
  float* o = C + (size_t)i * ldc + c;
  const float w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (c + e < n) o[e] = mode == 1 ? o[e] + w[e] : w[e];
}

// Mid[i][c] = silu(sum g) * (sum u), rounded to the operand type, from the
// partials of the gate/up GEMM (g at column c, u at c + f).  Grid (rows,
// column blocks of 4 * blockDim).
template <typename T>
__global__ void k_swiglu_combine(Parts pp, int rows, int f, T* __restrict__ Mid) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int c = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (i >= rows || c >= f) return;
  const float4 g4 = pp.sum4(i, c), u4 = pp.sum4(i, c + f);
  const float g[4] = {g4.x, g4.y, g4.z, g4.w}, u[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (c + e < f) Mid[(size_t)i * f + c + e] = from_f<T>(g[e] / (1.0f + expf(-g[e])) * u[e]);
}

// A[i] = [e ; s] rounded to the operand type (x = adapter . [e; s_{d-1}]).
template <typename T>
__global__ void k_concat(const float* __restrict__ E, int e_per_slot, const int* __restrict__ mslot,
                         const float* __restrict__ X, T* __restrict__ A, int rows, int d) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  if (i >= rows) return;
  const float* e = E + (size_t)(e_per_slot ? mslot[i] : i) * d;
  const float* s = X + (size_t)i * d;
  T* a = A + (size_t)i * 2 * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    a[c] = from_f<T>(e[c]);
    a[d + c] = from_f<T>(s[c]);
  }
}

// ---------------------------------------------------------------------------
// RoPE (rotate-half) + KV write into the depth-indexed cache
// ---------------------------------------------------------------------------

// Row i at position p and loop step r writes K,V into slot slot_base + r-1
// (core layers; slot_base + min(r, clamp) - 1 with a shared layout) or
// slot_base (prelude / coda layers, clamp = 0).  QKV arrives as split-K
// partials (qkv.ns >= 1; one partial is the plain GEMM output).
template <typename T>
__global__ void k_rope_kv(Parts qkv, int rows, const int* __restrict__ mslot,
                          const int* __restrict__ mpos, const int* __restrict__ mdepth,
                          int depth_uniform, int slot_base, int clamp, T* __restrict__ Q, KvGeom kv,
                          int H, int hd, const float2* __restrict__ rope, int* status) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  if (i >= rows) return;
  const int d = kv.d, half = hd / 2;
  const int pos = mpos[i];
  if (pos < 0 || (pos >> 4) >= kv.max_blocks || mslot[i] < 0) {  // past the block table (and the RoPE table)
    if (threadIdx.x == 0) atomicOr(status, kStatusBadRow);
    return;
  }
  const int r = depth_uniform > 0 ? depth_uniform : mdepth[i] + 1;
  const int blk = kv.bt[mslot[i] * kv.max_blocks + pos / 16];
  const int sl = slot_base + (clamp ? min(r, clamp) - 1 : 0);
  if (blk < 0 || blk >= kv.kv_blocks || sl < 0 || sl >= kv.nsl) {
    if (threadIdx.x == 0) atomicOr(status, kStatusBadBlock);
    return;
  }
  // Pool layout [block][slot][K|V][head][16][hd]: head h of this position
  // starts at (pos & 15) * hd inside its head's page.
  T* pool = reinterpret_cast<T*>(kv.pool);
  T* kdst = pool + (((size_t)blk * kv.nsl + sl) * 2 + 0) * 16 * d + (size_t)(pos & 15) * hd;
  T* vdst = kdst + (size_t)16 * d;
  const float2* cs = rope + (size_t)pos * half;
  // blockIdx.z: 0 = q (rotated, to Q), 1 = k (rotated, to the K page), 2 = v
  // (to the V page).  Four consecutive rotation pairs (j, j + half) per
  // thread; half is a multiple of 4 for every supported head dim.
  const int part = blockIdx.z;
  const int quads = H * half / 4;
  for (int u = blockIdx.y * blockDim.x + threadIdx.x; u < quads; u += gridDim.y * blockDim.x) {
    const int h = u / (half / 4), j0 = (u % (half / 4)) * 4;
    const int a = h * hd + j0, b = a + half;
    float2 r[4];
    if (part < 2) {
#pragma unroll
      for (int e = 0; e < 4; ++e) r[e] = cs[j0 + e];
    }
    const float4 xa = qkv.sum4(i, part * d + a), xb = qkv.sum4(i, part * d + b);
    const float a_[4] = {xa.x, xa.y, xa.z, xa.w}, b_[4] = {xb.x, xb.y, xb.z, xb.w};
    T lo[4], hi[4];
    if (part < 2) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float l, h;
        rope_pair(a_[e], b_[e], r[e], l, h);
        lo[e] = from_f<T>(l);
        hi[e] = from_f<T>(h);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        lo[e] = from_f<T>(a_[e]);
        hi[e] = from_f<T>(b_[e]);
      }
    }
    T* dst = part == 0 ? Q + (size_t)i * d + a : (part == 1 ? kdst : vdst) + (size_t)h * 16 * hd + j0;
    store4(dst, lo);
    store4(dst + half, hi);
  }
}

// cos/sin of pos * theta^(-2j/hd), evaluated in double and rounded once.
__global__ void k_rope_table(float2* tab, int max_ctx, int hd, float theta) {
  pdl_wait();
  pdl_trigger();
  const int half = hd / 2;
  const int n = max_ctx * half;
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < n; u += gridDim.x * blockDim.x) {
    const int p = u / half, j = u % half;
    const double inv = pow((double)theta, -2.0 * (double)j / (double)hd);
    const double a = (double)p * inv;
    tab[u] = make_float2((float)cos(a), (float)sin(a));
  }
}

// ---------------------------------------------------------------------------
// lookahead exit gate (§4.3)
// ---------------------------------------------------------------------------

// Probe gate (Sp == nullptr): z = w . rmsnorm(h) + b, fires when z > thr.
// Convergence gate (Sp = the states that entered this step, App. E.2):
// z = ||h - Sp|| / ||h||, fires when z < thr.  The flag set after step r makes
// the token exit after step r+1: live gate -> it fires and r >= r_min-1; a
// forced exit depth e -> r + 1 == e; fixed-depth mode never sets it.  z goes
// to the gate trace in either case.
template <typename T>
__global__ void k_gate(const float* __restrict__ X, const float* __restrict__ Sp, const T* __restrict__ w,
                       float bias, float thr,
                       float eps, int rows, int d, RowMeta m, int mode, int r_min, int r_max,
                       const int8_t* __restrict__ fexit, int cap, int* __restrict__ pend_new,
                       uint8_t* __restrict__ ring, float* __restrict__ gtrace) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sh[33];
  const int i = blockIdx.x;
  if (i >= rows) return;
  const float* x = X + (size_t)i * d;
  float ss = 0.f, dot = 0.f;
  if (Sp) {  // convergence statistic: dot accumulates ||s_d - s_{d-1}||^2
    const float* xp = Sp + (size_t)i * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      const float df = x[c] - xp[c];
      ss = fmaf(x[c], x[c], ss);
      dot = fmaf(df, df, dot);
    }
  } else {
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      ss = fmaf(x[c], x[c], ss);
      dot = fmaf(x[c], to_f(w[c]), dot);
    }
  }
  ss = block_sum(ss, sh);
  dot = block_sum(dot, sh);
  if (threadIdx.x != 0) return;
  const float z = Sp ? (ss > 0.f ? sqrtf(dot) / sqrtf(ss) : __int_as_float(0x7f800000))
                     : dot / sqrtf(ss / (float)d + eps) + bias;
  const int slot = m.slot[i], t = m.t[i];
  const int r = m.depth[i] + 1;
  int p = 0;
  if (mode != 2) {
    const int fe = fexit[slot * cap + t - 1];
    if (fe > 0) p = (r + 1 == fe);
    else p = (Sp ? z < thr : z > thr) && (r >= r_min - 1);
  }
  if (r + 1 >= r_max) p = 0;
  pend_new[i] = p;
  ring[slot] = (uint8_t)p;
  if (gtrace) gtrace[((size_t)slot * cap + (t - 1)) * r_max + (r - 1)] = z;
}

// ---------------------------------------------------------------------------
// compaction of the recurrent batch (Algorithm 2, lines 15-17)
// ---------------------------------------------------------------------------

// Row i exits after this step if its previous-step flag was set or it reached
// r_max.  Exits keep slot order and go to the coda rows after qc_off; the
// rest keep slot order at the front of the continuing rows.  One block per
// row; its destination is the exclusive prefix sum of the exit flags at row
// i, taken as a block-wide population count of the flags of rows j < i
// (__syncthreads_count, blockDim rows per round), and the row moves in
// 16-byte vectors.
// blockIdx.y == 0 compacts row blockIdx.x; blockIdx.y = 1 + l fills the exit
// gaps of core layer l: a row leaving after loop step r < r_max copies its
// slot-r K and V into slots r+1 .. r_max of that layer.  A later reader at
// step r' then finds in slot r' exactly the entry of slot min(r', r), the one
// the depth-clamped read rule selects, so every key of a page is read from
// one slot.
__global__ void k_compact(const float* __restrict__ X, RowMeta m, const int* __restrict__ pend_new,
                          int B, int d, int r_max, int qc_off, float* __restrict__ Xc, RowMeta mc,
                          float* __restrict__ Cb, RowMeta mb, KvGeom kv, int8_t* __restrict__ out_depth,
                          int cap, int core_slot0, int hd, int es, int* status) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  if (i >= B) return;
  auto exits = [&](int j) { return (m.depth[j] >= 1 && m.pend[j]) || (m.depth[j] + 1 >= r_max); };
  if (blockIdx.y > 0) {
    const int r = m.depth[i] + 1;
    if (!exits(i) || r >= r_max) return;
    const int pos = m.pos[i];
    const int blk = kv.bt[m.slot[i] * kv.max_blocks + pos / 16];
    if (blk < 0 || blk >= kv.kv_blocks) return;  // flagged by the compaction block
    const int base = core_slot0 + (blockIdx.y - 1) * r_max;
    // Per (block, slot): [K|V][head][16][hd]; this position's head rows are
    // hd elements at (pos & 15) * hd inside each head's page.
    const size_t row_b = (size_t)hd * es, page_b = 16 * row_b, kv_b = (size_t)16 * d * es;
    const int H = d / hd, cpr = (int)(row_b / 16);  // 16-byte chunks per head row
    const uint8_t* pool = reinterpret_cast<const uint8_t*>(kv.pool);
    const uint8_t* src = pool + ((size_t)blk * kv.nsl + base + r - 1) * 2 * kv_b + (size_t)(pos & 15) * row_b;
    for (int rr = r + 1; rr <= r_max; ++rr) {
      uint8_t* dst = const_cast<uint8_t*>(pool) + ((size_t)blk * kv.nsl + base + rr - 1) * 2 * kv_b +
                     (size_t)(pos & 15) * row_b;
      for (int u = threadIdx.x; u < 2 * H * cpr; u += blockDim.x) {
        const int kvh = u / (H * cpr), h = (u / cpr) % H, c = u % cpr;
        const size_t o = kvh * kv_b + h * page_b + (size_t)c * 16;
        *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(src + o);
      }
    }
    return;
  }
  int n_exit_before = 0;
  for (int j0 = 0; j0 < i; j0 += blockDim.x) {  // i is uniform across the block
    const int j = j0 + threadIdx.x;
    n_exit_before += __syncthreads_count(j < i && exits(j));
  }
  const bool ex = exits(i);
  const int r = m.depth[i] + 1;
  const int dst = ex ? qc_off + n_exit_before : i - n_exit_before;
  // Rows are d fp32 values, d a multiple of 4, at 256-byte aligned buffers.
  const float4* src4 = reinterpret_cast<const float4*>(X + (size_t)i * d);
  float4* dst4 = reinterpret_cast<float4*>((ex ? Cb : Xc) + (size_t)dst * d);
  for (int c = threadIdx.x; c < d / 4; c += blockDim.x) dst4[c] = src4[c];
  if (threadIdx.x == 0) {
    RowMeta o = ex ? mb : mc;
    const int slot = m.slot[i], pos = m.pos[i], t = m.t[i];
    o.slot[dst] = slot;
    o.pos[dst] = pos;
    o.t[dst] = t;
    o.depth[dst] = r;
    o.pend[dst] = ex ? 0 : pend_new[i];
    if (ex) {
      const int blk = kv.bt[slot * kv.max_blocks + pos / 16];
      if (blk < 0 || blk >= kv.kv_blocks) atomicOr(status, kStatusBadBlock);
      else kv.etab[blk * 16 + (pos & 15)] = (uint8_t)r;
      out_depth[slot * cap + t - 1] = (int8_t)r;
    }
  }
}

// Batch re-formation: continuing rows first, then refill rows (slot order).
__global__ void k_gather_core(const float* __restrict__ Xc, RowMeta mc, int B_cont,
                              const float* __restrict__ Pb, RowMeta mp, int n_ref,
                              float* __restrict__ X, RowMeta mx, int d, float* __restrict__ Sprev) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  if (i >= B_cont + n_ref) return;
  const bool c = i < B_cont;
  const int j = c ? i : i - B_cont;
  const float* src = (c ? Xc : Pb) + (size_t)j * d;
  const float4* s4 = reinterpret_cast<const float4*>(src);
  float4* d4 = reinterpret_cast<float4*>(X + (size_t)i * d);
  if (Sprev) {
    float4* p4 = reinterpret_cast<float4*>(Sprev + (size_t)i * d);
    for (int u = threadIdx.x; u < d / 4; u += blockDim.x) {
      const float4 v = s4[u];
      d4[u] = v;
      p4[u] = v;
    }
  } else {
    for (int u = threadIdx.x; u < d / 4; u += blockDim.x) d4[u] = s4[u];
  }
  if (threadIdx.x == 0) {
    const RowMeta& s = c ? mc : mp;
    mx.slot[i] = s.slot[j];
    mx.pos[i] = s.pos[j];
    mx.t[i] = s.t[j];
    mx.depth[i] = s.depth[j];
    mx.pend[i] = s.pend[j];
  }
}

// dst[k] = src[idx[k]] with metadata (prefill rows that finish a prompt).
__global__ void k_gather_rows(const float* __restrict__ src, const int* __restrict__ idx,
                              const int* __restrict__ rslot, const int* __restrict__ rpos, int n,
                              float* __restrict__ dst, RowMeta md, int d) {
  pdl_wait();
  pdl_trigger();
  const int k = blockIdx.x;
  if (k >= n) return;
  const int j = idx[k];
  for (int c = threadIdx.x; c < d; c += blockDim.x) dst[(size_t)k * d + c] = src[(size_t)j * d + c];
  if (threadIdx.x == 0) {
    md.slot[k] = rslot[j];
    md.pos[k] = rpos[j];
    md.t[k] = 0;
    md.depth[k] = 0;
    md.pend[k] = 0;
  }
}

__global__ void k_copy_rows(const float* __restrict__ src, float* __restrict__ dst, size_t n) {
  pdl_wait();
  pdl_trigger();
  for (size_t u = blockIdx.x * (size_t)blockDim.x + threadIdx.x; u < n;
       u += (size_t)gridDim.x * blockDim.x)
    dst[u] = src[u];
}

// ---------------------------------------------------------------------------
// coda: greedy argmax (ties -> lowest index), forced tokens, traces
// ---------------------------------------------------------------------------

__global__ void k_argmax(const float* __restrict__ logits, int rows, int V, RowMeta m,
                         const int* __restrict__ ftok, int cap, int* __restrict__ out_tok,
                         float* __restrict__ ltrace, int trace_T, const float* __restrict__ Hin,
                         float* __restrict__ htrace, int d, int* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sv[32];
  __shared__ int si[32];
  const int i = blockIdx.x;
  if (i >= rows) return;
  const float* lg = logits + (size_t)i * V;
  float best = -INFINITY;
  int bi = V;
  bool nan = false;
  auto take = [&](float v, int j) {
    if (v != v) nan = true;
    if (v > best) {  // strict: the lowest index wins a tie within a thread
      best = v;
      bi = j;
    }
  };
  if ((V & 3) == 0) {  // rows are 16-byte aligned: four logits per load, eight loads in flight
    const float4* lg4 = reinterpret_cast<const float4*>(lg);
#pragma unroll 8
    for (int j = threadIdx.x; j < V / 4; j += blockDim.x) {
      const float4 v = lg4[j];
      take(v.x, 4 * j);
      take(v.y, 4 * j + 1);
      take(v.z, 4 * j + 2);
      take(v.w, 4 * j + 3);
    }
  } else {
    for (int j = threadIdx.x; j < V; j += blockDim.x) take(lg[j], j);
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  if (lane == 0) {
    sv[w] = best;
    si[w] = bi;
  }
  if (nan) atomicOr(status, kStatusNaN);
  __syncthreads();
  const int slot = m.slot[i], t = m.t[i];
  if (threadIdx.x == 0) {
    for (int u = 1; u < (int)(blockDim.x >> 5); ++u)
      if (sv[u] > sv[0] || (sv[u] == sv[0] && si[u] < si[0])) {
        sv[0] = sv[u];
        si[0] = si[u];
      }
    int tok = si[0] >= V ? 0 : si[0];
    const int f = ftok[slot * cap + t];
    if (f >= 0) tok = f;
    out_tok[slot * cap + t] = tok;
  }
  if (ltrace && t < trace_T) {
    float* dst = ltrace + ((size_t)slot * trace_T + t) * V;
    for (int j = threadIdx.x; j < V; j += blockDim.x) dst[j] = lg[j];
    float* hd = htrace + ((size_t)slot * trace_T + t) * d;
    for (int j = threadIdx.x; j < d; j += blockDim.x) hd[j] = Hin[(size_t)i * d + j];
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

template <typename T>
void launch_embed_prefill(cudaStream_t s, const T* E, int d, int V, const int* rslot, const int* rpos,
                          const int* rtok, int rows, float* X, KvGeom kv, int r_max, int* status) {
  if (rows > 0) count_launch(), launch_pdl(k_embed_prefill<T>, dim3(rows), dim3(256), 0, s, E, d, V, rslot, rpos, rtok, rows, X, kv, r_max, status);
}
template <typename T>
void launch_embed_prelude(cudaStream_t s, const T* E, int d, int V, const int* lslot, const int* lt,
                          const int* lpos, int rows, const int* out_tok, int cap, float* X,
                          RowMeta meta, KvGeom kv, int r_max, int* status) {
  if (rows > 0)
    count_launch(), launch_pdl(k_embed_prelude<T>, dim3(rows), dim3(256), 0, s, E, d, V, lslot, lt, lpos, rows, out_tok, cap, X, meta, kv,
                                            r_max, status);
}
void launch_prelude_finish(cudaStream_t s, const float* Tp, RowMeta tm, int rows, float* Pb, RowMeta pm,
                           int dst_off, float* estore, int d, int adapter) {
  if (rows > 0) count_launch(), launch_pdl(k_prelude_finish, dim3(rows), dim3(256), 0, s, Tp, tm, rows, Pb, pm, dst_off, estore, d, adapter);
}
template <typename T>
void launch_rmsnorm(cudaStream_t s, float* X, const T* g, T* A, int rows, int d, float eps, int lda,
                    const float* P, int ns, int mode) {
  Parts pp{P, ns, (size_t)rows * d, d};
  if (rows <= 0) return;
  // d and lda are multiples of 4 (the model descriptor requires it of d_model).
  const int n4 = d / 4;
  const int kv = n4 <= 512 ? 1 : n4 <= 1024 ? 2 : n4 <= 2048 ? 4 : 8;
  const int threads = ((n4 + kv - 1) / kv + 31) / 32 * 32;
  count_launch();
  switch (kv) {
    case 1: launch_pdl(k_rmsnorm<T, 1>, dim3(rows), dim3(threads), 0, s, X, g, A, rows, d, eps, lda, pp, mode); break;
    case 2: launch_pdl(k_rmsnorm<T, 2>, dim3(rows), dim3(threads), 0, s, X, g, A, rows, d, eps, lda, pp, mode); break;
    case 4: launch_pdl(k_rmsnorm<T, 4>, dim3(rows), dim3(threads), 0, s, X, g, A, rows, d, eps, lda, pp, mode); break;
    default: launch_pdl(k_rmsnorm<T, 8>, dim3(rows), dim3(threads), 0, s, X, g, A, rows, d, eps, lda, pp, mode); break;
  }
}
void launch_fold(cudaStream_t s, const float* P, int ns, int rows, int n, float* C, int ldc, int mode) {
  Parts pp{P, ns, (size_t)rows * n, n};
  if (rows > 0 && ns > 0)
    count_launch(), launch_pdl(k_fold, dim3(rows, (n + 511) / 512), dim3(128), 0, s, pp, rows, n, C, ldc, mode);
}
template <typename T>
void launch_swiglu_combine(cudaStream_t s, const float* P, int ns, int rows, int f, T* Mid) {
  Parts pp{P, ns, (size_t)rows * 2 * f, 2 * f};
  if (rows > 0)
    count_launch(), launch_pdl(k_swiglu_combine<T>, dim3(rows, (f + 511) / 512), dim3(128), 0, s, pp, rows, f, Mid);
}
template <typename T>
void launch_concat(cudaStream_t s, const float* E, int e_per_slot, const int* mslot, const float* X, T* A,
                   int rows, int d) {
  if (rows > 0) count_launch(), launch_pdl(k_concat<T>, dim3(rows), dim3(256), 0, s, E, e_per_slot, mslot, X, A, rows, d);
}
template <typename T>
void launch_rope_kv(cudaStream_t s, const float* QKV, int ns, int rows, const int* mslot, const int* mpos,
                    const int* mdepth, int depth_uniform, int slot_base, int clamp, T* Q, KvGeom kv, int H,
                    int hd, const float2* rope, int* status) {
  Parts qkv{QKV, ns < 1 ? 1 : ns, (size_t)rows * 3 * kv.d, 3 * kv.d};
  const int quads = H * (hd / 2) / 4;
  const int gy = (quads + 63) / 64;
  if (rows > 0)
    count_launch(), launch_pdl(k_rope_kv<T>, dim3(rows, gy, 3), dim3(64), 0, s, qkv, rows, mslot, mpos, mdepth, depth_uniform, slot_base, clamp, Q,
                                      kv, H, hd, rope, status);
}
template <typename T>
void launch_gate(cudaStream_t s, const float* X, const float* Sprev, const T* w, float bias, float thr, float eps,
                 int rows, int d, RowMeta meta, int mode, int r_min, int r_max, const int8_t* fexit, int cap,
                 int* pend_new, uint8_t* ring, float* gtrace) {
  if (rows > 0)
    count_launch(), launch_pdl(k_gate<T>, dim3(rows), dim3(256), 0, s, X, Sprev, w, bias, thr, eps, rows, d, meta, mode,
                               r_min, r_max, fexit, cap, pend_new, ring, gtrace);
}
void launch_compact(cudaStream_t s, const float* X, RowMeta m, const int* pend_new, int B, int d, int r_max,
                    int qc_off, float* Xc, RowMeta mc, float* Cb, RowMeta mb, KvGeom kv, int8_t* out_depth,
                    int cap, int n_core, int core_slot0, int hd, int es, int* status) {
  if (B > 0)
    count_launch(), launch_pdl(k_compact, dim3(B, 1 + n_core), dim3(256), 0, s, X, m, pend_new, B, d, r_max, qc_off,
                               Xc, mc, Cb, mb, kv, out_depth, cap, core_slot0, hd, es, status);
}
void launch_gather_core(cudaStream_t s, const float* Xc, RowMeta mc, int B_cont, const float* Pb, RowMeta mp,
                        int n_ref, float* X, RowMeta mx, int d, float* Sprev) {
  if (B_cont + n_ref > 0)
    count_launch(), launch_pdl(k_gather_core, dim3(B_cont + n_ref), dim3(256), 0, s, Xc, mc, B_cont, Pb, mp, n_ref, X, mx, d,
                               Sprev);
}
void launch_gather_rows(cudaStream_t s, const float* src, const int* idx, const int* rslot, const int* rpos,
                        int n, float* dst, RowMeta md, int d) {
  if (n > 0) count_launch(), launch_pdl(k_gather_rows, dim3(n), dim3(256), 0, s, src, idx, rslot, rpos, n, dst, md, d);
}
void launch_argmax(cudaStream_t s, const float* logits, int rows, int V, RowMeta m, const int* ftok, int cap,
                   int* out_tok, float* ltrace, int trace_T, const float* H, float* htrace, int d,
                   int* status) {
  if (rows > 0)
    count_launch(), launch_pdl(k_argmax, dim3(rows), dim3(512), 0, s, logits, rows, V, m, ftok, cap, out_tok, ltrace, trace_T, H, htrace, d,
                                  status);
}
void launch_rope_table(cudaStream_t s, float2* tab, int max_ctx, int hd, float theta) {
  count_launch(), launch_pdl(k_rope_table, dim3(1024), dim3(256), 0, s, tab, max_ctx, hd, theta);
}
void launch_copy_rows(cudaStream_t s, const float* src, float* dst, int rows, int d) {
  if (rows > 0) count_launch(), launch_pdl(k_copy_rows, dim3(1024), dim3(256), 0, s, src, dst, (size_t)rows * d);
}

#define CDB_INST(T)                                                                                          \
  template void launch_embed_prefill<T>(cudaStream_t, const T*, int, int, const int*, const int*,          \
                                        const int*, int, float*, KvGeom, int, int*);                          \
  template void launch_embed_prelude<T>(cudaStream_t, const T*, int, int, const int*, const int*,          \
                                        const int*, int, const int*, int, float*, RowMeta, KvGeom, int,       \
                                        int*);                                                                \
  template void launch_rmsnorm<T>(cudaStream_t, float*, const T*, T*, int, int, float, int, const float*,   \
                                  int, int);                                                                \
  template void launch_swiglu_combine<T>(cudaStream_t, const float*, int, int, int, T*);                   \
  template void launch_concat<T>(cudaStream_t, const float*, int, const int*, const float*, T*, int, int);  \
  template void launch_rope_kv<T>(cudaStream_t, const float*, int, int, const int*, const int*, const int*,  \
                                  int, int, int, T*, KvGeom, int, int, const float2*, int*);                  \
  template void launch_gate<T>(cudaStream_t, const float*, const float*, const T*, float, float, float, int, \
                               int, RowMeta, int, int, int, const int8_t*, int, int*, uint8_t*, float*);
CDB_INST(float)
CDB_INST(__nv_bfloat16)
#undef CDB_INST

}  // namespace cdb
