// Paged decode attention over the depth-indexed looped KV cache.
//
// "Depth-adaptive Inference of Looped Language Models via Continuous Depth
// Batching", §4.2: each core layer keeps one KV slot per loop step.  A row at
// loop step r reads the key/value of an earlier position j from step
// min(r, e_j), where e_j is j's exit depth (r_max for prompt positions and for
// the row's own in-flight position), so the slots an early exit left empty are
// never read.  Appendix A.1: keys live in 16-token blocks found through the
// sequence's block table.
//
// Pool layout [block][slot][K|V][head][16 keys][head_dim]: one head's page of
// one slot is a contiguous run of 16 * head_dim elements.
//
// Keys are split in fixed-size ranges (split), independent of the batch, so a
// row's result does not depend on what else is in the batch.  A work item is
// (key split, group of kWarps heads, row); items are numbered split-major
// (every row has split 0) and handed out by a device counter to a grid of
// resident CTAs, so which CTA computes an item never changes its result.
// In a CTA a producer warp streams the item's pages (16 keys, each key from
// its own depth slot) through a ring of shared-memory stages with 16-byte
// async copies whose completion lands on the stage's mbarrier; rows are
// padded by 16 bytes so matrix loads of 8 keys hit 8 different banks.  One
// consumer warp per head computes:
//  - bf16, head_dim % 16 == 0: per page, scores s^T = K_page . q and
//    o^T += V_page^T . p on the warp-level bf16 MMA (m16n8k16, fp32
//    accumulate), q and p in column 0 of the B operand, p fed as a bf16 pair
//    p_hi + p_lo (about 16 significant bits); online softmax once per page;
//  - otherwise: LPK lanes per key, q.k reduced with shuffles, online softmax
//    per lane group, groups merged in a fixed order at the end.
// Scores are kept in the log2 domain (exp2).  With one split the warp writes
// the normalised output; otherwise (m, l, acc) partials that k_attn_combine
// merges in split order.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "tmap.h"

namespace cdb {

// Raw 16-byte chunk -> floats.
template <typename T>
struct Unpack;
template <>
struct Unpack<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void run(const uint4& r, float* o) {
    o[0] = __uint_as_float(r.x);
    o[1] = __uint_as_float(r.y);
    o[2] = __uint_as_float(r.z);
    o[3] = __uint_as_float(r.w);
  }
};
template <>
struct Unpack<__nv_bfloat16> {
  static constexpr int N = 8;
  // bf16 is the top half of an fp32: shift or mask, no conversion instruction.
  __device__ __forceinline__ static void run(const uint4& r, float* o) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

namespace attn {

constexpr int kWarps = 4;   // consumer warps per CTA, one head each
constexpr int kStages = 3;  // ring depth (pages)

// Per-stage record: item, flags (bit 0 first page of the item, bit 1 last,
// bit 2 end of work), valid-key mask, the row's split count.
struct StageMeta {
  int item, flags, mask, nsp;
};
enum : int { kFirst = 1, kLast = 2, kEnd = 4 };

// Stage layout: rows (K|V, head, key) of RS bytes, then kWarps q rows.
template <typename T, int HD>
struct Geo {
  static constexpr int ES = sizeof(T);
  static constexpr int RB = HD * ES;             // bytes of one head row
  static constexpr int RS = RB + 16;             // padded shared-memory row
  static constexpr int CR = RB / 16;             // 16-byte chunks per row
  static constexpr int NR = 2 * kWarps * 16;     // K and V rows of one page
  static constexpr int STAGE = (NR + kWarps) * RS;
  static constexpr size_t SMEM = (size_t)kStages * STAGE + kStages * (2 * 8 + sizeof(StageMeta));
  static_assert(RB % 16 == 0, "head row must be a multiple of 16 bytes");
  static_assert((NR * CR) % 32 == 0, "chunks per page");
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}
// Wait for the phase of the given parity; false after ~2 s of global time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = su32(bar);
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 63) == 0) {
      uint64_t t;
      asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
      if (t0 == 0) t0 = t;
      else if (t - t0 > 2000000000ull) return false;
    }
  }
}

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on the mbarrier once every earlier cp.async of this thread has
// landed (counted against the barrier's initial count).
__device__ __forceinline__ void cp_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(su32(bar)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D[16x8] += A[16x16] . B[16x8], bf16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace attn

// Lanes sharing one key in the CUDA-core path: each lane owns one 16-byte
// chunk of the head row.
template <typename T, int HD>
struct AttnShape {
  static constexpr int CPE = Unpack<T>::N;  // elements per chunk
  static constexpr int NCH = HD / CPE;      // chunks per head row
  static constexpr int LPK = NCH <= 1 ? 1 : NCH <= 2 ? 2 : NCH <= 4 ? 4 : NCH <= 8 ? 8 : NCH <= 16 ? 16 : 32;
  static constexpr int KPW = 32 / LPK;      // keys per warp per pass
  static_assert(HD % CPE == 0 && NCH <= 32, "head dim");
};

// Online-softmax state of one compute warp (one head) for the current item.
template <typename T, int HD, bool MMA>
struct Acc;

// MMA path: lane 4i holds head dims 16t + i (acc[t][0]) and 16t + i + 8
// (acc[t][2]); the other lanes' accumulators hold zero columns.
template <typename T, int HD>
struct Acc<T, HD, true> {
  static constexpr int NT = HD / 16;
  uint32_t qb[NT][2];
  float acc[NT][4];
  float m, l;

  __device__ __forceinline__ void start(const uint8_t* qrow, int lane) {
    const uint32_t* qs = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      qb[t][0] = lane < 4 ? qs[t * 8 + lane] : 0u;
      qb[t][1] = lane < 4 ? qs[t * 8 + 4 + lane] : 0u;
      acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    }
    m = -INFINITY;
    l = 0.f;
  }

  // sk / sv: shared addresses of this head's first K / V row in the stage.
  __device__ __forceinline__ void page(uint32_t sk, uint32_t sv, uint32_t mask, int lane) {
    using Gm = attn::Geo<T, HD>;
    const float scale = 1.4426950408889634f / sqrtf((float)HD);  // log2(e) / sqrt(HD)
    const bool real = (lane & 3) == 0;
    const uint32_t koff = sk + ((lane & 7) + 8 * ((lane >> 3) & 1)) * Gm::RS + 16 * (lane >> 4);
    const uint32_t voff = sv + ((lane & 7) + 8 * (lane >> 4)) * Gm::RS + 16 * ((lane >> 3) & 1);
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      uint32_t a[4];
      attn::ldsm_x4(koff + t * 32, a);
      attn::mma_bf16(sc, a, qb[t][0], qb[t][1]);
    }
    // sc[0]: key lane/4, sc[2]: key lane/4 + 8 (column 0 on real lanes).
    const int k0 = lane >> 2;
    const float s0 = (real && ((mask >> k0) & 1u)) ? sc[0] * scale : -INFINITY;
    const float s1 = (real && ((mask >> (k0 + 8)) & 1u)) ? sc[2] * scale : -INFINITY;
    float mx = fmaxf(s0, s1);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(m, __shfl_sync(0xffffffffu, mx, 0));
    if (mn == -INFINITY) return;
    const float corr = exp2f(m - mn);
    const float p0 = exp2f(s0 - mn), p1 = exp2f(s1 - mn);
    // p as the B operand: lane t < 4 needs keys 2t, 2t+1 (rows 0..7 of B)
    // and 2t+8, 2t+9; key k sits on lane 4(k & 7), in p0 for k < 8.
    const int t4 = lane & 3;
    const float x0 = __shfl_sync(0xffffffffu, p0, 8 * t4);
    const float x1 = __shfl_sync(0xffffffffu, p0, 8 * t4 + 4);
    const float x2 = __shfl_sync(0xffffffffu, p1, 8 * t4);
    const float x3 = __shfl_sync(0xffffffffu, p1, 8 * t4 + 4);
    uint32_t bh0 = 0, bh1 = 0, bl0 = 0, bl1 = 0;
    if (lane < 4) {
      const float h0 = __bfloat162float(__float2bfloat16_rn(x0)), h1 = __bfloat162float(__float2bfloat16_rn(x1));
      const float h2 = __bfloat162float(__float2bfloat16_rn(x2)), h3 = __bfloat162float(__float2bfloat16_rn(x3));
      bh0 = attn::pack_bf16(h0, h1);
      bh1 = attn::pack_bf16(h2, h3);
      bl0 = attn::pack_bf16(x0 - h0, x1 - h1);
      bl1 = attn::pack_bf16(x2 - h2, x3 - h3);
    }
    l = fmaf(l, corr, p0 + p1);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      acc[t][0] *= corr;
      acc[t][2] *= corr;
      uint32_t a[4];
      attn::ldsm_x4_t(voff + t * 32, a);
      attn::mma_bf16(acc[t], a, bh0, bh1);
      attn::mma_bf16(acc[t], a, bl0, bl1);
    }
    m = mn;
  }

  __device__ __forceinline__ void finish(int lane, bool write, bool single, T* out, float* po, float* pml) {
    float lt = l;
    lt += __shfl_xor_sync(0xffffffffu, lt, 4);
    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
    if (!write || (lane & 3) != 0) return;
    const int i = lane >> 2;
    if (single) {
      const float inv = 1.f / lt;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        out[16 * t + i] = from_f<T>(acc[t][0] * inv);
        out[16 * t + i + 8] = from_f<T>(acc[t][2] * inv);
      }
    } else {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        po[16 * t + i] = acc[t][0];
        po[16 * t + i + 8] = acc[t][2];
      }
      if (lane == 0) {
        pml[0] = m;  // log2 domain
        pml[1] = lt;
      }
    }
  }
};

// CUDA-core path (fp32 models and head rows too narrow for the MMA tiles).
template <typename T, int HD>
struct Acc<T, HD, false> {
  using S = AttnShape<T, HD>;
  static constexpr int CPE = S::CPE, NCH = S::NCH, LPK = S::LPK, KPW = S::KPW;
  float q[CPE], acc[CPE];
  float m, l;

  __device__ __forceinline__ void start(const uint8_t* qrow, int lane) {
    const int c = lane % LPK;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (c < NCH) raw = *reinterpret_cast<const uint4*>(qrow + c * 16);
    Unpack<T>::run(raw, q);
    const float scale = 1.4426950408889634f / sqrtf((float)HD);
#pragma unroll
    for (int e = 0; e < CPE; ++e) {
      q[e] *= scale;
      acc[e] = 0.f;
    }
    m = -INFINITY;
    l = 0.f;
  }

  // sk / sv: this head's first K / V row in the stage.
  __device__ __forceinline__ void page(const uint8_t* sk, const uint8_t* sv, uint32_t mask, int lane) {
    using Gm = attn::Geo<T, HD>;
    const int g = lane / LPK, c = lane % LPK;
    const bool act = c < NCH;
#pragma unroll 1
    for (int kb = 0; kb < 16; kb += KPW) {
      const int k = kb + g;
      const bool valid = k < 16 && ((mask >> k) & 1u);
      uint4 kr = make_uint4(0, 0, 0, 0), vr = make_uint4(0, 0, 0, 0);
      if (valid && act) {
        kr = *reinterpret_cast<const uint4*>(sk + k * Gm::RS + c * 16);
        vr = *reinterpret_cast<const uint4*>(sv + k * Gm::RS + c * 16);
      }
      float kf[CPE];
      Unpack<T>::run(kr, kf);
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < CPE; ++e) a = fmaf(q[e], kf[e], a);
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      const float sc = valid ? a : -INFINITY;
      const float mn = fmaxf(m, sc);
      if (mn != -INFINITY) {
        const float corr = exp2f(m - mn);
        const float p = exp2f(sc - mn);
        float vf[CPE];
        Unpack<T>::run(vr, vf);
        l = fmaf(l, corr, p);
#pragma unroll
        for (int e = 0; e < CPE; ++e) acc[e] = fmaf(acc[e], corr, p * vf[e]);
        m = mn;
      }
    }
  }

  __device__ __forceinline__ void finish(int lane, bool write, bool single, T* out, float* po, float* pml) {
    // Merge the KPW key groups of the warp (fixed butterfly order).
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
      const float mn = fmaxf(m, m2);
      const float c1 = (m == -INFINITY) ? 0.f : exp2f(m - mn);
      const float c2 = (m2 == -INFINITY) ? 0.f : exp2f(m2 - mn);
#pragma unroll
      for (int e = 0; e < CPE; ++e) {
        const float a2 = __shfl_xor_sync(0xffffffffu, acc[e], o);
        acc[e] = acc[e] * c1 + a2 * c2;
      }
      l = l * c1 + l2 * c2;
      m = mn;
    }
    const int g = lane / LPK, c = lane % LPK;
    if (!write || g != 0 || c >= NCH) return;
    if (single) {
      const float inv = 1.f / l;
#pragma unroll
      for (int e = 0; e < CPE; ++e) out[c * CPE + e] = from_f<T>(acc[e] * inv);
    } else {
#pragma unroll
      for (int e = 0; e < CPE; ++e) po[c * CPE + e] = acc[e];
      if (c == 0) {
        pml[0] = m;  // log2 domain
        pml[1] = l;
      }
    }
  }
};

namespace attn {
// A row's last key position must lie inside both the split partials
// (max_splits * split keys) and its block-table row (max_blocks pages), and
// its sequence slot must be a table row.  Rows that fail are skipped and
// flagged (kStatusBadRow), never read past those arrays.
__device__ __forceinline__ bool row_in_bounds(int pos, int slot, int split, int max_splits, int max_blocks) {
  return pos >= 0 && slot >= 0 && (long long)pos < (long long)split * max_splits && (pos >> 4) < max_blocks;
}
}  // namespace attn

template <typename T, int HD>
__global__ void __launch_bounds__((attn::kWarps + 1) * 32)
    k_attn(const T* __restrict__ Q, int rows, const int* __restrict__ mslot, const int* __restrict__ mpos,
           const int* __restrict__ mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp, int perkey, int H,
           int split,
           int max_splits, T* __restrict__ O, float* __restrict__ part_o, float* __restrict__ part_ml,
           int* status) {
  using Gm = attn::Geo<T, HD>;
  constexpr bool MMA = sizeof(T) == 2 && HD % 16 == 0;
  constexpr int G = attn::kWarps, NS = attn::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * Gm::STAGE);
  uint64_t* empty = full + NS;
  attn::StageMeta* meta = reinterpret_cast<attn::StageMeta*>(empty + NS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = (H + G - 1) / G;
  const int per_sp = rows * ngroups;
  const int n_items = max_splits * per_sp;
  int* counter = status + kWorkCounter;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      attn::mbar_init(&full[i], 33);  // 32 producer lanes' copies + lane 0's record
      attn::mbar_init(&empty[i], G);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  if (warp == G) {
    // ---------------- producer warp ----------------
    const T* pool = reinterpret_cast<const T*>(kv.pool);
    const size_t head_elems = (size_t)16 * HD;       // one head's page
    const size_t kv_elems = (size_t)H * head_elems;  // K (or V) of one block-slot
    auto fetch = [&]() -> int {  // next active item, or n_items when the queue is empty
      int it = 0;
      if (lane == 0) {
        do {
          it = atomicAdd(counter, 1);
          if (it >= n_items) break;
          const int sp = it / per_sp, row = (it - sp * per_sp) / ngroups;
          const int p = __ldg(&mpos[row]);
          if (!attn::row_in_bounds(p, __ldg(&mslot[row]), split, max_splits, kv.max_blocks)) {
            if (sp == 0) atomicOr(status, kStatusBadRow);
            continue;
          }
          if (sp * split <= p) break;  // split sp starts at or before the row's last key
        } while (true);
      }
      return __shfl_sync(0xffffffffu, it, 0);
    };
    int st = 0;
    bool fail = false;
    auto acquire = [&](int s) -> bool {  // stage s free for writing
      if (st < NS) return true;
      const bool ok = attn::mbar_wait(&empty[s], ((st / NS) - 1) & 1);
      return __all_sync(0xffffffffu, ok) != 0;
    };
    int item = fetch();
    while (true) {
      const int s = st % NS;
      if (item >= n_items) {  // end marker
        if (!acquire(s)) {
          fail = true;
          break;
        }
        if (lane == 0) meta[s].flags = attn::kEnd;
        __syncwarp();
        attn::cp_arrive(&full[s]);
        if (lane == 0) attn::mbar_arrive(&full[s]);
        break;
      }
      const int sp = item / per_sp;
      const int row = (item - sp * per_sp) / ngroups;
      const int h0 = (item - sp * per_sp - row * ngroups) * G;
      const int L = mpos[row] + 1;
      const int nsp = (L + split - 1) / split;
      const int k_lo = sp * split, k_hi = min(L, k_lo + split);
      const int npg = (k_hi - k_lo + 15) >> 4;
      const int r = depth_uniform > 0 ? depth_uniform : mdepth[row] + 1;
      const int* bt = kv.bt + mslot[row] * kv.max_blocks;
      const int next = fetch();  // overlaps this item's pages
      for (int pg = 0; pg < npg; ++pg) {
        const int s2 = st % NS;
        // Block-slot index of this lane's key (lanes 0..15), -1 if not read.
        const int key = k_lo + pg * 16 + (lane & 15);
        int kidx = -1;
        if (key < k_hi) {
          const int blk = bt[key >> 4];
          // clamp 0: the layer's single slot; else step min(r, clamp), and
          // with perkey also at most e_j from the exit-depth table.
          int dr = 1;
          if (clamp > 0) {
            dr = min(r, clamp);
            if (perkey && blk >= 0 && blk < kv.kv_blocks) dr = min(dr, (int)kv.etab[(size_t)blk * 16 + (key & 15)]);
          }
          const int sl = slot_base + dr - 1;
          if (blk < 0 || blk >= kv.kv_blocks || dr < 1 || sl >= kv.nsl) {
            if (lane < 16) atomicOr(status, kStatusBadDepth);
          } else {
            kidx = blk * kv.nsl + sl;
          }
        }
        const uint32_t mask = __ballot_sync(0xffffffffu, kidx >= 0) & 0xFFFFu;
        if (!acquire(s2)) {
          fail = true;
          break;
        }
        uint8_t* stage = smem + (size_t)s2 * Gm::STAGE;
        const uint32_t sdst = attn::su32(stage);
        // Rows (kv, head hh, key k) of CR chunks; chunk c*32 + lane.
#pragma unroll 4
        for (int c = 0; c < Gm::NR * Gm::CR / 32; ++c) {
          const int idx = c * 32 + lane;
          const int rw = idx / Gm::CR, ch = idx - rw * Gm::CR;
          const int k = rw & 15, hh = (rw >> 4) % G, kvh = rw / (16 * G);
          const int ki = __shfl_sync(0xffffffffu, kidx, k);
          const uint32_t dst = sdst + rw * Gm::RS + ch * 16;
          if (ki >= 0 && h0 + hh < H) {
            const T* src = pool + ((size_t)ki * 2 + kvh) * kv_elems + (size_t)(h0 + hh) * head_elems +
                           (size_t)k * HD + ch * (16 / Gm::ES);
            attn::cp16(dst, src);
          } else if (kvh == 1) {  // V rows not read hold zeros: p = 0 must not meet a stale NaN
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
          }
        }
        if (pg == 0) {  // the G heads' q rows
          for (int idx = lane; idx < G * Gm::CR; idx += 32) {
            const int hh = idx / Gm::CR, ch = idx - hh * Gm::CR;
            if (h0 + hh < H)
              attn::cp16(sdst + (Gm::NR + hh) * Gm::RS + ch * 16,
                         Q + (size_t)row * kv.d + (size_t)(h0 + hh) * HD + ch * (16 / Gm::ES));
          }
        }
        if (lane == 0) {
          meta[s2].item = item;
          meta[s2].flags = (pg == 0 ? attn::kFirst : 0) | (pg == npg - 1 ? attn::kLast : 0);
          meta[s2].mask = (int)mask;
          meta[s2].nsp = nsp;
        }
        __syncwarp();
        attn::cp_arrive(&full[s2]);
        if (lane == 0) attn::mbar_arrive(&full[s2]);
        ++st;
      }
      if (fail) break;
      item = next;
    }
    if (fail) {
      if (lane == 0) atomicOr(status, kStatusTimeout);
      // Copies already issued land before the CTA may exit.
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
    // The last CTA to finish with the queue resets it for the next launch.
    if (lane == 0) {
      __threadfence();
      if (atomicAdd(counter + 1, 1) == (int)gridDim.x - 1) {
        atomicExch(counter, 0);
        atomicExch(counter + 1, 0);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }

  // ---------------- consumer warps: warp w handles head h0 + w ----------------
  Acc<T, HD, MMA> A;
  for (int st = 0;; ++st) {
    const int s = st % NS;
    const bool ok = attn::mbar_wait(&full[s], (st / NS) & 1);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) atomicOr(status, kStatusTimeout);
      return;
    }
    const int flags = meta[s].flags;
    if (flags & attn::kEnd) return;
    const int item = meta[s].item;
    const uint32_t mask = (uint32_t)meta[s].mask;
    const int nsp = meta[s].nsp;
    const uint8_t* stage = smem + (size_t)s * Gm::STAGE;
    if (flags & attn::kFirst) A.start(stage + (Gm::NR + warp) * Gm::RS, lane);
    const uint8_t* sk = stage + (size_t)warp * 16 * Gm::RS;
    const uint8_t* sv = stage + (size_t)(G + warp) * 16 * Gm::RS;
    if constexpr (MMA) A.page(attn::su32(sk), attn::su32(sv), mask, lane);
    else A.page(sk, sv, mask, lane);
    __syncwarp();
    if (lane == 0) attn::mbar_arrive(&empty[s]);
    if (flags & attn::kLast) {
      const int sp = item / per_sp;
      const int row = (item - sp * per_sp) / ngroups;
      const int h = (item - sp * per_sp - row * ngroups) * G + warp;
      const size_t pi = ((size_t)row * H + h) * max_splits + sp;
      A.finish(lane, h < H, nsp == 1, O + (size_t)row * kv.d + (size_t)h * HD, part_o + pi * HD, part_ml + pi * 2);
    }
  }
}

// ---------------------------------------------------------------------------
// Uniform-slot variant (bf16, head_dim 32, 64, 96 or 128): every key of a row
// is read from the same slot (slot_base + r - 1 for core layers, slot_base
// otherwise).  The engine guarantees this by filling exit gaps when a token
// leaves the loop (k_compact), so the depth-clamped read rule needs no
// per-key slot here.  A page of the kWarps heads of one slot is then two
// rectangular tiles of the pool (K and V: 16 keys x kWarps heads rows of
// head_dim elements) that a producer thread moves with 2D TMA tensor copies,
// head_dim split into 64- (or 32-) element slices under the 128-byte (or
// 64-byte) swizzle, so the consumers' matrix loads of 8 keys hit 8 different
// bank groups.  One CTA per (key split, head group, row); consumers as in the
// MMA path above.
// ---------------------------------------------------------------------------
namespace attn {

// NSTG: pages in flight per CTA (two at three CTAs per SM; six when the grid
// has no more CTAs than the GPU has SMs, i.e. small decode batches, whose
// few CTAs each walk a split's pages as a latency chain).
template <int HD, int NSTG = 2>
struct TmaGeo {
  static constexpr int SWB = HD % 64 == 0 ? 128 : 64;  // swizzle span = bytes of one slice row
  static constexpr int XW = SWB / 2;                    // elements per slice
  static constexpr int NX = HD / XW;                    // slices per head row
  static constexpr int ROWS = 16 * kWarps;              // tile rows: kWarps heads x 16 keys
  static constexpr int SLICE = ROWS * SWB;              // bytes of one slice tile
  static constexpr int KREG = NX * SLICE;               // K (or V) of one page
  static constexpr int QB = kWarps * HD * 2;            // q rows of the item
  static constexpr int STAGE = (2 * KREG + QB + 1023) / 1024 * 1024;
  static constexpr int NS = NSTG;
  static constexpr size_t SMEM = 1024 + (size_t)NS * STAGE + NS * (2 * 8 + sizeof(StageMeta));
  // Fused RoPE / KV write: q, k and v rows (bf16) of each consumer warp's head.
  static constexpr size_t XOFF = ((size_t)NS * STAGE + NS * (2 * 8 + sizeof(StageMeta)) + 15) / 16 * 16;
  static constexpr size_t SMEM_FUSED = 1024 + XOFF + (size_t)kWarps * 3 * HD * 2;
  static_assert(HD % 32 == 0, "head dim");
};

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                       uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(map), "r"(su32(bar)), "r"(x), "r"(y), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_1d(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
}

// Shared address of 16-byte chunk c (within a slice row) of tile row `row`.
template <int SWB>
__device__ __forceinline__ uint32_t swz(uint32_t slice, int row, int c) {
  const int pc = SWB == 128 ? (c ^ (row & 7)) : (c ^ ((row >> 1) & 3));
  return slice + (uint32_t)row * SWB + (uint32_t)pc * 16;
}

}  // namespace attn

// FUSE: the row's query is not read from Q but formed here from the QKV
// GEMM's split-K partials (RoPE, then bf16), and the CTA holding the row's
// last split also forms the token's own K and V rows: it stores them in the
// pool for later steps and writes them into the tile of its last page, whose
// copy from the pool may predate them.  Same arithmetic as k_rope_kv.
template <int HD, bool FUSE, int NSTG>
__global__ void __launch_bounds__((attn::kWarps + 1) * 32)
    k_attn_tma(const __grid_constant__ CUtensorMap tm, const __nv_bfloat16* __restrict__ Q, int rows,
               const int* __restrict__ mslot, const int* __restrict__ mpos, const int* __restrict__ mdepth,
               int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int split, int max_splits,
               __nv_bfloat16* __restrict__ O, float* __restrict__ part_o, float* __restrict__ part_ml,
               int* status, Parts qkv, const float2* __restrict__ rope) {
  using Gm = attn::TmaGeo<HD, NSTG>;
  constexpr int G = attn::kWarps, NS = Gm::NS, NT = HD / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * Gm::STAGE);
  uint64_t* empty = full + NS;
  attn::StageMeta* meta = reinterpret_cast<attn::StageMeta*>(empty + NS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.z, h0 = blockIdx.y * G, sp = blockIdx.x;

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm) : "memory");
    for (int i = 0; i < NS; ++i) {
      attn::mbar_init(&full[i], 1);
      attn::mbar_init(&empty[i], G);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (row >= rows) return;
  const int L = mpos[row] + 1;
  if (!attn::row_in_bounds(L - 1, mslot[row], split, max_splits, kv.max_blocks)) {
    if (threadIdx.x == 0 && sp == 0 && blockIdx.y == 0) atomicOr(status, kStatusBadRow);
    return;
  }
  const int nsp = (L + split - 1) / split;
  if (sp >= nsp) return;
  const int k_lo = sp * split, k_hi = min(L, k_lo + split);
  const int npg = (k_hi - k_lo + 15) >> 4;
  const int Gc = min(G, H - h0);

  if (warp == G) {
    // ---------------- producer warp ----------------
    const int r = depth_uniform > 0 ? depth_uniform : mdepth[row] + 1;
    const int sl = slot_base + (clamp ? min(r, clamp) - 1 : 0);
    const int* bt = kv.bt + mslot[row] * kv.max_blocks;
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    const bool sl_ok = sl >= 0 && sl < kv.nsl;
    if (!sl_ok && lane == 0) atomicOr(status, kStatusBadDepth);
    int blk_l = -1;
    bool fail = false;
    for (int pg = 0; pg < npg; ++pg) {
      const int s = pg % NS;
      if ((pg & 31) == 0) {
        const int p = (k_lo >> 4) + pg + lane;
        blk_l = (pg + lane < npg) ? bt[p] : -1;
      }
      const int blk = __shfl_sync(0xffffffffu, blk_l, pg & 31);
      if (pg >= NS) {
        const bool ok = attn::mbar_wait(&empty[s], ((pg / NS) - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          fail = true;
          break;
        }
      }
      if (lane == 0) {
        const bool ok = sl_ok && blk >= 0 && blk < kv.kv_blocks;
        if (!ok && sl_ok) atomicOr(status, kStatusBadBlock);
        const int key0 = k_lo + pg * 16;
        const int nk = min(16, k_hi - key0);
        meta[s].flags = (pg == 0 ? attn::kFirst : 0) | (pg == npg - 1 ? attn::kLast : 0);
        meta[s].mask = ok ? (int)((1u << nk) - 1u) : 0;
        const uint32_t qb = FUSE ? 0u : (uint32_t)Gc * HD * 2;
        const uint32_t st = attn::su32(smem + (size_t)s * Gm::STAGE);
        attn::mbar_arrive_tx(&full[s], (ok ? 2u * Gm::KREG : 0u) + (pg == 0 ? qb : 0u));
        if (ok) {
          // Tile row 0 = head h0, key 0 of this page at this slot.
          const int y0 = (int)((((long long)blk * kv.nsl + sl) * 2) * H * 16 + (long long)h0 * 16);
          for (int kvh = 0; kvh < 2; ++kvh)
            for (int j = 0; j < Gm::NX; ++j)
              attn::tma_2d(st + kvh * Gm::KREG + j * Gm::SLICE, &tm, &full[s], j * Gm::XW, y0 + kvh * H * 16, pol);
        }
        if (!FUSE && pg == 0)
          attn::bulk_1d(st + 2 * Gm::KREG, Q + (size_t)row * kv.d + (size_t)h0 * HD, qb, &full[s]);
      }
      __syncwarp();
    }
    if (fail && lane == 0) atomicOr(status, kStatusTimeout);
    return;
  }

  // ---------------- consumer warps: warp w handles head h0 + w ----------------
  const int h = h0 + warp;
  // Fused RoPE / KV write: this warp's q (and, in the row's last split, k
  // and v) rows, rotated and rounded, in xs = [q | k | v] of HD each.
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem + Gm::XOFF) + warp * 3 * HD;
  const bool own = FUSE && sp == nsp - 1 && h < H;
  if constexpr (FUSE) {
    if (h < H) {
      const int pos = L - 1;
      const float2* cs = rope + (size_t)pos * (HD / 2);
      constexpr int QU = HD / 8;  // four-pair groups per part
      for (int u = lane; u < (own ? 3 : 1) * QU; u += 32) {
        const int part = u / QU, j0 = (u - part * QU) * 4;
        const int c = part * kv.d + h * HD + j0;
        const float4 xa = qkv.sum4(row, c), xb = qkv.sum4(row, c + HD / 2);
        const float a_[4] = {xa.x, xa.y, xa.z, xa.w}, b_[4] = {xb.x, xb.y, xb.z, xb.w};
        float lo[4], hi[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (part < 2) {
            rope_pair(a_[e], b_[e], cs[j0 + e], lo[e], hi[e]);
          } else {
            lo[e] = a_[e];
            hi[e] = b_[e];
          }
        }
        __nv_bfloat16* dst = xs + part * HD + j0;
        *reinterpret_cast<uint2*>(dst) = make_uint2(attn::pack_bf16(lo[0], lo[1]), attn::pack_bf16(lo[2], lo[3]));
        *reinterpret_cast<uint2*>(dst + HD / 2) =
            make_uint2(attn::pack_bf16(hi[0], hi[1]), attn::pack_bf16(hi[2], hi[3]));
      }
      __syncwarp();
      if (own) {
        // The token's K and V rows go to its page at this layer's slot.
        const int r = depth_uniform > 0 ? depth_uniform : mdepth[row] + 1;
        const int sl = slot_base + (clamp ? min(r, clamp) - 1 : 0);
        const int blk = kv.bt[mslot[row] * kv.max_blocks + (pos >> 4)];
        if (blk >= 0 && blk < kv.kv_blocks && sl >= 0 && sl < kv.nsl) {
          __nv_bfloat16* kdst = reinterpret_cast<__nv_bfloat16*>(kv.pool) +
                                (((size_t)blk * kv.nsl + sl) * 2) * 16 * kv.d + (size_t)h * 16 * HD +
                                (size_t)(pos & 15) * HD;
          for (int u = lane; u < HD / 4; u += 32) {
            *reinterpret_cast<uint2*>(kdst + 4 * u) = *reinterpret_cast<const uint2*>(xs + HD + 4 * u);
            *reinterpret_cast<uint2*>(kdst + (size_t)16 * kv.d + 4 * u) =
                *reinterpret_cast<const uint2*>(xs + 2 * HD + 4 * u);
          }
        } else if (lane == 0) {
          atomicOr(status, kStatusBadBlock);
        }
      }
    }
  }
  const float scale = 1.4426950408889634f / sqrtf((float)HD);
  const bool real = (lane & 3) == 0;
  uint32_t qb[NT][2];
  float acc[NT][4];
  float m = -INFINITY, l = 0.f;
  const uint32_t base = attn::su32(smem);
  // Tile rows of this lane's ldmatrix addresses (K: keys in matrix order 0-7,
  // 8-15 for lanes 0-15 and again for 16-31; V transposed: 0-7, 0-7, 8-15, 8-15).
  const int krow = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
  const int vrow = warp * 16 + (lane & 7) + 8 * (lane >> 4);
  for (int pg = 0; pg < npg; ++pg) {
    const int s = pg % NS;
    const bool ok = attn::mbar_wait(&full[s], (pg / NS) & 1);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) atomicOr(status, kStatusTimeout);
      return;
    }
    const uint32_t mask = (uint32_t)meta[s].mask;
    const int flags = meta[s].flags;
    const uint32_t st = base + (uint32_t)s * Gm::STAGE;
    if (flags & attn::kFirst) {
      const uint32_t* qs =
          FUSE ? reinterpret_cast<const uint32_t*>(xs)
               : reinterpret_cast<const uint32_t*>(smem + (size_t)s * Gm::STAGE + 2 * Gm::KREG) + warp * (HD / 2);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        qb[t][0] = (lane < 4 && warp < Gc) ? qs[t * 8 + lane] : 0u;
        qb[t][1] = (lane < 4 && warp < Gc) ? qs[t * 8 + 4 + lane] : 0u;
        acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      }
    }
    if (mask != 0xFFFFu) {
      // Keys past the row's end (or a bad page): zero their V rows so that
      // p = 0 never meets stale or NaN values in the MMA.
      uint8_t* vt = smem + (size_t)s * Gm::STAGE + Gm::KREG;
      for (int u = lane; u < 16 * Gm::NX * (Gm::SWB / 16); u += 32) {
        const int k = u / (Gm::NX * (Gm::SWB / 16));
        if ((mask >> k) & 1u) continue;
        const int rem = u - k * (Gm::NX * (Gm::SWB / 16));
        const int j = rem / (Gm::SWB / 16), c = rem % (Gm::SWB / 16);
        *reinterpret_cast<uint4*>(vt + (size_t)j * Gm::SLICE + (size_t)(warp * 16 + k) * Gm::SWB + c * 16) =
            make_uint4(0, 0, 0, 0);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    if (own && (flags & attn::kLast) && mask != 0u) {
      // Lanes 0-15: the K row, 16-31: the V row, one 16-byte chunk each (HD <= 128).
      const int kk = (L - 1) & 15;
      const int part = lane >> 4, e = (lane & 15) * 8;
      if (e < HD) {
        const int j = e / Gm::XW, c = (e % Gm::XW) / 8;
        const uint32_t dst = attn::swz<Gm::SWB>(st + part * Gm::KREG + j * Gm::SLICE, warp * 16 + kk, c);
        const uint4 v = *reinterpret_cast<const uint4*>(xs + (1 + part) * HD + e);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    // Scores s^T = K_page . q.
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int j = (16 * t) / Gm::XW, c = ((16 * t) % Gm::XW) / 8 + (lane >> 4);
      uint32_t a[4];
      attn::ldsm_x4(attn::swz<Gm::SWB>(st + j * Gm::SLICE, krow, c), a);
      attn::mma_bf16(sc, a, qb[t][0], qb[t][1]);
    }
    const int k0 = lane >> 2;
    const float s0 = (real && ((mask >> k0) & 1u)) ? sc[0] * scale : -INFINITY;
    const float s1 = (real && ((mask >> (k0 + 8)) & 1u)) ? sc[2] * scale : -INFINITY;
    float mx = fmaxf(s0, s1);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(m, __shfl_sync(0xffffffffu, mx, 0));
    if (mn != -INFINITY) {
      const float corr = exp2f(m - mn);
      const float p0 = exp2f(s0 - mn), p1 = exp2f(s1 - mn);
      const int t4 = lane & 3;
      const float x0 = __shfl_sync(0xffffffffu, p0, 8 * t4);
      const float x1 = __shfl_sync(0xffffffffu, p0, 8 * t4 + 4);
      const float x2 = __shfl_sync(0xffffffffu, p1, 8 * t4);
      const float x3 = __shfl_sync(0xffffffffu, p1, 8 * t4 + 4);
      uint32_t bh0 = 0, bh1 = 0, bl0 = 0, bl1 = 0;
      if (lane < 4) {
        const float e0 = __bfloat162float(__float2bfloat16_rn(x0)), e1 = __bfloat162float(__float2bfloat16_rn(x1));
        const float e2 = __bfloat162float(__float2bfloat16_rn(x2)), e3 = __bfloat162float(__float2bfloat16_rn(x3));
        bh0 = attn::pack_bf16(e0, e1);
        bh1 = attn::pack_bf16(e2, e3);
        bl0 = attn::pack_bf16(x0 - e0, x1 - e1);
        bl1 = attn::pack_bf16(x2 - e2, x3 - e3);
      }
      l = fmaf(l, corr, p0 + p1);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        acc[t][0] *= corr;
        acc[t][2] *= corr;
        const int j = (16 * t) / Gm::XW, c = ((16 * t) % Gm::XW) / 8 + ((lane >> 3) & 1);
        uint32_t a[4];
        attn::ldsm_x4_t(attn::swz<Gm::SWB>(st + Gm::KREG + j * Gm::SLICE, vrow, c), a);
        attn::mma_bf16(acc[t], a, bh0, bh1);
        attn::mma_bf16(acc[t], a, bl0, bl1);
      }
      m = mn;
    }
    __syncwarp();
    if (lane == 0) attn::mbar_arrive(&empty[s]);
  }
  float lt = l;
  lt += __shfl_xor_sync(0xffffffffu, lt, 4);
  lt += __shfl_xor_sync(0xffffffffu, lt, 8);
  lt += __shfl_xor_sync(0xffffffffu, lt, 16);
  if (h >= H || !real) return;
  const int i = lane >> 2;
  if (nsp == 1) {
    const float inv = 1.f / lt;
    __nv_bfloat16* out = O + (size_t)row * kv.d + (size_t)h * HD;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      out[16 * t + i] = __float2bfloat16_rn(acc[t][0] * inv);
      out[16 * t + i + 8] = __float2bfloat16_rn(acc[t][2] * inv);
    }
  } else {
    const size_t pi = ((size_t)row * H + h) * max_splits + sp;
    float* po = part_o + pi * HD;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      po[16 * t + i] = acc[t][0];
      po[16 * t + i + 8] = acc[t][2];
    }
    if (lane == 0) {
      part_ml[pi * 2] = m;  // log2 domain
      part_ml[pi * 2 + 1] = lt;
    }
  }
}

// ---------------------------------------------------------------------------
// Prefill attention (bf16, head_dim 32, 64, 96 or 128), causal, in the style
// of FlashAttention-2 on the warp-level MMA.  The rows of a prefill chunk come
// sequence by sequence with consecutive positions; the host cuts them into
// query tiles of up to kPfRows rows of one sequence.  One CTA per (tile,
// head): a producer warp moves the tile's q rows once and then streams the
// sequence's key pages (16 keys, every key from the same slot) through a ring
// with 2D TMA tensor copies under the same swizzle as the decode kernel; four
// consumer warps own 16 query rows each.  Per page: S = Q.K^T (m16n8k16, fp32
// accumulate), causal mask, online softmax per row, O += P.V with P fed as a
// bf16 hi/lo pair.  Each page is read once per tile instead of once per row.
// ---------------------------------------------------------------------------
namespace attn {

constexpr int kPfRows = 64;   // query rows per tile (4 warps x 16)
constexpr int kPfStages = 4;  // pages in flight per CTA

template <int HD>
struct PfGeo {
  using Tg = TmaGeo<HD>;
  static constexpr int SWB = Tg::SWB, XW = Tg::XW, NX = Tg::NX;
  static constexpr int QSLICE = kPfRows * SWB;           // q rows of one slice
  static constexpr int QBYTES = NX * QSLICE;
  static constexpr int PSLICE = 16 * SWB;                // one page slice (16 keys)
  static constexpr int KV = NX * PSLICE;                 // K (or V) of one page
  static constexpr int STAGE = (2 * KV + 1023) / 1024 * 1024;
  static constexpr size_t SMEM = 1024 + (size_t)QBYTES + (size_t)kPfStages * STAGE + 2 * kPfStages * 8 + 8;
};

}  // namespace attn

template <int HD>
__global__ void __launch_bounds__(5 * 32)
    k_attn_prefill(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const int4* __restrict__ tiles, KvGeom kv, int slot, int H, __nv_bfloat16* __restrict__ O,
                   int* status) {
  using Pg = attn::PfGeo<HD>;
  constexpr int NS = attn::kPfStages, NT = HD / 16, NV = HD / 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem;
  uint8_t* ring = smem + Pg::QBYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)NS * Pg::STAGE);
  uint64_t* empty = full + NS;
  uint64_t* qbar = empty + NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmq) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmk) : "memory");
    for (int i = 0; i < NS; ++i) {
      attn::mbar_init(&full[i], 1);
      attn::mbar_init(&empty[i], 4);
    }
    attn::mbar_init(qbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int4 tile = tiles[blockIdx.x];  // (first row, rows, sequence slot, position of the first row)
  const int row0 = tile.x, nq = tile.y, p0 = tile.w;
  const int npg = (p0 + nq + 15) >> 4;  // pages up to the tile's last position

  if (warp == 4) {
    // ---------------- producer warp ----------------
    if (lane == 0) {
      uint64_t pol;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
      attn::mbar_arrive_tx(qbar, Pg::QBYTES);
      for (int j = 0; j < Pg::NX; ++j)
        attn::tma_2d(attn::su32(qs + j * Pg::QSLICE), &tmq, qbar, h * HD + j * Pg::XW, row0, pol);
      const int* bt = kv.bt + tile.z * kv.max_blocks;
      const bool sl_ok = slot >= 0 && slot < kv.nsl;
      if (!sl_ok) atomicOr(status, kStatusBadDepth);
      for (int pg = 0; pg < npg; ++pg) {
        const int s = pg % NS;
        if (pg >= NS && !attn::mbar_wait(&empty[s], ((pg / NS) - 1) & 1)) {
          atomicOr(status, kStatusTimeout);
          break;
        }
        const int blk = bt[pg];
        const bool ok = sl_ok && blk >= 0 && blk < kv.kv_blocks;
        if (!ok && sl_ok) atomicOr(status, kStatusBadBlock);
        attn::mbar_arrive_tx(&full[s], ok ? 2u * Pg::KV : 0u);
        if (ok) {
          // Page rows of head h at this slot: K then V (H * 16 rows later).
          const int y = (int)((((long long)blk * kv.nsl + slot) * 2 * H + h) * 16);
          const uint32_t st = attn::su32(ring + (size_t)s * Pg::STAGE);
          for (int j = 0; j < Pg::NX; ++j) {
            attn::tma_2d(st + j * Pg::PSLICE, &tmk, &full[s], j * Pg::XW, y, pol);
            attn::tma_2d(st + Pg::KV + j * Pg::PSLICE, &tmk, &full[s], j * Pg::XW, y + H * 16, pol);
          }
        }
      }
    }
    return;
  }

  // ---------------- consumer warps: query rows 16 * warp .. + 15 ----------------
  const float scale = 1.4426950408889634f / sqrtf((float)HD);
  const int g = lane >> 2, q4 = lane & 3;
  const int qr0 = p0 + warp * 16 + g, qr1 = qr0 + 8;  // positions of this thread's two rows
  if (!attn::mbar_wait(qbar, 0)) {
    if (lane == 0) atomicOr(status, kStatusTimeout);
    return;
  }
  uint32_t qa[NT][4];
  {
    const uint32_t qb = attn::su32(qs);
    const int r = warp * 16 + (lane & 15);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int j = (16 * t) / Pg::XW, c = ((16 * t) % Pg::XW) / 8 + (lane >> 4);
      attn::ldsm_x4(attn::swz<Pg::SWB>(qb + j * Pg::QSLICE, r, c), qa[t]);
    }
  }
  float o[NV][4];
#pragma unroll
  for (int v = 0; v < NV; ++v) o[v][0] = o[v][1] = o[v][2] = o[v][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const uint32_t rb = attn::su32(ring);
  for (int pg = 0; pg < npg; ++pg) {
    const int s = pg % NS;
    if (!attn::mbar_wait(&full[s], (pg / NS) & 1)) {
      if (lane == 0) atomicOr(status, kStatusTimeout);
      return;
    }
    const uint32_t st = rb + (uint32_t)s * Pg::STAGE;
    // S = Q . K^T for keys 16 pg .. + 15 (two n-tiles of 8 keys).
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int key = (lane & 7) + 8 * (lane >> 4);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int j = (16 * t) / Pg::XW, c = ((16 * t) % Pg::XW) / 8 + ((lane >> 3) & 1);
        uint32_t b[4];
        attn::ldsm_x4(attn::swz<Pg::SWB>(st + j * Pg::PSLICE, key, c), b);
        attn::mma_bf16(sc[0], qa[t], b[0], b[1]);
        attn::mma_bf16(sc[1], qa[t], b[2], b[3]);
      }
    }
    // Causal mask and scale: element (row, key) of the C fragments.
    const int kb = pg * 16;
    float sv[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kb + 8 * u + 2 * q4 + (e & 1);
        const int qp = e < 2 ? qr0 : qr1;
        sv[u][e] = key <= qp ? sc[u][e] * scale : -INFINITY;
      }
    float mx0 = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
    float mx1 = fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // Rows with no visible key so far keep zero weights (no -inf - -inf).
    const float c0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0), c1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
    float p[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      p[u][0] = n0 == -INFINITY ? 0.f : exp2f(sv[u][0] - n0);
      p[u][1] = n0 == -INFINITY ? 0.f : exp2f(sv[u][1] - n0);
      p[u][2] = n1 == -INFINITY ? 0.f : exp2f(sv[u][2] - n1);
      p[u][3] = n1 == -INFINITY ? 0.f : exp2f(sv[u][3] - n1);
    }
    l0 = l0 * c0 + p[0][0] + p[0][1] + p[1][0] + p[1][1];
    l1 = l1 * c1 + p[0][2] + p[0][3] + p[1][2] + p[1][3];
    m0 = n0;
    m1 = n1;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      o[v][0] *= c0;
      o[v][1] *= c0;
      o[v][2] *= c1;
      o[v][3] *= c1;
    }
    // P as the A operand (rows x keys), hi and lo bf16 parts.
    uint32_t ph[4], pl[4];
    {
      const float* f[4] = {&p[0][0], &p[0][2], &p[1][0], &p[1][2]};  // a0a1, a2a3, a4a5, a6a7
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float x0 = f[r][0], x1 = f[r][1];
        const float e0 = __bfloat162float(__float2bfloat16_rn(x0)), e1 = __bfloat162float(__float2bfloat16_rn(x1));
        ph[r] = attn::pack_bf16(e0, e1);
        pl[r] = attn::pack_bf16(x0 - e0, x1 - e1);
      }
    }
    // Keys past the tile's last position may hold NaN in the pool: their
    // weights are 0, and their V values are zeroed in the B fragments.
    const int kmax = p0 + nq - 1;
    const bool tail = kb + 15 > kmax;
    {
      const int key = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int vp = 0; vp < NV / 2; ++vp) {
        const int j = (16 * vp) / Pg::XW, c = ((16 * vp) % Pg::XW) / 8 + (lane >> 4);
        uint32_t b[4];
        attn::ldsm_x4_t(attn::swz<Pg::SWB>(st + Pg::KV + j * Pg::PSLICE, key, c), b);
        if (tail) {
          // b[0], b[2]: keys 2q4, 2q4+1; b[1], b[3]: keys 2q4+8, 2q4+9.
          const int k0 = kb + 2 * q4;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int kk = k0 + ((r & 1) ? 8 : 0);
            uint32_t mk = 0;
            if (kk <= kmax) mk |= 0x0000FFFFu;
            if (kk + 1 <= kmax) mk |= 0xFFFF0000u;
            b[r] &= mk;
          }
        }
        attn::mma_bf16(o[2 * vp], ph, b[0], b[1]);
        attn::mma_bf16(o[2 * vp], pl, b[0], b[1]);
        attn::mma_bf16(o[2 * vp + 1], ph, b[2], b[3]);
        attn::mma_bf16(o[2 * vp + 1], pl, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) attn::mbar_arrive(&empty[s]);
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int r0 = warp * 16 + g, r1 = r0 + 8;
  const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int dcol = h * HD + 8 * v + 2 * q4;
    if (r0 < nq)
      *reinterpret_cast<__nv_bfloat162*>(O + (size_t)(row0 + r0) * kv.d + dcol) =
          __floats2bfloat162_rn(o[v][0] * i0, o[v][1] * i0);
    if (r1 < nq)
      *reinterpret_cast<__nv_bfloat162*>(O + (size_t)(row0 + r1) * kv.d + dcol) =
          __floats2bfloat162_rn(o[v][2] * i1, o[v][3] * i1);
  }
}

// Merge split partials in split order: o = sum_s e^{m_s - m} acc_s / sum_s e^{m_s - m} l_s.
// One warp per (row, head): lane j owns columns 4j..4j+3 (HDv <= 128).  The
// split weights 2^(m_s - m) are computed once per split by the lane that
// loaded (m_s, l_s) and broadcast; the output sums over splits in split order.
template <typename T>
__global__ void k_attn_combine(int rows, const int* __restrict__ mpos, int H, int HDv, int d, int split,
                               int max_splits, int max_keys, const float* __restrict__ part_o,
                               const float* __restrict__ part_ml, T* __restrict__ O) {
  // Trigger first: the O projection that follows reads only its weights
  // before its own wait, so its CTAs can start streaming them on SMs the
  // attention kernel's tail has freed.
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int row = item / H, h = item % H;
  if (row >= rows) return;
  const int L = mpos[row] + 1;
  if (L < 1 || L > max_keys) return;  // skipped and flagged by the attention kernel
  const int nsp = (L + split - 1) / split;
  if (nsp <= 1) return;
  const size_t pi = ((size_t)row * H + h) * max_splits;
  float m = -INFINITY;
  for (int s = lane; s < nsp; s += 32) m = fmaxf(m, part_ml[(pi + s) * 2]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const bool cols = 4 * lane < HDv;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  for (int s0 = 0; s0 < nsp; s0 += 32) {
    const int s = s0 + lane;
    const float w = s < nsp ? exp2f(part_ml[(pi + s) * 2] - m) : 0.f;
    const float ls = s < nsp ? part_ml[(pi + s) * 2 + 1] * w : 0.f;
    // l and the output accumulate over the broadcast splits in split order.
    const int n = min(32, nsp - s0);
    int k = 0;
    for (; k + 4 <= n; k += 4) {
      float wk[4];
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        wk[u] = __shfl_sync(0xffffffffu, w, k + u);
        l += __shfl_sync(0xffffffffu, ls, k + u);
        v[u] = cols ? *reinterpret_cast<const float4*>(part_o + (pi + s0 + k + u) * HDv + 4 * lane)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a.x += v[u].x * wk[u];
        a.y += v[u].y * wk[u];
        a.z += v[u].z * wk[u];
        a.w += v[u].w * wk[u];
      }
    }
    for (; k < n; ++k) {
      const float wk = __shfl_sync(0xffffffffu, w, k);
      l += __shfl_sync(0xffffffffu, ls, k);
      const float4 v = cols ? *reinterpret_cast<const float4*>(part_o + (pi + s0 + k) * HDv + 4 * lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      a.x += v.x * wk;
      a.y += v.y * wk;
      a.z += v.z * wk;
      a.w += v.w * wk;
    }
  }
  if (!cols) return;
  const float inv = 1.f / l;
  T out[4] = {from_f<T>(a.x * inv), from_f<T>(a.y * inv), from_f<T>(a.z * inv), from_f<T>(a.w * inv)};
  T* dst = O + (size_t)row * d + h * HDv + 4 * lane;
#pragma unroll
  for (int e = 0; e < 4; ++e) dst[e] = out[e];
}

// Uniform-slot TMA path; false when the shape or pool does not fit it.
// FUSE: q, k and v from the QKV partials (see k_attn_tma), Q unused.
template <int HD, bool FUSE, int NSTG>
static bool attn_tma_ns(cudaStream_t s, const CUtensorMap* tm, const __nv_bfloat16* Q, int rows, const int* mslot,
                        const int* mpos, const int* mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp,
                        int H, int split, int max_splits, __nv_bfloat16* O, float* part_o, float* part_ml,
                        int* status, Parts qkv, const float2* rope) {
  using Gm = attn::TmaGeo<HD, NSTG>;
  constexpr size_t smem = FUSE ? Gm::SMEM_FUSED : Gm::SMEM;
  static bool set[kMaxDevices] = {};
  const int dev = current_device();
  if (!set[dev]) {
    if (cudaFuncSetAttribute(k_attn_tma<HD, FUSE, NSTG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return false;
    set[dev] = true;
  }
  dim3 grid(max_splits, (H + attn::kWarps - 1) / attn::kWarps, rows);
  count_launch();
  launch_pdl(k_attn_tma<HD, FUSE, NSTG>, grid, dim3((attn::kWarps + 1) * 32), smem, s, *tm, Q, rows, mslot, mpos,
             mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, qkv, rope);
  return true;
}

static int attn_sm_count() {
  static int n[kMaxDevices] = {};
  const int dev = current_device();
  if (!n[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    n[dev] = v;
  }
  return n[dev];
}

// The ring depth changes neither the order in which a CTA takes its pages
// nor their arithmetic, so a row's result is the same with either.
template <int HD, bool FUSE>
static bool attn_tma(cudaStream_t s, const __nv_bfloat16* Q, int rows, const int* mslot, const int* mpos,
                     const int* mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int split,
                     int max_splits, __nv_bfloat16* O, float* part_o, float* part_ml, int* status, Parts qkv,
                     const float2* rope) {
  using Gm = attn::TmaGeo<HD>;
  const uint64_t pool_rows = (uint64_t)kv.kv_blocks * kv.nsl * 2 * H * 16;
  if (pool_rows + 16 * attn::kWarps >= (1ull << 31)) return false;  // tile row coordinates are int32
  const CUtensorMap* tm = tmap_bf16_2d(kv.pool, HD, pool_rows, (uint64_t)HD * 2, Gm::XW, Gm::ROWS, Gm::SWB);
  if (!tm) return false;
  const long long ctas = (long long)max_splits * ((H + attn::kWarps - 1) / attn::kWarps) * rows;
  if (ctas <= attn_sm_count())
    return attn_tma_ns<HD, FUSE, 6>(s, tm, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split,
                                    max_splits, O, part_o, part_ml, status, qkv, rope);
  return attn_tma_ns<HD, FUSE, 2>(s, tm, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split,
                                  max_splits, O, part_o, part_ml, status, qkv, rope);
}

// Merge of the split partials (rows whose keys span more than one split).
template <typename T>
static void attn_combine(cudaStream_t s, int rows, const int* mpos, int H, int hd, KvGeom kv, int split,
                         int max_splits, const float* part_o, const float* part_ml, T* O) {
  if (max_splits > 1)
    count_launch(), launch_pdl(k_attn_combine<T>, dim3((rows * H + 3) / 4), dim3(128), 0, s, rows, mpos, H, hd, kv.d,
                               split, max_splits, (int)std::min<long long>((long long)split * max_splits,
                                                                           (long long)kv.max_blocks * 16),
                               part_o, part_ml, O);
}

template <typename T, int HD>
static void attn_hd(cudaStream_t s, const T* Q, int rows, const int* mslot, const int* mpos, const int* mdepth,
                    int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int split, int max_splits,
                    T* O, float* part_o, float* part_ml, int* status, bool uniform) {
  bool done = false;
  if constexpr (sizeof(T) == 2 && HD % 32 == 0) {
    if (uniform)
      done = attn_tma<HD, false>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split,
                                 max_splits, O, part_o, part_ml, status, Parts{nullptr, 0, 0, 0}, nullptr);
  }
  if (!done) {
    using Gm = attn::Geo<T, HD>;
    // Grid size (SMs x resident CTAs) and the shared-memory attribute, per device.
    static int ctas[kMaxDevices] = {};
    const int dev = current_device();
    if (!ctas[dev]) {
      cudaFuncSetAttribute(k_attn<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Gm::SMEM);
      int sms = 0, per_sm = 0;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_attn<T, HD>, (attn::kWarps + 1) * 32, Gm::SMEM);
      ctas[dev] = (sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    }
    const long long items = (long long)max_splits * rows * ((H + attn::kWarps - 1) / attn::kWarps);
    const int grid = (int)(items < ctas[dev] ? items : ctas[dev]);
    count_launch();  // uniform reads never touch the exit-depth table
    launch_pdl(k_attn<T, HD>, dim3(grid), dim3((attn::kWarps + 1) * 32), Gm::SMEM, s, Q, rows, mslot, mpos, mdepth,
               depth_uniform, kv, slot_base, clamp, uniform ? 0 : 1, H, split, max_splits, O, part_o, part_ml, status);
  }
  attn_combine<T>(s, rows, mpos, H, HD, kv, split, max_splits, part_o, part_ml, O);
}

bool attention_rope_fusable(KvGeom kv, int H, int hd, int split) {
  const uint64_t pool_rows = (uint64_t)kv.kv_blocks * kv.nsl * 2 * H * 16;
  return (hd == 32 || hd == 64 || hd == 96 || hd == 128) && split % 16 == 0 &&
         pool_rows + 16 * attn::kWarps < (1ull << 31);
}

bool launch_attention_rope(cudaStream_t s, const float* QKV, int ns, int rows, const int* mslot, const int* mpos,
                           const int* mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int hd,
                           int split, int max_splits, const float2* rope, __nv_bfloat16* O, float* part_o,
                           float* part_ml, int* status) {
  if (rows <= 0) return true;
  if (split % 16 != 0) return false;
  const Parts qkv{QKV, ns < 1 ? 1 : ns, (size_t)rows * 3 * kv.d, 3 * kv.d};
  bool done = false;
  switch (hd) {
    case 32: done = attn_tma<32, true>(s, nullptr, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, qkv, rope); break;
    case 64: done = attn_tma<64, true>(s, nullptr, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, qkv, rope); break;
    case 96: done = attn_tma<96, true>(s, nullptr, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, qkv, rope); break;
    case 128: done = attn_tma<128, true>(s, nullptr, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, qkv, rope); break;
    default: return false;
  }
  if (done) attn_combine<__nv_bfloat16>(s, rows, mpos, H, hd, kv, split, max_splits, part_o, part_ml, O);
  return done;
}

template <int HD>
static bool prefill_hd(cudaStream_t s, const __nv_bfloat16* Q, int q_rows, const int4* tiles, int n_tiles, KvGeom kv,
                       int slot, int H, __nv_bfloat16* O, int* status) {
  using Pg = attn::PfGeo<HD>;
  const uint64_t pool_rows = (uint64_t)kv.kv_blocks * kv.nsl * 2 * H * 16;
  if (pool_rows + 16 >= (1ull << 31) || q_rows + attn::kPfRows >= (1 << 30)) return false;
  const CUtensorMap* tk = tmap_bf16_2d(kv.pool, HD, pool_rows, (uint64_t)HD * 2, Pg::XW, 16, Pg::SWB);
  const CUtensorMap* tq = tmap_bf16_2d(Q, (uint64_t)kv.d, q_rows, (uint64_t)kv.d * 2, Pg::XW, attn::kPfRows, Pg::SWB);
  if (!tk || !tq) return false;
  static bool set[kMaxDevices] = {};
  const int dev = current_device();
  if (!set[dev]) {
    if (cudaFuncSetAttribute(k_attn_prefill<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Pg::SMEM) !=
        cudaSuccess)
      return false;
    set[dev] = true;
  }
  count_launch();
  return launch_pdl(k_attn_prefill<HD>, dim3(n_tiles, H), dim3(5 * 32), Pg::SMEM, s, *tq, *tk, tiles, kv, slot, H, O,
                    status) == cudaSuccess;
}

bool launch_prefill_attention(cudaStream_t s, const __nv_bfloat16* Q, int q_rows, const int4* tiles, int n_tiles,
                              KvGeom kv, int slot, int H, int hd, __nv_bfloat16* O, int* status) {
  if (n_tiles <= 0) return true;
  switch (hd) {
    case 32: return prefill_hd<32>(s, Q, q_rows, tiles, n_tiles, kv, slot, H, O, status);
    case 64:
    case 128: return launch_prefill_attention_tc(s, Q, q_rows, tiles, n_tiles, kv, slot, H, hd, O, status);
    case 96: return prefill_hd<96>(s, Q, q_rows, tiles, n_tiles, kv, slot, H, O, status);
    default: return false;
  }
}

std::vector<int4> prefill_tiles(const int32_t* row_slot, const int32_t* row_pos, int rows, int hd) {
  const int T = prefill_tile_rows(hd);
  std::vector<int4> tiles;
  for (int i = 0; i < rows;) {
    int j = i + 1;
    while (j < rows && j - i < T && row_slot[j] == row_slot[i] && row_pos[j] == row_pos[i] + (j - i)) ++j;
    tiles.push_back(make_int4(i, j - i, row_slot[i], row_pos[i]));
    i = j;
  }
  // Work of a tile grows with its last position (keys 0 .. p0 + rows - 1).
  std::stable_sort(tiles.begin(), tiles.end(), [](const int4& a, const int4& b) { return a.w + a.y > b.w + b.y; });
  return tiles;
}

template <typename T>
void launch_attention(cudaStream_t s, const T* Q, int rows, const int* mslot, const int* mpos,
                      const int* mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int hd,
                      int split, int max_splits, T* O, float* part_o, float* part_ml, int* status,
                      bool uniform) {
  if (rows <= 0) return;
  switch (hd) {
    case 8: attn_hd<T, 8>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, uniform); break;
    case 16: attn_hd<T, 16>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, uniform); break;
    case 32: attn_hd<T, 32>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, uniform); break;
    case 64: attn_hd<T, 64>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, uniform); break;
    case 96: attn_hd<T, 96>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, uniform); break;
    case 128: attn_hd<T, 128>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status, uniform); break;
    default: break;  // rejected at init
  }
}

template void launch_attention<float>(cudaStream_t, const float*, int, const int*, const int*, const int*, int,
                                      KvGeom, int, int, int, int, int, int, float*, float*, float*, int*, bool);
template void launch_attention<__nv_bfloat16>(cudaStream_t, const __nv_bfloat16*, int, const int*, const int*,
                                              const int*, int, KvGeom, int, int, int, int, int, int,
                                              __nv_bfloat16*, float*, float*, int*, bool);

}  // namespace cdb
