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
// One warp handles one (row, head, key split).  Keys are split in fixed-size
// ranges (split), independent of the batch, so a row's result does not depend
// on what else is in the batch.  Inside a warp, groups of LPK (<= 4) lanes
// each own one key at a time; each lane loads CPL 16-byte chunks of the key
// row and of the value row, the group reduces q.k with shuffles and keeps its
// own online-softmax state, rescaled once per block of UNR keys (scores in the
// log2 domain, exp2).  The groups are merged in a fixed order at the end.
// With one split the warp writes the normalised output; otherwise it writes
// (m, l, acc) partials that k_attn_combine merges in split order.
#include "common.cuh"
#include "kernels.cuh"

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

// 16-byte load of streamed KV data: read-only path, no L1 allocation, so the
// block-table and exit-depth lines stay cached.
template <typename T>
__device__ __forceinline__ uint4 ld_stream(const T* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Lanes per key and 16-byte chunks per lane for a head row of HD elements.
template <typename T, int HD>
struct AttnShape {
  static constexpr int CPE = Unpack<T>::N;       // elements per chunk
  static constexpr int NCH = HD / CPE;           // chunks per head row
  static constexpr int LPK = NCH >= 4 ? 4 : 2;  // lanes sharing one key
  static constexpr int CPL = NCH >= LPK ? NCH / LPK : 1;  // chunks per lane
  static constexpr int KPW = 32 / LPK;           // keys per warp per pass
  static constexpr int UNR = 16 / KPW;           // passes per 16-key page
  static_assert(HD % CPE == 0 && (NCH < LPK || NCH % LPK == 0), "head dim");
};

template <typename T, int HD>
__global__ void __launch_bounds__(128)
    k_attn(const T* __restrict__ Q, int rows, const int* __restrict__ mslot, const int* __restrict__ mpos,
           const int* __restrict__ mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp, int H,
           int split, int max_splits, T* __restrict__ O, float* __restrict__ part_o,
           float* __restrict__ part_ml, int* status) {
  pdl_wait();
  pdl_trigger();
  using S = AttnShape<T, HD>;
  constexpr int CPE = S::CPE, LPK = S::LPK, CPL = S::CPL, KPW = S::KPW, UNR = S::UNR, NCH = S::NCH;
  constexpr int EPL = CPL * CPE;  // elements per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.z;
  const int h = blockIdx.y * 4 + warp;
  if (row >= rows || h >= H) return;
  const int pos = mpos[row];
  const int L = pos + 1;
  const int nsp = (L + split - 1) / split;
  const int sp = blockIdx.x;
  if (sp >= nsp) return;
  const int k_lo = sp * split;
  const int k_hi = min(L, k_lo + split);
  const int r = depth_uniform > 0 ? depth_uniform : mdepth[row] + 1;
  const int slot = mslot[row];
  const int d = kv.d;
  const int g = lane / LPK, c = lane % LPK;
  const bool act = c < NCH;  // a one-chunk head row leaves the second lane idle
  // Scores are kept in the log2 domain: s * log2(e) / sqrt(HD).
  const float scale = 1.4426950408889634f / sqrtf((float)HD);

  // Chunk cc of this lane covers elements (c + LPK*cc)*CPE .. +CPE of the head
  // row, so for each cc the LPK lanes of a key read 16*LPK contiguous bytes.
  float q[EPL];
  {
    const T* qp = Q + (size_t)row * d + h * HD;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) {
      const uint4 raw = act ? *reinterpret_cast<const uint4*>(qp + (c + LPK * cc) * CPE) : make_uint4(0, 0, 0, 0);
      Unpack<T>::run(raw, q + cc * CPE);
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) q[e] *= scale;
  }

  const T* pool = reinterpret_cast<const T*>(kv.pool);
  const int* bt = kv.bt + slot * kv.max_blocks;
  const size_t slot_stride = (size_t)2 * 16 * d;  // elements between slots of one block
  float m = -INFINITY, l = 0.f;
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;

  // Keys go in blocks of KPW*UNR = 16, one KV page each (split starts are
  // multiples of 16).  The page's physical block and exit depths are fetched
  // one block ahead so the address chain overlaps the previous block's loads.
  static_assert(KPW * UNR == 16, "one 16-key page per pass");
  int blk_n = bt[k_lo >> 4];
  uint4 e16_n = make_uint4(0, 0, 0, 0);
  if (clamp && blk_n >= 0 && blk_n < kv.kv_blocks) e16_n = *reinterpret_cast<const uint4*>(kv.etab + blk_n * 16);
  for (int j0 = k_lo; j0 < k_hi; j0 += 16) {
    const int blk = blk_n;
    const uint4 e16 = e16_n;
    const bool blk_ok = blk >= 0 && blk < kv.kv_blocks;
    uint4 kr[UNR][CPL], vr[UNR][CPL];
    bool valid[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int off = u * KPW + g;
      const int j = j0 + off;
      valid[u] = j < k_hi;
#pragma unroll
      for (int cc = 0; cc < CPL; ++cc) kr[u][cc] = vr[u][cc] = make_uint4(0, 0, 0, 0);
      if (valid[u]) {
        int dr = 1;
        if (clamp) {
          const uint32_t w = off < 4 ? e16.x : off < 8 ? e16.y : off < 12 ? e16.z : e16.w;
          dr = min(r, (int)((w >> (8 * (off & 3))) & 0xFFu));
        }
        const int sl = slot_base + dr - 1;
        if (!blk_ok || dr < 1 || sl >= kv.nsl) {
          valid[u] = false;
          if (c == 0) atomicOr(status, kStatusBadDepth);
        } else if (act) {
          const T* kp = pool + ((size_t)blk * kv.nsl + sl) * slot_stride + (size_t)off * d + h * HD;
          const T* vp = kp + (size_t)16 * d;
#pragma unroll
          for (int cc = 0; cc < CPL; ++cc) {
            kr[u][cc] = ld_stream(kp + (c + LPK * cc) * CPE);
            vr[u][cc] = ld_stream(vp + (c + LPK * cc) * CPE);
          }
        }
      }
    }
    if (j0 + 16 < k_hi) {
      blk_n = bt[(j0 + 16) >> 4];
      if (clamp && blk_n >= 0 && blk_n < kv.kv_blocks) e16_n = *reinterpret_cast<const uint4*>(kv.etab + blk_n * 16);
    }
    float s[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float a = 0.f;
#pragma unroll
      for (int cc = 0; cc < CPL; ++cc) {
        float kf[CPE];
        Unpack<T>::run(kr[u][cc], kf);
#pragma unroll
        for (int e = 0; e < CPE; ++e) a = fmaf(q[cc * CPE + e], kf[e], a);
      }
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      s[u] = valid[u] ? a : -INFINITY;
    }
    // One rescale per block of UNR keys.
    float mn = m;
#pragma unroll
    for (int u = 0; u < UNR; ++u) mn = fmaxf(mn, s[u]);
    if (mn == -INFINITY) continue;  // no valid key in this block for this group
    const float corr = exp2f(m - mn);
    l *= corr;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= corr;
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const float p = exp2f(s[u] - mn);  // 0 for invalid keys
      l += p;
#pragma unroll
      for (int cc = 0; cc < CPL; ++cc) {
        float vf[CPE];
        Unpack<T>::run(vr[u][cc], vf);
#pragma unroll
        for (int e = 0; e < CPE; ++e) acc[cc * CPE + e] = fmaf(p, vf[e], acc[cc * CPE + e]);
      }
    }
    m = mn;
  }
  // Merge the KPW key groups of the warp (fixed butterfly order).
#pragma unroll
  for (int o = LPK; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float mn = fmaxf(m, m2);
    const float c1 = (m == -INFINITY) ? 0.f : exp2f(m - mn);
    const float c2 = (m2 == -INFINITY) ? 0.f : exp2f(m2 - mn);
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float a2 = __shfl_xor_sync(0xffffffffu, acc[e], o);
      acc[e] = acc[e] * c1 + a2 * c2;
    }
    l = l * c1 + l2 * c2;
    m = mn;
  }
  if (g != 0 || !act) return;
  if (nsp == 1) {
    const float inv = 1.f / l;
    T* out = O + (size_t)row * d + h * HD;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc)
#pragma unroll
      for (int e = 0; e < CPE; ++e) out[(c + LPK * cc) * CPE + e] = from_f<T>(acc[cc * CPE + e] * inv);
  } else {
    const size_t pi = ((size_t)row * H + h) * max_splits + sp;
    float* po = part_o + pi * HD;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc)
#pragma unroll
      for (int e = 0; e < CPE; ++e) po[(c + LPK * cc) * CPE + e] = acc[cc * CPE + e];
    if (c == 0) {
      part_ml[pi * 2] = m;  // log2 domain
      part_ml[pi * 2 + 1] = l;
    }
  }
}

// Merge split partials in split order: o = sum_s e^{m_s - m} acc_s / sum_s e^{m_s - m} l_s.
template <typename T>
__global__ void k_attn_combine(int rows, const int* __restrict__ mpos, int H, int HDv, int d, int split,
                               int max_splits, const float* __restrict__ part_o,
                               const float* __restrict__ part_ml, T* __restrict__ O) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x / H, h = blockIdx.x % H;
  if (row >= rows) return;
  const int L = mpos[row] + 1;
  const int nsp = (L + split - 1) / split;
  if (nsp <= 1) return;
  const size_t pi = ((size_t)row * H + h) * max_splits;
  float m = -INFINITY;
  for (int s = 0; s < nsp; ++s) m = fmaxf(m, part_ml[(pi + s) * 2]);
  float l = 0.f;
  for (int s = 0; s < nsp; ++s) l += part_ml[(pi + s) * 2 + 1] * exp2f(part_ml[(pi + s) * 2] - m);
  const float inv = 1.f / l;
  for (int e = threadIdx.x; e < HDv; e += blockDim.x) {
    float a = 0.f;
    for (int s = 0; s < nsp; ++s) a += part_o[(pi + s) * HDv + e] * exp2f(part_ml[(pi + s) * 2] - m);
    O[(size_t)row * d + h * HDv + e] = from_f<T>(a * inv);
  }
}

template <typename T, int HD>
static void attn_hd(cudaStream_t s, const T* Q, int rows, const int* mslot, const int* mpos, const int* mdepth,
                    int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int split, int max_splits,
                    T* O, float* part_o, float* part_ml, int* status) {
  dim3 grid(max_splits, (H + 3) / 4, rows);
  count_launch();
  launch_pdl(k_attn<T, HD>, dim3(grid), dim3(128), 0, s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H,
                                     split, max_splits, O, part_o, part_ml, status);
  if (max_splits > 1)
    count_launch(), launch_pdl(k_attn_combine<T>, dim3(rows * H), dim3(128), 0, s, rows, mpos, H, HD, kv.d, split, max_splits, part_o, part_ml, O);
}

template <typename T>
void launch_attention(cudaStream_t s, const T* Q, int rows, const int* mslot, const int* mpos,
                      const int* mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int hd,
                      int split, int max_splits, T* O, float* part_o, float* part_ml, int* status) {
  if (rows <= 0) return;
  switch (hd) {
    case 8: attn_hd<T, 8>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status); break;
    case 16: attn_hd<T, 16>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status); break;
    case 32: attn_hd<T, 32>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status); break;
    case 64: attn_hd<T, 64>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status); break;
    case 96: attn_hd<T, 96>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status); break;
    case 128: attn_hd<T, 128>(s, Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H, split, max_splits, O, part_o, part_ml, status); break;
    default: break;  // rejected at init
  }
}

template void launch_attention<float>(cudaStream_t, const float*, int, const int*, const int*, const int*, int,
                                      KvGeom, int, int, int, int, int, int, float*, float*, float*, int*);
template void launch_attention<__nv_bfloat16>(cudaStream_t, const __nv_bfloat16*, int, const int*, const int*,
                                              const int*, int, KvGeom, int, int, int, int, int, int,
                                              __nv_bfloat16*, float*, float*, int*);

}  // namespace cdb
