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
// on what else is in the batch.  Inside a warp, groups of LPK lanes each own
// one key at a time: every lane loads one 16-byte chunk of the key row and of
// the value row, the group reduces q.k with shuffles, and keeps its own online
// softmax state; the groups are merged in a fixed order at the end.  With one
// split the warp writes the normalised output; otherwise it writes (m, l, acc)
// partials that k_attn_combine merges in split order.
#include "common.cuh"
#include "kernels.cuh"

namespace cdb {

template <typename T, int HD>
__global__ void __launch_bounds__(128)
    k_attn(const T* __restrict__ Q, int rows, const int* __restrict__ mslot, const int* __restrict__ mpos,
           const int* __restrict__ mdepth, int depth_uniform, KvGeom kv, int slot_base, int clamp, int H,
           int split, int max_splits, T* __restrict__ O, float* __restrict__ part_o,
           float* __restrict__ part_ml, int* status) {
  constexpr int CPE = Chunk<T>::N;
  constexpr int NCH = HD / CPE;
  constexpr int LPK = NCH <= 2 ? 2 : NCH <= 4 ? 4 : NCH <= 8 ? 8 : NCH <= 16 ? 16 : 32;
  constexpr int KPI = 32 / LPK;
  static_assert(HD % CPE == 0 && NCH <= 32, "head dim");
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
  const bool act = c < NCH;
  const float scale = 1.0f / sqrtf((float)HD);

  float q[CPE];
  if (act) Chunk<T>::load(Q + (size_t)row * d + h * HD + c * CPE, q);
  else
#pragma unroll
    for (int e = 0; e < CPE; ++e) q[e] = 0.f;

  const T* pool = reinterpret_cast<const T*>(kv.pool);
  const int* bt = kv.bt + slot * kv.max_blocks;
  float m = -INFINITY, l = 0.f;
  float acc[CPE];
#pragma unroll
  for (int e = 0; e < CPE; ++e) acc[e] = 0.f;

  constexpr int UNR = 4;  // keys per group in flight
  for (int j0 = k_lo; j0 < k_hi; j0 += KPI * UNR) {
    float kf[UNR][CPE], vf[UNR][CPE], s[UNR];
    bool valid[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int j = j0 + u * KPI + g;
      valid[u] = j < k_hi;
      s[u] = 0.f;
#pragma unroll
      for (int e = 0; e < CPE; ++e) kf[u][e] = vf[u][e] = 0.f;
      if (valid[u]) {
        const int blk = bt[j >> 4];
        const int off = j & 15;
        const bool blk_ok = blk >= 0 && blk < kv.kv_blocks;
        int dr = 1;
        if (clamp && blk_ok) dr = min(r, (int)kv.etab[blk * 16 + off]);
        const int sl = slot_base + dr - 1;
        if (!blk_ok || dr < 1 || sl >= kv.nsl) {
          if (c == 0) atomicOr(status, kStatusBadDepth);
        } else if (act) {
          const size_t base =
              (((size_t)blk * kv.nsl + sl) * 2) * 16 * d + (size_t)off * d + h * HD + c * CPE;
          Chunk<T>::load(pool + base, kf[u]);
          Chunk<T>::load(pool + base + 16 * (size_t)d, vf[u]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
#pragma unroll
      for (int e = 0; e < CPE; ++e) s[u] = fmaf(q[e], kf[u][e], s[u]);
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) s[u] += __shfl_xor_sync(0xffffffffu, s[u], o);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (!valid[u]) continue;
      const float su = s[u] * scale;
      const float mn = fmaxf(m, su);
      const float corr = expf(m - mn);
      const float p = expf(su - mn);
      l = l * corr + p;
#pragma unroll
      for (int e = 0; e < CPE; ++e) acc[e] = fmaf(p, vf[u][e], acc[e] * corr);
      m = mn;
    }
  }
  // Merge the KPI key groups (fixed butterfly order).
#pragma unroll
  for (int o = LPK; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float mn = fmaxf(m, m2);
    const float c1 = (m == -INFINITY) ? 0.f : expf(m - mn);
    const float c2 = (m2 == -INFINITY) ? 0.f : expf(m2 - mn);
#pragma unroll
    for (int e = 0; e < CPE; ++e) {
      const float a2 = __shfl_xor_sync(0xffffffffu, acc[e], o);
      acc[e] = acc[e] * c1 + a2 * c2;
    }
    l = l * c1 + l2 * c2;
    m = mn;
  }
  if (g != 0 || !act) return;
  if (nsp == 1) {
    const float inv = 1.f / l;
    T* out = O + (size_t)row * d + h * HD + c * CPE;
#pragma unroll
    for (int e = 0; e < CPE; ++e) out[e] = from_f<T>(acc[e] * inv);
  } else {
    const size_t pi = ((size_t)row * H + h) * max_splits + sp;
    float* po = part_o + pi * HD + c * CPE;
#pragma unroll
    for (int e = 0; e < CPE; ++e) po[e] = acc[e];
    if (c == 0) {
      part_ml[pi * 2] = m;
      part_ml[pi * 2 + 1] = l;
    }
  }
}

// Merge split partials in split order: o = sum_s e^{m_s - m} acc_s / sum_s e^{m_s - m} l_s.
template <typename T>
__global__ void k_attn_combine(int rows, const int* __restrict__ mpos, int H, int HDv, int d, int split,
                               int max_splits, const float* __restrict__ part_o,
                               const float* __restrict__ part_ml, T* __restrict__ O) {
  const int row = blockIdx.x / H, h = blockIdx.x % H;
  if (row >= rows) return;
  const int L = mpos[row] + 1;
  const int nsp = (L + split - 1) / split;
  if (nsp <= 1) return;
  const size_t pi = ((size_t)row * H + h) * max_splits;
  float m = -INFINITY;
  for (int s = 0; s < nsp; ++s) m = fmaxf(m, part_ml[(pi + s) * 2]);
  float l = 0.f;
  for (int s = 0; s < nsp; ++s) l += part_ml[(pi + s) * 2 + 1] * expf(part_ml[(pi + s) * 2] - m);
  const float inv = 1.f / l;
  for (int e = threadIdx.x; e < HDv; e += blockDim.x) {
    float a = 0.f;
    for (int s = 0; s < nsp; ++s) a += part_o[(pi + s) * HDv + e] * expf(part_ml[(pi + s) * 2] - m);
    O[(size_t)row * d + h * HDv + e] = from_f<T>(a * inv);
  }
}

template <typename T, int HD>
static void attn_hd(cudaStream_t s, const T* Q, int rows, const int* mslot, const int* mpos, const int* mdepth,
                    int depth_uniform, KvGeom kv, int slot_base, int clamp, int H, int split, int max_splits,
                    T* O, float* part_o, float* part_ml, int* status) {
  dim3 grid(max_splits, (H + 3) / 4, rows);
  count_launch();
  k_attn<T, HD><<<grid, 128, 0, s>>>(Q, rows, mslot, mpos, mdepth, depth_uniform, kv, slot_base, clamp, H,
                                     split, max_splits, O, part_o, part_ml, status);
  if (max_splits > 1)
    count_launch(), k_attn_combine<T><<<rows * H, 128, 0, s>>>(rows, mpos, H, HD, kv.d, split, max_splits, part_o, part_ml, O);
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
