// Causal prefill attention on the 5th-generation tensor cores (bf16, head_dim
// 64 or 128): the chunked prefill of "Depth-adaptive Inference of Looped
// Language Models via Continuous Depth Batching" (App. A.1, every prompt
// position at full depth; App. A.5 runs it as a varlen prefill attention).
//
// A prefill chunk's rows arrive sequence by sequence with consecutive
// positions; the host cuts them into query tiles of up to 128 rows of one
// sequence.  One CTA per (tile, head), six warps:
//   warp 4      TMA producer: the tile's q rows once, then the sequence's keys
//               in blocks of 64 (four 16-key pages of K and of V per block,
//               each page a 2D tensor copy per 64-element slice of the head,
//               128-byte swizzle) through a ring of kStages blocks;
//   warp 5      MMA issuer: S_j = Q K_j^T (M 128 rows, N 64 keys) into one of
//               two TMEM score buffers, then O_j = P_j V_j (N = head_dim) into
//               one of two TMEM output buffers, P fed as a bf16 hi/lo pair
//               (two MMAs, about 16 significant bits of each weight);
//   warps 0-3   softmax: thread t owns query row t (its TMEM lane).  It reads
//               its 64 scores, applies the causal mask and the online
//               softmax (log2 domain), writes P_j to shared memory in the
//               MMA's K-major swizzled layout, and accumulates O_j from TMEM
//               into registers rescaled by the running maximum.
// S_{j+1} is computed while the softmax warps work on block j, and P_{j+1} is
// formed while the tensor core runs P_j V_j.  V is the MMA's B operand in its
// stored [key][head_dim] order, i.e. N-major ("MN-major") under the 128-byte
// swizzle: 8-key groups 1024 bytes apart, 64-element column groups one slice
// apart.  Every mbarrier wait is bounded; on expiry the kernel records
// kStatusTimeout, waits (bounded) for its own copies and MMAs, frees TMEM and
// returns.
#include "common.cuh"
#include "kernels.cuh"
#include "tmap.h"

namespace cdb {
namespace pftc {

constexpr int kRows = 128;   // query rows per tile: MMA M, TMEM lanes
constexpr int kKeys = 64;    // keys per block: four 16-key pages
constexpr int kStages = 3;   // key blocks in flight

template <int HD>
struct Geo {
  static_assert(HD == 64 || HD == 128, "head dim");
  static constexpr int NX = HD / 64;             // 128-byte slices of a head row
  static constexpr int QSLICE = kRows * 128;     // one slice of the q tile
  static constexpr int QBYTES = NX * QSLICE;
  static constexpr int KSLICE = kKeys * 128;     // one slice of a key block
  static constexpr int KVB = NX * KSLICE;        // K (or V) of one block
  static constexpr int STAGE = 2 * KVB;
  static constexpr int PPART = kRows * kKeys * 2;  // P hi (or lo): 128 rows x 64 keys bf16
  static constexpr int PBUF = 2 * PPART;
  static constexpr int OFF_KV = QBYTES;
  static constexpr int OFF_P = OFF_KV + kStages * STAGE;
  static constexpr int OFF_XCH = OFF_P + 2 * PBUF;   // fp32 [6][kRows]: row maxima, then row sums
  static constexpr int OFF_BAR = OFF_XCH + 6 * kRows * 4;
  static constexpr int NBAR = 2 + 2 * kStages + 8 + 12;  // q, done, kv full/empty, s full/free, p full, o done, pairs
  static constexpr size_t SMEM = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr int S_COL = 0;                // two score buffers of kKeys columns
  static constexpr int O_COL = 2 * kKeys;        // the output accumulator, HD columns
  static constexpr int TMEM_COLS = O_COL + HD <= 256 ? 256 : 512;
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
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

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                       uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(map), "r"(su32(bar)), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

// 2^x on the special-function unit (ex2.approx, within a few fp32 ulp;
// results below 2^-126 flush to zero, a weight negligible against the row's
// maximum weight of 1).  One instruction per softmax weight, where exp2f adds
// range handling around the same instruction.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptors (tcgen05 version 1, 128-byte swizzle,
// 8-row groups 1024 bytes apart).  K-major: the K extent of one MMA lies
// inside a 128-byte row, stepped by moving the start address.  MN-major: N is
// contiguous inside a 128-byte row (64 elements), further 64-element groups
// `lbo` bytes apart.
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major or (b_mn) MN-major.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

}  // namespace pftc

template <int HD>
__global__ void __launch_bounds__(320, 1)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const int4* __restrict__ tiles, KvGeom kv, int slot, int H, __nv_bfloat16* __restrict__ O,
                      int* status) {
  using namespace pftc;
  using G = Geo<HD>;
  constexpr int HH = HD / 2;  // output columns of one softmax warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem;
  uint8_t* kvs = smem + G::OFF_KV;
  uint8_t* ps = smem + G::OFF_P;
  float* xch = reinterpret_cast<float*>(smem + G::OFF_XCH);  // [2 parities][2 halves][128 rows] maxima, then sums
  uint64_t* qbar = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* done = qbar + 1;
  uint64_t* kv_full = done + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* pair = o_done + 2;  // [quadrant][parity] exchange barriers, then one per quadrant for the sums
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pair + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmq) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmk) : "memory");
    mbar_init(qbar, 1);
    mbar_init(done, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 8);
      mbar_init(&p_full[b], 8);
      mbar_init(&o_done[b], 1);
    }
    for (int i = 0; i < 12; ++i) mbar_init(&pair[i], 64);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(G::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  const int4 tile = tiles[blockIdx.x];  // (first row, rows, sequence slot, position of the first row)
  const int row0 = tile.x, nq = tile.y, p0 = tile.w;
  const int kmax = p0 + nq - 1;  // the tile's last position: the last key any of its rows reads
  const int nb = kmax / kKeys + 1;
  const int npg = kmax / 16 + 1;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint64_t pol;  // keys and values are read again by the sequence's later tiles
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
      mbar_arrive_tx(qbar, G::QBYTES);
      for (int x = 0; x < G::NX; ++x) tma_2d(su32(qs + x * G::QSLICE), &tmq, qbar, h * HD + x * 64, row0, pol);
      const int* bt = kv.bt + tile.z * kv.max_blocks;
      const bool sl_ok = slot >= 0 && slot < kv.nsl;
      if (!sl_ok) atomicOr(status, kStatusBadDepth);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < nb; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !mbar_wait(&kv_empty[s], ((j / kStages) - 1) & 1)) {
          ok = false;
          break;
        }
        int blk[4];
        uint32_t bytes = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pg = 4 * j + i;
          blk[i] = -1;
          if (pg < npg) {
            const int b = bt[pg];
            if (sl_ok && b >= 0 && b < kv.kv_blocks) {
              blk[i] = b;
              bytes += 2u * G::NX * 16 * 128;
            } else if (sl_ok) {
              atomicOr(status, kStatusBadBlock);
            }
          }
        }
        mbar_arrive_tx(&kv_full[s], bytes);
        const uint32_t st = su32(kvs + (size_t)s * G::STAGE);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (blk[i] < 0) continue;
          // Rows of head h's page at this slot: K, then V (H * 16 rows later).
          const int y = (int)((((long long)blk[i] * kv.nsl + slot) * 2 * H + h) * 16);
          for (int x = 0; x < G::NX; ++x) {
            tma_2d(st + x * G::KSLICE + i * 16 * 128, &tmk, &kv_full[s], x * 64, y, pol);
            tma_2d(st + G::KVB + x * G::KSLICE + i * 16 * 128, &tmk, &kv_full[s], x * 64, y + H * 16, pol);
          }
        }
        issued = j + 1;
      }
      if (!ok) atomicOr(status, kStatusTimeout);
      // Copies already issued land before the CTA may leave (immediate when
      // the consumers have taken every block).
      mbar_wait(qbar, 0);
      for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
        mbar_wait(&kv_full[j % kStages], (j / kStages) & 1);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idS = idesc(kRows, kKeys, false), idO = idesc(kRows, HD, true);
      const uint32_t qa = su32(qs);
      bool ok = mbar_wait(qbar, 0);
      auto issue_qk = [&](int j) -> bool {
        const int s = j % kStages, b = j & 1;
        if (!mbar_wait(&kv_full[s], (j / kStages) & 1)) return false;
        if (j >= 2 && !mbar_wait(&s_free[b], ((j - 2) >> 1) & 1)) return false;
        fence_after();
        const uint32_t kb = su32(kvs + (size_t)s * G::STAGE);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma(tmem + G::S_COL + b * kKeys, desc_k(qa + (kk / 4) * G::QSLICE + (kk % 4) * 32),
              desc_k(kb + (kk / 4) * G::KSLICE + (kk % 4) * 32), idS, kk > 0 ? 1u : 0u);
        commit(&s_full[b]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; ok && j < nb; ++j) {
        if (j + 1 < nb && !(ok = issue_qk(j + 1))) break;
        const int s = j % kStages, b = j & 1;
        if (!(ok = mbar_wait(&p_full[b], (j >> 1) & 1))) break;
        fence_after();
        const uint32_t pb = su32(ps + b * G::PBUF);
        const uint32_t vb = su32(kvs + (size_t)s * G::STAGE + G::KVB);
        // O += P_hi V_j + P_lo V_j over the block's four 16-key steps; block 0
        // starts the accumulator.
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma(tmem + G::O_COL, desc_k(pb + kk * 32), desc_mn(vb + kk * 2048, G::KSLICE), idO,
              (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma(tmem + G::O_COL, desc_k(pb + G::PPART + kk * 32), desc_mn(vb + kk * 2048, G::KSLICE), idO, 1u);
        commit(&o_done[b]);
        commit(&kv_empty[s]);
      }
      if (!ok) atomicOr(status, kStatusTimeout);
      // Every MMA issued above completes before TMEM is released.
      commit(done);
      mbar_wait(done, 0);
    }
  } else {
    // ---------------- softmax warps ----------------
    // Warps w and w + 4 share query rows 32 (w % 4) .. + 31 (TMEM lanes of
    // that quadrant): warp half hf = w / 4 takes keys 32 hf .. + 31 of each
    // block and output columns hf * HD / 2 .. + HD / 2.  The pair exchanges
    // its row maxima through shared memory behind a bounded mbarrier.
    const int q4 = warp & 3, hf = warp >> 2;
    const int r = q4 * 32 + lane;
    const int lim = min(p0 + r, kmax);  // last key of row r (rows past the tile end stop at kmax)
    const float scale = 1.4426950408889634f / sqrtf((float)HD);
    constexpr float kTau = 8.f;  // rescale O only when the row maximum grows by more than 2^8
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t pbase = su32(ps) + (uint32_t)(r >> 3) * 1024 + (uint32_t)(r & 7) * 128;
    float m = -INFINITY, l = 0.f;  // m: log2-domain maximum the weights are taken against
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int b = j & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b], (j >> 1) & 1)))) break;
      fence_after();
      float sv[32];
      tmem_ld32(trow + G::S_COL + b * kKeys + hf * 32, sv);
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[b]);
      const int k0 = j * kKeys + hf * 32;
      float mx = -INFINITY;
      if (k0 + 31 <= p0) {  // every key of this half block precedes every row of the tile
#pragma unroll
        for (int c = 0; c < 32; ++c) mx = fmaxf(mx, sv[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          sv[c] = k0 + c <= lim ? sv[c] : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
      }
      mx *= scale;
      xch[(b * 2 + hf) * kRows + r] = mx;
      mbar_arrive(&pair[q4 * 2 + b]);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&pair[q4 * 2 + b], (j >> 1) & 1)))) break;
      mx = fmaxf(mx, xch[(b * 2 + (hf ^ 1)) * kRows + r]);  // finite: key 0 is visible to every row
      const float mnew = mx > m + kTau ? mx : m;
      const float factor = exp2f(m - mnew);  // 1 without a rescale, 0 for the first block
      if (j > 0 && __any_sync(0xffffffffu, mnew != m)) {
        // O holds blocks 0 .. j-1 against the old maximum: wait for P_{j-1} V_{j-1}.
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1))))
          break;
        fence_after();
#pragma unroll
        for (int c0 = 0; c0 < HH; c0 += 32) {
          float v[32];
          tmem_ld32(trow + G::O_COL + hf * HH + c0, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] *= factor;
          tmem_st32(trow + G::O_COL + hf * HH + c0, v);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      l *= factor;
      m = mnew;
      // P buffer b was last read by P_{j-2} V_{j-2}.
      if (j >= 2 && !(ok = __all_sync(0xffffffffu, mbar_wait(&o_done[b], ((j - 2) >> 1) & 1)))) break;
      const uint32_t ph = pbase + b * G::PBUF, pl = ph + G::PPART;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = ex2(fmaf(sv[8 * cc + 2 * e], scale, -m));
          const float x1 = ex2(fmaf(sv[8 * cc + 2 * e + 1], scale, -m));
          l += x0 + x1;
          hi[e] = pack_bf16(x0, x1);
          const float h0 = __uint_as_float(hi[e] << 16), h1 = __uint_as_float(hi[e] & 0xFFFF0000u);
          lo[e] = pack_bf16(x0 - h0, x1 - h1);
        }
        const uint32_t off = (uint32_t)(((hf * 4 + cc) ^ (r & 7)) * 16);
        st_shared_v4(ph + off, hi[0], hi[1], hi[2], hi[3]);
        st_shared_v4(pl + off, lo[0], lo[1], lo[2], lo[3]);
      }
      if (j == nb - 1 && kmax - j * kKeys < kKeys - 1) {
        // Keys past the tile's last position: their weights are 0, but their
        // V rows may hold NaN (unwritten positions) or a previous block's
        // keys; zero them so that 0 * NaN never reaches the accumulator.
        const int s = j % kStages;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&kv_full[s], (j / kStages) & 1)))) break;
        uint8_t* vt = kvs + (size_t)s * G::STAGE + G::KVB;
        const int first = kmax - j * kKeys + 1;
        for (int u = warp * 32 + lane; u < (kKeys - first) * G::NX * 8; u += 256) {
          const int row = first + u / (G::NX * 8), rem = u % (G::NX * 8);
          *reinterpret_cast<uint4*>(vt + (size_t)(rem / 8) * G::KSLICE + (size_t)row * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[(nb - 1) & 1], ((nb - 1) >> 1) & 1));
    float lt = 0.f;
    if (ok) {
      xch[(4 + hf) * kRows + r] = l;  // sums: a region the maxima never use
      mbar_arrive(&pair[8 + q4]);
      ok = __all_sync(0xffffffffu, mbar_wait(&pair[8 + q4], 0));
      lt = l + xch[(4 + (hf ^ 1)) * kRows + r];
    }
    if (!ok) {
      if (lane == 0) atomicOr(status, kStatusTimeout);
    } else {
      fence_after();
      const float inv = 1.f / lt;
      __nv_bfloat16* dst = O + (size_t)(row0 + r) * kv.d + (size_t)h * HD + hf * HH;
#pragma unroll
      for (int c0 = 0; c0 < HH; c0 += 32) {
        float v[32];
        tmem_ld32(trow + G::O_COL + hf * HH + c0, v);
        if (r < nq) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 u;
            u.x = pack_bf16(v[c] * inv, v[c + 1] * inv);
            u.y = pack_bf16(v[c + 2] * inv, v[c + 3] * inv);
            u.z = pack_bf16(v[c + 4] * inv, v[c + 5] * inv);
            u.w = pack_bf16(v[c + 6] * inv, v[c + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c0 + c) = u;
          }
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 9) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(G::TMEM_COLS));
  }
}

template <int HD>
static bool prefill_tc_hd(cudaStream_t s, const __nv_bfloat16* Q, int q_rows, const int4* tiles, int n_tiles,
                          KvGeom kv, int slot, int H, __nv_bfloat16* O, int* status) {
  using G = pftc::Geo<HD>;
  const uint64_t pool_rows = (uint64_t)kv.kv_blocks * kv.nsl * 2 * H * 16;
  if (pool_rows + 16 >= (1ull << 31) || q_rows + pftc::kRows >= (1 << 30)) return false;
  const CUtensorMap* tk = tmap_bf16_2d(kv.pool, HD, pool_rows, (uint64_t)HD * 2, 64, 16, 128);
  const CUtensorMap* tq = tmap_bf16_2d(Q, (uint64_t)kv.d, q_rows, (uint64_t)kv.d * 2, 64, pftc::kRows, 128);
  if (!tk || !tq) return false;
  static bool set[kMaxDevices] = {};
  const int dev = current_device();
  if (!set[dev]) {
    if (cudaFuncSetAttribute(k_attn_prefill_tc<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::SMEM) !=
        cudaSuccess)
      return false;
    set[dev] = true;
  }
  count_launch();
  return launch_pdl(k_attn_prefill_tc<HD>, dim3(n_tiles, H), dim3(320), G::SMEM, s, *tq, *tk, tiles, kv, slot, H, O,
                    status) == cudaSuccess;
}

bool launch_prefill_attention_tc(cudaStream_t s, const __nv_bfloat16* Q, int q_rows, const int4* tiles, int n_tiles,
                                 KvGeom kv, int slot, int H, int hd, __nv_bfloat16* O, int* status) {
  if (n_tiles <= 0) return true;
  switch (hd) {
    case 64: return prefill_tc_hd<64>(s, Q, q_rows, tiles, n_tiles, kv, slot, H, O, status);
    case 128: return prefill_tc_hd<128>(s, Q, q_rows, tiles, n_tiles, kv, slot, H, O, status);
    default: return false;
  }
}

}  // namespace cdb
