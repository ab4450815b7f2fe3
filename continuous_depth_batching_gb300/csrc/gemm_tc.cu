// Tensor-core GEMM for bf16 models: C = A[rows, K] . W[N, K]^T, fp32 accumulate.
//
// sm_103a, 5th-generation tensor cores.  One CTA computes a 128 (output
// features) x BN (activation rows) tile: the weight tile is the 128-row MMA
// operand and the activation rows form the N side, so a decode batch of a few
// dozen rows still fills the tensor core's M=128 (swap-AB).  Operands arrive
// in shared memory through TMA (128-byte swizzle, 64-element K slabs, a ring
// of STAGES buffers tracked by mbarriers); one thread issues tcgen05.mma into a
// TMEM accumulator; all four warps then read TMEM with tcgen05.ld and apply
// the epilogue (store, residual add, or SwiGLU of two accumulators).
//
// Split-K (decode tilings): the K range is cut into `splits` pieces whose
// count depends only on the weight shape, never on the number of rows, so a
// row's result is the same in every batch.  Each split CTA stores its fp32
// partial tile to a workspace P[split][row][ldp]; the kernel that consumes the
// GEMM's output (RoPE + KV write, residual + RMSNorm, the SwiGLU combine, or
// the residual fold) sums the partials in split order while it reads them.
// With one split the epilogue (store, residual add, SwiGLU) runs in place.
//
// Prefill (many rows, no split) runs a persistent variant, k_gemm_pf: one CTA
// per SM walks the tiles with separate producer, MMA and epilogue warps and
// two TMEM accumulators, so a tile's epilogue overlaps the next tile's MMAs.
//
// Every mbarrier wait is bounded by the global timer; on expiry the kernel
// records kStatusTimeout, skips the epilogue, releases TMEM and returns.
#include <cuda.h>

#include <cstdlib>
#include <cstring>
#include <unordered_map>

#include "common.cuh"
#include "kernels.cuh"

namespace cdb {
namespace tc {

constexpr int BM = 128;  // output features per tile (MMA M)
constexpr int BK = 64;   // K per stage: 128 bytes of bf16 = one swizzle row
constexpr int UK = 16;   // K per tcgen05.mma, kind::f16

__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes)
               : "memory");
}

// Wait for the phase with the given parity; false after ~2 s.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = su32(bar);
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 255) == 0) {
      const uint64_t t = gtimer();
      if (t0 == 0) t0 = t;
      else if (t - t0 > 2000000000ull) return false;
    }
  }
}

__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          su32(dst)),
      "l"(map), "r"(su32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (tcgen05 descriptor version 1).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Apply the epilogue to n (<= 16) consecutive rows of one output column:
// v = first accumulator, u = second (SwiGLU up); o = offset of the first row.
// All residual loads are issued before any store.
template <int EPI>
__device__ __forceinline__ void epilogue16(const float* v, const float* u, int n, float* __restrict__ Cf,
                                           __nv_bfloat16* __restrict__ Ct, size_t o, int ldc) {
  if (EPI == kEpiStore) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < n) Cf[o + (size_t)j * ldc] = v[j];
  } else if (EPI == kEpiResid) {
    float old[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) old[j] = j < n ? Cf[o + (size_t)j * ldc] : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < n) Cf[o + (size_t)j * ldc] = old[j] + v[j];
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < n) Ct[o + (size_t)j * ldc] = __float2bfloat16_rn(v[j] / (1.0f + expf(-v[j])) * u[j]);
  }
}

template <int BN, bool SW, bool DEEP>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES * (SW ? 2 : 1) + B_BYTES;
  // DEEP: one CTA per SM with a 160 KB ring (six weight slabs in flight, four
  // for SwiGLU), for grids of at most one wave: a decode split streams only
  // 5-11 slabs, so the bytes it requests before its first MMA set its
  // bandwidth.  Otherwise two CTAs per SM, so one CTA's prologue and
  // epilogue overlap the other's main loop.
  static constexpr int BUDGET = DEEP ? 160 * 1024 : BN == 64 ? 104 * 1024 : 100 * 1024;
  static_assert(DEEP || BN < 256, "256-row tiles run one CTA per SM (their SwiGLU accumulators fill TMEM)");
  static constexpr int STAGES = BUDGET / STAGE > 8 ? 8 : BUDGET / STAGE;
  static constexpr int ACC = BN * (SW ? 2 : 1);
  static constexpr int TMEM_COLS = ACC <= 32 ? 32 : ACC <= 64 ? 64 : ACC <= 128 ? 128 : ACC <= 256 ? 256 : 512;
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
};

template <int BN, int EPI, bool DEEP>
__global__ void __launch_bounds__(128, DEEP ? 1 : 2)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
              const __grid_constant__ CUtensorMap tmA, int N, int K, int rows, int splits,
              float* __restrict__ Cf, __nv_bfloat16* __restrict__ Ct, int ldc, float* __restrict__ ws,
              int* status) {
  constexpr bool SW = EPI == kEpiSwiglu;
  using C = Cfg<BN, SW, DEEP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* done = empty + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BM;
  const int m0 = blockIdx.y * BN;
  const int split = blockIdx.z;
  const int KT = (K + BK - 1) / BK;
  const int kt0 = (int)((long long)KT * split / splits);
  const int kt1 = (int)((long long)KT * (split + 1) / splits);
  const int nkt = kt1 - kt0;

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
    if (SW) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW2) : "memory");
    s_fail = 0;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // TMA producer.  Weights never change, so the first ring of weight tiles
    // is requested before waiting for the previous kernel; activation tiles
    // only after it has completed.
    const int pre = nkt < C::STAGES ? nkt : C::STAGES;
    for (int i = 0; i < pre; ++i) {
      uint8_t* st = smem + i * C::STAGE;
      mbar_expect_tx(&full[i], C::STAGE);
      const int kx = (kt0 + i) * BK;
      tma_load(st, &tmW, &full[i], kx, n0);
      if (SW) tma_load(st + C::A_BYTES, &tmW2, &full[i], kx, n0);
    }
    pdl_wait();
    pdl_trigger();
    for (int i = 0; i < pre; ++i)
      tma_load(smem + i * C::STAGE + C::A_BYTES * (SW ? 2 : 1), &tmA, &full[i], (kt0 + i) * BK, m0);
    for (int i = pre; i < nkt; ++i) {
      const int s = i % C::STAGES;
      if (!mbar_wait(&empty[s], ((i / C::STAGES) - 1) & 1)) {
        s_fail = 1;
        atomicOr(status, kStatusTimeout);
        break;
      }
      uint8_t* st = smem + s * C::STAGE;
      mbar_expect_tx(&full[s], C::STAGE);
      const int kx = (kt0 + i) * BK;
      tma_load(st, &tmW, &full[s], kx, n0);
      if (SW) tma_load(st + C::A_BYTES, &tmW2, &full[s], kx, n0);
      tma_load(st + C::A_BYTES * (SW ? 2 : 1), &tmA, &full[s], kx, m0);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t id = idesc(BM, BN);
    for (int i = 0; i < nkt; ++i) {
      const int s = i % C::STAGES;
      if (!mbar_wait(&full[s], (i / C::STAGES) & 1)) {
        s_fail = 1;
        atomicOr(status, kStatusTimeout);
        break;
      }
      fence_after();
      const uint32_t a = su32(smem + s * C::STAGE);
      const uint32_t a2 = a + C::A_BYTES;
      const uint32_t b = a + C::A_BYTES * (SW ? 2 : 1);
#pragma unroll
      for (int kk = 0; kk < BK / UK; ++kk) {
        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
        mma(tmem, sdesc(a + kk * 32), sdesc(b + kk * 32), id, acc);
        if (SW) mma(tmem + BN, sdesc(a2 + kk * 32), sdesc(b + kk * 32), id, acc);
      }
      mma_commit(&empty[s]);
    }
    mma_commit(done);
  }
  __syncwarp();
  pdl_wait();  // outputs (and residual inputs) belong to earlier kernels
  const bool ok = mbar_wait(done, 0) && !s_fail;
  fence_after();
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(status, kStatusTimeout);
  } else {
    const int f = n0 + warp * 32 + lane;  // output feature of this thread's TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    if (ws == nullptr) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16], u[16];
        tmem_ld16(lane_base + c0, v);
        if (SW) tmem_ld16(lane_base + BN + c0, u);
        const int jn = min(16, rows - (m0 + c0));
        if (f < N && jn > 0) epilogue16<EPI>(v, u, jn, Cf, Ct, (size_t)(m0 + c0) * ldc + f, ldc);
      }
    } else {
      // This split's partial tile: P[split][row][f] (SwiGLU: up at f + N).
      const size_t ldp = SW ? 2 * (size_t)N : (size_t)N;
      float* P = ws + (size_t)split * rows * ldp;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16], u[16];
        tmem_ld16(lane_base + c0, v);
        if (SW) tmem_ld16(lane_base + BN + c0, u);
        const int jn = min(16, rows - (m0 + c0));
        if (f < N && jn > 0) {
          float* o = P + (size_t)(m0 + c0) * ldp + f;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < jn) {
              o[(size_t)j * ldp] = v[j];
              if (SW) o[(size_t)j * ldp + N] = u[j];
            }
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
}

// ---------------------------------------------------------------------------
// Persistent prefill GEMM: one CTA per SM walks the output tiles (tile t, then
// t + gridDim.x, ...).  Warp 0 streams operand slabs through a STAGES-deep
// ring, warp 1 issues the MMAs, warps 2-5 drain accumulators.  Two TMEM
// accumulator buffers alternate between tiles, so the epilogue of one tile
// overlaps the main loop of the next: the MMA warp waits for `tempty[b]`
// (all four epilogue warps done with buffer b) before reusing it, the
// epilogue warps wait for `tfull[b]` (the tile's last MMA committed).  When
// the grid covers every tile once, buffer 1 is never used and only one is
// allocated, which lets a SwiGLU tile of 192 or 256 rows fit TMEM.  An
// epilogue warp reads the TMEM lane quadrant its warp index selects
// (warp % 4), i.e. output features n0 + 32 * (warp % 4) + lane.
// ---------------------------------------------------------------------------
template <int BN, bool SW>
struct PfCfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES * (SW ? 2 : 1) + B_BYTES;
  static constexpr int STAGES = (196 * 1024) / STAGE > 8 ? 8 : (196 * 1024) / STAGE;
  static constexpr int ACC = BN * (SW ? 2 : 1);  // TMEM columns of one tile's accumulators
  // TMEM columns to allocate (a power of two, at least 32): one buffer when
  // the grid covers every tile once, two when CTAs walk several tiles; 0 when
  // two buffers do not fit, so that such a tile runs in a single pass only.
  static constexpr int TMEM_ONE = ACC <= 32 ? 32 : ACC <= 64 ? 64 : ACC <= 128 ? 128 : ACC <= 256 ? 256 : 512;
  static constexpr int TMEM_TWO = 2 * ACC <= 128 ? 128 : 2 * ACC <= 256 ? 256 : 2 * ACC <= 512 ? 512 : 0;
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
  static_assert(ACC <= 512, "one accumulator buffer must fit TMEM");
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}

template <int BN, int EPI>
__global__ void __launch_bounds__(192, 1)
    k_gemm_pf(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
              const __grid_constant__ CUtensorMap tmA, int N, int K, int rows, float* __restrict__ Cf,
              __nv_bfloat16* __restrict__ Ct, int ldc, int* status) {
  constexpr bool SW = EPI == kEpiSwiglu;
  using C = PfCfg<BN, SW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_n = (N + BM - 1) / BM;
  const int tiles = tiles_n * ((rows + BN - 1) / BN);
  const int KT = (K + BK - 1) / BK;
  const uint32_t tmem_cols = tiles <= (int)gridDim.x ? C::TMEM_ONE : C::TMEM_TWO;
  if (tmem_cols == 0) {  // uniform over the grid: nothing allocated or waited on yet
    if (threadIdx.x == 0) atomicOr(status, kStatusBadLaunch);
    return;
  }

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
    if (SW) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW2) : "memory");
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // activations, residual inputs and outputs belong to earlier kernels
  pdl_trigger();
  bool fail = false;
  if (warp == 0) {
    if (lane == 0) {
      // TMA producer: k-slab `it` counts across all of this CTA's tiles.
      uint32_t it = 0;
      for (int t = blockIdx.x; t < tiles && !fail; t += gridDim.x) {
        const int n0 = (t % tiles_n) * BM, m0 = (t / tiles_n) * BN;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % C::STAGES;
          if (it >= (uint32_t)C::STAGES && !mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1)) {
            fail = true;
            break;
          }
          uint8_t* st = smem + s * C::STAGE;
          mbar_expect_tx(&full[s], C::STAGE);
          tma_load(st, &tmW, &full[s], kt * BK, n0);
          if (SW) tma_load(st + C::A_BYTES, &tmW2, &full[s], kt * BK, n0);
          tma_load(st + C::A_BYTES * (SW ? 2 : 1), &tmA, &full[s], kt * BK, m0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer.
      constexpr uint32_t id = idesc(BM, BN);
      uint32_t it = 0, tl = 0;
      for (int t = blockIdx.x; t < tiles && !fail; t += gridDim.x, ++tl) {
        const uint32_t b = tl & 1, acc0 = tmem + b * C::ACC;
        if (tl >= 2 && !mbar_wait(&tempty[b], ((tl / 2) - 1) & 1)) {
          fail = true;
          break;
        }
        fence_after();
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % C::STAGES;
          if (!mbar_wait(&full[s], (it / C::STAGES) & 1)) {
            fail = true;
            break;
          }
          fence_after();
          const uint32_t a = su32(smem + s * C::STAGE);
          const uint32_t a2 = a + C::A_BYTES;
          const uint32_t bb = a + C::A_BYTES * (SW ? 2 : 1);
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            const uint32_t accum = (kt > 0 || kk > 0) ? 1u : 0u;
            mma(acc0, sdesc(a + kk * 32), sdesc(bb + kk * 32), id, accum);
            if (SW) mma(acc0 + BN, sdesc(a2 + kk * 32), sdesc(bb + kk * 32), id, accum);
          }
          mma_commit(&empty[s]);
        }
        if (fail) break;
        mma_commit(&tfull[b]);
      }
    }
  } else {
    // Epilogue warps 2-5: TMEM lane quadrant warp % 4.
    const int q = warp & 3;
    uint32_t tl = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tl) {
      const uint32_t b = tl & 1;
      // Warp-uniform: tcgen05.ld below is a collective of the whole warp.
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[b], (tl / 2) & 1))) {
        fail = true;
        break;
      }
      fence_after();
      const int n0 = (t % tiles_n) * BM, m0 = (t / tiles_n) * BN;
      const int f = n0 + q * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + b * C::ACC;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16], u[16];
        tmem_ld16(lane_base + c0, v);
        if (SW) tmem_ld16(lane_base + BN + c0, u);
        const int jn = min(16, rows - (m0 + c0));
        if (f < N && jn > 0) epilogue16<EPI>(v, u, jn, Cf, Ct, (size_t)(m0 + c0) * ldc + f, ldc);
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
  }
  fence_before();
  __syncthreads();
  if (fail && lane == 0) atomicOr(status, kStatusTimeout);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols));
}

// ---------------------------------------------------------------------------
// host side: tensor maps (cached), launch
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

struct MapKey {
  const void* p;
  uint64_t inner, outer, stride;
  uint32_t box;
  bool operator==(const MapKey& o) const {
    return p == o.p && inner == o.inner && outer == o.outer && stride == o.stride && box == o.box;
  }
};
struct MapHash {
  size_t operator()(const MapKey& k) const {
    return std::hash<const void*>()(k.p) ^ (k.inner * 1315423911ull) ^ (k.outer << 20) ^ (k.stride << 7) ^ k.box;
  }
};

// bf16 [outer][inner] with row stride `stride` bytes, box 64 x box, 128-byte swizzle.
static const CUtensorMap* get_map(const void* p, uint64_t inner, uint64_t outer, uint64_t stride, uint32_t box) {
  static std::unordered_map<MapKey, CUtensorMap, MapHash> cache;
  MapKey k{p, inner, outer, stride, box};
  auto it = cache.find(k);
  if (it != cache.end()) return &it->second;
  EncodeFn enc = encoder();
  if (!enc) return nullptr;
  CUtensorMap m;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {stride};
  cuuint32_t boxd[2] = {(cuuint32_t)BK, box};
  cuuint32_t es[2] = {1, 1};
  if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, boxd, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return nullptr;
  return &cache.emplace(k, m).first->second;
}

template <int BN, int EPI, bool DEEP>
static bool launch_bn_cfg(cudaStream_t s, const CUtensorMap* mw, const CUtensorMap* mw2, const CUtensorMap* ma,
                          int N, int K, int rows, int splits, float* Cf, __nv_bfloat16* Ct, int ldc, float* ws,
                          int* status) {
  using C = Cfg<BN, EPI == kEpiSwiglu, DEEP>;
  static bool attr[kMaxDevices] = {};
  const int dev = current_device();
  if (!attr[dev]) {
    if (cudaFuncSetAttribute(k_gemm_tc<BN, EPI, DEEP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
      return false;
    attr[dev] = true;
  }
  count_launch();
  return launch_pdl(k_gemm_tc<BN, EPI, DEEP>, dim3((N + BM - 1) / BM, (rows + BN - 1) / BN, splits), dim3(128),
                    C::SMEM, s, *mw, *mw2, *ma, N, K, rows, splits, Cf, Ct, ldc, ws, status) == cudaSuccess;
}

// The ring depth changes neither the MMA order nor the split count, so a
// row's result is the same whichever configuration runs.
template <int BN, int EPI>
static bool launch_bn(cudaStream_t s, const __nv_bfloat16* A, int lda, int a_rows, const __nv_bfloat16* W,
                      const __nv_bfloat16* W2, int N, int K, int rows, int splits, float* Cf,
                      __nv_bfloat16* Ct, int ldc, float* ws, int* status, int sms) {
  const CUtensorMap* mw = get_map(W, K, N, (uint64_t)K * 2, BM);
  const CUtensorMap* mw2 = EPI == kEpiSwiglu ? get_map(W2, K, N, (uint64_t)K * 2, BM) : mw;
  const CUtensorMap* ma = get_map(A, K, a_rows, (uint64_t)lda * 2, BN);
  if (!mw || !mw2 || !ma) return false;
  const long long ctas = (long long)((N + BM - 1) / BM) * ((rows + BN - 1) / BN) * splits;
  if constexpr (BN == 256) {
    if (ctas > sms) return false;  // the caller takes 256-row tiles only for one-wave grids
    return launch_bn_cfg<BN, EPI, true>(s, mw, mw2, ma, N, K, rows, splits, Cf, Ct, ldc, ws, status);
  } else {
    return ctas <= sms ? launch_bn_cfg<BN, EPI, true>(s, mw, mw2, ma, N, K, rows, splits, Cf, Ct, ldc, ws, status)
                       : launch_bn_cfg<BN, EPI, false>(s, mw, mw2, ma, N, K, rows, splits, Cf, Ct, ldc, ws, status);
  }
}

// Persistent prefill launch: min(tiles, max_ctas) CTAs of 192 threads.
template <int BN, int EPI>
static bool launch_pf(cudaStream_t s, const __nv_bfloat16* A, int lda, int a_rows, const __nv_bfloat16* W,
                      const __nv_bfloat16* W2, int N, int K, int rows, float* Cf, __nv_bfloat16* Ct, int ldc,
                      int max_ctas, int* status) {
  using C = PfCfg<BN, EPI == kEpiSwiglu>;
  const CUtensorMap* mw = get_map(W, K, N, (uint64_t)K * 2, BM);
  const CUtensorMap* mw2 = EPI == kEpiSwiglu ? get_map(W2, K, N, (uint64_t)K * 2, BM) : mw;
  const CUtensorMap* ma = get_map(A, K, a_rows, (uint64_t)lda * 2, BN);
  if (!mw || !mw2 || !ma) return false;
  static bool attr[kMaxDevices] = {};
  const int dev = current_device();
  if (!attr[dev]) {
    if (cudaFuncSetAttribute(k_gemm_pf<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
      return false;
    attr[dev] = true;
  }
  const long long tiles = (long long)((N + BM - 1) / BM) * ((rows + BN - 1) / BN);
  const int grid = (int)(tiles < max_ctas ? tiles : max_ctas);
  count_launch();
  return launch_pdl(k_gemm_pf<BN, EPI>, dim3(grid), dim3(192), C::SMEM, s, *mw, *mw2, *ma, N, K, rows, Cf, Ct, ldc,
                    status) == cudaSuccess;
}

}  // namespace tc

static int sm_count() {
  static int n[kMaxDevices] = {};
  const int dev = current_device();
  if (!n[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    n[dev] = v;
  }
  return n[dev];
}

// Split count of a decode GEMM: at least four 64-element K slabs per split,
// at most kGemmMaxSplits, and about one CTA per SM for a 64-row tile of
// activations.  Depends only on the weight shape (and the device), never on
// the number of rows.
int gemm_tc_splits(int N, int K, bool decode) {
  if (!decode) return 1;
  const int tiles = (N + tc::BM - 1) / tc::BM;
  const int KT = (K + tc::BK - 1) / tc::BK;
  int s = sm_count() / tiles;
  if (s > KT / 4) s = KT / 4;
  if (s > kGemmMaxSplits) s = kGemmMaxSplits;
  return s < 1 ? 1 : s;
}

// Split count of a narrow weight (fewer than 32 tiles of 128 features) in a
// wide decode batch: about one CTA per SM for two 256-row activation tiles,
// at least four K slabs per split, at most kWideMaxSplits.  Depends only on
// the weight shape (and the device), never on the number of rows.
static int gemm_tc_wide_splits(int N, int K) {
  const int tiles = (N + tc::BM - 1) / tc::BM;
  const int KT = (K + tc::BK - 1) / tc::BK;
  int s = sm_count() / (2 * tiles);
  if (s > KT / 4) s = KT / 4;
  if (s > kWideMaxSplits) s = kWideMaxSplits;
  return s < 1 ? 1 : s;
}

int launch_gemm_tc(cudaStream_t s, int epi, const __nv_bfloat16* A, int lda, int a_rows, const __nv_bfloat16* W,
                   const __nv_bfloat16* W2, int N, int K, int rows, float* Cf, __nv_bfloat16* Ct, int ldc,
                   int tiling, float* ws, size_t ws_floats, int* status) {
  if (rows <= 0) return 0;
  if ((K * 2) % 16 != 0 || (lda * 2) % 16 != 0 || rows > a_rows) return -1;
  const int sm = sm_count();
  const long long tiles_n = (N + tc::BM - 1) / tc::BM;
  // Narrow weights in wide decode batches (the O and down projections):
  // their few feature tiles leave a CTA a long K loop of small tiles, so
  // they split K instead (consumers fold the partials, as for decode).
  const bool narrow = tiling == kTileWide && tiles_n < 32;
  int splits = !ws ? 1 : tiling == kTileSplit ? gemm_tc_splits(N, K, true) : narrow ? gemm_tc_wide_splits(N, K) : 1;
  const size_t ldp = epi == kEpiSwiglu ? 2 * (size_t)N : (size_t)N;
  // Consumers fold partials four columns at a time.
  if (splits > 1 && ((size_t)splits * rows * ldp > ws_floats || N % 4 != 0)) splits = 1;
  float* P = splits > 1 ? ws : nullptr;
  const bool decode = tiling == kTileSplit || (narrow && P);
  bool ok;
  if (decode) {
    // Activation tile height.  Decode tiling: the smallest of 64, 128 and
    // 256 rows that holds the batch, while the grid stays one wave (else
    // 128-row tiles).  Split narrow weights of wide batches: 64, 128 or 256
    // rows, whichever minimises waves x bytes per k-slab of a tile (weight
    // rows plus activation rows; the smallest on a tie).  The split count
    // comes from the weight shape alone and a tile's height does not change
    // the order in which a row's products are summed, so a row's result is
    // the same for every batch size.
    const long long one_wave = tiles_n * splits;
    int bn = rows <= 64 ? 64 : rows <= 128 ? 128 : rows <= 256 ? 256 : 128;
    if (bn == 256 && one_wave > sm) bn = 128;
    if (tiling == kTileWide) {
      const int wrows = epi == kEpiSwiglu ? 2 * tc::BM : tc::BM;
      long long best = -1;
      for (int b : {64, 128, 256}) {
        const long long waves = (one_wave * ((rows + b - 1) / b) + sm - 1) / sm;
        const long long cost = waves * (wrows + b);
        if (best < 0 || cost < best) {
          best = cost;
          bn = b;
        }
      }
    }
#define CDB_BN(B)                                                                                                \
  switch (epi) {                                                                                                 \
    case kEpiStore: ok = tc::launch_bn<B, kEpiStore>(s, A, lda, a_rows, W, W2, N, K, rows, splits, Cf, Ct, ldc, P, status, sm); break; \
    case kEpiResid: ok = tc::launch_bn<B, kEpiResid>(s, A, lda, a_rows, W, W2, N, K, rows, splits, Cf, Ct, ldc, P, status, sm); break; \
    default: ok = tc::launch_bn<B, kEpiSwiglu>(s, A, lda, a_rows, W, W2, N, K, rows, splits, Cf, Ct, ldc, P, status, sm); break; \
  }
    if (bn == 64) {
      CDB_BN(64)
    } else if (bn == 128) {
      CDB_BN(128)
    } else {
      CDB_BN(256)
    }
#undef CDB_BN
  } else {
    // Persistent: one CTA per SM, double-buffered accumulators.  Prefill:
    // 256-row tiles where one accumulator fits, 128-row tiles for SwiGLU.
    const bool wide = tiling == kTilePrefill && rows > 128;
    // Wide decode batches, narrow weights without a split workspace: 64-row
    // tiles, so the tiles outnumber the SMs.  Other wide decode GEMMs: 128,
    // 192 or 256 rows, whichever minimises waves x bytes per k-slab of a tile
    // (128 weight rows, 256 for SwiGLU, plus the tile's activation rows),
    // since a CTA streams a tile's slabs through a ring of fixed size; the
    // smallest on a tie.  SwiGLU takes 192 or 256 rows only in one wave,
    // where each CTA needs one accumulator buffer.  Without split-K a row's
    // result is the same for any tile height.
    int bn = wide ? 256 : narrow ? 64 : 128;
    if (tiling == kTileWide && !narrow) {
      const int wrows = epi == kEpiSwiglu ? 2 * tc::BM : tc::BM;
      long long best = -1;
      for (int b : {128, 192, 256}) {
        const long long waves = (tiles_n * ((rows + b - 1) / b) + sm - 1) / sm;
        if (epi == kEpiSwiglu && b > 128 && waves > 1) continue;
        const long long cost = waves * (wrows + b);
        if (best < 0 || cost < best) {
          best = cost;
          bn = b;
        }
      }
    }
    const int sbn = tiling == kTileWide && !narrow ? bn : 128;
#define CDB_PF(E)                                                                                          \
  ok = bn == 64    ? tc::launch_pf<64, E>(s, A, lda, a_rows, W, W2, N, K, rows, Cf, Ct, ldc, sm, status)  \
       : bn == 192 ? tc::launch_pf<192, E>(s, A, lda, a_rows, W, W2, N, K, rows, Cf, Ct, ldc, sm, status) \
       : bn == 256 ? tc::launch_pf<256, E>(s, A, lda, a_rows, W, W2, N, K, rows, Cf, Ct, ldc, sm, status) \
                   : tc::launch_pf<128, E>(s, A, lda, a_rows, W, W2, N, K, rows, Cf, Ct, ldc, sm, status);
    switch (epi) {
      case kEpiStore: CDB_PF(kEpiStore) break;
      case kEpiResid: CDB_PF(kEpiResid) break;
#undef CDB_PF
      default:
        ok = sbn == 192   ? tc::launch_pf<192, kEpiSwiglu>(s, A, lda, a_rows, W, W2, N, K, rows, Cf, Ct, ldc, sm, status)
             : sbn == 256 ? tc::launch_pf<256, kEpiSwiglu>(s, A, lda, a_rows, W, W2, N, K, rows, Cf, Ct, ldc, sm, status)
                          : tc::launch_pf<128, kEpiSwiglu>(s, A, lda, a_rows, W, W2, N, K, rows, Cf, Ct, ldc, sm, status);
        break;
    }
  }
  if (!ok) return -1;
  return P ? splits : 0;
}

}  // namespace cdb
