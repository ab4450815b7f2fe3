// Decode attention for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocating routine) at the
// point where they need attention: for example a plugin inside a host program
// whose memory manager owns every byte of device memory, or a latency-critical
// path that cannot afford an allocation's implicit device synchronisation.
// cdb_attention_noalloc serves them: it runs the same split-KV decode-attention
// kernel as cdb_test_attention, but its scratch (the per-split partial results
// and a status word) lives in a fixed array compiled into this library instead
// of memory the caller provides.  The caller still passes every input and the
// output buffer.
#include <mutex>

#include "../../include/cdb.h"
#include "../../include/cdb_testing.h"
#include "kernels.cuh"

namespace {

// Size of the built-in scratch.  Every GPU that loads this library keeps this
// much device memory reserved until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// The built-in scratch.  In host code this name is only a stand-in for the
// device array: its device address must be looked up with
// cudaGetSymbolAddress on each device before a kernel may use it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the built-in scratch on the current device (looked up
// once per device, with that device current).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

int cdb_attention_noalloc(const void* q, int rows, const int32_t* slot, const int32_t* pos, const int32_t* depth,
                          const void* kv_pool, const int32_t* block_table, int max_blocks, const uint8_t* exit_table,
                          int kv_blocks, int n_kv_slots, int slot_base, int n_heads, int head_dim, int dtype,
                          int split, int max_ctx, void* out, void* stream) {
  const bool hd_ok = head_dim == 8 || head_dim == 16 || head_dim == 32 || head_dim == 64 || head_dim == 96 ||
                     head_dim == 128;
  if (!q || rows < 1 || !slot || !pos || !depth || !kv_pool || !block_table || max_blocks < 1 || !exit_table ||
      kv_blocks < 1 || n_kv_slots < 1 || slot_base < 0 || n_heads < 1 || !hd_ok ||
      (dtype != CDB_FP32 && dtype != CDB_BF16) || split < 16 || split % 16 != 0 || max_ctx < 1 || !out)
    return CDB_ERR_ARG;
  // Scratch layout: status word, then per-(row, head, split) partial outputs,
  // then their (max, sum) pairs.
  const size_t splits = (size_t)(max_ctx + split - 1) / split;
  const size_t po_bytes = ((size_t)rows * n_heads * splits * head_dim * 4 + 255) / 256 * 256;
  const size_t ml_bytes = (size_t)rows * n_heads * splits * 2 * 4;
  if (256 + po_bytes + ml_bytes > kNoAllocScratchBytes) return CDB_ERR_ARG;  // too large for the built-in scratch
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return CDB_ERR_CUDA;
  char* w = static_cast<char*>(base);
  int* status = reinterpret_cast<int*>(w);
  float* part_o = reinterpret_cast<float*>(w + 256);
  float* part_ml = reinterpret_cast<float*>(w + 256 + po_bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents; only the status area must
  // start at zero (every partial read is written earlier in this call).
  if (cudaMemsetAsync(status, 0, cdb::kStatusBytes, s) != cudaSuccess) return CDB_ERR_CUDA;
  cdb::KvGeom g;
  g.pool = const_cast<void*>(kv_pool);
  g.bt = block_table;
  g.etab = const_cast<uint8_t*>(exit_table);
  g.max_blocks = max_blocks;
  g.kv_blocks = kv_blocks;
  g.nsl = n_kv_slots;
  g.d = n_heads * head_dim;
  if (dtype == CDB_BF16)
    cdb::launch_attention<__nv_bfloat16>(s, static_cast<const __nv_bfloat16*>(q), rows, slot, pos, depth, 0, g,
                                         slot_base, cdb::kNoSlotCap, n_heads, head_dim, split, (int)splits,
                                         static_cast<__nv_bfloat16*>(out), part_o, part_ml, status, false);
  else
    cdb::launch_attention<float>(s, static_cast<const float*>(q), rows, slot, pos, depth, 0, g, slot_base,
                                 cdb::kNoSlotCap,
                                 n_heads, head_dim, split, (int)splits, static_cast<float*>(out), part_o, part_ml,
                                 status, false);
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return CDB_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CDB_ERR_CUDA;
  return st ? CDB_ERR_DEVICE_BOUNDS : CDB_OK;
}

}  // extern "C"
