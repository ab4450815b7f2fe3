// Tensor-map encoding through the driver entry point exposed by the runtime
// (the library links no driver library directly).
#include "tmap.h"

#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

namespace cdb {

namespace {

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

struct Key {
  const void* p;
  uint64_t inner, outer, stride;
  uint32_t bi, bo;
  int sw;
  bool operator==(const Key& o) const {
    return p == o.p && inner == o.inner && outer == o.outer && stride == o.stride && bi == o.bi && bo == o.bo &&
           sw == o.sw;
  }
};
struct KeyHash {
  size_t operator()(const Key& k) const {
    size_t h = std::hash<const void*>()(k.p);
    for (uint64_t v : {k.inner, k.outer, k.stride, (uint64_t)k.bi, (uint64_t)k.bo, (uint64_t)k.sw})
      h = h * 1000003u ^ std::hash<uint64_t>()(v);
    return h;
  }
};

}  // namespace

const CUtensorMap* tmap_bf16_2d(const void* p, uint64_t inner, uint64_t outer, uint64_t stride, uint32_t box_inner,
                                uint32_t box_outer, int swizzle) {
  static std::mutex mu;
  static std::unordered_map<Key, CUtensorMap, KeyHash> cache;
  std::lock_guard<std::mutex> lock(mu);
  const Key k{p, inner, outer, stride, box_inner, box_outer, swizzle};
  auto it = cache.find(k);
  if (it != cache.end()) return &it->second;
  EncodeFn enc = encoder();
  if (!enc) return nullptr;
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  else if (swizzle == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  else if (swizzle == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  else if (swizzle != 0) return nullptr;
  CUtensorMap m;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {stride};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return nullptr;
  return &cache.emplace(k, m).first->second;
}

}  // namespace cdb
