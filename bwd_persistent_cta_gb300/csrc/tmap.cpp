// tmap.cpp - host-side TMA tensor-map encoding (bf16, 2-D, 128-byte swizzle).
// The driver entry point is looked up at run time through the CUDA runtime,
// so the library has no link-time dependency on the driver library.
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

#include "rnn_internal.h"

namespace rnn {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_once;

void lookup() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
}
}  // namespace

// Row-major matrix ptr[j * ld + i], i < dim0 (contiguous), j < dim1; the box is
// box0 x box1 elements with box0 * 2 == 128 bytes (the swizzle span).
int make_tmap_bf16_2d(void* map, const void* ptr, uint64_t dim0, uint64_t dim1, uint64_t ld_elems,
                      uint32_t box0, uint32_t box1) {
  std::call_once(g_once, lookup);
  if (!g_encode) return 3;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0 || (ld_elems * 2) % 16 != 0) return 2;
  cuuint64_t dims[2] = {dim0, dim1};
  cuuint64_t strides[1] = {ld_elems * 2};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : 2;
}

}  // namespace rnn
