// tmap.cpp - host-side TMA tensor-map encoding (bf16, 2-D and 4-D, 128-byte swizzle).
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
// box0 x box1 elements with box0 * 2 == swizzle_bytes (the swizzle span, 128
// or 64).
int make_tmap_bf16_2d(void* map, const void* ptr, uint64_t dim0, uint64_t dim1, uint64_t ld_elems,
                      uint32_t box0, uint32_t box1, int swizzle_bytes) {
  std::call_once(g_once, lookup);
  if (!g_encode) return 3;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0 || (ld_elems * 2) % 16 != 0) return 2;
  cuuint64_t dims[2] = {dim0, dim1};
  cuuint64_t strides[1] = {ld_elems * 2};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t estr[2] = {1, 1};
  if (swizzle_bytes != 128 && swizzle_bytes != 64) return 2;
  CUresult r = g_encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : 2;
}

// Four-dimensional view of bf16 data: element (i0, i1, i2, i3) at byte
// offset 2*i0 + i1*stride1 + i2*stride2 + i3*stride3 (strides in bytes, any
// order, multiples of 16); the box is box[0..3] elements with box[0]*2 == 128.
int make_tmap_bf16_4d(void* map, const void* ptr, const uint64_t* dims, const uint64_t* strides_bytes,
                      const uint32_t* box) {
  std::call_once(g_once, lookup);
  if (!g_encode) return 3;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0) return 2;
  cuuint64_t d[4];
  cuuint64_t st[3];
  cuuint32_t b[4];
  cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < 4; ++i) { d[i] = dims[i]; b[i] = box[i]; }
  for (int i = 0; i < 3; ++i) {
    if (strides_bytes[i] % 16 != 0) return 2;
    st[i] = strides_bytes[i];
  }
  CUresult r = g_encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), d,
                        st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : 2;
}

}  // namespace rnn
