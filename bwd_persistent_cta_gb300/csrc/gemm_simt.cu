// gemm_simt.cu - fp32-FMA GEMM for the fp32 path (where a 1e-5 bound rules
// out tensor-core TF32) and for operands whose layout the TMA-fed tensor-core
// GEMM cannot take.  64x64 output tile, 16-deep K slices staged in shared
// memory, 256 threads with a 4x4 register tile each.  The same epilogue as the
// tensor-core GEMM: column bias, optional accumulate into C, fp32 or bf16
// output, and the gate-slot row remap used to write weight gradients straight
// into the caller's gate order.
#include "common.cuh"

namespace rnn {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <typename T>
__device__ __forceinline__ float ld_op(const T* p, int64_t i) { return to_f<T>(p[i]); }

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B);
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int tid = threadIdx.x;
  const int tr = tid / 16, tc = tid % 16;   // 16 x 16 threads, 4x4 each
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int k0 = 0; k0 < g.K; k0 += TK) {
    // 64 x 16 elements per operand, 4 per thread
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + e * 256;
      int mm, kk;
      if (g.a_kmajor) { mm = idx / TK; kk = idx % TK; } else { kk = idx / TM; mm = idx % TM; }
      const int m = m0 + mm, k = k0 + kk;
      float v = 0.0f;
      if (m < g.M && k < g.K)
        v = ld_op(A, g.a_kmajor ? static_cast<int64_t>(m) * g.lda + k : static_cast<int64_t>(k) * g.lda + m);
      As[kk][mm] = v;
      int nn;
      if (g.b_kmajor) { nn = idx / TK; kk = idx % TK; } else { kk = idx / TN; nn = idx % TN; }
      const int n = n0 + nn, k2 = k0 + kk;
      float w = 0.0f;
      if (n < g.N && k2 < g.K)
        w = ld_op(B, g.b_kmajor ? static_cast<int64_t>(n) * g.ldb + k2 : static_cast<int64_t>(k2) * g.ldb + n);
      Bs[kk][nn] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tr * 4 + i;
    if (m >= g.M) continue;
    int64_t row = m;
    if (g.rowmap_H > 0) {
      const int p = g.perm[m & 3];
      if (p < 0) continue;
      row = static_cast<int64_t>(p) * g.rowmap_H + (m >> 2);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tc * 4 + j;
      if (n >= g.N) continue;
      float v = acc[i][j];
      if (g.bias) v += g.bias[n];
      const int64_t o = row * g.ldc + n;
      if (g.c_bf16) {
        __nv_bfloat16* C = static_cast<__nv_bfloat16*>(g.C);
        if (g.beta) v += __bfloat162float(C[o]);
        C[o] = __float2bfloat16_rn(v);
      } else {
        float* C = static_cast<float*>(g.C);
        if (g.beta) v += C[o];
        C[o] = v;
      }
    }
  }
}

}  // namespace

int launch_gemm_simt(const GemmArgs& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return 0;
  dim3 grid((g.N + TN - 1) / TN, (g.M + TM - 1) / TM);
  if (grid.y > 65535) return 2;
  if (g.in_bf16)
    gemm_simt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(g);
  else
    gemm_simt_kernel<float><<<grid, 256, 0, s>>>(g);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace rnn
