// gemm_tc.cu - bf16 GEMM on the 5th-generation tensor cores (tcgen05), fp32
// accumulation in tensor memory, operands fed by TMA.  Serves the three
// contractions around the recurrence on the bf16 path:
//   input projection  P  = X  * W_ih^T + b    (all timesteps at once; poplibs
//                                              Lstm.cpp calcSequenceWeightedInputs)
//   input gradient    dX = dG * W_ih          (Lstm.cpp backwardStepImpl, hoisted)
//   weight gradients  dW = dG^T * [X | H_prev] (basicLstmParamUpdate /
//                                              basicGruParamUpdate, one long-K GEMM)
//
// Structure: a persistent kernel, one CTA per SM, 128 x 128 output tiles,
// 64-deep K slices in a 4-stage shared-memory ring.
//   warp 0       TMA producer (one elected thread)
//   warp 1       TMEM owner and MMA issuer (one elected thread); M=128, N=128,
//                K=16 per tcgen05.mma, 128-byte swizzled operands
//   warps 2..5   epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//                lanes 32*(w%4) .. +31 = tile rows), bias / accumulate / cast,
//                global stores with the gate-slot row remap
// Two TMEM accumulators (2 x 128 columns) let the epilogue of one tile overlap
// the main loop of the next.  Operands may be K-major (row = M or N index, K
// contiguous) or MN-major (K = row index, M or N contiguous); the descriptor
// major-ness bits select which.  Every wait is bounded; on timeout the kernel
// records RNN_TIMEOUT in the status word and leaves its loops.
#include "common.cuh"

namespace rnn {

namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;

struct alignas(1024) GemmSmem {
  uint8_t stage[STAGES][STAGE_BYTES];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_base;
  int abort_flag;
};

struct TcGemmParams {
  int M, N, K;
  int a_kmajor, b_kmajor;
  void* C; int64_t ldc; int c_bf16;
  const float* bias;
  int beta;
  int rowmap_H;
  int perm[4];
  DevArea* dev;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kmajor, int kstep) {
  // base: 1024-aligned start of a 128 x 64 (rows x K) operand tile.
  if (kmajor) return sdesc_sw128(base + kstep * 32, 16, 1024);
  // MN-major: two 64-element MN chunks of 64 K-rows (8 KB each).
  return sdesc_sw128(base + kstep * 2048, 8192, 1024);
}

__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int kmajor,
                                             int row0, int k0) {
  if (kmajor) {
    tma_load_2d(dst, map, bar, k0, row0);
  } else {
    tma_load_2d(dst, map, bar, row0, k0);
    tma_load_2d(dst + 8192, map, bar, row0 + 64, k0);
  }
}

__device__ __forceinline__ void store_chunk(const TcGemmParams& p, int64_t row, int n0, const float (&v)[32]) {
  // 32 consecutive columns n0 .. n0+31 of one output row.
  const bool full = n0 + 32 <= p.N;
  if (p.c_bf16) {
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C) + row * p.ldc + n0;
    if (full && (p.ldc % 8 == 0) && !p.beta) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        uint4 q;
        uint32_t* w = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a0 = v[j + 2 * e], a1 = v[j + 2 * e + 1];
          if (p.bias) { a0 += p.bias[n0 + j + 2 * e]; a1 += p.bias[n0 + j + 2 * e + 1]; }
          __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
          w[e] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(C + j) = q;
      }
    } else {
      for (int j = 0; j < 32 && n0 + j < p.N; ++j) {
        float a = v[j];
        if (p.bias) a += p.bias[n0 + j];
        if (p.beta) a += __bfloat162float(C[j]);
        C[j] = __float2bfloat16_rn(a);
      }
    }
  } else {
    float* C = static_cast<float*>(p.C) + row * p.ldc + n0;
    if (full && (p.ldc % 4 == 0)) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float4 q = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        if (p.bias) { q.x += p.bias[n0 + j]; q.y += p.bias[n0 + j + 1]; q.z += p.bias[n0 + j + 2]; q.w += p.bias[n0 + j + 3]; }
        if (p.beta) {
          const float4 o = *reinterpret_cast<const float4*>(C + j);
          q.x += o.x; q.y += o.y; q.z += o.z; q.w += o.w;
        }
        *reinterpret_cast<float4*>(C + j) = q;
      }
    } else {
      for (int j = 0; j < 32 && n0 + j < p.N; ++j) {
        float a = v[j];
        if (p.bias) a += p.bias[n0 + j];
        if (p.beta) a += C[j];
        C[j] = a;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcGemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (p.M + BM - 1) / BM, nt = (p.N + BN - 1) / BN;
  const int ntiles = mt * nt;
  const int nk = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&sm.tfull[b], 1); mbar_init(&sm.tempty[b], 4); }
    sm.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t idesc = idesc_bf16(BM, BN, !p.a_kmajor, !p.b_kmajor);

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int m0 = (tile / nt) * BM, n0 = (tile % nt) * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&sm.empty[s], ph ^ 1, p.timeout_ns) || *(volatile int*)&sm.abort_flag) {
            report_status(p.dev, 4u, K_GEMM_TC, it, W_TMA);
            sm.abort_flag = 1;
            goto producer_done;
          }
          mbar_arrive_expect_tx(&sm.full[s], STAGE_BYTES);
          load_operand(sm.stage[s], &tmA, &sm.full[s], p.a_kmajor, m0, kb * BK);
          load_operand(sm.stage[s] + A_BYTES, &tmB, &sm.full[s], p.b_kmajor, n0, kb * BK);
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, acc = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++acc) {
        const int buf = acc & 1;
        const uint32_t aph = (acc >> 1) & 1;
        if (!mbar_wait(&sm.tempty[buf], aph ^ 1, p.timeout_ns) || *(volatile int*)&sm.abort_flag) {
          report_status(p.dev, 4u, K_GEMM_TC, acc, W_MMA);
          sm.abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem + buf * BN;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&sm.full[s], ph, p.timeout_ns) || *(volatile int*)&sm.abort_flag) {
            report_status(p.dev, 4u, K_GEMM_TC, it, W_TMA);
            sm.abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t abase = smem_u32(sm.stage[s]);
          const uint32_t bbase = abase + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            mma_bf16_ss(dt, operand_desc(abase, p.a_kmajor, k), operand_desc(bbase, p.b_kmajor, k), idesc,
                        (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&sm.empty[s]);
        }
        if (!ok) break;
        mma_commit(&sm.tfull[buf]);
      }
    }
  } else {
    const int q = warp & 3;              // TMEM lane quarter of this warp
    uint32_t acc = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++acc) {
      const int buf = acc & 1;
      const uint32_t aph = (acc >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&sm.tfull[buf], aph, p.timeout_ns) && !*(volatile int*)&sm.abort_flag;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) { report_status(p.dev, 4u, K_GEMM_TC, acc, W_MMA); sm.abort_flag = 1; }
        break;
      }
      tc_fence_after();
      const int m0 = (tile / nt) * BM, n0 = (tile % nt) * BN;
      const int m = m0 + q * 32 + lane;
      int64_t row = m;
      bool write = m < p.M;
      if (write && p.rowmap_H > 0) {
        const int pm = p.perm[m & 3];
        if (pm < 0) write = false;
        row = static_cast<int64_t>(pm) * p.rowmap_H + (m >> 2);
      }
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + c, v);
        if (write && n0 + c < p.N) store_chunk(p, row, n0 + c, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

constexpr size_t kSmemBytes = sizeof(GemmSmem) + 1024;

}  // namespace

bool gemm_tc_supported(const GemmArgs& g) {
  if (!g.in_bf16 || g.K <= 0 || g.M <= 0 || g.N <= 0) return false;
  if ((reinterpret_cast<uintptr_t>(g.A) & 15) || (reinterpret_cast<uintptr_t>(g.B) & 15)) return false;
  if ((g.lda * 2) % 16 || (g.ldb * 2) % 16) return false;
  return true;
}

int launch_gemm_tc(const GemmArgs& g, cudaStream_t s, int num_sms, DevArea* dev, uint64_t timeout_ns) {
  if (!gemm_tc_supported(g)) return 2;
  CUtensorMap ta, tb;
  int rc;
  // A: rows = M; B: rows = N.
  if (g.a_kmajor) rc = make_tmap_bf16_2d(&ta, g.A, g.K, g.M, g.lda, 64, BM);
  else rc = make_tmap_bf16_2d(&ta, g.A, g.M, g.K, g.lda, 64, BK);
  if (rc) return rc;
  if (g.b_kmajor) rc = make_tmap_bf16_2d(&tb, g.B, g.K, g.N, g.ldb, 64, BN);
  else rc = make_tmap_bf16_2d(&tb, g.B, g.N, g.K, g.ldb, 64, BK);
  if (rc) return rc;
  TcGemmParams p;
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.a_kmajor = g.a_kmajor; p.b_kmajor = g.b_kmajor;
  p.C = g.C; p.ldc = g.ldc; p.c_bf16 = g.c_bf16;
  p.bias = g.bias; p.beta = g.beta; p.rowmap_H = g.rowmap_H;
  for (int i = 0; i < 4; ++i) p.perm[i] = g.perm[i];
  p.dev = dev;
  p.timeout_ns = timeout_ns;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
      return 3;
    attr_set = true;
  }
  const int tiles = ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  gemm_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(ta, tb, p);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace rnn
