// gemm_tc.cu - bf16 GEMM on the 5th-generation tensor cores (tcgen05), fp32
// accumulation in tensor memory, operands fed by TMA.  Serves the three
// contractions around the recurrence on the bf16 path:
//   input projection  P  = X  * W_ih^T + b    (all timesteps at once; poplibs
//                                              Lstm.cpp calcSequenceWeightedInputs)
//   input gradient    dX = dG * W_ih          (Lstm.cpp backwardStepImpl, hoisted)
//   weight gradients  dW = dG^T * [X | H_prev] (basicLstmParamUpdate /
//                                              basicGruParamUpdate, one long-K GEMM)
//
// Structure: a persistent kernel, one CTA per SM, 128 x BN output tiles
// (BN = 256, or 128 when 256-wide tiles would leave most SMs idle), 64-deep K
// slices in a shared-memory ring (4 x 48 KB or 6 x 32 KB).
//   warp 0       TMA producer (one elected thread)
//   warp 1       TMEM owner and MMA issuer (one elected thread); M=128, N=BN,
//                K=16 per tcgen05.mma, 128-byte swizzled operands
//   warps 2..9   epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//                lanes 32*(w%4) .. +31 = tile rows; warps 2-5 the first half
//                of the tile's columns, warps 6-9 the second), bias /
//                accumulate / cast, global stores with the gate-slot row remap
// Two TMEM accumulators (2 x BN columns) let the epilogue of one tile overlap
// the main loop of the next.  Operands may be K-major (row = M or N index, K
// contiguous) or MN-major (K = row index, M or N contiguous); the descriptor
// major-ness bits select which.
//
// Split K (a long K with too few tiles to fill the GPU, i.e. the weight
// gradients): work item (tile, s) covers K slice s of S and stores its raw
// fp32 partial product to scratch; a second kernel sums the S partials of
// every element in split order (deterministic) and applies the epilogue.
// Every wait is bounded; on timeout the kernel records RNN_TIMEOUT in the
// status word and leaves its loops.
#include <atomic>
#include <cstdlib>

#include "common.cuh"

namespace rnn {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int kMaxSplits = 16;

template <int BN>
struct GemmCfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
};

template <int BN>
struct alignas(1024) GemmSmem {
  uint8_t stage[GemmCfg<BN>::STAGES][GemmCfg<BN>::STAGE_BYTES];
  uint64_t full[GemmCfg<BN>::STAGES];
  uint64_t empty[GemmCfg<BN>::STAGES];
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
  int splits;                 // S >= 1
  float* ws;                  // S > 1: partial products, [S][M][N] fp32
};

__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kmajor, int kstep) {
  // base: 1024-aligned start of a rows x 64 (rows x K) operand tile.
  if (kmajor) return sdesc_sw128(base + kstep * 32, 16, 1024);
  // MN-major: 64-element MN chunks of 64 K-rows (8 KB each).
  return sdesc_sw128(base + kstep * 2048, 8192, 1024);
}

// One rows x 64 operand tile: a single box (K-major, the map's box is
// 64 x rows) or rows/64 boxes of 64 x 64 (MN-major).
template <int ROWS>
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int kmajor,
                                             int row0, int k0) {
  if (kmajor) {
    tma_load_2d(dst, map, bar, k0, row0);
  } else {
#pragma unroll
    for (int c = 0; c < ROWS / 64; ++c) tma_load_2d(dst + 8192 * c, map, bar, row0 + 64 * c, k0);
  }
}

// 32 consecutive columns n0 .. n0+31 of one output row.  bias: added when
// non-null; beta: C's previous value is added (read through L2: another SM may
// have written it during this launch).
__device__ __forceinline__ void store_chunk(const TcGemmParams& p, int64_t row, int n0, const float (&v)[32],
                                            const float* bias, int beta) {
  const bool full = n0 + 32 <= p.N;
  if (p.c_bf16) {
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C) + row * p.ldc + n0;
    if (full && (p.ldc % 8 == 0) && !beta) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        uint4 q;
        uint32_t* w = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a0 = v[j + 2 * e], a1 = v[j + 2 * e + 1];
          if (bias) { a0 += bias[n0 + j + 2 * e]; a1 += bias[n0 + j + 2 * e + 1]; }
          __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
          w[e] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(C + j) = q;
      }
    } else {
      for (int j = 0; j < 32 && n0 + j < p.N; ++j) {
        float a = v[j];
        if (bias) a += bias[n0 + j];
        if (beta) a += __bfloat162float(__ldcg(C + j));
        C[j] = __float2bfloat16_rn(a);
      }
    }
  } else {
    float* C = static_cast<float*>(p.C) + row * p.ldc + n0;
    if (full && (p.ldc % 4 == 0)) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float4 q = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        if (bias) { q.x += bias[n0 + j]; q.y += bias[n0 + j + 1]; q.z += bias[n0 + j + 2]; q.w += bias[n0 + j + 3]; }
        if (beta) {
          const float4 o = __ldcg(reinterpret_cast<const float4*>(C + j));
          q.x += o.x; q.y += o.y; q.z += o.z; q.w += o.w;
        }
        *reinterpret_cast<float4*>(C + j) = q;
      }
    } else {
      for (int j = 0; j < 32 && n0 + j < p.N; ++j) {
        float a = v[j];
        if (bias) a += bias[n0 + j];
        if (beta) a += __ldcg(C + j);
        C[j] = a;
      }
    }
  }
}

// Raw fp32 partial product: 32 consecutive columns n0.. of row m of split s.
__device__ __forceinline__ void store_partial(const TcGemmParams& p, int s, int m, int n0, const float (&v)[32]) {
  float* W = p.ws + (static_cast<int64_t>(s) * p.M + m) * p.N + n0;
  if (n0 + 32 <= p.N && p.N % 4 == 0) {
#pragma unroll
    for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(W + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  } else {
    for (int j = 0; j < 32 && n0 + j < p.N; ++j) W[j] = v[j];
  }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcGemmParams p) {
  using Cfg = GemmCfg<BN>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  GemmSmem<BN>& sm = *reinterpret_cast<GemmSmem<BN>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (p.M + BM - 1) / BM, nt = (p.N + BN - 1) / BN;
  const int ntiles = mt * nt;
  const int nitems = ntiles * p.splits;
  const int nk = (p.K + BK - 1) / BK;
  // K blocks [kb_lo(s), kb_lo(s + 1)) belong to split s
  auto kb_lo = [&](int s) { return static_cast<int>((static_cast<int64_t>(nk) * s) / p.splits); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&sm.tfull[b], 1); mbar_init(&sm.tempty[b], kEpiWarps); }
    sm.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, Cfg::TMEM_COLS);
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
      for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
        const int tile = item % ntiles, sp = item / ntiles;
        const int m0 = (tile / nt) * BM, n0 = (tile % nt) * BN;
        for (int kb = kb_lo(sp); kb < kb_lo(sp + 1); ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&sm.empty[s], ph ^ 1, p.timeout_ns) || *(volatile int*)&sm.abort_flag) {
            report_status(p.dev, 4u, K_GEMM_TC, it, W_TMA);
            sm.abort_flag = 1;
            goto producer_done;
          }
          mbar_arrive_expect_tx(&sm.full[s], Cfg::STAGE_BYTES);
          load_operand<BM>(sm.stage[s], &tmA, &sm.full[s], p.a_kmajor, m0, kb * BK);
          load_operand<BN>(sm.stage[s] + A_BYTES, &tmB, &sm.full[s], p.b_kmajor, n0, kb * BK);
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, acc = 0;
      for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++acc) {
        const int sp = item / ntiles;
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
        const int k0 = kb_lo(sp), k1 = kb_lo(sp + 1);
        for (int kb = k0; kb < k1; ++kb, ++it) {
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
                        (kb > k0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&sm.empty[s]);
        }
        if (!ok) break;
        mma_commit(&sm.tfull[buf]);
      }
    }
  } else {
    const int q = warp & 3;              // TMEM lane quarter of this warp
    const int c_lo = (warp - 2) / 4 * (BN / 2), c_hi = c_lo + BN / 2;   // its half of the columns
    uint32_t acc = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++acc) {
      const int tile = item % ntiles, sp = item / ntiles;
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
      if (write && p.splits == 1 && p.rowmap_H > 0) {
        const int pm = p.perm[m & 3];
        if (pm < 0) write = false;
        row = static_cast<int64_t>(pm) * p.rowmap_H + (m >> 2);
      }
      for (int c = c_lo; c < c_hi; c += 32) {
        float v[32];
        tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + c, v);
        if (write && n0 + c < p.N) {
          if (p.splits > 1) store_partial(p, sp, m, n0 + c, v);
          else store_chunk(p, row, n0 + c, v, p.bias, p.beta);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

template <int BN>
constexpr size_t smem_bytes() { return sizeof(GemmSmem<BN>) + 1024; }

// C[row(m), n] = sum over s in order of ws[s][m][n] (+ bias[n]) (+ C if beta),
// four consecutive columns per thread.
__global__ void __launch_bounds__(256)
gemm_split_reduce_kernel(const float* __restrict__ ws, int S, int M, int N, TcGemmParams p) {
  const int nq = (N + 3) / 4;
  const int64_t total = static_cast<int64_t>(M) * nq;
  const int64_t plane = static_cast<int64_t>(M) * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(i / nq), n0 = static_cast<int>(i % nq) * 4;
    int64_t row = m;
    if (p.rowmap_H > 0) {
      const int pm = p.perm[m & 3];
      if (pm < 0) continue;
      row = static_cast<int64_t>(pm) * p.rowmap_H + (m >> 2);
    }
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    const float* w = ws + static_cast<int64_t>(m) * N + n0;
    if (n0 + 4 <= N && N % 4 == 0) {
      for (int s = 0; s < S; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(w + s * plane);
        a[0] += v.x; a[1] += v.y; a[2] += v.z; a[3] += v.w;
      }
    } else {
      for (int s = 0; s < S; ++s)
        for (int j = 0; j < 4 && n0 + j < N; ++j) a[j] += w[s * plane + j];
    }
    for (int j = 0; j < 4 && n0 + j < N; ++j) {
      float x = a[j];
      if (p.bias) x += p.bias[n0 + j];
      if (p.c_bf16) {
        __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C) + row * p.ldc + n0 + j;
        if (p.beta) x += __bfloat162float(*C);
        *C = __float2bfloat16_rn(x);
      } else {
        float* C = static_cast<float*>(p.C) + row * p.ldc + n0 + j;
        if (p.beta) x += *C;
        *C = x;
      }
    }
  }
}

struct GemmPlan { int BN, S; };

// Tile width and K split.  Items run in waves of num_sms.  128 x 256 tiles
// unless they would leave most SMs idle; then a long K is split when the
// scratch allows and that saves at least a sixth of the waves per unit of
// work, and otherwise 128-wide tiles double the tile count.
GemmPlan plan_gemm(const GemmArgs& g, int num_sms) {
  const int mt = (g.M + BM - 1) / BM;
  const int t256 = mt * ((g.N + 255) / 256), t128 = mt * ((g.N + 127) / 128);
  const int nk = (g.K + BK - 1) / BK;
  if (t256 >= num_sms) return {256, 1};
  const size_t plane = static_cast<size_t>(g.M) * g.N * 4;
  if (g.split_ws && nk >= 32) {
    int best = 1;
    double best_cost = 1.0;
    for (int S = 2; S <= kMaxSplits && nk / S >= 16 && S * plane <= g.split_ws_bytes; ++S) {
      const double cost = static_cast<double>((t256 * S + num_sms - 1) / num_sms) / S;
      if (cost < best_cost - 1e-9) { best_cost = cost; best = S; }
    }
    if (best > 1 && best_cost <= 5.0 / 6.0) return {256, best};
  }
  if (2 * t256 < num_sms && t128 > t256) return {128, 1};
  return {256, 1};
}

template <int BN>
int launch_bn(const GemmArgs& g, int S, cudaStream_t s, int num_sms, DevArea* dev, uint64_t timeout_ns) {
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
  p.splits = S;
  p.ws = static_cast<float*>(g.split_ws);
  // the shared-memory limit is a per-device attribute: set it once on each
  // device this instantiation launches on (any thread may get here first)
  static std::atomic<uint64_t> attr_set{0};
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return 3;
  const uint64_t bit = cur < 64 ? (1ull << cur) : 0ull;
  if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<BN>())) != cudaSuccess)
      return 3;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  const int items = ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN) * S;
  const int grid = items < num_sms ? items : num_sms;
  gemm_tc_kernel<BN><<<grid, kThreads, smem_bytes<BN>(), s>>>(ta, tb, p);
  if (cudaGetLastError() != cudaSuccess) return 3;
  if (S > 1) {
    gemm_split_reduce_kernel<<<4 * num_sms, 256, 0, s>>>(p.ws, S, g.M, g.N, p);
    if (cudaGetLastError() != cudaSuccess) return 3;
  }
  return 0;
}

}  // namespace

bool gemm_tc_supported(const GemmArgs& g) {
  if (!g.in_bf16 || g.K <= 0 || g.M <= 0 || g.N <= 0) return false;
  if ((reinterpret_cast<uintptr_t>(g.A) & 15) || (reinterpret_cast<uintptr_t>(g.B) & 15)) return false;
  if ((g.lda * 2) % 16 || (g.ldb * 2) % 16) return false;
  return true;
}

int launch_gemm_tc(const GemmArgs& g, cudaStream_t s, int num_sms, DevArea* dev, uint64_t timeout_ns,
                   int* launches) {
  if (!gemm_tc_supported(g)) return 2;
  GemmPlan pl = plan_gemm(g, num_sms);
  // test hook: a forced tile width (no K split)
  const int bn = plan_overrides().gemm_bn;
  if (bn == 128 || bn == 256) pl = {bn, 1};
  if (launches) *launches = pl.S > 1 ? 2 : 1;
  return pl.BN == 256 ? launch_bn<256>(g, pl.S, s, num_sms, dev, timeout_ns)
                      : launch_bn<128>(g, pl.S, s, num_sms, dev, timeout_ns);
}

}  // namespace rnn
