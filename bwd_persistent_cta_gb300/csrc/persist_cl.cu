// persist_cl.cu - cluster-resident persistent forward recurrence on the
// tcgen05 tensor cores, for layers whose 4H gate rows fit one thread-block
// cluster (H <= 512: at most 16 CTAs of 128 gate rows), bf16 LSTM / GRU
// resetAfter without sequence lengths or cell clipping.  An opt-in variant
// (environment RNN_CLUSTER_FWD=1) of the K-split kernel in
// persist_tc_kernels.cuh: see launch_persist_fwd_cl for the measurement.
//
// One cluster per direction; CTA m owns the 128 gate rows of hidden units
// [32m, 32m + 32) (all four gate slots) over the whole K = H, its W_hh rows
// resident in tensor memory as the A operand of tcgen05.mma (columns 256..),
// so there is no K split and no partial-sum exchange.  The state h_(t-1) of
// the whole direction sits in shared memory as nm 64-column-wide chunks (one
// per CTA, 64-byte swizzled K-major, double-buffered by step parity).  Per
// step every CTA
//   1. issues the MMAs of each chunk as soon as that chunk's mbarrier shows it
//      arrived (M=128, N=batch rounded up to 16, K=16; two per chunk);
//   2. reads the accumulator (tcgen05.ld) into shared memory as [unit][batch]
//      [4 slots], applies the cell in registers (the cell / GRU state never
//      leaves registers), and stores h_t of its 32 units into the layer
//      output (global memory);
//   3. fences those stores to the async proxy and issues ONE multicast TMA of
//      its 32-unit chunk of h_t (from the layer output, through L2) into the
//      next buffer of every CTA of the cluster, completing on each CTA's
//      mbarrier for that chunk.
// No grid-wide counter: the exchange and its synchronisation are the
// multicast copy and the receivers' mbarriers.  A buffer is rewritten two
// steps after it was read, and a sender reaches that step only after every
// CTA finished reading it (it needs their chunks of the step in between).
// Every wait is bounded; after a timeout the CTA records RNN_TIMEOUT and stops
// exchanging (no more barrier arrivals, MMAs or copies: a chunk that never
// came leaves its barrier phase open), its peers then time out on its missing
// chunks and stop too, and every CTA meets at the final cluster barrier; the
// outputs are invalid.
//
// This is the persistent-RNN design of the persistent backward-data kernel
// fragment (weights resident on chip, one launch for all steps) with the
// cross-CTA exchange moved from a polled global buffer to a cluster-wide
// multicast copy.  Cell math: Lstm.cpp lstmCellForwardPassCalcUnits, Gru.cpp
// gruCellForwardPassCalcUnitsResetAfter; sigmoid / tanh by tanh.approx.f32.
#include <cstdlib>

#include "common.cuh"

namespace rnn {

namespace {

constexpr int kThreadsCl = 256;
constexpr int kMaxChunks = 16;
constexpr uint32_t kWCol = 256;          // first TMEM column of the weight rows
constexpr uint64_t kShortWaitNs = 1000000ull;

struct ClParams {
  PersistArgs a;
  int nm;                 // CTAs per cluster = 4H / 128; CTA m owns units [32m, 32m + 32)
  int Npad;               // batch rounded up to 16 (MMA N)
  uint32_t chunk_bytes;   // Npad * 64: one 32-unit chunk of the state, all batch rows
  uint32_t off_tr, off_bar;
};

struct ClBars {
  uint64_t full[2][kMaxChunks];   // chunk j of buffer b landed (multicast TMA)
  uint64_t mma;                   // this step's MMAs finished
  uint32_t tmem;
};

__device__ __forceinline__ float tanh_fast_cl(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigm_fast_cl(float x) { return fmaf(0.5f, tanh_fast_cl(0.5f * x), 0.5f); }

template <int PP>
__global__ void __launch_bounds__(kThreadsCl, 1)
persist_fwd_cl_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ ClParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const PersistArgs& a = P.a;
  const int H = a.H, B = a.B, TT = a.T, D = a.D;
  const int dir = a.dir0 + blockIdx.y;
  const int m = static_cast<int>(cluster_ctarank());
  const int nm = P.nm, Npad = P.Npad;
  const uint32_t cb = P.chunk_bytes;
  uint8_t* buf = base;                                                   // [2][nm][cb]
  float* tr = reinterpret_cast<float*>(base + P.off_tr);                 // [32][TRS]
  ClBars& bars = *reinterpret_cast<ClBars*>(base + P.off_bar);
  const int TRS = 4 * Npad + 4;                                          // floats per unit row (+16 B pad)
  const bool lstm = a.mode == 0;
  const uint16_t mask = static_cast<uint16_t>((1u << nm) - 1u);
  const int u0 = 32 * m;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool skip = a.skip_cta == static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);

  // ---- setup: barriers, TMEM, the weight rows in TMEM
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i)
      for (int j = 0; j < nm; ++j) mbar_init(&bars.full[i][j], 1);
    mbar_init(&bars.mma, 1);
    fence_mbar_init();
    prefetch_tmap(&tmY);
  }
  if (warp == 0) {
    tmem_alloc(&bars.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem;
  {
    // rows dir*4H + 128m + r of the packed W_hh, K = H: warps w and w + 4 share
    // lane quarter w % 4 and split K into halves of H/4 32-bit columns
    const int q = warp & 3, half = warp >> 2;
    const int ncol = H / 4;
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.Wr) +
                               (static_cast<int64_t>(dir) * 4 * H + 128 * m + q * 32 + lane) * H + half * (H / 2);
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + kWCol + static_cast<uint32_t>(half * ncol);
    for (int c = 0; c < ncol; c += 32) {
      const uint4* p4 = reinterpret_cast<const uint4*>(src + 2 * c);
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = p4[i];
        r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
      }
      tmem_st_32x32b_x32(trow + c, r);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // every CTA's barriers are initialised before any multicast lands

  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.Y);
  const __nv_bfloat16* Pm = static_cast<const __nv_bfloat16*>(a.P);
  __nv_bfloat16* G = static_cast<__nv_bfloat16*>(a.gates);
  const int64_t ldY = static_cast<int64_t>(D) * H;
  const int64_t ldP = static_cast<int64_t>(D) * 4 * H;
  const int npairs = 32 * B;
  const int slot_h0 = dir ? TT + 1 : 0;
  const uint32_t idesc = idesc_bf16(128, Npad, false, false);

  // per pair (unit u0 + id % 32, batch id / 32): LSTM c / GRU h, GRU recurrent biases
  float st[PP];
  float bh[PP][3];
#pragma unroll
  for (int p = 0; p < PP; ++p) {
    st[p] = 0.f;
    bh[p][0] = bh[p][1] = bh[p][2] = 0.f;
    const int id = threadIdx.x + p * kThreadsCl;
    if (id >= npairs) continue;
    const int ul = id & 31, b = id >> 5, u = u0 + ul;
    if (lstm) {
      const __nv_bfloat16* c0 = static_cast<const __nv_bfloat16*>(a.c0);
      st[p] = c0 ? __bfloat162float(c0[(static_cast<int64_t>(dir) * B + b) * H + u]) : 0.f;
      if (a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? TT : 0)) * B + b) * H + u] = st[p];
    } else {
      st[p] = __bfloat162float(Y[(static_cast<int64_t>(slot_h0) * B + b) * ldY + dir * H + u]);
      const float* bb = a.bh + dir * 4 * H + 4 * u;
      bh[p][0] = bb[0]; bh[p][1] = bb[1]; bh[p][2] = bb[2];
    }
  }

  // this CTA's chunk of h0 to every CTA (buffer 0)
  if (threadIdx.x == 0) {
    for (int j = 0; j < nm; ++j) mbar_arrive_expect_tx(&bars.full[0][j], cb);
    if (!skip) tma_load_2d_multicast(buf + m * cb, &tmY, &bars.full[0][m], dir * H + u0, slot_h0 * B, mask);
  }

  bool aborted = false;   // a wait ran out: this CTA stops exchanging (uniform across the CTA)
  int stop_step = 0;
  for (int s = 0; s < TT; ++s) {
    stop_step = s;
    const int t = dir ? TT - 1 - s : s;
    const int so = t + 1;
    const int pb = s & 1;
    // this step's input projections: independent of the exchange
    uint2 pq[PP];
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreadsCl;
      const int ul = id & 31, b = id >> 5, u = u0 + ul;
      pq[p] = id < npairs ? *reinterpret_cast<const uint2*>(Pm + (static_cast<int64_t>(t) * B + b) * ldP + dir * 4 * H + 4 * u)
                          : make_uint2(0, 0);
    }
    int ok = 1;
    if (threadIdx.x == 0) {
      // each chunk barrier gets exactly one arrival per phase: arm the next
      // step's buffer (its previous phase completed a step ago)
      if (s + 1 < TT)
        for (int j = 0; j < nm; ++j) mbar_arrive_expect_tx(&bars.full[pb ^ 1][j], cb);
      const uint8_t* bb = buf + pb * nm * cb;
      for (int j = 0; j < nm; ++j) {
        if (!mbar_wait(&bars.full[pb][j], (s >> 1) & 1, a.timeout_ns)) {
          report_status(a.dev, 4u, K_FWD_CL, static_cast<unsigned>(s), W_PEER);
          ok = 0;
          break;
        }
        tc_fence_after();
        const uint64_t bd = sdesc_sw64(smem_u32(bb + j * cb), 512);
#pragma unroll
        for (int k = 0; k < 2; ++k)
          mma_bf16_ts(tmem, tmem + kWCol + static_cast<uint32_t>(16 * j + 8 * k), bd + 2 * k, idesc,
                      (j > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(&bars.mma);   // also when stopping: the MMAs issued so far finish before TMEM is freed
    }
    if (!__syncthreads_and(ok)) {
      aborted = true;
      break;
    }
    if (!__syncthreads_and(mbar_wait(&bars.mma, s & 1, a.timeout_ns) ? 1 : 0)) {
      if (threadIdx.x == 0) report_status(a.dev, 4u, K_FWD_CL, static_cast<unsigned>(s), W_MMA);
      aborted = true;
      break;
    }
    tc_fence_after();
    {
      // accumulator row r = 4 * unit + slot (lane r), column = batch
      const int q = warp & 3, half = warp >> 2;
      const int r = q * 32 + lane;
      float* dst = tr + (r >> 2) * TRS + (r & 3);
      for (int c = half * 32; c < Npad; c += 64) {
        float v[32];
        tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, v);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c + j < Npad) dst[(c + j) * 4] = v[j];
      }
    }
    tc_fence_before();
    __syncthreads();
    float hv[PP];
    float gq[PP][4];
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreadsCl;
      hv[p] = 0.f;
      if (id >= npairs) break;
      const int ul = id & 31, b = id >> 5, u = u0 + ul;
      const float4 acc = *reinterpret_cast<const float4*>(tr + ul * TRS + 4 * b);
      float pv[4];
      {
        __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&pq[p].x);
        __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162*>(&pq[p].y);
        const float2 fa = __bfloat1622float2(lo), fb = __bfloat1622float2(hi);
        pv[0] = fa.x; pv[1] = fa.y; pv[2] = fb.x; pv[3] = fb.y;
      }
      float h;
      if (lstm) {
        const float i = sigm_fast_cl(pv[0] + acc.x);
        const float f = sigm_fast_cl(pv[1] + acc.y);
        const float gg = tanh_fast_cl(pv[2] + acc.z);
        const float o = sigm_fast_cl(pv[3] + acc.w);
        const float c = f * st[p] + i * gg;
        h = o * tanh_fast_cl(c);
        st[p] = c;
        gq[p][0] = i; gq[p][1] = f; gq[p][2] = gg; gq[p][3] = o;
      } else {
        const float r = sigm_fast_cl(pv[0] + acc.x + bh[p][0]);
        const float z = sigm_fast_cl(pv[1] + acc.y + bh[p][1]);
        const float hn = acc.z + bh[p][2];
        const float n = tanh_fast_cl(pv[2] + r * hn);
        h = (1.f - z) * n + z * st[p];
        st[p] = h;
        gq[p][0] = r; gq[p][1] = z; gq[p][2] = n; gq[p][3] = hn;
      }
      hv[p] = h;
      Y[(static_cast<int64_t>(so) * B + b) * ldY + dir * H + u] = __float2bfloat16_rn(h);
    }
    // h_t of this CTA's units to every CTA: the stores, then one multicast copy
    fence_proxy_async_global();
    __syncthreads();
    if (threadIdx.x == 0 && s + 1 < TT && !skip)
      tma_load_2d_multicast(buf + (pb ^ 1) * nm * cb + m * cb, &tmY, &bars.full[pb ^ 1][m], dir * H + u0, so * B,
                            mask);
    // stores nothing in this launch waits for
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreadsCl;
      if (id >= npairs) break;
      const int ul = id & 31, b = id >> 5, u = u0 + ul;
      if (G) Vec4<__nv_bfloat16>::store(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * 4 * H + 4 * u, gq[p]);
      if (lstm && a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? t : t + 1)) * B + b) * H + u] = st[p];
      if (s == TT - 1) {
        const int64_t o = (static_cast<int64_t>(dir) * B + b) * H + u;
        if (a.hy) static_cast<__nv_bfloat16*>(a.hy)[o] = __float2bfloat16_rn(hv[p]);
        if (lstm && a.cy) static_cast<__nv_bfloat16*>(a.cy)[o] = __float2bfloat16_rn(st[p]);
      }
    }
  }
  if (aborted && threadIdx.x == 0) {
    // the MMAs issued before stopping finish before TMEM is freed (the commit
    // of the step that stopped), and a peer's copy still in flight lands
    // before this CTA leaves
    mbar_wait(&bars.mma, static_cast<uint32_t>(stop_step) & 1u, kShortWaitNs);
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

const void* cl_kernel(int pp) {
  switch (pp) {
    case 1: return reinterpret_cast<const void*>(&persist_fwd_cl_kernel<1>);
    case 2: return reinterpret_cast<const void*>(&persist_fwd_cl_kernel<2>);
    case 4: return reinterpret_cast<const void*>(&persist_fwd_cl_kernel<4>);
    default: return reinterpret_cast<const void*>(&persist_fwd_cl_kernel<8>);
  }
}

}  // namespace

int launch_persist_fwd_cl(const PersistArgs& a, cudaStream_t s, int num_sms) {
  (void)num_sms;
  // opt-in (RNN_CLUSTER_FWD=1): measured slower than the K-split kernel on
  // GRU T128 B64 H512 (0.72 vs 0.57 ms per forward): without a K split each
  // CTA issues H/16 MMAs per step (issue-bound at about 45 ns each) and runs
  // the cell for 4x the pairs, which outweighs the cheaper exchange
  const char* e = std::getenv("RNN_CLUSTER_FWD");
  if (!e || e[0] != '1') return 2;
  if (!a.is_bf16 || !(a.mode == 0 || (a.mode == 1 && a.reset_after)) || a.len || a.clip || a.y_out) return 2;
  const int H = a.H, B = a.B;
  if (H % 128 != 0 || 4 * H / 128 > kMaxChunks || B < 1 || B > 64) return 2;
  const int nm = 4 * H / 128;
  const int Npad = (B + 15) / 16 * 16;
  const int PP = B <= 8 ? 1 : B <= 16 ? 2 : B <= 32 ? 4 : 8;
  const uint32_t cb = static_cast<uint32_t>(Npad) * 64;
  const size_t buf_bytes = 2ull * nm * cb;
  const size_t tr_bytes = 32ull * (4 * Npad + 4) * 4;
  ClParams P;
  P.a = a;
  P.nm = nm;
  P.Npad = Npad;
  P.chunk_bytes = cb;
  P.off_tr = static_cast<uint32_t>((buf_bytes + 1023) / 1024 * 1024);
  P.off_bar = static_cast<uint32_t>((P.off_tr + tr_bytes + 1023) / 1024 * 1024);
  size_t smem = P.off_bar + sizeof(ClBars) + 1024;
  if (smem < 116 * 1024) smem = 116 * 1024;   // one CTA per SM: it holds all 512 TMEM columns
  if (smem > 227 * 1024) return 2;
  const void* fn = cl_kernel(PP);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return 2;
  }
  if (nm > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 2;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(nm, a.ndir, 1);
  cfg.blockDim = dim3(kThreadsCl, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nm;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 2;
  }
  if (max_clusters < a.ndir) return 2;
  CUtensorMap tmY;
  if (make_tmap_bf16_2d(&tmY, a.Y, static_cast<uint64_t>(a.D) * H, static_cast<uint64_t>(a.T + 2) * B,
                        static_cast<uint64_t>(a.D) * H, 32, static_cast<uint32_t>(Npad), 64) != 0)
    return 2;
  void* params[] = {&tmY, &P};
  if (cudaLaunchKernelExC(&cfg, fn, params) != cudaSuccess) return 3;
  return 0;
}

}  // namespace rnn
