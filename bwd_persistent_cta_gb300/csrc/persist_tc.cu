// persist_tc.cu - persistent recurrent kernels on the tcgen05 tensor cores
// (bf16 operands, fp32 accumulation in tensor memory), forward and backward
// through time, for LSTM and GRU resetAfter.
//
// Work split.  The per-step recurrent contraction is swapped so that the
// weights are the M=128 operand and the batch is N:
//   forward   S^T[4H, B]  = W_hh[4H, H] . h_{t-1}^T[H, B]
//   backward  dh^T[H, B]  = W_hh^T[H, 4H] . dG^T_{t+1}[4H, B]
// A cluster of KS CTAs owns one 128-row block of the weight operand; CTA rank
// ks owns the K slice [ks*K/KS, (ks+1)*K/KS) and keeps that 128 x K/KS bf16
// tile resident in shared memory (loaded once by TMA) for the whole sequence.
// Each step a CTA
//   1. waits (bounded) on its direction's gpu-scope step counter until every
//      CTA of the direction finished the previous step (acquire);
//   2. streams its K slice of the previous state (h_{t-1} rows of the layer
//      output, or the gate gradients of the step after) with TMA through a
//      ring of 64-column sub-tiles, issuing tcgen05.mma (M=128, N=B rounded up
//      to 16, K=16) into a TMEM accumulator as sub-tiles land;
//   3. moves the accumulator to shared memory (tcgen05.ld), and after a
//      cluster barrier sums the KS partial tiles of its own units over
//      distributed shared memory;
//   4. applies the cell (forward) or its derivative (backward) in registers -
//      the LSTM cell state, the GRU state and the backward carries never leave
//      registers - and writes its units' outputs;
//   5. arrives on the counter (release).
// Cluster-uniform abort: a CTA whose wait ran out publishes a flag in shared
// memory before the cluster barrier; every CTA reads all flags of its cluster
// after it, so all of them leave together (after one more cluster barrier, so
// no CTA exits while a peer may still read its shared memory).
//
// This is the persistent-RNN design of the persistent backward-data kernel
// fragment (one launch for all steps, weights resident on chip, a per-step
// exchange between CTAs through global memory) carried to tensor cores, TMA,
// TMEM and thread-block clusters; flag counters with acquire/release replace
// its -0.0 sentinel polling.  Cell math: Lstm.cpp
// lstmCellForwardPassCalcUnits / backwardStepImpl; Gru.cpp
// gruCellForwardPassCalcUnitsResetAfter / backwardStepImplResetAfter.
#include "common.cuh"

namespace rnn {

namespace {

constexpr int kThreads = 128;
constexpr int kSubK = 64;                 // K columns per TMA sub-tile (128 bytes)
constexpr int kWSub = 128 * kSubK * 2;    // bytes of one 128 x 64 weight sub-tile
constexpr size_t kSmemCap = 227 * 1024;
constexpr size_t kMinSmem = 80 * 1024;

struct TcPersistParams {
  PersistArgs a;
  int KS, Kc, nsub, R, Npad, UPC;
  unsigned int nblk_dir;   // CTAs per direction
  uint32_t tmem_cols;
  uint32_t off_ring, off_part, off_bar;
};

struct TcBars {
  uint64_t wbar;
  uint64_t mma;
  uint64_t full[16];
  uint64_t empty[16];
  int abort_flag[2];
  uint32_t tmem;
};

__device__ __forceinline__ size_t align1k(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

// One step's contraction: stream nsub sub-tiles of the exchange operand
// through the ring and accumulate into TMEM.  Called by thread 0 only.
// g: running sub-tile load counter (across steps).  Returns false on timeout.
__device__ bool contract_step(const TcPersistParams& P, const CUtensorMap* tmX, uint8_t* wsm, uint8_t* ring,
                              TcBars& bars, uint32_t tmem, uint32_t& g, int x0, int y0, uint32_t idesc,
                              uint32_t step_parity, bool first_use_w) {
  const int nsub = P.nsub, R = P.R;
  const uint32_t rbytes = static_cast<uint32_t>(P.Npad) * 128;
  const uint64_t to = P.a.timeout_ns;
  const uint32_t g0 = g;
  // prologue: first min(R, nsub) loads
  for (int j = 0; j < nsub && j < R; ++j) {
    const uint32_t gg = g0 + j;
    const int slot = gg % R;
    if (gg >= static_cast<uint32_t>(R)) {
      if (!mbar_wait(&bars.empty[slot], ((gg / R) - 1) & 1, to)) return false;
    }
    mbar_arrive_expect_tx(&bars.full[slot], rbytes);
    tma_load_2d(ring + slot * rbytes, tmX, &bars.full[slot], x0 + j * kSubK, y0);
  }
  if (first_use_w) {
    if (!mbar_wait(&bars.wbar, 0, to)) return false;
  }
  for (int j = 0; j < nsub; ++j) {
    const uint32_t gg = g0 + j;
    const int slot = gg % R;
    if (!mbar_wait(&bars.full[slot], (gg / R) & 1, to)) return false;
    tc_fence_after();
    const uint32_t abase = smem_u32(wsm + j * kWSub);
    const uint32_t bbase = smem_u32(ring + slot * rbytes);
#pragma unroll
    for (int k = 0; k < kSubK / 16; ++k) {
      mma_bf16_ss(tmem, sdesc_sw128(abase + k * 32, 16, 1024), sdesc_sw128(bbase + k * 32, 16, 1024), idesc,
                  (j > 0 || k > 0) ? 1u : 0u);
    }
    mma_commit(&bars.empty[slot]);
    const int jn = j + R;
    if (jn < nsub) {
      const uint32_t gn = g0 + jn;
      if (!mbar_wait(&bars.empty[slot], ((gn / R) - 1) & 1, to)) return false;
      mbar_arrive_expect_tx(&bars.full[slot], rbytes);
      tma_load_2d(ring + slot * rbytes, tmX, &bars.full[slot], x0 + jn * kSubK, y0);
    }
  }
  mma_commit(&bars.mma);
  g = g0 + nsub;
  (void)step_parity;
  return true;
}

// TMEM accumulator (128 lanes x Npad columns) -> part[b][row] (fp32).
__device__ __forceinline__ void tmem_to_part(uint32_t tmem, float* part, int Npad) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = warp * 32 + lane;
  for (int c = 0; c < Npad; c += 32) {
    float v[32];
    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c + j < Npad) part[(c + j) * 128 + row] = v[j];
  }
}

// Common per-step front half: wait, contract, stage partials, agree on abort.
// Returns true when the whole cluster may continue.
__device__ bool step_front(const TcPersistParams& P, const CUtensorMap* tmX, uint8_t* wsm, uint8_t* ring,
                           float* part, TcBars& bars, uint32_t tmem, uint32_t& g, int x0, int y0,
                           uint32_t idesc, bool do_contract, unsigned int wait_target, int s, int& n_mma,
                           bool& w_waited, unsigned int kernel) {
  const PersistArgs& a = P.a;
  const int dir = a.dir0 + blockIdx.y;
  unsigned int* ctr = &a.dev->counters[dir];
  int ok = 1;
  if (threadIdx.x == 0) {
    if (wait_target > 0 && !wait_counter_geq(ctr, wait_target, a.timeout_ns)) {
      ok = 0;
      report_status(a.dev, 4u, kernel, static_cast<unsigned>(s), W_COUNTER);
    }
    if (ok && do_contract) {
      fence_proxy_async_global();
      if (!contract_step(P, tmX, wsm, ring, bars, tmem, g, x0, y0, idesc, 0, !w_waited)) {
        ok = 0;
        report_status(a.dev, 4u, kernel, static_cast<unsigned>(s), W_TMA);
      }
      w_waited = true;
    }
  }
  ok = __syncthreads_and(ok);
  if (ok && do_contract) {
    const bool done = mbar_wait(&bars.mma, n_mma & 1, a.timeout_ns);
    ++n_mma;
    if (!done) report_status(a.dev, 4u, kernel, static_cast<unsigned>(s), W_MMA);
    ok = __syncthreads_and(done ? 1 : 0);
    if (ok) {
      tc_fence_after();
      tmem_to_part(tmem, part, P.Npad);
    }
  }
  if (threadIdx.x == 0) bars.abort_flag[s & 1] = ok ? 0 : 1;
  tc_fence_before();
  if (P.KS > 1) cluster_sync(); else __syncthreads();
  tc_fence_after();
  int any = 0;
  if (P.KS > 1) {
    const uint32_t fa = smem_u32(&bars.abort_flag[s & 1]);
    for (int r = 0; r < P.KS; ++r) any |= static_cast<int>(ld_shared_cluster_u32(mapa_shared(fa, r)));
  } else {
    any = bars.abort_flag[s & 1];
  }
  return any == 0;
}

__device__ __forceinline__ void step_arrive(const PersistArgs& a, bool skip) {
  fence_proxy_async_global();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (!skip) red_release_gpu_add(&a.dev->counters[a.dir0 + blockIdx.y], 1u);
  }
}

__device__ __forceinline__ float4 sum_partials(const TcPersistParams& P, const float* part, int b, int row4) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* p = part + b * 128 + row4;
  if (P.KS == 1) return *reinterpret_cast<const float4*>(p);
  const uint32_t addr = smem_u32(p);
  for (int r = 0; r < P.KS; ++r) {
    const float4 v = ld_shared_cluster_v4(mapa_shared(addr, r));
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  return acc;
}

__device__ __forceinline__ float sum_partial1(const TcPersistParams& P, const float* part, int b, int row) {
  const float* p = part + b * 128 + row;
  if (P.KS == 1) return *p;
  const uint32_t addr = smem_u32(p);
  float acc = 0.f;
  for (int r = 0; r < P.KS; ++r) acc += ld_shared_cluster_f32(mapa_shared(addr, r));
  return acc;
}

__device__ __forceinline__ void setup(const TcPersistParams& P, const CUtensorMap* tmW, uint8_t* wsm, TcBars& bars,
                                      int wx0, int wy0) {
  if (threadIdx.x == 0) {
    mbar_init(&bars.wbar, 1);
    mbar_init(&bars.mma, 1);
    for (int i = 0; i < P.R; ++i) { mbar_init(&bars.full[i], 1); mbar_init(&bars.empty[i], 1); }
    bars.abort_flag[0] = bars.abort_flag[1] = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&bars.wbar, static_cast<uint32_t>(P.nsub) * kWSub);
    for (int j = 0; j < P.nsub; ++j) tma_load_2d(wsm + j * kWSub, tmW, &bars.wbar, wx0 + j * kSubK, wy0);
  }
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(&bars.tmem, P.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ void teardown(const TcPersistParams& P, TcBars& bars) {
  tc_fence_before();
  if (P.KS > 1) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(bars.tmem, P.tmem_cols);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <int PP>
__global__ void __launch_bounds__(kThreads, 1)
persist_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ TcPersistParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* wsm = base;
  uint8_t* ring = base + P.off_ring;
  float* part = reinterpret_cast<float*>(base + P.off_part);
  TcBars& bars = *reinterpret_cast<TcBars*>(base + P.off_bar);
  const PersistArgs& a = P.a;
  const int H = a.H, B = a.B, TT = a.T, D = a.D;
  const int dir = a.dir0 + blockIdx.y;
  const int ks = static_cast<int>(blockIdx.x) % P.KS;
  const int rg = static_cast<int>(blockIdx.x) / P.KS;
  const bool lstm = a.mode == 0;

  setup(P, &tmW, wsm, bars, ks * P.Kc, dir * 4 * H + rg * 128);
  const uint32_t tmem = bars.tmem;
  const uint32_t idesc = idesc_bf16(128, P.Npad, false, false);

  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.Y);
  const __nv_bfloat16* Pm = static_cast<const __nv_bfloat16*>(a.P);
  __nv_bfloat16* G = static_cast<__nv_bfloat16*>(a.gates);
  const int64_t ldY = static_cast<int64_t>(D) * H;
  const int64_t ldP = static_cast<int64_t>(D) * 4 * H;
  const int UPC = P.UPC;
  const int npairs = UPC * B;
  const int ubase = rg * 32 + ks * UPC;     // first hidden unit of this CTA's epilogue
  const int slot_h0 = dir ? TT + 1 : 0;

  float st[PP];
#pragma unroll
  for (int p = 0; p < PP; ++p) {
    st[p] = 0.f;
    const int id = threadIdx.x + p * kThreads;
    if (id >= npairs) continue;
    const int ul = id % UPC, b = id / UPC, u = ubase + ul;
    if (lstm) {
      const __nv_bfloat16* c0 = static_cast<const __nv_bfloat16*>(a.c0);
      st[p] = c0 ? __bfloat162float(c0[(static_cast<int64_t>(dir) * B + b) * H + u]) : 0.f;
      if (a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? TT : 0)) * B + b) * H + u] = st[p];
    } else {
      st[p] = __bfloat162float(Y[(static_cast<int64_t>(slot_h0) * B + b) * ldY + dir * H + u]);
    }
  }

  const bool skip = a.skip_cta == static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);
  uint32_t g = 0;
  int n_mma = 0;
  bool w_waited = false;
  for (int s = 0; s < TT; ++s) {
    const int t = dir ? TT - 1 - s : s;
    const int sp = dir ? t + 2 : t;
    const int so = t + 1;
    const bool ok = step_front(P, &tmX, wsm, ring, part, bars, tmem, g, dir * H + ks * P.Kc, sp * B, idesc, true,
                               static_cast<unsigned int>(s) * P.nblk_dir, s, n_mma, w_waited, K_FWD_TC);
    if (!ok) break;
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      if (id >= npairs) break;
      const int ul = id % UPC, b = id / UPC, u = ubase + ul;
      const float4 acc = sum_partials(P, part, b, 4 * (u - rg * 32));
      float pv[4];
      Vec4<__nv_bfloat16>::load(Pm + (static_cast<int64_t>(t) * B + b) * ldP + dir * 4 * H + 4 * u, pv);
      float gv[4], h;
      if (lstm) {
        const float i = sigm(pv[0] + acc.x);
        const float f = sigm(pv[1] + acc.y);
        const float gg = tanhf(pv[2] + acc.z);
        const float o = sigm(pv[3] + acc.w);
        const float c = f * st[p] + i * gg;
        h = o * tanhf(c);
        st[p] = c;
        gv[0] = i; gv[1] = f; gv[2] = gg; gv[3] = o;
        if (a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? t : t + 1)) * B + b) * H + u] = c;
        if (s == TT - 1 && a.cy)
          static_cast<__nv_bfloat16*>(a.cy)[(static_cast<int64_t>(dir) * B + b) * H + u] = __float2bfloat16_rn(c);
      } else {
        const float* bh = a.bh + dir * 4 * H + 4 * u;
        const float r = sigm(pv[0] + acc.x + bh[0]);
        const float z = sigm(pv[1] + acc.y + bh[1]);
        const float hn = acc.z + bh[2];
        const float n = tanhf(pv[2] + r * hn);
        h = (1.f - z) * n + z * st[p];
        st[p] = h;
        gv[0] = r; gv[1] = z; gv[2] = n; gv[3] = hn;
      }
      Y[(static_cast<int64_t>(so) * B + b) * ldY + dir * H + u] = __float2bfloat16_rn(h);
      if (G) Vec4<__nv_bfloat16>::store(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * 4 * H + 4 * u, gv);
      if (s == TT - 1 && a.hy)
        static_cast<__nv_bfloat16*>(a.hy)[(static_cast<int64_t>(dir) * B + b) * H + u] = __float2bfloat16_rn(h);
    }
    step_arrive(a, skip);
  }
  teardown(P, bars);
}

// ---------------------------------------------------------------------------
// backward through time
// ---------------------------------------------------------------------------
template <int PP>
__global__ void __launch_bounds__(kThreads, 1)
persist_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ TcPersistParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* wsm = base;
  uint8_t* ring = base + P.off_ring;
  float* part = reinterpret_cast<float*>(base + P.off_part);
  TcBars& bars = *reinterpret_cast<TcBars*>(base + P.off_bar);
  const PersistArgs& a = P.a;
  const int H = a.H, B = a.B, TT = a.T, D = a.D;
  const int K4 = 4 * H;
  const int dir = a.dir0 + blockIdx.y;
  const int ks = static_cast<int>(blockIdx.x) % P.KS;
  const int rg = static_cast<int>(blockIdx.x) / P.KS;
  const bool lstm = a.mode == 0;

  setup(P, &tmW, wsm, bars, ks * P.Kc, dir * H + rg * 128);
  const uint32_t tmem = bars.tmem;
  const uint32_t idesc = idesc_bf16(128, P.Npad, false, false);

  const __nv_bfloat16* Y = static_cast<const __nv_bfloat16*>(a.Y);
  const __nv_bfloat16* G = static_cast<const __nv_bfloat16*>(a.gates);
  __nv_bfloat16* dG = static_cast<__nv_bfloat16*>(a.dG);
  const int64_t ldY = static_cast<int64_t>(D) * H;
  const int64_t ldG = static_cast<int64_t>(D) * K4;
  const int UPC = P.UPC;
  const int npairs = UPC * B;
  const int ubase = rg * 128 + ks * UPC;

  float carry[PP], db[PP][4];
#pragma unroll
  for (int p = 0; p < PP; ++p) {
    carry[p] = 0.f;
    db[p][0] = db[p][1] = db[p][2] = db[p][3] = 0.f;
    const int id = threadIdx.x + p * kThreads;
    if (id >= npairs) continue;
    const int ul = id % UPC, b = id / UPC, u = ubase + ul;
    if (lstm && a.dcT)
      carry[p] = __bfloat162float(static_cast<const __nv_bfloat16*>(a.dcT)[(static_cast<int64_t>(dir) * B + b) * H + u]);
  }

  const bool skip = a.skip_cta == static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);
  uint32_t g = 0;
  int n_mma = 0;
  bool w_waited = false;
  bool aborted = false;
  for (int s = 0; s <= TT; ++s) {
    const int tp = dir ? s - 1 : TT - s;     // step processed just before (s >= 1)
    const bool ok = step_front(P, &tmX, wsm, ring, part, bars, tmem, g, dir * K4 + ks * P.Kc, (s > 0 ? tp : 0) * B,
                               idesc, s > 0, static_cast<unsigned int>(s) * P.nblk_dir, s, n_mma, w_waited,
                               K_BWD_TC);
    if (!ok) { aborted = true; break; }
    const int t = dir ? s : TT - 1 - s;
    const int sp = dir ? t + 2 : t;
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      if (id >= npairs) break;
      const int ul = id % UPC, b = id / UPC, u = ubase + ul;
      float dhr;
      if (s == 0) {
        dhr = a.dhT ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.dhT)[(static_cast<int64_t>(dir) * B + b) * H + u])
                    : 0.f;
      } else {
        dhr = sum_partial1(P, part, b, u - rg * 128);
      }
      if (s == TT) {
        const int64_t o = (static_cast<int64_t>(dir) * B + b) * H + u;
        if (a.dh0) static_cast<__nv_bfloat16*>(a.dh0)[o] = __float2bfloat16_rn(lstm ? dhr : dhr + carry[p]);
        if (lstm && a.dc0) static_cast<__nv_bfloat16*>(a.dc0)[o] = __float2bfloat16_rn(carry[p]);
        continue;
      }
      float gv[4];
      Vec4<__nv_bfloat16>::load(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * K4 + 4 * u, gv);
      const float dy = a.dYi[(static_cast<int64_t>(t) * B + b) * ldY + dir * H + u];
      float da[4];
      if (lstm) {
        const float i = gv[0], f = gv[1], gg = gv[2], o = gv[3];
        const float* C = a.C + static_cast<int64_t>(dir) * (TT + 1) * B * H;
        const float c = C[(static_cast<int64_t>(dir ? t : t + 1) * B + b) * H + u];
        const float cp = C[(static_cast<int64_t>(dir ? t + 1 : t) * B + b) * H + u];
        const float dh = dy + dhr;
        const float tc = tanhf(c);
        const float dc = dh * o * (1.f - tc * tc) + carry[p];
        da[0] = dc * gg * i * (1.f - i);
        da[1] = dc * cp * f * (1.f - f);
        da[2] = dc * i * (1.f - gg * gg);
        da[3] = dh * tc * o * (1.f - o);
        carry[p] = dc * f;
      } else {
        const float r = gv[0], z = gv[1], n = gv[2], hn = gv[3];
        const float hp = __bfloat162float(Y[(static_cast<int64_t>(sp) * B + b) * ldY + dir * H + u]);
        const float dh = dy + dhr + carry[p];
        const float dn = dh * (1.f - z) * (1.f - n * n);
        const float dz = dh * (hp - n) * z * (1.f - z);
        const float dr = dn * hn * r * (1.f - r);
        da[0] = dr; da[1] = dz; da[2] = dn; da[3] = dn * r;
        carry[p] = dh * z;
      }
      Vec4<__nv_bfloat16>::store(dG + (static_cast<int64_t>(t) * B + b) * ldG + dir * K4 + 4 * u, da);
#pragma unroll
      for (int q = 0; q < 4; ++q) db[p][q] += da[q];
    }
    if (s < TT) step_arrive(a, skip);
  }

  if (!aborted) {
    // bias gradients: reduce each unit's four sums over the batch (reuses part,
    // after every peer has finished reading it)
    tc_fence_before();
    if (P.KS > 1) cluster_sync(); else __syncthreads();
    float* red = part;
    for (int i = threadIdx.x; i < 4 * UPC; i += kThreads) red[i] = 0.f;
    __syncthreads();
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      if (id >= npairs) break;
      const int ul = id % UPC;
#pragma unroll
      for (int q = 0; q < 4; ++q) atomicAdd(&red[ul * 4 + q], db[p][q]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * UPC; i += kThreads)
      a.db[static_cast<int64_t>(dir) * K4 + 4 * ubase + i] = red[i];
  }
  teardown(P, bars);
}

int pp_for(int pairs) {
  const int need = (pairs + kThreads - 1) / kThreads;
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 8 ? 8 : need <= 16 ? 16 : 0;
}

const void* fwd_fn(int pp) {
  switch (pp) {
    case 1: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<1>);
    case 2: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<2>);
    case 4: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<4>);
    case 8: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<8>);
    default: return reinterpret_cast<const void*>(&persist_fwd_tc_kernel<16>);
  }
}
const void* bwd_fn(int pp) {
  switch (pp) {
    case 1: return reinterpret_cast<const void*>(&persist_bwd_tc_kernel<1>);
    case 2: return reinterpret_cast<const void*>(&persist_bwd_tc_kernel<2>);
    case 4: return reinterpret_cast<const void*>(&persist_bwd_tc_kernel<4>);
    case 8: return reinterpret_cast<const void*>(&persist_bwd_tc_kernel<8>);
    default: return reinterpret_cast<const void*>(&persist_bwd_tc_kernel<16>);
  }
}

struct TcPlan {
  int KS = 0, Kc = 0, nsub = 0, R = 0, Npad = 0, UPC = 0, PP = 0, nrg = 0;
  uint32_t tmem_cols = 0, off_ring = 0, off_part = 0, off_bar = 0;
  size_t smem = 0;
};

size_t a1k(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

// Candidate K splits for one launch, preferred first: the largest split
// whose grid fits (shorter per-CTA contraction, less shared memory per CTA).
// Whether the clusters can all be resident at once is checked at launch.
int make_plans(int bwd, int H, int B, int ndir, int num_sms, TcPlan* out, int max_out) {
  if (B < 1 || B > 256) return 0;
  const int K = bwd ? 4 * H : H;
  const int nrg = bwd ? H / 128 : (4 * H) / 128;
  if (bwd ? (H % 128) : (H % 32)) return 0;
  const int Npad = (B + 15) / 16 * 16;
  int n = 0;
  for (int KS = 8; KS >= 1 && n < max_out; KS /= 2) {
    if (K % (KS * kSubK)) continue;
    const int Kc = K / KS;
    const int nsub = Kc / kSubK;
    const int UPC = (bwd ? 128 : 32) / KS;
    if (UPC < 1) continue;
    const int PP = pp_for(UPC * B);
    if (PP == 0) continue;
    if (nrg * KS * ndir > num_sms) continue;
    const size_t wbytes = static_cast<size_t>(nsub) * kWSub;
    const size_t rb = static_cast<size_t>(Npad) * 128;
    const size_t part = static_cast<size_t>(Npad) * 128 * 4;
    int R = nsub < 16 ? nsub : 16;
    size_t smem = 0;
    for (; R >= 1; --R) {
      smem = a1k(wbytes) + a1k(R * rb) + a1k(part) + a1k(sizeof(TcBars)) + 1024;
      if (smem <= kSmemCap) break;
    }
    if (R < 1 || (R < nsub && R < 2)) continue;
    TcPlan p;
    p.KS = KS; p.Kc = Kc; p.nsub = nsub; p.R = R; p.Npad = Npad; p.UPC = UPC; p.PP = PP; p.nrg = nrg;
    uint32_t tc = 32;
    while (tc < static_cast<uint32_t>(Npad)) tc *= 2;
    p.tmem_cols = tc;
    p.off_ring = static_cast<uint32_t>(a1k(wbytes));
    p.off_part = p.off_ring + static_cast<uint32_t>(a1k(R * rb));
    p.off_bar = p.off_part + static_cast<uint32_t>(a1k(part));
    // at least a third of an SM's shared memory: at most two CTAs per SM, so
    // their tensor-memory allocations (<= 256 columns each) always fit
    p.smem = smem < kMinSmem ? kMinSmem : smem;
    out[n++] = p;
  }
  return n;
}

const void* kernel_for(int bwd, int pp) { return bwd ? bwd_fn(pp) : fwd_fn(pp); }

void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, const TcPlan& pl, int ndir, cudaStream_t s) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(pl.nrg * pl.KS, ndir, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

// First candidate plan whose clusters can all be resident at once.
bool choose_plan(int bwd, int H, int B, int ndir, int num_sms, TcPlan* chosen) {
  TcPlan plans[4];
  const int n = make_plans(bwd, H, B, ndir, num_sms, plans, 4);
  for (int i = 0; i < n; ++i) {
    const TcPlan& pl = plans[i];
    const void* fn = kernel_for(bwd, pl.PP);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(pl.smem)) !=
        cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_config(cfg, attr, pl, ndir, nullptr);
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (max_clusters >= pl.nrg * ndir) {
      *chosen = pl;
      return true;
    }
  }
  return false;
}

int launch(const PersistArgs& a, int bwd, cudaStream_t s, int num_sms) {
  TcPlan pl;
  if (!choose_plan(bwd, a.H, a.B, a.ndir, num_sms, &pl)) return 2;
  const int H = a.H, D = a.D;
  CUtensorMap tmW, tmX;
  int rc;
  if (!bwd) {
    rc = make_tmap_bf16_2d(&tmW, a.Wr, H, static_cast<uint64_t>(D) * 4 * H, H, kSubK, 128);
    if (rc) return rc;
    rc = make_tmap_bf16_2d(&tmX, a.Y, static_cast<uint64_t>(D) * H, static_cast<uint64_t>(a.T + 2) * a.B,
                           static_cast<uint64_t>(D) * H, kSubK, pl.Npad);
  } else {
    rc = make_tmap_bf16_2d(&tmW, a.WrT, 4 * H, static_cast<uint64_t>(D) * H, 4 * H, kSubK, 128);
    if (rc) return rc;
    rc = make_tmap_bf16_2d(&tmX, a.dG, static_cast<uint64_t>(D) * 4 * H, static_cast<uint64_t>(a.T) * a.B,
                           static_cast<uint64_t>(D) * 4 * H, kSubK, pl.Npad);
  }
  if (rc) return rc;
  TcPersistParams P;
  P.a = a;
  P.KS = pl.KS; P.Kc = pl.Kc; P.nsub = pl.nsub; P.R = pl.R; P.Npad = pl.Npad; P.UPC = pl.UPC;
  P.nblk_dir = static_cast<unsigned int>(pl.nrg * pl.KS);
  P.tmem_cols = pl.tmem_cols;
  P.off_ring = pl.off_ring; P.off_part = pl.off_part; P.off_bar = pl.off_bar;
  const void* fn = kernel_for(bwd, pl.PP);
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_config(cfg, attr, pl, a.ndir, s);
  void* params[] = {&tmW, &tmX, &P};
  if (cudaLaunchKernelExC(&cfg, fn, params) != cudaSuccess) return 3;
  return 0;
}

}  // namespace

bool persist_tc_supported(int mode, int reset_after, int H, int B, int ndir, int num_sms) {
  if (!(mode == 0 || (mode == 1 && reset_after))) return false;
  TcPlan f, b;
  return choose_plan(0, H, B, ndir, num_sms, &f) && choose_plan(1, H, B, ndir, num_sms, &b);
}

int launch_persist_fwd_tc(const PersistArgs& a, cudaStream_t s, int num_sms) { return launch(a, 0, s, num_sms); }
int launch_persist_bwd_tc(const PersistArgs& a, cudaStream_t s, int num_sms) { return launch(a, 1, s, num_sms); }

}  // namespace rnn
