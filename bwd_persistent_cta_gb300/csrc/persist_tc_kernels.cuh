// persist_tc_kernels.cuh - persistent recurrent kernels on the tcgen05 tensor cores
// (bf16 operands, fp32 accumulation in tensor memory), forward and backward
// through time, for LSTM, GRU resetAfter and GRU reset-before (the latter in
// the extended variant).
//
// Work split.  The per-step recurrent contraction is swapped so that the
// weights are the M=128 operand and the batch is N:
//   forward   S^T[4H, B]  = W_hh[4H, H] . h_{t-1}^T[H, B]
//   backward  dh^T[H, B]  = W_hh^T[H, 4H] . dG^T_{t+1}[4H, B]
// KS CTAs own one 128-row block of the weight operand and one batch part (NB
// parts of Bp rows split the batch); CTA ks owns the K slice
// [ks*K/KS, (ks+1)*K/KS) and keeps that 128 x K/KS bf16 tile resident for the
// whole sequence - in shared memory (loaded once by TMA), in tensor memory as
// the MMA A operand, or split between the two - and owns the 128/KS rows
// [ks*128/KS, (ks+1)*128/KS) of the result for its batch part.  The KS CTAs
// are one thread-block cluster, or, for a backward whose clusters cannot all
// be resident, a group that exchanges through global memory.
//
// Each step a CTA
//   1. waits (bounded) on the step counter of the K slice it contracts: one
//      gpu-scope counter per (direction, batch part, K slice), advanced by
//      the CTAs whose outputs form that slice (release add / acquire poll);
//   2. brings its K slice of the previous state (h_{t-1} rows of the layer
//      output, or the gate gradients of the step after) into shared memory
//      with TMA (4-D boxes for the whole slice, or a ring of 64-column
//      sub-tiles), issuing tcgen05.mma (M=128, N=B rounded up to 16, K=16)
//      into a TMEM accumulator as the pieces land;
//   3. pushes each accumulator row (tcgen05.ld) into the shared memory of the
//      cluster peer that owns that row (posted distributed shared-memory
//      stores, one receive buffer per exchange parity), together with its
//      abort flag - or, without a cluster, writes them to the group's buffer
//      in global memory and copies its own rows back after the group's
//      counter says every peer has written;
//   4. after one cluster barrier sums the KS partial rows of its own units,
//      applies the cell (forward) or its derivative (backward) in registers -
//      the LSTM cell state, the GRU state and the backward carries never leave
//      registers - stores the exchanged values and arrives on the counter of
//      the slice they form.  The forward stores what no CTA of the launch
//      waits for (gates, c, the caller's y) during the next step's
//      contraction instead.
// Extended variant (template flag EXT, used when sequence lengths or LSTM cell
// clipping are set, and for GRU reset-before; the plain variant compiles
// without them):
//  * variable sequence lengths: at a step t >= len[b] the pair (u, b) keeps
//    its state (h, c) and stores it unchanged, and the backward step writes
//    zero gate gradients and passes the state gradients on (LSTM: an extra
//    register carries dh past such steps);
//  * LSTM cell clipping: every use of the raw cell state goes through
//    clip = min(max(c, lo), hi), and the backward multiplies by dclip;
//  * GRU reset-before: two exchanges per step.  Forward: the second is over
//    r * h_{t-1}, which each CTA stores for its units in between.  Backward:
//    the first contracts [0, 0, dn, 0] (d(rh) = W_hn^T dn), the second the
//    gate gradients [dr, dz, dn, 0].
// Cluster-uniform abort: every CTA reads the same set of flags after the same
// barrier, so all CTAs of a cluster leave at the same step (after one more
// cluster barrier, so no CTA exits while a peer may still touch its shared
// memory); a group without a cluster shares one abort flag in global memory.
//
// This is the persistent-RNN design of the persistent RNN backward-data kernel
// page (one launch for all steps, weights resident on chip, a per-step
// exchange between CTAs through global memory) carried to tensor cores, TMA,
// TMEM and thread-block clusters; that kernel polls its dgates buffer for a
// -0.0 sentinel where a release/acquire counter is used here.  Cell math:
// the popnn Lstm.cpp page's forward cell step and backward step, and the popnn
// Gru.cpp page's resetAfter forward cell step and backward step.  The
// sigmoid and tanh of this bf16 path use the hardware tanh.approx.f32
// instruction (sigma(x) = 1/2 + tanh(x/2)/2); its relative error (about 2^-11)
// is below the bf16 storage rounding of the stored states.
#pragma once

#include <cstdlib>

#include "common.cuh"

namespace rnn {

namespace {

#ifdef RNN_STEP_TRACE
// Step-phase timestamps (globaltimer, ns) of two CTAs, for latency studies;
// compiled only with -DRNN_STEP_TRACE.
__device__ unsigned long long g_step_trace[2][2][1100][16];
#define RNN_TRACE_AT(slot_, kind_, step_)                                                        \
  do {                                                                                          \
    if (threadIdx.x == 0 && (blockIdx.x == 0 || blockIdx.x == gridDim.x - 1) && blockIdx.y == 0 && \
        (step_) < 1100)                                                                          \
      g_step_trace[(kind_)][blockIdx.x == 0 ? 0 : 1][(step_)][(slot_)] = globaltimer_ns();       \
  } while (0)
// the same, recorded by thread tid_ instead of thread 0
#define RNN_TRACE_AT_T(tid_, slot_, kind_, step_)                                                  \
  do {                                                                                          \
    if (threadIdx.x == (tid_) && (blockIdx.x == 0 || blockIdx.x == gridDim.x - 1) && blockIdx.y == 0 && \
        (step_) < 1100)                                                                          \
      g_step_trace[(kind_)][blockIdx.x == 0 ? 0 : 1][(step_)][(slot_)] = globaltimer_ns();       \
  } while (0)
#else
#define RNN_TRACE_AT(slot_, kind_, step_) do { } while (0)
#define RNN_TRACE_AT_T(tid_, slot_, kind_, step_) do { } while (0)
#endif

constexpr int kThreads = 256;             // warps 0-3 read TMEM; all 8 run the cell epilogue
constexpr int kSubK = 64;                 // K columns per 128-byte swizzled sub-tile
constexpr int kWSub = 128 * kSubK * 2;    // bytes of one 128 x 64 weight sub-tile
constexpr int kMaxKS = 16;
constexpr int kMaxRing = 16;
constexpr size_t kSmemCap = 227 * 1024;
constexpr size_t kMinSmem = 80 * 1024;    // at most two CTAs per SM: TMEM (<= 256 cols each) fits
constexpr size_t kOneCtaSmem = 116 * 1024; // one CTA per SM (it holds all 512 TMEM columns)

struct TcPersistParams {
  PersistArgs a;
  int KS, Kc, nsub, R, Npad, UPC, RPC;
  int w_tmem;              // 64-column weight sub-tiles held in tensor memory (the A operand from TMEM):
                           // sub-tiles [0, w_tmem) there, [w_tmem, nsub) in shared memory
  int single;              // the whole K slice arrives with 4-D TMAs issued at the step's start (R == nsub)
  int nchunk;              // single: that many 4-D TMAs of nsub / nchunk sub-tiles, each on its own
                           // mbarrier, so the MMAs start when the first chunk lands
  int prefetch;            // forward: request later steps' projections into L2 (kPrefetchSteps)
  int nrg;                 // 128-row groups per direction
  int NB, Bp;              // batch parts per row group and batch rows per part (Npad = Bp rounded up to 16)
  uint32_t wcol;           // first TMEM column of the weight tile (w_tmem)
  unsigned int nblk_dir;   // CTAs per direction
  uint32_t tmem_cols;
  uint32_t off_ring, off_recv, off_bar;
  uint32_t off_stage;      // forward with a K split: warp 0's post-step stage, 0 = none
  int gk;                  // backward: the K-split partials go through global memory (a.gk_buf), no cluster
  int recv2;               // K split over a cluster: receive buffer (exchange index & 1); else one buffer
};

// Byte offset of exchange e's receive buffer: with a K split over a cluster
// a peer may push exchange e + 1's partials while this CTA still reads e's.
__device__ __forceinline__ uint32_t recv_off(const TcPersistParams& P, int e) {
  return (P.recv2 && (e & 1)) ? static_cast<uint32_t>(P.Npad) * 128 * 4 : 0u;
}

struct TcBars {
  uint64_t wbar;                 // resident weight tile landed (TMA)
  uint64_t mma;                  // this step's MMAs finished (tcgen05.commit)
  uint64_t full[kMaxRing];       // exchange sub-tile landed (TMA)
  uint64_t empty[kMaxRing];      // exchange sub-tile consumed (tcgen05.commit)
  int flags[2][kMaxKS];          // abort flags pushed by the peers, by step parity
  uint32_t tmem;
  // forward: thread 0's post-step values (4 gates, h, c, y) per pair, stored
  // by thread 32 during the next step while thread 0 drives the contraction
  float stage[8][7];
};

// The forward requests the input projections of the step this many steps
// ahead into L2 when they are too large to stay there after the projection
// GEMM (more than a quarter of L2): the step's own loads would otherwise wait
// on HBM inside the chain (GB300: LSTM T256 B32 H1024, 67 MB of projections,
// forward 1.09 -> 1.06 ms; 2-layer bidirectional T512 B128 H1024 8.77 ->
// 8.29 ms; GRU T128 B64 H512, 17 MB, still in L2: 0.57 -> 0.59 ms, so off).
// The same prefetch of the backward's saved gates, states and dy measured
// slower (17.4 -> 18.2 ms on the 2-layer LSTM) and is not done.
constexpr int kPrefetchSteps = 4;
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigm_fast(float x) { return fmaf(0.5f, tanh_fast(0.5f * x), 0.5f); }

// Generic address of ``p`` (a shared-memory location) in CTA ``rank`` of the
// cluster; plain loads and stores through it reach distributed shared memory.
template <typename T>
__device__ __forceinline__ T* peer_ptr(T* p, int rank) {
  uint64_t g;
  asm("mapa.u64 %0, %1, %2;" : "=l"(g) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
  return reinterpret_cast<T*>(g);
}

// The MMAs of sub-tile j (64 K columns) of the K slice, exchange operand in
// ring slot ``slot``.
__device__ __forceinline__ void mma_subtile(const TcPersistParams& P, uint32_t tmem, uint64_t adesc0,
                                            uint64_t bdesc0, uint32_t rbytes, uint32_t idesc, int j, int slot) {
  const uint64_t bd = bdesc0 + static_cast<uint64_t>((slot * rbytes) >> 4);
  if (j < P.w_tmem) {
    // K=16 bf16 = 8 TMEM columns
    const uint32_t at = tmem + P.wcol + static_cast<uint32_t>(j * (kSubK / 2));
#pragma unroll
    for (int k = 0; k < kSubK / 16; ++k) mma_bf16_ts(tmem, at + 8 * k, bd + 2 * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
  } else {
    const uint64_t ad = adesc0 + static_cast<uint64_t>(((j - P.w_tmem) * kWSub) >> 4);
#pragma unroll
    for (int k = 0; k < kSubK / 16; ++k)   // +32 bytes per K=16 step inside the swizzle atom
      mma_bf16_ss(tmem, ad + 2 * k, bd + 2 * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
  }
}

// One step's contraction: bring the exchange operand's K slice into shared
// memory and accumulate into TMEM.  Called by thread 0 only.  Either one 4-D
// TMA brings the whole slice (chunk j at ring + j * rbytes), or nsub 2-D loads
// stream through a ring of R slots.  g: running load counter (across steps).
// (x0, y0): 2-D coordinates of the slice; (y4, c2, dir): its row, chunk and
// direction coordinates in the 4-D view.  Returns false on timeout.
__device__ bool contract_step(const TcPersistParams& P, const CUtensorMap* tmX, const CUtensorMap* tmX4,
                              uint8_t* ring, TcBars& bars, uint32_t tmem, uint32_t& g, int x0, int y0, int y4, int c2,
                              int dir, uint32_t idesc, uint64_t adesc0, bool first_use_w, int tk, int s) {
  (void)tk; (void)s;
  const int nsub = P.nsub, R = P.R;
  const uint32_t rbytes = static_cast<uint32_t>(P.Npad) * 128;
  const uint64_t to = P.a.timeout_ns;
  const uint64_t bdesc0 = sdesc_sw128(smem_u32(ring), 16, 1024);
  if (P.single) {
    // the previous step's MMAs on the ring finished before this CTA released
    // that step, and every CTA's did before the counter let this load start
    const int nc = P.nchunk, per = nsub / nc;
    for (int c = 0; c < nc; ++c) {
      mbar_arrive_expect_tx(&bars.full[c], static_cast<uint32_t>(per) * rbytes);
      tma_load_4d(ring + static_cast<size_t>(c) * per * rbytes, tmX4, &bars.full[c], 0, y4, c2 + c * per, dir);
    }
    RNN_TRACE_AT(1, tk, s);
    if (first_use_w && P.w_tmem < P.nsub && !mbar_wait(&bars.wbar, 0, to)) return false;
    // descriptors in registers, advanced per sub-tile: the issue loop does
    // nothing but the MMAs (one K=16 instruction per 32 bytes of K)
    const int wt = P.w_tmem;
    const uint64_t bstep = static_cast<uint64_t>(rbytes >> 4);
    uint64_t bd = bdesc0;
    uint32_t at = tmem + P.wcol;
    uint64_t ad = adesc0;
    uint32_t acc = 0u;
    for (int c = 0; c < nc; ++c) {
      if (!mbar_wait(&bars.full[c], g & 1, to)) return false;
      if (c == 0) RNN_TRACE_AT(8, tk, s);
      if (c == nc - 1) RNN_TRACE_AT(14, tk, s);
      tc_fence_after();
      const int j1 = (c + 1) * per;
      int j = c * per;
      for (; j < j1 && j < wt; ++j, at += kSubK / 2, bd += bstep) {
        mma_bf16_ts(tmem, at, bd, idesc, acc);
        mma_bf16_ts(tmem, at + 8, bd + 2, idesc, 1u);
        mma_bf16_ts(tmem, at + 16, bd + 4, idesc, 1u);
        mma_bf16_ts(tmem, at + 24, bd + 6, idesc, 1u);
        acc = 1u;
      }
      for (; j < j1; ++j, ad += static_cast<uint64_t>(kWSub >> 4), bd += bstep) {
        mma_bf16_ss(tmem, ad, bd, idesc, acc);
        mma_bf16_ss(tmem, ad + 2, bd + 2, idesc, 1u);
        mma_bf16_ss(tmem, ad + 4, bd + 4, idesc, 1u);
        mma_bf16_ss(tmem, ad + 6, bd + 6, idesc, 1u);
        acc = 1u;
      }
    }
    mma_commit(&bars.mma);
    g += 1;
    return true;
  }
  const uint32_t g0 = g;
  for (int j = 0; j < nsub && j < R; ++j) {
    const uint32_t gg = g0 + j;
    const int slot = gg % R;
    if (gg >= static_cast<uint32_t>(R) && !mbar_wait(&bars.empty[slot], ((gg / R) - 1) & 1, to)) return false;
    mbar_arrive_expect_tx(&bars.full[slot], rbytes);
    tma_load_2d(ring + slot * rbytes, tmX, &bars.full[slot], x0 + j * kSubK, y0);
  }
  RNN_TRACE_AT(1, tk, s);
  if (first_use_w && P.w_tmem < P.nsub && !mbar_wait(&bars.wbar, 0, to)) return false;
  for (int j = 0; j < nsub; ++j) {
    const uint32_t gg = g0 + j;
    const int slot = gg % R;
    if (!mbar_wait(&bars.full[slot], (gg / R) & 1, to)) return false;
    if (j == 0) RNN_TRACE_AT(8, tk, s);
    if (j == nsub - 1) RNN_TRACE_AT(14, tk, s);
    tc_fence_after();
    mma_subtile(P, tmem, adesc0, bdesc0, rbytes, idesc, j, slot);
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
  return true;
}

// TMEM accumulator rows -> the owning peer's receive buffer
// recv[src = this rank][column][row within the owner].  Warps w and w + 4 read
// the same TMEM lane quarter (32 * (w % 4) ..) and split the 32-column chunks.
__device__ __forceinline__ void push_partials(const TcPersistParams& P, uint32_t tmem, float* recv, int ks) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3, half = warp >> 2;
  const int row = q * 32 + lane;
  const int owner = row / P.RPC, lr = row - owner * P.RPC;
  // the rows this CTA owns itself go by local shared-memory stores
  float* dst = (owner == ks ? recv : peer_ptr(recv, owner)) + static_cast<size_t>(ks) * P.Npad * P.RPC + lr;
  for (int c = half * 32; c < P.Npad; c += 64) {
    float v[32];
    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, v);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c + j < P.Npad) dst[(c + j) * P.RPC] = v[j];
  }
}

// The K split of a row group exchanged through global memory instead of
// distributed shared memory (a grid without clusters: shapes whose clusters
// cannot all be resident).  ctr: the group's arrival counter; buf: its
// partials, two exchange parities of [owner][source][column][row in owner],
// so an owner's rows from every source are one contiguous block laid out as
// the receive buffer.
struct GkGroup {
  unsigned int* ctr = nullptr;
  float* buf = nullptr;
};

// TMEM accumulator rows -> the group's partials in global memory (plain
// stores; published by the caller's fence and release).
__device__ __forceinline__ void push_partials_global(const TcPersistParams& P, uint32_t tmem, float* buf, int ks) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3, half = warp >> 2;
  const int row = q * 32 + lane;
  const int owner = row / P.RPC, lr = row - owner * P.RPC;
  float* dst = buf + (static_cast<size_t>(owner) * P.KS + ks) * P.Npad * P.RPC + lr;
  for (int c = half * 32; c < P.Npad; c += 64) {
    float v[32];
    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, v);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c + j < P.Npad) dst[(c + j) * P.RPC] = v[j];
  }
}

// The per-step exchange and contraction, up to the point where this CTA's
// units' summed pre-activations can be read from ``recv``.  Returns true when
// the whole cluster may continue.
// ``deferred`` runs on every thread while the step's contraction is under
// way: on thread 0 after it has passed the counter wait and issued the step's
// TMA and MMAs, on the others at once (the previous step's stores that no CTA
// of this launch waits for, kept off the wait's critical path).
struct NoDeferred {
  __device__ void operator()() const {}
};
template <typename Deferred = NoDeferred>
__device__ __forceinline__ bool step_exchange(const TcPersistParams& P, const CUtensorMap* tmX, const CUtensorMap* tmX4,
                              uint8_t* ring, float* recv, TcBars& bars, uint32_t tmem, uint32_t& g, int x0, int y0,
                              int y4, int c2, int dir, uint32_t idesc,
                              uint64_t adesc0, bool do_contract, unsigned int* ctr_in, unsigned int wait_target, int s,
                              int ks, int& n_mma, bool& w_waited, unsigned int kernel,
                              const Deferred& deferred = Deferred(), const GkGroup& gk = GkGroup()) {
  const PersistArgs& a = P.a;
  const int tk = kernel == K_BWD_TC ? 1 : 0;
  (void)tk;
  int ok = 1;
  // warp 0's other lanes first: they would otherwise run their share only
  // once thread 0 leaves its wait and issue (divergent paths of one warp)
  if ((threadIdx.x >> 5) == 0) {
    if (threadIdx.x != 0) deferred();
    __syncwarp();
  }
  if (threadIdx.x == 0) {
    if (wait_target > 0 && !wait_counter_geq(ctr_in, wait_target, a.timeout_ns)) {
      ok = 0;
      report_status(a.dev, 4u, kernel, static_cast<unsigned>(s), W_COUNTER);
    }
    RNN_TRACE_AT(7, tk, s);
    if (ok && do_contract) {
      if (!contract_step(P, tmX, tmX4, ring, bars, tmem, g, x0, y0, y4, c2, dir, idesc, adesc0, !w_waited, tk, s)) {
        ok = 0;
        report_status(a.dev, 4u, kernel, static_cast<unsigned>(s), W_TMA);
      }
      w_waited = true;
    }
    RNN_TRACE_AT(2, tk, s);
  }
  if ((threadIdx.x >> 5) != 0) deferred();
  RNN_TRACE_AT_T(32, 15, tk, s);
  ok = __syncthreads_and(ok);
  if (ok && do_contract) {
    const bool done = mbar_wait(&bars.mma, n_mma & 1, a.timeout_ns);
    ++n_mma;
    if (!done) report_status(a.dev, 4u, kernel, static_cast<unsigned>(s), W_MMA);
    RNN_TRACE_AT(3, tk, s);
    ok = __syncthreads_and(done ? 1 : 0);
    if (ok) {
      tc_fence_after();
      if (P.gk) push_partials_global(P, tmem, gk.buf + static_cast<size_t>(s & 1) * P.KS * P.Npad * 128, ks);
      else push_partials(P, tmem, recv + recv_off(P, s) / 4, ks);
    }
  }
  RNN_TRACE_AT(9, tk, s);
  if (P.gk) {
    // publish the partials (or this CTA's failure), then wait for the KS CTAs
    // of the row group: exchange s completes at s + 1 arrivals each
    const float* pbuf = gk.buf + static_cast<size_t>(s & 1) * P.KS * P.Npad * 128;
    __threadfence();
    tc_fence_before();
    const int all_ok = __syncthreads_and(ok);
    int pass = 1;
    if (threadIdx.x == 0) {
      if (!all_ok) atomicExch(&a.dev->gk_abort, 1u);
      red_release_gpu_add(gk.ctr, 1u);
      if (!wait_counter_geq(gk.ctr, static_cast<unsigned int>(s + 1) * P.KS, a.timeout_ns)) {
        pass = 0;
        report_status(a.dev, 4u, kernel, static_cast<unsigned>(s), W_COUNTER);
      } else {
        pass = all_ok && *reinterpret_cast<volatile unsigned int*>(&a.dev->gk_abort) == 0u;
      }
    }
    pass = __syncthreads_and(pass);
    tc_fence_after();
    if (pass && do_contract) {
      // this CTA's rows from every source, as the receive buffer lays them out
      const float4* src = reinterpret_cast<const float4*>(pbuf + static_cast<size_t>(ks) * P.KS * P.Npad * P.RPC);
      float4* dst = reinterpret_cast<float4*>(recv);
      const int n4 = P.Npad * 128 / 4;
      for (int i = threadIdx.x; i < n4; i += kThreads) dst[i] = __ldcg(src + i);
      __syncthreads();
    }
    RNN_TRACE_AT(4, tk, s);
    return pass != 0;
  }
  if (static_cast<int>(threadIdx.x) < P.KS) *peer_ptr(&bars.flags[s & 1][ks], threadIdx.x) = ok ? 0 : 1;
  tc_fence_before();
  if (P.KS > 1) cluster_sync(); else __syncthreads();
  tc_fence_after();
  RNN_TRACE_AT(10, tk, s);
  int any = 0;
#pragma unroll
  for (int r = 0; r < kMaxKS; ++r)
    if (r < P.KS) any |= bars.flags[s & 1][r];
  RNN_TRACE_AT(4, tk, s);
  return any == 0;
}

// Checking builds (-DRNN_CHECKS): the host fills the buffers the step
// exchanges go through with 0xFF bytes (bf16 0xFFFF, a NaN no kernel writes)
// before each persistent launch; after every contraction, all threads scan
// the slice that landed in shared memory (whole K slice per TMA only) for the
// pattern in this CTA's batch rows and record RNN_INTERNAL / W_CHECK with the
// step in the status word: a slice read before its producers wrote it.
__device__ __forceinline__ void check_slice(const TcPersistParams& P, const uint8_t* ring, int rows,
                                            unsigned int kernel, int s) {
#ifdef RNN_CHECKS
  if (!P.single) return;
  const int per_sub = P.Npad * 8;          // 16-byte pieces per sub-tile (Npad rows of 128 bytes)
  const int n16 = P.nsub * per_sub;
  const uint32_t rbytes = static_cast<uint32_t>(P.Npad) * 128;
  int bad = 0;
  for (int i = threadIdx.x; i < n16; i += kThreads) {
    const int j = i / per_sub, rem = i - j * per_sub;
    if (rem / 8 >= rows) continue;
    const uint4 q = *reinterpret_cast<const uint4*>(ring + j * rbytes + rem * 16);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) bad |= ((w[e] & 0xFFFFu) == 0xFFFFu) || ((w[e] >> 16) == 0xFFFFu);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0)
    report_status(P.a.dev, 6u /* RNN_INTERNAL */, kernel, static_cast<unsigned>(s), W_CHECK);
#else
  (void)P; (void)ring; (void)rows; (void)kernel; (void)s;
#endif
}

// After the exchange-critical stores of a step.  Each thread orders its own
// generic-proxy stores before the TMA (async-proxy) reads that other CTAs issue
// once they observe the counter; the barrier orders every thread's stores
// before the release add.  Fencing here, on the writer side, keeps the fence
// off the reader's critical path, where it would also wait for the reader's
// own outstanding prefetch loads.
__device__ __forceinline__ void step_arrive(unsigned int* ctr_out, bool skip, int s, int tk) {
  (void)s; (void)tk;
  fence_proxy_async_global();
  __syncthreads();
  RNN_TRACE_AT(11, tk, s);
  if (threadIdx.x == 0 && !skip) red_release_gpu_add(ctr_out, 1u);
}

// The step counter a CTA waits on (the K slice ks it contracts) or arrives on
// (the K slice its outputs fall in), of its direction and batch part.  Each of
// the KS slices of a batch part is written by exactly nrg CTAs: one CTA's
// outputs (forward 32/KS units, backward 4 x 128/KS gate-gradient columns)
// lie in one slice of H/KS units (forward) or 4H/KS columns (backward).
__device__ __forceinline__ unsigned int* slice_counter(const TcPersistParams& P, int nbp, int slice) {
  const int d = P.a.dir0 + static_cast<int>(blockIdx.y);
  return &P.a.dev->slice_ctr[(d * P.NB + nbp) * P.KS + slice];
}

__device__ __forceinline__ uint2 ld_u2(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }

// Explicit shared-memory loads: the compiler cannot mistake them for global
// accesses that might alias the epilogue's stores, so they issue together.
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ float lds_f1(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ void unpack4(uint2 q, float (&v)[4]) {
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&q.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&q.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}

// V (1, 2 or 4) consecutive values in one access: fp32, bf16 (widened to
// fp32), and V units' 4-slot bf16 rows (as raw 32-bit words / from fp32).
template <int V>
__device__ __forceinline__ void ld_f32v(const float* p, float (&o)[V]) {
  if constexpr (V == 4) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    o[0] = q.x; o[1] = q.y; o[2] = q.z; o[3] = q.w;
  } else if constexpr (V == 2) {
    const float2 q = *reinterpret_cast<const float2*>(p);
    o[0] = q.x; o[1] = q.y;
  } else {
    o[0] = *p;
  }
}
template <int V>
__device__ __forceinline__ void ld_bf16v(const __nv_bfloat16* p, float (&o)[V]) {
  if constexpr (V == 4) {
    float v[4];
    unpack4(*reinterpret_cast<const uint2*>(p), v);
    o[0] = v[0]; o[1] = v[1]; o[2] = v[2]; o[3] = v[3];
  } else if constexpr (V == 2) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    o[0] = f.x; o[1] = f.y;
  } else {
    o[0] = __bfloat162float(*p);
  }
}
template <int V>
__device__ __forceinline__ void st_bf16v(__nv_bfloat16* p, const float (&v)[V]) {
  if constexpr (V == 4) {
    Vec4<__nv_bfloat16>::store(p, v);
  } else if constexpr (V == 2) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v[0], v[1]);
  } else {
    *p = __float2bfloat16_rn(v[0]);
  }
}
template <int V>
__device__ __forceinline__ void ld_rows(const __nv_bfloat16* p, uint32_t (&w)[2 * V]) {
  if constexpr (V == 4) {
    const uint4 a = reinterpret_cast<const uint4*>(p)[0], b = reinterpret_cast<const uint4*>(p)[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else if constexpr (V == 2) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(p);
    w[0] = a.x; w[1] = a.y;
  }
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <int V>
__device__ __forceinline__ void st_rows(__nv_bfloat16* p, const float (&v)[V][4]) {
  uint32_t w[2 * V];
#pragma unroll
  for (int j = 0; j < V; ++j) {
    w[2 * j] = pack_bf16x2(v[j][0], v[j][1]);
    w[2 * j + 1] = pack_bf16x2(v[j][2], v[j][3]);
  }
  if constexpr (V == 4) {
    reinterpret_cast<uint4*>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else if constexpr (V == 2) {
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  }
}
__device__ __forceinline__ float2 lds_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
  return v;
}
template <int V>
__device__ __forceinline__ void lds_v(uint32_t a, float (&o)[V]) {
  if constexpr (V == 4) {
    const float4 q = lds_f4(a);
    o[0] = q.x; o[1] = q.y; o[2] = q.z; o[3] = q.w;
  } else if constexpr (V == 2) {
    const float2 q = lds_f2(a);
    o[0] = q.x; o[1] = q.y;
  } else {
    o[0] = lds_f1(a);
  }
}

// Barriers, TMEM, and the resident weight tile: 128 rows from row wy0, K
// columns from column wx0 of the packed weight matrix w (leading dimension
// ldw).  Its first w_tmem sub-tiles go by every thread through registers into
// TMEM columns [wcol, wcol + 32 * w_tmem) (lane = row), the others by TMA into
// shared memory.
__device__ __forceinline__ void setup(const TcPersistParams& P, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                      const CUtensorMap* tmX4, uint8_t* wsm, TcBars& bars, int wx0, int wy0,
                                      const __nv_bfloat16* w, int64_t ldw) {
  if (threadIdx.x == 0) {
    mbar_init(&bars.wbar, 1);
    mbar_init(&bars.mma, 1);
    for (int i = 0; i < P.R; ++i) { mbar_init(&bars.full[i], 1); mbar_init(&bars.empty[i], 1); }
    fence_mbar_init();
    fence_proxy_async_smem();
    if (P.single) prefetch_tmap(tmX4); else prefetch_tmap(tmX);
    if (P.w_tmem < P.nsub) {
      prefetch_tmap(tmW);
      mbar_arrive_expect_tx(&bars.wbar, static_cast<uint32_t>(P.nsub - P.w_tmem) * kWSub);
      for (int j = P.w_tmem; j < P.nsub; ++j)
        tma_load_2d(wsm + (j - P.w_tmem) * kWSub, tmW, &bars.wbar, wx0 + j * kSubK, wy0);
    }
  }
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(&bars.tmem, P.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (P.w_tmem) {
    // warps w and w + 4 share lane quarter w % 4 and split the K columns
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, half = warp >> 2;
    const int kt = P.w_tmem * kSubK;   // K columns held in TMEM (w_tmem even)
    const int ncol = kt / 4;           // 32-bit columns per half
    const __nv_bfloat16* src = w + (static_cast<int64_t>(wy0) + q * 32 + lane) * ldw + wx0 + half * (kt / 2);
    const uint32_t trow = bars.tmem + (static_cast<uint32_t>(q * 32) << 16) + P.wcol + static_cast<uint32_t>(half * ncol);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
}

__device__ __forceinline__ void teardown(const TcPersistParams& P, TcBars& bars) {
  tc_fence_before();
  if (P.KS > 1 && !P.gk) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(bars.tmem, P.tmem_cols);
}

#define RNN_TC_SMEM_VIEW                                                                              \
  extern __shared__ __align__(1024) uint8_t smem_raw[];                                              \
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &         \
                                             ~static_cast<uintptr_t>(1023));                          \
  uint8_t* wsm = base;                                                                                \
  uint8_t* ring = base + P.off_ring;                                                                  \
  float* recv = reinterpret_cast<float*>(base + P.off_recv);                                          \
  TcBars& bars = *reinterpret_cast<TcBars*>(base + P.off_bar)

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <int PP, int KS, bool EXT>
__global__ void __launch_bounds__(kThreads, 1)
persist_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmX4, const __grid_constant__ CUtensorMap tmR,
                      const __grid_constant__ CUtensorMap tmR4, const __grid_constant__ TcPersistParams P) {
  RNN_TC_SMEM_VIEW;
  const PersistArgs& a = P.a;
  const int H = a.H, B = a.B, TT = a.T, D = a.D;
  const int dir = a.dir0 + blockIdx.y;
  // blockIdx.x = (batch part * row groups + row group) * KS + K slice; a
  // cluster is the KS K slices of one row group and batch part
  const int ks = static_cast<int>(blockIdx.x) % KS;
  const int rg = (static_cast<int>(blockIdx.x) / KS) % P.nrg;
  const int b0 = (static_cast<int>(blockIdx.x) / KS / P.nrg) * P.Bp;   // first batch row of this part
  const int Bn = min(P.Bp, B - b0);
  const bool lstm = a.mode == 0;
  // GRU reset-before (extended variant only): two exchanges per step, the
  // second over r * h_{t-1} (tmR / tmR4: a view of RH [D][T*B][H])
  const bool rbm = EXT && a.mode == 1 && !a.reset_after;
  __nv_bfloat16* RHp = static_cast<__nv_bfloat16*>(a.RH);
  constexpr int RPC = 128 / KS;
  const bool clip = EXT && a.clip;
  const float clo = a.clip_lo, chi = a.clip_hi;

  setup(P, &tmW, &tmX, &tmX4, wsm, bars, ks * P.Kc, dir * 4 * H + rg * 128, static_cast<const __nv_bfloat16*>(a.Wr),
        H);
  const uint32_t tmem = bars.tmem;
  const uint32_t idesc = idesc_bf16(128, P.Npad, false, false);
  const uint64_t adesc0 = sdesc_sw128(smem_u32(wsm), 16, 1024);

  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.Y);
  const __nv_bfloat16* Pm = static_cast<const __nv_bfloat16*>(a.P);
  __nv_bfloat16* G = static_cast<__nv_bfloat16*>(a.gates);
  const int64_t ldY = static_cast<int64_t>(D) * H;
  const int64_t ldP = static_cast<int64_t>(D) * 4 * H;
  const int UPC = P.UPC;
  const int npairs = UPC * Bn;
  const int ubase = rg * 32 + ks * UPC;     // first hidden unit of this CTA's epilogue
  const int slot_h0 = dir ? TT + 1 : 0;
  const uint32_t recv_s = smem_u32(recv);
  const uint32_t src_bytes = static_cast<uint32_t>(P.Npad) * RPC * 4;   // bytes per source rank in recv

  float st[PP];      // LSTM: c_{t-1}; GRU: h_{t-1}
  float hl[PP];      // EXT, LSTM: h_{t-1} (held over masked steps)
  int lenp[PP];      // EXT: valid steps of the pair's sequence
  float bh[PP][3];
#pragma unroll
  for (int p = 0; p < PP; ++p) {
    st[p] = hl[p] = 0.f;
    lenp[p] = TT;
    bh[p][0] = bh[p][1] = bh[p][2] = 0.f;
    const int id = threadIdx.x + p * kThreads;
    if (id >= npairs) continue;
    const int ul = id % UPC, b = b0 + id / UPC, u = ubase + ul;
    if constexpr (EXT) lenp[p] = a.len ? a.len[b] : TT;   // clipping alone: no lengths
    if (lstm) {
      const __nv_bfloat16* c0 = static_cast<const __nv_bfloat16*>(a.c0);
      st[p] = c0 ? __bfloat162float(c0[(static_cast<int64_t>(dir) * B + b) * H + u]) : 0.f;
      if constexpr (EXT) hl[p] = __bfloat162float(Y[(static_cast<int64_t>(slot_h0) * B + b) * ldY + dir * H + u]);
      if (a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? TT : 0)) * B + b) * H + u] = st[p];
    } else {
      st[p] = __bfloat162float(Y[(static_cast<int64_t>(slot_h0) * B + b) * ldY + dir * H + u]);
      if (a.bh) {   // resetAfter's recurrent biases (reset-before has its biases in P)
        const float* bb = a.bh + dir * 4 * H + 4 * u;
        bh[p][0] = bb[0]; bh[p][1] = bb[1]; bh[p][2] = bb[2];
      }
    }
  }

  // the step counters: in, the K slice this CTA contracts; out, the slice its
  // units' new state falls in
  const int nbp = static_cast<int>(blockIdx.x) / KS / P.nrg;
  unsigned int* const ctr_in = slice_counter(P, nbp, ks);
  unsigned int* const ctr_out = slice_counter(P, nbp, (rg * 32) / P.Kc);
  const bool skip = a.skip_cta == static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);
  uint32_t g = 0;
  int n_mma = 0;
  bool w_waited = false;
  bool aborted = false;
  // the step's new state and gate values: the state goes out before the
  // step's release; the rest is stored during the next step's contraction
  float hv[PP];
  float gq[PP][4];
#pragma unroll
  for (int p = 0; p < PP; ++p) {
    hv[p] = 0.f;
    gq[p][0] = gq[p][1] = gq[p][2] = gq[p][3] = 0.f;
  }
  // stores of step sd that no CTA of this launch waits for (pair id: its 4
  // gate values, the new state h, the LSTM cell c and the output y), and the
  // L2 prefetch of a later step's projections
  auto store_pair = [&](int sd, int id, const float (&g4)[4], float h, float c, float yv) {
    const int t = dir ? TT - 1 - sd : sd;
    const int ul = id % UPC, b = b0 + id / UPC, u = ubase + ul;
    // one prefetch per 128-byte line of the projections (16 units)
    if (P.prefetch && sd + kPrefetchSteps < TT && ((u & 15) == 0 || ul == 0)) {
      const int tf = dir ? TT - 1 - (sd + kPrefetchSteps) : sd + kPrefetchSteps;
      prefetch_l2(Pm + (static_cast<int64_t>(tf) * B + b) * ldP + dir * 4 * H + 4 * u);
    }
    if (G) Vec4<__nv_bfloat16>::store(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * 4 * H + 4 * u, g4);
    if (lstm && a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? t : t + 1)) * B + b) * H + u] = c;
    if (a.y_out)
      static_cast<__nv_bfloat16*>(a.y_out)[(static_cast<int64_t>(t) * B + b) * ldY + dir * H + u] =
          __float2bfloat16_rn(yv);
    if (sd == TT - 1) {
      const int64_t o = (static_cast<int64_t>(dir) * B + b) * H + u;
      if (a.hy) static_cast<__nv_bfloat16*>(a.hy)[o] = __float2bfloat16_rn(h);
      if (lstm && a.cy) static_cast<__nv_bfloat16*>(a.cy)[o] = __float2bfloat16_rn(c);
    }
  };
  auto y_of = [&](int sd, int p) {
    float yv = hv[p];
    if constexpr (EXT) {
      const int t = dir ? TT - 1 - sd : sd;
      if (t >= lenp[p]) yv = 0.f;
    }
    return yv;
  };
  // The stores of a step take about 0.15 us per pair a thread owns and must
  // not delay thread 0, which drives the next step's wait, TMA and MMAs.
  // Warp 0 stages all its pairs' values (8 floats each: 4 gates, h, c, y)
  // and warps 1-7 store them: without a K split in the receive buffer, idle
  // from the end of a step until the next step's partials land; with a K
  // split (peers may write the receive buffer at any time) in a stage area of
  // its own where shared memory allows.  Otherwise thread 0 alone stages its
  // pairs (bars.stage) for thread 32, and warp 0's other lanes store theirs
  // before thread 0 starts its wait.
  float* const stage_w0 = KS == 1 ? recv : (P.off_stage ? reinterpret_cast<float*>(base + P.off_stage) : nullptr);
  const bool kStageWarp0 = stage_w0 != nullptr;
  auto post_stores = [&](int sd, bool own) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool mine = own || (kStageWarp0 ? warp != 0 : threadIdx.x != 0);
    if (mine) {
#pragma unroll
      for (int p = 0; p < PP; ++p) {
        const int id = threadIdx.x + p * kThreads;
        if (id >= npairs) break;
        store_pair(sd, id, gq[p], hv[p], st[p], y_of(sd, p));
      }
    }
    if (own) return;
    if (kStageWarp0) {
      if (warp != 0) {
        // staged entry j = warp-0 lane j % 32, pair j / 32
        for (int j = (warp - 1) * 32 + lane; j < 32 * PP; j += 7 * 32) {
          const int id = (j & 31) + (j >> 5) * kThreads;
          if (id >= npairs) continue;
          const float4 g = *reinterpret_cast<const float4*>(stage_w0 + 8 * j);
          const float4 r = *reinterpret_cast<const float4*>(stage_w0 + 8 * j + 4);
          const float g4[4] = {g.x, g.y, g.z, g.w};
          store_pair(sd, id, g4, r.x, r.y, r.z);
        }
      }
    } else if (threadIdx.x == 32) {
#pragma unroll
      for (int p = 0; p < PP; ++p) {
        const int id = p * kThreads;
        if (id >= npairs) break;
        const float* v = bars.stage[p];
        const float g4[4] = {v[0], v[1], v[2], v[3]};
        store_pair(sd, id, g4, v[4], v[5], v[6]);
      }
    }
  };
  // the staging of step sd's values (ordered before the readers by the
  // barrier of the step's release; without a K split after a barrier that
  // ends every read of the step's partial sums)
  auto stage_own = [&](int sd) {
    if (kStageWarp0) {
      if (KS == 1) __syncthreads();   // every read of the step's partial sums is done
      if ((threadIdx.x >> 5) != 0) return;
#pragma unroll
      for (int p = 0; p < PP; ++p) {
        if (static_cast<int>(threadIdx.x) + p * kThreads >= npairs) break;
        float* v = stage_w0 + 8 * (threadIdx.x + 32 * p);
        *reinterpret_cast<float4*>(v) = make_float4(gq[p][0], gq[p][1], gq[p][2], gq[p][3]);
        *reinterpret_cast<float4*>(v + 4) = make_float4(hv[p], st[p], y_of(sd, p), 0.f);
      }
    } else {
      if (threadIdx.x != 0) return;
#pragma unroll
      for (int p = 0; p < PP; ++p) {
        if (p * kThreads >= npairs) break;
        float* v = bars.stage[p];
        v[0] = gq[p][0]; v[1] = gq[p][1]; v[2] = gq[p][2]; v[3] = gq[p][3];
        v[4] = hv[p]; v[5] = st[p]; v[6] = y_of(sd, p);
      }
    }
  };
  for (int s = 0; s < TT; ++s) {
    const int t = dir ? TT - 1 - s : s;
    const int sp = dir ? t + 2 : t;
    const int so = t + 1;
    RNN_TRACE_AT(0, 0, s);
    // this step's input projections do not depend on the exchange: load them first
    uint2 pq[PP];
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      const int ul = id % UPC, b = b0 + id / UPC, u = ubase + ul;
      pq[p] = id < npairs ? ld_u2(Pm + (static_cast<int64_t>(t) * B + b) * ldP + dir * 4 * H + 4 * u) : make_uint2(0, 0);
    }
    const int ex = rbm ? 2 * s : s;   // exchanges (counter phases) before this step's first
    auto deferred = [&]() {
      if (s > 0) post_stores(s - 1, false);
    };
    if (!step_exchange(P, &tmX, &tmX4, ring, recv, bars, tmem, g, dir * H + ks * P.Kc, sp * B + b0, sp * B + b0,
                       ks * P.nsub, dir, idesc, adesc0, true, ctr_in, static_cast<unsigned int>(ex) * P.nrg, ex, ks,
                       n_mma, w_waited, K_FWD_TC, deferred)) {
      aborted = true;
      break;
    }
    check_slice(P, ring, Bn, K_FWD_TC, s);
    // partial sums of every pair first (all shared loads in flight), then the cell
    float4 acc[PP];
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      const int ul = id % UPC, bl = id / UPC;
      acc[p] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (id < npairs) {
        const uint32_t ra = recv_s + recv_off(P, ex) + static_cast<uint32_t>((bl * RPC + 4 * ul) * 4);
        float4 v[KS];
#pragma unroll
        for (int r = 0; r < KS; ++r) v[r] = lds_f4(ra + r * src_bytes);
#pragma unroll
        for (int r = 0; r < KS; ++r) {
          acc[p].x += v[r].x; acc[p].y += v[r].y; acc[p].z += v[r].z; acc[p].w += v[r].w;
        }
      }
    }
    RNN_TRACE_AT(12, 0, s);
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      hv[p] = 0.f;
      gq[p][0] = gq[p][1] = gq[p][2] = gq[p][3] = 0.f;
      if (id >= npairs) break;
      const int ul = id % UPC, b = b0 + id / UPC, u = ubase + ul;
      float pv[4];
      unpack4(pq[p], pv);
      float h;
      if (lstm) {
        const float i = sigm_fast(pv[0] + acc[p].x);
        const float f = sigm_fast(pv[1] + acc[p].y);
        const float gg = tanh_fast(pv[2] + acc[p].z);
        const float o = sigm_fast(pv[3] + acc[p].w);
        float c;
        if (clip) {
          c = f * clipv(st[p], clo, chi) + i * gg;
          h = o * tanh_fast(clipv(c, clo, chi));
        } else {
          c = f * st[p] + i * gg;
          h = o * tanh_fast(c);
        }
        if constexpr (EXT) {
          if (t >= lenp[p]) { c = st[p]; h = hl[p]; }
          hl[p] = h;
        }
        st[p] = c;
        pv[0] = i; pv[1] = f; pv[2] = gg; pv[3] = o;
      } else if (rbm) {
        // reset-before, phase A: r, z and the reset state the second contraction reads
        const float r = sigm_fast(pv[0] + acc[p].x);
        const float z = sigm_fast(pv[1] + acc[p].y);
        gq[p][0] = r; gq[p][1] = z;
        RHp[((static_cast<int64_t>(dir) * TT + t) * B + b) * H + u] = __float2bfloat16_rn(r * st[p]);
        continue;
      } else {
        const float r = sigm_fast(pv[0] + acc[p].x + bh[p][0]);
        const float z = sigm_fast(pv[1] + acc[p].y + bh[p][1]);
        const float hn = acc[p].z + bh[p][2];
        const float n = tanh_fast(pv[2] + r * hn);
        h = (1.f - z) * n + z * st[p];
        if constexpr (EXT) {
          if (t >= lenp[p]) h = st[p];
        }
        st[p] = h;
        pv[0] = r; pv[1] = z; pv[2] = n; pv[3] = hn;
      }
      hv[p] = h;
      gq[p][0] = pv[0]; gq[p][1] = pv[1]; gq[p][2] = pv[2]; gq[p][3] = pv[3];
      Y[(static_cast<int64_t>(so) * B + b) * ldY + dir * H + u] = __float2bfloat16_rn(h);
    }
    if constexpr (EXT) {
      if (rbm) {
        // reset-before, phase B: publish r * h_{t-1}, then n = tanh(W_in x + b_n + W_hn (r * h_{t-1}))
        step_arrive(ctr_out, skip, s, 0);
        if (!step_exchange(P, &tmR, &tmR4, ring, recv, bars, tmem, g, ks * P.Kc, (dir * TT + t) * B + b0, t * B + b0,
                           ks * P.nsub, dir, idesc, adesc0, true, ctr_in, static_cast<unsigned int>(ex + 1) * P.nrg,
                           ex + 1, ks, n_mma, w_waited, K_FWD_TC)) {
          aborted = true;
          break;
        }
        check_slice(P, ring, Bn, K_FWD_TC, s);
#pragma unroll
        for (int p = 0; p < PP; ++p) {
          const int id = threadIdx.x + p * kThreads;
          if (id >= npairs) break;
          const int ul = id % UPC, bl = id / UPC, b = b0 + bl, u = ubase + ul;
          const uint32_t ra = recv_s + recv_off(P, ex + 1) + static_cast<uint32_t>((bl * RPC + 4 * ul + 2) * 4);
          float sn = 0.f;
#pragma unroll
          for (int r = 0; r < KS; ++r) sn += lds_f1(ra + r * src_bytes);
          float pv[4];
          unpack4(pq[p], pv);
          const float n = tanh_fast(pv[2] + sn);
          const float z = gq[p][1];
          float h = (1.f - z) * n + z * st[p];
          if (t >= lenp[p]) h = st[p];
          st[p] = h;
          hv[p] = h;
          gq[p][2] = n; gq[p][3] = 0.f;
          Y[(static_cast<int64_t>(so) * B + b) * ldY + dir * H + u] = __float2bfloat16_rn(h);
        }
      }
    }
    RNN_TRACE_AT(13, 0, s);
    stage_own(s);
    RNN_TRACE_AT(5, 0, s);
    step_arrive(ctr_out, skip, s, 0);
    RNN_TRACE_AT(6, 0, s);
  }
  if (!aborted) post_stores(TT - 1, true);
  teardown(P, bars);
}

// ---------------------------------------------------------------------------
// backward through time
// ---------------------------------------------------------------------------
template <int PP, int KS, bool EXT>
__global__ void __launch_bounds__(kThreads, 1)
persist_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmX4, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmA4, const __grid_constant__ TcPersistParams P) {
  RNN_TC_SMEM_VIEW;
  const PersistArgs& a = P.a;
  const int H = a.H, B = a.B, TT = a.T, D = a.D;
  const int K4 = 4 * H;
  const int dir = a.dir0 + blockIdx.y;
  const int ks = static_cast<int>(blockIdx.x) % KS;
  const int rg = (static_cast<int>(blockIdx.x) / KS) % P.nrg;
  const int nb = static_cast<int>(blockIdx.x) / KS / P.nrg;   // batch part
  const int b0 = nb * P.Bp;
  const int Bn = min(P.Bp, B - b0);
  const bool lstm = a.mode == 0;
  constexpr int RPC = 128 / KS;
  const bool clip = EXT && a.clip;
  const float clo = a.clip_lo, chi = a.clip_hi;
  // GRU reset-before (extended variant only): two exchanges per step.  Phase
  // A publishes [0, 0, dn, 0] (XA), whose contraction with the resident
  // W_hh^T is d(rh) = W_hn^T dn; phase B publishes dG = [dr, dz, dn, 0], whose
  // contraction the next step reads: W_{h,rz}^T [dr, dz] + W_hn^T dn, so the
  // carry adds d(rh) (r - 1) + dh z to give
  //   dh_{t-1} = W_{h,rz}^T [dr, dz] + d(rh) r + dh z.
  const bool rbm = EXT && a.mode == 1 && !a.reset_after;
  const int ph = rbm ? 2 : 1;   // counter phases per step
  __nv_bfloat16* XA = static_cast<__nv_bfloat16*>(a.XA);

  setup(P, &tmW, &tmX, &tmX4, wsm, bars, ks * P.Kc, dir * H + rg * 128, static_cast<const __nv_bfloat16*>(a.WrT),
        4 * H);
  const uint32_t tmem = bars.tmem;
  const uint32_t idesc = idesc_bf16(128, P.Npad, false, false);
  const uint64_t adesc0 = sdesc_sw128(smem_u32(wsm), 16, 1024);

  const __nv_bfloat16* Y = static_cast<const __nv_bfloat16*>(a.Y);
  const __nv_bfloat16* G = static_cast<const __nv_bfloat16*>(a.gates);
  __nv_bfloat16* dG = static_cast<__nv_bfloat16*>(a.dG);
  const float* Cb = a.C ? a.C + static_cast<int64_t>(dir) * (TT + 1) * B * H : nullptr;
  const int64_t ldY = static_cast<int64_t>(D) * H;
  const int64_t ldG = static_cast<int64_t>(D) * K4;
  const int UPC = P.UPC;
  const int ubase = rg * 128 + ks * UPC;
  const uint32_t recv_s = smem_u32(recv);
  const uint32_t src_bytes = static_cast<uint32_t>(P.Npad) * RPC * 4;
  // Pairs: each thread owns V consecutive units of NQ batch rows (V = 4 from
  // 4 pairs per thread on), so every gate, state, gradient and partial-sum
  // access of the epilogue is one vector access per V pairs.  Pair p = q V + j:
  // unit ul0 + j of local batch row rl0 + q RPT.
  constexpr int V = PP >= 4 ? 4 : PP;
  constexpr int NQ = PP / V;
  const int TPR = UPC / V;               // threads per batch row (UPC is a power of two >= 8)
  const int RPT = kThreads / TPR;        // batch rows per round of the threads
  const int ul0 = V * (static_cast<int>(threadIdx.x) % TPR);
  const int u0 = ubase + ul0;
  const int rl0 = static_cast<int>(threadIdx.x) / TPR;

  // carry: LSTM dc_next, GRU dh*z (or the whole dh over a masked step);
  // carry_h: LSTM dh passed over masked steps
  float carry[PP], carry_h[PP], db[PP][4];
  float cnext[PP];   // LSTM: the cell state the next step needs as c_t
  float dhv[PP], dnv[PP], dzv[PP];   // reset-before: dh, dn, dz between the step's two phases
  int lenq[NQ];
#pragma unroll
  for (int p = 0; p < PP; ++p) {
    carry[p] = carry_h[p] = cnext[p] = 0.f;
    dhv[p] = dnv[p] = dzv[p] = 0.f;
    db[p][0] = db[p][1] = db[p][2] = db[p][3] = 0.f;
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    lenq[q] = TT;
    const int rl = rl0 + q * RPT;
    if (rl >= Bn) continue;
    const int b = b0 + rl;
    if constexpr (EXT) lenq[q] = a.len ? a.len[b] : TT;   // clipping alone: no lengths
    if (lstm && a.dcT) {
      float v[V];
      ld_bf16v<V>(static_cast<const __nv_bfloat16*>(a.dcT) + (static_cast<int64_t>(dir) * B + b) * H + u0, v);
#pragma unroll
      for (int jj = 0; jj < V; ++jj) carry[q * V + jj] = v[jj];
    }
  }

  // the step counters: in, the K slice this CTA contracts; out, the slice its
  // units' gate gradients fall in
  unsigned int* const ctr_in = slice_counter(P, nb, ks);
  unsigned int* const ctr_out = slice_counter(P, nb, (4 * ubase) / P.Kc);
  const bool skip = a.skip_cta == static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);
  // K split through global memory: this row group's counter and partials
  GkGroup gkg;
  if (P.gk) {
    const int grp = (static_cast<int>(blockIdx.y) * P.NB + nb) * P.nrg + rg;
    gkg.ctr = &a.dev->gk_ctr[grp];
    gkg.buf = a.gk_buf + static_cast<size_t>(grp) * 2 * KS * P.Npad * 128;
  }
  uint32_t g = 0;
  int n_mma = 0;
  bool w_waited = false;
  bool aborted = false;
  for (int s = 0; s <= TT; ++s) {
    const int tp = dir ? s - 1 : TT - s;     // step processed just before (s >= 1)
    const int t = dir ? s : TT - 1 - s;
    const int sp = dir ? t + 2 : t;
    RNN_TRACE_AT(0, 1, s);
    // this step's saved forward values and upstream gradient: load before the exchange
    // (LSTM: c_t is the c_{t-1} the previous step loaded, only c_{t-1} is read)
    uint32_t gw[NQ][2 * V];
    float e0[PP], e1[PP], dyv[PP];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
#pragma unroll
      for (int k = 0; k < 2 * V; ++k) gw[q][k] = 0u;
#pragma unroll
      for (int jj = 0; jj < V; ++jj) e0[q * V + jj] = e1[q * V + jj] = dyv[q * V + jj] = 0.f;
      const int rl = rl0 + q * RPT;
      if (rl >= Bn || s >= TT) continue;
      const int b = b0 + rl;
      ld_rows<V>(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * K4 + 4 * u0, gw[q]);
      float v[V];
      ld_f32v<V>(a.dYi + (static_cast<int64_t>(t) * B + b) * ldY + dir * H + u0, v);
#pragma unroll
      for (int jj = 0; jj < V; ++jj) dyv[q * V + jj] = v[jj];
      if (lstm) {
        if (s == 0) {
          ld_f32v<V>(Cb + (static_cast<int64_t>(dir ? t : t + 1) * B + b) * H + u0, v);
#pragma unroll
          for (int jj = 0; jj < V; ++jj) e0[q * V + jj] = v[jj];
        } else {
#pragma unroll
          for (int jj = 0; jj < V; ++jj) e0[q * V + jj] = cnext[q * V + jj];
        }
        ld_f32v<V>(Cb + (static_cast<int64_t>(dir ? t + 1 : t) * B + b) * H + u0, v);
#pragma unroll
        for (int jj = 0; jj < V; ++jj) e1[q * V + jj] = v[jj];
      } else {
        ld_bf16v<V>(Y + (static_cast<int64_t>(sp) * B + b) * ldY + dir * H + u0, v);
#pragma unroll
        for (int jj = 0; jj < V; ++jj) e0[q * V + jj] = v[jj];
      }
    }
    if (!step_exchange(P, &tmX, &tmX4, ring, recv, bars, tmem, g, dir * K4 + ks * P.Kc, (s > 0 ? tp : 0) * B + b0,
                       (s > 0 ? tp : 0) * B + b0, ks * P.nsub, dir, idesc, adesc0, s > 0, ctr_in,
                       static_cast<unsigned int>(s * ph) * P.nrg, s * ph, ks, n_mma, w_waited, K_BWD_TC,
                       NoDeferred(), gkg)) {
      aborted = true;
      break;
    }
    if (s > 0) check_slice(P, ring, Bn, K_BWD_TC, s);
    // recurrent gradient of every pair first (all shared loads in flight)
    float dhs[PP];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
#pragma unroll
      for (int jj = 0; jj < V; ++jj) dhs[q * V + jj] = 0.f;
      const int rl = rl0 + q * RPT;
      if (rl >= Bn) continue;
      if (s == 0) {
        if (a.dhT) {
          float v[V];
          ld_bf16v<V>(static_cast<const __nv_bfloat16*>(a.dhT) + (static_cast<int64_t>(dir) * B + b0 + rl) * H + u0, v);
#pragma unroll
          for (int jj = 0; jj < V; ++jj) dhs[q * V + jj] = v[jj];
        }
      } else {
        const uint32_t ra = recv_s + recv_off(P, s * ph) + static_cast<uint32_t>((rl * RPC + ul0) * 4);
        float v[KS][V];
#pragma unroll
        for (int r = 0; r < KS; ++r) lds_v<V>(ra + r * src_bytes, v[r]);
#pragma unroll
        for (int r = 0; r < KS; ++r) {
#pragma unroll
          for (int jj = 0; jj < V; ++jj) dhs[q * V + jj] += v[r][jj];
        }
      }
    }
    RNN_TRACE_AT(12, 1, s);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int rl = rl0 + q * RPT;
      if (rl >= Bn) break;
      const int b = b0 + rl;
      if (s == TT) {
        float h0v[V], c0v[V];
#pragma unroll
        for (int jj = 0; jj < V; ++jj) {
          const int p = q * V + jj;
          h0v[jj] = lstm ? dhs[p] + (EXT ? carry_h[p] : 0.f) : dhs[p] + carry[p];
          c0v[jj] = carry[p];
        }
        const int64_t o = (static_cast<int64_t>(dir) * B + b) * H + u0;
        if (a.dh0) st_bf16v<V>(static_cast<__nv_bfloat16*>(a.dh0) + o, h0v);
        if (lstm && a.dc0) st_bf16v<V>(static_cast<__nv_bfloat16*>(a.dc0) + o, c0v);
        continue;
      }
      bool live = true;
      if constexpr (EXT) live = t < lenq[q];
      float da[V][4];
      float xa[V][4];
#pragma unroll
      for (int jj = 0; jj < V; ++jj) {
        const int p = q * V + jj;
        const float dhr = dhs[p];
        float gv[4];
        unpack4(make_uint2(gw[q][2 * jj], gw[q][2 * jj + 1]), gv);
        da[jj][0] = da[jj][1] = da[jj][2] = da[jj][3] = 0.f;
        if (rbm) {
          // phase A: dn, dz; [0, 0, dn, 0] to XA for the first exchange
          const float gh = dhr + carry[p];
          float dn = 0.f, dz = 0.f;
          if (live) {
            const float z = gv[1], n = gv[2], hp = e0[p];
            const float dh = dyv[p] + gh;
            dn = dh * (1.f - z) * (1.f - n * n);
            dz = dh * (hp - n) * z * (1.f - z);
            dhv[p] = dh;
          } else {
            dhv[p] = gh;
          }
          dnv[p] = dn;
          dzv[p] = dz;
          xa[jj][0] = 0.f; xa[jj][1] = 0.f; xa[jj][2] = dn; xa[jj][3] = 0.f;
          continue;
        }
        if (lstm) {
          const float gh = EXT ? dhr + carry_h[p] : dhr;
          if (live) {
            const float i = gv[0], f = gv[1], gg = gv[2], o = gv[3];
            const float c = e0[p], cp = e1[p];
            const float dh = dyv[p] + gh;
            if (clip) {
              const float tc = tanh_fast(clipv(c, clo, chi));
              const float dc = dh * o * (1.f - tc * tc) * dclipv(c, clo, chi) + carry[p];
              da[jj][0] = dc * gg * i * (1.f - i);
              da[jj][1] = dc * clipv(cp, clo, chi) * f * (1.f - f);
              da[jj][2] = dc * i * (1.f - gg * gg);
              da[jj][3] = dh * tc * o * (1.f - o);
              carry[p] = dc * f * dclipv(cp, clo, chi);
            } else {
              const float tc = tanh_fast(c);
              const float dc = dh * o * (1.f - tc * tc) + carry[p];
              da[jj][0] = dc * gg * i * (1.f - i);
              da[jj][1] = dc * cp * f * (1.f - f);
              da[jj][2] = dc * i * (1.f - gg * gg);
              da[jj][3] = dh * tc * o * (1.f - o);
              carry[p] = dc * f;
            }
            if constexpr (EXT) carry_h[p] = 0.f;
          } else {
            carry_h[p] = gh;
          }
          cnext[p] = e1[p];
        } else {
          const float gh = dhr + carry[p];
          if (live) {
            const float r = gv[0], z = gv[1], n = gv[2], hn = gv[3];
            const float hp = e0[p];
            const float dh = dyv[p] + gh;
            const float dn = dh * (1.f - z) * (1.f - n * n);
            const float dz = dh * (hp - n) * z * (1.f - z);
            const float dr = dn * hn * r * (1.f - r);
            da[jj][0] = dr; da[jj][1] = dz; da[jj][2] = dn; da[jj][3] = dn * r;
            carry[p] = dh * z;
          } else {
            carry[p] = gh;
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) db[p][c] += da[jj][c];
      }
      const int64_t row = (static_cast<int64_t>(t) * B + b) * ldG + dir * K4 + 4 * u0;
      if (rbm) st_rows<V>(XA + row, xa);
      else st_rows<V>(dG + row, da);
    }
    if constexpr (EXT) {
      if (rbm && s < TT) {
        // publish [0, 0, dn, 0], contract it: d(rh) = W_hn^T dn
        step_arrive(ctr_out, skip, s, 1);
        if (!step_exchange(P, &tmA, &tmA4, ring, recv, bars, tmem, g, dir * K4 + ks * P.Kc, t * B + b0, t * B + b0,
                           ks * P.nsub, dir, idesc, adesc0, true, ctr_in, static_cast<unsigned int>(2 * s + 1) * P.nrg,
                           2 * s + 1, ks, n_mma, w_waited, K_BWD_TC, NoDeferred(), gkg)) {
          aborted = true;
          break;
        }
        check_slice(P, ring, Bn, K_BWD_TC, s);
        // phase B: dr; dG = [dr, dz, dn, 0]; the carry to the step before
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const int rl = rl0 + q * RPT;
          if (rl >= Bn) break;
          const int b = b0 + rl;
          const uint32_t ra = recv_s + recv_off(P, 2 * s + 1) + static_cast<uint32_t>((rl * RPC + ul0) * 4);
          float v[KS][V];
#pragma unroll
          for (int r = 0; r < KS; ++r) lds_v<V>(ra + r * src_bytes, v[r]);
          const bool live = t < lenq[q];
          float da[V][4];
#pragma unroll
          for (int jj = 0; jj < V; ++jj) {
            const int p = q * V + jj;
            float drh = 0.f;
#pragma unroll
            for (int r = 0; r < KS; ++r) drh += v[r][jj];
            float gv[4];
            unpack4(make_uint2(gw[q][2 * jj], gw[q][2 * jj + 1]), gv);
            const float r = gv[0], z = gv[1];
            const float dr = live ? drh * e0[p] * r * (1.f - r) : 0.f;
            da[jj][0] = dr; da[jj][1] = dzv[p]; da[jj][2] = dnv[p]; da[jj][3] = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) db[p][c] += da[jj][c];
            carry[p] = live ? dhv[p] * z + drh * (r - 1.f) : dhv[p];
          }
          st_rows<V>(dG + (static_cast<int64_t>(t) * B + b) * ldG + dir * K4 + 4 * u0, da);
        }
      }
    }
    RNN_TRACE_AT(5, 1, s);
    if (s < TT) step_arrive(ctr_out, skip, s, 1);
    RNN_TRACE_AT(6, 1, s);
  }

  if (!aborted) {
    // bias gradients: reduce each unit's four sums over the batch (reuses recv,
    // after every peer has finished with it), one unit slot j of the threads'
    // V units per pass.  Deterministic order throughout: each thread sums its
    // batch rows in order, then unit V w + j adds threads w, w + TPR, ... in
    // index order.
    tc_fence_before();
    if (KS > 1 && !P.gk) cluster_sync(); else __syncthreads();
    float* red = recv;
    // this batch part's sums to plane nb of db [NB][D][4H]; with several
    // parts, part 0 then adds planes 1.. in order once every CTA of the
    // direction has arrived once more
    float* plane = a.db + (static_cast<int64_t>(nb) * D + dir) * K4 + 4 * ubase;
#pragma unroll
    for (int jj = 0; jj < V; ++jj) {
      float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (rl0 + q * RPT >= Bn) break;
#pragma unroll
        for (int c = 0; c < 4; ++c) part[c] += db[q * V + jj][c];
      }
      if (jj > 0) __syncthreads();   // the previous pass's reads of red are done
#pragma unroll
      for (int c = 0; c < 4; ++c) red[threadIdx.x * 4 + c] = part[c];
      __syncthreads();
      for (int i = threadIdx.x; i < 4 * TPR; i += kThreads) {
        const int w = i >> 2, c = i & 3;
        float v = 0.f;
        for (int t2 = w; t2 < kThreads; t2 += TPR) v += red[t2 * 4 + c];
        plane[4 * (V * w + jj) + c] = v;
      }
    }
    if (P.NB > 1) {
      // every CTA of the direction arrives once on the direction's counter
      // after writing its plane; part 0 then sums the planes
      step_arrive(&a.dev->counters[a.dir0 + blockIdx.y], skip, TT, 1);
      if (nb == 0) {
        int ok = 1;
        if (threadIdx.x == 0) {
          ok = wait_counter_geq(&a.dev->counters[a.dir0 + blockIdx.y], P.nblk_dir, a.timeout_ns) ? 1 : 0;
          if (!ok) report_status(a.dev, 4u, K_BWD_TC, static_cast<unsigned>(TT), W_COUNTER);
        }
        if (__syncthreads_and(ok)) {
          for (int i = threadIdx.x; i < 4 * UPC; i += kThreads) {
            float v = __ldcg(plane + i);
            for (int q = 1; q < P.NB; ++q) v += __ldcg(a.db + (static_cast<int64_t>(q) * D + dir) * K4 + 4 * ubase + i);
            plane[i] = v;
          }
        }
      }
    }
  }
  teardown(P, bars);
}

}  // namespace

// Kernel entry points by template arguments (PP pairs per thread in 1, 2, 4, 8;
// K split KS in 1, 2, 4, 8, 16; ext = the extended variant), defined in
// persist_tc_fwd.cu / persist_tc_bwd.cu so the instances compile in parallel.
const void* persist_tc_fwd_kernel_ptr(int pp, int ks, int ext);
const void* persist_tc_bwd_kernel_ptr(int pp, int ks, int ext);

}  // namespace rnn
