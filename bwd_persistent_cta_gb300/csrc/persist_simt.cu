// persist_simt.cu - persistent recurrent kernels on fp32 FMA (SIMT).
//
// One launch runs every timestep of one layer (both directions when they fit
// together).  Each CTA owns NU hidden units of one direction and keeps their
// recurrent weights resident in shared memory for the whole sequence:
//   forward: the 4 gate rows W_hh[gate][u][0:H] of each owned unit;
//   backward: the column W_hh[:, u] of each owned unit over all 4H gate rows.
// Each step a CTA stages the full previous state (h_{t-1}, or the gate
// gradients of the step after) from L2 in chunks, forms its units'
// contractions, applies the cell (forward) or its derivative (backward) in
// registers, writes its slice, and arrives on a gpu-scope step counter.
// Before the next step every CTA waits - with a time limit - until all CTAs of
// its direction have arrived.  This is the persistent-RNN structure of the
// persistent RNN backward-data kernel page (one launch for all steps,
// register/shared-resident weights, a per-step exchange through global memory
// between CTAs), with acquire/release counters in place of its -0.0 sentinel
// polling.
//
// When the weights of the grid do not fit in shared memory (e.g. H = 2048), the
// kernels stream them instead: each step reads the owned rows / columns
// through the read-only data cache from L2 (the packed recurrent weights of a
// layer, at most 32 MiB in bf16, stay L2-resident across steps).
//
// These kernels serve the fp32 path (the 1e-5 bound needs fp32 FMA, not
// TF32), the plain RNN cells, the GRU reset-before backward (two dependent
// contractions per step: r/z, then W_hn(r*h)) and its forward below batch 4,
// and any shape the tensor-core kernels do not take.
//
// Cell math: the popnn Lstm.cpp page's forward cell step and backward step;
// the popnn Gru.cpp page's reset-before and resetAfter forward cell steps and
// backward steps; the LSTM and GRU branches of the persistent RNN
// backward-data kernel page.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace rnn {

namespace {

constexpr int kThreads = 256;

#ifdef RNN_STEP_TRACE
// Step-phase timestamps (globaltimer, ns) of CTA 0 and the last CTA of the
// latency-mode forward, for latency studies; compiled only with -DRNN_STEP_TRACE.
__device__ unsigned long long g_lat_trace[2][1100][8];
#define RNN_LAT_TRACE(slot_, step_)                                                              \
  do {                                                                                          \
    if (threadIdx.x == 0 && (blockIdx.x == 0 || blockIdx.x == gridDim.x - 1) && blockIdx.y == 0 && \
        (step_) < 1100)                                                                          \
      g_lat_trace[blockIdx.x == 0 ? 0 : 1][(step_)][(slot_)] = globaltimer_ns();                 \
  } while (0)
#else
#define RNN_LAT_TRACE(slot_, step_) do { } while (0)
#endif

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

template <typename T> __host__ __device__ inline int row_pad() { return sizeof(T) == 4 ? 1 : 2; }

__device__ __forceinline__ float ldcg_f(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float ldcg_f(const __nv_bfloat16* p) { return __bfloat162float(__ldcg(p)); }

// thread 0 waits on the counter; the outcome is shared with the whole CTA.
// A direction run by one CTA needs no counter: the block barrier orders its
// own global writes before its reads.
__device__ __forceinline__ bool cta_wait(const PersistArgs& a, const unsigned int* ctr, unsigned int target,
                                         unsigned int kernel, int step) {
  int ok = 1;
  if (threadIdx.x == 0 && gridDim.x > 1) {
    ok = wait_counter_geq(ctr, target, a.timeout_ns) ? 1 : 0;
    if (!ok) report_status(a.dev, 4u /* RNN_TIMEOUT */, kernel, static_cast<unsigned>(step), W_COUNTER);
  }
  return __syncthreads_and(ok) != 0;
}

// All stores of this phase by the CTA are ordered before the arrival (the
// barrier, then the release add).
__device__ __forceinline__ void cta_arrive(unsigned int* ctr, bool skip) {
  __syncthreads();
  if (threadIdx.x == 0 && !skip && gridDim.x > 1) red_release_gpu_add(ctr, 1u);
}

// The recurrent weights as seen by one CTA: resident in shared memory
// (row stride WS), or streamed from the packed global copy.
template <typename T, bool STREAM>
struct WView {
  const T* base;   // smem tile, or this direction's packed global matrix
  int NU, WS, u0, H;
  __device__ __forceinline__ const T* fwd_row(int s, int ul, int k0) const {
    return STREAM ? base + static_cast<size_t>(4 * (u0 + ul) + s) * H + k0 : base + (s * NU + ul) * WS + k0;
  }
  __device__ __forceinline__ const T* bwd_row(int ul, int k0) const {
    return STREAM ? base + static_cast<size_t>(u0 + ul) * 4 * H + k0 : base + ul * WS + k0;
  }
};
template <typename T, bool STREAM>
__device__ __forceinline__ float ldw(const T* p) {
  if (STREAM) return to_f<T>(__ldg(p));
  return to_f<T>(*p);
}

// acc[p][s] += sum_k W[s][ul][k] * src[b][k] over k in [0, K), slots in MASK.
// src row b starts at src + b * ld.
template <typename T, bool STREAM, int PP, int MASK>
__device__ __forceinline__ void contract_fwd(float (&acc)[PP][4], const WView<T, STREAM>& W, float* hs, int KC,
                                             const T* src, int64_t ld, int K, int B, int nu, int npairs) {
  const int HS = KC + 1;
  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    for (int idx = threadIdx.x; idx < B * kc; idx += kThreads) {
      const int b = idx / kc, kk = idx - b * kc;
      hs[b * HS + kk] = ldcg_f(src + b * ld + k0 + kk);
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      if (id >= npairs) break;
      const int ul = id % nu, b = id / nu;
      const float* hr = hs + b * HS;
      const T* w0 = W.fwd_row(0, ul, k0);
      const T* w1 = W.fwd_row(1, ul, k0);
      const T* w2 = W.fwd_row(2, ul, k0);
      const T* w3 = W.fwd_row(3, ul, k0);
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      for (int kk = 0; kk < kc; ++kk) {
        const float hv = hr[kk];
        if (MASK & 1) a0 = fmaf(ldw<T, STREAM>(w0 + kk), hv, a0);
        if (MASK & 2) a1 = fmaf(ldw<T, STREAM>(w1 + kk), hv, a1);
        if (MASK & 4) a2 = fmaf(ldw<T, STREAM>(w2 + kk), hv, a2);
        if (MASK & 8) a3 = fmaf(ldw<T, STREAM>(w3 + kk), hv, a3);
      }
      acc[p][0] += a0; acc[p][1] += a1; acc[p][2] += a2; acc[p][3] += a3;
    }
  }
}

// acc[p] += sum_k WT[ul][k] * src[b][k] over k in [0, K) with (k & 3) in MASK.
template <typename T, bool STREAM, int PP, int MASK>
__device__ __forceinline__ void contract_bwd(float (&acc)[PP], const WView<T, STREAM>& W, float* hs, int KC,
                                             const T* src, int64_t ld, int K, int B, int nu, int npairs) {
  const int HS = KC + 1;
  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    for (int idx = threadIdx.x; idx < B * kc; idx += kThreads) {
      const int b = idx / kc, kk = idx - b * kc;
      hs[b * HS + kk] = ldcg_f(src + b * ld + k0 + kk);
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      if (id >= npairs) break;
      const int ul = id % nu, b = id / nu;
      const float* hr = hs + b * HS;
      const T* w = W.bwd_row(ul, k0);
      float sacc = 0.f;
      if (MASK == 0xF) {
        for (int kk = 0; kk < kc; ++kk) sacc = fmaf(ldw<T, STREAM>(w + kk), hr[kk], sacc);
      } else {
        for (int kk = 0; kk < kc; ++kk)
          if ((MASK >> (kk & 3)) & 1) sacc = fmaf(ldw<T, STREAM>(w + kk), hr[kk], sacc);
      }
      acc[p] += sacc;
    }
  }
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <typename T, int PP, bool STREAM>
__global__ void __launch_bounds__(kThreads, 1) persist_fwd_simt_kernel(PersistArgs a, int NU, int KC) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int H = a.H, B = a.B, TT = a.T, D = a.D;
  const int dir = a.dir0 + blockIdx.y;
  const int u0 = blockIdx.x * NU;
  const int nu = min(NU, H - u0);
  const int WS = H + row_pad<T>();
  T* Ws = reinterpret_cast<T*>(smem);
  float* hs = reinterpret_cast<float*>(STREAM ? smem : smem + align16(static_cast<size_t>(4) * NU * WS * sizeof(T)));
  const bool lstm = a.mode == 0;
  const bool plain = a.mode >= 2;
  const bool rb = a.mode == 1 && !a.reset_after;
  const float clo = a.clip ? a.clip_lo : -INFINITY, chi = a.clip ? a.clip_hi : INFINITY;

  const T* Wr = static_cast<const T*>(a.Wr) + static_cast<size_t>(dir) * 4 * H * H;
  if (!STREAM) {
    for (int idx = threadIdx.x; idx < 4 * nu * H; idx += kThreads) {
      const int s = idx / (nu * H);
      const int rem = idx - s * nu * H;
      const int ul = rem / H, k = rem - ul * H;
      Ws[(s * NU + ul) * WS + k] = Wr[static_cast<size_t>(4 * (u0 + ul) + s) * H + k];
    }
  }
  const WView<T, STREAM> W{STREAM ? Wr : Ws, NU, WS, u0, H};

  T* Y = static_cast<T*>(a.Y);
  const T* P = static_cast<const T*>(a.P);
  T* G = static_cast<T*>(a.gates);
  T* RH = static_cast<T*>(a.RH);
  const int64_t ldY = static_cast<int64_t>(D) * H;
  const int64_t ldP = static_cast<int64_t>(D) * 4 * H;
  const int npairs = nu * B;
  float st[PP];      // LSTM: c_{t-1}; GRU: h_{t-1} (fp32 copy)
  float hl[PP];      // LSTM: h_{t-1}, held over masked steps
  int lenp[PP];      // valid steps of the pair's sequence (later steps are masked)
  float zr[PP][2];   // GRU reset-before: r, z between the two phases
  const int slot_h0 = dir ? TT + 1 : 0;
#pragma unroll
  for (int p = 0; p < PP; ++p) {
    st[p] = hl[p] = 0.f;
    lenp[p] = TT;
    zr[p][0] = zr[p][1] = 0.f;
    const int id = threadIdx.x + p * kThreads;
    if (id >= npairs) continue;
    const int ul = id % nu, b = id / nu, u = u0 + ul;
    if (a.len) lenp[p] = a.len[b];
    const float h0 = to_f<T>(Y[(static_cast<int64_t>(slot_h0) * B + b) * ldY + dir * H + u]);
    if (lstm) {
      const T* c0 = static_cast<const T*>(a.c0);
      st[p] = c0 ? to_f<T>(c0[(static_cast<int64_t>(dir) * B + b) * H + u]) : 0.f;
      hl[p] = h0;
      if (a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? TT : 0)) * B + b) * H + u] = st[p];
    } else {
      st[p] = h0;
    }
  }

  unsigned int* ctr = &a.dev->counters[dir];
  const unsigned int nblk = gridDim.x;
  const bool skip = a.skip_cta == static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);
  unsigned int phases = 0;

  for (int s = 0; s < TT; ++s) {
    const int t = dir ? TT - 1 - s : s;
    const int sp = dir ? t + 2 : t;     // Y slot of h_{t-1}
    const int so = t + 1;               // Y slot of h_t
    if (phases > 0 && !cta_wait(a, ctr, phases * nblk, K_FWD_SIMT, s)) return;
    float acc[PP][4];
#pragma unroll
    for (int p = 0; p < PP; ++p) acc[p][0] = acc[p][1] = acc[p][2] = acc[p][3] = 0.f;
    const T* hsrc = Y + static_cast<int64_t>(sp) * B * ldY + dir * H;
    if (rb)
      contract_fwd<T, STREAM, PP, 0x3>(acc, W, hs, KC, hsrc, ldY, H, B, nu, npairs);
    else if (lstm)
      contract_fwd<T, STREAM, PP, 0xF>(acc, W, hs, KC, hsrc, ldY, H, B, nu, npairs);
    else if (plain)
      contract_fwd<T, STREAM, PP, 0x1>(acc, W, hs, KC, hsrc, ldY, H, B, nu, npairs);
    else
      contract_fwd<T, STREAM, PP, 0x7>(acc, W, hs, KC, hsrc, ldY, H, B, nu, npairs);

    if (rb) {
      // phase 1: r, z and the reset state r * h_{t-1}
#pragma unroll
      for (int p = 0; p < PP; ++p) {
        const int id = threadIdx.x + p * kThreads;
        if (id >= npairs) break;
        const int ul = id % nu, b = id / nu, u = u0 + ul;
        float pv[4];
        Vec4<T>::load(P + (static_cast<int64_t>(t) * B + b) * ldP + dir * 4 * H + 4 * u, pv);
        const float r = sigm(pv[0] + acc[p][0]);
        const float z = sigm(pv[1] + acc[p][1]);
        zr[p][0] = r;
        zr[p][1] = z;
        RH[((static_cast<int64_t>(dir) * TT + t) * B + b) * H + u] = from_f<T>(r * st[p]);
      }
      cta_arrive(ctr, skip);
      ++phases;
      if (!cta_wait(a, ctr, phases * nblk, K_FWD_SIMT, s)) return;
#pragma unroll
      for (int p = 0; p < PP; ++p) acc[p][2] = 0.f;
      const T* rsrc = RH + (static_cast<int64_t>(dir) * TT + t) * B * H;
      contract_fwd<T, STREAM, PP, 0x4>(acc, W, hs, KC, rsrc, H, H, B, nu, npairs);
    }

#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      if (id >= npairs) break;
      const int ul = id % nu, b = id / nu, u = u0 + ul;
      float pv[4];
      Vec4<T>::load(P + (static_cast<int64_t>(t) * B + b) * ldP + dir * 4 * H + 4 * u, pv);
      float gv[4];
      float h;
      const bool live = t < lenp[p];
      if (lstm) {
        const float i = sigm(pv[0] + acc[p][0]);
        const float f = sigm(pv[1] + acc[p][1]);
        const float g = tanhf(pv[2] + acc[p][2]);
        const float o = sigm(pv[3] + acc[p][3]);
        float c = f * clipv(st[p], clo, chi) + i * g;
        h = o * tanhf(clipv(c, clo, chi));
        if (!live) { c = st[p]; h = hl[p]; }
        st[p] = c;
        hl[p] = h;
        gv[0] = i; gv[1] = f; gv[2] = g; gv[3] = o;
        if (a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? t : t + 1)) * B + b) * H + u] = c;
        if (s == TT - 1 && a.cy)
          static_cast<T*>(a.cy)[(static_cast<int64_t>(dir) * B + b) * H + u] = from_f<T>(c);
      } else if (plain) {
        const float hn = plain_act(a.mode, pv[0] + acc[p][0]);
        h = live ? hn : st[p];
        st[p] = h;
        gv[0] = hn; gv[1] = gv[2] = gv[3] = 0.f;
      } else if (!rb) {
        const float* bh = a.bh + dir * 4 * H + 4 * u;
        const float r = sigm(pv[0] + acc[p][0] + bh[0]);
        const float z = sigm(pv[1] + acc[p][1] + bh[1]);
        const float hn = acc[p][2] + bh[2];
        const float n = tanhf(pv[2] + r * hn);
        h = live ? (1.f - z) * n + z * st[p] : st[p];
        st[p] = h;
        gv[0] = r; gv[1] = z; gv[2] = n; gv[3] = hn;
      } else {
        const float r = zr[p][0], z = zr[p][1];
        const float n = tanhf(pv[2] + acc[p][2]);
        h = live ? (1.f - z) * n + z * st[p] : st[p];
        st[p] = h;
        gv[0] = r; gv[1] = z; gv[2] = n; gv[3] = 0.f;
      }
      Y[(static_cast<int64_t>(so) * B + b) * ldY + dir * H + u] = from_f<T>(h);
      if (G) Vec4<T>::store(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * 4 * H + 4 * u, gv);
      if (s == TT - 1 && a.hy)
        static_cast<T*>(a.hy)[(static_cast<int64_t>(dir) * B + b) * H + u] = from_f<T>(h);
    }
    cta_arrive(ctr, skip);
    ++phases;
  }
}

// ---------------------------------------------------------------------------
// backward through time
// ---------------------------------------------------------------------------
// Floats of the staging tile hs (B rows of KC + 1), rounded up to 16 bytes.
__host__ __device__ inline int hs_floats(int B, int KC) { return (B * (KC + 1) + 3) & ~3; }

// Per-step work bounds for accumulating dW_hh inside the backward kernel.
// Anywhere (mode 2): NU * H * B <= kDwhhWork, at most 4 * kDwhhWork / 256 =
// 256 multiply-adds per thread.  By default (mode 1) only where the work
// hides behind the wait for the step exchange: each thread's share of the
// (unit, column) items times the batch at most kDwhhIters (measured on
// GB300: GRU resetAfter fp32 H128 B16, 1 x 16, and GRU reset-before bf16
// H128 B8, 1 x 8, gained 30 and 13 us per step; LSTM fp32 H256 B8, 4 x 8,
// lost 20 us).
constexpr int kDwhhWork = 16384;
constexpr int kDwhhIters = 16;

// 4-byte asynchronous global -> shared copy (completes at cp_async_wait_all)
__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gsrc) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Stages the step's second operand of the dW_hh accumulation into shared
// memory, vs[b][k] = h_{t-1}[b][k] (Y slot sp), and for the reset-before
// candidate vs[B + b][k] = (r * h_{t-1})[b][k] (RH), in 4-byte copies (H even
// for bf16) issued early in the step so that they land during the contraction.
template <typename T>
__device__ __forceinline__ void dwhh_stage(const PersistArgs& a, T* vs, int dir, int t, int sp, bool rb) {
  const int H = a.H, B = a.B;
  const int64_t ldY = static_cast<int64_t>(a.D) * H;
  constexpr int E = 4 / static_cast<int>(sizeof(T));
  const int HW = H / E;
  const T* hp = static_cast<const T*>(a.Y) + static_cast<int64_t>(sp) * B * ldY + dir * H;
  for (int i = threadIdx.x; i < B * HW; i += kThreads) {
    const int b = i / HW, kw = i - b * HW;
    cp_async_4(vs + b * H + kw * E, hp + b * ldY + kw * E);
  }
  if (rb) {
    const T* rh = static_cast<const T*>(a.RH) + (static_cast<int64_t>(dir) * a.T + t) * B * H;
    for (int i = threadIdx.x; i < B * HW; i += kThreads) cp_async_4(vs + B * H + i * E, rh + i * E);
  }
}

// dW_hh accumulation of one step (the weight update interleaved with the
// backward pass: the popnn Lstm.cpp and Gru.cpp pages accumulate the weight
// gradients inside the backward loop, their interleaved weight update).  The CTA's rows are
// its units' 4 gate slots, row j = 4 * ul + slot; for column k
//   acc[j][k] += sum_b dG_t[b][j] * v_b[k],
// v = h_{t-1}, or r * h_{t-1} for the reset-before candidate (both staged in
// vs).  Work items are (unit, column) pairs, k fastest, spread over all
// threads; a warp reads one unit's four gate gradients as a broadcast float4
// from dgs[b][4 * NU], and the four sums of an item stay in registers over
// the batch.
template <typename T>
__device__ __forceinline__ void dwhh_step(float* accs, const float* dgs, const T* vs, int NU, int nu, int H, int B,
                                          bool rb) {
  const int ld = 4 * NU;
  for (int item = threadIdx.x; item < nu * H; item += kThreads) {
    const int ul = item / H, k = item - ul * H;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll 4
    for (int b = 0; b < B; ++b) {
      const float4 g = *reinterpret_cast<const float4*>(dgs + b * ld + 4 * ul);
      const float v = to_f<T>(vs[b * H + k]);
      s0 = fmaf(g.x, v, s0);
      s1 = fmaf(g.y, v, s1);
      s2 = fmaf(g.z, rb ? to_f<T>(vs[(B + b) * H + k]) : v, s2);
      s3 = fmaf(g.w, v, s3);
    }
    float* acc = accs + 4 * ul * H + k;
    acc[0] += s0;
    acc[H] += s1;
    acc[2 * H] += s2;
    acc[3 * H] += s3;
  }
}

template <typename T, int PP, bool STREAM>
__global__ void __launch_bounds__(kThreads, 1) persist_bwd_simt_kernel(PersistArgs a, int NU, int KC) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int H = a.H, B = a.B, TT = a.T, D = a.D;
  const int dir = a.dir0 + blockIdx.y;
  const int u0 = blockIdx.x * NU;
  const int nu = min(NU, H - u0);
  const int K4 = 4 * H;
  const int WS = K4 + row_pad<T>();
  T* Ws = reinterpret_cast<T*>(smem);
  float* hs = reinterpret_cast<float*>(STREAM ? smem : smem + align16(static_cast<size_t>(NU) * WS * sizeof(T)));
  __shared__ float dbs[4 * 64];
  const bool lstm = a.mode == 0;
  const bool plain = a.mode >= 2;
  const bool rb = a.mode == 1 && !a.reset_after;
  const float clo = a.clip ? a.clip_lo : -INFINITY, chi = a.clip ? a.clip_hi : INFINITY;

  const T* WT = static_cast<const T*>(a.WrT) + static_cast<size_t>(dir) * H * K4;
  if (!STREAM) {
    for (int idx = threadIdx.x; idx < nu * K4; idx += kThreads) {
      const int ul = idx / K4, k = idx - ul * K4;
      Ws[ul * WS + k] = WT[static_cast<size_t>(u0 + ul) * K4 + k];
    }
  }
  const WView<T, STREAM> W{STREAM ? WT : Ws, NU, WS, u0, H};
  // interleaved dW_hh: accumulator [4 * NU][H] and the step's gate gradients
  // [B][4 * NU] after the staging tile
  const bool dw = a.dwhh != nullptr;
  float* accs = hs + hs_floats(B, KC);
  float* dgs = accs + 4 * NU * H;
  T* vs = reinterpret_cast<T*>(dgs + 4 * NU * B);
  if (dw)
    for (int i = threadIdx.x; i < 4 * nu * H; i += kThreads) accs[i] = 0.f;

  const T* Y = static_cast<const T*>(a.Y);
  const T* G = static_cast<const T*>(a.gates);
  T* dG = static_cast<T*>(a.dG);
  const int64_t ldY = static_cast<int64_t>(D) * H;
  const int64_t ldG = static_cast<int64_t>(D) * K4;
  const int npairs = nu * B;
  float carry[PP];     // LSTM dc_next; GRU resetAfter dh*z; reset-before d(rh)*r + dh*z
                       // (GRU: the whole state gradient over a masked step)
  float carry_h[PP];   // LSTM: dh passed over masked steps
  float dhv[PP];       // reset-before: dh_t (masked: the passed gradient) between its two phases
  int lenp[PP];
  float db[PP][4];
#pragma unroll
  for (int p = 0; p < PP; ++p) {
    carry[p] = carry_h[p] = 0.f;
    dhv[p] = 0.f;
    lenp[p] = TT;
    db[p][0] = db[p][1] = db[p][2] = db[p][3] = 0.f;
    const int id = threadIdx.x + p * kThreads;
    if (id >= npairs) continue;
    const int ul = id % nu, b = id / nu, u = u0 + ul;
    if (a.len) lenp[p] = a.len[b];
    if (lstm && a.dcT) carry[p] = to_f<T>(static_cast<const T*>(a.dcT)[(static_cast<int64_t>(dir) * B + b) * H + u]);
  }

  unsigned int* ctr = &a.dev->counters[dir];
  const unsigned int nblk = gridDim.x;
  const bool skip = a.skip_cta == static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);
  unsigned int phases = 0;

  for (int s = 0; s <= TT; ++s) {
    float dhr[PP];
#pragma unroll
    for (int p = 0; p < PP; ++p) dhr[p] = 0.f;
    if (dw && s == 0) dwhh_stage<T>(a, vs, dir, dir ? 0 : TT - 1, dir ? 2 : TT - 1, rb);
    if (s == 0) {
      if (a.dhT) {
#pragma unroll
        for (int p = 0; p < PP; ++p) {
          const int id = threadIdx.x + p * kThreads;
          if (id >= npairs) break;
          const int ul = id % nu, b = id / nu;
          dhr[p] = to_f<T>(static_cast<const T*>(a.dhT)[(static_cast<int64_t>(dir) * B + b) * H + u0 + ul]);
        }
      }
    } else {
      if (!cta_wait(a, ctr, phases * nblk, K_BWD_SIMT, s)) return;
      if (dw && s < TT) dwhh_stage<T>(a, vs, dir, dir ? s : TT - 1 - s, dir ? s + 2 : TT - 1 - s, rb);
      const int tp = dir ? s - 1 : TT - s;   // step processed just before
      const T* src = dG + static_cast<int64_t>(tp) * B * ldG + dir * K4;
      if (rb)
        contract_bwd<T, STREAM, PP, 0x3>(dhr, W, hs, KC, src, ldG, K4, B, nu, npairs);
      else if (plain)
        contract_bwd<T, STREAM, PP, 0x1>(dhr, W, hs, KC, src, ldG, K4, B, nu, npairs);
      else
        contract_bwd<T, STREAM, PP, 0xF>(dhr, W, hs, KC, src, ldG, K4, B, nu, npairs);
    }
    if (s == TT) {
#pragma unroll
      for (int p = 0; p < PP; ++p) {
        const int id = threadIdx.x + p * kThreads;
        if (id >= npairs) break;
        const int ul = id % nu, b = id / nu, u = u0 + ul;
        const int64_t o = (static_cast<int64_t>(dir) * B + b) * H + u;
        if (a.dh0) static_cast<T*>(a.dh0)[o] = from_f<T>(lstm ? dhr[p] + carry_h[p] : dhr[p] + carry[p]);
        if (lstm && a.dc0) static_cast<T*>(a.dc0)[o] = from_f<T>(carry[p]);
      }
      break;
    }
    const int t = dir ? s : TT - 1 - s;
    const int sp = dir ? t + 2 : t;          // Y slot of h_{t-1}
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      if (id >= npairs) break;
      const int ul = id % nu, b = id / nu, u = u0 + ul;
      float gv[4];
      Vec4<T>::load(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * K4 + 4 * u, gv);
      const float dy = a.dYi[(static_cast<int64_t>(t) * B + b) * ldY + dir * H + u];
      T* dg = dG + (static_cast<int64_t>(t) * B + b) * ldG + dir * K4 + 4 * u;
      const bool live = t < lenp[p];
      if (lstm) {
        const float gh = dhr[p] + carry_h[p];
        float da[4] = {0.f, 0.f, 0.f, 0.f};
        if (live) {
          const float i = gv[0], f = gv[1], g = gv[2], o = gv[3];
          const float* C = a.C + static_cast<int64_t>(dir) * (TT + 1) * B * H;
          const float c = C[(static_cast<int64_t>(dir ? t : t + 1) * B + b) * H + u];
          const float cp = C[(static_cast<int64_t>(dir ? t + 1 : t) * B + b) * H + u];
          const float dh = dy + gh;
          const float tc = tanhf(clipv(c, clo, chi));
          const float dc = dh * o * (1.f - tc * tc) * (a.clip ? dclipv(c, clo, chi) : 1.f) + carry[p];
          da[0] = dc * g * i * (1.f - i);
          da[1] = dc * clipv(cp, clo, chi) * f * (1.f - f);
          da[2] = dc * i * (1.f - g * g);
          da[3] = dh * tc * o * (1.f - o);
          carry[p] = dc * f * (a.clip ? dclipv(cp, clo, chi) : 1.f);
          carry_h[p] = 0.f;
        } else {
          carry_h[p] = gh;
        }
        Vec4<T>::store(dg, da);
        if (dw) *reinterpret_cast<float4*>(dgs + b * 4 * NU + 4 * ul) = make_float4(da[0], da[1], da[2], da[3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) db[p][q] += da[q];
      } else if (plain) {
        const float gh = dhr[p] + carry[p];
        float da[4] = {0.f, 0.f, 0.f, 0.f};
        if (live) {
          da[0] = (dy + gh) * plain_dact(a.mode, gv[0]);
          carry[p] = 0.f;
        } else {
          carry[p] = gh;
        }
        Vec4<T>::store(dg, da);
        if (dw) *reinterpret_cast<float4*>(dgs + b * 4 * NU + 4 * ul) = make_float4(da[0], 0.f, 0.f, 0.f);
        db[p][0] += da[0];
      } else if (!rb) {
        const float gh = dhr[p] + carry[p];
        float da[4] = {0.f, 0.f, 0.f, 0.f};
        if (live) {
          const float r = gv[0], z = gv[1], n = gv[2], hn = gv[3];
          const float hp = to_f<T>(Y[(static_cast<int64_t>(sp) * B + b) * ldY + dir * H + u]);
          const float dh = dy + gh;
          const float dn = dh * (1.f - z) * (1.f - n * n);
          const float dz = dh * (hp - n) * z * (1.f - z);
          const float dr = dn * hn * r * (1.f - r);
          da[0] = dr; da[1] = dz; da[2] = dn; da[3] = dn * r;
          carry[p] = dh * z;
        } else {
          carry[p] = gh;
        }
        Vec4<T>::store(dg, da);
        if (dw) *reinterpret_cast<float4*>(dgs + b * 4 * NU + 4 * ul) = make_float4(da[0], da[1], da[2], da[3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) db[p][q] += da[q];
      } else {
        // reset-before, phase A: dn, dz
        const float gh = dhr[p] + carry[p];
        float dn = 0.f, dz = 0.f;
        if (live) {
          const float z = gv[1], n = gv[2];
          const float hp = to_f<T>(Y[(static_cast<int64_t>(sp) * B + b) * ldY + dir * H + u]);
          const float dh = dy + gh;
          dn = dh * (1.f - z) * (1.f - n * n);
          dz = dh * (hp - n) * z * (1.f - z);
          dhv[p] = dh;
        } else {
          dhv[p] = gh;
        }
        dg[1] = from_f<T>(dz);
        dg[2] = from_f<T>(dn);
        dg[3] = from_f<T>(0.f);
        if (dw) {
          dgs[b * 4 * NU + 4 * ul + 1] = dz;
          dgs[b * 4 * NU + 4 * ul + 2] = dn;
          dgs[b * 4 * NU + 4 * ul + 3] = 0.f;
        }
        db[p][1] += dz;
        db[p][2] += dn;
      }
    }
    if (dw) cp_async_wait_all();
    cta_arrive(ctr, skip);
    ++phases;
    // the weight-gradient work of the step overlaps the wait for the other CTAs
    // (cta_arrive's barrier made dgs and vs complete; the next cta_wait's
    // barrier orders these reads before the next step's writes)
    if (dw && !rb) dwhh_step<T>(accs, dgs, vs, NU, nu, H, B, false);
    if (rb) {
      // phase B: d(rh) = W_hn^T dn, then dr
      if (!cta_wait(a, ctr, phases * nblk, K_BWD_SIMT, s)) return;
      float drh[PP];
#pragma unroll
      for (int p = 0; p < PP; ++p) drh[p] = 0.f;
      const T* src = dG + static_cast<int64_t>(t) * B * ldG + dir * K4;
      contract_bwd<T, STREAM, PP, 0x4>(drh, W, hs, KC, src, ldG, K4, B, nu, npairs);
#pragma unroll
      for (int p = 0; p < PP; ++p) {
        const int id = threadIdx.x + p * kThreads;
        if (id >= npairs) break;
        const int ul = id % nu, b = id / nu, u = u0 + ul;
        float gv[4];
        Vec4<T>::load(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * K4 + 4 * u, gv);
        const float r = gv[0], z = gv[1];
        const float hp = to_f<T>(Y[(static_cast<int64_t>(sp) * B + b) * ldY + dir * H + u]);
        const bool live = t < lenp[p];
        const float dr = live ? drh[p] * hp * r * (1.f - r) : 0.f;
        dG[(static_cast<int64_t>(t) * B + b) * ldG + dir * K4 + 4 * u] = from_f<T>(dr);
        if (dw) dgs[b * 4 * NU + 4 * ul] = dr;
        db[p][0] += dr;
        carry[p] = live ? drh[p] * r + dhv[p] * z : dhv[p];
      }
      cta_arrive(ctr, skip);
      ++phases;
      if (dw) dwhh_step<T>(accs, dgs, vs, NU, nu, H, B, true);
    }
  }

  // bias gradients: reduce each unit's four sums over the batch
  for (int base = 0; base < nu; base += 64) {
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * 64; i += kThreads) dbs[i] = 0.f;
    __syncthreads();
#pragma unroll
    for (int p = 0; p < PP; ++p) {
      const int id = threadIdx.x + p * kThreads;
      if (id >= npairs) break;
      const int ul = id % nu;
      if (ul < base || ul >= base + 64) continue;
#pragma unroll
      for (int q = 0; q < 4; ++q) atomicAdd(&dbs[(ul - base) * 4 + q], db[p][q]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * 64; i += kThreads) {
      const int ul = base + i / 4;
      if (ul < nu) a.db[static_cast<int64_t>(dir) * K4 + 4 * (u0 + ul) + (i & 3)] = dbs[i];
    }
  }

  // interleaved dW_hh: each row of the CTA to its caller gate block
  if (dw) {
    __syncthreads();
    const int G = lstm ? 4 : (plain ? 1 : 3);
    float* dst = a.dwhh + static_cast<int64_t>(dir) * G * H * H;
    for (int i = threadIdx.x; i < 4 * nu * H; i += kThreads) {
      const int j = i / H, k = i - j * H;
      const int m = a.whh_map[j & 3];
      if (m >= 0) dst[(static_cast<int64_t>(m) * H + u0 + (j >> 2)) * H + k] = accs[i];
    }
  }
}

// ---------------------------------------------------------------------------
// forward, large weights, small batch (latency mode)
// ---------------------------------------------------------------------------
// For layers whose recurrent weights do not fit the per-unit layout above
// (e.g. H = 2048) and batch <= 8.  Each CTA owns NU units; as many of their
// weight rows as fit stay resident in shared memory for the whole sequence,
// the remaining rows are streamed from L2 each step (read-only path).  Each
// warp owns rows r = warp, warp + 8, ...; its lanes split K in 16-byte
// vectors.  Per K vector a lane loads its slice of h_{t-1} for every batch
// column once (from shared memory, staged per step) and reuses it across its
// rows; the per-row partial sums are combined with warp shuffles.  At batch 8
// the step is FP32-issue bound, at batch 1 bound by the exchange.
constexpr int kLatRows = 8;    // max rows per warp (4 * NU <= 64)

template <typename T, int BB>
__device__ __forceinline__ void latency_rows(const T* Ws, int WSR, int Rs, const T* Wg, int H, const int* rowmap,
                                             int row0, int nrows, const T* hs, int B, float* out) {
  constexpr int VE = 16 / sizeof(T);           // elements per 16-byte vector
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = H / (32 * VE);
  float acc[kLatRows][BB];
#pragma unroll
  for (int j = 0; j < kLatRows; ++j)
#pragma unroll
    for (int b = 0; b < BB; ++b) acc[j][b] = 0.f;
  for (int v = 0; v < nv; ++v) {
    const int k = (v * 32 + lane) * VE;
    float hv[BB][VE];
#pragma unroll
    for (int b = 0; b < BB; ++b) {
      if (b < B) {
        const uint4 q = *reinterpret_cast<const uint4*>(hs + static_cast<size_t>(b) * H + k);
        if (sizeof(T) == 2) {
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
          for (int e = 0; e < VE / 2; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            hv[b][2 * e] = f.x; hv[b][2 * e + 1] = f.y;
          }
        } else {
          const float* f = reinterpret_cast<const float*>(&q);
#pragma unroll
          for (int e = 0; e < VE; ++e) hv[b][e] = f[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) hv[b][e] = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < kLatRows; ++j) {
      const int r = row0 + warp + 8 * j;
      if (r < nrows) {
        const uint4 q = r < Rs ? *reinterpret_cast<const uint4*>(Ws + static_cast<size_t>(r) * WSR + k)
                               : __ldg(reinterpret_cast<const uint4*>(Wg + static_cast<size_t>(rowmap[r]) * H + k));
        float w[VE];
        if (sizeof(T) == 2) {
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
          for (int e = 0; e < VE / 2; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            w[2 * e] = f.x; w[2 * e + 1] = f.y;
          }
        } else {
          const float* f = reinterpret_cast<const float*>(&q);
#pragma unroll
          for (int e = 0; e < VE; ++e) w[e] = f[e];
        }
#pragma unroll
        for (int b = 0; b < BB; ++b)
#pragma unroll
          for (int e = 0; e < VE; ++e) acc[j][b] = fmaf(w[e], hv[b][e], acc[j][b]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kLatRows; ++j) {
    const int r = row0 + warp + 8 * j;
#pragma unroll
    for (int b = 0; b < BB; ++b) {
      float x = acc[j][b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == 0 && r < nrows && b < B) out[r * BB + b] = x;
    }
  }
}

// B rows of a state (storage type, row stride ld) -> hs[b][k] in shared memory.
template <typename T>
__device__ __forceinline__ void stage_state(const T* src, int64_t ld, int H, int B, T* hs) {
  constexpr int VE = 16 / sizeof(T);
  const int per_row = H / VE;
  for (int i = threadIdx.x; i < B * per_row; i += kThreads) {
    const int b = i / per_row, c = i - b * per_row;
    const uint4 q = __ldcg(reinterpret_cast<const uint4*>(src + b * ld) + c);
    *reinterpret_cast<uint4*>(hs + static_cast<size_t>(b) * H + c * VE) = q;
  }
}

template <typename T, int BB>
__global__ void __launch_bounds__(kThreads, 1) persist_fwd_latency_kernel(PersistArgs a, int NU, int Rs) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int H = a.H, B = a.B, TT = a.T, D = a.D;
  const int dir = a.dir0 + blockIdx.y;
  const int u0 = blockIdx.x * NU;
  const int nu = min(NU, H - u0);
  const bool lstm = a.mode == 0;
  const bool plain = a.mode >= 2;
  const bool rb = a.mode == 1 && !a.reset_after;
  const int na = lstm ? 4 : (rb ? 2 : (plain ? 1 : 3));     // phase-A rows per unit
  const float clo = a.clip ? a.clip_lo : -INFINITY, chi = a.clip ? a.clip_hi : INFINITY;
  const int WSR = H + 16 / static_cast<int>(sizeof(T));   // resident row stride (16-byte aligned)
  T* hs = reinterpret_cast<T*>(smem);                                   // [BB][H]
  float* out = reinterpret_cast<float*>(smem + static_cast<size_t>(BB) * H * sizeof(T));   // [4*NU][BB]
  int* rows = reinterpret_cast<int*>(out + 4 * NU * BB);                // local row -> packed row
  T* Ws = reinterpret_cast<T*>(rows + 4 * NU);                          // [Rs][WSR]
  int nA = 0, nAB = 0;
  {
    // phase A rows: LSTM i,f,g,o; GRU resetAfter r,z,n; reset-before r,z.  Phase B (reset-before): n.
    for (int ul = 0; ul < nu; ++ul)
      for (int sl = 0; sl < na; ++sl) {
        if (threadIdx.x == 0) rows[nA] = 4 * (u0 + ul) + sl;
        ++nA;
      }
    nAB = nA;
    if (rb)
      for (int ul = 0; ul < nu; ++ul) {
        if (threadIdx.x == 0) rows[nAB] = 4 * (u0 + ul) + 2;
        ++nAB;
      }
  }
  __syncthreads();
  const T* Wr = static_cast<const T*>(a.Wr) + static_cast<size_t>(dir) * 4 * H * H;
  const int rs = min(Rs, nAB);
  {
    constexpr int VE = 16 / sizeof(T);
    const int per_row = H / VE;
    for (int i = threadIdx.x; i < rs * per_row; i += kThreads) {
      const int r = i / per_row, c = i - r * per_row;
      *reinterpret_cast<uint4*>(Ws + static_cast<size_t>(r) * WSR + c * VE) =
          __ldg(reinterpret_cast<const uint4*>(Wr + static_cast<size_t>(rows[r]) * H) + c);
    }
  }

  T* Y = static_cast<T*>(a.Y);
  const T* P = static_cast<const T*>(a.P);
  T* G = static_cast<T*>(a.gates);
  T* RH = static_cast<T*>(a.RH);
  const int64_t ldY = static_cast<int64_t>(D) * H;
  const int64_t ldP = static_cast<int64_t>(D) * 4 * H;
  const int npairs = nu * B;          // <= kThreads: one pair per thread
  const int id = threadIdx.x;
  const bool has = id < npairs;
  const int ul = has ? id % nu : 0, b = has ? id / nu : 0, u = u0 + ul;
  const int slot_h0 = dir ? TT + 1 : 0;
  float st = 0.f;     // LSTM: c_{t-1}; GRU: h_{t-1}
  float hl = 0.f;     // LSTM: h_{t-1}, held over masked steps
  int lenb = TT;      // valid steps of the pair's sequence
  if (has) {
    if (a.len) lenb = a.len[b];
    const float h0 = to_f<T>(Y[(static_cast<int64_t>(slot_h0) * B + b) * ldY + dir * H + u]);
    if (lstm) {
      const T* c0 = static_cast<const T*>(a.c0);
      st = c0 ? to_f<T>(c0[(static_cast<int64_t>(dir) * B + b) * H + u]) : 0.f;
      hl = h0;
      if (a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? TT : 0)) * B + b) * H + u] = st;
    } else {
      st = h0;
    }
  }
  unsigned int* ctr = &a.dev->counters[dir];
  const unsigned int nblk = gridDim.x;
  const bool skip = a.skip_cta == static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);
  unsigned int phases = 0;

  for (int s = 0; s < TT; ++s) {
    const int t = dir ? TT - 1 - s : s;
    const int sp = dir ? t + 2 : t;
    float pv[4] = {0.f, 0.f, 0.f, 0.f};
    RNN_LAT_TRACE(0, s);
    if (has) Vec4<T>::load(P + (static_cast<int64_t>(t) * B + b) * ldP + dir * 4 * H + 4 * u, pv);
    if (phases > 0 && !cta_wait(a, ctr, phases * nblk, K_FWD_SIMT, s)) return;
    RNN_LAT_TRACE(1, s);
    stage_state<T>(Y + static_cast<int64_t>(sp) * B * ldY + dir * H, ldY, H, B, hs);
    __syncthreads();
    RNN_LAT_TRACE(2, s);
    latency_rows<T, BB>(Ws, WSR, rs, Wr, H, rows, 0, nA, hs, B, out);
    __syncthreads();
    RNN_LAT_TRACE(3, s);
    float gv[4] = {0.f, 0.f, 0.f, 0.f}, h = 0.f;
    float r = 0.f, z = 0.f;
    if (has) {
      const float* o = out + (ul * na) * BB + b;   // this unit's rows in phase-A order
      if (lstm) {
        const float i = sigm(pv[0] + o[0]);
        const float f = sigm(pv[1] + o[BB]);
        const float g = tanhf(pv[2] + o[2 * BB]);
        const float oo = sigm(pv[3] + o[3 * BB]);
        float c = f * clipv(st, clo, chi) + i * g;
        h = oo * tanhf(clipv(c, clo, chi));
        if (t >= lenb) { c = st; h = hl; }
        st = c;
        hl = h;
        gv[0] = i; gv[1] = f; gv[2] = g; gv[3] = oo;
      } else if (plain) {
        const float hn = plain_act(a.mode, pv[0] + o[0]);
        h = t < lenb ? hn : st;
        gv[0] = hn;
      } else if (!rb) {
        const float* bh = a.bh + dir * 4 * H + 4 * u;
        r = sigm(pv[0] + o[0] + bh[0]);
        z = sigm(pv[1] + o[BB] + bh[1]);
        const float hn = o[2 * BB] + bh[2];
        const float n = tanhf(pv[2] + r * hn);
        h = t < lenb ? (1.f - z) * n + z * st : st;
        gv[0] = r; gv[1] = z; gv[2] = n; gv[3] = hn;
      } else {
        r = sigm(pv[0] + o[0]);
        z = sigm(pv[1] + o[BB]);
        RH[((static_cast<int64_t>(dir) * TT + t) * B + b) * H + u] = from_f<T>(r * st);
      }
    }
    if (rb) {
      cta_arrive(ctr, skip);
      ++phases;
      if (!cta_wait(a, ctr, phases * nblk, K_FWD_SIMT, s)) return;
      stage_state<T>(RH + (static_cast<int64_t>(dir) * TT + t) * B * H, H, H, B, hs);
      __syncthreads();
      latency_rows<T, BB>(Ws, WSR, rs, Wr, H, rows, nA, nAB, hs, B, out);
      __syncthreads();
      if (has) {
        const float n = tanhf(pv[2] + out[(nA + ul) * BB + b]);
        h = t < lenb ? (1.f - z) * n + z * st : st;
        gv[0] = r; gv[1] = z; gv[2] = n; gv[3] = 0.f;
      }
    }
    if (has) {
      if (!lstm) st = h;
      Y[(static_cast<int64_t>(t + 1) * B + b) * ldY + dir * H + u] = from_f<T>(h);
    }
    RNN_LAT_TRACE(4, s);
    cta_arrive(ctr, skip);
    RNN_LAT_TRACE(5, s);
    ++phases;
    if (has) {
      if (G) Vec4<T>::store(G + ((static_cast<int64_t>(dir) * TT + t) * B + b) * 4 * H + 4 * u, gv);
      if (lstm && a.C) a.C[((static_cast<int64_t>(dir) * (TT + 1) + (dir ? t : t + 1)) * B + b) * H + u] = st;
      if (s == TT - 1) {
        const int64_t o = (static_cast<int64_t>(dir) * B + b) * H + u;
        if (a.hy) static_cast<T*>(a.hy)[o] = from_f<T>(h);
        if (lstm && a.cy) static_cast<T*>(a.cy)[o] = from_f<T>(st);
      }
    }
  }
}

template <typename T, bool STREAM>
struct SimtKernels {
  static const void* fwd(int pp) {
    switch (pp) {
      case 1: return reinterpret_cast<const void*>(&persist_fwd_simt_kernel<T, 1, STREAM>);
      case 2: return reinterpret_cast<const void*>(&persist_fwd_simt_kernel<T, 2, STREAM>);
      case 4: return reinterpret_cast<const void*>(&persist_fwd_simt_kernel<T, 4, STREAM>);
      default: return reinterpret_cast<const void*>(&persist_fwd_simt_kernel<T, 8, STREAM>);
    }
  }
  static const void* bwd(int pp) {
    switch (pp) {
      case 1: return reinterpret_cast<const void*>(&persist_bwd_simt_kernel<T, 1, STREAM>);
      case 2: return reinterpret_cast<const void*>(&persist_bwd_simt_kernel<T, 2, STREAM>);
      case 4: return reinterpret_cast<const void*>(&persist_bwd_simt_kernel<T, 4, STREAM>);
      default: return reinterpret_cast<const void*>(&persist_bwd_simt_kernel<T, 8, STREAM>);
    }
  }
};

struct SimtPlan {
  int NU = 0, nblk = 0, KC = 0, PP = 0;
  bool stream = false;
  size_t smem = 0;
};

int pp_for(int pairs) {
  const int need = (pairs + kThreads - 1) / kThreads;
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 8 ? 8 : 0;
}

const void* kernel_for(const PersistArgs& a, bool bwd, const SimtPlan& pl) {
  if (a.is_bf16)
    return pl.stream ? (bwd ? SimtKernels<__nv_bfloat16, true>::bwd(pl.PP) : SimtKernels<__nv_bfloat16, true>::fwd(pl.PP))
                     : (bwd ? SimtKernels<__nv_bfloat16, false>::bwd(pl.PP) : SimtKernels<__nv_bfloat16, false>::fwd(pl.PP));
  return pl.stream ? (bwd ? SimtKernels<float, true>::bwd(pl.PP) : SimtKernels<float, true>::fwd(pl.PP))
                   : (bwd ? SimtKernels<float, false>::bwd(pl.PP) : SimtKernels<float, false>::fwd(pl.PP));
}

// Pick units per CTA: minimise an estimated step time (a fixed cost for the
// cross-CTA exchange when there is more than one CTA, plus the per-thread FMA
// count) subject to shared memory, registers and co-residency of the grid.
// The exchange weight (500 serial FMAs per thread) is from GB300 timings: a
// step exchange costs about 2-3 us, one serial FMA per thread (weights and
// state from shared memory) about 6 ns; e.g. GRU reset-before bf16, H = 128,
// batch 8: one CTA with 4 pairs per thread took 30 us per backward step,
// 8 CTAs with one pair each 12 us.
// Without a resident fit, stream the weights and spread them over the most
// CTAs that fit (more read bandwidth).
int make_plan(const PersistArgs& a, bool bwd, int num_sms, SimtPlan* out) {
  const int H = a.H, B = a.B;
  const size_t es = a.is_bf16 ? 2 : 4;
  const size_t smem_cap = 200 * 1024;
  int KC = (8192 / B) - 1;
  KC = (KC / 4) * 4;
  if (KC < 4) return 2;
  const int Kmax = bwd ? 4 * H : H;
  if (KC > Kmax) KC = (Kmax + 3) / 4 * 4;
  const size_t hs_bytes = static_cast<size_t>(B) * (KC + 1) * 4;
  const bool dw = bwd && a.dwhh != nullptr;
  double best = 1e300;
  SimtPlan bp;
  for (int NU = 1; NU <= H; ++NU) {
    const int nblk = (H + NU - 1) / NU;
    if (nblk * a.ndir > num_sms) continue;
    const int pp = pp_for(NU * B);
    if (pp == 0) break;
    if (dw && (static_cast<int64_t>(NU) * H * B > kDwhhWork || (a.is_bf16 && (H & 1)))) break;
    const size_t wbytes = bwd ? static_cast<size_t>(NU) * (4 * H + (a.is_bf16 ? 2 : 1)) * es
                              : static_cast<size_t>(4) * NU * (H + (a.is_bf16 ? 2 : 1)) * es;
    // interleaved dW_hh: accumulator [4 NU][H] and gate gradients [B][4 NU],
    // fp32, then the staged h_{t-1} (and r * h_{t-1}) tiles [B][H]
    const bool rb = a.mode == 1 && !a.reset_after;
    const size_t smem = dw ? align16(wbytes) + static_cast<size_t>(hs_floats(B, KC)) * 4 +
                                 static_cast<size_t>(4) * NU * (H + B) * 4 +
                                 static_cast<size_t>(rb ? 2 : 1) * B * H * es
                           : align16(wbytes) + hs_bytes;
    if (smem > smem_cap) break;
    const double cost = (nblk > 1 ? 500.0 : 0.0) + static_cast<double>(pp) * 4.0 * H +
                        static_cast<double>(B) * (bwd ? 4 * H : H) / kThreads;
    if (cost < best) {
      best = cost;
      bp.NU = NU; bp.nblk = nblk; bp.KC = KC; bp.PP = pp; bp.smem = smem; bp.stream = false;
    }
  }
  if (bp.NU == 0) {
    if (dw) return 2;   // streamed weights: no interleaved dW_hh
    const int max_ctas = num_sms / a.ndir;
    if (max_ctas < 1) return 2;
    const int NU = (H + max_ctas - 1) / max_ctas;
    const int pp = pp_for(NU * B);
    if (pp == 0) return 2;
    bp.NU = NU; bp.nblk = (H + NU - 1) / NU; bp.KC = KC; bp.PP = pp; bp.smem = hs_bytes; bp.stream = true;
  }
  *out = bp;
  return 0;
}

const void* latency_fwd_fn(const PersistArgs& a) {
  const int bb = a.B <= 1 ? 1 : a.B <= 2 ? 2 : a.B <= 4 ? 4 : 8;
  if (a.is_bf16) {
    switch (bb) {
      case 1: return reinterpret_cast<const void*>(&persist_fwd_latency_kernel<__nv_bfloat16, 1>);
      case 2: return reinterpret_cast<const void*>(&persist_fwd_latency_kernel<__nv_bfloat16, 2>);
      case 4: return reinterpret_cast<const void*>(&persist_fwd_latency_kernel<__nv_bfloat16, 4>);
      default: return reinterpret_cast<const void*>(&persist_fwd_latency_kernel<__nv_bfloat16, 8>);
    }
  }
  switch (bb) {
    case 1: return reinterpret_cast<const void*>(&persist_fwd_latency_kernel<float, 1>);
    case 2: return reinterpret_cast<const void*>(&persist_fwd_latency_kernel<float, 2>);
    case 4: return reinterpret_cast<const void*>(&persist_fwd_latency_kernel<float, 4>);
    default: return reinterpret_cast<const void*>(&persist_fwd_latency_kernel<float, 8>);
  }
}

// Host-side plan cache: the occupancy queries behind a launch cost host time
// that the GPU would wait for at every persistent launch.  Dynamic shared
// memory limits only ever rise, so a cached plan never meets a lower limit set
// for another shape.
struct SimtKey {
  int v[11];
  bool operator<(const SimtKey& o) const { return std::lexicographical_compare(v, v + 11, o.v, o.v + 11); }
};
struct SimtEntry {
  int rc = 0;
  SimtPlan pl;
  int lat = 0;          // latency-mode forward chosen
  int lat_NU = 0, lat_Rs = 0, lat_nblk = 0;
  size_t lat_smem = 0;
};
std::mutex g_simt_mu;
std::map<SimtKey, SimtEntry> g_simt;
std::map<std::pair<const void*, int>, int> g_simt_smem;

bool raise_smem(const void* fn, int dev, size_t bytes) {
  int& cur = g_simt_smem[{fn, dev}];
  if (static_cast<int>(bytes) <= cur) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cur = static_cast<int>(bytes);
  return true;
}

// Latency-mode forward (large weights, batch <= 8): one pair per thread, as
// many weight rows resident in shared memory as fit.  Plans only (0, or 2 when
// it does not apply); the caller launches.
int plan_latency_fwd(const PersistArgs& a, int num_sms, int dev, SimtEntry* e) {
  const int max_ctas = num_sms / a.ndir;
  const int NU = (a.H + max_ctas - 1) / max_ctas;
  if (NU * a.B > kThreads || 4 * NU > 8 * kLatRows) return 2;
  const int nblk = (a.H + NU - 1) / NU;
  const int bb = a.B <= 1 ? 1 : a.B <= 2 ? 2 : a.B <= 4 ? 4 : 8;
  const size_t es = a.is_bf16 ? 2 : 4;
  const size_t fixed = static_cast<size_t>(bb) * a.H * es + static_cast<size_t>(4) * NU * bb * 4 + 4 * NU * 4;
  const size_t row_bytes = (static_cast<size_t>(a.H) + 16 / es) * es;
  const size_t cap = 220 * 1024;
  if (fixed > cap) return 2;
  int Rs = static_cast<int>((cap - fixed) / row_bytes);
  if (Rs > 4 * NU) Rs = 4 * NU;
  const size_t smem = fixed + static_cast<size_t>(Rs) * row_bytes;
  const void* fn = latency_fwd_fn(a);
  if (!raise_smem(fn, dev, smem)) return 3;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem) != cudaSuccess) return 3;
  if (per_sm * num_sms < nblk * a.ndir) return 2;
  e->lat = 1;
  e->lat_NU = NU; e->lat_Rs = Rs; e->lat_nblk = nblk; e->lat_smem = smem;
  return 0;
}

// RNN_TRACE=1: one stderr line per launch shape, when its plan is chosen.
void trace_entry(const PersistArgs& a, bool bwd, const SimtEntry& e) {
  const char* env = std::getenv("RNN_TRACE");
  if (!env || env[0] != '1') return;
  const char* pass = bwd ? "backward" : "forward";
  if (e.rc) {
    std::fprintf(stderr, "[rnn] SIMT %s H=%d B=%d dirs=%d: no plan fits\n", pass, a.H, a.B, a.ndir);
  } else if (e.lat) {
    std::fprintf(stderr,
                 "[rnn] SIMT %s H=%d B=%d dirs=%d: latency mode, %d CTAs of %d units, %d weight rows resident, "
                 "%zu B shared memory\n",
                 pass, a.H, a.B, a.ndir, e.lat_nblk * a.ndir, e.lat_NU, e.lat_Rs, e.lat_smem);
  } else {
    std::fprintf(stderr,
                 "[rnn] SIMT %s H=%d B=%d dirs=%d: %d CTAs of %d units, %d pair(s) per thread, weights %s, "
                 "%zu B shared memory%s\n",
                 pass, a.H, a.B, a.ndir, e.pl.nblk * a.ndir, e.pl.NU, e.pl.PP,
                 e.pl.stream ? "streamed from L2" : "resident", e.pl.smem,
                 a.dwhh ? ", dW_hh accumulated per step" : "");
  }
}

// The plan of one launch (cached per shape and device).
SimtEntry simt_entry(const PersistArgs& a, bool bwd, int num_sms) {
  int dev = 0;
  cudaGetDevice(&dev);
  const SimtKey key{{bwd ? 1 : 0, a.mode, a.reset_after, a.is_bf16, a.H, a.B, a.ndir, a.dwhh ? 1 : 0, num_sms, dev,
                     a.D}};
  std::lock_guard<std::mutex> lock(g_simt_mu);
  const auto hit = g_simt.find(key);
  if (hit != g_simt.end()) return hit->second;
  SimtEntry e;
  e.rc = make_plan(a, bwd, num_sms, &e.pl);
  if (e.rc == 0) {
    const int span = 32 * (a.is_bf16 ? 8 : 4);
    int lrc = 2;
    if (e.pl.stream && !bwd && a.B <= 8 && a.H % span == 0) lrc = plan_latency_fwd(a, num_sms, dev, &e);
    if (lrc == 3) {
      e.rc = 3;
    } else if (!e.lat) {
      const void* fn = kernel_for(a, bwd, e.pl);
      int per_sm = 0;
      if (!raise_smem(fn, dev, e.pl.smem) ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, e.pl.smem) != cudaSuccess)
        e.rc = 3;
      else if (per_sm * num_sms < e.pl.nblk * a.ndir)
        e.rc = 2;
    }
  }
  if (e.rc != 3) {   // a CUDA error is not cached
    g_simt[key] = e;
    trace_entry(a, bwd, e);
  }
  return e;
}

int launch_simt(const PersistArgs& a, bool bwd, cudaStream_t s, int num_sms) {
  const SimtEntry e = simt_entry(a, bwd, num_sms);
  if (e.rc) return e.rc;
  if (e.lat) {
    PersistArgs args = a;
    int nu = e.lat_NU, rs = e.lat_Rs;
    void* params[] = {&args, &nu, &rs};
    if (cudaLaunchKernel(latency_fwd_fn(a), dim3(e.lat_nblk, a.ndir), dim3(kThreads), params, e.lat_smem, s) !=
        cudaSuccess)
      return 3;
    return 0;
  }
  const SimtPlan& pl = e.pl;
  const void* fn = kernel_for(a, bwd, pl);
  dim3 grid(pl.nblk, a.ndir);
  PersistArgs args = a;
  int NU = pl.NU, KC = pl.KC;
  void* params[] = {&args, &NU, &KC};
  if (cudaLaunchKernel(fn, grid, dim3(kThreads), params, pl.smem, s) != cudaSuccess) return 3;
  return 0;
}

}  // namespace

#ifdef RNN_STEP_TRACE
extern "C" int rnn_debug_read_lat_trace(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, g_lat_trace, bytes) == cudaSuccess ? 0 : 3;
}
#endif

int plan_persist_simt(const PersistArgs& a, int num_sms, int* nblk, size_t* smem) {
  SimtPlan pf, pb;
  int rc = make_plan(a, false, num_sms, &pf);
  if (rc) return rc;
  rc = make_plan(a, true, num_sms, &pb);
  if (rc) return rc;
  if (nblk) *nblk = pf.nblk > pb.nblk ? pf.nblk : pb.nblk;
  if (smem) *smem = pf.smem > pb.smem ? pf.smem : pb.smem;
  return 0;
}

// hidden_only (mode 1): the backward kernel's own plan must stay as without
// the accumulation, span several CTAs per direction (a lone CTA has no wait
// to hide the work behind: LSTM fp32 T16 B4 H32 measured +20 us in the
// backward kernel against 10 us for the dW_hh GEMM) and give each thread at
// most kDwhhIters item-batch iterations per step.  The launch tries both
// directions at once first, then one at a time.
bool persist_simt_dwhh_ok(const PersistArgs& a, int num_sms, bool hidden_only) {
  PersistArgs b = a;
  float probe = 0.f;
  for (int nd : {a.D, 1}) {
    b.ndir = nd;
    SimtPlan nat, dwp;
    b.dwhh = nullptr;
    const int rn = make_plan(b, true, num_sms, &nat);
    b.dwhh = &probe;   // only tested for null by the planner
    const int rd = make_plan(b, true, num_sms, &dwp);
    if (!hidden_only) {
      if (rd == 0) return true;
      continue;
    }
    if (rn != 0) continue;
    return rd == 0 && dwp.NU == nat.NU && nat.nblk > 1 && !nat.stream &&
           (nat.NU * a.H + kThreads - 1) / kThreads * a.B <= kDwhhIters;
  }
  return false;
}

extern "C" int rnn_debug_simt_plan(int mode, int reset_after, int is_bf16, int bwd, int hidden, int batch,
                                   int ndir, int num_sms, int dwhh, int* out) {
  if (!out) return 0;
  PersistArgs a;
  a.mode = mode; a.reset_after = reset_after; a.is_bf16 = is_bf16;
  a.H = hidden; a.B = batch; a.D = ndir; a.ndir = ndir;
  float probe = 0.f;
  if (dwhh) a.dwhh = &probe;   // only tested for null by the planner
  SimtPlan pl;
  if (make_plan(a, bwd != 0, num_sms, &pl) != 0) return 0;
  out[0] = pl.NU; out[1] = pl.nblk; out[2] = pl.PP; out[3] = pl.stream ? 1 : 0;
  out[4] = static_cast<int>(pl.smem);
  a.dwhh = nullptr;
  out[5] = persist_simt_dwhh_ok(a, num_sms, true) ? 1 : 0;
  out[6] = persist_simt_dwhh_ok(a, num_sms, false) ? 1 : 0;
  return 1;
}

int launch_persist_fwd_simt(const PersistArgs& a, cudaStream_t s, int num_sms) {
  return launch_simt(a, false, s, num_sms);
}

int launch_persist_bwd_simt(const PersistArgs& a, cudaStream_t s, int num_sms) {
  return launch_simt(a, true, s, num_sms);
}

}  // namespace rnn
