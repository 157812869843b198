// api.cpp - the C ABI: descriptor validation, buffer sizing, weight layout,
// and the per-call launch sequence (host orchestration, one CUDA stream).
//
// Forward, per layer:   pack W_ih / W_hh / biases into the 4-slot order ->
//   input-projection GEMM over all timesteps -> h0 into the output buffer's
//   boundary slot -> one persistent recurrent launch for all steps (both
//   directions together when they fit) -> (last layer) copy / transpose y out.
// Backward data, per layer from the top: pack W_hh^T and W_ih^T -> one
//   persistent BPTT launch (writes dG and the bias-gradient sums) -> input-
//   gradient GEMM dX = dG W_ih (feeds the layer below).
// Backward weights, per layer and direction: dW_ih = dG^T X and
//   dW_hh = dG^T H_prev as long-K GEMMs writing straight into the caller's gate
//   order, and the bias gradients scattered from the sums.
// The split mirrors cuDNN's forward-training / backward-data / backward-weights
// calls as the SystemDS LibMatrixCuDNN.java page's LSTM operators make them.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "rnn.h"
#include "rnn_internal.h"

using namespace rnn;

#include "handle.h"

namespace {

size_t al(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct Bump {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = al(off + bytes);
    return o;
  }
};

int layer_in(const rnn_handle_s* h, int l) { return l == 0 ? h->I : h->D * h->H; }

rnn_status_t st(int rc) { return static_cast<rnn_status_t>(rc); }

// A layout launch, timed in its class with its algorithmic bytes.
#define RNN_LAYOUT(cls, bytes, expr)          \
  do {                                        \
    TimeScope _ts(h, (cls), s, (bytes));      \
    int _rc = (expr);                         \
    if (_rc) return st(_rc);                  \
  } while (0)
#define RNN_TRY(expr)                         \
  do {                                        \
    int _rc = (expr);                         \
    if (_rc) return st(_rc);                  \
  } while (0)

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

void trace(rnn_handle_s* h, const char* what) {
  if (h->trace) std::fprintf(stderr, "[rnn] %s\n", what);
}

void fill_layout(rnn_handle_s* h) {
  const int L = h->L, D = h->D, T = h->T, B = h->B, H = h->H, G = h->G;
  const size_t es = h->es;
  // weights
  size_t o = 0;
  h->off_ih.assign(L * D, 0); h->off_hh.assign(L * D, 0); h->off_b.assign(L * D, 0); h->off_bh.assign(L * D, 0);
  for (int l = 0; l < L; ++l)
    for (int d = 0; d < D; ++d) {
      const int i = l * D + d;
      h->off_ih[i] = o; o += static_cast<size_t>(G) * H * layer_in(h, l);
      h->off_hh[i] = o; o += static_cast<size_t>(G) * H * H;
      h->off_b[i] = o; o += static_cast<size_t>(G) * H;
      if (h->ra) { h->off_bh[i] = o; o += static_cast<size_t>(G) * H; }
    }
  h->weight_elems = o;
  // reserve
  Bump r;
  h->r_y.assign(L, 0); h->r_g.assign(L, 0); h->r_c.assign(L, 0); h->r_rh.assign(L, 0);
  h->r_dg.assign(L, 0); h->r_db.assign(L, 0); h->r_dwhh.assign(L, 0);
  const size_t TB = static_cast<size_t>(T) * B;
  for (int l = 0; l < L; ++l) {
    h->r_y[l] = r.take(static_cast<size_t>(T + 2) * B * D * H * es);
    h->r_g[l] = r.take(static_cast<size_t>(D) * TB * 4 * H * es);
    if (h->lstm && !h->recompute) h->r_c[l] = r.take(static_cast<size_t>(D) * (T + 1) * B * H * 4);
    if (h->rb) h->r_rh[l] = r.take(static_cast<size_t>(D) * TB * H * es);
    h->r_dg[l] = r.take(TB * D * 4 * H * es);
    // bias-gradient sums, one plane per batch part of the tensor-core backward
    // (plane 0 holds the total when it returns)
    h->r_db[l] = r.take(static_cast<size_t>(kMaxBatchParts) * D * 4 * H * 4);
    if (h->dw_bptt) h->r_dwhh[l] = r.take(static_cast<size_t>(D) * G * H * H * 4);
  }
  h->reserve_bytes = r.off;
  // workspace
  int Imax = h->I > D * H ? h->I : D * H;
  Bump w;
  h->w_p = w.take(TB * D * 4 * H * es);
  h->w_xin = h->bfirst ? w.take(TB * h->I * es) : 0;
  h->w_dyi = w.take(TB * D * H * 4);
  h->w_dx0 = h->bfirst ? w.take(TB * h->I * es) : 0;
  h->w_wx = w.take(static_cast<size_t>(D) * 4 * H * Imax * es);
  h->w_wxt = w.take(static_cast<size_t>(Imax) * D * 4 * H * es);
  h->w_wr = w.take(static_cast<size_t>(D) * 4 * H * H * es);
  h->w_wrt = w.take(static_cast<size_t>(D) * H * 4 * H * es);
  h->w_bx = w.take(static_cast<size_t>(D) * 4 * H * 4);
  h->w_bh = w.take(static_cast<size_t>(D) * 4 * H * 4);
  // inference (reserve == NULL): two output buffers and the reset-before exchange
  h->w_y0 = w.take(static_cast<size_t>(T + 2) * B * D * H * es);
  h->w_y1 = w.take(static_cast<size_t>(T + 2) * B * D * H * es);
  h->w_rh = h->rb ? w.take(static_cast<size_t>(D) * TB * H * es) : 0;
  h->w_g = 0;
  // the backward's K-split partials where its plan runs without clusters
  // (both directions in one launch, or one at a time)
  h->gk_bytes = 0;
  if (h->algo == RNN_ALGO_PERSIST_TC) {
    const size_t a = persist_tc_bwd_gk_bytes(h->desc.mode, h->ra, H, B, D, h->num_sms);
    const size_t b = D > 1 ? persist_tc_bwd_gk_bytes(h->desc.mode, h->ra, H, B, 1, h->num_sms) : 0;
    h->gk_bytes = a > b ? a : b;
  }
  h->w_gk = h->gk_bytes ? w.take(h->gk_bytes) : 0;
  h->workspace_bytes = w.off;
}

// internal slot s -> caller's gate block (-1: zero / not used)
void slots_fwd(const rnn_handle_s* h, int* m) {
  if (h->plain) { m[0] = 0; m[1] = m[2] = m[3] = -1; }
  else if (h->lstm) { for (int s = 0; s < 4; ++s) m[s] = h->pos[s]; }
  else { m[0] = h->pos[0]; m[1] = h->pos[1]; m[2] = h->pos[2]; m[3] = -1; }
}
void slots_bwd_rec(const rnn_handle_s* h, int* m) {
  if (h->plain) { m[0] = 0; m[1] = m[2] = m[3] = -1; }
  else if (h->lstm) { for (int s = 0; s < 4; ++s) m[s] = h->pos[s]; }
  else if (h->ra) { m[0] = h->pos[0]; m[1] = h->pos[1]; m[2] = -1; m[3] = h->pos[2]; }
  else { m[0] = h->pos[0]; m[1] = h->pos[1]; m[2] = h->pos[2]; m[3] = -1; }
}

// Interleaved dW_hh (the weight update inside the backward pass) where the
// SIMT backward kernel runs the layer and can hide the per-step work; the
// reserve then holds the accumulated gradient between the backward calls.
void update_dw_bptt(rnn_handle_s* h) {
  PersistArgs probe;
  probe.mode = h->desc.mode; probe.reset_after = h->ra; probe.is_bf16 = h->bf16;
  probe.T = h->T; probe.B = h->B; probe.H = h->H; probe.D = h->D;
  h->dw_bptt = h->dw_mode && h->algo == RNN_ALGO_PERSIST_SIMT &&
                persist_simt_dwhh_ok(probe, h->num_sms, h->dw_mode == 1);
}

int count(rnn_handle_s* h, int rc, int n = 1) {
  if (rc == 0) h->launches += n;
  return rc;
}

// Records an event pair around the launches made while it lives (timing on).
struct TimeScope {
  rnn_handle_s* h;
  cudaStream_t s;
  rnn_handle_s::Ev ev{};
  bool on;
  TimeScope(rnn_handle_s* h_, int cls, cudaStream_t s_, double bytes = 0.0) : h(h_), s(s_), on(h_->timing) {
    if (!on) return;
    if (!h->pool.empty()) {
      ev = h->pool.back();
      h->pool.pop_back();
    } else if (cudaEventCreate(&ev.a) != cudaSuccess || cudaEventCreate(&ev.b) != cudaSuccess) {
      on = false;
      return;
    }
    ev.cls = cls;
    ev.bytes = bytes;
    cudaEventRecord(ev.a, s);
  }
  ~TimeScope() {
    if (!on) return;
    cudaEventRecord(ev.b, s);
    h->events.push_back(ev);
  }
};

// Timing classes of the layout kernels and their algorithmic bytes (every
// element read once and written once at its storage size).
constexpr int kClsSeq = 5, kClsPack = 6, kClsRecompute = 7;
double seq_bytes(int T, int B, int F, int in_bf16, int out_bf16) {
  return static_cast<double>(T) * B * F * ((in_bf16 ? 2 : 4) + (out_bf16 ? 2 : 4));
}
double pack_bytes(const PackBatch& pb, int es) {
  double b = 0.0;
  for (int i = 0; i < pb.n; ++i) {
    const PackJob& j = pb.job[i];
    int mapped = 0;
    for (int k = 0; k < 4; ++k) mapped += j.map[k] >= 0;
    const double HK = static_cast<double>(j.H) * j.K;
    switch (j.kind) {
      case PACK_ROWS:
      case PACK_ROWS_T: b += (mapped + 4.0) * HK * es; break;
      case PACK_BIAS: b += (j.in ? mapped * es : 0) * static_cast<double>(j.H) + 16.0 * j.H; break;
      case SCATTER_DB: b += 16.0 * j.H + 4.0 * mapped * j.H; break;
      default: b += (j.in ? 2.0 : 1.0) * j.B * j.H * es;   // H0_TO_Y
    }
  }
  return b;
}

int run_gemm(rnn_handle_s* h, GemmArgs g, cudaStream_t s, int cls) {
  if (g.M <= 0 || g.N <= 0) return 0;
  TimeScope ts(h, cls, s);
  if (g.K <= 0) return 2;
  g.in_bf16 = h->bf16;
  if (h->bf16 && gemm_tc_supported(g)) {
    int n = 1;
    const int rc = launch_gemm_tc(g, s, h->num_sms, h->dev, h->timeout_ns, &n);
    return count(h, rc, n);
  }
  return count(h, launch_gemm_simt(g, s));
}

int reset_counters(rnn_handle_s* h, cudaStream_t s) {
  // counters, slice counters, the global-K-split counters and abort flag
  return cudaMemsetAsync(h->dev->counters, 0, offsetof(DevArea, status), s) == cudaSuccess ? 0 : 3;
}

// One persistent launch per layer (both directions), or one per direction
// when both do not fit on the GPU at once.
int run_persist(rnn_handle_s* h, PersistArgs a, bool bwd, cudaStream_t s) {
  a.dev = h->dev;
  a.timeout_ns = h->timeout_ns;
  a.skip_cta = h->skip_cta;
#ifdef RNN_CHECKS
  // checking builds: every buffer the steps exchange through starts as 0xFF
  // bytes (a NaN no kernel writes), so a slice read before its producers
  // wrote it shows (the kernels scan each landed slice).  Once per layer,
  // before the first launch: per-direction launches share the buffers.
  {
    const size_t es = h->bf16 ? 2 : 4;
    const size_t TB = static_cast<size_t>(a.T) * a.B;
    const size_t slot = static_cast<size_t>(a.B) * a.D * a.H * es;   // one step of Y
    auto poison = [&](void* p, size_t bytes) { return !p || cudaMemsetAsync(p, 0xFF, bytes, s) == cudaSuccess; };
    bool ok = true;
    if (!bwd) {
      ok = poison(static_cast<char*>(a.Y) + slot, slot * a.T) && ok;   // slots 1 .. T (0 and T + 1 hold h0)
      if (a.mode == 1 && !a.reset_after && a.RH) ok = poison(a.RH, TB * a.D * a.H * es) && ok;
    } else {
      ok = poison(a.dG, TB * a.D * 4 * a.H * es) && ok;
      if (a.XA) ok = poison(a.XA, TB * a.D * 4 * a.H * es) && ok;
    }
    if (!ok) return 3;
  }
#endif
  auto go = [&](PersistArgs& x) -> int {
    int rc = reset_counters(h, s);
    if (rc) return rc;
    TimeScope ts(h, bwd ? 1 : 0, s);
    if (bwd ? h->algo == RNN_ALGO_PERSIST_TC : h->fwd_tc != 0)
      rc = bwd ? launch_persist_bwd_tc(x, s, h->num_sms) : launch_persist_fwd_tc(x, s, h->num_sms);
    else
      rc = bwd ? launch_persist_bwd_simt(x, s, h->num_sms) : launch_persist_fwd_simt(x, s, h->num_sms);
    return count(h, rc);
  };
  a.dir0 = 0;
  a.ndir = h->D;
  int rc = go(a);
  if (rc != 2 || h->D == 1) return rc;
  for (int d = 0; d < h->D; ++d) {
    a.dir0 = d;
    a.ndir = 1;
    rc = go(a);
    if (rc) return rc;
  }
  return 0;
}

// GRU reset-before forward on the tensor-core kernel from this batch on.
constexpr int kRbTcMinBatch = 4;

rnn_status_t check_desc(const rnn_desc_t* d) {
  if (!d) return RNN_BAD_PARAM;
  if (d->mode != RNN_LSTM && d->mode != RNN_GRU && d->mode != RNN_RNN_RELU && d->mode != RNN_RNN_TANH)
    return RNN_BAD_PARAM;
  if (d->dtype != RNN_F32 && d->dtype != RNN_BF16) return RNN_BAD_PARAM;
  if (d->num_layers < 1 || d->num_layers > 8) return RNN_BAD_PARAM;
  if (d->seq_len < 1 || d->batch < 1 || d->input_size < 1 || d->hidden_size < 1) return RNN_BAD_PARAM;
  if (d->bidirectional != 0 && d->bidirectional != 1) return RNN_BAD_PARAM;
  if (d->reset_after != 0 && d->reset_after != 1) return RNN_BAD_PARAM;
  if (d->batch_first != 0 && d->batch_first != 1) return RNN_BAD_PARAM;
  if (d->algo < RNN_ALGO_AUTO || d->algo > RNN_ALGO_PERSIST_SIMT) return RNN_BAD_PARAM;
  const int G = d->mode == RNN_LSTM ? 4 : (d->mode == RNN_GRU ? 3 : 1);
  bool all_zero = true;
  for (int k = 0; k < 4; ++k) all_zero = all_zero && d->gate_order[k] == 0;
  if (!all_zero) {
    int seen = 0;
    for (int k = 0; k < G; ++k) {
      const int c = d->gate_order[k];
      if (c < 0 || c >= G || (seen >> c) & 1) return RNN_BAD_PARAM;
      seen |= 1 << c;
    }
  }
  // element counts must stay addressable with 32-bit grid dimensions
  const long long TB = static_cast<long long>(d->seq_len) * d->batch;
  if (TB > (1LL << 30)) return RNN_BAD_PARAM;
  // vectorised 4-slot accesses need 16-byte aligned rows
  if (d->dtype == RNN_BF16 && (d->hidden_size % 8 || d->input_size % 8)) return RNN_NOT_SUPPORTED;
  if (d->dtype == RNN_F32 && (d->hidden_size % 4 || d->input_size % 4)) return RNN_NOT_SUPPORTED;
  return RNN_OK;
}

}  // namespace

namespace rnn {

int init_handle_host(rnn_handle_s* h, const rnn_desc_t* desc) {
  rnn_status_t rs = check_desc(desc);
  if (rs != RNN_OK) return rs;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_CUDA_ERROR;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return RNN_CUDA_ERROR;
  if (!(prop.major == 10 && prop.minor == 3)) return RNN_NOT_SUPPORTED;
  h->desc = *desc;
  h->L = desc->num_layers; h->D = desc->bidirectional ? 2 : 1;
  h->T = desc->seq_len; h->B = desc->batch; h->H = desc->hidden_size; h->I = desc->input_size;
  h->lstm = desc->mode == RNN_LSTM;
  h->plain = desc->mode == RNN_RNN_RELU || desc->mode == RNN_RNN_TANH;
  h->G = h->lstm ? 4 : (h->plain ? 1 : 3);
  h->ra = desc->mode == RNN_GRU && desc->reset_after;
  h->rb = desc->mode == RNN_GRU && !desc->reset_after;
  h->bf16 = desc->dtype == RNN_BF16;
  h->bfirst = desc->batch_first;
  h->es = h->bf16 ? 2 : 4;
  bool all_zero = true;
  for (int k = 0; k < 4; ++k) all_zero = all_zero && desc->gate_order[k] == 0;
  for (int c = 0; c < 4; ++c) h->pos[c] = c;
  if (!all_zero)
    for (int k = 0; k < h->G; ++k) h->pos[desc->gate_order[k]] = k;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->timeout_ns = 2000000000ull;
  h->skip_cta = -1;
  h->launches = 0;
  h->d_len = nullptr;
  h->has_len = 0;
  h->recompute = 0;
  h->dw_mode = 1;
  h->dw_bptt = 0;
  h->clip = 0;
  h->clip_lo = h->clip_hi = 0.f;
  h->trace = false;
  h->timing = false;
  h->dev = nullptr;
  fill_layout(h);
  // GRU reset-before below batch kRbTcMinBatch keeps the SIMT kernels (its
  // latency-mode forward is faster there)
  const bool tc_ok = h->bf16 && (!h->rb || h->B >= kRbTcMinBatch) &&
                     persist_tc_supported(desc->mode, h->ra, h->H, h->B, 1, h->num_sms);
  PersistArgs probe;
  probe.mode = desc->mode; probe.reset_after = h->ra; probe.is_bf16 = h->bf16;
  probe.T = h->T; probe.B = h->B; probe.H = h->H; probe.D = h->D; probe.ndir = 1;
  const bool simt_ok = plan_persist_simt(probe, h->num_sms, nullptr, nullptr) == 0;
  if (desc->algo == RNN_ALGO_PERSIST_TC) h->algo = tc_ok ? RNN_ALGO_PERSIST_TC : 0;
  else if (desc->algo == RNN_ALGO_PERSIST_SIMT) h->algo = simt_ok ? RNN_ALGO_PERSIST_SIMT : 0;
  else h->algo = tc_ok ? RNN_ALGO_PERSIST_TC : (simt_ok ? RNN_ALGO_PERSIST_SIMT : 0);
  // automatic choice: a tensor-core forward even where only the backward
  // lacks a tensor-core plan (e.g. hidden 2048: the forward splits its weight
  // tile between tensor and shared memory; GRU reset-before, whose forward
  // exchanges twice per step, from batch kRbTcMinBatch on)
  h->fwd_tc = h->algo == RNN_ALGO_PERSIST_TC ||
              (desc->algo == RNN_ALGO_AUTO && h->algo == RNN_ALGO_PERSIST_SIMT && h->bf16 &&
               (!h->rb || h->B >= kRbTcMinBatch) &&
               persist_tc_fwd_supported(desc->mode, h->ra, h->H, h->B, 1, h->num_sms));
  update_dw_bptt(h);
  fill_layout(h);
  return h->algo == 0 ? RNN_NOT_SUPPORTED : RNN_OK;
}

}  // namespace rnn

namespace {

// Makes the handle's device current for one call and puts the caller's
// current device back afterwards (nothing to do when it already is current).
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) { ok = false; return; }
    if (cur == dev) return;
    if (cudaSetDevice(dev) != cudaSuccess) { ok = false; return; }
    prev = cur;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
};

}  // namespace

namespace rnn {
namespace {
std::mutex g_override_mu;
PlanOverrides g_override{0, 0, 0, 0, 0, 0, 0, 0};
}  // namespace
PlanOverrides plan_overrides() {
  std::lock_guard<std::mutex> lock(g_override_mu);
  return g_override;
}
}  // namespace rnn

extern "C" {

const char* rnn_status_string(rnn_status_t s) {
  switch (s) {
    case RNN_OK: return "RNN_OK";
    case RNN_BAD_PARAM: return "RNN_BAD_PARAM: invalid descriptor field or pointer";
    case RNN_NOT_SUPPORTED: return "RNN_NOT_SUPPORTED: valid, but the library or GPU cannot run it";
    case RNN_CUDA_ERROR: return "RNN_CUDA_ERROR: a CUDA call failed";
    case RNN_TIMEOUT: return "RNN_TIMEOUT: a device spin-wait ran out of time";
    case RNN_BAD_WORKSPACE: return "RNN_BAD_WORKSPACE: workspace / reserve missing or misaligned";
    case RNN_INTERNAL: return "RNN_INTERNAL: internal error";
  }
  return "unknown rnn_status_t";
}

rnn_status_t rnn_create(const rnn_desc_t* desc, rnn_handle_t* out) {
  if (!out) return RNN_BAD_PARAM;
  *out = nullptr;
  rnn_handle_s* h = new (std::nothrow) rnn_handle_s();
  if (!h) return RNN_INTERNAL;
  const int rc = rnn::init_handle_host(h, desc);
  if (rc != RNN_OK) { delete h; return static_cast<rnn_status_t>(rc); }
  const char* tr = std::getenv("RNN_TRACE");
  h->trace = tr && tr[0] == '1';

  if (cudaMalloc(&h->dev, sizeof(DevArea)) != cudaSuccess) { delete h; return RNN_CUDA_ERROR; }
  if (cudaMemset(h->dev, 0, sizeof(DevArea)) != cudaSuccess) { cudaFree(h->dev); delete h; return RNN_CUDA_ERROR; }
  *out = h;
  return RNN_OK;
}

rnn_status_t rnn_destroy(rnn_handle_t h) {
  if (!h) return RNN_OK;
  DeviceGuard dg(h->device);
  for (auto& e : h->events) { cudaEventDestroy(e.a); cudaEventDestroy(e.b); }
  for (auto& e : h->pool) { cudaEventDestroy(e.a); cudaEventDestroy(e.b); }
  if (h->dev) cudaFree(h->dev);
  if (h->d_len) cudaFree(h->d_len);
  delete h;
  return RNN_OK;
}

rnn_status_t rnn_get_sizes(rnn_handle_t h, size_t* wb, size_t* ws, size_t* rs) {
  if (!h) return RNN_BAD_PARAM;
  if (wb) *wb = h->weight_elems * h->es;
  if (ws) *ws = h->workspace_bytes;
  if (rs) *rs = h->reserve_bytes;
  return RNN_OK;
}

rnn_status_t rnn_set_timeout_ns(rnn_handle_t h, uint64_t ns) {
  if (!h || ns == 0) return RNN_BAD_PARAM;
  h->timeout_ns = ns;
  return RNN_OK;
}

rnn_status_t rnn_set_seq_lengths(rnn_handle_t h, const int* lengths) {
  if (!h) return RNN_BAD_PARAM;
  DeviceGuard dg(h->device);
  if (!dg.ok) return RNN_CUDA_ERROR;
  if (!lengths) {
    h->has_len = 0;
    return RNN_OK;
  }
  for (int b = 0; b < h->B; ++b)
    if (lengths[b] < 0 || lengths[b] > h->T) return RNN_BAD_PARAM;
  if (!h->d_len && cudaMalloc(&h->d_len, sizeof(int) * h->B) != cudaSuccess) {
    h->d_len = nullptr;
    return RNN_CUDA_ERROR;
  }
  if (cudaMemcpy(h->d_len, lengths, sizeof(int) * h->B, cudaMemcpyHostToDevice) != cudaSuccess)
    return RNN_CUDA_ERROR;
  h->has_len = 1;
  return RNN_OK;
}

rnn_status_t rnn_set_recomputation(rnn_handle_t h, int mode) {
  if (!h || mode < 0 || mode > 1) return RNN_BAD_PARAM;
  DeviceGuard dg(h->device);
  if (!dg.ok) return RNN_CUDA_ERROR;
  h->recompute = h->lstm ? mode : 0;
  fill_layout(h);
  return RNN_OK;
}

rnn_status_t rnn_set_interleaved_dw(rnn_handle_t h, int mode) {
  if (!h || mode < 0 || mode > 2) return RNN_BAD_PARAM;
  DeviceGuard dg(h->device);
  if (!dg.ok) return RNN_CUDA_ERROR;
  h->dw_mode = mode;
  update_dw_bptt(h);
  fill_layout(h);
  return RNN_OK;
}

int rnn_interleaved_dw_active(rnn_handle_t h) { return h ? h->dw_bptt : 0; }

rnn_status_t rnn_set_cell_clip(rnn_handle_t h, int enable, double lo, double hi) {
  if (!h) return RNN_BAD_PARAM;
  if (!enable) {
    h->clip = 0;
    return RNN_OK;
  }
  if (!h->lstm || !(lo < hi)) return RNN_BAD_PARAM;
  h->clip = 1;
  h->clip_lo = static_cast<float>(lo);
  h->clip_hi = static_cast<float>(hi);
  return RNN_OK;
}

rnn_status_t rnn_set_timing(rnn_handle_t h, int enable) {
  if (!h) return RNN_BAD_PARAM;
  h->timing = enable != 0;
  return RNN_OK;
}

rnn_status_t rnn_get_timing_ex(rnn_handle_t h, double* ms, uint64_t* n, double* bytes) {
  if (!h) return RNN_BAD_PARAM;
  double acc[RNN_TIMING_CLASSES] = {0}, by[RNN_TIMING_CLASSES] = {0};
  uint64_t cnt[RNN_TIMING_CLASSES] = {0};
  rnn_status_t rs = RNN_OK;
  for (auto& e : h->events) {
    float t = 0.f;
    if (cudaEventSynchronize(e.b) != cudaSuccess || cudaEventElapsedTime(&t, e.a, e.b) != cudaSuccess)
      rs = RNN_CUDA_ERROR;
    acc[e.cls] += t;
    cnt[e.cls] += 1;
    by[e.cls] += e.bytes;
    h->pool.push_back(e);
  }
  h->events.clear();
  for (int i = 0; i < RNN_TIMING_CLASSES; ++i) {
    if (ms) ms[i] = acc[i];
    if (n) n[i] = cnt[i];
    if (bytes) bytes[i] = by[i];
  }
  return rs;
}

rnn_status_t rnn_get_timing(rnn_handle_t h, double* ms, uint64_t* n) { return rnn_get_timing_ex(h, ms, n, nullptr); }

uint64_t rnn_launch_count(rnn_handle_t h) { return h ? h->launches : 0; }

int rnn_selected_algo(rnn_handle_t h) { return h ? h->algo : 0; }

int rnn_selected_fwd_algo(rnn_handle_t h) {
  return h ? (h->fwd_tc ? RNN_ALGO_PERSIST_TC : h->algo) : 0;
}

rnn_status_t rnn_debug_set_plan_overrides(int max_ks_fwd, int max_ks_bwd, int nb_fwd, int nb_bwd, int gemm_bn,
                                          int gemm_splits, int gemm_tm, int bwd_global_ks) {
  auto ks_ok = [](int v) { return v >= 0 && v <= 16; };
  auto nb_ok = [](int v) { return v == 0 || v == 1 || v == 2 || v == 4; };
  if (!ks_ok(max_ks_fwd) || !ks_ok(max_ks_bwd) || !nb_ok(nb_fwd) || !nb_ok(nb_bwd) ||
      !(gemm_bn == 0 || gemm_bn == 128 || gemm_bn == 256) || !ks_ok(gemm_splits) ||
      !(gemm_tm == 0 || gemm_tm == 128 || gemm_tm == 256) || (gemm_tm == 256 && gemm_bn == 128) ||
      !(bwd_global_ks == 0 || bwd_global_ks == 1))
    return RNN_BAD_PARAM;
  std::lock_guard<std::mutex> lock(rnn::g_override_mu);
  rnn::g_override = {max_ks_fwd, max_ks_bwd, nb_fwd, nb_bwd, gemm_bn, gemm_splits, gemm_tm, bwd_global_ks};
  return RNN_OK;
}

rnn_status_t rnn_debug_skip_arrival(rnn_handle_t h, int cta) {
  if (!h || cta < -1) return RNN_BAD_PARAM;
  h->skip_cta = cta;
  return RNN_OK;
}

rnn_status_t rnn_sync_status(rnn_handle_t h, void* stream) {
  if (!h) return RNN_BAD_PARAM;
  DeviceGuard dg(h->device);
  if (!dg.ok) return RNN_CUDA_ERROR;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return RNN_CUDA_ERROR;
  unsigned int code = 0;
  if (cudaMemcpy(&code, &h->dev->status, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess) return RNN_CUDA_ERROR;
  if (code != 0) {
    unsigned int where[4] = {0, 0, 0, 0};
    cudaMemcpy(where, h->dev->where, sizeof(where), cudaMemcpyDeviceToHost);
    if (h->trace)
      std::fprintf(stderr, "[rnn] device status %u: kernel %u block %u step %u wait %u\n", code, where[0], where[1],
                   where[2], where[3]);
    if (cudaMemset(h->dev, 0, sizeof(DevArea)) != cudaSuccess) return RNN_CUDA_ERROR;
  }
  return static_cast<rnn_status_t>(code);
}

rnn_status_t rnn_forward(rnn_handle_t h, const void* x, const void* hx, const void* cx, const void* w, void* y,
                         void* hy, void* cy, void* workspace, void* reserve, void* stream) {
  if (!h || !x || !w || !y) return RNN_BAD_PARAM;
  if (!workspace) return RNN_BAD_WORKSPACE;
  DeviceGuard dg(h->device);
  if (!dg.ok) return RNN_CUDA_ERROR;
  const void* ptrs[] = {x, hx, cx, w, y, hy, cy, workspace, reserve};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return RNN_BAD_PARAM;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int L = h->L, D = h->D, T = h->T, B = h->B, H = h->H;
  const size_t es = h->es;
  const size_t TB = static_cast<size_t>(T) * B;
  const bool train = reserve != nullptr;
  trace(h, train ? "forward (training)" : "forward (inference)");
  int sf[4];
  slots_fwd(h, sf);
  const void* layer_x = x;
  if (h->bfirst) {
    RNN_LAYOUT(kClsSeq, seq_bytes(T, B, h->I, h->bf16, h->bf16),
               count(h, launch_seq_transpose(x, at<char>(workspace, h->w_xin), T, B, h->I, h->bf16, h->bf16, 1, 0,
                                             h->I, s)));
    layer_x = at<char>(workspace, h->w_xin);
  }
  void* Ybuf = nullptr;
  const bool y_direct = h->fwd_tc && !h->bfirst;
  for (int l = 0; l < L; ++l) {
    const int Il = layer_in(h, l);
    char* wb = static_cast<char*>(const_cast<void*>(w));
    // layer output buffer (h0 goes into its boundary slots)
    Ybuf = train ? at<char>(reserve, h->r_y[l]) : at<char>(workspace, (l & 1) ? h->w_y1 : h->w_y0);
    // one launch: packed W_ih, W_hh, biases of both directions, h0 into Ybuf
    PackBatch pb;
    for (int d = 0; d < D; ++d) {
      const int i = l * D + d;
      PackJob j;
      for (int k = 0; k < 4; ++k) j.map[k] = sf[k];
      j.H = H;
      j.kind = PACK_ROWS; j.K = Il; j.in = wb + h->off_ih[i] * es; j.ld_out = Il;
      j.out = at<char>(workspace, h->w_wx) + static_cast<size_t>(d) * 4 * H * Il * es;
      pb.add(j);
      j.K = H; j.in = wb + h->off_hh[i] * es; j.ld_out = H;
      j.out = at<char>(workspace, h->w_wr) + static_cast<size_t>(d) * 4 * H * H * es;
      pb.add(j);
      j.kind = PACK_BIAS; j.in = wb + h->off_b[i] * es; j.out = at<float>(workspace, h->w_bx) + static_cast<size_t>(d) * 4 * H;
      pb.add(j);
      if (h->ra) {
        j.in = wb + h->off_bh[i] * es; j.out = at<float>(workspace, h->w_bh) + static_cast<size_t>(d) * 4 * H;
        pb.add(j);
      }
      PackJob y;
      y.kind = H0_TO_Y; y.H = H; y.T = T; y.B = B; y.D = D; y.dir = d; y.out = Ybuf;
      y.in = hx ? static_cast<const char*>(hx) + (static_cast<size_t>(l) * D + d) * B * H * es : nullptr;
      pb.add(y);
    }
    RNN_LAYOUT(kClsPack, pack_bytes(pb, static_cast<int>(es)), count(h, launch_pack_batch(pb, h->bf16, s)));
    // hoisted input projection for every timestep and direction
    GemmArgs g;
    g.M = static_cast<int>(TB); g.N = D * 4 * H; g.K = Il;
    g.A = layer_x; g.lda = Il; g.a_kmajor = 1;
    g.B = at<char>(workspace, h->w_wx); g.ldb = Il; g.b_kmajor = 1;
    g.C = at<char>(workspace, h->w_p); g.ldc = D * 4 * H; g.c_bf16 = h->bf16;
    g.bias = at<float>(workspace, h->w_bx);
    RNN_TRY(run_gemm(h, g, s, 2));
    PersistArgs a;
    a.mode = h->desc.mode; a.reset_after = h->ra; a.is_bf16 = h->bf16;
    a.T = T; a.B = B; a.H = H; a.D = D;
    a.P = at<char>(workspace, h->w_p);
    a.bh = h->ra ? at<float>(workspace, h->w_bh) : nullptr;
    a.Wr = at<char>(workspace, h->w_wr);
    a.Y = Ybuf;
    a.gates = train ? at<char>(reserve, h->r_g[l]) : nullptr;
    a.C = (train && h->lstm && !h->recompute) ? at<float>(reserve, h->r_c[l]) : nullptr;
    a.RH = h->rb ? (train ? at<char>(reserve, h->r_rh[l]) : at<char>(workspace, h->w_rh)) : nullptr;
    a.c0 = (h->lstm && cx) ? static_cast<const char*>(cx) + static_cast<size_t>(l) * D * B * H * es : nullptr;
    a.hy = hy ? static_cast<char*>(hy) + static_cast<size_t>(l) * D * B * H * es : nullptr;
    a.cy = (h->lstm && cy) ? static_cast<char*>(cy) + static_cast<size_t>(l) * D * B * H * es : nullptr;
    a.len = h->has_len ? h->d_len : nullptr;
    a.clip = h->clip; a.clip_lo = h->clip_lo; a.clip_hi = h->clip_hi;
    // the tensor-core kernels write the caller's seq-major y themselves
    if (l == L - 1 && y_direct) a.y_out = y;
    RNN_TRY(run_persist(h, a, false, s));
    layer_x = static_cast<char*>(Ybuf) + static_cast<size_t>(B) * D * H * es;   // slot 1
  }
  // y out (rows of slots 1..T)
  if (!y_direct)
    RNN_LAYOUT(kClsSeq, seq_bytes(T, B, D * H, h->bf16, h->bf16),
               count(h, launch_seq_transpose(layer_x, y, T, B, D * H, h->bf16, h->bf16, 0, h->bfirst, D * H, s,
                                             h->has_len ? h->d_len : nullptr)));
  return cudaGetLastError() == cudaSuccess ? RNN_OK : RNN_CUDA_ERROR;
}

rnn_status_t rnn_backward_data(rnn_handle_t h, const void* y, const void* dy, const void* dhy, const void* dcy,
                               const void* w, const void* hx, const void* cx, void* dx, void* dhx, void* dcx,
                               void* workspace, void* reserve, void* stream) {
  (void)y; (void)hx;   // cx: read only with recomputation (the cell states' initial value)
  if (!h || !dy || !w || !dx) return RNN_BAD_PARAM;
  if (!workspace || !reserve) return RNN_BAD_WORKSPACE;
  DeviceGuard dg(h->device);
  if (!dg.ok) return RNN_CUDA_ERROR;
  const void* ptrs[] = {dy, dhy, dcy, w, cx, dx, dhx, dcx, workspace, reserve};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return RNN_BAD_PARAM;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int L = h->L, D = h->D, T = h->T, B = h->B, H = h->H;
  const size_t es = h->es;
  const size_t TB = static_cast<size_t>(T) * B;
  trace(h, "backward data");
  int sr[4], sx[4];
  slots_bwd_rec(h, sr);
  slots_fwd(h, sx);
  float* dyi = at<float>(workspace, h->w_dyi);
  RNN_LAYOUT(kClsSeq, seq_bytes(T, B, D * H, h->bf16, 0),
             count(h, launch_seq_transpose(dy, dyi, T, B, D * H, h->bf16, 0, h->bfirst, 0, D * H, s)));
  char* wb = static_cast<char*>(const_cast<void*>(w));
  for (int l = L - 1; l >= 0; --l) {
    const int Il = layer_in(h, l);
    // one launch: W_hh^T and W_ih^T of both directions
    PackBatch pb;
    for (int d = 0; d < D; ++d) {
      const int i = l * D + d;
      PackJob j;
      j.kind = PACK_ROWS_T; j.H = H;
      for (int k = 0; k < 4; ++k) j.map[k] = sr[k];
      j.K = H; j.in = wb + h->off_hh[i] * es; j.ld_out = 4 * H;
      j.out = at<char>(workspace, h->w_wrt) + static_cast<size_t>(d) * H * 4 * H * es;
      pb.add(j);
      for (int k = 0; k < 4; ++k) j.map[k] = sx[k];
      j.K = Il; j.in = wb + h->off_ih[i] * es; j.ld_out = static_cast<int64_t>(D) * 4 * H;
      j.out = at<char>(workspace, h->w_wxt) + static_cast<size_t>(d) * 4 * H * es;
      pb.add(j);
    }
    RNN_LAYOUT(kClsPack, pack_bytes(pb, static_cast<int>(es)), count(h, launch_pack_batch(pb, h->bf16, s)));
    PersistArgs a;
    a.mode = h->desc.mode; a.reset_after = h->ra; a.is_bf16 = h->bf16;
    a.T = T; a.B = B; a.H = H; a.D = D;
    a.Y = at<char>(reserve, h->r_y[l]);
    a.gates = at<char>(reserve, h->r_g[l]);
    a.C = h->lstm ? at<float>(reserve, h->r_c[l]) : nullptr;
    if (h->lstm && h->recompute) {
      // cell states recomputed from the saved gates into the projection
      // buffer, idle in the backward pass (D*(T+1)*B*H*4 <= T*B*D*4H*es bytes)
      float* Cw = at<float>(workspace, h->w_p);
      const void* c0 = cx ? static_cast<const char*>(cx) + static_cast<size_t>(l) * D * B * H * es : nullptr;
      RNN_LAYOUT(kClsRecompute, static_cast<double>(D) * T * B * H * (3.0 * es + 4.0),
                 count(h, launch_recompute_cells(a.gates, c0, Cw, T, B, H, D, h->bf16,
                                                 h->has_len ? h->d_len : nullptr, h->clip, h->clip_lo, h->clip_hi,
                                                 s)));
      a.C = Cw;
    }
    a.WrT = at<char>(workspace, h->w_wrt);
    a.dYi = dyi;
    a.dG = at<char>(reserve, h->r_dg[l]);
    a.db = at<float>(reserve, h->r_db[l]);
    const size_t so = static_cast<size_t>(l) * D * B * H * es;
    a.dhT = dhy ? static_cast<const char*>(dhy) + so : nullptr;
    a.dcT = (h->lstm && dcy) ? static_cast<const char*>(dcy) + so : nullptr;
    a.len = h->has_len ? h->d_len : nullptr;
    a.clip = h->clip; a.clip_lo = h->clip_lo; a.clip_hi = h->clip_hi;
    a.dh0 = dhx ? static_cast<char*>(dhx) + so : nullptr;
    a.dc0 = (h->lstm && dcx) ? static_cast<char*>(dcx) + so : nullptr;
    // the projection buffer, idle in the backward, holds the tensor-core
    // reset-before backward's first-exchange operand [T, B, D*4H]
    if (h->rb) a.XA = at<char>(workspace, h->w_p);
    if (h->dw_bptt) {
      a.dwhh = at<float>(reserve, h->r_dwhh[l]);
      for (int k = 0; k < 4; ++k) a.whh_map[k] = sr[k];
      a.RH = h->rb ? at<char>(reserve, h->r_rh[l]) : nullptr;
    }
    a.gk_buf = h->gk_bytes ? at<float>(workspace, h->w_gk) : nullptr;
    RNN_TRY(run_persist(h, a, true, s));
    // input gradient dX = dG * W_ih (both directions summed through K)
    GemmArgs g;
    g.M = static_cast<int>(TB); g.N = Il; g.K = D * 4 * H;
    g.A = at<char>(reserve, h->r_dg[l]); g.lda = D * 4 * H; g.a_kmajor = 1;
    g.B = at<char>(workspace, h->w_wxt); g.ldb = D * 4 * H; g.b_kmajor = 1;
    if (l > 0) {
      g.C = dyi; g.ldc = Il; g.c_bf16 = 0;
    } else {
      g.C = h->bfirst ? at<char>(workspace, h->w_dx0) : dx; g.ldc = Il; g.c_bf16 = h->bf16;
    }
    RNN_TRY(run_gemm(h, g, s, 3));
  }
  if (h->bfirst)
    RNN_LAYOUT(kClsSeq, seq_bytes(T, B, h->I, h->bf16, h->bf16),
               count(h, launch_seq_transpose(at<char>(workspace, h->w_dx0), dx, T, B, h->I, h->bf16, h->bf16, 0, 1,
                                             h->I, s)));
  return cudaGetLastError() == cudaSuccess ? RNN_OK : RNN_CUDA_ERROR;
}

rnn_status_t rnn_backward_weights(rnn_handle_t h, const void* x, const void* hx, const void* y, void* workspace,
                                  const void* reserve, void* dw, void* stream) {
  (void)hx; (void)y;
  if (!h || !x || !dw) return RNN_BAD_PARAM;
  if (!workspace || !reserve) return RNN_BAD_WORKSPACE;
  DeviceGuard dg(h->device);
  if (!dg.ok) return RNN_CUDA_ERROR;
  const void* ptrs[] = {x, workspace, reserve, dw};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RNN_BAD_PARAM;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int L = h->L, D = h->D, T = h->T, B = h->B, H = h->H;
  const size_t es = h->es;
  const size_t TB = static_cast<size_t>(T) * B;
  trace(h, "backward weights");
  const void* x0 = x;
  if (h->bfirst) {
    RNN_LAYOUT(kClsSeq, seq_bytes(T, B, h->I, h->bf16, h->bf16),
               count(h, launch_seq_transpose(x, at<char>(workspace, h->w_xin), T, B, h->I, h->bf16, h->bf16, 1, 0,
                                             h->I, s)));
    x0 = at<char>(workspace, h->w_xin);
  }
  char* rs = static_cast<char*>(const_cast<void*>(reserve));
  float* dwf = static_cast<float*>(dw);
  const int* pos = h->pos;
  int m_ih[4], m_hh[4], m_b[4], m_bh[4];
  if (h->plain) {
    for (int k = 0; k < 4; ++k) m_ih[k] = m_hh[k] = m_b[k] = m_bh[k] = k == 0 ? 0 : -1;
  } else if (h->lstm) {
    for (int k = 0; k < 4; ++k) m_ih[k] = m_hh[k] = m_b[k] = m_bh[k] = pos[k];
  } else {
    m_ih[0] = pos[0]; m_ih[1] = pos[1]; m_ih[2] = pos[2]; m_ih[3] = -1;
    m_b[0] = pos[0]; m_b[1] = pos[1]; m_b[2] = pos[2]; m_b[3] = -1;
    if (h->ra) {
      m_hh[0] = pos[0]; m_hh[1] = pos[1]; m_hh[2] = -1; m_hh[3] = pos[2];
      m_bh[0] = pos[0]; m_bh[1] = pos[1]; m_bh[2] = -1; m_bh[3] = pos[2];
    } else {
      m_hh[0] = pos[0]; m_hh[1] = pos[1]; m_hh[2] = -1; m_hh[3] = -1;
    }
  }
  PackBatch scatter;
  for (int l = 0; l < L; ++l) {
    const int Il = layer_in(h, l);
    const void* Xl = l == 0 ? x0 : rs + h->r_y[l - 1] + static_cast<size_t>(B) * D * H * es;
    // the layer's weight-gradient GEMMs (every direction, W_ih and W_hh):
    // one grouped launch on the tensor cores, else one SIMT launch each
    GemmArgs grp[6];
    int ng = 0;
    for (int d = 0; d < D; ++d) {
      const int i = l * D + d;
      const char* dG = rs + h->r_dg[l] + static_cast<size_t>(d) * 4 * H * es;
      GemmArgs g;
      g.M = 4 * H; g.K = static_cast<int>(TB);
      g.A = dG; g.lda = D * 4 * H; g.a_kmajor = 0;
      g.rowmap_H = H;
      // long K = T*B: the projection buffer (idle here) holds split-K partials
      g.split_ws = at<char>(workspace, h->w_p);
      g.split_ws_bytes = TB * D * 4 * H * es;
      g.in_bf16 = h->bf16;
      // dW_ih = sum over (t, b) of dG x^T
      g.N = Il;
      g.B = Xl; g.ldb = Il; g.b_kmajor = 0;
      g.C = dwf + h->off_ih[i]; g.ldc = Il; g.c_bf16 = 0;
      for (int k = 0; k < 4; ++k) g.perm[k] = m_ih[k];
      grp[ng++] = g;
      if (h->dw_bptt) {
        // accumulated by the backward-data pass, already in the caller's rows
        const size_t bytes = static_cast<size_t>(h->G) * H * H * 4;
        if (cudaMemcpyAsync(dwf + h->off_hh[i], rs + h->r_dwhh[l] + d * bytes, bytes, cudaMemcpyDeviceToDevice,
                            s) != cudaSuccess)
          return RNN_CUDA_ERROR;
      } else {
        // dW_hh = sum over (t, b) of dG^h h_prev^T ; h_prev rows are Y slots t (forward) / t+2 (reverse)
        const char* hp =
            rs + h->r_y[l] + (static_cast<size_t>(d == 0 ? 0 : 2) * B * D * H + static_cast<size_t>(d) * H) * es;
        g.N = H;
        g.B = hp; g.ldb = D * H; g.b_kmajor = 0;
        g.C = dwf + h->off_hh[i]; g.ldc = H;
        for (int k = 0; k < 4; ++k) g.perm[k] = m_hh[k];
        grp[ng++] = g;
        if (h->rb) {
          // reset-before candidate rows: dW_hn = sum dn (r * h_prev)^T
          g.B = rs + h->r_rh[l] + static_cast<size_t>(d) * TB * H * es; g.ldb = H;
          g.perm[0] = -1; g.perm[1] = -1; g.perm[2] = pos[2]; g.perm[3] = -1;
          grp[ng++] = g;
        }
      }
    }
    bool tc = h->bf16;
    for (int k = 0; k < ng && tc; ++k) tc = gemm_tc_supported(grp[k]);
    if (tc) {
      TimeScope ts(h, 4, s);
      RNN_TRY(count(h, launch_gemm_tc_grouped(grp, ng, s, h->num_sms, h->dev, h->timeout_ns)));
    } else {
      for (int k = 0; k < ng; ++k) RNN_TRY(run_gemm(h, grp[k], s, 4));
    }
    for (int d = 0; d < D; ++d) {
      const int i = l * D + d;
      // bias gradients back to the caller's gate blocks (batched below)
      PackJob j;
      j.kind = SCATTER_DB; j.H = H;
      j.in = reinterpret_cast<const float*>(rs + h->r_db[l]) + static_cast<size_t>(d) * 4 * H;
      for (int k = 0; k < 4; ++k) j.map[k] = m_b[k];
      j.out = dwf + h->off_b[i];
      if (!scatter.add(j)) {
        RNN_LAYOUT(kClsPack, pack_bytes(scatter, 4), count(h, launch_pack_batch(scatter, 0, s)));
        scatter.n = 0;
        scatter.add(j);
      }
      if (h->ra) {
        for (int k = 0; k < 4; ++k) j.map[k] = m_bh[k];
        j.out = dwf + h->off_bh[i];
        if (!scatter.add(j)) {
          RNN_LAYOUT(kClsPack, pack_bytes(scatter, 4), count(h, launch_pack_batch(scatter, 0, s)));
          scatter.n = 0;
          scatter.add(j);
        }
      }
    }
  }
  RNN_LAYOUT(kClsPack, pack_bytes(scatter, 4), count(h, launch_pack_batch(scatter, 0, s)));
  return cudaGetLastError() == cudaSuccess ? RNN_OK : RNN_CUDA_ERROR;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// test hook: the internal GEMM on its own (include/rnn_debug.h)
// ---------------------------------------------------------------------------
#include "rnn_debug.h"

extern "C" rnn_status_t rnn_debug_gemm(int M, int N, int K, const void* A, int64_t lda, int a_kmajor, const void* B,
                                       int64_t ldb, int b_kmajor, void* C, int64_t ldc, int c_bf16,
                                       const float* bias, int beta, int rowmap_H, const int* perm, int in_bf16,
                                       int use_tc, void* stream) {
  if (M <= 0 || N <= 0 || K <= 0 || !A || !B || !C) return RNN_BAD_PARAM;
  GemmArgs g;
  g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.a_kmajor = a_kmajor;
  g.B = B; g.ldb = ldb; g.b_kmajor = b_kmajor;
  g.C = C; g.ldc = ldc; g.c_bf16 = c_bf16;
  g.bias = bias; g.beta = beta; g.rowmap_H = rowmap_H;
  for (int k = 0; k < 4; ++k) g.perm[k] = perm ? perm[k] : k;
  g.in_bf16 = in_bf16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // scratch for a K split of fp32 outputs, as the weight gradients get (kept
  // across calls, grown on demand; only this test hook allocates it)
  static void* ws = nullptr;
  static size_t ws_bytes = 0;
  if (!c_bf16 && use_tc) {
    const size_t need = gemm_tc_split_scratch_bytes(M, N);
    if (need > ws_bytes) {
      if (ws) cudaFree(ws);
      ws = nullptr;
      ws_bytes = 0;
      if (cudaMalloc(&ws, need) != cudaSuccess) return RNN_CUDA_ERROR;
      ws_bytes = need;
    }
    g.split_ws = ws;
    g.split_ws_bytes = ws_bytes;
  }
  static DevArea* dev = nullptr;
  if (!dev) {
    if (cudaMalloc(&dev, sizeof(DevArea)) != cudaSuccess) return RNN_CUDA_ERROR;
    if (cudaMemset(dev, 0, sizeof(DevArea)) != cudaSuccess) return RNN_CUDA_ERROR;
  }
  int nsm = 0, d = 0;
  cudaGetDevice(&d);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, d);
  int rc = use_tc ? launch_gemm_tc(g, s, nsm, dev, 2000000000ull) : launch_gemm_simt(g, s);
  return static_cast<rnn_status_t>(rc);
}
