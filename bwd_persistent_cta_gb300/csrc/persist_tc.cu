// persist_tc.cu - plans and launches of the persistent tensor-core kernels
// (the kernels themselves: persist_tc_kernels.cuh; their instances:
// persist_tc_fwd.cu, persist_tc_bwd.cu).
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "persist_tc_kernels.cuh"

namespace rnn {

namespace {

int pp_for(int pairs) {
  const int need = (pairs + kThreads - 1) / kThreads;
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 8 ? 8 : 0;
}

struct TcPlan {
  int KS = 0, Kc = 0, nsub = 0, R = 0, Npad = 0, UPC = 0, PP = 0, nrg = 0, w_tmem = 0;
  int NB = 1, Bp = 0;   // batch parts per row group, batch rows per part
  uint32_t tmem_cols = 0, off_ring = 0, off_recv = 0, off_bar = 0;
  uint32_t wcol = 0;   // first TMEM column of the weight sub-tiles (w_tmem > 0)
  uint32_t off_stage = 0;   // forward K split: warp 0's post-step stage (0: none)
  size_t smem = 0;
  int gk = 0;               // backward: K-split partials through global memory, no clusters
  int recv2 = 0;            // K split over a cluster: one receive buffer per exchange parity
};

size_t a1k(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

// Estimated per-step cost (us) of a plan, fitted to GB300 step-phase traces
// (timestamps inside the kernels) of the LSTM at hidden 1024 with batch 32 and
// 128 and the GRU at hidden 512:
//   MMA      about 40 ns + 0.07 ns per batch column for each K=16 instruction
//            (42 ns at N=32, 49 ns at N=128: a fixed cost per instruction
//            dominates, so wide N is almost free);
//   TMA      the step's K slice of the exchanged state, 0.3 us + 4 ns per KB;
//   push     the K-split partials over distributed shared memory, 0.2 us +
//            35 ns per KB (51 ns per KB in clusters of 16), none without a
//            K split;
//   cluster  the cluster barrier with the abort flags, about 0.6 us (1.6 us
//            in clusters of 16);
//   epilogue partial sums and cell math, about 0.15 us per (unit, batch row)
//            pair each thread owns, and in the forward as much again for the
//            stores after the step's release.
// The counter wait and release (about 1.8 us) are the same for every plan.
// Measured against these estimates: LSTM B128 H1024 forward, K split 2 x one
// batch part, 9.2 us per step (both directions); backward, K split 4 x 4 batch
// parts, 7.3 us per direction; LSTM B32 H1024 forward 4 x 1, 4.4 us; backward
// 8 x 1, 5.3 us.
// A K split exchanged through global memory instead (gk) is estimated at
// 0.3 us + 30 ns per KB to write the partials, a counter round trip of about
// 1.5 us, and 0.3 us + 30 ns per KB to read the owned rows back.
double plan_cost(int bwd, int KS, int Kc, int Npad, int pairs, int gk = 0) {
  const double n_mma = Kc / 16;
  const double mma = (0.040 + 0.00007 * Npad) * n_mma;
  const double tma = 0.3 + 0.004 * (static_cast<double>(Kc) * Npad * 2 / 1024.0);
  const double push_kb = 128.0 * Npad * 4 * (KS - 1) / KS / 1024.0;
  double push = KS > 1 ? 0.2 + push_kb * (KS >= 16 ? 0.051 : 0.035) : 0.1;
  double cl = KS >= 16 ? 1.6 : KS > 1 ? 0.62 : 0.05;
  if (gk && KS > 1) {
    const double kb = 128.0 * Npad * 4 / 1024.0;
    push = 0.6 + 0.06 * kb;
    cl = 1.5;
  }
  const double per_thread = (pairs + kThreads - 1) / kThreads;
  const double epi = bwd ? 0.14 + 0.14 * per_thread : 0.09 + 0.15 * per_thread;
  const double post = bwd ? 0.0 : 0.15 * per_thread;
  return mma + tma + push + cl + epi + post;
}

// Candidate plans for one launch (K split x batch parts), cheapest first by
// plan_cost.  Whether their clusters can all be resident at once is checked
// at launch.
// gk: backward plans whose K split is exchanged through global memory (no
// clusters; at most 64 row-group counters over directions and batch parts).
int make_plans(int mode, int bwd, int H, int B, int ndir, int num_sms, TcPlan* out, int max_out, int gk = 0) {
  (void)mode;
  if (gk && !bwd) return 0;
  if (B < 1 || B > 256 * kMaxBatchParts) return 0;
  const int K = bwd ? 4 * H : H;
  const int nrg = bwd ? H / 128 : (4 * H) / 128;
  if (bwd ? (H % 128) : (H % 32)) return 0;
  // test hook: a K-split cap (1..16) and a fixed batch-part count (1, 2, 4)
  const PlanOverrides ov = plan_overrides();
  int cap = kMaxKS;
  if (const int v = bwd ? ov.max_ks_bwd : ov.max_ks_fwd) cap = v;
  const int nb_only = bwd ? ov.nb_bwd : ov.nb_fwd;
  std::vector<std::pair<double, TcPlan>> cands;
  for (int NB = 1; NB <= kMaxBatchParts; NB *= 2) {
    // each batch part: Bp rows (at least 8; every part non-empty), the MMA N
    // dimension padded to 16
    const int Bp = (B + NB - 1) / NB;
    if (Bp > 256) continue;   // one part's MMA N stays within 256
    if (NB > 1 && (Bp < 8 || (NB - 1) * Bp >= B)) continue;
    if (nb_only && NB != nb_only && !(NB == 1 && (B + nb_only - 1) / nb_only < 8)) continue;
    const int Npad = (Bp + 15) / 16 * 16;
    for (int KS = kMaxKS; KS >= 1; KS /= 2) {
      if (KS > cap) continue;
      if (K % (KS * kSubK)) continue;
      const int Kc = K / KS;
      const int nsub = Kc / kSubK;
      const int UPC = (bwd ? 128 : 32) / KS;
      if (UPC < 1) continue;
      const int PP = pp_for(UPC * Bp);
      if (PP == 0) continue;
      if (nrg * KS * NB * ndir > num_sms) continue;
      if (gk && (KS == 1 || ndir * NB * nrg > 64)) continue;
      const size_t wbytes = static_cast<size_t>(nsub) * kWSub;
      const size_t rb = static_cast<size_t>(Npad) * 128;
      // a K split over a cluster receives into one buffer per exchange
      // parity: a peer may push the next exchange's partials while this CTA
      // still reads the current ones (it can push the one after only once this
      // CTA has passed the next cluster barrier, after those reads)
      const size_t recv1 = static_cast<size_t>(Npad) * 128 * 4;
      const size_t recv = (KS > 1 && !gk) ? 2 * recv1 : recv1;
      // without a K split the forward stages warp 0's post-step values (32 B
      // per pair) in the receive buffer
      if (KS == 1 && !bwd && recv1 < static_cast<size_t>(32) * PP * 32) continue;
      // weight tile in shared memory, with the deepest exchange ring that fits
      int R = nsub < kMaxRing ? nsub : kMaxRing;
      size_t smem = 0;
      for (; R >= 1; --R) {
        smem = a1k(wbytes) + a1k(R * rb) + a1k(recv) + a1k(sizeof(TcBars)) + 1024;
        if (smem <= kSmemCap) break;
      }
      // else the first wt weight sub-tiles (an even count) in tensor memory as
      // the MMA A operand, in the columns the accumulator leaves free at the top
      // (wcol = 512 - 32 * wt >= Npad), the others in shared memory, and the
      // whole K slice of the exchange operand in flight at once; the fewest
      // sub-tiles in tensor memory that fit
      int wt = 0;
      if (R < nsub && Npad <= 256) {
        const int tmax = std::min(nsub, (512 - Npad) / 32) & ~1;
        for (int t = 2; t <= tmax; t += 2) {
          const size_t sm2 = a1k(static_cast<size_t>(nsub - t) * kWSub) + a1k(static_cast<size_t>(nsub) * rb) +
                             a1k(recv) + a1k(sizeof(TcBars)) + 1024;
          if (sm2 <= kSmemCap) {
            wt = t;
            R = nsub;
            smem = sm2;
            break;
          }
        }
      }
      if (!wt && (R < 1 || (R < nsub && R < 2))) continue;
      TcPlan p;
      p.KS = KS; p.Kc = Kc; p.nsub = nsub; p.R = R; p.Npad = Npad; p.UPC = UPC; p.PP = PP; p.nrg = nrg;
      p.NB = NB; p.Bp = Bp;
      p.w_tmem = wt;
      uint32_t tc = 32;
      while (tc < static_cast<uint32_t>(Npad)) tc *= 2;
      p.tmem_cols = wt ? 512 : tc;
      p.off_ring = static_cast<uint32_t>(a1k(static_cast<size_t>(nsub - wt) * kWSub));
      p.off_recv = p.off_ring + static_cast<uint32_t>(a1k(R * rb));
      p.off_bar = p.off_recv + static_cast<uint32_t>(a1k(recv));
      // forward with a K split: room for warp 0's post-step values (32 B per
      // pair) after the barriers, when shared memory allows
      p.off_stage = 0;
      if (!bwd && KS > 1) {
        const size_t st_bytes = static_cast<size_t>(32) * PP * 32;
        if (smem + a1k(st_bytes) <= kSmemCap) {
          p.off_stage = p.off_bar + static_cast<uint32_t>(a1k(sizeof(TcBars)));
          smem += a1k(st_bytes);
        }
      }
      // all 512 TMEM columns: the shared-memory request alone must keep a
      // second CTA off the SM
      const size_t floor = wt ? kOneCtaSmem : kMinSmem;
      p.smem = smem < floor ? floor : smem;
      p.wcol = wt ? 512u - 32u * static_cast<uint32_t>(wt) : 0u;
      p.gk = gk;
      p.recv2 = (KS > 1 && !gk) ? 1 : 0;
      cands.emplace_back(plan_cost(bwd, KS, Kc, Npad, UPC * Bp, gk), p);
    }
  }
  std::stable_sort(cands.begin(), cands.end(),
                   [](const std::pair<double, TcPlan>& x, const std::pair<double, TcPlan>& y) {
                     return x.first < y.first;
                   });
  int n = 0;
  for (const auto& c : cands) {
    if (n >= max_out) break;
    out[n++] = c.second;
  }
  return n;
}

const void* kernel_for(int bwd, int pp, int ks, int ext) {
  return bwd ? persist_tc_bwd_kernel_ptr(pp, ks, ext) : persist_tc_fwd_kernel_ptr(pp, ks, ext);
}

void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, const TcPlan& pl, int ndir, cudaStream_t s) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(pl.nrg * pl.KS * pl.NB, ndir, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.gk ? 1 : pl.KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

// Chosen plans per shape and device, and the dynamic shared-memory limit set
// on each kernel (only ever raised, so that a cached plan never meets a lower
// limit set for another shape).  The occupancy query behind a plan costs tens
// of microseconds of host time, which the GPU would otherwise wait for at the
// start of every persistent launch.
struct PlanKey {
  int v[13];
  bool operator<(const PlanKey& o) const { return std::lexicographical_compare(v, v + 13, o.v, o.v + 13); }
};

std::mutex g_plan_mu;
std::map<PlanKey, std::pair<bool, TcPlan>> g_plans;
std::map<std::pair<const void*, int>, int> g_smem_limit;

bool raise_smem_limit(const void* fn, int dev, int bytes) {
  int& cur = g_smem_limit[{fn, dev}];
  if (bytes <= cur) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cur = bytes;
  return true;
}

// First candidate plan whose clusters can all be resident at once.
// RNN_TRACE=1: one stderr line per launch shape, when its plan is chosen.
void trace_plan(int bwd, int H, int B, int ndir, int ext, const TcPlan* p) {
  const char* e = std::getenv("RNN_TRACE");
  if (!e || e[0] != '1') return;
  const char* pass = bwd ? "backward" : "forward";
  if (!p) {
    std::fprintf(stderr, "[rnn] tensor-core %s H=%d B=%d dirs=%d: no plan fits\n", pass, H, B, ndir);
    return;
  }
  std::fprintf(stderr,
               "[rnn] tensor-core %s H=%d B=%d dirs=%d%s: K split %d%s, %d batch part(s) of %d rows, %d CTAs, "
               "%d pair(s) per thread, %d weight sub-tiles in tensor memory, %zu B shared memory\n",
               pass, H, B, ndir, ext ? " (extended)" : "", p->KS, p->gk ? " (through global memory)" : "", p->NB,
               p->Bp, p->nrg * p->KS * p->NB * ndir, p->PP, p->w_tmem, p->smem);
}

bool choose_plan(int mode, int bwd, int H, int B, int ndir, int num_sms, int ext, TcPlan* chosen) {
  int dev = 0;
  cudaGetDevice(&dev);
  const PlanOverrides ov = plan_overrides();
  const PlanKey key{{mode, bwd, H, B, ndir, num_sms, ext, dev, ov.max_ks_fwd, ov.max_ks_bwd, ov.nb_fwd, ov.nb_bwd,
                     ov.bwd_global_ks}};
  std::lock_guard<std::mutex> lock(g_plan_mu);
  const auto hit = g_plans.find(key);
  if (hit != g_plans.end()) {
    *chosen = hit->second.second;
    return hit->second.first;
  }
  TcPlan plans[12];
  // test hook: the backward's K split through global memory only
  const int n = bwd && ov.bwd_global_ks ? 0 : make_plans(mode, bwd, H, B, ndir, num_sms, plans, 12);
  for (int i = 0; i < n; ++i) {
    const TcPlan& pl = plans[i];
    const void* fn = kernel_for(bwd, pl.PP, pl.KS, ext);
    if (!raise_smem_limit(fn, dev, static_cast<int>(pl.smem))) continue;
    if (pl.KS > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
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
    if (max_clusters >= pl.nrg * pl.NB * ndir) {
      *chosen = pl;
      g_plans[key] = {true, pl};
      trace_plan(bwd, H, B, ndir, ext, &pl);
      return true;
    }
  }
  // no cluster plan can be resident: the backward's K split through global
  // memory, every CTA of the grid resident at once (one per SM)
  const int ng = bwd ? make_plans(mode, bwd, H, B, ndir, num_sms, plans, 12, 1) : 0;
  for (int i = 0; i < ng; ++i) {
    const TcPlan& pl = plans[i];
    const void* fn = kernel_for(bwd, pl.PP, pl.KS, ext);
    if (!raise_smem_limit(fn, dev, static_cast<int>(pl.smem))) continue;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, pl.smem) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (per_sm >= 1 && pl.nrg * pl.KS * pl.NB * ndir <= num_sms) {
      *chosen = pl;
      g_plans[key] = {true, pl};
      trace_plan(bwd, H, B, ndir, ext, &pl);
      return true;
    }
  }
  g_plans[key] = {false, TcPlan()};
  trace_plan(bwd, H, B, ndir, ext, nullptr);
  return false;
}

int launch(const PersistArgs& a, int bwd, cudaStream_t s, int num_sms) {
  TcPlan pl;
  // the extended kernel variant takes sequence lengths, cell clipping and the
  // GRU reset-before forward
  const bool rb = a.mode == 1 && !a.reset_after;
  if (rb && (bwd ? a.XA == nullptr : a.RH == nullptr)) return 2;
  const int ext = (a.len != nullptr || a.clip || rb) ? 1 : 0;
  if (!choose_plan(a.mode, bwd, a.H, a.B, a.ndir, num_sms, ext, &pl)) return 2;
  if (pl.gk && !a.gk_buf) return 2;
  const int H = a.H, D = a.D;
  CUtensorMap tmW, tmX, tmX4;
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
  // 4-D view of the exchange operand: (64 columns, row, 64-column chunk,
  // direction), so that one box {64, Npad, nsub, 1} lands as nsub consecutive
  // swizzled 64-column sub-tiles
  int single = pl.R >= pl.nsub ? 1 : 0;
  // a slice of 64 KB or more in two chunks of whole sub-tiles (each TMA issue
  // costs about 0.1 us of the step: four chunks measured no faster, and a
  // smaller slice lands too soon to gain)
  const size_t slice_bytes = static_cast<size_t>(pl.nsub) * pl.Npad * 128;
  const int nchunk = pl.nsub % 2 == 0 && pl.nsub >= 4 && slice_bytes >= (64u << 10) ? 2 : 1;
  if (single) {
    const uint64_t Kd = bwd ? 4ull * H : static_cast<uint64_t>(H);
    const uint64_t rows = bwd ? static_cast<uint64_t>(a.T) * a.B : static_cast<uint64_t>(a.T + 2) * a.B;
    const uint64_t dims[4] = {static_cast<uint64_t>(kSubK), rows, Kd / kSubK, static_cast<uint64_t>(D)};
    const uint64_t strides[3] = {static_cast<uint64_t>(D) * Kd * 2, static_cast<uint64_t>(kSubK) * 2, Kd * 2};
    const uint32_t box[4] = {static_cast<uint32_t>(kSubK), static_cast<uint32_t>(pl.Npad),
                             static_cast<uint32_t>(pl.nsub / nchunk), 1u};
    if (make_tmap_bf16_4d(&tmX4, bwd ? a.dG : a.Y, dims, strides, box) != 0) single = 0;
  }
  if (!single) tmX4 = tmX;
  // reset-before: views of RH [D][T*B][H] for the forward's second exchange
  // of a step, of XA [T*B][D*4H] for the backward's first (whole K slice per
  // TMA only)
  CUtensorMap tmR = tmX, tmR4 = tmX4;
  if (rb && bwd) {
    if (!single) return 2;
    const uint64_t TB = static_cast<uint64_t>(a.T) * a.B;
    if (make_tmap_bf16_2d(&tmR, a.XA, static_cast<uint64_t>(D) * 4 * H, TB, static_cast<uint64_t>(D) * 4 * H, kSubK,
                          pl.Npad) != 0)
      return 2;
    const uint64_t Kd = 4ull * H;
    const uint64_t dims[4] = {static_cast<uint64_t>(kSubK), TB, Kd / kSubK, static_cast<uint64_t>(D)};
    const uint64_t strides[3] = {static_cast<uint64_t>(D) * Kd * 2, static_cast<uint64_t>(kSubK) * 2, Kd * 2};
    const uint32_t box[4] = {static_cast<uint32_t>(kSubK), static_cast<uint32_t>(pl.Npad),
                             static_cast<uint32_t>(pl.nsub / nchunk), 1u};
    if (make_tmap_bf16_4d(&tmR4, a.XA, dims, strides, box) != 0) return 2;
  } else if (rb) {
    if (!single) return 2;
    const uint64_t TB = static_cast<uint64_t>(a.T) * a.B;
    if (make_tmap_bf16_2d(&tmR, a.RH, H, D * TB, H, kSubK, pl.Npad) != 0) return 2;
    const uint64_t dims[4] = {static_cast<uint64_t>(kSubK), TB, static_cast<uint64_t>(H) / kSubK,
                              static_cast<uint64_t>(D)};
    const uint64_t strides[3] = {static_cast<uint64_t>(H) * 2, static_cast<uint64_t>(kSubK) * 2, TB * H * 2};
    const uint32_t box[4] = {static_cast<uint32_t>(kSubK), static_cast<uint32_t>(pl.Npad),
                             static_cast<uint32_t>(pl.nsub / nchunk), 1u};
    if (make_tmap_bf16_4d(&tmR4, a.RH, dims, strides, box) != 0) return 2;
  }
  TcPersistParams P;
  P.a = a;
  P.KS = pl.KS; P.Kc = pl.Kc; P.nsub = pl.nsub; P.R = pl.R; P.Npad = pl.Npad; P.UPC = pl.UPC;
  P.RPC = 128 / pl.KS;
  P.nblk_dir = static_cast<unsigned int>(pl.nrg * pl.KS * pl.NB);
  P.nrg = pl.nrg;
  P.NB = pl.NB;
  P.Bp = pl.Bp;
  P.tmem_cols = pl.tmem_cols;
  P.off_ring = pl.off_ring; P.off_recv = pl.off_recv; P.off_bar = pl.off_bar; P.off_stage = pl.off_stage;
  P.w_tmem = pl.w_tmem;
  P.single = single;
  P.nchunk = nchunk;
  const uint64_t proj_bytes = static_cast<uint64_t>(a.T) * a.B * D * 4 * H * 2;
  P.prefetch = !bwd && proj_bytes > (32ull << 20);
  P.wcol = pl.wcol;
  P.gk = pl.gk;
  P.recv2 = pl.recv2;
  const void* fn = kernel_for(bwd, pl.PP, pl.KS, ext);
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_config(cfg, attr, pl, a.ndir, s);
  void* params_fwd[] = {&tmW, &tmX, &tmX4, &tmR, &tmR4, &P};
  void* params_bwd[] = {&tmW, &tmX, &tmX4, &tmR, &tmR4, &P};
  if (cudaLaunchKernelExC(&cfg, fn, bwd ? params_bwd : params_fwd) != cudaSuccess) return 3;
  return 0;
}

}  // namespace


bool persist_tc_supported(int mode, int reset_after, int H, int B, int ndir, int num_sms) {
  if (!(mode == 0 || mode == 1)) return false;
  // GRU reset-before: the extended variant, two exchanges per step, each a
  // whole K slice per TMA
  const bool rb = mode == 1 && !reset_after;
  const int ext = rb ? 1 : 0;
  TcPlan f, b;
  if (!choose_plan(mode, 0, H, B, ndir, num_sms, ext, &f) || !choose_plan(mode, 1, H, B, ndir, num_sms, ext, &b))
    return false;
  return !rb || (f.R >= f.nsub && b.R >= b.nsub);
}

size_t persist_tc_bwd_gk_bytes(int mode, int reset_after, int H, int B, int ndir, int num_sms) {
  if (!(mode == 0 || mode == 1)) return 0;
  size_t most = 0;
  for (int ext = 0; ext <= 1; ++ext) {
    TcPlan b;
    if (!choose_plan(mode, 1, H, B, ndir, num_sms, ext, &b) || !b.gk) continue;
    // two exchange parities x row groups x KS sources x Npad columns x 128 rows
    const size_t bytes = static_cast<size_t>(2) * ndir * b.NB * b.nrg * b.KS * b.Npad * 128 * 4;
    most = std::max(most, bytes);
  }
  (void)reset_after;
  return most;
}

bool persist_tc_fwd_supported(int mode, int reset_after, int H, int B, int ndir, int num_sms) {
  if (mode != 0 && mode != 1) return false;
  const bool rb = mode == 1 && !reset_after;
  TcPlan f;
  if (!choose_plan(mode, 0, H, B, ndir, num_sms, rb ? 1 : 0, &f)) return false;
  // reset-before exchanges r * h_{t-1} as one whole K slice per step
  return !rb || f.R >= f.nsub;
}

extern "C" int rnn_debug_tc_plans(int mode, int bwd, int hidden, int batch, int ndir, int num_sms, int* out,
                                  int max_out) {
  if (!out || max_out <= 0) return 0;
  TcPlan plans[32];
  const int n = make_plans(mode, bwd ? 1 : 0, hidden, batch, ndir, num_sms, plans, max_out < 32 ? max_out : 32);
  for (int i = 0; i < n; ++i) {
    const TcPlan& p = plans[i];
    int* o = out + 7 * i;
    o[0] = p.KS; o[1] = p.NB; o[2] = p.nrg * p.KS * p.NB * ndir; o[3] = p.Npad; o[4] = p.PP; o[5] = p.w_tmem;
    o[6] = static_cast<int>(p.smem);
  }
  return n;
}

int launch_persist_fwd_tc(const PersistArgs& a, cudaStream_t s, int num_sms) { return launch(a, 0, s, num_sms); }
int launch_persist_bwd_tc(const PersistArgs& a, cudaStream_t s, int num_sms) { return launch(a, 1, s, num_sms); }

}  // namespace rnn
