// rnn_internal.h - internal data layouts and kernel launch interfaces.
//
// Internal layouts (all seq-major; s = storage element, fp32 or bf16):
//   * Gate slots are unit-interleaved: column 4*u + slot of a [.., 4H] array
//     belongs to hidden unit u.  Slots (canonical gate order):
//       LSTM            i, f, g, o
//       GRU resetAfter  r, z, n, hn (hn = W_hn h + b_hn, forward reserve only)
//       GRU reset-before r, z, n, (unused)
//     GRU's fourth slot is padding in every weight matrix (zero rows).
//   * P  [T, B, D*4H]  s    input projection W_ih x_t + b (all directions)
//   * Y  [T+2, B, D*H] s    layer output; slot t+1 holds y_t.  Slot 0 holds
//     the forward direction's h0 (columns [0, H)), slot T+1 the reverse
//     direction's h0 (columns [H, 2H)), so h_{t-1} of the forward direction
//     is slot t and h_{t+1} of the reverse direction is slot t+2.
//   * GATES [D][T, B, 4H] s  post-activation gates (reserve).
//   * C [D][T+1, B, H] fp32  LSTM cell state: forward c_t at slot t+1 (c0 at 0);
//     reverse c_t at slot t (c0 at T).
//   * RH [D][T, B, H] s      GRU reset-before r * h_{t-1} (reserve).
//   * DG [T, B, D*4H] s      gate pre-activation gradients: LSTM (da_i, da_f,
//     da_g, da_o); GRU resetAfter (dr, dz, dn, dn*r); reset-before (dr, dz, dn, 0).
//   * DB [D][4H] fp32        batch- and time-summed DG, slot order (GRU
//     resetAfter: slots r, z, n give the input-side bias gradient and slots
//     r, z, n*r the recurrent-side one).
//   * Packed weights: WX [D*4H, I_l] (row d*4H + 4u + s = W_ih of gate s, unit u),
//     WXT [I_l, D*4H], WR [D][4H, H] (row 4u + s = W_hh row of gate s, unit u),
//     WRT [D][H, 4H] (element (j, 4u+s) = W_hh[gate(s)][u][j]; for GRU
//     resetAfter slot 2 is zero and slot 3 holds W_hn, matching the DG slots
//     of the recurrent side), BX [D*4H] fp32, BH [D*4H] fp32.
#pragma once

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

namespace rnn {

constexpr int kSlots = 4;

struct DevArea {
  unsigned int counters[32];   // step counters of the running persistent launch (per direction)
  // tensor-core persistent kernels: per (direction, batch part, K slice), the
  // arrivals of the CTAs whose outputs form that K slice of the exchanged state
  unsigned int slice_ctr[128];
  // tensor-core backward with its K split exchanged through global memory
  // (no cluster): per (direction, batch part, row group) the arrivals of its
  // KS CTAs, and a flag any of them sets when it gives up
  unsigned int gk_ctr[64];
  unsigned int gk_abort;
  unsigned int status;         // 0, or the first rnn_status_t a kernel reported
  unsigned int where[4];       // kernel id, block, step, wait kind of that report
  unsigned int pad[26];        // to 1 KB
};
static_assert(sizeof(DevArea) == 1024, "DevArea is 1 KB");

enum KernelId : unsigned int { K_FWD_SIMT = 1, K_BWD_SIMT = 2, K_FWD_TC = 3, K_BWD_TC = 4, K_GEMM_TC = 5 };
// W_CHECK (checking builds, -DRNN_CHECKS): an exchanged slice held the poison
// pattern, i.e. it was read before its producer wrote it.
enum WaitKind : unsigned int { W_COUNTER = 1, W_TMA = 2, W_MMA = 3, W_CHECK = 4 };

// C[row(m), n] = sum_k A(m, k) * B(n, k)  (+ bias[n]) (+ C_old if beta)
//   A(m, k) = A[m*lda + k] (a_kmajor) or A[k*lda + m];  same for B with n.
//   row(m) = m, or with rowmap_H > 0: m = 4u + s -> perm[s]*rowmap_H + u
//   (rows whose perm[s] < 0 are not written).
struct GemmArgs {
  int M = 0, N = 0, K = 0;
  const void* A = nullptr; int64_t lda = 0; int a_kmajor = 1;
  const void* B = nullptr; int64_t ldb = 0; int b_kmajor = 1;
  void* C = nullptr; int64_t ldc = 0; int c_bf16 = 0;
  const float* bias = nullptr;
  int beta = 0;
  int rowmap_H = 0;
  int perm[4] = {0, 1, 2, 3};
  int in_bf16 = 1;            // operand element type (SIMT kernel takes fp32 too)
  // scratch the tcgen05 kernel may use to split K across CTAs (one fp32
  // partial per output tile, summed in split order); null: no split
  void* split_ws = nullptr;
  size_t split_ws_bytes = 0;
};

struct PersistArgs {
  int mode = 0, reset_after = 0, is_bf16 = 0;   // mode: rnn_mode_t (0 LSTM, 1 GRU, 2 / 3 plain ReLU / tanh)
  // LSTM cell clipping: every use of the (raw) cell state goes through
  // clip(x) = min(max(x, clip_lo), clip_hi)
  int clip = 0;
  float clip_lo = 0.f, clip_hi = 0.f;
  // valid steps per sequence ([B], device) or null = all T; step t of
  // sequence b is masked when t >= len[b] (state held, zero gate gradients)
  const int* len = nullptr;
  int T = 0, B = 0, H = 0, D = 1;   // D = directions of the layer (buffer strides)
  int dir0 = 0, ndir = 1;            // directions handled by this launch
  // forward
  const void* P = nullptr;
  const float* bh = nullptr;
  const void* Wr = nullptr;
  void* Y = nullptr;
  void* gates = nullptr;
  float* C = nullptr;
  void* RH = nullptr;
  const void* c0 = nullptr;          // [D][B, H] slice of cx for this layer
  void* hy = nullptr;                // [D][B, H]
  void* cy = nullptr;
  void* y_out = nullptr;             // tensor-core forward: also writes y_t to [T, B, D*H] (zero at masked steps)
  // backward
  const void* WrT = nullptr;
  const float* dYi = nullptr;        // [T, B, D*H]
  void* dG = nullptr;
  float* db = nullptr;
  const void* dhT = nullptr;         // [D][B, H] slice of dhy
  const void* dcT = nullptr;
  void* dh0 = nullptr;               // [D][B, H] slice of dhx
  void* dc0 = nullptr;
  // tensor-core GRU reset-before backward: [T, B, D*4H] operand of the step's
  // first exchange, rows [0, 0, dn, 0] per unit (the contraction W_hn^T dn)
  void* XA = nullptr;
  // recurrent weight gradient accumulated inside the backward kernel (SIMT
  // kernel only): [D][G*H][H] fp32 in the caller's gate blocks, internal slot s
  // of unit u -> row whh_map[s] * H + u (-1: the slot is no W_hh row); the
  // reset-before candidate rows take r * h_{t-1} from RH.  null = the weight
  // gradient is left to the GEMM of the backward-weights call
  float* dwhh = nullptr;
  int whh_map[4] = {-1, -1, -1, -1};
  // tensor-core backward without clusters: the K-split partials of every
  // row group, two exchange parities (persist_tc_bwd_gk_bytes)
  float* gk_buf = nullptr;
  DevArea* dev = nullptr;
  uint64_t timeout_ns = 2000000000ull;
  int skip_cta = -1;
};

// Host-side launch status: 0 = launched, otherwise an rnn_status_t value.
int launch_gemm_simt(const GemmArgs& g, cudaStream_t s);
// *launches (optional) receives the number of kernels launched (2 with a K split).
int launch_gemm_tc(const GemmArgs& g, cudaStream_t s, int num_sms, DevArea* dev, uint64_t timeout_ns,
                   int* launches = nullptr);
bool gemm_tc_supported(const GemmArgs& g);
// Up to 6 GEMMs with the same K and operand major-ness in one launch (their
// tiles share the grid); the split-K scratch of gs[0] serves all of them.
int launch_gemm_tc_grouped(const GemmArgs* gs, int n, cudaStream_t s, int num_sms, DevArea* dev,
                           uint64_t timeout_ns);
// Scratch bytes that let the tensor-core GEMM split the K of an M x N output.
size_t gemm_tc_split_scratch_bytes(int M, int N);

int plan_persist_simt(const PersistArgs& a, int num_sms, int* nblk, size_t* smem);
// Whether the SIMT backward kernel can accumulate dW_hh in its step loop for
// this shape (the per-step work small, the accumulator within shared memory);
// with hidden_only, also that the work hides behind the step exchange.
bool persist_simt_dwhh_ok(const PersistArgs& a, int num_sms, bool hidden_only);
int launch_persist_fwd_simt(const PersistArgs& a, cudaStream_t s, int num_sms);
int launch_persist_bwd_simt(const PersistArgs& a, cudaStream_t s, int num_sms);

// Batch parts the tensor-core backward may split a row group into; its bias
// gradients take one [D][4H] fp32 plane per part (the sum lands in plane 0).
constexpr int kMaxBatchParts = 4;
bool persist_tc_supported(int mode, int reset_after, int H, int B, int ndir, int num_sms);
// The forward kernel alone (a layer whose backward has no tensor-core plan).
bool persist_tc_fwd_supported(int mode, int reset_after, int H, int B, int ndir, int num_sms);
int launch_persist_fwd_tc(const PersistArgs& a, cudaStream_t s, int num_sms);
int launch_persist_bwd_tc(const PersistArgs& a, cudaStream_t s, int num_sms);
// Bytes of PersistArgs::gk_buf the tensor-core backward needs for this shape:
// 0 when its plan exchanges the K split within clusters.
size_t persist_tc_bwd_gk_bytes(int mode, int reset_after, int H, int B, int ndir, int num_sms);

// TMA tensor map (CUtensorMap, 128 bytes) over a bf16 row-major matrix
// ptr[j * ld + i], i < dim0, j < dim1, box box0 x box1, 128-byte swizzle.
int make_tmap_bf16_2d(void* map, const void* ptr, uint64_t dim0, uint64_t dim1, uint64_t ld_elems,
                      uint32_t box0, uint32_t box1, int swizzle_bytes = 128);
// 4-D view: element (i0..i3) at 2*i0 + i1*strides[0] + i2*strides[1] + i3*strides[2]
// bytes; box[0] * 2 == 128 (the swizzle span).
int make_tmap_bf16_4d(void* map, const void* ptr, const uint64_t* dims, const uint64_t* strides_bytes,
                      const uint32_t* box);

// layout / cast / pack kernels (layout.cu)
// Sequence copy [T,B,F] <-> [B,T,F] with casts; len (optional, device [B]):
// output rows (t, b) with t >= len[b] are zero.
int launch_seq_transpose(const void* in, void* out, int T, int B, int F, int in_bf16,
                         int out_bf16, int in_batch_first, int out_batch_first,
                         int64_t out_ld, cudaStream_t s, const int* len = nullptr);
// Several layout jobs in one launch (the forward's weight / bias packing and
// h0 placement, the backward's transposed packing, the bias-gradient scatter).
enum PackKind { PACK_ROWS = 0, PACK_ROWS_T = 1, PACK_BIAS = 2, SCATTER_DB = 3, H0_TO_Y = 4 };
struct PackJob {
  int kind = PACK_ROWS;
  int H = 0, K = 0;
  // PACK_*: internal slot -> caller gate block to read; SCATTER_DB: slot ->
  // caller block to write; -1: zero / skipped
  int map[4] = {-1, -1, -1, -1};
  const void* in = nullptr;   // may be null for PACK_BIAS (zeros) and H0_TO_Y (zero state)
  void* out = nullptr;
  int64_t ld_out = 0;         // PACK_ROWS / PACK_ROWS_T row stride of out
  int T = 0, B = 0, D = 1, dir = 0;   // H0_TO_Y
};
constexpr int kMaxPackJobs = 12;
struct PackBatch {
  int n = 0;
  PackJob job[kMaxPackJobs];
  bool add(const PackJob& j) {
    if (n >= kMaxPackJobs) return false;
    job[n++] = j;
    return true;
  }
};
int launch_pack_batch(const PackBatch& pb, int is_bf16, cudaStream_t s);
int launch_fill_zero(void* p, size_t bytes, cudaStream_t s);
// LSTM cell states c_t of every step from the saved gate activations
// ([D][T, B, 4H], slots i, f, g, o) and c0 ([D, B, H] or null = zero) into C
// ([D][T+1, B, H] fp32, the forward kernels' layout); len / clip as in
// PersistArgs.
int launch_recompute_cells(const void* gates, const void* c0, float* C, int T, int B, int H, int D, int is_bf16,
                           const int* len, int clip, float lo, float hi, cudaStream_t s);

// Plan overrides set by the rnn_debug_set_plan_overrides test hook (0 = the
// planner's choice): K-split caps and batch parts of the tensor-core
// persistent kernels, the tensor-core GEMM's tile width and K split.
struct PlanOverrides {
  int max_ks_fwd, max_ks_bwd, nb_fwd, nb_bwd, gemm_bn, gemm_splits, gemm_tm;
  int bwd_global_ks;           // 1: the tensor-core backward exchanges its K split through global memory
};
PlanOverrides plan_overrides();

}  // namespace rnn
