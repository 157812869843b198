// handle.h - the library handle's host-side state (shared by the C-ABI
// translation units).
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "rnn.h"
#include "rnn_internal.h"

struct rnn_handle_s {
  using DevArea = rnn::DevArea;
  rnn_desc_t desc;
  int L, D, T, B, H, I, G;
  int lstm, ra, rb, plain, bf16, bfirst;   // plain: RNN_RNN_RELU / RNN_RNN_TANH (one gate)
  int pos[4];          // canonical gate c sits in the caller's block pos[c]
  int algo;            // RNN_ALGO_PERSIST_TC or RNN_ALGO_PERSIST_SIMT
  int fwd_tc;          // the forward runs the tensor-core kernel (also when algo is SIMT: a
                       // shape whose backward has no tensor-core plan)
  int device, num_sms;
  size_t es;
  DevArea* dev;
  uint64_t timeout_ns;
  int skip_cta;
  uint64_t launches;
  int* d_len;                  // device copy of the sequence lengths (B ints), or null
  int has_len;                 // 1: the lengths in d_len apply
  int recompute;               // LSTM: no cell states in the reserve; the backward recomputes them
  int dw_mode;                 // interleaved dW_hh: 0 never, 1 where the SIMT backward kernel hides it, 2 where it fits
  int dw_bptt;                 // 1: rnn_backward_data accumulates dW_hh into the reserve
  int clip;                    // LSTM cell clipping on, bounds [clip_lo, clip_hi]
  float clip_lo, clip_hi;
  bool trace;
  bool timing;
  struct Ev { cudaEvent_t a, b; int cls; double bytes; };
  std::vector<Ev> events;      // recorded, not yet read
  std::vector<Ev> pool;        // created, free
  // weight offsets (elements), per layer and direction
  std::vector<size_t> off_ih, off_hh, off_b, off_bh;
  size_t weight_elems;
  // reserve offsets (bytes), per layer
  std::vector<size_t> r_y, r_g, r_c, r_rh, r_dg, r_db, r_dwhh;
  size_t reserve_bytes;
  // workspace offsets (bytes)
  size_t w_p, w_xin, w_dyi, w_dx0, w_wx, w_wxt, w_wr, w_wrt, w_bx, w_bh, w_y0, w_y1, w_rh, w_g;
  size_t w_gk, gk_bytes;       // tensor-core backward: K-split partials through global memory (0: none)
  size_t workspace_bytes;
};


namespace rnn {
// Host-side initialisation of a handle for ``desc`` on the current device
// (validation, layout, kernel choice); allocates no device memory and leaves
// h->dev unset.  Returns an rnn_status_t.
int init_handle_host(rnn_handle_s* h, const rnn_desc_t* desc);
}  // namespace rnn
