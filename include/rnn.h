/*
 * rnn.h - C ABI of the GB300 (sm_103a) multi-timestep LSTM / GRU library.
 *
 * One layer stack (1..8 layers, uni- or bidirectional) of LSTM, GRU or plain
 * RNN cells, run forward over a whole sequence and back-propagated through
 * time.  The
 * three-phase split (forward, backward-data, backward-weights) follows the
 * SystemDS LibMatrixCuDNN.java page (its LSTM forward and backward operators
 * run cuDNN's forward-training, backward-data and backward-weights calls) and
 * the forward, backward and weight-update entry points of the popnn Lstm.cpp
 * and Gru.cpp pages (Graphcore poplibs).
 *
 * Cell definitions (canonical gate order; sigma = logistic sigmoid):
 *   LSTM (the popnn Lstm.cpp page, forward cell step):
 *     a = W_ih x_t + W_hh h_{t-1} + b
 *     i = sigma(a_i), f = sigma(a_f), g = tanh(a_g), o = sigma(a_o)
 *     c_t = f c_{t-1} + i g,  h_t = o tanh(c_t)
 *   GRU resetAfter (the popnn Gru.cpp page, resetAfter forward cell step):
 *     r = sigma(W_ir x + b_ir + W_hr h + b_hr), z = sigma(W_iz x + b_iz + W_hz h + b_hz)
 *     n = tanh(W_in x + b_in + r * (W_hn h + b_hn)),  h_t = (1 - z) n + z h_{t-1}
 *   GRU reset-before (the popnn Gru.cpp page, reset-before forward cell step):
 *     r, z as above with one bias b_r, b_z;  n = tanh(W_in x + b_n + W_hn (r * h_{t-1}))
 *     h_t = (1 - z) n + z h_{t-1}
 * Backward: the BPTT recurrences of the backward steps of the popnn Lstm.cpp
 * and Gru.cpp pages (identical to the LSTM and GRU branches of the persistent
 * RNN backward-data kernel page), and the weight-gradient sums of their weight
 * updates.
 *
 * Conventions shared by every call
 *   - All pointers marked "device" are device memory owned by the caller; the
 *     library never frees them.  The handle owns only host metadata and a small
 *     device area (status word, step counters) allocated in rnn_create.
 *   - A handle belongs to the device that was current in rnn_create.  Each
 *     call that touches the GPU makes that device current for its duration
 *     and restores the caller's current device before it returns; ``stream``
 *     and every device pointer must belong to that device.
 *   - Calls are asynchronous on ``stream`` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).  Errors found on the host are returned;
 *     errors found on the device (a spin-wait that ran out, RNN_TIMEOUT) are
 *     recorded in the handle's status word and returned by rnn_sync_status.
 *   - No call throws or aborts; every failure is a status code.
 *   - One handle serves one host thread at a time; different handles may be
 *     used from different threads (the library's shared plan caches are
 *     locked).  The recurrent kernels are persistent grids sized to be
 *     resident at once on an otherwise idle GPU: a call that overlaps other
 *     kernels holding SMs (another handle's calls on a concurrent stream,
 *     another client under MPS) may find some of its CTAs not resident, and
 *     its waits then end in RNN_TIMEOUT rather than a hang.  Order such
 *     calls on one stream.
 *   - Sequences are seq-major [T, B, F] unless desc.batch_first != 0, in which
 *     case x, y, dy and dx are [B, T, F].  States (hx, cx, hy, cy, dhy, dcy,
 *     dhx, dcx) are [L*D, B, H] with index l*D + d (d = 0 forward, 1 reverse).
 *     A bidirectional layer's output row is [y_fwd (H) | y_bwd (H)].
 *   - Element type of x, y, dy, dx, w and all states is desc.dtype (fp32 or
 *     bf16).  Accumulation and the cell state are always fp32.  dw is fp32.
 *   - State pointers may be NULL: NULL inputs (hx, cx, dhy, dcy) mean zero,
 *     NULL outputs (hy, cy, dhx, dcx) are skipped - the same convention as the
 *     ``cx == NULL`` / ``dhx != NULL`` tests of the persistent RNN
 *     backward-data kernel page and the absent final-state gradient of the
 *     SystemDS LibMatrixCuDNN.java page's LSTM backward operator.
 *   - Every device pointer must be 16-byte aligned.
 *
 * Environment variables (read by the library; none is needed in normal use)
 *   RNN_TRACE=1            stderr: each recurrent-kernel plan when it is first
 *                          chosen for a shape (grid, K split, batch parts,
 *                          shared memory), and the device status record
 *                          (kernel, block, step, wait) when rnn_sync_status
 *                          finds an error.
 * The status-record part of RNN_TRACE is fixed at rnn_create.
 */
#ifndef GB300_RNN_H
#define GB300_RNN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RNN_OK = 0,
  RNN_BAD_PARAM = 1,       /* a descriptor field or pointer is invalid         */
  RNN_NOT_SUPPORTED = 2,   /* valid, but the library or GPU cannot run it      */
  RNN_CUDA_ERROR = 3,      /* a CUDA runtime / driver call failed              */
  RNN_TIMEOUT = 4,         /* a device spin-wait gave up (see rnn_sync_status) */
  RNN_BAD_WORKSPACE = 5,   /* workspace / reserve pointer NULL or misaligned   */
  RNN_INTERNAL = 6
} rnn_status_t;

/* RNN_RNN_RELU / RNN_RNN_TANH: the plain recurrent cell h' = act(W_ih x +
 * W_hh h + b) of the persistent RNN backward-data kernel page's ReLU / tanh
 * branch (one gate, G = 1). */
typedef enum { RNN_LSTM = 0, RNN_GRU = 1, RNN_RNN_RELU = 2, RNN_RNN_TANH = 3 } rnn_mode_t;
typedef enum { RNN_F32 = 0, RNN_BF16 = 1 } rnn_dtype_t;

/* Recurrent-kernel choice.  AUTO picks the tensor-core persistent kernels
 * (bf16 LSTM and GRU whose W_hh slices fit on chip; GRU reset-before from
 * batch 4) and the SIMT persistent kernels otherwise (every fp32 problem,
 * plain RNN cells, GRU reset-before below batch 4, shapes the tensor-core
 * kernels do not take); with AUTO the
 * forward alone may still run on the tensor cores (see
 * rnn_selected_fwd_algo).  The two explicit values force one kernel family
 * for both passes. */
typedef enum { RNN_ALGO_AUTO = 0, RNN_ALGO_PERSIST_TC = 1, RNN_ALGO_PERSIST_SIMT = 2 } rnn_algo_t;

typedef struct {
  int mode;            /* rnn_mode_t                                                */
  int gate_order[4];   /* block k of every per-gate matrix holds canonical gate
                          gate_order[k] (LSTM 0..3 = i,f,g,o; GRU 0..2 = r,z,n;
                          plain RNN: one gate, only 0).  All zero = canonical.      */
  int reset_after;     /* 0 or 1; GRU only: 1 = resetAfter form, 0 = reset-before */
  int bidirectional;   /* 0 or 1                                                    */
  int num_layers;      /* 1..8                                                      */
  int seq_len;         /* T >= 1                                                    */
  int batch;           /* B >= 1                                                    */
  int input_size;      /* I >= 1 (layer 0 input; later layers take D*H)             */
  int hidden_size;     /* H >= 1                                                    */
  int dtype;           /* rnn_dtype_t                                               */
  int batch_first;     /* 0 = [T,B,F], 1 = [B,T,F] for x, y, dy, dx                 */
  int algo;            /* rnn_algo_t                                                */
} rnn_desc_t;

typedef struct rnn_handle_s* rnn_handle_t;

/* Validate ``desc`` and make a handle.  Allocates the handle's small device
 * area on the current device (which the handle is then bound to).
 * Returns RNN_BAD_PARAM for an invalid descriptor (a field outside the range
 * given above, a gate_order that is not a permutation of 0..G-1, or
 * seq_len * batch above 2^30), checked before any device call;
 * RNN_NOT_SUPPORTED when input_size or hidden_size is not a multiple of 8
 * (bf16) or 4 (fp32) - rows are moved in 16-byte vectors - when the current
 * GPU is not sm_103, or when the forced algo cannot take the shape;
 * RNN_CUDA_ERROR when the device allocation fails (no device included).
 * ``*handle`` is NULL after any failure. */
rnn_status_t rnn_create(const rnn_desc_t* desc, rnn_handle_t* handle);

/* Free the handle and its device area.  NULL is accepted. */
rnn_status_t rnn_destroy(rnn_handle_t handle);

/* Byte sizes the caller must allocate (device memory, 256-byte aligned):
 *   weight_bytes    - the packed weight buffer w (desc.dtype elements); dw
 *                     has the same element count at 4 bytes per element.
 *                     Per layer l, per direction d, in this order:
 *                     W_ih [G*H, I_l] row-major, W_hh [G*H, H], b [G*H], and
 *                     for GRU resetAfter b_h [G*H].  G = 4 (LSTM), 3 (GRU) or
 *                     1 (plain RNN);
 *                     gate blocks in desc.gate_order.  LSTM and GRU
 *                     reset-before have one bias vector per direction.
 *   workspace_bytes - scratch for any one call; contents need not persist.
 *   reserve_bytes   - state kept from rnn_forward (training) to the two
 *                     backward calls, and from rnn_backward_data to
 *                     rnn_backward_weights; must not be touched in between.
 * Any output pointer may be NULL. */
rnn_status_t rnn_get_sizes(rnn_handle_t handle, size_t* weight_bytes,
                           size_t* workspace_bytes, size_t* reserve_bytes);

/* Forward over the whole sequence.
 *   x  [T,B,I] (device, in)         hx, cx [L*D,B,H] (device, in, may be NULL)
 *   w  weight_bytes (device, in)    y  [T,B,D*H] (device, out)
 *   hy, cy [L*D,B,H] (device, out, may be NULL; cy and cx are LSTM only)
 *   workspace (device, workspace_bytes, scratch)
 *   reserve (device, reserve_bytes, out) - NULL runs inference: nothing is
 *     kept for a backward pass.
 * cx is ignored for GRU. */
rnn_status_t rnn_forward(rnn_handle_t handle, const void* x, const void* hx, const void* cx,
                         const void* w, void* y, void* hy, void* cy,
                         void* workspace, void* reserve, void* stream);

/* Backward through time (data gradients).  Needs the reserve written by
 * rnn_forward with the same x, hx, cx and w.
 *   y     forward output; accepted for interface symmetry, the reserve holds
 *         the copy the kernels read (may be NULL)
 *   dy    [T,B,D*H] (device, in)     dhy, dcy [L*D,B,H] (device, in, may be NULL)
 *   w     (device, in)               hx: accepted for symmetry (may be NULL)
 *   cx    (device, in, may be NULL = zero) read only with recomputation
 *         (rnn_set_recomputation): it must then be the cx of rnn_forward
 *   dx    [T,B,I] (device, out)      dhx, dcx [L*D,B,H] (device, out, may be NULL)
 * Writes the gate and bias gradients into the reserve for
 * rnn_backward_weights. */
rnn_status_t rnn_backward_data(rnn_handle_t handle, const void* y, const void* dy,
                               const void* dhy, const void* dcy, const void* w,
                               const void* hx, const void* cx, void* dx, void* dhx,
                               void* dcx, void* workspace, void* reserve, void* stream);

/* Weight gradients dW_ih = sum_t dA_t x_t^T, dW_hh = sum_t dA^h_t h_{t-1}^T,
 * db = sum_t dA_t (GRU resetAfter also db_h = sum_t dA^h_t), summed over the
 * batch, written (overwritten, never accumulated) into dw: fp32, same layout
 * as w.  Needs the reserve after rnn_backward_data.  x (device, in, not NULL)
 * is read: it is the input operand of layer 0's dW_ih, and must be the x of
 * rnn_forward.  hx, y: accepted for symmetry with cuDNN's backward-weights
 * call (may be NULL); the reserve holds the states and gate gradients that are
 * read. */
rnn_status_t rnn_backward_weights(rnn_handle_t handle, const void* x, const void* hx,
                                  const void* y, void* workspace, const void* reserve,
                                  void* dw, void* stream);

/* Synchronise ``stream`` and return (then clear) the device status word:
 * RNN_OK, or RNN_TIMEOUT when a persistent kernel's bounded spin-wait gave up
 * (its outputs are then invalid), or RNN_CUDA_ERROR. */
rnn_status_t rnn_sync_status(rnn_handle_t handle, void* stream);

/* Upper bound, in nanoseconds, of every device spin-wait (default 2 s). */
rnn_status_t rnn_set_timeout_ns(rnn_handle_t handle, uint64_t ns);

/* Variable sequence lengths (the popnn Gru.cpp and Lstm.cpp pages: the
 * batchwise time-step limit of the forward and backward loops).  ``lengths``: host
 * array of desc.batch ints, each in [0, seq_len]; sequence b then has
 * lengths[b] valid steps, and at every later step t >= lengths[b] (in time
 * order, for both directions) the step is masked: the state h (and c) is
 * carried unchanged, the output y_t is zero, and in the backward calls the
 * state gradients pass through the step while its gate gradients are zero
 * (so padded positions contribute nothing to dx, dW and db, and dy there is
 * ignored).  hy / cy are the states after each sequence's last valid step;
 * the reverse direction starts from hx at t = lengths[b] - 1.
 * NULL restores full length for every sequence.  The lengths apply to the
 * following rnn_forward / rnn_backward_data calls (which must see the same
 * lengths) and are copied synchronously to the handle's device memory, so
 * call this between uses of the handle.  Returns RNN_BAD_PARAM for a length
 * outside [0, seq_len], RNN_CUDA_ERROR if the copy fails. */
rnn_status_t rnn_set_seq_lengths(rnn_handle_t handle, const int* lengths);

/* Recomputation (the popnn Lstm.cpp page's recomputation mode that rebuilds
 * the cell state and its tanh in the backward pass).
 * mode 1: the LSTM forward keeps no cell states in the reserve (smaller by
 * num_layers * D * (seq_len+1) * batch * hidden * 4 bytes); rnn_backward_data
 * recomputes them from the saved gate activations (c_t = f * c_{t-1} + i * g,
 * with the cell clipping and sequence lengths in force) before each layer's
 * backward pass, into its workspace, and tanh(c_t) is recomputed in the
 * backward step as always.  rnn_backward_data must then receive the same cx
 * as rnn_forward.  mode 0 (the default) stores the cell states.  A GRU or
 * plain-RNN handle has no cell state and ignores the mode.  Changes the sizes
 * rnn_get_sizes reports: set it before allocating.  RNN_BAD_PARAM for other
 * modes. */
rnn_status_t rnn_set_recomputation(rnn_handle_t handle, int mode);

/* LSTM cell clipping (the clip / dclip of the persistent RNN backward-data
 * kernel page's LSTM branch).  With enable != 0 and lo < hi the cell state stays
 * the raw value c, and every use of it goes through clip(x) = min(max(x, lo),
 * hi) (a NaN stays NaN): c_t = f * clip(c_{t-1}) + i * g and
 * h_t = o * tanh(clip(c_t)); cy is the raw c_T; the backward uses
 * dclip(x) = 1 on [lo, hi], 0 outside.  enable = 0 turns it off (the
 * default).  Applies to the following forward / backward calls, which must
 * agree.  RNN_BAD_PARAM for a non-LSTM handle or lo >= hi. */
rnn_status_t rnn_set_cell_clip(rnn_handle_t handle, int enable, double lo, double hi);

/* Interleaved weight update (the popnn Lstm.cpp and Gru.cpp pages' interleaved
 * weight update: the weight gradients accumulated inside the backward loop).
 * Where the SIMT persistent backward kernel runs the layers and its per-step
 * share of the recurrent weight gradient is small (units per CTA x hidden x
 * batch <= 16384 multiply-adds; small layers and batches), rnn_backward_data
 * can accumulate dW_hh in fp32 step by step inside that kernel into the
 * reserve, and rnn_backward_weights then copies it to dw instead of running
 * the dW_hh GEMM; dW_ih and the biases are unchanged.  The result is the same
 * sum in another summation order.
 *   mode 0: always the GEMM;
 *   mode 1 (the default): interleaved where, in addition, the work hides
 *     behind the wait for the step exchange: each direction spans several
 *     CTAs (a lone CTA has nothing to hide it behind) and each thread's
 *     per-step share is at most 16 batch-length passes over its (unit,
 *     column) items;
 *   mode 2: interleaved wherever the kernel can.
 * Changes the reserve size rnn_get_sizes reports (by num_layers * D * G *
 * hidden^2 * 4 bytes when active): set it before allocating.  RNN_BAD_PARAM
 * for other modes. */
rnn_status_t rnn_set_interleaved_dw(rnn_handle_t handle, int mode);

/* 1 when rnn_backward_data accumulates dW_hh (see rnn_set_interleaved_dw),
 * else 0. */
int rnn_interleaved_dw_active(rnn_handle_t handle);

/* Number of kernels this handle has launched since it was created. */
uint64_t rnn_launch_count(rnn_handle_t handle);

/* Which recurrent kernel the handle runs: 1 = tensor-core persistent,
 * 2 = SIMT persistent (rnn_algo_t values). */
int rnn_selected_algo(rnn_handle_t handle);

/* Which recurrent kernel the forward runs (rnn_algo_t values).  Equal to
 * rnn_selected_algo except where the automatic choice runs the forward on the
 * tensor-core kernel and the backward on the SIMT kernel: a bf16 LSTM or GRU
 * layer whose backward has no tensor-core plan (a hidden size that is a
 * multiple of 64 but not of 128: the forward's K slices fit, the backward's
 * 128-unit row groups do not).  Hidden 2048 runs both on tensor cores (the
 * backward exchanging its K split through global memory). */
int rnn_selected_fwd_algo(rnn_handle_t handle);

/* Per-kernel-class timing with CUDA events recorded on the launching stream
 * around every launch (off by default; costs two event records per launch).
 * Classes: 0 persistent forward, 1 persistent backward, 2 input-projection
 * GEMM, 3 input-gradient GEMM, 4 weight-gradient GEMMs (with their split-K
 * reduction), 5 sequence layout copies / casts (batch-first transposes, the
 * upstream gradient's fp32 copy, y out), 6 weight / bias / state packing and
 * the bias-gradient scatter, 7 the cell-state recomputation sweep.
 * rnn_get_timing waits for the recorded events, writes the summed
 * milliseconds (ms[8]) and launch counts (n[8]) since the last read, and
 * clears them.  rnn_get_timing_ex also writes, per class, the algorithmic
 * bytes of the timed launches (bytes[8]: every element read once and written
 * once at its storage size; 0 for the classes that are bound by arithmetic,
 * 0 to 4).  Any output pointer may be NULL. */
#define RNN_TIMING_CLASSES 8
rnn_status_t rnn_set_timing(rnn_handle_t handle, int enable);
rnn_status_t rnn_get_timing(rnn_handle_t handle, double* ms, uint64_t* n);
rnn_status_t rnn_get_timing_ex(rnn_handle_t handle, double* ms, uint64_t* n, double* bytes);

/* Inference forward that allocates nothing on the device.
 *
 * The paper has no counterpart; this entry point exists for callers that
 * cannot let a library call cudaMalloc - a process whose device memory is all
 * pre-reserved by its own allocator or a framework's caching pool, or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device
 * synchronisation.  It computes what rnn_forward computes with reserve == NULL
 * (same kernels, same results) but takes no handle and no workspace: its
 * scratch is a fixed array of RNN_NOALLOC_SCRATCH_BYTES built into the library,
 * which every GPU that loads the library holds until the process exits.
 *   desc                  as for rnn_create
 *   x, hx, cx, w, y, hy, cy  as for rnn_forward (caller-owned device memory)
 *   sync                  nonzero: synchronise ``stream`` and return the
 *                         device status (RNN_TIMEOUT when a spin-wait gave up);
 *                         zero: return once the work is queued - a device
 *                         timeout of that call is then reported only by
 *                         rnn_noalloc_status, which must run before the next
 *                         call on the device (each call clears the status)
 * Returns RNN_NOT_SUPPORTED when the problem's workspace plus 1 KB of
 * counters exceeds RNN_NOALLOC_SCRATCH_BYTES (nothing is launched then).
 * The first call on each device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  All calls share the array, which keeps the last call's contents:
 * the counters and status are cleared by each call; calls that overlap on the
 * GPU race on the array and must be serialised by the caller. */
#define RNN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
rnn_status_t rnn_forward_noalloc(const rnn_desc_t* desc, const void* x, const void* hx, const void* cx,
                                 const void* w, void* y, void* hy, void* cy, int sync, void* stream);

/* Status of the last rnn_forward_noalloc call on the current device: waits
 * for ``stream`` (the stream that call used), reads the device status word
 * (RNN_OK, or RNN_TIMEOUT when a spin-wait of that call gave up, in which case
 * its y / hy / cy are incomplete) and clears it.  Allocates nothing.
 * RNN_OK when no call has run on this device yet; RNN_CUDA_ERROR when the
 * stream cannot be synchronised. */
rnn_status_t rnn_noalloc_status(void* stream);

/* Static text for a status code. */
const char* rnn_status_string(rnn_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* GB300_RNN_H */
