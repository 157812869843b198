/*
 * rnn_debug.h - test hooks of librnn.so: the library's internal GEMM, run
 * directly so tests can check it element by element in isolation, the
 * tensor-core planner's candidate ranking, plan overrides that force a kernel
 * configuration, and a withheld arrival that exercises the timeout path.
 * None of them is needed in normal use.
 *
 * C[row(m), n] = sum_k A(m,k) B(n,k) (+ bias[n]) (+ C if beta != 0)
 *   A(m,k) = A[m*lda + k] when a_kmajor, else A[k*lda + m] (same for B, n)
 *   row(m) = m, or with rowmap_H > 0: m = 4u + s -> perm[s]*rowmap_H + u
 *   (rows with perm[s] < 0 are not written) - the gate-slot remap the weight
 *   gradients use.
 * A, B: device, in_bf16 ? bf16 : fp32.  C: device, c_bf16 ? bf16 : fp32.
 * bias: device fp32 [N] or NULL.  use_tc = 1 runs the tcgen05 kernel (bf16
 * operands, 16-byte aligned pointers and row strides), 0 the SIMT kernel.
 * Asynchronous on ``stream``; returns an rnn_status_t.  A test hook: its
 * split-K scratch and status area are allocated on first use on the device
 * current then and kept for the process, so call it from one thread and on
 * one device only.
 */
#ifndef GB300_RNN_DEBUG_H
#define GB300_RNN_DEBUG_H

#include <stdint.h>
#include "rnn.h"

#ifdef __cplusplus
extern "C" {
#endif

rnn_status_t rnn_debug_gemm(int M, int N, int K, const void* A, int64_t lda, int a_kmajor, const void* B,
                            int64_t ldb, int b_kmajor, void* C, int64_t ldc, int c_bf16, const float* bias,
                            int beta, int rowmap_H, const int* perm, int in_bf16, int use_tc, void* stream);

/* Planner hook: the candidate plans of the tensor-core persistent kernel for
 * one launch shape, cheapest first by the per-step cost estimate, before the
 * launch-time check that their clusters can all be resident (host arithmetic
 * only; needs no GPU).  mode: rnn_mode_t; bwd: 0 forward, 1 backward; ndir:
 * directions in the launch; num_sms: SMs of the device.  For candidate i,
 * out[7*i ...] = {K split (CTAs per cluster), batch parts, CTAs, padded
 * batch rows per part, pairs per thread (1/2/4/8), weight sub-tiles held in
 * tensor memory, shared memory bytes}.  Returns the number of candidates
 * written (at most max_out). */
int rnn_debug_tc_plans(int mode, int bwd, int hidden, int batch, int ndir, int num_sms, int* out, int max_out);

/* Planner hook: the tensor-core GEMM's plan for one grouped launch (host
 * arithmetic only): n GEMMs (1..6) of M[i] x N[i] with the common depth K;
 * fp32_out != 0: fp32 outputs with ws_bytes of split-K scratch (0: no K
 * split), else bf16 outputs.  out[0..2] = {tile width (128 or 256), K split,
 * tile rows (128 or 256)}.  Returns 1, or 0 for invalid arguments. */
int rnn_debug_gemm_plan(int n, const int* M, const int* N, int K, int fp32_out, size_t ws_bytes, int num_sms,
                        int* out);

/* Planner hook: the SIMT persistent kernel's plan for one launch shape (host
 * arithmetic only).  dwhh != 0 plans with the interleaved dW_hh accumulator.
 * out[0..6] = {units per CTA, CTAs per direction, pairs per thread, weights
 * streamed (1) or resident (0), shared memory bytes, interleaved dW_hh taken
 * by default (mode 1), interleaved dW_hh possible at all (mode 2)}.  Returns 1,
 * or 0 when the kernel cannot take the shape. */
int rnn_debug_simt_plan(int mode, int reset_after, int is_bf16, int bwd, int hidden, int batch, int ndir,
                        int num_sms, int dwhh, int* out);

/* Test hook for the timeout path: CTA ``cta`` (>= 0) of the next persistent
 * launches of this handle skips its per-step arrival, so its peers' bounded
 * waits run out and the call ends with RNN_TIMEOUT instead of hanging.
 * -1 (default) = off.  RNN_BAD_PARAM for a NULL handle or cta < -1. */
rnn_status_t rnn_debug_skip_arrival(rnn_handle_t handle, int cta);

/* Test hook: process-wide overrides of the kernel plans, for tests that must
 * reach a given configuration.  0 leaves a choice to the planner.
 *   max_ks_fwd, max_ks_bwd  1..16: cap the tensor-core persistent kernels' K
 *                           split (CTAs per cluster), forward / backward;
 *   nb_fwd, nb_bwd          1, 2 or 4: fix their number of batch parts;
 *   gemm_bn                 128 or 256: force the tensor-core GEMM's tile
 *                           width (no K split);
 *   gemm_splits             1..16: force the K split of a tensor-core GEMM
 *                           with fp32 output and split scratch (256-wide
 *                           tiles), where it has at least 16 K blocks of 64
 *                           per split;
 *   gemm_tm                 128 or 256: force the tensor-core GEMM's tile
 *                           rows (256 rows go with 256-wide tiles, so 256
 *                           together with gemm_bn 128 is rejected);
 *   bwd_global_ks           1: the tensor-core backward exchanges its K-split
 *                           partials through global memory (no thread-block
 *                           clusters), as it does by itself only where no
 *                           cluster plan can be resident.  Takes effect for
 *                           handles created after it is set (the workspace
 *                           size depends on it).
 * Other values are RNN_BAD_PARAM and change nothing.  Plans are cached per
 * shape and per override set; set the overrides while no call of the library
 * runs on another thread. */
rnn_status_t rnn_debug_set_plan_overrides(int max_ks_fwd, int max_ks_bwd, int nb_fwd, int nb_bwd, int gemm_bn,
                                          int gemm_splits, int gemm_tm, int bwd_global_ks);

#ifdef __cplusplus
}
#endif

#endif /* GB300_RNN_DEBUG_H */
