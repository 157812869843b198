"""rnn_forward_noalloc against rnn_forward, on the GPU.

rnn_forward_noalloc is the inference forward for callers that cannot let a
library allocate device memory (their device memory is pre-reserved by their
own allocator or a caching pool, or they cannot afford cudaMalloc's implicit
synchronisation).  It keeps its scratch in a fixed array inside librnn.so.
This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It must pass both alone in a
fresh process and after the other tests (which leave the shared scratch array
holding whatever their last call wrote)."""
import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

AREA = 1024  # the counters and status word in front of the workspace


def _desc(R, wl):
    d = R.rnn_desc_t()
    d.mode = R.RNN_LSTM if wl.mode == "lstm" else R.RNN_GRU
    d.reset_after = int(wl.reset_after)
    d.bidirectional = int(wl.bidirectional)
    d.num_layers, d.seq_len, d.batch = wl.num_layers, wl.seq_len, wl.batch
    d.input_size, d.hidden_size = wl.input_size, wl.hidden_size
    d.dtype = R.RNN_BF16 if wl.dtype == "bf16" else R.RNN_F32
    return d


def _workspace_bytes(R, wl):
    rnn = R.RNN(wl.mode, wl.input_size, wl.hidden_size, wl.seq_len, wl.batch, wl.num_layers, wl.bidirectional,
                wl.reset_after, wl.dtype)
    try:
        return rnn.workspace_bytes
    finally:
        rnn.close()


def _near_limit_workload(R):
    """A bf16 LSTM whose workspace is the largest of its family (sequence
    length varied) that still fits the fixed scratch, and the same shape one
    step longer than fits."""
    base = synth.Workload("na_lstm_near", "lstm", False, 1, False, 8, 48, 256, 256, "bf16", 93, state_std=0.5)
    import dataclasses
    fits, over = None, None
    lo, hi = 1, 4096
    while lo <= hi:                              # workspace grows with the sequence length
        mid = (lo + hi) // 2
        wl = dataclasses.replace(base, seq_len=mid)
        if _workspace_bytes(R, wl) + AREA <= R.RNN_NOALLOC_SCRATCH_BYTES:
            fits, lo = wl, mid + 1
        else:
            over, hi = wl, mid - 1
    return fits, over


def _compare_two_calls(R, wl, inp):
    import torch
    w = Hn.to_dev(synth.flatten_params(wl, inp.params), wl)
    x = Hn.to_dev(inp.x, wl)
    hx, cx = Hn.to_dev(inp.h0, wl), Hn.to_dev(inp.c0, wl)
    # existing entry point (handle + caller workspace), inference
    rnn = R.RNN(wl.mode, wl.input_size, wl.hidden_size, wl.seq_len, wl.batch, wl.num_layers, wl.bidirectional,
                wl.reset_after, wl.dtype)
    try:
        y_ref, hy_ref, cy_ref = rnn.forward(x, w, hx, cx, train=False)
        rnn.sync()
    finally:
        rnn.close()
    tol = Hn.TOL[wl.dtype]
    desc = _desc(R, wl)
    stream = torch.cuda.current_stream().cuda_stream
    outs = [(torch.full_like(y_ref, float("nan")), torch.full_like(hy_ref, float("nan")),
             torch.full_like(cy_ref, float("nan")) if cy_ref is not None else None) for _ in range(2)]
    torch.cuda.synchronize()
    free = []
    for y, hy, cy in outs:
        rc = R.rnn_forward_noalloc(desc, x.data_ptr(), hx.data_ptr() if hx is not None else None,
                                   cx.data_ptr() if cx is not None else None, w.data_ptr(), y.data_ptr(),
                                   hy.data_ptr(), cy.data_ptr() if cy is not None else None, 1, stream)
        assert rc == R.RNN_OK, R.rnn_status_string(rc)
        free.append(torch.cuda.mem_get_info()[0])
        assert Hn.max_rel_err(Hn.to_np(y), Hn.to_np(y_ref)) <= tol
        assert Hn.max_rel_err(Hn.to_np(hy), Hn.to_np(hy_ref)) <= tol
        if cy is not None:
            assert Hn.max_rel_err(Hn.to_np(cy), Hn.to_np(cy_ref)) <= tol
    return free


@pytest.mark.parametrize("wl", [
    synth.Workload("na_lstm", "lstm", False, 2, True, 9, 20, 72, 128, "bf16", 91, state_std=0.5),
    synth.Workload("na_gru", "gru", True, 1, False, 7, 5, 12, 16, "f32", 92, state_std=0.5),
    # the tensor-core forward with batch parts
    synth.Workload("na_lstm_parts", "lstm", False, 1, False, 6, 300, 64, 128, "bf16", 94, state_std=0.5),
    # GRU reset-before: its r * h buffer lives in the scratch too
    synth.Workload("na_gru_rb", "gru", False, 1, True, 8, 16, 48, 128, "bf16", 95, state_std=0.5),
], ids=lambda w: w.name)
def test_noalloc_forward_matches_rnn_forward_on_two_calls(wl):
    import bwd_persistent_cta_gb300 as R
    from bwd_persistent_cta_gb300 import build
    build.build()
    _compare_two_calls(R, wl, synth.make_inputs(wl))


def test_noalloc_near_the_limit_and_allocates_nothing():
    import torch
    import bwd_persistent_cta_gb300 as R
    from bwd_persistent_cta_gb300 import build
    build.build()
    fits, over = _near_limit_workload(R)
    assert fits is not None and over is not None and over.seq_len == fits.seq_len + 1
    assert _workspace_bytes(R, fits) + AREA > R.RNN_NOALLOC_SCRATCH_BYTES * 0.95
    # the first call has looked up the scratch (the library image is loaded);
    # a call allocates no device memory: free memory is the same after the
    # first and the second call
    free = _compare_two_calls(R, fits, synth.make_inputs(fits))
    assert free[0] == free[1]
    # one step longer does not fit: rejected before anything is launched
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream
    rc = R.rnn_forward_noalloc(_desc(R, over), p, None, None, p, p, None, None, 1, stream)
    assert rc == R.RNN_NOT_SUPPORTED


def test_noalloc_async_call_status():
    import torch
    import bwd_persistent_cta_gb300 as R
    from bwd_persistent_cta_gb300 import build
    build.build()
    wl = synth.Workload("na_async", "lstm", False, 1, False, 5, 8, 32, 64, "bf16", 96, state_std=0.5)
    inp = synth.make_inputs(wl)
    w = Hn.to_dev(synth.flatten_params(wl, inp.params), wl)
    x = Hn.to_dev(inp.x, wl)
    y = torch.empty(wl.seq_len, wl.batch, wl.hidden_size, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = R.rnn_forward_noalloc(_desc(R, wl), x.data_ptr(), None, None, w.data_ptr(), y.data_ptr(), None, None, 0,
                               stream)
    assert rc == R.RNN_OK
    assert R.rnn_noalloc_status(stream) == R.RNN_OK
    assert np.isfinite(Hn.to_np(y)).all()


def test_noalloc_rejects_problems_beyond_the_scratch_limit():
    import torch
    import bwd_persistent_cta_gb300 as R
    from bwd_persistent_cta_gb300 import build
    build.build()
    wl = synth.WORKLOADS["lstm2bi_bf16_T512_B128_H1024"]
    desc = _desc(R, wl)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    rc = R.rnn_forward_noalloc(desc, p, None, None, p, p, None, None, 1, torch.cuda.current_stream().cuda_stream)
    assert rc == R.RNN_NOT_SUPPORTED
