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


def _desc(R, wl):
    d = R.rnn_desc_t()
    d.mode = R.RNN_LSTM if wl.mode == "lstm" else R.RNN_GRU
    d.reset_after = int(wl.reset_after)
    d.bidirectional = int(wl.bidirectional)
    d.num_layers, d.seq_len, d.batch = wl.num_layers, wl.seq_len, wl.batch
    d.input_size, d.hidden_size = wl.input_size, wl.hidden_size
    d.dtype = R.RNN_BF16 if wl.dtype == "bf16" else R.RNN_F32
    return d


@pytest.mark.parametrize("wl", [
    synth.Workload("na_lstm", "lstm", False, 2, True, 9, 20, 72, 128, "bf16", 91, state_std=0.5),
    synth.Workload("na_gru", "gru", True, 1, False, 7, 5, 12, 16, "f32", 92, state_std=0.5),
], ids=lambda w: w.name)
def test_noalloc_forward_matches_rnn_forward_on_two_calls(wl):
    import torch
    import bwd_persistent_cta_gb300 as R
    from bwd_persistent_cta_gb300 import build
    build.build()
    inp = synth.make_inputs(wl)
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
    for _ in range(2):
        y = torch.full_like(y_ref, float("nan"))
        hy = torch.full_like(hy_ref, float("nan"))
        cy = torch.full_like(cy_ref, float("nan")) if cy_ref is not None else None
        rc = R.rnn_forward_noalloc(desc, x.data_ptr(), hx.data_ptr() if hx is not None else None,
                                   cx.data_ptr() if cx is not None else None, w.data_ptr(), y.data_ptr(),
                                   hy.data_ptr(), cy.data_ptr() if cy is not None else None, 1, stream)
        assert rc == R.RNN_OK, R.rnn_status_string(rc)
        assert Hn.max_rel_err(Hn.to_np(y), Hn.to_np(y_ref)) <= tol
        assert Hn.max_rel_err(Hn.to_np(hy), Hn.to_np(hy_ref)) <= tol
        if cy is not None:
            assert Hn.max_rel_err(Hn.to_np(cy), Hn.to_np(cy_ref)) <= tol


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
