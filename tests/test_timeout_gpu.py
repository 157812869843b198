"""The bounded spin-waits: one CTA of a persistent launch skips its per-step
arrival (a flag that nothing else sets), so its peers' waits run out.  The
call must end with RNN_TIMEOUT reported through rnn_sync_status - no hang, no
fault - and the context must stay usable for a normal call afterwards."""
import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("algo", [1, 2])
def test_skipped_arrival_times_out_and_context_survives(algo):
    import torch
    import bwd_persistent_cta_gb300 as R
    from bwd_persistent_cta_gb300 import build
    build.build()
    wl = synth.Workload("t", "lstm", False, 1, False, 6, 16, 64, 128, "bf16", 5, state_std=0.5)
    inp = synth.make_inputs(wl)
    rnn = R.RNN("lstm", 64, 128, 6, 16, algo=algo)
    try:
        w = Hn.to_dev(synth.flatten_params(wl, inp.params), wl)
        x = Hn.to_dev(inp.x, wl)
        hx, cx = Hn.to_dev(inp.h0, wl), Hn.to_dev(inp.c0, wl)
        rnn.set_timeout_ns(200_000_000)
        rnn.debug_skip_arrival(0)
        rnn.forward(x, w, hx, cx)
        rc = R.rnn_sync_status(rnn.handle, torch.cuda.current_stream().cuda_stream)
        assert rc == R.RNN_TIMEOUT, R.rnn_status_string(rc)
        rnn.debug_skip_arrival(-1)
        y, hy, cy = rnn.forward(x, w, hx, cx)
        rnn.sync()
        ref = Hn.run_oracle(inp, backward=False)
        assert Hn.max_rel_err(Hn.to_np(y), ref["y"]) <= Hn.TOL["bf16"]
    finally:
        rnn.close()
