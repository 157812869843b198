"""The cluster-resident forward (opt-in with RNN_CLUSTER_FWD=1): parity with the
fp64 oracle for LSTM and GRU resetAfter, several hidden sizes (4, 8 and 16
CTAs per cluster), batch paddings and both directions, and the bounded waits
(one CTA withholding its chunk ends in RNN_TIMEOUT, the context survives)."""
import os

import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cluster_forward(monkeypatch):
    monkeypatch.setenv("RNN_CLUSTER_FWD", "1")
    yield


@pytest.mark.parametrize("mode,ra,L,bidir,T,B,H", [
    ("lstm", False, 1, False, 12, 16, 128), ("gru", True, 1, True, 12, 5, 256),
    ("lstm", False, 2, True, 10, 40, 256), ("gru", True, 1, False, 16, 64, 512),
])
def test_cluster_forward_parity(mode, ra, L, bidir, T, B, H):
    wl = synth.Workload(f"cl_{mode}_T{T}_B{B}_H{H}", mode, ra, L, bidir, T, B, 64, H, "bf16", 500 + H + B,
                        state_std=0.5)
    inp = synth.make_inputs(wl)
    Hn.compare(Hn.run_gpu(inp, algo=1), Hn.run_oracle(inp), wl)


def test_cluster_forward_full_gru_ra_bf16_T128_B64_H512():
    wl = synth.WORKLOADS["gru_ra_bf16_T128_B64_H512"]
    inp = synth.make_inputs(wl)
    Hn.compare(Hn.run_gpu(inp, backward=False), Hn.run_oracle(inp, backward=False), wl)


def test_cluster_forward_withheld_chunk_times_out():
    import torch
    import bwd_persistent_cta_gb300 as R
    wl = synth.Workload("t", "lstm", False, 1, False, 6, 16, 64, 128, "bf16", 5, state_std=0.5)
    inp = synth.make_inputs(wl)
    rnn = R.RNN("lstm", 64, 128, 6, 16, algo=1)
    try:
        w = Hn.to_dev(synth.flatten_params(wl, inp.params), wl)
        x = Hn.to_dev(inp.x, wl)
        hx, cx = Hn.to_dev(inp.h0, wl), Hn.to_dev(inp.c0, wl)
        rnn.set_timeout_ns(200_000_000)
        rnn.debug_skip_arrival(2)
        rnn.forward(x, w, hx, cx)
        rc = R.rnn_sync_status(rnn.handle, torch.cuda.current_stream().cuda_stream)
        assert rc == R.RNN_TIMEOUT, R.rnn_status_string(rc)
        rnn.debug_skip_arrival(-1)
        y, hy, cy = rnn.forward(x, w, hx, cx)
        rnn.sync()
        assert Hn.max_rel_err(Hn.to_np(y), Hn.run_oracle(inp, backward=False)["y"]) <= Hn.TOL["bf16"]
    finally:
        rnn.close()
