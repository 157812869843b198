"""The tensor-core BPTT with its K split exchanged through global memory
instead of thread-block clusters: taken by itself where no cluster plan can
be resident (hidden 2048: 16 row groups x a K split of 8 would need 16
clusters of 8), forced by the bwd_global_ks test hook elsewhere.  Against the
fp64 oracle (bf16 tolerance): LSTM, GRU resetAfter and reset-before at
hidden 2048; forced on small shapes with two layers, both directions,
sequence lengths, batch parts; bit-identical repeated calls; and a skipped
arrival that must end in RNN_TIMEOUT with the context still usable."""
import dataclasses

import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TC = 1


def _wl(mode, ra, L, bidir, T, B, I, H, seed):
    return synth.Workload(f"gk_{mode}_T{T}_B{B}_I{I}_H{H}_L{L}{'bi' if bidir else ''}", mode, ra, L, bidir, T, B, I,
                          H, "bf16", seed, state_std=0.5)


@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", True), ("gru", False)])
def test_hidden_2048_backward_on_tensor_cores(mode, ra):
    wl = _wl(mode, ra, 1, False, 5, 8, 64, 2048, 900 + int(ra))
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["algo"] == TC and gpu["fwd_algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


@pytest.mark.parametrize("B", [32, 64])
def test_hidden_2048_backward_wider_batch(B):
    # N = 32 / 64 per MMA (one batch part), 2 or 4 pairs per thread
    wl = _wl("lstm", False, 1, False, 4, B, 64, 2048, 903 + B)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_hidden_2048_bidirectional_one_direction_per_launch():
    # both directions need 256 CTAs: the layer runs as one launch per
    # direction, each with its K split through global memory
    wl = _wl("gru", True, 1, True, 4, 8, 64, 2048, 905)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


@pytest.mark.parametrize("mode,ra,L,bidir,T,B,H", [("lstm", False, 2, True, 7, 16, 256),
                                                   ("gru", True, 1, True, 6, 33, 128),
                                                   ("gru", False, 2, False, 5, 8, 256),
                                                   ("lstm", False, 1, False, 4, 300, 128)])
def test_forced_global_ksplit(plan_overrides, mode, ra, L, bidir, T, B, H):
    plan_overrides(bwd_global_ks=1)
    wl = _wl(mode, ra, L, bidir, T, B, 48, H, 910 + H + B)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp, algo=TC)
    assert gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


@pytest.mark.parametrize("nb", [1, 2])
def test_forced_global_ksplit_lengths_and_parts(plan_overrides, nb):
    plan_overrides(bwd_global_ks=1, nb_bwd=nb)
    wl = _wl("lstm", False, 2, True, 9, 16, 32, 128, 920 + nb)
    lengths = np.array([9, 0, 1, 5, 8, 3, 9, 7, 2, 9, 6, 4, 9, 1, 8, 5])
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=lengths)
    gpu = Hn.run_gpu(inp, algo=TC)
    assert gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)
    for b, n in enumerate(lengths):
        assert np.all(gpu["y"][n:, b] == 0.0)


def test_forced_global_ksplit_repeatable(plan_overrides):
    plan_overrides(bwd_global_ks=1)
    wl = _wl("gru", True, 1, True, 8, 16, 32, 256, 930)
    inp = synth.make_inputs(wl)
    a = Hn.run_gpu(inp, algo=TC)
    b = Hn.run_gpu(inp, algo=TC, repeat=2)
    for k in ("y", "hy", "dx", "dhx"):
        np.testing.assert_array_equal(a[k], b[k])
    for name, v in a["dparams"][0][1].items():
        np.testing.assert_array_equal(v, b["dparams"][0][1][name])


def test_forced_global_ksplit_skipped_arrival_times_out(plan_overrides):
    import torch
    import bwd_persistent_cta_gb300 as R
    plan_overrides(bwd_global_ks=1)
    wl = _wl("lstm", False, 1, False, 6, 16, 64, 256, 940)
    inp = synth.make_inputs(wl)
    rnn = R.RNN("lstm", 64, 256, 6, 16, algo=TC)
    try:
        w = Hn.to_dev(synth.flatten_params(wl, inp.params), wl)
        x = Hn.to_dev(inp.x, wl)
        hx, cx = Hn.to_dev(inp.h0, wl), Hn.to_dev(inp.c0, wl)
        dy = Hn.to_dev(inp.dy, wl)
        rnn.set_timeout_ns(200_000_000)
        rnn.forward(x, w, hx, cx, train=True)
        rnn.sync()
        rnn.debug_skip_arrival(0)
        rnn.backward_data(dy, w, None, None, cx=cx)
        rc = R.rnn_sync_status(rnn.handle, torch.cuda.current_stream().cuda_stream)
        assert rc == R.RNN_TIMEOUT, R.rnn_status_string(rc)
        rnn.debug_skip_arrival(-1)
        rnn.forward(x, w, hx, cx, train=True)
        dx, _, _ = rnn.backward_data(dy, w, Hn.to_dev(inp.dhy, wl), Hn.to_dev(inp.dcy, wl), cx=cx)
        rnn.sync()
        ref = Hn.run_oracle(inp)
        assert Hn.max_rel_err(Hn.to_np(dx), ref["dx"]) <= Hn.TOL["bf16"]
    finally:
        rnn.close()
