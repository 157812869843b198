"""Recomputation mode (LSTM cell states recomputed from the saved gates in the
backward pass, the popnn Lstm.cpp page's recomputation of the cell state and
its tanh) on the GPU, through the C ABI:
parity with the fp64 oracle (the mode changes storage, not the mathematics),
the smaller reserve, and agreement with the storing mode.  Tolerances: 1e-5
(fp32), 2e-2 (bf16)."""
import dataclasses

import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TC, SIMT = 1, 2


def _wl(mode, L, bidir, T, B, I, H, dtype, seed, **kw):
    return synth.Workload(f"{mode}_{dtype}_T{T}_B{B}_I{I}_H{H}_L{L}{'bi' if bidir else ''}_rc",
                          mode, True, L, bidir, T, B, I, H, dtype, seed, **kw)


@pytest.mark.parametrize("dtype,algo,T,B,H", [("bf16", TC, 20, 24, 128), ("f32", SIMT, 9, 5, 40)])
def test_recompute_matches_oracle_and_storing_mode(dtype, algo, T, B, H):
    wl = _wl("lstm", 2, True, T, B, 64 if dtype == "bf16" else 24, H, dtype, 400 + H, state_std=0.5)
    inp = synth.make_inputs(wl)
    ref = Hn.run_oracle(inp)
    store = Hn.run_gpu(inp, algo=algo)
    rc = Hn.run_gpu(dataclasses.replace(inp, wl=wl.with_(recompute=True)), algo=algo)
    Hn.compare(rc, ref, wl)
    # the forward is untouched by the mode; the backward agrees closely
    np.testing.assert_array_equal(rc["y"], store["y"])
    tol = 1e-6 if dtype == "f32" else 2e-2
    for k in ("dx", "dhx", "dcx"):
        assert Hn.max_rel_err(rc[k], store[k]) <= tol, k


def test_recompute_with_lengths_and_clip():
    wl = _wl("lstm", 2, True, 12, 16, 64, 128, "bf16", 405, state_std=None, recompute=True)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=np.array([12, 0, 3, 7, 1, 12, 11, 5] * 2))
    Hn.compare(Hn.run_gpu(inp, algo=TC), Hn.run_oracle(inp), wl)


def test_recompute_reserve_is_smaller_by_the_cell_states():
    import bwd_persistent_cta_gb300 as R
    L, T, B, H = 2, 12, 16, 128
    a = R.RNN("lstm", 64, H, T, B, L, True, dtype="bf16")
    b = R.RNN("lstm", 64, H, T, B, L, True, dtype="bf16", recompute=True)
    g0 = R.RNN("gru", 64, H, T, B, L, True, dtype="bf16")
    g1 = R.RNN("gru", 64, H, T, B, L, True, dtype="bf16", recompute=True)
    try:
        assert a.reserve_bytes - b.reserve_bytes == L * 2 * (T + 1) * B * H * 4
        assert g0.reserve_bytes == g1.reserve_bytes          # no cell state: nothing changes
    finally:
        for r in (a, b, g0, g1):
            r.close()


def test_recompute_full_lstm2bi_bf16_T512_B128_H1024_sampled():
    wl = synth.WORKLOADS["lstm2bi_bf16_T512_B128_H1024_recompute"]
    keep = [5, 127]
    full = Hn.masked_dy(synth.make_inputs(wl), keep)
    gpu = Hn.run_gpu(full)
    ref = Hn.run_oracle(synth.make_inputs(wl, batch_subset=keep))
    Hn.compare(gpu, ref, wl, batch_idx=keep)
