"""Interleaved weight update on the GPU: dW_hh accumulated step by step inside
the SIMT persistent backward kernel (rnn_set_interleaved_dw), against the fp64
oracle, and against the same handle with the dW_hh GEMM.  Cases cover every
cell (LSTM, GRU resetAfter, GRU reset-before with its r * h_{t-1} rows, plain
ReLU / tanh), one and several CTAs per direction, both directions, stacked
layers, sequence lengths, T = 1 and B = 1, and repeated calls (the accumulator
starts from zero each call).  Mode 2 forces the interleaved path wherever it
fits; the default mode 1 takes it only where a direction spans several CTAs.
Tolerances: 1e-5 (fp32), 2e-2 (bf16)."""
import dataclasses

import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

SIMT = 2


def _wl(mode, ra, L, bidir, T, B, I, H, dtype, seed, **kw):
    return synth.Workload(f"{mode}{'_ra' if ra else ''}_{dtype}_T{T}_B{B}_I{I}_H{H}_L{L}{'bi' if bidir else ''}_idw",
                          mode, ra, L, bidir, T, B, I, H, dtype, seed, **kw)


CASES = [
    # mode, reset_after, layers, bidirectional, T, B, I, H, dtype
    ("lstm", False, 1, False, 16, 4, 32, 32, "f32"),
    ("lstm", False, 2, True, 9, 8, 24, 256, "f32"),      # several CTAs per direction
    ("gru", True, 2, True, 9, 6, 24, 40, "f32"),
    ("gru", False, 2, True, 9, 6, 24, 40, "f32"),
    ("gru", False, 1, True, 12, 6, 32, 64, "bf16"),
    ("rnn_relu", False, 2, True, 9, 5, 24, 40, "f32"),
    ("rnn_tanh", False, 1, False, 9, 5, 24, 40, "f32"),
    ("lstm", False, 1, False, 1, 3, 16, 48, "f32"),       # T = 1
    ("gru", True, 1, True, 7, 1, 16, 48, "f32"),          # B = 1
]


@pytest.mark.parametrize("mode,ra,L,bidir,T,B,I,H,dtype", CASES)
def test_interleaved_dw_parity(mode, ra, L, bidir, T, B, I, H, dtype):
    wl = _wl(mode, ra, L, bidir, T, B, I, H, dtype, 400 + T + H + B, state_std=0.5)
    inp = synth.make_inputs(wl)
    on = Hn.run_gpu(inp, algo=SIMT, repeat=2, interleaved_dw=2)
    assert on["algo"] == SIMT and on["interleaved_dw"]
    ref = Hn.run_oracle(inp)
    Hn.compare(on, ref, wl)
    off = Hn.run_gpu(inp, algo=SIMT, interleaved_dw=0)
    assert not off["interleaved_dw"]
    Hn.compare(off, ref, wl)
    # the same gradient in another summation order
    G = {"lstm": 4, "gru": 3}.get(mode, 1)
    for l in range(L):
        for d in range(2 if bidir else 1):
            a, b = on["dparams"][l][d]["W_hh"], off["dparams"][l][d]["W_hh"]
            assert Hn.max_rel_err(a, b) <= Hn.TOL[dtype]
    # the reserve holds the accumulator; backward-weights runs one GEMM fewer per (layer, direction):
    # one launch fewer each on the fp32 path, while the bf16 path runs a layer's weight-gradient
    # GEMMs as one grouped launch either way
    D = 2 if bidir else 1
    assert on["reserve_bytes"] - off["reserve_bytes"] == L * D * G * H * H * 4
    if dtype == "f32":
        assert on["launches"] / 2 < off["launches"]      # two calls on, one off
    else:
        assert on["launches"] / 2 <= off["launches"]


def test_interleaved_dw_with_lengths():
    wl = _wl("lstm", False, 2, True, 10, 6, 24, 40, "f32", 431, state_std=0.5)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=np.array([10, 0, 1, 9, 4, 7]))
    gpu = Hn.run_gpu(inp, algo=SIMT, interleaved_dw=2)
    assert gpu["interleaved_dw"]
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_interleaved_dw_reset_before_bf16_lengths():
    wl = _wl("gru", False, 2, True, 12, 8, 32, 64, "bf16", 432, state_std=0.5)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=np.array([12, 0, 1, 11, 5, 7, 12, 3]))
    gpu = Hn.run_gpu(inp, algo=SIMT, interleaved_dw=2)
    assert gpu["interleaved_dw"]
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_interleaved_dw_full_lstm_f32_T16_B4_I32_H32():
    wl = synth.WORKLOADS["lstm_f32_T16_B4_I32_H32"]
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp, interleaved_dw=2)
    assert gpu["algo"] == SIMT and gpu["interleaved_dw"]
    Hn.compare(gpu, Hn.run_oracle(inp), wl)
    # the default leaves this shape (one CTA per direction) to the GEMM
    assert not Hn.run_gpu(inp, backward=False)["interleaved_dw"]


def test_interleaved_dw_default_on_several_ctas():
    wl = _wl("gru", True, 1, False, 24, 16, 64, 128, "f32", 433, state_std=0.5)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["algo"] == SIMT and gpu["interleaved_dw"]
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_interleaved_dw_not_on_tensor_core_or_large_layers():
    import bwd_persistent_cta_gb300 as R
    tc = R.RNN("lstm", 64, 128, 8, 16, dtype="bf16")          # tcgen05 kernels: the GEMM
    big = R.RNN("lstm", 64, 1024, 8, 64, dtype="f32")         # per-step share too large
    try:
        assert tc.algo == 1 and not tc.interleaved_dw
        assert big.algo == SIMT and not big.interleaved_dw
        assert R.rnn_set_interleaved_dw(tc.handle, 3) == R.RNN_BAD_PARAM
        assert R.rnn_set_interleaved_dw(big.handle, 2) == R.RNN_OK and not big.interleaved_dw
    finally:
        tc.close()
        big.close()
