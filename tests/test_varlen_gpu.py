"""Variable sequence lengths on the GPU, through the C ABI, against the fp64
oracle run with the same lengths (the batchwise step mask: at t >= len_b the
state is held, y_t = 0, and the backward passes the state gradients through
with zero gate gradients).  Lengths cover 0, 1, T and values in between, on
every kernel family: tcgen05 persistent (bf16 LSTM / GRU resetAfter), SIMT
persistent (fp32, GRU reset-before), the latency-mode forward (batch <= 8,
H = 2048) and the full-size sampled workloads.  Tolerances as in the parity
tests: 1e-5 (fp32), 2e-2 (bf16)."""
import dataclasses

import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TC, SIMT = 1, 2


def _wl(mode, ra, L, bidir, T, B, I, H, dtype, seed, **kw):
    return synth.Workload(f"{mode}{'_ra' if ra else ''}_{dtype}_T{T}_B{B}_I{I}_H{H}_L{L}{'bi' if bidir else ''}_len",
                          mode, ra, L, bidir, T, B, I, H, dtype, seed, **kw)


def _lengths(T, B, seed):
    """0, 1, T, T-1 first, then seeded values in [0, T]."""
    fixed = [0, 1, T, T - 1]
    rng = np.random.default_rng(seed)
    rest = rng.integers(0, T + 1, size=max(0, B - len(fixed)))
    return np.asarray((fixed + list(rest))[:B], dtype=np.int64)


CASES = [
    # mode, reset_after, layers, bidirectional, T, B, I, H, dtype, algo
    ("lstm", False, 2, True, 9, 6, 24, 40, "f32", SIMT),
    ("gru", True, 2, True, 9, 6, 24, 40, "f32", SIMT),
    ("gru", False, 2, True, 9, 6, 24, 40, "f32", SIMT),
    ("lstm", False, 2, True, 20, 24, 64, 128, "bf16", TC),
    ("gru", True, 1, False, 24, 20, 64, 128, "bf16", TC),
    ("gru", True, 1, True, 24, 20, 64, 128, "bf16", TC),
    ("gru", False, 1, True, 12, 6, 32, 64, "bf16", SIMT),
]


@pytest.mark.parametrize("mode,ra,L,bidir,T,B,I,H,dtype,algo", CASES)
def test_varlen_small(mode, ra, L, bidir, T, B, I, H, dtype, algo):
    wl = _wl(mode, ra, L, bidir, T, B, I, H, dtype, 200 + T + H, state_std=0.5)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=_lengths(T, B, 7 + L))
    gpu = Hn.run_gpu(inp, algo=algo)
    assert gpu["algo"] == algo
    ref = Hn.run_oracle(inp)
    Hn.compare(gpu, ref, wl)
    # padded positions of y and dx are exactly zero
    for b, n in enumerate(inp.lengths):
        assert np.all(gpu["y"][n:, b] == 0.0)
        assert np.all(gpu["dx"][n:, b] == 0.0)


def test_varlen_full_length_equals_no_lengths():
    wl = _wl("lstm", False, 1, True, 16, 16, 64, 128, "bf16", 211, state_std=0.5)
    inp = synth.make_inputs(wl)
    a = Hn.run_gpu(inp, algo=TC)
    b = Hn.run_gpu(dataclasses.replace(inp, lengths=np.full(16, 16)), algo=TC)
    for k in ("y", "hy", "cy", "dx", "dhx", "dcx"):
        np.testing.assert_array_equal(a[k], b[k])


def test_varlen_set_and_clear():
    import torch
    import bwd_persistent_cta_gb300 as R
    wl = _wl("gru", True, 1, False, 8, 16, 32, 128, "bf16", 212, state_std=0.5)
    inp = synth.make_inputs(wl)
    base = Hn.run_gpu(inp, algo=TC)
    rnn = R.RNN("gru", 32, 128, 8, 16, 1, False, True, "bf16", algo=TC)
    try:
        with pytest.raises(R.RnnError):
            rnn.set_seq_lengths([9] + [8] * 15)          # longer than seq_len
        with pytest.raises(R.RnnError):
            rnn.set_seq_lengths([-1] + [8] * 15)
        rnn.set_seq_lengths([3] * 16)
        rnn.set_seq_lengths(None)                        # back to full length
        w = Hn.to_dev(synth.flatten_params(wl, inp.params), wl)
        y, hy, _ = rnn.forward(Hn.to_dev(inp.x, wl), w, Hn.to_dev(inp.h0, wl), None, train=False)
        rnn.sync()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(Hn.to_np(y), base["y"])
        np.testing.assert_array_equal(Hn.to_np(hy), base["hy"])
    finally:
        rnn.close()


@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", False)])
def test_varlen_latency_forward(mode, ra):
    # batch <= 8 with H = 2048: the latency-mode forward kernel
    wl = _wl(mode, ra, 1, False, 12, 8, 2048, 2048, "bf16", 213, state_std=None, forward_only=True)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=_lengths(12, 8, 9))
    gpu = Hn.run_gpu(inp, backward=False)
    ref = Hn.run_oracle(inp, backward=False)
    Hn.compare(gpu, ref, wl)
    for b, n in enumerate(inp.lengths):
        assert np.all(gpu["y"][n:, b] == 0.0)


def test_varlen_full_gru_ra_bf16_T128_B64_H512():
    wl = synth.WORKLOADS["gru_ra_bf16_T128_B64_H512_varlen"]
    inp = synth.make_inputs(wl)
    assert inp.lengths.min() >= 64 and inp.lengths.max() <= 128
    Hn.compare(Hn.run_gpu(inp), Hn.run_oracle(inp), wl)


def test_varlen_full_lstm2bi_bf16_T512_B128_H1024_sampled():
    wl = synth.WORKLOADS["lstm2bi_bf16_T512_B128_H1024_varlen"]
    keep = [5, 127]
    full = Hn.masked_dy(synth.make_inputs(wl), keep)
    gpu = Hn.run_gpu(full)
    ref = Hn.run_oracle(synth.make_inputs(wl, batch_subset=keep))
    Hn.compare(gpu, ref, wl, batch_idx=keep)
