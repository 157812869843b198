"""GRU reset-before on the tensor-core kernels, chosen automatically from
batch 4 on.  The forward exchanges twice per step (r, z from W_hh h_{t-1},
then n from W_hn (r * h_{t-1})); so does the backward (d(rh) = W_hn^T dn from
a [0, 0, dn, 0] operand, then the recurrent gradient from dG = [dr, dz, dn, 0]
with W_hn^T dn taken back out).  Hidden sizes that are not a multiple of 128
have no tensor-core backward plan and pair the tensor-core forward with the
SIMT backward.  Against the fp64 oracle, tolerance 2e-2 (bf16): forward and
backward, one and two layers, both directions, sequence lengths, batch parts,
hidden sizes that take one or several K slices, the full-size T128 B64 H512
layer, bit-identical repeated calls, and the small-batch case that stays on
the SIMT kernels."""
import dataclasses

import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TC, SIMT = 1, 2


def _wl(L, bidir, T, B, I, H, seed):
    return synth.Workload(f"rb_tc_T{T}_B{B}_I{I}_H{H}_L{L}{'bi' if bidir else ''}", "gru", False, L, bidir, T, B, I,
                          H, "bf16", seed, state_std=0.5)


@pytest.mark.parametrize("L,bidir,T,B,H", [(1, False, 10, 8, 128), (1, True, 9, 16, 256), (2, True, 7, 4, 192),
                                           (1, False, 6, 8, 1024), (1, False, 5, 33, 512)])
def test_reset_before_tc_forward(L, bidir, T, B, H):
    wl = _wl(L, bidir, T, B, 64, H, 700 + H + B)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["fwd_algo"] == TC and gpu["algo"] == (TC if H % 128 == 0 else SIMT)
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


@pytest.mark.parametrize("L,bidir,T,B,H", [(1, False, 8, 4, 128), (2, True, 6, 16, 256), (1, True, 5, 33, 128),
                                           (1, False, 4, 300, 128), (1, False, 5, 8, 1024)])
def test_reset_before_tc_backward(L, bidir, T, B, H):
    wl = _wl(L, bidir, T, B, 48, H, 730 + H + B + L)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp, algo=TC)
    assert gpu["algo"] == TC and gpu["fwd_algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_reset_before_tc_backward_with_lengths_and_parts(plan_overrides):
    plan_overrides(nb_fwd=2, nb_bwd=2)
    wl = _wl(2, True, 9, 16, 32, 128, 741)
    lengths = np.array([9, 0, 1, 5, 8, 3, 9, 7, 2, 9, 6, 4, 9, 1, 8, 5])
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=lengths)
    gpu = Hn.run_gpu(inp, algo=TC)
    assert gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)
    for b, n in enumerate(lengths):
        assert np.all(gpu["y"][n:, b] == 0.0)


def test_reset_before_tc_backward_repeatable():
    wl = _wl(1, True, 8, 16, 32, 128, 742)
    inp = synth.make_inputs(wl)
    a = Hn.run_gpu(inp, algo=TC)
    b = Hn.run_gpu(inp, algo=TC, repeat=2)
    for k in ("y", "hy", "dx", "dhx"):
        np.testing.assert_array_equal(a[k], b[k])
    for name, v in a["dparams"][0][1].items():
        np.testing.assert_array_equal(v, b["dparams"][0][1][name])


def test_full_gru_rb_bf16_T128_B64_H512():
    # the shape of the GRU resetAfter workload, reset-before form, forward and backward
    wl = synth.Workload("gru_rb_bf16_T128_B64_H512", "gru", False, 1, False, 128, 64, 512, 512, "bf16", 1)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["algo"] == TC and gpu["fwd_algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_reset_before_tc_forward_with_lengths():
    wl = _wl(2, True, 9, 8, 32, 128, 711)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=np.array([9, 0, 1, 5, 8, 3, 9, 7]))
    gpu = Hn.run_gpu(inp)
    assert gpu["fwd_algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)
    for b, n in enumerate(inp.lengths):
        assert np.all(gpu["y"][n:, b] == 0.0)


def test_reset_before_small_batch_stays_simt():
    wl = _wl(1, False, 6, 2, 32, 128, 712)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["fwd_algo"] == SIMT
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_reset_before_tc_inference_matches_training():
    import torch
    import bwd_persistent_cta_gb300 as R
    wl = _wl(1, True, 8, 8, 32, 128, 713)
    inp = synth.make_inputs(wl)
    rnn = R.RNN("gru", 32, 128, 8, 8, 1, True, False, "bf16")
    try:
        assert rnn.fwd_algo == TC
        w = Hn.to_dev(synth.flatten_params(wl, inp.params), wl)
        x, hx = Hn.to_dev(inp.x, wl), Hn.to_dev(inp.h0, wl)
        y1, h1, _ = rnn.forward(x, w, hx, None, train=True)
        y0, h0, _ = rnn.forward(x, w, hx, None, train=False)
        rnn.sync()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(Hn.to_np(y0), Hn.to_np(y1))
        np.testing.assert_array_equal(Hn.to_np(h0), Hn.to_np(h1))
    finally:
        rnn.close()
