"""Plain RNN cells (ReLU / tanh) and LSTM cell clipping on the GPU, through the
C ABI, against the fp64 oracle.

Clipping and ReLU have discontinuous derivatives: a value that lies within
rounding distance of a clip bound (or a ReLU pre-activation that lies within
rounding distance of zero) can legitimately take the other branch of the
derivative on the GPU.  So the backward is compared where the cases keep every
such value clear of the discontinuity: fp32 cases (rounding ~1e-6) with the
oracle's cell values checked to stay 1e-4 away from the bounds, and a bf16
tensor-core case whose saturated gates keep every cell value at least 0.4 away
from the bounds.  In bf16 with random inputs only the (continuous) forward
outputs are compared.  Tolerances: 1e-5 (fp32), 2e-2 (bf16)."""
import dataclasses

import numpy as np
import pytest

import synth
from oracle import rnn_oracle
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TC, SIMT = 1, 2


def _wl(mode, ra, L, bidir, T, B, I, H, dtype, seed, **kw):
    return synth.Workload(f"{mode}_{dtype}_T{T}_B{B}_I{I}_H{H}_L{L}{'bi' if bidir else ''}_cell",
                          mode, ra, L, bidir, T, B, I, H, dtype, seed, **kw)


def _cell_margin(inp, bounds):
    """Smallest distance of any oracle cell value (c_t and c_{t-1}) to a bound."""
    ref = Hn.run_oracle(inp, backward=False)
    vals = np.concatenate([k[n].ravel() for _, per in ref["fwd"]["cache"] for k in per for n in ("c", "c_prev")])
    return float(np.min(np.minimum(np.abs(vals - bounds[0]), np.abs(vals - bounds[1])))), \
        float(np.mean((vals < bounds[0]) | (vals > bounds[1])))


# ---------------------------------------------------------------------------
# plain RNN cells
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["rnn_relu", "rnn_tanh"])
@pytest.mark.parametrize("L,bidir", [(1, False), (2, True)])
def test_plain_rnn_fp32(mode, L, bidir):
    wl = _wl(mode, False, L, bidir, 9, 5, 24, 40, "f32", 300 + L, state_std=0.5)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["algo"] == SIMT
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_plain_rnn_tanh_bf16_with_lengths():
    wl = _wl("rnn_tanh", False, 2, True, 12, 16, 64, 96, "bf16", 303, state_std=0.5)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=np.array([12, 0, 1, 5, 11, 7, 12, 3] * 2))
    gpu = Hn.run_gpu(inp)
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_plain_rnn_relu_bf16_forward():
    wl = _wl("rnn_relu", False, 2, True, 12, 16, 64, 96, "bf16", 304, state_std=0.5)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp, backward=False)
    Hn.compare(gpu, Hn.run_oracle(inp, backward=False), wl)


@pytest.mark.parametrize("mode", ["rnn_relu", "rnn_tanh"])
def test_plain_rnn_latency_forward(mode):
    # batch <= 8, H = 2048: the latency-mode forward kernel with one gate
    wl = _wl(mode, False, 1, False, 10, 4, 2048, 2048, "bf16", 305, state_std=None, forward_only=True)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp, backward=False)
    Hn.compare(gpu, Hn.run_oracle(inp, backward=False), wl)


# ---------------------------------------------------------------------------
# LSTM cell clipping
# ---------------------------------------------------------------------------
def test_clip_fp32_simt_full():
    bounds = (-0.45, 0.5)
    wl = _wl("lstm", False, 2, True, 7, 5, 24, 40, "f32", 311, state_std=1.0)
    inp = dataclasses.replace(synth.make_inputs(wl), clip=bounds)
    margin, frac = _cell_margin(inp, bounds)
    assert margin > 1e-4 and frac > 0.05        # clipping active, no value at a bound
    gpu = Hn.run_gpu(inp, algo=SIMT)
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_clip_bf16_tc_forward_random():
    bounds = (-0.4, 0.45)
    wl = _wl("lstm", False, 2, True, 16, 24, 64, 128, "bf16", 312, state_std=1.0)
    inp = dataclasses.replace(synth.make_inputs(wl), clip=bounds)
    gpu = Hn.run_gpu(inp, algo=TC, backward=False)
    assert gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp, backward=False), wl)
    assert _cell_margin(inp, bounds)[1] > 0.05


def _saturated_inputs(seed, T, B, I, H, L, bidir, dtype):
    """LSTM with saturated input / forget gates (bias +8) and candidates of
    alternating sign (bias +-8 by unit), tiny weights: c grows by about one per
    step from c0 = 0, so every cell value sits near an integer, far from the
    half-integer bounds used with it; the output gate stays unsaturated."""
    wl = _wl("lstm", False, L, bidir, T, B, I, H, dtype, seed, state_std=None)
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(seed)
    rnd = synth.round_bf16 if dtype == "bf16" else (lambda a: a)
    for per in inp.params:
        for p in per:
            p["W_ih"] = rnd(rng.uniform(-0.002, 0.002, p["W_ih"].shape))
            p["W_hh"] = rnd(rng.uniform(-0.002, 0.002, p["W_hh"].shape))
            b = np.zeros(4 * H)
            b[0:H] = 8.0                                        # input gate
            b[H:2 * H] = 8.0                                    # forget gate
            b[2 * H:3 * H] = np.where(np.arange(H) % 2 == 0, 8.0, -8.0)   # candidate +-1
            b[3 * H:4 * H] = rnd(rng.uniform(-1.0, 1.0, H))     # output gate
            p["b"] = b
    return wl, inp


def test_clip_bf16_tc_full_saturated():
    bounds = (-2.5, 2.5)
    wl, inp = _saturated_inputs(313, 8, 16, 64, 128, 1, True, "bf16")
    inp = dataclasses.replace(inp, clip=bounds)
    margin, frac = _cell_margin(inp, bounds)
    assert margin > 0.4 and frac > 0.1
    gpu = Hn.run_gpu(inp, algo=TC)
    Hn.compare(gpu, Hn.run_oracle(inp), wl)
    # the clipping matters: without it the cell states grow past the bounds
    ref_free = rnn_oracle.run_inputs(dataclasses.replace(inp, clip=None), with_backward=False)
    assert np.max(np.abs(ref_free["cy"] - gpu["cy"])) > 1.0


def test_clip_bf16_tc_with_lengths_saturated():
    bounds = (-2.5, 2.5)
    wl, inp = _saturated_inputs(314, 8, 16, 64, 128, 2, True, "bf16")
    inp = dataclasses.replace(inp, clip=bounds, lengths=np.array([8, 0, 3, 5, 1, 8, 7, 2] * 2))
    gpu = Hn.run_gpu(inp, algo=TC)
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_clip_latency_forward():
    bounds = (-0.3, 0.35)
    wl = _wl("lstm", False, 1, False, 10, 4, 2048, 2048, "bf16", 315, state_std=None, forward_only=True)
    inp = dataclasses.replace(synth.make_inputs(wl), clip=bounds)
    gpu = Hn.run_gpu(inp, backward=False)
    Hn.compare(gpu, Hn.run_oracle(inp, backward=False), wl)


def test_clip_setter_errors():
    import bwd_persistent_cta_gb300 as R
    g = R.RNN("gru", 32, 64, 4, 2, dtype="f32")
    try:
        with pytest.raises(R.RnnError):
            g.set_cell_clip((-1.0, 1.0))                 # clipping is an LSTM option
    finally:
        g.close()
    m = R.RNN("lstm", 32, 64, 4, 2, dtype="f32")
    try:
        with pytest.raises(R.RnnError):
            m.set_cell_clip((1.0, 1.0))                  # needs lo < hi
        m.set_cell_clip((-1.0, 1.0))
        m.set_cell_clip(None)
    finally:
        m.close()
