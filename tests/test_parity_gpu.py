"""GPU parity against the fp64 oracle, through the C ABI.

Small cases (several tiles plus a ragged tail) run the oracle in full; the
full-size workloads run the GPU on the whole batch and the oracle on sampled
batch columns (sequences are independent), with dy zero outside the sampled
columns so the weight gradients equal the sampled oracle's exactly.
Tolerance (max over each output tensor of |gpu - ref| / max|ref|): 1e-5 on the
fp32 path, 2e-2 on the bf16 path (bf16 storage, fp32 accumulation)."""
import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TC, SIMT = 1, 2


def _wl(mode, ra, L, bidir, T, B, I, H, dtype, seed, **kw):
    return synth.Workload(f"{mode}{'_ra' if ra else ''}_{dtype}_T{T}_B{B}_I{I}_H{H}_L{L}{'bi' if bidir else ''}",
                          mode, ra, L, bidir, T, B, I, H, dtype, seed, **kw)


def test_config_lstm_f32_T16_B4_I32_H32():
    wl = synth.WORKLOADS["lstm_f32_T16_B4_I32_H32"]
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    Hn.compare(gpu, Hn.run_oracle(inp), wl, tol=1e-5)


FP32_CASES = [
    ("lstm", False, 1, False), ("lstm", False, 2, True),
    ("gru", True, 1, False), ("gru", True, 2, True),
    ("gru", False, 1, False), ("gru", False, 2, True),
]


@pytest.mark.parametrize("mode,ra,L,bidir", FP32_CASES)
def test_fp32_small(mode, ra, L, bidir):
    wl = _wl(mode, ra, L, bidir, 7, 5, 12, 16, "f32", 31, state_std=0.5)
    inp = synth.make_inputs(wl)
    inp.dhy = np.random.default_rng(1).normal(size=inp.h0.shape) * 0.5
    if mode == "lstm":
        inp.dcy = np.random.default_rng(2).normal(size=inp.c0.shape) * 0.5
    Hn.compare(Hn.run_gpu(inp), Hn.run_oracle(inp), wl, tol=1e-5)


BF16_CASES = [
    ("lstm", False, 1, False, TC), ("lstm", False, 1, False, SIMT),
    ("lstm", False, 2, True, TC), ("lstm", False, 2, True, SIMT),
    ("gru", True, 1, False, TC), ("gru", True, 1, False, SIMT),
    ("gru", True, 2, True, TC),
    ("gru", False, 1, False, SIMT), ("gru", False, 2, True, SIMT),
]


@pytest.mark.parametrize("mode,ra,L,bidir,algo", BF16_CASES)
def test_bf16_small(mode, ra, L, bidir, algo):
    wl = _wl(mode, ra, L, bidir, 9, 20, 72, 128, "bf16", 41, state_std=0.5)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp, algo=algo)
    assert gpu["algo"] == algo
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", True), ("gru", False)])
def test_batch_first_gate_order_and_state_grads(mode, ra):
    order = (2, 0, 3, 1) if mode == "lstm" else (1, 2, 0)
    wl = _wl(mode, ra, 1, True, 6, 17, 40, 128, "bf16", 51, state_std=0.5, gate_order=order, batch_first=True)
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(3)
    inp.dhy = synth.round_bf16(rng.normal(size=inp.h0.shape))
    if mode == "lstm":
        inp.dcy = synth.round_bf16(rng.normal(size=inp.c0.shape))
    Hn.compare(Hn.run_gpu(inp), Hn.run_oracle(inp), wl)


@pytest.mark.parametrize("T,B,H,algo", [(1, 1, 128, TC), (1, 16, 128, TC), (3, 1, 128, TC), (2, 256, 256, 0),
                                        (4, 3, 8, 0)])
@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", True)])
def test_edge_sizes(T, B, H, algo, mode, ra):
    wl = _wl(mode, ra, 1, False, T, B, 64, H, "bf16", 61, state_std=0.5)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp, algo=algo)
    if algo:
        assert gpu["algo"] == algo
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_inference_forward_only_matches_training_forward():
    wl = _wl("lstm", False, 2, True, 8, 24, 64, 128, "bf16", 71, state_std=0.5)
    inp = synth.make_inputs(wl)
    a = Hn.run_gpu(inp, backward=False)
    b = Hn.run_gpu(inp, backward=True)
    np.testing.assert_array_equal(a["y"], b["y"])
    Hn.compare(a, Hn.run_oracle(inp, backward=False), wl)


def test_repeated_calls_are_deterministic():
    wl = _wl("gru", True, 1, False, 10, 32, 64, 128, "bf16", 81, state_std=0.5)
    inp = synth.make_inputs(wl)
    a = Hn.run_gpu(inp, repeat=1)
    b = Hn.run_gpu(inp, repeat=3)
    for k in ("y", "hy", "dx", "dhx"):
        np.testing.assert_array_equal(a[k], b[k])
    # weight and bias gradients too: split-K and bias sums run in a fixed order
    for name, v in a["dparams"][0][0].items():
        np.testing.assert_array_equal(v, b["dparams"][0][0][name])


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------
def test_full_gru_ra_bf16_T128_B64_H512():
    wl = synth.WORKLOADS["gru_ra_bf16_T128_B64_H512"]
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_full_lstm_bf16_T256_B32_H1024_sampled():
    wl = synth.WORKLOADS["lstm_bf16_T256_B32_H1024"]
    keep = [0, 13, 20, 31]      # one column in each quarter: every batch part of any plan (at most 4)
    full = Hn.masked_dy(synth.make_inputs(wl), keep)
    gpu = Hn.run_gpu(full)
    ref = Hn.run_oracle(synth.make_inputs(wl, batch_subset=keep))
    Hn.compare(gpu, ref, wl, batch_idx=keep)


def test_full_lstm2bi_bf16_T512_B128_H1024_sampled():
    wl = synth.WORKLOADS["lstm2bi_bf16_T512_B128_H1024"]
    keep = [5, 40, 77, 127]     # one column in each quarter: every batch part of any plan (at most 4)
    full = Hn.masked_dy(synth.make_inputs(wl), keep)
    gpu = Hn.run_gpu(full)
    ref = Hn.run_oracle(synth.make_inputs(wl, batch_subset=keep))
    Hn.compare(gpu, ref, wl, batch_idx=keep)


@pytest.mark.parametrize("name,keep", [("lstm_bf16_T1024_B8_H2048", [3, 6]), ("gru_rb_bf16_T1024_B8_H2048", [0, 7])])
def test_full_hidden_2048_training_sampled(name, keep):
    # the latency workloads' shapes trained: tensor-core forward and backward
    # (the backward's K split through global memory)
    wl = synth.WORKLOADS[name]
    full = Hn.masked_dy(synth.make_inputs(wl), keep)
    gpu = Hn.run_gpu(full)
    assert gpu["algo"] == 1 and gpu["fwd_algo"] == 1
    ref = Hn.run_oracle(synth.make_inputs(wl, batch_subset=keep))
    Hn.compare(gpu, ref, wl, batch_idx=keep)


# ---------------------------------------------------------------------------
# weights that do not fit on chip: the SIMT kernels stream them from L2
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", False), ("gru", True)])
def test_streamed_weights_fp32(mode, ra):
    wl = _wl(mode, ra, 1, False, 4, 3, 16, 2048, "f32", 101, state_std=0.5)
    inp = synth.make_inputs(wl)
    Hn.compare(Hn.run_gpu(inp), Hn.run_oracle(inp), wl, tol=1e-5)


@pytest.mark.parametrize("name,keep", [("gru_rb_bf16_T1024_B1_H2048", [0]), ("gru_rb_bf16_T1024_B8_H2048", [0, 7]),
                                       ("lstm_bf16_T1024_B1_H2048", [0]), ("lstm_bf16_T1024_B8_H2048", [3, 6])])
def test_full_latency_workloads_forward(name, keep):
    wl = synth.WORKLOADS[name]
    gpu = Hn.run_gpu(synth.make_inputs(wl), backward=False)
    ref = Hn.run_oracle(synth.make_inputs(wl, batch_subset=keep), backward=False)
    Hn.compare(gpu, ref, wl, batch_idx=keep)
