"""The tensor-core forward with its weight tile split between tensor memory
(8 sub-tiles of 64 columns, the MMA A operand) and shared memory (the rest),
for K slices of more than 512 columns, at hidden 2048 with the tensor-core
backward; and the automatic mixed choice, a tensor-core forward with the SIMT
backward, for layers whose backward has no tensor-core plan (hidden not a
multiple of 128).  Against the fp64 oracle, tolerance 2e-2
(bf16).  A K-split cap of 1 (the plan-override test hook) makes a hidden-1024 forward run
one 1024-column K slice per 128 gate rows, which takes the split tile."""
import dataclasses

import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TC, SIMT = 1, 2


@pytest.fixture
def one_k_slice(plan_overrides):
    plan_overrides(max_ks_fwd=1)
    yield


def _wl(mode, ra, L, bidir, T, B, I, H, seed):
    return synth.Workload(f"split_{mode}{'_ra' if ra else ''}_T{T}_B{B}_H{H}_L{L}{'bi' if bidir else ''}",
                          mode, ra, L, bidir, T, B, I, H, "bf16", seed, state_std=0.5)


@pytest.mark.parametrize("mode,ra,L,bidir,B", [("lstm", False, 1, False, 16), ("gru", True, 1, False, 8),
                                               ("lstm", False, 1, False, 3), ("lstm", False, 2, True, 8)])
def test_split_weight_tile_forward(one_k_slice, mode, ra, L, bidir, B):
    wl = _wl(mode, ra, L, bidir, 10, B, 64, 1024, 600 + B + L)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["fwd_algo"] == TC and gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_split_weight_tile_forward_with_lengths_and_clip(one_k_slice):
    wl = _wl("lstm", False, 1, True, 9, 8, 64, 1024, 611)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=np.array([9, 0, 1, 5, 8, 3, 9, 7]))
    gpu = Hn.run_gpu(inp, backward=False)
    assert gpu["fwd_algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp, backward=False), wl)
    for b, n in enumerate(inp.lengths):
        assert np.all(gpu["y"][n:, b] == 0.0)


@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", True)])
def test_hidden_2048_tensor_core_forward_and_backward(mode, ra):
    # the backward's K split of 8 goes through global memory (16 clusters of
    # 8 cannot all be resident)
    wl = _wl(mode, ra, 1, False, 6, 4, 64, 2048, 612)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["fwd_algo"] == TC and gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", True)])
def test_tensor_core_forward_simt_backward(mode, ra):
    # hidden 320: the forward's 64-column K slices fit, the backward's
    # 128-unit row groups do not; the automatic choice mixes the two
    wl = _wl(mode, ra, 1, False, 6, 8, 64, 320, 614)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["fwd_algo"] == TC and gpu["algo"] == SIMT
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_forced_simt_keeps_the_simt_forward():
    wl = _wl("lstm", False, 1, False, 5, 4, 64, 2048, 613)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp, algo=SIMT, backward=False)
    assert gpu["fwd_algo"] == SIMT
    Hn.compare(gpu, Hn.run_oracle(inp, backward=False), wl)
