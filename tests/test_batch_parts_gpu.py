"""Batch parts in the tensor-core persistent kernels: a row group's batch split
over 1, 2 or 4 clusters (the plan-override test hook forces the count; by
default a per-step cost estimate chooses).  Against the fp64 oracle, tolerance
2e-2 (bf16), and bit-identical results over repeated calls (the bias
gradients of the parts are summed in part order)."""
import dataclasses

import numpy as np
import pytest

import synth
from tests import harness as Hn

pytestmark = pytest.mark.gpu

TC = 1


def _wl(mode, ra, L, bidir, T, B, I, H, seed):
    return synth.Workload(f"nb_{mode}{'_ra' if ra else ''}_T{T}_B{B}_H{H}_L{L}{'bi' if bidir else ''}", mode, ra, L,
                          bidir, T, B, I, H, "bf16", seed, state_std=0.5)


@pytest.mark.parametrize("nb", [1, 2, 4])
@pytest.mark.parametrize("mode,ra,L,bidir,T,B,H", [("lstm", False, 1, False, 12, 64, 256),
                                                   ("gru", True, 2, True, 9, 40, 128),
                                                   ("lstm", False, 1, True, 8, 33, 128)])
def test_batch_parts_parity(plan_overrides, nb, mode, ra, L, bidir, T, B, H):
    plan_overrides(nb_fwd=nb, nb_bwd=nb)
    wl = _wl(mode, ra, L, bidir, T, B, 64, H, 800 + nb + B)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


@pytest.mark.parametrize("nb", [2, 4])
def test_batch_parts_with_lengths(plan_overrides, nb):
    plan_overrides(nb_fwd=nb, nb_bwd=nb)
    wl = _wl("lstm", False, 1, True, 10, 32, 64, 128, 810 + nb)
    lengths = np.array([10, 0, 1, 9, 5, 7, 10, 3] * 4)
    inp = dataclasses.replace(synth.make_inputs(wl), lengths=lengths)
    gpu = Hn.run_gpu(inp)
    Hn.compare(gpu, Hn.run_oracle(inp), wl)
    for b, n in enumerate(lengths):
        assert np.all(gpu["y"][n:, b] == 0.0)


@pytest.mark.parametrize("nb", [2, 4])
def test_batch_parts_reset_before_forward(plan_overrides, nb):
    plan_overrides(nb_fwd=nb)
    wl = _wl("gru", False, 1, False, 8, 32, 64, 128, 820 + nb)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["fwd_algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)


def test_batch_parts_repeatable(plan_overrides):
    plan_overrides(nb_fwd=2, nb_bwd=4)
    wl = _wl("gru", True, 1, False, 10, 64, 64, 256, 830)
    inp = synth.make_inputs(wl)
    a = Hn.run_gpu(inp)
    b = Hn.run_gpu(inp)
    for k in ("y", "hy", "dx", "dhx"):
        np.testing.assert_array_equal(a[k], b[k])
    for name, v in a["dparams"][0][0].items():
        np.testing.assert_array_equal(v, b["dparams"][0][0][name])


@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", True)])
def test_batch_above_256_on_tensor_cores(mode, ra):
    # 300 sequences: the MMA N limit of 256 needs 2 batch parts of 150 (N 160)
    wl = _wl(mode, ra, 1, False, 6, 300, 64, 128, 840)
    inp = synth.make_inputs(wl)
    gpu = Hn.run_gpu(inp)
    assert gpu["algo"] == TC
    Hn.compare(gpu, Hn.run_oracle(inp), wl)
