"""The parity comparator itself (no GPU): a comparison that could not fail
would make every parity test vacuous.  It must accept the oracle's own
result, reject one perturbed element in any output tensor, a NaN, a missing
output and a shape mismatch, and compare only the sampled batch columns when
asked to."""
import copy
import re

import numpy as np
import pytest

import synth
from tests import harness as Hn


def _case(mode, ra, dtype="f32"):
    wl = synth.Workload(f"h_{mode}", mode, ra, 2, True, 4, 3, 8, 8, dtype, 5, state_std=0.5)
    inp = synth.make_inputs(wl)
    return wl, inp, Hn.run_oracle(inp)


def _as_gpu(ref):
    return {k: copy.deepcopy(v) for k, v in ref.items() if k in ("y", "hy", "cy", "dx", "dhx", "dcx", "dparams")}


def _failing(gpu, ref, wl):
    """The outputs compare() reports above tolerance (it must report some)."""
    with pytest.raises(AssertionError) as ei:
        Hn.compare(gpu, ref, wl)
    bad = str(ei.value).split("(all:")[0]
    return sorted(re.findall(r"'([^']+)':", bad))


def test_max_rel_err_definition():
    r = np.array([[1.0, -4.0], [2.0, 0.5]])
    g = r.copy()
    g[1, 0] += 0.04
    assert Hn.max_rel_err(g, r) == pytest.approx(0.01)
    assert Hn.max_rel_err(np.zeros(3), np.zeros(3)) == 0.0
    with pytest.raises(AssertionError):
        Hn.max_rel_err(np.zeros(3), np.zeros(4))


@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", True), ("gru", False)])
def test_identical_results_pass(mode, ra):
    wl, _, ref = _case(mode, ra)
    errs = Hn.compare(_as_gpu(ref), ref, wl)
    assert set(errs) >= {"y", "hy", "dx", "dhx"} and all(v == 0.0 for v in errs.values())
    assert any(k.startswith("dW_hh") for k in errs) and any(k.startswith("dW_ih") for k in errs)


@pytest.mark.parametrize("mode,ra", [("lstm", False), ("gru", True)])
def test_each_output_can_fail(mode, ra):
    wl, _, ref = _case(mode, ra)
    keys = ["y", "hy", "dx", "dhx"] + (["cy", "dcx"] if mode == "lstm" else [])
    for k in keys:
        gpu = _as_gpu(ref)
        a = gpu[k]
        a[(0,) * a.ndim] += 1e-3 * np.max(np.abs(ref[k])) + 1e-3
        assert _failing(gpu, ref, wl) == [k]
    for l in range(2):
        for d in range(2):
            for name in ref["dparams"][l][d]:
                gpu = _as_gpu(ref)
                v = gpu["dparams"][l][d][name]
                v.flat[-1] += 1e-3 * np.max(np.abs(v)) + 1e-3
                assert _failing(gpu, ref, wl) == [f"d{name}[{l},{d}]"]


def test_nan_missing_output_and_shape_mismatch_fail():
    wl, _, ref = _case("lstm", False)
    gpu = _as_gpu(ref)
    gpu["y"][1, 1, 1] = np.nan
    with pytest.raises(AssertionError):
        Hn.compare(gpu, ref, wl)
    gpu = _as_gpu(ref)
    del gpu["dcx"]
    with pytest.raises(AssertionError, match="lacks"):
        Hn.compare(gpu, ref, wl)
    gpu = _as_gpu(ref)
    gpu["dx"] = gpu["dx"][:, :2]
    with pytest.raises(AssertionError):
        Hn.compare(gpu, ref, wl)


def test_bf16_tolerance_is_looser_than_f32():
    wl, _, ref = _case("gru", True)
    gpu = _as_gpu(ref)
    gpu["y"] = gpu["y"] * (1 + 5e-3)
    with pytest.raises(AssertionError):
        Hn.compare(gpu, ref, wl)                                   # 5e-3 > 1e-5
    Hn.compare(gpu, ref, synth.Workload("h_bf", "gru", True, 2, True, 4, 3, 8, 8, "bf16", 5))


def test_sampled_columns():
    wl = synth.Workload("h_s", "lstm", False, 1, False, 4, 6, 8, 8, "f32", 6, state_std=0.5)
    keep = [1, 4]
    full = Hn.masked_dy(synth.make_inputs(wl), keep)
    ref_full = Hn.run_oracle(full)
    ref = Hn.run_oracle(synth.make_inputs(wl, batch_subset=keep))
    # the full run's sampled columns and weight gradients (dy zero elsewhere)
    # equal the run on the sampled columns alone
    Hn.compare(_as_gpu(ref_full), ref, wl, batch_idx=keep)
    gpu = _as_gpu(ref_full)
    gpu["y"][:, 0] += 1.0                        # a column that is not sampled
    Hn.compare(gpu, ref, wl, batch_idx=keep)
    gpu["y"][:, 4] += 1.0                        # a sampled one
    with pytest.raises(AssertionError):
        Hn.compare(gpu, ref, wl, batch_idx=keep)


def test_elementwise_error_definition():
    # floor 1e-3 of the tensor's scale: 0.5 is held to itself, 1e-6 to 4e-3
    r = np.array([4.0, 0.5, 1e-6])
    g = r + np.array([0.0, 0.05, 0.0])
    assert Hn.max_elem_rel_err(g, r) == pytest.approx(0.1)
    g = r + np.array([0.0, 0.0, 4e-4])
    assert Hn.max_elem_rel_err(g, r) == pytest.approx(0.1)
    assert Hn.max_elem_rel_err(np.zeros(2), np.zeros(2)) == 0.0
    assert Hn.max_elem_rel_err(np.ones(2), np.zeros(2)) == float("inf")


def test_elementwise_bound_catches_a_small_element():
    # an element near the floor (1e-3 of the tensor's scale) off by 1e-2 of
    # the scale passes the norm-wise bound (2e-2) but not the elementwise one
    # (about 10 > 6)
    wl, _, ref = _case("lstm", False, "bf16")
    gpu = _as_gpu(ref)
    y = ref["y"]
    scale = float(np.max(np.abs(y)))
    idx = np.unravel_index(np.argmin(np.abs(np.abs(y) - 1e-3 * scale)), y.shape)
    gpu["y"][idx] = y[idx] + 1e-2 * scale
    assert Hn.max_rel_err(gpu["y"], y) <= Hn.TOL["bf16"]
    with pytest.raises(AssertionError, match="elementwise"):
        Hn.compare(gpu, ref, wl)
