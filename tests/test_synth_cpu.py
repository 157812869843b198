"""The seeded input generator (synth) that both the GPU path and the oracle
take their inputs from: the same seed gives the same draws; a batch subset is
exactly those columns of the full draw (the sampled full-size parity tests
rely on it); bf16 workloads hold bf16-representable values; the
variable-length workloads draw lengths in [ceil(T/2), T] and change no other
input."""
import math

import numpy as np
import pytest

import synth


def _small(name, **kw):
    base = dict(mode="lstm", reset_after=False, num_layers=2, bidirectional=True, seq_len=7, batch=6,
                input_size=5, hidden_size=8, dtype="bf16", seed=3, state_std=0.5)
    base.update(kw)
    return synth.Workload(name, base.pop("mode"), base.pop("reset_after"), base.pop("num_layers"),
                          base.pop("bidirectional"), base.pop("seq_len"), base.pop("batch"), base.pop("input_size"),
                          base.pop("hidden_size"), base.pop("dtype"), base.pop("seed"), **base)


def test_same_seed_same_draws():
    wl = _small("a")
    a, b = synth.make_inputs(wl), synth.make_inputs(wl)
    for k in ("x", "h0", "c0", "dy"):
        np.testing.assert_array_equal(getattr(a, k), getattr(b, k))
    for pa, pb in zip(a.params, b.params):
        for da, db in zip(pa, pb):
            for n in da:
                np.testing.assert_array_equal(da[n], db[n])


@pytest.mark.parametrize("keep", [[0], [5], [1, 4], [0, 2, 5]])
def test_batch_subset_is_the_full_draws_columns(keep):
    wl = _small("s", mode="gru", reset_after=True)
    full, sub = synth.make_inputs(wl), synth.make_inputs(wl, batch_subset=keep)
    np.testing.assert_array_equal(sub.x, full.x[:, keep])
    np.testing.assert_array_equal(sub.dy, full.dy[:, keep])
    np.testing.assert_array_equal(sub.h0, full.h0[:, keep])
    for pf, ps in zip(full.params, sub.params):
        for df, ds in zip(pf, ps):
            for n in df:
                np.testing.assert_array_equal(df[n], ds[n])


def test_bf16_values_are_representable():
    inp = synth.make_inputs(_small("b"))
    for arr in [inp.x, inp.dy, inp.h0] + [v for per in inp.params for d in per for v in d.values()]:
        assert np.array_equal(synth.round_bf16(arr), arr)


def test_varlen_lengths_range_and_other_draws_unchanged():
    for name in ("gru_ra_bf16_T128_B64_H512", "lstm2bi_bf16_T512_B128_H1024"):
        fixed = synth.WORKLOADS[name]
        var = synth.WORKLOADS[name + "_varlen"]
        T = var.seq_len
        small_fixed = synth.Workload("f", fixed.mode, fixed.reset_after, 1, False, T, 16, 8, 16, fixed.dtype,
                                     fixed.seed)
        small_var = synth.Workload("v", fixed.mode, fixed.reset_after, 1, False, T, 16, 8, 16, fixed.dtype,
                                   fixed.seed, min_len_frac=var.min_len_frac)
        a, b = synth.make_inputs(small_fixed), synth.make_inputs(small_var)
        np.testing.assert_array_equal(a.x, b.x)
        np.testing.assert_array_equal(a.dy, b.dy)
        assert a.lengths is None
        lo = math.ceil(var.min_len_frac * T)
        assert b.lengths.min() >= lo and b.lengths.max() <= T
