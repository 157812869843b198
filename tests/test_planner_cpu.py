"""Host logic of the tensor-core planners (no GPU): the persistent kernels'
candidate ranking by the per-step cost estimate, followed by the co-residency
filter the launch applies (emulated here with the limits measured on the
152-SM GB300: 7 clusters of 16 CTAs, 15 of 8, 36 of 4 at one CTA per SM), and
the GEMM's tile shape and K split.  Each pinned choice is the plan measured
fastest for that shape."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

LSTM, GRU = 0, 1
SMS = 152
MAX_CLUSTERS = {16: 7, 8: 15, 4: 36, 2: 76, 1: 152}


@pytest.fixture(scope="module")
def R():
    from bwd_persistent_cta_gb300 import build as B
    B.build()
    import bwd_persistent_cta_gb300 as mod
    return mod


def chosen(R, mode, bwd, H, B, ndir):
    """First candidate whose clusters can all be resident, as the launch picks it."""
    for p in R.rnn_debug_tc_plans(mode, bwd, H, B, ndir, SMS):
        if p["ctas"] // p["ks"] <= MAX_CLUSTERS[p["ks"]]:
            return p["ks"], p["nb"]
    return None


@pytest.mark.parametrize("mode,bwd,H,B,ndir,expect", [
    (GRU, 0, 512, 64, 1, (4, 2)),      # 0.586 -> 0.477 ms against (4, 1)
    (GRU, 1, 512, 64, 1, (8, 2)),      # 0.819 -> 0.606 ms against (8, 1)
    (LSTM, 0, 1024, 32, 1, (4, 1)),    # (2, 2): 1.08 -> 1.18 ms
    (LSTM, 1, 1024, 32, 1, (8, 1)),    # (4, 2): 1.30 -> 1.56 ms
    (LSTM, 0, 1024, 128, 2, (1, 2)),   # both directions in one launch, no K split: 12 weight
                                       # sub-tiles in tensor memory, no partial push
    (LSTM, 1, 1024, 128, 2, (4, 2)),   # both directions at once (12 sub-tiles in tensor memory)
    (LSTM, 1, 1024, 128, 1, (4, 4)),   # one direction alone: 17.8 -> 14.0 ms against (8, 1)
    (LSTM, 0, 2048, 8, 1, (2, 1)),     # split weight tile, 128 CTAs
])
def test_planner_choice(R, mode, bwd, H, B, ndir, expect):
    assert chosen(R, mode, bwd, H, B, ndir) == expect


def test_candidates_respect_resources(R):
    for mode, bwd, H, B in [(LSTM, 0, 1024, 128), (GRU, 1, 512, 64), (LSTM, 0, 2048, 8), (GRU, 1, 256, 200)]:
        plans = R.rnn_debug_tc_plans(mode, bwd, H, B, 1, SMS)
        assert plans
        for p in plans:
            assert p["ctas"] <= SMS
            assert p["smem"] <= 227 * 1024
            assert p["npad"] % 16 == 0 and p["npad"] <= 256
            assert p["pp"] in (1, 2, 4, 8)
            # weight sub-tiles in tensor memory sit above the accumulator's columns
            assert p["w_tmem"] % 2 == 0 and 512 - 32 * p["w_tmem"] >= p["npad"]
            # every batch part non-empty, at least 8 rows when split
            bp = -(-B // p["nb"])
            assert p["nb"] == 1 or (bp >= 8 and (p["nb"] - 1) * bp < B)


def test_no_plan_for_unsupported_shapes(R):
    assert R.rnn_debug_tc_plans(LSTM, 1, 96, 16, 1, SMS) == []    # backward needs H % 128 == 0
    assert R.rnn_debug_tc_plans(LSTM, 0, 512, 1100, 1, SMS) == []  # batch above 4 parts of 256


def test_large_batch_takes_batch_parts(R):
    # above 256 rows the MMA N limit needs 2 or 4 batch parts
    for H, B, nb_min in [(512, 300, 2), (512, 512, 2), (256, 600, 4)]:
        plans = R.rnn_debug_tc_plans(LSTM, 0, H, B, 1, SMS)
        assert plans and all(p["nb"] >= nb_min and p["npad"] <= 256 for p in plans)
    # hidden 512, batch 1000: 4 parts of 250 rows leave at most a K split of 2
    # on the 152 SMs, i.e. 16 pairs per thread: no tensor-core plan
    assert R.rnn_debug_tc_plans(LSTM, 0, 512, 1000, 1, SMS) == []


# SIMT persistent kernels: units per CTA from the cost model (exchange weighted
# as 500 serial FMAs, calibrated on GB300), and where the interleaved weight
# update is taken by default (several CTAs per direction and at most 16
# item-batch passes per thread per step).
@pytest.mark.parametrize("args,nblk_gt1,dw_default", [
    ((LSTM, 0, 0, 1, 32, 4, 1), False, False),     # fp32 T16 B4 H32: one CTA (148 vs 165 us with it)
    ((GRU, 0, 1, 1, 128, 8, 1), True, True),       # reset-before bf16: 8+ CTAs (30 -> 12 us per step)
    ((GRU, 1, 0, 1, 128, 16, 1), True, True),      # 1172 -> 1143 us per step with the interleave
    ((LSTM, 0, 0, 1, 256, 8, 2), True, False),     # 4 units x 8 rows = 32 passes: 974 vs 994 us
])
def test_simt_plan_choice(R, args, nblk_gt1, dw_default):
    p = R.rnn_debug_simt_plan(*args, num_sms=SMS)
    assert p is not None and not p["stream"]
    assert (p["nblk"] > 1) == nblk_gt1
    assert bool(p["dwhh_default"]) == dw_default
    assert p["dwhh_possible"]


def test_simt_streams_weights_that_do_not_fit(R):
    p = R.rnn_debug_simt_plan(LSTM, 0, 1, 0, 2048, 8, 1, SMS)
    assert p is not None and p["stream"] and p["nblk"] <= SMS
    assert not R.rnn_debug_simt_plan(LSTM, 0, 1, 1, 2048, 8, 1, SMS)["dwhh_possible"]


# Structural invariants over a sweep of shapes: what the kernel itself needs of
# a plan, independent of the cost ranking.  Each CTA owns 128 output rows of
# one direction (forward: 32 units x 4 gate slots of h W_hh^T; backward: 128
# units of dG W_hh), one 1/KS slice of the contraction dimension (forward H,
# backward 4H, in 64-column sub-tiles) and one batch part; its 256 threads
# cover the part's (unit, row) pairs of the epilogue PP at a time.
@pytest.mark.parametrize("mode", [LSTM, GRU])
@pytest.mark.parametrize("bwd", [0, 1])
@pytest.mark.parametrize("ndir", [1, 2])
def test_plan_invariants_sweep(R, mode, bwd, ndir):
    n_shapes = n_planned = 0
    for H in (32, 64, 96, 128, 192, 256, 384, 512, 768, 1024, 1536, 2048):
        for B in (1, 3, 8, 16, 33, 64, 100, 128, 200, 256, 300, 512, 600, 1024):
            n_shapes += 1
            plans = R.rnn_debug_tc_plans(mode, bwd, H, B, ndir, SMS, max_out=32)
            if bwd and H % 128:
                assert plans == []
                continue
            n_planned += bool(plans)
            rows, K = (H, 4 * H) if bwd else (4 * H, H)
            seen = set()
            for p in plans:
                ks, nb, npad, pp = p["ks"], p["nb"], p["npad"], p["pp"]
                assert (ks, nb) not in seen
                seen.add((ks, nb))
                assert ks in (1, 2, 4, 8, 16) and nb in (1, 2, 4) and pp in (1, 2, 4, 8)
                assert K % (ks * 64) == 0
                assert p["ctas"] == (rows // 128) * ks * nb * ndir <= SMS
                bp = -(-B // nb)
                assert bp <= 256 and npad == -(-bp // 16) * 16
                assert nb == 1 or (bp >= 8 and (nb - 1) * bp < B)
                units = (128 if bwd else 32) // ks
                assert units >= 1 and units * bp <= 256 * pp
                assert p["smem"] <= 227 * 1024
                assert p["w_tmem"] % 2 == 0 and 0 <= p["w_tmem"] <= K // ks // 64
                assert p["w_tmem"] == 0 or 512 - 32 * p["w_tmem"] >= npad
            if ndir == 2 and plans:
                assert R.rnn_debug_tc_plans(mode, bwd, H, B, 1, SMS, max_out=32)
    assert n_planned > n_shapes // 4


# The SIMT planner over a sweep: units per CTA cover the hidden size with no
# empty CTA, every CTA of the launch fits on its own SM, the 256 threads cover
# the (unit, row) pairs PP at a time, a resident weight slice stays within the
# shared-memory budget, and the interleaved weight update is only offered where
# the kernel can hold its accumulator (at most 16384 unit x hidden x batch
# products per CTA) and only taken by default with several CTAs per direction.
@pytest.mark.parametrize("mode,ra,bf16", [(LSTM, 0, 0), (LSTM, 0, 1), (GRU, 1, 1), (GRU, 0, 0), (GRU, 0, 1),
                                          (2, 0, 0), (3, 0, 1)])
@pytest.mark.parametrize("bwd", [0, 1])
def test_simt_plan_invariants_sweep(R, mode, ra, bf16, bwd):
    planned = 0
    for H in (8, 32, 40, 64, 128, 256, 512, 1024, 2048):
        for B in (1, 2, 5, 8, 16, 32, 64, 128):
            for ndir in (1, 2):
                p = R.rnn_debug_simt_plan(mode, ra, bf16, bwd, H, B, ndir, SMS)
                if p is None:
                    continue
                planned += 1
                nu, nblk, pp = p["nu"], p["nblk"], p["pp"]
                assert nblk == -(-H // nu) and (nblk - 1) * nu < H
                assert nblk * ndir <= SMS
                assert pp in (1, 2, 4, 8) and nu * B <= 256 * pp
                if not p["stream"]:
                    assert p["smem"] <= 200 * 1024
                if p["dwhh_default"]:
                    assert p["dwhh_possible"] and nblk > 1 and not p["stream"]
                q = R.rnn_debug_simt_plan(mode, ra, bf16, bwd, H, B, ndir, SMS, dwhh=1)
                if bwd and q is not None:
                    assert q["nu"] * H * B <= 16384 and not q["stream"] and q["smem"] <= 200 * 1024
    assert planned > 0


# ---------------------------------------------------------------------------
# tensor-core GEMM planner (host arithmetic): tile width, K split, tile rows
# ---------------------------------------------------------------------------
GIB = 1 << 30


@pytest.mark.parametrize("shapes,K,fp32,ws,expect", [
    # 2-layer bidirectional LSTM H1024 weight gradients (one launch per layer): 256-row tiles, no split
    ([(4096, 1024)] * 4, 65536, True, GIB, (256, 1, 256)),
    ([(4096, 2048), (4096, 1024)] * 2, 65536, True, GIB, (256, 1, 256)),
    # its dX (K = 8192) and projections (K = 1024 / 2048, bf16 output)
    ([(65536, 1024)], 8192, False, 0, (256, 1, 256)),
    ([(65536, 8192)], 1024, False, 0, (256, 1, 128)),
    ([(65536, 8192)], 2048, False, 0, (256, 1, 128)),
    # GRU H512 T128 B64 weight gradients: 64 tiles of 128 x 256 split in two
    ([(2048, 512)] * 2, 8192, True, 32 << 20, (256, 2, 128)),
    # without split scratch the same launch cannot split: 128-wide tiles double the tile count
    ([(2048, 512)] * 2, 8192, True, 0, (128, 1, 128)),
    # LSTM H1024 T256 B32 weight gradients: 128 tiles of 256 x 256 fill one wave
    ([(4096, 1024)] * 2, 8192, True, 64 << 20, (256, 1, 256)),
    # a small GEMM: 128-wide tiles double the tile count
    ([(256, 256)], 64, False, 0, (128, 1, 128)),
])
def test_gemm_plan(R, shapes, K, fp32, ws, expect):
    assert R.rnn_debug_gemm_plan(shapes, K, fp32, ws, SMS) == expect


def test_gemm_plan_rejects_bad_queries(R):
    with pytest.raises(ValueError):
        R.rnn_debug_gemm_plan([(0, 16)], 64, False, 0, SMS)
    with pytest.raises(ValueError):
        R.rnn_debug_gemm_plan([(16, 16)] * 7, 64, False, 0, SMS)
