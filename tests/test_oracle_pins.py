"""Pins for the fp64 oracle: checks against things other than the oracle itself.

* hand-derived single-unit cases with closed-form values (tests/golden);
* closed forms for zero weights and saturated gates;
* PyTorch's own fp64 CPU nn.LSTM / nn.GRU (a library special case: same i,f,g,o
  and r,z,n gate order, GRU in the resetAfter form) with autograd gradients;
* GRU reset-before equals resetAfter exactly when W_hn is diagonal and b_hn = 0
  (diagonal matrices commute with the elementwise reset product), and differs
  otherwise;
* central finite differences of the loss sum <dy, y> + <dhy, h_T> + <dcy, c_T>;
* structural invariants: reverse direction = forward on the time-reversed input;
  stacked layers = sequential single-layer calls;
* variable sequence lengths: a masked batch equals each sequence run alone on
  its own truncated length (outputs, final states, all gradients), full lengths
  equal no lengths, and the masked backward matches finite differences.
A final group plants mistakes in a copy of the oracle and checks that the pins
catch each one.
"""
import inspect
import math
import os
import types

import numpy as np
import pytest
import torch

from oracle import rnn_oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scalar_cells.txt")


def _parse_golden(path):
    cases, cur = {}, None
    env = {"log": math.log, "tanh": math.tanh, "atanh": math.atanh, "exp": math.exp}
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            cur = cases.setdefault(line.strip("[]"), {})
            continue
        k, v = line.split("=", 1)
        cur[k.strip()] = eval(v.strip(), {"__builtins__": {}}, env)
    return cases


GOLDEN_CASES = _parse_golden(GOLDEN)


def _scalar_params(case):
    p = {"W_ih": np.array(case["W_ih"], float).reshape(-1, 1),
         "W_hh": np.array(case["W_hh"], float).reshape(-1, 1),
         "b": np.array(case["b"], float)}
    if "b_h" in case:
        p["b_h"] = np.array(case["b_h"], float)
    return p


@pytest.mark.parametrize("name", sorted(GOLDEN_CASES))
def test_golden_scalar_cases(name):
    case = GOLDEN_CASES[name]
    x = np.array(case["x"], float).reshape(-1, 1, 1)
    p = _scalar_params(case)
    h0 = np.full((1, 1, 1), case["h0"])
    c0 = np.full((1, 1, 1), case["c0"])
    clip = tuple(case["clip"]) if "clip" in case else None
    f = O.rnn_forward(case["mode"], case["reset_after"], [[p]], x, h0, c0, clip=clip)
    np.testing.assert_allclose(f["y"][:, 0, 0], case["expect_h"], rtol=0, atol=1e-14)
    if "expect_c" in case:
        keep = f["cache"][0][1][0]
        np.testing.assert_allclose(keep["c"][:, 0, 0], case["expect_c"], rtol=0, atol=1e-14)
    if "expect_dc0_for_unit_dy" in case:
        b = O.rnn_backward(case["mode"], case["reset_after"], [[p]], f, np.ones_like(f["y"]))
        assert abs(b["dcx"][0, 0, 0] - case["expect_dc0_for_unit_dy"]) < 1e-14


def _rand_params(rng, mode, reset_after, L, D, I, H, scale=0.5):
    G = 4 if mode == "lstm" else (3 if mode == "gru" else 1)
    params = []
    for l in range(L):
        per = []
        for _ in range(D):
            Il = I if l == 0 else D * H
            p = {"W_ih": rng.uniform(-scale, scale, (G * H, Il)),
                 "W_hh": rng.uniform(-scale, scale, (G * H, H)),
                 "b": rng.uniform(-scale, scale, G * H)}
            if mode == "gru" and reset_after:
                p["b_h"] = rng.uniform(-scale, scale, G * H)
            per.append(p)
        params.append(per)
    return params


def test_lstm_zero_weights_closed_form():
    """W = 0: c_t = s_f c_{t-1} + s_i tanh(b_g) is a geometric recurrence with
    c_t = s_f^t c_0 + s_i g (1 - s_f^t) / (1 - s_f); h_t = s_o tanh(c_t)."""
    rng = np.random.default_rng(5)
    T, B, I, H = 9, 3, 4, 5
    p = {"W_ih": np.zeros((4 * H, I)), "W_hh": np.zeros((4 * H, H)), "b": rng.normal(size=4 * H)}
    x = rng.normal(size=(T, B, I))
    h0 = rng.normal(size=(1, B, H))
    c0 = rng.normal(size=(1, B, H))
    f = O.rnn_forward("lstm", False, [[p]], x, h0, c0)
    s = lambda v: 1 / (1 + math.e ** (-v))
    si, sf, g, so = (np.array([s(v) for v in p["b"][0:H]]), np.array([s(v) for v in p["b"][H:2 * H]]),
                     np.tanh(p["b"][2 * H:3 * H]), np.array([s(v) for v in p["b"][3 * H:]]))
    for t in range(1, T + 1):
        ct = sf ** t * c0[0] + si * g * (1 - sf ** t) / (1 - sf)
        np.testing.assert_allclose(f["y"][t - 1], so * np.tanh(ct), rtol=1e-13, atol=1e-14)


def test_lstm_saturated_gates_copy_and_reset():
    rng = np.random.default_rng(6)
    T, B, I, H = 7, 2, 3, 4
    p = {"W_ih": rng.uniform(-.1, .1, (4 * H, I)), "W_hh": rng.uniform(-.1, .1, (4 * H, H)),
         "b": rng.uniform(-.1, .1, 4 * H)}
    x = rng.uniform(-1, 1, (T, B, I))
    c0 = rng.normal(size=(1, B, H))
    # forget = 1, input = 0: the cell state is copied through all steps
    pc = {k: v.copy() for k, v in p.items()}
    pc["b"][0:H] = -60.0
    pc["b"][H:2 * H] = 60.0
    f = O.rnn_forward("lstm", False, [[pc]], x, None, c0)
    np.testing.assert_allclose(f["cy"][0], c0[0], rtol=0, atol=1e-15)
    # forget = 0, input = 1: c_t = g_t exactly, |c_t| < 1
    pr = {k: v.copy() for k, v in p.items()}
    pr["b"][0:H] = 60.0
    pr["b"][H:2 * H] = -60.0
    f = O.rnn_forward("lstm", False, [[pr]], x, None, c0)
    keep = f["cache"][0][1][0]
    np.testing.assert_allclose(keep["c"], keep["g"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("reset_after", [True, False])
def test_gru_saturated_update_gate(reset_after):
    """z = 1 keeps the state (h_T = h_0); z = 0 with W_hh = 0 gives h_t = n_t
    = tanh of the input-side candidate pre-activation (plus r * b_hn)."""
    rng = np.random.default_rng(7)
    T, B, I, H = 6, 2, 3, 4
    p = _rand_params(rng, "gru", reset_after, 1, 1, I, H, 0.3)[0][0]
    x = rng.uniform(-1, 1, (T, B, I))
    h0 = rng.normal(size=(1, B, H))
    pk = {k: v.copy() for k, v in p.items()}
    pk["b"][H:2 * H] = 60.0
    f = O.rnn_forward("gru", reset_after, [[pk]], x, h0)
    np.testing.assert_allclose(f["hy"][0], h0[0], rtol=0, atol=1e-14)
    pn = {k: v.copy() for k, v in p.items()}
    pn["b"][H:2 * H] = -60.0
    pn["W_hh"][:] = 0.0
    if reset_after:
        pn["b_h"][2 * H:] = 0.0
    f = O.rnn_forward("gru", reset_after, [[pn]], x, h0)
    expect = np.tanh(x @ pn["W_ih"][2 * H:].T + pn["b"][2 * H:])
    np.testing.assert_allclose(f["y"], expect, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# PyTorch fp64 nn.LSTM / nn.GRU as a library special case
# ---------------------------------------------------------------------------
def _torch_run(mode, params, x, h0, c0, dy, dhy, dcy, bidirectional):
    L, D = len(params), len(params[0])
    T, B, I = x.shape
    H = params[0][0]["W_hh"].shape[1]
    if mode in ("rnn_relu", "rnn_tanh"):
        m = torch.nn.RNN(I, H, num_layers=L, nonlinearity=mode[4:], bidirectional=bidirectional,
                         dtype=torch.float64)
    else:
        cls = torch.nn.LSTM if mode == "lstm" else torch.nn.GRU
        m = cls(I, H, num_layers=L, bidirectional=bidirectional, dtype=torch.float64)
    with torch.no_grad():
        for l in range(L):
            for d in range(D):
                sfx = f"_l{l}" + ("_reverse" if d else "")
                p = params[l][d]
                getattr(m, "weight_ih" + sfx).copy_(torch.from_numpy(p["W_ih"]))
                getattr(m, "weight_hh" + sfx).copy_(torch.from_numpy(p["W_hh"]))
                getattr(m, "bias_ih" + sfx).copy_(torch.from_numpy(p["b"]))
                getattr(m, "bias_hh" + sfx).copy_(
                    torch.from_numpy(p["b_h"]) if "b_h" in p else torch.zeros(p["b"].shape, dtype=torch.float64))
    xt = torch.from_numpy(x).requires_grad_(True)
    h0t = torch.from_numpy(h0).requires_grad_(True)
    if mode == "lstm":
        c0t = torch.from_numpy(c0).requires_grad_(True)
        y, (hy, cy) = m(xt, (h0t, c0t))
        loss = (y * torch.from_numpy(dy)).sum() + (hy * torch.from_numpy(dhy)).sum() + \
            (cy * torch.from_numpy(dcy)).sum()
    else:
        y, hy = m(xt, h0t)
        cy = None
        loss = (y * torch.from_numpy(dy)).sum() + (hy * torch.from_numpy(dhy)).sum()
    loss.backward()
    out = {"y": y.detach().numpy(), "hy": hy.detach().numpy(), "dx": xt.grad.numpy(),
           "dhx": h0t.grad.numpy(), "m": m}
    if mode == "lstm":
        out["cy"] = cy.detach().numpy()
        out["dcx"] = c0t.grad.numpy()
    return out


@pytest.mark.parametrize("mode,L,bidir", [("lstm", 1, False), ("lstm", 2, True),
                                          ("gru", 1, False), ("gru", 2, True),
                                          ("rnn_relu", 1, False), ("rnn_relu", 2, True),
                                          ("rnn_tanh", 1, False), ("rnn_tanh", 2, True)])
def test_matches_torch_fp64(mode, L, bidir):
    rng = np.random.default_rng(11)
    T, B, I, H = 6, 3, 5, 4
    D = 2 if bidir else 1
    params = _rand_params(rng, mode, True, L, D, I, H)
    x = rng.normal(size=(T, B, I))
    h0 = rng.normal(size=(L * D, B, H))
    c0 = rng.normal(size=(L * D, B, H))
    dy = rng.normal(size=(T, B, D * H))
    dhy = rng.normal(size=(L * D, B, H))
    dcy = rng.normal(size=(L * D, B, H))
    ref = _torch_run(mode, params, x, h0, c0, dy, dhy, dcy, bidir)
    f = O.rnn_forward(mode, True, params, x, h0, c0 if mode == "lstm" else None, bidir)
    b = O.rnn_backward(mode, True, params, f, dy, dhy, dcy if mode == "lstm" else None, bidir)
    tol = dict(rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f["y"], ref["y"], **tol)
    np.testing.assert_allclose(f["hy"], ref["hy"], **tol)
    np.testing.assert_allclose(b["dx"], ref["dx"], **tol)
    np.testing.assert_allclose(b["dhx"], ref["dhx"], **tol)
    if mode == "lstm":
        np.testing.assert_allclose(f["cy"], ref["cy"], **tol)
        np.testing.assert_allclose(b["dcx"], ref["dcx"], **tol)
    m = ref["m"]
    for l in range(L):
        for d in range(D):
            sfx = f"_l{l}" + ("_reverse" if d else "")
            g = b["dparams"][l][d]
            np.testing.assert_allclose(g["W_ih"], getattr(m, "weight_ih" + sfx).grad.numpy(), **tol)
            np.testing.assert_allclose(g["W_hh"], getattr(m, "weight_hh" + sfx).grad.numpy(), **tol)
            np.testing.assert_allclose(g["b"], getattr(m, "bias_ih" + sfx).grad.numpy(), **tol)
            if mode == "gru":
                np.testing.assert_allclose(g["b_h"], getattr(m, "bias_hh" + sfx).grad.numpy(), **tol)
            else:  # one LSTM / plain-RNN bias: its gradient equals both of torch's
                np.testing.assert_allclose(g["b"], getattr(m, "bias_hh" + sfx).grad.numpy(), **tol)


# ---------------------------------------------------------------------------
# reset-before vs resetAfter
# ---------------------------------------------------------------------------
def _rb_from_ra(p_ra):
    H = p_ra["W_hh"].shape[1]
    b = p_ra["b"].copy()
    b[0:2 * H] += p_ra["b_h"][0:2 * H]
    return {"W_ih": p_ra["W_ih"].copy(), "W_hh": p_ra["W_hh"].copy(), "b": b}


def test_gru_reset_before_equals_reset_after_for_diagonal_Whn():
    rng = np.random.default_rng(12)
    T, B, I, H = 7, 3, 4, 5
    p = _rand_params(rng, "gru", True, 1, 1, I, H)[0][0]
    p["W_hh"][2 * H:] = np.diag(rng.uniform(-1, 1, H))
    p["b_h"][2 * H:] = 0.0
    q = _rb_from_ra(p)
    x = rng.normal(size=(T, B, I))
    h0 = rng.normal(size=(1, B, H))
    dy = rng.normal(size=(T, B, H))
    fa = O.rnn_forward("gru", True, [[p]], x, h0)
    fb = O.rnn_forward("gru", False, [[q]], x, h0)
    np.testing.assert_allclose(fb["y"], fa["y"], rtol=1e-13, atol=1e-14)
    ba = O.rnn_backward("gru", True, [[p]], fa, dy)
    bb = O.rnn_backward("gru", False, [[q]], fb, dy)
    np.testing.assert_allclose(bb["dx"], ba["dx"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(bb["dhx"], ba["dhx"], rtol=1e-12, atol=1e-13)
    ga, gb = ba["dparams"][0][0], bb["dparams"][0][0]
    np.testing.assert_allclose(gb["W_ih"], ga["W_ih"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(gb["W_hh"][0:2 * H], ga["W_hh"][0:2 * H], rtol=1e-12, atol=1e-13)
    # on the diagonal of W_hn both parametrisations have the same derivative
    np.testing.assert_allclose(np.diag(gb["W_hh"][2 * H:]), np.diag(ga["W_hh"][2 * H:]),
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(gb["b"], ga["b"], rtol=1e-12, atol=1e-13)
    # a full W_hn separates the two forms
    p2 = dict(p)
    p2["W_hh"] = p["W_hh"].copy()
    p2["W_hh"][2 * H:] = rng.uniform(-1, 1, (H, H))
    q2 = _rb_from_ra(p2)
    ya = O.rnn_forward("gru", True, [[p2]], x, h0)["y"]
    yb = O.rnn_forward("gru", False, [[q2]], x, h0)["y"]
    assert np.max(np.abs(ya - yb)) > 1e-3


# ---------------------------------------------------------------------------
# central finite differences
# ---------------------------------------------------------------------------
def _fd_check(mode, reset_after, L, bidir, oracle=O, seed=13, T=3, B=2, I=3, H=2, rtol=1e-7, lengths=None,
              clip=None, state_scale=1.0):
    rng = np.random.default_rng(seed)
    D = 2 if bidir else 1
    params = _rand_params(rng, mode, reset_after, L, D, I, H, 0.8)
    x = rng.normal(size=(T, B, I))
    h0 = rng.normal(size=(L * D, B, H))
    c0 = rng.normal(size=(L * D, B, H)) * state_scale if mode == "lstm" else None
    dy = rng.normal(size=(T, B, D * H))
    dhy = rng.normal(size=(L * D, B, H))
    dcy = rng.normal(size=(L * D, B, H)) if mode == "lstm" else None

    def loss():
        f = oracle.rnn_forward(mode, reset_after, params, x, h0, c0, bidir, lengths=lengths, clip=clip)
        return oracle.rnn_loss(mode, f, dy, dhy, dcy)

    f = oracle.rnn_forward(mode, reset_after, params, x, h0, c0, bidir, lengths=lengths, clip=clip)
    g = oracle.rnn_backward(mode, reset_after, params, f, dy, dhy, dcy, bidir)
    checks = [(x, g["dx"]), (h0, g["dhx"])]
    if mode == "lstm":
        checks.append((c0, g["dcx"]))
    for l in range(L):
        for d in range(D):
            for k in params[l][d]:
                checks.append((params[l][d][k], g["dparams"][l][d][k]))
    eps = 1e-6
    worst = 0.0
    for arr, grad in checks:
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        scale = max(1.0, float(np.max(np.abs(num))))
        worst = max(worst, float(np.max(np.abs(num - grad))) / scale)
    return worst


@pytest.mark.parametrize("mode,reset_after", [("lstm", False), ("gru", True), ("gru", False), ("rnn_tanh", False)])
@pytest.mark.parametrize("L,bidir", [(1, False), (2, True)])
def test_finite_differences(mode, reset_after, L, bidir):
    assert _fd_check(mode, reset_after, L, bidir) < 1e-7


# ---------------------------------------------------------------------------
# structural invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode,reset_after", [("lstm", False), ("gru", True), ("gru", False)])
def test_reverse_direction_is_forward_on_reversed_time(mode, reset_after):
    rng = np.random.default_rng(14)
    T, B, I, H = 5, 2, 3, 4
    params = _rand_params(rng, mode, reset_after, 1, 2, I, H)
    x = rng.normal(size=(T, B, I))
    h0 = rng.normal(size=(2, B, H))
    c0 = rng.normal(size=(2, B, H)) if mode == "lstm" else None
    bi = O.rnn_forward(mode, reset_after, params, x, h0, c0, True)
    rev = O.rnn_forward(mode, reset_after, [[params[0][1]]], x[::-1].copy(), h0[1:2],
                        None if c0 is None else c0[1:2])
    np.testing.assert_allclose(bi["y"][:, :, H:], rev["y"][::-1], rtol=1e-14, atol=1e-15)
    fwd = O.rnn_forward(mode, reset_after, [[params[0][0]]], x, h0[0:1],
                        None if c0 is None else c0[0:1])
    np.testing.assert_allclose(bi["y"][:, :, :H], fwd["y"], rtol=1e-14, atol=1e-15)


def test_stacked_layers_equal_sequential_calls():
    rng = np.random.default_rng(15)
    T, B, I, H = 4, 2, 3, 5
    params = _rand_params(rng, "lstm", False, 2, 2, I, H)
    x = rng.normal(size=(T, B, I))
    both = O.rnn_forward("lstm", False, params, x, None, None, True)
    l0 = O.rnn_forward("lstm", False, params[0:1], x, None, None, True)
    l1 = O.rnn_forward("lstm", False, params[1:2], l0["y"], None, None, True)
    np.testing.assert_allclose(both["y"], l1["y"], rtol=0, atol=0)


def test_synth_flatten_roundtrip_and_gate_order():
    wl = synth.WORKLOADS["lstm_f32_T16_B4_I32_H32"].with_(gate_order=(1, 0, 3, 2), num_layers=2,
                                                          bidirectional=True)
    inp = synth.make_inputs(wl)
    flat = synth.flatten_params(wl, inp.params)
    assert flat.size == synth.weight_count(wl)
    back = synth.unflatten_params(wl, flat)
    H = wl.hidden_size
    for l in range(2):
        for d in range(2):
            for k in inp.params[l][d]:
                np.testing.assert_array_equal(back[l][d][k], inp.params[l][d][k])
    # block 0 of the flat W_ih holds canonical gate 1 (forget)
    np.testing.assert_array_equal(flat[0:H * wl.input_size].reshape(H, wl.input_size),
                                  inp.params[0][0]["W_ih"][H:2 * H])


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by a pin above
# ---------------------------------------------------------------------------
def _mutant(old, new):
    src = inspect.getsource(O)
    assert src.count(old) >= 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = [
    # (mode, reset_after, old text, new text)
    ("lstm", False, "dc = dh * o * (1.0 - tc * tc) * _dclip(ct, clip) + m * dc_next",
     "dc = dh * o * (1.0 - tc * tc) * _dclip(ct, clip)"),
    ("lstm", False, "dc_next = dc * f", "dc_next = dc * i"),
    ("lstm", False, "dA[t, :, 3 * H:4 * H] = dh * tc * o * (1.0 - o)",
     "dA[t, :, 3 * H:4 * H] = dc * tc * o * (1.0 - o)"),
    ("lstm", False, "dh_rec = dA[t] @ p[\"W_hh\"]", "dh_rec = dA[t] @ p[\"W_hh\"] * 0.5"),
    ("gru", True, "dz = dh * (hp - n) * z * (1.0 - z)", "dz = dh * (n - hp) * z * (1.0 - z)"),
    ("gru", True, "dAh[t] = np.concatenate([dr, dz, dn * r], axis=1)",
     "dAh[t] = np.concatenate([dr, dz, dn], axis=1)"),
    ("gru", True, "dh_rec = dAh[t] @ p[\"W_hh\"] + dh * z", "dh_rec = dAh[t] @ p[\"W_hh\"]"),
    ("gru", False, "dh_rec = drh * r + dA[t, :, 0:2 * H] @ Wh[0:2 * H] + dh * z",
     "dh_rec = drh + dA[t, :, 0:2 * H] @ Wh[0:2 * H] + dh * z"),
    ("gru", False, "f[:, 2 * H:3 * H].T @ keep[\"rh\"].reshape(T * B, H)",
     "f[:, 2 * H:3 * H].T @ keep[\"h_prev\"].reshape(T * B, H)"),
    ("rnn_tanh", False, "else 1.0 - h * h", "else 1.0 - h"),
    ("rnn_tanh", False, "dh_rec = dA[t] @ p[\"W_hh\"] + (1.0 - m) * dh_rec\n    dx = dA @ p[\"W_ih\"]\n    flat = dA.reshape(T * B, H)",
     "dh_rec = dA[t] @ p[\"W_ih\"][:, :H] + (1.0 - m) * dh_rec\n    dx = dA @ p[\"W_ih\"]\n    flat = dA.reshape(T * B, H)"),
]


@pytest.mark.parametrize("mode,reset_after,old,new", MUTATIONS)
def test_planted_backward_mistakes_fail_finite_differences(mode, reset_after, old, new):
    mut = _mutant(old, new)
    assert _fd_check(mode, reset_after, 1, False, oracle=mut, seed=21) > 1e-4


@pytest.mark.parametrize("old,new", [
    ("n = np.tanh(ax[:, 2 * H:3 * H] + r * hn)", "n = np.tanh(ax[:, 2 * H:3 * H] + hn)"),
    ("h_new = (1.0 - z) * n + z * h\n        for k, v in ((\"r\", r), (\"z\", z), (\"n\", n), (\"hn\"",
     "h_new = z * n + (1.0 - z) * h\n        for k, v in ((\"r\", r), (\"z\", z), (\"n\", n), (\"hn\""),
])
def test_planted_forward_mistakes_fail_golden_or_torch(old, new):
    mut = _mutant(old, new)
    case = GOLDEN_CASES["gru_reset_after_bias_inside_reset"]
    x = np.array(case["x"], float).reshape(-1, 1, 1)
    f = mut.rnn_forward("gru", True, [[_scalar_params(case)]], x, np.full((1, 1, 1), case["h0"]))
    assert abs(f["y"][0, 0, 0] - case["expect_h"][0]) > 1e-3


# ---------------------------------------------------------------------------
# variable sequence lengths
# ---------------------------------------------------------------------------
def _len_case(mode, reset_after, L, bidir, seed, T=6, B=4, I=3, H=4):
    rng = np.random.default_rng(seed)
    D = 2 if bidir else 1
    params = _rand_params(rng, mode, reset_after, L, D, I, H)
    x = rng.normal(size=(T, B, I))
    h0 = rng.normal(size=(L * D, B, H))
    c0 = rng.normal(size=(L * D, B, H)) if mode == "lstm" else None
    dy = rng.normal(size=(T, B, D * H))
    dhy = rng.normal(size=(L * D, B, H))
    dcy = rng.normal(size=(L * D, B, H)) if mode == "lstm" else None
    return params, x, h0, c0, dy, dhy, dcy


CELLS = [("lstm", False), ("gru", True), ("gru", False), ("rnn_relu", False), ("rnn_tanh", False)]


@pytest.mark.parametrize("mode,reset_after", CELLS)
def test_lengths_all_full_equal_no_lengths(mode, reset_after):
    params, x, h0, c0, dy, dhy, dcy = _len_case(mode, reset_after, 2, True, 31)
    T, B = x.shape[:2]
    a = O.rnn_forward(mode, reset_after, params, x, h0, c0, True)
    b = O.rnn_forward(mode, reset_after, params, x, h0, c0, True, lengths=[T] * B)
    ga = O.rnn_backward(mode, reset_after, params, a, dy, dhy, dcy, True)
    gb = O.rnn_backward(mode, reset_after, params, b, dy, dhy, dcy, True)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["hy"], b["hy"])
    assert np.array_equal(ga["dx"], gb["dx"]) and np.array_equal(ga["dhx"], gb["dhx"])
    for l in range(2):
        for d in range(2):
            for k in ga["dparams"][l][d]:
                assert np.array_equal(ga["dparams"][l][d][k], gb["dparams"][l][d][k])


@pytest.mark.parametrize("mode,reset_after", CELLS)
@pytest.mark.parametrize("L,bidir", [(1, False), (2, True)])
def test_lengths_equal_truncated_sequences(mode, reset_after, L, bidir):
    """Each sequence of a masked batch behaves as if run alone on its first
    len_b steps: outputs (zero beyond len_b), final states, input and state
    gradients; weight gradients are the sum over sequences of those runs."""
    params, x, h0, c0, dy, dhy, dcy = _len_case(mode, reset_after, L, bidir, 32 + L)
    T, B = x.shape[:2]
    D = 2 if bidir else 1
    lengths = [4, 6, 0, 1]
    f = O.rnn_forward(mode, reset_after, params, x, h0, c0, bidir, lengths=lengths)
    g = O.rnn_backward(mode, reset_after, params, f, dy, dhy, dcy, bidir)
    dw_sum = [[{k: np.zeros_like(v) for k, v in params[l][d].items()} for d in range(D)] for l in range(L)]
    for b, n in enumerate(lengths):
        assert np.all(f["y"][n:, b] == 0.0) and np.all(g["dx"][n:, b] == 0.0)
        if n == 0:
            assert np.array_equal(f["hy"][:, b], h0[:, b])
            assert np.array_equal(g["dhx"][:, b], dhy[:, b])
            if mode == "lstm":
                assert np.array_equal(f["cy"][:, b], c0[:, b])
                assert np.array_equal(g["dcx"][:, b], dcy[:, b])
            continue
        sl = slice(b, b + 1)
        c0b = c0[:, sl] if mode == "lstm" else None
        dcyb = dcy[:, sl] if mode == "lstm" else None
        fb = O.rnn_forward(mode, reset_after, params, x[:n, sl], h0[:, sl], c0b, bidir)
        gb = O.rnn_backward(mode, reset_after, params, fb, dy[:n, sl], dhy[:, sl], dcyb, bidir)
        assert np.allclose(f["y"][:n, sl], fb["y"], rtol=1e-12, atol=1e-13)
        assert np.allclose(f["hy"][:, sl], fb["hy"], rtol=1e-12, atol=1e-13)
        assert np.allclose(g["dx"][:n, sl], gb["dx"], rtol=1e-11, atol=1e-12)
        assert np.allclose(g["dhx"][:, sl], gb["dhx"], rtol=1e-11, atol=1e-12)
        if mode == "lstm":
            assert np.allclose(f["cy"][:, sl], fb["cy"], rtol=1e-12, atol=1e-13)
            assert np.allclose(g["dcx"][:, sl], gb["dcx"], rtol=1e-11, atol=1e-12)
        for l in range(L):
            for d in range(D):
                for k in dw_sum[l][d]:
                    dw_sum[l][d][k] += gb["dparams"][l][d][k]
    for l in range(L):
        for d in range(D):
            for k in dw_sum[l][d]:
                assert np.allclose(g["dparams"][l][d][k], dw_sum[l][d][k], rtol=1e-10, atol=1e-11), (l, d, k)


@pytest.mark.parametrize("mode,reset_after", CELLS)
def test_lengths_finite_differences(mode, reset_after):
    assert _fd_check(mode, reset_after, 2, True, seed=33, T=4, B=3, lengths=[4, 2, 0]) < 1e-7


@pytest.mark.parametrize("mode,reset_after,old,new", [
    ("lstm", False, "dh = m * (dy[t] + dh_rec)", "dh = dy[t] + dh_rec"),
    ("lstm", False, "dc_next = dc * f * _dclip(cp, clip) + (1.0 - m) * dc_next", "dc_next = dc * f * _dclip(cp, clip)"),
    ("gru", True, "dh_rec = dAh[t] @ p[\"W_hh\"] + dh * z + (1.0 - m) * dh_rec",
     "dh_rec = dAh[t] @ p[\"W_hh\"] + dh * z"),
    ("gru", False, "Wh[0:2 * H] + dh * z + (1.0 - m) * dh_rec", "Wh[0:2 * H] + dh * z + dh_rec"),
])
def test_planted_mask_mistakes_fail_finite_differences(mode, reset_after, old, new):
    mut = _mutant(old, new)
    assert _fd_check(mode, reset_after, 1, False, oracle=mut, seed=34, T=4, B=3, lengths=[4, 2, 0]) > 1e-4


@pytest.mark.parametrize("old,new", [
    ("        y[t] = m * h_new\n        h, c = m * h_new", "        y[t] = h_new\n        h, c = m * h_new"),
    ("h, c = m * h_new + (1.0 - m) * h, m * c_new + (1.0 - m) * c", "h, c = m * h_new, m * c_new"),
])
def test_planted_mask_forward_mistakes_fail_truncation(old, new):
    mut = _mutant(old, new)
    params, x, h0, c0, dy, dhy, dcy = _len_case("lstm", False, 1, True, 35)
    lengths = [4, 6, 0, 1]
    f = mut.rnn_forward("lstm", False, params, x, h0, c0, True, lengths=lengths)
    ok = True
    for b, n in enumerate(lengths):
        if n == 0:
            ok = ok and np.array_equal(f["hy"][:, b], h0[:, b]) and np.all(f["y"][:, b] == 0)
            continue
        fb = O.rnn_forward("lstm", False, params, x[:n, b:b + 1], h0[:, b:b + 1], c0[:, b:b + 1], True)
        ok = ok and np.allclose(f["y"][:, b:b + 1], np.concatenate(
            [fb["y"], np.zeros((x.shape[0] - n, 1, fb["y"].shape[2]))], axis=0)) and np.allclose(
            f["hy"][:, b:b + 1], fb["hy"])
    assert not ok


# ---------------------------------------------------------------------------
# LSTM cell clipping
# ---------------------------------------------------------------------------
def test_clip_with_unreached_bounds_is_identity():
    params, x, h0, c0, dy, dhy, dcy = _len_case("lstm", False, 2, True, 41)
    a = O.rnn_forward("lstm", False, params, x, h0, c0, True)
    b = O.rnn_forward("lstm", False, params, x, h0, c0, True, clip=(-1e9, 1e9))
    ga = O.rnn_backward("lstm", False, params, a, dy, dhy, dcy, True)
    gb = O.rnn_backward("lstm", False, params, b, dy, dhy, dcy, True)
    for k in ("y", "hy", "cy"):
        assert np.array_equal(a[k], b[k])
    for k in ("dx", "dhx", "dcx"):
        assert np.array_equal(ga[k], gb[k])


def _clip_case_is_active(seed, clip):
    """The clipped run differs from the unclipped one, and no cell value sits
    within the finite-difference step of a bound."""
    rng = np.random.default_rng(seed)
    params = _rand_params(rng, "lstm", False, 2, 2, 3, 2, 0.8)
    x = rng.normal(size=(4, 3, 3))
    f = O.rnn_forward("lstm", False, params, x, rng.normal(size=(4, 3, 2)), 3.0 * rng.normal(size=(4, 3, 2)), True,
                      clip=clip)
    cs = np.concatenate([k["c"].ravel() for _, per in f["cache"] for k in per] +
                        [k["c_prev"].ravel() for _, per in f["cache"] for k in per])
    outside = np.sum((cs < clip[0]) | (cs > clip[1]))
    margin = np.min(np.minimum(np.abs(cs - clip[0]), np.abs(cs - clip[1])))
    return outside, margin


def test_clip_finite_differences():
    clip = (-0.6, 0.7)
    outside, margin = _clip_case_is_active(42, clip)
    assert outside >= 5 and margin > 1e-4
    assert _fd_check("lstm", False, 2, True, seed=42, T=4, B=3, clip=clip, state_scale=3.0) < 1e-7


@pytest.mark.parametrize("old,new", [
    ("dc = dh * o * (1.0 - tc * tc) * _dclip(ct, clip) + m * dc_next", "dc = dh * o * (1.0 - tc * tc) + m * dc_next"),
    ("dc_next = dc * f * _dclip(cp, clip) + (1.0 - m) * dc_next", "dc_next = dc * f + (1.0 - m) * dc_next"),
    ("dc * _clip(cp, clip) * f * (1.0 - f)", "dc * cp * f * (1.0 - f)"),
])
def test_planted_clip_mistakes_fail_finite_differences(old, new):
    mut = _mutant(old, new)
    assert _fd_check("lstm", False, 2, True, oracle=mut, seed=42, T=4, B=3, clip=(-0.6, 0.7), state_scale=3.0) > 1e-4
