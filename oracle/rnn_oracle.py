"""fp64 CPU oracle for the multi-timestep LSTM / GRU layer, forward and BPTT.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or runs
this module: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm do.  It shares no code with the CUDA library.

It is a plain, slow, obviously correct restatement of the cell equations in
float64: one Python loop over time, numpy matrix products per step, no
blocking, fusion or reordering.  Gate blocks are in canonical order
(LSTM i, f, g, o; GRU r, z, n).  Sequences are seq-major [T, B, F]; states are
[L*D, B, H] indexed l*D + d.

Sources (the pages the method is taken from, by title, and the part of each):
  * The popnn Lstm.cpp page (Graphcore poplibs LSTM): the forward cell step,
    the backward step, and the weight update (weight-gradient accumulation
    into zeroed accumulators).
  * The popnn Gru.cpp page (Graphcore poplibs GRU): the reset-before and the
    resetAfter forward cell steps, their backward steps, and the weight
    update.
  * The persistent RNN backward-data kernel page (a recovered CUDA listing):
    the LSTM and GRU gate-gradient branches, the direction mapping of the
    step loop, and the initial-state gradients at step zero.
  * The SystemDS LibMatrixCuDNN.java page: the LSTM forward and backward
    operators (the forward / backward-data / backward-weights split, the
    absent final-state gradient).
  * Plain RNN cells (the persistent kernel page's ReLU / tanh branch):
    h' = act(W_ih x + W_hh h + b) with one gate; its backward step multiplies
    the state gradient by the activation's derivative (ReLU: zero where the
    output is not positive; tanh: 1 - h'^2).

Readings where the pages are silent:
  * LSTM cell clipping (the persistent kernel page's clip / dclip on the cell state), when
    enabled with bounds lo < hi: the state is the raw c, and every use of it
    goes through clip(x) = min(max(x, lo), hi) (a NaN stays NaN):
    c_t = f clip(c_{t-1}) + i g, h_t = o tanh(clip(c_t)); cy is the raw c_T;
    dclip(x) = 1 on [lo, hi], else 0; off by default (identity);
  * LSTM has one bias vector per direction (the sum of cuDNN's two);
  * the GRU update is h' = (1 - z) * n + z * h (both GRU sources agree);
  * resetAfter keeps separate input / recurrent biases, with the recurrent
    candidate bias inside the reset product: n = tanh(a^x_n + r * (W_hn h + b_hn));
  * reset-before has one bias; its candidate bias is on the input side:
    n = tanh(W_in x + b_n + W_hn (r * h));
  * dhy / dcy default to zero; weight gradients overwrite (never accumulate
    across calls).
  * variable sequence lengths (the popnn Gru.cpp and Lstm.cpp pages, the
    batchwise time-step mask of the forward and backward loops): sequence b has
    len_b <= T valid steps; at a step t >= len_b the mask m = 0 holds the
    state (h, c carried unchanged, the latched final state) and zeroes the
    output, h_t = m h' + (1 - m) h_{t-1}, c_t = m c' + (1 - m) c_{t-1},
    y_t = m h'.  The backward is the exact derivative of that: the gate
    gradients of a masked step are zero and the state gradients pass through
    it unchanged.  The reverse direction therefore starts from h0 at
    t = len_b - 1.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

LSTM, GRU = "lstm", "gru"
RNN_RELU, RNN_TANH = "rnn_relu", "rnn_tanh"   # plain RNN: h' = act(W_ih x + W_hh h + b)


def sigmoid(a: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-a))


def _time_order(T: int, reverse: bool):
    """The reverse direction walks t = T-1 .. 0 over the same inputs
    (direction mapping of the persistent kernel's step loop)."""
    return range(T - 1, -1, -1) if reverse else range(T)


def _clip(x, clip):
    """clip(x) = min(max(x, lo), hi); identity when ``clip`` is None."""
    if clip is None:
        return x
    lo, hi = clip
    return np.where(x < lo, lo, np.where(x > hi, hi, x))


def _dclip(x, clip):
    """Derivative of _clip: 1 on [lo, hi], 0 outside."""
    if clip is None:
        return np.ones_like(x)
    lo, hi = clip
    return ((x >= lo) & (x <= hi)).astype(float)


def _masks(T: int, B: int, lengths) -> np.ndarray:
    """m[t, b, 0] = 1 when step t is inside sequence b (t < len_b), else 0;
    all ones without lengths (the batchwise time-step mask)."""
    m = np.ones((T, B, 1))
    if lengths is not None:
        for b, n in enumerate(lengths):
            m[int(n):, b, 0] = 0.0
    return m


# ----------------------------------------------------------------------------
# LSTM, one direction of one layer
# ----------------------------------------------------------------------------
def lstm_forward_dir(x, p, h0, c0, reverse=False, lengths=None, clip=None):
    """The popnn Lstm.cpp page, forward cell step:
    a = W_ih x_t + W_hh h_{t-1} + b; i, f, o = sigmoid; g = tanh;
    c' = f c_{t-1} + i g; h' = o tanh(c').  With the step mask m:
    c_t = m c' + (1-m) c_{t-1}; h_t = m h' + (1-m) h_{t-1}; y_t = m h'.
    With cell clipping (bounds ``clip``): c' = f clip(c_{t-1}) + i g and
    h' = o tanh(clip(c'))."""
    T, B, _ = x.shape
    H = p["W_hh"].shape[1]
    M = _masks(T, B, lengths)
    h, c = h0, c0
    y = np.zeros((T, B, H))
    keep = {k: np.zeros((T, B, H)) for k in ("i", "f", "g", "o", "c", "c_prev", "h_prev")}
    keep["m"] = M
    keep["clip"] = clip
    for t in _time_order(T, reverse):
        m = M[t]
        a = x[t] @ p["W_ih"].T + h @ p["W_hh"].T + p["b"]
        i = sigmoid(a[:, 0 * H:1 * H])
        f = sigmoid(a[:, 1 * H:2 * H])
        g = np.tanh(a[:, 2 * H:3 * H])
        o = sigmoid(a[:, 3 * H:4 * H])
        c_new = f * _clip(c, clip) + i * g
        h_new = o * np.tanh(_clip(c_new, clip))
        for k, v in (("i", i), ("f", f), ("g", g), ("o", o), ("c", c_new),
                     ("c_prev", c), ("h_prev", h)):
            keep[k][t] = v
        y[t] = m * h_new
        h, c = m * h_new + (1.0 - m) * h, m * c_new + (1.0 - m) * c
    return y, h, c, keep


def lstm_backward_dir(x, p, keep, dy, dhT, dcT, reverse=False):
    """The popnn Lstm.cpp page, backward step, identical to the LSTM branch
    of the persistent RNN backward-data kernel page:
      dh = dy_t + dh_rec
      dc = dh o (1 - tanh^2 c_t) + dc_next
      da_i = dc g i(1-i); da_f = dc c_{t-1} f(1-f); da_g = dc i (1-g^2);
      da_o = dh tanh(c_t) o(1-o)
      dh_rec <- W_hh^T da; dc_next <- dc f
    Weight gradients (the page's weight update): dW_ih = sum da x^T,
    dW_hh = sum da h_{t-1}^T, db = sum da.
    Masked step (m = 0): the gate gradients are zero and dh_rec, dc_next pass
    through unchanged; dy_t does not reach the state.  With cell clipping
    (the persistent kernel page's LSTM branch): dc = dh o (1 - tanh^2 clip(c_t)) dclip(c_t)
    + dc_next, da_f uses clip(c_{t-1}), da_o uses tanh(clip(c_t)), and
    dc_next <- dc f dclip(c_{t-1})."""
    T, B, I = x.shape
    H = p["W_hh"].shape[1]
    M = keep["m"]
    clip = keep.get("clip")
    dA = np.zeros((T, B, 4 * H))
    dh_rec, dc_next = dhT, dcT
    for t in reversed(list(_time_order(T, reverse))):
        m = M[t]
        i, f, g, o = keep["i"][t], keep["f"][t], keep["g"][t], keep["o"][t]
        ct, cp = keep["c"][t], keep["c_prev"][t]
        tc = np.tanh(_clip(ct, clip))
        dh = m * (dy[t] + dh_rec)
        dc = dh * o * (1.0 - tc * tc) * _dclip(ct, clip) + m * dc_next
        dA[t, :, 0 * H:1 * H] = dc * g * i * (1.0 - i)
        dA[t, :, 1 * H:2 * H] = dc * _clip(cp, clip) * f * (1.0 - f)
        dA[t, :, 2 * H:3 * H] = dc * i * (1.0 - g * g)
        dA[t, :, 3 * H:4 * H] = dh * tc * o * (1.0 - o)
        dh_rec = dA[t] @ p["W_hh"] + (1.0 - m) * dh_rec
        dc_next = dc * f * _dclip(cp, clip) + (1.0 - m) * dc_next
    dx = dA @ p["W_ih"]
    flat = dA.reshape(T * B, 4 * H)
    grads = {"W_ih": flat.T @ x.reshape(T * B, I),
             "W_hh": flat.T @ keep["h_prev"].reshape(T * B, H),
             "b": flat.sum(axis=0)}
    return dx, dh_rec, dc_next, grads, dA


# ----------------------------------------------------------------------------
# GRU resetAfter, one direction of one layer
# ----------------------------------------------------------------------------
def gru_ra_forward_dir(x, p, h0, reverse=False, lengths=None):
    """The popnn Gru.cpp page, resetAfter forward cell step:
    a^x = W_ih x + b_i; a^h = W_hh h + b_h; r = s(a^x_r + a^h_r);
    z = s(a^x_z + a^h_z); n = tanh(a^x_n + r a^h_n); h' = (1-z) n + z h.
    With the step mask m: h_t = m h' + (1-m) h_{t-1}; y_t = m h'."""
    T, B, _ = x.shape
    H = p["W_hh"].shape[1]
    M = _masks(T, B, lengths)
    h = h0
    y = np.zeros((T, B, H))
    keep = {k: np.zeros((T, B, H)) for k in ("r", "z", "n", "hn", "h_prev")}
    keep["m"] = M
    for t in _time_order(T, reverse):
        m = M[t]
        ax = x[t] @ p["W_ih"].T + p["b"]
        ah = h @ p["W_hh"].T + p["b_h"]
        r = sigmoid(ax[:, 0:H] + ah[:, 0:H])
        z = sigmoid(ax[:, H:2 * H] + ah[:, H:2 * H])
        hn = ah[:, 2 * H:3 * H]
        n = np.tanh(ax[:, 2 * H:3 * H] + r * hn)
        h_new = (1.0 - z) * n + z * h
        for k, v in (("r", r), ("z", z), ("n", n), ("hn", hn), ("h_prev", h)):
            keep[k][t] = v
        y[t] = m * h_new
        h = m * h_new + (1.0 - m) * h
    return y, h, keep


def gru_ra_backward_dir(x, p, keep, dy, dhT, reverse=False):
    """The popnn Gru.cpp page, resetAfter backward step, identical to the GRU
    branch of the persistent RNN backward-data kernel page:
      dh = dy_t + dh_rec
      dn = dh (1-z)(1-n^2); dz = dh (h_{t-1} - n) z(1-z); dr = dn a^h_n r(1-r)
      input side dA^x = [dr, dz, dn]; recurrent side dA^h = [dr, dz, dn r]
      dh_rec <- W_hh^T dA^h + dh z
    Weight gradients: dW_ih = sum dA^x x^T, dW_hh = sum dA^h h^T,
    db_i = sum dA^x, db_h = sum dA^h.
    Masked step (m = 0): zero gate gradients, dh_rec passes through."""
    T, B, I = x.shape
    H = p["W_hh"].shape[1]
    M = keep["m"]
    dAx = np.zeros((T, B, 3 * H))
    dAh = np.zeros((T, B, 3 * H))
    dh_rec = dhT
    for t in reversed(list(_time_order(T, reverse))):
        m = M[t]
        r, z, n, hn, hp = (keep[k][t] for k in ("r", "z", "n", "hn", "h_prev"))
        dh = m * (dy[t] + dh_rec)
        dn = dh * (1.0 - z) * (1.0 - n * n)
        dz = dh * (hp - n) * z * (1.0 - z)
        dr = dn * hn * r * (1.0 - r)
        dAx[t] = np.concatenate([dr, dz, dn], axis=1)
        dAh[t] = np.concatenate([dr, dz, dn * r], axis=1)
        dh_rec = dAh[t] @ p["W_hh"] + dh * z + (1.0 - m) * dh_rec
    dx = dAx @ p["W_ih"]
    fx = dAx.reshape(T * B, 3 * H)
    fh = dAh.reshape(T * B, 3 * H)
    grads = {"W_ih": fx.T @ x.reshape(T * B, I),
             "W_hh": fh.T @ keep["h_prev"].reshape(T * B, H),
             "b": fx.sum(axis=0), "b_h": fh.sum(axis=0)}
    return dx, dh_rec, grads, (dAx, dAh)


# ----------------------------------------------------------------------------
# GRU reset-before, one direction of one layer
# ----------------------------------------------------------------------------
def gru_rb_forward_dir(x, p, h0, reverse=False, lengths=None):
    """The popnn Gru.cpp page, reset-before forward cell step:
    [r, z] = s(W_{ih,rz} x + W_{hh,rz} h + b_rz);
    n = tanh(W_in x + W_hn (r * h) + b_n); h' = (1-z) n + z h.
    With the step mask m: h_t = m h' + (1-m) h_{t-1}; y_t = m h'."""
    T, B, _ = x.shape
    H = p["W_hh"].shape[1]
    M = _masks(T, B, lengths)
    h = h0
    y = np.zeros((T, B, H))
    keep = {k: np.zeros((T, B, H)) for k in ("r", "z", "n", "rh", "h_prev")}
    keep["m"] = M
    Wi, Wh, b = p["W_ih"], p["W_hh"], p["b"]
    for t in _time_order(T, reverse):
        m = M[t]
        a_rz = x[t] @ Wi[0:2 * H].T + h @ Wh[0:2 * H].T + b[0:2 * H]
        r = sigmoid(a_rz[:, 0:H])
        z = sigmoid(a_rz[:, H:2 * H])
        rh = r * h
        n = np.tanh(x[t] @ Wi[2 * H:3 * H].T + rh @ Wh[2 * H:3 * H].T + b[2 * H:3 * H])
        h_new = (1.0 - z) * n + z * h
        for k, v in (("r", r), ("z", z), ("n", n), ("rh", rh), ("h_prev", h)):
            keep[k][t] = v
        y[t] = m * h_new
        h = m * h_new + (1.0 - m) * h
    return y, h, keep


def gru_rb_backward_dir(x, p, keep, dy, dhT, reverse=False):
    """The popnn Gru.cpp page, reset-before backward step:
      dh = dy_t + dh_rec
      dn = dh (1-z)(1-n^2); dz = dh (h_{t-1} - n) z(1-z)
      d(rh) = W_hn^T dn; dr = d(rh) * h_{t-1} * r(1-r)
      dh_rec <- d(rh) * r + W_{hh,rz}^T [dr, dz] + dh z
    Weight gradients (the page's weight update): dW_ih = sum [dr,dz,dn] x^T,
    dW_{hh,rz} = sum [dr,dz] h_{t-1}^T, dW_hn = sum dn (r*h_{t-1})^T,
    db = sum [dr, dz, dn].
    Masked step (m = 0): zero gate gradients, dh_rec passes through."""
    T, B, I = x.shape
    H = p["W_hh"].shape[1]
    Wh = p["W_hh"]
    M = keep["m"]
    dA = np.zeros((T, B, 3 * H))
    dh_rec = dhT
    for t in reversed(list(_time_order(T, reverse))):
        m = M[t]
        r, z, n, hp = (keep[k][t] for k in ("r", "z", "n", "h_prev"))
        dh = m * (dy[t] + dh_rec)
        dn = dh * (1.0 - z) * (1.0 - n * n)
        dz = dh * (hp - n) * z * (1.0 - z)
        drh = dn @ Wh[2 * H:3 * H]
        dr = drh * hp * r * (1.0 - r)
        dA[t] = np.concatenate([dr, dz, dn], axis=1)
        dh_rec = drh * r + dA[t, :, 0:2 * H] @ Wh[0:2 * H] + dh * z + (1.0 - m) * dh_rec
    dx = dA @ p["W_ih"]
    f = dA.reshape(T * B, 3 * H)
    dW_hh = np.concatenate([
        f[:, 0:2 * H].T @ keep["h_prev"].reshape(T * B, H),
        f[:, 2 * H:3 * H].T @ keep["rh"].reshape(T * B, H)], axis=0)
    grads = {"W_ih": f.T @ x.reshape(T * B, I), "W_hh": dW_hh, "b": f.sum(axis=0)}
    return dx, dh_rec, grads, dA


# ----------------------------------------------------------------------------
# plain RNN (ReLU / tanh), one direction of one layer
# ----------------------------------------------------------------------------
def _act(mode, a):
    return np.maximum(a, 0.0) if mode == RNN_RELU else np.tanh(a)


def _dact_from_out(mode, h):
    """Activation derivative expressed through its output, as the persistent kernel page's
    backward branch does: ReLU 1 where h > 0 else 0; tanh 1 - h^2."""
    return (h > 0.0).astype(float) if mode == RNN_RELU else 1.0 - h * h


def rnn_plain_forward_dir(mode, x, p, h0, reverse=False, lengths=None):
    """h' = act(W_ih x_t + W_hh h_{t-1} + b); with the step mask m:
    h_t = m h' + (1-m) h_{t-1}; y_t = m h'."""
    T, B, _ = x.shape
    H = p["W_hh"].shape[1]
    M = _masks(T, B, lengths)
    h = h0
    y = np.zeros((T, B, H))
    keep = {k: np.zeros((T, B, H)) for k in ("h", "h_prev")}
    keep["m"] = M
    for t in _time_order(T, reverse):
        m = M[t]
        h_new = _act(mode, x[t] @ p["W_ih"].T + h @ p["W_hh"].T + p["b"])
        keep["h"][t], keep["h_prev"][t] = h_new, h
        y[t] = m * h_new
        h = m * h_new + (1.0 - m) * h
    return y, h, keep


def rnn_plain_backward_dir(mode, x, p, keep, dy, dhT, reverse=False):
    """The persistent kernel page's plain-RNN branch: da = (dy_t + dh_rec) act'(h'),
    dh_rec <- W_hh^T da (masked steps: da = 0, dh_rec passes through).
    Weight gradients dW_ih = sum da x^T, dW_hh = sum da h_{t-1}^T,
    db = sum da."""
    T, B, I = x.shape
    H = p["W_hh"].shape[1]
    M = keep["m"]
    dA = np.zeros((T, B, H))
    dh_rec = dhT
    for t in reversed(list(_time_order(T, reverse))):
        m = M[t]
        dA[t] = m * (dy[t] + dh_rec) * _dact_from_out(mode, keep["h"][t])
        dh_rec = dA[t] @ p["W_hh"] + (1.0 - m) * dh_rec
    dx = dA @ p["W_ih"]
    flat = dA.reshape(T * B, H)
    grads = {"W_ih": flat.T @ x.reshape(T * B, I),
             "W_hh": flat.T @ keep["h_prev"].reshape(T * B, H),
             "b": flat.sum(axis=0)}
    return dx, dh_rec, grads, dA


# ----------------------------------------------------------------------------
# Stacked, optionally bidirectional layer
# ----------------------------------------------------------------------------
def rnn_forward(mode: str, reset_after: bool, params, x, h0=None, c0=None,
                bidirectional: bool = False, lengths=None, clip=None) -> Dict:
    """Layer l+1 reads layer l's output; a bidirectional layer's output is
    [y_fwd | y_bwd] on the feature axis; NULL initial states are zero.
    ``lengths`` (optional, [B] ints <= T): valid steps per sequence, the same
    for every layer and direction.  ``clip`` (optional, (lo, hi)): LSTM cell
    clipping bounds.
    Returns y [T,B,D*H], hy [L*D,B,H], cy (LSTM) and a cache for rnn_backward."""
    L, D = len(params), (2 if bidirectional else 1)
    T, B, _ = x.shape
    H = params[0][0]["W_hh"].shape[1]
    zeros = np.zeros((L * D, B, H))
    h0 = zeros if h0 is None else h0
    c0 = zeros if c0 is None else c0
    hy, cy = np.zeros((L * D, B, H)), np.zeros((L * D, B, H))
    layer_in, caches = x, []
    for l in range(L):
        outs, per_dir = [], []
        for d in range(D):
            s = l * D + d
            p = params[l][d]
            if mode == LSTM:
                y, hT, cT, keep = lstm_forward_dir(layer_in, p, h0[s], c0[s], reverse=(d == 1),
                                                   lengths=lengths, clip=clip)
                cy[s] = cT
            elif mode in (RNN_RELU, RNN_TANH):
                y, hT, keep = rnn_plain_forward_dir(mode, layer_in, p, h0[s], reverse=(d == 1), lengths=lengths)
            elif reset_after:
                y, hT, keep = gru_ra_forward_dir(layer_in, p, h0[s], reverse=(d == 1), lengths=lengths)
            else:
                y, hT, keep = gru_rb_forward_dir(layer_in, p, h0[s], reverse=(d == 1), lengths=lengths)
            hy[s] = hT
            outs.append(y)
            per_dir.append(keep)
        caches.append((layer_in, per_dir))
        layer_in = np.concatenate(outs, axis=2)
    out = {"y": layer_in, "hy": hy, "cache": caches}
    if mode == LSTM:
        out["cy"] = cy
    return out


def rnn_backward(mode: str, reset_after: bool, params, fwd: Dict, dy,
                 dhy=None, dcy=None, bidirectional: bool = False) -> Dict:
    """Backward through time and layers.  Layer l's output gradient is the
    caller's dy for the top layer, else the input gradient of layer l+1
    (summed over its directions).  Returns dx, dhx, dcx (LSTM), per-(layer,
    direction) canonical weight gradients ``dparams`` and the gate gradients
    ``dgates[l][d]``."""
    L, D = len(params), (2 if bidirectional else 1)
    T, B, _ = dy.shape
    H = params[0][0]["W_hh"].shape[1]
    zeros = np.zeros((L * D, B, H))
    dhy = zeros if dhy is None else dhy
    dcy = zeros if dcy is None else dcy
    dhx, dcx = np.zeros((L * D, B, H)), np.zeros((L * D, B, H))
    dparams: List[List[Optional[Dict]]] = [[None] * D for _ in range(L)]
    dgates: List[List[Optional[object]]] = [[None] * D for _ in range(L)]
    dout = dy
    dx = None
    for l in range(L - 1, -1, -1):
        layer_in, per_dir = fwd["cache"][l]
        dx = np.zeros(layer_in.shape)
        for d in range(D):
            s = l * D + d
            p = params[l][d]
            dyd = dout[:, :, d * H:(d + 1) * H]
            if mode == LSTM:
                dxd, dh0, dc0, g, dg = lstm_backward_dir(layer_in, p, per_dir[d], dyd,
                                                         dhy[s], dcy[s], reverse=(d == 1))
                dcx[s] = dc0
            elif mode in (RNN_RELU, RNN_TANH):
                dxd, dh0, g, dg = rnn_plain_backward_dir(mode, layer_in, p, per_dir[d], dyd,
                                                         dhy[s], reverse=(d == 1))
            elif reset_after:
                dxd, dh0, g, dg = gru_ra_backward_dir(layer_in, p, per_dir[d], dyd,
                                                      dhy[s], reverse=(d == 1))
            else:
                dxd, dh0, g, dg = gru_rb_backward_dir(layer_in, p, per_dir[d], dyd,
                                                      dhy[s], reverse=(d == 1))
            dhx[s] = dh0
            dx += dxd
            dparams[l][d] = g
            dgates[l][d] = dg
        dout = dx
    out = {"dx": dx, "dhx": dhx, "dparams": dparams, "dgates": dgates}
    if mode == LSTM:
        out["dcx"] = dcx
    return out


def rnn_loss(mode: str, fwd: Dict, dy, dhy=None, dcy=None) -> float:
    """The scalar whose gradient rnn_backward returns:
    L = sum_t sum_b <dy_t, y_t> + <dhy, h_T> + <dcy, c_T>."""
    L = float(np.sum(dy * fwd["y"]))
    if dhy is not None:
        L += float(np.sum(dhy * fwd["hy"]))
    if dcy is not None and mode == LSTM:
        L += float(np.sum(dcy * fwd["cy"]))
    return L


def run_inputs(inp, with_backward: bool = True) -> Dict:
    """Convenience: run a ``synth.Inputs`` bundle (duck-typed: .wl, .params,
    .x, .h0, .c0, .dy, .dhy, .dcy) through forward (+ backward)."""
    wl = inp.wl
    f = rnn_forward(wl.mode, wl.reset_after, inp.params, inp.x, inp.h0, inp.c0, wl.bidirectional,
                    lengths=getattr(inp, "lengths", None), clip=getattr(inp, "clip", None))
    out = {"y": f["y"], "hy": f["hy"]}
    if wl.mode == LSTM:
        out["cy"] = f["cy"]
    if with_backward:
        b = rnn_backward(wl.mode, wl.reset_after, inp.params, f, inp.dy, inp.dhy, inp.dcy,
                         wl.bidirectional)
        out.update({k: v for k, v in b.items()})
    out["fwd"] = f
    return out
