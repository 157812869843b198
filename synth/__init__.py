"""Seeded synthetic inputs for the multi-timestep LSTM / GRU layer.

This module is shared by the fp64 oracle side (tests, the CPU baseline) and the
CUDA side (tests, bench).  It draws random numbers and moves values between
layouts; it holds none of the recurrence's arithmetic.

Draw order (one ``torch.Generator('cpu')`` seeded per workload): for each layer,
for each direction: W_ih, W_hh, b (and b_h for GRU resetAfter); then x, h0, c0,
dy.  dhy and dcy are zero unless a test sets them.

Weights and biases are U(-1/sqrt(H), 1/sqrt(H)); the LSTM forget bias may get a
constant added (the "forget-gate bias +1.0" workload).  For bf16 workloads every
input is rounded to bf16 (round to nearest even) once, here, so the oracle and
the GPU see identical values.

Canonical gate order inside this module and the oracle:
  LSTM  i, f, g, o        (input, forget, candidate, output)
  GRU   r, z, n           (reset, update, candidate)
The flat weight buffer the C ABI takes stores the gate blocks in the caller's
``gate_order``: block k of every per-gate matrix holds canonical gate
``gate_order[k]``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

LSTM, GRU = "lstm", "gru"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str                    # "lstm" | "gru"
    reset_after: bool            # GRU only
    num_layers: int
    bidirectional: bool
    seq_len: int
    batch: int
    input_size: int
    hidden_size: int
    dtype: str                   # "f32" | "bf16"
    seed: int
    x_std: float = 1.0
    state_std: Optional[float] = 1.0   # None -> zero initial states
    dy_std: float = 1.0
    forget_bias: float = 0.0
    gate_order: Tuple[int, ...] = ()   # empty -> canonical
    forward_only: bool = False
    batch_first: bool = False
    # variable sequence lengths: None = every sequence has T steps; else the
    # lengths are drawn uniformly from [ceil(min_len_frac * T), T]
    min_len_frac: Optional[float] = None
    # LSTM recomputation mode: the backward pass recomputes the cell states
    recompute: bool = False

    @property
    def gates(self) -> int:
        return 4 if self.mode == LSTM else (3 if self.mode == GRU else 1)

    @property
    def dirs(self) -> int:
        return 2 if self.bidirectional else 1

    def layer_input(self, layer: int) -> int:
        return self.input_size if layer == 0 else self.dirs * self.hidden_size

    def order(self) -> Tuple[int, ...]:
        return tuple(self.gate_order) if self.gate_order else tuple(range(self.gates))

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def flops(self) -> float:
        """Algorithmic FLOPs of forward + backward-data + backward-weights:
        sum over layers and directions of 3 * 2*G*H*(I_l + H)*B*T."""
        G, H, B, T = self.gates, self.hidden_size, self.batch, self.seq_len
        f = 0.0
        for l in range(self.num_layers):
            f += self.dirs * 2.0 * G * H * (self.layer_input(l) + H) * B * T
        return f if self.forward_only else 3.0 * f


# The five workloads of the problem statement (sizes, seeds, distributions),
# and variable-length versions of two of them.
WORKLOADS: Dict[str, Workload] = {
    "lstm_f32_T16_B4_I32_H32": Workload(
        "lstm_f32_T16_B4_I32_H32", LSTM, False, 1, False, 16, 4, 32, 32, "f32", 0,
        state_std=1.0),
    "gru_ra_bf16_T128_B64_H512": Workload(
        "gru_ra_bf16_T128_B64_H512", GRU, True, 1, False, 128, 64, 512, 512, "bf16", 1,
        state_std=None),
    "lstm_bf16_T256_B32_H1024": Workload(
        "lstm_bf16_T256_B32_H1024", LSTM, False, 1, False, 256, 32, 1024, 1024, "bf16", 2,
        state_std=0.1, forget_bias=1.0),
    "lstm2bi_bf16_T512_B128_H1024": Workload(
        "lstm2bi_bf16_T512_B128_H1024", LSTM, False, 2, True, 512, 128, 1024, 1024, "bf16", 3,
        state_std=None),
    "gru_rb_bf16_T1024_B1_H2048": Workload(
        "gru_rb_bf16_T1024_B1_H2048", GRU, False, 1, False, 1024, 1, 2048, 2048, "bf16", 4,
        state_std=None, forward_only=True),
    "gru_rb_bf16_T1024_B8_H2048": Workload(
        "gru_rb_bf16_T1024_B8_H2048", GRU, False, 1, False, 1024, 8, 2048, 2048, "bf16", 4,
        state_std=None, forward_only=True),
    "lstm_bf16_T1024_B1_H2048": Workload(
        "lstm_bf16_T1024_B1_H2048", LSTM, False, 1, False, 1024, 1, 2048, 2048, "bf16", 4,
        state_std=None, forward_only=True),
    "lstm_bf16_T1024_B8_H2048": Workload(
        "lstm_bf16_T1024_B8_H2048", LSTM, False, 1, False, 1024, 8, 2048, 2048, "bf16", 4,
        state_std=None, forward_only=True),
    # variable sequence lengths (lengths uniform in [T/2, T]) on two of the shapes above
    "gru_ra_bf16_T128_B64_H512_varlen": Workload(
        "gru_ra_bf16_T128_B64_H512_varlen", GRU, True, 1, False, 128, 64, 512, 512, "bf16", 1,
        state_std=None, min_len_frac=0.5),
    "lstm2bi_bf16_T512_B128_H1024_varlen": Workload(
        "lstm2bi_bf16_T512_B128_H1024_varlen", LSTM, False, 2, True, 512, 128, 1024, 1024, "bf16", 3,
        state_std=None, min_len_frac=0.5),
    # the 2-layer bidirectional LSTM with the cell states recomputed in the backward pass
    "lstm2bi_bf16_T512_B128_H1024_recompute": Workload(
        "lstm2bi_bf16_T512_B128_H1024_recompute", LSTM, False, 2, True, 512, 128, 1024, 1024, "bf16", 3,
        state_std=None, recompute=True),
}


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even) and return float64."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


@dataclasses.dataclass
class Inputs:
    """One workload's values, all float64 (already bf16-rounded where the
    workload is bf16).  ``params[l][d]`` is a dict with canonical-order
    ``W_ih [G*H, I_l]``, ``W_hh [G*H, H]``, ``b [G*H]`` and, for GRU resetAfter,
    ``b_h [G*H]``.  Sequences are seq-major: x [T, B, I], dy [T, B, D*H];
    states are [L*D, B, H] with index l*D + d."""
    wl: Workload
    params: List[List[Dict[str, np.ndarray]]]
    x: np.ndarray
    h0: Optional[np.ndarray]
    c0: Optional[np.ndarray]
    dy: np.ndarray
    dhy: Optional[np.ndarray] = None
    dcy: Optional[np.ndarray] = None
    lengths: Optional[np.ndarray] = None   # [B] valid steps per sequence, or None (all T)
    clip: Optional[Tuple[float, float]] = None   # LSTM cell clipping bounds, or None


def make_lengths(wl: Workload) -> Optional[np.ndarray]:
    """The workload's [B] sequence lengths (None: every sequence has T steps),
    drawn from a generator of their own so that no other draw depends on them."""
    if wl.min_len_frac is None:
        return None
    T = wl.seq_len
    gl = torch.Generator(device="cpu").manual_seed(wl.seed + 7919)
    lo = min(T, int(math.ceil(wl.min_len_frac * T)))
    return torch.randint(lo, T + 1, (wl.batch,), generator=gl).numpy().astype(np.int64)


def make_inputs(wl: Workload, batch_subset: Optional[Sequence[int]] = None) -> Inputs:
    """Draw the workload's inputs.  ``batch_subset`` keeps only those batch
    columns of x, h0, c0 and dy (the draws themselves are unchanged)."""
    g = torch.Generator(device="cpu").manual_seed(wl.seed)
    G, H, T, B = wl.gates, wl.hidden_size, wl.seq_len, wl.batch
    k = 1.0 / math.sqrt(H)

    def uni(*shape):
        return (torch.rand(*shape, generator=g, dtype=torch.float64) * 2.0 - 1.0) * k

    def nrm(std, *shape):
        return torch.randn(*shape, generator=g, dtype=torch.float64) * std

    rnd = round_bf16 if wl.dtype == "bf16" else (lambda a: np.asarray(a, dtype=np.float64))
    params: List[List[Dict[str, np.ndarray]]] = []
    for l in range(wl.num_layers):
        per_dir = []
        for _d in range(wl.dirs):
            p = {"W_ih": uni(G * H, wl.layer_input(l)), "W_hh": uni(G * H, H), "b": uni(G * H)}
            if wl.mode == GRU and wl.reset_after:
                p["b_h"] = uni(G * H)
            if wl.mode == LSTM and wl.forget_bias:
                p["b"][H:2 * H] += wl.forget_bias
            per_dir.append({n: rnd(v.numpy()) for n, v in p.items()})
        params.append(per_dir)
    x = nrm(wl.x_std, T, B, wl.input_size).numpy()
    S = wl.num_layers * wl.dirs
    if wl.state_std is None:
        h0 = c0 = None
    else:
        h0 = nrm(wl.state_std, S, B, H).numpy()
        c0 = nrm(wl.state_std, S, B, H).numpy() if wl.mode == LSTM else None
    dy = nrm(wl.dy_std, T, B, wl.dirs * H).numpy()
    lengths = make_lengths(wl)
    if batch_subset is not None:
        idx = np.asarray(list(batch_subset))
        x, dy = x[:, idx], dy[:, idx]
        h0 = None if h0 is None else h0[:, idx]
        c0 = None if c0 is None else c0[:, idx]
        lengths = None if lengths is None else lengths[idx]
    return Inputs(wl, params, rnd(x), None if h0 is None else rnd(h0),
                  None if c0 is None else rnd(c0), rnd(dy), lengths=lengths)


# ----------------------------------------------------------------------------
# Flat weight buffer layout of the C ABI (pure index bookkeeping).
# ----------------------------------------------------------------------------
def param_names(wl: Workload) -> List[str]:
    names = ["W_ih", "W_hh", "b"]
    if wl.mode == GRU and wl.reset_after:
        names.append("b_h")
    return names


def param_shape(wl: Workload, layer: int, name: str) -> Tuple[int, ...]:
    GH = wl.gates * wl.hidden_size
    return {"W_ih": (GH, wl.layer_input(layer)), "W_hh": (GH, wl.hidden_size),
            "b": (GH,), "b_h": (GH,)}[name]


def weight_count(wl: Workload) -> int:
    n = 0
    for l in range(wl.num_layers):
        for _d in range(wl.dirs):
            for name in param_names(wl):
                n += int(np.prod(param_shape(wl, l, name)))
    return n


def _to_user_order(wl: Workload, a: np.ndarray) -> np.ndarray:
    H = wl.hidden_size
    blocks = [a[c * H:(c + 1) * H] for c in wl.order()]
    return np.concatenate(blocks, axis=0)


def _from_user_order(wl: Workload, a: np.ndarray) -> np.ndarray:
    H = wl.hidden_size
    out = np.empty_like(a)
    for k, c in enumerate(wl.order()):
        out[c * H:(c + 1) * H] = a[k * H:(k + 1) * H]
    return out


def flatten_params(wl: Workload, params) -> np.ndarray:
    """Canonical per-(layer, direction) dicts -> the flat buffer (float64)."""
    parts = []
    for l in range(wl.num_layers):
        for d in range(wl.dirs):
            for name in param_names(wl):
                parts.append(_to_user_order(wl, params[l][d][name]).reshape(-1))
    return np.concatenate(parts)


def unflatten_params(wl: Workload, flat: np.ndarray):
    """Flat buffer (weights or weight gradients) -> canonical dicts."""
    flat = np.asarray(flat, dtype=np.float64).reshape(-1)
    assert flat.size == weight_count(wl), (flat.size, weight_count(wl))
    out, off = [], 0
    for l in range(wl.num_layers):
        per_dir = []
        for _d in range(wl.dirs):
            p = {}
            for name in param_names(wl):
                shp = param_shape(wl, l, name)
                n = int(np.prod(shp))
                p[name] = _from_user_order(wl, flat[off:off + n].reshape(shp))
                off += n
            per_dir.append(p)
        out.append(per_dir)
    return out


def to_batch_first(a: np.ndarray) -> np.ndarray:
    """[T, B, F] -> [B, T, F]."""
    return np.ascontiguousarray(np.swapaxes(a, 0, 1))
