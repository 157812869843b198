"""Shared test helpers: run a synthetic workload through the C ABI on the GPU
and through the fp64 oracle, and compare them.

The GPU side goes through ``bwd_persistent_cta_gb300`` (ctypes over
librnn.so); the oracle side through ``oracle.rnn_oracle``.  Both get the same
seeded inputs from ``synth``.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import os

import numpy as np

import synth

TOL = {"f32": 1e-5, "bf16": 2e-2}
# Elementwise bound on |gpu - ref| / max(|ref|, 1e-3 ||ref||_inf), checked
# beside the norm-wise error: an element far below its tensor's scale is held
# to the floor 1e-3 ||ref||_inf instead of to its own size.  Rounding errors
# are absolute at the scale of the operands (bf16 storage of states, gates and
# gate gradients: about 2^-8 of the scale), not relative to each element, so
# at the floor the metric is the norm-wise error divided by 1e-3: with bf16
# storage norm-wise errors of 3-6e-3 give elementwise values up to about 4
# (3.8 the largest over all GPU parity cases), fp32 up to about 5e-4.  The
# bounds leave a margin of 1.6 (bf16) and 4 (fp32) over those; the norm-wise
# bounds alone would allow 20 and 1e-2.
ELEM_TOL = {"f32": 2e-3, "bf16": 6.0}
ELEM_FLOOR = 1e-3


def max_elem_rel_err(gpu: np.ndarray, ref: np.ndarray, floor: float = ELEM_FLOOR) -> float:
    """max |gpu - ref| / max(|ref|, floor * ||ref||_inf) over the elements (0
    when ref vanishes)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if not ref.size:
        return 0.0
    scale = float(np.max(np.abs(ref)))
    if scale == 0.0:
        return 0.0 if np.all(gpu == 0.0) else float("inf")
    den = np.maximum(np.abs(ref), floor * scale)
    return float(np.max(np.abs(gpu - ref) / den))


def max_rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """||gpu - ref||_inf / ||ref||_inf (0 when both vanish)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


def torch_dtype(wl):
    import torch
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def to_dev(a: Optional[np.ndarray], wl, device="cuda"):
    import torch
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=torch_dtype(wl))


def to_np(t) -> Optional[np.ndarray]:
    if t is None:
        return None
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_gpu(inp: "synth.Inputs", algo: int = 0, backward: bool = True, repeat: int = 1,
            interleaved_dw: int = 1) -> Dict:
    """Forward (+ backward data + weights) through the C ABI.  Results are
    returned seq-major and in canonical gate order (float64)."""
    import torch
    import bwd_persistent_cta_gb300 as R
    from bwd_persistent_cta_gb300 import build as B

    B.build()
    wl = inp.wl
    T, Bt, _ = inp.x.shape
    rnn = R.RNN(wl.mode, wl.input_size, wl.hidden_size, T, Bt, wl.num_layers, wl.bidirectional, wl.reset_after,
                wl.dtype, wl.gate_order, wl.batch_first, algo, recompute=wl.recompute,
                interleaved_dw=interleaved_dw)
    try:
        if inp.lengths is not None:
            rnn.set_seq_lengths([int(v) for v in inp.lengths])
        if inp.clip is not None:
            rnn.set_cell_clip(inp.clip)
        w = to_dev(synth.flatten_params(wl, inp.params), wl)
        xs = synth.to_batch_first(inp.x) if wl.batch_first else inp.x
        x = to_dev(xs, wl)
        hx, cx = to_dev(inp.h0, wl), to_dev(inp.c0, wl)
        out = {}
        for _ in range(repeat):
            y, hy, cy = rnn.forward(x, w, hx, cx, train=backward)
            if backward:
                dys = synth.to_batch_first(inp.dy) if wl.batch_first else inp.dy
                dy = to_dev(dys, wl)
                dx, dhx, dcx = rnn.backward_data(dy, w, to_dev(inp.dhy, wl), to_dev(inp.dcy, wl), cx=cx)
                dw = rnn.backward_weights(x)
            rnn.sync()
        yn = to_np(y)
        out["y"] = np.swapaxes(yn, 0, 1) if wl.batch_first else yn
        out["hy"] = to_np(hy)
        if wl.mode == "lstm":
            out["cy"] = to_np(cy)
        if backward:
            dxn = to_np(dx)
            out["dx"] = np.swapaxes(dxn, 0, 1) if wl.batch_first else dxn
            out["dhx"] = to_np(dhx)
            if wl.mode == "lstm":
                out["dcx"] = to_np(dcx)
            out["dparams"] = synth.unflatten_params(wl, dw.cpu().numpy())
        out["algo"] = rnn.algo
        out["fwd_algo"] = rnn.fwd_algo
        out["launches"] = rnn.launches()
        out["interleaved_dw"] = rnn.interleaved_dw
        out["reserve_bytes"] = rnn.reserve_bytes
        torch.cuda.synchronize()
        return out
    finally:
        rnn.close()


def run_oracle(inp: "synth.Inputs", backward: bool = True) -> Dict:
    from oracle import rnn_oracle
    return rnn_oracle.run_inputs(inp, with_backward=backward)


def compare(gpu: Dict, ref: Dict, wl, tol: Optional[float] = None, batch_idx: Optional[Sequence[int]] = None,
            skip: Sequence[str] = (), elem_tol: Optional[float] = None) -> Dict[str, float]:
    """Max relative error per output tensor (||gpu - ref||_inf / ||ref||_inf);
    asserts each is within ``tol``, and the elementwise error (see
    max_elem_rel_err) within ``elem_tol``.  ``batch_idx`` restricts the GPU's
    sequence and state outputs to the batch columns the oracle ran.  Returns
    the norm-wise errors; the elementwise ones are in ``compare.last_elem``.
    With RNN_PARITY_LOG set, appends both to that file (one JSON line)."""
    tol = TOL[wl.dtype] if tol is None else tol
    elem_tol = ELEM_TOL[wl.dtype] if elem_tol is None else elem_tol
    errs = {}
    elem = {}
    # every output the oracle produced must be there to compare
    missing = [k for k in ("y", "hy", "cy", "dx", "dhx", "dcx", "dparams") if k in ref and k not in skip
               and k not in gpu]
    assert not missing, f"GPU result lacks {missing}"

    def sel(a, axis):
        return a if batch_idx is None else np.take(a, list(batch_idx), axis=axis)

    for k in ("y", "dx", "hy", "cy", "dhx", "dcx"):
        if k in ref and k in gpu and k not in skip:
            errs[k] = max_rel_err(sel(gpu[k], 1), ref[k])
            elem[k] = max_elem_rel_err(sel(gpu[k], 1), ref[k])
    if "dparams" in ref and "dparams" in gpu and "dparams" not in skip:
        for l, per in enumerate(ref["dparams"]):
            for d, g in enumerate(per):
                for name, v in g.items():
                    errs[f"d{name}[{l},{d}]"] = max_rel_err(gpu["dparams"][l][d][name], v)
                    elem[f"d{name}[{l},{d}]"] = max_elem_rel_err(gpu["dparams"][l][d][name], v)
    assert "y" in errs or "y" in skip, "nothing compared"
    compare.last_elem = elem
    log = os.environ.get("RNN_PARITY_LOG")
    if log:
        import json
        with open(log, "a") as f:
            f.write(json.dumps({"workload": wl.name, "dtype": wl.dtype, "norm": errs, "elem": elem}) + "\n")
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"max rel err above {tol}: {bad} (all: {errs})"
    bad = {k: v for k, v in elem.items() if not (v <= elem_tol)}
    assert not bad, f"elementwise rel err above {elem_tol}: {bad} (all: {elem})"
    return errs


def masked_dy(inp: "synth.Inputs", keep: Sequence[int]) -> "synth.Inputs":
    """Copy of ``inp`` whose dy is zero outside the batch columns ``keep``."""
    import dataclasses
    dy = np.zeros_like(inp.dy)
    dy[:, list(keep)] = inp.dy[:, list(keep)]
    return dataclasses.replace(inp, dy=dy)
