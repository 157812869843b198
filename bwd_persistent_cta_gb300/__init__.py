"""GB300 (sm_103a) multi-timestep LSTM / GRU layer: forward and BPTT.

Thin Python binding over the C ABI in ``include/rnn.h`` (library
``librnn.so`` built in-tree by ``build.py``).  The functions below carry the C
names and only marshal arguments: every step of forward, backward-data and
backward-weights runs in the library's CUDA kernels.  PyTorch is used for
device memory and the current stream.

``RNN`` is a convenience wrapper that allocates the workspace / reserve with
torch and calls the same entry points.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librnn.so")

RNN_OK, RNN_BAD_PARAM, RNN_NOT_SUPPORTED, RNN_CUDA_ERROR, RNN_TIMEOUT, RNN_BAD_WORKSPACE, RNN_INTERNAL = range(7)
RNN_LSTM, RNN_GRU, RNN_RNN_RELU, RNN_RNN_TANH = 0, 1, 2, 3
RNN_F32, RNN_BF16 = 0, 1
RNN_ALGO_AUTO, RNN_ALGO_PERSIST_TC, RNN_ALGO_PERSIST_SIMT = 0, 1, 2


class rnn_desc_t(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("gate_order", ctypes.c_int * 4), ("reset_after", ctypes.c_int),
                ("bidirectional", ctypes.c_int), ("num_layers", ctypes.c_int), ("seq_len", ctypes.c_int),
                ("batch", ctypes.c_int), ("input_size", ctypes.c_int), ("hidden_size", ctypes.c_int),
                ("dtype", ctypes.c_int), ("batch_first", ctypes.c_int), ("algo", ctypes.c_int)]


class RnnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {rnn_status_string(status)}" if what else rnn_status_string(status))


_lib = None
_P = ctypes.c_void_p
_SIGS = {
    "rnn_create": (ctypes.c_int, [ctypes.POINTER(rnn_desc_t), ctypes.POINTER(_P)]),
    "rnn_destroy": (ctypes.c_int, [_P]),
    "rnn_get_sizes": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_size_t)]),
    "rnn_forward": (ctypes.c_int, [_P] * 11),
    "rnn_backward_data": (ctypes.c_int, [_P] * 14),
    "rnn_backward_weights": (ctypes.c_int, [_P] * 8),
    "rnn_sync_status": (ctypes.c_int, [_P, _P]),
    "rnn_set_timeout_ns": (ctypes.c_int, [_P, ctypes.c_uint64]),
    "rnn_set_seq_lengths": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int)]),
    "rnn_set_cell_clip": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_double, ctypes.c_double]),
    "rnn_set_recomputation": (ctypes.c_int, [_P, ctypes.c_int]),
    "rnn_set_interleaved_dw": (ctypes.c_int, [_P, ctypes.c_int]),
    "rnn_interleaved_dw_active": (ctypes.c_int, [_P]),
    "rnn_launch_count": (ctypes.c_uint64, [_P]),
    "rnn_selected_algo": (ctypes.c_int, [_P]),
    "rnn_selected_fwd_algo": (ctypes.c_int, [_P]),
    "rnn_debug_skip_arrival": (ctypes.c_int, [_P, ctypes.c_int]),
    "rnn_debug_set_plan_overrides": (ctypes.c_int, [ctypes.c_int] * 8),
    "rnn_debug_gemm_plan": (ctypes.c_int, [ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                                            ctypes.c_int, _P]),
    "rnn_debug_tc_plans": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
    "rnn_debug_simt_plan": (ctypes.c_int, [ctypes.c_int] * 9 + [ctypes.POINTER(ctypes.c_int)]),
    "rnn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "rnn_set_timing": (ctypes.c_int, [_P, ctypes.c_int]),
    "rnn_get_timing": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint64)]),
    "rnn_get_timing_ex": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint64),
                                         ctypes.POINTER(ctypes.c_double)]),
    "rnn_forward_noalloc": (ctypes.c_int, [ctypes.POINTER(rnn_desc_t)] + [_P] * 7 + [ctypes.c_int, _P]),
    "rnn_noalloc_status": (ctypes.c_int, [_P]),
    "rnn_debug_gemm": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int64, ctypes.c_int,
                                      _P, ctypes.c_int64, ctypes.c_int, _P, ctypes.c_int64, ctypes.c_int, _P,
                                      ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int,
                                      ctypes.c_int, _P]),
}


def lib() -> ctypes.CDLL:
    """Load librnn.so (fails loudly when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with bwd_persistent_cta_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(t) -> Optional[int]:
    """Device pointer of a tensor (or None)."""
    return None if t is None else t.data_ptr()


def _stream(stream=None, device=None) -> int:
    """cudaStream_t of ``stream``, else of the current stream of ``device``
    (default: the current device)."""
    import torch
    return (stream if stream is not None else torch.cuda.current_stream(device)).cuda_stream


# --- the C entry points, same names -----------------------------------------
def rnn_status_string(status: int) -> str:
    return lib().rnn_status_string(int(status)).decode()


def rnn_create(desc: rnn_desc_t) -> int:
    h = _P()
    rc = lib().rnn_create(ctypes.byref(desc), ctypes.byref(h))
    if rc != RNN_OK:
        raise RnnError(rc, "rnn_create")
    return h.value


def rnn_destroy(handle: int) -> None:
    lib().rnn_destroy(handle)


def rnn_get_sizes(handle: int) -> Tuple[int, int, int]:
    w, ws, rs = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    rc = lib().rnn_get_sizes(handle, ctypes.byref(w), ctypes.byref(ws), ctypes.byref(rs))
    if rc != RNN_OK:
        raise RnnError(rc, "rnn_get_sizes")
    return w.value, ws.value, rs.value


def rnn_forward(handle, x, hx, cx, w, y, hy, cy, workspace, reserve, stream=None) -> int:
    return lib().rnn_forward(handle, x, hx, cx, w, y, hy, cy, workspace, reserve, stream)


def rnn_backward_data(handle, y, dy, dhy, dcy, w, hx, cx, dx, dhx, dcx, workspace, reserve, stream=None) -> int:
    return lib().rnn_backward_data(handle, y, dy, dhy, dcy, w, hx, cx, dx, dhx, dcx, workspace, reserve, stream)


def rnn_backward_weights(handle, x, hx, y, workspace, reserve, dw, stream=None) -> int:
    return lib().rnn_backward_weights(handle, x, hx, y, workspace, reserve, dw, stream)


def rnn_forward_noalloc(desc: rnn_desc_t, x, hx, cx, w, y, hy, cy, sync: int = 1, stream=None) -> int:
    """Inference forward with no device allocation by the library (scratch is
    a fixed array inside librnn.so); see include/rnn.h."""
    return lib().rnn_forward_noalloc(ctypes.byref(desc), x, hx, cx, w, y, hy, cy, int(sync), stream)


def rnn_noalloc_status(stream=None) -> int:
    """Status of the last rnn_forward_noalloc call on the current device (waits
    for ``stream`` and clears the status)."""
    return lib().rnn_noalloc_status(stream)


RNN_NOALLOC_SCRATCH_BYTES = 32 << 20


def rnn_sync_status(handle, stream=None) -> int:
    return lib().rnn_sync_status(handle, stream)


def rnn_set_timeout_ns(handle, ns: int) -> int:
    return lib().rnn_set_timeout_ns(handle, int(ns))


def rnn_set_seq_lengths(handle, lengths) -> int:
    """lengths: a sequence of batch ints in [0, seq_len], or None for full length."""
    if lengths is None:
        return lib().rnn_set_seq_lengths(handle, None)
    arr = (ctypes.c_int * len(lengths))(*[int(v) for v in lengths])
    return lib().rnn_set_seq_lengths(handle, arr)


def rnn_set_recomputation(handle, mode: int) -> int:
    return lib().rnn_set_recomputation(handle, int(mode))


def rnn_set_interleaved_dw(handle, mode: int) -> int:
    return lib().rnn_set_interleaved_dw(handle, int(mode))


def rnn_interleaved_dw_active(handle) -> int:
    return int(lib().rnn_interleaved_dw_active(handle))


def rnn_set_cell_clip(handle, enable: int, lo: float = 0.0, hi: float = 0.0) -> int:
    return lib().rnn_set_cell_clip(handle, int(enable), float(lo), float(hi))


def rnn_launch_count(handle) -> int:
    return int(lib().rnn_launch_count(handle))


def rnn_selected_algo(handle) -> int:
    return int(lib().rnn_selected_algo(handle))


def rnn_selected_fwd_algo(handle) -> int:
    return int(lib().rnn_selected_fwd_algo(handle))


RNN_TIMING_CLASSES = 8
TIMING_CLASS_NAMES = ("persist_fwd", "persist_bwd", "gemm_proj", "gemm_dx", "gemm_dw", "layout_seq", "layout_pack",
                      "recompute_cells")


def rnn_set_timing(handle, enable: bool) -> int:
    return lib().rnn_set_timing(handle, int(bool(enable)))


def rnn_get_timing(handle):
    """(ms[8], counts[8]) since the last read; waits for the recorded events."""
    ms = (ctypes.c_double * RNN_TIMING_CLASSES)()
    n = (ctypes.c_uint64 * RNN_TIMING_CLASSES)()
    rc = lib().rnn_get_timing(handle, ms, n)
    if rc != RNN_OK:
        raise RnnError(rc, "rnn_get_timing")
    return list(ms), [int(v) for v in n]


def rnn_get_timing_ex(handle):
    """(ms[8], counts[8], algorithmic bytes[8]) since the last read."""
    ms = (ctypes.c_double * RNN_TIMING_CLASSES)()
    n = (ctypes.c_uint64 * RNN_TIMING_CLASSES)()
    by = (ctypes.c_double * RNN_TIMING_CLASSES)()
    rc = lib().rnn_get_timing_ex(handle, ms, n, by)
    if rc != RNN_OK:
        raise RnnError(rc, "rnn_get_timing_ex")
    return list(ms), [int(v) for v in n], list(by)


def rnn_debug_gemm_plan(shapes, K: int, fp32_out: bool, ws_bytes: int, num_sms: int):
    """(tile width, K split, tile rows) the tensor-core GEMM planner picks for
    one grouped launch of GEMMs [(M, N), ...] of depth K (host arithmetic)."""
    n = len(shapes)
    Ms = (ctypes.c_int * n)(*[int(m) for m, _ in shapes])
    Ns = (ctypes.c_int * n)(*[int(nn) for _, nn in shapes])
    out = (ctypes.c_int * 3)()
    if not lib().rnn_debug_gemm_plan(n, Ms, Ns, int(K), int(bool(fp32_out)), int(ws_bytes), int(num_sms), out):
        raise ValueError("invalid GEMM plan query")
    return tuple(out)


def rnn_debug_tc_plans(mode: int, bwd: int, hidden: int, batch: int, ndir: int, num_sms: int, max_out: int = 16):
    """Candidate tensor-core plans, cheapest first: a list of dicts."""
    buf = (ctypes.c_int * (7 * max_out))()
    n = lib().rnn_debug_tc_plans(int(mode), int(bwd), int(hidden), int(batch), int(ndir), int(num_sms), buf,
                                 int(max_out))
    keys = ("ks", "nb", "ctas", "npad", "pp", "w_tmem", "smem")
    return [dict(zip(keys, buf[7 * i:7 * i + 7])) for i in range(n)]


def rnn_debug_simt_plan(mode: int, reset_after: int, is_bf16: int, bwd: int, hidden: int, batch: int, ndir: int,
                        num_sms: int, dwhh: int = 0):
    """The SIMT persistent kernel's plan for one launch shape (a dict), or None."""
    buf = (ctypes.c_int * 7)()
    ok = lib().rnn_debug_simt_plan(int(mode), int(reset_after), int(is_bf16), int(bwd), int(hidden), int(batch),
                                   int(ndir), int(num_sms), int(dwhh), buf)
    keys = ("nu", "nblk", "pp", "stream", "smem", "dwhh_default", "dwhh_possible")
    return dict(zip(keys, buf[:7])) if ok else None


def rnn_debug_skip_arrival(handle, cta: int) -> int:
    return lib().rnn_debug_skip_arrival(handle, int(cta))


def rnn_debug_set_plan_overrides(max_ks_fwd: int = 0, max_ks_bwd: int = 0, nb_fwd: int = 0, nb_bwd: int = 0,
                                 gemm_bn: int = 0, gemm_splits: int = 0, gemm_tm: int = 0,
                                 bwd_global_ks: int = 0) -> int:
    return lib().rnn_debug_set_plan_overrides(int(max_ks_fwd), int(max_ks_bwd), int(nb_fwd), int(nb_bwd),
                                              int(gemm_bn), int(gemm_splits), int(gemm_tm), int(bwd_global_ks))


def rnn_debug_gemm(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, C, ldc, c_bf16, bias, beta, rowmap_H, perm,
                   in_bf16, use_tc, stream=None) -> int:
    arr = (ctypes.c_int * 4)(*perm)
    return lib().rnn_debug_gemm(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, C, ldc, c_bf16, bias, beta,
                                rowmap_H, arr, in_bf16, use_tc, stream)


# --- convenience wrapper (torch allocation + the calls above) ----------------
class RNN:
    """One LSTM / GRU layer stack bound to a device.

    Tensors are seq-major [T, B, F] (or [B, T, F] with batch_first), states
    [L*D, B, H], weights a flat buffer in the layout ``rnn_get_sizes``
    documents.  dtype is torch.float32 or torch.bfloat16 for every tensor
    except dw (fp32)."""

    def __init__(self, mode: str, input_size: int, hidden_size: int, seq_len: int, batch: int,
                 num_layers: int = 1, bidirectional: bool = False, reset_after: bool = True,
                 dtype: str = "bf16", gate_order: Sequence[int] = (), batch_first: bool = False,
                 algo: int = RNN_ALGO_AUTO, device=None, recompute: bool = False, interleaved_dw: int = 1):
        modes = {"lstm": RNN_LSTM, "gru": RNN_GRU, "rnn_relu": RNN_RNN_RELU, "rnn_tanh": RNN_RNN_TANH}
        if mode not in modes:
            raise ValueError(f"mode must be one of {sorted(modes)}, not {mode!r}")
        if dtype not in ("bf16", "f32"):
            raise ValueError(f"dtype must be 'bf16' or 'f32', not {dtype!r}")
        if len(gate_order) > 4:
            raise ValueError(f"gate_order has at most 4 entries, not {len(gate_order)}")
        import torch
        self.torch = torch
        self.device = torch.device(device if device is not None else "cuda")
        if self.device.index is None:     # pin the device current now: the handle is bound to it
            self.device = torch.device("cuda", torch.cuda.current_device())
        d = rnn_desc_t()
        d.mode = modes[mode]
        for k, v in enumerate(gate_order):
            d.gate_order[k] = int(v)
        d.reset_after = int(bool(reset_after))
        d.bidirectional = int(bool(bidirectional))
        d.num_layers, d.seq_len, d.batch = num_layers, seq_len, batch
        d.input_size, d.hidden_size = input_size, hidden_size
        d.dtype = RNN_BF16 if dtype == "bf16" else RNN_F32
        d.batch_first = int(bool(batch_first))
        d.algo = int(algo)
        self.desc = d
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        with torch.cuda.device(self.device):
            self.handle = rnn_create(d)
        if recompute:
            self._check(rnn_set_recomputation(self.handle, 1), "rnn_set_recomputation")
        if int(interleaved_dw) != 1:
            self._check(rnn_set_interleaved_dw(self.handle, int(interleaved_dw)), "rnn_set_interleaved_dw")
        self.weight_bytes, self.workspace_bytes, self.reserve_bytes = rnn_get_sizes(self.handle)
        self.weight_count = self.weight_bytes // (2 if dtype == "bf16" else 4)
        self.workspace = torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=self.device)
        self.reserve = torch.empty(max(self.reserve_bytes, 256), dtype=torch.uint8, device=self.device)

    def close(self):
        if getattr(self, "handle", None):
            rnn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def algo(self) -> int:
        return rnn_selected_algo(self.handle)

    @property
    def fwd_algo(self) -> int:
        return rnn_selected_fwd_algo(self.handle)

    @property
    def interleaved_dw(self) -> bool:
        return bool(rnn_interleaved_dw_active(self.handle))

    def launches(self) -> int:
        return rnn_launch_count(self.handle)

    def _check(self, rc, what):
        if rc != RNN_OK:
            raise RnnError(rc, what)

    def _state_shape(self):
        d = self.desc
        return (d.num_layers * (2 if d.bidirectional else 1), d.batch, d.hidden_size)

    def _seq_shape(self, features: int):
        d = self.desc
        return (d.batch, d.seq_len, features) if d.batch_first else (d.seq_len, d.batch, features)

    def _want(self, t, name: str, shape=None, numel=None, dtype=None):
        """Raise unless ``t`` (None passes) can be handed to the C ABI as
        ``name``: a tensor on this handle's device, of the given shape (or
        element count) and dtype, contiguous and 16-byte aligned.  The library
        sees only pointers, so a wrong shape here would be an out-of-bounds
        access there."""
        if t is None:
            return
        torch = self.torch
        dtype = self.tdtype if dtype is None else dtype
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor, not {type(t).__name__}")
        if t.device != self.device:
            raise ValueError(f"{name} is on {t.device}; the handle is on {self.device}")
        if t.dtype != dtype:
            raise ValueError(f"{name} has dtype {t.dtype}; expected {dtype}")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}; expected {tuple(shape)}")
        if numel is not None and t.numel() != numel:
            raise ValueError(f"{name} has {t.numel()} elements; expected {numel}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.data_ptr() % 16:
            raise ValueError(f"{name} must start on a 16-byte boundary")

    def _check_forward(self, x, w, hx, cx, y, hy, cy):
        d = self.desc
        S = self._state_shape()
        self._want(x, "x", self._seq_shape(d.input_size))
        self._want(w, "w", numel=self.weight_count)
        for t, n in ((hx, "hx"), (cx, "cx"), (hy, "hy"), (cy, "cy")):
            self._want(t, n, S)
        self._want(y, "y", self._seq_shape((2 if d.bidirectional else 1) * d.hidden_size))

    def _check_backward_data(self, dy, w, dhy, dcy, dx, dhx, dcx, cx):
        d = self.desc
        S = self._state_shape()
        self._want(dy, "dy", self._seq_shape((2 if d.bidirectional else 1) * d.hidden_size))
        self._want(w, "w", numel=self.weight_count)
        for t, n in ((dhy, "dhy"), (dcy, "dcy"), (dhx, "dhx"), (dcx, "dcx"), (cx, "cx")):
            self._want(t, n, S)
        self._want(dx, "dx", self._seq_shape(d.input_size))

    def _check_backward_weights(self, x, dw):
        self._want(x, "x", self._seq_shape(self.desc.input_size))
        self._want(dw, "dw", numel=self.weight_count, dtype=self.torch.float32)

    def forward(self, x, w, hx=None, cx=None, train=True, y=None, hy=None, cy=None, stream=None):
        torch = self.torch
        d = self.desc
        D = 2 if d.bidirectional else 1
        shp = (d.batch, d.seq_len, D * d.hidden_size) if d.batch_first else (d.seq_len, d.batch, D * d.hidden_size)
        y = torch.empty(shp, dtype=self.tdtype, device=self.device) if y is None else y
        hy = torch.empty(self._state_shape(), dtype=self.tdtype, device=self.device) if hy is None else hy
        if d.mode == RNN_LSTM and cy is None:
            cy = torch.empty(self._state_shape(), dtype=self.tdtype, device=self.device)
        if x is None or w is None:
            raise ValueError("x and w are required")
        self._check_forward(x, w, hx, cx, y, hy, cy)
        rc = rnn_forward(self.handle, _p(x), _p(hx), _p(cx), _p(w), _p(y), _p(hy), _p(cy),
                         _p(self.workspace), _p(self.reserve) if train else None, _stream(stream, self.device))
        self._check(rc, "rnn_forward")
        return y, hy, cy

    def backward_data(self, dy, w, dhy=None, dcy=None, dx=None, dhx=None, dcx=None, stream=None, cx=None):
        torch = self.torch
        d = self.desc
        shp = (d.batch, d.seq_len, d.input_size) if d.batch_first else (d.seq_len, d.batch, d.input_size)
        dx = torch.empty(shp, dtype=self.tdtype, device=self.device) if dx is None else dx
        dhx = torch.empty(self._state_shape(), dtype=self.tdtype, device=self.device) if dhx is None else dhx
        if d.mode == RNN_LSTM and dcx is None:
            dcx = torch.empty(self._state_shape(), dtype=self.tdtype, device=self.device)
        if dy is None or w is None:
            raise ValueError("dy and w are required")
        self._check_backward_data(dy, w, dhy, dcy, dx, dhx, dcx, cx)
        rc = rnn_backward_data(self.handle, None, _p(dy), _p(dhy), _p(dcy), _p(w), None, _p(cx), _p(dx), _p(dhx),
                               _p(dcx), _p(self.workspace), _p(self.reserve), _stream(stream, self.device))
        self._check(rc, "rnn_backward_data")
        return dx, dhx, dcx

    def backward_weights(self, x, dw=None, stream=None):
        torch = self.torch
        dw = torch.empty(self.weight_count, dtype=torch.float32, device=self.device) if dw is None else dw
        if x is None:
            raise ValueError("x is required")
        self._check_backward_weights(x, dw)
        rc = rnn_backward_weights(self.handle, _p(x), None, None, _p(self.workspace), _p(self.reserve), _p(dw),
                                  _stream(stream, self.device))
        self._check(rc, "rnn_backward_weights")
        return dw

    def sync(self, stream=None):
        rc = rnn_sync_status(self.handle, _stream(stream, self.device))
        self._check(rc, "rnn_sync_status")

    def set_timeout_ns(self, ns: int):
        self._check(rnn_set_timeout_ns(self.handle, ns), "rnn_set_timeout_ns")

    def set_cell_clip(self, bounds):
        """LSTM cell clipping to (lo, hi), or None to turn it off."""
        if bounds is None:
            self._check(rnn_set_cell_clip(self.handle, 0), "rnn_set_cell_clip")
        else:
            self._check(rnn_set_cell_clip(self.handle, 1, bounds[0], bounds[1]), "rnn_set_cell_clip")

    def set_seq_lengths(self, lengths):
        """Valid steps per sequence (batch ints), or None for full length."""
        if lengths is not None and len(lengths) != self.desc.batch:
            raise ValueError("one length per sequence of the batch")
        self._check(rnn_set_seq_lengths(self.handle, lengths), "rnn_set_seq_lengths")

    def debug_skip_arrival(self, cta: int):
        self._check(rnn_debug_skip_arrival(self.handle, cta), "rnn_debug_skip_arrival")
