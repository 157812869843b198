"""Host-side checks that need no GPU: the library builds and loads, exports
every function the public headers declare, reports status strings, and fails
cleanly (an error code, no crash) when no CUDA device is present."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in ("rnn.h", "rnn_debug.h"):
        txt = open(os.path.join(ROOT, "include", h)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names |= set(re.findall(r"\b(rnn_[a-z_]+)\s*\(", txt))
    return names


@pytest.fixture(scope="module")
def lib():
    from bwd_persistent_cta_gb300 import build
    build.build()
    import bwd_persistent_cta_gb300 as R
    return R.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"rnn_create", "rnn_forward", "rnn_backward_data", "rnn_backward_weights"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_status_strings(lib):
    import bwd_persistent_cta_gb300 as R
    for code in range(7):
        s = R.rnn_status_string(code)
        assert s.startswith("RNN_")
    assert "unknown" in R.rnn_status_string(99)


def test_binding_names_match_header():
    import bwd_persistent_cta_gb300 as R
    for n in _declared():
        assert callable(getattr(R, n)), n


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-device path")
def test_create_without_device_fails_cleanly(lib):
    import bwd_persistent_cta_gb300 as R
    d = R.rnn_desc_t()
    d.mode, d.num_layers, d.seq_len, d.batch, d.input_size, d.hidden_size = 0, 1, 4, 2, 8, 8
    d.dtype = R.RNN_BF16
    h = ctypes.c_void_p()
    rc = lib.rnn_create(ctypes.byref(d), ctypes.byref(h))
    assert rc in (R.RNN_CUDA_ERROR, R.RNN_NOT_SUPPORTED)
    assert not h.value


def test_bad_descriptor_rejected_before_any_device_call(lib):
    import bwd_persistent_cta_gb300 as R
    d = R.rnn_desc_t()
    d.mode, d.num_layers, d.seq_len, d.batch, d.input_size, d.hidden_size = 7, 1, 4, 2, 8, 8
    h = ctypes.c_void_p()
    assert lib.rnn_create(ctypes.byref(d), ctypes.byref(h)) == R.RNN_BAD_PARAM
    d.mode = 0
    d.num_layers = 0
    assert lib.rnn_create(ctypes.byref(d), ctypes.byref(h)) == R.RNN_BAD_PARAM
    d.num_layers = 1
    d.gate_order[0], d.gate_order[1], d.gate_order[2], d.gate_order[3] = 0, 0, 1, 2
    assert lib.rnn_create(ctypes.byref(d), ctypes.byref(h)) == R.RNN_BAD_PARAM


# ---------------------------------------------------------------------------
# the header and the binding agree (a drift here is a silent ABI mismatch)
# ---------------------------------------------------------------------------
def _header_text():
    txt = ""
    for h in ("rnn.h", "rnn_debug.h"):
        txt += open(os.path.join(ROOT, "include", h)).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return re.sub(r"//[^\n]*", "", txt)


def test_binding_argument_counts_match_header():
    import bwd_persistent_cta_gb300 as R
    protos = re.findall(r"\b(rnn_[a-z_]+)\s*\(([^()]*)\)\s*;", _header_text())
    assert len(protos) >= 20
    for name, args in protos:
        args = args.strip()
        n = 0 if args in ("", "void") else args.count(",") + 1
        assert name in R._SIGS, name
        assert len(R._SIGS[name][1]) == n, (name, n, len(R._SIGS[name][1]))


def test_descriptor_struct_matches_header():
    import bwd_persistent_cta_gb300 as R
    body = re.search(r"typedef struct\s*\{(.*?)\}\s*rnn_desc_t\s*;", _header_text(), flags=re.S).group(1)
    fields = re.findall(r"\bint\s+([a-z_]+)\s*(?:\[(\d+)\])?\s*;", body)
    assert [f for f, _ in fields] == [f for f, _ in R.rnn_desc_t._fields_]
    assert ctypes.sizeof(R.rnn_desc_t) == 4 * sum(int(n) if n else 1 for _, n in fields)
    for (name, n), (_, ct) in zip(fields, R.rnn_desc_t._fields_):
        assert ctypes.sizeof(ct) == 4 * (int(n) if n else 1), name


def test_enum_values_match_header():
    import bwd_persistent_cta_gb300 as R
    vals = dict(re.findall(r"\b(RNN_[A-Z0-9_]+)\s*=\s*(\d+)", _header_text()))
    assert {"RNN_OK", "RNN_BF16", "RNN_GRU", "RNN_ALGO_PERSIST_SIMT"} <= set(vals)
    for name, v in vals.items():
        assert getattr(R, name) == int(v), name


# ---------------------------------------------------------------------------
# descriptor validation: every rule of rnn_create is checked on the host
# before any device call, so each answer is the same with or without a GPU
# ---------------------------------------------------------------------------
def _desc(R, **kw):
    d = R.rnn_desc_t()
    base = dict(mode=R.RNN_LSTM, reset_after=0, bidirectional=0, num_layers=1, seq_len=4, batch=2, input_size=8,
                hidden_size=8, dtype=R.RNN_BF16, batch_first=0, algo=R.RNN_ALGO_AUTO)
    base.update(kw)
    order = base.pop("gate_order", (0, 0, 0, 0))
    for k, v in base.items():
        setattr(d, k, v)
    for k in range(4):
        d.gate_order[k] = order[k]
    return d


BAD = [
    dict(mode=4), dict(mode=-1), dict(dtype=2), dict(num_layers=0), dict(num_layers=9), dict(seq_len=0),
    dict(batch=0), dict(input_size=0), dict(hidden_size=-8), dict(bidirectional=2), dict(reset_after=2),
    dict(batch_first=-1), dict(algo=3), dict(algo=-1),
    dict(gate_order=(1, 0, 3, 3)), dict(gate_order=(0, 1, 2, 4)),
    dict(mode=1, gate_order=(0, 1, 3, 0)), dict(mode=1, gate_order=(2, 2, 1, 0)),
    dict(mode=2, gate_order=(1, 0, 0, 0)),
    dict(seq_len=1 << 16, batch=1 << 15),          # T * B = 2^31 rows
]
UNSUPPORTED = [dict(hidden_size=12), dict(input_size=4), dict(dtype=0, hidden_size=6), dict(dtype=0, input_size=2)]
VALID = [dict(), dict(mode=1, gate_order=(2, 0, 1, 0)), dict(gate_order=(3, 2, 1, 0)), dict(dtype=0, hidden_size=4,
         input_size=4), dict(mode=3, num_layers=8, bidirectional=1, batch_first=1, algo=2),
         dict(seq_len=1 << 15, batch=1 << 15)]


@pytest.mark.parametrize("kw", BAD, ids=[str(k) for k in BAD])
def test_invalid_descriptor_is_bad_param(lib, kw):
    import bwd_persistent_cta_gb300 as R
    h = ctypes.c_void_p(16)
    assert lib.rnn_create(ctypes.byref(_desc(R, **kw)), ctypes.byref(h)) == R.RNN_BAD_PARAM
    assert not h.value
    # the allocation-free forward validates the same descriptor first
    assert lib.rnn_forward_noalloc(ctypes.byref(_desc(R, **kw)), 16, None, None, 16, 16, None, None, 0,
                                   None) == R.RNN_BAD_PARAM


@pytest.mark.parametrize("kw", UNSUPPORTED, ids=[str(k) for k in UNSUPPORTED])
def test_unaligned_rows_not_supported(lib, kw):
    import bwd_persistent_cta_gb300 as R
    h = ctypes.c_void_p(16)
    assert lib.rnn_create(ctypes.byref(_desc(R, **kw)), ctypes.byref(h)) == R.RNN_NOT_SUPPORTED
    assert not h.value


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-device path")
@pytest.mark.parametrize("kw", VALID, ids=[str(k) for k in VALID])
def test_valid_descriptor_reaches_the_device_query(lib, kw):
    import bwd_persistent_cta_gb300 as R
    h = ctypes.c_void_p(16)
    assert lib.rnn_create(ctypes.byref(_desc(R, **kw)), ctypes.byref(h)) in (R.RNN_CUDA_ERROR, R.RNN_NOT_SUPPORTED)
    assert not h.value


def test_null_arguments(lib):
    import bwd_persistent_cta_gb300 as R
    h = ctypes.c_void_p()
    assert lib.rnn_create(None, ctypes.byref(h)) == R.RNN_BAD_PARAM
    assert lib.rnn_create(ctypes.byref(_desc(R)), None) == R.RNN_BAD_PARAM
    assert lib.rnn_forward_noalloc(None, 16, None, None, 16, 16, None, None, 0, None) == R.RNN_BAD_PARAM
    assert lib.rnn_destroy(None) == R.RNN_OK
    bad = R.RNN_BAD_PARAM
    assert lib.rnn_get_sizes(None, None, None, None) == bad
    assert lib.rnn_forward(None, *([None] * 10)) == bad
    assert lib.rnn_backward_data(None, *([None] * 13)) == bad
    assert lib.rnn_backward_weights(None, *([None] * 7)) == bad
    assert lib.rnn_sync_status(None, None) == bad
    assert lib.rnn_set_timeout_ns(None, 1) == bad
    assert lib.rnn_set_seq_lengths(None, None) == bad
    assert lib.rnn_set_cell_clip(None, 1, -1.0, 1.0) == bad
    assert lib.rnn_set_recomputation(None, 0) == bad
    assert lib.rnn_set_interleaved_dw(None, 1) == bad
    assert lib.rnn_set_timing(None, 1) == bad
    assert lib.rnn_get_timing(None, None, None) == bad
    assert lib.rnn_debug_skip_arrival(None, 0) == bad
    # plan overrides: out-of-range values are rejected and change nothing
    for args in ((17, 0, 0, 0, 0, 0, 0, 0), (-1, 0, 0, 0, 0, 0, 0, 0), (0, 0, 3, 0, 0, 0, 0, 0),
                 (0, 0, 0, 8, 0, 0, 0, 0), (0, 0, 0, 0, 64, 0, 0, 0), (0, 0, 0, 0, 0, 17, 0, 0),
                 (0, 0, 0, 0, 0, 0, 64, 0), (0, 0, 0, 0, 128, 0, 256, 0), (0, 0, 0, 0, 0, 0, 0, 2)):
        assert lib.rnn_debug_set_plan_overrides(*args) == bad, args
    assert lib.rnn_debug_set_plan_overrides(0, 0, 0, 0, 0, 0, 0, 0) == 0
    for q in ("rnn_interleaved_dw_active", "rnn_launch_count", "rnn_selected_algo", "rnn_selected_fwd_algo"):
        assert getattr(lib, q)(None) == 0, q


C_CALLER = r"""
#include "rnn.h"
#include "rnn_debug.h"
#include <stdio.h>
int main(void) {
  rnn_desc_t d = {0};
  rnn_handle_t h = 0;
  rnn_status_t rc;
  d.mode = RNN_GRU; d.reset_after = 1; d.num_layers = 1; d.seq_len = 4; d.batch = 2;
  d.input_size = 8; d.hidden_size = 8; d.dtype = RNN_BF16; d.algo = RNN_ALGO_AUTO;
  d.gate_order[0] = 2; d.gate_order[1] = 2;            /* not a permutation */
  rc = rnn_create(&d, &h);
  printf("%d %d %s\n", (int)rc, h == 0, rnn_status_string(rc));
  return rc == RNN_BAD_PARAM && h == 0 && rnn_destroy(0) == RNN_OK ? 0 : 1;
}
"""


def test_headers_are_plain_c_and_the_library_links_from_c(lib, tmp_path):
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    import bwd_persistent_cta_gb300 as R
    src, exe = tmp_path / "caller.c", tmp_path / "caller"
    src.write_text(C_CALLER)
    libdir = os.path.dirname(R.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", libdir, "-lrnn", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("1 1 RNN_BAD_PARAM")


@pytest.mark.parametrize("kw", [dict(mode="lstm2"), dict(dtype="fp16"), dict(dtype="bfloat16"),
                                dict(gate_order=(0, 1, 2, 3, 0))])
def test_binding_rejects_bad_arguments_before_any_device_call(kw):
    import bwd_persistent_cta_gb300 as R
    args = dict(mode="lstm", input_size=8, hidden_size=8, seq_len=4, batch=2)
    args.update(kw)
    with pytest.raises(ValueError):
        R.RNN(**args)


def _unbound_rnn(mode="lstm", bidirectional=True, batch_first=False, dtype="bf16"):
    """An RNN wrapper without a handle, on the CPU device: enough to exercise
    its argument checks, which run before any library call."""
    import torch
    import bwd_persistent_cta_gb300 as R
    r = object.__new__(R.RNN)
    r.torch = torch
    r.device = torch.device("cpu")
    r.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
    d = R.rnn_desc_t()
    d.mode = R.RNN_LSTM if mode == "lstm" else R.RNN_GRU
    d.num_layers, d.seq_len, d.batch, d.input_size, d.hidden_size = 2, 5, 3, 8, 16
    d.bidirectional, d.batch_first = int(bidirectional), int(batch_first)
    r.desc = d
    r.weight_count = 1000
    r.handle = None
    return r


@pytest.mark.parametrize("batch_first", [False, True])
def test_wrapper_checks_tensors_before_calling_the_library(batch_first):
    import torch
    r = _unbound_rnn(batch_first=batch_first)
    bf = torch.bfloat16
    seq = (lambda F: (3, 5, F)) if batch_first else (lambda F: (5, 3, F))
    x, y, w = torch.zeros(seq(8), dtype=bf), torch.zeros(seq(32), dtype=bf), torch.zeros(1000, dtype=bf)
    S = torch.zeros(4, 3, 16, dtype=bf)
    r._check_forward(x, w, S, S, y, S, S)                       # all consistent
    r._check_forward(x, w, None, None, y, None, None)
    r._check_backward_data(y, w, S, None, x, S, S, None)
    r._check_backward_weights(x, torch.zeros(1000, dtype=torch.float32))
    bad = [
        lambda: r._check_forward(torch.zeros(seq(9), dtype=bf), w, None, None, y, None, None),    # input size
        lambda: r._check_forward(x.transpose(0, 1), w, None, None, y, None, None),                # layout
        lambda: r._check_forward(x, torch.zeros(999, dtype=bf), None, None, y, None, None),       # weights
        lambda: r._check_forward(x, w, torch.zeros(2, 3, 16, dtype=bf), None, y, None, None),     # state layers
        lambda: r._check_forward(x, w, None, None, torch.zeros(seq(16), dtype=bf), None, None),   # y width (D*H)
        lambda: r._check_forward(x.float(), w, None, None, y, None, None),                        # dtype
        lambda: r._check_forward(torch.zeros(seq(16), dtype=bf)[..., ::2], w, None, None, y, None, None),
        lambda: r._check_backward_data(y, w, None, None, torch.zeros(seq(4), dtype=bf), None, None, None),
        lambda: r._check_backward_data(y, w, None, torch.zeros(4, 2, 16, dtype=bf), x, None, None, None),
        lambda: r._check_backward_weights(x, torch.zeros(1000, dtype=bf)),                        # dw is fp32
        lambda: r._check_backward_weights(x, torch.zeros(1001, dtype=torch.float32)),
        lambda: r._check_forward([0.0], w, None, None, y, None, None),                            # not a tensor
    ]
    for f in bad:
        with pytest.raises((ValueError, TypeError)):
            f()


def test_wrapper_checks_alignment_and_device():
    import torch
    r = _unbound_rnn(bidirectional=False)
    bf = torch.bfloat16
    x = torch.zeros(5 * 3 * 8 + 1, dtype=bf)[1:].view(5, 3, 8)           # 2-byte offset
    with pytest.raises(ValueError, match="16-byte"):
        r._want(x, "x", (5, 3, 8))
    with pytest.raises(ValueError, match="handle is on"):
        r._want(torch.zeros(5, 3, 8, dtype=bf, device="meta"), "x", (5, 3, 8))


def test_wrapper_marshals_the_calls(monkeypatch):
    """forward / backward_data / backward_weights of the wrapper, with the C
    entry points replaced by recorders: outputs are allocated with the right
    shapes, the arguments reach the library in its order, inference passes no
    reserve, and a library error becomes RnnError."""
    import torch
    import bwd_persistent_cta_gb300 as R
    r = _unbound_rnn(bidirectional=True)
    r.handle = 1234
    try:
        r.workspace = torch.zeros(256, dtype=torch.uint8)
        r.reserve = torch.zeros(256, dtype=torch.uint8)
        calls = []

        def rec(name, rc=R.RNN_OK):
            def f(*args):
                calls.append((name, args))
                return rc
            return f

        monkeypatch.setattr(R, "_stream", lambda stream=None, device=None: 77)
        monkeypatch.setattr(R, "rnn_forward", rec("fwd"))
        monkeypatch.setattr(R, "rnn_backward_data", rec("bwd"))
        monkeypatch.setattr(R, "rnn_backward_weights", rec("wu"))
        bf = torch.bfloat16
        x, w = torch.zeros(5, 3, 8, dtype=bf), torch.zeros(1000, dtype=bf)
        hx = torch.zeros(4, 3, 16, dtype=bf)
        y, hy, cy = r.forward(x, w, hx, None)
        assert y.shape == (5, 3, 32) and hy.shape == cy.shape == (4, 3, 16)
        name, a = calls[-1]
        assert a[0] == 1234 and a[1] == x.data_ptr() and a[2] == hx.data_ptr() and a[3] is None
        assert a[4] == w.data_ptr() and a[5] == y.data_ptr() and a[6] == hy.data_ptr() and a[7] == cy.data_ptr()
        assert a[8] == r.workspace.data_ptr() and a[9] == r.reserve.data_ptr() and a[10] == 77
        r.forward(x, w, train=False)
        assert calls[-1][1][9] is None                                   # inference: no reserve
        dy = torch.zeros(5, 3, 32, dtype=bf)
        dx, dhx, dcx = r.backward_data(dy, w)
        assert dx.shape == (5, 3, 8) and dhx.shape == dcx.shape == (4, 3, 16)
        a = calls[-1][1]
        assert a[2] == dy.data_ptr() and a[5] == w.data_ptr() and a[8] == dx.data_ptr() and a[9] == dhx.data_ptr()
        assert a[10] == dcx.data_ptr() and a[12] == r.reserve.data_ptr()
        dw = r.backward_weights(x)
        assert dw.dtype == torch.float32 and dw.numel() == 1000
        a = calls[-1][1]
        assert a[1] == x.data_ptr() and a[5] == r.reserve.data_ptr() and a[6] == dw.data_ptr()
        with pytest.raises(ValueError):
            r.forward(x, torch.zeros(10, dtype=bf))
        monkeypatch.setattr(R, "rnn_forward", rec("fwd", R.RNN_NOT_SUPPORTED))
        with pytest.raises(R.RnnError):
            r.forward(x, w)
    finally:
        r.handle = None      # a fake handle must never reach rnn_destroy
