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
