"""Runs the exchange-checking build of the library (compiled with
-DRNN_CHECKS into _build_checks/) on shapes that exchange across CTAs and
clusters, against the fp64 oracle; prints one line per case.  A step that
read an exchanged slice before its producers wrote it ends the call with
RNN_INTERNAL, which the binding raises.  Run by tests/test_checks_gpu.py in a
process of its own (the binding loads one library per process)."""
import dataclasses
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from bwd_persistent_cta_gb300 import build as B  # noqa: E402

LIB = B.build(extra_flags=["-DRNN_CHECKS"], lib_path=os.path.join(B.HERE, "_build_checks", "librnn_checks.so"),
              build_dir=os.path.join(B.HERE, "_build_checks"))
import bwd_persistent_cta_gb300 as R  # noqa: E402

R.LIB_PATH = LIB
import synth  # noqa: E402
from tests import harness as Hn  # noqa: E402


def wl_(name, mode, ra, L, bidir, T, Bt, I, H, seed):
    return synth.Workload(name, mode, ra, L, bidir, T, Bt, I, H, "bf16", seed, state_std=0.5)


CASES = [
    # name, workload, overrides, lengths
    ("lstm K split fwd 4 / bwd 8", wl_("c_lstm", "lstm", False, 1, False, 8, 32, 64, 1024, 970), {}, None),
    ("gru resetAfter 2 layers bidirectional", wl_("c_gru", "gru", True, 2, True, 6, 64, 64, 512, 971), {}, None),
    ("gru reset-before", wl_("c_grb", "gru", False, 1, True, 6, 16, 32, 256, 972), {}, None),
    ("lstm batch parts with lengths", wl_("c_len", "lstm", False, 2, True, 7, 16, 32, 128, 973),
     {"nb_fwd": 2, "nb_bwd": 2}, np.array([7, 0, 1, 5, 7, 3, 6, 7, 2, 7, 6, 4, 7, 1, 7, 5])),
    ("lstm backward K split through global memory", wl_("c_gk", "lstm", False, 1, True, 6, 16, 32, 256, 974),
     {"bwd_global_ks": 1}, None),
]

for name, wl, ov, lengths in CASES:
    R.rnn_debug_set_plan_overrides(**ov)
    inp = synth.make_inputs(wl)
    if lengths is not None:
        inp = dataclasses.replace(inp, lengths=lengths)
    gpu = Hn.run_gpu(inp)          # raises on RNN_INTERNAL (a slice read before it was written)
    R.rnn_debug_set_plan_overrides()
    Hn.compare(gpu, Hn.run_oracle(inp), wl)
    print(f"checked: {name}: algo {gpu['algo']}, forward {gpu['fwd_algo']}", flush=True)
# the checker itself: an initial state holding the poison pattern (bf16 bits
# 0xFFFF, a NaN) in one batch row is what a slice read before its write looks
# like to the first step, which must report it
import torch  # noqa: E402

wl = wl_("c_neg", "lstm", False, 1, False, 4, 16, 32, 128, 975)
inp = synth.make_inputs(wl)
rnn = R.RNN("lstm", 32, 128, 4, 16, algo=1)
try:
    w = Hn.to_dev(synth.flatten_params(wl, inp.params), wl)
    x = Hn.to_dev(inp.x, wl)
    hx, cx = Hn.to_dev(inp.h0, wl), Hn.to_dev(inp.c0, wl)
    hx.view(torch.int16)[0, 3, 5] = -1
    rnn.forward(x, w, hx, cx, train=False)
    rc = R.rnn_sync_status(rnn.handle, torch.cuda.current_stream().cuda_stream)
    assert rc == R.RNN_INTERNAL, R.rnn_status_string(rc)
    hx.view(torch.int16)[0, 3, 5] = 0
    rnn.forward(x, w, hx, cx, train=False)
    rnn.sync()
finally:
    rnn.close()
print("checker fired on the poison pattern")
print("all checked")
