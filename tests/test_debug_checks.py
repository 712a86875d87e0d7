"""The debug build: the same library with the kernels' index checks compiled in
(FCM_DEBUG_CHECKS).  A failed check never traps; it records itself in the handle's error word,
which fcm_check reports as FCM_ERR_DEVICE_FAULT with the check's id and the offending index.

The CPU test builds it (nvcc cross-compiles); the GPU test runs the tensor-core modules through
it, in every mode, on shapes with ragged tiles, and requires no check to fire and the results to
equal the oracle's bit for bit."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_compiles():
    from pointwise_conv_cnn_gb300 import build
    lib = build.build(debug=True)
    assert os.path.exists(lib) and lib.endswith("libfcm_debug.so")


_RUN = r'''
import sys
sys.path.insert(0, %(root)r); sys.path.insert(0, %(root)r + "/tests")
import numpy as np
import pointwise_conv_cnn_gb300 as fcm
from pointwise_conv_cnn_gb300 import workloads as wk
from helpers import assert_bitexact, oracle_conv1, oracle_fused, run_case, make_module
assert fcm.load_library()._name.endswith("libfcm_debug.so")
cases = [
    ("mobilenet_dwpw_f16", dict(n=2, h=23, w=37), "tc_roles"),
    ("wide5x5_dwpw_bf16", dict(n=2, h=13, w=21), "tc_workers"),
    ("stride2_dwpw_bf16", dict(n=1, h=31, w=45), "tc_workers"),
    ("mobilenet_dwpw_i8", dict(n=2, h=19, w=29), "tc_roles"),
    ("b2b_dense3x3_f16", dict(n=1, h=13, w=30), "tc"),
    ("pwdw_i8", dict(n=1, h=11, w=17), "tc"),
]
for name, shape, kernel in cases:
    wl = wk.BY_NAME[name].with_(**shape)
    if wl.dtype == "i8":
        case = wk.make_case(wl)
    else:
        case = wk.make_case(wl, kind="integer" if wk.integer_safe(wl) else "integer1")
    mod = make_module(case, kernel)
    ref = oracle_fused(case)
    for mode in ("fused", "unfused"):
        got, _ = run_case(case, mode, module=mod)   # run_case calls fcm_check: raises on a check
        assert_bitexact(got, ref, wl.dtype)
    got, _ = run_case(case, "conv1", module=mod)
    assert_bitexact(got, oracle_conv1(case), wl.dtype)
    print("ok", name, kernel)
'''


@pytest.mark.gpu
def test_debug_checks_stay_quiet_on_parity_cases(cuda):
    from pointwise_conv_cnn_gb300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, FCM_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", _RUN % {"root": ROOT}], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("ok ") == 6, r.stdout
