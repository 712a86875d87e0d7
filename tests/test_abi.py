"""The C ABI library loads, exports every symbol include/fcm.h declares, and rejects bad
arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import pointwise_conv_cnn_gb300 as fcm
from pointwise_conv_cnn_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "fcm.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fcm.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FCM_API\s+[\w\s\*]+?\b(fcm_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_symbols() == sorted(fcm.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_only_the_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fcm.LIB_PATH], capture_output=True,
                         text=True).stdout
    text_syms = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert text_syms == set(declared_symbols())


def test_desc_struct_matches_header():
    text = open(HEADER).read()
    body = re.search(r"typedef struct fcm_desc \{(.*?)\} fcm_desc;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = [n for decl in body.split(";") for n in re.findall(r"(\w+)\s*(?:,|$)", decl.replace("int", "", 1).strip())]
    assert [f for f, _ in fcm.FcmDesc._fields_] == names
    assert ctypes.sizeof(fcm.FcmDesc) == 16 * 4
    assert ctypes.sizeof(fcm.FcmPlanInfo) == 11 * 4 + 4 + 6 * 8 + 8   # tc_variant + tail padding


def good_desc(**kw):
    base = dict(n=2, h=8, w=8, c=16, k_out=16, ksize=3, stride=1, pad=1, dtype="f16")
    base.update(kw)
    return fcm.make_desc(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(n=0), 1), (dict(ksize=9), 2), (dict(stride=3), 2), (dict(pad=3), 1),
    (dict(c=12), 3), (dict(k_out=20, dtype="bf16"), 3), (dict(c=4, k_out=4, dtype="f32"), 0),
    (dict(c=6, k_out=4, dtype="f32"), 3), (dict(mid=32), 1), (dict(h=1, w=1, pad=0), 1),
])
def test_plan_desc_validation(lib, kw, status):
    d = good_desc(**kw)
    if status == 0:
        info = fcm.fcm_plan_desc(d)
        assert info["ho"] == 8
    else:
        with pytest.raises(fcm.FcmError) as e:
            fcm.fcm_plan_desc(d)
        assert e.value.status == status
        assert fcm.fcm_last_error()


def test_tensor_bytes(lib):
    d = good_desc(stride=2)
    assert fcm.fcm_tensor_bytes(d) == (2 * 8 * 8 * 16 * 2, 2 * 4 * 4 * 16 * 2, 2 * 4 * 4 * 16 * 2)


def test_null_handle_rejected(lib):
    assert lib.fcm_run(None, 0, None, None, None) == 1
    assert lib.fcm_check(None, None) == 1
    lib.fcm_destroy(None)  # ignored


def test_create_without_gpu_reports_no_device(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import numpy as np
    w = np.zeros(16 * 9, np.float16)
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_create(good_desc(), w.ctypes.data, w.ctypes.data, w.ctypes.data, w.ctypes.data,
                       w.ctypes.data, w.ctypes.data)
    assert e.value.status == 8


def test_product_path_never_touches_the_oracle():
    """The package (binding, build, workloads, CUDA sources) neither imports nor links the
    oracle, and a missing library raises instead of falling back to anything."""
    import subprocess
    import sys
    pkg = os.path.dirname(fcm.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text and "fcm_oracle" not in text, f
    code = ("import sys, pointwise_conv_cnn_gb300 as fcm, pointwise_conv_cnn_gb300.workloads; "
            "assert 'oracle' not in sys.modules; "
            "fcm._lib = None\n"
            "try:\n    fcm.load_library('/nonexistent/libfcm.so')\n"
            "except FileNotFoundError:\n    print('raised')\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         cwd=os.path.dirname(pkg))
    assert out.returncode == 0 and "raised" in out.stdout, out.stderr


def test_selftest_limit_checked_on_the_host(lib):
    """The wait self-test validates its limit before touching a device."""
    for bad in (0, 10_000_000_001):
        with pytest.raises(fcm.FcmError) as e:
            fcm.fcm_selftest_wait_timeout(bad)
        assert e.value.status == 1
