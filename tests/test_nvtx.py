"""The entry points mark their calls with NVTX ranges (visible on a profiler's timeline).  A tiny
NVTX tool (tests/nvtx/nvtx_recorder.c, injected through NVTX_INJECTION64_PATH) records the
ranges of calls that need no GPU: a run on a NULL handle still opens and closes its range."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_entry_points_open_and_close_nvtx_ranges(tmp_path):
    import pointwise_conv_cnn_gb300 as fcm
    fcm.load_library()
    so = tmp_path / "libnvtx_recorder.so"
    cuda_inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
    r = subprocess.run(["gcc", "-shared", "-fPIC", "-O2", "-I", cuda_inc, "-o", str(so),
                        os.path.join(HERE, "nvtx", "nvtx_recorder.c")], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip(f"cannot build the NVTX recorder: {r.stderr[:200]}")
    log = tmp_path / "ranges.log"
    code = ("import sys; sys.path.insert(0, %r); import pointwise_conv_cnn_gb300 as fcm; "
            "lib = fcm.load_library(); "
            "assert lib.fcm_run(None, 0, None, None, None) == 1; "
            "assert lib.fcm_check(None, None) == 1; "
            "assert lib.fcm_run_unfused_static(None, None, None, None) == 1" % ROOT)
    env = dict(os.environ, NVTX_INJECTION64_PATH=str(so), FCM_NVTX_LOG=str(log))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lines = log.read_text().split("\n")
    pushes = [l[5:] for l in lines if l.startswith("push ")]
    assert pushes == ["fcm_run", "fcm_check", "fcm_run_unfused_static"], lines
    assert sum(l == "pop" for l in lines) == 3
