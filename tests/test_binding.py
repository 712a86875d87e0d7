"""The Python binding's own checks (CPU only): the byte counts each fcm_run mode reads and
writes, and the refusal of tensors the library would read or write past."""
import numpy as np
import pytest

import pointwise_conv_cnn_gb300 as fcm
from pointwise_conv_cnn_gb300 import workloads as wk

torch = pytest.importorskip("torch")
TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "i8": torch.int8}
# (mode, input tensor, output tensor) as the layers' shapes name them
MODE_TENSORS = (("fused", "x", "y"), ("conv1", "x", "m"), ("pw", "m", "y"), ("unfused", "x", "y"))


@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_mode_bytes_match_the_layer_shapes(wl):
    need = fcm.mode_bytes(fcm.desc_from_workload(wl))
    sh = wl.shapes()
    for mode, a, b in MODE_TENSORS:
        got = need[fcm.MODES[mode]]
        assert got == (int(np.prod(sh[a])) * wl.esize, int(np.prod(sh[b])) * wl.esize), mode


@pytest.mark.parametrize("wl", [w.with_(n=2, h=min(w.h, 12), w=min(w.w, 12))
                                for w in wk.WORKLOADS], ids=lambda w: w.name)
def test_exact_tensors_pass_and_short_ones_are_refused(wl):
    need = fcm.mode_bytes(fcm.desc_from_workload(wl))
    sh = wl.shapes()
    for mode, a, b in MODE_TENSORS:
        m = fcm.MODES[mode]
        inp = torch.empty(sh[a], dtype=TDT[wl.dtype])
        out = torch.empty(sh[b], dtype=TDT[wl.dtype])
        fcm.check_run_buffers(need, m, inp, out, on_device=False)
        # one image fewer in either tensor: refused before any pointer reaches the library
        for short_in in (True, False):
            si = inp[:1].contiguous() if short_in else inp
            so = out if short_in else out[:1].contiguous()
            with pytest.raises(fcm.FcmError) as e:
                fcm.check_run_buffers(need, m, si, so, on_device=False)
            assert e.value.status == 1 and ("input" if short_in else "output") in str(e.value)


def test_device_contiguity_and_mode_are_checked():
    wl = wk.BY_NAME["tiny_dwpw_f32"]
    need = fcm.mode_bytes(fcm.desc_from_workload(wl))
    sh = wl.shapes()
    x, y = torch.empty(sh["x"]), torch.empty(sh["y"])
    with pytest.raises(fcm.FcmError, match="CUDA tensor"):
        fcm.check_run_buffers(need, 0, x, y, on_device=True)       # host tensors to fcm_run
    with pytest.raises(fcm.FcmError, match="contiguous"):
        xt = torch.empty(sh["x"][0], sh["x"][3], sh["x"][1], sh["x"][2]).permute(0, 2, 3, 1)
        fcm.check_run_buffers(need, 0, xt, y, on_device=False)     # an NCHW tensor viewed NHWC
    with pytest.raises(fcm.FcmError, match="mode"):
        fcm.check_run_buffers(need, 9, x, y, on_device=False)
    # a larger output (a slice of a bigger buffer's worth) is accepted: only too small is refused
    fcm.check_run_buffers(need, 0, x, torch.empty(2 * y.numel()), on_device=False)
