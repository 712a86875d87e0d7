"""fcm_run_host_async (needs a GB300): calls enqueued back to back on one handle overlap their
copies but give exactly what the synchronous fcm_run_host gives, including when one call's
output buffer is the next call's input (the copies in must wait for the copies out), when the
mode changes between calls, and when the batch is not split (the layer-by-layer mode)."""
import numpy as np
import pytest

from pointwise_conv_cnn_gb300 import workloads as wk

from helpers import empty, make_module, to_device, to_host

pytestmark = pytest.mark.gpu


def _pinned(arr, dtype):
    return to_device(arr, dtype, "cpu").pin_memory()


@pytest.mark.parametrize("name,n", [("mobilenet_dwpw_f16", 5), ("mobilenet_dwpw_i8", 8),
                                    ("b2b_dense3x3_f16", 3)])
def test_async_calls_equal_sync_calls(cuda, name, n):
    import torch
    base = wk.BY_NAME[name]
    wl = base.with_(n=n, h=min(base.h, 20), w=min(base.w, 20))
    assert wl.shapes()["x"] == wl.shapes()["y"]          # so that outputs can be inputs
    mod = make_module(wk.make_case(wl))
    xs = [_pinned(wk.make_case(wl, seed=40 + i).x, wl.dtype) for i in range(3)]
    ys = [empty(wl.shapes()["y"], wl.dtype, "cpu", fill=float("nan")).pin_memory()
          for _ in range(6)]
    # the same sequence, synchronous: three independent calls, a chain through host memory,
    # and the layer-by-layer mode (not split) in between
    plan = [(xs[0], 0, "fused"), (xs[1], 1, "fused"), (None, 2, "fused"),   # input = ys[1]
            (xs[2], 3, "unfused"), (None, 4, "fused"), (xs[0], 5, "fused")]  # input = ys[3]
    want = []
    for inp, o, mode in plan:
        src = inp if inp is not None else ys[o - 1]
        out = empty(wl.shapes()["y"], wl.dtype, "cpu", fill=float("nan")).pin_memory()
        mod.run_host(src, out, mode)
        want.append(to_host(out, wl.dtype))
        ys[o].copy_(out)
    for y in ys:
        y.fill_(float("nan") if wl.dtype != "i8" else -77)
    stream = torch.cuda.Stream()
    for inp, o, mode in plan:
        src = inp if inp is not None else ys[o - 1]
        mod.run_host_async(src, ys[o], mode, stream=stream)
    stream.synchronize()
    for o, w in enumerate(want):
        assert np.array_equal(to_host(ys[o], wl.dtype), w), (name, o)
    # a synchronous call between asynchronous ones (the batch split differently), then an
    # asynchronous call reading the synchronous call's output
    z1 = empty(wl.shapes()["y"], wl.dtype, "cpu", fill=float("nan")).pin_memory()
    z2 = empty(wl.shapes()["y"], wl.dtype, "cpu", fill=float("nan")).pin_memory()
    mod.run_host_async(xs[1], ys[0], "fused", stream=stream)
    mod.run_host(xs[0], z1, "fused", stream=stream)
    mod.run_host_async(z1, z2, "fused", stream=stream)
    stream.synchronize()
    assert np.array_equal(to_host(ys[0], wl.dtype), want[1])
    assert np.array_equal(to_host(z1, wl.dtype), want[0])
    ref = empty(wl.shapes()["y"], wl.dtype, "cpu", fill=float("nan")).pin_memory()
    mod.run_host(z1, ref, "fused")
    assert np.array_equal(to_host(z2, wl.dtype), to_host(ref, wl.dtype))
    mod.check(stream)
    mod.close()
