"""fcm_run_unfused_static: the layer-by-layer evaluation that allocates nothing.

Some callers cannot call cudaMalloc while they run (a serving loop whose device memory is
budgeted up front, a thread that must not take the allocator's locks or wait on its implicit
synchronisation).  For them the library keeps the intermediate in a fixed device array of
16 MiB instead of a buffer the handle allocates.  These tests call that entry point through
the C ABI and compare it with the allocating path (fcm_run, FCM_MODE_UNFUSED), twice in a row,
since consecutive calls share the array.  This file is collected last on purpose.
"""
import numpy as np
import pytest

import pointwise_conv_cnn_gb300 as fcm
from pointwise_conv_cnn_gb300 import workloads as wk

from helpers import assert_parity, empty, make_module, oracle_fused, parity_error, to_device, to_host

pytestmark = pytest.mark.gpu

MODE_UNFUSED = 3


def _run_both(wl, kernel):
    import torch
    case = wk.make_case(wl)
    mod = make_module(case, kernel)
    x = to_device(case.x, wl.dtype)
    shape = wl.shapes()["y"]
    s = torch.cuda.current_stream().cuda_stream
    ref = empty(shape, wl.dtype, fill=float("nan"))
    fcm.fcm_run(mod.handle, MODE_UNFUSED, x.data_ptr(), ref.data_ptr(), s)
    outs = []
    for _ in range(2):   # two calls in a row reuse the same static array
        y = empty(shape, wl.dtype, fill=float("nan"))
        fcm.fcm_run_unfused_static(mod.handle, x.data_ptr(), y.data_ptr(), s)
        outs.append(y)
    torch.cuda.synchronize()
    mod.check()
    return case, to_host(ref, wl.dtype), [to_host(y, wl.dtype) for y in outs]


@pytest.mark.parametrize("name,kernel", [("mobilenet_dwpw_f16", "auto"), ("stride2_dwpw_bf16", "auto"),
                                         ("mobilenet_dwpw_f16", "simt"), ("tiny_dwpw_f32", "auto"),
                                         ("mobilenet_dwpw_i8", "auto")])
def test_static_scratch_matches_allocating_path(cuda, name, kernel):
    wl = wk.BY_NAME[name]
    wl = wl.with_(n=min(wl.n, 2))
    case, ref, outs = _run_both(wl, kernel)
    bar = {"f32": 1e-4 * np.sqrt(wl.cm), "i8": 0.0}.get(wl.dtype, 2e-2)
    f_ref = wk.to_f64(ref, wl.dtype)
    for got in outs:
        err = float(np.abs(wk.to_f64(got, wl.dtype) - f_ref).max())
        if wl.dtype not in ("f32", "i8"):
            err /= max(float(np.abs(f_ref).max()), 1e-6)
        assert err <= bar, (name, kernel, err)
    # and both paths against the oracle
    assert_parity(outs[1], oracle_fused(case), wl.dtype, wl.cm)


def test_static_scratch_rejects_large_intermediate(cuda):
    wl = wk.BY_NAME["mobilenet_dwpw_f16"]          # 64 x 56 x 56 x 128 x 2 B = 51 MB > 16 MiB
    case = wk.make_case(wl.with_(n=1))
    mod = fcm.FusedConvModule(fcm.desc_from_workload(wl), case.w1, case.wp, case.s1, case.b1,
                              case.s2, case.b2)
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_run_unfused_static(mod.handle, 16, 16, 0)
    assert e.value.status == 2 and "static scratch" in str(e.value)
