"""fcm_run_unfused_static: the layer-by-layer evaluation that allocates nothing.

Some callers cannot call cudaMalloc while they run (a serving loop whose device memory is
budgeted up front, a thread that must not take the allocator's locks or wait on its implicit
synchronisation).  For them the library keeps the intermediate in a fixed device array of
16 MiB instead of a buffer the handle allocates.  These tests call that entry point through
the C ABI and compare it bit for bit with the allocating path (fcm_run, FCM_MODE_UNFUSED) on
consecutive calls with different inputs and handles, since all calls share the array.  This
file is collected last on purpose.
"""
import numpy as np
import pytest

import pointwise_conv_cnn_gb300 as fcm
from pointwise_conv_cnn_gb300 import workloads as wk

from helpers import assert_parity, empty, make_module, oracle_fused, to_device, to_host

pytestmark = pytest.mark.gpu

MODE_UNFUSED = 3


def _unfused_pair(mod, wl, x, s):
    """The allocating layer-by-layer path and the static-scratch one on the same input."""
    shape = wl.shapes()["y"]
    ref = empty(shape, wl.dtype, fill=float("nan"))
    fcm.fcm_run(mod.handle, MODE_UNFUSED, x.data_ptr(), ref.data_ptr(), s)
    y = empty(shape, wl.dtype, fill=float("nan"))
    fcm.fcm_run_unfused_static(mod.handle, x.data_ptr(), y.data_ptr(), s)
    return ref, y


@pytest.mark.parametrize("name,kernel", [("mobilenet_dwpw_f16", "auto"), ("stride2_dwpw_bf16", "auto"),
                                         ("mobilenet_dwpw_f16", "simt"), ("tiny_dwpw_f32", "auto"),
                                         ("mobilenet_dwpw_i8", "auto")])
def test_static_scratch_matches_allocating_path(cuda, name, kernel):
    """Both paths run the same kernels, so their outputs must agree bit for bit.  Consecutive
    calls share the array: the second call takes a different input (a call that left part of
    the array unwritten would read the first call's intermediate there), and a third goes
    through another handle of a different shape."""
    import torch
    wl = wk.BY_NAME[name]
    wl = wl.with_(n=min(wl.n, 2))
    s = torch.cuda.current_stream().cuda_stream
    mod = make_module(wk.make_case(wl), kernel)
    pairs = []
    for seed in (11, 12):
        x = to_device(wk.make_case(wl, seed=seed).x, wl.dtype)
        pairs.append(_unfused_pair(mod, wl, x, s) + (x,))
    wl2 = wl.with_(n=1, h=wl.h // 2 + 3, w=wl.w // 2 + 1)
    case2 = wk.make_case(wl2, seed=13)
    mod2 = make_module(case2, kernel)
    x2 = to_device(case2.x, wl2.dtype)
    ref2, y2 = _unfused_pair(mod2, wl2, x2, s)
    torch.cuda.synchronize()
    mod.check()
    mod2.check()
    for ref, y, _ in pairs:
        assert np.array_equal(to_host(ref, wl.dtype), to_host(y, wl.dtype)), (name, kernel)
    assert not np.array_equal(to_host(pairs[0][1], wl.dtype), to_host(pairs[1][1], wl.dtype))
    assert np.array_equal(to_host(ref2, wl2.dtype), to_host(y2, wl2.dtype)), (name, kernel, "2nd handle")
    # and against the oracle
    assert_parity(to_host(y2, wl2.dtype), oracle_fused(case2), wl2.dtype, wl2.cm)


def test_static_scratch_rejects_large_intermediate(cuda):
    wl = wk.BY_NAME["mobilenet_dwpw_f16"]          # 64 x 56 x 56 x 128 x 2 B = 51 MB > 16 MiB
    case = wk.make_case(wl.with_(n=1))
    mod = fcm.FusedConvModule(fcm.desc_from_workload(wl), case.w1, case.wp, case.s1, case.b1,
                              case.s2, case.b2)
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_run_unfused_static(mod.handle, 16, 16, 0)
    assert e.value.status == 2 and "static scratch" in str(e.value)
