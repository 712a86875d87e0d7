"""Launch order on one stream (needs a GB300).

The tensor-core kernels let the next kernel on the stream start before they finish, and wait for
the previous kernel before they read their input (programmatic dependent launch).  A chain of
layers whose output feeds the next layer's input -- ping-ponging between two buffers, so that
each launch also overwrites the buffer the launch before it read -- must give exactly the same
bytes enqueued back to back as with the host waiting after every launch.
"""
import numpy as np
import pytest

from pointwise_conv_cnn_gb300 import workloads as wk

from helpers import empty, make_module, to_device, to_host

pytestmark = pytest.mark.gpu

# layers whose output has the input's shape (C == K, stride 1), on each tensor-core kernel
CHAIN = [
    (wk.Workload("chain_dw3_f16", 3, 30, 34, 64, 64, "dw", 3, 1, 1, "relu6", "relu6", "f16",
                 "normal"), "tc_roles"),
    (wk.Workload("chain_dw5_bf16", 3, 30, 34, 64, 64, "dw", 5, 1, 2, "relu", "none", "bf16",
                 "normal"), "tc_workers"),
    (wk.Workload("chain_dense3_f16", 2, 24, 40, 64, 64, "dense", 3, 1, 1, "relu", "relu6", "f16",
                 "normal", mid=64), "tc"),
    (wk.Workload("chain_pwdw_f16", 2, 24, 40, 64, 64, "pwdw", 3, 1, 1, "relu6", "relu6", "f16",
                 "normal", mid=64), "tc"),
    (wk.Workload("chain_dw3_i8", 3, 30, 34, 64, 64, "dw", 3, 1, 1, "relu", "none", "i8",
                 "int8"), "tc_roles"),
]
MODES = ["fused", "unfused", "fused", "fused", "unfused", "fused", "fused", "fused"]


@pytest.mark.parametrize("wl,kernel", CHAIN, ids=lambda v: v.name if hasattr(v, "name") else v)
def test_chain_back_to_back_equals_synchronised(cuda, wl, kernel):
    import torch
    case = wk.make_case(wl)
    mod = make_module(case, kernel)
    shape = wl.shapes()["y"]
    assert tuple(shape) == tuple(wl.shapes()["x"])

    def chain(sync: bool) -> list[np.ndarray]:
        bufs = [to_device(case.x, wl.dtype), empty(shape, wl.dtype, fill=float("nan"))]
        outs = []
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            for i, mode in enumerate(MODES):
                mod.run(bufs[i % 2], bufs[(i + 1) % 2], mode, stream=stream)
                if sync:
                    stream.synchronize()
                    outs.append(to_host(bufs[(i + 1) % 2], wl.dtype))
            stream.synchronize()
        mod.check(stream)
        if not sync:
            outs.append(to_host(bufs[len(MODES) % 2], wl.dtype))
        return outs

    want = chain(sync=True)
    got = chain(sync=False)
    assert np.array_equal(got[-1], want[-1])
    # the chain did not settle into a fixed point early (every step changed the values)
    assert not np.array_equal(want[-1], want[-2])
    mod.close()
