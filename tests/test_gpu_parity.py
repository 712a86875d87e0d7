"""Parity of the CUDA kernels with the fp64 oracle, through the C ABI (needs a GB300).

Bars: bit-exact on integer-valued inputs (index, halo, stride and padding handling); fp32
max-abs error <= 1e-4*sqrt(C); fp16/bf16 max-norm relative error <= 2e-2.
"""
import numpy as np
import pytest

import pointwise_conv_cnn_gb300 as fcm
from pointwise_conv_cnn_gb300 import workloads as wk

from helpers import (assert_bitexact, assert_parity, empty, make_module, oracle_conv1,
                     oracle_fused, oracle_pw, parity_error, run_case, to_device, to_host)

pytestmark = pytest.mark.gpu

# the depthwise module's two tensor-core kernels: "tc_roles" (dedicated warp roles) and
# "tc_workers" (worker warps running the stencil and the epilogue); for the other modules both
# mean "tc"
KERNELS = ["simt", "tc_roles", "tc_workers"]


def reduced(wl: wk.Workload, n=2, hw=None) -> wk.Workload:
    """Smaller batch (and optionally spatial size) with the layer's own channels, filter,
    stride, padding, activations and dtype."""
    kw = {"n": n}
    if hw is not None:
        kw.update(h=hw, w=hw)
    return wl.with_(**kw)


def module_or_skip(case, kernel):
    if kernel == "tc_workers" and case.wl.conv1 != "dw":
        pytest.skip("only the depthwise module has a second tensor-core kernel")
    if case.wl.dtype == "i8" and kernel == "simt":
        # INT8 has no CUDA-core kernels: the request is refused, not served by another path
        with pytest.raises(fcm.FcmError) as e:
            make_module(case, kernel)
        assert e.value.status == 2
        pytest.skip("INT8 runs on the tensor-core kernels only")
    try:
        return make_module(case, kernel)
    except fcm.FcmError as e:
        if kernel in ("tc", "tc_roles", "tc_workers") and e.status == 2:
            pytest.skip(f"tensor-core kernels do not take this shape: {e}")
        raise


def integer_variant(wl: wk.Workload) -> tuple[wk.Workload, str]:
    """The integer kind that keeps the case exact end to end (+-1 values for wide dense
    layers)."""
    if wk.integer_safe(wl):
        return wl, "integer"
    if wk.integer_safe(wl, "integer1"):
        return wl, "integer1"
    raise AssertionError(wl)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_integer_bitexact_fused_and_unfused(cuda, wl, kernel):
    small, kind = integer_variant(reduced(wl, n=2, hw=min(wl.h, 30)))
    case = wk.make_case(small, kind=kind)
    mod = module_or_skip(case, kernel)
    ref = oracle_fused(case)
    for mode in ("fused", "unfused"):
        got, _ = run_case(case, mode, module=mod)
        assert_bitexact(got, ref, small.dtype)
    m_gpu, _ = run_case(case, "conv1", module=mod)
    assert_bitexact(m_gpu, oracle_conv1(case), small.dtype)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_integer_pow2_scales_bitexact(cuda, wl, kernel):
    """Integer inputs with a scale of 1/2, 1 or 2 per channel (exact in every format): a scale
    or bias read for the wrong channel changes the result, so this pins their indexing bit for
    bit in every mode.  Where the intermediate of the integer case exceeds the format's exact
    range (the dense 3x3 layer), the oracle rounds it to the storage format as the kernels do
    (its mirror mode); the fp32 sums stay exact either way."""
    if wl.dtype == "i8":
        pytest.skip("INT8 scales are arbitrary fp32 values already, replicated exactly")
    small = reduced(wl, n=2, hw=min(wl.h, 30))
    kind = next((k for k in ("integer_pow2", "integer1_pow2") if wk.integer_safe(small, k)), None)
    mid = "exact" if kind else small.dtype
    case = wk.make_case(small, seed=31, kind=kind or "integer1_pow2")
    assert len(set(np.asarray(case.s1).tolist())) == 3 and len(set(np.asarray(case.s2).tolist())) > 1
    mod = module_or_skip(case, kernel)
    ref = oracle_fused(case, mid=mid)
    for mode in ("fused", "unfused"):
        got, _ = run_case(case, mode, module=mod)
        assert_bitexact(got, ref, small.dtype)
    m_gpu, _ = run_case(case, "conv1", module=mod)
    m_ref = oracle_conv1(case)
    if mid == "exact":
        assert_bitexact(m_gpu, m_ref, small.dtype)


def storage_ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """The spacing of the storage format at |v| (its subnormal spacing at 0)."""
    mant, emin = {"f16": (10, -14), "bf16": (7, -126)}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return np.exp2(e - mant)


@pytest.mark.parametrize("kernel", ["tc_roles", "tc_workers"])
@pytest.mark.parametrize("wl", [w for w in wk.WORKLOADS if w.dtype in ("f16", "bf16")],
                         ids=lambda w: w.name)
def test_mirror_within_storage_ulps(cuda, wl, kernel):
    """The tensor-core result against the oracle's mirror mode, which rounds the intermediate
    to the storage format as the kernels do.  What remains is the kernels' fp32 sums (the
    depthwise or dense sum, the 1x1 GEMM's accumulator) against the oracle's fp64 ones, and one
    rounding of the output.  Bar, element by element: one storage ulp at the value, plus one
    storage ulp at the largest output magnitude -- the room for an intermediate that rounds to
    the other neighbour when its fp32 sum and its fp64 sum straddle a rounding boundary, which
    moves an output near zero by many of its own ulps but by far less than the largest
    output's ulp.  At least 99.9% of the outputs must be within one ulp of the mirror."""
    small = reduced(wl, n=2, hw=min(wl.h, 40))
    case = wk.make_case(small)
    mod = module_or_skip(case, kernel)
    got = wk.to_f64(run_case(case, "fused", module=mod)[0], small.dtype)
    ref = oracle_fused(case, mid=small.dtype)
    ref_s = wk.to_f64(wk.to_storage(ref, small.dtype), small.dtype)
    err = np.abs(got - ref_s)
    bar = storage_ulp(ref_s, small.dtype) + storage_ulp(np.abs(ref_s).max(), small.dtype)
    worst = np.unravel_index(np.argmax(err - bar), err.shape)
    assert np.all(err <= bar), (float(err[worst]), float(bar[worst]), float(ref[worst]))
    within1 = float(np.mean(err <= storage_ulp(ref_s, small.dtype)))
    assert within1 >= 0.999, within1


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_tolerance_reduced_batch(cuda, wl, kernel):
    small = reduced(wl, n=2)
    case = wk.make_case(small)
    mod = module_or_skip(case, kernel)
    ref = oracle_fused(case)
    got, _ = run_case(case, "fused", module=mod)
    e_f = assert_parity(got, ref, small.dtype, small.cm)
    got_u, _ = run_case(case, "unfused", module=mod)
    assert_parity(got_u, ref, small.dtype, small.cm)
    # the fused and the layer-by-layer path use the same per-element arithmetic
    assert np.array_equal(wk.to_f64(got, small.dtype), wk.to_f64(got_u, small.dtype)), (
        "fused and unfused differ", e_f)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_pw_only_on_oracle_intermediate(cuda, wl, kernel):
    """PW_ONLY on a stored intermediate equals the oracle's 1x1 stage on the same values."""
    small = reduced(wl, n=1)
    case = wk.make_case(small)
    mod = module_or_skip(case, kernel)
    m_store = wk.to_storage(oracle_conv1(case), small.dtype)
    ref = oracle_pw(case, wk.to_f64(m_store, small.dtype))
    import torch
    y = empty(small.shapes()["y"], small.dtype, fill=float("nan"))
    mod.run(to_device(m_store, small.dtype), y, "pw")
    torch.cuda.synchronize()
    assert_parity(to_host(y, small.dtype), ref, small.dtype, small.cm)


EDGE = [  # (N, H, W, C, K, k, s, p, dtype, act1, act2)
    (1, 1, 1, 16, 16, 3, 1, 1, "f16", "relu", "relu"),
    (1, 13, 17, 32, 48, 3, 1, 1, "f16", "relu6", "none"),
    (3, 9, 30, 64, 32, 5, 2, 2, "bf16", "relu", "relu6"),
    (1, 7, 7, 16, 256, 7, 1, 3, "bf16", "none", "relu"),
    (2, 11, 5, 48, 16, 1, 1, 0, "f16", "relu", "none"),
    (1, 20, 131, 16, 16, 3, 1, 1, "f16", "relu", "relu"),
    (1, 15, 15, 8, 8, 3, 2, 0, "f32", "relu", "relu"),
    (2, 6, 9, 12, 20, 5, 1, 2, "f32", "relu6", "relu6"),
    # channel counts that leave the last 64-channel chunk partly empty, 3 and 4 chunks,
    # quadrants of 16 x 2 pixels, several tiles across, K = 256 with stride 2
    (2, 14, 14, 96, 64, 3, 1, 1, "f16", "relu6", "relu6"),
    (1, 33, 33, 192, 80, 5, 1, 2, "bf16", "relu", "none"),
    (2, 9, 70, 256, 256, 3, 2, 1, "f16", "none", "relu"),
    (1, 5, 9, 240, 80, 5, 1, 2, "bf16", "relu", "none"),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "x".join(map(str, s[:8])) + s[8])
def test_edge_shapes(cuda, shape, kernel):
    N, H, W, C, K, k, s, p, dt, a1, a2 = shape
    wl = wk.Workload("edge", N, H, W, C, K, "dw", k, s, p, a1, a2, dt, "normal")
    if kernel in ("tc", "tc_roles", "tc_workers") and dt == "f32":
        pytest.skip("fp32 runs on CUDA cores")
    case = wk.make_case(wl, seed=77)
    mod = module_or_skip(case, kernel)
    got, _ = run_case(case, "fused", module=mod)
    assert_parity(got, oracle_fused(case), dt, C)
    icase = wk.make_case(wl, seed=78, kind="integer")
    if wk.integer_safe(wl):
        imod = make_module(icase, kernel)
        got, _ = run_case(icase, "fused", module=imod)
        assert_bitexact(got, oracle_fused(icase), dt)


DENSE_EDGE = [  # (N, H, W, C, mid, K, k, p, dtype, act1, act2)
    (2, 9, 13, 32, 32, 48, 3, 1, "f16", "relu", "relu6"),
    (2, 9, 13, 64, 32, 48, 3, 1, "f16", "relu", "relu6"),
    (1, 11, 60, 128, 64, 64, 5, 2, "bf16", "relu", "none"),
    (3, 7, 100, 64, 16, 32, 3, 1, "f16", "none", "relu"),
    (1, 5, 21, 64, 48, 16, 1, 0, "bf16", "relu6", "relu"),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shape", DENSE_EDGE, ids=lambda s: "x".join(map(str, s[:8])) + s[8])
def test_dense_edge_shapes(cuda, shape, kernel):
    N, H, W, C, mid, K, k, p, dt, a1, a2 = shape
    wl = wk.Workload("dense_edge", N, H, W, C, K, "dense", k, 1, p, a1, a2, dt, "normal", mid=mid)
    case = wk.make_case(wl, seed=5)
    mod = module_or_skip(case, kernel)
    got, _ = run_case(case, "fused", module=mod)
    assert_parity(got, oracle_fused(case), dt, mid)
    got_u, _ = run_case(case, "unfused", module=mod)
    assert_parity(got_u, oracle_fused(case), dt, mid)
    if wk.integer_safe(wl, "integer1"):
        icase = wk.make_case(wl, seed=6, kind="integer1")
        got, _ = run_case(icase, "fused", module=make_module(icase, kernel))
        assert_bitexact(got, oracle_fused(icase), dt)


PWDW_EDGE = [  # (N, H, W, C, Cm, k, s, p, dtype, act1, act2): 1x1 C -> Cm, then depthwise k x k
    (2, 9, 13, 64, 64, 3, 1, 1, "f16", "relu6", "relu6"),
    (1, 11, 60, 64, 128, 3, 2, 1, "bf16", "relu", "none"),
    (3, 7, 20, 128, 64, 5, 1, 2, "f16", "none", "relu"),
    (1, 5, 100, 64, 64, 3, 1, 1, "f16", "relu", "relu"),
    (2, 6, 6, 64, 192, 1, 1, 0, "bf16", "relu", "relu"),
    (1, 13, 17, 32, 48, 3, 1, 1, "f16", "relu6", "none"),
    (1, 9, 9, 8, 16, 3, 2, 1, "f32", "relu", "relu6"),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shape", PWDW_EDGE, ids=lambda s: "x".join(map(str, s[:8])) + s[8])
def test_pwdw_edge_shapes(cuda, shape, kernel):
    """PWDW: tiles whose halo crosses the image border (the intermediate is zero there, not
    act(bias)), stride 2, 5x5, several M blocks per halo, k = 1."""
    N, H, W, C, mid, k, s, p, dt, a1, a2 = shape
    wl = wk.Workload("pwdw_edge", N, H, W, C, mid, "pwdw", k, s, p, a1, a2, dt, "normal", mid=mid)
    case = wk.make_case(wl, seed=7)
    mod = module_or_skip(case, kernel)
    ref = oracle_fused(case)
    got, _ = run_case(case, "fused", module=mod)
    assert_parity(got, ref, dt, max(C, k * k))   # longest reduction on the path (fp32 bar)
    got_u, _ = run_case(case, "unfused", module=mod)
    assert_parity(got_u, ref, dt, max(C, k * k))
    kind = "integer" if wk.integer_safe(wl) else "integer1"
    if wk.integer_safe(wl, kind):
        icase = wk.make_case(wl, seed=8, kind=kind)
        imod = make_module(icase, kernel) if kernel == "simt" else module_or_skip(icase, kernel)
        iref = oracle_fused(icase)
        for mode in ("fused", "unfused"):
            got, _ = run_case(icase, mode, module=imod)
            assert_bitexact(got, iref, dt)


I8_EDGE = [  # (N, H, W, C, K, k, s, p, act1, act2): the INT8 module, int8 over the full range
    (1, 1, 1, 16, 16, 3, 1, 1, "relu", "none"),
    (2, 13, 17, 32, 48, 3, 1, 1, "none", "relu6"),
    (3, 9, 30, 64, 32, 5, 2, 2, "relu", "relu"),
    (1, 7, 7, 16, 256, 7, 1, 3, "none", "none"),
    (2, 11, 5, 48, 16, 1, 1, 0, "relu", "none"),
    (1, 20, 131, 16, 16, 3, 1, 1, "relu", "relu"),
    (2, 12, 14, 256, 64, 3, 2, 1, "relu6", "none"),
    (1, 9, 40, 96, 80, 7, 2, 3, "relu", "relu6"),
]


@pytest.mark.parametrize("kernel", ["tc_roles", "tc_workers"])
@pytest.mark.parametrize("shape", I8_EDGE, ids=lambda s: "x".join(map(str, s[:8])))
def test_int8_edge_shapes(cuda, shape, kernel):
    """INT8 DW -> PW: bit-exact with the oracle in every mode (fused, layer by layer, the
    depthwise layer alone, the 1x1 on the oracle's intermediate): ragged tiles, 1x1 images,
    stride 2, k = 1, 5, 7, the widest channel counts."""
    import torch
    N, H, W, C, K, k, s, p, a1, a2 = shape
    wl = wk.Workload("i8_edge", N, H, W, C, K, "dw", k, s, p, a1, a2, "i8", "int8")
    case = wk.make_case(wl, seed=91)
    mod = make_module(case, kernel)
    ref = oracle_fused(case)
    for mode in ("fused", "unfused"):
        got, _ = run_case(case, mode, module=mod)
        assert_bitexact(got, ref, "i8")
    m_ref = oracle_conv1(case)
    m_gpu, _ = run_case(case, "conv1", module=mod)
    assert_bitexact(m_gpu, m_ref, "i8")
    y = empty(wl.shapes()["y"], "i8", fill=float("nan"))
    mod.run(to_device(m_ref.astype(np.int8), "i8"), y, "pw")
    torch.cuda.synchronize()
    mod.check()
    assert_bitexact(to_host(y, "i8"), oracle_pw(case, m_ref), "i8")


PWDW_I8_EDGE = [  # (N, H, W, C, Cm, k, s, p, act1, act2): the INT8 PWDW module
    (2, 9, 13, 64, 64, 3, 1, 1, "relu", "none"),
    (1, 11, 60, 64, 128, 3, 2, 1, "relu", "relu"),
    (3, 7, 20, 128, 64, 5, 1, 2, "none", "relu"),
    (2, 6, 6, 64, 192, 1, 1, 0, "relu", "none"),
    (1, 13, 17, 64, 128, 7, 1, 3, "relu6", "none"),
    (1, 9, 9, 256, 64, 3, 1, 1, "relu", "relu"),
]


@pytest.mark.parametrize("shape", PWDW_I8_EDGE, ids=lambda s: "x".join(map(str, s[:8])))
def test_int8_pwdw_edge_shapes(cuda, shape):
    """INT8 1x1 -> depthwise: bit-exact with the oracle fused (the int8 intermediate recomputed
    under every depthwise tap, int8 zero in the padding), layer by layer, the 1x1 layer alone,
    and the depthwise layer on the oracle's intermediate; halos across the image border, stride
    2, k = 1, 5, 7, and C = 256 (the 1x1's widest exact reduction; with a 3x3 halo, since a
    7x7 one of 256 channels does not fit shared memory)."""
    import torch
    N, H, W, C, Cm, k, s, p, a1, a2 = shape
    wl = wk.Workload("i8_pwdw", N, H, W, C, Cm, "pwdw", k, s, p, a1, a2, "i8", "int8", mid=Cm)
    case = wk.make_case(wl, seed=95)
    mod = make_module(case, "tc")
    ref = oracle_fused(case)
    for mode in ("fused", "unfused"):
        got, _ = run_case(case, mode, module=mod)
        assert_bitexact(got, ref, "i8")
    m_ref = oracle_conv1(case)
    m_gpu, _ = run_case(case, "conv1", module=mod)
    assert_bitexact(m_gpu, m_ref, "i8")
    y = empty(wl.shapes()["y"], "i8", fill=float("nan"))
    mod.run(to_device(m_ref.astype(np.int8), "i8"), y, "pw")
    torch.cuda.synchronize()
    mod.check()
    assert_bitexact(to_host(y, "i8"), oracle_pw(case, m_ref), "i8")


def test_int8_shapes_refused(cuda):
    """INT8 requests outside the tensor-core kernels fail with FCM_ERR_UNSUPPORTED (a dense
    3x3 first layer, more than 256 channels, a PWDW input that is not a multiple of 64)."""
    for kw in ({"conv1": "dense", "mid": 32}, {"c": 512, "k_out": 64},
               {"conv1": "pwdw", "mid": 32}):
        wl = wk.Workload("i8_no", 1, 8, 8, kw.get("c", 32), kw.get("k_out", 32),
                         kw.get("conv1", "dw"), 3, 1, 1, "relu", "none", "i8", "int8",
                         mid=kw.get("mid", 0))
        with pytest.raises(fcm.FcmError) as e:
            make_module(wk.make_case(wl))
        assert e.value.status == 2, kw


def test_run_host_matches_run(cuda):
    import torch
    wl = reduced(wk.BY_NAME["mobilenet_dwpw_f16"], n=2)
    case = wk.make_case(wl)
    mod = make_module(case)
    got, _ = run_case(case, "fused", module=mod)
    x_h = to_device(case.x, wl.dtype, "cpu").pin_memory()
    y_h = torch.empty(wl.shapes()["y"], dtype=torch.float16).pin_memory()
    mod.run_host(x_h, y_h, "fused")
    assert np.array_equal(y_h.numpy(), got)


@pytest.mark.parametrize("name,n", [("mobilenet_dwpw_f16", 5), ("b2b_dense3x3_f16", 3),
                                    ("pwdw_f16", 9), ("tiny_dwpw_f32", 1),
                                    ("mobilenet_dwpw_i8", 6)])
def test_run_host_pipelined_chunks(cuda, name, n):
    """fcm_run_host splits the batch into chunks whose copies overlap the kernels (uneven
    chunks for n = 5 and 9): the result equals fcm_run on the device for every mode."""
    import torch
    wl = wk.BY_NAME[name].with_(n=n, h=min(wk.BY_NAME[name].h, 20), w=min(wk.BY_NAME[name].w, 20))
    case = wk.make_case(wl)
    mod = make_module(case)
    x_h = to_device(case.x, wl.dtype, "cpu").pin_memory()
    for mode, out_key in (("fused", "y"), ("conv1", "m"), ("unfused", "y")):
        want, _ = run_case(case, mode, module=mod)
        got = empty(wl.shapes()[out_key], wl.dtype, "cpu", fill=float("nan")).pin_memory()
        mod.run_host(x_h, got, mode)
        assert np.array_equal(to_host(got, wl.dtype), want), mode


def test_argument_errors(cuda):
    import torch
    wl = reduced(wk.BY_NAME["mobilenet_dwpw_f16"], n=1)
    case = wk.make_case(wl)
    mod = make_module(case)
    x = to_device(case.x, wl.dtype)
    y = empty(wl.shapes()["y"], wl.dtype)
    raw = torch.empty(x.numel() * 2 + 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_run(mod.handle, 0, raw.data_ptr() + 2, y.data_ptr(), 0)
    assert e.value.status == 3
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_run(mod.handle, 0, x.data_ptr(), x.data_ptr(), 0)
    assert e.value.status == 1
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_run(mod.handle, 9, x.data_ptr(), y.data_ptr(), 0)
    assert e.value.status == 1
    mod.check()


def test_weights_from_device_memory(cuda):
    import torch
    wl = reduced(wk.BY_NAME["stride2_dwpw_bf16"], n=1, hw=20)
    case = wk.make_case(wl)
    d = fcm.desc_from_workload(wl)
    dev = [to_device(a, wl.dtype) for a in (case.w1, case.wp)]
    sb = [torch.from_numpy(a).cuda() for a in (case.s1, case.b1, case.s2, case.b2)]
    mod = fcm.FusedConvModule(d, dev[0], dev[1], *sb)
    got, _ = run_case(case, "fused", module=mod)
    assert_parity(got, oracle_fused(case), wl.dtype, wl.cm)


# ---------------------------------------------------------------- full-size, sampled images
SAMPLE_IMAGES = 2


@pytest.mark.slow
@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_full_size_sampled(cuda, wl):
    """The full batch in the launch configuration the benchmark times (planner's choice);
    the oracle recomputes the first and the last image."""
    case = wk.make_case(wl)
    got, mod = run_case(case, "fused")
    picks = [0, wl.n - 1][:SAMPLE_IMAGES]
    for i in picks:
        sub = wk.Case(wl.with_(n=1), case.seed, case.x[i:i + 1], case.w1, case.wp, case.s1,
                      case.b1, case.s2, case.b2)
        assert_parity(got[i:i + 1], oracle_fused(sub), wl.dtype, wl.cm)
    assert np.all(np.isfinite(wk.to_f64(got, wl.dtype)))


def test_bounded_wait_reports_timeout_and_context_survives(cuda):
    """Failure detection: a kernel's bounded wait on an mbarrier phase that nothing completes
    gives up after its limit and reports FCM_ERR_TIMEOUT; the CUDA context stays usable."""
    import time
    t0 = time.monotonic()
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_selftest_wait_timeout(2_000_000)   # 2 ms
    assert e.value.status == 6, e.value
    assert time.monotonic() - t0 < 5.0
    wl = reduced(wk.BY_NAME["mobilenet_dwpw_i8"], n=1, hw=14)
    case = wk.make_case(wl)
    got, _ = run_case(case, "fused")
    assert_bitexact(got, oracle_fused(case), "i8")


I8_PWPW_EDGE = [  # (N, H, W, C, Cm, K, act1, act2): the INT8 PWPW module (two 1x1 convolutions)
    (2, 9, 13, 64, 64, 64, "relu", "none"),
    (1, 11, 60, 128, 64, 128, "none", "relu6"),
    (3, 7, 100, 64, 32, 48, "relu6", "relu"),
    (1, 5, 21, 128, 64, 128, "relu", "none"),
    (2, 1, 1, 64, 16, 16, "none", "none"),
]


@pytest.mark.parametrize("shape", I8_PWPW_EDGE, ids=lambda s: "x".join(map(str, s[:6])))
def test_int8_pwpw_edge_shapes(cuda, shape):
    """INT8 1x1 -> 1x1 on the back-to-back kernel (int8 tiles widened to f16 by converter
    warps): bit-exact with the oracle fused, layer by layer, first layer alone, and the second
    layer on the oracle's intermediate; pitches of 64 and 128 columns, C up to 128 (the int8
    and the f16 input rings of wider layers do not fit next to the weights)."""
    import torch
    N, H, W, C, Cm, K, a1, a2 = shape
    wl = wk.Workload("i8_pwpw", N, H, W, C, K, "dense", 1, 1, 0, a1, a2, "i8", "int8", mid=Cm)
    case = wk.make_case(wl, seed=93)
    mod = make_module(case, "tc")
    ref = oracle_fused(case)
    for mode in ("fused", "unfused"):
        got, _ = run_case(case, mode, module=mod)
        assert_bitexact(got, ref, "i8")
    m_ref = oracle_conv1(case)
    m_gpu, _ = run_case(case, "conv1", module=mod)
    assert_bitexact(m_gpu, m_ref, "i8")
    y = empty(wl.shapes()["y"], "i8", fill=float("nan"))
    mod.run(to_device(m_ref.astype(np.int8), "i8"), y, "pw")
    torch.cuda.synchronize()
    mod.check()
    assert_bitexact(to_host(y, "i8"), oracle_pw(case, m_ref), "i8")


def test_output_guards_detect_a_stray_write(cuda):
    """The guard zones run_case puts around every output catch a write outside the output: one
    byte just past the end (written by torch inside the same allocation) trips the check, an
    untouched buffer passes it."""
    import torch
    from helpers import GUARD_BYTES, guarded_empty
    t, check = guarded_empty((2, 3, 5, 16), "f16", fill=0.0)
    check()
    flat = t.view(torch.uint8).view(-1)
    # the first byte past the output (as_strided takes an offset into the whole allocation)
    raw = torch.as_strided(flat, (1,), (1,), flat.storage_offset() + flat.numel())
    raw.fill_(0)
    torch.cuda.synchronize()
    with pytest.raises(AssertionError):
        check()
    assert GUARD_BYTES >= 16
