"""Shared helpers of the GPU tests: storage <-> torch, running a module through the C ABI,
and the parity bars."""
from __future__ import annotations

import numpy as np

import oracle
import pointwise_conv_cnn_gb300 as fcm
from pointwise_conv_cnn_gb300 import workloads as wk

# Parity bars: fp32 max-abs error <= 1e-4 * sqrt(C) with C the 1x1 reduction length;
# fp16/bf16 max-norm relative error <= 2e-2 (max|gpu - ref| / max|ref|); INT8 exact.
F32_ABS_PER_SQRT_C = 1e-4
HALF_REL = 2e-2


def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
            "i8": torch.int8}[dtype]


def to_device(arr: np.ndarray, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.to(device)


def to_host(t, dtype: str) -> np.ndarray:
    import torch
    t = t.detach().cpu()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def empty(shape, dtype: str, device="cuda", fill=None):
    import torch
    t = torch.empty(shape, dtype=torch_dtype(dtype), device=device)
    if fill is not None:
        # int8 has no NaN: a value the kernels must overwrite (compared element by element)
        t.fill_(I8_FILL if dtype == "i8" and fill != fill else fill)
    return t


I8_FILL = -77
GUARD_BYTES = 256      # guard zone on each side of an output buffer
GUARD_BYTE = 0xA5


def guarded_empty(shape, dtype: str, fill=None):
    """An output tensor on the GPU inside one allocation with a guard zone of GUARD_BYTES
    before and after it, filled with GUARD_BYTE.  Returns (tensor, check); check() raises if a
    kernel wrote into either zone (a store outside the output it was given)."""
    import torch
    tdt = torch_dtype(dtype)
    n = int(np.prod(shape)) * torch.empty((), dtype=tdt).element_size()
    buf = torch.full((n + 2 * GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
    t = buf[GUARD_BYTES:GUARD_BYTES + n].view(tdt).view(shape)
    if fill is not None:
        t.fill_(I8_FILL if dtype == "i8" and fill != fill else fill)

    def check():
        lo = buf[:GUARD_BYTES].cpu().numpy()
        hi = buf[GUARD_BYTES + n:].cpu().numpy()
        bad = int((lo != GUARD_BYTE).sum() + (hi != GUARD_BYTE).sum())
        assert bad == 0, f"{bad} guard bytes around the output were overwritten"
    return t, check


def make_module(case: wk.Case, kernel: str = "auto", **desc_over) -> fcm.FusedConvModule:
    d = fcm.desc_from_workload(case.wl, kernel=kernel, **desc_over)
    return fcm.FusedConvModule(d, case.w1, case.wp, case.s1, case.b1, case.s2, case.b2)


def run_case(case: wk.Case, mode: str = "fused", kernel: str = "auto", inp=None,
             module=None):
    """Run one mode on the GPU; returns (output storage array, module)."""
    import torch
    wl = case.wl
    mod = module or make_module(case, kernel)
    sh = wl.shapes()
    x = to_device(case.x if inp is None else inp, wl.dtype)
    out_shape = sh["m"] if mode == "conv1" else sh["y"]
    y, guards = guarded_empty(out_shape, wl.dtype, fill=float("nan"))
    mod.run(x, y, mode)
    torch.cuda.synchronize()
    mod.check()
    guards()
    return to_host(y, wl.dtype), mod


def oracle_fused(case: wk.Case, mid: str = "exact", nthreads: int = 0) -> np.ndarray:
    wl = case.wl
    if wl.dtype == "i8":   # int8 results, as float64 for the shared comparisons
        fn = {"dense": oracle.fused_dense_i8, "pwdw": oracle.pwdw_i8}.get(wl.conv1, oracle.fused_i8)
        return fn(case.x, case.w1, case.s1, case.b1, case.wp, case.s2, case.b2, wl.act1, wl.act2,
                  wl.stride, wl.pad, nthreads=nthreads).astype(np.float64)
    f = case.f64()
    if wl.conv1 == "pwdw":
        return oracle.pwdw(f["x"], f["w1"], f["s1"], f["b1"], f["wp"], f["s2"], f["b2"],
                           wl.act1, wl.act2, wl.stride, wl.pad, mid=mid, nthreads=nthreads)
    return oracle.fused(f["x"], f["w1"], f["s1"], f["b1"], f["wp"], f["s2"], f["b2"], wl.act1,
                        wl.act2, wl.stride, wl.pad, conv1=wl.conv1, mid=mid, nthreads=nthreads)


def oracle_conv1(case: wk.Case) -> np.ndarray:
    wl = case.wl
    if wl.dtype == "i8":
        if wl.conv1 == "pwdw":   # the 1x1 layer, over the input's extent
            return oracle.pw_i8(case.x, case.w1, case.s1, case.b1, wl.act1).astype(np.float64)
        fn = oracle.dense_i8 if wl.conv1 == "dense" else oracle.dw_i8
        return fn(case.x, case.w1, case.s1, case.b1, wl.act1, wl.stride, wl.pad).astype(np.float64)
    f = case.f64()
    if wl.conv1 == "pwdw":   # the 1x1 layer, over the input's extent
        return oracle.pw(f["x"], f["w1"], f["s1"], f["b1"], wl.act1)
    if wl.conv1 == "dw":
        return oracle.dw(f["x"], f["w1"], f["s1"], f["b1"], wl.act1, wl.stride, wl.pad)
    return oracle.dense(f["x"], f["w1"], f["s1"], f["b1"], wl.act1, wl.stride, wl.pad)


def oracle_pw(case: wk.Case, m: np.ndarray) -> np.ndarray:
    """The module's second convolution on an intermediate (the depthwise one for PWDW)."""
    wl = case.wl
    if wl.dtype == "i8":
        if wl.conv1 == "pwdw":   # the depthwise layer over the intermediate
            return oracle.dw_i8(np.asarray(m).astype(np.int8), case.wp, case.s2, case.b2, wl.act2,
                                wl.stride, wl.pad).astype(np.float64)
        return oracle.pw_i8(np.asarray(m).astype(np.int8), case.wp, case.s2, case.b2,
                            wl.act2).astype(np.float64)
    f = case.f64()
    if wl.conv1 == "pwdw":
        return oracle.dw(m, f["wp"], f["s2"], f["b2"], wl.act2, wl.stride, wl.pad)
    return oracle.pw(m, f["wp"], f["s2"], f["b2"], wl.act2)


def parity_error(gpu_storage: np.ndarray, ref: np.ndarray, dtype: str) -> float:
    g = wk.to_f64(gpu_storage, dtype)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "non-finite output"
    err = float(np.abs(g - ref).max(initial=0.0))
    if dtype in ("f32", "i8"):
        return err
    return err / max(float(np.abs(ref).max(initial=0.0)), 1e-6)


def assert_parity(gpu_storage: np.ndarray, ref: np.ndarray, dtype: str, c_red: int) -> float:
    e = parity_error(gpu_storage, ref, dtype)
    bar = {"f32": F32_ABS_PER_SQRT_C * np.sqrt(c_red), "i8": 0.0}.get(dtype, HALF_REL)
    assert e <= bar, f"parity error {e:.3e} above bar {bar:.3e}"
    return e


def assert_bitexact(gpu_storage: np.ndarray, ref: np.ndarray, dtype: str) -> None:
    """Exact equality with the oracle rounded once to the storage format (values compared,
    so +0 and -0 count as equal)."""
    want = wk.to_f64(wk.to_storage(ref, dtype), dtype)
    got_f = wk.to_f64(np.asarray(gpu_storage), dtype)
    got = np.asarray(gpu_storage)
    eq = got_f == want
    if not eq.all():
        idx = np.argwhere(~eq)[:5]
        raise AssertionError(
            f"{int((~eq).sum())} of {eq.size} outputs differ; first at {idx.tolist()}: "
            f"got {[wk.to_f64(got[tuple(i)], dtype) for i in idx]} want {[ref[tuple(i)] for i in idx]}")
