"""fp64 CPU oracle for the fused DW/dense k x k -> 1x1 convolution module.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers.  The product path (the CUDA library in
``pointwise_conv_cnn_gb300``) never imports this package, and this package imports nothing
from it.

The arithmetic lives in ``fcm_oracle.c`` (plain loops, fp64).  This module only builds that
file with gcc, loads it with ctypes and marshals numpy arrays.  Inputs of any float dtype are
upcast to float64 exactly before the call; outputs are float64.  The INT8 functions
(``dw_i8``, ``pw_i8``, ``fused_i8``, ``dense_i8``, ``fused_dense_i8``, ``pwdw_i8``) take int8
activations and weights and fp32 scales and biases, and return int8 (section III-B's INT8
FCMs).

Definitions followed (see the C file for the full list): "Fusing Depthwise and Pointwise
Convolutions for Efficient Inference on GPUs", section II-B (DW and PW convolutions),
section II-D / Figure 3(b) (PWDW_R) and section III-A (conv -> norm -> activation, up to six
fused layers); "Fusing two back-to-back
convolutions" (CUTLASS discussion #208), the CONV1 3x3 -> CONV2 1x1 scale_bias_relu example.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fcm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ACT = {"none": 0, "relu": 1, "relu6": 2}
MID = {"exact": 0, "f32": 1, "f16": 2, "bf16": 3}


def build(force: bool = False) -> str:
    """Compile fcm_oracle.c into liboracle.so next to it (OpenMP when gcc supports it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def bind(path: str):
    """Load an oracle shared library from `path` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_dw.argtypes = [i] * 7 + [dp] * 4 + [i, dp, i]
    lib.oracle_pw.argtypes = [i] * 5 + [dp] * 4 + [i, dp, i]
    lib.oracle_dense.argtypes = [i] * 8 + [dp] * 4 + [i, dp, i]
    lib.oracle_fused.argtypes = [i] * 10 + [dp] * 4 + [i] + [dp] * 3 + [i, i, dp, i]
    lib.oracle_pwdw.argtypes = [i] * 8 + [dp] * 4 + [i] + [dp] * 3 + [i, i, dp, i]
    lib.oracle_round_format.argtypes = [ctypes.c_double, i, i, ctypes.c_double]
    lib.oracle_round_format.restype = ctypes.c_double
    lib.oracle_max_threads.argtypes = [i]
    bp = ctypes.POINTER(ctypes.c_int8)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.oracle_dw_i8.argtypes = [i] * 7 + [bp, bp, fp, fp, i, bp, i]
    lib.oracle_pw_i8.argtypes = [i] * 5 + [bp, bp, fp, fp, i, bp, i]
    lib.oracle_fused_i8.argtypes = [i] * 8 + [bp, bp, fp, fp, i, bp, fp, fp, i, bp, i]
    lib.oracle_requant_i8.argtypes = [ctypes.c_longlong, ctypes.c_float, ctypes.c_float, i]
    lib.oracle_dense_i8.argtypes = [i] * 8 + [bp, bp, fp, fp, i, bp, i]
    lib.oracle_fused_dense_i8.argtypes = [i] * 9 + [bp, bp, fp, fp, i, bp, fp, fp, i, bp, i]
    lib.oracle_pwdw_i8.argtypes = [i] * 8 + [bp, bp, fp, fp, i, bp, fp, fp, i, bp, i]
    for f in (lib.oracle_dw, lib.oracle_pw, lib.oracle_dense, lib.oracle_fused, lib.oracle_pwdw,
              lib.oracle_max_threads, lib.oracle_dw_i8, lib.oracle_pw_i8, lib.oracle_fused_i8,
              lib.oracle_requant_i8, lib.oracle_dense_i8, lib.oracle_fused_dense_i8,
              lib.oracle_pwdw_i8):
        f.restype = ctypes.c_int
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            build()
            _lib = bind(_LIB)
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def out_extent(n: int, k: int, s: int, p: int) -> int:
    """Output extent floor((n + 2p - k)/s) + 1 (zero padding, cross-correlation)."""
    return (n + 2 * p - k) // s + 1


def max_threads(nthreads: int = 0, lib=None) -> int:
    return int(_load(lib).oracle_max_threads(int(nthreads)))


def dw(x, wd, s1, b1, act1="none", stride=1, pad=0, nthreads=0, lib=None) -> np.ndarray:
    """Depthwise conv: x [N,H,W,C], wd [C,k,k] -> act1(s1*conv + b1) as [N,Ho,Wo,C]."""
    x, wd, s1, b1 = map(_f64, (x, wd, s1, b1))
    N, H, W, C = x.shape
    k = wd.shape[1]
    assert wd.shape == (C, k, k) and s1.shape == (C,) and b1.shape == (C,)
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    m = np.empty((N, Ho, Wo, C), np.float64)
    rc = _load(lib).oracle_dw(N, H, W, C, k, stride, pad, _ptr(x), _ptr(wd), _ptr(s1), _ptr(b1),
                           ACT[act1], _ptr(m), nthreads)
    if rc != 0:
        raise ValueError("oracle_dw: invalid shape")
    return m


def pw(m, wp, s2, b2, act2="none", nthreads=0, lib=None) -> np.ndarray:
    """Pointwise conv: m [N,Ho,Wo,Cm], wp [K,Cm] -> act2(s2*(m.wp^T) + b2) as [N,Ho,Wo,K]."""
    m, wp, s2, b2 = map(_f64, (m, wp, s2, b2))
    N, Ho, Wo, Cm = m.shape
    K = wp.shape[0]
    assert wp.shape == (K, Cm) and s2.shape == (K,) and b2.shape == (K,)
    y = np.empty((N, Ho, Wo, K), np.float64)
    rc = _load(lib).oracle_pw(N, Ho, Wo, Cm, K, _ptr(m), _ptr(wp), _ptr(s2), _ptr(b2), ACT[act2],
                           _ptr(y), nthreads)
    if rc != 0:
        raise ValueError("oracle_pw: invalid shape")
    return y


def dense(x, w1, s1, b1, act1="none", stride=1, pad=0, nthreads=0, lib=None) -> np.ndarray:
    """Dense conv: x [N,H,W,C], w1 [K1,k,k,C] -> act1(s1*conv + b1) as [N,Ho,Wo,K1]."""
    x, w1, s1, b1 = map(_f64, (x, w1, s1, b1))
    N, H, W, C = x.shape
    K1, k = w1.shape[0], w1.shape[1]
    assert w1.shape == (K1, k, k, C) and s1.shape == (K1,) and b1.shape == (K1,)
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    m = np.empty((N, Ho, Wo, K1), np.float64)
    rc = _load(lib).oracle_dense(N, H, W, C, K1, k, stride, pad, _ptr(x), _ptr(w1), _ptr(s1),
                              _ptr(b1), ACT[act1], _ptr(m), nthreads)
    if rc != 0:
        raise ValueError("oracle_dense: invalid shape")
    return m


def fused(x, w1, s1, b1, wp, s2, b2, act1="none", act2="none", stride=1, pad=0,
          conv1="dw", mid="exact", nthreads=0, lib=None) -> np.ndarray:
    """Fused module in one pass: conv1 (``"dw"`` with w1 [C,k,k] or ``"dense"`` with
    w1 [K1,k,k,C]) + scale/bias/act1, then 1x1 conv wp [K,Cm] + scale/bias/act2."""
    x, w1, s1, b1, wp, s2, b2 = map(_f64, (x, w1, s1, b1, wp, s2, b2))
    N, H, W, C = x.shape
    is_dense = conv1 == "dense"
    if is_dense:
        Cm, k = w1.shape[0], w1.shape[1]
        assert w1.shape == (Cm, k, k, C)
    else:
        Cm, k = C, w1.shape[1]
        assert w1.shape == (C, k, k)
    K = wp.shape[0]
    assert wp.shape == (K, Cm) and s1.shape == (Cm,) and b1.shape == (Cm,)
    assert s2.shape == (K,) and b2.shape == (K,)
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    y = np.empty((N, Ho, Wo, K), np.float64)
    rc = _load(lib).oracle_fused(int(is_dense), N, H, W, C, Cm, K, k, stride, pad, _ptr(x),
                              _ptr(w1), _ptr(s1), _ptr(b1), ACT[act1], _ptr(wp), _ptr(s2),
                              _ptr(b2), ACT[act2], MID[mid], _ptr(y), nthreads)
    if rc != 0:
        raise ValueError("oracle_fused: invalid shape")
    return y


def pwdw(x, wq, s1, b1, wd2, s2, b2, act1="none", act2="none", stride=1, pad=0, mid="exact",
         nthreads=0, lib=None) -> np.ndarray:
    """PWDW module in one pass: 1x1 conv wq [Cm,C] + scale/bias/act1, then depthwise
    wd2 [Cm,k,k] over the intermediate (zero padding of the intermediate) + scale/bias/act2;
    x [N,H,W,C] -> [N,Ho,Wo,Cm]."""
    x, wq, s1, b1, wd2, s2, b2 = map(_f64, (x, wq, s1, b1, wd2, s2, b2))
    N, H, W, C = x.shape
    Cm, k = wd2.shape[0], wd2.shape[1]
    assert wq.shape == (Cm, C) and wd2.shape == (Cm, k, k)
    assert s1.shape == (Cm,) and b1.shape == (Cm,) and s2.shape == (Cm,) and b2.shape == (Cm,)
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    y = np.empty((N, Ho, Wo, Cm), np.float64)
    rc = _load(lib).oracle_pwdw(N, H, W, C, Cm, k, stride, pad, _ptr(x), _ptr(wq), _ptr(s1),
                                _ptr(b1), ACT[act1], _ptr(wd2), _ptr(s2), _ptr(b2), ACT[act2],
                                MID[mid], _ptr(y), nthreads)
    if rc != 0:
        raise ValueError("oracle_pwdw: invalid shape")
    return y


def _i8(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.int8:
        if not np.issubdtype(a.dtype, np.integer) or a.min(initial=0) < -128 or a.max(initial=0) > 127:
            raise ValueError("int8 operand expected")
        a = a.astype(np.int8)
    return np.ascontiguousarray(a)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _p8(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))


def _p32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def requant_i8(acc: int, s: float, b: float, act: str = "none", lib=None) -> int:
    """int8 requantization of one accumulator: clamp(rint(act(fma32(s, acc, b))), -128, 127)."""
    return int(_load(lib).oracle_requant_i8(int(acc), float(s), float(b), ACT[act]))


def dw_i8(x, wd, s1, b1, act1="none", stride=1, pad=0, nthreads=0, lib=None) -> np.ndarray:
    """INT8 depthwise conv: x [N,H,W,C] int8, wd [C,k,k] int8, s1/b1 fp32 -> m int8."""
    x, wd = _i8(x), _i8(wd)
    s1, b1 = _f32(s1), _f32(b1)
    N, H, W, C = x.shape
    k = wd.shape[1]
    assert wd.shape == (C, k, k) and s1.shape == (C,) and b1.shape == (C,)
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    m = np.empty((N, Ho, Wo, C), np.int8)
    rc = _load(lib).oracle_dw_i8(N, H, W, C, k, stride, pad, _p8(x), _p8(wd), _p32(s1),
                                 _p32(b1), ACT[act1], _p8(m), nthreads)
    if rc != 0:
        raise ValueError("oracle_dw_i8: invalid shape")
    return m


def pw_i8(m, wp, s2, b2, act2="none", nthreads=0, lib=None) -> np.ndarray:
    """INT8 pointwise conv: m [N,Ho,Wo,Cm] int8, wp [K,Cm] int8, s2/b2 fp32 -> y int8."""
    m, wp = _i8(m), _i8(wp)
    s2, b2 = _f32(s2), _f32(b2)
    N, Ho, Wo, Cm = m.shape
    K = wp.shape[0]
    assert wp.shape == (K, Cm) and s2.shape == (K,) and b2.shape == (K,)
    y = np.empty((N, Ho, Wo, K), np.int8)
    rc = _load(lib).oracle_pw_i8(N, Ho, Wo, Cm, K, _p8(m), _p8(wp), _p32(s2), _p32(b2),
                                 ACT[act2], _p8(y), nthreads)
    if rc != 0:
        raise ValueError("oracle_pw_i8: invalid shape")
    return y


def fused_i8(x, wd, s1, b1, wp, s2, b2, act1="none", act2="none", stride=1, pad=0,
             nthreads=0, lib=None) -> np.ndarray:
    """INT8 DW -> PW module in one pass (int8 intermediate): x [N,H,W,C], wd [C,k,k],
    wp [K,C] int8; s1/b1 [C], s2/b2 [K] fp32 -> y [N,Ho,Wo,K] int8."""
    x, wd, wp = _i8(x), _i8(wd), _i8(wp)
    s1, b1, s2, b2 = map(_f32, (s1, b1, s2, b2))
    N, H, W, C = x.shape
    k = wd.shape[1]
    K = wp.shape[0]
    assert wd.shape == (C, k, k) and wp.shape == (K, C)
    assert s1.shape == (C,) and b1.shape == (C,) and s2.shape == (K,) and b2.shape == (K,)
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    y = np.empty((N, Ho, Wo, K), np.int8)
    rc = _load(lib).oracle_fused_i8(N, H, W, C, K, k, stride, pad, _p8(x), _p8(wd), _p32(s1),
                                    _p32(b1), ACT[act1], _p8(wp), _p32(s2), _p32(b2), ACT[act2],
                                    _p8(y), nthreads)
    if rc != 0:
        raise ValueError("oracle_fused_i8: invalid shape")
    return y


def dense_i8(x, w1, s1, b1, act1="none", stride=1, pad=0, nthreads=0, lib=None) -> np.ndarray:
    """INT8 dense conv: x [N,H,W,C] int8, w1 [Cm,k,k,C] int8, s1/b1 fp32 -> m int8."""
    x, w1 = _i8(x), _i8(w1)
    s1, b1 = _f32(s1), _f32(b1)
    N, H, W, C = x.shape
    Cm, k = w1.shape[0], w1.shape[1]
    assert w1.shape == (Cm, k, k, C) and s1.shape == (Cm,) and b1.shape == (Cm,)
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    m = np.empty((N, Ho, Wo, Cm), np.int8)
    rc = _load(lib).oracle_dense_i8(N, H, W, C, Cm, k, stride, pad, _p8(x), _p8(w1), _p32(s1),
                                    _p32(b1), ACT[act1], _p8(m), nthreads)
    if rc != 0:
        raise ValueError("oracle_dense_i8: invalid shape")
    return m


def fused_dense_i8(x, w1, s1, b1, wp, s2, b2, act1="none", act2="none", stride=1, pad=0,
                   nthreads=0, lib=None) -> np.ndarray:
    """INT8 dense k x k -> 1x1 module in one pass (PWPW for k = 1): x [N,H,W,C], w1 [Cm,k,k,C],
    wp [K,Cm] int8; s1/b1 [Cm], s2/b2 [K] fp32 -> y [N,Ho,Wo,K] int8."""
    x, w1, wp = _i8(x), _i8(w1), _i8(wp)
    s1, b1, s2, b2 = map(_f32, (s1, b1, s2, b2))
    N, H, W, C = x.shape
    Cm, k = w1.shape[0], w1.shape[1]
    K = wp.shape[0]
    assert w1.shape == (Cm, k, k, C) and wp.shape == (K, Cm)
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    y = np.empty((N, Ho, Wo, K), np.int8)
    rc = _load(lib).oracle_fused_dense_i8(N, H, W, C, Cm, K, k, stride, pad, _p8(x), _p8(w1),
                                          _p32(s1), _p32(b1), ACT[act1], _p8(wp), _p32(s2),
                                          _p32(b2), ACT[act2], _p8(y), nthreads)
    if rc != 0:
        raise ValueError("oracle_fused_dense_i8: invalid shape")
    return y


def pwdw_i8(x, wq, s1, b1, wd2, s2, b2, act1="none", act2="none", stride=1, pad=0,
            nthreads=0, lib=None) -> np.ndarray:
    """INT8 PWDW module in one pass (int8 intermediate, recomputed under each depthwise tap):
    x [N,H,W,C], wq [Cm,C], wd2 [Cm,k,k] int8; s1/b1, s2/b2 [Cm] fp32 -> y [N,Ho,Wo,Cm] int8."""
    x, wq, wd2 = _i8(x), _i8(wq), _i8(wd2)
    s1, b1, s2, b2 = map(_f32, (s1, b1, s2, b2))
    N, H, W, C = x.shape
    Cm, k = wd2.shape[0], wd2.shape[1]
    assert wq.shape == (Cm, C) and wd2.shape == (Cm, k, k)
    assert all(v.shape == (Cm,) for v in (s1, b1, s2, b2))
    Ho, Wo = out_extent(H, k, stride, pad), out_extent(W, k, stride, pad)
    y = np.empty((N, Ho, Wo, Cm), np.int8)
    rc = _load(lib).oracle_pwdw_i8(N, H, W, C, Cm, k, stride, pad, _p8(x), _p8(wq), _p32(s1),
                                   _p32(b1), ACT[act1], _p8(wd2), _p32(s2), _p32(b2), ACT[act2],
                                   _p8(y), nthreads)
    if rc != 0:
        raise ValueError("oracle_pwdw_i8: invalid shape")
    return y


def round_format(v: float, prec: int, emin: int, maxf: float, lib=None) -> float:
    """Round to nearest, ties to even, into a binary format (used by the mirror mode)."""
    return float(_load(lib).oracle_round_format(float(v), prec, emin, float(maxf)))


def build_variant(src_text: str, out_path: str) -> str:
    """Compile C source text (e.g. a deliberately mutated copy of fcm_oracle.c, used by the
    tests that show the pins catch planted mistakes) into `out_path`."""
    c_path = out_path[:-3] + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", c_path, "-o", out_path, "-lm"],
                   check=True, capture_output=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()
