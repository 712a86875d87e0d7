"""Thin Python binding of the FCM C ABI (``include/fcm.h``) for GB300.

Argument marshalling only: every step of the computation runs in the CUDA kernels of
``libfcm.so``.  PyTorch provides device memory and streams (``tensor.data_ptr()``,
``torch.cuda.current_stream().cuda_stream``); nothing here computes on the CPU, and a missing
library raises instead of falling back.

The functions keep the C names (``fcm_create``, ``fcm_run``, ...).  ``FusedConvModule`` wraps
a handle for convenience.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "FCM_OK", "FcmError", "FcmDesc", "FcmPlanInfo", "FusedConvModule", "load_library",
    "fcm_create", "fcm_run", "fcm_run_host", "fcm_run_host_async", "fcm_check", "fcm_plan",
    "fcm_plan_desc",
    "fcm_tensor_bytes", "fcm_destroy", "fcm_last_error", "fcm_model_overlap",
    "fcm_model_pw_gma", "fcm_model_dw_gma", "fcm_model_dwpw_gma", "fcm_model_pwdw_gma",
    "fcm_model_pwpw_gma", "fcm_fuse_plan", "FcmLayer", "FcmLayerPlan", "LAYER_KINDS", "MODULES",
    "EXPORTED_SYMBOLS",
    "fcm_run_unfused_static", "fcm_selftest_wait_timeout",
    "DTYPES", "ACTS", "MODES",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfcm.so")

FCM_OK = 0
FCM_ERR_INVALID_ARG = 1
STATUS_NAMES = {0: "FCM_OK", 1: "FCM_ERR_INVALID_ARG", 2: "FCM_ERR_UNSUPPORTED",
                3: "FCM_ERR_ALIGNMENT", 4: "FCM_ERR_SMEM_BUDGET", 5: "FCM_ERR_CUDA",
                6: "FCM_ERR_TIMEOUT", 7: "FCM_ERR_DEVICE_FAULT", 8: "FCM_ERR_NO_DEVICE"}
DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "i8": 3}
ACTS = {"none": 0, "relu": 1, "relu6": 2}
CONV1 = {"dw": 0, "dense": 1, "pwdw": 2}
MODES = {"fused": 0, "conv1": 1, "pw": 2, "unfused": 3}
KERNELS = {"auto": 0, "simt": 1, "tc": 2, "tc_roles": 3, "tc_workers": 4}

EXPORTED_SYMBOLS = (
    "fcm_create", "fcm_run", "fcm_run_host", "fcm_run_host_async", "fcm_check", "fcm_plan",
    "fcm_plan_desc", "fcm_tensor_bytes", "fcm_destroy", "fcm_last_error", "fcm_model_overlap",
    "fcm_model_pw_gma", "fcm_model_dw_gma", "fcm_model_dwpw_gma", "fcm_run_unfused_static",
    "fcm_selftest_wait_timeout",
    "fcm_model_pwdw_gma", "fcm_model_pwpw_gma", "fcm_fuse_plan",
)


class FcmError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


class FcmDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n", "h", "w", "c", "k_out", "mid", "ksize", "stride", "pad", "conv1", "dtype", "act1",
        "act2", "tile_h", "tile_w", "kernel")]


class FcmPlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "ho", "wo", "cm", "kernel", "tile_h", "tile_w", "chunk_c", "stages", "ctas", "threads",
        "smem_bytes")] + [(n, ctypes.c_longlong) for n in (
            "num_tiles", "bytes_fused_min", "bytes_unfused_min", "gma_fused_model",
            "gma_lbl_model", "overlap_elems")] + [("tc_variant", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


LAYER_KINDS = {"dw": 0, "pw": 1}
MODULES = {0: "lbl_dw", 1: "lbl_pw", 2: "dwpw", 3: "pwdw", 4: "pwpw", 5: "fused_second", -1: None}


class FcmLayer(ctypes.Structure):
    """Mirror of fcm_layer."""
    _fields_ = [(n, ctypes.c_int) for n in ("kind", "h", "w", "c", "k_out", "ksize", "stride", "pad")]


class FcmLayerPlan(ctypes.Structure):
    """Mirror of fcm_layer_plan."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "fuse_with_next", "module", "fcm_module", "tile_h", "tile_w", "tile_c", "fcm_tile_h",
        "fcm_tile_w", "fcm_tile_c", "tiles_ok", "fcm_tiles_ok")] + [("gma_lbl", ctypes.c_longlong),
                                        ("gma_fcm", ctypes.c_longlong)]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["module"] = MODULES[d["module"]]
        d["fcm_module"] = MODULES[d["fcm_module"]]
        return d


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None):
    """Load libfcm.so (built in-tree by ``pointwise_conv_cnn_gb300.build``).  Raises if the
    library is missing: there is no fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or os.environ.get("FCM_LIBRARY") or LIB_PATH
        if not os.path.exists(p):
            raise FileNotFoundError(
                f"{p} is missing: build it with `python -m pointwise_conv_cnn_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        fp = ctypes.POINTER(ctypes.c_float)
        lib.fcm_create.argtypes = [ctypes.POINTER(FcmDesc), vp, vp, vp, vp, vp, vp,
                                   ctypes.POINTER(vp)]
        lib.fcm_run.argtypes = [vp, i, vp, vp, vp]
        lib.fcm_run_host.argtypes = [vp, i, vp, vp, vp]
        lib.fcm_run_host_async.argtypes = [vp, i, vp, vp, vp]
        lib.fcm_run_unfused_static.argtypes = [vp, vp, vp, vp]
        lib.fcm_check.argtypes = [vp, vp]
        lib.fcm_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong]
        lib.fcm_plan.argtypes = [vp, ctypes.POINTER(FcmPlanInfo)]
        lib.fcm_plan_desc.argtypes = [ctypes.POINTER(FcmDesc), i, i, ctypes.POINTER(FcmPlanInfo)]
        lib.fcm_tensor_bytes.argtypes = [ctypes.POINTER(FcmDesc)] + [ctypes.POINTER(ctypes.c_size_t)] * 3
        for f in ("fcm_create", "fcm_run", "fcm_run_host", "fcm_run_host_async",
                  "fcm_run_unfused_static", "fcm_check", "fcm_plan",
                  "fcm_plan_desc", "fcm_tensor_bytes", "fcm_selftest_wait_timeout"):
            getattr(lib, f).restype = i
        lib.fcm_destroy.argtypes = [vp]
        lib.fcm_destroy.restype = None
        lib.fcm_last_error.argtypes = []
        lib.fcm_last_error.restype = ctypes.c_char_p
        lib.fcm_model_overlap.argtypes = [ll] * 7
        lib.fcm_model_pw_gma.argtypes = [ll] * 5
        lib.fcm_model_dw_gma.argtypes = [ll] * 7
        lib.fcm_model_dwpw_gma.argtypes = [ll] * 9
        lib.fcm_model_pwdw_gma.argtypes = [ll] * 11
        lib.fcm_model_pwpw_gma.argtypes = [ll] * 7
        for f in ("fcm_model_overlap", "fcm_model_pw_gma", "fcm_model_dw_gma",
                  "fcm_model_dwpw_gma", "fcm_model_pwdw_gma", "fcm_model_pwpw_gma"):
            getattr(lib, f).restype = ll
        lib.fcm_fuse_plan.argtypes = [ctypes.POINTER(FcmLayer), i, i, i, ll, i,
                                      ctypes.POINTER(FcmLayerPlan), ctypes.POINTER(ll)]
        lib.fcm_fuse_plan.restype = i
        del fp
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != FCM_OK:
        raise FcmError(status, fcm_last_error())


def fcm_last_error() -> str:
    return load_library().fcm_last_error().decode(errors="replace")


def make_desc(n, h, w, c, k_out, ksize, stride, pad, conv1="dw", dtype="f16", act1="relu",
              act2="relu", mid=0, tile_h=0, tile_w=0, kernel="auto") -> FcmDesc:
    return FcmDesc(n, h, w, c, k_out, mid, ksize, stride, pad, CONV1[conv1], DTYPES[dtype],
                   ACTS[act1], ACTS[act2], tile_h, tile_w, KERNELS[kernel])


def desc_from_workload(wl, **over) -> FcmDesc:
    kw = dict(n=wl.n, h=wl.h, w=wl.w, c=wl.c, k_out=wl.k_out, ksize=wl.ksize, stride=wl.stride,
              pad=wl.pad, conv1=wl.conv1, dtype=wl.dtype, act1=wl.act1, act2=wl.act2,
              mid=wl.mid if wl.conv1 in ("dense", "pwdw") else 0)
    kw.update(over)
    return make_desc(**kw)


def fcm_create(desc: FcmDesc, w1: int, wp: int, s1: int, b1: int, s2: int, b2: int) -> int:
    """Raw C call; pointers are integers (host or device addresses).  Returns the handle."""
    out = ctypes.c_void_p()
    _check(load_library().fcm_create(ctypes.byref(desc), w1, wp, s1, b1, s2, b2,
                                     ctypes.byref(out)))
    return out.value


def fcm_run(handle: int, mode: int, inp: int, out: int, stream: int = 0) -> None:
    _check(load_library().fcm_run(handle, mode, inp, out, stream))


def fcm_run_host(handle: int, mode: int, host_in: int, host_out: int, stream: int = 0) -> None:
    _check(load_library().fcm_run_host(handle, mode, host_in, host_out, stream))


def fcm_run_host_async(handle: int, mode: int, host_in: int, host_out: int,
                       stream: int = 0) -> None:
    _check(load_library().fcm_run_host_async(handle, mode, host_in, host_out, stream))


def fcm_run_unfused_static(handle: int, inp: int, out: int, stream: int = 0) -> None:
    """Layer-by-layer evaluation with the intermediate in the library's fixed device array:
    allocates nothing (for callers that cannot call cudaMalloc); see include/fcm.h."""
    _check(load_library().fcm_run_unfused_static(handle, inp, out, stream))


def fcm_check(handle: int, stream: int = 0) -> None:
    _check(load_library().fcm_check(handle, stream))


def fcm_selftest_wait_timeout(limit_ns: int) -> None:
    """Make one bounded device wait run out (see include/fcm.h); raises FcmError with status
    FCM_ERR_TIMEOUT (6) when the failure detection works as designed."""
    _check(load_library().fcm_selftest_wait_timeout(int(limit_ns)))


def fcm_plan(handle: int) -> dict:
    info = FcmPlanInfo()
    _check(load_library().fcm_plan(handle, ctypes.byref(info)))
    return info.as_dict()


def fcm_plan_desc(desc: FcmDesc, num_sms: int = 152, smem_per_block: int = 232448) -> dict:
    info = FcmPlanInfo()
    _check(load_library().fcm_plan_desc(ctypes.byref(desc), num_sms, smem_per_block,
                                        ctypes.byref(info)))
    return info.as_dict()


def fcm_tensor_bytes(desc: FcmDesc) -> tuple[int, int, int]:
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().fcm_tensor_bytes(ctypes.byref(desc), ctypes.byref(a),
                                           ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def fcm_destroy(handle: int) -> None:
    if handle:
        load_library().fcm_destroy(handle)


def fcm_model_overlap(*a) -> int:
    return load_library().fcm_model_overlap(*a)


def fcm_model_pw_gma(*a) -> int:
    return load_library().fcm_model_pw_gma(*a)


def fcm_model_dw_gma(*a) -> int:
    return load_library().fcm_model_dw_gma(*a)


def fcm_model_dwpw_gma(*a) -> int:
    return load_library().fcm_model_dwpw_gma(*a)


def fcm_model_pwdw_gma(*a) -> int:
    return load_library().fcm_model_pwdw_gma(*a)


def fcm_model_pwpw_gma(*a) -> int:
    return load_library().fcm_model_pwpw_gma(*a)


def fcm_fuse_plan(layers, batch: int = 1, num_sms: int = 152, l1_bytes: int = 232448,
                  elem_bytes: int = 2) -> tuple[list[dict], int]:
    """FusePlanner over a chain of layers.  Each layer is a dict with kind ("dw" or "pw"),
    h, w, c, and k_out (PW) or ksize/stride/pad (DW).  Returns the per-layer plans and the
    chain total (elements per image)."""
    n = len(layers)
    arr = (FcmLayer * n)()
    for i, L in enumerate(layers):
        arr[i] = FcmLayer(LAYER_KINDS[L["kind"]], L["h"], L["w"], L["c"], L.get("k_out", 0),
                          L.get("ksize", 1), L.get("stride", 1), L.get("pad", 0))
    out = (FcmLayerPlan * n)()
    total = ctypes.c_longlong()
    _check(load_library().fcm_fuse_plan(arr, n, batch, num_sms, l1_bytes, elem_bytes, out,
                                        ctypes.byref(total)))
    return [o.as_dict() for o in out], total.value


def mode_bytes(desc: FcmDesc) -> dict[int, tuple[int, int]]:
    """Bytes each fcm_run mode reads and writes: {mode: (input bytes, output bytes)}."""
    x, m, y = fcm_tensor_bytes(desc)
    return {MODES["fused"]: (x, y), MODES["conv1"]: (x, m), MODES["pw"]: (m, y),
            MODES["unfused"]: (x, y)}


def check_run_buffers(need: dict, mode: int, inp, out, on_device: bool) -> None:
    """Refuse tensors the library would read or write past: the C ABI takes bare pointers, so
    the binding checks what only it can see -- device, contiguity and size."""
    sizes = need.get(mode)
    if sizes is None:
        raise FcmError(FCM_ERR_INVALID_ARG, f"mode {mode}")
    if (inp.is_cuda == on_device and out.is_cuda == on_device and inp.is_contiguous()
            and out.is_contiguous() and inp.nbytes >= sizes[0] and out.nbytes >= sizes[1]):
        return
    where = "a CUDA" if on_device else "a host"
    for t, nbytes, what in ((inp, sizes[0], "input"), (out, sizes[1], "output")):
        if bool(t.is_cuda) != on_device:
            raise FcmError(FCM_ERR_INVALID_ARG, f"{what} must be {where} tensor")
        if not t.is_contiguous():
            raise FcmError(FCM_ERR_INVALID_ARG, f"{what} must be contiguous (NHWC)")
        if t.nbytes < nbytes:
            raise FcmError(FCM_ERR_INVALID_ARG,
                           f"{what} holds {t.nbytes} bytes; the mode needs {nbytes}")


class FusedConvModule:
    """Owns one FCM handle.  Weights are torch tensors or numpy arrays in the storage dtype
    (bf16 may be given as uint16 bit patterns, INT8 as int8); scales/biases float32."""

    def __init__(self, desc: FcmDesc, w1, wp, s1, b1, s2, b2):
        import numpy as np
        self.desc = desc
        keep = []

        def addr(a):
            if hasattr(a, "data_ptr"):
                t = a.contiguous()
                keep.append(t)
                return t.data_ptr()
            arr = np.ascontiguousarray(a)
            keep.append(arr)
            return arr.ctypes.data

        self.handle = fcm_create(desc, addr(w1), addr(wp), addr(s1), addr(b1), addr(s2),
                                 addr(b2))
        self.plan = fcm_plan(self.handle)
        self.mode_bytes = mode_bytes(desc)
        self._streams = set()   # streams work was enqueued on (waited for before destroying)

    def run(self, inp, out, mode: str | int = "fused", stream=None) -> None:
        """Enqueue on `stream` (torch.cuda.Stream, raw handle int, or None = current stream).
        `inp`/`out` are contiguous CUDA tensors holding at least the mode's bytes."""
        import torch
        m = MODES[mode] if isinstance(mode, str) else mode
        check_run_buffers(self.mode_bytes, m, inp, out, on_device=True)
        if stream is None:
            s = torch.cuda.current_stream().cuda_stream
        elif hasattr(stream, "cuda_stream"):
            s = stream.cuda_stream
        else:
            s = int(stream)
        self._streams.add(s)
        fcm_run(self.handle, m, inp.data_ptr(), out.data_ptr(), s)

    def run_host(self, host_in, host_out, mode: str | int = "fused", stream=None) -> None:
        """`host_in`/`host_out`: contiguous host tensors (pinned for overlapped copies)."""
        import torch
        m = MODES[mode] if isinstance(mode, str) else mode
        check_run_buffers(self.mode_bytes, m, host_in, host_out, on_device=False)
        s = (torch.cuda.current_stream().cuda_stream if stream is None
             else getattr(stream, "cuda_stream", stream))
        fcm_run_host(self.handle, m, host_in.data_ptr(), host_out.data_ptr(), s)

    def run_host_async(self, host_in, host_out, mode: str | int = "fused", stream=None) -> None:
        """fcm_run_host_async: enqueue without waiting; `host_out` holds the result once `stream`
        has completed.  Keep both tensors alive and unchanged until then."""
        import torch
        m = MODES[mode] if isinstance(mode, str) else mode
        check_run_buffers(self.mode_bytes, m, host_in, host_out, on_device=False)
        s = (torch.cuda.current_stream().cuda_stream if stream is None
             else getattr(stream, "cuda_stream", stream))
        self._streams.add(s)
        fcm_run_host_async(self.handle, m, host_in.data_ptr(), host_out.data_ptr(), s)

    def check(self, stream=None) -> None:
        import torch
        s = (torch.cuda.current_stream().cuda_stream if stream is None
             else getattr(stream, "cuda_stream", stream))
        fcm_check(self.handle, s)

    def close(self) -> None:
        """Wait for the work enqueued through run() on its streams, then free the handle
        (fcm_destroy waits only for the handle's own copy streams)."""
        if getattr(self, "handle", None):
            if self._streams:
                import torch
                for s in self._streams:
                    torch.cuda.ExternalStream(s).synchronize()
                self._streams.clear()
            fcm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
