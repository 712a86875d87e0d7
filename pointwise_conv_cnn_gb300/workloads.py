"""Seeded synthetic workloads: layer shapes and counter-based input generators.

This module is shared by the oracle side (tests, CPU baseline) and the CUDA side (tests,
benchmark) and holds none of the convolution arithmetic: it only draws numbers, rounds them to
the storage format and describes the five layer shapes.

Layer shapes stand in for the workloads of "Fusing Depthwise and Pointwise Convolutions for
Efficient Inference on GPUs" (section V-B: DW/PW pairs of MobileNet-style depthwise separable
blocks) and of "Fusing two back-to-back convolutions" (the ResNet-50 56x56x64 3x3 -> 1x1 pair).
No dataset and no trained weights are used.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) evaluated at counter n: value = mix(seed + (n + 1) * golden), with the
counter n = (tensor_id << 40) + element index, so every tensor has its own stream and any
element can be regenerated alone.  Uniform values take the top 53 bits; normals use the
Box-Muller transform of two uniforms (the cosine branch only).  Values are drawn in float64,
rounded to float32 and then, round-to-nearest-even, to the storage format (f16 or bf16).
Scales and biases stay float32.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "i8": 1}
BASE_SEED = 20240430


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """splitmix64 output for each counter (uint64 array), state = seed + (n+1)*golden."""
    z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (counters.astype(np.uint64) + np.uint64(1)) * _GOLDEN
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform01(seed: int, tensor_id: int, count: int, offset: int = 0) -> np.ndarray:
    """count uniforms in [0, 1) from stream `tensor_id`, starting at element `offset`."""
    out = np.empty(count, np.float64)
    base = (tensor_id << 40) + offset
    for lo in range(0, count, _CHUNK):
        hi = min(count, lo + _CHUNK)
        ctr = np.arange(base + lo, base + hi, dtype=np.uint64)
        out[lo:hi] = (splitmix64(seed, ctr) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return out


def uniform(seed: int, tensor_id: int, count: int, lo: float, hi: float) -> np.ndarray:
    return lo + (hi - lo) * uniform01(seed, tensor_id, count)


def normal(seed: int, tensor_id: int, count: int, std: float = 1.0) -> np.ndarray:
    """Box-Muller (cosine branch): element i uses uniforms 2i and 2i+1 of the stream."""
    out = np.empty(count, np.float64)
    for lo in range(0, count, _CHUNK):
        hi = min(count, lo + _CHUNK)
        u = uniform01(seed, tensor_id, 2 * (hi - lo), offset=2 * lo)
        u1, u2 = u[0::2], u[1::2]
        out[lo:hi] = np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2) * std
    return out


def integers(seed: int, tensor_id: int, count: int, lo: int, hi: int) -> np.ndarray:
    """Uniform integers in [lo, hi] (inclusive), as float64."""
    u = uniform01(seed, tensor_id, count)
    return np.floor(lo + (hi - lo + 1) * u).clip(lo, hi)


# ---------------------------------------------------------------------------- storage formats
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    r = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64/float32 values to the storage format (RN-even through float32)."""
    a32 = np.asarray(a, dtype=np.float32)
    if dtype == "f32":
        return a32
    if dtype == "f16":
        return a32.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(a32)
    if dtype == "i8":
        a = np.asarray(a, dtype=np.float64)
        if not np.array_equal(a, np.rint(a)) or a.min(initial=0) < -128 or a.max(initial=0) > 127:
            raise ValueError("int8 storage takes integers in [-128, 127]")
        return a.astype(np.int8)
    raise ValueError(dtype)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of storage values (f32 / f16 / bf16 bit patterns) to float64."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def numpy_storage_dtype(dtype: str):
    return {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "i8": np.int8}[dtype]


# ---------------------------------------------------------------------------- layer shapes
@dataclass(frozen=True)
class Workload:
    """One fused layer pair.  conv1 is "dw" (weights [C,k,k]) or "dense" (weights
    [Cm,k,k,C]) followed by the 1x1 conv with weights [K,Cm]; or "pwdw": a 1x1 conv with
    weights [Cm,C] followed by a depthwise k x k conv with weights [Cm,k,k] (K = Cm).
    Activations are NHWC."""
    name: str
    n: int
    h: int
    w: int
    c: int
    k_out: int
    conv1: str
    ksize: int
    stride: int
    pad: int
    act1: str
    act2: str
    dtype: str
    dist: str
    mid: int = 0          # first convolution's output channels (0: equal to c)

    @property
    def cm(self) -> int:
        return self.c if self.conv1 == "dw" or self.mid == 0 else self.mid

    @property
    def ho(self) -> int:
        return (self.h + 2 * self.pad - self.ksize) // self.stride + 1

    @property
    def wo(self) -> int:
        return (self.w + 2 * self.pad - self.ksize) // self.stride + 1

    @property
    def esize(self) -> int:
        return DTYPE_BYTES[self.dtype]

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def shapes(self) -> dict:
        k, C, Cm, K = self.ksize, self.c, self.cm, self.k_out
        if self.conv1 == "pwdw":
            return {"x": (self.n, self.h, self.w, C), "w1": (Cm, C), "wp": (Cm, k, k),
                    "s1": (Cm,), "b1": (Cm,), "s2": (Cm,), "b2": (Cm,),
                    "y": (self.n, self.ho, self.wo, Cm), "m": (self.n, self.h, self.w, Cm)}
        w1 = (C, k, k) if self.conv1 == "dw" else (Cm, k, k, C)
        return {"x": (self.n, self.h, self.w, C), "w1": w1, "wp": (K, Cm),
                "s1": (Cm,), "b1": (Cm,), "s2": (K,), "b2": (K,),
                "y": (self.n, self.ho, self.wo, K), "m": (self.n, self.ho, self.wo, Cm)}

    def fan_in(self) -> tuple[int, int]:
        k = self.ksize
        if self.conv1 == "pwdw":
            return self.c, k * k
        return (k * k if self.conv1 == "dw" else k * k * self.c), self.cm

    def min_bytes(self) -> dict:
        """Algorithmic bytes: every tensor moved once (input, weights, scale/bias, output);
        the unfused pair adds one write and one read of the intermediate."""
        sh = self.shapes()
        e = self.esize
        size = lambda s: int(np.prod(s))
        wbytes = (size(sh["w1"]) + size(sh["wp"])) * e
        sb = 4 * (2 * self.cm + 2 * self.k_out)
        fused = size(sh["x"]) * e + wbytes + sb + size(sh["y"]) * e
        mid = size(sh["m"]) * e
        return {"fused": fused, "unfused": fused + 2 * mid, "mid": mid,
                "x": size(sh["x"]) * e, "y": size(sh["y"]) * e, "weights": wbytes + sb}

    def flops(self) -> dict:
        P = self.n * self.ho * self.wo
        k = self.ksize
        if self.conv1 == "pwdw":   # algorithmic: the 1x1 over H x W, the depthwise over Ho x Wo
            pw = 2 * self.c * self.cm * self.n * self.h * self.w
            dw = 2 * k * k * self.cm * P
            return {"conv1": pw, "pw": dw, "total": pw + dw}
        conv1 = 2 * k * k * (self.c if self.conv1 == "dw" else self.c * self.cm) * P
        if self.conv1 == "dw":
            conv1 = 2 * k * k * self.c * P
        pw = 2 * self.cm * self.k_out * P
        return {"conv1": conv1, "pw": pw, "total": conv1 + pw}


WORKLOADS = (
    Workload("tiny_dwpw_f32", 1, 14, 14, 32, 32, "dw", 3, 1, 1, "relu", "relu", "f32", "uniform"),
    Workload("mobilenet_dwpw_f16", 64, 56, 56, 128, 128, "dw", 3, 1, 1, "relu6", "relu6", "f16",
             "normal"),
    Workload("stride2_dwpw_bf16", 128, 112, 112, 64, 128, "dw", 3, 2, 1, "relu", "relu", "bf16",
             "normal"),
    Workload("wide5x5_dwpw_bf16", 128, 28, 28, 240, 80, "dw", 5, 1, 2, "relu", "none", "bf16",
             "normal"),
    Workload("b2b_dense3x3_f16", 64, 56, 56, 64, 64, "dense", 3, 1, 1, "relu", "relu", "f16",
             "normal", mid=64),
    # two 1x1 convolutions back to back (the PWPW pair): 64 -> 128 (ReLU6) -> 64 (linear)
    Workload("pwpw_f16", 64, 56, 56, 64, 64, "dense", 1, 1, 0, "relu6", "none", "f16", "normal",
             mid=128),
    # an inverted residual's expansion and depthwise layers (the PWDW pair): 1x1 64 -> 192
    # (ReLU6), then depthwise 3x3 s1 over the 192 channels (ReLU6)
    Workload("pwdw_f16", 64, 56, 56, 64, 192, "pwdw", 3, 1, 1, "relu6", "relu6", "f16", "normal",
             mid=192),
    # the MobileNet DW -> PW pair in INT8 (int8 activations and weights, fp32 requantization
    # scales); ReLU after the depthwise layer, none after the pointwise one
    Workload("mobilenet_dwpw_i8", 64, 56, 56, 128, 128, "dw", 3, 1, 1, "relu", "none", "i8",
             "int8"),
    # the PWPW pair in INT8: 1x1 64 -> 128 (ReLU), 1x1 128 -> 64 (none)
    Workload("pwpw_i8", 64, 56, 56, 64, 64, "dense", 1, 1, 0, "relu", "none", "i8", "int8",
             mid=128),
    # the PWDW pair in INT8: 1x1 64 -> 192 (ReLU), then depthwise 3x3 s1 over the 192 channels
    # (ReLU)
    Workload("pwdw_i8", 64, 56, 56, 64, 192, "pwdw", 3, 1, 1, "relu", "relu", "i8", "int8",
             mid=192),
)
BY_NAME = {w.name: w for w in WORKLOADS}


@dataclass
class Case:
    """Storage-format tensors of one workload (numpy, host)."""
    wl: Workload
    seed: int
    x: np.ndarray
    w1: np.ndarray
    wp: np.ndarray
    s1: np.ndarray
    b1: np.ndarray
    s2: np.ndarray
    b2: np.ndarray

    def f64(self) -> dict:
        d = self.wl.dtype
        return {"x": to_f64(self.x, d), "w1": to_f64(self.w1, d), "wp": to_f64(self.wp, d),
                "s1": self.s1.astype(np.float64), "b1": self.b1.astype(np.float64),
                "s2": self.s2.astype(np.float64), "b2": self.b2.astype(np.float64)}


# stream ids of the tensors of one case
_TID = {"x": 1, "w1": 2, "wp": 3, "s1": 4, "b1": 5, "s2": 6, "b2": 7}


def make_case(wl: Workload, seed: int | None = None, kind: str | None = None) -> Case:
    """Draw a case.  kind: None -> the workload's own distribution ("uniform" or "normal");
    "integer" -> small integers (x in [-3,3], weights in [-2,2]) chosen so that every partial
    sum is exact in fp32 and the intermediate is exact in the storage format (bit-exact
    checks); "integer1" -> the same with x and weights in [-1,1], for wide dense layers;
    "integer_pow2" / "integer1_pow2" -> the same with scales 1/2, 1 or 2 per channel (exact in
    every format, so that the scale of each channel is checked bit for bit too);
    "int8" -> int8 activations and weights uniform over [-128, 127] with fp32 requantization
    scales that put the intermediate's and the output's spread near 32 (their tails saturate)
    and biases uniform in [-4, 4] (int8 units)."""
    seed = BASE_SEED if seed is None else seed
    kind = wl.dist if kind is None else kind
    sh = wl.shapes()
    cnt = {name: int(np.prod(sh[name])) for name in _TID}
    fan1, fan2 = wl.fan_in()
    d = wl.dtype
    if kind in ("integer", "integer1", "integer_pow2", "integer1_pow2"):
        xr, wr = (3, 2) if kind.startswith("integer_") or kind == "integer" else (1, 1)
        x = integers(seed, _TID["x"], cnt["x"], -xr, xr)
        w1 = integers(seed, _TID["w1"], cnt["w1"], -wr, wr)
        wp = integers(seed, _TID["wp"], cnt["wp"], -wr, wr)
        if kind.endswith("_pow2"):
            s1 = np.exp2(integers(seed, _TID["s1"], cnt["s1"], -1, 1))
            s2 = np.exp2(integers(seed, _TID["s2"], cnt["s2"], -1, 1))
        else:
            s1 = np.ones(cnt["s1"])
            s2 = np.ones(cnt["s2"])
        b1 = integers(seed, _TID["b1"], cnt["b1"], -2, 2)
        b2 = integers(seed, _TID["b2"], cnt["b2"], -2, 2)
    else:
        if kind == "uniform":
            x = uniform(seed, _TID["x"], cnt["x"], -1.0, 1.0)
            w1 = uniform(seed, _TID["w1"], cnt["w1"], -1.0, 1.0)
            wp = uniform(seed, _TID["wp"], cnt["wp"], -1.0, 1.0)
        elif kind == "normal":
            x = normal(seed, _TID["x"], cnt["x"], 1.0)
            w1 = normal(seed, _TID["w1"], cnt["w1"], (1.0 / fan1) ** 0.5)
            wp = normal(seed, _TID["wp"], cnt["wp"], (1.0 / fan2) ** 0.5)
        elif kind == "int8":
            x = integers(seed, _TID["x"], cnt["x"], -128, 127)
            w1 = integers(seed, _TID["w1"], cnt["w1"], -128, 127)
            wp = integers(seed, _TID["wp"], cnt["wp"], -128, 127)
            sd = 73.9   # standard deviation of a uniform integer on [-128, 127]
            rms_m = 32.0 / 2 ** 0.5 if wl.act1 in ("relu", "relu6") else 32.0
            s1 = uniform(seed, _TID["s1"], cnt["s1"], 0.5, 1.5) * (32.0 / (sd * sd * fan1 ** 0.5))
            s2 = uniform(seed, _TID["s2"], cnt["s2"], 0.5, 1.5) * (32.0 / (rms_m * sd * fan2 ** 0.5))
            b1 = uniform(seed, _TID["b1"], cnt["b1"], -4.0, 4.0)
            b2 = uniform(seed, _TID["b2"], cnt["b2"], -4.0, 4.0)
        else:
            raise ValueError(kind)
        if kind != "int8":
            s1 = uniform(seed, _TID["s1"], cnt["s1"], 0.5, 1.5)
            b1 = uniform(seed, _TID["b1"], cnt["b1"], -0.1, 0.1)
            s2 = uniform(seed, _TID["s2"], cnt["s2"], 0.5, 1.5)
            b2 = uniform(seed, _TID["b2"], cnt["b2"], -0.1, 0.1)
    st = lambda a, name: to_storage(a.reshape(sh[name]), d)
    f32 = lambda a, name: a.reshape(sh[name]).astype(np.float32)
    return Case(wl, seed, st(x, "x"), st(w1, "w1"), st(wp, "wp"), f32(s1, "s1"), f32(b1, "b1"),
                f32(s2, "s2"), f32(b2, "b2"))


# largest magnitude up to which a format holds every integer (the "_half" entries: every
# multiple of 1/2)
_EXACT_LIM = {"f32": 1 << 24, "f16": 1 << 11, "bf16": 1 << 8, "f16_half": 1 << 10,
              "bf16_half": 1 << 7}


def integer_safe(wl: Workload, kind: str = "integer") -> bool:
    """True when the integer case of `wl` is exact end to end: fp32 partial sums stay below
    2^24 and the intermediate (|m| <= k*k*max|x*w| + 2, before the activation) is exactly
    representable in the storage format (2^8 for bf16, 2^11 for f16)."""
    if wl.dtype == "i8":
        return True   # int8 arithmetic is exact integer arithmetic at every size
    k = wl.ksize
    prod = 6 if kind in ("integer", "integer_pow2") else 1
    if kind.endswith("_pow2"):
        # scales up to 2 double the values, scales of 1/2 need one bit below the integers: check
        # the doubled sums against half the format's exact range
        prod *= 2
        wl = wl.with_(dtype={"f16": "f16_half", "bf16": "bf16_half"}.get(wl.dtype, wl.dtype))
    if wl.conv1 == "pwdw":
        # the 1x1 sum over C, then k*k depthwise products of the intermediate
        per1 = wl.c * prod + 2
        lim = _EXACT_LIM[wl.dtype]
        mid_max = min(per1, 6) if wl.act1 == "relu6" else per1
        return per1 <= lim and k * k * mid_max * (prod // 3 + 1) + 2 < (1 << 24)
    per1 = k * k * (wl.c if wl.conv1 == "dense" else 1) * prod + 2
    lim = _EXACT_LIM[wl.dtype]
    mid_max = min(per1, 6) if wl.act1 == "relu6" else per1
    return per1 < (1 << 24) and mid_max <= lim and wl.cm * mid_max * (prod // 3 + 1) + 2 < (1 << 24)
