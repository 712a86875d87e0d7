"""Pins of the INT8 oracle (section III-B's INT8 FCMs) to things other than itself (CPU only).

* a hand-computed example, with ties that round to even and a saturating output;
* the requantization against an independent numpy formulation: the fp32 fused multiply-add
  emulated exactly in float64 (the product of two 24-bit significands is exact in float64,
  and only samples whose float64 sum is exact -- TwoSum error zero -- are kept, so the one
  rounding to float32 is the fma's), then numpy's round-half-even and a clip; on values drawn
  next to the rounding ties;
* the convolutions against a direct numpy formulation in int64 (sliding windows of the
  zero-padded input, an integer matrix product for the 1x1);
* fused == pointwise(depthwise(x)) exactly (the single-pass function against the two layer
  functions), and the PWDW module == depthwise(pointwise(x)) likewise, with a hand case that
  separates padding the intermediate from padding the input;
* planted mistakes in a copy of the oracle source must fail at least one pin.
"""
import numpy as np
import pytest

import oracle

ACT_NP = {"none": lambda v: v, "relu": lambda v: np.maximum(v, 0.0),
          "relu6": lambda v: np.minimum(np.maximum(v, 0.0), 6.0)}


def rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ independent formulation
def fma32_exact(s, acc, b):
    """float32 fma(s, acc, b) for float32 s, b and integer acc (|acc| < 2^24), with a mask of
    the samples where the float64 evaluation is exact (the others are not used)."""
    s64 = np.asarray(s, np.float32).astype(np.float64)
    b64 = np.asarray(b, np.float32).astype(np.float64)
    p = s64 * np.asarray(acc, np.float64)          # exact: 24 x 24 significand bits
    tot = p + b64
    bb = tot - p                                   # TwoSum (Knuth): err == 0 <=> tot exact
    err = (p - (tot - bb)) + (b64 - bb)
    return tot.astype(np.float32), err == 0.0


def requant_np(acc, s, b, act):
    v, exact = fma32_exact(s, acc, b)
    q = np.clip(np.rint(ACT_NP[act](v.astype(np.float64))), -128, 127)
    return q.astype(np.int8), exact


def dw_np(x, wd, s1, b1, act, stride, pad):
    N, H, W, C = x.shape
    k = wd.shape[1]
    Ho, Wo = (H + 2 * pad - k) // stride + 1, (W + 2 * pad - k) // stride + 1
    xp = np.zeros((N, H + 2 * pad, W + 2 * pad, C), np.int64)
    xp[:, pad:pad + H, pad:pad + W, :] = x
    acc = np.zeros((N, Ho, Wo, C), np.int64)
    for i in range(k):
        for j in range(k):
            win = xp[:, i:i + (Ho - 1) * stride + 1:stride, j:j + (Wo - 1) * stride + 1:stride, :]
            acc += win * wd[:, i, j].astype(np.int64)
    q, exact = requant_np(acc, np.broadcast_to(s1, acc.shape), np.broadcast_to(b1, acc.shape), act)
    assert exact.all()
    return q


def pw_np(m, wp, s2, b2, act):
    acc = m.astype(np.int64) @ wp.astype(np.int64).T
    q, exact = requant_np(acc, np.broadcast_to(s2, acc.shape), np.broadcast_to(b2, acc.shape), act)
    assert exact.all()
    return q


def draw(r, N, H, W, C, K, k):
    x = r.integers(-128, 128, (N, H, W, C)).astype(np.int8)
    wd = r.integers(-128, 128, (C, k, k)).astype(np.int8)
    wp = r.integers(-128, 128, (K, C)).astype(np.int8)
    s1 = (r.uniform(0.5, 1.5, C) * 32 / (5461 * k)).astype(np.float32)
    b1 = r.uniform(-4, 4, C).astype(np.float32)
    s2 = (r.uniform(0.5, 1.5, K) * 32 / (74 * 23 * np.sqrt(C))).astype(np.float32)
    b2 = r.uniform(-4, 4, K).astype(np.float32)
    return x, wd, wp, s1, b1, s2, b2


CASES = [  # (N, H, W, C, K, k, stride, pad, act1, act2)
    (1, 5, 6, 3, 4, 3, 1, 1, "relu", "none"),
    (2, 7, 5, 4, 2, 3, 2, 1, "none", "relu6"),
    (1, 6, 6, 2, 3, 5, 1, 2, "relu6", "relu"),
    (1, 4, 9, 5, 3, 1, 1, 0, "relu", "relu"),
    (1, 9, 7, 3, 2, 5, 2, 1, "none", "none"),
]


# --------------------------------------------------------------------------------- pins
def pin_i8_hand(lib=None):
    """x = 1..9 on a 3x3 plane (one channel), all-ones 3x3 depthwise filter, pad 1:
    accumulators 12 (corner), 21 (top row, middle), 27 (middle row, left) and 45 (centre).
    Scale 1/4, bias 0, ReLU: 3, 5.25 -> 5, 6.75 -> 7 and 11.25 -> 11.  1x1 weights (2, -3),
    scale 1, bias 0.5: at the centre 2*11 + 0.5 = 22.5 -> 22 and -33 + 0.5 = -32.5 -> -32 (ties to even); at the corner
    6.5 -> 6 and -8.5 -> -8.  Third output channel, weight 100, scale 1: 1100.5 at the centre
    saturates to 127."""
    x = np.arange(1, 10, dtype=np.int8).reshape(1, 3, 3, 1)
    y = oracle.fused_i8(x, np.ones((1, 3, 3), np.int8), [0.25], [0.0],
                        np.array([[2], [-3], [100]], np.int8), [1.0, 1.0, 1.0], [0.5, 0.5, 0.5],
                        "relu", "none", 1, 1, lib=lib)
    m = oracle.dw_i8(x, np.ones((1, 3, 3), np.int8), [0.25], [0.0], "relu", 1, 1, lib=lib)
    return (m[0, 0, 0, 0] == 3 and m[0, 0, 1, 0] == 5 and m[0, 1, 0, 0] == 7 and
            m[0, 1, 1, 0] == 11 and
            list(y[0, 1, 1]) == [22, -32, 127] and list(y[0, 0, 0]) == [6, -8, 127])


def pin_i8_requant_near_ties(lib=None):
    """Requantization of one accumulator next to its rounding ties, against numpy."""
    r = rng(7)
    n = 4000
    acc = r.integers(-(1 << 20), 1 << 20, n)
    s = (r.uniform(1.0 / 8192, 1.0 / 128, n)).astype(np.float32)
    sa = s.astype(np.float64) * acc
    target = np.rint(sa) + 0.5 + r.integers(-3, 3, n)       # near x.5 ties
    b = (target - sa + r.choice([0.0, 1e-7, -1e-7, 3e-6], n)).astype(np.float32)
    ok = True
    for act in ("none", "relu", "relu6"):
        want, exact = requant_np(acc, s, b, act)
        for i in np.flatnonzero(exact)[:1500]:
            if oracle.requant_i8(int(acc[i]), float(s[i]), float(b[i]), act, lib=lib) != want[i]:
                ok = False
    return ok


def pin_i8_requant_closed_forms(lib=None):
    """Ties to even in both signs, saturation at both ends, the activations' clamps."""
    q = lambda acc, s, b, act="none": oracle.requant_i8(acc, s, b, act, lib=lib)
    cases = [(5, 0.5, 0.0, "none", 2), (7, 0.5, 0.0, "none", 4), (-5, 0.5, 0.0, "none", -2),
             (-7, 0.5, 0.0, "none", -4), (1, 0.5, 0.0, "none", 0), (3, 0.5, 0.0, "none", 2),
             (1000, 1.0, 0.0, "none", 127), (-1000, 1.0, 0.0, "none", -128),
             (-128, 1.0, 0.0, "none", -128), (127, 1.0, 0.0, "none", 127),
             (-1000, 1.0, 0.0, "relu", 0), (13, 1.0, 0.0, "relu6", 6), (11, 0.5, 0.0, "relu6", 6),
             (-3, 1.0, 0.0, "relu6", 0), (9, 0.5, 0.0, "relu6", 4), (0, 1.0, -0.5, "none", 0),
             (0, 1.0, -1.5, "none", -2), (2, 1.0, 125.5, "none", 127),
             FMA_CASE + ("none", 1)]
    return all(q(a, s, b, act) == want for a, s, b, act, want in cases)


def pin_i8_dw_numpy(lib=None):
    r = rng(11)
    for (N, H, W, C, K, k, st, p, a1, a2) in CASES:
        x, wd, wp, s1, b1, s2, b2 = draw(r, N, H, W, C, K, k)
        if not np.array_equal(oracle.dw_i8(x, wd, s1, b1, a1, st, p, lib=lib),
                              dw_np(x, wd, s1, b1, a1, st, p)):
            return False
    return True


def pin_i8_pw_numpy(lib=None):
    r = rng(13)
    for (N, H, W, C, K, k, st, p, a1, a2) in CASES:
        x, wd, wp, s1, b1, s2, b2 = draw(r, N, H, W, C, K, k)
        if not np.array_equal(oracle.pw_i8(x, wp, s2, b2, a2, lib=lib), pw_np(x, wp, s2, b2, a2)):
            return False
    return True


def pin_i8_fused_numpy(lib=None):
    """The single-pass module against the numpy composition."""
    r = rng(17)
    for (N, H, W, C, K, k, st, p, a1, a2) in CASES:
        x, wd, wp, s1, b1, s2, b2 = draw(r, N, H, W, C, K, k)
        got = oracle.fused_i8(x, wd, s1, b1, wp, s2, b2, a1, a2, st, p, lib=lib)
        want = pw_np(dw_np(x, wd, s1, b1, a1, st, p), wp, s2, b2, a2)
        if not np.array_equal(got, want):
            return False
    return True


def pin_i8_fused_composition(lib=None):
    """fused_i8 == pw_i8(dw_i8(x)) (the oracle's own two paths)."""
    r = rng(19)
    for (N, H, W, C, K, k, st, p, a1, a2) in CASES:
        x, wd, wp, s1, b1, s2, b2 = draw(r, N, H, W, C, K, k)
        got = oracle.fused_i8(x, wd, s1, b1, wp, s2, b2, a1, a2, st, p, lib=lib)
        m = oracle.dw_i8(x, wd, s1, b1, a1, st, p, lib=lib)
        if not np.array_equal(got, oracle.pw_i8(m, wp, s2, b2, a2, lib=lib)):
            return False
    return True


def dense_np(x, w1, s1, b1, act, stride, pad):
    """Dense k x k conv in int64 (w1 [Cm,k,k,C]) from sliding windows, then requantization."""
    N, H, W, C = x.shape
    Cm, k = w1.shape[0], w1.shape[1]
    Ho, Wo = (H + 2 * pad - k) // stride + 1, (W + 2 * pad - k) // stride + 1
    xp = np.zeros((N, H + 2 * pad, W + 2 * pad, C), np.int64)
    xp[:, pad:pad + H, pad:pad + W, :] = x
    acc = np.zeros((N, Ho, Wo, Cm), np.int64)
    for i in range(k):
        for j in range(k):
            win = xp[:, i:i + (Ho - 1) * stride + 1:stride, j:j + (Wo - 1) * stride + 1:stride, :]
            acc += win @ w1[:, i, j, :].astype(np.int64).T
    q, exact = requant_np(acc, np.broadcast_to(s1, acc.shape), np.broadcast_to(b1, acc.shape), act)
    assert exact.all()
    return q


DENSE_CASES = [  # (N, H, W, C, Cm, K, k, stride, pad, act1, act2)
    (1, 5, 6, 3, 4, 2, 1, 1, 0, "relu", "none"),
    (2, 4, 7, 8, 5, 3, 1, 1, 0, "none", "relu6"),
    (1, 6, 5, 3, 4, 2, 3, 1, 1, "relu", "relu"),
    (1, 7, 7, 2, 3, 4, 3, 2, 1, "none", "none"),
]


def draw_dense(r, N, H, W, C, Cm, K, k):
    x = r.integers(-128, 128, (N, H, W, C)).astype(np.int8)
    w1 = r.integers(-128, 128, (Cm, k, k, C)).astype(np.int8)
    wp = r.integers(-128, 128, (K, Cm)).astype(np.int8)
    s1 = (r.uniform(0.5, 1.5, Cm) * 32 / (5461 * k * np.sqrt(C))).astype(np.float32)
    b1 = r.uniform(-4, 4, Cm).astype(np.float32)
    s2 = (r.uniform(0.5, 1.5, K) * 32 / (74 * 23 * np.sqrt(Cm))).astype(np.float32)
    b2 = r.uniform(-4, 4, K).astype(np.float32)
    return x, w1, wp, s1, b1, s2, b2


def pin_i8_dense_numpy(lib=None):
    """The dense layer and the single-pass dense -> 1x1 module against int64 numpy."""
    r = rng(23)
    for (N, H, W, C, Cm, K, k, st, p, a1, a2) in DENSE_CASES:
        x, w1, wp, s1, b1, s2, b2 = draw_dense(r, N, H, W, C, Cm, K, k)
        m = dense_np(x, w1, s1, b1, a1, st, p)
        if not np.array_equal(oracle.dense_i8(x, w1, s1, b1, a1, st, p, lib=lib), m):
            return False
        got = oracle.fused_dense_i8(x, w1, s1, b1, wp, s2, b2, a1, a2, st, p, lib=lib)
        if not np.array_equal(got, pw_np(m, wp, s2, b2, a2)):
            return False
    return True


def pin_i8_pwpw_composition(lib=None):
    """k = 1: the dense module is two 1x1 layers, pw_i8(pw_i8(x)) (the oracle's own paths)."""
    r = rng(29)
    for (N, H, W, C, Cm, K, k, st, p, a1, a2) in DENSE_CASES[:2]:
        x, w1, wp, s1, b1, s2, b2 = draw_dense(r, N, H, W, C, Cm, K, k)
        m = oracle.pw_i8(x, w1.reshape(Cm, C), s1, b1, a1, lib=lib)
        want = oracle.pw_i8(m, wp, s2, b2, a2, lib=lib)
        if not np.array_equal(oracle.fused_dense_i8(x, w1, s1, b1, wp, s2, b2, a1, a2, lib=lib),
                              want):
            return False
    return True


PWDW_CASES = [  # (N, H, W, C, Cm, k, stride, pad, act1, act2): 1x1 C -> Cm, then depthwise
    (1, 5, 6, 3, 4, 3, 1, 1, "relu6", "relu"),
    (2, 6, 5, 4, 3, 3, 2, 1, "none", "relu6"),
    (1, 7, 6, 2, 5, 5, 1, 2, "relu", "none"),
    (1, 4, 4, 3, 2, 1, 1, 0, "none", "none"),
]


def draw_pwdw(r, N, H, W, C, Cm, k):
    x = r.integers(-128, 128, (N, H, W, C)).astype(np.int8)
    wq = r.integers(-128, 128, (Cm, C)).astype(np.int8)
    wd2 = r.integers(-128, 128, (Cm, k, k)).astype(np.int8)
    s1 = (r.uniform(0.5, 1.5, Cm) * 32 / (74 * 74 * np.sqrt(C))).astype(np.float32)
    b1 = r.uniform(-4, 4, Cm).astype(np.float32)
    s2 = (r.uniform(0.5, 1.5, Cm) * 32 / (74 * 23 * k)).astype(np.float32)
    b2 = r.uniform(-4, 4, Cm).astype(np.float32)
    return x, wq, s1, b1, wd2, s2, b2


def pin_i8_pwdw_numpy(lib=None):
    """The INT8 PWDW module against int64 numpy: the 1x1 over the input's extent, requantized,
    then the depthwise layer over that int8 intermediate zero-padded."""
    r = rng(31)
    for (N, H, W, C, Cm, k, st, p, a1, a2) in PWDW_CASES:
        x, wq, s1, b1, wd2, s2, b2 = draw_pwdw(r, N, H, W, C, Cm, k)
        want = dw_np(pw_np(x, wq, s1, b1, a1), wd2, s2, b2, a2, st, p)
        got = oracle.pwdw_i8(x, wq, s1, b1, wd2, s2, b2, a1, a2, st, p, lib=lib)
        if not np.array_equal(got, want):
            return False
    return True


def pin_i8_pwdw_composition(lib=None):
    """pwdw_i8 == dw_i8(pw_i8(x)) (the oracle's own two layer functions)."""
    r = rng(37)
    for (N, H, W, C, Cm, k, st, p, a1, a2) in PWDW_CASES:
        x, wq, s1, b1, wd2, s2, b2 = draw_pwdw(r, N, H, W, C, Cm, k)
        m = oracle.pw_i8(x, wq, s1, b1, a1, lib=lib)
        want = oracle.dw_i8(m, wd2, s2, b2, a2, st, p, lib=lib)
        if not np.array_equal(oracle.pwdw_i8(x, wq, s1, b1, wd2, s2, b2, a1, a2, st, p, lib=lib),
                              want):
            return False
    return True


def pin_i8_pwdw_padding_by_hand(lib=None):
    """One pixel x = 2, 1x1 weight 3, bias 4: the intermediate is 3*2 + 4 = 10.  A 3x3
    all-ones depthwise filter with pad 1 sees only that pixel, so y = 10.  Padding the input
    instead (the 1x1 of a zero pixel is the bias, 4, at each of the eight border taps) would
    give 10 + 8*4 = 42."""
    y = oracle.pwdw_i8(np.full((1, 1, 1, 1), 2, np.int8), np.full((1, 1), 3, np.int8), [1.0],
                       [4.0], np.ones((1, 3, 3), np.int8), [1.0], [0.0], "none", "none", 1, 1,
                       lib=lib)
    return y.shape == (1, 1, 1, 1) and int(y[0, 0, 0, 0]) == 10


PINS = [pin_i8_hand, pin_i8_requant_near_ties, pin_i8_requant_closed_forms, pin_i8_dw_numpy,
        pin_i8_pw_numpy, pin_i8_fused_numpy, pin_i8_fused_composition, pin_i8_dense_numpy,
        pin_i8_pwpw_composition, pin_i8_pwdw_numpy, pin_i8_pwdw_composition,
        pin_i8_pwdw_padding_by_hand]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    assert pin()


# s = 1 + 2^-23, acc = 5, b = -4.5 - 2^-21: the exact s*acc + b is 0.5 + 2^-23 (a float32),
# which rounds to 1; a product rounded to float32 first (5 + 2^-21) plus b gives the tie 0.5,
# which rounds to 0.
FMA_CASE = (5, 1.0 + 2.0 ** -23, -4.5 - 2.0 ** -21)


def test_numpy_formulation_sees_fma():
    acc, s, b = FMA_CASE
    q, exact = requant_np(np.array([acc]), np.array([s], np.float32), np.array([b], np.float32),
                          "none")
    assert exact.all() and q[0] == 1
    rounded_first = np.float32(np.float32(s) * np.float32(acc)) + np.float32(b)
    assert rounded_first == np.float32(0.5) and np.rint(rounded_first) == 0


def test_int8_operands_checked():
    with pytest.raises(ValueError):
        oracle.dw_i8(np.full((1, 2, 2, 1), 200), np.ones((1, 1, 1), np.int8), [1.0], [0.0])


# ------------------------------------------------------------------------ planted mistakes
MUTANTS = {
    "round_half_away": ("double r = nearbyint(a);", "double r = round(a);"),
    "no_low_saturation": ("if (r < -128.0) r = -128.0;", ""),
    "no_high_saturation": ("if (r > 127.0) r = 127.0;", ""),
    "mul_then_add": ("float v = fmaf(s, (float)acc, b);", "float v = (float)(s * (float)acc) + b;"),
    "act_dropped": ("double a = act_apply((double)v, act);", "double a = (double)v;"),
    "dw_i8_tap_transposed": (
        "t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *\n                                 (int64_t)wd[((size_t)c * k + i) * k + j];",
        "t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *\n                                 (int64_t)wd[((size_t)c * k + j) * k + i];"),
    "fused_i8_tap_transposed": (
        "t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *\n                                     (int64_t)wd[((size_t)c * k + i) * k + j];",
        "t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *\n                                     (int64_t)wd[((size_t)c * k + j) * k + i];"),
    "pw_i8_weight_transposed": ("t += (int64_t)m[(size_t)q * Cm + c] * (int64_t)wp[(size_t)kk * Cm + c];",
                                "t += (int64_t)m[(size_t)q * Cm + c] * (int64_t)wp[(size_t)c * K + kk];"),
    "fused_i8_pw_bias_dropped": (
        "(int64_t)wp[(size_t)kk * C + c];\n                        y[IDX4(n, ho, wo, kk, Ho, Wo, K)] = requant_i8(t, s2[kk], b2[kk], act2);",
        "(int64_t)wp[(size_t)kk * C + c];\n                        y[IDX4(n, ho, wo, kk, Ho, Wo, K)] = requant_i8(t, s2[kk], 0.0f, act2);"),
    "dense_i8_taps_swapped": (
        "t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *\n                                     (int64_t)w1[IDX4(j, r, u, c, k, k, C)];",
        "t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *\n                                     (int64_t)w1[IDX4(j, u, r, c, k, k, C)];"),
    "fused_dense_i8_pw_weight_transposed": (
        "t += (int64_t)mid[j] * (int64_t)wp[(size_t)kk * Cm + j];",
        "t += (int64_t)mid[j] * (int64_t)wp[(size_t)j * K + kk];"),
    "dw_i8_pad_sign": ("int hi = ho * s - p + i;\n                        if (hi < 0 || hi >= H) continue;\n                        for (int j = 0; j < k; j++) {\n                            int wi = wo * s - p + j;\n                            if (wi < 0 || wi >= W) continue;\n                            t += (int64_t)",
                       "int hi = ho * s + p + i;\n                        if (hi < 0 || hi >= H) continue;\n                        for (int j = 0; j < k; j++) {\n                            int wi = wo * s - p + j;\n                            if (wi < 0 || wi >= W) continue;\n                            t += (int64_t)"),
    "pwdw_i8_pads_the_input": (
        "if (wi < 0 || wi >= W) continue;\n                            int64_t q = 0;\n                            for (int c = 0; c < C; c++)",
        "int64_t q = 0;\n                            if (wi >= 0 && wi < W) for (int c = 0; c < C; c++)"),
    "pwdw_i8_wq_transposed": ("(int64_t)wq[(size_t)j * C + c];", "(int64_t)wq[(size_t)c * Cm + j];"),
    "pwdw_i8_dw_taps_transposed": ("(int64_t)wd2[((size_t)j * k + i) * k + u];",
                                   "(int64_t)wd2[((size_t)j * k + u) * k + i];"),
    "pwdw_i8_mid_not_requantized": ("int8_t mval = requant_i8(q, s1[j], b1[j], act1);",
                                    "int64_t mval = q;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor missing or ambiguous: {name}"
    lib = oracle.bind(oracle.build_variant(src.replace(old, new, 1), str(tmp_path / "mut.so")))
    failures = [p.__name__ for p in PINS if not p(lib)]
    assert failures, f"no pin caught mutant {name}"
