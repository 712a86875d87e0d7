"""Pins of the fp64 oracle to things other than itself (CPU only).

* hand-computed examples (tests/golden/*.json, derivations inside);
* library routines the definitions reduce to: torch.nn.functional.conv2d in float64
  (grouped for depthwise, 1x1 for pointwise, dense for the back-to-back conv1) and
  scipy.signal.correlate2d per channel;
* closed forms and invariants: delta filter + identity 1x1 reproduces act(x); linearity;
  fused == pointwise(depthwise(x)) exactly on integer data;
* the mirror rounding against numpy's float16 and torch's bfloat16 conversions;
* planted mistakes: mutated copies of the oracle source must fail at least one pin.
"""
import json
import os

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
F = torch.nn.functional

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ACT_T = {"none": lambda t: t, "relu": F.relu, "relu6": F.relu6}


def rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ library formulations
def lib_dw(x, wd, s1, b1, act, stride, pad):
    """DW conv + norm + act via torch conv2d(groups=C), NHWC in/out, float64."""
    xt = torch.from_numpy(np.ascontiguousarray(x.transpose(0, 3, 1, 2)))
    C = x.shape[3]
    w = torch.from_numpy(wd[:, None, :, :] * s1[:, None, None, None])
    y = F.conv2d(xt, w, torch.from_numpy(b1), stride=stride, padding=pad, groups=C)
    return ACT_T[act](y).numpy().transpose(0, 2, 3, 1)


def lib_dense(x, w1, s1, b1, act, stride, pad):
    xt = torch.from_numpy(np.ascontiguousarray(x.transpose(0, 3, 1, 2)))
    w = torch.from_numpy(np.ascontiguousarray(w1.transpose(0, 3, 1, 2)) * s1[:, None, None, None])
    y = F.conv2d(xt, w, torch.from_numpy(b1), stride=stride, padding=pad)
    return ACT_T[act](y).numpy().transpose(0, 2, 3, 1)


def lib_pw(m, wp, s2, b2, act):
    mt = torch.from_numpy(np.ascontiguousarray(m.transpose(0, 3, 1, 2)))
    w = torch.from_numpy(wp[:, :, None, None] * s2[:, None, None, None])
    y = F.conv2d(mt, w, torch.from_numpy(b2))
    return ACT_T[act](y).numpy().transpose(0, 2, 3, 1)


def close(a, b, tol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape
    scale = max(1.0, float(np.abs(b).max(initial=0.0)))
    return float(np.abs(a - b).max(initial=0.0)) <= tol * scale


DW_CASES = [  # N, H, W, C, k, s, p, act
    (1, 1, 1, 1, 1, 1, 0, "none"), (1, 2, 3, 2, 3, 1, 1, "relu"), (1, 5, 5, 8, 3, 2, 1, "relu6"),
    (2, 5, 4, 3, 5, 1, 2, "none"), (1, 3, 5, 2, 5, 2, 2, "relu"), (1, 6, 7, 4, 3, 2, 0, "none"),
    (1, 7, 7, 2, 7, 1, 3, "relu6"), (1, 4, 4, 1, 2, 1, 0, "none"),
]


def draw_dw(case, seed):
    N, H, W, C, k, s, p, act = case
    r = rng(seed)
    x = r.uniform(-2, 2, (N, H, W, C))
    wd = r.uniform(-1, 1, (C, k, k))
    s1 = r.uniform(0.5, 1.5, C)
    b1 = r.uniform(-0.5, 0.5, C)
    return x, wd, s1, b1


def pin_dw(lib=None):
    for i, case in enumerate(DW_CASES):
        N, H, W, C, k, s, p, act = case
        x, wd, s1, b1 = draw_dw(case, 100 + i)
        got = oracle.dw(x, wd, s1, b1, act, s, p, lib=lib)
        if not close(got, lib_dw(x, wd, s1, b1, act, s, p)):
            return False
    return True


def pin_pw(lib=None):
    r = rng(7)
    for (N, Ho, Wo, Cm, K, act) in [(1, 1, 1, 1, 1, "none"), (2, 3, 4, 5, 7, "relu"),
                                    (1, 4, 2, 16, 3, "relu6")]:
        m = r.uniform(-2, 2, (N, Ho, Wo, Cm))
        wp = r.uniform(-1, 1, (K, Cm))
        s2, b2 = r.uniform(0.5, 1.5, K), r.uniform(-0.5, 0.5, K)
        if not close(oracle.pw(m, wp, s2, b2, act, lib=lib), lib_pw(m, wp, s2, b2, act)):
            return False
    return True


def pin_dense(lib=None):
    r = rng(11)
    for (N, H, W, C, K1, k, s, p, act) in [(1, 3, 3, 2, 3, 3, 1, 1, "none"),
                                           (2, 5, 6, 3, 4, 3, 2, 1, "relu"),
                                           (1, 4, 5, 4, 2, 5, 1, 2, "relu6"),
                                           (1, 3, 4, 2, 2, 1, 1, 0, "none")]:
        x = r.uniform(-2, 2, (N, H, W, C))
        w1 = r.uniform(-1, 1, (K1, k, k, C))
        s1, b1 = r.uniform(0.5, 1.5, K1), r.uniform(-0.5, 0.5, K1)
        if not close(oracle.dense(x, w1, s1, b1, act, s, p, lib=lib),
                     lib_dense(x, w1, s1, b1, act, s, p)):
            return False
    return True


def pin_fused(lib=None):
    r = rng(13)
    for conv1, (N, H, W, C, Cm, K, k, s, p, a1, a2) in [
            ("dw", (1, 5, 5, 3, 3, 4, 3, 1, 1, "relu", "relu6")),
            ("dw", (2, 6, 5, 4, 4, 2, 5, 2, 2, "relu6", "none")),
            ("dw", (1, 4, 3, 2, 2, 3, 3, 2, 0, "none", "relu")),
            ("dense", (1, 5, 4, 3, 2, 3, 3, 1, 1, "relu", "relu")),
            ("dense", (2, 6, 6, 2, 3, 2, 3, 2, 1, "none", "relu6"))]:
        x = r.uniform(-2, 2, (N, H, W, C))
        w1 = r.uniform(-1, 1, (C, k, k) if conv1 == "dw" else (Cm, k, k, C))
        s1, b1 = r.uniform(0.5, 1.5, Cm), r.uniform(-0.5, 0.5, Cm)
        wp = r.uniform(-1, 1, (K, Cm))
        s2, b2 = r.uniform(0.5, 1.5, K), r.uniform(-0.5, 0.5, K)
        mid = (lib_dw(x, w1, s1, b1, a1, s, p) if conv1 == "dw"
               else lib_dense(x, w1, s1, b1, a1, s, p))
        want = lib_pw(mid, wp, s2, b2, a2)
        got = oracle.fused(x, w1, s1, b1, wp, s2, b2, a1, a2, s, p, conv1=conv1, lib=lib)
        if not close(got, want):
            return False
    return True


def pin_golden_dw(lib=None):
    g = json.load(open(os.path.join(GOLDEN, "dw3x3_s2p1_hand.json")))
    x = np.array(g["x_hw"], float)[None, :, :, None]
    wd = np.array(g["wd_kk"], float)[None]
    raw = oracle.dw(x, wd, [1.0], [0.0], "none", g["stride"], g["pad"], lib=lib)[0, :, :, 0]
    m = oracle.dw(x, wd, g["s1"], g["b1"], g["act1"], g["stride"], g["pad"], lib=lib)
    y = oracle.pw(m, g["wp"], g["s2"], g["b2"], g["act2"], lib=lib)
    yf = oracle.fused(x, wd, g["s1"], g["b1"], g["wp"], g["s2"], g["b2"], g["act1"], g["act2"],
                      g["stride"], g["pad"], lib=lib)
    return (np.array_equal(raw, g["dw_raw"]) and np.array_equal(m[0, :, :, 0], g["m"])
            and np.array_equal(y[0], g["y"]) and np.array_equal(yf[0], g["y"]))


def pin_golden_dense(lib=None):
    g = json.load(open(os.path.join(GOLDEN, "dense3x3_p1_hand.json")))
    x = np.stack([np.array(g["x_c0"], float), np.array(g["x_c1"], float)], -1)[None]
    w = np.stack([np.array(g["w_c0"], float), np.array(g["w_c1"], float)], -1)[None]
    out = oracle.dense(x, w, [1.0], [0.0], "none", g["stride"], g["pad"], lib=lib)
    return np.array_equal(out[0, :, :, 0], g["out"])


def pin_delta_identity(lib=None):
    """DW filter = delta at the centre, 1x1 = identity, scales 1, biases 0: y = act2(act1(x))
    for stride 1 and pad (k-1)/2, and the stride-2 subsample x[::2, ::2] for stride 2."""
    r = rng(17)
    for k in (1, 3, 5):
        for s in (1, 2):
            C = 4
            x = r.uniform(-3, 3, (2, 7, 6, C))
            wd = np.zeros((C, k, k))
            wd[:, k // 2, k // 2] = 1.0
            eye = np.eye(C)
            one, zero = np.ones(C), np.zeros(C)
            y = oracle.fused(x, wd, one, zero, eye, one, zero, "none", "none", s, k // 2, lib=lib)
            if not np.array_equal(y, x[:, ::s, ::s, :]):
                return False
            y = oracle.fused(x, wd, one, zero, eye, one, zero, "relu", "none", s, k // 2, lib=lib)
            if not np.array_equal(y, np.maximum(x[:, ::s, ::s, :], 0.0)):
                return False
    return True


def pin_linearity(lib=None):
    r = rng(19)
    C, K, k = 3, 5, 3
    x1, x2 = r.uniform(-1, 1, (2, 1, 6, 5, C))
    wd, wp = r.uniform(-1, 1, (C, k, k)), r.uniform(-1, 1, (K, C))
    s1, s2 = r.uniform(0.5, 1.5, C), r.uniform(0.5, 1.5, K)
    z1, z2 = np.zeros(C), np.zeros(K)
    f = lambda x: oracle.fused(x, wd, s1, z1, wp, s2, z2, "none", "none", 2, 1, lib=lib)
    a, b = 1.75, -0.5
    return close(f(a * x1 + b * x2), a * f(x1) + b * f(x2), 1e-12)


def pin_composition_integers(lib=None):
    """fused == pw(dw(x)) and fused == pw(dense(x)) bit for bit on integer data."""
    r = rng(23)
    for conv1 in ("dw", "dense"):
        C, Cm, K, k = 4, (4 if conv1 == "dw" else 3), 5, 3
        x = r.integers(-3, 4, (2, 6, 7, C)).astype(float)
        w1 = r.integers(-2, 3, (C, k, k) if conv1 == "dw" else (Cm, k, k, C)).astype(float)
        b1 = r.integers(-2, 3, Cm).astype(float)
        wp = r.integers(-2, 3, (K, Cm)).astype(float)
        b2 = r.integers(-2, 3, K).astype(float)
        s1, s2 = np.ones(Cm), np.ones(K)
        for s in (1, 2):
            m = (oracle.dw(x, w1, s1, b1, "relu", s, 1, lib=lib) if conv1 == "dw"
                 else oracle.dense(x, w1, s1, b1, "relu", s, 1, lib=lib))
            y = oracle.pw(m, wp, s2, b2, "relu6", lib=lib)
            yf = oracle.fused(x, w1, s1, b1, wp, s2, b2, "relu", "relu6", s, 1, conv1=conv1,
                              lib=lib)
            if not np.array_equal(y, yf):
                return False
    return True


def lib_pwdw(x, wq, s1, b1, wd2, s2, b2, a1, a2, stride, pad):
    """1x1 conv (torch, float64) then grouped k x k conv with zero padding of the
    intermediate."""
    m = lib_pw(x, wq, s1, b1, a1)
    return lib_dw(m, wd2, s2, b2, a2, stride, pad)


PWDW_CASES = [  # N, H, W, C, Cm, k, s, p, act1, act2
    (1, 1, 1, 1, 1, 3, 1, 1, "none", "none"), (1, 5, 5, 3, 4, 3, 1, 1, "relu6", "relu6"),
    (2, 6, 5, 2, 3, 3, 2, 1, "relu", "none"), (1, 7, 6, 4, 2, 5, 1, 2, "none", "relu"),
    (1, 6, 7, 3, 5, 3, 2, 0, "relu", "relu6"), (1, 3, 4, 2, 2, 1, 1, 0, "none", "none"),
]


def pin_pwdw(lib=None):
    r = rng(41)
    for (N, H, W, C, Cm, k, s, p, a1, a2) in PWDW_CASES:
        x = r.uniform(-2, 2, (N, H, W, C))
        wq = r.uniform(-1, 1, (Cm, C))
        wd2 = r.uniform(-1, 1, (Cm, k, k))
        s1, b1 = r.uniform(0.5, 1.5, Cm), r.uniform(-0.5, 0.5, Cm)
        s2, b2 = r.uniform(0.5, 1.5, Cm), r.uniform(-0.5, 0.5, Cm)
        got = oracle.pwdw(x, wq, s1, b1, wd2, s2, b2, a1, a2, s, p, lib=lib)
        if not close(got, lib_pwdw(x, wq, s1, b1, wd2, s2, b2, a1, a2, s, p)):
            return False
    return True


def pin_pwdw_padding_by_hand(lib=None):
    """One pixel, one channel, 3x3 depthwise with pad 1: x = 2, 1x1 weight 3, scale 1, bias 5,
    no activation -> the intermediate is 11; all taps 1, so only the centre tap is inside and
    y = 2 * 11 + 1 = 23 (scale 2, bias 1).  Padding the input instead of the intermediate
    would add act(0*3 + 5) = 5 for each of the 8 outer taps: 2 * 51 + 1 = 103."""
    y = oracle.pwdw(np.full((1, 1, 1, 1), 2.0), [[3.0]], [1.0], [5.0], np.ones((1, 3, 3)), [2.0],
                    [1.0], "none", "none", 1, 1, lib=lib)
    return y.shape == (1, 1, 1, 1) and y[0, 0, 0, 0] == 23.0


def pin_pwdw_composition_integers(lib=None):
    """pwdw == dw(pw(x)) bit for bit on integer data (both oracle paths, stride 1 and 2)."""
    r = rng(43)
    C, Cm, k = 3, 4, 3
    x = r.integers(-3, 4, (2, 6, 7, C)).astype(float)
    wq = r.integers(-2, 3, (Cm, C)).astype(float)
    wd2 = r.integers(-2, 3, (Cm, k, k)).astype(float)
    b1 = r.integers(-2, 3, Cm).astype(float)
    b2 = r.integers(-2, 3, Cm).astype(float)
    one = np.ones(Cm)
    for s in (1, 2):
        m = oracle.pw(x, wq, one, b1, "relu6", lib=lib)
        y = oracle.dw(m, wd2, one, b2, "relu", s, 1, lib=lib)
        yf = oracle.pwdw(x, wq, one, b1, wd2, one, b2, "relu6", "relu", s, 1, lib=lib)
        if not np.array_equal(y, yf):
            return False
    return True


PINS = [pin_dw, pin_pw, pin_dense, pin_fused, pin_golden_dw, pin_golden_dense,
        pin_delta_identity, pin_linearity, pin_composition_integers, pin_pwdw,
        pin_pwdw_padding_by_hand, pin_pwdw_composition_integers]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    assert pin()


def test_dw_scipy_correlate2d():
    """Second library routine: scipy.signal.correlate2d per channel (zero fill, stride 1)."""
    signal = pytest.importorskip("scipy.signal")
    r = rng(29)
    x = r.uniform(-1, 1, (1, 6, 7, 3))
    wd = r.uniform(-1, 1, (3, 3, 3))
    got = oracle.dw(x, wd, np.ones(3), np.zeros(3), "none", 1, 1)
    for c in range(3):
        want = signal.correlate2d(x[0, :, :, c], wd[c], mode="same", boundary="fill")
        assert np.allclose(got[0, :, :, c], want, rtol=0, atol=1e-13)


def test_fig1_toy_tiling_shapes():
    """Section II-D's toy: a 2x2 DW filter over a 4x4 IFM tile gives a 3x3 OFM tile."""
    x = np.ones((1, 4, 4, 1))
    out = oracle.dw(x, np.ones((1, 2, 2)), [1.0], [0.0], "none", 1, 0)
    assert out.shape == (1, 3, 3, 1) and np.all(out == 4.0)


def test_invalid_shapes_rejected():
    with pytest.raises(ValueError):
        oracle.dw(np.zeros((1, 2, 2, 1)), np.zeros((1, 5, 5)), [1.0], [0.0], "none", 1, 0)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_mirror_round_f16_matches_numpy(seed):
    r = rng(seed)
    vals = np.concatenate([r.normal(0, 1, 2000), r.normal(0, 1e-5, 500), r.uniform(-7e4, 7e4, 500),
                           [0.0, -0.0, 65504.0, 65519.99, 65520.0, 2 ** -24, 2 ** -25,
                            3 * 2 ** -26, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11]])
    for v in vals:
        with np.errstate(over="ignore"):
            want = float(np.float16(v))  # numpy float64 -> float16 rounds to nearest even
        got = oracle.round_format(v, 11, -14, 65504.0)
        assert got == want or (np.isinf(got) and np.isinf(want) and np.sign(got) == np.sign(want)), v


def test_mirror_round_bf16_matches_torch():
    r = rng(5)
    vals = np.concatenate([r.normal(0, 1, 3000), r.normal(0, 1e-38, 200),
                           [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895e38]]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    maxf = float(np.ldexp(255.0, 120))
    got = np.array([oracle.round_format(float(v), 8, -126, maxf) for v in vals])
    assert np.array_equal(got, want)


def test_mirror_mode_rounds_the_intermediate():
    """mid='f16' must equal running pw on f16-rounded dw output (both oracle paths)."""
    r = rng(31)
    x = r.normal(0, 1, (1, 5, 5, 4))
    wd = r.normal(0, 0.3, (4, 3, 3))
    wp = r.normal(0, 0.5, (3, 4))
    s1, b1, s2, b2 = np.ones(4), np.zeros(4), np.ones(3), np.zeros(3)
    m = oracle.dw(x, wd, s1, b1, "relu", 1, 1)
    want = oracle.pw(m.astype(np.float16).astype(np.float64), wp, s2, b2, "none")
    got = oracle.fused(x, wd, s1, b1, wp, s2, b2, "relu", "none", 1, 1, mid="f16")
    assert np.array_equal(got, want)


# ------------------------------------------------------------------------ planted mistakes
MUTANTS = {
    "dw_filter_transposed": ("wd[((size_t)c * k + i) * k + j]", "wd[((size_t)c * k + j) * k + i]"),
    "dw_bias_dropped": ("act_apply(s1[c] * t + b1[c], act1)", "act_apply(s1[c] * t, act1)"),
    "dw_pad_sign": ("int hi = ho * s - p + i;", "int hi = ho * s + p + i;"),
    "relu6_no_clamp": ("if (v > 6.0) return 6.0;", "if (v > 6.0) return v;"),
    "relu_sign": ("return v > 0.0 ? v : 0.0;", "return v < 0.0 ? v : 0.0;"),
    "pw_operand_transposed": ("m[(size_t)q * Cm + c] * wp[(size_t)kk * Cm + c]",
                              "m[(size_t)q * Cm + c] * wp[(size_t)c * K + kk]"),
    "dense_taps_swapped": ("t += x[IDX4(n, hi, wi, c, H, W, C)] *\n                                     w1[IDX4(j, r, u, c, k, k, C)];",
                           "t += x[IDX4(n, hi, wi, c, H, W, C)] *\n                                     w1[IDX4(j, u, r, c, k, k, C)];"),
    "dense_stride_dropped": ("int wi = wo * s - p + u;", "int wi = wo - p + u;"),
    "fused_dw_wrong_channel": ("t += x[IDX4(n, hi, wi, j, H, W, C)] *", "t += x[IDX4(n, hi, wi, 0, H, W, C)] *"),
    "fused_pw_scale_dropped": ("y[IDX4(n, ho, wo, kk, Ho, Wo, K)] = act_apply(s2[kk] * t + b2[kk], act2);",
                               "y[IDX4(n, ho, wo, kk, Ho, Wo, K)] = act_apply(t + b2[kk], act2);"),
    "f16_round_precision": ("return oracle_round_format(v, 11, -14, 65504.0);",
                            "return oracle_round_format(v, 10, -14, 65504.0);"),
    # taps left or right of the image read act1(s1*0 + b1), as if the input were padded
    "pwdw_pads_the_input": ("                            if (wi < 0 || wi >= W) continue;\n                            double q = 0.0;",
                            "                            if (wi < 0 || wi >= W) { t += act_apply(b1[j], act1) * wd2[((size_t)j * k + i) * k + u]; continue; }\n                            double q = 0.0;"),
    "pwdw_pw_weight_transposed": ("q += x[IDX4(n, hi, wi, c, H, W, C)] * wq[(size_t)j * C + c];",
                                  "q += x[IDX4(n, hi, wi, c, H, W, C)] * wq[(size_t)c * Cm + j];"),
    "pwdw_pw_scale_dropped": ("double mval = mid_round(act_apply(s1[j] * q + b1[j], act1), mid_mode);",
                              "double mval = mid_round(act_apply(q + b1[j], act1), mid_mode);"),
    "pwdw_dw_tap_transposed": ("t += mval * wd2[((size_t)j * k + i) * k + u];",
                               "t += mval * wd2[((size_t)j * k + u) * k + i];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation anchor missing: {name}"
    lib = oracle.bind(oracle.build_variant(src.replace(old, new, 1), str(tmp_path / "mut.so")))
    failures = [p.__name__ for p in PINS if not p(lib)]
    if name == "f16_round_precision":
        # the mirror rounding is pinned by the numpy comparison instead
        got = oracle.fused(np.full((1, 1, 1, 1), 1.0 + 2 ** -10), np.ones((1, 1, 1)), [1.0], [0.0],
                           [[1.0]], [1.0], [0.0], mid="f16", lib=lib)
        failures.append("mirror") if got[0, 0, 0, 0] != float(np.float16(1.0 + 2 ** -10)) else None
    assert failures, f"no pin caught mutant {name}"
