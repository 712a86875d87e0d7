"""Randomised pins of the oracle (CPU only): shapes, strides, paddings and activations drawn by
hypothesis, each result checked against a library formulation of the same definition.

* fp64 functions: torch.nn.functional.conv2d in float64 (grouped for the depthwise
  convolution, dense for the k x k one, 1x1 for the pointwise one), composed in the module's
  order ("Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs",
  section II-B for DW and PW, section II-D for PWDW; CUTLASS discussion #208 for the
  back-to-back pair).
* INT8 functions (section III-B's INT8 FCMs): the same convolutions over integer data, which
  float64 holds exactly, and a requantization written with numpy.  Scales are powers of two
  and biases multiples of 1/4, so the fp32 fused multiply-add the oracle uses is exact and
  ``clip(rint(act(s * acc + b)))`` in float64 must agree with it element for element,
  ties to even included.
"""
import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
torch = pytest.importorskip("torch")
st = hyp.strategies
given, settings, assume = hyp.given, hyp.settings, hyp.assume
F = torch.nn.functional

ACTS = ("none", "relu", "relu6")
ACT_NP = {"none": lambda v: v, "relu": lambda v: np.maximum(v, 0.0),
          "relu6": lambda v: np.minimum(np.maximum(v, 0.0), 6.0)}
SETTINGS = dict(max_examples=60, deadline=None, derandomize=True)


@st.composite
def geometry(draw):
    """(N, H, W, k, s, p) with at least one output pixel."""
    k = draw(st.sampled_from((1, 2, 3, 5, 7)))
    s = draw(st.integers(1, 3))
    p = draw(st.integers(0, k - 1))
    N = draw(st.integers(1, 2))
    H = draw(st.integers(1, 9))
    W = draw(st.integers(1, 9))
    assume(H + 2 * p >= k and W + 2 * p >= k)
    return N, H, W, k, s, p


def nchw(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.float64).transpose(0, 3, 1, 2)))


def nhwc(t):
    return t.numpy().transpose(0, 2, 3, 1)


def t_dw(x, wd, s, p):
    C = x.shape[3]
    return nhwc(F.conv2d(nchw(x), torch.from_numpy(np.asarray(wd, np.float64)[:, None]),
                         stride=s, padding=p, groups=C))


def t_dense(x, w1, s, p):
    w = torch.from_numpy(np.ascontiguousarray(np.asarray(w1, np.float64).transpose(0, 3, 1, 2)))
    return nhwc(F.conv2d(nchw(x), w, stride=s, padding=p))


def t_pw(m, wp):
    return nhwc(F.conv2d(nchw(m), torch.from_numpy(np.asarray(wp, np.float64)[:, :, None, None])))


def norm_act(t, sc, b, act):
    return ACT_NP[act](t * sc + b)


def close(got, want, tol=1e-12):
    assert got.shape == want.shape, (got.shape, want.shape)
    scale = max(1.0, float(np.abs(want).max(initial=0.0)))
    err = float(np.abs(got - want).max(initial=0.0))
    assert err <= tol * scale, err


# ------------------------------------------------------------------------------ fp64
@settings(**SETTINGS)
@given(geometry(), st.integers(1, 6), st.integers(1, 5), st.sampled_from(ACTS),
       st.sampled_from(ACTS), st.sampled_from(("dw", "dense")), st.integers(0, 2**31 - 1))
def test_fused_matches_library_composition(g, C, K, a1, a2, conv1, seed):
    N, H, W, k, s, p = g
    r = np.random.default_rng(seed)
    Cm = C if conv1 == "dw" else int(r.integers(1, 6))
    x = r.uniform(-2, 2, (N, H, W, C))
    w1 = r.uniform(-1, 1, (C, k, k) if conv1 == "dw" else (Cm, k, k, C))
    s1, b1 = r.uniform(0.5, 1.5, Cm), r.uniform(-0.5, 0.5, Cm)
    wp = r.uniform(-1, 1, (K, Cm))
    s2, b2 = r.uniform(0.5, 1.5, K), r.uniform(-0.5, 0.5, K)

    conv = t_dw(x, w1, s, p) if conv1 == "dw" else t_dense(x, w1, s, p)
    mid = norm_act(conv, s1, b1, a1)
    want = norm_act(t_pw(mid, wp), s2, b2, a2)

    first = (oracle.dw if conv1 == "dw" else oracle.dense)(x, w1, s1, b1, a1, s, p)
    close(first, mid)
    close(oracle.pw(mid, wp, s2, b2, a2), want)
    close(oracle.fused(x, w1, s1, b1, wp, s2, b2, a1, a2, s, p, conv1=conv1), want)


@settings(**SETTINGS)
@given(geometry(), st.integers(1, 5), st.integers(1, 6), st.sampled_from(ACTS),
       st.sampled_from(ACTS), st.integers(0, 2**31 - 1))
def test_pwdw_matches_library_composition(g, C, Cm, a1, a2, seed):
    N, H, W, k, s, p = g
    r = np.random.default_rng(seed)
    x = r.uniform(-2, 2, (N, H, W, C))
    wq = r.uniform(-1, 1, (Cm, C))
    wd = r.uniform(-1, 1, (Cm, k, k))
    s1, b1 = r.uniform(0.5, 1.5, Cm), r.uniform(-0.5, 0.5, Cm)
    s2, b2 = r.uniform(0.5, 1.5, Cm), r.uniform(-0.5, 0.5, Cm)
    mid = norm_act(t_pw(x, wq), s1, b1, a1)
    want = norm_act(t_dw(mid, wd, s, p), s2, b2, a2)
    close(oracle.pwdw(x, wq, s1, b1, wd, s2, b2, a1, a2, s, p), want)


# ------------------------------------------------------------------------------ INT8
def requant(acc, sc, b, act):
    """clamp(rint(act(s*acc + b)), -128, 127) in float64 (exact for these scales/biases)."""
    return np.clip(np.rint(ACT_NP[act](acc * sc + b)), -128, 127).astype(np.int8)


def draw_norm(r, n):
    sc = np.float32(2.0) ** r.integers(-3, 2, n).astype(np.float32)
    b = (r.integers(-32, 33, n) / 4.0).astype(np.float32)
    return sc, b


@settings(**SETTINGS)
@given(geometry(), st.integers(1, 6), st.integers(1, 5), st.sampled_from(ACTS),
       st.sampled_from(ACTS), st.sampled_from(("dw", "dense")), st.integers(0, 2**31 - 1))
def test_int8_matches_library_composition(g, C, K, a1, a2, conv1, seed):
    N, H, W, k, s, p = g
    r = np.random.default_rng(seed)
    Cm = C if conv1 == "dw" else int(r.integers(1, 6))
    x = r.integers(-128, 128, (N, H, W, C)).astype(np.int8)
    w1 = r.integers(-128, 128, (C, k, k) if conv1 == "dw" else (Cm, k, k, C)).astype(np.int8)
    wp = r.integers(-128, 128, (K, Cm)).astype(np.int8)
    s1, b1 = draw_norm(r, Cm)
    s2, b2 = draw_norm(r, K)

    conv = t_dw(x, w1, s, p) if conv1 == "dw" else t_dense(x, w1, s, p)
    mid = requant(conv, s1.astype(np.float64), b1.astype(np.float64), a1)
    want = requant(t_pw(mid, wp), s2.astype(np.float64), b2.astype(np.float64), a2)

    first = (oracle.dw_i8 if conv1 == "dw" else oracle.dense_i8)(x, w1, s1, b1, a1, s, p)
    np.testing.assert_array_equal(first, mid)
    np.testing.assert_array_equal(oracle.pw_i8(mid, wp, s2, b2, a2), want)
    fused = oracle.fused_i8 if conv1 == "dw" else oracle.fused_dense_i8
    np.testing.assert_array_equal(fused(x, w1, s1, b1, wp, s2, b2, a1, a2, s, p), want)


@settings(**SETTINGS)
@given(st.integers(-2**20, 2**20), st.integers(-3, 1), st.integers(-32, 32),
       st.sampled_from(ACTS))
def test_int8_requant_single_values(acc, e, b4, act):
    sc, b = 2.0 ** e, b4 / 4.0
    want = int(requant(np.float64(acc), sc, b, act))
    assert oracle.requant_i8(acc, sc, b, act) == want


@settings(**SETTINGS)
@given(geometry(), st.integers(1, 5), st.integers(1, 6), st.sampled_from(ACTS),
       st.sampled_from(ACTS), st.integers(0, 2**31 - 1))
def test_int8_pwdw_matches_library_composition(g, C, Cm, a1, a2, seed):
    N, H, W, k, s, p = g
    r = np.random.default_rng(seed)
    x = r.integers(-128, 128, (N, H, W, C)).astype(np.int8)
    wq = r.integers(-128, 128, (Cm, C)).astype(np.int8)
    wd = r.integers(-128, 128, (Cm, k, k)).astype(np.int8)
    s1, b1 = draw_norm(r, Cm)
    s2, b2 = draw_norm(r, Cm)
    mid = requant(t_pw(x, wq), s1.astype(np.float64), b1.astype(np.float64), a1)
    want = requant(t_dw(mid, wd, s, p), s2.astype(np.float64), b2.astype(np.float64), a2)
    got = oracle.pwdw_i8(x, wq, s1, b1, wd, s2, b2, a1, a2, s, p)
    np.testing.assert_array_equal(got, want)
