"""The seeded input generator and storage conversions (CPU only)."""
import numpy as np
import pytest

from pointwise_conv_cnn_gb300 import workloads as wk


def test_splitmix64_reference_values():
    # splitmix64 with state 0: the first outputs of the published generator
    out = wk.splitmix64(0, np.arange(3, dtype=np.uint64))
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_deterministic_and_independent():
    a = wk.uniform01(7, 1, 1000)
    b = wk.uniform01(7, 1, 1000)
    c = wk.uniform01(7, 2, 1000)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    # element i can be regenerated alone (counter-based)
    assert wk.uniform01(7, 1, 10, offset=500)[3] == a[503]
    assert a.min() >= 0.0 and a.max() < 1.0


def test_distributions_moments():
    u = wk.uniform(3, 1, 200000, -1.0, 1.0)
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01
    z = wk.normal(3, 2, 200000, 2.0)
    assert abs(z.mean()) < 0.02 and abs(z.std() - 2.0) < 0.02
    i = wk.integers(3, 4, 50000, -3, 3)
    assert set(np.unique(i)) == set(range(-3, 4))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(0)
    v = np.concatenate([r.normal(0, 1, 10000), r.normal(0, 1e-30, 100),
                        [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wk.f32_to_bf16_bits(v), want)
    back = wk.bf16_bits_to_f32(want)
    assert np.array_equal(back, torch.from_numpy(v).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_case_shapes_and_storage(wl):
    small = wl.with_(n=1)
    case = wk.make_case(small)
    sh = small.shapes()
    assert case.x.shape == sh["x"] and case.w1.shape == sh["w1"] and case.wp.shape == sh["wp"]
    assert case.x.dtype == wk.numpy_storage_dtype(wl.dtype)
    f = case.f64()
    if wl.dist == "int8":
        # int8 over the full range; requantization scales positive, biases within +-4
        assert case.x.min() == -128 and case.x.max() == 127 and case.wp.min() == -128
        assert case.s1.dtype == np.float32 and case.s1.min() > 0 and case.s2.min() > 0
        assert np.abs(case.b1).max() <= 4.0 and np.abs(case.b2).max() <= 4.0
        return
    assert case.s1.dtype == np.float32 and case.s1.min() >= 0.5 and case.s1.max() <= 1.5
    assert np.abs(case.b2).max() <= 0.1
    if wl.dist == "normal":
        fan1, fan2 = wl.fan_in()
        assert abs(f["w1"].std() - fan1 ** -0.5) < 0.25 * fan1 ** -0.5
        assert abs(f["x"].std() - 1.0) < 0.05
    else:
        assert np.abs(f["x"]).max() <= 1.0


def test_integer_case_exactness():
    wl = wk.BY_NAME["mobilenet_dwpw_f16"].with_(n=1, h=8, w=8)
    case = wk.make_case(wl, kind="integer")
    f = case.f64()
    assert np.all(f["x"] == np.round(f["x"])) and np.abs(f["x"]).max() <= 3
    assert wk.integer_safe(wl)
    assert not wk.integer_safe(wk.BY_NAME["b2b_dense3x3_f16"])   # 9*64*6 > 2^11
    assert wk.integer_safe(wk.BY_NAME["b2b_dense3x3_f16"], "integer1")   # 9*64*1 + 2 < 2^11
    c1 = wk.make_case(wk.BY_NAME["b2b_dense3x3_f16"].with_(n=1, h=4, w=4), kind="integer1")
    assert set(np.unique(c1.f64()["x"])) <= {-1.0, 0.0, 1.0}


def test_min_bytes_closed_form():
    # config 2 (MobileNet): in + out = 2 * 64*56*56*128*2 bytes; unfused adds 2x the mid
    wl = wk.BY_NAME["mobilenet_dwpw_f16"]
    b = wl.min_bytes()
    io = 64 * 56 * 56 * 128 * 2
    assert b["x"] == io and b["y"] == io
    assert b["fused"] == 2 * io + (128 * 9 + 128 * 128) * 2 + 4 * (2 * 128 + 2 * 128)
    assert b["unfused"] - b["fused"] == 2 * io
