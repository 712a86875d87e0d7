"""Randomised checks of the host planner (CPU only, no device): for any module description
it either returns a plan the kernels can be launched with, or refuses with a status code.

A plan must fit the launch limits of a GB300 (152 SMs, 227 KB of dynamic shared memory a
block, at most 1024 threads), cover every output pixel with its tiles, and report the byte
counts of section IV's minimum-traffic reading: input, weights, scale/bias and output once
fused, plus one write and one read of the intermediate layer by layer.  Its Eq. 1-4 estimates
for the chosen tile must equal the literal equations (oracle/planner_model.py).
"""
import pytest

import pointwise_conv_cnn_gb300 as fcm
from oracle import planner_model as pm

hyp = pytest.importorskip("hypothesis")
st = hyp.strategies
given, settings = hyp.given, hyp.settings

NUM_SMS, SMEM = 152, 232448
ESIZE = {"f32": 4, "f16": 2, "bf16": 2, "i8": 1}
# mostly multiples of 16 (the tensor-core kernels' rule), sometimes of 8, sometimes anything
CHANNELS = st.one_of(st.integers(1, 16).map(lambda i: 16 * i), st.integers(1, 16).map(lambda i: 16 * i),
                     st.sampled_from((8, 24, 40, 240, 320, 512)), st.integers(1, 300))


def out_extent(n, k, s, p):
    return (n + 2 * p - k) // s + 1


@st.composite
def descs(draw):
    conv1 = draw(st.sampled_from(("dw", "dense", "pwdw")))
    dtype = draw(st.sampled_from(("f32", "f16", "bf16", "i8")))
    k = draw(st.sampled_from((1, 3, 3, 5, 7, 2, 4, 6)))
    s = draw(st.integers(1, 2))
    p = draw(st.integers(0, k - 1))
    c = draw(CHANNELS)
    mid = c if conv1 == "dw" else draw(CHANNELS)
    k_out = mid if conv1 == "pwdw" else draw(CHANNELS)
    kw = dict(n=draw(st.integers(1, 256)), h=draw(st.integers(k, 130)),
              w=draw(st.integers(k, 130)), c=c, k_out=k_out, ksize=k, stride=s, pad=p,
              conv1=conv1, dtype=dtype, act1=draw(st.sampled_from(("none", "relu", "relu6"))),
              act2=draw(st.sampled_from(("none", "relu", "relu6"))),
              mid=0 if conv1 == "dw" else mid,
              kernel=draw(st.sampled_from(("auto", "simt", "tc"))))
    return kw


def expected_refusal(kw):
    """Requests the planner must refuse whatever the tile search finds, with their status."""
    e = ESIZE[kw["dtype"]]
    cm = kw["mid"] or kw["c"]
    if any((v * e) % 16 for v in (kw["c"], cm, kw["k_out"])):
        return 3                                     # FCM_ERR_ALIGNMENT
    if kw["dtype"] == "i8" and kw["kernel"] == "simt":
        return 2                                     # INT8 has no CUDA-core kernels
    if kw["dtype"] == "f32" and kw["kernel"] == "tc":
        return 2                                     # fp32 runs on CUDA cores
    return None


@settings(max_examples=800, deadline=None, derandomize=True)
@given(descs())
def test_plan_fits_or_refuses(kw):
    want_err = expected_refusal(kw)
    try:
        info = fcm.fcm_plan_desc(fcm.make_desc(**kw), NUM_SMS, SMEM)
    except fcm.FcmError as err:
        assert err.status in (2, 3, 4), (err.status, kw)
        if want_err is not None:
            assert err.status == want_err, (err.status, kw)
        return
    assert want_err is None, kw
    check_plan(kw, info)


@st.composite
def tc_descs(draw):
    """Descriptions inside the tensor-core kernels' shape rules (one per module kind)."""
    conv1 = draw(st.sampled_from(("dw", "dense", "pwdw")))
    dtype = draw(st.sampled_from(("f16", "bf16", "i8") if conv1 != "pwdw" else ("f16", "bf16")))
    ch16 = st.integers(1, 16).map(lambda i: 16 * i)
    if conv1 == "dw":
        k = draw(st.sampled_from((1, 3, 5, 7)))
        s = draw(st.integers(1, 2))
        c, mid, k_out = draw(ch16), 0, draw(ch16)
        w_max = 130
    elif conv1 == "dense":
        k = 1 if dtype == "i8" else draw(st.sampled_from((1, 3, 5)))
        s = 1
        c = draw(st.sampled_from((64, 128) if dtype == "i8" else (64, 128, 192, 256)))
        mid = draw(st.integers(1, 15).map(lambda i: 16 * i))
        k_out = draw(st.integers(1, 16 - mid // 16).map(lambda i: 16 * i))
        w_max = 128
    else:
        k = draw(st.sampled_from((1, 3, 5, 7)))
        s = draw(st.integers(1, 2))
        c, mid = draw(st.sampled_from((64, 128, 192, 256))), draw(st.sampled_from((64, 128, 192, 256)))
        k_out = mid
        w_max = 128
    p = 0 if (dtype == "i8" and conv1 == "dense") else draw(st.integers(0, k - 1))
    h = draw(st.integers(k, 130))
    w = draw(st.integers(max(k, 1), w_max))
    return dict(n=draw(st.integers(1, 64)), h=h, w=w, c=c, k_out=k_out, ksize=k, stride=s, pad=p,
                conv1=conv1, dtype=dtype, act1="relu", act2="none", mid=mid, kernel="tc")


@settings(max_examples=600, deadline=None, derandomize=True)
@given(tc_descs())
def test_tensor_core_plans(kw):
    """Inside the tensor-core kernels' shape rules a plan exists unless no tile fits shared
    memory (or a PWDW or dense output row is too wide for one tile), and `auto` then takes the
    tensor cores too."""
    try:
        info = fcm.fcm_plan_desc(fcm.make_desc(**kw), NUM_SMS, SMEM)
    except fcm.FcmError as err:
        assert err.status == 2 and any(w in str(err) for w in (
            "no tile fits", "too wide", "above 128")), (str(err), kw)
        return
    assert info["kernel"] == 2
    check_plan(kw, info)
    auto = fcm.fcm_plan_desc(fcm.make_desc(**dict(kw, kernel="auto")), NUM_SMS, SMEM)
    assert auto == info


def check_plan(kw, info):
    N, H, W, C, K, k, s, p = (kw[x] for x in ("n", "h", "w", "c", "k_out", "ksize", "stride",
                                              "pad"))
    ho, wo, cm = out_extent(H, k, s, p), out_extent(W, k, s, p), kw["mid"] or C
    assert (info["ho"], info["wo"], info["cm"]) == (ho, wo, cm)

    # launch limits
    assert 0 < info["smem_bytes"] <= SMEM or (info["kernel"] == 1 and kw["conv1"] == "pwdw")
    assert info["threads"] % 32 == 0 and 0 < info["threads"] <= 1024
    if kw["dtype"] == "f32" or kw["kernel"] == "simt":
        assert info["kernel"] == 1
    if kw["dtype"] == "i8":
        assert info["kernel"] == 2
    th, tw = info["tile_h"], info["tile_w"]
    if info["kernel"] == 2:
        assert info["stages"] >= 2
        assert 0 < info["ctas"] <= min(info["num_tiles"], NUM_SMS)
        assert info["num_tiles"] == N * -(-ho // th) * -(-wo // tw)   # covers every pixel
        # TMA boxes start at channel offsets that are multiples of the chunk: the innermost
        # coordinate times the element size must be a multiple of 16 bytes
        assert info["chunk_c"] > 0 and (info["chunk_c"] * ESIZE[kw["dtype"]]) % 16 == 0
        if kw["conv1"] == "dw":
            assert th * tw <= 128
            if info["tc_variant"] == 1:   # worker-warp kernel: 64-channel chunks, last one padded
                assert info["chunk_c"] == 64 and cm <= 256
            else:
                assert info["tc_variant"] == 2 and cm % info["chunk_c"] == 0
    else:
        assert 0 < info["ctas"] <= min(info["num_tiles"], 8 * NUM_SMS)
        # flattened tiles of 32 output pixels (tile_w reports min(32, Wo) for the cost models)
        assert info["num_tiles"] == -(-N * ho * wo // 32) and tw == min(32, wo)

    # minimum bytes (section IV, read as each tensor moved once)
    e = ESIZE[kw["dtype"]]
    w1 = {"dw": C * k * k, "dense": cm * k * k * C, "pwdw": cm * C}[kw["conv1"]]
    wp = cm * k * k if kw["conv1"] == "pwdw" else K * cm
    fused = (N * H * W * C + N * ho * wo * K + w1 + wp) * e + 4 * (2 * cm + 2 * K)
    mid_px = H * W if kw["conv1"] == "pwdw" else ho * wo
    assert info["bytes_fused_min"] == fused
    assert info["bytes_unfused_min"] - fused == 2 * N * mid_px * cm * e
    assert info["overlap_elems"] >= 0 and info["gma_fused_model"] > 0

    # section IV's estimates for the plan's own tile, against the literal equations
    if kw["conv1"] == "dw":
        g = pm.layer_pair_gma(H, W, C, K, k, s, p, th, tw)
        assert info["overlap_elems"] == g["overlap"]
        assert info["gma_fused_model"] == g["fused"] * N * e
        assert info["gma_lbl_model"] == g["lbl"] * N * e
    elif kw["conv1"] == "pwdw":
        ov = pm.overlap(W, H, tw * s, th * s, k, k, s)
        wq, wd = cm * C, cm * k * k
        lbl = (pm.pw_gma(wq, wq, H * W * C, H * W * cm, th * tw * cm)
               + pm.dw_gma(cm, ov, H * W * cm, ho * wo * cm, ho * wo, th * tw, wd))
        fused = pm.pwdw_gma(C, ov, H * W * C, wq, wq, wd, wd, ho * wo * cm, th * tw * cm,
                            ho * wo, th * tw)
        assert info["overlap_elems"] == ov
        assert info["gma_lbl_model"] == lbl * N * e
        assert info["gma_fused_model"] == fused * N * e
