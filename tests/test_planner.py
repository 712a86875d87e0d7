"""FusePlanner cost models (section IV, Eq. 1-4) and the tile planner (CPU only)."""
import numpy as np
import pytest

import pointwise_conv_cnn_gb300 as fcm
from oracle import planner_model as pm
from pointwise_conv_cnn_gb300 import build
from pointwise_conv_cnn_gb300 import workloads as wk


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fcm.load_library()


def test_eq1_overlap_by_hand():
    # (ceil(56/28)-1)*(3-1)*56 + (ceil(56/14)-1)*(3-1)*56 = 112 + 336
    assert pm.overlap(56, 56, 28, 14, 3, 3, 1) == 448
    assert fcm.fcm_model_overlap(56, 56, 28, 14, 3, 3, 1) == 448
    # one tile: no overlap
    assert fcm.fcm_model_overlap(56, 56, 56, 56, 3, 3, 1) == 0
    # filter no wider than the stride: windows of neighbouring tiles share nothing
    for f in (pm.overlap, fcm.fcm_model_overlap):
        assert f(9, 9, 2, 2, 1, 1, 2) == 0 and f(8, 8, 4, 4, 2, 2, 2) == 0
        # 3 wide at stride 2: one shared column per tile boundary, (ceil(9/4)-1)*1*9 = 18 per axis
        assert f(9, 9, 4, 4, 3, 3, 2) == 36


def test_eq2_eq3_dwpw_by_hand():
    # Eq. 2: ceil(100/30)*1000 + 500 + ceil(500/64)*100 = 4000 + 500 + 800
    assert pm.pw_gma(100, 30, 1000, 500, 64) == 5300
    assert fcm.fcm_model_pw_gma(100, 30, 1000, 500, 64) == 5300
    # Eq. 3: 2*8*10 + 1000 + 900 + ceil(100/32)*72 = 160 + 1000 + 900 + 288
    assert pm.dw_gma(8, 10, 1000, 900, 100, 32, 72) == 2348
    assert fcm.fcm_model_dw_gma(8, 10, 1000, 900, 100, 32, 72) == 2348
    # DWPW: (2*8*10 + 1000)*ceil(64/32) + 800 + ceil(100/32)*(72+64) = 2320 + 800 + 544
    assert pm.dwpw_gma(8, 10, 1000, 64, 32, 800, 100, 32, 72) == 3664
    assert fcm.fcm_model_dwpw_gma(8, 10, 1000, 64, 32, 800, 100, 32, 72) == 3664


def test_eq4_pwdw_as_printed():
    # (2*16*5 + 400) * max(ceil(64/32), ceil(72/72)) + ceil(300/100)*64 + ceil(50/25)*72
    #   = 560*2 + 3*64 + 2*72
    assert pm.pwdw_gma(16, 5, 400, 64, 32, 72, 72, 300, 100, 50, 25) == 1120 + 192 + 144


def test_c_models_match_literal_models_randomised():
    r = np.random.default_rng(0)
    for _ in range(300):
        a = [int(v) for v in r.integers(1, 500, 12)]
        assert fcm.fcm_model_overlap(a[0], a[1], a[2], a[3], a[4] % 7 + 1, a[5] % 7 + 1, a[6] % 2 + 1) == \
            pm.overlap(a[0], a[1], a[2], a[3], a[4] % 7 + 1, a[5] % 7 + 1, a[6] % 2 + 1)
        assert fcm.fcm_model_pw_gma(*a[:5]) == pm.pw_gma(*a[:5])
        assert fcm.fcm_model_dw_gma(*a[:7]) == pm.dw_gma(*a[:7])
        assert fcm.fcm_model_dwpw_gma(*a[:9]) == pm.dwpw_gma(*a[:9])


def test_fig1_fusion_saves_half_of_activation_traffic():
    """Figure 1 / section I: fusing DW+PW saves 50% of their off-chip accesses (C = K,
    stride 1, one tile over the image, weights set aside)."""
    H = W = 56
    C = K = 128
    g = pm.layer_pair_gma(H, W, C, K, 3, 1, 1, H, W)
    weights = C * 9 + K * C
    lbl = g["lbl"] - weights  # each layer reads its weights once
    fused = g["fused"] - weights
    assert g["overlap"] == 0
    assert fused * 2 == lbl


@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_plan_bytes_match_closed_form(wl):
    info = fcm.fcm_plan_desc(fcm.desc_from_workload(wl))
    mb = wl.min_bytes()
    assert info["bytes_fused_min"] == mb["fused"]
    assert info["bytes_unfused_min"] == mb["unfused"]
    assert info["ho"] == wl.ho and info["wo"] == wl.wo


@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_plan_model_matches_literal(wl):
    if wl.conv1 != "dw":
        pytest.skip("Eq. 3 models the depthwise layer")
    info = fcm.fcm_plan_desc(fcm.desc_from_workload(wl))
    g = pm.layer_pair_gma(wl.h, wl.w, wl.c, wl.k_out, wl.ksize, wl.stride, wl.pad,
                          info["tile_h"], info["tile_w"])
    e = wl.esize
    assert info["overlap_elems"] == g["overlap"]
    assert info["gma_fused_model"] == g["fused"] * wl.n * e
    assert info["gma_lbl_model"] == g["lbl"] * wl.n * e


def test_fused_saving_closed_forms():
    """Saving of fusion vs the unfused pair, from the tensor sizes alone: 50% for C=K stride 1
    (MobileNet), 25% for the stride-2 64->128 layer, 60% for the 240->80 5x5 layer."""
    expect = {"mobilenet_dwpw_f16": 0.50, "stride2_dwpw_bf16": 0.25, "wide5x5_dwpw_bf16": 0.60,
              "b2b_dense3x3_f16": 0.50}
    for name, saving in expect.items():
        b = wk.BY_NAME[name].min_bytes()
        io_f = b["x"] + b["y"]
        io_u = io_f + 2 * b["mid"]
        assert abs((1 - io_f / io_u) - saving) < 1e-12, name


def test_pwdw_plan_models_match_literal():
    """The PWDW module's plan reports Eq. 2 + Eq. 3 layer by layer (the 1x1 over H x W, the
    depthwise over its output) and Eq. 4 fused, for the plan's own tile, as printed."""
    wl = wk.BY_NAME["pwdw_f16"]
    info = fcm.fcm_plan_desc(fcm.desc_from_workload(wl))
    H, W, C, Cm, k, s = wl.h, wl.w, wl.c, wl.cm, wl.ksize, wl.stride
    Ho, Wo, th, tw = info["ho"], info["wo"], info["tile_h"], info["tile_w"]
    ov = pm.overlap(W, H, tw * s, th * s, k, k, s)
    w1, wd = Cm * C, Cm * k * k
    lbl = (pm.pw_gma(w1, w1, H * W * C, H * W * Cm, th * tw * Cm)
           + pm.dw_gma(Cm, ov, H * W * Cm, Ho * Wo * Cm, Ho * Wo, th * tw, wd))
    fused = pm.pwdw_gma(C, ov, H * W * C, w1, w1, wd, wd, Ho * Wo * Cm, th * tw * Cm, Ho * Wo,
                        th * tw)
    e = wl.esize
    assert info["overlap_elems"] == ov
    assert info["gma_lbl_model"] == lbl * wl.n * e
    assert info["gma_fused_model"] == fused * wl.n * e
    # the intermediate (N x H x W x Cm) is what fusion keeps out of HBM
    assert info["bytes_unfused_min"] - info["bytes_fused_min"] == 2 * wl.n * H * W * Cm * e


def test_int8_plans_and_refusals():
    """INT8 (FCM_I8): the depthwise module plans on the tensor-core kernels with 1-byte
    activations and weights (scales and biases stay fp32); requests without an INT8 kernel are
    refused with FCM_ERR_UNSUPPORTED, never served by another path."""
    f16 = wk.BY_NAME["mobilenet_dwpw_f16"]
    i8 = wk.BY_NAME["mobilenet_dwpw_i8"]
    pi = fcm.fcm_plan_desc(fcm.desc_from_workload(i8))
    pf = fcm.fcm_plan_desc(fcm.desc_from_workload(f16))
    assert pi["kernel"] == 2
    sb = 4 * (2 * i8.c + 2 * i8.k_out)
    assert pi["bytes_fused_min"] - sb == (pf["bytes_fused_min"] - sb) // 2
    refused = [i8.with_(conv1="dense", mid=128), i8.with_(conv1="pwdw", c=96, mid=128, k_out=128),
               i8.with_(c=512, k_out=64)]
    for wl in refused:
        with pytest.raises(fcm.FcmError) as e:
            fcm.fcm_plan_desc(fcm.desc_from_workload(wl))
        assert e.value.status == 2, wl
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_plan_desc(fcm.desc_from_workload(i8, kernel="simt"))
    assert e.value.status == 2


@pytest.mark.parametrize("wl", wk.WORKLOADS, ids=lambda w: w.name)
def test_plans_fit_the_gb300_limits(wl):
    """Every workload's plan (planned on the host for 152 SMs and 227 KB of shared memory a
    block) fits the limits the kernels are launched under: dynamic shared memory, whole warps,
    at most 1024 threads, a persistent grid of at most one CTA per SM, at least two stages."""
    info = fcm.fcm_plan_desc(fcm.desc_from_workload(wl), 152, 232448)
    assert info["smem_bytes"] <= 232448
    assert info["threads"] % 32 == 0 and 0 < info["threads"] <= 1024
    assert 0 < info["ctas"] <= 152 * (8 if info["kernel"] == 1 else 1)
    if info["kernel"] == 2:
        assert info["stages"] >= 2
        assert info["tile_h"] * info["tile_w"] <= 128 or wl.conv1 == "pwdw"


@pytest.mark.parametrize("n,ok", [(1 << 18, True), (1 << 24, False)])
def test_huge_batches_plan_or_refuse_cleanly(n, ok):
    """A batch of 2^18 MobileNet images plans (7.3 M tiles, 32-bit tile indices); 2^24 images
    (6.7e12 input elements, above the 2^40 guard) is refused with FCM_ERR_UNSUPPORTED."""
    wl = wk.BY_NAME["mobilenet_dwpw_f16"].with_(n=n)
    if ok:
        info = fcm.fcm_plan_desc(fcm.desc_from_workload(wl), 152, 232448)
        assert info["num_tiles"] == n * 28 and info["ctas"] == 152
    else:
        with pytest.raises(fcm.FcmError) as e:
            fcm.fcm_plan_desc(fcm.desc_from_workload(wl), 152, 232448)
        assert e.value.status == 2


DW_DESCS = [  # (N, H, W, C, K, k, s, p, dtype)
    (64, 56, 56, 128, 128, 3, 1, 1, "f16"),
    (128, 112, 112, 64, 128, 3, 2, 1, "bf16"),
    (128, 28, 28, 240, 80, 5, 1, 2, "bf16"),
    (8, 14, 14, 256, 64, 3, 1, 1, "f16"),
    (4, 7, 7, 96, 32, 7, 1, 3, "i8"),
    (2, 20, 131, 64, 64, 3, 1, 1, "f16"),
]


def _work_eff(info, ho, wo, stencil):
    """Useful output pixels over the MMA rows the tiles occupy (the worker-warp kernel also
    counts the stencil pixels its 4-pixel units compute past the image)."""
    tiles_w = -(-wo // info["tile_w"])
    tiles_h = -(-ho // info["tile_h"])
    eff = ho * wo / (tiles_w * tiles_h * 128)
    if stencil:
        pitch = info["tile_w"]   # reported as min(pitch, Wo): the pitch is a multiple of 8
        ngroups = -(-min(pitch, wo) // 4)
        eff *= ho * wo / (tiles_w * tiles_h * info["tile_h"] * ngroups * 4)
    return eff


@pytest.mark.parametrize("shape", DW_DESCS, ids=lambda s: "x".join(map(str, s[:8])) + s[8])
@pytest.mark.parametrize("kernel", ["tc_roles", "tc_workers"])
def test_tile_choice_minimises_the_section4_estimate(shape, kernel):
    """The planner ranks by the bytes it models (FusePlanner, section IV): among the tiles whose
    work efficiency is within 3% of the best one's, the chosen tile has the smallest DWPW
    global-memory-access estimate (gma_fused_model, Eq. 1-4 form).  Every tile the kernel can
    take is planned on its own through the tile override and compared."""
    N, H, W, C, K, k, s, p, dt = shape
    base = dict(n=N, h=H, w=W, c=C, k_out=K, ksize=k, stride=s, pad=p, conv1="dw", dtype=dt,
                act1="relu", act2="none", kernel=kernel)
    try:
        auto = fcm.fcm_plan_desc(fcm.make_desc(**base))
    except fcm.FcmError:
        pytest.skip("the kernel does not take this shape")
    ho, wo = auto["ho"], auto["wo"]
    if kernel == "tc_workers":
        tiles = [(32 // qw * (4 // nqx), qw * nqx) for qw in (32, 16, 8) for nqx in (1, 2, 4)]
    else:
        tiles = [(th, 0) for th in range(1, 129)]
    forced = []
    for th, tw in tiles:
        try:
            forced.append(fcm.fcm_plan_desc(fcm.make_desc(**dict(base, tile_h=th, tile_w=tw))))
        except fcm.FcmError:
            continue
    stencil = kernel == "tc_workers"
    best = max(_work_eff(f, ho, wo, stencil) for f in forced)
    assert _work_eff(auto, ho, wo, stencil) >= 0.97 * best - 1e-12
    admissible = [f for f in forced if _work_eff(f, ho, wo, stencil) >= 0.97 * best - 1e-12]
    assert auto["gma_fused_model"] == min(f["gma_fused_model"] for f in admissible)
