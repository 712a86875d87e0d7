"""FusePlanner over a chain of DW/PW layers (fcm_fuse_plan) against hand-computed cases and
the literal Python model of the equations (CPU only).

"Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs", section IV:
Equations 1-3 (layer by layer), Equation 4 (PWDW) and the FCM estimators built like it."""
import random

import pytest

import pointwise_conv_cnn_gb300 as fcm
from pointwise_conv_cnn_gb300 import build
from oracle import planner_model as pm


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fcm.load_library()


def test_eq4_pwdw_by_hand():
    # PW 8 -> 16 channels on 6x6, DW 3x3 s1 over 2 tiles along W (tile 3 wide): overlap
    # (2-1)*(3-1)*6 = 12 elements per channel.  Weight tiles: PW 128 of 16*8 -> 1 tile, DW
    # 72 of 144 -> 2 tiles, so max(1, 2) = 2.  DW OFM 576 in tiles of 3*6*8 = 144 -> 4.
    # (2*8*12 + 288) * 2 + 4*128 + ceil(36/18)*144 = 960 + 512 + 288 = 1760
    args = (8, 12, 288, 128, 128, 144, 72, 576, 144, 36, 18)
    assert pm.pwdw_gma(*args) == 1760
    assert fcm.fcm_model_pwdw_gma(*args) == 1760


def test_pwpw_estimator_by_hand():
    # IFM 512 re-read per 2nd-layer weight tile (8192 / 4096 -> 2), OFM 512, one spatial tile
    # reads both weights (8192 + 8192): 1024 + 512 + 16384
    args = (512, 8192, 8192, 4096, 512, 16, 16)
    assert pm.pwpw_gma(*args) == 17920
    assert fcm.fcm_model_pwpw_gma(*args) == 17920


def test_dwpw_pair_fuses_by_hand():
    """DW 3x3 on 4x4x32 then PW 32->32, one SM, unbounded L1: the only pixel tile is the whole
    plane (16 < 32 pixels).  Eq. 3: 0 + 512 + 512 + 288 = 1312; Eq. 2: 512 + 512 + 1024 = 2048;
    DWPW: 512 + 512 + (288 + 1024) = 2336 < 3360, so the pair is fused (the intermediate's write
    and read, 2 x 512, are saved)."""
    layers = [dict(kind="dw", h=4, w=4, c=32, ksize=3, stride=1, pad=1),
              dict(kind="pw", h=4, w=4, c=32, k_out=32)]
    plans, total = fcm.fcm_fuse_plan(layers, 1, 1, 2 * 10**9, 2)
    assert [p["gma_lbl"] for p in plans] == [1312, 2048]
    assert plans[0]["gma_fcm"] == 2336 and plans[0]["fcm_module"] == "dwpw"
    assert plans[0]["fuse_with_next"] == 1 and plans[0]["module"] == "dwpw"
    assert plans[1]["module"] == "fused_second"
    assert total == 2336


def test_pwpw_weights_do_not_fit_so_layers_stay_apart():
    """PW 32->256 then PW 256->32 on 4x4: each layer fits 20000 elements of L1 (16*32 +
    16*256 + 256*32 = 12800) but the FCM's five tiles need 16*32 + 16*32 + 8192 + 8192 + 4096 =
    21504 with the smallest filter tile, so no FCM exists (section IV-B: two weight tiles make
    PWPW fusion less likely).  With room for it, the FCM (512 + 512 + 16384 = 17408) beats the
    two layers (12800 each) and is chosen."""
    layers = [dict(kind="pw", h=4, w=4, c=32, k_out=256), dict(kind="pw", h=4, w=4, c=256, k_out=32)]
    plans, total = fcm.fcm_fuse_plan(layers, 1, 1, 20000 * 2, 2)
    assert [p["gma_lbl"] for p in plans] == [12800, 12800]
    assert plans[0]["gma_fcm"] == -1 and plans[0]["fuse_with_next"] == 0 and total == 25600
    plans, total = fcm.fcm_fuse_plan(layers, 1, 1, 10**9, 2)
    assert plans[0]["gma_fcm"] == 17408 and plans[0]["fuse_with_next"] == 1 and total == 17408


def random_chain(rng):
    H = W = rng.choice([4, 6, 8, 12])
    C = rng.choice([16, 32, 48, 64])
    layers = []
    for _ in range(rng.randint(2, 5)):
        if rng.random() < 0.5:
            k = rng.choice([1, 3, 5])
            s = rng.choice([1, 2]) if H >= 4 else 1
            p = k // 2
            layers.append(dict(kind="dw", h=H, w=W, c=C, ksize=k, stride=s, pad=p))
            H = (H + 2 * p - k) // s + 1
            W = (W + 2 * p - k) // s + 1
        else:
            K = rng.choice([16, 32, 40, 64, 96])
            layers.append(dict(kind="pw", h=H, w=W, c=C, k_out=K))
            C = K
    return layers


@pytest.mark.parametrize("seed", range(30))
def test_chain_matches_literal_model(seed):
    rng = random.Random(seed)
    layers = random_chain(rng)
    batch = rng.choice([1, 2, 8])
    sms = rng.choice([1, 4, 16, 152])
    l1 = rng.choice([2000, 6000, 20000, 10**7])
    try:
        ref, ref_total = pm.plan_chain(layers, batch, sms, l1)
    except ValueError:   # the model found no admissible tile for some layer
        with pytest.raises(fcm.FcmError):
            fcm.fcm_fuse_plan(layers, batch, sms, l1 * 2, 2)
        return
    plans, total = fcm.fcm_fuse_plan(layers, batch, sms, l1 * 2, 2)
    assert total == ref_total
    for p, r in zip(plans, ref):
        assert p["gma_lbl"] == r["gma_lbl"]
        assert p["gma_fcm"] == r["gma_fcm"]
        assert p["fuse_with_next"] == r["fuse_with_next"]
        assert p["fcm_module"] == r["fcm_module"]
    # the chain total is never above running every layer alone, and fused pairs do not overlap
    assert total <= sum(p["gma_lbl"] for p in plans)
    for a, b in zip(plans, plans[1:]):
        assert not (a["fuse_with_next"] and b["fuse_with_next"])


def test_chain_validation():
    with pytest.raises(fcm.FcmError) as e:
        fcm.fcm_fuse_plan([dict(kind="pw", h=8, w=8, c=16, k_out=32),
                           dict(kind="pw", h=8, w=8, c=16, k_out=16)])
    assert e.value.status == 1
    with pytest.raises(fcm.FcmError):
        fcm.fcm_fuse_plan([dict(kind="dw", h=8, w=8, c=16, k_out=8, ksize=3, stride=1, pad=1)])


def test_int8_bit_width_changes_the_fusion_decision():
    """Section V-B: changing the bit width changes the tiles, so FusePlanner chooses differently
    (most INT8 FCMs are fusions not feasible in FP32).  The PWPW pair above with 64 KiB of L1:
    FP32 holds 16384 elements, fewer than the FCM's five tiles need (21504), so the layers stay
    apart; INT8 holds 65536 and the pair is fused.  The literal model agrees in both cases."""
    layers = [dict(kind="pw", h=4, w=4, c=32, k_out=256), dict(kind="pw", h=4, w=4, c=256, k_out=32)]
    l1 = 64 * 1024
    for elem_bytes, fused in ((4, 0), (1, 1)):
        plans, total = fcm.fcm_fuse_plan(layers, 1, 1, l1, elem_bytes)
        ref, ref_total = pm.plan_chain(layers, 1, 1, l1 // elem_bytes)
        assert plans[0]["fuse_with_next"] == fused == ref[0]["fuse_with_next"], elem_bytes
        assert total == ref_total
    assert fcm.fcm_fuse_plan(layers, 1, 1, l1, 1)[1] == 17408


def inverted_residual_chain(blocks=4):
    """A MobileNetV2-style stack written here (not a model's table): per block a 1x1 expansion
    (x6), a 3x3 depthwise layer (stride 2 or 1) and a 1x1 projection, from 112x112x16."""
    layers, H, c = [], 112, 16
    for cout, s in ((24, 2), (24, 1), (32, 2), (32, 1))[:blocks]:
        e = 6 * c
        layers.append(dict(kind="pw", h=H, w=H, c=c, k_out=e))
        layers.append(dict(kind="dw", h=H, w=H, c=e, ksize=3, stride=s, pad=1))
        H = (H + 2 - 3) // s + 1
        layers.append(dict(kind="pw", h=H, w=H, c=e, k_out=cout))
        c = cout
    return layers


def test_int8_chain_fuses_more_kinds_of_pairs():
    """Section V-B on a chain: with 64 KiB of L1 and 152 SMs, FP32 fuses only the four
    expansion -> depthwise pairs (PWDW), while INT8's smaller elements also admit a PWPW and a
    DWPW fusion; the literal model makes the same decisions."""
    layers = inverted_residual_chain()
    kinds = {}
    for e in (4, 1):
        plans, total = fcm.fcm_fuse_plan(layers, 1, 152, 64 * 1024, e)
        ref, ref_total = pm.plan_chain(layers, 1, 152, 64 * 1024 // e)
        assert total == ref_total
        assert [p["fuse_with_next"] for p in plans] == [r["fuse_with_next"] for r in ref]
        kinds[e] = sorted(p["fcm_module"] for p in plans if p["fuse_with_next"])
    assert kinds[4] == ["pwdw"] * 4
    assert kinds[1] == sorted(["pwdw"] * 3 + ["pwpw", "dwpw"])
