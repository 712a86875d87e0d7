"""Randomised checks of FusePlanner over chains of DW and PW layers (CPU only).

"Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs", section IV:
each layer's layer-by-layer estimate (Equations 1-3), each adjacent pair's FCM estimate
(Equation 4 for PWDW, DWPW and PWPW built from Equations 2 and 3), and the chain's choice of
pairs.  Chains of any DW geometry (k 1-7, stride 1-2, every padding, filters narrower than
the stride included) are drawn by hypothesis and checked three ways:

* against the literal Python model of the equations, decision by decision;
* the chosen pairs against a brute-force search over every set of disjoint adjacent pairs
  (the planner's dynamic programme must reach the same minimum total);
* invariants: a fused pair is a DWPW, PWDW or PWPW module whose estimate is below its two
  layers' sum, and no estimate is negative.
"""
import itertools

import pytest

import pointwise_conv_cnn_gb300 as fcm
from oracle import planner_model as pm

hyp = pytest.importorskip("hypothesis")
st = hyp.strategies
given, settings = hyp.given, hyp.settings

PAIR_KIND = {("dw", "pw"): "dwpw", ("pw", "dw"): "pwdw", ("pw", "pw"): "pwpw"}


@st.composite
def chains(draw):
    H = draw(st.integers(2, 10))
    W = draw(st.integers(2, 10))
    C = draw(st.sampled_from((8, 16, 24, 32, 48, 64)))
    layers = []
    for _ in range(draw(st.integers(1, 6))):
        if draw(st.booleans()):
            k = draw(st.sampled_from((1, 2, 3, 5, 7)))
            p = draw(st.integers(0, k - 1))
            if H + 2 * p < k or W + 2 * p < k:
                p = k - 1
            s = draw(st.integers(1, 2))
            layers.append(dict(kind="dw", h=H, w=W, c=C, ksize=k, stride=s, pad=p))
            H = (H + 2 * p - k) // s + 1
            W = (W + 2 * p - k) // s + 1
        else:
            K = draw(st.sampled_from((8, 16, 32, 40, 64, 96)))
            layers.append(dict(kind="pw", h=H, w=W, c=C, k_out=K))
            C = K
    return layers


def brute_force_total(plans):
    """Minimum chain total over every set of disjoint adjacent pairs that have an FCM."""
    n = len(plans)
    cands = [i for i in range(n - 1) if plans[i]["gma_fcm"] >= 0]
    best = sum(p["gma_lbl"] for p in plans)
    for r in range(1, len(cands) + 1):
        for pick in itertools.combinations(cands, r):
            if any(b - a < 2 for a, b in zip(pick, pick[1:])):
                continue
            t = sum(p["gma_lbl"] for p in plans)
            for i in pick:
                t += plans[i]["gma_fcm"] - plans[i]["gma_lbl"] - plans[i + 1]["gma_lbl"]
            best = min(best, t)
    return best


@settings(max_examples=150, deadline=None, derandomize=True)
@given(chains(), st.sampled_from((1, 2, 8)), st.sampled_from((1, 4, 16, 152)),
       st.sampled_from((1500, 4000, 20000, 10**7)), st.sampled_from((1, 2, 4)))
def test_chain_plans(layers, batch, sms, l1_elems, elem_bytes):
    l1_bytes = l1_elems * elem_bytes
    try:
        ref, ref_total = pm.plan_chain(layers, batch, sms, l1_elems)
    except ValueError:   # some layer has no admissible tile in this L1
        with pytest.raises(fcm.FcmError) as e:
            fcm.fcm_fuse_plan(layers, batch, sms, l1_bytes, elem_bytes)
        assert e.value.status == 4
        return
    plans, total = fcm.fcm_fuse_plan(layers, batch, sms, l1_bytes, elem_bytes)

    # the literal model, decision by decision
    assert total == ref_total
    for p, r in zip(plans, ref):
        assert (p["gma_lbl"], p["gma_fcm"], p["fuse_with_next"], p["fcm_module"]) == \
            (r["gma_lbl"], r["gma_fcm"], r["fuse_with_next"], r["fcm_module"])

    # the dynamic programme reaches the brute-force minimum, and its pairs add up to it
    assert total == brute_force_total(plans)
    picked = sum(p["gma_fcm"] - p["gma_lbl"] - q["gma_lbl"]
                 for p, q in zip(plans, plans[1:]) if p["fuse_with_next"])
    assert total == sum(p["gma_lbl"] for p in plans) + picked

    # invariants
    second = False
    for i, p in enumerate(plans):
        assert p["gma_lbl"] > 0
        kind = PAIR_KIND.get((layers[i]["kind"], layers[i + 1]["kind"])) \
            if i + 1 < len(plans) else None
        assert p["fcm_module"] == kind                  # DW -> DW has no FCM
        assert p["gma_fcm"] == -1 or (kind is not None and p["gma_fcm"] > 0)
        if second:
            assert p["module"] == "fused_second" and not p["fuse_with_next"]
        elif p["fuse_with_next"]:
            assert p["module"] == kind
            assert p["gma_fcm"] < p["gma_lbl"] + plans[i + 1]["gma_lbl"]
        else:
            assert p["module"] == "lbl_" + layers[i]["kind"]
        second = bool(p["fuse_with_next"])
