"""Literal global-memory-access cost models of FusePlanner, written out from the equations.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``): the C++ tile planner in the
library is checked against these functions; the library never imports them.

Source: "Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs",
section IV-A (Equations 1-3) and section IV-B (Equation 4 and the DWPW estimator the text says
is "constructed similarly").  All quantities are element counts per image, as printed; the
caller multiplies by the batch and the element size.  Readings of garbled or unprinted parts:

* Eq. 1 is used as printed, with ChannelW/ChannelH the IFM extent and TileW/TileH the IFM
  distance between consecutive OFM tiles (the OFM tile extent times the stride), so that
  ceil(ChannelW / TileW) is the number of tiles along W.
* Eq. 2 and 3 are used as printed, including the factor 2 of Eq. 3.
* Eq. 4 (PWDW) is used as printed (it has no OFM term; that is how it is printed).
* The DWPW estimator, not printed, is built from Eq. 2 and 3 with the two changes section IV-B
  names: the intermediate is neither written nor read, and the DW input is re-read once per
  PW weight tile because the all-channels rule (section II-D) forces recomputation:
      DwPwGMA = (2*C*Overlap + DwIFMsSz) * ceil(PwWeightsSz / PwWeightsTileSz)
                + PwOFMsSz + ceil(OFMsHW / OFMsTileHW) * (DwWeightsSz + PwWeightsSz)
"""
from __future__ import annotations


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def overlap(channel_w: int, channel_h: int, tile_w: int, tile_h: int,
            filter_w: int, filter_h: int, strides: int) -> int:
    """Equation 1: halo elements (per channel) re-read across neighbouring tiles.  The
    equation is stated for overlapping windows (filter at least as wide as the stride); a
    narrower filter leaves gaps and re-reads nothing, so FilterW - Strides is taken as 0 there
    instead of a negative count."""
    return ((ceil_div(channel_w, tile_w) - 1) * max(filter_w - strides, 0) * channel_h
            + (ceil_div(channel_h, tile_h) - 1) * max(filter_h - strides, 0) * channel_w)


def pw_gma(weights_sz: int, weights_tile_sz: int, ifms_sz: int, ofms_sz: int,
           ofms_tile_sz: int) -> int:
    """Equation 2: PW layer global memory accesses."""
    return (ceil_div(weights_sz, weights_tile_sz) * ifms_sz + ofms_sz
            + ceil_div(ofms_sz, ofms_tile_sz) * weights_sz)


def dw_gma(ifms_d: int, overlap_elems: int, ifms_sz: int, ofms_sz: int, ofms_hw: int,
           ofms_tile_hw: int, weights_sz: int) -> int:
    """Equation 3: DW layer global memory accesses."""
    return (2 * ifms_d * overlap_elems + ifms_sz + ofms_sz
            + ceil_div(ofms_hw, ofms_tile_hw) * weights_sz)


def pwdw_gma(pw_ifms_d: int, dw_overlap: int, pw_ifms_sz: int, pw_weights_sz: int,
             pw_weights_tile_sz: int, dw_weights_sz: int, dw_weights_tile_sz: int,
             dw_ofms_sz: int, dw_ofms_tile_sz: int, dw_ofms_hw: int,
             dw_ofms_tile_hw: int) -> int:
    """Equation 4 (PWDW FCM), as printed."""
    return ((2 * pw_ifms_d * dw_overlap + pw_ifms_sz)
            * max(ceil_div(pw_weights_sz, pw_weights_tile_sz),
                  ceil_div(dw_weights_sz, dw_weights_tile_sz))
            + ceil_div(dw_ofms_sz, dw_ofms_tile_sz) * pw_weights_sz
            + ceil_div(dw_ofms_hw, dw_ofms_tile_hw) * dw_weights_sz)


def dwpw_gma(c: int, overlap_elems: int, dw_ifms_sz: int, pw_weights_sz: int,
             pw_weights_tile_sz: int, pw_ofms_sz: int, ofms_hw: int, ofms_tile_hw: int,
             dw_weights_sz: int) -> int:
    """DWPW FCM estimator built like Eq. 4 from Eq. 2 and 3 (reading in the module doc)."""
    return ((2 * c * overlap_elems + dw_ifms_sz) * ceil_div(pw_weights_sz, pw_weights_tile_sz)
            + pw_ofms_sz + ceil_div(ofms_hw, ofms_tile_hw) * (dw_weights_sz + pw_weights_sz))


def layer_pair_gma(H: int, W: int, C: int, K: int, k: int, s: int, p: int,
                   tile_h: int, tile_w: int, k_tile: int | None = None) -> dict:
    """Per-image element counts for one DW k x k (stride s, pad p) -> PW C->K pair tiled into
    OFM tiles of tile_h x tile_w pixels (all channels) and PW weight tiles of k_tile filters.

    Returns the LBL estimate (Eq. 3 for DW + Eq. 2 for PW) and the fused DWPW estimate."""
    Ho = (H + 2 * p - k) // s + 1
    Wo = (W + 2 * p - k) // s + 1
    k_tile = K if k_tile is None else k_tile
    ov = overlap(W, H, tile_w * s, tile_h * s, k, k, s)
    ifm = H * W * C
    mid = Ho * Wo * C
    ofm = Ho * Wo * K
    dw_w = C * k * k
    pw_w = K * C
    n_tiles_hw = ceil_div(Ho, tile_h) * ceil_div(Wo, tile_w)
    lbl_dw = dw_gma(C, ov, ifm, mid, Ho * Wo, tile_h * tile_w, dw_w)
    # Eq. 2 for the PW layer with OFM tiles of tile_h*tile_w pixels x k_tile channels and the
    # weight tile holding k_tile filters of C.
    lbl_pw = pw_gma(pw_w, k_tile * C, mid, ofm, tile_h * tile_w * k_tile)
    fused = dwpw_gma(C, ov, ifm, pw_w, k_tile * C, ofm, Ho * Wo, tile_h * tile_w, dw_w)
    return {"overlap": ov, "lbl_dw": lbl_dw, "lbl_pw": lbl_pw, "lbl": lbl_dw + lbl_pw,
            "fused": fused, "tiles": n_tiles_hw}


def pwpw_gma(pw1_ifms_sz: int, pw1_weights_sz: int, pw2_weights_sz: int,
             pw2_weights_tile_sz: int, pw2_ofms_sz: int, ofms_hw: int, ofms_tile_hw: int) -> int:
    """PWPW FCM estimator, built from Eq. 2 like the DWPW one (reading in the module doc of
    the chain planner below): the first layer's input is re-read once per weight tile of the
    second layer, the output is written once, both weights are read once per spatial tile."""
    return (pw1_ifms_sz * ceil_div(pw2_weights_sz, pw2_weights_tile_sz) + pw2_ofms_sz
            + ceil_div(ofms_hw, ofms_tile_hw) * (pw1_weights_sz + pw2_weights_sz))


# ------------------------------------------------------------- FusePlanner over a layer chain
# Section IV ("FusePlanner overview", IV-A, IV-B): minimum layer-by-layer estimate of every
# layer, minimum FCM estimate of every adjacent pair, both over the tiles that (a) fit in L1
# (three tiles for a layer: IFM, OFM, weights; five for an FCM: both layers' input/output
# tiles, both weight tiles, the communication buffer) and (b) give at least #SMs output tiles;
# tile sizes are multiples of the warp size.  Readings: pixels per tile and channels per tile
# are the sizes restricted to multiples of 32 (a whole plane, or all channels, when smaller);
# output tiles are counted over the batch; when no tile reaches #SMs the tiles with the most
# output tiles are used; a pair is fused when its FCM estimate is below the sum of its layers'
# estimates, and overlapping candidate pairs are resolved by the smallest chain total.

WARP = 32


def _chan_tiles(n):
    return [c for c in range(WARP, n, WARP)] + [n]


def _pixel_tiles(Ho, Wo):
    for th in range(1, Ho + 1):
        for tw in range(1, Wo + 1):
            if (th * tw) % WARP == 0 or (th == Ho and tw == Wo):
                yield th, tw


def _geometry(layer):
    kind = layer["kind"]
    H, W, C = layer["h"], layer["w"], layer["c"]
    if kind == "dw":
        k, s, p = layer["ksize"], layer["stride"], layer["pad"]
        K = C
    else:
        k, s, p = 1, 1, 0
        K = layer["k_out"]
    Ho = (H + 2 * p - k) // s + 1
    Wo = (W + 2 * p - k) // s + 1
    return dict(kind=kind, H=H, W=W, C=C, K=K, k=k, s=s, p=p, Ho=Ho, Wo=Wo)


def _pick(cands):
    """cands: (gma, ntiles, ok, th, tw, tc); the rule of the module comment."""
    if not cands:
        return None
    ok = [c for c in cands if c[2]]
    if ok:
        return min(ok, key=lambda c: c[0])
    most = max(c[1] for c in cands)
    return min((c for c in cands if c[1] == most), key=lambda c: c[0])


def _lbl(g, batch, sms, l1):
    cands = []
    hw = g["Ho"] * g["Wo"]
    if g["kind"] == "dw":
        for ct in _chan_tiles(g["C"]):
            for th, tw in _pixel_tiles(g["Ho"], g["Wo"]):
                ih, iw = (th - 1) * g["s"] + g["k"], (tw - 1) * g["s"] + g["k"]
                if ih * iw * ct + th * tw * ct + ct * g["k"] ** 2 > l1:
                    continue
                n = batch * ceil_div(g["Ho"], th) * ceil_div(g["Wo"], tw) * ceil_div(g["C"], ct)
                ov = overlap(g["W"], g["H"], tw * g["s"], th * g["s"], g["k"], g["k"], g["s"])
                cands.append((dw_gma(g["C"], ov, g["H"] * g["W"] * g["C"], hw * g["C"], hw,
                                     th * tw, g["C"] * g["k"] ** 2), n, n >= sms, th, tw, ct))
    else:
        for kt in _chan_tiles(g["K"]):
            for th, tw in _pixel_tiles(g["Ho"], g["Wo"]):
                px = th * tw
                if px * g["C"] + px * kt + kt * g["C"] > l1:
                    continue
                n = batch * ceil_div(g["Ho"], th) * ceil_div(g["Wo"], tw) * ceil_div(g["K"], kt)
                cands.append((pw_gma(g["K"] * g["C"], kt * g["C"], hw * g["C"], hw * g["K"],
                                     px * kt), n, n >= sms, th, tw, kt))
    return _pick(cands)


def _fcm(a, b, batch, sms, l1):
    cands = []
    if a["kind"] == "dw" and b["kind"] == "pw":
        d, q = a, b
        hw = d["Ho"] * d["Wo"]
        for kt in _chan_tiles(q["K"]):
            for th, tw in _pixel_tiles(d["Ho"], d["Wo"]):
                px = th * tw
                ih, iw = (th - 1) * d["s"] + d["k"], (tw - 1) * d["s"] + d["k"]
                need = ih * iw * d["C"] + px * kt + kt * d["C"] + d["C"] * d["k"] ** 2 + px * d["C"]
                if need > l1:
                    continue
                n = batch * ceil_div(d["Ho"], th) * ceil_div(d["Wo"], tw) * ceil_div(q["K"], kt)
                ov = overlap(d["W"], d["H"], tw * d["s"], th * d["s"], d["k"], d["k"], d["s"])
                cands.append((dwpw_gma(d["C"], ov, d["H"] * d["W"] * d["C"], q["K"] * q["C"],
                                       kt * q["C"], hw * q["K"], hw, px, d["C"] * d["k"] ** 2),
                              n, n >= sms, th, tw, kt))
        return "dwpw", _pick(cands)
    if a["kind"] == "pw" and b["kind"] == "dw":
        q, d = a, b
        hw = d["Ho"] * d["Wo"]
        for ct in _chan_tiles(d["C"]):
            for th, tw in _pixel_tiles(d["Ho"], d["Wo"]):
                px = th * tw
                ih, iw = (th - 1) * d["s"] + d["k"], (tw - 1) * d["s"] + d["k"]
                need = (ih * iw * q["C"] + px * ct + ct * q["C"] + ct * d["k"] ** 2
                        + ih * iw * ct)
                if need > l1:
                    continue
                n = batch * ceil_div(d["Ho"], th) * ceil_div(d["Wo"], tw) * ceil_div(d["C"], ct)
                ov = overlap(d["W"], d["H"], tw * d["s"], th * d["s"], d["k"], d["k"], d["s"])
                cands.append((pwdw_gma(q["C"], ov, q["H"] * q["W"] * q["C"], q["K"] * q["C"],
                                       ct * q["C"], d["C"] * d["k"] ** 2, ct * d["k"] ** 2,
                                       hw * d["C"], px * ct, hw, px), n, n >= sms, th, tw, ct))
        return "pwdw", _pick(cands)
    if a["kind"] == "pw" and b["kind"] == "pw":
        q1, q2 = a, b
        hw = q2["Ho"] * q2["Wo"]
        for kt in _chan_tiles(q2["K"]):
            for th, tw in _pixel_tiles(q2["Ho"], q2["Wo"]):
                px = th * tw
                need = px * q1["C"] + px * kt + q1["K"] * q1["C"] + kt * q2["C"] + px * q1["K"]
                if need > l1:
                    continue
                n = batch * ceil_div(q2["Ho"], th) * ceil_div(q2["Wo"], tw) * ceil_div(q2["K"], kt)
                cands.append((pwpw_gma(q1["H"] * q1["W"] * q1["C"], q1["K"] * q1["C"],
                                       q2["K"] * q2["C"], kt * q2["C"], hw * q2["K"], hw, px),
                              n, n >= sms, th, tw, kt))
        return "pwpw", _pick(cands)
    return None, None


def plan_chain(layers, batch, sms, l1_elems):
    """Returns (per-layer dicts, chain total).  Written as a plain recursion over the chain."""
    geo = [_geometry(L) for L in layers]
    lbl = [_lbl(g, batch, sms, l1_elems) for g in geo]
    if any(x is None for x in lbl):
        raise ValueError("a layer has no tile that fits in L1")
    fcm = [(None, None)] * len(geo)
    for i in range(len(geo) - 1):
        fcm[i] = _fcm(geo[i], geo[i + 1], batch, sms, l1_elems)
    memo = {}

    def best(i):
        """(total, decisions) for layers i.. of the chain."""
        if i >= len(geo):
            return 0, []
        if i in memo:
            return memo[i]
        t_alone, d_alone = best(i + 1)
        choice = (lbl[i][0] + t_alone, [False] + d_alone)
        kind, f = fcm[i] if i + 1 < len(geo) else (None, None)
        if f is not None and f[0] < lbl[i][0] + lbl[i + 1][0]:
            t_pair, d_pair = best(i + 2)
            if f[0] + t_pair < choice[0]:
                choice = (f[0] + t_pair, [True, False] + d_pair)
        memo[i] = choice
        return choice

    total, fuse = best(0)
    out = []
    for i, g in enumerate(geo):
        kind, f = fcm[i]
        out.append({"fuse_with_next": int(fuse[i]), "gma_lbl": lbl[i][0],
                    "gma_fcm": f[0] if f is not None else -1, "fcm_module": kind,
                    "tile": lbl[i][3:6], "fcm_tile": f[3:6] if f else (0, 0, 0)})
    return out, total
