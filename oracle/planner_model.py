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
    """Equation 1: halo elements (per channel) re-read across neighbouring tiles."""
    return ((ceil_div(channel_w, tile_w) - 1) * (filter_w - strides) * channel_h
            + (ceil_div(channel_h, tile_h) - 1) * (filter_h - strides) * channel_w)


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
