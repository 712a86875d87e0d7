// fuse_planner.cu -- FusePlanner over a chain of DW and PW layers (host only).
//
// "Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs", section IV:
// a first pass estimates each layer's minimum global-memory accesses layer by layer
// (Equations 2 and 3 with the overlap of Equation 1), a second pass estimates every possible
// two-layer FCM (Equation 4 for PWDW; DWPW and PWPW built from Equations 2 and 3 the way
// section IV-B builds Equation 4), each minimised over the tile sizes that satisfy the two
// constraints of section IV-A: the tiles fit in L1 (five tiles for an FCM, three for a
// layer) and there are at least as many output tiles as SMs.  Tile sizes are restricted to
// multiples of the warp size (pixels per tile and channels per tile; a dimension smaller than
// that is taken whole).  The output tiles are counted over the batch; when no admissible tile
// reaches #SMs (a small layer), the tiles with the most output tiles are taken.  A pair is fused when its FCM estimate is below the sum of its two
// layers' estimates; along a chain, where two candidate pairs share a layer, the choice that
// minimises the chain's total is taken (dynamic programming over the chain).
//
// All counts are elements per image, as the equations are printed.
#include <limits.h>
#include <string.h>

#include <vector>

#include "fcm_internal.h"

namespace {

constexpr int kWarp = 32;
constexpr long long kNone = -1;

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

struct Geo {
    int kind, H, W, C, K, k, s, p, Ho, Wo;
};

// The cheapest admissible tile.  Tiles that give at least #SMs output tiles (over the batch)
// come first; when none does (a small layer on many SMs), the tiles with the most output tiles
// are taken instead, the cheapest of them.
struct Best {
    long long gma = kNone;
    int th = 0, tw = 0, tc = 0;
    bool enough = false;     // the chosen tile meets the #SMs constraint
    long long tiles = 0;
    void offer(long long g, long long ntiles, bool ok, int h, int w, int c) {
        bool better;
        if (gma == kNone) better = true;
        else if (ok != enough) better = ok;
        else if (ok) better = g < gma;
        else better = ntiles > tiles || (ntiles == tiles && g < gma);
        if (better) {
            gma = g;
            tiles = ntiles;
            enough = ok;
            th = h;
            tw = w;
            tc = c;
        }
    }
};

// channel tiles: multiples of the warp size up to n, and n itself
std::vector<int> chan_tiles(int n) {
    std::vector<int> v;
    for (int c = kWarp; c < n; c += kWarp) v.push_back(c);
    v.push_back(n);
    return v;
}

// pixel tiles th x tw of an Ho x Wo plane whose pixel count is a multiple of the warp size, or
// the whole plane
template <typename F>
void for_pixel_tiles(int Ho, int Wo, F &&f) {
    for (int th = 1; th <= Ho; th++)
        for (int tw = 1; tw <= Wo; tw++)
            if ((th * tw) % kWarp == 0 || (th == Ho && tw == Wo)) f(th, tw);
}

long long eq1_overlap(const Geo &g, int th, int tw) {
    return fcm_model_overlap(g.W, g.H, (long long)tw * g.s, (long long)th * g.s, g.k, g.k, g.s);
}

Best lbl_dw(const Geo &g, long long batch, int sms, long long l1) {
    Best b;
    const long long hw = (long long)g.Ho * g.Wo;
    for (int ct : chan_tiles(g.C))
        for_pixel_tiles(g.Ho, g.Wo, [&](int th, int tw) {
            const long long tiles = batch * cdiv(g.Ho, th) * cdiv(g.Wo, tw) * cdiv(g.C, ct);
            const long long ih = (long long)(th - 1) * g.s + g.k, iw = (long long)(tw - 1) * g.s + g.k;
            const long long need = ih * iw * ct + (long long)th * tw * ct + (long long)ct * g.k * g.k;
            if (need > l1) return;
            b.offer(fcm_model_dw_gma(g.C, eq1_overlap(g, th, tw), (long long)g.H * g.W * g.C,
                                     hw * g.C, hw, (long long)th * tw, (long long)g.C * g.k * g.k),
                    tiles, tiles >= sms, th, tw, ct);
        });
    return b;
}

Best lbl_pw(const Geo &g, long long batch, int sms, long long l1) {
    Best b;
    const long long hw = (long long)g.Ho * g.Wo;
    for (int kt : chan_tiles(g.K))
        for_pixel_tiles(g.Ho, g.Wo, [&](int th, int tw) {
            const long long px = (long long)th * tw;
            const long long tiles = batch * cdiv(g.Ho, th) * cdiv(g.Wo, tw) * cdiv(g.K, kt);
            if (px * g.C + px * kt + (long long)kt * g.C > l1) return;
            b.offer(fcm_model_pw_gma((long long)g.K * g.C, (long long)kt * g.C, hw * g.C, hw * g.K,
                                     px * kt),
                    tiles, tiles >= sms, th, tw, kt);
        });
    return b;
}

// DW (C -> C, k x k) then PW (C -> K): OFM tiles of th x tw pixels x kt filters; the DW tile
// holds all C channels (section II-D)
Best fcm_dwpw(const Geo &d, const Geo &q, long long batch, int sms, long long l1) {
    Best b;
    const long long hw = (long long)d.Ho * d.Wo;
    for (int kt : chan_tiles(q.K))
        for_pixel_tiles(d.Ho, d.Wo, [&](int th, int tw) {
            const long long px = (long long)th * tw;
            const long long tiles = batch * cdiv(d.Ho, th) * cdiv(d.Wo, tw) * cdiv(q.K, kt);
            const long long ih = (long long)(th - 1) * d.s + d.k, iw = (long long)(tw - 1) * d.s + d.k;
            const long long need = ih * iw * d.C + px * kt + (long long)kt * d.C +
                                   (long long)d.C * d.k * d.k + px * d.C;
            if (need > l1) return;
            b.offer(fcm_model_dwpw_gma(d.C, eq1_overlap(d, th, tw), (long long)d.H * d.W * d.C,
                                       (long long)q.K * q.C, (long long)kt * q.C, hw * q.K, hw, px,
                                       (long long)d.C * d.k * d.k),
                    tiles, tiles >= sms, th, tw, kt);
        });
    return b;
}

// PW (Cin -> Cm) then DW (Cm -> Cm, k x k): DW OFM tiles of th x tw pixels x ct channels; the
// PW computes the ct channels of the DW's input halo tile (Equation 4)
Best fcm_pwdw(const Geo &q, const Geo &d, long long batch, int sms, long long l1) {
    Best b;
    const long long hw = (long long)d.Ho * d.Wo;
    for (int ct : chan_tiles(d.C))
        for_pixel_tiles(d.Ho, d.Wo, [&](int th, int tw) {
            const long long px = (long long)th * tw;
            const long long tiles = batch * cdiv(d.Ho, th) * cdiv(d.Wo, tw) * cdiv(d.C, ct);
            const long long ih = (long long)(th - 1) * d.s + d.k, iw = (long long)(tw - 1) * d.s + d.k;
            const long long need = ih * iw * q.C + px * ct + (long long)ct * q.C +
                                   (long long)ct * d.k * d.k + ih * iw * ct;
            if (need > l1) return;
            b.offer(fcm_model_pwdw_gma(q.C, eq1_overlap(d, th, tw), (long long)q.H * q.W * q.C,
                                       (long long)q.K * q.C, (long long)ct * q.C,
                                       (long long)d.C * d.k * d.k, (long long)ct * d.k * d.k,
                                       hw * d.C, px * ct, hw, px),
                    tiles, tiles >= sms, th, tw, ct);
        });
    return b;
}

// PW (C -> Cm) then PW (Cm -> K): OFM tiles of th x tw pixels x kt filters; the first layer
// produces all Cm channels of the tile
Best fcm_pwpw(const Geo &q1, const Geo &q2, long long batch, int sms, long long l1) {
    Best b;
    const long long hw = (long long)q2.Ho * q2.Wo;
    for (int kt : chan_tiles(q2.K))
        for_pixel_tiles(q2.Ho, q2.Wo, [&](int th, int tw) {
            const long long px = (long long)th * tw;
            const long long tiles = batch * cdiv(q2.Ho, th) * cdiv(q2.Wo, tw) * cdiv(q2.K, kt);
            const long long need = px * q1.C + px * kt + (long long)q1.K * q1.C +
                                   (long long)kt * q2.C + px * q1.K;
            if (need > l1) return;
            b.offer(fcm_model_pwpw_gma((long long)q1.H * q1.W * q1.C, (long long)q1.K * q1.C,
                                       (long long)q2.K * q2.C, (long long)kt * q2.C, hw * q2.K,
                                       hw, px),
                    tiles, tiles >= sms, th, tw, kt);
        });
    return b;
}

}  // namespace

extern "C" {

long long fcm_model_pwdw_gma(long long pw_ifms_d, long long dw_overlap, long long pw_ifms_sz,
                             long long pw_weights_sz, long long pw_weights_tile_sz,
                             long long dw_weights_sz, long long dw_weights_tile_sz,
                             long long dw_ofms_sz, long long dw_ofms_tile_sz, long long dw_ofms_hw,
                             long long dw_ofms_tile_hw) {
    if (pw_weights_tile_sz <= 0 || dw_weights_tile_sz <= 0 || dw_ofms_tile_sz <= 0 ||
        dw_ofms_tile_hw <= 0)
        return -1;
    const long long wt = cdiv(pw_weights_sz, pw_weights_tile_sz);
    const long long dt = cdiv(dw_weights_sz, dw_weights_tile_sz);
    return (2 * pw_ifms_d * dw_overlap + pw_ifms_sz) * (wt > dt ? wt : dt) +
           cdiv(dw_ofms_sz, dw_ofms_tile_sz) * pw_weights_sz +
           cdiv(dw_ofms_hw, dw_ofms_tile_hw) * dw_weights_sz;
}

long long fcm_model_pwpw_gma(long long pw1_ifms_sz, long long pw1_weights_sz,
                             long long pw2_weights_sz, long long pw2_weights_tile_sz,
                             long long pw2_ofms_sz, long long ofms_hw, long long ofms_tile_hw) {
    if (pw2_weights_tile_sz <= 0 || ofms_tile_hw <= 0) return -1;
    return pw1_ifms_sz * cdiv(pw2_weights_sz, pw2_weights_tile_sz) + pw2_ofms_sz +
           cdiv(ofms_hw, ofms_tile_hw) * (pw1_weights_sz + pw2_weights_sz);
}

fcm_status fcm_fuse_plan(const fcm_layer *layers, int n_layers, int batch, int num_sms,
                         long long l1_bytes, int elem_bytes, fcm_layer_plan *out,
                         long long *total_gma) {
    if (!layers || !out || n_layers < 1 || batch < 1 || num_sms < 1 || l1_bytes < 1 ||
        elem_bytes < 1)
        return fcm_fail(FCM_ERR_INVALID_ARG, "fcm_fuse_plan: bad arguments");
    const long long l1 = l1_bytes / elem_bytes;
    std::vector<Geo> g(n_layers);
    for (int i = 0; i < n_layers; i++) {
        const fcm_layer &L = layers[i];
        Geo &x = g[i];
        x.kind = L.kind;
        x.H = L.h;
        x.W = L.w;
        x.C = L.c;
        x.K = L.kind == FCM_LAYER_DW ? L.c : L.k_out;
        x.k = L.kind == FCM_LAYER_DW ? L.ksize : 1;
        x.s = L.kind == FCM_LAYER_DW ? L.stride : 1;
        x.p = L.kind == FCM_LAYER_DW ? L.pad : 0;
        if ((L.kind != FCM_LAYER_DW && L.kind != FCM_LAYER_PW) || x.H < 1 || x.W < 1 || x.C < 1 ||
            x.K < 1 || x.k < 1 || x.s < 1 || x.p < 0 || x.H + 2 * x.p < x.k || x.W + 2 * x.p < x.k)
            return fcm_fail(FCM_ERR_INVALID_ARG, "layer %d: bad shape", i);
        if (L.kind == FCM_LAYER_DW && L.k_out != 0 && L.k_out != L.c)
            return fcm_fail(FCM_ERR_INVALID_ARG, "layer %d: a DW layer has k_out == c", i);
        x.Ho = (x.H + 2 * x.p - x.k) / x.s + 1;
        x.Wo = (x.W + 2 * x.p - x.k) / x.s + 1;
        if (i > 0 && (x.H != g[i - 1].Ho || x.W != g[i - 1].Wo || x.C != g[i - 1].K))
            return fcm_fail(FCM_ERR_INVALID_ARG,
                            "layer %d: input %dx%dx%d does not match the output of layer %d", i,
                            x.H, x.W, x.C, i - 1);
    }
    std::vector<Best> lbl(n_layers), fcm(n_layers);
    std::vector<int> fcm_kind(n_layers, -1);
    for (int i = 0; i < n_layers; i++) {
        lbl[i] = g[i].kind == FCM_LAYER_DW ? lbl_dw(g[i], batch, num_sms, l1)
                                           : lbl_pw(g[i], batch, num_sms, l1);
        if (lbl[i].gma == kNone)
            return fcm_fail(FCM_ERR_SMEM_BUDGET, "layer %d: no tile fits in %lld elements of L1", i,
                            l1);
        if (i + 1 < n_layers) {
            const Geo &a = g[i], &b = g[i + 1];
            if (a.kind == FCM_LAYER_DW && b.kind == FCM_LAYER_PW) {
                fcm[i] = fcm_dwpw(a, b, batch, num_sms, l1);
                fcm_kind[i] = FCM_MODULE_DWPW;
            } else if (a.kind == FCM_LAYER_PW && b.kind == FCM_LAYER_DW) {
                fcm[i] = fcm_pwdw(a, b, batch, num_sms, l1);
                fcm_kind[i] = FCM_MODULE_PWDW;
            } else if (a.kind == FCM_LAYER_PW && b.kind == FCM_LAYER_PW) {
                fcm[i] = fcm_pwpw(a, b, batch, num_sms, l1);
                fcm_kind[i] = FCM_MODULE_PWPW;
            }
        }
    }
    // best[i]: minimum total of layers i.. ; fuse[i]: layers i and i+1 form one FCM
    std::vector<long long> best(n_layers + 1, 0);
    std::vector<int> fuse(n_layers, 0);
    for (int i = n_layers - 1; i >= 0; i--) {
        best[i] = lbl[i].gma + best[i + 1];
        if (i + 1 < n_layers && fcm[i].gma != kNone &&
            fcm[i].gma < lbl[i].gma + lbl[i + 1].gma) {
            const long long f = fcm[i].gma + best[i + 2];
            if (f < best[i]) {
                best[i] = f;
                fuse[i] = 1;
            }
        }
    }
    for (int i = 0; i < n_layers; i++) {
        fcm_layer_plan &o = out[i];
        memset(&o, 0, sizeof(o));
        o.gma_lbl = lbl[i].gma;
        o.gma_fcm = fcm[i].gma;
        o.fcm_module = fcm_kind[i];
        o.fcm_tile_h = fcm[i].th;
        o.fcm_tile_w = fcm[i].tw;
        o.fcm_tile_c = fcm[i].tc;
        o.tile_h = lbl[i].th;
        o.tile_w = lbl[i].tw;
        o.tile_c = lbl[i].tc;
        o.tiles_ok = lbl[i].enough ? 1 : 0;
        o.fcm_tiles_ok = fcm[i].enough ? 1 : 0;
    }
    // walk the chosen decomposition
    for (int i = 0; i < n_layers;) {
        if (fuse[i]) {
            out[i].fuse_with_next = 1;
            out[i].module = fcm_kind[i];
            out[i + 1].module = FCM_MODULE_FUSED_SECOND;
            i += 2;
        } else {
            out[i].module = g[i].kind == FCM_LAYER_DW ? FCM_MODULE_LBL_DW : FCM_MODULE_LBL_PW;
            i += 1;
        }
    }
    if (total_gma) *total_gma = best[0];
    return FCM_OK;
}

}  // extern "C"
