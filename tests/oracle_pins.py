"""Pins for the CPU oracle: facts fixed by the pages or by mathematics.

Each ``pin_*`` function takes an oracle (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with the fact it checks.  None of
them re-derives the oracle's own code path: they use closed forms that
bilinear interpolation must reproduce, special cases, identities that follow
from linearity, finite differences, a library bilinear sampler
(``torch.nn.functional.grid_sample``) and a hand-worked example.

What the pages fix ("MS Deformable Attention Kernel API Reference" and its
backward page, Parameters / Returns / Notes):
  * align_corners=True maps [0,1] onto [0, H-1]; False onto [-0.5, H-0.5];
  * "zeros" padding reads 0 out of bounds, "border" clamps to the edge;
  * value BLNC (B,L,N_h,C_h) / BNLC (B,N_h,L,C_h), locations BQHLP2 / B2QHLP,
    output (B, N_q, N_h*C_h);
  * gradients are the bilinear-interpolation derivatives.
The same functions run against planted-mistake copies of the oracle (see
test_oracle_mutants.py), where at least one of them must fail.
"""
from __future__ import annotations

import json
import os

import numpy as np

from scale_deformable_attention_forward_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- helpers
def _starts(levels):
    s, out = 0, []
    for h, w in levels:
        out.append(s)
        s += h * w
    return tuple(out)


def _u_from_pixel(pix, size, align):
    """Normalised coordinate whose pixel coordinate is ``pix``, by the page's
    mapping: align_corners=True sends [0,1] to [0, size-1], False to
    [-0.5, size-0.5] (both linear)."""
    if align:
        return pix / (size - 1) if size > 1 else np.zeros_like(pix)
    return (pix + 0.5) / size


def _du_dpix(size, align):
    """Pixels per unit of normalised coordinate, from the same mapping."""
    return (size - 1) if align else size


def _problem(rng, levels, B, N_q, N_h, C_h, N_p, loc_lo=-0.1, loc_hi=1.1):
    L = sum(h * w for h, w in levels)
    N_l = len(levels)
    value = rng.standard_normal((B, L, N_h, C_h))
    loc = rng.uniform(loc_lo, loc_hi, size=(B, N_q, N_h, N_l, N_p, 2))
    attn = rng.uniform(0.05, 1.0, size=(B, N_q, N_h, N_l, N_p))
    g = rng.standard_normal((B, N_q, N_h * C_h))
    return dict(value=value, loc=loc, attn=attn, g=g, levels=tuple(levels), starts=_starts(levels))


def _fwd(orc, P, value=None, loc=None, attn=None, **kw):
    return orc.forward(P["value"] if value is None else value, P["levels"], P["starts"],
                       P["loc"] if loc is None else loc, P["attn"] if attn is None else attn, **kw)


def _bwd(orc, P, value=None, loc=None, attn=None, g=None, **kw):
    return orc.backward(P["g"] if g is None else g, P["value"] if value is None else value,
                        P["levels"], P["starts"], P["loc"] if loc is None else loc,
                        P["attn"] if attn is None else attn, **kw)


def _level_map(value, starts, levels, l):
    """(B, H, W, N_h, C_h) view of level l of a BLNC value tensor."""
    h, w = levels[l]
    return value[:, starts[l]:starts[l] + h * w].reshape(value.shape[0], h, w, *value.shape[2:])


def _close(a, b, rtol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= rtol * scale, f"{what}: max abs err {err:.3e} > {rtol:.1e} * {scale:.3e}"


# --------------------------------------------------------------------------- pins
def pin_pixel_centre(orc):
    """A sample at the exact centre of pixel (i, j) of level l, with all
    attention on it, returns value[b, start_l + i*W + j, h, :] -- for both
    align_corners mappings, both paddings and both layouts.  Non-square and
    single-row/column levels; distinct values per head and channel."""
    rng = np.random.default_rng(101)
    levels = ((3, 5), (4, 2), (1, 6), (7, 1))
    B, N_q, N_h, C_h, N_p = 2, 7, 3, 4, 2
    N_l = len(levels)
    for align in (False, True):
        P = _problem(rng, levels, B, N_q, N_h, C_h, N_p)
        loc = np.empty((B, N_q, N_h, N_l, N_p, 2))
        attn = np.zeros((B, N_q, N_h, N_l, N_p))
        expect = np.empty((B, N_q, N_h, C_h))
        for b in range(B):
            for q in range(N_q):
                for h in range(N_h):
                    for l, (H, W) in enumerate(levels):
                        i = rng.integers(0, H, size=N_p)
                        j = rng.integers(0, W, size=N_p)
                        loc[b, q, h, l, :, 0] = _u_from_pixel(j.astype(float), W, align)
                        loc[b, q, h, l, :, 1] = _u_from_pixel(i.astype(float), H, align)
                        if align and W == 1:
                            loc[b, q, h, l, :, 0] = rng.uniform(0, 1, size=N_p)
                        if align and H == 1:
                            loc[b, q, h, l, :, 1] = rng.uniform(0, 1, size=N_p)
                    l, p = rng.integers(0, N_l), rng.integers(0, N_p)
                    attn[b, q, h, l, p] = 1.0
                    H, W = levels[l]
                    y = int(round(loc[b, q, h, l, p, 1] * (H - 1))) if align else \
                        int(round(loc[b, q, h, l, p, 1] * H - 0.5))
                    x = int(round(loc[b, q, h, l, p, 0] * (W - 1))) if align else \
                        int(round(loc[b, q, h, l, p, 0] * W - 0.5))
                    expect[b, q, h] = P["value"][b, P["starts"][l] + y * W + x, h]
        expect = expect.reshape(B, N_q, N_h * C_h)
        for pad in ("zeros", "border"):
            for vl in ("BLNC", "BNLC"):
                for ll in ("BQHLP2", "B2QHLP"):
                    out = orc.forward(gen.to_value_layout(P["value"], vl), levels, P["starts"],
                                      gen.to_loc_layout(loc, ll), attn, value_layout=vl,
                                      sampling_locations_layout=ll, align_corners=align,
                                      padding_mode=pad)
                    _close(out, expect, 1e-12, f"pixel centre align={align} {pad} {vl}/{ll}")


def pin_corner_points(orc):
    """align_corners=True: location (0,0) is the first pixel of a level and
    (1,1) its last pixel."""
    rng = np.random.default_rng(102)
    levels = ((3, 5), (6, 4))
    P = _problem(rng, levels, 1, 2, 2, 3, 1)
    loc = np.zeros((1, 2, 2, 2, 1, 2))
    loc[0, 1] = 1.0
    for l, (H, W) in enumerate(levels):
        attn = np.zeros((1, 2, 2, 2, 1))
        attn[:, :, :, l, 0] = 1.0
        out = _fwd(orc, P, loc=loc, attn=attn, align_corners=True).reshape(1, 2, 2, 3)
        m = _level_map(P["value"], P["starts"], levels, l)
        _close(out[0, 0], m[0, 0, 0], 1e-13, f"(0,0) level {l}")
        _close(out[0, 1], m[0, H - 1, W - 1], 1e-13, f"(1,1) level {l}")


def pin_affine_bilinear_closed_form(orc):
    """Bilinear interpolation reproduces a + b*x + c*y + d*x*y exactly.

    With value_l[y, x] = a + b x + c y + d x y (per level, head, channel) and
    in-bounds samples at pixel coordinates (x, y):
      out            = sum_s A_s (a + b x_s + c y_s + d x_s y_s)
      grad_attn_s    = <g, a + b x_s + c y_s + d x_s y_s>
      grad_loc_x_s   = A_s <g, b + d y_s> * dx/du,  grad_loc_y_s = A_s <g, c + d x_s> * dy/du
    where dx/du is W (align_corners=False) or W-1 (True)."""
    rng = np.random.default_rng(103)
    levels = ((4, 6), (5, 3), (2, 9))
    B, N_q, N_h, C_h, N_p = 2, 5, 2, 3, 3
    N_l = len(levels)
    for align in (False, True):
        for pad in ("zeros", "border"):
            P = _problem(rng, levels, B, N_q, N_h, C_h, N_p)
            coef = rng.standard_normal((N_l, 4, N_h, C_h))
            value = np.empty_like(P["value"])
            for l, (H, W) in enumerate(levels):
                ys, xs = np.meshgrid(np.arange(H, dtype=float), np.arange(W, dtype=float), indexing="ij")
                a, bb, c, d = coef[l]
                m = (a[None, None] + bb[None, None] * xs[..., None, None] + c[None, None] * ys[..., None, None]
                     + d[None, None] * (xs * ys)[..., None, None])
                value[:, P["starts"][l]:P["starts"][l] + H * W] = m.reshape(H * W, N_h, C_h)[None]
            xpix = np.empty((B, N_q, N_h, N_l, N_p))
            ypix = np.empty_like(xpix)
            loc = np.empty((B, N_q, N_h, N_l, N_p, 2))
            for l, (H, W) in enumerate(levels):
                xpix[..., l, :] = rng.uniform(0, W - 1, size=xpix[..., l, :].shape)
                ypix[..., l, :] = rng.uniform(0, H - 1, size=ypix[..., l, :].shape)
                loc[..., l, :, 0] = _u_from_pixel(xpix[..., l, :], W, align)
                loc[..., l, :, 1] = _u_from_pixel(ypix[..., l, :], H, align)
            attn, g = P["attn"], P["g"].reshape(B, N_q, N_h, C_h)
            S = np.empty((B, N_q, N_h, N_l, N_p, C_h))
            dSx = np.empty_like(S)
            dSy = np.empty_like(S)
            for l in range(N_l):
                a, bb, c, d = (coef[l, k][None, None, :, None, :] for k in range(4))
                x = xpix[..., l, :, None]
                y = ypix[..., l, :, None]
                S[..., l, :, :] = a + bb * x + c * y + d * x * y
                dSx[..., l, :, :] = bb + d * y
                dSy[..., l, :, :] = c + d * x
            expect_out = np.einsum("bqhlp,bqhlpc->bqhc", attn, S).reshape(B, N_q, N_h * C_h)
            kw = dict(align_corners=align, padding_mode=pad)
            _close(_fwd(orc, P, value=value, loc=loc, **kw), expect_out, 1e-12, f"affine out {align} {pad}")
            _, gl, ga = _bwd(orc, P, value=value, loc=loc, compute_grad_value=False, **kw)
            _close(ga, np.einsum("bqhc,bqhlpc->bqhlp", g, S), 1e-12, "affine grad_attn")
            sx = np.array([_du_dpix(W, align) for _, W in levels], dtype=float)[None, None, None, :, None]
            sy = np.array([_du_dpix(H, align) for H, _ in levels], dtype=float)[None, None, None, :, None]
            ex = attn * np.einsum("bqhc,bqhlpc->bqhlp", g, dSx) * sx
            ey = attn * np.einsum("bqhc,bqhlpc->bqhlp", g, dSy) * sy
            _close(gl[..., 0], ex, 1e-11, f"affine grad_loc x {align} {pad}")
            _close(gl[..., 1], ey, 1e-11, f"affine grad_loc y {align} {pad}")


def pin_constant_map(orc):
    """value == k_h everywhere and attention summing to 1: the output is k_h
    for in-bounds samples under both paddings, and for every sample under
    "border"; the location gradient of a constant map is 0."""
    rng = np.random.default_rng(104)
    levels = ((5, 7), (3, 4))
    B, N_q, N_h, C_h, N_p = 2, 6, 3, 2, 3
    P = _problem(rng, levels, B, N_q, N_h, C_h, N_p)
    k = rng.standard_normal(N_h)
    value = np.broadcast_to(k[None, None, :, None], P["value"].shape).copy()
    attn = P["attn"] / P["attn"].sum(axis=(3, 4), keepdims=True)
    expect = np.broadcast_to(np.repeat(k, C_h)[None, None], (B, N_q, N_h * C_h))
    for align in (False, True):
        loc_in = np.empty_like(P["loc"])
        for l, (H, W) in enumerate(levels):
            loc_in[..., l, :, 0] = _u_from_pixel(rng.uniform(0, W - 1, size=loc_in[..., l, :, 0].shape), W, align)
            loc_in[..., l, :, 1] = _u_from_pixel(rng.uniform(0, H - 1, size=loc_in[..., l, :, 1].shape), H, align)
        for pad in ("zeros", "border"):
            _close(_fwd(orc, P, value=value, loc=loc_in, attn=attn, align_corners=align, padding_mode=pad),
                   expect, 1e-13, f"constant in-bounds {align} {pad}")
            _, gl, _ = _bwd(orc, P, value=value, loc=loc_in, attn=attn, align_corners=align,
                            padding_mode=pad, compute_grad_value=False, compute_grad_attention_weights=False)
            _close(gl, np.zeros_like(gl), 1e-12, "constant map grad_loc")
        loc_any = rng.uniform(-3.0, 4.0, size=P["loc"].shape)
        _close(_fwd(orc, P, value=value, loc=loc_any, attn=attn, align_corners=align, padding_mode="border"),
               expect, 1e-13, f"constant border anywhere {align}")


def pin_zeros_padding(orc):
    """"zeros": a sample whose pixel coordinate is <= -1 or >= W (or the same
    in y) reads only outside the map and returns exactly 0 with zero
    gradients; a sample half a pixel outside the first/last column (pixel
    coordinate -0.5 or W-0.5, i.e. u = 0 or 1 with align_corners=False) at a
    row centre returns half of the edge pixel."""
    rng = np.random.default_rng(105)
    levels = ((4, 6),)
    H, W = levels[0]
    B, N_q, N_h, C_h, N_p = 1, 8, 2, 3, 1
    P = _problem(rng, levels, B, N_q, N_h, C_h, N_p)
    attn = np.ones((B, N_q, N_h, 1, N_p))
    far = np.array([-1.0, W + 0.0, W + 3.7, -1e6, 1e6, -2.5, 1e30, -1e30])
    for axis in (0, 1):
        loc = np.empty((B, N_q, N_h, 1, N_p, 2))
        size = W if axis == 0 else H
        other = H if axis == 0 else W
        pix = far.copy()
        pix[1] = size
        loc[..., 0, 0, axis] = _u_from_pixel(pix, size, False)[None, :, None]
        loc[..., 0, 0, 1 - axis] = _u_from_pixel(rng.uniform(0, other - 1, size=(N_q, N_h)), other, False)[None]
        out = _fwd(orc, P, loc=loc, attn=attn, padding_mode="zeros")
        assert np.all(out == 0.0), f"zeros padding outside the map (axis {axis}) is not 0"
        # At exactly -1 the cell [-1, 0] is used and its right-sided
        # derivative is not 0; strictly below -1 every corner is outside.
        loc[0, 0, :, 0, 0, axis] = _u_from_pixel(np.float64(-1.25), size, False)
        gv, gl, ga = _bwd(orc, P, loc=loc, attn=attn, padding_mode="zeros")
        assert np.all(gv == 0.0) and np.all(gl == 0.0) and np.all(ga == 0.0), "zeros padding gradients"
    # half a pixel outside the first / last column, at the centre of row i
    m = _level_map(P["value"], P["starts"], levels, 0)
    for u, col in ((0.0, 0), (1.0, W - 1)):
        loc = np.empty((B, N_q, N_h, 1, N_p, 2))
        rows = rng.integers(0, H, size=N_q)
        loc[..., 0] = u
        loc[0, :, :, 0, 0, 1] = ((rows + 0.5) / H)[:, None]
        out = _fwd(orc, P, loc=loc, attn=attn, padding_mode="zeros").reshape(N_q, N_h, C_h)
        _close(out, 0.5 * m[0, rows, col], 1e-13, f"half-pixel edge u={u}")


def pin_border_padding(orc):
    """"border": far outside the map a sample returns the nearest edge pixel
    (corners for both axes outside), and its location gradient along a
    clamped axis is 0."""
    rng = np.random.default_rng(106)
    levels = ((4, 6), (3, 2))
    B, N_q, N_h, C_h, N_p = 1, 4, 2, 3, 1
    P = _problem(rng, levels, B, N_q, N_h, C_h, N_p)
    for align in (False, True):
        for l, (H, W) in enumerate(levels):
            m = _level_map(P["value"], P["starts"], levels, l)
            attn = np.zeros((B, N_q, N_h, 2, N_p))
            attn[..., l, :] = 1.0
            loc = np.zeros((B, N_q, N_h, 2, N_p, 2))
            loc[0, 0, :, l, 0] = (-5.0, -5.0)
            loc[0, 1, :, l, 0] = (5.0, 5.0)
            loc[0, 2, :, l, 0] = (-1e6, 5.0)
            loc[0, 3, :, l, 0] = (1e30, -1e30)
            out = _fwd(orc, P, loc=loc, attn=attn, align_corners=align, padding_mode="border")
            out = out.reshape(N_q, N_h, C_h)
            _close(out[0], m[0, 0, 0], 1e-14, "border (-,-)")
            _close(out[1], m[0, H - 1, W - 1], 1e-14, "border (+,+)")
            _close(out[2], m[0, H - 1, 0], 1e-14, "border (-,+)")
            _close(out[3], m[0, 0, W - 1], 1e-14, "border (+,-)")
            _, gl, _ = _bwd(orc, P, loc=loc, attn=attn, align_corners=align, padding_mode="border")
            assert np.all(gl == 0.0), "border: gradient along a clamped axis is not 0"
            # x clamped, y inside: the sample equals the edge column's linear interpolation in y
            loc2 = np.zeros((B, N_q, N_h, 2, N_p, 2))
            ypix = rng.uniform(0, H - 1, size=(N_q,))
            loc2[0, :, :, l, 0, 0] = -7.0
            loc2[0, :, :, l, 0, 1] = _u_from_pixel(ypix, H, align)[:, None]
            out2 = _fwd(orc, P, loc=loc2, attn=attn, align_corners=align, padding_mode="border")
            y0 = np.floor(ypix).astype(int)
            y1 = np.minimum(y0 + 1, H - 1)
            fy = (ypix - y0)[:, None, None]
            expect = (1 - fy) * m[0, y0, 0] + fy * m[0, y1, 0]
            _close(out2.reshape(N_q, N_h, C_h), expect, 1e-13, "border clamped column")
            _, gl2, _ = _bwd(orc, P, loc=loc2, attn=attn, align_corners=align, padding_mode="border",
                             compute_grad_value=False, compute_grad_attention_weights=False)
            assert np.all(gl2[..., l, :, 0] == 0.0), "border: x gradient not 0 when x is clamped"


def pin_grid_sample(orc):
    """One level and one point with weight 1 is the textbook bilinear sampler:
    torch.nn.functional.grid_sample(value_l, grid = 2*loc - 1) (CPU, float64),
    forward and -- through autograd -- grad_value and grad_loc
    (d grid / d loc = 2), for both paddings and both align_corners."""
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(107)
    H, W = 5, 7
    B, N_q, N_h, C_h = 2, 9, 3, 4
    for align in (False, True):
        for pad in ("zeros", "border"):
            P = _problem(rng, ((H, W),), B, N_q, N_h, C_h, 1, loc_lo=-0.25, loc_hi=1.25)
            attn = np.ones((B, N_q, N_h, 1, 1))
            img = torch.tensor(P["value"].reshape(B, H, W, N_h, C_h).transpose(0, 3, 4, 1, 2)
                               .reshape(B * N_h, C_h, H, W), dtype=torch.float64, requires_grad=True)
            grid = torch.tensor((2.0 * P["loc"][:, :, :, 0, 0, :] - 1.0).transpose(0, 2, 1, 3)
                                .reshape(B * N_h, N_q, 1, 2), dtype=torch.float64, requires_grad=True)
            ref = F.grid_sample(img, grid, mode="bilinear", padding_mode=pad, align_corners=align)
            ref_out = ref.detach().numpy().reshape(B, N_h, C_h, N_q).transpose(0, 3, 1, 2).reshape(B, N_q, N_h * C_h)
            _close(_fwd(orc, P, attn=attn, align_corners=align, padding_mode=pad), ref_out, 1e-12,
                   f"grid_sample fwd {align} {pad}")
            gt = torch.tensor(P["g"].reshape(B, N_q, N_h, C_h).transpose(0, 2, 3, 1).reshape(B * N_h, C_h, N_q, 1))
            (ref * gt).sum().backward()
            gv, gl, ga = _bwd(orc, P, attn=attn, align_corners=align, padding_mode=pad)
            ref_gv = img.grad.numpy().reshape(B, N_h, C_h, H, W).transpose(0, 3, 4, 1, 2).reshape(B, H * W, N_h, C_h)
            ref_gl = 2.0 * grid.grad.numpy().reshape(B, N_h, N_q, 2).transpose(0, 2, 1, 3)
            _close(gv, ref_gv, 1e-12, f"grid_sample grad_value {align} {pad}")
            _close(gl[:, :, :, 0, 0, :], ref_gl, 1e-11, f"grid_sample grad_loc {align} {pad}")
            _close(ga[..., 0, 0], np.einsum("bqhc,bqhc->bqh", P["g"].reshape(B, N_q, N_h, C_h),
                                              ref_out.reshape(B, N_q, N_h, C_h)), 1e-12, "grid_sample grad_attn")


def pin_linearity(orc):
    """out is linear in value and in attention_weights."""
    rng = np.random.default_rng(108)
    levels = ((5, 4), (2, 3))
    P = _problem(rng, levels, 2, 4, 2, 3, 2)
    V2 = rng.standard_normal(P["value"].shape)
    A2 = rng.uniform(0, 1, size=P["attn"].shape)
    al, be = 0.7, -1.3
    for pad in ("zeros", "border"):
        kw = dict(padding_mode=pad)
        _close(_fwd(orc, P, value=al * P["value"] + be * V2, **kw),
               al * _fwd(orc, P, **kw) + be * _fwd(orc, P, value=V2, **kw), 1e-12, "linear in value")
        _close(_fwd(orc, P, attn=al * P["attn"] + be * A2, **kw),
               al * _fwd(orc, P, **kw) + be * _fwd(orc, P, attn=A2, **kw), 1e-12, "linear in attention")


def pin_layouts(orc):
    """BNLC / B2QHLP give the same numbers as BLNC / BQHLP2 on the permuted
    tensors, forward and all three gradients (returned in the input's layout)."""
    rng = np.random.default_rng(109)
    levels = ((4, 5), (3, 3))
    P = _problem(rng, levels, 2, 5, 3, 2, 2)
    for pad in ("zeros", "border"):
        base = _fwd(orc, P, padding_mode=pad)
        bgv, bgl, bga = _bwd(orc, P, padding_mode=pad)
        for vl in ("BLNC", "BNLC"):
            for ll in ("BQHLP2", "B2QHLP"):
                v = gen.to_value_layout(P["value"], vl)
                loc = gen.to_loc_layout(P["loc"], ll)
                kw = dict(value_layout=vl, sampling_locations_layout=ll, padding_mode=pad)
                _close(orc.forward(v, levels, P["starts"], loc, P["attn"], **kw), base, 1e-14, "layout fwd")
                gv, gl, ga = orc.backward(P["g"], v, levels, P["starts"], loc, P["attn"], **kw)
                _close(gen.from_value_layout(gv, vl), bgv, 1e-14, f"layout grad_value {vl}")
                _close(gen.from_loc_layout(gl, ll), bgl, 1e-14, f"layout grad_loc {ll}")
                _close(ga, bga, 1e-14, "layout grad_attn")


def pin_grad_attention_is_sample_dot(orc):
    """grad_attention_weights[s] = <g, S_s>, with S_s read off a forward call
    whose attention is one-hot at (l, p); and sum_s A_s grad_attn_s = <g, out>."""
    rng = np.random.default_rng(110)
    levels = ((4, 6), (3, 2))
    B, N_q, N_h, C_h, N_p = 2, 4, 2, 3, 2
    for pad in ("zeros", "border"):
        P = _problem(rng, levels, B, N_q, N_h, C_h, N_p, loc_lo=-0.3, loc_hi=1.3)
        _, _, ga = _bwd(orc, P, padding_mode=pad)
        g = P["g"].reshape(B, N_q, N_h, C_h)
        for l in range(len(levels)):
            for p in range(N_p):
                onehot = np.zeros_like(P["attn"])
                onehot[..., l, p] = 1.0
                S = _fwd(orc, P, attn=onehot, padding_mode=pad).reshape(B, N_q, N_h, C_h)
                _close(ga[..., l, p], np.einsum("bqhc,bqhc->bqh", g, S), 1e-13, f"grad_attn (l={l},p={p})")
        out = _fwd(orc, P, padding_mode=pad).reshape(B, N_q, N_h, C_h)
        _close(np.einsum("bqhlp,bqhlp->bqh", ga, P["attn"]), np.einsum("bqhc,bqhc->bqh", g, out),
               1e-12, "sum A*grad_attn = <g,out>")


def pin_adjoint(orc):
    """out is linear in value, so <grad_value, V'> = <g, out(V')> for any V'."""
    rng = np.random.default_rng(111)
    levels = ((6, 5), (3, 3), (2, 1))
    for pad in ("zeros", "border"):
        for align in (False, True):
            P = _problem(rng, levels, 2, 7, 2, 3, 3, loc_lo=-0.2, loc_hi=1.2)
            gv, _, _ = _bwd(orc, P, padding_mode=pad, align_corners=align,
                            compute_grad_sampling_locations=False, compute_grad_attention_weights=False)
            for _ in range(3):
                Vp = rng.standard_normal(P["value"].shape)
                lhs = float(np.sum(gv * Vp))
                rhs = float(np.sum(P["g"] * _fwd(orc, P, value=Vp, padding_mode=pad, align_corners=align)))
                assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(rhs)), f"adjoint {pad} {align}: {lhs} vs {rhs}"


def pin_finite_differences(orc):
    """Central differences of J = <g, out> match every gradient.

    The sample is affine in each pixel coordinate inside one bilinear cell, so
    with step h the difference is exact up to rounding as long as no integer
    pixel line lies within h of the coordinate (such coordinates are skipped).
    J is linear in value and in attention, so those differences are exact."""
    rng = np.random.default_rng(112)
    levels = ((5, 7), (3, 4))
    B, N_q, N_h, C_h, N_p = 1, 3, 2, 3, 2
    h = 1e-7
    for pad in ("zeros", "border"):
        for align in (False, True):
            P = _problem(rng, levels, B, N_q, N_h, C_h, N_p, loc_lo=-0.15, loc_hi=1.15)
            kw = dict(padding_mode=pad, align_corners=align)
            gv, gl, ga = _bwd(orc, P, **kw)

            def J(**over):
                return float(np.sum(P["g"] * _fwd(orc, P, **over, **kw)))

            checked = 0
            for idx in np.ndindex(*P["loc"].shape):
                l, axis = idx[3], idx[5]
                H, W = levels[l]
                size = W if axis == 0 else H
                pix = P["loc"][idx] * _du_dpix(size, align) - (0.0 if align else 0.5)
                if abs(pix - np.round(pix)) < 20 * h * size:
                    continue
                lp, lm = P["loc"].copy(), P["loc"].copy()
                lp[idx] += h
                lm[idx] -= h
                fd = (J(loc=lp) - J(loc=lm)) / (2 * h)
                assert abs(fd - gl[idx]) <= 1e-6 * max(1.0, abs(gl[idx])), f"FD loc {idx}: {fd} vs {gl[idx]}"
                checked += 1
            assert checked > 0.8 * P["loc"].size
            for idx in list(np.ndindex(*P["attn"].shape))[::3]:
                ap, am = P["attn"].copy(), P["attn"].copy()
                ap[idx] += 0.5
                am[idx] -= 0.5
                fd = J(attn=ap) - J(attn=am)
                assert abs(fd - ga[idx]) <= 1e-12 * max(1.0, abs(ga[idx])), f"FD attn {idx}"
            for idx in [tuple(rng.integers(0, s) for s in P["value"].shape) for _ in range(25)]:
                vp, vm = P["value"].copy(), P["value"].copy()
                vp[idx] += 0.5
                vm[idx] -= 0.5
                fd = J(value=vp) - J(value=vm)
                assert abs(fd - gv[idx]) <= 1e-12 * max(1.0, abs(gv[idx])), f"FD value {idx}"


def pin_compute_flags(orc):
    """compute_grad_* select outputs independently (a disabled output is not
    produced) and do not change the enabled ones; all three off is rejected
    ("at least one ... must be True")."""
    rng = np.random.default_rng(113)
    P = _problem(rng, ((4, 4), (2, 3)), 1, 3, 2, 2, 2)
    full = _bwd(orc, P)
    for flags in [(1, 0, 0), (0, 1, 0), (0, 0, 1), (1, 1, 0), (0, 1, 1), (1, 0, 1)]:
        got = _bwd(orc, P, compute_grad_value=bool(flags[0]), compute_grad_sampling_locations=bool(flags[1]),
                   compute_grad_attention_weights=bool(flags[2]))
        for f, a, b in zip(flags, got, full):
            if f:
                _close(a, b, 0.0, f"flags {flags}")
            else:
                assert a is None
    try:
        _bwd(orc, P, compute_grad_value=False, compute_grad_sampling_locations=False,
             compute_grad_attention_weights=False)
    except ValueError:
        pass
    else:
        raise AssertionError("all compute_grad_* False was accepted")


def pin_hand_worked_example(orc):
    """The hand-computed fixture tests/golden/hand_worked.json (every number
    derived on paper from the pages' definitions; the derivation is in the
    file)."""
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        case = json.load(f)
    value = np.array(case["value_BLNC"], dtype=float)
    loc = np.array(case["sampling_locations_BQHLP2"], dtype=float)
    attn = np.array(case["attention_weights"], dtype=float)
    g = np.array(case["grad_output"], dtype=float)
    shapes = [tuple(s) for s in case["spatial_shapes"]]
    starts = case["level_start_index"]
    for exp in case["expected"]:
        kw = dict(align_corners=exp["align_corners"], padding_mode=exp["padding_mode"])
        out = orc.forward(value, shapes, starts, loc, attn, **kw)
        _close(out, np.array(exp["out"]), 0.0, f"hand-worked out {kw}")
        if "grad_value" in exp:
            gv, gl, ga = orc.backward(g, value, shapes, starts, loc, attn, **kw)
            _close(gv, np.array(exp["grad_value"]), 0.0, f"hand-worked grad_value {kw}")
            _close(gl, np.array(exp["grad_sampling_locations"]), 0.0, f"hand-worked grad_loc {kw}")
            _close(ga, np.array(exp["grad_attention_weights"]), 0.0, f"hand-worked grad_attn {kw}")


def pin_cell_decision_in_binary32(orc):
    """coord_f32 rounds the pixel coordinate to binary32 before floor(): a
    binary32 location whose exact pixel coordinate lies just below the integer
    k but rounds to k takes the cell [k, k+1] (one-sided derivative from the
    right), while exact arithmetic takes [k-1, k].  On value[x] = x^2 the two
    slopes are 2k+1 and 2k-1."""
    W = 167
    found = None
    for k in range(2, W - 2):
        u0 = np.float32((k + 0.5) / W)
        for step in range(-4, 5):
            u = np.nextafter(u0, np.float32(np.inf if step > 0 else -np.inf), dtype=np.float32) if step else u0
            for _ in range(abs(step) - 1):
                u = np.nextafter(u, np.float32(np.inf if step > 0 else -np.inf), dtype=np.float32)
            x = float(u) * W - 0.5
            if x < k and float(np.float32(x)) == float(k):
                found = (k, float(u))
                break
        if found:
            break
    assert found is not None
    k, u = found
    levels = ((1, W),)
    value = (np.arange(W, dtype=float) ** 2).reshape(1, W, 1, 1)
    loc = np.array([u, 0.5]).reshape(1, 1, 1, 1, 1, 2)
    attn = np.ones((1, 1, 1, 1, 1))
    g = np.ones((1, 1, 1))
    _, gl_exact, _ = orc.backward(g, value, levels, (0,), loc, attn, coord_f32=False)
    _, gl_f32, _ = orc.backward(g, value, levels, (0,), loc, attn, coord_f32=True)
    assert gl_exact[0, 0, 0, 0, 0, 0] == (2 * k - 1) * W, gl_exact
    assert gl_f32[0, 0, 0, 0, 0, 0] == (2 * k + 1) * W, gl_f32
    out_f32 = orc.forward(value, levels, (0,), loc, attn, coord_f32=True)
    assert out_f32[0, 0, 0] == float(k * k)


def pin_attention_logits(orc):
    """Attention logits (the fused softmax producer): the weights are a
    softmax over each (b, q, h)'s N_l*N_p slots.  Pinned by: equal logits give
    equal weights 1/(N_l*N_p); adding a constant to a row's logits changes
    nothing; one dominant logit selects that sample; the logits' gradient sums
    to zero over every row and matches central differences of <g, out>."""
    rng = np.random.default_rng(131)
    levels = ((5, 7), (3, 4))
    B, N_q, N_h, C_h, N_p = 2, 3, 2, 3, 2
    P = _problem(rng, levels, B, N_q, N_h, C_h, N_p)
    nlp = len(levels) * N_p
    z = rng.standard_normal(P["attn"].shape)
    kw = dict(padding_mode="zeros", align_corners=False)

    def fwd_z(zz):
        return orc.forward_logits(P["value"], P["levels"], P["starts"], P["loc"], zz, **kw)

    # equal logits
    _close(fwd_z(np.full_like(z, 0.3)), _fwd(orc, P, attn=np.full_like(z, 1.0 / nlp), **kw), 1e-14, "equal logits")
    # row shift
    shift = rng.standard_normal(z.shape[:3])[..., None, None] * 5.0
    _close(fwd_z(z + shift), fwd_z(z), 1e-13, "row shift")
    # one dominant logit: sample (l=1, p=0) of every row
    zd = np.zeros_like(z)
    zd[..., 1, 0] = 60.0
    onehot = np.zeros_like(z)
    onehot[..., 1, 0] = 1.0
    _close(fwd_z(zd), _fwd(orc, P, attn=onehot, **kw), 1e-13, "dominant logit")
    # gradient: rows sum to zero; central differences of J = <g, out>
    gv, gl, gz = orc.backward_logits(P["g"], P["value"], P["levels"], P["starts"], P["loc"], z, **kw)
    assert np.max(np.abs(gz.reshape(B, N_q, N_h, -1).sum(-1))) < 1e-12, "logit gradient rows must sum to 0"
    h = 1e-5
    for idx in np.ndindex(*z.shape):
        zp, zm = z.copy(), z.copy()
        zp[idx] += h
        zm[idx] -= h
        fd = (np.sum(P["g"] * fwd_z(zp)) - np.sum(P["g"] * fwd_z(zm))) / (2 * h)
        assert abs(fd - gz[idx]) <= 1e-8 * max(1.0, abs(gz[idx])), f"FD logits {idx}: {fd} vs {gz[idx]}"
    # grad_value / grad_loc are those of the softmaxed weights
    A = np.exp(z - z.max(axis=(-2, -1), keepdims=True))
    A /= A.sum(axis=(-2, -1), keepdims=True)
    gv2, gl2, _ = _bwd(orc, P, attn=A, **kw)
    _close(gv, gv2, 1e-13, "grad_value with logits")
    _close(gl, gl2, 1e-13, "grad_loc with logits")


ALL_PINS = [
    pin_pixel_centre, pin_corner_points, pin_affine_bilinear_closed_form, pin_constant_map,
    pin_zeros_padding, pin_border_padding, pin_grid_sample, pin_linearity, pin_layouts,
    pin_grad_attention_is_sample_dot, pin_adjoint, pin_finite_differences, pin_compute_flags,
    pin_hand_worked_example, pin_cell_decision_in_binary32, pin_attention_logits,
]
