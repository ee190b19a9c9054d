"""Planted mistakes in the oracle must be caught by the pins (CPU only).

Each case copies ``oracle/msda_oracle.c`` to a temporary directory, applies
one plausible slip (a dropped term, a wrong sign, a transposed index, a wrong
scale, a wrong layout), compiles the copy and runs the pin suite against it.
At least one pin has to fail; otherwise the pins would not notice that slip in
the real oracle either.  Every mutation keeps memory accesses in bounds.
"""
import os

import pytest

import oracle
import oracle_pins

MUTATIONS = {
    "x/y weights confused": ("const double wx[4] = {1.0 - fx, fx, 1.0 - fx, fx};",
                             "const double wx[4] = {1.0 - fx, 1.0 - fx, fx, fx};"),
    "no half-pixel shift": ("u * (double)size - 0.5", "u * (double)size"),
    "align_corners scale W": ("u * (double)(size - 1)", "u * (double)size"),
    "gradient scale W-1 always": ("P->align_corners ? (double)(size - 1) : (double)size",
                                  "(double)(size - 1)"),
    "border clamps one short": ("ix > (double)(W - 1) ? (double)(W - 1) : ix",
                                "ix > (double)(W - 1) ? (double)(W - 2) : ix"),
    "zeros drops column 0": ("ix >= 0.0 && ix <= (double)(W - 1)", "ix >= 1.0 && ix <= (double)(W - 1)"),
    "x derivative sign": ("const double dwx[4] = {-1.0, 1.0, -1.0, 1.0};",
                          "const double dwx[4] = {1.0, -1.0, 1.0, -1.0};"),
    "grad_attn drops weight": ("s += k.w[i] * gv[i];", "s += gv[i];"),
    "grad_value drops A": ("A * k.w[i] * g[c];", "k.w[i] * g[c];"),
    "grad_loc drops A": ("grad_loc[loc_offset(&P, b, q, h, l, p, 0)] = A * sx",
                         "grad_loc[loc_offset(&P, b, q, h, l, p, 0)] = sx"),
    "BNLC read as BLNC": ("return ((b * P->N_h + h) * P->L + pix) * P->C_h + c;",
                          "return ((b * P->L + pix) * P->N_h + h) * P->C_h + c;"),
    "B2QHLP x/y swapped": ("return ((((b * 2 + xy) * P->N_q", "return ((((b * 2 + (1 - xy)) * P->N_q"),
    "BQHLP2 x/y swapped": ("* P->N_p + p) * 2) + xy;", "* P->N_p + p) * 2) + (1 - xy);"),
    "output channel-major": ("h * P->C_h + c;\n}", "c * P->N_h + h;\n}"),
    "forward ignores attention": ("out[out_offset(&P, b, q, h, c)] += A * S[c];",
                                  "out[out_offset(&P, b, q, h, c)] += S[c];"),
    "round instead of floor": ("const double x0 = floor(x), y0 = floor(y);",
                               "const double x0 = round(x), y0 = round(y);"),
    "y gradient scaled by W": ("A * sy * pixel_scale(&P, H)", "A * sy * pixel_scale(&P, W)"),
    "binary32 decision ignored": ("t = (double)(float)t;", "t = t;"),
    "level start ignored": ("P->starts[l] + (int64_t)iy * W + (int64_t)ix",
                            "(int64_t)iy * W + (int64_t)ix"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    mutant = oracle.Oracle(oracle.build(force=True, src=path, out=os.path.join(tmp_path, "libmutant.so")))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError) as e:
            caught.append((pin.__name__, str(e)[:80]))
            break
    assert caught, f"no pin caught the planted mistake {name!r}"
