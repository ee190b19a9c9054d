"""The kernels at the largest problem the library accepts (GPU).

The C ABI bounds the value map so that every element offset the kernels form
in 32-bit arithmetic stays below 2^31: (L + 2*max(W) + 4) * N_h * C_h <
2^31 - 1.  These tests run a value map just inside that bound -- one level of
1021 x 1024 pixels (one row more is refused), N_h = 8 heads of C_h = 256
channels, 2.14e9 elements -- with samples crowded into the last rows and
columns (the largest offsets) and beyond the edge (clamped / zero corners),
in both value layouts.

Every output of a head depends on that head's slice of value only, so the
oracle checks the last head (whose offsets are the largest) as a one-head
problem: its forward output, all three gradients of that head -- grad_value
element by element over the whole slice -- against the float64 oracle.
Inputs are drawn on the GPU from a seeded generator; the oracle receives the
same numbers.
"""
import numpy as np
import pytest

from parity_util import RTOL, assert_close, np64

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

H, W = 1021, 1024
N_h, C_h, N_q, N_p, B = 8, 256, 48, 4, 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_forward_gb300 import build
    build.build()


def _inputs(vl, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    L = H * W
    vt = torch.bfloat16 if dtype == "bf16" else torch.float32
    shape = (B, L, N_h, C_h) if vl == "BLNC" else (B, N_h, L, C_h)
    value = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(vt)
    # half the points in the last 3% of rows and columns, a quarter anywhere, a quarter past the edge
    u = torch.rand((B, N_q, N_h, 1, N_p, 2), generator=g, device="cuda")
    far = 0.97 + 0.03 * u
    anywhere = u
    past = 0.99 + 0.03 * u
    pick = torch.arange(N_p, device="cuda").view(1, 1, 1, 1, N_p, 1) % 4
    loc = torch.where(pick < 2, far, torch.where(pick == 2, anywhere, past)).contiguous()
    logits = torch.randn((B, N_q, N_h, 1, N_p), generator=g, device="cuda")
    attn = torch.softmax(logits.view(B, N_q, N_h, N_p), -1).view(B, N_q, N_h, 1, N_p).contiguous()
    go = torch.randn((B, N_q, N_h * C_h), generator=g, device="cuda", dtype=torch.float32).to(vt)
    return value, loc, attn, go


@pytest.mark.parametrize("vl,dtype,pad,align", [("BLNC", "f32", "zeros", False), ("BNLC", "f32", "border", True),
                                                ("BLNC", "bf16", "border", False)])
def test_largest_value_map(vl, dtype, pad, align):
    import scale_deformable_attention_forward_gb300 as msda
    L = H * W
    assert (L + 2 * W + 4) * N_h * C_h < 2**31 - 1 < (L + W + 2 * W + 4) * N_h * C_h  # the largest height accepted
    value, loc, attn, go = _inputs(vl, dtype, seed=501)
    kw = dict(value_layout=vl, sampling_locations_layout="BQHLP2", align_corners=align, padding_mode=pad)
    shapes, starts = ((H, W),), (0,)
    out = msda.msda_forward(value, shapes, starts, loc, attn, **kw)
    gv, gl, ga = msda.msda_backward(go, value, shapes, starts, loc, attn, **kw)
    torch.cuda.synchronize()

    h = N_h - 1  # the last head: the largest offsets
    v_h = value[:, :, h:h + 1, :] if vl == "BLNC" else value[:, h:h + 1, :, :]
    d = {
        "value": np64(v_h.contiguous()),
        "sampling_locations": np64(loc[:, :, h:h + 1]),
        "attention_weights": np64(attn[:, :, h:h + 1]),
        "grad_output": np64(go[:, :, h * C_h:(h + 1) * C_h].contiguous()),
    }
    okw = dict(value_layout=vl, sampling_locations_layout="BQHLP2", align_corners=align, padding_mode=pad,
               coord_f32=True)
    ref_out = oracle.forward(d["value"], shapes, starts, d["sampling_locations"], d["attention_weights"], **okw)
    rt = RTOL[(dtype, "fwd")]
    assert_close(np64(out[:, :, h * C_h:(h + 1) * C_h].contiguous()), ref_out, rt, "out, last head")
    ref = oracle.backward(d["grad_output"], d["value"], shapes, starts, d["sampling_locations"],
                          d["attention_weights"], **okw)
    rb = RTOL[(dtype, "bwd")]
    gv_h = gv[:, :, h:h + 1, :] if vl == "BLNC" else gv[:, h:h + 1, :, :]
    assert_close(np64(gv_h.contiguous()), ref[0], rb, "grad_value, last head")
    assert_close(np64(gl[:, :, h:h + 1]), ref[1], rb, "grad_sampling_locations, last head")
    assert_close(np64(ga[:, :, h:h + 1]), ref[2], rb, "grad_attention_weights, last head")
    # the corners near the end of the map were actually read and written
    assert float(np.abs(ref[0][0, -W:] if vl == "BLNC" else ref[0][0, 0, -W:]).max()) > 0.0
    del value, gv, out
    torch.cuda.empty_cache()


def test_one_row_too_many_is_rejected():
    """One more row than the largest accepted map: refused before any launch."""
    import scale_deformable_attention_forward_gb300 as msda
    lib = msda.load_library()
    Hb = H + 1
    desc = msda.make_desc((B, N_q, N_h, C_h, 1, N_p, Hb * W), ((Hb, W),), (0,))
    out = torch.empty(1, device="cuda")
    rc = lib.msda_forward(desc.ref(), out.data_ptr(), out.data_ptr(), out.data_ptr(), out.data_ptr(), None)
    assert rc == -7
