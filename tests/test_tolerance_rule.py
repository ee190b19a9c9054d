"""The parity rule itself (CPU only): it must catch an error confined to the
fine level of the bfloat16 workloads' grad_value, which a floor of max|ref|
over the whole tensor let through.

The reference is the oracle's grad_value of the encoder workload with
bfloat16 value and gradients (one batch item); the "GPU" side is that
reference rounded to bfloat16 as the kernels store it, with a planted
mistake.  Rule: "MS Deformable Attention Backward Kernel API Reference",
Returns (grad_value has value's shape; each pyramid level is a slice of it).
"""
import numpy as np
import pytest

from parity_util import RTOL, assert_close, tensor_groups
from scale_deformable_attention_forward_gb300 import inputs as gen


@pytest.fixture(scope="module")
def encoder16_grad_value():
    import oracle
    w = gen.WORKLOADS["encoder16"].with_(B=1)
    d = gen.generate(w)
    kw = dict(value_layout=w.value_layout, sampling_locations_layout=w.loc_layout,
              align_corners=w.align_corners, padding_mode=w.padding_mode)
    gv = oracle.backward(d["grad_output"], d["value"], d["spatial_shapes"], d["level_start_index"],
                         d["sampling_locations"], d["attention_weights"], compute_grad_sampling_locations=False,
                         compute_grad_attention_weights=False, coord_f32=True, **kw)[0]
    return w, gv


def _level0(w):
    n0 = w.levels[0][0] * w.levels[0][1]
    return (slice(None), slice(None), slice(0, n0)) if w.value_layout == "BNLC" else (slice(None), slice(0, n0))


def test_rounded_reference_passes(encoder16_grad_value):
    w, ref = encoder16_grad_value
    stored = gen.round_to_bf16(ref).astype(np.float64)  # what a correct kernel stores
    assert_close(stored, ref, RTOL[("bf16", "bwd")], "rounded", groups=tensor_groups(w, "grad_value"))


def test_level0_scale_error_fails(encoder16_grad_value):
    """A 5% scale error on level 0 only, in bfloat16: the per-level rule
    rejects it, while the old global max|ref| floor did not."""
    w, ref = encoder16_grad_value
    bad = ref.copy()
    bad[_level0(w)] *= 1.05
    bad = gen.round_to_bf16(bad).astype(np.float64)
    rtol = RTOL[("bf16", "bwd")]
    old_bound = rtol * (np.abs(ref) + np.max(np.abs(ref)))
    assert np.all(np.abs(bad - ref) <= old_bound), "the planted error was meant to pass the old rule"
    with pytest.raises(AssertionError):
        assert_close(bad, ref, rtol, "planted", groups=tensor_groups(w, "grad_value"))


def test_level0_noise_fails(encoder16_grad_value):
    """Level-0 elements off by noise of 5% of that level's RMS (no scale
    change) are caught by the per-group norm check."""
    w, ref = encoder16_grad_value
    rng = np.random.default_rng(0)
    bad = ref.copy()
    sl = _level0(w)
    lvl = bad[sl]
    bad[sl] = lvl + 0.05 * np.sqrt(np.mean(lvl * lvl)) * rng.standard_normal(lvl.shape)
    with pytest.raises(AssertionError):
        assert_close(bad, ref, RTOL[("bf16", "bwd")], "planted noise", groups=tensor_groups(w, "grad_value"))


def test_groups_cover_every_element():
    """Every element of each tensor lies in exactly one comparison group."""
    for name in ("encoder32", "encoder16", "hires16"):
        w = gen.WORKLOADS[name].with_(B=1)
        Q, H, C, Nl, Np, L = w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L
        shapes = {
            "grad_value": (1, L, H, C) if w.value_layout == "BLNC" else (1, H, L, C),
            "grad_sampling_locations": (1, Q, H, Nl, Np, 2) if w.loc_layout == "BQHLP2" else (1, 2, Q, H, Nl, Np),
            "grad_attention_weights": (1, Q, H, Nl, Np),
            "out": (1, Q, H * C),
        }
        for t, shp in shapes.items():
            cover = np.zeros(shp, dtype=np.int32)
            for idx in tensor_groups(w, t):
                cover[idx] += 1
            assert np.all(cover == 1), f"{name} {t}"
