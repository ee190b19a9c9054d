"""The seeded workload generator (CPU only)."""
import numpy as np
import pytest

from scale_deformable_attention_forward_gb300 import inputs as gen


def test_workload_table():
    w = gen.WORKLOADS
    assert w["tiny"].L == 80 and w["tiny"].samples == 1 * 16 * 2 * 2 * 2
    assert w["decoder"].L == 22223 and w["decoder"].samples == 76800
    assert w["encoder32"].n_queries == 22223 and w["encoder32"].samples == 5689088
    assert w["encoder16"].samples == 22756352 and w["encoder16"].value_layout == "BNLC"
    assert w["hires16"].L == 21760 and w["hires16"].samples == 22282240
    assert w["decoder"].level_start_index == (0, 16700, 20900, 21950)
    assert sorted(v.seed for v in w.values()) == [0, 1, 2, 3, 4]


def test_deterministic_and_layout_independent():
    w = gen.WORKLOADS["tiny"]
    a, b = gen.generate(w), gen.generate(w)
    for k in ("value", "sampling_locations", "attention_weights", "grad_output"):
        assert np.array_equal(a[k], b[k])
    c = gen.generate(w.with_(value_layout="BNLC", loc_layout="B2QHLP"))
    assert np.array_equal(gen.from_value_layout(c["value"], "BNLC"), a["value"])
    assert np.array_equal(gen.from_loc_layout(c["sampling_locations"], "B2QHLP"), a["sampling_locations"])
    assert c["value"].flags.c_contiguous and c["sampling_locations"].flags.c_contiguous


def test_shapes_and_distributions():
    w = gen.WORKLOADS["tiny"].with_(B=2, N_q=64)
    d = gen.generate(w)
    assert d["value"].shape == (2, 80, 2, 8) and d["value"].dtype == np.float32
    assert d["sampling_locations"].shape == (2, 64, 2, 2, 2, 2)
    assert d["attention_weights"].shape == (2, 64, 2, 2, 2)
    assert d["grad_output"].shape == (2, 64, 16)
    s = d["attention_weights"].reshape(2, 64, 2, 4).sum(-1)
    assert np.allclose(s, 1.0, atol=1e-6)
    loc = d["sampling_locations"]
    assert loc.min() >= -0.1 and loc.max() <= 1.1


def test_pixel_centre_recipe():
    w = gen.Workload("t", B=1, N_q=None, N_h=1, C_h=4, N_p=64, levels=((4, 6), (2, 3)),
                     loc_recipe="pixel_centre", seed=7)
    d = gen.generate(w)
    loc = d["sampling_locations"].astype(np.float64)  # (1, L, 1, 2, 64, 2)
    mean = loc.mean(axis=(0, 2, 4))  # (L, N_l, 2): reference point per query
    # query 0 is pixel (0,0) of level 0: centre (0.5/6, 0.5/4); offsets are zero-mean
    assert abs(mean[0, 0, 0] - 0.5 / 6) < 0.1 and abs(mean[0, 0, 1] - 0.5 / 4) < 0.1
    # last query is pixel (1,2) of level 1: centre (2.5/3, 1.5/2)
    assert abs(mean[-1, 1, 0] - 2.5 / 3) < 0.3 and abs(mean[-1, 1, 1] - 1.5 / 2) < 0.3


@pytest.mark.parametrize("x", [0.0, 1.0, -2.5, 3.14159, 1e-3, 65504.0, 1.00390625, 1.01171875])
def test_bf16_rounding_ties_to_even(x):
    r = gen.round_to_bf16(np.array([x]))[0]
    assert (np.array([r], dtype=np.float32).view(np.uint32)[0] & 0xFFFF) == 0
    # the nearest bf16 (8 significant bits) to x
    if x != 0.0:
        e = np.floor(np.log2(abs(x)))
        ulp = 2.0 ** (e - 7)
        assert abs(r - x) <= ulp / 2 + 1e-12
    # exact ties go to the even significand
    assert gen.round_to_bf16(np.array([1.00390625]))[0] == 1.0      # 1 + 2^-8 -> 1
    assert gen.round_to_bf16(np.array([1.01171875]))[0] == 1.015625  # 1 + 3*2^-8 -> 1 + 2^-6


def test_bf16_workload_values_representable():
    d = gen.generate(gen.WORKLOADS["tiny"].with_(dtype="bf16"))
    for k in ("value", "grad_output"):
        assert np.all((d[k].view(np.uint32) & 0xFFFF) == 0)
