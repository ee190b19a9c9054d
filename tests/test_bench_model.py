"""The benchmark's byte and line models (CPU): the compulsory-byte count the
HBM roofline divides by, and the corner-row line count of the forward's L1
roofline, checked against counts written out by hand for the workloads."""
import importlib.util
import os

import pytest

from scale_deformable_attention_forward_gb300 import inputs as gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_compulsory_bytes_encoder32(bench):
    w = gen.WORKLOADS["encoder32"]
    samples = 2 * 22223 * 8 * 4 * 4
    value = 2 * 22223 * 8 * 32 * 4  # BLNC binary32, = out / grad_output at N_q = L
    fwd, bwd = bench.compulsory_bytes(w)
    assert w.samples == samples
    assert fwd == value + 8 * samples + 4 * samples + value  # value, locations, weights, out
    assert bwd == 2 * value + 8 * samples + 4 * samples + value + 8 * samples + 4 * samples
    assert fwd + bwd == 432370688  # the step's bytes in the bench line


def test_compulsory_bytes_bf16_halves_the_maps(bench):
    w16 = gen.WORKLOADS["encoder32"].with_(dtype="bf16")
    w32 = gen.WORKLOADS["encoder32"]
    (f16, b16), (f32, b32) = bench.compulsory_bytes(w16), bench.compulsory_bytes(w32)
    maps = 2 * 22223 * 8 * 32  # elements of value (= out)
    assert f32 - f16 == 2 * maps * 2  # value and out, 2 bytes fewer each
    assert b32 - b16 == 3 * maps * 2  # value, grad_output, grad_value


def test_gather_roofline_lines_and_fraction(bench):
    w = gen.WORKLOADS["encoder32"]
    r = bench.gather_roofline(w, fwd_ms=0.2, n_sm=100, sm_mhz=2000.0)
    lines = w.samples * 4  # one 128-byte line per binary32 32-channel corner row
    assert r["achieved"] == pytest.approx(lines / 0.2e-3 / 1e9, abs=0.01)
    assert r["peak"] == pytest.approx(200.0)  # 100 SMs x 2 GHz, one line a cycle each
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], abs=1e-4)
    # a bfloat16 row of 32 channels is 64 bytes: still one line
    assert bench.gather_roofline(w.with_(dtype="bf16"), 0.2, 100, 2000.0)["achieved"] == r["achieved"]
    # 64 binary32 channels span two lines
    r64 = bench.gather_roofline(w.with_(C_h=64), 0.2, 100, 2000.0)
    assert r64["achieved"] == pytest.approx(2 * r["achieved"], abs=0.02)
    # without a clock sample the maximum clock stands in, and says so
    assert "maximum clock" in bench.gather_roofline(w, 0.2, 100, None)["peak_source"]
