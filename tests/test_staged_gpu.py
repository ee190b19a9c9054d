"""msda_forward_staged (the staged-level gather) against msda_forward and the
oracle (GPU).

The staged kernel copies the coarsest levels of a head into shared memory
with TMA and gathers those levels from there; its arithmetic is the direct
kernel's, so the two outputs must be bit-identical, and both within the
forward tolerance of the float64 oracle.  Covers full and partial staging
(every level / only the coarse ones), both layouts, both paddings, both
align_corners, both value dtypes, every staged lane shape, queries that do
not fill the last block, extreme locations, and the shapes that fall back to
the direct kernel.
"""
import numpy as np
import pytest

from parity_util import RTOL, assert_close, kw_of, np64, oracle_forward, tensor_groups, to_device
from scale_deformable_attention_forward_gb300 import inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ALL_FIT = ((11, 13), (7, 9), (3, 4), (1, 1))     # 288 staged pixels (36 KB at 128 B): every level staged
COARSE_FIT = ((40, 50), (7, 9), (3, 4), (1, 1))  # level 0 (2000 px) too big at 128 B a pixel


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_forward_gb300 import build
    build.build()


def _desc(w):
    import scale_deformable_attention_forward_gb300 as msda
    return msda.make_desc((w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L), w.levels, w.level_start_index,
                          w.value_layout, w.loc_layout, w.align_corners, w.padding_mode,
                          msda.DTYPE_BF16 if w.dtype == "bf16" else msda.DTYPE_F32,
                          {"f32": msda.DTYPE_F32, "bf16": msda.DTYPE_BF16, "f16": msda.DTYPE_F16}[w.loc_dtype])


def _both(w, d=None):
    import scale_deformable_attention_forward_gb300 as msda
    d = gen.generate(w) if d is None else d
    t = to_device(d, w.dtype, loc_dtype=w.loc_dtype)
    args = (t["value"], d["spatial_shapes"], d["level_start_index"], t["sampling_locations"], t["attention_weights"])
    direct = msda.msda_forward(*args, **kw_of(w))
    staged = msda.msda_forward_staged(*args, **kw_of(w))
    torch.cuda.synchronize()
    return d, direct, staged


def _check(w, d=None, oracle=True):
    d, direct, staged = _both(w, d)
    assert torch.equal(staged, direct), f"{w.name}: staged and direct outputs differ"
    if oracle:
        assert_close(np64(staged), oracle_forward(w, d), RTOL[(w.dtype, "fwd")], f"{w.name} staged out",
                     groups=tensor_groups(w, "out"))


def _small(dtype, vl, ll, align, pad, levels, C_h=32, N_q=150, N_h=3, N_p=3, B=2, seed=401):
    return gen.Workload(f"st-{dtype}-{vl}-{ll}-{align}-{pad}-C{C_h}", B=B, N_q=N_q, N_h=N_h, C_h=C_h, N_p=N_p,
                        levels=levels, dtype=dtype, value_layout=vl, loc_layout=ll, align_corners=align,
                        padding_mode=pad, loc_recipe="uniform", loc_lo=-0.15, loc_hi=1.15, seed=seed)


@pytest.mark.parametrize("name", ["decoder", "encoder32", "encoder16", "hires16"])
def test_staged_full_size(name):
    """Bit-identical to the direct kernel on the full workloads (the direct
    kernel itself is checked against the oracle at full size elsewhere); the
    oracle too on the two binary32 ones."""
    w = gen.WORKLOADS[name]
    import scale_deformable_attention_forward_gb300 as msda
    assert msda.staged_levels(_desc(w)) < w.N_l, "expected a staged level"
    _check(w, oracle=name in ("decoder", "encoder32"))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vl", ["BLNC", "BNLC"])
@pytest.mark.parametrize("ll", ["BQHLP2", "B2QHLP"])
@pytest.mark.parametrize("align", [False, True])
@pytest.mark.parametrize("pad", ["zeros", "border"])
@pytest.mark.parametrize("levels", [ALL_FIT, COARSE_FIT], ids=["all", "coarse"])
def test_staged_option_matrix(dtype, vl, ll, align, pad, levels):
    import scale_deformable_attention_forward_gb300 as msda
    w = _small(dtype, vl, ll, align, pad, levels)
    first = msda.staged_levels(_desc(w))
    # level 0 of COARSE_FIT is 2016 staged pixels: 252 KB (binary32) or 126 KB (bfloat16)
    assert first == (0 if levels is ALL_FIT else 1)
    _check(w)


@pytest.mark.parametrize("dtype,C_h", [("f32", 4), ("f32", 8), ("f32", 16), ("f32", 64), ("bf16", 8),
                                       ("bf16", 16), ("bf16", 64)])
def test_staged_lane_shapes(dtype, C_h):
    """Every staged (lanes per row, chunks per lane) shape: G = 1, 2, 4, 8 and
    two chunks a lane."""
    import scale_deformable_attention_forward_gb300 as msda
    w = _small(dtype, "BLNC", "BQHLP2", False, "zeros", COARSE_FIT, C_h=C_h, N_q=70, N_h=2, seed=410 + C_h)
    assert msda.staged_levels(_desc(w)) < w.N_l
    _check(w)


@pytest.mark.parametrize("case", ["scalar", "wide", "bf16_8byte_rows", "loc_bf16", "one_big_level"])
def test_staged_falls_back_to_direct(case):
    """Shapes the staged kernel does not cover run the direct kernel: same
    output, still within the oracle's tolerance."""
    import scale_deformable_attention_forward_gb300 as msda
    w = {
        "scalar": _small("f32", "BLNC", "BQHLP2", False, "zeros", ALL_FIT, C_h=5, N_q=40),
        "wide": _small("f32", "BLNC", "BQHLP2", False, "zeros", ALL_FIT, C_h=96, N_q=40),
        "bf16_8byte_rows": _small("bf16", "BLNC", "BQHLP2", False, "zeros", ALL_FIT, C_h=4, N_q=40),
        "loc_bf16": _small("f32", "BLNC", "BQHLP2", False, "zeros", ALL_FIT, N_q=40).with_(loc_dtype="bf16"),
        "one_big_level": _small("f32", "BLNC", "BQHLP2", False, "zeros", ((250, 200),), N_q=40, N_p=4),
    }[case]
    assert msda.staged_levels(_desc(w)) == w.N_l
    d, direct, staged = _both(w)
    assert torch.equal(staged, direct)
    if w.loc_dtype == "f32":
        assert_close(np64(staged), oracle_forward(w, d), RTOL[(w.dtype, "fwd")], f"{w.name} fallback")


@pytest.mark.parametrize("N_q,B,N_h", [(1, 1, 1), (65, 1, 2), (129, 3, 1)])
def test_staged_block_tails(N_q, B, N_h):
    """Query runs that do not fill their last block, and a single query."""
    w = _small("f32", "BNLC", "B2QHLP", True, "border", ALL_FIT, N_q=N_q, B=B, N_h=N_h, seed=420 + N_q)
    _check(w)


@pytest.mark.parametrize("pad", ["zeros", "border"])
def test_staged_extreme_locations(pad):
    """Locations far outside, on and next to the pixel grid of staged levels."""
    levels = ((5, 7), (3, 2), (1, 4), (2, 2))
    specials = np.array([-1e30, -1e6, -5.0, -1.0, -0.5, -1e-7, 0.0, 1e-7, 0.25, 0.5, 1.0 - 1e-7, 1.0,
                         1.0 + 1e-7, 1.5, 5.0, 1e6, 1e30] + [k / 7 for k in range(8)] + [(k + 0.5) / 5 for k in range(5)],
                        dtype=np.float32)
    w = gen.Workload("st-extreme", B=2, N_q=40, N_h=2, C_h=8, N_p=4, levels=levels, dtype="f32",
                     padding_mode=pad, loc_recipe="uniform", seed=430)
    d = gen.generate(w)
    rng = np.random.default_rng(431)
    d["sampling_locations"] = gen.to_loc_layout(rng.choice(specials, size=(2, 40, 2, len(levels), 4, 2)),
                                                w.loc_layout).astype(np.float32)
    _check(w, d)


def test_staged_kernel_runs_and_never_times_out():
    """encoder32 takes the staged kernel (the library's level choice stages at
    least one level, so the launch is the staged one and not the direct
    fallback), its output is the direct kernel's, and no block of any test of
    this module gave up waiting for its shared-memory copy."""
    import scale_deformable_attention_forward_gb300 as msda
    w = gen.WORKLOADS["encoder32"]
    desc = msda.make_desc((w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L), w.levels, w.level_start_index)
    first = msda.staged_levels(desc)
    assert first < w.N_l, "encoder32 stages no level: the direct kernel would run instead"
    d, direct, staged = _both(w)
    assert torch.equal(staged, direct)
    torch.cuda.synchronize()
    assert msda.staged_timeouts() == 0


# ------------------------------------------------------------------ staged backward
FLAGS_GV = [(True, True, True), (True, False, False), (True, True, False), (True, False, True)]


def _bwd_both(w, flags, d=None):
    import scale_deformable_attention_forward_gb300 as msda
    d = gen.generate(w) if d is None else d
    t = to_device(d, w.dtype)
    args = (t["grad_output"], t["value"], d["spatial_shapes"], d["level_start_index"], t["sampling_locations"],
            t["attention_weights"])
    kw = dict(compute_grad_value=flags[0], compute_grad_sampling_locations=flags[1],
              compute_grad_attention_weights=flags[2], **kw_of(w))
    direct = [x.clone() if x is not None else None for x in msda.msda_backward(*args, **kw)]
    staged = msda.msda_backward_staged(*args, **kw)
    torch.cuda.synchronize()
    return d, direct, staged


def _bwd_check(w, flag_sets=FLAGS_GV, d=None, oracle=True):
    from parity_util import oracle_backward
    d = gen.generate(w) if d is None else d
    for flags in flag_sets:
        d, direct, staged = _bwd_both(w, flags, d)
        for name, a, b, f in zip(("grad_value", "grad_sampling_locations", "grad_attention_weights"), staged, direct,
                                 flags):
            if not f:
                assert a is None and b is None
                continue
            if name == "grad_value":  # summation order differs: within the backward tolerance of each other
                assert_close(np64(a), np64(b), RTOL[(w.dtype, "bwd")], f"{w.name} {name} staged vs direct",
                             groups=tensor_groups(w, name))
            else:  # the direct kernel's arithmetic
                assert torch.equal(a, b), f"{w.name} {name} {flags}: staged and direct differ"
        if oracle:
            ref = oracle_backward(w, d, flags)
            for name, a, r, f in zip(("grad_value", "grad_sampling_locations", "grad_attention_weights"), staged,
                                     ref, flags):
                if f:
                    assert_close(np64(a), r, RTOL[(w.dtype, "bwd")], f"{w.name} {name} {flags} staged vs oracle",
                                 groups=tensor_groups(w, name))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vl,ll,align,pad", [("BLNC", "BQHLP2", False, "zeros"), ("BNLC", "B2QHLP", True, "border"),
                                             ("BLNC", "B2QHLP", True, "zeros"), ("BNLC", "BQHLP2", False, "border")])
@pytest.mark.parametrize("levels", [ALL_FIT, COARSE_FIT], ids=["all", "coarse"])
def test_backward_staged_matrix(dtype, vl, ll, align, pad, levels):
    import scale_deformable_attention_forward_gb300 as msda
    w = _small(dtype, vl, ll, align, pad, levels)
    assert msda.backward_staged_levels(_desc(w)) == (0 if levels is ALL_FIT else 1)
    _bwd_check(w)


@pytest.mark.parametrize("dtype,C_h", [("f32", 4), ("f32", 8), ("f32", 12), ("f32", 16), ("f32", 64), ("bf16", 8),
                                       ("bf16", 16), ("bf16", 64)])
def test_backward_staged_lane_shapes(dtype, C_h):
    """Every staged lane shape, and C_h = 12 (three chunks: no bank rotation,
    one lane of four past the channels)."""
    w = _small(dtype, "BLNC", "BQHLP2", False, "zeros", COARSE_FIT, C_h=C_h, N_q=70, N_h=2, seed=440 + C_h)
    _bwd_check(w, flag_sets=FLAGS_GV[:2])


@pytest.mark.parametrize("case", ["scalar", "wide", "no_grad_value"])
def test_backward_staged_falls_back(case):
    import scale_deformable_attention_forward_gb300 as msda
    w = {"scalar": _small("f32", "BLNC", "BQHLP2", False, "zeros", ALL_FIT, C_h=5, N_q=40),
         "wide": _small("f32", "BLNC", "BQHLP2", False, "zeros", ALL_FIT, C_h=96, N_q=40),
         "no_grad_value": _small("f32", "BLNC", "BQHLP2", False, "zeros", ALL_FIT, N_q=40)}[case]
    flags = [(False, True, True)] if case == "no_grad_value" else FLAGS_GV[:1]
    if case != "no_grad_value":
        assert msda.backward_staged_levels(_desc(w)) == w.N_l
    _bwd_check(w, flag_sets=flags)


@pytest.mark.parametrize("N_q,B,N_h", [(1, 1, 1), (65, 1, 2), (129, 3, 1)])
def test_backward_staged_block_tails(N_q, B, N_h):
    _bwd_check(_small("f32", "BNLC", "B2QHLP", True, "border", ALL_FIT, N_q=N_q, B=B, N_h=N_h, seed=450 + N_q),
               flag_sets=FLAGS_GV[:1])


@pytest.mark.parametrize("name", ["encoder32", "hires16"])
def test_backward_staged_full_size(name):
    """Full workloads: the location and attention gradients bit-identical to
    msda_backward, grad_value within tolerance of it (and of the oracle for
    the binary32 encoder)."""
    w = gen.WORKLOADS[name]
    _bwd_check(w, flag_sets=FLAGS_GV[:1], oracle=name == "encoder32")
