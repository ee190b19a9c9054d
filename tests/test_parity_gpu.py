"""GPU parity: the sm_103a kernels (through the Python binding and the C ABI)
against the float64 CPU oracle, element by element, on seeded inputs.

Covers the five Deformable-DETR-shaped workloads at full size, the layout x
padding x align_corners x dtype matrix on a multi-tile problem with ragged
tails, every compute_grad_* combination, channel counts that exercise every
kernel shape (vector and scalar paths, masked lanes), unaligned pointers,
degenerate levels, extreme and exactly-on-grid locations, and empty inputs.
"""
import numpy as np
import pytest

from parity_util import (RTOL, assert_close, check_workload, gpu_backward, gpu_forward, np64, oracle_backward,
                         tensor_groups,
                         oracle_forward, to_device)
from scale_deformable_attention_forward_gb300 import inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ALL_FLAGS = [(True, True, True), (True, False, False), (False, True, False), (False, False, True),
             (True, True, False), (False, True, True), (True, False, True)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_forward_gb300 import build
    build.build()


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["tiny", "decoder", "encoder32", "encoder16", "hires16"])
def test_workload_full_size(name):
    w = gen.WORKLOADS[name]
    flag_sets = [(True, True, True)]
    if name in ("hires16", "encoder32"):  # grad_value alone: the tile-sorted path at full size, both dtypes
        flag_sets += [(True, False, False), (False, True, True)]
    if name == "tiny":
        flag_sets = ALL_FLAGS
    check_workload(w, flag_sets=flag_sets)


# ------------------------------------------------------------------ option matrix
MATRIX_LEVELS = ((13, 17), (7, 9), (3, 4), (1, 1))


def _small(dtype, vl, ll, align, pad, C_h=32, N_q=37, N_p=3, B=2, N_h=3, levels=MATRIX_LEVELS, seed=11,
           lo=-0.15, hi=1.15):
    return gen.Workload(f"m-{dtype}-{vl}-{ll}-{align}-{pad}-C{C_h}", B=B, N_q=N_q, N_h=N_h, C_h=C_h, N_p=N_p,
                        levels=levels, dtype=dtype, value_layout=vl, loc_layout=ll, align_corners=align,
                        padding_mode=pad, loc_recipe="uniform", loc_lo=lo, loc_hi=hi, seed=seed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vl", ["BLNC", "BNLC"])
@pytest.mark.parametrize("ll", ["BQHLP2", "B2QHLP"])
@pytest.mark.parametrize("align", [False, True])
@pytest.mark.parametrize("pad", ["zeros", "border"])
def test_option_matrix(dtype, vl, ll, align, pad):
    check_workload(_small(dtype, vl, ll, align, pad), flag_sets=[(True, True, True), (False, True, True)])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("C_h", [1, 3, 4, 5, 8, 12, 16, 24, 40, 64, 96, 200, 256])
def test_channel_counts(dtype, C_h):
    """Every (vector width, lanes per sample, chunks per lane) instantiation,
    including masked lanes and the scalar fallback."""
    w = _small(dtype, "BLNC", "BQHLP2", False, "zeros", C_h=C_h, N_q=9, N_h=2, N_p=2, seed=C_h)
    check_workload(w, flag_sets=[(True, True, True)])


# The cell-sorted grad_value (count, scan, append, per-cell reduction) runs
# when a problem has at least two samples per cell key; the problems above are
# sparser and take the direct-atomic grad_value.  These repeat the option
# matrix and the channel counts on problems dense enough for the sorted path.
def _dense(w):
    keys = w.B * w.N_h * sum((h + 1) * (wd + 1) for h, wd in w.levels)
    samples = w.B * w.n_queries * w.N_h * w.N_l * w.N_p
    assert samples >= 2 * keys, "not dense enough for the cell-sorted grad_value"
    return w


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vl", ["BLNC", "BNLC"])
@pytest.mark.parametrize("ll", ["BQHLP2", "B2QHLP"])
@pytest.mark.parametrize("align", [False, True])
@pytest.mark.parametrize("pad", ["zeros", "border"])
def test_option_matrix_sorted(dtype, vl, ll, align, pad):
    w = _dense(_small(dtype, vl, ll, align, pad, N_q=150, seed=13))
    check_workload(w, flag_sets=[(True, True, True), (True, False, False)], check_forward=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("C_h", [1, 3, 4, 5, 8, 12, 40, 96, 256])
def test_channel_counts_sorted(dtype, C_h):
    w = _dense(_small(dtype, "BLNC", "BQHLP2", False, "zeros", C_h=C_h, N_q=120, N_h=2, N_p=2, seed=C_h + 100))
    # grad_value alone takes the tile-sorted path; with the other gradients
    # the direct row kernel runs on the same dense problem
    check_workload(w, flag_sets=[(True, False, False), (True, True, True), (True, True, False), (True, False, True)],
                   check_forward=False)


@pytest.mark.parametrize("pad,align", [("zeros", False), ("border", True)])
def test_sorted_many_levels(pad, align):
    """The tile-sorted grad_value on 16 levels including 1-pixel rows and
    columns (tile tables, level boundaries, border clamps)."""
    levels = tuple((3 + i, 1 + (i * 5) % 7) for i in range(15)) + ((1, 1),)
    w = _dense(_small("f32", "BNLC", "B2QHLP", align, pad, levels=levels, N_q=100, N_p=2, seed=62))
    check_workload(w, flag_sets=[(True, False, False), (True, True, True)], check_forward=False)


@pytest.mark.parametrize("loc_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N_q,ll", [(37, "BQHLP2"), (150, "B2QHLP")])  # 150: cell-sorted grad_value too
def test_16bit_locations(loc_dtype, dtype, N_q, ll):
    """Locations, weights and their gradients stored in bfloat16 or binary16
    (arithmetic binary32); the oracle reads the same 16-bit numbers."""
    w = _small(dtype, "BLNC", ll, False, "zeros", N_q=N_q, seed=31).with_(loc_dtype=loc_dtype)
    check_workload(w, flag_sets=[(True, True, True), (True, False, False), (False, False, True)])


@pytest.mark.parametrize("N_p", [1, 5, 8, 13])
def test_points_per_level(N_p):
    """N_l*N_p not a multiple of the samples in flight per warp."""
    check_workload(_small("f32", "BLNC", "BQHLP2", False, "zeros", N_p=N_p, N_q=11, seed=50 + N_p),
                   flag_sets=ALL_FLAGS[:4])


def test_many_levels():
    levels = tuple((3 + i, 2 + (i * 5) % 7) for i in range(16))
    check_workload(_small("f32", "BNLC", "B2QHLP", True, "border", levels=levels, N_q=7, N_p=2, seed=61))


# ------------------------------------------------------------------ flags and untouched outputs
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N_q", [37, 150])  # 150: grad_value-only calls take the tile-sorted path
def test_disabled_outputs_untouched(dtype, N_q):
    w = _small(dtype, "BLNC", "BQHLP2", False, "zeros", N_q=N_q, seed=71)
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    for flags in ALL_FLAGS:
        sentinels = {
            "grad_value": torch.full_like(t["value"], 7.0),
            "grad_sampling_locations": torch.full_like(t["sampling_locations"], 7.0),
            "grad_attention_weights": torch.full_like(t["attention_weights"], 7.0),
        }
        import scale_deformable_attention_forward_gb300 as msda
        lib = msda.load_library()
        desc = msda.make_desc((w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L), d["spatial_shapes"],
                              d["level_start_index"], w.value_layout, w.loc_layout, w.align_corners,
                              w.padding_mode, msda.DTYPE_BF16 if dtype == "bf16" else msda.DTYPE_F32)
        ws_n = lib.msda_backward_workspace_size(desc.ref(), int(flags[0]))
        ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
        P = lambda x: x.data_ptr()
        rc = lib.msda_backward(desc.ref(), P(t["grad_output"]), P(t["value"]), P(t["sampling_locations"]),
                               P(t["attention_weights"]), *[int(f) for f in flags],
                               P(sentinels["grad_value"]), P(sentinels["grad_sampling_locations"]),
                               P(sentinels["grad_attention_weights"]), P(ws), ws_n,
                               torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        ref = oracle_backward(w, d, flags)
        for (name, buf), f, r in zip(sentinels.items(), flags, ref):
            if f:
                assert_close(np64(buf), r, RTOL[(dtype, "bwd")], f"{name} {flags}", groups=tensor_groups(w, name))
            else:
                assert torch.all(buf == 7.0), f"{name} written although disabled ({flags})"


# ------------------------------------------------------------------ special locations
def _custom(levels, loc, value=None, attn=None, g=None, N_h=2, C_h=8, dtype="f32", **opt):
    B, N_q = loc.shape[0], loc.shape[1]
    N_p = loc.shape[4]
    rng = np.random.default_rng(5)
    L = sum(h * w for h, w in levels)
    w = gen.Workload("custom", B=B, N_q=N_q, N_h=N_h, C_h=C_h, N_p=N_p, levels=levels, dtype=dtype, **opt)
    d = {
        "value": gen.to_value_layout(gen.store_dtype(rng.standard_normal((B, L, N_h, C_h)) if value is None
                                                     else value, dtype), w.value_layout),
        "sampling_locations": gen.to_loc_layout(np.asarray(loc, dtype=np.float32), w.loc_layout),
        "attention_weights": np.asarray(rng.uniform(0.1, 1.0, (B, N_q, N_h, len(levels), N_p))
                                        if attn is None else attn, dtype=np.float32),
        "grad_output": gen.store_dtype(rng.standard_normal((B, N_q, N_h * C_h)) if g is None else g, dtype),
        "spatial_shapes": levels,
        "level_start_index": w.level_start_index,
    }
    return w, d


@pytest.mark.parametrize("pad", ["zeros", "border"])
@pytest.mark.parametrize("align", [False, True])
def test_extreme_and_on_grid_locations(pad, align):
    levels = ((5, 7), (3, 2), (1, 4))
    specials = [-1e30, -1e6, -5.0, -1.0, -0.5, -1e-7, 0.0, 1e-7, 0.25, 0.5, 1.0 - 1e-7, 1.0, 1.0 + 1e-7, 1.5,
                5.0, 1e6, 1e30]
    # integer pixel coordinates and pixel centres of every level, in both mappings
    for H, W in levels:
        for n in (H, W):
            specials += [k / n for k in range(n + 1)] + [(k + 0.5) / n for k in range(n)]
            if n > 1:
                specials += [k / (n - 1) for k in range(n)]
    sp = np.array(specials, dtype=np.float32)
    rng = np.random.default_rng(9)
    N_q, N_p = 40, 4
    loc = rng.choice(sp, size=(2, N_q, 2, len(levels), N_p, 2))
    w, d = _custom(levels, loc, padding_mode=pad, align_corners=align)
    check_workload(w, d=d, flag_sets=[(True, True, True)])


def test_single_pixel_and_single_row_levels_align_corners():
    """W_l = 1 or H_l = 1 with align_corners=True: that axis always maps to 0
    and its location gradient is 0."""
    levels = ((1, 1), (1, 6), (5, 1))
    rng = np.random.default_rng(10)
    loc = rng.uniform(-0.2, 1.2, size=(1, 16, 2, 3, 3, 2))
    for pad in ("zeros", "border"):
        w, d = _custom(levels, loc, padding_mode=pad, align_corners=True)
        check_workload(w, d=d, flag_sets=ALL_FLAGS[:1])


# ------------------------------------------------------------------ pointers, streams, empties
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unaligned_pointers_take_scalar_path(dtype):
    """Tensors that start one element past a 16-byte boundary are still
    accepted (element-aligned) and give the same results."""
    w = _small(dtype, "BLNC", "BQHLP2", False, "zeros", C_h=32, N_q=13, seed=81)
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    shifted = {}
    for k, v in t.items():
        buf = torch.empty(v.numel() + 1, dtype=v.dtype, device=v.device)
        s = buf[1:].view(v.shape)
        s.copy_(v)
        shifted[k] = s
    out = gpu_forward(w, shifted, d)
    gv_buf = torch.empty(t["value"].numel() + 1, dtype=t["value"].dtype, device="cuda")
    got = gpu_backward(w, shifted, d, grad_value=gv_buf[1:].view(t["value"].shape))
    torch.cuda.synchronize()
    assert_close(np64(out), oracle_forward(w, d), RTOL[(dtype, "fwd")], "unaligned out",
                 groups=tensor_groups(w, "out"))
    for g, r, n in zip(got, oracle_backward(w, d), ("grad_value", "grad_sampling_locations", "grad_attention_weights")):
        assert_close(np64(g), r, RTOL[(dtype, "bwd")], f"unaligned {n}", groups=tensor_groups(w, n))


def test_non_default_stream():
    w = _small("f32", "BLNC", "BQHLP2", False, "zeros", seed=91)
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = gpu_forward(w, t, d)
        got = gpu_backward(w, t, d)
    s.synchronize()
    assert_close(np64(out), oracle_forward(w, d), RTOL[("f32", "fwd")], "stream out")
    assert_close(np64(got[0]), oracle_backward(w, d)[0], RTOL[("f32", "bwd")], "stream gv",
                 groups=tensor_groups(w, "grad_value"))


@pytest.mark.parametrize("dims", [dict(B=0), dict(N_q=0), dict(N_p=0), dict(C_h=0), dict(N_h=0)])
def test_empty_inputs(dims):
    base = dict(B=2, N_q=5, N_h=2, C_h=8, N_p=2)
    base.update(dims)
    w = gen.Workload("empty", levels=((4, 5), (2, 2)), loc_recipe="uniform", seed=3, **base)
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    out = gpu_forward(w, t, d)
    got = gpu_backward(w, t, d)
    torch.cuda.synchronize()
    assert_close(np64(out), oracle_forward(w, d), 1e-5, "empty out")
    for g, r in zip(got, oracle_backward(w, d)):
        assert_close(np64(g), r, 1e-4, "empty grads")


def test_repeatable():
    """The forward and the location/attention gradients are bit-identical
    from run to run (no atomics there); grad_value stays within tolerance."""
    w = gen.WORKLOADS["decoder"]
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    o1, o2 = gpu_forward(w, t, d).clone(), gpu_forward(w, t, d).clone()
    a = [x.clone() for x in gpu_backward(w, t, d)]
    b = [x.clone() for x in gpu_backward(w, t, d)]
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert_close(np64(a[0]), np64(b[0]), 1e-5, "grad_value run to run")


@pytest.mark.parametrize("pad", ["zeros", "border"])
def test_repeatable_sorted(pad):
    """On a problem dense enough for the tile-sorted grad_value: the location
    and attention gradients are bit-identical from run to run, and grad_value
    (summed by cell runs in an order that changes from run to run) stays
    within tolerance, whether it comes alone or with the other two."""
    w = _dense(_small("f32", "BLNC", "BQHLP2", False, pad, N_q=150, seed=17))
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    runs = []
    for _ in range(3):
        runs.append([x.clone() for x in gpu_backward(w, t, d)])
    gvs = [gpu_backward(w, t, d, (True, False, False))[0].clone() for _ in range(3)]
    torch.cuda.synchronize()
    for a in runs[1:]:
        assert torch.equal(a[1], runs[0][1]) and torch.equal(a[2], runs[0][2])
        assert_close(np64(a[0]), np64(runs[0][0]), 1e-5, "grad_value run to run")
    for g in gvs:
        assert_close(np64(g), np64(runs[0][0]), 1e-5, "tile-sorted grad_value run to run")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cuda_graph_capture(dtype):
    """Every call only enqueues work on the caller's stream, so a training
    step can be captured in a CUDA graph (after one call outside the capture):
    replays reproduce the eager results -- forward, full backward, the
    tile-sorted grad_value-only backward, and both staged variants."""
    import scale_deformable_attention_forward_gb300 as msda
    w = _dense(_small(dtype, "BLNC", "BQHLP2", False, "zeros", N_q=150, seed=19))
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    kw = dict(value_layout=w.value_layout, sampling_locations_layout=w.loc_layout,
              align_corners=w.align_corners, padding_mode=w.padding_mode)
    a = (d["spatial_shapes"], d["level_start_index"], t["sampling_locations"], t["attention_weights"])
    ws = torch.empty(max(1, msda.msda_backward_workspace_size(t["value"], d["spatial_shapes"], d["level_start_index"],
                                                              t["sampling_locations"], w.value_layout,
                                                              w.loc_layout)), dtype=torch.uint8, device="cuda")

    def buffers():
        return dict(out=torch.empty((w.B, w.n_queries, w.N_h * w.C_h), dtype=t["value"].dtype, device="cuda"),
                    out_st=torch.empty((w.B, w.n_queries, w.N_h * w.C_h), dtype=t["value"].dtype, device="cuda"),
                    gv=torch.empty_like(t["value"]), gl=torch.empty_like(t["sampling_locations"]),
                    ga=torch.empty_like(t["attention_weights"]), gv1=torch.empty_like(t["value"]),
                    gv_st=torch.empty_like(t["value"]), gl_st=torch.empty_like(t["sampling_locations"]),
                    ga_st=torch.empty_like(t["attention_weights"]))

    def step(b):
        msda.msda_forward(t["value"], *a, out=b["out"], **kw)
        msda.msda_backward(t["grad_output"], t["value"], *a, grad_value=b["gv"], grad_sampling_locations=b["gl"],
                           grad_attention_weights=b["ga"], workspace=ws, **kw)
        msda.msda_backward(t["grad_output"], t["value"], *a, compute_grad_sampling_locations=False,
                           compute_grad_attention_weights=False, grad_value=b["gv1"], workspace=ws, **kw)
        msda.msda_forward_staged(t["value"], *a, out=b["out_st"], **kw)
        msda.msda_backward_staged(t["grad_output"], t["value"], *a, grad_value=b["gv_st"],
                                  grad_sampling_locations=b["gl_st"], grad_attention_weights=b["ga_st"],
                                  workspace=ws, **kw)

    eager = buffers()
    step(eager)
    torch.cuda.synchronize()
    cap = buffers()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(cap)  # one call on the capture stream first
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for v in cap.values():
        v.zero_()
    with torch.cuda.graph(g):
        step(cap)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for k in ("out", "out_st", "gl", "ga", "gl_st", "ga_st"):
        assert torch.equal(cap[k], eager[k]), k
    for k in ("gv", "gv1", "gv_st"):
        assert_close(np64(cap[k]), np64(eager[k]), RTOL[(dtype, "bwd")], f"{k} replay")


# ------------------------------------------------------------------ plain atomics
@pytest.mark.parametrize("name", ["encoder32", "hires16"])
def test_plain_atomics_full_size(name, monkeypatch):
    """The backward with the warp-aggregated grad_value scatter switched off
    (MSDA_BWD_AGGREGATE=0: one reduction per corner and sample), against the
    oracle at full size."""
    monkeypatch.setenv("MSDA_BWD_AGGREGATE", "0")
    check_workload(gen.WORKLOADS[name], flag_sets=[(True, True, True)], check_forward=False)


# Enough rows (B * N_h * N_q > 9.7 K on 152 multiprocessors) that the
# whole-row kernels run, not the row split of small problems: the
# aggregated scatter and, switched off, the plain atomics of the same shape.
# N_p = 4 (16 samples a row, C_h = 32): full rows, the guard-free kernels;
# N_p = 3: a partial last batch, the guarded ones.
def _whole_rows(dtype, vl, ll, align, pad, seed, N_p=3):
    return _small(dtype, vl, ll, align, pad, N_q=701, N_h=8, B=2, N_p=N_p, seed=seed)


@pytest.mark.parametrize("N_p", [3, 4])
@pytest.mark.parametrize("aggregate", ["1", "0"])
@pytest.mark.parametrize("vl,ll", [("BLNC", "BQHLP2"), ("BNLC", "B2QHLP")])
@pytest.mark.parametrize("pad,align", [("zeros", False), ("border", True)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_whole_row_scatter_matrix(dtype, pad, align, vl, ll, aggregate, N_p, monkeypatch):
    monkeypatch.setenv("MSDA_BWD_AGGREGATE", aggregate)
    check_workload(_whole_rows(dtype, vl, ll, align, pad, seed=17 + N_p, N_p=N_p),
                   flag_sets=[(True, True, True), (True, True, False), (True, False, True), (False, True, True)],
                   check_forward=N_p == 4)


@pytest.mark.parametrize("aggregate", ["1", "0"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grad_value_only_row_kernel(dtype, aggregate, monkeypatch):
    """grad_value alone on a problem too sparse for the tile-sorted path but
    with whole rows (decoder-style queries, 2 x 2000 x 8 rows): the row
    kernel's grad_value-only instantiation, aggregated and plain."""
    monkeypatch.setenv("MSDA_BWD_AGGREGATE", aggregate)
    w = gen.WORKLOADS["decoder"].with_(N_q=2000, dtype=dtype, seed=27)
    check_workload(w, flag_sets=[(True, False, False), (True, True, True)], check_forward=False)
