"""msda_backward_accumulate against the oracle (GPU).

The backward page lets a call add into persistent grad_value buffers instead
of zeroing them ("MS Deformable Attention Backward Kernel API Reference",
Parameters: grad_value_buffers_in, prev_reduced_grad_value,
dump_reduced_grad_value), so that calls over query chunks or micro-batches
build one total.  Here the persistent state is a caller-owned float32 tensor:
after the calls it must equal its starting contents plus the sum of the
calls' grad_value, each computed by the float64 oracle.  The accumulator is
never rounded to bfloat16, so the float32 tolerance applies for both value
dtypes.
"""
import numpy as np
import pytest

from parity_util import RTOL, assert_close, kw_of, np64, oracle_backward, tensor_groups, to_device
from scale_deformable_attention_forward_gb300 import inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LEVELS = ((13, 17), (7, 9), (3, 4), (1, 1))


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_forward_gb300 import build
    build.build()


def _workload(dtype, N_q, seed, vl="BLNC", ll="BQHLP2", pad="zeros", align=False):
    return gen.Workload(f"acc-{dtype}-{N_q}-{seed}", B=2, N_q=N_q, N_h=3, C_h=32, N_p=3, levels=LEVELS,
                        dtype=dtype, value_layout=vl, loc_layout=ll, align_corners=align, padding_mode=pad,
                        loc_recipe="uniform", loc_lo=-0.15, loc_hi=1.15, seed=seed)


def _accumulate(w, d, t, acc, flags=(True, True, True)):
    import scale_deformable_attention_forward_gb300 as msda
    return msda.msda_backward_accumulate(t["grad_output"], t["value"], d["spatial_shapes"], d["level_start_index"],
                                         t["sampling_locations"], t["attention_weights"], acc,
                                         compute_grad_value=flags[0], compute_grad_sampling_locations=flags[1],
                                         compute_grad_attention_weights=flags[2], **kw_of(w))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N_q", [37, 150])  # 150: dense enough for the cell-sorted grad_value
def test_two_calls_add_up(dtype, N_q):
    """start + grad_value(g1) + grad_value(g2), and the other two gradients of
    each call as msda_backward gives them."""
    w = _workload(dtype, N_q, seed=201)
    d1 = gen.generate(w)
    d2 = dict(d1)
    rng = np.random.default_rng(7)
    d2["grad_output"] = rng.standard_normal(d1["grad_output"].shape)
    if dtype == "bf16":  # the oracle sees the numbers the GPU sees
        d2["grad_output"] = torch.from_numpy(d2["grad_output"]).to(torch.bfloat16).double().numpy()
    start = rng.standard_normal(d1["value"].shape)
    acc = torch.from_numpy(start).to("cuda", torch.float32)
    start32 = np64(acc)
    for flags in ((True, True, True), (True, False, False)):
        acc.copy_(torch.from_numpy(start32))
        total = start32.copy()
        for d in (d1, d2):
            t = to_device(d, dtype)
            gv, gl, ga = _accumulate(w, d, t, acc, flags)
            torch.cuda.synchronize()
            assert gv is acc
            ref = oracle_backward(w, d, flags)
            total = total + ref[0]
            if flags[1]:
                assert_close(np64(gl), ref[1], RTOL[(dtype, "bwd")], "grad_sampling_locations",
                             groups=tensor_groups(w, "grad_sampling_locations"))
                assert_close(np64(ga), ref[2], RTOL[(dtype, "bwd")], "grad_attention_weights",
                             groups=tensor_groups(w, "grad_attention_weights"))
            else:
                assert gl is None and ga is None
        assert_close(np64(acc), total, RTOL[("f32", "bwd")], f"accumulator {flags}",
                     groups=tensor_groups(w, "grad_value"))


@pytest.mark.parametrize("ll", ["BQHLP2", "B2QHLP"])
@pytest.mark.parametrize("vl", ["BLNC", "BNLC"])
def test_query_chunks_sum_to_full_call(vl, ll):
    """The grad_value of all queries equals the accumulation over two query
    chunks (each chunk a call with its own N_q)."""
    w = _workload("f32", 60, seed=202, vl=vl, ll=ll, pad="border", align=True)
    d = gen.generate(w)
    full = oracle_backward(w, d, (True, False, False))[0]
    acc = torch.zeros(d["value"].shape, dtype=torch.float32, device="cuda")
    qax = 1 if ll == "BQHLP2" else 2
    for q0, q1 in ((0, 23), (23, 60)):
        wc = _workload("f32", q1 - q0, seed=202, vl=vl, ll=ll, pad="border", align=True)
        dc = dict(d)
        dc["sampling_locations"] = np.ascontiguousarray(np.take(d["sampling_locations"], range(q0, q1), axis=qax))
        dc["attention_weights"] = np.ascontiguousarray(d["attention_weights"][:, q0:q1])
        dc["grad_output"] = np.ascontiguousarray(d["grad_output"][:, q0:q1])
        _accumulate(wc, dc, to_device(dc, "f32"), acc, (True, False, False))
    torch.cuda.synchronize()
    assert_close(np64(acc), full, RTOL[("f32", "bwd")], "chunked accumulator", groups=tensor_groups(w, "grad_value"))


def test_rejects_misaligned_accumulator():
    import scale_deformable_attention_forward_gb300 as msda
    w = _workload("f32", 8, seed=203)
    d = gen.generate(w)
    t = to_device(d, "f32")
    acc = torch.zeros(d["value"].size + 1, dtype=torch.uint8, device="cuda")
    bad = acc[1:]  # not 4-byte aligned
    lib = msda.load_library()
    desc = msda.make_desc((w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L), d["spatial_shapes"],
                          d["level_start_index"])
    gl = torch.empty_like(t["sampling_locations"])
    ga = torch.empty_like(t["attention_weights"])
    rc = lib.msda_backward_accumulate(desc.ref(), t["grad_output"].data_ptr(), t["value"].data_ptr(),
                                      t["sampling_locations"].data_ptr(), t["attention_weights"].data_ptr(),
                                      1, 1, 1, bad.data_ptr(), gl.data_ptr(), ga.data_ptr(), None, 0,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == -9
