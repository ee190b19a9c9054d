"""msda_forward_logits / msda_backward_logits against the oracle (GPU).

The weights are the softmax of each (b, q, h)'s N_l*N_p attention logits,
computed inside the kernels; the oracle composes a float64 softmax with its
forward and backward (and the softmax's chain rule for the logits' gradient).
Same tolerances as the weight-input entry points.
"""
import pytest

from parity_util import RTOL, assert_close, kw_of, np64, tensor_groups, to_device
from scale_deformable_attention_forward_gb300 import inputs as gen

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LEVELS = ((13, 17), (7, 9), (3, 4), (1, 1))
FLAG_SETS = [(True, True, True), (False, False, True), (True, False, False), (False, True, False)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_forward_gb300 import build
    build.build()


def _check(w, flag_sets, check_forward=True):
    import scale_deformable_attention_forward_gb300 as msda
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    z = torch.from_numpy(d["attention_logits"]).cuda()
    if check_forward:
        out = msda.msda_forward_logits(t["value"], d["spatial_shapes"], d["level_start_index"],
                                       t["sampling_locations"], z, **kw_of(w))
        torch.cuda.synchronize()
        ref = oracle.forward_logits(d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
                                    d["attention_logits"], coord_f32=True, **kw_of(w))
        assert_close(np64(out), ref, RTOL[(w.dtype, "fwd")], f"{w.name} out", groups=tensor_groups(w, "out"))
    for flags in flag_sets:
        got = msda.msda_backward_logits(t["grad_output"], t["value"], d["spatial_shapes"], d["level_start_index"],
                                        t["sampling_locations"], z, compute_grad_value=flags[0],
                                        compute_grad_sampling_locations=flags[1],
                                        compute_grad_attention_logits=flags[2], **kw_of(w))
        torch.cuda.synchronize()
        ref = oracle.backward_logits(d["grad_output"], d["value"], d["spatial_shapes"], d["level_start_index"],
                                     d["sampling_locations"], d["attention_logits"], compute_grad_value=flags[0],
                                     compute_grad_sampling_locations=flags[1],
                                     compute_grad_attention_logits=flags[2], coord_f32=True, **kw_of(w))
        for name, g, r, f in zip(("grad_value", "grad_sampling_locations", "grad_attention_logits"), got, ref,
                                 flags):
            if f:
                grp = tensor_groups(w, "grad_attention_weights" if name == "grad_attention_logits" else name)
                assert_close(np64(g), r, RTOL[(w.dtype, "bwd")], f"{w.name} {name} flags={flags}", groups=grp)
            else:
                assert g is None


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("vl,ll,align,pad", [("BLNC", "BQHLP2", False, "zeros"), ("BNLC", "B2QHLP", True, "border")])
@pytest.mark.parametrize("N_q", [37, 150])  # 150: dense enough for the cell-sorted grad_value
def test_logits_matrix(dtype, vl, ll, align, pad, N_q):
    w = gen.Workload(f"z-{dtype}-{vl}-{ll}-{N_q}", B=2, N_q=N_q, N_h=3, C_h=32, N_p=3, levels=LEVELS, dtype=dtype,
                     value_layout=vl, loc_layout=ll, align_corners=align, padding_mode=pad, loc_recipe="uniform",
                     loc_lo=-0.15, loc_hi=1.15, seed=301)
    _check(w, FLAG_SETS)


@pytest.mark.parametrize("C_h,N_p", [(5, 5), (96, 2)])  # scalar path / wide rows; N_l*N_p not a multiple of G
def test_logits_shapes(C_h, N_p):
    w = gen.Workload(f"z-C{C_h}", B=1, N_q=11, N_h=2, C_h=C_h, N_p=N_p, levels=LEVELS, dtype="f32",
                     value_layout="BLNC", loc_layout="BQHLP2", align_corners=False, padding_mode="zeros",
                     loc_recipe="uniform", loc_lo=-0.15, loc_hi=1.15, seed=302)
    _check(w, FLAG_SETS[:2])


def test_logits_encoder_full_size():
    _check(gen.WORKLOADS["encoder32"], [(True, True, True)])
