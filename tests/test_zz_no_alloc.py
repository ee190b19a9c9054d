"""msda_backward_noalloc against the CPU oracle and against msda_backward,
through the C ABI (GPU).

msda_backward_noalloc serves callers that may not allocate device memory
(for example a plug-in that must stay inside its host application's memory
pool): instead of a caller-provided workspace it accumulates bfloat16
grad_value in a fixed array owned by the library.  This file runs last so
that a failure here never hides the other GPU tests; it also passes on its
own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from parity_util import assert_close, np64, oracle_backward, tensor_groups, to_device
from scale_deformable_attention_forward_gb300 import inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_forward_gb300 import build
    build.build()
    import scale_deformable_attention_forward_gb300 as msda
    lib = msda.load_library()
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.msda_backward_noalloc.argtypes = [ctypes.POINTER(msda.msda_desc), P, P, P, P, I, I, I, P, P, P, P]
    lib.msda_backward_noalloc.restype = I
    return lib


def _desc(w, d):
    import scale_deformable_attention_forward_gb300 as msda
    return msda.make_desc((w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L), d["spatial_shapes"],
                          d["level_start_index"], w.value_layout, w.loc_layout, w.align_corners, w.padding_mode,
                          msda.DTYPE_BF16 if w.dtype == "bf16" else msda.DTYPE_F32)


def _call(lib, fn, desc, t, outs, flags, ws=None, ws_bytes=0):
    P = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [desc.ref(), P(t["grad_output"]), P(t["value"]), P(t["sampling_locations"]),
            P(t["attention_weights"]), *[int(f) for f in flags], P(outs[0]), P(outs[1]), P(outs[2])]
    if fn == "noalloc":
        return lib.msda_backward_noalloc(*args, s)
    return lib.msda_backward(*args, P(ws), ws_bytes, s)


def _outs(t, flags):
    return (torch.empty_like(t["value"]) if flags[0] else None,
            torch.empty_like(t["sampling_locations"]) if flags[1] else None,
            torch.empty_like(t["attention_weights"]) if flags[2] else None)


@pytest.mark.parametrize("name,dtype,flags", [
    ("decoder-1img-bf16", "bf16", (1, 1, 1)),
    ("decoder-1img-bf16", "bf16", (1, 0, 0)),
    ("encoder-1img-bf16", "bf16", (1, 0, 0)),
    ("tiny-bf16", "bf16", (1, 1, 1)),
    ("tiny-f32", "f32", (1, 1, 1)),
])
def test_noalloc_matches_backward_twice(lib, name, dtype, flags):
    if name.startswith("decoder"):
        # one image of the Deformable-DETR pyramid: a 5.7M-element accumulator
        w = gen.WORKLOADS["decoder"].with_(B=1, dtype=dtype, seed=21)
    elif name.startswith("encoder"):
        # one image, one query per pixel: whole rows, grad_value by the row kernel
        # (msda_backward takes the tile-sorted path for this grad_value-only call)
        w = gen.WORKLOADS["encoder32"].with_(B=1, dtype=dtype, seed=23)
    else:
        w = gen.WORKLOADS["tiny"].with_(dtype=dtype, seed=22)
    assert 4 * w.B * w.L * w.N_h * w.C_h <= SCRATCH_BYTES
    d = gen.generate(w)
    t = to_device(d, w.dtype)
    desc = _desc(w, d)
    ws_bytes = lib.msda_backward_workspace_size(desc.ref(), int(flags[0]))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    ref = _outs(t, flags)
    assert _call(lib, "backward", desc, t, ref, flags, ws, ws_bytes) == 0
    rtol = 2e-2 if dtype == "bf16" else 1e-4
    oref = oracle_backward(w, d, tuple(bool(f) for f in flags))
    names = ("grad_value", "grad_sampling_locations", "grad_attention_weights")
    for call in range(2):  # the second call starts from the first call's scratch contents
        got = _outs(t, flags)
        assert _call(lib, "noalloc", desc, t, got, flags) == 0
        torch.cuda.synchronize()
        for g, r, o, n in zip(got, ref, oref, names):
            if r is None:
                assert o is None
                continue
            grp = tensor_groups(w, n)
            assert_close(np64(g), o, rtol, f"call {call}: {n} vs the oracle", groups=grp)
            assert_close(np64(g), np64(r), rtol, f"call {call}: {n} vs msda_backward", groups=grp)


def test_noalloc_refuses_oversized_accumulator(lib):
    """A bfloat16 problem whose accumulator exceeds the array is refused
    before anything is enqueued (all tensor pointers are NULL here, so even a
    regression could not launch: validation would then reject the NULLs)."""
    import scale_deformable_attention_forward_gb300 as msda
    levels = ((100, 167), (50, 84), (25, 42), (13, 21))
    starts = (0, 16700, 20900, 21950)
    big = msda.make_desc((2, 10, 8, 32, 4, 4, 22223), levels, starts, value_dtype=msda.DTYPE_BF16)
    rc = lib.msda_backward_noalloc(big.ref(), None, None, None, None, 1, 1, 1, None, None, None, None)
    assert rc == -6, msda.msda_status_string(rc)
    # without grad_value no scratch is needed, so the size limit does not apply
    rc = lib.msda_backward_noalloc(big.ref(), None, None, None, None, 0, 1, 1, None, None, None, None)
    assert rc == -1
