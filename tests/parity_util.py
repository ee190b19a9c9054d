"""Shared helpers for the GPU parity tests: run a workload through the CUDA
path (Python binding -> C ABI -> kernels) and through the CPU oracle on the
same seeded inputs, and compare element by element.

Tolerance (elementwise, per tensor):
    |gpu - ref| <= rtol * (|ref| + max|ref|)
with rtol 1e-5 for the binary32 forward, 1e-4 for the binary32 backward
(grad_value is summed by atomics in a run-dependent order) and 2e-2 when value
and gradients are stored in bfloat16 (arithmetic stays binary32).  The
max|ref| term is a normwise floor, so values near zero that come from
cancellation do not fail on rounding noise.
"""
from __future__ import annotations

import numpy as np

import oracle
from scale_deformable_attention_forward_gb300 import inputs as gen

RTOL = {("f32", "fwd"): 1e-5, ("f32", "bwd"): 1e-4, ("bf16", "fwd"): 2e-2, ("bf16", "bwd"): 2e-2}
# gradients stored in a 16-bit location dtype (rounding to nearest even on store)
LOC_RTOL = {"f32": None, "bf16": 2e-2, "f16": 2e-3}


def torch_dtype(dtype):
    import torch
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def loc_torch_dtype(loc_dtype):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[loc_dtype]


def to_device(d: dict, dtype: str, device="cuda", loc_dtype: str = "f32"):
    import torch
    vt, lt = torch_dtype(dtype), loc_torch_dtype(loc_dtype)
    return {
        "value": torch.from_numpy(d["value"]).to(device=device, dtype=vt),
        "sampling_locations": torch.from_numpy(d["sampling_locations"]).to(device=device, dtype=lt),
        "attention_weights": torch.from_numpy(d["attention_weights"]).to(device=device, dtype=lt),
        "grad_output": torch.from_numpy(d["grad_output"]).to(device=device, dtype=vt),
    }


def np64(t):
    return None if t is None else t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu, ref, rtol, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, f"{what}: shape {gpu.shape} vs {ref.shape}"
    if ref.size == 0:
        return
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    bound = rtol * (np.abs(ref) + np.max(np.abs(ref)))
    err = np.abs(gpu - ref)
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {ref.size} elements out of tolerance; worst at {i}: "
                             f"gpu {gpu[i]!r} ref {ref[i]!r} (rtol {rtol}, bound {bound[i]:.3e})")


def kw_of(w: gen.Workload):
    return dict(value_layout=w.value_layout, sampling_locations_layout=w.loc_layout,
                align_corners=w.align_corners, padding_mode=w.padding_mode)


def oracle_forward(w, d):
    return oracle.forward(d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
                          d["attention_weights"], coord_f32=True, **kw_of(w))


def oracle_backward(w, d, flags=(True, True, True)):
    return oracle.backward(d["grad_output"], d["value"], d["spatial_shapes"], d["level_start_index"],
                           d["sampling_locations"], d["attention_weights"], compute_grad_value=flags[0],
                           compute_grad_sampling_locations=flags[1], compute_grad_attention_weights=flags[2],
                           coord_f32=True, **kw_of(w))


def gpu_forward(w, t, d):
    import scale_deformable_attention_forward_gb300 as msda
    return msda.msda_forward(t["value"], d["spatial_shapes"], d["level_start_index"], t["sampling_locations"],
                             t["attention_weights"], **kw_of(w))


def gpu_backward(w, t, d, flags=(True, True, True), **outs):
    import scale_deformable_attention_forward_gb300 as msda
    return msda.msda_backward(t["grad_output"], t["value"], d["spatial_shapes"], d["level_start_index"],
                              t["sampling_locations"], t["attention_weights"], compute_grad_value=flags[0],
                              compute_grad_sampling_locations=flags[1], compute_grad_attention_weights=flags[2],
                              **outs, **kw_of(w))


def check_workload(w, d=None, flag_sets=((True, True, True),), check_forward=True):
    """Forward and backward of one workload on the GPU against the oracle."""
    import torch
    d = gen.generate(w) if d is None else d
    t = to_device(d, w.dtype, loc_dtype=w.loc_dtype)
    if check_forward:
        out = gpu_forward(w, t, d)
        torch.cuda.synchronize()
        assert_close(np64(out), oracle_forward(w, d), RTOL[(w.dtype, "fwd")], f"{w.name} out")
    for flags in flag_sets:
        got = gpu_backward(w, t, d, flags)
        torch.cuda.synchronize()
        ref = oracle_backward(w, d, flags)
        for name, g, r, f in zip(("grad_value", "grad_sampling_locations", "grad_attention_weights"), got, ref,
                                 flags):
            if f:
                rtol = RTOL[(w.dtype, "bwd")]
                if name != "grad_value" and LOC_RTOL[w.loc_dtype]:
                    rtol = max(rtol, LOC_RTOL[w.loc_dtype])
                assert_close(np64(g), r, rtol, f"{w.name} {name} flags={flags}")
            else:
                assert g is None and r is None
