"""Shared helpers for the GPU parity tests: run a workload through the CUDA
path (Python binding -> C ABI -> kernels) and through the CPU oracle on the
same seeded inputs, and compare element by element.

Tolerance (per tensor, per group of elements):
    |gpu - ref| <= rtol * (|ref| + rms_group(ref))      for every element, and
    ||gpu - ref||_2 <= rtol * ||ref||_2                   over every group,
with rtol 1e-5 for the binary32 forward, 1e-4 for the binary32 backward
(grad_value is summed by atomics in a run-dependent order) and 2e-2 when value
and gradients are stored in bfloat16 (arithmetic stays binary32).  The groups
follow the pyramid: grad_value per (level, head) slice, the location gradient
per (level, axis), the attention-weight gradient per level, the output per
head.  The RMS floor of an element's own group keeps values near zero that
come from cancellation from failing on rounding noise, without letting the
large coarse-level magnitudes set the floor of the fine levels (a floor of
max|ref| over the whole tensor was larger than the typical level-0 element of
the bfloat16 workloads' grad_value).  A group whose exact values are all zero
(the location gradient along a one-pixel axis, where border padding or
align_corners fixes the sample) holds only the oracle's float64 rounding
noise, so each group's RMS is floored at 1e-6 of the whole tensor's RMS.
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


def assert_close(gpu, ref, rtol, what, groups=None, report=None):
    """Check gpu against ref under the rule above.

    ``groups``: a list of index tuples (each selects one group of elements);
    None makes the whole tensor one group.  ``report``, if a dict, receives
    the worst |gpu - ref| / bound of every group (1.0 is the limit).
    """
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, f"{what}: shape {gpu.shape} vs {ref.shape}"
    if ref.size == 0:
        return
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    rms_all = float(np.sqrt(np.mean(ref * ref)))
    for gi, idx in enumerate([(Ellipsis,)] if groups is None else groups):
        r = ref[idx]
        if r.size == 0:
            continue
        g = gpu[idx]
        rms = max(float(np.sqrt(np.mean(r * r))), 1e-6 * rms_all)
        bound = rtol * (np.abs(r) + rms)
        err = np.abs(g - r)
        label = "" if groups is None else f" group {gi} {_fmt_idx(idx)}"
        worst = float(np.max(err / np.where(bound > 0, bound, np.inf))) if rms > 0 else float(np.max(err) > 0)
        if report is not None:
            report[label.strip() or "all"] = worst
        bad = err > bound
        if np.any(bad):
            i = np.unravel_index(np.argmax(err - bound), err.shape)
            raise AssertionError(f"{what}{label}: {int(bad.sum())} of {r.size} elements out of tolerance; worst at "
                                 f"{i}: gpu {g[i]!r} ref {r[i]!r} (rtol {rtol}, bound {bound[i]:.3e}, "
                                 f"group rms {rms:.3e})")
        nerr, nref = float(np.linalg.norm(err)), max(float(np.linalg.norm(r)), rms * np.sqrt(r.size))
        if nerr > rtol * nref:
            raise AssertionError(f"{what}{label}: relative error norm {nerr / nref:.3e} above rtol {rtol}")


def _fmt_idx(idx):
    def one(x):
        if x is Ellipsis:
            return "..."
        if isinstance(x, slice):
            return ":" if x.start is None and x.stop is None else f"{x.start}:{x.stop}"
        return str(x)
    return "[" + ",".join(one(x) for x in idx) + "]"


def tensor_groups(w: gen.Workload, name: str):
    """The comparison groups of one tensor of workload ``w`` (see the module
    docstring), as index tuples into the tensor in the workload's layout."""
    starts = list(w.level_start_index) + [w.L]
    nl = w.N_l
    if name == "grad_value":  # BLNC (B, L, N_h, C_h) or BNLC (B, N_h, L, C_h)
        out = []
        for l in range(nl):
            ls = slice(starts[l], starts[l + 1])
            for h in range(w.N_h):
                out.append((slice(None), ls, h) if w.value_layout == "BLNC" else (slice(None), h, ls))
        return out
    if name == "grad_sampling_locations":  # BQHLP2 (B, N_q, N_h, N_l, N_p, 2) or B2QHLP (B, 2, N_q, N_h, N_l, N_p)
        out = []
        for l in range(nl):
            for a in range(2):
                out.append((Ellipsis, l, slice(None), a) if w.loc_layout == "BQHLP2" else
                           (slice(None), a, Ellipsis, l, slice(None)))
        return out
    if name == "grad_attention_weights":  # (B, N_q, N_h, N_l, N_p)
        return [(Ellipsis, l, slice(None)) for l in range(nl)]
    if name == "out":  # (B, N_q, N_h * C_h)
        return [(slice(None), slice(None), slice(h * w.C_h, (h + 1) * w.C_h)) for h in range(w.N_h)]
    raise ValueError(name)


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


def check_workload(w, d=None, flag_sets=((True, True, True),), check_forward=True, verbose=True):
    """Forward and backward of one workload on the GPU against the oracle;
    prints the worst error / bound ratio of every tensor and group."""
    import torch
    d = gen.generate(w) if d is None else d
    t = to_device(d, w.dtype, loc_dtype=w.loc_dtype)
    margins = {}
    if check_forward:
        out = gpu_forward(w, t, d)
        torch.cuda.synchronize()
        rep = {}
        assert_close(np64(out), oracle_forward(w, d), RTOL[(w.dtype, "fwd")], f"{w.name} out",
                     groups=tensor_groups(w, "out"), report=rep)
        margins["out"] = rep
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
                rep = {}
                assert_close(np64(g), r, rtol, f"{w.name} {name} flags={flags}", groups=tensor_groups(w, name),
                             report=rep)
                margins[f"{name} {flags}"] = rep
            else:
                assert g is None and r is None
    if verbose:
        for k, rep in margins.items():
            worst = max(rep.values()) if rep else 0.0
            per_level = ", ".join(f"{g}: {v:.3f}" for g, v in rep.items())
            print(f"[margin] {w.name} {k}: worst err/bound {worst:.3f} ({per_level})")
    return margins
