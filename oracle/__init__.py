"""CPU oracle for multi-scale deformable attention -- TEST INFRASTRUCTURE ONLY.

A ctypes wrapper around ``msda_oracle.c`` (plain float64 loops; that file
states what it follows and which readings it takes).  Only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this package; the CUDA library never does, and the two share no code.

Arrays are numpy; every input is widened to float64 here (inputs stored as
float32 or bfloat16 are widened exactly, so the oracle sees the numbers the
GPU sees).  Outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "msda_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmsda_oracle.so")

VALUE_LAYOUTS = {"BLNC": 0, "BNLC": 1}
LOC_LAYOUTS = {"BQHLP2": 0, "B2QHLP": 1}
PADDING_MODES = {"zeros": 0, "border": 1}

_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = SOURCE, out: str = _LIB) -> str:
    """Compile the oracle with gcc and return the shared library's path.

    -ffp-contract=off keeps the float64 arithmetic identical on x86-64 and
    aarch64 (no fused multiply-adds).  ``src``/``out`` let a test compile a
    modified copy of the source elsewhere.
    """
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(out), exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                        "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, out)
    return out


def _f64(x) -> np.ndarray:
    a = np.asarray(x)
    if a.dtype != np.float64 or not a.flags.c_contiguous:
        a = np.ascontiguousarray(a, dtype=np.float64)
    return a


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dims(value, spatial_shapes, sampling_locations, value_layout, loc_layout):
    if value_layout == "BLNC":
        B, L, N_h, C_h = value.shape
    else:
        B, N_h, L, C_h = value.shape
    if loc_layout == "BQHLP2":
        _, N_q, _, N_l, N_p, _ = sampling_locations.shape
    else:
        _, _, N_q, _, N_l, N_p = sampling_locations.shape
    if N_l != len(spatial_shapes):
        raise ValueError("sampling_locations' level axis does not match spatial_shapes")
    return B, N_q, N_h, C_h, N_l, N_p, L


def _level_arrays(spatial_shapes, level_start_index):
    shapes = np.ascontiguousarray(np.array(spatial_shapes, dtype=np.int64).reshape(-1, 2))
    starts = np.ascontiguousarray(np.array(level_start_index, dtype=np.int64).reshape(-1))
    return shapes, starts


class Oracle:
    """Forward/backward calls bound to one compiled copy of the oracle."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        common = [i64] * 7 + [p, p] + [i32] * 5
        lib.msda_oracle_forward.argtypes = common + [p, p, p, p]
        lib.msda_oracle_forward.restype = i32
        lib.msda_oracle_backward.argtypes = common + [p, p, p, p, i32, i32, i32, p, p, p]
        lib.msda_oracle_backward.restype = i32
        self.lib = lib

    def forward(self, value, spatial_shapes: Sequence[Tuple[int, int]],
                level_start_index: Sequence[int], sampling_locations, attention_weights,
                value_layout: str = "BLNC", sampling_locations_layout: str = "BQHLP2",
                align_corners: bool = False, padding_mode: str = "zeros",
                coord_f32: bool = False) -> np.ndarray:
        """MSDA forward in float64; returns out of shape (B, N_q, N_h*C_h)."""
        value, loc, attn = _f64(value), _f64(sampling_locations), _f64(attention_weights)
        B, N_q, N_h, C_h, N_l, N_p, L = _dims(value, spatial_shapes, loc, value_layout,
                                              sampling_locations_layout)
        shapes, starts = _level_arrays(spatial_shapes, level_start_index)
        out = np.empty((B, N_q, N_h * C_h), dtype=np.float64)
        rc = self.lib.msda_oracle_forward(
            B, N_q, N_h, C_h, N_l, N_p, L, _ptr(shapes), _ptr(starts),
            VALUE_LAYOUTS[value_layout], LOC_LAYOUTS[sampling_locations_layout],
            int(bool(align_corners)), PADDING_MODES[padding_mode], int(bool(coord_f32)),
            _ptr(value), _ptr(loc), _ptr(attn), _ptr(out))
        if rc != 0:
            raise ValueError(f"oracle rejected the problem (status {rc})")
        return out

    def backward(self, grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                 attention_weights, value_layout: str = "BLNC",
                 sampling_locations_layout: str = "BQHLP2", align_corners: bool = False,
                 padding_mode: str = "zeros", compute_grad_value: bool = True,
                 compute_grad_sampling_locations: bool = True,
                 compute_grad_attention_weights: bool = True, coord_f32: bool = False):
        """MSDA backward in float64.

        Returns (grad_value, grad_sampling_locations, grad_attention_weights)
        in the inputs' shapes and layouts; a disabled output is ``None``.
        """
        g, value = _f64(grad_output), _f64(value)
        loc, attn = _f64(sampling_locations), _f64(attention_weights)
        B, N_q, N_h, C_h, N_l, N_p, L = _dims(value, spatial_shapes, loc, value_layout,
                                              sampling_locations_layout)
        shapes, starts = _level_arrays(spatial_shapes, level_start_index)
        gv = np.empty(value.shape, dtype=np.float64) if compute_grad_value else None
        gl = np.empty(loc.shape, dtype=np.float64) if compute_grad_sampling_locations else None
        ga = np.empty(attn.shape, dtype=np.float64) if compute_grad_attention_weights else None
        rc = self.lib.msda_oracle_backward(
            B, N_q, N_h, C_h, N_l, N_p, L, _ptr(shapes), _ptr(starts),
            VALUE_LAYOUTS[value_layout], LOC_LAYOUTS[sampling_locations_layout],
            int(bool(align_corners)), PADDING_MODES[padding_mode], int(bool(coord_f32)),
            _ptr(g), _ptr(value), _ptr(loc), _ptr(attn),
            int(bool(compute_grad_value)), int(bool(compute_grad_sampling_locations)),
            int(bool(compute_grad_attention_weights)), _ptr(gv), _ptr(gl), _ptr(ga))
        if rc != 0:
            raise ValueError(f"oracle rejected the problem (status {rc})")
        return gv, gl, ga


def softmax_rows(attention_logits) -> np.ndarray:
    """Attention weights from logits (B, N_q, N_h, N_l, N_p): the softmax over
    the N_l*N_p (level, point) slots of each (b, q, h), in float64 -- how the
    workloads build their weights from N(0,1) logits."""
    z = _f64(attention_logits)
    flat = z.reshape(z.shape[:3] + (-1,))
    e = np.exp(flat - flat.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True)).reshape(z.shape)


def _forward_logits(self, value, spatial_shapes, level_start_index, sampling_locations, attention_logits,
                    **kw) -> np.ndarray:
    """The forward with the weights softmax(logits) (see softmax_rows)."""
    return self.forward(value, spatial_shapes, level_start_index, sampling_locations,
                        softmax_rows(attention_logits), **kw)


def _backward_logits(self, grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                     attention_logits, compute_grad_value: bool = True,
                     compute_grad_sampling_locations: bool = True, compute_grad_attention_logits: bool = True,
                     **kw):
    """The backward with the weights softmax(logits): grad_value and
    grad_sampling_locations as for those weights, and for the logits the
    chain rule of the softmax, dz = A * (gA - sum over the row of A * gA)."""
    A = softmax_rows(attention_logits)
    gv, gl, gA = self.backward(grad_output, value, spatial_shapes, level_start_index, sampling_locations, A,
                               compute_grad_value=compute_grad_value,
                               compute_grad_sampling_locations=compute_grad_sampling_locations,
                               compute_grad_attention_weights=compute_grad_attention_logits, **kw)
    gz = None
    if compute_grad_attention_logits:
        s = (A * gA).reshape(A.shape[:3] + (-1,)).sum(axis=-1)[..., None, None]
        gz = A * (gA - s)
    return gv, gl, gz


Oracle.forward_logits = _forward_logits
Oracle.backward_logits = _backward_logits


def default() -> Oracle:
    """The oracle built from ``msda_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def forward(*args, **kwargs) -> np.ndarray:
    """MSDA forward in float64 (see :meth:`Oracle.forward`)."""
    return default().forward(*args, **kwargs)


def backward(*args, **kwargs):
    """MSDA backward in float64 (see :meth:`Oracle.backward`)."""
    return default().backward(*args, **kwargs)


def forward_logits(*args, **kwargs) -> np.ndarray:
    """MSDA forward with attention logits (see :func:`softmax_rows`)."""
    return default().forward_logits(*args, **kwargs)


def backward_logits(*args, **kwargs):
    """MSDA backward with attention logits; returns the logits' gradient third."""
    return default().backward_logits(*args, **kwargs)
