"""GB300-native multi-scale deformable attention (MSDA), forward and backward.

A thin ctypes binding of ``libmsda.so`` (declared in ``include/msda.h``).
This module only marshals arguments: it checks tensor shapes, dtypes and
devices, allocates outputs with PyTorch when the caller does not pass them,
and hands raw device pointers plus the current CUDA stream to the library.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback -- if the library is missing, calls raise.

The functions follow the pages "MS Deformable Attention Kernel API
Reference" (``msda_forward``) and "MS Deformable Attention Backward Kernel API
Reference" (``msda_backward``): same argument names, layouts
(value ``BLNC``/``BNLC``, sampling_locations ``BQHLP2``/``B2QHLP``),
``align_corners``, ``padding_mode`` and ``compute_grad_*`` flags.  Beside
them: ``msda_backward_accumulate`` (adds into a persistent float32
grad_value), ``msda_forward_logits`` / ``msda_backward_logits`` (softmax of
attention logits inside the kernels), and the staged variants
``msda_forward_staged`` / ``msda_backward_staged`` (coarse levels held in
shared memory; same results, measured slower on GB300 than the direct
kernels the plain calls use).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple, Union

__all__ = ["msda_forward", "msda_backward", "msda_backward_workspace_size", "msda_status_string",
           "msda_backward_accumulate", "msda_forward_logits", "msda_backward_logits", "msda_forward_staged",
           "msda_backward_staged", "staged_levels", "backward_staged_levels", "staged_timeouts",
           "MSDAError", "library_path", "load_library", "make_desc"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libmsda.so")

VALUE_LAYOUTS = {"BLNC": 0, "BNLC": 1}
LOC_LAYOUTS = {"BQHLP2": 0, "B2QHLP": 1}
PADDING_MODES = {"zeros": 0, "border": 1}
DTYPE_F32, DTYPE_BF16, DTYPE_F16 = 0, 1, 2
MAX_LEVELS = 16


class msda_desc(ctypes.Structure):
    """Mirror of ``struct msda_desc`` in include/msda.h."""

    _fields_ = [("B", ctypes.c_int64), ("N_q", ctypes.c_int64), ("N_h", ctypes.c_int64),
                ("C_h", ctypes.c_int64), ("N_l", ctypes.c_int64), ("N_p", ctypes.c_int64),
                ("L", ctypes.c_int64), ("spatial_shapes", ctypes.c_void_p),
                ("level_start_index", ctypes.c_void_p), ("value_layout", ctypes.c_int32),
                ("loc_layout", ctypes.c_int32), ("align_corners", ctypes.c_int32),
                ("padding_mode", ctypes.c_int32), ("value_dtype", ctypes.c_int32),
                ("loc_dtype", ctypes.c_int32)]


STATUS_STAGE_COPY = -11  # msda_staged_timeouts: a staged block exited with its copy in flight


class MSDAError(RuntimeError):
    """A non-zero status returned by libmsda."""

    def __init__(self, status: int, where: str):
        self.status = status
        msg = msda_status_string(status)
        if status == -10:
            msg += f" (cudaError {load_library().msda_last_cuda_error()})"
        super().__init__(f"{where}: libmsda status {status}: {msg}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libmsda.so (built by ``scale_deformable_attention_forward_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"libmsda.so is not built ({_LIB_PATH}); run "
                                   "`python -m scale_deformable_attention_forward_gb300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            D = ctypes.POINTER(msda_desc)
            lib.msda_forward.argtypes = [D, P, P, P, P, P]
            lib.msda_forward.restype = I
            lib.msda_backward_workspace_size.argtypes = [D, I]
            lib.msda_backward_workspace_size.restype = Z
            lib.msda_backward.argtypes = [D, P, P, P, P, I, I, I, P, P, P, P, Z, P]
            lib.msda_backward.restype = I
            lib.msda_backward_accumulate.argtypes = [D, P, P, P, P, I, I, I, P, P, P, P, Z, P]
            lib.msda_backward_accumulate.restype = I
            lib.msda_forward_logits.argtypes = [D, P, P, P, P, P]
            lib.msda_forward_logits.restype = I
            lib.msda_forward_staged.argtypes = [D, P, P, P, P, P]
            lib.msda_forward_staged.restype = I
            lib.msda_staged_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint)]
            lib.msda_staged_timeouts.restype = I
            lib.msda_forward_staged_levels.argtypes = [D, ctypes.POINTER(ctypes.c_int)]
            lib.msda_forward_staged_levels.restype = I
            lib.msda_backward_staged.argtypes = [D, P, P, P, P, I, I, I, P, P, P, P, Z, P]
            lib.msda_backward_staged.restype = I
            lib.msda_backward_staged_levels.argtypes = [D, ctypes.POINTER(ctypes.c_int)]
            lib.msda_backward_staged_levels.restype = I
            lib.msda_backward_logits.argtypes = [D, P, P, P, P, I, I, I, P, P, P, P, Z, P]
            lib.msda_backward_logits.restype = I
            lib.msda_status_string.argtypes = [I]
            lib.msda_status_string.restype = ctypes.c_char_p
            lib.msda_last_cuda_error.argtypes = []
            lib.msda_last_cuda_error.restype = I
            _lib = lib
    return _lib


def msda_status_string(status: int) -> str:
    return load_library().msda_status_string(int(status)).decode()


class _Desc:
    """A msda_desc plus the host arrays it points to (kept alive together)."""

    def __init__(self, dims, spatial_shapes, level_start_index, value_layout, loc_layout,
                 align_corners, padding_mode, value_dtype, loc_dtype=DTYPE_F32):
        B, N_q, N_h, C_h, N_l, N_p, L = (int(x) for x in dims)
        shapes = [int(v) for hw in spatial_shapes for v in hw]
        starts = [int(v) for v in level_start_index]
        self._shapes = (ctypes.c_int64 * max(1, len(shapes)))(*shapes)
        self._starts = (ctypes.c_int64 * max(1, len(starts)))(*starts)
        if value_layout not in VALUE_LAYOUTS:
            raise ValueError(f"value_layout must be one of {sorted(VALUE_LAYOUTS)}, got {value_layout!r}")
        if loc_layout not in LOC_LAYOUTS:
            raise ValueError(f"sampling_locations_layout must be one of {sorted(LOC_LAYOUTS)}, got {loc_layout!r}")
        if padding_mode not in PADDING_MODES:
            raise ValueError(f"padding_mode must be one of {sorted(PADDING_MODES)}, got {padding_mode!r}")
        self.c = msda_desc(B, N_q, N_h, C_h, N_l, N_p, L,
                           ctypes.cast(self._shapes, ctypes.c_void_p),
                           ctypes.cast(self._starts, ctypes.c_void_p),
                           VALUE_LAYOUTS[value_layout], LOC_LAYOUTS[loc_layout], int(bool(align_corners)),
                           PADDING_MODES[padding_mode], value_dtype, loc_dtype)

    def ref(self):
        return ctypes.byref(self.c)


def make_desc(dims, spatial_shapes, level_start_index, value_layout="BLNC",
              sampling_locations_layout="BQHLP2", align_corners=False, padding_mode="zeros",
              value_dtype=DTYPE_F32, loc_dtype=DTYPE_F32) -> _Desc:
    """Build a descriptor from (B, N_q, N_h, C_h, N_l, N_p, L) and level tuples."""
    return _Desc(dims, spatial_shapes, level_start_index, value_layout, sampling_locations_layout,
                 align_corners, padding_mode, value_dtype, loc_dtype)


# ----------------------------------------------------------------------------- tensors
def _torch():
    import torch
    return torch


def _levels(spatial_shapes, level_start_index):
    torch = _torch()
    if isinstance(spatial_shapes, torch.Tensor):
        spatial_shapes = spatial_shapes.detach().cpu().reshape(-1, 2).tolist()
    if isinstance(level_start_index, torch.Tensor):
        level_start_index = level_start_index.detach().cpu().reshape(-1).tolist()
    shapes = [(int(h), int(w)) for h, w in spatial_shapes]
    return shapes, [int(s) for s in level_start_index]


def _dims(value, sampling_locations, value_layout, loc_layout):
    if value.dim() != 4:
        raise ValueError(f"value must be 4-D ({value_layout}), got shape {tuple(value.shape)}")
    if value_layout == "BLNC":
        B, L, N_h, C_h = value.shape
    elif value_layout == "BNLC":
        B, N_h, L, C_h = value.shape
    else:
        raise ValueError(f"value_layout must be 'BLNC' or 'BNLC', got {value_layout!r}")
    if sampling_locations.dim() != 6:
        raise ValueError(f"sampling_locations must be 6-D ({loc_layout}), got {tuple(sampling_locations.shape)}")
    if loc_layout == "BQHLP2":
        b2, N_q, h2, N_l, N_p, two = sampling_locations.shape
    elif loc_layout == "B2QHLP":
        b2, two, N_q, h2, N_l, N_p = sampling_locations.shape
    else:
        raise ValueError(f"sampling_locations_layout must be 'BQHLP2' or 'B2QHLP', got {loc_layout!r}")
    if b2 != B or h2 != N_h or two != 2:
        raise ValueError(f"sampling_locations {tuple(sampling_locations.shape)} does not match value "
                         f"{tuple(value.shape)} in layouts {value_layout}/{loc_layout}")
    return B, N_q, N_h, C_h, N_l, N_p, L


def _value_dtype(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"value must be float32 or bfloat16, got {t.dtype}")


def _loc_dtype(t):
    """msda_dtype of sampling_locations / attention weights (and their gradients)."""
    torch = _torch()
    codes = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16}
    if t.dtype not in codes:
        raise TypeError(f"sampling_locations must be float32, bfloat16 or float16, got {t.dtype}")
    return codes[t.dtype]


def _check(t, name, dtype, shape, device):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(_torch().cuda.current_stream(device).cuda_stream)


def msda_forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                 value_layout: str = "BLNC", sampling_locations_layout: str = "BQHLP2",
                 align_corners: bool = False, padding_mode: str = "zeros", out=None, _logits: bool = False,
                 _staged: bool = False):
    """Multi-scale deformable attention forward on the GPU.

    value (B,L,N_h,C_h) or (B,N_h,L,C_h), float32 or bfloat16;
    sampling_locations (B,N_q,N_h,N_l,N_p,2) or (B,2,N_q,N_h,N_l,N_p), float32;
    attention_weights (B,N_q,N_h,N_l,N_p), float32.  All CUDA tensors on one
    device, contiguous.  Returns out (B, N_q, N_h*C_h) in value's dtype,
    enqueued on the current stream.
    """
    torch = _torch()
    lib = load_library()
    B, N_q, N_h, C_h, N_l, N_p, L = _dims(value, sampling_locations, value_layout, sampling_locations_layout)
    if value.device.type != "cuda":
        raise ValueError("msda_forward runs on CUDA tensors only")
    dev = value.device
    shapes, starts = _levels(spatial_shapes, level_start_index)
    if len(shapes) != N_l or len(starts) != N_l:
        raise ValueError(f"spatial_shapes/level_start_index have {len(shapes)}/{len(starts)} levels, "
                         f"sampling_locations has {N_l}")
    vdt = _value_dtype(value)
    _check(value, "value", value.dtype, value.shape, dev)
    ldt = _loc_dtype(sampling_locations)
    _check(sampling_locations, "sampling_locations", sampling_locations.dtype, sampling_locations.shape, dev)
    _check(attention_weights, "attention_weights", sampling_locations.dtype, (B, N_q, N_h, N_l, N_p), dev)
    if out is None:
        out = torch.empty((B, N_q, N_h * C_h), dtype=value.dtype, device=dev)
    else:
        _check(out, "out", value.dtype, (B, N_q, N_h * C_h), dev)
    d = make_desc((B, N_q, N_h, C_h, N_l, N_p, L), shapes, starts, value_layout,
                  sampling_locations_layout, align_corners, padding_mode, vdt, ldt)
    fn, name = ((lib.msda_forward_logits, "msda_forward_logits") if _logits else
                (lib.msda_forward_staged, "msda_forward_staged") if _staged else (lib.msda_forward, "msda_forward"))
    with torch.cuda.device(dev):
        rc = fn(d.ref(), _ptr(value), _ptr(sampling_locations), _ptr(attention_weights), _ptr(out), _stream(dev))
    if rc != 0:
        raise MSDAError(rc, name)
    return out


def msda_forward_staged(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                        value_layout: str = "BLNC", sampling_locations_layout: str = "BQHLP2",
                        align_corners: bool = False, padding_mode: str = "zeros", out=None):
    """msda_forward through the staged-level kernel: each thread block copies
    the coarsest levels of its head that fit in shared memory there (TMA) and
    gathers those levels' corners from it.  Same arguments and the same (bit
    for bit) result as msda_forward; shapes the staged kernel does not cover
    run msda_forward's kernel."""
    return msda_forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                        value_layout, sampling_locations_layout, align_corners, padding_mode, out, _staged=True)


def staged_levels(desc) -> int:
    """First level msda_forward_staged stages for descriptor `desc` (from
    make_desc); N_l when it runs msda_forward's kernel."""
    lib = load_library()
    n = ctypes.c_int(0)
    rc = lib.msda_forward_staged_levels(desc.ref(), ctypes.byref(n))
    if rc != 0:
        raise MSDAError(rc, "msda_forward_staged_levels")
    return int(n.value)


def staged_timeouts() -> int:
    """Staged-forward blocks (since the library was loaded) that gave up
    waiting for their shared-memory copy; synchronises with the device.
    Raises MSDAError (status STATUS_STAGE_COPY) if such a block exited while
    its copy was still in flight."""
    lib = load_library()
    n = ctypes.c_uint(0)
    rc = lib.msda_staged_timeouts(ctypes.byref(n))
    if rc != 0:
        raise MSDAError(rc, "msda_staged_timeouts")
    return int(n.value)


def msda_forward_logits(value, spatial_shapes, level_start_index, sampling_locations, attention_logits,
                        value_layout: str = "BLNC", sampling_locations_layout: str = "BQHLP2",
                        align_corners: bool = False, padding_mode: str = "zeros", out=None):
    """msda_forward with attention logits (B,N_q,N_h,N_l,N_p), float32: the
    weights are the softmax over each (b, q, h)'s N_l*N_p logits, computed in
    the kernel."""
    return msda_forward(value, spatial_shapes, level_start_index, sampling_locations, attention_logits,
                        value_layout, sampling_locations_layout, align_corners, padding_mode, out, _logits=True)


def msda_backward_workspace_size(value, spatial_shapes, level_start_index, sampling_locations,
                                 value_layout: str = "BLNC", sampling_locations_layout: str = "BQHLP2",
                                 compute_grad_value: bool = True) -> int:
    """Bytes of workspace msda_backward needs for these tensors."""
    B, N_q, N_h, C_h, N_l, N_p, L = _dims(value, sampling_locations, value_layout, sampling_locations_layout)
    shapes, starts = _levels(spatial_shapes, level_start_index)
    d = make_desc((B, N_q, N_h, C_h, N_l, N_p, L), shapes, starts, value_layout,
                  sampling_locations_layout, False, "zeros", _value_dtype(value))
    return int(load_library().msda_backward_workspace_size(d.ref(), int(bool(compute_grad_value))))


def msda_backward(grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                  attention_weights, value_layout: str = "BLNC", sampling_locations_layout: str = "BQHLP2",
                  align_corners: bool = False, padding_mode: str = "zeros", compute_grad_value: bool = True,
                  compute_grad_sampling_locations: bool = True, compute_grad_attention_weights: bool = True,
                  grad_value=None, grad_sampling_locations=None, grad_attention_weights=None,
                  workspace=None, _accumulate: bool = False, _logits: bool = False,
                  _staged: bool = False) -> Tuple:
    """Multi-scale deformable attention backward on the GPU.

    Returns (grad_value, grad_sampling_locations, grad_attention_weights);
    a disabled output is None.  grad_value has value's shape, layout and
    dtype; grad_sampling_locations sampling_locations' shape and layout
    (float32); grad_attention_weights (B,N_q,N_h,N_l,N_p) float32.  For
    bfloat16 value with compute_grad_value, a float32 accumulator of
    ``msda_backward_workspace_size`` bytes is needed; it is allocated here
    when ``workspace`` is None.
    """
    torch = _torch()
    lib = load_library()
    B, N_q, N_h, C_h, N_l, N_p, L = _dims(value, sampling_locations, value_layout, sampling_locations_layout)
    if value.device.type != "cuda":
        raise ValueError("msda_backward runs on CUDA tensors only")
    dev = value.device
    shapes, starts = _levels(spatial_shapes, level_start_index)
    if len(shapes) != N_l or len(starts) != N_l:
        raise ValueError("spatial_shapes/level_start_index do not match sampling_locations' level axis")
    vdt = _value_dtype(value)
    _check(value, "value", value.dtype, value.shape, dev)
    _check(grad_output, "grad_output", value.dtype, (B, N_q, N_h * C_h), dev)
    ldt = _loc_dtype(sampling_locations)
    _check(sampling_locations, "sampling_locations", sampling_locations.dtype, sampling_locations.shape, dev)
    _check(attention_weights, "attention_weights", sampling_locations.dtype, (B, N_q, N_h, N_l, N_p), dev)
    fv, fl, fa = (bool(compute_grad_value), bool(compute_grad_sampling_locations),
                  bool(compute_grad_attention_weights))
    if not (fv or fl or fa):
        raise ValueError("at least one of compute_grad_value / compute_grad_sampling_locations / "
                         "compute_grad_attention_weights must be True")
    if fv:
        if _accumulate:
            if grad_value is None:
                raise ValueError("msda_backward_accumulate needs grad_value_accum")
            _check(grad_value, "grad_value_accum", torch.float32, value.shape, dev)
        else:
            if grad_value is None:
                grad_value = torch.empty_like(value)
            _check(grad_value, "grad_value", value.dtype, value.shape, dev)
    else:
        grad_value = None
    if fl:
        if grad_sampling_locations is None:
            grad_sampling_locations = torch.empty_like(sampling_locations)
        _check(grad_sampling_locations, "grad_sampling_locations", sampling_locations.dtype,
               sampling_locations.shape, dev)
    else:
        grad_sampling_locations = None
    if fa:
        if grad_attention_weights is None:
            grad_attention_weights = torch.empty_like(attention_weights)
        _check(grad_attention_weights, "grad_attention_weights", sampling_locations.dtype,
               attention_weights.shape, dev)
    else:
        grad_attention_weights = None
    d = make_desc((B, N_q, N_h, C_h, N_l, N_p, L), shapes, starts, value_layout,
                  sampling_locations_layout, align_corners, padding_mode, vdt, ldt)
    ws_bytes = int(lib.msda_backward_workspace_size(d.ref(), int(fv)))
    if ws_bytes > 0:
        if workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        elif workspace.device != dev or workspace.numel() * workspace.element_size() < ws_bytes:
            raise ValueError(f"workspace must hold {ws_bytes} bytes on {dev}")
    with torch.cuda.device(dev):
        fn = (lib.msda_backward_accumulate if _accumulate else
              lib.msda_backward_logits if _logits else
              lib.msda_backward_staged if _staged else lib.msda_backward)
        rc = fn(d.ref(), _ptr(grad_output), _ptr(value), _ptr(sampling_locations),
                               _ptr(attention_weights), int(fv), int(fl), int(fa), _ptr(grad_value),
                               _ptr(grad_sampling_locations), _ptr(grad_attention_weights),
                               _ptr(workspace) if ws_bytes > 0 else None, ws_bytes, _stream(dev))
    if rc != 0:
        raise MSDAError(rc, "msda_backward_accumulate" if _accumulate else
                        "msda_backward_logits" if _logits else
                        "msda_backward_staged" if _staged else "msda_backward")
    return grad_value, grad_sampling_locations, grad_attention_weights


def msda_backward_staged(grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, value_layout: str = "BLNC", sampling_locations_layout: str = "BQHLP2",
                         align_corners: bool = False, padding_mode: str = "zeros", compute_grad_value: bool = True,
                         compute_grad_sampling_locations: bool = True, compute_grad_attention_weights: bool = True,
                         grad_value=None, grad_sampling_locations=None, grad_attention_weights=None,
                         workspace=None) -> Tuple:
    """msda_backward with grad_value of the coarse levels accumulated per
    thread block in shared memory (then added in once per block); the same
    arguments and results (grad_value up to summation order)."""
    return msda_backward(grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, value_layout, sampling_locations_layout, align_corners, padding_mode,
                         compute_grad_value, compute_grad_sampling_locations, compute_grad_attention_weights,
                         grad_value=grad_value, grad_sampling_locations=grad_sampling_locations,
                         grad_attention_weights=grad_attention_weights, workspace=workspace, _staged=True)


def backward_staged_levels(desc) -> int:
    """First level msda_backward_staged accumulates in shared memory for
    descriptor `desc` (from make_desc); N_l when it runs msda_backward's
    kernels."""
    lib = load_library()
    n = ctypes.c_int(0)
    rc = lib.msda_backward_staged_levels(desc.ref(), ctypes.byref(n))
    if rc != 0:
        raise MSDAError(rc, "msda_backward_staged_levels")
    return int(n.value)



def msda_backward_accumulate(grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                             attention_weights, grad_value_accum, value_layout: str = "BLNC",
                             sampling_locations_layout: str = "BQHLP2", align_corners: bool = False,
                             padding_mode: str = "zeros", compute_grad_value: bool = True,
                             compute_grad_sampling_locations: bool = True,
                             compute_grad_attention_weights: bool = True, grad_sampling_locations=None,
                             grad_attention_weights=None, workspace=None) -> Tuple:
    """msda_backward that ADDS this call's grad_value into ``grad_value_accum``
    (a float32 tensor of value's shape and layout, never zeroed by the call),
    for query-chunked calls or gradient accumulation over micro-batches.
    Returns (grad_value_accum, grad_sampling_locations, grad_attention_weights)."""
    return msda_backward(grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, value_layout, sampling_locations_layout, align_corners, padding_mode,
                         compute_grad_value, compute_grad_sampling_locations, compute_grad_attention_weights,
                         grad_value=grad_value_accum, grad_sampling_locations=grad_sampling_locations,
                         grad_attention_weights=grad_attention_weights, workspace=workspace, _accumulate=True)


def msda_backward_logits(grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_logits, value_layout: str = "BLNC", sampling_locations_layout: str = "BQHLP2",
                         align_corners: bool = False, padding_mode: str = "zeros", compute_grad_value: bool = True,
                         compute_grad_sampling_locations: bool = True, compute_grad_attention_logits: bool = True,
                         grad_value=None, grad_sampling_locations=None, grad_attention_logits=None,
                         workspace=None) -> Tuple:
    """msda_backward with attention logits (see msda_forward_logits).
    Returns (grad_value, grad_sampling_locations, grad_attention_logits)."""
    return msda_backward(grad_output, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_logits, value_layout, sampling_locations_layout, align_corners, padding_mode,
                         compute_grad_value, compute_grad_sampling_locations, compute_grad_attention_logits,
                         grad_value=grad_value, grad_sampling_locations=grad_sampling_locations,
                         grad_attention_weights=grad_attention_logits, workspace=workspace, _logits=True)
