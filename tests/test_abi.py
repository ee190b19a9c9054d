"""The C-ABI library on the CPU: it loads, exports every symbol include/*.h
declares, and rejects invalid arguments before any CUDA call (no GPU is
touched by these tests)."""
import ctypes
import glob
import os
import re

import pytest

import scale_deformable_attention_forward_gb300 as msda
from scale_deformable_attention_forward_gb300 import build as msda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    msda_build.build()
    return msda.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"msda_forward", "msda_backward", "msda_backward_workspace_size", "msda_status_string",
            "msda_last_cuda_error"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code in range(-11, 1):
        s = msda.msda_status_string(code)
        assert s and s != "unknown status"
    assert msda.msda_status_string(-99) == "unknown status"
    assert lib.msda_last_cuda_error() == 0


def test_staged_copy_status_reaches_the_caller(lib):
    """MSDA_ERR_STAGE_COPY (a staged-forward block exited with its copy in
    flight, reported by msda_staged_timeouts) has its own code and message,
    and the binding turns it into an exception naming it.  (The condition
    itself needs a copy that never lands, which no test provokes on a GPU.)"""
    assert msda.STATUS_STAGE_COPY == -11
    err = msda.MSDAError(msda.STATUS_STAGE_COPY, "msda_staged_timeouts")
    assert "shared-memory copy" in str(err) and "-11" in str(err)


LEVELS = ((4, 6), (2, 3))
STARTS = (0, 24)
DIMS = (2, 5, 3, 8, 2, 4, 30)  # B, N_q, N_h, C_h, N_l, N_p, L
FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every case below fails validation

# The rejection tests hand the library placeholder pointers.  They are meant
# to fail validation before any launch; to rule out a launch on a placeholder
# should validation ever regress, they run only where no GPU is visible.
no_gpu = pytest.mark.skipif(
    __import__("torch").cuda.is_available(), reason="placeholder-pointer tests run only without a GPU")


def _fwd(lib, desc, value=FAKE, loc=FAKE, attn=FAKE, out=FAKE):
    return lib.msda_forward(desc.ref() if desc is not None else None, value, loc, attn, out, None)


def _fwd_staged(lib, desc, value=FAKE, loc=FAKE, attn=FAKE, out=FAKE):
    return lib.msda_forward_staged(desc.ref() if desc is not None else None, value, loc, attn, out, None)


def _bwd(lib, desc, flags=(1, 1, 1), ws=None, ws_bytes=0, **ptrs):
    p = dict(go=FAKE, value=FAKE, loc=FAKE, attn=FAKE, gv=FAKE, gl=FAKE, ga=FAKE)
    p.update(ptrs)
    return lib.msda_backward(desc.ref(), p["go"], p["value"], p["loc"], p["attn"], *flags, p["gv"], p["gl"],
                             p["ga"], ws, ws_bytes, None)


@no_gpu
@pytest.mark.parametrize("entry", ["msda_forward", "msda_forward_staged"])
def test_rejections_forward(lib, entry):
    """Both forward entry points validate the same way."""
    d = msda.make_desc
    _fwd = globals()["_fwd_staged" if entry == "msda_forward_staged" else "_fwd"]
    assert _fwd(lib, None) == -1
    assert _fwd(lib, d(DIMS, LEVELS, STARTS), out=None) == -1
    assert _fwd(lib, d(DIMS, LEVELS, STARTS), value=None) == -1
    bad = d(DIMS, LEVELS, STARTS)
    bad.c.value_layout = 7
    assert _fwd(lib, bad) == -2
    bad = d(DIMS, LEVELS, STARTS)
    bad.c.padding_mode = 2
    assert _fwd(lib, bad) == -2
    bad = d(DIMS, LEVELS, STARTS)
    bad.c.align_corners = 3
    assert _fwd(lib, bad) == -2
    assert _fwd(lib, d((2, -1, 3, 8, 2, 4, 30), LEVELS, STARTS)) == -3
    assert _fwd(lib, d((2, 5, 3, 8, 17, 4, 30), LEVELS * 9, STARTS * 9)) == -3
    assert _fwd(lib, d(DIMS, LEVELS, (1, 24))) == -5          # start[0] != 0
    assert _fwd(lib, d(DIMS, LEVELS, (0, 23))) == -5          # start[1] != H0*W0
    assert _fwd(lib, d((2, 5, 3, 8, 2, 4, 31), LEVELS, STARTS)) == -5  # L != sum
    assert _fwd(lib, d(DIMS, ((0, 6), (2, 3)), (0, 0))) == -5  # empty level
    assert _fwd(lib, d(DIMS, LEVELS, STARTS, value_dtype=msda.DTYPE_F16)) == -8  # binary16 value
    assert _fwd(lib, d(DIMS, LEVELS, STARTS, loc_dtype=7)) == -2
    assert _fwd(lib, d(DIMS, LEVELS, STARTS, loc_dtype=msda.DTYPE_BF16), loc=ctypes.c_void_p(0x10001)) == -9
    assert _fwd(lib, d(DIMS, LEVELS, STARTS), value=ctypes.c_void_p(0x10002)) == -9
    big = ((46341, 46341),)
    assert _fwd(lib, d((1, 1, 1, 1, 1, 1, 46341 * 46341), big, (0,))) == -7
    assert _fwd(lib, d((1, 1, 64, 64, 1, 1, 1 << 20), ((1024, 1024),), (0,))) == -7


@no_gpu
@pytest.mark.parametrize("entry", ["msda_backward", "msda_backward_staged"])
def test_rejections_backward(lib, entry):
    """Both backward entry points validate the same way."""
    d = msda.make_desc(DIMS, LEVELS, STARTS)

    def _bwd(lib, desc, flags=(1, 1, 1), ws=None, ws_bytes=0, **ptrs):
        p = dict(go=FAKE, value=FAKE, loc=FAKE, attn=FAKE, gv=FAKE, gl=FAKE, ga=FAKE)
        p.update(ptrs)
        return getattr(lib, entry)(desc.ref(), p["go"], p["value"], p["loc"], p["attn"], *flags, p["gv"], p["gl"],
                                   p["ga"], ws, ws_bytes, None)
    assert _bwd(lib, d, flags=(0, 0, 0)) == -4
    assert _bwd(lib, d, flags=(2, 0, 0)) == -2
    assert _bwd(lib, d, gv=None) == -1
    assert _bwd(lib, d, flags=(0, 1, 0), gl=None) == -1
    assert _bwd(lib, d, flags=(0, 0, 1), ga=None) == -1
    assert _bwd(lib, d, flags=(0, 1, 0), value=None) == -1
    assert _bwd(lib, d, flags=(1, 0, 0), attn=None) == -1     # grad_value needs the weights
    assert _bwd(lib, d, flags=(1, 0, 0), gv=ctypes.c_void_p(0x10001)) == -9
    bf = msda.make_desc(DIMS, LEVELS, STARTS, value_dtype=msda.DTYPE_BF16)
    need = lib.msda_backward_workspace_size(bf.ref(), 1)
    assert need == 2 * 30 * 3 * 8 * 4
    assert lib.msda_backward_workspace_size(bf.ref(), 0) == 0
    assert lib.msda_backward_workspace_size(d.ref(), 1) == 0
    assert _bwd(lib, bf, ws=None, ws_bytes=0) == -6
    assert _bwd(lib, bf, ws=FAKE, ws_bytes=need - 1) == -6
    assert _bwd(lib, bf, ws=None, ws_bytes=need) == -1
    assert _bwd(lib, bf, ws=ctypes.c_void_p(0x10004), ws_bytes=need) == -9


@no_gpu
def test_rejections_backward_accumulate(lib):
    d = msda.make_desc(DIMS, LEVELS, STARTS)
    P = ctypes.c_void_p

    def acc_call(acc, flags=(1, 1, 1)):
        lib.msda_backward_accumulate.argtypes = [ctypes.POINTER(msda.msda_desc), P, P, P, P, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, P, P, P, P, ctypes.c_size_t, P]
        return lib.msda_backward_accumulate(d.ref(), FAKE, FAKE, FAKE, FAKE, *flags, acc, FAKE, FAKE, None, 0, None)

    assert acc_call(None) == -1                       # grad_value requested, no accumulator
    assert acc_call(ctypes.c_void_p(0x10002)) == -9   # binary32 accumulator must be 4-byte aligned
    assert acc_call(FAKE, flags=(0, 0, 0)) == -4


def test_python_binding_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    v = torch.zeros(1, 30, 1, 4)
    loc = torch.zeros(1, 2, 1, 2, 1, 2)
    a = torch.zeros(1, 2, 1, 2, 1)
    with pytest.raises(ValueError):
        msda.msda_forward(v, LEVELS, STARTS, loc, a)
    with pytest.raises(ValueError):
        msda.msda_backward(torch.zeros(1, 2, 4), v, LEVELS, STARTS, loc, a)


def test_staged_timeouts_rejects_null(lib):
    assert lib.msda_staged_timeouts(None) == -1


def _staged_levels(w, **over):
    from scale_deformable_attention_forward_gb300 import inputs as gen
    kw = dict(value_layout=w.value_layout, sampling_locations_layout=w.loc_layout, align_corners=w.align_corners,
              padding_mode=w.padding_mode, value_dtype=msda.DTYPE_BF16 if w.dtype == "bf16" else msda.DTYPE_F32)
    kw.update(over)
    dims = over.pop("dims", None) or (w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L)
    kw.pop("dims", None)
    return msda.staged_levels(msda.make_desc(dims, w.levels, w.level_start_index, **kw))


def test_staged_level_choice():
    """The coarsest levels whose pixels of one head fit 40 KB, each rounded up
    to whole 32-pixel boxes: level 3 only for every workload (encoder32,
    binary32 at 128 B a pixel: 288 px = 36 KB, with level 2 1344 px = 168 KB;
    the bfloat16 workloads at 64 B a pixel: 18 KB and 16 KB, with level 2
    84 KB and 80 KB)."""
    from scale_deformable_attention_forward_gb300 import inputs as gen
    W = gen.WORKLOADS
    assert _staged_levels(W["encoder32"]) == 3
    assert _staged_levels(W["decoder"]) == 3
    assert _staged_levels(W["encoder16"]) == 3
    assert _staged_levels(W["hires16"]) == 3
    w = W["encoder32"]
    N_l = w.N_l
    assert _staged_levels(w, loc_dtype=msda.DTYPE_BF16) == N_l  # 16-bit locations: the direct kernel
    B, N_q, N_h, C_h, _, N_p, L = w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L
    assert _staged_levels(w, dims=(B, N_q, N_h, 5, N_l, N_p, L)) == N_l    # scalar path
    assert _staged_levels(w, dims=(B, N_q, N_h, 96, N_l, N_p, L)) == N_l   # wide rows
    assert _staged_levels(w, dims=(B, N_q, N_h, 64, N_l, N_p, L)) == N_l   # 288 px x 256 B = 72 KB: none fits
    assert _staged_levels(w, dims=(B, N_q, N_h, 32, N_l, N_p, L), value_dtype=msda.DTYPE_BF16) == 3
    assert _staged_levels(w, dims=(B, N_q, N_h, 4, N_l, N_p, L), value_dtype=msda.DTYPE_BF16) == N_l  # 8-byte rows
    # 16-byte pixels: levels 2-3 fit (1344 px = 21 KB), with level 1 87 KB
    assert _staged_levels(w, dims=(B, N_q, N_h, 8, N_l, N_p, L), value_dtype=msda.DTYPE_BF16) == 2
    one = msda.make_desc((1, 4, 1, 32, 1, 1, 40000), ((200, 200),), (0,))
    assert msda.staged_levels(one) == 1  # 5 MB: no level fits
    small = msda.make_desc((1, 4, 1, 32, 1, 1, 20), ((4, 5),), (0,))
    assert msda.staged_levels(small) == 1  # L < 32 pixels


def test_staged_levels_rejects_bad_input(lib):
    d = msda.make_desc(DIMS, LEVELS, STARTS)
    assert lib.msda_forward_staged_levels(d.ref(), None) == -1
    bad = msda.make_desc(DIMS, LEVELS, (1, 24))
    n = ctypes.c_int(0)
    assert lib.msda_forward_staged_levels(bad.ref(), ctypes.byref(n)) == -5


def test_backward_staged_level_choice():
    """The shared accumulator is binary32 whatever value's dtype (C_h * 4
    bytes a pixel, 40 KB): level 3 for every workload; none at C_h = 64
    (73 KB); C_h = 12 (48 B a pixel) keeps level 3 only (level 2 would make it
    64 KB); not for the scalar path or wide rows."""
    from scale_deformable_attention_forward_gb300 import inputs as gen
    W = gen.WORKLOADS

    def lv(w, C_h=None, **over):
        kw = dict(value_layout=w.value_layout, sampling_locations_layout=w.loc_layout,
                  align_corners=w.align_corners, padding_mode=w.padding_mode,
                  value_dtype=msda.DTYPE_BF16 if w.dtype == "bf16" else msda.DTYPE_F32)
        kw.update(over)
        dims = (w.B, w.n_queries, w.N_h, C_h or w.C_h, w.N_l, w.N_p, w.L)
        return msda.backward_staged_levels(msda.make_desc(dims, w.levels, w.level_start_index, **kw))

    for name in ("encoder32", "decoder", "encoder16", "hires16"):
        assert lv(W[name]) == 3, name
    w = W["encoder32"]
    assert lv(w, 64) == w.N_l
    assert lv(w, 12) == 3
    assert lv(w, 5) == w.N_l
    assert lv(w, 96) == w.N_l
    d = msda.make_desc(DIMS, LEVELS, STARTS)
    assert lib_staged_rejects(d)


def lib_staged_rejects(d):
    lib = msda.load_library()
    return lib.msda_backward_staged_levels(d.ref(), None) == -1
