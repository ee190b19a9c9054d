"""Seeded synthetic workloads for multi-scale deformable attention (MSDA).

This module is the one piece shared by the CUDA path's tests/benchmark and by
the CPU oracle's tests: it draws the inputs and nothing else.  It holds none of
the method's arithmetic (no coordinate mapping, no interpolation, no
gradients).  Every array is drawn from ``numpy.random.Generator(PCG64(seed))``
in float64 and then rounded once to the dtype it is stored in, so both sides
see bit-identical numbers.

Tensor shapes and layouts follow "MS Deformable Attention Kernel API
Reference", Parameters:
  value               BLNC (B, L, N_h, C_h)  or BNLC (B, N_h, L, C_h)
  sampling_locations  BQHLP2 (B, N_q, N_h, N_l, N_p, 2) or B2QHLP (B, 2, N_q, N_h, N_l, N_p)
  attention_weights   (B, N_q, N_h, N_l, N_p)
and grad_output (B, N_q, N_h*C_h) from "MS Deformable Attention Backward
Kernel API Reference", Parameters.  The last axis of BQHLP2 (and the "2" axis
of B2QHLP) holds (x, y): x runs along the width W_i, y along the height H_i.

There is no public dataset for this operator; the workloads below are
Deformable-DETR-shaped stand-ins (a 4-level feature pyramid, 8 heads, 32
channels per head, 4 or 8 points per level).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional, Sequence, Tuple

import numpy as np

# Deformable-DETR pyramid for an ~800x1333 image: strides 8, 16, 32, 64.
LEVELS_DETR: Tuple[Tuple[int, int], ...] = ((100, 167), (50, 84), (25, 42), (13, 21))
# Square high-resolution pyramid.
LEVELS_HIRES: Tuple[Tuple[int, int], ...] = ((128, 128), (64, 64), (32, 32), (16, 16))


@dataclass(frozen=True)
class Workload:
    """One synthetic MSDA problem.

    ``N_q`` of ``None`` means one query per pyramid pixel (N_q = L, encoder
    style).  ``loc_recipe`` is one of:
      * ``"uniform"``: every coordinate iid U(loc_lo, loc_hi);
      * ``"ref_uniform"``: a reference point U(0,1)^2 per (b, q), shared by
        all heads/levels/points, plus an offset N(0, sigma = 2/W_l) on each
        axis at sampled level l (decoder style);
      * ``"pixel_centre"``: query i is pyramid pixel i (flattened order); its
        reference point is that pixel's centre ((x+0.5)/W, (y+0.5)/H) at its
        own level, plus the same N(0, 2/W_l) offsets (encoder style).
    Attention weights are a softmax over the N_l*N_p (level, point) slots of
    N(0,1) logits, per (b, q, h).
    """

    name: str
    B: int
    N_q: Optional[int]
    N_h: int
    C_h: int
    N_p: int
    levels: Tuple[Tuple[int, int], ...]
    dtype: str = "f32"  # storage dtype of value / out / grad_output / grad_value
    loc_dtype: str = "f32"  # storage dtype of locations, attention weights / logits and their gradients
    value_layout: str = "BLNC"
    loc_layout: str = "BQHLP2"
    align_corners: bool = False
    padding_mode: str = "zeros"
    loc_recipe: str = "uniform"
    loc_lo: float = -0.1
    loc_hi: float = 1.1
    seed: int = 0

    @property
    def N_l(self) -> int:
        return len(self.levels)

    @property
    def L(self) -> int:
        return int(sum(h * w for h, w in self.levels))

    @property
    def n_queries(self) -> int:
        return self.L if self.N_q is None else int(self.N_q)

    @property
    def level_start_index(self) -> Tuple[int, ...]:
        starts, s = [], 0
        for h, w in self.levels:
            starts.append(s)
            s += h * w
        return tuple(starts)

    @property
    def samples(self) -> int:
        """Sample count B*N_q*N_h*N_l*N_p (the throughput unit)."""
        return self.B * self.n_queries * self.N_h * self.N_l * self.N_p

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five Deformable-DETR-shaped workloads, seed = position in this table.
WORKLOADS = {
    "tiny": Workload("tiny", B=1, N_q=16, N_h=2, C_h=8, N_p=2, levels=((8, 8), (4, 4)),
                     loc_recipe="uniform", loc_lo=-0.1, loc_hi=1.1, seed=0),
    "decoder": Workload("decoder", B=2, N_q=300, N_h=8, C_h=32, N_p=4, levels=LEVELS_DETR,
                        loc_recipe="ref_uniform", seed=1),
    "encoder32": Workload("encoder32", B=2, N_q=None, N_h=8, C_h=32, N_p=4, levels=LEVELS_DETR,
                          loc_recipe="pixel_centre", seed=2),
    "encoder16": Workload("encoder16", B=8, N_q=None, N_h=8, C_h=32, N_p=4, levels=LEVELS_DETR,
                          dtype="bf16", value_layout="BNLC", loc_layout="B2QHLP",
                          align_corners=True, padding_mode="border",
                          loc_recipe="uniform", loc_lo=-0.05, loc_hi=1.05, seed=3),
    "hires16": Workload("hires16", B=4, N_q=None, N_h=8, C_h=32, N_p=8, levels=LEVELS_HIRES,
                        dtype="bf16", loc_recipe="pixel_centre", seed=4),
}

WORKLOAD_DESCRIPTIONS = {
    "tiny": "tiny fp32: B=1 Nq=16 Nh=2 Ch=8 Nl=2 Np=2 levels (8,8),(4,4) L=80, BLNC/BQHLP2, "
            "loc~U(-0.1,1.1), zeros, align_corners=False",
    "decoder": "decoder fp32: B=2 Nq=300 Nh=8 Ch=32 Nl=4 Np=4 levels (100,167),(50,84),(25,42),(13,21) "
               "L=22223, ref U(0,1)+N(0,2/W_l), zeros",
    "encoder32": "encoder fp32: B=2 Nq=L=22223 Nh=8 Ch=32 Nl=4 Np=4 levels (100,167),(50,84),(25,42),(13,21), "
                 "pixel-centre ref + N(0,2/W_l), zeros, align_corners=False, BLNC/BQHLP2",
    "encoder16": "encoder bf16 value/grads, fp32 accumulation: B=8 Nq=L=22223 Nh=8 Ch=32 Nl=4 Np=4, "
                 "BNLC/B2QHLP, align_corners=True, border, loc~U(-0.05,1.05)",
    "hires16": "high-res bf16: B=4 Nq=L=21760 Nh=8 Ch=32 Nl=4 Np=8 levels (128,128),(64,64),(32,32),(16,16), "
               "BLNC/BQHLP2, zeros, pixel-centre ref + N(0,2/W_l)",
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64/float32 values to the nearest bfloat16 (ties to even).

    Returns float32 values that are exactly representable in bfloat16.  NaN
    and infinities do not occur in generated inputs.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def store_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round to the storage dtype; the result is float32 holding exact values."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f16":
        return np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float16), dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def _pixel_centre_refs(levels: Sequence[Tuple[int, int]]) -> np.ndarray:
    """(L, 2) reference points (x, y): the centre of every pyramid pixel."""
    refs = []
    for h, w in levels:
        ys, xs = np.meshgrid(np.arange(h, dtype=np.float64), np.arange(w, dtype=np.float64),
                             indexing="ij")
        refs.append(np.stack([(xs.ravel() + 0.5) / w, (ys.ravel() + 0.5) / h], axis=1))
    return np.concatenate(refs, axis=0)


def to_value_layout(v_blnc: np.ndarray, layout: str) -> np.ndarray:
    """(B, L, N_h, C_h) -> the requested value layout (a pure permutation)."""
    if layout == "BLNC":
        return np.ascontiguousarray(v_blnc)
    if layout == "BNLC":
        return np.ascontiguousarray(v_blnc.transpose(0, 2, 1, 3))
    raise ValueError(f"unknown value layout {layout!r}")


def from_value_layout(v: np.ndarray, layout: str) -> np.ndarray:
    """The requested value layout -> (B, L, N_h, C_h)."""
    if layout == "BLNC":
        return v
    if layout == "BNLC":
        return v.transpose(0, 2, 1, 3)
    raise ValueError(f"unknown value layout {layout!r}")


def to_loc_layout(loc_qhlp2: np.ndarray, layout: str) -> np.ndarray:
    """(B, N_q, N_h, N_l, N_p, 2) -> the requested location layout."""
    if layout == "BQHLP2":
        return np.ascontiguousarray(loc_qhlp2)
    if layout == "B2QHLP":
        return np.ascontiguousarray(np.moveaxis(loc_qhlp2, -1, 1))
    raise ValueError(f"unknown sampling_locations layout {layout!r}")


def from_loc_layout(loc: np.ndarray, layout: str) -> np.ndarray:
    """The requested location layout -> (B, N_q, N_h, N_l, N_p, 2)."""
    if layout == "BQHLP2":
        return loc
    if layout == "B2QHLP":
        return np.moveaxis(loc, 1, -1)
    raise ValueError(f"unknown sampling_locations layout {layout!r}")


def generate(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw one workload's inputs.

    Returns a dict of C-contiguous float32 numpy arrays in the workload's
    layouts (``value``, ``sampling_locations``, ``attention_weights``,
    ``grad_output``) plus ``spatial_shapes`` and ``level_start_index`` tuples.
    value and grad_output hold values exactly representable in ``w.dtype``.
    The logical tensors do not depend on the layouts: the same seed gives the
    same numbers, permuted.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    B, Nq, Nh, Ch, Nl, Np, L = w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L

    value = rng.standard_normal((B, L, Nh, Ch))

    widths = np.array([lw for _, lw in w.levels], dtype=np.float64)
    shape6 = (B, Nq, Nh, Nl, Np, 2)
    if w.loc_recipe == "uniform":
        loc = rng.uniform(w.loc_lo, w.loc_hi, size=shape6)
    elif w.loc_recipe in ("ref_uniform", "pixel_centre"):
        if w.loc_recipe == "ref_uniform":
            ref = rng.uniform(0.0, 1.0, size=(B, Nq, 2))
        else:
            if Nq != L:
                raise ValueError("pixel_centre locations need one query per pyramid pixel")
            ref = np.broadcast_to(_pixel_centre_refs(w.levels)[None], (B, Nq, 2))
        sigma = (2.0 / widths).reshape(1, 1, 1, Nl, 1, 1)
        offset = rng.standard_normal(shape6) * sigma
        loc = ref[:, :, None, None, None, :] + offset
    else:
        raise ValueError(f"unknown location recipe {w.loc_recipe!r}")

    logits = rng.standard_normal((B, Nq, Nh, Nl * Np))
    raw_logits = logits.reshape(B, Nq, Nh, Nl, Np).copy()
    if logits.size:
        logits -= logits.max(axis=-1, keepdims=True)
        e = np.exp(logits)
        attn = (e / e.sum(axis=-1, keepdims=True)).reshape(B, Nq, Nh, Nl, Np)
    else:
        attn = np.zeros((B, Nq, Nh, Nl, Np))

    grad_output = rng.standard_normal((B, Nq, Nh * Ch))

    return {
        "value": to_value_layout(store_dtype(value, w.dtype), w.value_layout),
        "sampling_locations": to_loc_layout(store_dtype(loc, w.loc_dtype), w.loc_layout),
        "attention_weights": store_dtype(attn, w.loc_dtype),
        "attention_logits": store_dtype(raw_logits, w.loc_dtype),  # the logits the weights come from
        "grad_output": store_dtype(grad_output, w.dtype),
        "spatial_shapes": tuple(tuple(int(x) for x in hw) for hw in w.levels),
        "level_start_index": w.level_start_index,
    }
