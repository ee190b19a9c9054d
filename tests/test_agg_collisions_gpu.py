"""The warp-aggregated grad_value scatter when its merge table overflows (GPU).

The backward's warp-aggregated scatter merges a warp batch's corner
contributions (four rows x eight samples) in a per-warp table keyed by the
pixel's element offset, with linear probing from a multiplicative hash and
at most eight probes; a contribution that finds no slot is added directly by
its row's group.  On the workloads' inputs that path is rare.  Here one
64 x 64 level, two heads and eight points per query put every sample at the
exact centre of one of sixteen pixels whose keys share one home slot, so each
batch fills that slot's run of eight, sends the other distinct pixels down
the direct path and still merges the repeated ones (32 samples on 16 pixels:
enough repeats that the warp does not back off to plain atomics).  N_l*N_p =
8 keeps the rows whole (no row split), so the aggregated kernel runs.

The hash below restates the kernel's (key * 0x9E3779B1 mod 2^32, top eight
bits of a 256-slot table); if the kernel's hash changes, this test still
checks the results against the oracle but may exercise fewer overflows.
Rule: "MS Deformable Attention Backward Kernel API Reference", Returns
(grad_value, grad_sampling_locations, grad_attention_weights).
"""
import numpy as np
import pytest

from parity_util import check_workload
from scale_deformable_attention_forward_gb300 import inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SIDE, N_H, C_H, N_P, N_Q = 64, 2, 32, 8, 64


def _colliding_pixels(count=16):
    key = np.arange(SIDE * SIDE, dtype=np.uint64) * (N_H * C_H)  # element offset in a BLNC (b, h) slice
    home = ((key * 0x9E3779B1) & 0xFFFFFFFF) >> 24
    best = np.bincount(home.astype(np.int64), minlength=256).argmax()
    pixels = np.flatnonzero(home == best)
    assert len(pixels) >= count, "not enough pixels share a home slot"
    return pixels[:count]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_overflowing_merge_table_matches_oracle(dtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = gen.Workload("collide", B=1, N_q=N_Q, N_h=N_H, C_h=C_H, N_p=N_P, levels=((SIDE, SIDE),), dtype=dtype,
                     seed=71)
    d = gen.generate(w)
    pix = _colliding_pixels()
    loc = np.empty((1, N_Q, N_H, 1, N_P, 2), dtype=np.float32)  # BQHLP2
    for q in range(N_Q):
        for h in range(N_H):
            for s in range(N_P):
                p = int(pix[(q * N_P + s + 3 * h) % len(pix)])
                # pixel centres, exact in binary32 (the side is a power of two):
                # weight A on the pixel itself, zero on the other three corners
                loc[0, q, h, 0, s] = ((p % SIDE + 0.5) / SIDE, (p // SIDE + 0.5) / SIDE)
    d["sampling_locations"] = loc
    check_workload(w, d=d, flag_sets=((True, True, True), (True, False, False)))
