"""The boundary sweeps of test_gpu_quantize_boundaries.py really reach the rounding boundaries:
checked on the CPU with the oracle's own scales and zero points."""
import numpy as np

from oracle import oracle as orc

from test_gpu_quantize_boundaries import RANGES, _head


def test_sweeps_hold_exact_ties_and_near_ties():
    Wb = _head(RANGES, 128)
    _, _, _, sc, zp = orc.quantize(Wb, with_params=True)
    w = (Wb.astype(np.uint32) << 16).view(np.float32).reshape(Wb.shape[0], -1, 128)
    t = w.astype(np.float64) / sc[..., None].astype(np.float64) + zp[..., None]
    dist = np.abs(np.abs(t - np.rint(t)) - 0.5)        # distance to the nearest half-integer
    inside = (t > 0) & (t < 3)
    assert np.count_nonzero(inside & (dist == 0)) >= 6          # exact ties
    assert np.count_nonzero(inside & (dist > 0) & (dist < 2.0 ** -6)) >= 6  # one ulp away


def test_sweeps_cover_every_bf16_value_of_each_range():
    Wb = _head(RANGES, 128)
    present = set(np.unique(Wb).tolist())
    for lo, hi in RANGES:
        vals = np.arange(1 << 16, dtype=np.uint32)
        f = (vals << 16).view(np.float32)
        want = vals[np.isfinite(f) & (f >= np.float32(lo)) & (f <= np.float32(hi))]
        assert set(want.tolist()) <= present
