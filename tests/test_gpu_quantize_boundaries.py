"""GPU quantisers bit-exact with the oracle on weights at and next to the rounding boundaries.

The quantisers compute each code from a product with the group's reciprocal and fall back to
the defining division only where that product lands within a small margin of a half-integer
(dh_quantize.cu).  Random weights almost never land there, so these groups are built to: each
group holds its chosen minimum and maximum plus every bf16 value between them (spread over as
many groups as needed, in a seeded order).  With a power-of-two scale sc = (hi - lo) / L the
half-integer points (j + 1/2) sc are themselves bf16 values, so the exact ties (rounded to even
by the definition) and their neighbours one ulp away are all present; the other ranges give
scales that are not powers of two.  The fp8 quantiser gets the same treatment with every e4m3
value in the range and a power-of-two and an arbitrary row scale.
"""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from oracle import oracle as orc

from parity import host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _bf16_bits(v: float) -> int:
    """Round-to-nearest-even of an fp32 value to bf16 bits (the value is chosen representable)."""
    b = int(np.array([v], np.float32).view(np.uint32)[0])
    return (b + 0x7FFF + ((b >> 16) & 1)) >> 16


def _all_bf16_between(lo_bits: int, hi_bits: int) -> np.ndarray:
    every = np.arange(1 << 16, dtype=np.uint32)
    vals = (every << 16).view(np.float32)
    lo = float((np.array([lo_bits], np.uint32) << 16).view(np.float32)[0])
    hi = float((np.array([hi_bits], np.uint32) << 16).view(np.float32)[0])
    keep = np.isfinite(vals) & (vals >= lo) & (vals <= hi)
    return every[keep].astype(np.uint16)


def _groups(lo_bits, hi_bits, payload, G, rng):
    """Groups of G values: lo, hi and G - 2 payload values each (the payload cycled to fill the
    last group), every group in a seeded order."""
    per = G - 2
    n = -(-len(payload) // per)
    pay = np.resize(payload, n * per).reshape(n, per)
    out = np.empty((n, G), np.uint16)
    out[:, 0] = lo_bits
    out[:, 1] = hi_bits
    out[:, 2:] = pay
    for g in range(n):
        out[g] = out[g, rng.permutation(G)]
    return out


def _head(ranges, G, H=512, seed=0):
    """A [V, H] bf16 head (raw bits) whose groups sweep every bf16 value of each range."""
    rng = np.random.default_rng(seed)
    groups = []
    for lo, hi in ranges:
        lb, hb = _bf16_bits(lo), _bf16_bits(hi)
        groups.append(_groups(lb, hb, _all_bf16_between(lb, hb), G, rng))
    flat = np.concatenate(groups).reshape(-1)
    per_row = H
    V = -(-flat.size // per_row)
    flat = np.resize(flat, V * per_row)          # the last row repeats whole groups
    return flat.reshape(V, per_row)


def _to_device(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16).copy()).to(DEV).view(torch.bfloat16)


# (lo, hi) per sweep: power-of-two scales for L = 3 and for L = 15 (exact ties present), a range
# whose scale for L = 3 is 5 2^-8 (ties present too), and an arbitrary range
RANGES = [(0.0, 3 * 2.0 ** -6), (-1.5 * 2.0 ** -5, 1.5 * 2.0 ** -5), (0.0, 15 * 2.0 ** -8),
          (-0.69921875, 1.296875)]


def _alloc(V, H, cols_per_byte, G):
    packed = torch.empty(V, H // cols_per_byte, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // G, dtype=torch.bfloat16, device=DEV)
    return packed, S, torch.empty_like(S)


@pytest.mark.parametrize("kind", ["quarter", "half4", "c4", "g64"])
def test_quantizers_at_rounding_boundaries(kind):
    G = 64 if kind == "g64" else 128
    Wb = _head(RANGES, G)
    V, H = Wb.shape
    W = _to_device(Wb)
    fn, ref, cpb = {"quarter": (dh.dh_quantize, orc.quantize, 4),
                    "half4": (dh.dh_quantize4, orc.quantize4, 2),
                    "c4": (dh.dh_quantize_c4, orc.quantize_c4, 4),
                    "g64": (dh.dh_quantize_g64, orc.quantize_g64, 4)}[kind]
    packed, S, ZS = _alloc(V, H, cpb, G)
    fn(W, packed, S, ZS)
    torch.cuda.synchronize()
    rp, rS, rZS = ref(Wb)
    assert np.array_equal(host(packed), rp)
    assert np.array_equal(host(S), rS)
    assert np.array_equal(host(ZS), rZS)


def test_quantize_fp8_at_rounding_boundaries():
    """e4m3 rows: groups of lo = 0, hi = 0.375 (scale 2^-3 for L = 3: the ties 1/16, 3/16, 5/16
    are e4m3 values) and of lo = -0.375, hi = 0.375, filled with every e4m3 value between, at
    row scales 1 (ties kept), 2^-7 and 0.1 (products off the grid)."""
    codes = np.arange(256, dtype=np.uint32)
    mag = codes & 0x7F
    # decode e4m3 by its definition: subnormal m 2^-9, normal (1 + m/8) 2^(e - 7)
    e = (mag >> 3).astype(np.int64)
    m = (mag & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8) * np.exp2(e - 7.0))
    val = np.where(codes & 0x80, -val, val)
    finite = mag != 0x7F
    rng = np.random.default_rng(1)
    groups = []
    for lo, hi in [(0.0, 0.375), (-0.375, 0.375)]:
        lo_c = int(np.flatnonzero(finite & (val == lo))[0])
        hi_c = int(np.flatnonzero(finite & (val == hi))[0])
        inside = codes[finite & (val >= lo) & (val <= hi)].astype(np.uint16)
        groups.append(_groups(lo_c, hi_c, inside, 128, rng))
    g = np.concatenate(groups)                    # [ng, 128] codes
    H = 512
    rows = []
    for _ in range(3):                            # one copy of every group per row scale
        flat = np.resize(g.reshape(-1), -(-g.size // H) * H)
        rows.append(flat.reshape(-1, H))
    W8 = np.concatenate(rows).astype(np.uint8)
    per = rows[0].shape[0]
    rs = np.concatenate([np.full(per, 1.0), np.full(per, 2.0 ** -7), np.full(per, 0.1)]
                        ).astype(np.float32)
    V = W8.shape[0]
    packed, S, ZS = _alloc(V, H, 4, 128)
    dh.dh_quantize_fp8(torch.from_numpy(W8).to(DEV), torch.from_numpy(rs).to(DEV), packed, S, ZS)
    torch.cuda.synchronize()
    rp, rS, rZS = orc.quantize_fp8(W8, rs)
    assert np.array_equal(host(packed), rp)
    assert np.array_equal(host(S), rS)
    assert np.array_equal(host(ZS), rZS)

