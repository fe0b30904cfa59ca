"""GPU parity of the contiguous-4 layout (the page's packing ablation): dh_quantize_c4
bit-exact with the oracle, and the forward on that packing judged by the rules in parity.py
against the oracle's contiguous-4 forward.  Its coarse values must also agree with the
quarter-split forward of the same head within the coarse tolerance (same codes, S and ZS)."""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from oracle import oracle as orc

from parity import check_coarse, full_compare, gpu_forward, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _quantize(W, fn):
    V, H = W.shape
    packed = torch.empty(V, H // 4, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // 128, dtype=torch.bfloat16, device=DEV)
    ZS = torch.empty_like(S)
    fn(W, packed, S, ZS)
    return packed, S, ZS


@pytest.mark.parametrize("V, H", [(4096, 1024), (1000, 512), (2003, 1536), (1, 512)])
def test_quantize_c4_bit_exact(V, H):
    wl = synth.custom(1, H, V, hot_rows=min(V, 37), hot_scale=4.0)
    W = synth.make_w(wl, 0, DEV)
    W[0, :128] = 0.25
    packed, S, ZS = _quantize(W, dh.dh_quantize_c4)
    torch.cuda.synchronize()
    rp, rS, rZS = orc.quantize_c4(host(W))
    assert np.array_equal(host(packed), rp)
    assert np.array_equal(host(S), rS)
    assert np.array_equal(host(ZS), rZS)


@pytest.mark.parametrize("M, H, V, kcand, R, k", [
    (1, 1024, 8192, 8, 32, 1),
    (16, 5120, 12288 + 37, 8, 32, 4),     # ragged tail block
    (33, 1536, 6144, 4, 24, 5),           # two batch chunks (32 + 16 rows)
    (16, 5120, 40000 + 37, 8, 32, 1),     # 313 tiles of 128 rows: every CTA runs two or more
])
def test_forward_c4_matches_the_oracle_and_the_quarter_split(M, H, V, kcand, R, k):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = _quantize(W, dh.dh_quantize_c4)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, k, bits="c4")
    pq, Sq, Zq = _quantize(W, dh.dh_quantize)
    assert torch.equal(S, Sq) and torch.equal(ZS, Zq)
    quarter = gpu_forward(x, pq, Sq, Zq, W, kcand, R, k)
    check_coarse(gpu["coarse"], quarter["coarse"].astype(np.float64))
    print("c4", M, H, V, rep["coarse_worst"], "tie rows", len(rep["ties"]))
