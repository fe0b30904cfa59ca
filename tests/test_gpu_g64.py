"""GPU parity of the 2-bit head with groups of 64 (the page's group-size ablation):
dh_quantize_g64 bit-exact with the oracle, and the forward on that head judged by the rules in
parity.py against the oracle's 64-group forward (M <= 16, the sizes the ablation runs at)."""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from oracle import oracle as orc

from parity import full_compare, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _quantize_g64(W):
    V, H = W.shape
    packed = torch.empty(V, H // 4, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // 64, dtype=torch.bfloat16, device=DEV)
    ZS = torch.empty_like(S)
    dh.dh_quantize_g64(W, packed, S, ZS)
    return packed, S, ZS


@pytest.mark.parametrize("V, H", [(4096, 1024), (1000, 512), (2003, 1536), (1, 512)])
def test_quantize_g64_bit_exact(V, H):
    wl = synth.custom(1, H, V, hot_rows=min(V, 37), hot_scale=4.0)
    W = synth.make_w(wl, 0, DEV)
    W[0, :64] = 0.25                                     # a constant 64-group
    packed, S, ZS = _quantize_g64(W)
    torch.cuda.synchronize()
    rp, rS, rZS = orc.quantize_g64(host(W))
    assert np.array_equal(host(packed), rp)
    assert np.array_equal(host(S), rS)
    assert np.array_equal(host(ZS), rZS)


@pytest.mark.parametrize("M, H, V, kcand, R, k", [
    (1, 1024, 8192, 8, 32, 1),
    (5, 1024, 8192 + 37, 8, 32, 4),       # ragged tail block
    (16, 5120, 12288, 8, 32, 1),
    (16, 5120, 40000 + 37, 8, 32, 1),     # 313 tiles of 128 rows: every CTA runs two or more
])
def test_forward_g64_matches_the_oracle(M, H, V, kcand, R, k):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = _quantize_g64(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, k, bits="g64")
    print("g64", M, H, V, rep["coarse_worst"], "tie rows", len(rep["ties"]))


def test_forward_g64_rejects_batches_above_16():
    M, H, V = 17, 1024, 4096
    x = torch.zeros(M, H, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(V, H, dtype=torch.bfloat16, device=DEV)
    packed, S, ZS = _quantize_g64(W)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, 8, 32), dtype=torch.uint8, device=DEV)
    idx = torch.empty(M, 1, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, 1, dtype=torch.float32, device=DEV)
    with pytest.raises(dh.DHError) as e:
        dh.dh_forward_g64_debug(x, packed, S, ZS, W, 8, 32, 1, idx, logit, ws)
    assert e.value.code == -8
