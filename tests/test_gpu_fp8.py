"""GPU parity of the fp8 head (e4m3 rows with one fp32 scale per row): dh_quantize_fp8 must be
bit-exact with the oracle's fp8 quantiser, and dh_forward_fp8w is judged by the rules in
parity.py against the oracle's fp8 forward (exact values from the fp32 products
e4m3 * row scale).  A head whose row scales are powers of two is exactly a bf16 head, so
there the fp8 entry points must return bit for bit what the bf16 ones return.
"""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from oracle import oracle as orc

from parity import check_result, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _alloc(V, H):
    packed = torch.empty(V, H // 4, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // 128, dtype=torch.bfloat16, device=DEV)
    return packed, S, torch.empty_like(S)


def _quantize_fp8(W8, rs):
    packed, S, ZS = _alloc(*W8.shape)
    dh.dh_quantize_fp8(W8, rs, packed, S, ZS)
    return packed, S, ZS


def _forward_fp8w(x, packed, S, ZS, W8, rs, kcand, R, k):
    M, H = x.shape
    V = W8.shape[0]
    ws = torch.randint(0, 255, (dh.dh_workspace_bytes(M, H, V, kcand, R),), dtype=torch.uint8,
                       device=DEV)
    idx = torch.full((M, k), -7, dtype=torch.int32, device=DEV)
    logit = torch.full((M, k), float("nan"), dtype=torch.float32, device=DEV)
    dh.dh_forward_fp8w(x, packed, S, ZS, W8, rs, kcand, R, k, idx, logit, ws)
    torch.cuda.synchronize()
    assert dh.dh_device_status(reset=True) == 0
    return idx, logit


@pytest.mark.parametrize("V, H", [(4096, 1024), (1000, 512), (2003, 1536), (1, 512)])
def test_quantize_fp8_bit_exact(V, H):
    wl = synth.custom(1, H, V, hot_rows=min(V, 37), hot_scale=4.0)
    W8, rs = synth.make_w_fp8(wl, 0, DEV)
    # edge rows: all-zero codes, a zero scale, subnormal and negative-zero codes, extreme scales
    W8[0, :] = 0
    if V > 4:
        rs[1] = 0.0
        W8[2, :128] = torch.arange(128, device=DEV, dtype=torch.int64).remainder(8).to(torch.uint8)
        W8[2, 128:256] = 0x80
        rs[3] = 1e-30
        rs[4] = 3.0e30
    packed, S, ZS = _quantize_fp8(W8, rs)
    torch.cuda.synchronize()
    rp, rS, rZS = orc.quantize_fp8(W8.cpu().numpy(), rs.cpu().numpy())
    assert np.array_equal(host(packed), rp)
    assert np.array_equal(host(S), rS)
    assert np.array_equal(host(ZS), rZS)


@pytest.mark.parametrize("M, H, V, kcand, R, k", [
    (1, 1024, 8192, 8, 32, 1),
    (5, 1024, 8192 + 37, 8, 32, 4),     # ragged tail block
    (16, 2048, 16384, 8, 32, 1),
    (33, 1536, 6144, 4, 24, 5),         # two batch chunks
    (64, 1024, 4096, 8, 64, 16),        # the half-span tcgen05 configuration, RERANK 64
])
def test_forward_fp8w_matches_the_oracle(M, H, V, kcand, R, k):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x = synth.make_x(wl, 0, DEV)
    W8, rs = synth.make_w_fp8(wl, 0, DEV)
    packed, S, ZS = _quantize_fp8(W8, rs)
    idx, logit = _forward_fp8w(x, packed, S, ZS, W8, rs, kcand, R, k)
    xb, W8h, rsh = host(x), W8.cpu().numpy(), rs.cpu().numpy()
    ref = orc.forward_fp8(xb, host(packed), host(S), host(ZS), W8h, rsh, kcand, R, k)
    gpu = {"idx": idx.cpu().numpy(), "logit": logit.cpu().numpy()}

    def rerank_fn(xr, ix):
        return orc.rerank_fp8(xr, W8h, rsh, ix)

    ties = check_result(gpu, ref, kcand, k, xb, None, rerank_fn=rerank_fn)
    print("fp8 forward", M, H, V, "tie rows", len(ties), "differing", sum(t[4] for t in ties))


@pytest.mark.parametrize("M, H, V, k", [(4, 1024, 8192, 4), (16, 5120, 12288, 1)])
def test_power_of_two_row_scales_give_the_bf16_head_bit_for_bit(M, H, V, k):
    """e4m3 values times 2^j are exact in bf16: the fp8 head then IS a bf16 head, and both
    entry-point pairs must agree on every packed byte, every index and every logit bit."""
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x = synth.make_x(wl, 0, DEV)
    W8, rs = synth.make_w_fp8(wl, 0, DEV)
    rs = torch.exp2(torch.round(torch.log2(rs)))          # nearest power of two per row
    Wbf = (W8.view(torch.float8_e4m3fn).float() * rs[:, None]).to(torch.bfloat16)
    assert torch.equal(Wbf.float(), W8.view(torch.float8_e4m3fn).float() * rs[:, None])
    p8, S8, Z8 = _quantize_fp8(W8, rs)
    pb, Sb, Zb = _alloc(V, H)
    dh.dh_quantize(Wbf, pb, Sb, Zb)
    torch.cuda.synchronize()
    assert torch.equal(p8, pb) and torch.equal(S8, Sb) and torch.equal(Z8, Zb)
    i8, l8 = _forward_fp8w(x, p8, S8, Z8, W8, rs, 8, 32, k)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, 8, 32), dtype=torch.uint8, device=DEV)
    ib = torch.empty_like(i8)
    lb = torch.empty_like(l8)
    dh.dh_forward(x, pb, Sb, Zb, Wbf, 8, 32, k, ib, lb, ws)
    torch.cuda.synchronize()
    assert torch.equal(i8, ib) and torch.equal(l8, lb)


def test_draft_head_class_takes_an_fp8_weight():
    M, H, V = 3, 1024, 4096
    wl = synth.custom(M, H, V)
    x = synth.make_x(wl, 0, DEV)
    W8, rs = synth.make_w_fp8(wl, 0, DEV)
    head = dh.DraftHead(W8.view(torch.float8_e4m3fn), kcand=8, rerank=32, row_scale=rs)
    idx, logit = head.forward(x, topk=2)
    i2, l2 = _forward_fp8w(x, head.packed, head.scales, head.zeros, W8, rs, 8, 32, 2)
    torch.cuda.synchronize()
    assert torch.equal(idx, i2) and torch.equal(logit, l2)
