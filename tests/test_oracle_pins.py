"""Pins for the CPU oracle: it is checked against what the page and the mathematics fix,
never against itself.  Page: radiance_drafthead.py (module docstring and functions).

* hand-worked quantiser groups and packed bytes (tests/golden/*.json)
* the bit-pattern identity 0x3F80 | ((b << (5-2q)) & 0x60) == bf16(1 + v/4), exhaustively
* collapsed accumulator form == direct dequant-and-dot
* special cases that reduce to textbook routines (grid weights -> exact head; KCAND=64 and
  RERANK=V -> exact top-k of x W^T)
* brute force on tiny inputs for the selections; exact integer arithmetic for the dots
"""
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def f2bf_exact(vals):
    """Float values that are exactly representable in bf16 -> their bit patterns."""
    out = []
    for v in np.asarray(vals, dtype=np.float64).ravel():
        b = struct.unpack("<I", struct.pack("<f", float(v)))[0]
        assert b & 0xFFFF == 0, f"{v} is not a bf16 value"
        out.append(b >> 16)
    return np.array(out, dtype=np.uint16).reshape(np.shape(vals))


def bf2f(bits):
    return orc.bf16_bits_to_f64(bits)


def f32_bits(x):
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def my_unpack(packed, H):
    """Test-side unpack, written from the docstring: byte j carries k = j + p*Q in bits 2p."""
    Q = H // 4
    planes = [(packed >> (2 * p)) & 3 for p in range(4)]
    return np.concatenate(planes, axis=1).astype(np.uint8)  # k = p*Q + j


# ------------------------------------------------------------------------------------------
# quantiser and packing
# ------------------------------------------------------------------------------------------

def test_quantize_golden_groups():
    spec = json.load(open(os.path.join(GOLD, "quantize_groups.json")))
    for case in spec["cases"]:
        group = np.tile(np.array(case["pattern"]), 32)          # 128 values
        W = f2bf_exact(np.tile(group, 4)[None, :])              # H = 512: four equal groups
        packed, S, ZS, sc, zp = orc.quantize(W, with_params=True)
        codes = my_unpack(packed, 512)[0]
        want = np.tile(np.array(case["codes"]), 128)
        assert np.array_equal(codes, want), case["name"]
        for g in range(4):
            assert f32_bits(sc[0, g]) == int(case["sc_bits"], 16), case["name"]
            assert zp[0, g] == case["zp"], case["name"]
            assert S[0, g] == int(case["S"], 16), case["name"]
            assert ZS[0, g] == int(case["ZS"], 16), case["name"]


def test_packing_golden_bytes():
    spec = json.load(open(os.path.join(GOLD, "packing.json")))
    for row in spec["rows"]:
        H = row["H"]
        groups = [np.array([-0.75, 0.75] + [f] * 126) for f in row["group_fill"]]
        W = f2bf_exact(np.concatenate(groups)[None, :])
        packed, S, ZS = orc.quantize(W)
        want = np.zeros(H // 4, np.uint8)
        for start, count, val in row["bytes"]:
            want[start:start + count] = int(val, 16)
        assert np.array_equal(packed[0], want), H
        assert np.all(S == int(row["S"], 16)) and np.all(ZS == int(row["ZS"], 16))


def test_unpack_inverts_quarter_split_packing():
    rng = np.random.default_rng(1)
    for H in (512, 1024, 5120):
        Q = H // 4
        codes = rng.integers(0, 4, size=(7, H), dtype=np.uint8)
        packed = (codes[:, :Q] | (codes[:, Q:2 * Q] << 2) | (codes[:, 2 * Q:3 * Q] << 4)
                  | (codes[:, 3 * Q:] << 6)).astype(np.uint8)
        assert np.array_equal(orc.unpack(packed, H), codes)
    # plane placement: a byte with only plane p set decodes to k = p*Q + j only
    H, Q = 1024, 256
    for p in range(4):
        packed = np.zeros((1, Q), np.uint8)
        packed[0, 5] = 1 << (2 * p)
        codes = orc.unpack(packed, H)[0]
        assert np.flatnonzero(codes).tolist() == [p * Q + 5]


def test_quantize_invariants_and_error_bound():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((48, 1024)) * 0.02).astype(np.float32)
    w[3] *= 4.0
    w[7, :128] = 0.37                     # constant group
    w[9, 128:256] = np.abs(w[9, 128:256]) + 0.01   # all-positive group
    W = (w.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16 bits
    packed, S, ZS, sc, zp = orc.quantize(W, with_params=True)
    wv = bf2f(W)
    codes = my_unpack(packed, 1024).astype(np.float64)
    assert np.all(sc >= np.float32(1e-8))
    assert set(np.unique(zp).tolist()) <= {0.0, 1.0, 2.0, 3.0}
    g = wv.reshape(48, 8, 128)
    lo, hi = g.min(-1), g.max(-1)
    deq = sc[..., None].astype(np.float64) * (codes.reshape(48, 8, 128) - zp[..., None])
    err = np.abs(g - deq)
    straddle = (lo <= 0) & (hi >= 0)
    bound = 0.5 * sc.astype(np.float64) * (1 + 1e-5)
    assert np.all(err[straddle] <= bound[straddle][:, None])
    assert straddle.sum() >= 40
    # the stored pair is the premultiplied scale and zero within bf16 rounding (half an
    # ulp of an 8-bit significand: 2^-8 relative)
    s = bf2f(S)
    zs = bf2f(ZS)
    sc64 = sc.astype(np.float64)
    assert np.all(np.abs(s - 4 * sc64) <= 2.0 ** -8 * 4 * sc64)
    assert np.all(np.abs(zs - (4 + zp) * sc64) <= 2.0 ** -8 * (1 + 1e-6) * (4 + zp) * sc64)


def test_quantize_cross_check_with_torch_fp32():
    """Cross-check of platform fp32 semantics against the page's own library ops (torch
    amin/amax/round/clamp on CPU).  Not counted as a pin: it restates the arithmetic."""
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(3)
    wt = (torch.randn(64, 1024, generator=g) * 0.02).to(torch.bfloat16)
    W = wt.view(torch.int16).numpy().view(np.uint16)
    packed, S, ZS = orc.quantize(W)
    wg = wt.float().reshape(64, 8, 128)
    lo, hi = wg.amin(dim=2), wg.amax(dim=2)
    sc = ((hi - lo) / 3).clamp(min=1e-8)
    zp = torch.round(-lo / sc).clamp(0, 3)
    q = torch.round(wg / sc[:, :, None] + zp[:, :, None]).clamp(0, 3).to(torch.uint8)
    q = q.reshape(64, 1024)
    Q = 256
    tp = (q[:, :Q] | (q[:, Q:2 * Q] << 2) | (q[:, 2 * Q:3 * Q] << 4) | (q[:, 3 * Q:] << 6))
    assert np.array_equal(tp.numpy(), packed)
    assert np.array_equal((4.0 * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16), S)
    assert np.array_equal((4.0 * sc + zp * sc).to(torch.bfloat16).view(torch.int16).numpy()
                          .view(np.uint16), ZS)


def test_quantize_rejects_partial_quarter_groups():
    with pytest.raises(ValueError):
        orc.quantize(np.zeros((2, 256), np.uint16))


# ------------------------------------------------------------------------------------------
# bit-pattern dequant (module docstring, 'Bit-pattern dequant, hoisted' bullet)
# ------------------------------------------------------------------------------------------

def test_bit_pattern_identity_exhaustive():
    for b in range(256):
        for q in range(4):
            if q < 3:
                bits = 0x3F80 | ((b << (5 - 2 * q)) & 0x60)
            else:
                bits = 0x3F80 | ((b >> 1) & 0x60)
            v = (b >> (2 * q)) & 3
            assert bf2f(np.array([bits], np.uint16))[0] == 1.0 + v / 4.0


def test_bit_pattern_on_32bit_words_pairs_bytes_0_2_and_1_3():
    """The word form of the identity: one shift and one mask turn bytes (0, 2) or (1, 3) of a
    packed 32-bit word into a bf16 pair, both halves equal to 1 + v/4 of that byte."""
    rng = np.random.default_rng(4)
    words = rng.integers(0, 2 ** 32, size=4096, dtype=np.uint64)
    for wd in words.tolist() + [0, 0xFFFFFFFF, 0x1B1B1B1B]:
        bs = [(wd >> (8 * i)) & 0xFF for i in range(4)]
        for q in range(4):
            s = 5 - 2 * q
            even = ((wd << s) if s >= 0 else (wd >> -s)) & 0x00600060 | 0x3F803F80
            odd = (wd >> (3 + 2 * q)) & 0x00600060 | 0x3F803F80
            for word, (blo, bhi) in ((even, (bs[0], bs[2])), (odd, (bs[1], bs[3]))):
                lo = bf2f(np.array([word & 0xFFFF], np.uint16))[0]
                hi = bf2f(np.array([(word >> 16) & 0xFFFF], np.uint16))[0]
                assert lo == 1 + ((blo >> (2 * q)) & 3) / 4
                assert hi == 1 + ((bhi >> (2 * q)) & 3) / 4


# ------------------------------------------------------------------------------------------
# coarse value
# ------------------------------------------------------------------------------------------

def _grid_weights(rng, V, H):
    """Rows on the exact 2-bit grid {-1, -0.5, 0, 0.5} * 2^e (each group holds -1 and 0.5, so
    lo, hi fix sc = 0.5 * 2^e and zp = 2 and every value is reproduced exactly)."""
    vals = rng.choice(np.array([-1.0, -0.5, 0.0, 0.5]), size=(V, H))
    vals.reshape(V, H // 128, 128)[:, :, 0] = -1.0
    vals.reshape(V, H // 128, 128)[:, :, 1] = 0.5
    e = rng.integers(-9, -3, size=(V, 1)).astype(np.float64)
    return vals * 2.0 ** e


def test_coarse_on_grid_weights_is_the_exact_head():
    rng = np.random.default_rng(5)
    V, H, M = 96, 1024, 3
    W = f2bf_exact(_grid_weights(rng, V, H))
    x = f2bf_exact(np.round(rng.standard_normal((M, H)) * 64) / 64)
    packed, S, ZS = orc.quantize(W)
    c = orc.coarse(x, packed, S, ZS)
    ref = bf2f(x) @ bf2f(W).T
    np.testing.assert_allclose(c, ref, rtol=1e-12, atol=1e-12)


def test_coarse_collapsed_form_equals_direct_dequant():
    """c = sum_g S p - ZS xs must equal sum_k x_k (S_g (1 + v_k/4) - ZS_g), the per-element
    dequant-and-dot, computed here from a test-side unpack and a plain matmul."""
    rng = np.random.default_rng(6)
    V, H, M = 200, 1536, 5
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    packed, S, ZS = orc.quantize(W)
    v = my_unpack(packed, H).astype(np.float64)
    s = np.repeat(bf2f(S), 128, axis=1)
    zs = np.repeat(bf2f(ZS), 128, axis=1)
    What = s * (1.0 + v / 4.0) - zs
    ref = bf2f(x) @ What.T
    c = orc.coarse(x, packed, S, ZS)
    np.testing.assert_allclose(c, ref, rtol=1e-11, atol=1e-11)
    # and the quantised head tracks the bf16 head (2-bit noise, not a wrong term)
    exact = bf2f(x) @ bf2f(W).T
    corr = np.corrcoef(c.ravel(), exact.ravel())[0, 1]
    assert corr > 0.85


# ------------------------------------------------------------------------------------------
# selections (brute force on tiny inputs)
# ------------------------------------------------------------------------------------------

def _order(vals, idx):
    """Value descending, equal values -> lower index."""
    return np.lexsort((idx, -vals))


@pytest.mark.parametrize("kcand", [1, 3, 8, 64])
def test_block_topk_brute_force(kcand):
    rng = np.random.default_rng(7 + kcand)
    M, V = 3, 200                                   # blocks of 64, 64, 64, 8 (ragged tail)
    cf = np.round(rng.standard_normal((M, V)) * 4).astype(np.float32)  # many exact ties
    cval, cidx, _ = orc.block_topk(cf, kcand)
    nblk = 4
    for m in range(M):
        for b in range(nblk):
            cols = np.arange(64 * b, min(V, 64 * b + 64))
            o = _order(cf[m, cols], cols)[:kcand]
            got_i = cidx[m, b * kcand:(b + 1) * kcand]
            got_v = cval[m, b * kcand:(b + 1) * kcand]
            n = len(o)
            assert np.array_equal(got_i[:n], cols[o])
            assert np.array_equal(got_v[:n], cf[m, cols[o]])
            assert np.all(got_i[n:] == -1) and np.all(np.isneginf(got_v[n:]))


def test_select_topr_brute_force():
    rng = np.random.default_rng(8)
    M, V, kc = 4, 300, 8
    cf = np.round(rng.standard_normal((M, V)) * 3).astype(np.float32)
    cval, cidx, _ = orc.block_topk(cf, kc)
    for R in (1, 5, 17, 37):
        sel, selv = orc.select_topr(cval, cidx, R)
        for m in range(M):
            ok = cidx[m] >= 0
            o = _order(cval[m][ok], cidx[m][ok])[:R]
            assert np.array_equal(sel[m], cidx[m][ok][o])
            assert np.array_equal(selv[m], cval[m][ok][o])
    # KCAND = 64 makes the candidates every column: top-R of the full row
    cval, cidx, n = orc.block_topk(cf, 64)
    assert n == V
    sel, _ = orc.select_topr(cval, cidx, 50)
    for m in range(M):
        assert np.array_equal(sel[m], _order(cf[m], np.arange(V))[:50])


def test_forward_with_full_candidate_pool_is_exact_topk():
    """KCAND=64 and RERANK=V rerank every column, so the result is the exact head's top-k."""
    rng = np.random.default_rng(9)
    M, V, H, k = 4, 130, 512, 5
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    packed, S, ZS = orc.quantize(W)
    res = orc.forward(x, packed, S, ZS, W, 64, V, k)
    ex = bf2f(x) @ bf2f(W).T
    for m in range(M):
        o = _order(ex[m].astype(np.float32), np.arange(V))[:k]
        assert np.array_equal(res["idx"][m], o)
        np.testing.assert_allclose(res["logit"][m], ex[m, o], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------------------------------
# exact dots (integer arithmetic)
# ------------------------------------------------------------------------------------------

def test_rerank_and_exact_head_match_exact_rational_sums():
    rng = np.random.default_rng(10)
    M, V, H = 2, 40, 512
    xv = rng.integers(-128, 128, size=(M, H)) / 64.0          # bf16-exact (8-bit mantissas)
    wv = rng.integers(-128, 128, size=(V, H)) / 4096.0
    x, W = f2bf_exact(xv), f2bf_exact(wv)
    exact = np.array([[float(sum(Fraction(int(a)) * int(b) for a, b in
                                 zip(np.round(xv[m] * 64), np.round(wv[n] * 4096))) / (64 * 4096))
                       for n in range(V)] for m in range(M)])
    idx = np.array([[3, 17, 0, 39], [5, 5, 22, 1]], np.int32)
    e = orc.rerank(x, W, idx)
    for m in range(M):
        for j in range(4):
            assert e[m, j] == exact[m, idx[m, j]]
    assert np.array_equal(orc.exact_head(x, W), exact)


# ------------------------------------------------------------------------------------------
# decision gaps
# ------------------------------------------------------------------------------------------

def test_decision_gap_flags_a_planted_tie():
    rng = np.random.default_rng(11)
    M, V, H = 2, 256, 512
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    W[77] = W[12]                       # identical rows: identical coarse and exact values
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    packed, S, ZS = orc.quantize(W)
    ex = bf2f(x) @ bf2f(W).T
    res = orc.forward(x, packed, S, ZS, W, 8, 32, 1)
    gaps = orc.decision_gaps(res, 8, 1)
    assert gaps.shape == (M,)
    # make row 0's winner one of the twins: its exact gap to the (k+1)-th is 0
    x2 = x.copy()
    x2[0] = (((bf2f(W[12]) * 50).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    res2 = orc.forward(x2, packed, S, ZS, W, 8, 32, 1)
    assert set(res2["idx"][0].tolist()) <= {12, 77}
    assert res2["idx"][0, 0] == 12               # equal values -> lower index
    assert orc.decision_gaps(res2, 8, 1)[0] == 0.0


def _res_from_coarse(rows, exact, kcand, R):
    """A forward() result built from hand-set coarse rows (fp32 [M, V]) through the oracle's
    brute-force-pinned block_topk / select_topr, with the given exact values of the selected
    entries (one list of R per row)."""
    cf = np.asarray(rows, dtype=np.float32)
    cval, cidx, _ = orc.block_topk(cf, kcand)
    sel, selv = orc.select_topr(cval, cidx, R)
    return dict(coarse_f32=cf, cand_val=cval, cand_idx=cidx, sel_idx=sel, sel_val=selv,
                exact=np.asarray(exact, dtype=np.float64))


def _row(V, entries, fill=-8.0):
    r = np.full(V, fill, np.float32)
    for c, v in entries.items():
        r[c] = v
    return r


def _check_margin_pins(gaps_fn):
    """The decision margins on hand-built coarse rows, each worked out by hand.

    Page: radiance_drafthead.py, _emit (each block of 64 emits its top KC by successive
    max-and-mask) and the top-RERANK gather over the block candidates in _apply_head_int2.
    A coarse value that moves by its rounding error can change the returned indices only at
    those two boundaries (a block's KC-th / (KC+1)-th entry, when the latter could have made
    the reranked set; the R-th / (R+1)-th candidate) or in the final exact top-k.
    """
    d = 2.0 ** -10
    # (a) KC boundary inside a block whose (KC+1)-th value reaches the R-th selected value:
    #     block 0 = {10, 9, 9 - d}, block 1 = {3, 2}; KC = 2, R = 2 -> selected {10, 9},
    #     R-th = 9, block 0's 3rd value 9 - d reaches it.  margin 1 = d / (1 + 9).
    a = _row(128, {3: 10.0, 5: 9.0, 9: 9.0 - d, 70: 3.0, 71: 2.0})
    # (b) the same near-tie (5 | 5 - d) in a block that cannot reach the R-th value 9:
    #     block 0 = {10, 5, 5 - d}, block 1 = {9, 8} -> selected {10, 9}; only margin 2 applies,
    #     (9 - 8) / (1 + 9) = 0.1.
    b = _row(128, {3: 10.0, 5: 5.0, 9: 5.0 - d, 70: 9.0, 71: 8.0})
    # (c) R boundary: block 0 = {10, 9}, block 1 = {9 - d, 2} -> candidates 10, 9, 9 - d, 2;
    #     margin 2 = d / (1 + 9).  No block's 3rd value reaches 9.
    c = _row(128, {3: 10.0, 5: 9.0, 70: 9.0 - d, 71: 2.0})
    res = _res_from_coarse([a, b, c], [[5.0, 1.0]] * 3, 2, 2)
    assert res["sel_idx"].tolist() == [[3, 5], [3, 70], [3, 5]]
    g = gaps_fn(res, 2, 1)
    assert g[0] == d / 10.0 and g[0] <= 1e-3          # flagged
    assert g[1] == 0.1                                 # not flagged: the near-tie cannot reach
    assert g[2] == d / 10.0 and g[2] <= 1e-3          # flagged

    # (d) clear rows, KC = 1, R = 2, three blocks.
    #     row 0: block 0 = {10, 9.75}, block 1 = {9.5}, block 2 = {3}; selected {10, 9.5}; block
    #     0's 2nd value 9.75 is above the R-th (9.5), so margin 1 = (10 - 9.75) / (1 + 10);
    #     margin 2 = (9.5 - 3) / (1 + 9.5); exact gap 5 - 1 = 4.
    #     row 1: block 0 = {4}, block 1 = {-5, -5.5}, block 2 = {-2}; selected {4, -2}, R-th -2;
    #     block 1's 2nd value -5.5 does not reach it; margin 2 = (-2 - -5) / (1 + 2) = 1;
    #     exact gap 0.5 (absolute, unscaled) is the minimum.
    r0 = _row(192, {3: 10.0, 4: 9.75, 70: 9.5, 130: 3.0})
    r1 = _row(192, {10: 4.0, 80: -5.0, 81: -5.5, 150: -2.0})
    res = _res_from_coarse([r0, r1], [[5.0, 1.0], [7.0, 6.5]], 1, 2)
    assert res["sel_idx"].tolist() == [[3, 70], [10, 150]]
    g = gaps_fn(res, 1, 1)
    assert g[0] == 0.25 / 11.0
    assert g[1] == 0.5
    # the same rows judged at k = 2 (both reranked entries returned): no (k+1)-th exact value
    # exists, so the exact margin is the gap between the two
    g2 = gaps_fn(res, 1, 2)
    assert g2[0] == 0.25 / 11.0 and g2[1] == 0.5

    # (e) fewer than R + 1 candidates: no R boundary; a ragged last block (V = 129) whose only
    #     column cannot have a (KC+1)-th value.  KC = 1, R = 3: blocks {10, 9.9}, {8}, {7}.
    #     Block 0's 2nd value 9.9 reaches the R-th (7): margin 1 = 0.1 / 11 in fp32 values.
    e = _row(129, {0: 10.0, 1: 9.9, 64: 8.0, 128: 7.0})
    res = _res_from_coarse([e], [[3.0, 2.0, 1.0]], 1, 3)
    assert res["sel_idx"].tolist() == [[0, 64, 128]]
    g = gaps_fn(res, 1, 1)
    assert g[0] == (10.0 - float(np.float32(9.9))) / 11.0


def test_decision_gap_margins_on_hand_built_rows():
    _check_margin_pins(orc.decision_gaps)


_GAP_MUTANTS = {
    "drop the reach condition": (
        "reach = np.isfinite(k1) & (k1 >= r_th - 1e-3 * (1.0 + abs(r_th)))",
        "reach = np.isfinite(k1)"),
    "drop the (1 + |v|) scaling of margin 1": (
        "/ (1.0 + np.abs(kth[reach]))", "/ 1.0"),
    "drop the (1 + |v|) scaling of margin 2": (
        "/ (1.0 + abs(cv[R - 1]))", "/ 1.0"),
    "R boundary one place early": (
        "(cv[R - 1] - cv[R])", "(cv[R - 2] - cv[R - 1])"),
    "KC boundary one place late": (
        "blocks[:, kcand - 1], blocks[:, kcand]", "blocks[:, kcand], blocks[:, kcand + 1]"),
    "reach measured against the top candidate": (
        "r_th = cv[R - 1]", "r_th = cv[0]"),
}


@pytest.mark.parametrize("name", sorted(_GAP_MUTANTS))
def test_decision_gap_pins_catch_planted_mistakes(name):
    """Each mutant is the oracle's decision_gaps with one plausible mistake planted in its
    source (on the CPU); the hand-worked margins must reject every one."""
    import inspect
    import textwrap
    old, new = _GAP_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(orc.decision_gaps))
    assert src.count(old) == 1, f"mutation site for {name!r} not found"
    ns = dict(vars(orc))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    with pytest.raises(AssertionError):
        _check_margin_pins(ns["decision_gaps"])


# ------------------------------------------------------------------------------------------
# fp8 head (e4m3 rows, per-row fp32 scale): decode, quantise, rerank
# ------------------------------------------------------------------------------------------

def _finite_e4m3_codes():
    codes = np.arange(256, dtype=np.uint8)
    return codes[(codes & 0x7F) != 0x7F]           # 0x7F / 0xFF are NaN in e4m3fn


def test_e4m3_decode_matches_torch_float8_for_every_finite_code():
    torch = pytest.importorskip("torch")
    codes = _finite_e4m3_codes()
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    got = orc.decode_e4m3(codes)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))   # -0.0 included
    # spot values from the format: largest finite, smallest subnormal, one
    assert orc.decode_e4m3(np.array([0x7E, 0x01, 0x38], np.uint8)).tolist() == [448.0, 2.0**-9, 1.0]


def _fp8_head(rng, V, H, pow2_scales):
    codes = rng.choice(_finite_e4m3_codes(), size=(V, H)).astype(np.uint8)
    if pow2_scales:
        wsc = np.exp2(rng.integers(-12, -4, size=V)).astype(np.float32)
    else:
        wsc = (rng.uniform(0.5, 2.0, size=V) * 1e-3).astype(np.float32)
    return codes, wsc


def _as_bf16_bits(f32):
    bits = np.asarray(f32, np.float32).view(np.uint32)
    assert not (bits & 0xFFFF).any()                  # exactly representable in bf16
    return (bits >> 16).astype(np.uint16)


def test_fp8_quantise_and_rerank_with_power_of_two_scales_reduce_to_the_bf16_head():
    """e4m3 has 4 significant bits, so e4m3 * 2^k is an exact bf16 value: the fp8 head is
    then the bf16 head with those values, and both oracle paths must agree bit for bit."""
    rng = np.random.default_rng(21)
    V, H, M = 96, 1024, 3
    codes, wsc = _fp8_head(rng, V, H, pow2_scales=True)
    Wb = _as_bf16_bits(orc.decode_e4m3(codes) * wsc[:, None])
    p8, S8, Z8 = orc.quantize_fp8(codes, wsc)
    pb, Sb, Zb = orc.quantize(Wb)
    assert np.array_equal(p8, pb) and np.array_equal(S8, Sb) and np.array_equal(Z8, Zb)
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    idx = rng.integers(0, V, size=(M, 7)).astype(np.int32)
    assert np.array_equal(orc.rerank_fp8(x, codes, wsc, idx), orc.rerank(x, Wb, idx))


def test_fp8_rerank_rounds_each_weight_to_fp32_before_the_sum():
    """General row scales: weight k is the fp32 product e4m3(b) * scale, as the page's
    decoder computes it; the sum is checked against torch's float8 decode and numpy."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(22)
    V, H, M = 40, 512, 2
    codes, wsc = _fp8_head(rng, V, H, pow2_scales=False)
    dec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    w32 = (dec * wsc[:, None]).astype(np.float32)                 # one fp32 rounding
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    idx = rng.integers(0, V, size=(M, 5)).astype(np.int32)
    ref = np.einsum("mk,mjk->mj", bf2f(x).astype(np.float64), w32[idx].astype(np.float64))
    np.testing.assert_allclose(orc.rerank_fp8(x, codes, wsc, idx), ref, rtol=1e-12, atol=1e-14)
    # the fp32 rounding of the product matters: the fp64 product gives other sums
    raw = np.einsum("mk,mjk->mj", bf2f(x).astype(np.float64),
                    dec[idx].astype(np.float64) * wsc[idx][..., None].astype(np.float64))
    assert not np.array_equal(orc.rerank_fp8(x, codes, wsc, idx), raw)


# ------------------------------------------------------------------------------------------
# the 4-bit head (BITS = 4: half split, bias 16)
# ------------------------------------------------------------------------------------------

def my_unpack4(packed, H):
    """Test-side unpack of the half split: low nibble -> k = j, high nibble -> k = H/2 + j."""
    return np.concatenate([packed & 15, packed >> 4], axis=1).astype(np.uint8)


def test_quantize4_golden_groups():
    spec = json.load(open(os.path.join(GOLD, "quantize4_groups.json")))
    for case in spec["cases"]:
        group = np.tile(np.array(case["pattern"]), 32)
        W = f2bf_exact(np.tile(group, 4)[None, :])              # H = 512: four equal groups
        packed, S, ZS, sc, zp = orc.quantize4(W, with_params=True)
        codes = my_unpack4(packed, 512)[0]
        want = np.tile(np.array(case["codes"]), 128)
        assert np.array_equal(codes, want), case["name"]
        for g in range(4):
            assert f32_bits(sc[0, g]) == int(case["sc_bits"], 16), case["name"]
            assert zp[0, g] == case["zp"], case["name"]
            assert S[0, g] == int(case["S"], 16), case["name"]
            assert ZS[0, g] == int(case["ZS"], 16), case["name"]


def test_packing4_golden_bytes():
    spec = json.load(open(os.path.join(GOLD, "packing4.json")))
    for row in spec["rows"]:
        H = row["H"]
        groups = [np.array([-0.875, 1.0] + [f] * 126) for f in row["group_fill"]]
        W = f2bf_exact(np.concatenate(groups)[None, :])
        packed, S, ZS = orc.quantize4(W)
        want = np.zeros(H // 2, np.uint8)
        for start, count, val in row["bytes"]:
            want[start:start + count] = int(val, 16)
        assert np.array_equal(packed[0], want), H
        assert np.all(S == int(row["S"], 16)) and np.all(ZS == int(row["ZS"], 16))


def test_quantize4_invariants_and_error_bound():
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((40, 1536)) * 0.02).astype(np.float32)
    w[5] *= 4.0
    w[7, :128] = 0.37
    W = (w.view(np.uint32) >> 16).astype(np.uint16)
    packed, S, ZS, sc, zp = orc.quantize4(W, with_params=True)
    codes = my_unpack4(packed, 1536).astype(np.float64)
    assert codes.max() <= 15 and set(np.unique(zp).tolist()) <= set(range(16))
    g = bf2f(W).reshape(40, 12, 128)
    lo, hi = g.min(-1), g.max(-1)
    deq = sc[..., None].astype(np.float64) * (codes.reshape(40, 12, 128) - zp[..., None])
    straddle = (lo <= 0) & (hi >= 0)
    assert straddle.sum() >= 400
    bound = 0.5 * sc.astype(np.float64) * (1 + 1e-5)
    assert np.all(np.abs(g - deq)[straddle] <= bound[straddle][:, None])
    sc64 = sc.astype(np.float64)
    assert np.all(np.abs(bf2f(S) - 16 * sc64) <= 2.0 ** -8 * 16 * sc64)
    assert np.all(np.abs(bf2f(ZS) - (16 + zp) * sc64) <= 2.0 ** -8 * (1 + 1e-6) * (16 + zp) * sc64)
    # the same groups at 2 bits: a step of range/3 against range/15
    sc2 = orc.quantize(W, with_params=True)[3]
    assert np.allclose(sc2[sc2 > 1e-8], 5 * sc[sc2 > 1e-8], rtol=1e-6)


def test_quantize4_rejects_partial_half_groups():
    with pytest.raises(ValueError):
        orc.quantize4(np.zeros((2, 128), np.uint16))


def _grid_weights4(rng, V, H):
    """Rows on an exact 4-bit grid: per group codes in 0..15 with 0 and 15 present, a zero
    point zp and a power-of-two step, w = (code - zp) * 2^e; lo, hi then fix sc = 2^e and
    zp exactly and every value is reproduced."""
    codes = rng.integers(0, 16, size=(V, H // 128, 128))
    codes[:, :, 0] = 0
    codes[:, :, 1] = 15
    zp = rng.integers(0, 16, size=(V, H // 128, 1))
    e = rng.integers(-12, -6, size=(V, 1, 1)).astype(np.float64)
    return ((codes - zp) * 2.0 ** e).reshape(V, H)


def test_coarse4_on_grid_weights_is_the_exact_head():
    rng = np.random.default_rng(13)
    V, H, M = 80, 1024, 3
    W = f2bf_exact(_grid_weights4(rng, V, H))
    x = f2bf_exact(np.round(rng.standard_normal((M, H)) * 64) / 64)
    packed, S, ZS = orc.quantize4(W)
    c = orc.coarse4(x, packed, S, ZS)
    np.testing.assert_allclose(c, bf2f(x) @ bf2f(W).T, rtol=1e-12, atol=1e-12)


def test_coarse4_collapsed_form_equals_direct_dequant():
    """c = sum_g S p - ZS xs must equal sum_k x_k (S_g (1 + v_k/16) - ZS_g) from a test-side
    unpack of the half split and a plain matmul."""
    rng = np.random.default_rng(14)
    V, H, M = 150, 1536, 4
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    packed, S, ZS = orc.quantize4(W)
    v = my_unpack4(packed, H).astype(np.float64)
    s = np.repeat(bf2f(S), 128, axis=1)
    zs = np.repeat(bf2f(ZS), 128, axis=1)
    ref = bf2f(x) @ (s * (1.0 + v / 16.0) - zs).T
    c = orc.coarse4(x, packed, S, ZS)
    np.testing.assert_allclose(c, ref, rtol=1e-11, atol=1e-11)
    exact = bf2f(x) @ bf2f(W).T
    assert np.corrcoef(c.ravel(), exact.ravel())[0, 1] > 0.97


def test_forward4_with_full_candidate_pool_is_exact_topk():
    rng = np.random.default_rng(15)
    M, V, H, k = 3, 130, 512, 4
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    packed, S, ZS = orc.quantize4(W)
    res = orc.forward4(x, packed, S, ZS, W, 64, V, k)
    ex = bf2f(x) @ bf2f(W).T
    for m in range(M):
        o = _order(ex[m].astype(np.float32), np.arange(V))[:k]
        assert np.array_equal(res["idx"][m], o)


# ------------------------------------------------------------------------------------------
# the contiguous-4 layout (the page's packing ablation)
# ------------------------------------------------------------------------------------------

def test_packing_c4_golden_bytes():
    spec = json.load(open(os.path.join(GOLD, "packing_c4.json")))
    for row in spec["rows"]:
        H = row["H"]
        groups = [np.array([-0.75, 0.75] + [f] * 126) for f in row["group_fill"]]
        W = f2bf_exact(np.concatenate(groups)[None, :])
        packed, S, ZS = orc.quantize_c4(W)
        want = np.zeros(H // 4, np.uint8)
        for start, count, val in row["bytes"]:
            want[start:start + count] = int(val, 16)
        assert np.array_equal(packed[0], want), H
        assert np.all(S == int(row["S"], 16)) and np.all(ZS == int(row["ZS"], 16))


def test_c4_layout_holds_the_quarter_split_codes_and_coarse_values():
    """Only the byte layout differs: unpacking either layout (test-side) gives the same codes,
    S and ZS agree, and the coarse values of the two packings are identical."""
    rng = np.random.default_rng(16)
    V, H, M = 120, 1536, 3
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    pq, Sq, Zq = orc.quantize(W)
    pc, Sc, Zc = orc.quantize_c4(W)
    codes_c4 = np.stack([(pc >> (2 * f)) & 3 for f in range(4)], axis=2).reshape(V, H)
    assert np.array_equal(codes_c4, my_unpack(pq, H))
    assert np.array_equal(Sq, Sc) and np.array_equal(Zq, Zc)
    assert np.array_equal(orc.coarse_c4(x, pc, Sc, Zc), orc.coarse(x, pq, Sq, Zq))


# ------------------------------------------------------------------------------------------
# groups of 64 (the page's group-size ablation)
# ------------------------------------------------------------------------------------------

def test_quantize_g64_golden_groups():
    """The hand-worked 128-groups of quantize_groups.json hold a 4-value pattern, so the same
    pattern over 64 values has the same statistics, codes, S and ZS."""
    spec = json.load(open(os.path.join(GOLD, "quantize_groups.json")))
    for case in spec["cases"]:
        group = np.tile(np.array(case["pattern"]), 16)          # 64 values
        W = f2bf_exact(np.tile(group, 8)[None, :])              # H = 512: eight equal groups
        packed, S, ZS = orc.quantize_g64(W)
        assert np.array_equal(my_unpack(packed, 512)[0], np.tile(np.array(case["codes"]), 128))
        assert np.all(S == int(case["S"], 16)) and np.all(ZS == int(case["ZS"], 16))


def test_quantize_g64_equals_128_groups_of_doubled_values():
    """Group g of 64 values quantises like a 128-group holding each of them twice (same min,
    max and codes): the g64 quantiser against the pinned 128-group one."""
    rng = np.random.default_rng(17)
    V, H = 30, 1024
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    p64, S64, Z64 = orc.quantize_g64(W)
    W2 = np.repeat(W, 2, axis=1)                                # [V, 2H]: 128-group g = 64-group g
    p2, S2, Z2 = orc.quantize(W2)
    assert np.array_equal(S64, S2) and np.array_equal(Z64, Z2)
    assert np.array_equal(np.repeat(my_unpack(p64, H), 2, axis=1), my_unpack(p2, 2 * H))


def test_coarse_g64_collapsed_form_equals_direct_dequant():
    rng = np.random.default_rng(18)
    V, H, M = 150, 1024, 4
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    packed, S, ZS = orc.quantize_g64(W)
    v = my_unpack(packed, H).astype(np.float64)
    s = np.repeat(bf2f(S), 64, axis=1)
    zs = np.repeat(bf2f(ZS), 64, axis=1)
    ref = bf2f(x) @ (s * (1.0 + v / 4.0) - zs).T
    np.testing.assert_allclose(orc.coarse_g64(x, packed, S, ZS), ref, rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------------------------------
# weight-side dequant (the page's scale-placement ablation)
# ------------------------------------------------------------------------------------------

def test_coarse_wside_on_grid_weights_equals_the_activation_side_value():
    """With power-of-two steps every dequantised weight sc (v - zp) is a bf16 value, so the
    weight-side sum and the group form are the same number up to fp64 summation order."""
    rng = np.random.default_rng(19)
    V, H, M = 64, 1024, 3
    W = f2bf_exact(_grid_weights(rng, V, H))
    x = f2bf_exact(np.round(rng.standard_normal((M, H)) * 64) / 64)
    packed, S, ZS = orc.quantize(W)
    np.testing.assert_allclose(orc.coarse_wside(x, packed, S, ZS), orc.coarse(x, packed, S, ZS),
                               rtol=1e-12, atol=1e-12)


def test_coarse_wside_is_a_dot_with_bf16_rounded_weights():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(20)
    V, H, M = 90, 1024, 4
    W = (((rng.standard_normal((V, H)) * 0.02).astype(np.float32)).view(np.uint32) >> 16
         ).astype(np.uint16)
    x = ((rng.standard_normal((M, H)).astype(np.float32)).view(np.uint32) >> 16).astype(np.uint16)
    packed, S, ZS = orc.quantize(W)
    v = my_unpack(packed, H).astype(np.float64)
    s = np.repeat(bf2f(S), 128, axis=1)
    zs = np.repeat(bf2f(ZS), 128, axis=1)
    wq = torch.from_numpy(s * (1.0 + v / 4.0) - zs).to(torch.bfloat16).double().numpy()
    np.testing.assert_allclose(orc.coarse_wside(x, packed, S, ZS), bf2f(x) @ wq.T,
                               rtol=1e-11, atol=1e-11)
    # and it departs from the group form only by the bf16 rounding of the weights
    assert np.abs(orc.coarse_wside(x, packed, S, ZS) - orc.coarse(x, packed, S, ZS)).max() < 0.05
