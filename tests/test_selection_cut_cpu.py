"""The selection the forward runs on the GPU for RERANK <= 32, modelled on the host and checked
against the oracle's plain global top-R (no GPU).

The fused kernel splits a row's blocks into eight slices; each slice keeps the 32 best block
maxima, gathers those blocks' candidates and keeps the 32 best of them; the eight lists are
merged and the first R kept.  Exactness rests on two facts: a block list is in rank order (its
first entry is its best), so a candidate among the row's 32 best has a block among its slice's
32 best maxima; and fewer than 32 candidates of that slice's gathered set beat it.  The model
below follows those steps literally; the inputs have many exact ties, so the order rule
(value descending, lower vocabulary index first) is exercised.
"""
import numpy as np
import pytest

from oracle import oracle as orc

SLICES = 8
KEEP = 32


def _rank(vals, ids):
    """Order of (value desc, id asc) over valid entries (id >= 0)."""
    ok = ids >= 0
    o = np.lexsort((ids[ok], -vals[ok].astype(np.float64)))
    return vals[ok][o], ids[ok][o]


def model_select(cval, cidx, kcand, R):
    nblk = len(cval) // kcand
    per = -(-nblk // SLICES)
    lists_v, lists_i = [], []
    for p in range(SLICES):
        b0, b1 = p * per, min(nblk, p * per + per)
        if b0 >= b1:
            continue
        blocks = np.arange(b0, b1)
        mv, mi = cval[blocks * kcand], cidx[blocks * kcand]        # block maxima
        keep = mi >= 0
        order = np.lexsort((mi[keep], -mv[keep].astype(np.float64)))[:KEEP]
        best_blocks = blocks[keep][order]
        e = (best_blocks[:, None] * kcand + np.arange(kcand)[None, :]).ravel()
        v, i = _rank(cval[e], cidx[e])
        lists_v.append(v[:KEEP])
        lists_i.append(i[:KEEP])
    v, i = _rank(np.concatenate(lists_v), np.concatenate(lists_i))
    return i[:R], v[:R]


@pytest.mark.parametrize("V, kcand, R, levels, seed", [
    (8192, 8, 32, 7, 0),          # heavy ties: seven distinct values
    (8192 + 37, 8, 32, 1000, 1),  # ragged tail block
    (248320 // 4, 8, 32, 50, 2),  # a quarter of the full head, ties
    (4096, 64, 32, 20, 3),        # whole blocks as candidates
    (640, 1, 5, 3, 4),            # ten blocks, one candidate each
    (100000, 2, 1, 10, 5),        # RERANK 1
])
def test_cut_selection_equals_the_global_top_r(V, kcand, R, levels, seed):
    orc.build()
    rng = np.random.default_rng(seed)
    M = 3
    cf = (rng.integers(0, levels, size=(M, V)) / levels).astype(np.float32)
    cf[1] = rng.standard_normal(V).astype(np.float32)             # one row without ties
    cval, cidx, _ = orc.block_topk(cf, kcand)
    ref_idx, ref_val = orc.select_topr(cval, cidx, R)
    for m in range(M):
        ids, vals = model_select(cval[m], cidx[m], kcand, R)
        assert np.array_equal(ids, ref_idx[m]), m
        assert np.array_equal(vals, ref_val[m]), m
