"""Helpers for the GPU-vs-oracle parity tests (test infrastructure; never imported by the
product).  The comparison rules are the ones the draft head is judged by:

* coarse values within 1e-3 * (1 + |ref|) of the fp64 oracle;
* reranked (exact) logits within 1e-5 * max(|ref|, 1);
* indices bit-exact wherever the oracle's decision gap exceeds 1e-3; rows at or below it are
  tie rows, listed, and there the returned entries must still be valid (exact logits right,
  order right, drawn from the reranked set).
"""
from __future__ import annotations

import numpy as np
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from oracle import oracle as orc

COARSE_RTOL = 1e-3
EXACT_RTOL = 1e-5
GAP = 1e-3


def gpu_quantize(W: torch.Tensor):
    V, H = W.shape
    packed = torch.empty(V, H // 4, dtype=torch.uint8, device=W.device)
    S = torch.empty(V, H // 128, dtype=torch.bfloat16, device=W.device)
    ZS = torch.empty(V, H // 128, dtype=torch.bfloat16, device=W.device)
    dh.dh_quantize(W, packed, S, ZS)
    return packed, S, ZS


def gpu_forward(x, packed, S, ZS, W, kcand, rerank, topk, debug=True, path=None, bits=2):
    """Run the CUDA path (dh_forward_debug, or dh_forward4_debug for the 4-bit head) on device
    tensors; return numpy outputs."""
    fwd_dbg = {4: dh.dh_forward4_debug, "c4": dh.dh_forward_c4_debug,
               "g64": dh.dh_forward_g64_debug,
               "wside": dh.dh_forward_wside_debug}.get(bits, dh.dh_forward_debug)
    fwd = dh.dh_forward4 if bits == 4 else dh.dh_forward
    assert debug or bits not in ("c4", "g64", "wside")
    M, H = x.shape
    V = W.shape[0]
    dev = x.device
    nblk = (V + 63) // 64
    ws = torch.randint(0, 255, (dh.dh_workspace_bytes(M, H, V, kcand, rerank),),
                       dtype=torch.uint8, device=dev)  # garbage: nothing may rely on it
    idx = torch.full((M, topk), -7, dtype=torch.int32, device=dev)
    logit = torch.full((M, topk), float("nan"), dtype=torch.float32, device=dev)
    out = {}
    prev = None
    if path is not None:
        prev = dh.dh_set_coarse_path(path)
    try:
        if debug:
            coarse = torch.full((M, V), float("nan"), dtype=torch.float32, device=dev)
            cval = torch.full((M, nblk * kcand), float("nan"), dtype=torch.float32, device=dev)
            cidx = torch.full((M, nblk * kcand), -7, dtype=torch.int32, device=dev)
            sel = torch.full((M, rerank), -7, dtype=torch.int32, device=dev)
            sex = torch.full((M, rerank), float("nan"), dtype=torch.float32, device=dev)
            fwd_dbg(x, packed, S, ZS, W, kcand, rerank, topk, idx, logit, ws, coarse=coarse,
                    cand_val=cval, cand_idx=cidx, sel_idx=sel, sel_exact=sex)
            torch.cuda.synchronize()
            out.update(coarse=coarse.cpu().numpy(), cand_val=cval.cpu().numpy(),
                       cand_idx=cidx.cpu().numpy(), sel_idx=sel.cpu().numpy(),
                       sel_exact=sex.cpu().numpy())
        else:
            fwd(x, packed, S, ZS, W, kcand, rerank, topk, idx, logit, ws)
            torch.cuda.synchronize()
    finally:
        if prev is not None:
            dh.dh_set_coarse_path(prev)
    assert dh.dh_device_status(reset=True) == 0, "a device-side wait timed out"
    out.update(idx=idx.cpu().numpy(), logit=logit.cpu().numpy())
    return out


def host(t: torch.Tensor):
    """bf16 / u8 device tensor -> host numpy array of its raw bits."""
    if t.dtype == torch.bfloat16:
        return synth.bits(t)
    return t.cpu().numpy()


def check_coarse(gpu_c, ref_c):
    err = np.abs(gpu_c.astype(np.float64) - ref_c)
    tol = COARSE_RTOL * (1.0 + np.abs(ref_c))
    bad = err > tol
    if bad.any():
        r, c = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{bad.sum()} coarse values off (rows {sorted(set(np.nonzero(bad)[0].tolist()))[:10]}); "
                             f"worst ratio {(err / tol).max():.3g} at row {r} column {c}: "
                             f"GPU {gpu_c[r, c]!r} oracle {ref_c[r, c]!r}")
    return float((err / tol).max())


def check_block_candidates(gpu, ref, kcand, V):
    """Candidate sets per (row, block) equal, except at near-ties on the KCAND boundary."""
    M = ref["coarse"].shape[0]
    nblk = (V + 63) // 64
    cf = ref["coarse"]
    tie_blocks = {}
    for m in range(M):
        gi = gpu["cand_idx"][m].reshape(nblk, kcand)
        ri = ref["cand_idx"][m].reshape(nblk, kcand)
        for b in np.flatnonzero((gi != ri).any(axis=1)):
            gs, rs = set(gi[b].tolist()), set(ri[b].tolist())
            if gs == rs:
                # same set in another order: only equal-within-tolerance values may swap
                continue
            cols = np.arange(64 * b, min(V, 64 * b + 64))
            vals = np.sort(cf[m, cols])[::-1]
            kth = vals[kcand - 1]
            diff = (gs ^ rs) - {-1}
            assert -1 not in (gs ^ rs), f"row {m} block {b}: slot counts differ"
            for n in diff:
                assert abs(cf[m, n] - kth) <= 2 * COARSE_RTOL * (1 + abs(kth)), (
                    f"row {m} block {b}: candidate {n} differs beyond a near-tie")
            tie_blocks[(m, int(b))] = float(kth)
    return tie_blocks


def check_selection(gpu, ref, R, tie_blocks):
    """Reranked sets equal, except for members near the R-th coarse value or near the KCAND
    boundary of a block whose candidate list was already vetted as a near-tie."""
    M = gpu["sel_idx"].shape[0]
    cf = ref["coarse"]
    tie_rows = 0
    for m in range(M):
        gs, rs = set(gpu["sel_idx"][m].tolist()), set(ref["sel_idx"][m].tolist())
        assert -1 not in gs and len(gs) == R, f"row {m}: GPU selected {len(gs)} distinct"
        if gs == rs:
            continue
        rth = np.sort(cf[m, list(rs)])[0]
        for n in gs ^ rs:
            near_r = abs(cf[m, n] - rth) <= 2 * COARSE_RTOL * (1 + abs(rth))
            kth = tie_blocks.get((m, n // 64))
            near_k = kth is not None and abs(cf[m, n] - kth) <= 2 * COARSE_RTOL * (1 + abs(kth))
            assert near_r or near_k, f"row {m}: selected {n} differs beyond a near-tie"
        tie_rows += 1
    return tie_rows


def check_exact_values(gpu, x_bits, W_bits):
    """The GPU's exact logits of ITS selected rows against the oracle's fp64 rerank."""
    e = orc.rerank(x_bits, W_bits, gpu["sel_idx"])
    err = np.abs(gpu["sel_exact"].astype(np.float64) - e)
    tol = EXACT_RTOL * np.maximum(np.abs(e), 1.0)
    assert (err <= tol).all(), f"exact logits off: worst ratio {(err / tol).max():.3g}"
    return float((err / tol).max())


def check_result(gpu, ref, kcand, topk, x_bits, W_bits, rerank_fn=None):
    """Final indices: bit-exact where the decision gap is clear; where it is not (a tie row),
    the returned list must still be the top-k of the GPU's own reranked set under the
    oracle's exact values, within the exact-logit tolerance.  Returns the tie rows as
    (row, gap, oracle indices, GPU indices, differs).  rerank_fn(x_rows, idx) gives the
    oracle's exact values (default: the bf16 head W_bits)."""
    if rerank_fn is None:
        def rerank_fn(xr, ix):
            return orc.rerank(xr, W_bits, ix)
    gaps = orc.decision_gaps(ref, kcand, topk)
    ties = []
    M = gpu["idx"].shape[0]
    for m in range(M):
        gi, gl = gpu["idx"][m], gpu["logit"][m]
        assert (gi >= 0).all() and len(set(gi.tolist())) == topk, f"row {m}: bad result {gi}"
        e = rerank_fn(x_bits[m:m + 1], gi[None, :].astype(np.int32))[0]
        tol = EXACT_RTOL * np.maximum(np.abs(e), 1.0)
        assert (np.abs(gl - e) <= tol).all(), f"row {m}: returned logits off"
        order_ok = all((gl[i] > gl[i + 1]) or (gl[i] == gl[i + 1] and gi[i] < gi[i + 1])
                       for i in range(topk - 1))
        assert order_ok, f"row {m}: result not ordered"
        if gaps[m] > GAP:
            assert np.array_equal(gi, ref["idx"][m]), (
                f"row {m}: indices {gi} != oracle {ref['idx'][m]} with decision gap "
                f"{gaps[m]:.3g}")
            rtol = EXACT_RTOL * np.maximum(np.abs(ref["logit"][m]), 1.0)
            assert (np.abs(gl - ref["logit"][m]) <= rtol).all()
            continue
        differs = not np.array_equal(gi, ref["idx"][m])
        if differs and "sel_idx" in gpu:
            sel = gpu["sel_idx"][m]
            assert set(gi.tolist()) <= set(sel.tolist()), f"row {m}: result outside reranked set"
            es = rerank_fn(x_bits[m:m + 1], sel[None, :].astype(np.int32))[0]
            rest = es[~np.isin(sel, gi)]
            floor = e.min()
            slack = 2 * EXACT_RTOL * max(abs(floor), 1.0)
            assert rest.size == 0 or rest.max() <= floor + slack, (
                f"row {m}: a reranked entry above the returned top-k beyond tolerance")
            for i in range(topk - 1):
                assert e[i] + 2 * EXACT_RTOL * max(abs(e[i]), 1.0) >= e[i + 1], (
                    f"row {m}: order of the returned list contradicts the exact values")
        ties.append((m, float(gaps[m]), ref["idx"][m].tolist(), gi.tolist(), differs))
    return ties


_ORACLE_FWD = {4: orc.forward4, "c4": orc.forward_c4, "g64": orc.forward_g64,
               "wside": orc.forward_wside}


def _apply_checks(gpu, ref, xb, Wb, kcand, rerank, topk, V):
    rep = {}
    rep["coarse_worst"] = check_coarse(gpu["coarse"], ref["coarse"])
    tb = check_block_candidates(gpu, ref, kcand, V)
    rep["tie_blocks"] = len(tb)
    rep["tie_sel_rows"] = check_selection(gpu, ref, rerank, tb)
    rep["exact_worst"] = check_exact_values(gpu, xb, Wb)
    rep["ties"] = check_result(gpu, ref, kcand, topk, xb, Wb)
    return rep


def full_compare(x, W, packed, S, ZS, kcand, rerank, topk, path=None, bits=2):
    """Run GPU and oracle on the same tensors and apply every check.  Returns a report."""
    gpu = gpu_forward(x, packed, S, ZS, W, kcand, rerank, topk, path=path, bits=bits)
    xb, Wb = host(x), host(W)
    pb, Sb, ZSb = host(packed), host(S), host(ZS)
    ref = _ORACLE_FWD.get(bits, orc.forward)(xb, pb, Sb, ZSb, Wb, kcand, rerank, topk)
    rep = _apply_checks(gpu, ref, xb, Wb, kcand, rerank, topk, W.shape[0])
    return rep, gpu, ref


def rows_compare(gpu, rows, x, W, packed, S, ZS, kcand, rerank, topk, bits=2):
    """Every check of full_compare on a subset of the batch rows: the oracle runs the whole
    path (all V coarse values, both selections, the rerank) for x[rows] only, and the GPU's
    outputs for those rows -- taken from a launch over the whole batch -- are judged against
    it.  For workloads too large for the oracle to run on every row in seconds."""
    rows = np.asarray(rows)
    sub = {k: v[rows] for k, v in gpu.items()}
    xb, Wb = host(x)[rows], host(W)
    pb, Sb, ZSb = host(packed), host(S), host(ZS)
    ref = _ORACLE_FWD.get(bits, orc.forward)(xb, pb, Sb, ZSb, Wb, kcand, rerank, topk)
    rep = _apply_checks(sub, ref, xb, Wb, kcand, rerank, topk, W.shape[0])
    return rep, ref
