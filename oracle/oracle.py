"""CPU oracle for the 2-bit draft head with exact rerank (numpy front end over dh_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference leg may import this module.  The product library never does, and
this module never touches the CUDA library: the two share no code.

Every function restates one step of the page "radiance_drafthead.py":

* :func:`quantize`     -- ``_quantize_head_now`` (fp32, asymmetric min/max, group 128,
                          quarter-split packing, premultiplied bf16 scale/zero pair)
* :func:`coarse`       -- the coarse value of ``_draft_head_int2`` written as its definition:
                          ``c = sum_g S*p - ZS*xs`` with ``p = sum x (1 + v/4)`` (fp64)
* :func:`block_topk`   -- ``_emit``: the KCAND best of every 64-column block
* :func:`select_topr`  -- ``BI.gather(BM.topk(RERANK))`` in ``_apply_head_int2``
* :func:`rerank`       -- ``_rerank_exact`` (bf16 branch), fp64
* :func:`topk`         -- the top-k / argmax over the reranked entries only
* :func:`exact_head`   -- the stock bf16 head ``x @ W^T`` in fp64, for recall
* :func:`decision_gaps`-- the margins that decide whether an index comparison is strict

bf16 arrays travel as ``uint16`` numpy arrays holding the raw bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dh_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()

GROUP = 128
BLOCK_N = 64


def build(force: bool = False) -> str:
    """Compile dh_oracle.c with gcc (fp-contract off, no fast-math).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.orc_quantize.argtypes = [P, I64, I64, P, P, P, P, P]
        lib.orc_quantize.restype = I
        lib.orc_unpack.argtypes = [P, I64, I64, P]
        lib.orc_unpack.restype = None
        lib.orc_coarse.argtypes = [P, P, P, P, I, I64, I64, P, I]
        lib.orc_coarse.restype = None
        lib.orc_block_topk.argtypes = [P, I, I64, I, P, P]
        lib.orc_block_topk.restype = I64
        lib.orc_select_topr.argtypes = [P, P, I, I64, I, P, P]
        lib.orc_select_topr.restype = I
        lib.orc_rerank.argtypes = [P, P, I, I64, P, I, P]
        lib.orc_rerank.restype = None
        lib.orc_topk.argtypes = [P, P, I, I, I, P, P]
        lib.orc_topk.restype = None
        lib.orc_exact_head.argtypes = [P, P, I, I64, I64, P, I]
        lib.orc_exact_head.restype = None
        lib.orc_decode_e4m3.argtypes = [P, I64, P]
        lib.orc_decode_e4m3.restype = None
        lib.orc_quantize_fp8.argtypes = [P, P, I64, I64, P, P, P]
        lib.orc_quantize_fp8.restype = I
        lib.orc_rerank_fp8.argtypes = [P, P, P, I, I64, P, I, P]
        lib.orc_rerank_fp8.restype = None
        lib.orc_quantize4.argtypes = [P, I64, I64, P, P, P, P, P]
        lib.orc_quantize4.restype = I
        lib.orc_coarse4.argtypes = [P, P, P, P, I, I64, I64, P, I]
        lib.orc_coarse4.restype = None
        lib.orc_quantize_c4.argtypes = [P, I64, I64, P, P, P]
        lib.orc_quantize_c4.restype = I
        lib.orc_coarse_c4.argtypes = [P, P, P, P, I, I64, I64, P, I]
        lib.orc_coarse_c4.restype = None
        lib.orc_quantize_g64.argtypes = [P, I64, I64, P, P, P]
        lib.orc_quantize_g64.restype = I
        lib.orc_coarse_g64.argtypes = [P, P, P, P, I, I64, I64, P, I]
        lib.orc_coarse_g64.restype = None
        lib.orc_coarse_wside.argtypes = [P, P, P, P, I, I64, I64, P]
        lib.orc_coarse_wside.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------------------
# bf16 helpers (for the tests and recipes; the C side has its own)
# --------------------------------------------------------------------------------------

def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Raw bf16 bit patterns -> exact float64 values."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


# --------------------------------------------------------------------------------------
# Steps
# --------------------------------------------------------------------------------------

def quantize(W: np.ndarray, with_params: bool = False):
    """W: uint16 [V, H] bf16 bits -> (packed u8 [V, H/4], S u16 [V, H/128], ZS u16 [V, H/128])
    and, with ``with_params``, the fp32 scale ``sc`` and zero point ``zp`` per group."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    V, H = W.shape
    packed = np.empty((V, H // 4), np.uint8)
    S = np.empty((V, H // GROUP), np.uint16)
    ZS = np.empty((V, H // GROUP), np.uint16)
    sc = np.empty((V, H // GROUP), np.float32) if with_params else None
    zp = np.empty((V, H // GROUP), np.float32) if with_params else None
    rc = _load().orc_quantize(_ptr(W), V, H, _ptr(packed), _ptr(S), _ptr(ZS),
                              _ptr(sc) if with_params else None,
                              _ptr(zp) if with_params else None)
    if rc != 0:
        raise ValueError(f"orc_quantize: status {rc} (H must be a positive multiple of 512)")
    if with_params:
        return packed, S, ZS, sc, zp
    return packed, S, ZS


def quantize4(W: np.ndarray, with_params: bool = False):
    """The 4-bit head: W uint16 [V, H] bf16 bits -> (packed u8 [V, H/2] half split,
    S u16 [V, H/128] = bf16(16 sc), ZS u16 = bf16(16 sc + zp sc)) [+ sc, zp]."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    V, H = W.shape
    packed = np.empty((V, H // 2), np.uint8)
    S = np.empty((V, H // GROUP), np.uint16)
    ZS = np.empty((V, H // GROUP), np.uint16)
    sc = np.empty((V, H // GROUP), np.float32) if with_params else None
    zp = np.empty((V, H // GROUP), np.float32) if with_params else None
    rc = _load().orc_quantize4(_ptr(W), V, H, _ptr(packed), _ptr(S), _ptr(ZS),
                               _ptr(sc) if with_params else None,
                               _ptr(zp) if with_params else None)
    if rc != 0:
        raise ValueError(f"orc_quantize4: status {rc} (H must be a positive multiple of 256)")
    if with_params:
        return packed, S, ZS, sc, zp
    return packed, S, ZS


def quantize_c4(W: np.ndarray):
    """The 2-bit head packed in the contiguous-4 layout: (packed u8 [V, H/4], S, ZS)."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    V, H = W.shape
    packed = np.empty((V, H // 4), np.uint8)
    S = np.empty((V, H // GROUP), np.uint16)
    ZS = np.empty((V, H // GROUP), np.uint16)
    rc = _load().orc_quantize_c4(_ptr(W), V, H, _ptr(packed), _ptr(S), _ptr(ZS))
    if rc != 0:
        raise ValueError(f"orc_quantize_c4: status {rc} (H must be a positive multiple of 512)")
    return packed, S, ZS


def quantize_g64(W: np.ndarray):
    """The 2-bit head with groups of 64: (packed u8 [V, H/4], S u16 [V, H/64], ZS)."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    V, H = W.shape
    packed = np.empty((V, H // 4), np.uint8)
    S = np.empty((V, H // 64), np.uint16)
    ZS = np.empty((V, H // 64), np.uint16)
    rc = _load().orc_quantize_g64(_ptr(W), V, H, _ptr(packed), _ptr(S), _ptr(ZS))
    if rc != 0:
        raise ValueError(f"orc_quantize_g64: status {rc} (H must be a positive multiple of 512)")
    return packed, S, ZS


def unpack(packed: np.ndarray, H: int) -> np.ndarray:
    """Quarter-split packed bytes [V, H/4] -> 2-bit codes [V, H] (u8)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    V = packed.shape[0]
    codes = np.empty((V, H), np.uint8)
    _load().orc_unpack(_ptr(packed), V, H, _ptr(codes))
    return codes


def coarse(x, packed, S, ZS, nthreads: int | None = None) -> np.ndarray:
    """Coarse values c [M, V] in fp64 from the stored int2 head."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    S = np.ascontiguousarray(S, dtype=np.uint16)
    ZS = np.ascontiguousarray(ZS, dtype=np.uint16)
    M, H = x.shape
    V = packed.shape[0]
    c = np.empty((M, V), np.float64)
    _load().orc_coarse(_ptr(x), _ptr(packed), _ptr(S), _ptr(ZS), M, H, V, _ptr(c),
                       nthreads or default_threads())
    return c


def coarse4(x, packed, S, ZS, nthreads: int | None = None) -> np.ndarray:
    """Coarse values c [M, V] in fp64 from the stored 4-bit head (packed [V, H/2])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    S = np.ascontiguousarray(S, dtype=np.uint16)
    ZS = np.ascontiguousarray(ZS, dtype=np.uint16)
    M, H = x.shape
    V = packed.shape[0]
    assert packed.shape[1] * 2 == H
    c = np.empty((M, V), np.float64)
    _load().orc_coarse4(_ptr(x), _ptr(packed), _ptr(S), _ptr(ZS), M, H, V, _ptr(c),
                        nthreads or default_threads())
    return c


def coarse_c4(x, packed, S, ZS, nthreads: int | None = None) -> np.ndarray:
    """Coarse values c [M, V] in fp64 from the contiguous-4 packed 2-bit head."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    S = np.ascontiguousarray(S, dtype=np.uint16)
    ZS = np.ascontiguousarray(ZS, dtype=np.uint16)
    M, H = x.shape
    V = packed.shape[0]
    c = np.empty((M, V), np.float64)
    _load().orc_coarse_c4(_ptr(x), _ptr(packed), _ptr(S), _ptr(ZS), M, H, V, _ptr(c),
                          nthreads or default_threads())
    return c


def coarse_g64(x, packed, S, ZS, nthreads: int | None = None) -> np.ndarray:
    """Coarse values c [M, V] in fp64 from the 2-bit head with 64-groups."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    S = np.ascontiguousarray(S, dtype=np.uint16)
    ZS = np.ascontiguousarray(ZS, dtype=np.uint16)
    M, H = x.shape
    V = packed.shape[0]
    assert S.shape[1] * 64 == H
    c = np.empty((M, V), np.float64)
    _load().orc_coarse_g64(_ptr(x), _ptr(packed), _ptr(S), _ptr(ZS), M, H, V, _ptr(c),
                           nthreads or default_threads())
    return c


def coarse_wside(x, packed, S, ZS, nthreads: int | None = None) -> np.ndarray:
    """Coarse values of the weight-side variant: sum_k x_k bf16(S (1 + v/4) - ZS), fp64."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    S = np.ascontiguousarray(S, dtype=np.uint16)
    ZS = np.ascontiguousarray(ZS, dtype=np.uint16)
    M, H = x.shape
    V = packed.shape[0]
    c = np.empty((M, V), np.float64)
    _load().orc_coarse_wside(_ptr(x), _ptr(packed), _ptr(S), _ptr(ZS), M, H, V, _ptr(c))
    return c


def block_topk(cf: np.ndarray, kcand: int):
    """cf: fp32 coarse [M, V].  Returns (cval f32 [M, nblk*kcand], cidx i32, nvalid per row)."""
    cf = np.ascontiguousarray(cf, dtype=np.float32)
    M, V = cf.shape
    nblk = (V + BLOCK_N - 1) // BLOCK_N
    cval = np.empty((M, nblk * kcand), np.float32)
    cidx = np.empty((M, nblk * kcand), np.int32)
    nvalid = _load().orc_block_topk(_ptr(cf), M, V, kcand, _ptr(cval), _ptr(cidx))
    return cval, cidx, int(nvalid)


def select_topr(cval: np.ndarray, cidx: np.ndarray, R: int):
    """Top-R of the block candidates per row.  Returns (sel_idx i32 [M, R], sel_val f32)."""
    cval = np.ascontiguousarray(cval, dtype=np.float32)
    cidx = np.ascontiguousarray(cidx, dtype=np.int32)
    M, ncand = cval.shape
    sel_idx = np.empty((M, R), np.int32)
    sel_val = np.empty((M, R), np.float32)
    rc = _load().orc_select_topr(_ptr(cval), _ptr(cidx), M, ncand, R, _ptr(sel_idx),
                                 _ptr(sel_val))
    if rc != 0:
        raise ValueError(f"orc_select_topr: status {rc} (fewer than R valid candidates)")
    return sel_idx, sel_val


def rerank(x: np.ndarray, W: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Exact fp64 logits e [M, R] of the candidate rows idx [M, R]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    M, H = x.shape
    R = idx.shape[1]
    e = np.empty((M, R), np.float64)
    _load().orc_rerank(_ptr(x), _ptr(W), M, H, _ptr(idx), R, _ptr(e))
    return e


def topk(e: np.ndarray, idx: np.ndarray, k: int):
    """Top-k of the reranked entries: (out_idx i32 [M, k], out_val f64 [M, k])."""
    e = np.ascontiguousarray(e, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    M, R = e.shape
    out_idx = np.empty((M, k), np.int32)
    out_val = np.empty((M, k), np.float64)
    _load().orc_topk(_ptr(e), _ptr(idx), M, R, k, _ptr(out_idx), _ptr(out_val))
    return out_idx, out_val


def decode_e4m3(b: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) -> float32 values, from the format's definition."""
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.empty(b.shape, np.float32)
    _load().orc_decode_e4m3(_ptr(b), b.size, _ptr(out))
    return out


def quantize_fp8(W8: np.ndarray, wsc: np.ndarray):
    """An fp8 head (e4m3 rows [V, H] uint8, per-row fp32 scale [V]) -> (packed, S, ZS)."""
    W8 = np.ascontiguousarray(W8, dtype=np.uint8)
    wsc = np.ascontiguousarray(wsc, dtype=np.float32)
    V, H = W8.shape
    packed = np.empty((V, H // 4), np.uint8)
    S = np.empty((V, H // GROUP), np.uint16)
    ZS = np.empty((V, H // GROUP), np.uint16)
    rc = _load().orc_quantize_fp8(_ptr(W8), _ptr(wsc), V, H, _ptr(packed), _ptr(S), _ptr(ZS))
    if rc != 0:
        raise ValueError(f"orc_quantize_fp8: status {rc}")
    return packed, S, ZS


def rerank_fp8(x: np.ndarray, W8: np.ndarray, wsc: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Exact fp64 logits [M, R] against fp8 rows: weight = fp32(e4m3 * row scale)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    W8 = np.ascontiguousarray(W8, dtype=np.uint8)
    wsc = np.ascontiguousarray(wsc, dtype=np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    M, H = x.shape
    R = idx.shape[1]
    e = np.empty((M, R), np.float64)
    _load().orc_rerank_fp8(_ptr(x), _ptr(W8), _ptr(wsc), M, H, _ptr(idx), R, _ptr(e))
    return e


def forward_fp8(x, packed, S, ZS, W8, wsc, kcand: int, rerank_n: int, k: int,
                nthreads: int | None = None) -> dict:
    """The draft-head path with the fp8 rerank arm (the coarse part is the same)."""
    c = coarse(x, packed, S, ZS, nthreads)
    cf = c.astype(np.float32)
    cval, cidx, nvalid = block_topk(cf, kcand)
    sel_idx, sel_val = select_topr(cval, cidx, rerank_n)
    e = rerank_fp8(x, W8, wsc, sel_idx)
    out_idx, out_val = topk(e, sel_idx, k)
    return dict(coarse=c, coarse_f32=cf, cand_val=cval, cand_idx=cidx, sel_idx=sel_idx,
                sel_val=sel_val, exact=e, idx=out_idx, logit=out_val)


def forward4(x, packed, S, ZS, W, kcand: int, rerank_n: int, k: int,
             nthreads: int | None = None, coarse_fn=None) -> dict:
    """The draft-head path on the 4-bit head (the rerank is the same bf16 one).  coarse_fn
    replaces the coarse step (forward_c4 passes the contiguous-4 one)."""
    c = (coarse_fn or coarse4)(x, packed, S, ZS, nthreads)
    cf = c.astype(np.float32)
    cval, cidx, nvalid = block_topk(cf, kcand)
    sel_idx, sel_val = select_topr(cval, cidx, rerank_n)
    e = rerank(x, W, sel_idx)
    out_idx, out_val = topk(e, sel_idx, k)
    return dict(coarse=c, coarse_f32=cf, cand_val=cval, cand_idx=cidx, sel_idx=sel_idx,
                sel_val=sel_val, exact=e, idx=out_idx, logit=out_val)


def forward_c4(x, packed, S, ZS, W, kcand: int, rerank_n: int, k: int,
               nthreads: int | None = None) -> dict:
    """The draft-head path on the contiguous-4 packed 2-bit head."""
    return forward4(x, packed, S, ZS, W, kcand, rerank_n, k, nthreads, coarse_fn=coarse_c4)


def forward_g64(x, packed, S, ZS, W, kcand: int, rerank_n: int, k: int,
                nthreads: int | None = None) -> dict:
    """The draft-head path on the 64-group 2-bit head."""
    return forward4(x, packed, S, ZS, W, kcand, rerank_n, k, nthreads, coarse_fn=coarse_g64)


def forward_wside(x, packed, S, ZS, W, kcand: int, rerank_n: int, k: int,
                  nthreads: int | None = None) -> dict:
    """The draft-head path with the weight-side coarse variant."""
    return forward4(x, packed, S, ZS, W, kcand, rerank_n, k, nthreads, coarse_fn=coarse_wside)


def exact_head(x: np.ndarray, W: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """The stock bf16 head in fp64: logits [M, V]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    M, H = x.shape
    V = W.shape[0]
    out = np.empty((M, V), np.float64)
    _load().orc_exact_head(_ptr(x), _ptr(W), M, H, V, _ptr(out), nthreads or default_threads())
    return out


def forward(x, packed, S, ZS, W, kcand: int, rerank_n: int, k: int,
            nthreads: int | None = None) -> dict:
    """The whole draft-head path.  Returns every intermediate the parity tests compare."""
    c = coarse(x, packed, S, ZS, nthreads)
    cf = c.astype(np.float32)
    cval, cidx, nvalid = block_topk(cf, kcand)
    sel_idx, sel_val = select_topr(cval, cidx, rerank_n)
    e = rerank(x, W, sel_idx)
    out_idx, out_val = topk(e, sel_idx, k)
    return dict(coarse=c, coarse_f32=cf, cand_val=cval, cand_idx=cidx, sel_idx=sel_idx,
                sel_val=sel_val, exact=e, idx=out_idx, logit=out_val)


def decision_gaps(res: dict, kcand: int, k: int) -> np.ndarray:
    """Smallest decision margin per row, each scaled to the tolerance it is judged by.

    Three kinds of margin decide the returned indices:
      1. in every block whose (KC+1)-th coarse value reaches the R-th selected value, the
         gap between its KC-th and (KC+1)-th coarse values (a swap there changes the
         reranked set);
      2. the gap between the R-th and (R+1)-th candidate coarse values;
      3. the gaps between consecutive exact values among the top-k and the (k+1)-th.
    Coarse margins are divided by (1 + |value|), exact margins are absolute.  A row whose
    minimum is <= 1e-3 is a tie row.  Returns that minimum per row (inf when none applies).

    Margins 1 and 2 are the two selections the page makes on coarse values (radiance_drafthead.py:
    ``_emit``, the per-block top KCAND by successive max-and-mask, and the top-RERANK gather
    over the block candidates in ``_apply_head_int2``); margin 3 is the final ordering on exact
    values.  Pinned on hand-worked rows, with planted mistakes that must be caught.
    """
    cf = res["coarse_f32"].astype(np.float64)
    M, V = cf.shape
    nblk = (V + BLOCK_N - 1) // BLOCK_N
    cval = res["cand_val"].astype(np.float64)
    cidx = res["cand_idx"]
    e = res["exact"]
    R = res["sel_idx"].shape[1]
    out = np.full(M, np.inf)
    for m in range(M):
        gaps = []
        valid = cidx[m] >= 0
        cv = np.sort(cval[m][valid])[::-1]
        r_th = cv[R - 1]
        # 2. R boundary among the candidates
        if cv.size > R:
            gaps.append((cv[R - 1] - cv[R]) / (1.0 + abs(cv[R - 1])))
        # 1. KC boundary in every block where it can reach the reranked set
        if kcand < BLOCK_N:
            row = np.full(nblk * BLOCK_N, -np.inf)
            row[:V] = cf[m]
            blocks = -np.sort(-row.reshape(nblk, BLOCK_N), axis=1)
            kth, k1 = blocks[:, kcand - 1], blocks[:, kcand]
            reach = np.isfinite(k1) & (k1 >= r_th - 1e-3 * (1.0 + abs(r_th)))
            if reach.any():
                gaps.extend(((kth[reach] - k1[reach]) / (1.0 + np.abs(kth[reach]))).tolist())
        # 3. exact-value gaps at the top-k
        ev = np.sort(e[m])[::-1]
        upto = min(k + 1, ev.size)
        for i in range(upto - 1):
            gaps.append(ev[i] - ev[i + 1])
        if gaps:
            out[m] = float(min(gaps))
    return out
