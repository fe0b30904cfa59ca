"""GB300 2-bit draft head with exact rerank: Python binding of the C ABI in include/dh.h.

This module only marshals arguments: every step of the path runs in the CUDA library
``_build/libdh.so`` (build it with :func:`build`).  There is no fallback: if the library is
missing or a call fails, an exception is raised.

Functions mirror the C entry points one to one and take torch tensors (device memory owned by
the caller); ``stream`` defaults to torch's current CUDA stream.  :class:`DraftHead` bundles the
packed weight, its scale/zero pair, the bf16 weight and a workspace for repeated calls.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB as _LIB_PATH
from .build import build

__all__ = [
    "build", "DHError", "dh_quantize", "dh_workspace_bytes", "dh_forward", "dh_forward_debug",
    "dh_forward_timed", "dh_set_coarse_path", "dh_coarse_path_for", "dh_device_status",
    "dh_forward_launch_count", "dh_forward_noalloc", "NOALLOC_WORKSPACE_BYTES",
    "dh_last_error", "dh_version", "DraftHead", "dh_shard_candidates",
    "dh_shard_rerank_workspace_bytes", "dh_shard_rerank", "dh_rerank", "dh_shard_topk", "dh_quantize_fp8",
    "dh_forward_fp8w", "dh_quantize4", "dh_forward4", "dh_forward4_debug", "dh_forward4_timed",
    "dh_quantize_c4", "dh_forward_c4_debug", "dh_quantize_g64", "dh_forward_g64_debug",
    "dh_forward_wside_debug",
    "PATH_AUTO", "PATH_WARP", "PATH_TC", "PATH_TC_BF16", "PATH_CORE", "NUM_STAGE_EVENTS", "library_path",
]

PATH_AUTO, PATH_WARP, PATH_TC, PATH_TC_BF16, PATH_CORE = 0, 1, 2, 3, 4
NUM_STAGE_EVENTS = 6
NOALLOC_WORKSPACE_BYTES = 16 << 20
GROUP = 128
BLOCK_N = 64

_STATUS = {0: "DH_OK", -1: "DH_ERR_NULL", -2: "DH_ERR_SHAPE", -3: "DH_ERR_SELECT",
           -4: "DH_ERR_WORKSPACE", -5: "DH_ERR_ALIGN", -6: "DH_ERR_CUDA",
           -7: "DH_ERR_DEVICE_TIMEOUT", -8: "DH_ERR_ARG"}

_lib = None
_lock = threading.Lock()


class DHError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_STATUS.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"CUDA library {_LIB_PATH} is not built; call "
                               "quantised_speculative_draft_gb300.build() first")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.dh_quantize.argtypes = [P, I, I, P, P, P, P]
        lib.dh_quantize.restype = I
        lib.dh_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.dh_workspace_bytes.restype = S
        fwd = [P, P, P, P, P, I, I, I, I, I, I, P, P, P, S]
        lib.dh_forward.argtypes = fwd + [P]
        lib.dh_forward.restype = I
        lib.dh_forward_debug.argtypes = fwd + [P, P, P, P, P, P]
        lib.dh_forward_debug.restype = I
        lib.dh_forward_timed.argtypes = fwd + [P, P]
        lib.dh_forward_timed.restype = I
        lib.dh_forward_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P, P]
        lib.dh_forward_noalloc.restype = I
        lib.dh_set_coarse_path.argtypes = [I]
        lib.dh_set_coarse_path.restype = I
        lib.dh_coarse_path_for.argtypes = [I]
        lib.dh_coarse_path_for.restype = I
        lib.dh_forward_launch_count.argtypes = [I, I, I, I, I]
        lib.dh_forward_launch_count.restype = I
        lib.dh_device_status.argtypes = [I]
        lib.dh_device_status.restype = I
        lib.dh_last_error.argtypes = []
        lib.dh_last_error.restype = ctypes.c_char_p
        lib.dh_version.argtypes = []
        lib.dh_version.restype = I
        L = ctypes.c_longlong
        lib.dh_shard_candidates.argtypes = [P, P, P, P, I, I, I, L, I, I, P, P, P, S, P]
        lib.dh_shard_candidates.restype = I
        lib.dh_shard_rerank_workspace_bytes.argtypes = [I, L, I]
        lib.dh_shard_rerank_workspace_bytes.restype = S
        lib.dh_shard_rerank.argtypes = [P, P, I, I, I, L, P, P, L, I, P, P, P, S, P]
        lib.dh_shard_rerank.restype = I
        lib.dh_shard_topk.argtypes = [P, P, I, I, I, I, P, P, P]
        lib.dh_rerank.restype = I
        lib.dh_rerank.argtypes = [P, P, I, I, I, P, L, P, P]
        lib.dh_shard_topk.restype = I
        lib.dh_quantize_fp8.argtypes = [P, P, I, I, P, P, P, P]
        lib.dh_quantize_fp8.restype = I
        lib.dh_forward_fp8w.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, S, P]
        lib.dh_forward_fp8w.restype = I
        lib.dh_quantize4.argtypes = [P, I, I, P, P, P, P]
        lib.dh_quantize4.restype = I
        lib.dh_forward4.argtypes = fwd + [P]
        lib.dh_forward4.restype = I
        lib.dh_forward4_debug.argtypes = fwd + [P, P, P, P, P, P]
        lib.dh_forward4_debug.restype = I
        lib.dh_forward4_timed.argtypes = fwd + [P, P]
        lib.dh_forward4_timed.restype = I
        lib.dh_quantize_c4.argtypes = [P, I, I, P, P, P, P]
        lib.dh_quantize_c4.restype = I
        lib.dh_forward_c4_debug.argtypes = fwd + [P, P, P, P, P, P, P]
        lib.dh_forward_c4_debug.restype = I
        lib.dh_quantize_g64.argtypes = [P, I, I, P, P, P, P]
        lib.dh_quantize_g64.restype = I
        lib.dh_forward_host.argtypes = fwd + [P]
        lib.dh_forward_host.restype = I
        lib.dh_forward_g64_debug.argtypes = fwd + [P, P, P, P, P, P, P]
        lib.dh_forward_g64_debug.restype = I
        lib.dh_forward_wside_debug.argtypes = fwd + [P, P, P, P, P, P, P]
        lib.dh_forward_wside_debug.restype = I
        _lib = lib
        return lib


def dh_last_error() -> str:
    return _load().dh_last_error().decode()


def _check(rc: int):
    if rc != 0:
        raise DHError(rc, dh_last_error())
    return rc


def _p(t):
    """Device pointer of a tensor (or an int address, or None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dh_version() -> int:
    return _load().dh_version()


def dh_quantize(W, packed, scales, zeros, stream=None):
    """Quantise the bf16 head W [V, H] into packed [V, H/4] u8, scales/zeros [V, H/128] bf16."""
    V, H = W.shape
    _check(_load().dh_quantize(_p(W), V, H, _p(packed), _p(scales), _p(zeros), _stream(stream)))


def dh_workspace_bytes(M: int, H: int, V: int, kcand: int, rerank: int) -> int:
    return int(_load().dh_workspace_bytes(M, H, V, kcand, rerank))


def _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace):
    M, H = x.shape
    V = packed.shape[0]
    nbytes = workspace.numel() * workspace.element_size()
    return [_p(x), _p(packed), _p(scales), _p(zeros), _p(W), M, H, V, kcand, rerank, topk,
            _p(idx), _p(logit), _p(workspace), nbytes]


def dh_forward(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace,
               stream=None):
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    _check(_load().dh_forward(*args, _stream(stream)))


def dh_forward_host(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace,
                    stream=None):
    """dh_forward with x [M, H] bf16, idx [M, topk] int32 and logit [M, topk] fp32 in pinned
    host memory (CPU tensors with ``pin_memory()``); the head and the workspace stay on the
    device.  idx and logit hold the result once the stream has been synchronised."""
    for name, t in (("x", x), ("idx", idx), ("logit", logit)):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous pinned host tensor")
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    _check(_load().dh_forward_host(*args, _stream(stream)))


def dh_forward_debug(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace,
                     coarse=None, cand_val=None, cand_idx=None, sel_idx=None, sel_exact=None,
                     stream=None):
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    _check(_load().dh_forward_debug(*args, _p(coarse), _p(cand_val), _p(cand_idx), _p(sel_idx),
                                    _p(sel_exact), _stream(stream)))


def dh_forward_timed(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace,
                     events, stream=None):
    """``events``: NUM_STAGE_EVENTS torch.cuda.Event objects (created with enable_timing)."""
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    arr = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[e.cuda_event for e in events])
    _check(_load().dh_forward_timed(*args, arr, _stream(stream)))


def dh_forward_noalloc(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit,
                       stream=None):
    """dh_forward without a workspace: scratch is the library's fixed device array
    (NOALLOC_WORKSPACE_BYTES), for callers that cannot allocate device memory."""
    M, H = x.shape
    V = packed.shape[0]
    _check(_load().dh_forward_noalloc(_p(x), _p(packed), _p(scales), _p(zeros), _p(W), M, H, V,
                                      kcand, rerank, topk, _p(idx), _p(logit), _stream(stream)))


def dh_quantize_fp8(W8, row_scale, packed, scales, zeros, stream=None):
    """Quantise an fp8 head: W8 [V, H] e4m3 codes (uint8 or float8_e4m3fn), row_scale [V]
    fp32; outputs as dh_quantize."""
    V, H = W8.shape
    _check(_load().dh_quantize_fp8(_p(W8), _p(row_scale), V, H, _p(packed), _p(scales),
                                   _p(zeros), _stream(stream)))


def dh_forward_fp8w(x, packed, scales, zeros, W8, row_scale, kcand, rerank, topk, idx, logit,
                    workspace, stream=None):
    """dh_forward with the rerank against the fp8 rows W8 [V, H] scaled by row_scale [V]."""
    M, H = x.shape
    V = packed.shape[0]
    nbytes = workspace.numel() * workspace.element_size()
    _check(_load().dh_forward_fp8w(_p(x), _p(packed), _p(scales), _p(zeros), _p(W8),
                                   _p(row_scale), M, H, V, kcand, rerank, topk, _p(idx),
                                   _p(logit), _p(workspace), nbytes, _stream(stream)))


def dh_quantize4(W, packed, scales, zeros, stream=None):
    """Quantise the bf16 head W [V, H] to 4 bits: packed [V, H/2] u8 (half split),
    scales/zeros [V, H/128] bf16."""
    V, H = W.shape
    _check(_load().dh_quantize4(_p(W), V, H, _p(packed), _p(scales), _p(zeros), _stream(stream)))


def dh_forward4(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace,
                stream=None):
    """dh_forward on the 4-bit head (packed [V, H/2] from dh_quantize4)."""
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    _check(_load().dh_forward4(*args, _stream(stream)))


def dh_forward4_debug(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace,
                      coarse=None, cand_val=None, cand_idx=None, sel_idx=None, sel_exact=None,
                      stream=None):
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    _check(_load().dh_forward4_debug(*args, _p(coarse), _p(cand_val), _p(cand_idx), _p(sel_idx),
                                     _p(sel_exact), _stream(stream)))


def dh_forward4_timed(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace,
                      events, stream=None):
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    arr = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[e.cuda_event for e in events])
    _check(_load().dh_forward4_timed(*args, arr, _stream(stream)))


def dh_quantize_c4(W, packed, scales, zeros, stream=None):
    """The 2-bit head in the contiguous-4 layout (the packing ablation): packed [V, H/4]."""
    V, H = W.shape
    _check(_load().dh_quantize_c4(_p(W), V, H, _p(packed), _p(scales), _p(zeros),
                                  _stream(stream)))


def dh_forward_c4_debug(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace,
                        coarse=None, cand_val=None, cand_idx=None, sel_idx=None, sel_exact=None,
                        events=None, stream=None):
    """The forward on the contiguous-4 packing; optional debug outputs and stage events."""
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    arr = None
    if events is not None:
        arr = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[e.cuda_event for e in events])
    _check(_load().dh_forward_c4_debug(*args, _p(coarse), _p(cand_val), _p(cand_idx),
                                       _p(sel_idx), _p(sel_exact), arr, _stream(stream)))


def dh_quantize_g64(W, packed, scales, zeros, stream=None):
    """The 2-bit head with groups of 64 (the group-size ablation): scales/zeros [V, H/64]."""
    V, H = W.shape
    _check(_load().dh_quantize_g64(_p(W), V, H, _p(packed), _p(scales), _p(zeros),
                                   _stream(stream)))


def dh_forward_g64_debug(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit,
                         workspace, coarse=None, cand_val=None, cand_idx=None, sel_idx=None,
                         sel_exact=None, events=None, stream=None):
    """The forward on the 64-group head (M <= 16); optional debug outputs and stage events."""
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    arr = None
    if events is not None:
        arr = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[e.cuda_event for e in events])
    _check(_load().dh_forward_g64_debug(*args, _p(coarse), _p(cand_val), _p(cand_idx),
                                        _p(sel_idx), _p(sel_exact), arr, _stream(stream)))


def dh_forward_wside_debug(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit,
                           workspace, coarse=None, cand_val=None, cand_idx=None, sel_idx=None,
                           sel_exact=None, events=None, stream=None):
    """The forward with the weight-side dequant coarse pass (the scale-placement ablation)."""
    args = _fwd_args(x, packed, scales, zeros, W, kcand, rerank, topk, idx, logit, workspace)
    arr = None
    if events is not None:
        arr = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[e.cuda_event for e in events])
    _check(_load().dh_forward_wside_debug(*args, _p(coarse), _p(cand_val), _p(cand_idx),
                                          _p(sel_idx), _p(sel_exact), arr, _stream(stream)))


def dh_shard_candidates(x, packed, scales, zeros, vocab_offset, kcand, rerank, out_val, out_idx,
                        workspace, stream=None):
    """A vocabulary shard's top-``rerank`` candidates: out_val/out_idx [M, rerank] (global ids)."""
    M, H = x.shape
    Vs = packed.shape[0]
    nbytes = workspace.numel() * workspace.element_size()
    _check(_load().dh_shard_candidates(_p(x), _p(packed), _p(scales), _p(zeros), M, H, Vs,
                                       int(vocab_offset), kcand, rerank, _p(out_val),
                                       _p(out_idx), _p(workspace), nbytes, _stream(stream)))


def dh_shard_rerank_workspace_bytes(M: int, ncand_all: int, rerank: int) -> int:
    return int(_load().dh_shard_rerank_workspace_bytes(M, ncand_all, rerank))


def dh_shard_rerank(x, W_shard, vocab_offset, all_val, all_idx, rerank, sel_idx, exact,
                    workspace, stream=None):
    """Global top-``rerank`` of the gathered lists, exact logits of the ids this shard owns."""
    M, H = x.shape
    Vs = W_shard.shape[0]
    nbytes = workspace.numel() * workspace.element_size()
    _check(_load().dh_shard_rerank(_p(x), _p(W_shard), M, H, Vs, int(vocab_offset), _p(all_val),
                                   _p(all_idx), all_val.shape[1], rerank, _p(sel_idx), _p(exact),
                                   _p(workspace), nbytes, _stream(stream)))


def dh_rerank(x, W, idx, exact, stream=None):
    """Exact logits exact[m, j] = x[m] . W[idx[m, j]] (int32 ids; outside [0, V) -> -inf)."""
    M, H = x.shape
    _check(_load().dh_rerank(_p(x), _p(W), M, H, W.shape[0], _p(idx), idx.shape[1], _p(exact),
                             _stream(stream)))


def dh_shard_topk(exact_parts, sel_idx, topk, idx, logit, stream=None):
    """Merge the ranks' partial exact logits [P, M, rerank] and write the top-``topk``."""
    P, M, R = exact_parts.shape
    _check(_load().dh_shard_topk(_p(exact_parts), _p(sel_idx), P, M, R, topk, _p(idx), _p(logit),
                                 _stream(stream)))


def dh_set_coarse_path(path: int) -> int:
    rc = _load().dh_set_coarse_path(path)
    if rc < 0:
        raise DHError(rc, dh_last_error())
    return rc


def dh_coarse_path_for(M: int) -> int:
    rc = _load().dh_coarse_path_for(M)
    if rc < 0:
        raise DHError(rc, dh_last_error())
    return rc


def dh_forward_launch_count(M: int, H: int, V: int, kcand: int, rerank: int) -> int:
    return int(_load().dh_forward_launch_count(M, H, V, kcand, rerank))


def dh_device_status(reset: bool = False) -> int:
    return _load().dh_device_status(1 if reset else 0)


class DraftHead:
    """A quantised head ready for repeated forwards: owns packed/scales/zeros and a workspace.

    The head weight W stays owned by the caller and is kept by reference (the rerank reads
    it): bf16 [V, H], or e4m3 codes [V, H] (uint8 or float8_e4m3fn) with ``row_scale`` [V]
    fp32 for an fp8 head.  ``bits=4`` builds the 4-bit head (bf16 weight only; the page pairs
    it with ``kcand=1``).
    """

    def __init__(self, W, kcand: int = 8, rerank: int = 32, max_m: int = 128, stream=None,
                 row_scale=None, bits: int = 2):
        import torch
        fp8 = row_scale is not None
        if bits not in (2, 4) or (bits == 4 and fp8):
            raise ValueError("bits must be 2, or 4 with a bf16 weight")
        self.bits = bits
        ok_dtype = W.dtype in (torch.uint8, torch.float8_e4m3fn) if fp8 else \
            W.dtype == torch.bfloat16
        if not ok_dtype or not W.is_cuda or not W.is_contiguous():
            raise ValueError("W must be a contiguous CUDA tensor [V, H]: bf16, or e4m3 codes "
                             "with row_scale")
        if fp8 and (row_scale.dtype != torch.float32 or row_scale.shape != (W.shape[0],)
                    or not row_scale.is_cuda or not row_scale.is_contiguous()):
            raise ValueError("row_scale must be a contiguous fp32 CUDA tensor [V]")
        self.W, self.row_scale = W, row_scale
        self.V, self.H = W.shape
        dev = W.device
        self.packed = torch.empty(self.V, self.H * bits // 8, dtype=torch.uint8, device=dev)
        self.scales = torch.empty(self.V, self.H // GROUP, dtype=torch.bfloat16, device=dev)
        self.zeros = torch.empty(self.V, self.H // GROUP, dtype=torch.bfloat16, device=dev)
        if fp8:
            dh_quantize_fp8(W, row_scale, self.packed, self.scales, self.zeros, stream)
        elif bits == 4:
            dh_quantize4(W, self.packed, self.scales, self.zeros, stream)
        else:
            dh_quantize(W, self.packed, self.scales, self.zeros, stream)
        self.kcand, self.rerank = kcand, rerank
        self._ws = None
        self._ws_key = None

    def workspace(self, M: int):
        import torch
        key = (M, self.kcand, self.rerank)
        if self._ws_key != key:
            n = dh_workspace_bytes(M, self.H, self.V, self.kcand, self.rerank)
            if n == 0:
                raise DHError(-2, dh_last_error())
            self._ws = torch.empty(n, dtype=torch.uint8, device=self.W.device)
            self._ws_key = key
        return self._ws

    def forward(self, x, topk: int = 1, stream=None):
        """x [M, H] bf16 -> (idx int32 [M, topk], logit fp32 [M, topk]).  A pinned host x (the
        bf16 2-bit head) goes through dh_forward_host: the results come back in pinned host
        tensors, complete on return (the stream is synchronised)."""
        import torch
        M = x.shape[0]
        if not x.is_cuda:
            if self.bits == 4 or self.row_scale is not None:
                raise ValueError("a host x is taken by the bf16 2-bit head only")
            idx = torch.empty(M, topk, dtype=torch.int32).pin_memory()
            logit = torch.empty(M, topk, dtype=torch.float32).pin_memory()
            dh_forward_host(x, self.packed, self.scales, self.zeros, self.W, self.kcand,
                            self.rerank, topk, idx, logit, self.workspace(M), stream)
            (torch.cuda.current_stream() if stream is None else stream).synchronize()
            return idx, logit
        idx = torch.empty(M, topk, dtype=torch.int32, device=x.device)
        logit = torch.empty(M, topk, dtype=torch.float32, device=x.device)
        if self.bits == 4:
            dh_forward4(x, self.packed, self.scales, self.zeros, self.W, self.kcand, self.rerank,
                        topk, idx, logit, self.workspace(M), stream)
        elif self.row_scale is not None:
            dh_forward_fp8w(x, self.packed, self.scales, self.zeros, self.W, self.row_scale,
                            self.kcand, self.rerank, topk, idx, logit, self.workspace(M), stream)
        else:
            dh_forward(x, self.packed, self.scales, self.zeros, self.W, self.kcand, self.rerank,
                       topk, idx, logit, self.workspace(M), stream)
        return idx, logit
