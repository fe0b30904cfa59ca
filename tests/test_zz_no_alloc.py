"""dh_forward_noalloc: the forward for callers that cannot allocate device memory (for
example an engine that has already reserved almost all free memory for its KV cache).
It runs on the library's fixed device scratch instead of a caller workspace.

This file is collected last on purpose: if it fails, a run that stops at the first failure has
already run every other test.
"""
import ctypes

import pytest

import quantised_speculative_draft_gb300 as dh


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch():
    """A size whose workspace exceeds the fixed array is refused before anything runs."""
    dh.build()
    lib = dh._load()
    fake = 0x7F0000000000
    need = dh.dh_workspace_bytes(128, 5120, 248320, 8, 32)
    assert need > dh.NOALLOC_WORKSPACE_BYTES
    rc = lib.dh_forward_noalloc(fake, fake, fake, fake, fake, 128, 5120, 248320, 8, 32, 1, fake,
                                fake, None)
    assert rc == -4
    assert "fixed" in dh.dh_last_error()


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_forward_on_two_calls():
    import torch
    from quantised_speculative_draft_gb300 import synth

    dh.build()
    dev = "cuda:0"
    M, H, V, kc, R, k = 16, 5120, 124160, 8, 32, 4
    wl = synth.custom(M, H, V, hot_rows=512, hot_scale=4.0)
    W = synth.make_w(wl, 0, dev)
    xs = [synth.make_x(wl, seed, dev) for seed in (0, 1)]
    assert dh.dh_workspace_bytes(M, H, V, kc, R) <= dh.NOALLOC_WORKSPACE_BYTES
    packed = torch.empty(V, H // 4, dtype=torch.uint8, device=dev)
    S = torch.empty(V, H // 128, dtype=torch.bfloat16, device=dev)
    ZS = torch.empty_like(S)
    dh.dh_quantize(W, packed, S, ZS)

    # the existing entry point, with a caller-owned workspace
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, kc, R), dtype=torch.uint8, device=dev)
    refs = []
    for x in xs:
        idx = torch.empty(M, k, dtype=torch.int32, device=dev)
        logit = torch.empty(M, k, dtype=torch.float32, device=dev)
        dh.dh_forward(x, packed, S, ZS, W, kc, R, k, idx, logit, ws)
        refs.append((idx, logit))

    # two calls in a row through the C ABI on the fixed scratch (the second one finds the
    # first one's leftovers in it)
    lib = dh._load()
    stream = torch.cuda.current_stream().cuda_stream
    for x, (ridx, rlogit) in zip(xs, refs):
        idx = torch.full((M, k), -7, dtype=torch.int32, device=dev)
        logit = torch.full((M, k), float("nan"), dtype=torch.float32, device=dev)
        rc = lib.dh_forward_noalloc(x.data_ptr(), packed.data_ptr(), S.data_ptr(),
                                    ZS.data_ptr(), W.data_ptr(), M, H, V, kc, R, k,
                                    idx.data_ptr(), logit.data_ptr(), ctypes.c_void_p(stream))
        assert rc == 0, dh.dh_last_error()
        torch.cuda.synchronize()
        assert dh.dh_device_status(reset=True) == 0
        # the same kernels on the same inputs: bit for bit, indices and logits
        assert torch.equal(idx, ridx)
        assert torch.equal(logit, rlogit)
