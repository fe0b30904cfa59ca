"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded
inputs.  Quantise/pack must be bit-exact; the forward is judged by the rules in parity.py.
"""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from oracle import oracle as orc

from parity import full_compare, gpu_forward, gpu_quantize, host, check_coarse, rows_compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _inputs(M, H, V, seed=0, **kw):
    wl = synth.custom(M, H, V, **kw)
    return synth.make_x(wl, seed, DEV), synth.make_w(wl, seed, DEV)


def _paths():
    """The coarse paths this build can run: the warp path always, tcgen05 where supported."""
    out = [dh.PATH_WARP]
    for path in (dh.PATH_TC, dh.PATH_TC_BF16):
        prev = dh.dh_set_coarse_path(path)
        try:
            if dh.dh_coarse_path_for(16) == path:
                out.append(path)
        except dh.DHError:
            pass
        finally:
            dh.dh_set_coarse_path(prev)
    return out


# ------------------------------------------------------------------------------------------
# kernel (1): quantise + pack, bit-exact
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("V, H", [(8192, 1024), (1000, 512), (2003, 1536), (4096, 5120), (1, 512)])
def test_quantize_bit_exact(V, H):
    _, W = _inputs(1, H, V, hot_rows=min(V, 37), hot_scale=4.0)
    # edge groups: a constant group, an all-positive group, an all-negative group
    W[0, :128] = 0.25
    if V > 2:
        W[1, 128:256] = W[1, 128:256].abs() + 0.01
        W[2, :128] = -W[2, :128].abs() - 0.01
    packed, S, ZS = gpu_quantize(W)
    torch.cuda.synchronize()
    rp, rS, rZS = orc.quantize(host(W))
    assert np.array_equal(host(packed), rp)
    assert np.array_equal(host(S), rS)
    assert np.array_equal(host(ZS), rZS)


def test_quantize_bit_exact_one_shard_sampled():
    """The one-shard head (124160 x 5120, the pack workload) on sampled rows."""
    wl = synth.shard(16)
    W = synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, wl.V - 1], rng.choice(wl.V, 3000, replace=False)]))
    rows_t = torch.from_numpy(rows).to(DEV)
    rp, rS, rZS = orc.quantize(host(W[rows_t]))
    assert np.array_equal(host(packed[rows_t]), rp)
    assert np.array_equal(host(S[rows_t]), rS)
    assert np.array_equal(host(ZS[rows_t]), rZS)


# ------------------------------------------------------------------------------------------
# forward
# ------------------------------------------------------------------------------------------

def test_forward_tiny_head():
    """M=1, H=1024, V=8192, KCAND=8, RERANK=32, argmax (the tiny workload)."""
    wl = synth.tiny(1)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    for path in _paths():
        rep, gpu, ref = full_compare(x, W, packed, S, ZS, 8, 32, 1, path=path)
        print("tiny", path, rep)


@pytest.mark.parametrize("M, H, V, kcand, rerank, topk", [
    (5, 1024, 8192 + 37, 8, 32, 1),     # ragged tail block of 37
    (13, 512, 3000, 8, 64, 16),         # one span per row, top-k caller
    (16, 1536, 4099, 3, 40, 5),         # tail block of 3 < kcand
    (17, 1024, 2000, 64, 200, 16),      # two batch chunks, whole blocks as candidates
    (33, 1024, 5000, 8, 32, 4),         # three batch chunks
    (1, 512, 70, 64, 70, 7),            # two blocks, rerank everything
    (8, 2048, 1, 1, 1, 1),              # a one-row head
])
def test_forward_ragged(M, H, V, kcand, rerank, topk):
    x, W = _inputs(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    packed, S, ZS = gpu_quantize(W)
    for path in _paths():
        rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, rerank, topk, path=path)
        print((M, H, V, kcand, rerank, topk), path, rep["coarse_worst"], rep["exact_worst"],
              "tie rows", len(rep["ties"]), "differing", sum(t[4] for t in rep["ties"]))


@pytest.mark.parametrize("M, H, V, kcand, rerank, topk", [
    (128, 512, 4096, 64, 32, 32),       # largest batch, whole blocks as candidates, top-k = R
    (2, 1024, 100000 + 13, 8, 32, 32),  # 1563 blocks: ~196 per CTA of the row's cluster
    (4, 512, 64 * 3 + 1, 1, 4, 2),      # four blocks, one candidate each: rerank all
    (6, 1024, 8192, 2, 1, 1),           # RERANK 1
])
def test_forward_fused_selection_edges(M, H, V, kcand, rerank, topk):
    """Sizes at the edges of the one-launch selection + rerank + top-k (RERANK <= 32)."""
    x, W = _inputs(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, rerank, topk)
    print((M, H, V, kcand, rerank, topk), rep["coarse_worst"], rep["exact_worst"],
          "tie rows", len(rep["ties"]))


def test_forward_full_pool_is_the_exact_head():
    """KCAND=64 and RERANK=V rerank every column: the result is the exact bf16 head's top-k."""
    M, H, V, k = 3, 512, 1000, 10
    x, W = _inputs(M, H, V)
    packed, S, ZS = gpu_quantize(W)
    gpu = gpu_forward(x, packed, S, ZS, W, 64, V, k)
    exact = orc.exact_head(host(x), host(W))
    for m in range(M):
        order = np.lexsort((np.arange(V), -exact[m].astype(np.float32)))[:k]
        assert np.array_equal(gpu["idx"][m], order)
        np.testing.assert_allclose(gpu["logit"][m], exact[m, order], rtol=1e-5, atol=1e-5)


def test_forward_zero_input_breaks_ties_by_lower_index():
    """x = 0 makes every coarse and exact value 0: all selections fall to the lower index."""
    M, H, V = 4, 1024, 3000
    _, W = _inputs(M, H, V)
    x = torch.zeros(M, H, dtype=torch.bfloat16, device=DEV)
    packed, S, ZS = gpu_quantize(W)
    gpu = gpu_forward(x, packed, S, ZS, W, 8, 32, 5)
    assert (gpu["idx"] == np.arange(5)[None, :]).all()
    assert (gpu["logit"] == 0).all()


def test_forward_duplicate_rows_tie_to_lower_index():
    """Two identical rows of W have identical coarse and exact values: the lower index wins."""
    M, H, V = 2, 1024, 4096
    x, W = _inputs(M, H, V)
    W[3000] = W[2000]
    x[0] = (W[2000].float() * 40).to(torch.bfloat16)   # steer row 0 onto the twins
    packed, S, ZS = gpu_quantize(W)
    gpu = gpu_forward(x, packed, S, ZS, W, 8, 32, 2)
    assert gpu["idx"][0].tolist() == [2000, 3000]
    assert gpu["logit"][0, 0] == gpu["logit"][0, 1]


def test_forward_is_deterministic_and_graph_capturable():
    M, H, V = 16, 1024, 8192
    x, W = _inputs(M, H, V)
    packed, S, ZS = gpu_quantize(W)
    n = dh.dh_workspace_bytes(M, H, V, 8, 32)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    idx = torch.empty(M, 4, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, 4, dtype=torch.float32, device=DEV)
    dh.dh_forward(x, packed, S, ZS, W, 8, 32, 4, idx, logit, ws)
    torch.cuda.synchronize()
    first = (idx.clone(), logit.clone())
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dh.dh_forward(x, packed, S, ZS, W, 8, 32, 4, idx, logit, ws)
    for _ in range(3):
        idx.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(idx, first[0]) and torch.equal(logit, first[1])


def test_forward_one_shard_head():
    """M=16, H=5120, V=124160 with 512 hot rows (the one-shard memory-bound workload)."""
    wl = synth.shard(16)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    for path in _paths():
        rep, gpu, ref = full_compare(x, W, packed, S, ZS, 8, 32, 1, path=path)
        print("shard", path, rep["coarse_worst"], rep["exact_worst"], rep["ties"])
        exact = orc.exact_head(host(x), host(W))
        recall = np.mean([gpu["idx"][m, 0] == np.argmax(exact[m]) for m in range(16)])
        print("argmax recall vs exact bf16 head:", recall)


@pytest.mark.parametrize("rerank", [32, 64])
def test_forward_topk_caller_full_vocab(rerank):
    """M=16, V=248320, top-16 with RERANK 32/64 (the top-k caller workload)."""
    wl = synth.topk_caller(rerank)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, 8, rerank, 16)
    print("topk", rerank, rep["coarse_worst"], rep["exact_worst"], "tie rows", len(rep["ties"]),
          "differing", sum(t[4] for t in rep["ties"]))
    exact = orc.exact_head(host(x), host(W))
    rec = np.mean([len(set(gpu["idx"][m]) & set(np.argsort(-exact[m])[:16])) / 16
                   for m in range(16)])
    print(f"top-16 recall vs exact bf16 head at RERANK={rerank}: {rec:.3f}")


def test_forward_full_head_m16_full_compare():
    """The headline workload whole: M=16, H=5120, V=248320, KCAND 8, RERANK 32, argmax, on the
    default coarse path; every coarse value, both selections and the result against the
    oracle."""
    wl = synth.full(16)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, 8, 32, 1)
    print("full M=16", rep["coarse_worst"], rep["exact_worst"], "tie rows", len(rep["ties"]),
          "differing", sum(t[4] for t in rep["ties"]))


@pytest.mark.parametrize("wl", [synth.full(72), synth.shard(64)],
                         ids=["full-vocab-M72", "one-shard-M64"])
def test_forward_full_size_sampled(wl):
    """The full-size workloads the oracle cannot run whole in seconds -- M=72 on the full head
    (the largest point of the M sweep) and M=64 on the one-shard head (the compute-bound
    regime): sampled coarse values against the oracle, the selection checked for consistency,
    exact values against the oracle."""
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    gpu = gpu_forward(x, packed, S, ZS, W, 8, 32, 1)
    xb = host(x)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(wl.V, 2000, replace=False),
                                     gpu["sel_idx"].ravel(), [wl.V - 1]]))
    rows_t = torch.from_numpy(rows).to(DEV)
    ref_c = orc.coarse(xb, host(packed[rows_t]), host(S[rows_t]), host(ZS[rows_t]))
    check_coarse(gpu["coarse"][:, rows], ref_c)
    # every candidate's value is its coarse value, and each block's list is its best kcand
    M, V = wl.M, wl.V
    for m in range(0, M, 7):
        for b in rng.choice((V + 63) // 64, 20, replace=False):
            cols = np.arange(64 * b, 64 * b + 64)
            vals = gpu["coarse"][m, cols]
            best = cols[np.lexsort((cols, -vals))][:8]
            assert gpu["cand_idx"][m, b * 8:(b + 1) * 8].tolist() == best.tolist()
    # the reranked set is the best RERANK of the candidates (GPU's own fp32 values)
    for m in range(M):
        cv, ci = gpu["cand_val"][m], gpu["cand_idx"][m]
        top = ci[np.lexsort((ci, -cv))][:32]
        assert set(top.tolist()) == set(gpu["sel_idx"][m].tolist())
    # exact values of the reranked rows, and the result is their argmax
    from parity import check_exact_values
    check_exact_values(gpu, xb, host(W))
    for m in range(M):
        e, i = gpu["sel_exact"][m], gpu["sel_idx"][m]
        assert gpu["idx"][m, 0] == i[np.lexsort((i, -e))][0]
    # four whole batch rows against the oracle's own path: all V coarse values, its block
    # candidates and top-R selection (not the GPU's), the rerank and the argmax
    sample = np.unique(np.linspace(0, M - 1, 4).astype(int))
    rep, _ = rows_compare(gpu, sample, x, W, packed, S, ZS, 8, 32, 1)
    print(wl.name, "rows", sample.tolist(), rep["coarse_worst"],
          "tie rows", len(rep["ties"]))


def test_rerank_entry_on_arbitrary_lists_and_the_whole_vocabulary():
    """dh_rerank: exact logits of arbitrary id lists (repeats, out-of-range ids -> -inf), and
    with every id of a ragged head it is the stock bf16 head, against the oracle."""
    M, H, V = 5, 1536, 3000 + 17
    x, W = _inputs(M, H, V, hot_rows=60, hot_scale=4.0)
    xb, Wb = host(x), host(W)
    rng = np.random.default_rng(3)
    n = 77
    ids = rng.integers(0, V, (M, n)).astype(np.int32)
    ids[:, 5] = ids[:, 4]                       # a repeated id
    ids[0, 10], ids[1, 11], ids[2, 12] = -1, V, 2 ** 31 - 1
    idx = torch.from_numpy(ids).to(DEV)
    ex = torch.full((M, n), float("nan"), dtype=torch.float32, device=DEV)
    dh.dh_rerank(x, W, idx, ex)
    torch.cuda.synchronize()
    g = ex.cpu().numpy()
    bad = (ids < 0) | (ids >= V)
    assert np.isneginf(g[bad]).all()
    e = orc.rerank(xb, Wb, np.where(bad, 0, ids))
    tol = 1e-5 * np.maximum(np.abs(e), 1.0)
    assert (np.abs(g - e)[~bad] <= tol[~bad]).all()
    assert g[0, 5] == g[0, 4]
    # the whole vocabulary: the exact bf16 head
    full = torch.arange(V, dtype=torch.int32, device=DEV).repeat(M, 1).contiguous()
    exf = torch.empty(M, V, dtype=torch.float32, device=DEV)
    dh.dh_rerank(x, W, full, exf)
    torch.cuda.synchronize()
    ref = orc.exact_head(xb, Wb)
    assert (np.abs(exf.cpu().numpy() - ref) <= 1e-5 * np.maximum(np.abs(ref), 1.0)).all()
    with pytest.raises(dh.DHError):
        dh.dh_rerank(x, W, full[:, :0], exf[:, :0])
