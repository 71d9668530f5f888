"""dh_draft_head_argmax: the coarse pass, global top-R, exact rerank and argmax in one call (the
coarse and rerank kernels, validated together), against the oracle and against the two calls
dh_draft_head_coarse_topk + dh_draft_head_rerank_argmax on the same inputs.

Bars: the oracle's (tests/_parity.py); against the two calls, every output bit-identical (the
same kernels in the same order).
"""
import numpy as np
import pytest
import torch

import oracle
from bit_draft_lm_gb300 import build as dh_build
from bit_draft_lm_gb300 import drafthead as dh
from bit_draft_lm_gb300 import synth

from _parity import coarse_tol, dev_bf16, near_tie_rows, rerank_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dh_build.build()
    dh.lib()


def _quant(W_u16, G, bits):
    W = dev_bf16(W_u16)
    f = dh.dh_quantize_pack_int2 if bits == 2 else dh.dh_quantize_pack_int4
    packed, S, ZS = f(W, G)
    return W, packed, S, ZS


def _two_launch(x, W, packed, S, ZS, G, bits, kcand, R):
    M, K = x.shape
    N = W.shape[0]
    ws = dh.new_workspace(M, N, K, kcand, R)
    cv, ci = dh.dh_draft_head_coarse_topk(x, packed, S, ZS, N, G, bits, kcand, workspace=ws)
    rr, rl, am = dh.dh_draft_head_rerank_argmax(x, W, cv, ci, R, workspace=ws)
    torch.cuda.synchronize()
    assert dh.dh_workspace_status(ws) == 0
    return rr, rl, am, cv, ci


def _call(x, W, packed, S, ZS, G, bits, kcand, R, ws=None):
    M, K = x.shape
    N = W.shape[0]
    if ws is None:
        ws = dh.new_workspace(M, N, K, kcand, R)
    out = dh.dh_draft_head_argmax(x, packed, S, ZS, W, G, bits, kcand, R, workspace=ws)
    torch.cuda.synchronize()
    assert dh.dh_workspace_status(ws) == 0
    return out, ws


def _same_as_two_calls(one, two):
    for a, b in zip(one, two):  # rr_id, rr_logit, argmax_id, cand_val, cand_id
        assert torch.equal(a, b)


CASES = [
    # M, K, N, G, bits, kcand, R, seed
    (1, 1024, 8192, 128, 2, 8, 16, 60),      # the small draft head
    (1, 1024, 8232, 128, 2, 8, 32, 61),      # ragged N, R = 32
    (2, 2048, 20000, 64, 2, 4, 16, 62),      # G = 64, two hidden rows
    (4, 1024, 9000, 128, 4, 1, 8, 63),       # int4, KCAND = 1
    (8, 1024, 3000, 128, 2, 8, 4, 64),       # eight hidden rows
    (1, 5120, 124160, 128, 2, 8, 16, 65),    # the vocabulary-scale head
    (12, 1024, 4096, 128, 2, 8, 2, 68),      # two coarse passes
    (24, 2048, 9000, 128, 2, 8, 16, 66),     # the tensor-core coarse pass
]


@pytest.mark.parametrize("M,K,N,G,bits,kcand,R,seed", CASES)
def test_argmax_call_parity(M, K, N, G, bits, kcand, R, seed):
    w = synth.make_workload(M, K, N, seed, plant=N >= 128)
    W, packed, S, ZS = _quant(w.W, G, bits)
    x = dev_bf16(w.x)
    one, _ = _call(x, W, packed, S, ZS, G, bits, kcand, R)
    rr, rl, am, cv, ci = one
    # against the oracle
    op, oS, oZS = oracle.quantize_pack(w.W, G, bits)
    c = oracle.coarse(w.x, op, oS, oZS, G, bits)
    ov, oi = oracle.block_topk(c, kcand)
    o_rr, _ = oracle.global_topr(ov, oi, R)
    e_o = oracle.rerank(w.x, w.W, o_rr)
    o_am = oracle.argmax(e_o, o_rr)
    g_rr = rr.cpu().numpy()
    tol = coarse_tol(c)
    for m in range(M):
        d = g_rr[m] != o_rr[m]
        if d.any():  # only near-tied coarse values may swap at the top-R boundary
            assert np.all(np.abs(c[m, g_rr[m][d]] - c[m, o_rr[m][d]]) <=
                          np.maximum(tol[m, g_rr[m][d]], tol[m, o_rr[m][d]]))
    e_g = oracle.rerank(w.x, w.W, g_rr)
    gl = rl.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gl - e_g) <= rerank_tol(w.x, w.W, g_rr, e_g))
    ok = ~near_tie_rows(e_o)
    assert np.array_equal(am.cpu().numpy()[ok], o_am[ok])
    _same_as_two_calls(one, _two_launch(x, W, packed, S, ZS, G, bits, kcand, R))


def test_argmax_call_padding_slots():
    """N = 70: two blocks, the second with 6 rows, so the top 16 of the 16 slots include its two
    empty slots (-inf, id -1), which score -inf."""
    M, K, N, G, kcand, R = 1, 1024, 70, 128, 8, 16
    w = synth.make_workload(M, K, N, 69, plant=False)
    W, packed, S, ZS = _quant(w.W, G, 2)
    x = dev_bf16(w.x)
    one, _ = _call(x, W, packed, S, ZS, G, 2, kcand, R)
    rr, rl, am, _, _ = one
    ids = [i for i in rr[0].tolist() if i >= 0]
    assert len(ids) == 14 and len(set(ids)) == 14 and set(range(64, 70)) <= set(ids)
    assert bool(torch.all(torch.isneginf(rl[0][rr[0] < 0])))
    _same_as_two_calls(one, _two_launch(x, W, packed, S, ZS, G, 2, kcand, R))
    e = oracle.exact_logits(w.x, w.W)[0]
    assert int(am[0]) == ids[int(np.argmax(e[ids]))]


def test_argmax_call_all_ties():
    """x = 0: every coarse value and every exact logit is 0, so selection falls to the ids: block
    b's candidates are rows 64b .. 64b + 7, the top 16 are blocks 0 and 1's, the argmax is id 0."""
    M, K, N, G, kcand, R = 1, 1024, 8192, 128, 8, 16
    w = synth.make_workload(M, K, N, 70)
    W, packed, S, ZS = _quant(w.W, G, 2)
    x = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    one, _ = _call(x, W, packed, S, ZS, G, 2, kcand, R)
    rr, rl, am, _, _ = one
    assert rr[0].tolist() == list(range(8)) + list(range(64, 72))
    assert bool(torch.all(rl == 0)) and int(am[0]) == 0
    _same_as_two_calls(one, _two_launch(x, W, packed, S, ZS, G, 2, kcand, R))


def test_argmax_call_repeated_and_graph_replay():
    """Back-to-back calls on one workspace give the two calls' results for every new x; a
    captured CUDA graph of the call replays them."""
    M, K, N, G, kcand, R = 1, 2048, 30000, 128, 8, 16
    w = synth.make_workload(M, K, N, 71, plant=True)
    W, packed, S, ZS = _quant(w.W, G, 2)
    ws = dh.new_workspace(M, N, K, kcand, R)
    rng = np.random.default_rng(72)
    outs = [torch.empty(M, R, dtype=torch.int32, device="cuda"),
            torch.empty(M, R, dtype=torch.float32, device="cuda"),
            torch.empty(M, dtype=torch.int32, device="cuda")]
    x = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    for _ in range(4):
        xs = rng.standard_normal((M, K)).astype(np.float32)
        x.copy_(torch.from_numpy(xs).to(torch.bfloat16))
        dh.dh_draft_head_argmax(x, packed, S, ZS, W, G, 2, kcand, R, rr_id=outs[0],
                                rr_logit=outs[1], argmax_id=outs[2], workspace=ws)
        torch.cuda.synchronize()
        two = _two_launch(x, W, packed, S, ZS, G, 2, kcand, R)
        for a, b in zip(outs, two[:3]):
            assert torch.equal(a, b)
    ref = [t.clone() for t in outs]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        dh.dh_draft_head_argmax(x, packed, S, ZS, W, G, 2, kcand, R, rr_id=outs[0],
                                rr_logit=outs[1], argmax_id=outs[2], workspace=ws)
    for t in outs:
        t.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, outs):
        assert torch.equal(a, b)
    assert dh.dh_workspace_status(ws) == 0
