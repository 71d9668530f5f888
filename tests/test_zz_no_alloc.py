"""dh_draft_head_rerank_argmax_noalloc, the rerank + argmax entry point for callers that cannot
allocate device memory (a plug-in handed only its input and output buffers, code inside another
framework's memory pool): instead of a caller workspace it uses a fixed scratch array among the
library's device globals. Through the C ABI, its outputs must agree with the oracle and with
dh_draft_head_rerank_argmax (which takes a caller workspace) on calls in a row, each with other
sizes and candidates so that nothing left in the shared scratch by one call can pass for the
next call's result; one call carries a candidate id past the head, which must score -inf
without disturbing the clean call after it.

This file is named to be collected last: if it fails, a run that stops at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_draft_lm_gb300 import build as dh_build
from bit_draft_lm_gb300 import drafthead as dh
from bit_draft_lm_gb300 import synth

from _parity import bf16_to_f64, dev_bf16, near_tie_rows, rerank_tol, RERANK_ABS, RERANK_RTOL


@pytest.fixture(scope="module")
def lib():
    dh_build.build()
    return dh.lib()


A16 = 0x10000  # a 16-byte aligned fake address: never dereferenced by a refused call


@pytest.mark.parametrize("M,K,N,ncand,R,what", [
    (0, 1024, 8192, 64, 16, "M=0"),
    (5000, 1024, 8192, 64, 16, "M=5000"),
    (1, 1004, 8192, 64, 16, "K=1004"),
    (1, 1024, 8192, 8, 16, "ncand=8"),
    (1, 1024, 8192, 64, 0, "rerank=0"),
    (1, 1024, 8192, 300, 300, "rerank=300"),
])
def test_noalloc_refuses_bad_sizes_before_any_cuda_call(lib, M, K, N, ncand, R, what):
    """Sizes out of range are refused by the argument checks, before the scratch is looked up
    or cleared (the fake addresses are never touched, and no GPU is needed)."""
    rc = lib.dh_draft_head_rerank_argmax_noalloc(A16, M, K, A16, N, A16, A16, ncand, R, A16, A16,
                                                 A16, None, None)
    assert rc in (dh.DH_ERR_SHAPE, dh.DH_ERR_PARAM), what
    assert "noalloc" in dh.dh_last_error()


def test_noalloc_refuses_null_and_misaligned(lib):
    rc = lib.dh_draft_head_rerank_argmax_noalloc(A16, 1, 1024, None, 8192, A16, A16, 64, 16, A16,
                                                 A16, A16, None, None)
    assert rc == dh.DH_ERR_NULL
    rc = lib.dh_draft_head_rerank_argmax_noalloc(A16 + 8, 1, 1024, A16, 8192, A16, A16, 64, 16,
                                                 A16, A16, A16, None, None)
    assert rc == dh.DH_ERR_ALIGN


def _inputs(M, K, N, ncand, seed, bad_id=False):
    rng = np.random.default_rng(seed)
    w = synth.make_workload(M, K, N, seed, plant=False)
    val = rng.standard_normal((M, ncand)).astype(np.float32)
    ids = np.stack([rng.choice(N, ncand, replace=False) for _ in range(M)]).astype(np.int32)
    val[:, -2:] = -np.inf  # empty slots, as short blocks leave them
    ids[:, -2:] = -1
    if bad_id:  # row 0's largest candidate names a row past the head
        j = int(np.argmax(val[0]))
        ids[0, j] = N + 5
    return (w, val, ids, dev_bf16(w.x), dev_bf16(w.W), torch.from_numpy(val).cuda(),
            torch.from_numpy(ids).cuda())


def _oracle(w, val, ids, R):
    """The oracle's top-R, exact logits and argmax; an id past the head scores -inf (the
    library's stated convention for such a slot)."""
    rr, _ = oracle.global_topr(val.astype(np.float64), ids, R)
    safe = np.where(rr >= w.N, -1, rr).astype(np.int32)
    e = oracle.rerank(w.x, w.W, safe)
    return rr, safe, e, oracle.argmax(e, rr)


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_workspace_entry_point(lib):
    # calls in a row, each with other sizes and candidates: a larger one, one with an id past the
    # head (DH_DEV_BAD_ID inside the kernel), then a clean one
    cases = ((8, 5120, 20000, 15520, 16, 60, False),
             (2, 1024, 8192, 3000, 16, 62, True),
             (3, 1024, 8192, 1000, 32, 61, False))
    for M, K, N, ncand, R, seed, bad in cases:
        w, val, ids, x, W, cv, ci = _inputs(M, K, N, ncand, seed, bad)
        ws = dh.new_workspace(M, N, K, 1, R)
        rr0, rl0, am0 = dh.dh_draft_head_rerank_argmax(x, W, cv, ci, R, workspace=ws)
        rr1, rl1, am1 = dh.dh_draft_head_rerank_argmax_noalloc(x, W, cv, ci, R)
        torch.cuda.synchronize()
        # the workspace call reports the bad id in its status word, and only then
        status = dh.dh_workspace_status(ws)
        assert status == (dh.DH_DEV_BAD_ID if bad else 0)
        rr0, rr1 = rr0.cpu().numpy(), rr1.cpu().numpy()
        rl0 = rl0.cpu().numpy().astype(np.float64)
        rl1 = rl1.cpu().numpy().astype(np.float64)
        am0, am1 = am0.cpu().numpy(), am1.cpu().numpy()
        o_rr, safe, e, o_am = _oracle(w, val, ids, R)
        # against the oracle: ids exact, logits within the rerank tolerance, -inf where the oracle
        # has -inf (empty slots and the id past the head), argmax on every non-tied row
        assert np.array_equal(rr1, o_rr)
        fin = np.isfinite(e)
        assert np.array_equal(np.isfinite(rl1), fin)
        if bad:
            assert np.isneginf(rl1[rr1 >= N]).all() and (rr1 >= N).sum() == 1
        tol = rerank_tol(w.x, w.W, safe, e)
        assert np.all(np.abs(rl1[fin] - e[fin]) <= tol[fin])
        ok = ~near_tie_rows(e)
        assert np.array_equal(am1[ok], o_am[ok])
        # against the workspace entry point: the same kernels, so the same values
        assert np.array_equal(rr1, rr0)
        assert np.array_equal(np.isfinite(rl1), np.isfinite(rl0))
        xf, Wf = bf16_to_f64(w.x), bf16_to_f64(w.W)
        absdot = np.array([[np.abs(xf[m] * Wf[n]).sum() if 0 <= n < N else 0.0 for n in rr0[m]]
                           for m in range(M)])
        tol0 = RERANK_RTOL * np.abs(np.where(fin, rl0, 0.0)) + RERANK_ABS * absdot
        assert np.all(np.abs(rl1[fin] - rl0[fin]) <= tol0[fin])
        assert np.array_equal(am1[ok], am0[ok])
